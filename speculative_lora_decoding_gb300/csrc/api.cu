// C-ABI front end: argument checks, workspace layout and kernel launches.
// Nothing here computes a result; every step runs in the CUDA kernels.
#include <algorithm>
#include <atomic>
#include <cstring>

#include "common.cuh"
#include "launch.h"

namespace mlora {

static std::atomic<uint64_t> g_launches{0};
void note_launch() { g_launches.fetch_add(1, std::memory_order_relaxed); }

static int device_sms() {
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
  return sms;
}

static bool aligned(const void *p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

struct LinearLayout {
  size_t plan, T, tw, xs, sk, total;  // tw == 0: no token windows (draft only); sk == 0: no stream-K scratch
};

// Flag words of the stream-K GEMM: the upper half of the counter array.
constexpr size_t SK_FLAGS_OFF = WS_COUNTERS_OFF + 4 * (WS_MAX_COUNTERS / 2);

// Workspace of a layer call with n_slices output slices and K inputs: the
// plan (at the same offset for every call, so one plan serves all of them),
// then T (fp32, one per slice), the token windows of the tensor-core expand
// (one buffer per slice) and the token rows in adapter-sorted order, then
// the stream-K GEMM's partial sums.
static LinearLayout linear_layout(int M, int K, int n_ad, int n_slices, int sms) {
  LinearLayout L;
  const PlanLayout P = plan_layout(M, n_ad);
  size_t o = WS_SCRATCH_OFF;
  L.plan = o;
  o = align_up(o + P.words * 4, 256);
  L.T = o;
  o = align_up(o + (size_t)n_slices * M * T_STRIDE * 4, 256);
  L.tw = 0;
  L.xs = 0;
  if (n_ad > 0) {
    L.tw = o;
    o = align_up(o + (size_t)n_slices * max_window_rows(M, n_ad) * 32, 256);
    L.xs = o;
    o = align_up(o + (size_t)M * K * 2, 256);
  }
  // Partial sums of the stream-K GEMM (one tile's worth per SM).
  L.sk = 0;
  const size_t skb = sk_partial_bytes(M, sms);
  if (skb) {
    L.sk = o;
    o = align_up(o + skb, 256);
  }
  L.total = o;
  return L;
}

// Test knob (mlora_debug_set_flag_wait_ns): nonzero makes the stream-K GEMM's
// tile owners wait that long on flags nothing sets.
static std::atomic<uint32_t> g_test_flag_wait_ns{0};
static std::atomic<int> g_shrink_path{MLORA_SHRINK_AUTO};

// Slice ends: increasing, every one but the last a multiple of 128 (the
// GEMM's tile height), the last equal to N.
static bool slices_ok(int N, int n_slices, const int32_t *slice_end) {
  if (n_slices < 1 || n_slices > MLORA_MAX_SLICES || !slice_end) return false;
  int prev = 0;
  for (int i = 0; i < n_slices; ++i) {
    const int e = slice_end[i];
    if (e <= prev) return false;
    if (i + 1 < n_slices && (e % 128) != 0) return false;
    prev = e;
  }
  return prev == N;
}

static bool linear_sizes_ok(int M, int N, int K, int n_ad) {
  if (M < 1 || M > MLORA_MAX_ROWS || N < 1 || K < 8 || (K % 8) != 0) return false;
  if (n_ad < 0 || n_ad > MLORA_MAX_ADAPTERS) return false;
  if ((long long)((N + 127) / 128) * ((M + 511) / 512) * 4 > (long long)WS_MAX_COUNTERS) return false;
  return true;
}

static mlora_status cuda_status(cudaError_t e) { return e == cudaSuccess ? MLORA_OK : MLORA_ERR_CUDA; }

// Which GEMM kernel a layer call runs.  The cluster split-K kernel wins when
// its tiles fill at least 80% of the SMs in a single wave (70% past 256 rows):
// the weights then stream at the full HBM rate and its on-chip reduction is
// the shortest tail.  Otherwise (a partial last wave, several waves, or idle
// SMs) the persistent stream-K kernel runs, if it can: batches of up to 1024
// rows whose CTAs fit on every SM at once, in verify mode with the token
// windows.  Measured on the 32B block at 640 verify rows: q|k|v (112 cluster
// CTAs in one wave) 100 us on the cluster kernel, 111 us on stream-K; gate|up
// (5.7 cluster waves) 437 us against 377 us on stream-K.
static bool use_stream_k(int M, int N, int K, bool verify, bool have_tw, bool have_sk, int sms, const GemmShape &gs,
                         SkShape *sk_out) {
  // Draft mode (LoRA off) always streams on the stream-K kernel when it
  // fits: measured on the 8B shapes at 64 and 256 rows, o and down (one
  // cluster wave of 84%) took 121 -> 114 us and 158 -> 148 us per pass there.
  bool cluster_good = verify && gs.waves == 1 && (long long)gs.n_units * gs.C * 5 >= (long long)sms * 4;
  // Past 256 rows the cluster kernel keeps up to 512 rows in one token group
  // (two sub-accumulators).  Measured on GB300 at 384 rows (the 32B block at
  // k = 2) it lost to the stream-K kernel's two groups of 192 (q|k|v 100 ->
  // 70 us; o, gate|up and down within 2 us), while at 512 rows (8B o and
  // down: 84 and 137 us against 95 and 143) and at 640 rows it held its own
  // when one wave fills 70% of the SMs.
  if (M > 256)
    cluster_good = M > 384 && verify && gs.waves == 1 && (long long)gs.n_units * gs.C * 10 >= (long long)sms * 7;
  const SkShape sk = sk_shape(M, N, K, sms);
  if (sk_out) *sk_out = sk;
  const bool fits = sk.ok && have_sk && (!verify || have_tw);
  return fits && !cluster_good;
}

// Which shrink writes the verify pass's token windows: the tensor-core tile
// (launch_shrink_mma) or the warp items (launch_shrink), unless a path was
// forced with mlora_set_shrink_path.  Both read each A row from DRAM once;
// the warp items re-read it from L2 once per 4 tokens of its segment, the
// tiles once per unit of 8 blocks, but the tiles use fewer SMs.  Measured on
// GB300 (whole verify call, 640 and 512 rows, K 5120 and 14336): the tiles
// win by 7-21% at rank 64 with 8..128 rows per adapter, lose by 4-44% with
// fewer adapters (too few units to fill the SMs) or at rank 16 (little
// re-reading to save), and by up to 8% with 4 rows per adapter.
static bool shrink_on_tensor_cores(int M, int K, int n_ad, int r_max, int n_slices) {
  const int forced = g_shrink_path.load(std::memory_order_relaxed);
  if (forced == MLORA_SHRINK_WARP) return false;
  if (forced == MLORA_SHRINK_TENSOR) return true;
  (void)K, (void)n_slices;
  const int m_ad = M < n_ad ? M : n_ad;
  const int rows_per_adapter = M / m_ad;
  return r_max >= 64 && M >= 512 && rows_per_adapter >= 8 && rows_per_adapter <= 128;
}

}  // namespace mlora

using namespace mlora;

extern "C" {

size_t mlora_linear_workspace_bytes(int M, int N, int K, int n_adapters) {
  if (!linear_sizes_ok(M, N, K, n_adapters)) return 0;
  int sms = device_sms();
  if (sms <= 0) sms = 160;
  return linear_layout(M, K, n_adapters, 1, sms).total;
}

size_t mlora_linear_sliced_workspace_bytes(int M, int N, int K, int n_adapters, int n_slices) {
  if (!linear_sizes_ok(M, N, K, n_adapters) || n_slices < 1 || n_slices > MLORA_MAX_SLICES) return 0;
  int sms = device_sms();
  if (sms <= 0) sms = 160;
  return linear_layout(M, K, n_adapters, n_slices, sms).total;
}

size_t mlora_accept_workspace_bytes(int B, int k, int V) {
  if (B < 1 || B > (int)WS_MAX_COUNTERS / 2 || k < 1 || k > 16 || V < 1 || V > MLORA_MAX_VOCAB) return 0;
  int sms = device_sms();
  if (sms <= 0) sms = 160;
  return align_up(WS_SCRATCH_OFF + accept_shape(B, k, V, sms).scratch_bytes, 256);
}

mlora_status mlora_workspace_init(void *workspace, size_t ws_bytes, mlora_stream stream) {
  if (!workspace) return MLORA_ERR_WORKSPACE;
  if (ws_bytes < WS_INIT_BYTES || !aligned(workspace, 256)) return MLORA_ERR_WORKSPACE;
  return cuda_status(cudaMemsetAsync(workspace, 0, WS_INIT_BYTES, (cudaStream_t)stream));
}

mlora_status mlora_read_device_status(void *workspace, uint32_t *bits, int clear, mlora_stream stream) {
  if (!workspace || !bits) return MLORA_ERR_ARG;
  cudaStream_t s = (cudaStream_t)stream;
  uint32_t v = 0;
  cudaError_t e = cudaMemcpyAsync(&v, (uint8_t *)workspace + WS_STATUS_OFF, 4, cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess && clear) e = cudaMemsetAsync((uint8_t *)workspace + WS_STATUS_OFF, 0, 4, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return MLORA_ERR_CUDA;
  *bits = v;
  if (v & MLORA_DEV_TIMEOUT) return MLORA_ERR_TIMEOUT;
  return v ? MLORA_ERR_DEVICE_STATUS : MLORA_OK;
}

mlora_status mlora_plan_segments(const int32_t *adapter_idx, int M, const int32_t *rank_of, int n_adapters,
                                 int r_max, void *workspace, size_t ws_bytes, const int32_t **seg_offsets,
                                 const int32_t **perm, mlora_stream stream) {
  if (!adapter_idx || !rank_of) return MLORA_ERR_ARG;
  if (M < 1 || M > MLORA_MAX_ROWS || n_adapters < 1 || n_adapters > MLORA_MAX_ADAPTERS) return MLORA_ERR_SHAPE;
  if (r_max < 8 || r_max > MLORA_MAX_RANK || (r_max % 8) != 0) return MLORA_ERR_SHAPE;
  if (!workspace || !aligned(workspace, 256)) return MLORA_ERR_WORKSPACE;
  const PlanLayout P = plan_layout(M, n_adapters);
  if (ws_bytes < WS_SCRATCH_OFF + P.words * 4) return MLORA_ERR_WORKSPACE;
  int32_t *plan = reinterpret_cast<int32_t *>((uint8_t *)workspace + WS_SCRATCH_OFF);
  uint32_t *status = reinterpret_cast<uint32_t *>((uint8_t *)workspace + WS_STATUS_OFF);
  cudaError_t e = launch_plan(adapter_idx, M, rank_of, n_adapters, r_max, plan, status, (cudaStream_t)stream);
  if (e != cudaSuccess) return MLORA_ERR_CUDA;
  if (seg_offsets) *seg_offsets = plan + P.seg_offsets;
  if (perm) *perm = plan + P.perm;
  return MLORA_OK;
}

mlora_status mlora_shrink(const mlora_bf16 *x, int M, int K, const mlora_bf16 *A_stack, int n_adapters, int r_max,
                          const int32_t *seg_offsets, float *T, void *workspace, size_t ws_bytes,
                          mlora_stream stream) {
  if (!x || !A_stack || !T || !seg_offsets) return MLORA_ERR_ARG;
  if (M < 1 || M > MLORA_MAX_ROWS || K < 8 || (K % 8) != 0 || n_adapters < 1 || n_adapters > MLORA_MAX_ADAPTERS)
    return MLORA_ERR_SHAPE;
  if (r_max < 8 || r_max > MLORA_MAX_RANK || (r_max % 8) != 0) return MLORA_ERR_SHAPE;
  if (!aligned(x, 16) || !aligned(A_stack, 16)) return MLORA_ERR_ARG;
  if (!workspace || !aligned(workspace, 256)) return MLORA_ERR_WORKSPACE;
  const PlanLayout P = plan_layout(M, n_adapters);
  if (ws_bytes < WS_SCRATCH_OFF + P.words * 4) return MLORA_ERR_WORKSPACE;
  int32_t *plan = reinterpret_cast<int32_t *>((uint8_t *)workspace + WS_SCRATCH_OFF);
  if (seg_offsets != plan + P.seg_offsets) return MLORA_ERR_ARG;
  const int sms = device_sms();
  if (sms <= 0) return MLORA_ERR_CUDA;
  cudaError_t e =
      launch_shrink(x, M, K, A_stack, n_adapters, r_max, plan, T, r_max, true, sms, nullptr, 1.f, 1,
                    reinterpret_cast<uint32_t *>((uint8_t *)workspace + WS_STATUS_OFF), (cudaStream_t)stream);
  return cuda_status(e);
}

static mlora_status linear_impl(const mlora_bf16 *x, int M, int K, const mlora_bf16 *W, int N, int n_slices,
                                const int32_t *slice_end, const mlora_bf16 *A_stack, const mlora_bf16 *B_stack,
                                int n_adapters, int r_max, const int32_t *rank_of, const int32_t *adapter_idx,
                                const int32_t *seg_offsets, float scale, int mode, mlora_bf16 *y, void *workspace,
                                size_t ws_bytes, mlora_stream stream) {
  if (!x || !W || !y) return MLORA_ERR_ARG;
  const int prefetch_w = (mode & MLORA_PREFETCH_WEIGHTS) ? 1 : 0;
  const int base_mode = mode & ~MLORA_PREFETCH_WEIGHTS;
  if (base_mode != MLORA_DRAFT && base_mode != MLORA_VERIFY) return MLORA_ERR_ARG;
  const bool verify = base_mode == MLORA_VERIFY;
  if (verify && (!A_stack || !B_stack || !rank_of || !adapter_idx)) return MLORA_ERR_ARG;
  if (!linear_sizes_ok(M, N, K, verify ? n_adapters : 0)) return MLORA_ERR_SHAPE;
  if (!slices_ok(N, n_slices, slice_end)) return MLORA_ERR_SHAPE;
  if (verify && (n_adapters < 1 || r_max < 8 || r_max > MLORA_MAX_RANK || (r_max % 8) != 0)) return MLORA_ERR_SHAPE;
  if (!aligned(x, 16) || !aligned(W, 16)) return MLORA_ERR_ARG;
  if (verify && (!aligned(A_stack, 16) || !aligned(B_stack, 16))) return MLORA_ERR_ARG;
  if (!workspace || !aligned(workspace, 256)) return MLORA_ERR_WORKSPACE;
  const int sms = device_sms();
  if (sms <= 0) return MLORA_ERR_CUDA;
  const int n_ad = verify ? n_adapters : 0;
  const int S = verify ? n_slices : 1;  // the draft pass is one plain GEMM over all slices
  const LinearLayout L = linear_layout(M, K, n_ad, S, sms);
  if (ws_bytes < L.total) return MLORA_ERR_WORKSPACE;

  cudaStream_t s = (cudaStream_t)stream;
  uint8_t *ws = (uint8_t *)workspace;
  uint32_t *status = reinterpret_cast<uint32_t *>(ws + WS_STATUS_OFF);
  int32_t *plan = reinterpret_cast<int32_t *>(ws + L.plan);
  float *T = reinterpret_cast<float *>(ws + L.T);
  uint16_t *tw = L.tw ? reinterpret_cast<uint16_t *>(ws + L.tw) : nullptr;
  uint16_t *xs = L.xs ? reinterpret_cast<uint16_t *>(ws + L.xs) : nullptr;
  cudaError_t e;
  if (verify) {
    const PlanLayout P = plan_layout(M, n_ad);
    if (seg_offsets == nullptr) {
      e = launch_plan(adapter_idx, M, rank_of, n_ad, r_max, plan, status, s);
      if (e != cudaSuccess) return MLORA_ERR_CUDA;
    } else if (seg_offsets != plan + P.seg_offsets) {
      return MLORA_ERR_ARG;
    }
    // Token rows in adapter-sorted order for the GEMM, then T and the
    // windows of the tensor-core expand.
    e = launch_gather_rows(x, M, K, plan + P.perm, xs, sms, status, s);
    if (e != cudaSuccess) return MLORA_ERR_CUDA;
    if (shrink_on_tensor_cores(M, K, n_ad, r_max, S)) {
      e = launch_shrink_mma(xs, M, K, A_stack, n_ad, r_max, plan, tw, scale, S, sms, status, s);
    } else {
      e = launch_shrink(x, M, K, A_stack, n_ad, r_max, plan, T, T_STRIDE, false, sms, tw, scale, S, status, s);
    }
    if (e != cudaSuccess) return MLORA_ERR_CUDA;
  }
  GemmLaunch g;
  g.x = verify ? xs : x;
  g.W = W;
  g.M = M;
  g.N = N;
  g.K = K;
  g.n_slices = S;
  for (int i = 0; i < MLORA_MAX_SLICES; ++i) g.slice_end[i] = (verify && i < S) ? slice_end[i] : N;
  g.mode = base_mode;
  g.prefetch_w = prefetch_w;
  g.after_shrink = verify ? 1 : 0;
  g.scale = scale;
  g.y = y;
  g.B_stack = B_stack;
  g.r_max = r_max;
  g.n_ad = n_ad;
  g.T = T;
  g.plan = plan;
  g.status = status;
  g.tw = verify ? tw : nullptr;
  g.test_flag_wait_ns = g_test_flag_wait_ns.load(std::memory_order_relaxed);
  int err = 0;
  const GemmShape gs = gemm_shape(M, N, K, sms);
  SkShape sk;
  if (use_stream_k(M, N, K, verify, tw != nullptr, L.sk != 0, sms, gs, &sk)) {
    e = launch_gemm_sk(g, sk, reinterpret_cast<float *>(ws + L.sk), reinterpret_cast<uint32_t *>(ws + SK_FLAGS_OFF), s,
                       &err);
  } else {
    e = launch_gemm(g, gs, s, &err);
  }
  if (err) return MLORA_ERR_ARG;
  return cuda_status(e);
}

mlora_status mlora_linear(const mlora_bf16 *x, int M, int K, const mlora_bf16 *W, int N, const mlora_bf16 *A_stack,
                          const mlora_bf16 *B_stack, int n_adapters, int r_max, const int32_t *rank_of,
                          const int32_t *adapter_idx, const int32_t *seg_offsets, float scale, int mode,
                          mlora_bf16 *y, void *workspace, size_t ws_bytes, mlora_stream stream) {
  const int32_t end[1] = {N};
  return linear_impl(x, M, K, W, N, 1, end, A_stack, B_stack, n_adapters, r_max, rank_of, adapter_idx, seg_offsets,
                     scale, mode, y, workspace, ws_bytes, stream);
}

mlora_status mlora_linear_sliced(const mlora_bf16 *x, int M, int K, const mlora_bf16 *W, int N, int n_slices,
                                 const int32_t *slice_end, const mlora_bf16 *A_stack, const mlora_bf16 *B_stack,
                                 int n_adapters, int r_max, const int32_t *rank_of, const int32_t *adapter_idx,
                                 const int32_t *seg_offsets, float scale, int mode, mlora_bf16 *y, void *workspace,
                                 size_t ws_bytes, mlora_stream stream) {
  return linear_impl(x, M, K, W, N, n_slices, slice_end, A_stack, B_stack, n_adapters, r_max, rank_of, adapter_idx,
                     seg_offsets, scale, mode, y, workspace, ws_bytes, stream);
}

int mlora_linear_gemm_kernel(int M, int N, int K, int n_adapters, int r_max, int mode) {
  const int base_mode = mode & ~MLORA_PREFETCH_WEIGHTS;
  if (base_mode != MLORA_DRAFT && base_mode != MLORA_VERIFY) return -1;
  const bool verify = base_mode == MLORA_VERIFY;
  const int n_ad = verify ? n_adapters : 0;
  if (!linear_sizes_ok(M, N, K, n_ad)) return -1;
  if (verify && (n_ad < 1 || r_max < 8 || r_max > MLORA_MAX_RANK || (r_max % 8) != 0)) return -1;
  const int sms = device_sms();
  if (sms <= 0) return -1;
  const LinearLayout L = linear_layout(M, K, n_ad, 1, sms);
  const GemmShape gs = gemm_shape(M, N, K, sms);
  return use_stream_k(M, N, K, verify, L.tw != 0, L.sk != 0, sms, gs, nullptr) ? 1 : 0;
}

void mlora_debug_set_flag_wait_ns(uint32_t ns) { g_test_flag_wait_ns.store(ns, std::memory_order_relaxed); }

mlora_status mlora_debug_q40_mismatches(uint32_t first_bits, uint32_t count, unsigned long long *mismatches,
                                        mlora_stream stream) {
  if (!mismatches || (uint64_t)first_bits + count > (1ull << 32)) return MLORA_ERR_ARG;
  if (count == 0) return MLORA_OK;
  const int sms = device_sms();
  if (sms <= 0) return MLORA_ERR_CUDA;
  return cuda_status(launch_q40_check(first_bits, count, mismatches, sms, (cudaStream_t)stream));
}

mlora_status mlora_debug_exp_max_rel_error(uint32_t first_bits, uint32_t count, unsigned int *max_rel_bits,
                                          mlora_stream stream) {
  if (!max_rel_bits || (uint64_t)first_bits + count > (1ull << 32)) return MLORA_ERR_ARG;
  if (count == 0) return MLORA_OK;
  const int sms = device_sms();
  if (sms <= 0) return MLORA_ERR_CUDA;
  return cuda_status(launch_exp_check(first_bits, count, max_rel_bits, sms, (cudaStream_t)stream));
}

mlora_status mlora_set_shrink_path(int path) {
  if (path != MLORA_SHRINK_AUTO && path != MLORA_SHRINK_WARP && path != MLORA_SHRINK_TENSOR) return MLORA_ERR_ARG;
  g_shrink_path.store(path, std::memory_order_relaxed);
  return MLORA_OK;
}

static mlora_status accept_impl(const float *p, const float *q, const int32_t *draft_tok, const float *uniforms, int B,
                                int k, int V, int32_t *out_tok, int32_t *accepted, void *workspace, size_t ws_bytes,
                                mlora_stream stream, bool logits) {
  if (!p || !q || !draft_tok || !uniforms || !out_tok || !accepted) return MLORA_ERR_ARG;
  // B <= half the counters: the other half holds the stream-K GEMM's flags.
  if (B < 1 || B > (int)WS_MAX_COUNTERS / 2 || k < 1 || k > 16 || V < 1 || V > MLORA_MAX_VOCAB) return MLORA_ERR_SHAPE;
  if (!workspace || !aligned(workspace, 256)) return MLORA_ERR_WORKSPACE;
  const int sms = device_sms();
  if (sms <= 0) return MLORA_ERR_CUDA;
  const AcceptShape sh = accept_shape(B, k, V, sms);
  if (ws_bytes < WS_SCRATCH_OFF + sh.scratch_bytes) return MLORA_ERR_WORKSPACE;
  uint8_t *ws = (uint8_t *)workspace;
  cudaStream_t s = (cudaStream_t)stream;
  float2 *sp = nullptr, *sq = nullptr;
  if (logits) {
    // Row statistics of the target rows followed by the draft rows (sq = sp +
    // B (k + 1)), at most WS_MAX_COUNTERS rows per launch (the block
    // partials' scratch is sized for that many rows).
    sp = reinterpret_cast<float2 *>(ws + WS_SCRATCH_OFF + sh.stats_off);
    sq = sp + (size_t)B * (k + 1);
    void *part = ws + WS_SCRATCH_OFF + sh.part_off;
    const long long Rp = (long long)B * (k + 1), R = Rp + (long long)B * k;
    cudaError_t e = cudaSuccess;
    for (long long r0 = 0; r0 < R && e == cudaSuccess; r0 += (long long)WS_MAX_COUNTERS) {
      const long long r1 = std::min(R, r0 + (long long)WS_MAX_COUNTERS);
      const long long n1 = std::max(0ll, std::min(r1, Rp) - r0);  // target rows of this launch
      const float *z1 = n1 > 0 ? p + (size_t)r0 * V : q + (size_t)(r0 - Rp) * V;
      const long long q0 = std::max(r0, Rp) - Rp;                  // first draft row of this launch
      e = n1 > 0 ? launch_row_stats(z1, (int)n1, q + (size_t)q0 * V, (int)(r1 - r0 - n1), V, sp + r0, part, s)
                 : launch_row_stats(z1, (int)(r1 - r0), nullptr, 0, V, sp + r0, part, s);
    }
    if (e != cudaSuccess) return MLORA_ERR_CUDA;
  }
  cudaError_t e = launch_accept(p, q, draft_tok, uniforms, B, k, V, out_tok, accepted,
                                reinterpret_cast<uint32_t *>(ws + WS_COUNTERS_OFF), ws + WS_SCRATCH_OFF,
                                reinterpret_cast<uint32_t *>(ws + WS_STATUS_OFF), sh, sp, sq, s);
  return cuda_status(e);
}

mlora_status mlora_verify_accept(const float *p_target, const float *q_draft, const int32_t *draft_tok,
                                 const float *uniforms, int B, int k, int V, int32_t *out_tok, int32_t *accepted,
                                 void *workspace, size_t ws_bytes, mlora_stream stream) {
  return accept_impl(p_target, q_draft, draft_tok, uniforms, B, k, V, out_tok, accepted, workspace, ws_bytes, stream,
                     false);
}

mlora_status mlora_verify_accept_logits(const float *z_target, const float *z_draft, const int32_t *draft_tok,
                                        const float *uniforms, int B, int k, int V, int32_t *out_tok,
                                        int32_t *accepted, void *workspace, size_t ws_bytes, mlora_stream stream) {
  return accept_impl(z_target, z_draft, draft_tok, uniforms, B, k, V, out_tok, accepted, workspace, ws_bytes, stream,
                     true);
}

size_t mlora_softmax_workspace_bytes(int rows, int V) {
  if (rows < 1 || rows > MLORA_MAX_ROWS || V < 1 || V > MLORA_MAX_VOCAB) return 0;
  return align_up(WS_SCRATCH_OFF + align_up((size_t)rows * sizeof(float2), 256) + row_stats_scratch_bytes(rows, V),
                  256);
}

mlora_status mlora_softmax(const float *z, int rows, int V, float *p, void *workspace, size_t ws_bytes,
                           mlora_stream stream) {
  if (!z || !p) return MLORA_ERR_ARG;
  if (rows < 1 || rows > MLORA_MAX_ROWS || V < 1 || V > MLORA_MAX_VOCAB) return MLORA_ERR_SHAPE;
  if (!workspace || !aligned(workspace, 256) || ws_bytes < mlora_softmax_workspace_bytes(rows, V))
    return MLORA_ERR_WORKSPACE;
  const int sms = device_sms();
  if (sms <= 0) return MLORA_ERR_CUDA;
  uint8_t *ws = (uint8_t *)workspace;
  float2 *stats = reinterpret_cast<float2 *>(ws + WS_SCRATCH_OFF);
  void *part = ws + WS_SCRATCH_OFF + align_up((size_t)rows * sizeof(float2), 256);
  cudaStream_t s = (cudaStream_t)stream;
  cudaError_t e = launch_row_stats(z, rows, nullptr, 0, V, stats, part, s);
  if (e == cudaSuccess) e = launch_softmax_write(z, rows, V, stats, p, s);
  return cuda_status(e);
}

size_t mlora_draft_sample_workspace_bytes(int B, int V) {
  if (B < 1 || B > (int)WS_MAX_COUNTERS || V < 1 || V > MLORA_MAX_VOCAB) return 0;
  return align_up(WS_SCRATCH_OFF + align_up((size_t)B * sizeof(float2), 256) + draft_sample_scratch_bytes(B, V), 256);
}

mlora_status mlora_draft_sample(const float *z_draft, int B, int V, const float *uniforms, int32_t *draft_tok,
                                float *q_out, void *workspace, size_t ws_bytes, mlora_stream stream) {
  if (!z_draft || !uniforms || !draft_tok) return MLORA_ERR_ARG;
  if (B < 1 || B > (int)WS_MAX_COUNTERS || V < 1 || V > MLORA_MAX_VOCAB) return MLORA_ERR_SHAPE;
  if (!workspace || !aligned(workspace, 256) || ws_bytes < mlora_draft_sample_workspace_bytes(B, V))
    return MLORA_ERR_WORKSPACE;
  const int sms = device_sms();
  if (sms <= 0) return MLORA_ERR_CUDA;
  uint8_t *ws = (uint8_t *)workspace;
  float2 *stats = reinterpret_cast<float2 *>(ws + WS_SCRATCH_OFF);
  void *blk = ws + WS_SCRATCH_OFF + align_up((size_t)B * sizeof(float2), 256);
  cudaError_t e = launch_draft_sample(z_draft, B, V, uniforms, draft_tok, stats, q_out, blk,
                                      reinterpret_cast<uint32_t *>(ws + WS_STATUS_OFF), (cudaStream_t)stream);
  return cuda_status(e);
}

mlora_status mlora_quantize_rows_fp8(const mlora_bf16 *src, int R, int K, uint8_t *q, float *scale,
                                     mlora_stream stream) {
  if (R < 1 || K < 16 || (K % 16) != 0) return MLORA_ERR_SHAPE;
  if (!src || !q || !scale) return MLORA_ERR_ARG;
  if (!aligned(src, 16) || !aligned(q, 16)) return MLORA_ERR_ARG;
  const int sms = device_sms();
  if (sms <= 0) return MLORA_ERR_CUDA;
  return cuda_status(launch_quantize_rows_e4m3((const uint16_t *)src, R, K, q, scale, sms, (cudaStream_t)stream));
}

// Workspace of the FP8 draft layer: the activations' codes and scales, then
// the stream-K GEMM's partial sums.
struct F8Layout {
  size_t x8, xs, sk, total;
};
static F8Layout f8_layout(int M, int K, int sms) {
  F8Layout L;
  size_t o = WS_SCRATCH_OFF;
  L.x8 = o;
  o = align_up(o + (size_t)M * K, 256);
  L.xs = o;
  o = align_up(o + (size_t)M * 4, 256);
  L.sk = o;
  o = align_up(o + sk_partial_bytes(M, sms), 256);
  L.total = o;
  return L;
}

static bool f8_sizes_ok(int M, int N, int K) {
  return M >= 1 && M <= 256 && N >= 1 && K >= 16 && (K % 16) == 0;
}

size_t mlora_linear_fp8_workspace_bytes(int M, int N, int K) {
  if (!f8_sizes_ok(M, N, K)) return 0;
  int sms = device_sms();
  if (sms <= 0) sms = 160;
  return f8_layout(M, K, sms).total;
}

mlora_status mlora_linear_fp8(const mlora_bf16 *x, int M, int K, const uint8_t *W8, const float *w_scale, int N,
                              mlora_bf16 *y, int flags, void *workspace, size_t ws_bytes, mlora_stream stream) {
  if (!f8_sizes_ok(M, N, K)) return MLORA_ERR_SHAPE;
  if (!x || !W8 || !w_scale || !y) return MLORA_ERR_ARG;
  if ((flags & ~MLORA_PREFETCH_WEIGHTS) != 0) return MLORA_ERR_ARG;
  if (!aligned(x, 16) || !aligned(W8, 16)) return MLORA_ERR_ARG;
  if (!workspace || !aligned(workspace, 256)) return MLORA_ERR_WORKSPACE;
  const int sms = device_sms();
  if (sms <= 0) return MLORA_ERR_CUDA;
  const F8Layout L = f8_layout(M, K, sms);
  if (ws_bytes < L.total) return MLORA_ERR_WORKSPACE;
  const SkShape sk = sk_shape(M, N, K, sms, true);
  if (!sk.ok) return MLORA_ERR_UNSUPPORTED;  // a CTA of this shape does not fit on every SM
  uint8_t *ws = (uint8_t *)workspace;
  cudaStream_t s = (cudaStream_t)stream;
  uint8_t *x8 = ws + L.x8;
  float *xs = reinterpret_cast<float *>(ws + L.xs);
  cudaError_t e = launch_quantize_rows_e4m3((const uint16_t *)x, M, K, x8, xs, sms, s);
  if (e != cudaSuccess) return MLORA_ERR_CUDA;
  F8Launch g;
  g.x8 = x8;
  g.W8 = W8;
  g.x_scale = xs;
  g.w_scale = w_scale;
  g.M = M;
  g.N = N;
  g.K = K;
  g.prefetch_w = (flags & MLORA_PREFETCH_WEIGHTS) ? 1 : 0;
  g.y = (uint16_t *)y;
  g.status = reinterpret_cast<uint32_t *>(ws + WS_STATUS_OFF);
  int err = 0;
  e = launch_gemm_sk_f8(g, sk, reinterpret_cast<float *>(ws + L.sk), reinterpret_cast<uint32_t *>(ws + SK_FLAGS_OFF), s,
                        &err);
  if (err) return MLORA_ERR_ARG;
  return cuda_status(e);
}

size_t mlora_kv_workspace_bytes(void) { return WS_INIT_BYTES; }

mlora_status mlora_kv_write(const void *y, int M, int ld, int k_col, int v_col, int H, int D,
                            const int32_t *block_table, int B, int max_blocks, const int32_t *seq_len,
                            int rows_per_req, int t0, void *k_cache, void *v_cache, int num_blocks, int block_size,
                            void *workspace, size_t ws_bytes, mlora_stream stream) {
  if (M < 0 || M > MLORA_MAX_ROWS || B < 1 || B > MLORA_MAX_ROWS || rows_per_req < 1 ||
      (long long)M > (long long)B * rows_per_req || H < 1 || D < 1 || (long long)H * D > (1 << 20) || t0 < 0 ||
      max_blocks < 1 || num_blocks < 1 || block_size < 1 || k_col < 0 || v_col < 0 ||
      (long long)k_col + (long long)H * D > ld || (long long)v_col + (long long)H * D > ld)
    return MLORA_ERR_SHAPE;
  if ((M > 0 && !y) || !block_table || !seq_len || !k_cache || !v_cache) return MLORA_ERR_ARG;  // y may be empty
  if (!workspace || !aligned(workspace, 256) || ws_bytes < mlora_kv_workspace_bytes()) return MLORA_ERR_WORKSPACE;
  const int sms = device_sms();
  if (sms <= 0) return MLORA_ERR_CUDA;
  KvWrite a;
  a.y = (const uint16_t *)y;
  a.M = M;
  a.ld = ld;
  a.k_col = k_col;
  a.v_col = v_col;
  a.HD = H * D;
  a.block_table = block_table;
  a.B = B;
  a.max_blocks = max_blocks;
  a.seq_len = seq_len;
  a.rows_per_req = rows_per_req;
  a.t0 = t0;
  a.k_cache = (uint16_t *)k_cache;
  a.v_cache = (uint16_t *)v_cache;
  a.num_blocks = num_blocks;
  a.block_size = block_size;
  a.status = reinterpret_cast<uint32_t *>((uint8_t *)workspace + WS_STATUS_OFF);
  return cuda_status(launch_kv_write(a, sms, (cudaStream_t)stream));
}

mlora_status mlora_kv_commit(const int32_t *accepted, int B, int32_t *seq_len, mlora_stream stream) {
  if (B < 1 || B > MLORA_MAX_ROWS) return MLORA_ERR_SHAPE;
  if (!accepted || !seq_len) return MLORA_ERR_ARG;
  return cuda_status(launch_kv_commit(accepted, B, seq_len, (cudaStream_t)stream));
}

double mlora_expected_tokens(double alpha, int k) {
  if (k < 0 || !(alpha >= 0.0 && alpha <= 1.0)) return 0.0;
  // 1 + alpha + ... + alpha^k by Horner's rule (stable as alpha -> 1).
  double e = 1.0;
  for (int i = 0; i < k; ++i) e = 1.0 + alpha * e;
  return e;
}

int mlora_draft_gate(const double *t_cycle, int k_max, double t_plain, double alpha, double *gain) {
  if (!t_cycle || k_max < 1 || k_max > 64 || !(t_plain > 0.0) || !(alpha >= 0.0 && alpha <= 1.0)) return -1;
  for (int k = 1; k <= k_max; ++k)
    if (!(t_cycle[k] > 0.0)) return -1;
  int best_k = 0;
  double best_rate = 1.0 / t_plain;
  for (int k = 1; k <= k_max; ++k) {
    const double rate = mlora_expected_tokens(alpha, k) / t_cycle[k];
    if (rate > best_rate) {
      best_k = k;
      best_rate = rate;
    }
  }
  if (gain) *gain = best_rate * t_plain;
  return best_k;
}

double mlora_estimate_acceptance(const int32_t *accepted, int B, int k) {
  if (!accepted || B < 1 || k < 1) return 0.0;
  long long kept = 0, short_ = 0;
  for (int b = 0; b < B; ++b) {
    const int n = accepted[b] < 0 ? 0 : (accepted[b] > k ? k : accepted[b]);
    kept += n;
    short_ += n < k ? 1 : 0;
  }
  return kept + short_ == 0 ? 0.0 : (double)kept / (double)(kept + short_);
}

const char *mlora_status_string(mlora_status s) {
  switch (s) {
    case MLORA_OK: return "ok";
    case MLORA_ERR_ARG: return "invalid argument (null pointer, bad mode or misaligned pointer)";
    case MLORA_ERR_SHAPE: return "size outside the supported range";
    case MLORA_ERR_WORKSPACE: return "workspace missing, too small or misaligned";
    case MLORA_ERR_CUDA: return "CUDA call failed";
    case MLORA_ERR_DEVICE_STATUS: return "device raised status bits (bad input rows were handled by the fallback)";
    case MLORA_ERR_TIMEOUT: return "a bounded wait inside a kernel gave up";
    case MLORA_ERR_UNSUPPORTED: return "device is not supported (needs sm_103)";
  }
  return "unknown status";
}

int mlora_device_supported(void) {
  int dev = 0, major = 0, minor = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess) return 0;
  if (cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess) return 0;
  return (major == 10 && minor == 3) ? 1 : 0;
}

uint64_t mlora_launch_count(void) { return g_launches.load(std::memory_order_relaxed); }

}  // extern "C"
