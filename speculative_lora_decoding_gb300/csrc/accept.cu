// Steps a5 + a6: per-request accept test and residual / bonus draw.
//
// The InvisibleLoRA abstract has one LoRA-on pass verify all drafted tokens
// while keeping the output distribution of plain multi-LoRA decoding.  The
// rule used is standard speculative sampling (Leviathan et al. 2023; Chen et
// al. 2023) with exact arithmetic, so that every decision is reproducible:
//
//   keep draft x_i while (double)u_i * q_i(x_i) < p_i(x_i)       -> n kept
//   w(v) = max(0, Q(p_n(v)) - Q(q_n(v)))  if n < k   (residual)
//   w(v) = Q(p_k(v))                      if n = k   (bonus)      Q(f) = floor(f * 2^40)
//   token = smallest v with sum_{v' <= v} w(v') > floor(U * S / 2^32),
//           S = sum_v w(v), U = floor(u_k * 2^32)
//
// Layout: a request's vocabulary row is cut into chunks of CHUNK = 4096
// entries.  The accept test is repeated wherever a chunk of the request is
// handled (its k gathers hit L2), one lane per draft position.  Because
// almost every draft is accepted, the bonus row p_k is requested before the
// test resolves; when a draft was rejected p_n and q_n are read instead.
// Each chunk's exact uint64 sums (residual mass and target mass) are
// published; the last arrival for a request (atomic counter, no spinning)
// scans the chunk sums, computes the draw, re-reads only the chunk holding it
// and locates the token with prefix scans.  All sums are integers, so the
// order of addition cannot change a result.
//
// Two forms compute this.  The streaming form (rows of 16-byte aligned
// float4, V % 4 == 0) runs one CTA per SM over a contiguous range of
// (request, chunk) units, streaming chunks through a shared-memory ring with
// bulk copies so that each SM keeps 208 KB of reads in flight; it also
// publishes the sums of each 512-entry block, so its draw reads 512 entries.
// The per-chunk form (any V) runs one CTA per (request, chunk), plain loads.
//
// Q(f) = floor(f * 2^40): in the per-chunk form and the draws, one fp32
// multiply (exact: a power-of-two scale of a value in [0, 1]) and one
// conversion rounding toward minus infinity to an unsigned 64-bit integer
// (exact: the scaled value is representable and its integer part is below
// 2^41); in the streaming form's sums, three fused multiply-adds (q_bits).
#include <algorithm>

#include "common.cuh"
#include "launch.h"

namespace mlora {

constexpr int ACC_THREADS = 256;
constexpr int ACC_WARPS = ACC_THREADS / 32;
constexpr int CHUNK = 4096;                       // vocabulary entries per unit
constexpr int PER_THREAD = CHUNK / ACC_THREADS;   // 16 entries per thread (per-chunk form)
constexpr float TWO_POW_32 = 4294967296.0f;
constexpr float TWO_POW_40 = 1099511627776.0f;

__device__ __forceinline__ float sanitize_prob(float f, uint32_t &flags) {
  if (!(f >= 0.f)) {  // NaN or negative
    flags |= MLORA_DEV_BAD_PROB;
    return 0.f;
  }
  if (f > 1.f) {
    flags |= MLORA_DEV_BAD_PROB;
    return 1.f;
  }
  return f;
}

__device__ __forceinline__ float sanitize_uniform(float u, uint32_t &flags) {
  if (!(u >= 0.f)) {
    flags |= MLORA_DEV_BAD_PROB;
    return 0.f;
  }
  if (u >= 1.f) {
    flags |= MLORA_DEV_BAD_PROB;
    return __uint_as_float(0x3F7FFFFFu);  // largest float below 1
  }
  return u;
}

// Clamp to [0, 1] (NaN and negatives to 0) and note an out-of-range value.
__device__ __forceinline__ float clamp_prob(float f, bool &bad) {
  const float c = fminf(fmaxf(f, 0.f), 1.f);  // fmaxf(NaN, 0) = 0
  bad |= !(c == f);
  return c;
}

// Q(f) = floor(f * 2^40) for f in [0, 1].
__device__ __forceinline__ uint64_t fixq(float f) { return __float2ull_rd(f * TWO_POW_40); }

// Logits mode (LG): rows hold logits z and the probability of an entry is
// expf(z - m) / S with the row's statistics st = (m, S) from row_stats, the
// one expression softmax.cu uses everywhere (so the decisions equal the ones
// taken on the probabilities mlora_softmax writes).  Otherwise rows hold
// probabilities and are read as they are.
template <bool LG>
__device__ __forceinline__ float as_prob(float f, float2 st) {
  if (LG) return expf(f - st.x) / st.y;
  return f;
}

__device__ __forceinline__ uint64_t res_weight(uint64_t qp, uint64_t qq) { return qp > qq ? qp - qq : 0ull; }

__device__ __forceinline__ uint64_t warp_sum_u64(uint64_t v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

__device__ __forceinline__ uint64_t warp_incl_scan_u64(uint64_t v) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint64_t t = __shfl_up_sync(0xffffffffu, v, o);
    if (lane >= o) v += t;
  }
  return v;
}

// Exclusive block scan of one uint64 per thread; *total gets the sum.
__device__ __forceinline__ uint64_t block_excl_scan_u64(uint64_t v, uint64_t *sh, uint64_t *total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const uint64_t inc = warp_incl_scan_u64(v);
  if (lane == 31) sh[warp] = inc;
  block_sync();
  uint64_t before = 0, all = 0;
#pragma unroll
  for (int w = 0; w < ACC_WARPS; ++w) {
    const uint64_t t = sh[w];
    if (w < warp) before += t;
    all += t;
  }
  block_sync();
  *total = all;
  return before + inc - v;
}

// The 16 entries thread `tid` covers in the chunk starting at v0: v0 + tid +
// 256 j, j < 16 (each warp load is 128 contiguous bytes).  All loads are
// issued before any value is used.  Entries at or past V read as 0: in
// range, weight 0.
template <bool LG>
__device__ __forceinline__ void load_chunk(const float *row, int v0, int V, int tid, float (&f)[PER_THREAD],
                                           float2 st) {
#pragma unroll
  for (int j = 0; j < PER_THREAD; ++j) {
    const int v = v0 + tid + ACC_THREADS * j;
    f[j] = v < V ? __ldcs(row + v) : 0.f;
  }
  if (LG) {
#pragma unroll
    for (int j = 0; j < PER_THREAD; ++j)
      if (v0 + tid + ACC_THREADS * j < V) f[j] = as_prob<LG>(f[j], st);
  }
}

// Statistics of row `row` (zeros when not in logits mode).
template <bool LG>
__device__ __forceinline__ float2 row_st(const float2 *st, size_t row) {
  if (LG) return st[row];
  return make_float2(0.f, 1.f);
}

template <bool LG>
__global__ void __launch_bounds__(ACC_THREADS)
    accept_kernel(const float *__restrict__ p, const float *__restrict__ q, const int32_t *__restrict__ draft_tok,
                  const float *__restrict__ uni, int B, int k, int V, int chunks,
                  int32_t *__restrict__ out_tok, int32_t *__restrict__ accepted, uint32_t *counters,
                  uint64_t *sums, uint32_t *status, const float2 *__restrict__ sp, const float2 *__restrict__ sq) {
  __shared__ uint64_t sh_scan[ACC_WARPS];
  __shared__ uint64_t sh_red[2][ACC_WARPS];
  __shared__ int sh_n, sh_last, sh_tok, sh_mode, sh_chunk;
  __shared__ uint32_t sh_flags, sh_uflags;
  __shared__ float sh_uk;
  __shared__ uint64_t sh_T, sh_Tloc;

  grid_launch_dependents();
  grid_dependency_wait();
  const int b = blockIdx.x / chunks, c = blockIdx.x % chunks;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int k1 = k + 1;
  const int v0 = c * CHUNK;

  // Speculatively request this chunk of the bonus row p_k.
  float fp[PER_THREAD];
  load_chunk<LG>(p + ((size_t)b * k1 + k) * V, v0, V, tid, fp, row_st<LG>(sp, (size_t)b * k1 + k));

  // Step a5: the accept tests, position i on lane i of warp 0 (k <= 16).
  // The result is what the sequential rule gives: n = the first position
  // whose draft token is out of range or fails u*q < p, or k; flags come
  // from positions up to and including n only.
  if (warp == 0) {
    uint32_t f = 0;
    bool pass = true;
    if (lane < k) {
      const int x = draft_tok[(size_t)b * k + lane];
      if (x < 0 || x >= V) {
        f |= MLORA_DEV_BAD_TOKEN;
        pass = false;
      } else {
        const float pi = sanitize_prob(
            as_prob<LG>(p[((size_t)b * k1 + lane) * V + x], row_st<LG>(sp, (size_t)b * k1 + lane)), f);
        const float qi = sanitize_prob(
            as_prob<LG>(q[((size_t)b * k + lane) * V + x], row_st<LG>(sq, (size_t)b * k + lane)), f);
        const float ui = sanitize_uniform(uni[(size_t)b * k1 + lane], f);
        pass = (double)ui * (double)qi < (double)pi;
      }
    }
    const uint32_t fail = __ballot_sync(0xffffffffu, lane < k && !pass);
    const int n = fail ? __ffs(fail) - 1 : k;
    const uint32_t fl = __reduce_or_sync(0xffffffffu, (lane <= n && lane < k) ? f : 0u);
    if (lane == 0) {
      sh_n = n;
      sh_flags = fl;
    }
    if (lane == k) {  // the draw's uniform, needed by the last CTA only, read early
      uint32_t fu = 0;
      sh_uk = sanitize_uniform(uni[(size_t)b * k1 + k], fu);
      sh_uflags = fu;
    }
  }
  // Step a6, pass 1, on the bonus row while the accept tests resolve: exact
  // sums over this chunk (kept only if every draft was accepted).
  bool bad = false;
  uint64_t s_res = 0, s_tgt = 0;
#pragma unroll
  for (int j = 0; j < PER_THREAD; ++j) s_tgt += fixq(clamp_prob(fp[j], bad));
  block_sync();
  const int n = sh_n;
  const bool residual = n < k;
  if (residual) {
    bad = false;
    s_tgt = 0;
    float fq[PER_THREAD];
    load_chunk<LG>(p + ((size_t)b * k1 + n) * V, v0, V, tid, fp, row_st<LG>(sp, (size_t)b * k1 + n));
    load_chunk<LG>(q + ((size_t)b * k + n) * V, v0, V, tid, fq, row_st<LG>(sq, (size_t)b * k + n));
#pragma unroll
    for (int j = 0; j < PER_THREAD; ++j) {
      const uint64_t qp = fixq(clamp_prob(fp[j], bad));
      const uint64_t qq = fixq(clamp_prob(fq[j], bad));
      s_tgt += qp;
      s_res += res_weight(qp, qq);
    }
  }
  s_res = warp_sum_u64(s_res);
  s_tgt = warp_sum_u64(s_tgt);
  if (lane == 0) {
    sh_red[0][warp] = s_res;
    sh_red[1][warp] = s_tgt;
  }
  if (bad) atomicOr(&sh_flags, MLORA_DEV_BAD_PROB);
  block_sync();
  if (tid == 0) {
    uint64_t a = 0, t = 0;
#pragma unroll
    for (int w = 0; w < ACC_WARPS; ++w) {
      a += sh_red[0][w];
      t += sh_red[1][w];
    }
    const size_t at = ((size_t)b * chunks + c) * 2;
    sums[at + 0] = a;
    sums[at + 1] = t;
    __threadfence();
    const uint32_t old = atomicAdd(&counters[b], 1u);
    sh_last = (old == (uint32_t)(chunks - 1));
  }
  block_sync();
  if (!sh_last) {
    if (tid == 0 && sh_flags) raise_status(status, sh_flags);
    return;
  }

  // Last CTA of this request: scan the chunk sums (vocabulary order), choose
  // the weights and the draw, and find the chunk holding it.
  __threadfence();
  const int per = (chunks + ACC_THREADS - 1) / ACC_THREADS;
  const int c0 = min(chunks, tid * per), c1 = min(chunks, c0 + per);
  uint64_t my_res = 0, my_tgt = 0;
  for (int e = c0; e < c1; ++e) {
    my_res += __ldcg(&sums[((size_t)b * chunks + e) * 2 + 0]);
    my_tgt += __ldcg(&sums[((size_t)b * chunks + e) * 2 + 1]);
  }
  // With one chunk per thread (chunks <= 256) the search below needs no
  // second read of the sums.
  const bool one_each = per == 1;
  uint64_t S_res, S_tgt;
  const uint64_t ex_res = block_excl_scan_u64(my_res, sh_scan, &S_res);
  const uint64_t ex_tgt = block_excl_scan_u64(my_tgt, sh_scan, &S_tgt);
  if (tid == 0) {
    counters[b] = 0u;
    uint32_t f2 = sh_flags;
    int mode = residual ? 0 : 1;  // 0: residual weights, 1: target weights
    if (residual && S_res == 0) {
      f2 |= MLORA_DEV_ZERO_MASS;
      mode = 1;
    }
    const uint64_t S = mode == 0 ? S_res : S_tgt;
    const float uk = sh_uk;
    f2 |= sh_uflags;
    sh_tok = -1;
    sh_chunk = -1;
    if (S == 0) {
      f2 |= MLORA_DEV_ZERO_MASS;
      sh_tok = 0;
    } else {
      const uint64_t U = __float2ull_rz(uk * TWO_POW_32);
      const uint64_t lo = U * S, hi = __umul64hi(U, S);
      sh_T = (hi << 32) | (lo >> 32);  // floor(U * S / 2^32) < S
    }
    sh_mode = mode;
    if (f2) raise_status(status, f2);
  }
  block_sync();
  const int mode = sh_mode;
  if (sh_tok < 0) {
    const uint64_t T = sh_T;
    uint64_t run = mode == 0 ? ex_res : ex_tgt;
    for (int e = c0; e < c1; ++e) {
      const uint64_t w = one_each ? (mode == 0 ? my_res : my_tgt) : __ldcg(&sums[((size_t)b * chunks + e) * 2 + mode]);
      if (run <= T && T < run + w) {
        sh_chunk = e;
        sh_Tloc = T - run;  // the draw inside the chunk; exactly one thread gets here
      }
      run += w;
    }
  }
  block_sync();

  if (sh_tok < 0) {
    // Pass 2: one round over the chosen chunk, a contiguous run of 16
    // entries per thread (entries past V weigh 0).
    const int cv0 = sh_chunk * CHUNK + tid * PER_THREAD;
    const uint64_t T = sh_Tloc;
    const float *prow = p + ((size_t)b * k1 + n) * V;
    const float *qrow = q + ((size_t)b * k + (residual ? n : 0)) * V;
    const bool use_q = mode == 0;
    const float2 stp = row_st<LG>(sp, (size_t)b * k1 + n);
    const float2 stq = row_st<LG>(sq, (size_t)b * k + (residual ? n : 0));
    uint64_t w[PER_THREAD];
    {
      float a[PER_THREAD], bq[PER_THREAD];
#pragma unroll
      for (int j = 0; j < PER_THREAD; ++j) {
        a[j] = cv0 + j < V ? as_prob<LG>(__ldcg(prow + cv0 + j), stp) : 0.f;
        bq[j] = (use_q && cv0 + j < V) ? as_prob<LG>(__ldcg(qrow + cv0 + j), stq) : 0.f;
      }
      bool dummy = false;
#pragma unroll
      for (int j = 0; j < PER_THREAD; ++j) {
        const uint64_t qp = fixq(clamp_prob(a[j], dummy));
        w[j] = use_q ? res_weight(qp, fixq(clamp_prob(bq[j], dummy))) : qp;
      }
    }
    uint64_t mine = 0;
#pragma unroll
    for (int j = 0; j < PER_THREAD; ++j) mine += w[j];
    uint64_t tot;
    uint64_t run = block_excl_scan_u64(mine, sh_scan, &tot);
    if (run <= T && T < run + mine) {
#pragma unroll
      for (int j = 0; j < PER_THREAD; ++j) {
        if (T < run + w[j]) {
          sh_tok = cv0 + j;
          break;
        }
        run += w[j];
      }
    }
  }
  block_sync();
  if (tid == 0) {
    int tok = sh_tok;
    if (tok < 0) tok = 0;  // unreachable when the sums are consistent
    for (int i = 0; i < k1; ++i) {
      int v = -1;
      if (i < n) v = draft_tok[(size_t)b * k + i];
      else if (i == n) v = tok;
      out_tok[(size_t)b * k1 + i] = v;
    }
    accepted[b] = n;
  }
}

// ---------------------------------------------------------------------------
// Streaming form, for rows of 16-byte aligned float4 (V % 4 == 0), in two
// kernels.
//
// accept_stream_kernel: one CTA per SM at most; CTA g owns the units
// (request, chunk) u = g + i G, so a rejected request's reloads spread over
// many SMs.  Warp 8 streams chunks into a ring of RING_STAGES shared-memory
// stages with bulk copies; warps 0-7 run the accept tests of the units'
// requests, then each takes its own 512-entry block of every ring item and
// writes the block's exact sums.  Every wait is on an mbarrier, bounded,
// and taken in order by every thread that takes it (so each parity wait is
// on its current phase).
//
// accept_draw_kernel (programmatic dependent launch, one warp per request):
// the block sums give the totals, the chunk and then the block holding the
// draw; one read of that block's 512 entries finds the token.
// ---------------------------------------------------------------------------
constexpr int RING_STAGES = 14;
constexpr int RING_CONSUMERS = 8;
constexpr int PRODUCER_WARP = RING_CONSUMERS;
constexpr int RING_THREADS = (RING_CONSUMERS + 1) * 32;
constexpr int BLOCK = CHUNK / RING_CONSUMERS;  // 512 entries of an item per consumer warp
constexpr int RING_MAX_UNITS = 128;            // units of one CTA
constexpr int STAGE_FLOATS = CHUNK;
constexpr int DRAW_WARPS = 4;  // small CTAs: they fit beside a streaming CTA while they wait
constexpr uint32_t ONE_BITS = 0x3F800000u;  // bit pattern of 1.0f: every f in [0, 1] has bits <= it
constexpr uint32_t BIAS_BITS = 0x4B000000u; // bit pattern of 2^23

enum : int { ITEM_DISCARD = 0, ITEM_BONUS = 1, ITEM_RESIDUAL = 2 };

struct RingShared {
  uint64_t full[RING_STAGES], empty[RING_STAGES];
  uint64_t a5_done;
  int n[RING_MAX_UNITS];  // accepted count of each unit's request
  int abort_flag, zero_word;
};
constexpr size_t RING_SMEM = (size_t)RING_STAGES * STAGE_FLOATS * 4 + sizeof(RingShared) + 1024;
static_assert(RING_SMEM <= 232448, "ring exceeds the shared memory of a CTA");

// Q(f) = floor(f * 2^40) for f in [0, 1] as hi * 2^23 + lo, with FP32
// operations only: y = 2^23 + floor(f 2^17) (fused multiply-add rounding
// toward minus infinity: the exact sum lies in [2^23, 2^24), where floats
// are the integers), hi = y - 2^23, and z = 2^23 + floor(f 2^40 - hi 2^23)
// (again an exact sum in [2^23, 2^24) rounded down; the addend 2^23 - hi 2^23
// is exact).  The returned pair is the biased bit patterns of y and z: hi =
// bits(y) - bits(2^23), lo = bits(z) - bits(2^23) < 2^23.
struct QBits {
  uint32_t y, z;
};
__device__ __forceinline__ QBits q_bits(float f) {
  const float y = __fmaf_rd(f, 131072.0f, 8388608.0f);
  const float c = __fmaf_rn(-(y - 8388608.0f), 8388608.0f, 8388608.0f);
  const float z = __fmaf_rd(f, TWO_POW_40, c);
  return {__float_as_uint(y), __float_as_uint(z)};
}

__device__ __forceinline__ void ring_abort(RingShared &rs, uint32_t *status) {
  *reinterpret_cast<volatile int *>(&rs.abort_flag) = 1;
  raise_status(status, MLORA_DEV_TIMEOUT);
}

// blk: [B * chunks units][8 blocks][2] uint64 (residual, target);
// n_out: [B] accepted count, written by the unit holding chunk 0.
template <bool LG>
__global__ void __launch_bounds__(RING_THREADS, 1)
    accept_stream_kernel(const float *__restrict__ p, const float *__restrict__ q,
                         const int32_t *__restrict__ draft_tok, const float *__restrict__ uni, int B, int k, int V,
                         int chunks, uint64_t *__restrict__ blk, int32_t *__restrict__ n_out, uint32_t *status,
                         const float2 *__restrict__ sp, const float2 *__restrict__ sq) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t *smem = align_smem_1024(smem_raw);
  float *stages = reinterpret_cast<float *>(smem);
  RingShared &rs = *reinterpret_cast<RingShared *>(smem + (size_t)RING_STAGES * STAGE_FLOATS * 4);

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int k1 = k + 1;
  const int U = B * chunks, G = gridDim.x, g = blockIdx.x;
  const int nU = g < U ? (U - g + G - 1) / G : 0;
  if (nU <= 0) return;
  if (nU > RING_MAX_UNITS) {  // excluded by the host's choice of grid
    if (tid == 0) raise_status(status, MLORA_DEV_TIMEOUT);
    return;
  }
  const int R = min(RING_STAGES, nU);

  if (tid == 0) {
    for (int s = 0; s < RING_STAGES; ++s) {
      mbar_init(&rs.full[s], 1);
      mbar_init(&rs.empty[s], RING_CONSUMERS);
    }
    mbar_init(&rs.a5_done, RING_CONSUMERS);
    rs.abort_flag = 0;
    rs.zero_word = 0;
    fence_mbar_init();
  }
  grid_launch_dependents();
  block_sync();
  grid_dependency_wait();
  volatile int *ab = &rs.abort_flag;

  // The issue order (and the order producer and consumers walk the items
  // in), over this CTA's units i < nU:
  //  1. the bonus chunks of units i < R, before the tests resolve;
  //  2. p_n and q_n chunks of those units whose request was rejected (their
  //     bonus chunks are dropped);
  //  3. units i >= R: the bonus chunk, or p_n and q_n.
  // ITEM_RESIDUAL items take two consecutive slots, the others one.
  auto rejected = [&](int i) { return rs.n[i] < k; };
  auto walk = [&](auto &&f) {
    for (int i = 0; i < R; ++i)
      if (!f(i, rejected(i) ? ITEM_DISCARD : ITEM_BONUS)) return;
    for (int i = 0; i < R; ++i)
      if (rejected(i) && !f(i, ITEM_RESIDUAL)) return;
    for (int i = R; i < nU; ++i)
      if (!f(i, rejected(i) ? ITEM_RESIDUAL : ITEM_BONUS)) return;
  };

  if (warp == PRODUCER_WARP) {
    // Phase 1, lane i: unit i into stage i (no stage is in use yet).
    if (lane < R) {
      const int u = g + lane * G, b = u / chunks, c = u - b * chunks;
      const uint32_t bytes = (uint32_t)min(CHUNK, V - c * CHUNK) * 4u;
      mbar_arrive_expect_tx(&rs.full[lane], bytes);
      bulk_load(stages + (size_t)lane * STAGE_FLOATS, p + ((size_t)b * k1 + k) * V + (size_t)c * CHUNK, bytes,
                &rs.full[lane]);
    }
    if (lane != 0) return;
    int issued = R, st = R == RING_STAGES ? 0 : R;
    uint32_t ph = R == RING_STAGES ? 1u : 0u;
    auto issue = [&](const float *row, int c) -> bool {
      if (issued >= RING_STAGES && !mbar_wait_bounded(&rs.empty[st], ph ^ 1u, ab)) return false;
      const uint32_t bytes = (uint32_t)min(CHUNK, V - c * CHUNK) * 4u;
      mbar_arrive_expect_tx(&rs.full[st], bytes);
      bulk_load(stages + (size_t)st * STAGE_FLOATS, row + (size_t)c * CHUNK, bytes, &rs.full[st]);
      ++issued;
      if (++st == RING_STAGES) {
        st = 0;
        ph ^= 1u;
      }
      return true;
    };
    bool ok = mbar_wait_bounded(&rs.a5_done, 0u, ab);
    if (ok) {
      int item = 0;
      walk([&](int i, int kind) -> bool {
        if (item++ < R) return true;  // phase 1, issued above
        const int u = g + i * G, b = u / chunks, c = u - b * chunks, n = rs.n[i];
        if (kind == ITEM_BONUS) return ok = issue(p + ((size_t)b * k1 + k) * V, c);
        return ok = issue(p + ((size_t)b * k1 + n) * V, c) && issue(q + ((size_t)b * k + n) * V, c);
      });
    }
    if (!ok) ring_abort(rs, status);
    // Copies still in flight land before the CTA may exit.
    for (int s = max(0, issued - RING_STAGES); s < issued; ++s)
      if (!mbar_wait_bounded(&rs.full[s % RING_STAGES], (uint32_t)(s / RING_STAGES) & 1u, &rs.zero_word))
        raise_status(status, MLORA_DEV_TIMEOUT);
    return;
  }

  // Step a5 for every unit's request: kp = k rounded up to a power of two
  // lanes per request, 32 / kp requests per warp and round.
  {
    const int kp = k <= 1 ? 1 : 1 << (32 - __clz(k - 1));
    const int per = 32 / kp, slot = lane / kp, pos = lane % kp;
    for (int i0 = warp * per; i0 < nU; i0 += RING_CONSUMERS * per) {
      const int i = i0 + slot;
      const bool live = i < nU && pos < k;
      uint32_t f = 0;
      bool pass = true;
      int b = 0;
      if (i < nU) b = (g + i * G) / chunks;
      if (live) {
        const int x = draft_tok[(size_t)b * k + pos];
        if (x < 0 || x >= V) {
          f |= MLORA_DEV_BAD_TOKEN;
          pass = false;
        } else {
          const float pi = sanitize_prob(
              as_prob<LG>(p[((size_t)b * k1 + pos) * V + x], row_st<LG>(sp, (size_t)b * k1 + pos)), f);
          const float qi = sanitize_prob(
              as_prob<LG>(q[((size_t)b * k + pos) * V + x], row_st<LG>(sq, (size_t)b * k + pos)), f);
          const float ui = sanitize_uniform(uni[(size_t)b * k1 + pos], f);
          pass = (double)ui * (double)qi < (double)pi;
        }
      }
      // n = the first failing position of this lane's request, else k;
      // flags count from positions up to and including n only.
      const uint32_t fails = __ballot_sync(0xffffffffu, live && !pass);
      const uint32_t mine = kp == 32 ? fails : (fails >> (slot * kp)) & ((1u << kp) - 1u);
      const int n = mine ? __ffs(mine) - 1 : k;
      if (live && pos <= n && f) raise_status(status, f);
      if (i < nU && pos == 0) {
        rs.n[i] = n;
        if ((g + i * G) - b * chunks == 0) n_out[b] = n;
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&rs.a5_done);
  }
  if (!mbar_wait_bounded(&rs.a5_done, 0u, ab)) {
    if (lane == 0) ring_abort(rs, status);
    return;
  }

  // Consumer: this warp's block [512 warp, 512 warp + 512) of every item.
  int st = 0;
  uint32_t ph = 0;
  auto next_stage = [&](int &s, uint32_t &parity) {
    s = st;
    parity = ph;
    if (++st == RING_STAGES) {
      st = 0;
      ph ^= 1u;
    }
  };
  walk([&](int i, int kind) -> bool {
    int s0, s1 = 0;
    uint32_t p0, p1 = 0;
    next_stage(s0, p0);
    const bool resid = kind == ITEM_RESIDUAL;
    if (resid) next_stage(s1, p1);
    bool landed = mbar_wait_bounded(&rs.full[s0], p0, ab);
    if (landed && resid) landed = mbar_wait_bounded(&rs.full[s1], p1, ab);
    if (!__all_sync(0xffffffffu, landed)) {
      if (lane == 0) ring_abort(rs, status);
      return false;
    }
    if (kind == ITEM_DISCARD) {
      __syncwarp();
      if (lane == 0) mbar_arrive(&rs.empty[s0]);
      return true;
    }
    const int u = g + i * G, c = u % chunks;
    const int len4 = min(CHUNK, V - c * CHUNK) / 4;
    const float4 *a4 = reinterpret_cast<const float4 *>(stages + (size_t)s0 * STAGE_FLOATS);
    const float4 *c4 = reinterpret_cast<const float4 *>(stages + (size_t)s1 * STAGE_FLOATS);
    float pa[16], qa[16];
    bool inr[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int e4 = warp * (BLOCK / 4) + lane + 32 * j;  // entries past V read as 0 (weight 0)
      inr[j] = e4 < len4;
      const float4 z4 = make_float4(0.f, 0.f, 0.f, 0.f);
      const float4 a = e4 < len4 ? a4[e4] : z4;
      const float4 cq = (resid && e4 < len4) ? c4[e4] : z4;
      pa[4 * j + 0] = a.x, pa[4 * j + 1] = a.y, pa[4 * j + 2] = a.z, pa[4 * j + 3] = a.w;
      qa[4 * j + 0] = cq.x, qa[4 * j + 1] = cq.y, qa[4 * j + 2] = cq.z, qa[4 * j + 3] = cq.w;
    }
    __syncwarp();
    if (lane == 0) {
      mbar_arrive(&rs.empty[s0]);
      if (resid) mbar_arrive(&rs.empty[s1]);
    }
    if (LG) {
      // Logits to probabilities (entries past V stay 0).
      const int b = u / chunks, prow = resid ? rs.n[i] : k;
      const float2 stp = sp[(size_t)b * k1 + prow];
      const float2 stq = resid ? sq[(size_t)b * k + prow] : make_float2(0.f, 1.f);
#pragma unroll
      for (int e = 0; e < 16; ++e) {
        if (inr[e >> 2]) {
          pa[e] = as_prob<LG>(pa[e], stp);
          if (resid) qa[e] = as_prob<LG>(qa[e], stq);
        }
      }
    }
    uint32_t mx = 0, sy = 0, sz = 0, my = 0, mz = 0;
#pragma unroll
    for (int e = 0; e < 16; ++e) {
      mx = max(mx, __float_as_uint(pa[e]));
      const QBits t = q_bits(pa[e]);
      sy += t.y;
      sz += t.z;
      if (resid) {
        mx = max(mx, __float_as_uint(qa[e]));
        const QBits m = q_bits(fminf(pa[e], qa[e]));  // Q is monotone: Q(min(p, q)) = min(Q(p), Q(q))
        my += m.y;
        mz += m.z;
      }
    }
    uint64_t s_res, s_tgt;
    if (!__any_sync(0xffffffffu, mx > ONE_BITS)) {
      // Per lane the sums of hi stay <= 16 * 2^17 and of lo < 16 * 2^23, so
      // the warp sums stay below 2^32.
      const uint32_t bias16 = 16u * BIAS_BITS;
      s_tgt = ((uint64_t)__reduce_add_sync(0xffffffffu, sy - bias16) << 23) +
              __reduce_add_sync(0xffffffffu, sz - bias16);
      s_res = 0;
      if (resid) {
        const uint64_t s_min = ((uint64_t)__reduce_add_sync(0xffffffffu, my - bias16) << 23) +
                               __reduce_add_sync(0xffffffffu, mz - bias16);
        s_res = s_tgt - s_min;
      }
    } else {
      // An entry outside [0, 1] or NaN: clamp every entry and note it, as the
      // per-chunk form does.
      bool bad = false;
      s_res = 0;
      s_tgt = 0;
#pragma unroll
      for (int e = 0; e < 16; ++e) {
        const uint64_t qp = fixq(clamp_prob(pa[e], bad));
        s_tgt += qp;
        if (resid) s_res += res_weight(qp, fixq(clamp_prob(qa[e], bad)));
      }
      s_res = warp_sum_u64(s_res);
      s_tgt = warp_sum_u64(s_tgt);
      if (__any_sync(0xffffffffu, bad) && lane == 0) raise_status(status, MLORA_DEV_BAD_PROB);
    }
    if (lane == 0) {
      blk[((size_t)u * RING_CONSUMERS + warp) * 2 + 0] = s_res;
      blk[((size_t)u * RING_CONSUMERS + warp) * 2 + 1] = s_tgt;
    }
    return true;
  });
}

// The draw of request b by one warp, from the block sums: the totals, the
// weights (residual, else target), T = floor(U * S / 2^32), the chunk
// holding T (32 chunks per round, lane e summing chunk e's 8 blocks), the
// block within it, then the block's entries, 16 contiguous per lane.
template <bool LG>
__global__ void __launch_bounds__(DRAW_WARPS * 32)
    accept_draw_kernel(const float *__restrict__ p, const float *__restrict__ q,
                       const int32_t *__restrict__ draft_tok, const float *__restrict__ uni, int B, int k, int V,
                       int chunks, const uint64_t *blk, const int32_t *n_in, int32_t *__restrict__ out_tok,
                       int32_t *__restrict__ accepted, uint32_t *status, const float2 *__restrict__ sp,
                       const float2 *__restrict__ sq) {
  grid_launch_dependents();
  grid_dependency_wait();
  const int lane = threadIdx.x & 31;
  const int b = blockIdx.x * DRAW_WARPS + (threadIdx.x >> 5);
  if (b >= B) return;
  const int k1 = k + 1;
  const int n = __ldcg(n_in + b);
  const bool residual = n < k;
  uint32_t fl = 0;
  float uk = 0.f;
  if (lane == 0) uk = sanitize_uniform(uni[(size_t)b * k1 + k], fl);
  int dt = -1;
  if (lane < k) dt = draft_tok[(size_t)b * k + lane];
  const ulonglong2 *bb = reinterpret_cast<const ulonglong2 *>(blk) + (size_t)b * chunks * RING_CONSUMERS;
  // Group 0's block sums stay in registers (chunks <= 32 needs no reload).
  ulonglong2 g0[RING_CONSUMERS];
  uint64_t S_res = 0, S_tgt = 0;
  for (int e0 = 0; e0 < chunks; e0 += 32) {
    const int e = e0 + lane;
    ulonglong2 v[RING_CONSUMERS];
#pragma unroll
    for (int j = 0; j < RING_CONSUMERS; ++j) v[j] = e < chunks ? __ldcg(bb + (size_t)e * RING_CONSUMERS + j) : make_ulonglong2(0, 0);
#pragma unroll
    for (int j = 0; j < RING_CONSUMERS; ++j) {
      S_res += v[j].x;
      S_tgt += v[j].y;
      if (e0 == 0) g0[j] = v[j];
    }
  }
  S_res = warp_sum_u64(S_res);
  S_tgt = warp_sum_u64(S_tgt);
  int mode = residual ? 0 : 1;  // 0: residual weights, 1: target weights
  if (residual && S_res == 0) {
    fl |= MLORA_DEV_ZERO_MASS;
    mode = 1;
  }
  const uint64_t S = mode == 0 ? S_res : S_tgt;
  int tok = 0;
  if (S == 0) {
    fl |= MLORA_DEV_ZERO_MASS;
  } else {
    uk = __shfl_sync(0xffffffffu, uk, 0);
    const uint64_t Ud = __float2ull_rz(uk * TWO_POW_32);
    const uint64_t T = (__umul64hi(Ud, S) << 32) | ((Ud * S) >> 32);  // floor(U * S / 2^32) < S
    int found = -1;
    uint64_t base = 0;
    for (int e0 = 0; e0 < chunks && found < 0; e0 += 32) {
      const int e = e0 + lane;
      ulonglong2 v[RING_CONSUMERS];
#pragma unroll
      for (int j = 0; j < RING_CONSUMERS; ++j)
        v[j] = e0 == 0 ? g0[j] : (e < chunks ? __ldcg(bb + (size_t)e * RING_CONSUMERS + j) : make_ulonglong2(0, 0));
      uint64_t w = 0;
#pragma unroll
      for (int j = 0; j < RING_CONSUMERS; ++j) w += mode == 0 ? v[j].x : v[j].y;
      const uint64_t inc = warp_incl_scan_u64(w);
      uint64_t run = base + inc - w;
      const uint32_t hit = __ballot_sync(0xffffffffu, run <= T && T < run + w);
      if (hit) {
        // The hit lane walks its chunk's 8 blocks.
        const int h = __ffs(hit) - 1;
        int blkid = 0;
        uint64_t Tb = 0;
        if (lane == h) {
          uint64_t t = T - run;
#pragma unroll
          for (int j = 0; j < RING_CONSUMERS; ++j) {
            const uint64_t wj = mode == 0 ? v[j].x : v[j].y;
            if (t < wj) {
              blkid = j;
              Tb = t;
              break;
            }
            t -= wj;
          }
        }
        blkid = __shfl_sync(0xffffffffu, blkid, h);
        Tb = __shfl_sync(0xffffffffu, Tb, h);
        const int chunk = e0 + h;
        const int v0 = chunk * CHUNK + blkid * BLOCK + 16 * lane;  // 16 entries, a multiple of 4
        const bool use_q = mode == 0;
        const float4 *p4 = reinterpret_cast<const float4 *>(p + ((size_t)b * k1 + n) * V + v0);
        const float4 *q4 = reinterpret_cast<const float4 *>(q + ((size_t)b * k + (residual ? n : 0)) * V + v0);
        float a[16], c[16];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const bool in = v0 + 4 * j < V;
          const float4 z4 = make_float4(0.f, 0.f, 0.f, 0.f);
          const float4 t4 = in ? __ldcg(p4 + j) : z4;
          const float4 u4 = (in && use_q) ? __ldcg(q4 + j) : z4;
          a[4 * j + 0] = t4.x, a[4 * j + 1] = t4.y, a[4 * j + 2] = t4.z, a[4 * j + 3] = t4.w;
          c[4 * j + 0] = u4.x, c[4 * j + 1] = u4.y, c[4 * j + 2] = u4.z, c[4 * j + 3] = u4.w;
        }
        if (LG) {
          const float2 stp = sp[(size_t)b * k1 + n];
          const float2 stq = use_q ? sq[(size_t)b * k + n] : make_float2(0.f, 1.f);
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            if (v0 + j < V) {
              a[j] = as_prob<LG>(a[j], stp);
              if (use_q) c[j] = as_prob<LG>(c[j], stq);
            }
          }
        }
        uint64_t wv[16];
        uint64_t mine = 0;
        bool dummy = false;
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          const uint64_t qp = fixq(clamp_prob(a[j], dummy));
          wv[j] = use_q ? res_weight(qp, fixq(clamp_prob(c[j], dummy))) : qp;
          mine += wv[j];
        }
        const uint64_t inc2 = warp_incl_scan_u64(mine);
        uint64_t run2 = inc2 - mine;
        const uint32_t hit2 = __ballot_sync(0xffffffffu, run2 <= Tb && Tb < run2 + mine);
        int t = -1;
        if (hit2 && lane == __ffs(hit2) - 1) {
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            if (t < 0 && Tb < run2 + wv[j]) t = v0 + j;
            run2 += wv[j];
          }
        }
        if (hit2) found = __shfl_sync(0xffffffffu, t, __ffs(hit2) - 1);
        if (found < 0) found = 0;  // unreachable when the sums are consistent
      }
      base += __shfl_sync(0xffffffffu, inc, 31);
    }
    tok = found < 0 ? 0 : found;
  }
  if (lane < k1) {
    int v = -1;
    if (lane < n) v = dt;
    else if (lane == n) v = tok;
    out_tok[(size_t)b * k1 + lane] = v;
  }
  if (lane == 0) {
    accepted[b] = n;
    if (fl) raise_status(status, fl);
  }
}

AcceptShape accept_shape(int B, int k, int V, int num_sms) {
  AcceptShape s;
  s.slice_len = CHUNK;
  s.slices = (V + CHUNK - 1) / CHUNK;
  s.threads = ACC_THREADS;
  // Per-chunk form: chunk sums (residual, target).  Streaming form: the 8
  // block sums of every chunk, then the accepted count of every request.
  const size_t units = (size_t)B * s.slices;
  s.stats_off = units * RING_CONSUMERS * 2 * sizeof(uint64_t) + align_up((size_t)B * 4, 256);
  s.part_off = s.stats_off + align_up((size_t)B * (2 * k + 1) * sizeof(float2), 256);
  const size_t rows_per_launch = std::min((size_t)B * (k + 1), (size_t)WS_MAX_COUNTERS);
  s.scratch_bytes = s.part_off + row_stats_scratch_bytes((int)rows_per_launch, V);
  // Streaming form: one CTA per SM, more when a CTA would own more than
  // RING_MAX_UNITS units.
  long long g = (long long)units < num_sms ? (long long)units : num_sms;
  const long long g_units = ((long long)units + RING_MAX_UNITS - 1) / RING_MAX_UNITS;
  if (g < g_units) g = g_units;
  s.ring_grid = (int)(g > 0 ? g : 1);
  return s;
}

template <bool LG>
static cudaError_t launch_accept_t(const float *p, const float *q, const int32_t *draft_tok, const float *u, int B,
                                   int k, int V, int32_t *out_tok, int32_t *accepted, uint32_t *counters, void *scratch,
                                   uint32_t *status, const AcceptShape &sh, const float2 *sp, const float2 *sq,
                                   cudaStream_t s) {
  const bool vec = ((V & 3) == 0) && ((reinterpret_cast<uintptr_t>(p) & 15) == 0) &&
                   ((reinterpret_cast<uintptr_t>(q) & 15) == 0);
  uint64_t *sums = reinterpret_cast<uint64_t *>(scratch);
  cudaError_t e;
  if (vec) {
    static int attr_done[64] = {0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return cudaErrorInvalidValue;
    if (dev >= 0 && dev < 64 && !attr_done[dev]) {
      e = cudaFuncSetAttribute(accept_stream_kernel<LG>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)RING_SMEM);
      if (e != cudaSuccess) return e;
      attr_done[dev] = 1;
    }
    int32_t *n_buf = reinterpret_cast<int32_t *>(sums + (size_t)B * sh.slices * RING_CONSUMERS * 2);
    e = launch_pdl(accept_stream_kernel<LG>, dim3((unsigned)sh.ring_grid), dim3(RING_THREADS), RING_SMEM, s, p, q,
                   draft_tok, u, B, k, V, sh.slices, sums, n_buf, status, sp, sq);
    if (e != cudaSuccess) return e;
    e = launch_pdl(accept_draw_kernel<LG>, dim3((unsigned)((B + DRAW_WARPS - 1) / DRAW_WARPS)),
                   dim3(DRAW_WARPS * 32), 0, s, p, q, draft_tok, u, B, k, V, sh.slices, (const uint64_t *)sums,
                   (const int32_t *)n_buf, out_tok, accepted, status, sp, sq);
  } else {
    const long long grid = (long long)B * sh.slices;
    e = launch_pdl(accept_kernel<LG>, dim3((unsigned)grid), dim3(ACC_THREADS), 0, s, p, q, draft_tok, u, B, k, V,
                   sh.slices, out_tok, accepted, counters, sums, status, sp, sq);
  }
  return e != cudaSuccess ? e : cudaGetLastError();
}

cudaError_t launch_accept(const float *p, const float *q, const int32_t *draft_tok, const float *u, int B, int k, int V,
                          int32_t *out_tok, int32_t *accepted, uint32_t *counters, void *scratch, uint32_t *status,
                          const AcceptShape &sh, const float2 *stats_p, const float2 *stats_q, cudaStream_t s) {
  if (stats_p && stats_q)
    return launch_accept_t<true>(p, q, draft_tok, u, B, k, V, out_tok, accepted, counters, scratch, status, sh,
                                 stats_p, stats_q, s);
  return launch_accept_t<false>(p, q, draft_tok, u, B, k, V, out_tok, accepted, counters, scratch, status, sh, nullptr,
                                nullptr, s);
}

}  // namespace mlora
