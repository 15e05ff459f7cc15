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
#include "prob.cuh"

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
// prob_from_logit(z, st) with the row's pair st = (m, 1/S) from the row
// statistics, the one expression the softmax uses everywhere (so the
// decisions equal the ones taken on the probabilities mlora_softmax writes).
// Otherwise rows hold probabilities and are read as they are.
template <bool LG>
__device__ __forceinline__ float as_prob(float f, float2 st) {
  if (LG) return prob_from_logit(f, st);
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
// Streaming form, for rows of 16-byte aligned float4 (V % 4 == 0), in three
// kernels chained by programmatic dependent launch.
//
// accept_test_kernel: step a5 for every request (kp = k rounded up to a
// power of two lanes per request, 32 / kp requests per warp): n_out[b] = the
// first rejected position, or k.
//
// accept_blocks_kernel: one CTA of 8 warps per unit (request, 4096-entry
// chunk); warp w sums block w (512 entries, 16 per lane loaded as four
// 16-byte pieces before any is used) of the row the draw needs: p_k (bonus)
// when all k drafts were kept, else p_n and q_n (residual).  Every unit's
// loads are in flight at once across the resident CTAs (no shared-memory
// staging: the latency is hidden by the number of warps, not by a ring), and
// bonus and residual units take separate code paths, so neither issues the
// other's instructions.  Its output: the exact fixed-point sums of each
// block, (residual, target).
//
// accept_draw_kernel (one warp per request): the block sums give the totals,
// the chunk and then the block holding the draw; one read of that block's
// 512 entries finds the token.
// ---------------------------------------------------------------------------
constexpr int BLK_WARPS = 8;
constexpr int BLK_THREADS = BLK_WARPS * 32;
constexpr int BLOCK = CHUNK / BLK_WARPS;  // 512 entries of a unit per warp
constexpr int TEST_THREADS = 256;
constexpr int DRAW_WARPS = 4;
constexpr uint32_t ONE_BITS = 0x3F800000u;  // bit pattern of 1.0f: every f in [0, 1] has bits <= it
constexpr uint32_t BIAS_BITS = 0x4B000000u; // bit pattern of 2^23

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

template <bool LG>
__global__ void __launch_bounds__(TEST_THREADS)
    accept_test_kernel(const float *__restrict__ p, const float *__restrict__ q,
                       const int32_t *__restrict__ draft_tok, const float *__restrict__ uni, int B, int k, int V,
                       int32_t *__restrict__ n_out, uint32_t *status, const float2 *__restrict__ sp,
                       const float2 *__restrict__ sq) {
  grid_launch_dependents();
  grid_dependency_wait();
  const int lane = threadIdx.x & 31;
  const int k1 = k + 1;
  const int kp = k <= 1 ? 1 : 1 << (32 - __clz(k - 1));
  const int per = 32 / kp, slot = lane / kp, pos = lane % kp;
  const int b = (blockIdx.x * TEST_THREADS + threadIdx.x) / 32 * per + slot;
  const bool live = b < B && pos < k;
  uint32_t f = 0;
  bool pass = true;
  if (live) {
    const int x = draft_tok[(size_t)b * k + pos];
    if (x < 0 || x >= V) {
      f |= MLORA_DEV_BAD_TOKEN;
      pass = false;
    } else {
      const float pi =
          sanitize_prob(as_prob<LG>(p[((size_t)b * k1 + pos) * V + x], row_st<LG>(sp, (size_t)b * k1 + pos)), f);
      const float qi =
          sanitize_prob(as_prob<LG>(q[((size_t)b * k + pos) * V + x], row_st<LG>(sq, (size_t)b * k + pos)), f);
      const float ui = sanitize_uniform(uni[(size_t)b * k1 + pos], f);
      pass = (double)ui * (double)qi < (double)pi;
    }
  }
  // n = the first failing position of this lane's request, else k; flags
  // count from positions up to and including n only.
  const uint32_t fails = __ballot_sync(0xffffffffu, live && !pass);
  const uint32_t mine = kp == 32 ? fails : (fails >> (slot * kp)) & ((1u << kp) - 1u);
  const int n = mine ? __ffs(mine) - 1 : k;
  if (live && pos <= n && f) raise_status(status, f);
  if (b < B && pos == 0) n_out[b] = n;
}

// The four 16-byte pieces of lane `lane` in block `w` of the chunk at float4
// index c4 of `row` (entries past V read as 0: weight 0).
template <bool LG>
__device__ __forceinline__ void load_block(const float *row, int c4, int len4, int w, int lane, float (&a)[16],
                                           float2 st) {
  const float4 *r4 = reinterpret_cast<const float4 *>(row) + c4;
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const int e4 = w * (BLOCK / 4) + lane + 32 * j;
    const float4 v = e4 < len4 ? __ldcs(r4 + e4) : make_float4(0.f, 0.f, 0.f, 0.f);
    a[4 * j + 0] = v.x, a[4 * j + 1] = v.y, a[4 * j + 2] = v.z, a[4 * j + 3] = v.w;
  }
  if (LG) {
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      if (w * (BLOCK / 4) + lane + 32 * j < len4) {
#pragma unroll
        for (int i = 0; i < 4; ++i) a[4 * j + i] = as_prob<LG>(a[4 * j + i], st);
      }
    }
  }
}

// blk: [B * chunks units][8 blocks][2] uint64 (residual, target).
template <bool LG>
__global__ void __launch_bounds__(BLK_THREADS)
    accept_blocks_kernel(const float *__restrict__ p, const float *__restrict__ q, int B, int k, int V, int chunks,
                         const int32_t *__restrict__ n_in, uint64_t *__restrict__ blk, uint32_t *status,
                         const float2 *__restrict__ sp, const float2 *__restrict__ sq) {
  grid_launch_dependents();
  grid_dependency_wait();  // the accepted counts come from accept_test_kernel
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  const int k1 = k + 1;
  const int U = B * chunks;
  for (int u = blockIdx.x; u < U; u += gridDim.x) {
    const int b = u / chunks, c = u - b * chunks;
    const int n = __ldcg(n_in + b);
    const bool resid = n < k;
    const int len4 = min(CHUNK, V - c * CHUNK) / 4;
    const size_t prow = (size_t)b * k1 + (resid ? n : k);
    float pa[16];
    uint32_t mx = 0, sy = 0, sz = 0, my = 0, mz = 0;
    if (!resid) {
      load_block<LG>(p + prow * V, c * (CHUNK / 4), len4, w, lane, pa, row_st<LG>(sp, prow));
#pragma unroll
      for (int e = 0; e < 16; ++e) {
        mx = max(mx, __float_as_uint(pa[e]));
        const QBits t = q_bits(pa[e]);
        sy += t.y;
        sz += t.z;
      }
    } else {
      const size_t qrow = (size_t)b * k + n;
      float qa[16];
      load_block<LG>(p + prow * V, c * (CHUNK / 4), len4, w, lane, pa, row_st<LG>(sp, prow));
      load_block<LG>(q + qrow * V, c * (CHUNK / 4), len4, w, lane, qa, row_st<LG>(sq, qrow));
#pragma unroll
      for (int e = 0; e < 16; ++e) {
        mx = max(mx, max(__float_as_uint(pa[e]), __float_as_uint(qa[e])));
        const QBits t = q_bits(pa[e]);
        sy += t.y;
        sz += t.z;
        const QBits m = q_bits(fminf(pa[e], qa[e]));  // Q is monotone: Q(min(p, q)) = min(Q(p), Q(q))
        my += m.y;
        mz += m.z;
      }
      if (__any_sync(0xffffffffu, mx > ONE_BITS)) {
        // An entry outside [0, 1] or NaN: clamp every entry and note it, as
        // the per-chunk form does (here, where qa is in scope).
        bool bad = false;
        uint64_t s_res = 0, s_tgt = 0;
#pragma unroll
        for (int e = 0; e < 16; ++e) {
          const uint64_t qp = fixq(clamp_prob(pa[e], bad));
          s_tgt += qp;
          s_res += res_weight(qp, fixq(clamp_prob(qa[e], bad)));
        }
        s_res = warp_sum_u64(s_res);
        s_tgt = warp_sum_u64(s_tgt);
        if (__any_sync(0xffffffffu, bad) && lane == 0) raise_status(status, MLORA_DEV_BAD_PROB);
        if (lane == 0) {
          blk[((size_t)u * BLK_WARPS + w) * 2 + 0] = s_res;
          blk[((size_t)u * BLK_WARPS + w) * 2 + 1] = s_tgt;
        }
        continue;
      }
    }
    uint64_t s_res = 0, s_tgt = 0;
    if (!__any_sync(0xffffffffu, mx > ONE_BITS)) {
      // Per lane the sums of hi stay <= 16 * 2^17 and of lo < 16 * 2^23, so
      // the warp sums stay below 2^32.
      const uint32_t bias16 = 16u * BIAS_BITS;
      s_tgt = ((uint64_t)__reduce_add_sync(0xffffffffu, sy - bias16) << 23) +
              __reduce_add_sync(0xffffffffu, sz - bias16);
      if (resid) {
        const uint64_t s_min = ((uint64_t)__reduce_add_sync(0xffffffffu, my - bias16) << 23) +
                               __reduce_add_sync(0xffffffffu, mz - bias16);
        s_res = s_tgt - s_min;
      }
    } else {
      // A bonus-row entry outside [0, 1] or NaN: clamp every entry and note
      // it, as the per-chunk form does.
      bool bad = false;
#pragma unroll
      for (int e = 0; e < 16; ++e) s_tgt += fixq(clamp_prob(pa[e], bad));
      s_tgt = warp_sum_u64(s_tgt);
      if (__any_sync(0xffffffffu, bad) && lane == 0) raise_status(status, MLORA_DEV_BAD_PROB);
    }
    if (lane == 0) {
      blk[((size_t)u * BLK_WARPS + w) * 2 + 0] = s_res;
      blk[((size_t)u * BLK_WARPS + w) * 2 + 1] = s_tgt;
    }
  }
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
  const ulonglong2 *bb = reinterpret_cast<const ulonglong2 *>(blk) + (size_t)b * chunks * BLK_WARPS;
  // Group 0's block sums stay in registers (chunks <= 32 needs no reload).
  ulonglong2 g0[BLK_WARPS];
  uint64_t S_res = 0, S_tgt = 0;
  for (int e0 = 0; e0 < chunks; e0 += 32) {
    const int e = e0 + lane;
    ulonglong2 v[BLK_WARPS];
#pragma unroll
    for (int j = 0; j < BLK_WARPS; ++j) v[j] = e < chunks ? __ldcg(bb + (size_t)e * BLK_WARPS + j) : make_ulonglong2(0, 0);
#pragma unroll
    for (int j = 0; j < BLK_WARPS; ++j) {
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
      ulonglong2 v[BLK_WARPS];
#pragma unroll
      for (int j = 0; j < BLK_WARPS; ++j)
        v[j] = e0 == 0 ? g0[j] : (e < chunks ? __ldcg(bb + (size_t)e * BLK_WARPS + j) : make_ulonglong2(0, 0));
      uint64_t w = 0;
#pragma unroll
      for (int j = 0; j < BLK_WARPS; ++j) w += mode == 0 ? v[j].x : v[j].y;
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
          for (int j = 0; j < BLK_WARPS; ++j) {
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
  s.stats_off = units * BLK_WARPS * 2 * sizeof(uint64_t) + align_up((size_t)B * 4, 256);
  s.part_off = s.stats_off + align_up((size_t)B * (2 * k + 1) * sizeof(float2), 256);
  const size_t rows_per_launch = std::min((size_t)B * (2 * k + 1), (size_t)WS_MAX_COUNTERS);
  s.scratch_bytes = s.part_off + row_stats_scratch_bytes((int)rows_per_launch, V);
  // Streaming form: one CTA per unit, up to 64 per SM (a grid-stride loop
  // takes the rest).
  const long long cap = (long long)(num_sms > 0 ? num_sms : 1) * 64;
  const long long g = (long long)units < cap ? (long long)units : cap;
  s.blocks_grid = (int)(g > 0 ? g : 1);
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
    int32_t *n_buf = reinterpret_cast<int32_t *>(sums + (size_t)B * sh.slices * BLK_WARPS * 2);
    const int kp = k <= 1 ? 1 : 1 << (32 - __builtin_clz((unsigned)(k - 1)));
    const long long test_threads = (long long)(B + 32 / kp - 1) / (32 / kp) * 32;
    e = launch_pdl(accept_test_kernel<LG>, dim3((unsigned)((test_threads + TEST_THREADS - 1) / TEST_THREADS)),
                   dim3(TEST_THREADS), 0, s, p, q, draft_tok, u, B, k, V, n_buf, status, sp, sq);
    if (e != cudaSuccess) return e;
    e = launch_pdl(accept_blocks_kernel<LG>, dim3((unsigned)sh.blocks_grid), dim3(BLK_THREADS), 0, s, p, q, B, k, V,
                   sh.slices, (const int32_t *)n_buf, sums, status, sp, sq);
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
