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
// Layout: each request's vocabulary row is cut into `slices` contiguous
// slices, one CTA each, so a small batch still spreads over every SM; each
// slice is cut into one contiguous sub-range per warp.  A warp reads its
// sub-range once (coalesced 16-byte loads) and publishes two exact uint64
// sums (residual mass and target mass).  The last CTA of a request to arrive
// (atomic counter, no spinning) scans the per-warp sums in vocabulary order,
// picks the sub-range holding the draw, re-reads only that sub-range in one
// round (a contiguous run per thread) and locates the token with a block-wide
// prefix scan.  All sums are integers, so the order of addition cannot change
// a result.
#include "common.cuh"
#include "launch.h"

namespace mlora {

constexpr int ACC_THREADS = 256;
constexpr int ACC_WARPS = ACC_THREADS / 32;
constexpr int MIN_SLICE = 4096;
constexpr float TWO_POW_32 = 4294967296.0f;

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

// Q(f) = floor(f * 2^40) for f in [0, 1], from the IEEE-754 fields: a normal
// f is (2^23 + mantissa) * 2^(exponent - 150), so Q(f) is that 24-bit integer
// shifted left by (exponent - 110) or, for smaller exponents, right by
// (110 - exponent) (the right shift is the floor).  Below 2^-40 the result
// is 0; subnormals are far below that.  Integer operations only.
__device__ __forceinline__ uint64_t fixq(float f) {
  const uint32_t bits = __float_as_uint(f);
  const int e = (int)(bits >> 23) & 0xFF;
  const uint32_t m = (bits & 0x7FFFFFu) | 0x800000u;
  const int sh = e - 110;  // e <= 127 for f <= 1, so sh <= 17
  const uint64_t up = (uint64_t)m << (sh > 0 ? sh : 0);
  const uint64_t down = (uint64_t)(m >> min(-sh, 31));  // m < 2^24: shifts of 24 or more give 0
  return sh >= 0 ? up : down;
}

// Clamp to [0, 1] (NaN and negatives to 0) and note whether the value was
// out of range.
__device__ __forceinline__ float clamp_prob(float f, uint32_t &flags) {
  if (!(f >= 0.f && f <= 1.f)) flags |= MLORA_DEV_BAD_PROB;
  return fminf(fmaxf(f, 0.f), 1.f);
}

struct Weights {
  uint64_t res, tgt;
};

__device__ __forceinline__ Weights weight_of(float p, float q, bool residual, uint32_t &flags) {
  Weights w;
  const uint64_t qp = fixq(sanitize_prob(p, flags));
  w.tgt = qp;
  if (residual) {
    const uint64_t qq = fixq(sanitize_prob(q, flags));
    w.res = qp > qq ? qp - qq : 0ull;
  } else {
    w.res = 0ull;
  }
  return w;
}

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

// Exact sums over [w0, w1) of one vocabulary row: the target mass sum Q(p)
// and, when a draft was rejected, the residual mass sum max(0, Q(p) - Q(q)).
// Eight 16-byte loads per operand are in flight per lane before any is used.
template <bool RESIDUAL>
__device__ __forceinline__ void pass1_sums(const float *prow, const float *qrow, int w0, int w1, int lane, int vec,
                                           uint32_t &flags, uint64_t &s_res, uint64_t &s_tgt) {
  auto add = [&](float pf, float qf) {
    const uint64_t qp = fixq(clamp_prob(pf, flags));
    s_tgt += qp;
    if (RESIDUAL) {
      const uint64_t qq = fixq(clamp_prob(qf, flags));
      s_res += qp > qq ? qp - qq : 0ull;
    }
  };
  if (vec) {
    const float4 *p4 = reinterpret_cast<const float4 *>(prow);
    const float4 *q4 = reinterpret_cast<const float4 *>(qrow);
    const int e0 = w0 >> 2, e1 = w1 >> 2;  // w0, V multiples of 4 on this path
    int e = e0 + lane;
    for (; e + 7 * 32 < e1; e += 8 * 32) {
      float4 pv[8], qv[8];
#pragma unroll
      for (int r = 0; r < 8; ++r) {
        pv[r] = __ldcs(p4 + e + 32 * r);
        if (RESIDUAL) qv[r] = __ldcs(q4 + e + 32 * r);
      }
#pragma unroll
      for (int r = 0; r < 8; ++r) {
        add(pv[r].x, RESIDUAL ? qv[r].x : 0.f);
        add(pv[r].y, RESIDUAL ? qv[r].y : 0.f);
        add(pv[r].z, RESIDUAL ? qv[r].z : 0.f);
        add(pv[r].w, RESIDUAL ? qv[r].w : 0.f);
      }
    }
    for (; e < e1; e += 32) {
      const float4 pv = __ldcs(p4 + e);
      const float4 qv = RESIDUAL ? __ldcs(q4 + e) : make_float4(0.f, 0.f, 0.f, 0.f);
      add(pv.x, qv.x);
      add(pv.y, qv.y);
      add(pv.z, qv.z);
      add(pv.w, qv.w);
    }
  } else {
    for (int v = w0 + lane; v < w1; v += 32) add(prow[v], RESIDUAL ? qrow[v] : 0.f);
  }
}

// Vocabulary row of request b: slices of slice_len (one CTA each), each slice
// cut into ACC_WARPS contiguous sub-ranges of sub_len (one warp each).
__global__ void __launch_bounds__(ACC_THREADS)
    accept_kernel(const float *__restrict__ p, const float *__restrict__ q, const int32_t *__restrict__ draft_tok,
                  const float *__restrict__ uni, int B, int k, int V, int slices, int slice_len, int vec,
                  int32_t *__restrict__ out_tok, int32_t *__restrict__ accepted, uint32_t *counters,
                  uint64_t *sums, uint32_t *status) {
  __shared__ uint64_t sh_scan[ACC_WARPS];
  __shared__ int sh_n, sh_last, sh_tok, sh_mode, sh_entry;
  __shared__ uint32_t sh_flags;
  __shared__ uint64_t sh_T, sh_Tloc;

  grid_launch_dependents();
  grid_dependency_wait();
  const int b = blockIdx.x / slices, g = blockIdx.x % slices;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int k1 = k + 1;
  const int sub_len = slice_len / ACC_WARPS;
  uint32_t flags = 0;

  // Step a5: accept tests (cheap gathers; every CTA of the request agrees).
  if (tid == 0) {
    sh_flags = 0;
    int n = k;
    for (int i = 0; i < k; ++i) {
      const int x = draft_tok[(size_t)b * k + i];
      if (x < 0 || x >= V) {
        flags |= MLORA_DEV_BAD_TOKEN;
        n = i;
        break;
      }
      const float pi = sanitize_prob(p[((size_t)b * k1 + i) * V + x], flags);
      const float qi = sanitize_prob(q[((size_t)b * k + i) * V + x], flags);
      const float ui = sanitize_uniform(uni[(size_t)b * k1 + i], flags);
      if (!((double)ui * (double)qi < (double)pi)) {
        n = i;
        break;
      }
    }
    sh_n = n;
  }
  block_sync();
  const int n = sh_n;
  const bool residual = n < k;
  const float *prow = p + ((size_t)b * k1 + n) * V;
  const float *qrow = residual ? q + ((size_t)b * k + n) * V : prow;

  // Step a6, pass 1: exact sums over this warp's sub-range.
  const int w0 = min(V, g * slice_len + warp * sub_len), w1 = min(V, w0 + sub_len);
  uint64_t s_res = 0, s_tgt = 0;
  if (residual)
    pass1_sums<true>(prow, qrow, w0, w1, lane, vec, flags, s_res, s_tgt);
  else
    pass1_sums<false>(prow, qrow, w0, w1, lane, vec, flags, s_res, s_tgt);
  s_res = warp_sum_u64(s_res);
  s_tgt = warp_sum_u64(s_tgt);
  const size_t entries = (size_t)slices * ACC_WARPS;
  if (lane == 0) {
    const size_t at = ((size_t)b * entries + (size_t)g * ACC_WARPS + warp) * 2;
    sums[at + 0] = s_res;
    sums[at + 1] = s_tgt;
    __threadfence();
  }
  if (flags) atomicOr(&sh_flags, flags);
  block_sync();
  if (tid == 0) {
    const uint32_t old = atomicAdd(&counters[b], 1u);
    sh_last = (old == (uint32_t)(slices - 1));
  }
  block_sync();
  if (!sh_last) {
    if (tid == 0 && sh_flags) raise_status(status, sh_flags);
    return;
  }

  // Last CTA of this request: scan the per-warp sums (vocabulary order),
  // choose the weights and the draw, and find the sub-range holding it.
  __threadfence();
  const int per = (int)((entries + ACC_THREADS - 1) / ACC_THREADS);
  const int c0 = min((int)entries, tid * per), c1 = min((int)entries, c0 + per);
  uint64_t my_res = 0, my_tgt = 0;
  for (int c = c0; c < c1; ++c) {
    my_res += __ldcg(&sums[((size_t)b * entries + c) * 2 + 0]);
    my_tgt += __ldcg(&sums[((size_t)b * entries + c) * 2 + 1]);
  }
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
    const float uk = sanitize_uniform(uni[(size_t)b * k1 + k], f2);
    sh_tok = -1;
    sh_entry = -1;
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
    for (int c = c0; c < c1; ++c) {
      const uint64_t w = __ldcg(&sums[((size_t)b * entries + c) * 2 + mode]);
      if (run <= T && T < run + w) {
        sh_entry = c;
        sh_Tloc = T - run;  // the draw inside the entry; exactly one thread gets here
      }
      run += w;
    }
  }
  block_sync();

  if (sh_tok < 0) {
    // Pass 2: one round over the chosen sub-range, a contiguous run per thread.
    const int ent = sh_entry;
    const uint64_t T = sh_Tloc;
    const int gs = ent / ACC_WARPS, ws = ent % ACC_WARPS;
    const int r0 = min(V, gs * slice_len + ws * sub_len), r1 = min(V, r0 + sub_len);
    const int len = r1 - r0;
    const int per2 = (len + ACC_THREADS - 1) / ACC_THREADS;
    const int t0 = min(len, tid * per2), t1 = min(len, t0 + per2);
    uint64_t mine = 0;
    uint32_t dummy = 0;
    for (int v = r0 + t0; v < r0 + t1; ++v) {
      const Weights w = weight_of(prow[v], residual ? qrow[v] : 0.f, mode == 0, dummy);
      mine += mode == 0 ? w.res : w.tgt;
    }
    uint64_t tot;
    uint64_t run = block_excl_scan_u64(mine, sh_scan, &tot);
    if (run <= T && T < run + mine) {
      for (int v = r0 + t0; v < r0 + t1; ++v) {
        const Weights w = weight_of(prow[v], residual ? qrow[v] : 0.f, mode == 0, dummy);
        const uint64_t wv = mode == 0 ? w.res : w.tgt;
        if (T < run + wv) {
          sh_tok = v;
          break;
        }
        run += wv;
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

AcceptShape accept_shape(int B, int k, int V, int num_sms) {
  (void)k;
  AcceptShape s;
  int want = (2 * num_sms + B - 1) / B;  // about two CTAs per SM
  const int max_slices = (V + MIN_SLICE - 1) / MIN_SLICE;
  if (want > max_slices) want = max_slices;
  if (want < 1) want = 1;
  const int quantum = 4 * ACC_WARPS;  // every warp sub-range starts on a float4
  int len = (V + want - 1) / want;
  len = (len + quantum - 1) / quantum * quantum;
  s.slice_len = len;
  s.slices = (V + len - 1) / len;
  s.threads = ACC_THREADS;
  s.scratch_bytes = (size_t)B * s.slices * ACC_WARPS * 2 * sizeof(uint64_t);
  return s;
}

cudaError_t launch_accept(const float *p, const float *q, const int32_t *draft_tok, const float *u, int B, int k, int V,
                          int32_t *out_tok, int32_t *accepted, uint32_t *counters, void *scratch, uint32_t *status,
                          const AcceptShape &sh, cudaStream_t s) {
  const int vec = ((V & 3) == 0) && ((reinterpret_cast<uintptr_t>(p) & 15) == 0) &&
                  ((reinterpret_cast<uintptr_t>(q) & 15) == 0);
  const long long grid = (long long)B * sh.slices;
  cudaError_t e = launch_pdl(accept_kernel, dim3((unsigned)grid), dim3(ACC_THREADS), 0, s, p, q, draft_tok, u, B, k, V,
                             sh.slices, sh.slice_len, vec, out_tok, accepted, counters,
                             reinterpret_cast<uint64_t *>(scratch), status);
  return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace mlora
