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
// entries, one CTA each, so that a small batch still gives every SM several
// CTAs and each SM has many 16-byte loads in flight.  Every CTA of a request
// repeats the accept test (its k gathers hit L2), one lane per draft
// position.  Because almost every draft is accepted, the CTA requests its
// chunk of the bonus row p_k before the test resolves; when a draft was
// rejected it reads p_n and q_n instead.  It publishes the chunk's exact
// uint64 sums (residual mass and target mass); the last CTA of the request
// to arrive (atomic counter, no spinning) scans the chunk sums, computes the
// draw, re-reads only the chunk holding it (one round, a contiguous run per
// thread) and locates the token with a block-wide prefix scan.  All sums are
// integers, so the order of addition cannot change a result.
//
// Q(f) = floor(f * 2^40) is one fp32 multiply (exact: a power-of-two scale of
// a value in [0, 1]) and one conversion rounding toward minus infinity to an
// unsigned 64-bit integer (exact: the scaled value is representable and its
// integer part is below 2^41).
#include "common.cuh"
#include "launch.h"

namespace mlora {

constexpr int ACC_THREADS = 256;
constexpr int ACC_WARPS = ACC_THREADS / 32;
constexpr int CHUNK = 4096;                       // vocabulary entries per CTA
constexpr int PER_THREAD = CHUNK / ACC_THREADS;   // 16: four float4 per thread
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

// The 16 entries thread `tid` covers in the chunk starting at v0: with
// 16-byte loads, four float4 at v0 + 4 * (tid + 256 j), j < 4 (a warp reads
// 512 contiguous bytes per load); otherwise v0 + tid + 256 j, j < 16.  All
// loads are issued before any value is used.  Entries at or past V read as
// 0: in range, weight 0.
__device__ __forceinline__ void load_chunk(const float *row, int v0, int V, int tid, bool vec, float (&f)[PER_THREAD]) {
  if (vec && v0 + CHUNK <= V) {
    const float4 *r4 = reinterpret_cast<const float4 *>(row + v0);
    float4 t[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) t[j] = __ldcs(r4 + tid + ACC_THREADS * j);
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      f[4 * j + 0] = t[j].x;
      f[4 * j + 1] = t[j].y;
      f[4 * j + 2] = t[j].z;
      f[4 * j + 3] = t[j].w;
    }
  } else {
#pragma unroll
    for (int j = 0; j < PER_THREAD; ++j) {
      const int v = v0 + tid + ACC_THREADS * j;
      f[j] = v < V ? __ldcs(row + v) : 0.f;
    }
  }
}

__global__ void __launch_bounds__(ACC_THREADS)
    accept_kernel(const float *__restrict__ p, const float *__restrict__ q, const int32_t *__restrict__ draft_tok,
                  const float *__restrict__ uni, int B, int k, int V, int chunks, int vec,
                  int32_t *__restrict__ out_tok, int32_t *__restrict__ accepted, uint32_t *counters,
                  uint64_t *sums, uint32_t *status) {
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
  const bool vec_ok = vec != 0;

  // Speculatively request this chunk of the bonus row p_k.
  float fp[PER_THREAD];
  load_chunk(p + ((size_t)b * k1 + k) * V, v0, V, tid, vec_ok, fp);

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
        const float pi = sanitize_prob(p[((size_t)b * k1 + lane) * V + x], f);
        const float qi = sanitize_prob(q[((size_t)b * k + lane) * V + x], f);
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
    load_chunk(p + ((size_t)b * k1 + n) * V, v0, V, tid, vec_ok, fp);
    load_chunk(q + ((size_t)b * k + n) * V, v0, V, tid, vec_ok, fq);
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
    uint64_t w[PER_THREAD];
    {
      float a[PER_THREAD], bq[PER_THREAD];
#pragma unroll
      for (int j = 0; j < PER_THREAD; ++j) {
        a[j] = cv0 + j < V ? __ldcg(prow + cv0 + j) : 0.f;
        bq[j] = (use_q && cv0 + j < V) ? __ldcg(qrow + cv0 + j) : 0.f;
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

AcceptShape accept_shape(int B, int k, int V, int num_sms) {
  (void)k;
  (void)num_sms;
  AcceptShape s;
  s.slice_len = CHUNK;
  s.slices = (V + CHUNK - 1) / CHUNK;
  s.threads = ACC_THREADS;
  s.scratch_bytes = (size_t)B * s.slices * 2 * sizeof(uint64_t);
  return s;
}

cudaError_t launch_accept(const float *p, const float *q, const int32_t *draft_tok, const float *u, int B, int k, int V,
                          int32_t *out_tok, int32_t *accepted, uint32_t *counters, void *scratch, uint32_t *status,
                          const AcceptShape &sh, cudaStream_t s) {
  const int vec = ((V & 3) == 0) && ((reinterpret_cast<uintptr_t>(p) & 15) == 0) &&
                  ((reinterpret_cast<uintptr_t>(q) & 15) == 0);
  const long long grid = (long long)B * sh.slices;
  cudaError_t e = launch_pdl(accept_kernel, dim3((unsigned)grid), dim3(ACC_THREADS), 0, s, p, q, draft_tok, u, B, k, V,
                             sh.slices, vec, out_tok, accepted, counters, reinterpret_cast<uint64_t *>(scratch),
                             status);
  return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace mlora
