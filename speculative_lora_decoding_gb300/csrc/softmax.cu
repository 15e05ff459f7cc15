// The steps on either side of the accept step: the softmax that turns a
// pass's logits into the distributions the accept step compares, and the draw
// of each request's draft token from the draft distribution q (the InvisibleLoRA
// abstract: a LoRA-off pass proposes the next token for every request, one
// LoRA-on pass verifies the proposals).
//
// One definition of a probability serves every kernel of the library:
//
//   p(v) = expf(z(v) - m) / S,   m = max_w z(w),   S = the row sum below
//
// computed in fp32 with CUDA's expf and an IEEE division.  The row statistics
// (m, S) come from row_stats (one CTA per row, online softmax: every thread
// keeps a running maximum and a sum rescaled whenever the maximum grows, over
// a fixed set of entries in a fixed order, and the partial results are merged
// in a fixed tree), so they are deterministic; because every entry of p is
// computed from (m, S) by the same expression, the probabilities the accept
// step derives from logits are bit-identical to the ones softmax_write
// writes.
//
// The draft draw uses the accept step's exact integer inverse CDF on
// Q(q(v)) = floor(q(v) * 2^40): S_w = sum of the weights, U = floor(u * 2^32),
// T = floor(U * S_w / 2^32), token = the smallest v whose running sum of
// weights exceeds T.  Sums of the weights of 512-entry blocks are kept (exact
// in uint64), the block holding T is found by a scan over them, then the token
// inside it by a warp scan.
#include <algorithm>

#include "common.cuh"
#include "launch.h"

namespace mlora {

constexpr int SM_THREADS = 256;
constexpr int SM_WARPS = SM_THREADS / 32;
constexpr int SM_CHUNK = 4096;   // vocabulary entries per (row, chunk) unit: 16 per thread
constexpr int DRAW_BLOCK = 512;  // vocabulary entries per weight block of the draw
constexpr float SM_TWO_POW_32 = 4294967296.0f;
constexpr float SM_TWO_POW_40 = 1099511627776.0f;

// The probability of an entry from its logit and the row's statistics.
__device__ __forceinline__ float prob_of(float z, float2 st) { return expf(z - st.x) / st.y; }

// Merge two (running maximum, sum relative to it) pairs.
__device__ __forceinline__ void merge_stats(float &m, float &s, float m2, float s2) {
  if (m2 == -INFINITY) return;
  if (m == -INFINITY) {
    m = m2;
    s = s2;
    return;
  }
  const float mm = fmaxf(m, m2);
  s = s * expf(m - mm) + s2 * expf(m2 - mm);
  m = mm;
}

__device__ __forceinline__ void online_add(float &m, float &s, float z) {
  if (z > m) {
    s = (m == -INFINITY ? 0.f : s * expf(m - z)) + 1.f;
    m = z;
  } else if (m != -INFINITY) {  // z = -inf before any finite logit adds nothing
    s += expf(z - m);
  }
}

// Statistics of one (row, 4096-entry chunk) unit by a CTA of 256 threads:
// thread t takes entries 4t + 1024 j, j < 4 (float4 loads when the row
// allows), an online pass over its 16 entries in index order, then a fixed
// butterfly over the warp and a fixed sequential merge of the eight warps.
__device__ float2 chunk_stats(const float *row, int v0, int V, bool vec, float2 *sh) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  float m = -INFINITY, s = 0.f;
  float v[16];
  if (vec) {
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int e = v0 + 4 * tid + 1024 * j;
      const float4 f = e < V ? __ldcs(reinterpret_cast<const float4 *>(row + e))
                             : make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
      v[4 * j] = f.x, v[4 * j + 1] = f.y, v[4 * j + 2] = f.z, v[4 * j + 3] = f.w;
    }
  } else {
#pragma unroll
    for (int j = 0; j < 16; ++j) {
      const int e = v0 + 4 * tid + 1024 * (j >> 2) + (j & 3);
      v[j] = e < V ? __ldcs(row + e) : -INFINITY;
    }
  }
#pragma unroll
  for (int j = 0; j < 16; ++j) online_add(m, s, v[j]);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float m2 = __shfl_xor_sync(0xffffffffu, m, o);
    const float s2 = __shfl_xor_sync(0xffffffffu, s, o);
    // Both lanes of a pair merge the same two values in the same order.
    if (lane & o) {
      float mm = m2, ss = s2;
      merge_stats(mm, ss, m, s);
      m = mm;
      s = ss;
    } else {
      merge_stats(m, s, m2, s2);
    }
  }
  if (lane == 0) sh[warp] = make_float2(m, s);
  __syncthreads();
  float2 res = make_float2(0.f, 0.f);
  if (tid == 0) {
    float mt = sh[0].x, st = sh[0].y;
    for (int w = 1; w < SM_WARPS; ++w) merge_stats(mt, st, sh[w].x, sh[w].y);
    res = make_float2(mt, st);
  }
  return res;  // valid in thread 0
}

// stats[r] = (m, S) of row r of z [R, V].  One CTA per (row, chunk) unit;
// each writes its chunk's (maximum, sum) to part[r][c], and the last unit of
// the row to arrive (counter, no spinning) merges the chunks in chunk order,
// so the result does not depend on which unit finishes last.  The counters
// return to zero.
__global__ void __launch_bounds__(SM_THREADS)
    row_stats_kernel(const float *__restrict__ z, int R, int V, int chunks, float2 *__restrict__ part,
                     uint32_t *counters, float2 *__restrict__ stats) {
  __shared__ float2 sh[SM_WARPS];
  __shared__ int last;
  grid_dependency_wait();
  grid_launch_dependents();
  const bool vec = (V & 3) == 0 && (reinterpret_cast<uintptr_t>(z) & 15) == 0;
  const int r = blockIdx.x / chunks, c = blockIdx.x - r * chunks;
  const float2 cs = chunk_stats(z + (size_t)r * V, c * SM_CHUNK, V, vec, sh);
  if (threadIdx.x == 0) {
    part[(size_t)r * chunks + c] = cs;
    __threadfence();
    last = atomicAdd(&counters[r], 1u) == (uint32_t)(chunks - 1);
  }
  __syncthreads();
  if (last && threadIdx.x == 0) {
    __threadfence();
    float m = -INFINITY, sm = 0.f;
    for (int k = 0; k < chunks; ++k) {
      const float2 p2 = __ldcg(&part[(size_t)r * chunks + k]);
      merge_stats(m, sm, p2.x, p2.y);
    }
    stats[r] = make_float2(m, sm);
    counters[r] = 0u;
  }
}

// p[r, v] = prob_of(z[r, v], stats[r]).
__global__ void __launch_bounds__(256)
    softmax_write_kernel(const float *__restrict__ z, int R, int V, const float2 *__restrict__ stats,
                         float *__restrict__ p) {
  grid_dependency_wait();
  grid_launch_dependents();
  const long long total = (long long)R * V;
  const long long stride = (long long)gridDim.x * blockDim.x;
  for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < total; i += stride) {
    const int r = (int)(i / V);
    p[i] = prob_of(__ldcs(z + i), stats[r]);
  }
}

__device__ __forceinline__ uint64_t q40(float f) { return __float2ull_rd(fminf(fmaxf(f, 0.f), 1.f) * SM_TWO_POW_40); }

__device__ __forceinline__ uint64_t warp_sum_u64_sm(uint64_t v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

__device__ __forceinline__ uint64_t warp_incl_scan_u64_sm(uint64_t v) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint64_t t = __shfl_up_sync(0xffffffffu, v, o);
    if (lane >= o) v += t;
  }
  return v;
}

// Draft draw.  One CTA per (request b, 4096-entry chunk) unit: warp w takes
// the chunk's 512-entry block w (16 consecutive entries per lane), writes the
// probabilities (when q_out is given) and the block's exact uint64 weight sum
// blk[b][8 c + w].  The last unit of the request to arrive (counter) totals
// the weights, finds the block holding T (a block scan over contiguous runs
// of blocks) and then the token inside it (a warp scan), and writes it.
__global__ void __launch_bounds__(SM_THREADS)
    draft_sample_kernel(const float *__restrict__ z, int B, int V, int chunks, const float2 *__restrict__ stats,
                        const float *__restrict__ u, int32_t *__restrict__ tok, float *__restrict__ q_out,
                        uint64_t *__restrict__ blk, uint32_t *counters, uint32_t *status) {
  __shared__ uint64_t shu[SM_WARPS];
  __shared__ int sh_block, last;
  __shared__ uint64_t sh_T, sh_Tloc;
  grid_dependency_wait();
  grid_launch_dependents();
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int b = blockIdx.x / chunks, c = blockIdx.x - b * chunks;
  const int nblk = chunks * (SM_CHUNK / DRAW_BLOCK);
  const float *row = z + (size_t)b * V;
  const float2 st = stats[b];
  uint64_t *bw = blk + (size_t)b * nblk;
  {
    const int k = c * (SM_CHUNK / DRAW_BLOCK) + warp;
    const int v0 = k * DRAW_BLOCK + 16 * lane;
    uint64_t w = 0;
#pragma unroll
    for (int j = 0; j < 16; ++j) {
      const int v = v0 + j;
      if (v < V) {
        const float q = prob_of(row[v], st);
        if (q_out) q_out[(size_t)b * V + v] = q;
        w += q40(q);
      }
    }
    w = warp_sum_u64_sm(w);
    if (lane == 0) bw[k] = w;
  }
  __syncthreads();
  if (tid == 0) {
    __threadfence();
    last = atomicAdd(&counters[b], 1u) == (uint32_t)(chunks - 1);
  }
  __syncthreads();
  if (!last) return;
  __threadfence();
  // Total and the block holding T: thread t sums a contiguous run of blocks.
  const int per = (nblk + SM_THREADS - 1) / SM_THREADS;
  const int k0 = min(nblk, tid * per), k1 = min(nblk, k0 + per);
  uint64_t mine = 0;
  for (int k = k0; k < k1; ++k) mine += __ldcg(&bw[k]);
  const uint64_t inc = warp_incl_scan_u64_sm(mine);
  if (lane == 31) shu[warp] = inc;
  __syncthreads();
  uint64_t before = 0, total = 0;
  for (int w = 0; w < SM_WARPS; ++w) {
    if (w < warp) before += shu[w];
    total += shu[w];
  }
  if (tid == 0) {
    counters[b] = 0u;
    sh_block = -1;
    float uu = u[b];
    uint32_t fl = 0;
    if (!(uu >= 0.f)) {
      uu = 0.f;
      fl |= MLORA_DEV_BAD_PROB;
    } else if (uu >= 1.f) {
      uu = __uint_as_float(0x3F7FFFFFu);
      fl |= MLORA_DEV_BAD_PROB;
    }
    if (total == 0) fl |= MLORA_DEV_ZERO_MASS;
    const uint64_t U = __float2ull_rz(uu * SM_TWO_POW_32);
    sh_T = total == 0 ? 0 : (__umul64hi(U, total) << 32) | ((U * total) >> 32);  // floor(U * S / 2^32) < S
    if (fl) raise_status(status, fl);
  }
  __syncthreads();
  const uint64_t T = sh_T;
  if (total != 0) {
    uint64_t run = before + inc - mine;
    if (run <= T && T < run + mine) {
      for (int k = k0; k < k1; ++k) {
        const uint64_t w = __ldcg(&bw[k]);
        if (T < run + w) {
          sh_block = k;
          sh_Tloc = T - run;
          break;
        }
        run += w;
      }
    }
  }
  __syncthreads();
  if (warp == 0) {
    int t = 0;
    const int kb = sh_block;
    if (kb >= 0) {
      const uint64_t Tl = sh_Tloc;
      const int v0 = kb * DRAW_BLOCK + 16 * lane;
      uint64_t wv[16];
      uint64_t mw = 0;
#pragma unroll
      for (int j = 0; j < 16; ++j) {
        wv[j] = v0 + j < V ? q40(prob_of(row[v0 + j], st)) : 0ull;
        mw += wv[j];
      }
      const uint64_t inc2 = warp_incl_scan_u64_sm(mw);
      uint64_t run2 = inc2 - mw;
      const uint32_t hit = __ballot_sync(0xffffffffu, run2 <= Tl && Tl < run2 + mw);
      int found = -1;
      if (hit && lane == __ffs(hit) - 1) {
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          if (found < 0 && Tl < run2 + wv[j]) found = v0 + j;
          run2 += wv[j];
        }
      }
      t = hit ? __shfl_sync(0xffffffffu, found, __ffs(hit) - 1) : 0;
      if (t < 0) t = 0;  // unreachable when the sums are consistent
    }
    if (lane == 0) tok[b] = t;
  }
}

static int chunks_of(int V) { return (V + SM_CHUNK - 1) / SM_CHUNK; }

size_t row_stats_scratch_bytes(int R, int V) { return align_up((size_t)R * chunks_of(V) * sizeof(float2), 256); }

cudaError_t launch_row_stats(const float *z, int R, int V, float2 *stats, void *scratch, uint32_t *counters,
                             cudaStream_t s) {
  const int chunks = chunks_of(V);
  cudaError_t e = launch_pdl(row_stats_kernel, dim3((unsigned)((long long)R * chunks)), dim3(SM_THREADS), 0, s, z, R,
                             V, chunks, reinterpret_cast<float2 *>(scratch), counters, stats);
  return e != cudaSuccess ? e : cudaGetLastError();
}

cudaError_t launch_softmax_write(const float *z, int R, int V, const float2 *stats, float *p, int num_sms,
                                 cudaStream_t s) {
  const long long total = (long long)R * V;
  const int grid = (int)std::max<long long>(1, std::min<long long>((total + 255) / 256, (long long)num_sms * 8));
  cudaError_t e = launch_pdl(softmax_write_kernel, dim3(grid), dim3(256), 0, s, z, R, V, stats, p);
  return e != cudaSuccess ? e : cudaGetLastError();
}

size_t draft_sample_scratch_bytes(int B, int V) {
  return align_up((size_t)B * chunks_of(V) * (SM_CHUNK / DRAW_BLOCK) * sizeof(uint64_t), 256) +
         row_stats_scratch_bytes(B, V);
}

cudaError_t launch_draft_sample(const float *z, int B, int V, const float *u, int32_t *tok, float2 *stats, float *q,
                                void *scratch, uint32_t *counters, uint32_t *status, cudaStream_t s) {
  const int chunks = chunks_of(V);
  uint8_t *sc = static_cast<uint8_t *>(scratch);
  uint64_t *blk = reinterpret_cast<uint64_t *>(sc);
  void *stats_scratch = sc + align_up((size_t)B * chunks * (SM_CHUNK / DRAW_BLOCK) * sizeof(uint64_t), 256);
  cudaError_t e = launch_row_stats(z, B, V, stats, stats_scratch, counters, s);
  if (e != cudaSuccess) return e;
  e = launch_pdl(draft_sample_kernel, dim3((unsigned)((long long)B * chunks)), dim3(SM_THREADS), 0, s, z, B, V,
                 chunks, (const float2 *)stats, u, tok, q, blk, counters, status);
  return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace mlora
