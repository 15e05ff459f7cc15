// Step a2, the shrink: T[m, j] = sum_k A_a[j, k] x[m, k] for j < rank_of[a],
// the inner product A·x of "output = W·x + scale · B(A·x)" ("Multi-LoRA
// Serving in Practice", section "Core Principle: Shared Base Model,
// Per-Request Adapter Selection").
//
// Work item = (adapter a, block of SHRINK_J = 8 rows of A_a, chunk of
// SHRINK_TOK = 4 rows of the adapter's group).  One CTA of 8 warps takes an
// item and splits K across its warps; each lane streams 16-byte pieces of
// the 8 A rows (coalesced: a warp reads 512 contiguous bytes per row per
// step) and of the 4 x rows, and keeps 8 x 4 fp32 partial sums in registers.
// Every A element is used by exactly one thread, for all 4 tokens, so A goes
// from global memory straight to registers; nothing would be reused from a
// shared-memory copy.  Warp sums are combined in a fixed order, so T is
// deterministic.  Rank rows past rank_of[a] are never loaded.
#include "common.cuh"
#include "launch.h"

namespace mlora {

constexpr int SHRINK_THREADS = 256;
constexpr int SHRINK_WARPS = SHRINK_THREADS / 32;

__device__ __forceinline__ void bf16x8_to_f32(const uint4 v, float (&f)[8]) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    f[2 * i] = __uint_as_float(w[i] << 16);
    f[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
  }
}

__device__ __forceinline__ uint4 ldg_stream(const uint16_t *p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

__global__ void __launch_bounds__(SHRINK_THREADS)
    shrink_kernel(const uint16_t *__restrict__ x, int M, int K, const uint16_t *__restrict__ A, int n_ad, int r_max,
                  const int32_t *__restrict__ plan, float *__restrict__ T, int t_stride) {
  __shared__ float red[SHRINK_WARPS][SHRINK_J][SHRINK_TOK];
  const PlanLayout L = plan_layout(M, n_ad);
  const int n_active = plan[L.hdr + 0];
  const int total_items = plan[L.hdr + 1];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int kchunks = K >> 3;  // 16-byte pieces per row

  for (int item = blockIdx.x; item < total_items; item += gridDim.x) {
    // Active-list slot holding this item (item_off is increasing).
    int lo = 0, hi = n_active;
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (plan[L.item_off + mid] <= item) lo = mid; else hi = mid;
    }
    const int a = plan[L.active + lo];
    const int r = plan[L.rank_eff + a];
    const int s0 = plan[L.seg_offsets + a];
    const int cnt = plan[L.seg_offsets + a + 1] - s0;
    const int local = item - plan[L.item_off + lo];
    const int nj = (r + SHRINK_J - 1) / SHRINK_J;
    const int j0 = (local % nj) * SHRINK_J;
    const int t0 = (local / nj) * SHRINK_TOK;
    const int ntok = min(SHRINK_TOK, cnt - t0);
    const int nrow = min(SHRINK_J, r - j0);

    int rows[SHRINK_TOK];
#pragma unroll
    for (int t = 0; t < SHRINK_TOK; ++t) rows[t] = (t < ntok) ? plan[L.perm + s0 + t0 + t] : 0;

    const uint16_t *Abase = A + ((size_t)a * r_max + j0) * (size_t)K;
    float acc[SHRINK_J][SHRINK_TOK];
#pragma unroll
    for (int j = 0; j < SHRINK_J; ++j)
#pragma unroll
      for (int t = 0; t < SHRINK_TOK; ++t) acc[j][t] = 0.f;

    for (int c = warp * 32 + lane; c < kchunks; c += SHRINK_THREADS) {
      float xf[SHRINK_TOK][8];
#pragma unroll
      for (int t = 0; t < SHRINK_TOK; ++t) {
        uint4 v = make_uint4(0, 0, 0, 0);
        if (t < ntok) v = __ldg(reinterpret_cast<const uint4 *>(x + (size_t)rows[t] * K) + c);
        bf16x8_to_f32(v, xf[t]);
      }
#pragma unroll
      for (int j = 0; j < SHRINK_J; ++j) {
        if (j < nrow) {
          float af[8];
          bf16x8_to_f32(ldg_stream(Abase + (size_t)j * K + (size_t)c * 8), af);
#pragma unroll
          for (int t = 0; t < SHRINK_TOK; ++t)
#pragma unroll
            for (int e = 0; e < 8; ++e) acc[j][t] = fmaf(af[e], xf[t][e], acc[j][t]);
        }
      }
    }
    // Warp sums (butterfly), then a fixed-order sum over warps.
#pragma unroll
    for (int j = 0; j < SHRINK_J; ++j)
#pragma unroll
      for (int t = 0; t < SHRINK_TOK; ++t) {
        float v = acc[j][t];
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
        acc[j][t] = v;
      }
    if (lane == 0) {
#pragma unroll
      for (int j = 0; j < SHRINK_J; ++j)
#pragma unroll
        for (int t = 0; t < SHRINK_TOK; ++t) red[warp][j][t] = acc[j][t];
    }
    __syncthreads();
    if (threadIdx.x < SHRINK_J * SHRINK_TOK) {
      const int j = threadIdx.x / SHRINK_TOK, t = threadIdx.x % SHRINK_TOK;
      float s = 0.f;
#pragma unroll
      for (int w = 0; w < SHRINK_WARPS; ++w) s += red[w][j][t];
      if (t < ntok) T[(size_t)rows[t] * t_stride + j0 + j] = (j < nrow) ? s : 0.f;
    }
    __syncthreads();
  }
}

cudaError_t launch_shrink(const uint16_t *x, int M, int K, const uint16_t *A, int n_ad, int r_max,
                          const int32_t *plan, float *T, int t_stride, bool zero_first, int num_sms, cudaStream_t s) {
  if (zero_first) {
    cudaError_t e = cudaMemsetAsync(T, 0, (size_t)M * t_stride * sizeof(float), s);
    if (e != cudaSuccess) return e;
  }
  // Upper bound on work items: ceil(r_max/J) * (ceil(M/TOK) + min(M, n_ad)).
  const long long bound =
      (long long)((r_max + SHRINK_J - 1) / SHRINK_J) * ((M + SHRINK_TOK - 1) / SHRINK_TOK + min(M, n_ad));
  const int grid = (int)max(1LL, min(bound, (long long)num_sms * 4));
  shrink_kernel<<<grid, SHRINK_THREADS, 0, s>>>(x, M, K, A, n_ad, r_max, plan, T, t_stride);
  note_launch();
  return cudaGetLastError();
}

}  // namespace mlora
