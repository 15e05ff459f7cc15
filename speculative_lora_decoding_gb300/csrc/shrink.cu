// Step a2, the shrink: T[m, j] = sum_k A_a[j, k] x[m, k] for j < rank_of[a],
// the inner product A·x of "output = W·x + scale · B(A·x)" ("Multi-LoRA
// Serving in Practice", section "Core Principle: Shared Base Model,
// Per-Request Adapter Selection").
//
// Work item = (adapter a, block of SHRINK_J = 8 rows of A_a, chunk of
// SHRINK_TOK = 4 rows of the adapter's group), read as one 32-byte record
// the plan kernel wrote.  One CTA of 4 warps takes an item and splits K
// across its warps; each lane streams 16-byte pieces of
// the 8 A rows (coalesced: a warp reads 512 contiguous bytes per row per
// step) and of the 4 x rows, and keeps 8 x 4 fp32 partial sums in registers.
// Every A element is used by exactly one thread, for all 4 tokens, so A goes
// from global memory straight to registers; nothing would be reused from a
// shared-memory copy.  Warp sums are combined in a fixed order, so T is
// deterministic.  Rank rows past rank_of[a] are never loaded.
//
// Output slices: a call may cover several projections that read the same
// rows x (q, k and v; gate and up), each with its own A stack; slice s reads
// A + s * n_ad * r_max * K and writes T + s * M * t_stride.  The grid has
// three CTAs per SM (all that fit), each taking (slice, item) units in turn.
//
// The low-rank operand of the tensor-core expand, when requested (tw):
// for each expand block (adapter a, 16-rank block j0) the window of sorted
// positions [w0, w0 + W) that covers a's rows (see common.cuh), W rows of
// 16 bf16: scale * T[row, j0:j0+16] on a's rows and 0 on the others.  The
// work items write the member entries of the rank columns below ceil8(rank);
// a pass over the windows writes zeros to exactly the other 16-byte halves,
// so the two never touch the same bytes and no earlier zeroing is needed.
// Rows are stored as the GEMM's shared memory wants them for a
// 32-byte-swizzled operand (the two 16-byte halves of window row i swapped
// when bit 2 of i is set), so that the GEMM fetches a window with one plain
// bulk copy.
//
// gather_rows_kernel: the verify pass's token rows in adapter-sorted order,
// xs[p] = x[perm[p]], which the GEMM reads so that each adapter's rows are
// adjacent accumulator columns.
#include "common.cuh"
#include "launch.h"

namespace mlora {

constexpr int SHRINK_THREADS = 128;
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

// Sums of 32 per-lane values across the warp: after the five exchange rounds
// lane l holds the warp total of value l (31 shuffles instead of 160).
__device__ __forceinline__ float warp_transpose_sum(float (&v)[32]) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int off = 16, n = 32; off >= 1; off >>= 1, n >>= 1) {
    const bool upper = (lane & off) != 0;
#pragma unroll
    for (int i = 0; i < n / 2; ++i) {
      const float send = upper ? v[i] : v[i + n / 2];
      const float keep = upper ? v[i + n / 2] : v[i];
      v[i] = keep + __shfl_xor_sync(0xffffffffu, send, off);
    }
  }
  return v[0];
}

#ifndef SHRINK_MIN_BLOCKS
#define SHRINK_MIN_BLOCKS 3  // caps registers at 170: three CTAs fit on an SM
#endif
__global__ void __launch_bounds__(SHRINK_THREADS, SHRINK_MIN_BLOCKS)
    shrink_kernel(const uint16_t *__restrict__ x, int M, int K, const uint16_t *__restrict__ A_all, int n_ad, int r_max,
                  const int32_t *__restrict__ plan, float *__restrict__ T_all, int t_stride,
                  uint16_t *__restrict__ tw_all, float scale, int n_slices, uint32_t *status) {
  __shared__ float red[SHRINK_WARPS][SHRINK_J * SHRINK_TOK];
  // Wait for the preceding kernel first, then let the GEMM that follows
  // launch: by then everything the GEMM's mainloop reads (x, W) is complete,
  // so it may stream while this kernel computes T; the GEMM waits for T only
  // in its epilogue.
  grid_dependency_wait();
  grid_launch_dependents();
  const PlanLayout L = plan_layout(M, n_ad);
  const int total_items = plan[L.hdr + 1];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int kchunks = K >> 3;  // 16-byte pieces per row
  const size_t tw_rows = max_window_rows(M, n_ad);
  const size_t tw_slice = tw_rows * 16;  // bf16 elements of one slice's operand buffer
  const int n_exp = plan[L.hdr + 4];

  if (tw_all) {
    // Zero halves: (slice, block, window row i, half h) not written by an item.
    for (int bu = blockIdx.x; bu < n_exp * n_slices; bu += gridDim.x) {
      const int sl = bu / n_exp, b = bu - sl * n_exp;
      const int4 e0 = *reinterpret_cast<const int4 *>(plan + L.slices + (size_t)b * EXP_WORDS);
      const int4 e1 = *reinterpret_cast<const int4 *>(plan + L.slices + (size_t)b * EXP_WORDS + 4);
      const int a = e0.x, j0 = e0.y, win = e0.w, w0 = e1.x, W = e1.y;
      // A record out of range (a plan overwritten or made for other sizes) is skipped.
      if ((unsigned)a >= (unsigned)n_ad || win < 0 || W < 0 || (size_t)win + W > tw_rows) {
        if (threadIdx.x == 0) raise_status(status, MLORA_DEV_BAD_PLAN);
        continue;
      }
      const int s0 = plan[L.seg_offsets + a], s1 = plan[L.seg_offsets + a + 1];
      const int r = plan[L.rank_eff + a];
      uint16_t *tw = tw_all + (size_t)sl * tw_slice + (size_t)win * 16;
      for (int hh = threadIdx.x; hh < 2 * W; hh += SHRINK_THREADS) {
        const int i = hh >> 1, h = hh & 1;
        const int p = w0 + i;
        const bool member = p >= s0 && p < s1;
        if (!(member && j0 + 8 * h < r))
          *reinterpret_cast<uint4 *>(tw + (size_t)i * 16 + 8 * (h ^ ((i >> 2) & 1))) = make_uint4(0u, 0u, 0u, 0u);
      }
    }
  }

  // Work units (slice, item), slice-major, one CTA each in turn.
  for (int wu = blockIdx.x; wu < total_items * n_slices; wu += gridDim.x) {
    const int sl = wu / total_items, item = wu - sl * total_items;
    const uint16_t *A = A_all + (size_t)sl * n_ad * r_max * K;
    float *T = T_all + (size_t)sl * M * t_stride;
    uint16_t *tw = tw_all ? tw_all + (size_t)sl * tw_slice : nullptr;
    const int4 *rec = reinterpret_cast<const int4 *>(plan + L.items + (size_t)item * ITEM_WORDS);
    const int4 h = rec[0], rw = rec[1];
    const int a = h.x, j0 = h.y & 0xFF, nrow = (h.y >> 8) & 0xFF, ntok = h.y >> 16;
    const int pos0 = h.z, blk0 = h.w;
    const int rows[SHRINK_TOK] = {rw.x, rw.y, rw.z, rw.w};
    // A record out of range (a plan overwritten or made for other sizes) is skipped.
    bool rec_ok = (unsigned)a < (unsigned)n_ad && j0 + nrow <= r_max && nrow <= SHRINK_J && ntok <= SHRINK_TOK &&
                  pos0 >= 0 && pos0 + ntok <= M;
#pragma unroll
    for (int t = 0; t < SHRINK_TOK; ++t) rec_ok &= t >= ntok || (unsigned)rows[t] < (unsigned)M;
    if (!rec_ok) {
      if (threadIdx.x == 0) raise_status(status, MLORA_DEV_BAD_PLAN);
      continue;
    }

    const uint16_t *Abase = A + ((size_t)a * r_max + j0) * (size_t)K;
    float acc[SHRINK_J * SHRINK_TOK];
#pragma unroll
    for (int i = 0; i < SHRINK_J * SHRINK_TOK; ++i) acc[i] = 0.f;

    // Two 16-byte pieces per row per iteration: all 24 loads of an
    // iteration are issued before any is used.
    for (int c = warp * 32 + lane; c < kchunks; c += 2 * SHRINK_THREADS) {
      const int c2 = c + SHRINK_THREADS;
      const bool has2 = c2 < kchunks;
      uint4 xv[2][SHRINK_TOK], av[2][SHRINK_J];
#pragma unroll
      for (int t = 0; t < SHRINK_TOK; ++t) {
        xv[0][t] = make_uint4(0, 0, 0, 0);
        xv[1][t] = make_uint4(0, 0, 0, 0);
        if (t < ntok) {
          const uint4 *xr = reinterpret_cast<const uint4 *>(x + (size_t)rows[t] * K);
          xv[0][t] = __ldg(xr + c);
          if (has2) xv[1][t] = __ldg(xr + c2);
        }
      }
#pragma unroll
      for (int j = 0; j < SHRINK_J; ++j) {
        av[0][j] = make_uint4(0, 0, 0, 0);
        av[1][j] = make_uint4(0, 0, 0, 0);
        if (j < nrow) {
          av[0][j] = ldg_stream(Abase + (size_t)j * K + (size_t)c * 8);
          if (has2) av[1][j] = ldg_stream(Abase + (size_t)j * K + (size_t)c2 * 8);
        }
      }
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {
        float xf[SHRINK_TOK][8];
#pragma unroll
        for (int t = 0; t < SHRINK_TOK; ++t) bf16x8_to_f32(xv[hh][t], xf[t]);
#pragma unroll
        for (int j = 0; j < SHRINK_J; ++j) {
          float af[8];
          bf16x8_to_f32(av[hh][j], af);
#pragma unroll
          for (int t = 0; t < SHRINK_TOK; ++t)
#pragma unroll
            for (int e = 0; e < 8; ++e) acc[j * SHRINK_TOK + t] = fmaf(af[e], xf[t][e], acc[j * SHRINK_TOK + t]);
        }
      }
    }
    // Warp totals (lane l holds value l), then a fixed-order sum over warps.
    red[warp][lane] = warp_transpose_sum(acc);
    block_sync();
    if (threadIdx.x < SHRINK_J * SHRINK_TOK) {
      const int j = threadIdx.x / SHRINK_TOK, t = threadIdx.x % SHRINK_TOK;
      float s = 0.f;
#pragma unroll
      for (int w = 0; w < SHRINK_WARPS; ++w) s += red[w][threadIdx.x];
      if (t < ntok) {
        const float v = (j < nrow) ? s : 0.f;
        T[(size_t)rows[t] * t_stride + j0 + j] = v;
        if (tw) {
          // Member row of the window of block (j0 + j) / 16 of adapter a.
          const int b = blk0 + (j0 + j) / 16;
          const int win = b >= 0 && b < n_exp ? plan[L.slices + (size_t)b * EXP_WORDS + 3] : -1;
          const int w0 = b >= 0 && b < n_exp ? plan[L.slices + (size_t)b * EXP_WORDS + 4] : 0;
          const int W = b >= 0 && b < n_exp ? plan[L.slices + (size_t)b * EXP_WORDS + 5] : 0;
          const int c = (j0 + j) % 16, i = pos0 + t - w0;
          if (win >= 0 && i >= 0 && i < W && (size_t)win + W <= tw_rows) {
            const int pc = (((c >> 3) ^ ((i >> 2) & 1)) << 3) | (c & 7);  // swizzled column
            tw[((size_t)win + i) * 16 + pc] = float_to_bf16_bits(scale * v);
          } else {
            raise_status(status, MLORA_DEV_BAD_PLAN);
          }
        }
      }
    }
    block_sync();
  }
}

// xs[p, :] = x[perm[p], :] for p < M (16-byte pieces, four in flight per
// thread).  Waits for the plan, then lets the shrink kernel launch.
__global__ void __launch_bounds__(256)
    gather_rows_kernel(const uint16_t *__restrict__ x, int M, int K, const int32_t *__restrict__ perm,
                       uint16_t *__restrict__ xs, uint32_t *status) {
  grid_dependency_wait();
  grid_launch_dependents();
  const int kv = K >> 3;
  const long long total = (long long)M * kv;
  const long long stride = (long long)gridDim.x * blockDim.x;
  for (long long i0 = (long long)blockIdx.x * blockDim.x + threadIdx.x; i0 < total; i0 += 4 * stride) {
    uint4 v[4];
    long long dst[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const long long i = i0 + u * stride;
      dst[u] = -1;
      if (i < total) {
        const int p = (int)(i / kv), c = (int)(i - (long long)p * kv);
        const int m = perm[p];
        if ((unsigned)m < (unsigned)M) {
          v[u] = __ldg(reinterpret_cast<const uint4 *>(x + (size_t)m * K) + c);
          dst[u] = (long long)p * kv + c;
        } else {
          raise_status(status, MLORA_DEV_BAD_PLAN);  // a permutation entry out of range: skipped
        }
      }
    }
#pragma unroll
    for (int u = 0; u < 4; ++u)
      if (dst[u] >= 0) reinterpret_cast<uint4 *>(xs)[dst[u]] = v[u];
  }
}

cudaError_t launch_gather_rows(const uint16_t *x, int M, int K, const int32_t *perm, uint16_t *xs, int num_sms,
                               uint32_t *status, cudaStream_t s) {
  const long long pieces = (long long)M * (K >> 3);
  const long long want = (pieces + 4 * 256 - 1) / (4 * 256);
  const int grid = (int)max(1LL, min(want, (long long)num_sms * 4));
  cudaError_t e = launch_pdl(gather_rows_kernel, dim3(grid), dim3(256), 0, s, x, M, K, perm, xs, status);
  return e != cudaSuccess ? e : cudaGetLastError();
}

cudaError_t launch_shrink(const uint16_t *x, int M, int K, const uint16_t *A, int n_ad, int r_max,
                          const int32_t *plan, float *T, int t_stride, bool zero_first, int num_sms, uint16_t *tw,
                          float scale, int n_slices, uint32_t *status, cudaStream_t s) {
  if (zero_first) {
    cudaError_t e = cudaMemsetAsync(T, 0, (size_t)n_slices * M * t_stride * sizeof(float), s);
    if (e != cudaSuccess) return e;
  }
  // Upper bound on work items: ceil(r_max/J) * (ceil(M/TOK) + min(M, n_ad)).
  const long long bound =
      (long long)((r_max + SHRINK_J - 1) / SHRINK_J) * ((M + SHRINK_TOK - 1) / SHRINK_TOK + min(M, n_ad));
  // Three CTAs per SM (all that fit: 128 threads x 168 registers each).
  // Measured on the 32B block at 640 verify rows: one CTA per SM, leaving
  // registers for the GEMM that follows to stream beside it, made the verify
  // pass 908 us; three, with the GEMM's CTAs starting as the shrink's leave,
  // 825 us.
  const int grid = (int)max(1LL, min(bound * n_slices, (long long)num_sms * 3));
  cudaError_t e = launch_pdl(shrink_kernel, dim3(grid), dim3(SHRINK_THREADS), 0, s, x, M, K, A, n_ad, r_max, plan, T,
                             t_stride, tw, scale, n_slices, status);
  return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace mlora
