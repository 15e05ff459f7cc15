// Host-side launchers shared between the kernel translation units and the
// C-ABI front end (api.cu).  Internal to the library.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace mlora {

void note_launch();

// Step a1: stable counting sort of rows by adapter into `plan` (int32 words).
cudaError_t launch_plan(const int32_t *adapter_idx, int M, const int32_t *rank_of, int n_ad, int r_max,
                        int32_t *plan, uint32_t *status, cudaStream_t s);

// Step a2: T[m, j] for j < rank (fp32, row stride t_stride).  `zero_first`
// clears T first so that padding and rows without an adapter read 0.
cudaError_t launch_shrink(const uint16_t *x, int M, int K, const uint16_t *A, int n_ad, int r_max,
                          const int32_t *plan, float *T, int t_stride, bool zero_first, int num_sms, cudaStream_t s);

// Steps a3 + a4: base GEMM on tcgen05 with the expand epilogue.
struct GemmShape {
  int Mb, nsub, sub_n, n_tgroups, n_units, kblocks, total_iters, stages, nbuf, tmem_cols, grid;
  size_t smem_bytes, partial_floats;
};
GemmShape gemm_shape(int M, int N, int K, int num_sms);

struct GemmLaunch {
  const uint16_t *x;
  const uint16_t *W;
  int M, N, K;
  int mode;
  float scale;
  uint16_t *y;
  const uint16_t *B_stack;
  int r_max, n_ad;
  const float *T;
  const int32_t *plan;
  float *partials;
  uint32_t *counters;
  uint32_t *status;
};
cudaError_t launch_gemm(const GemmLaunch &g, const GemmShape &sh, cudaStream_t s, int *err_code);

// Steps a5 + a6.
struct AcceptShape {
  int slices, slice_len, threads;
  size_t scratch_bytes;
};
AcceptShape accept_shape(int B, int k, int V, int num_sms);
cudaError_t launch_accept(const float *p, const float *q, const int32_t *draft_tok, const float *u, int B, int k, int V,
                          int32_t *out_tok, int32_t *accepted, uint32_t *counters, void *scratch, uint32_t *status,
                          const AcceptShape &sh, cudaStream_t s);

}  // namespace mlora
