// Host-side launchers shared between the kernel translation units and the
// C-ABI front end (api.cu).  Internal to the library.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/mlora.h"

namespace mlora {

void note_launch();

// Launch with programmatic dependent launch allowed: the kernel may start
// while the preceding kernel in the stream finishes; every kernel of this
// library calls griddepcontrol.wait before it reads anything an earlier
// kernel may have written.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                       Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cudaError_t e = cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
  note_launch();
  return e;
}

// Step a1: stable counting sort of rows by adapter into `plan` (int32 words).
cudaError_t launch_plan(const int32_t *adapter_idx, int M, const int32_t *rank_of, int n_ad, int r_max,
                        int32_t *plan, uint32_t *status, cudaStream_t s);

// The verify pass's token rows in adapter-sorted order: xs[p] = x[perm[p]]
// for p < M (bf16 [M, K]).
cudaError_t launch_gather_rows(const uint16_t *x, int M, int K, const int32_t *perm, uint16_t *xs, int num_sms,
                               uint32_t *status, cudaStream_t s);

// Step a2: T[m, j] for j < rank (fp32, row stride t_stride), for n_slices
// output slices (A: [n_slices][n_ad][r_max][K]; T: [n_slices][M][t_stride]).
// `zero_first` clears T first so that padding and rows without an adapter
// read 0.  With `tw` non-null it also writes the token windows of the
// tensor-core expand, [n_slices][max_window_rows(M, n_ad)][16] bf16 (see
// common.cuh): scale * T on member rows, 0 elsewhere.
cudaError_t launch_shrink(const uint16_t *x, int M, int K, const uint16_t *A, int n_ad, int r_max,
                          const int32_t *plan, float *T, int t_stride, bool zero_first, int num_sms, uint16_t *tw,
                          float scale, int n_slices, uint32_t *status, cudaStream_t s);

// The token windows alone (as launch_shrink writes them into `tw`), on the
// tensor cores: one 128 x (up to 256) MMA tile per 8 consecutive expand
// blocks over their tokens in adapter-sorted order `xs` [M, K], split-K
// over a thread-block cluster.  Reads the plan; writes no T.
cudaError_t launch_shrink_mma(const uint16_t *xs, int M, int K, const uint16_t *A, int n_ad, int r_max,
                              const int32_t *plan, uint16_t *tw, float scale, int n_slices, int num_sms,
                              uint32_t *status, cudaStream_t s);

// Steps a3 + a4: base GEMM on tcgen05 with the expand epilogue.
struct GemmShape {
  int Mb, nsub, sub_n, n_tgroups, n_units, kblocks, total_iters, stages, nbuf, tmem_cols, grid;
  int C;          // CTAs per cluster splitting K (1: no split)
  int waves;      // rounds of resident clusters the launch takes
  int red_bytes;  // shared memory for the cluster reduction
  size_t smem_bytes, partial_floats;
};
GemmShape gemm_shape(int M, int N, int K, int num_sms);

struct GemmLaunch {
  const uint16_t *x;
  const uint16_t *W;
  int M, N, K;
  int n_slices;                      // output slices, each with its own T and masked operand
  int slice_end[MLORA_MAX_SLICES];   // end row of each slice in W / y; all but the last multiples of 128
  int mode;
  int prefetch_w;    // W may be requested before the preceding kernel finishes
  int after_shrink;  // the preceding kernel on the stream is launch_shrink's
  float scale;
  uint16_t *y;
  const uint16_t *B_stack;
  int r_max, n_ad;
  const float *T;      // [n_slices][M][T_STRIDE]
  const int32_t *plan;
  uint32_t *status;
  const uint16_t *tw;  // token windows [n_slices][max_window_rows][16] with x in sorted order, or null
                       // (x in row order, bucket-walk epilogue)
  uint32_t test_flag_wait_ns;  // stream-K only: nonzero makes owners wait on never-set flags (timeout test)
};
cudaError_t launch_gemm(const GemmLaunch &g, const GemmShape &sh, cudaStream_t s, int *err_code);

// Steps a3 + a4 as a persistent stream-K kernel (gemm_sk.cu): one CTA per SM,
// equal shares of the (tile, token group, k-block) triples, at most 1024 token
// rows in groups of at most 256, draft mode
// or verify mode with the tensor-core expand.  Needs sk_partial_bytes(M, SMs)
// of scratch for partial sums and one flag word per CTA (zero between calls).
// `ok` is false when a CTA of that shape would not fit on every SM at once
// (the cross-CTA waits need the whole grid resident).
struct SkShape {
  bool ok;
  int Mb, n_tg, cols, stages, n_tiles, kblocks, total, P, Pg;  // Mb rows in each of n_tg groups, Pg CTAs per group
  size_t smem_bytes;
};
SkShape sk_shape(int M, int N, int K, int num_sms, bool f8 = false);
size_t sk_partial_bytes(int M, int num_sms);
cudaError_t launch_gemm_sk(const GemmLaunch &g, const SkShape &sh, float *partials, uint32_t *flags, cudaStream_t s,
                           int *err_code);

// The draft layer on E4M3 codes (fp8.cu quantizes; the stream-K kernel with
// kind::f8f6f4 MMAs multiplies): y = bf16(acc * w_scale[n] * x_scale[m]).
struct F8Launch {
  const uint8_t *x8, *W8;
  const float *x_scale, *w_scale;
  int M, N, K, prefetch_w;
  uint16_t *y;
  uint32_t *status;
};
cudaError_t launch_gemm_sk_f8(const F8Launch &g, const SkShape &sh, float *partials, uint32_t *flags, cudaStream_t s,
                              int *err_code);
// Per-row E4M3 quantization of bf16 rows [R, K]: scale[r] = amax / 448,
// q[r, k] = e4m3_rn_satfinite(src[r, k] / scale[r]); a zero row gets scale 1.
cudaError_t launch_quantize_rows_e4m3(const uint16_t *src, int R, int K, uint8_t *q, float *scale, int num_sms,
                                      cudaStream_t s);

// Steps a5 + a6.  With stats_p and stats_q non-null, p and q hold logits and
// the kernels read probabilities expf(z - m) / S from the rows' statistics.
struct AcceptShape {
  int slices, slice_len, threads;
  int blocks_grid;  // CTAs of the streaming form's block sums (rows of aligned float4)
  size_t stats_off;      // scratch offset of the row statistics (logits form): float2 [B(k+1) + Bk]
  size_t part_off;       // scratch offset of the statistics' chunk partials (logits form)
  size_t scratch_bytes;
};
AcceptShape accept_shape(int B, int k, int V, int num_sms);
cudaError_t launch_accept(const float *p, const float *q, const int32_t *draft_tok, const float *u, int B, int k, int V,
                          int32_t *out_tok, int32_t *accepted, uint32_t *counters, void *scratch, uint32_t *status,
                          const AcceptShape &sh, const float2 *stats_p, const float2 *stats_q, cudaStream_t s);

// Softmax of logit rows (softmax.cu): stats[r] = (max, sum) of row r; the
// probabilities expf(z - max) / sum written out; the draft draw.
// Row statistics take one warp per (row, 512-entry block) and keep the
// blocks' partial pairs in `scratch` (row_stats_scratch_bytes(R1 + R2, V));
// a second launch merges each row's pairs.  The rows are those of z1 [R1, V]
// followed by those of z2 [R2, V] (z2 may be null when R2 = 0); stats gets
// R1 + R2 pairs in that order.
size_t row_stats_scratch_bytes(int R, int V);
cudaError_t launch_row_stats(const float *z1, int R1, const float *z2, int R2, int V, float2 *stats, void *scratch,
                             cudaStream_t s);
cudaError_t launch_softmax_write(const float *z, int R, int V, const float2 *stats, float *p, cudaStream_t s);
size_t draft_sample_scratch_bytes(int B, int V);
cudaError_t launch_draft_sample(const float *z, int B, int V, const float *u, int32_t *tok, float2 *stats, float *q,
                                void *scratch, uint32_t *status, cudaStream_t s);
cudaError_t launch_q40_check(uint32_t first, uint32_t count, unsigned long long *mismatches, int num_sms,
                             cudaStream_t s);
cudaError_t launch_exp_check(uint32_t first, uint32_t count, unsigned int *max_rel_bits, int num_sms,
                             cudaStream_t s);

// Hybrid KV cache (kvcache.cu): the K/V rows of one pass into the paged
// cache, and the committed lengths after the accept step.
struct KvWrite {
  const uint16_t *y;
  int M, ld, k_col, v_col, HD;
  const int32_t *block_table;
  int B, max_blocks;
  const int32_t *seq_len;
  int rows_per_req, t0;
  uint16_t *k_cache, *v_cache;
  int num_blocks, block_size;
  uint32_t *status;
};
cudaError_t launch_kv_write(const KvWrite &a, int num_sms, cudaStream_t s);
cudaError_t launch_kv_commit(const int32_t *accepted, int B, int32_t *seq_len, cudaStream_t s);

}  // namespace mlora
