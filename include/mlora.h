/*
 * mlora.h - C ABI of the multi-LoRA decode hot path for GB300 (sm_103a).
 *
 * Two operations, as the InvisibleLoRA abstract ("InvisibleLoRA: Fast
 * Multi-LoRA Serving Without Per-Token LoRA Decoding") uses them:
 *
 *   mlora_linear         the batched multi-adapter linear layer
 *                          draft  (LoRA off):  y = W x
 *                          verify (LoRA on):   y = W x + scale * B_a (A_a x)
 *                        with a = adapter_idx[row] chosen per token row.  The
 *                        formula is "output = W·x + scale · B(A·x)" of "Multi-
 *                        LoRA Serving in Practice", section "Core Principle:
 *                        Shared Base Model, Per-Request Adapter Selection".
 *   mlora_linear_sliced  the same layer for projections that share their
 *                        input rows (q/k/v, gate/up), in one launch
 *   mlora_verify_accept  the per-request accept / resample step that ends the
 *                        verify pass and keeps the target distribution
 *                        (speculative sampling; exact integer residual draw).
 *
 * Conventions for every entry point:
 *   - All array pointers are DEVICE pointers to caller-owned memory, unless a
 *     parameter says otherwise.  The library never allocates, frees or keeps
 *     a pointer past the call.
 *   - Every call is asynchronous on `stream` (a cudaStream_t; NULL = legacy
 *     default stream) and never synchronises, except mlora_read_device_status.
 *   - Errors a host can see (null pointers, sizes, alignment, workspace size)
 *     are returned at once and nothing is launched.  Errors only the device can
 *     see (bad adapter index, bad rank, NaN probability, timed-out wait) set
 *     bits in a status word inside the workspace; the affected rows are
 *     computed by the documented fallback and no kernel traps.
 *   - bf16 tensors are passed as uint16_t bit patterns (mlora_bf16).
 *   - Row-major layouts throughout.  Pointers to bf16 matrices read by the
 *     tensor-memory engine (x, W) must be 16-byte aligned and K % 8 == 0.
 *
 * Workspace: one caller-allocated device buffer, at least the size the
 * matching *_workspace_bytes function returns and 256-byte aligned.  It holds
 * a status word, zero-initialised arrival counters and scratch.  Call
 * mlora_workspace_init once after allocating it (and after any call that
 * returned MLORA_ERR_TIMEOUT).  Kernels leave the counters at zero when they
 * finish, so one workspace serves any sequence of calls on one stream.  Calls
 * that use the same workspace must not overlap in time (e.g. on two streams):
 * layer calls of either mode may use its scratch (the stream-K GEMM keeps
 * partial sums there).  A decode step that plans its verify pass on a second
 * stream while it drafts gives the draft calls a workspace of their own.
 */
#ifndef MLORA_H
#define MLORA_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define MLORA_API __attribute__((visibility("default")))
#else
#define MLORA_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef uint16_t mlora_bf16;   /* bf16 bit pattern */
typedef void *mlora_stream;    /* cudaStream_t */

typedef enum {
  MLORA_OK = 0,
  MLORA_ERR_ARG = 1,           /* null pointer, bad enum, misaligned pointer */
  MLORA_ERR_SHAPE = 2,         /* a size outside the supported range */
  MLORA_ERR_WORKSPACE = 3,     /* workspace missing, too small or misaligned */
  MLORA_ERR_CUDA = 4,          /* a CUDA runtime / driver call failed */
  MLORA_ERR_DEVICE_STATUS = 5, /* returned by mlora_read_device_status when bits are set */
  MLORA_ERR_TIMEOUT = 6,       /* returned by mlora_read_device_status when a device wait gave up */
  MLORA_ERR_UNSUPPORTED = 7    /* current device is not compute capability 10.3 */
} mlora_status;

typedef enum {
  MLORA_DRAFT = 0,   /* LoRA off: y = W x */
  MLORA_VERIFY = 1,  /* LoRA on:  y = W x + scale * B_a (A_a x) */
  /* Flag, OR-ed into the mode: W is constant while the stream runs (model
   * weights), so the call may start streaming W before the preceding kernel
   * on the stream has finished.  Activations, rank_of, adapter_idx, A and B
   * are still read only after it finishes. */
  MLORA_PREFETCH_WEIGHTS = 0x100
} mlora_mode;

/* Device status bits (mlora_read_device_status). */
#define MLORA_DEV_BAD_ADAPTER (1u << 0) /* adapter_idx outside [-1, n_adapters): row ran base-only */
#define MLORA_DEV_BAD_RANK    (1u << 1) /* rank_of[a] outside [0, r_max]: adapter ran base-only   */
#define MLORA_DEV_BAD_PROB    (1u << 2) /* a probability or uniform read was NaN or outside [0,1] */
#define MLORA_DEV_BAD_TOKEN   (1u << 3) /* a draft token outside [0, V): rejected at its position */
#define MLORA_DEV_ZERO_MASS   (1u << 4) /* residual mass 0: drew from p_n, or emitted token 0     */
#define MLORA_DEV_TIMEOUT     (1u << 5) /* a bounded wait inside a kernel gave up                 */
#define MLORA_DEV_BAD_PLAN    (1u << 6) /* a plan entry read by a layer kernel was out of range (the
                                           workspace's plan was overwritten, or made for other
                                           sizes): the access was skipped, outputs are wrong    */
#define MLORA_DEV_BAD_SLOT    (1u << 7) /* a KV row's slot was outside the cache or the request's
                                           block table: the row was not written                 */

/* Supported ranges. */
#define MLORA_MAX_RANK 64          /* r_max <= 64, r_max % 8 == 0 */
#define MLORA_MAX_ADAPTERS 4096
#define MLORA_MAX_ROWS 65536
#define MLORA_MAX_VOCAB (1 << 24)
#define MLORA_MAX_SLICES 4         /* output slices of one mlora_linear_sliced call */

/* ------------------------------------------------------------------------- */
/* Workspace                                                                  */
/* ------------------------------------------------------------------------- */

/* Bytes of workspace mlora_plan_segments / mlora_shrink / mlora_linear need for
 * M rows, N outputs, K inputs and n_adapters resident adapters, on the
 * current device (it grows with M * K: verify mode keeps a copy of the token
 * rows in adapter-sorted order).  One workspace sized for the largest
 * (M, N, K) of a set of projections serves all of them.  Returns 0 for sizes
 * outside the ranges. */
MLORA_API size_t mlora_linear_workspace_bytes(int M, int N, int K, int n_adapters);

/* Bytes of workspace mlora_linear_sliced needs with n_slices output slices
 * (1..MLORA_MAX_SLICES); equal to mlora_linear_workspace_bytes for one. */
MLORA_API size_t mlora_linear_sliced_workspace_bytes(int M, int N, int K, int n_adapters, int n_slices);

/* Bytes of workspace mlora_verify_accept needs (B requests, k drafts, V vocab). */
MLORA_API size_t mlora_accept_workspace_bytes(int B, int k, int V);

/* Zero the status word and the arrival counters (asynchronous memset). */
MLORA_API mlora_status mlora_workspace_init(void *workspace, size_t ws_bytes, mlora_stream stream);

/* Copy the device status bits to *bits (host pointer), optionally clearing
 * them.  Synchronises `stream`.  Returns MLORA_OK if no bit is set,
 * MLORA_ERR_TIMEOUT if MLORA_DEV_TIMEOUT is set, else MLORA_ERR_DEVICE_STATUS. */
MLORA_API mlora_status mlora_read_device_status(void *workspace, uint32_t *bits, int clear, mlora_stream stream);

/* ------------------------------------------------------------------------- */
/* Segment plan (step a1)                                                     */
/* ------------------------------------------------------------------------- */

/* Group token rows by adapter: a stable counting sort of adapter_idx.
 * The InvisibleLoRA abstract notes that requests are partitioned across the
 * active adapters; "Multi-LoRA Serving in Practice", section "4. Batching:
 * Heterogeneous LoRAs Break 'Neat' Batches", asks to aggregate requests of
 * the same adapter.
 *
 *   adapter_idx  int32 [M]   adapter of each row; -1 = base only
 *   rank_of      int32 [n_adapters]  rank of each resident adapter
 *   r_max        row stride of A_stack / column stride of B_stack (<= 64, % 8 == 0)
 *
 * Writes the plan into the workspace and returns device pointers into it:
 *   *seg_offsets  int32 [n_adapters + 2]: rows of adapter a sit at sorted
 *                 positions [seg_offsets[a], seg_offsets[a+1]); bucket
 *                 n_adapters holds rows without a (valid) adapter.
 *   *perm         int32 [M]: perm[sorted position] = row; increasing within
 *                 a bucket.
 * Either output pointer may be NULL.  The plan depends only on adapter_idx,
 * rank_of, n_adapters and r_max, so one plan serves every projection of a
 * decode step that shares them (pass *seg_offsets to mlora_linear). */
MLORA_API mlora_status mlora_plan_segments(const int32_t *adapter_idx, int M, const int32_t *rank_of, int n_adapters,
                                 int r_max, void *workspace, size_t ws_bytes, const int32_t **seg_offsets,
                                 const int32_t **perm, mlora_stream stream);

/* ------------------------------------------------------------------------- */
/* Shrink (step a2)                                                           */
/* ------------------------------------------------------------------------- */

/* Low-rank activations T[m, j] = sum_k A_a[j, k] x[m, k] for j < rank_of[a],
 * a = adapter_idx[m] (the inner product A·x of "output = W·x + scale · B(A·x)").
 *
 *   x        bf16 [M, K]          A_stack  bf16 [n_adapters, r_max, K]
 *   T        fp32 [M, r_max] out: zero where j >= rank and on rows without
 *            a valid adapter; fp32 accumulation.
 *   seg_offsets  the pointer mlora_plan_segments returned for this workspace.
 * Rows of A past rank_of[a] are never read. */
MLORA_API mlora_status mlora_shrink(const mlora_bf16 *x, int M, int K, const mlora_bf16 *A_stack, int n_adapters, int r_max,
                          const int32_t *seg_offsets, float *T, void *workspace, size_t ws_bytes,
                          mlora_stream stream);

/* ------------------------------------------------------------------------- */
/* Multi-adapter linear layer (steps a1-a4)                                   */
/* ------------------------------------------------------------------------- */

/* y = W x (mode MLORA_DRAFT) or y = W x + scale * B_a[:, :r] (A_a[:r, :] x)
 * (mode MLORA_VERIFY), per row, a = adapter_idx[row], r = rank_of[a].
 *
 *   x        bf16 [M, K]   token rows (verify rows are request-major:
 *                          row = request * (k+1) + t)
 *   W        bf16 [N, K]   base weight (out x in)
 *   A_stack  bf16 [n_adapters, r_max, K]   B_stack  bf16 [n_adapters, N, r_max]
 *            (only the first rank_of[a] rows of A_a / columns of B_a are read;
 *            may be NULL in draft mode, as may rank_of and adapter_idx)
 *   seg_offsets  NULL: plan first (step a1) into the workspace.  Otherwise the
 *            pointer mlora_plan_segments returned for this workspace and the
 *            same adapter_idx / rank_of / n_adapters / r_max.
 *   scale    LoRA scaling (alpha / r), one scalar per call
 *   y        bf16 [M, N] out, rows in input order; fp32 accumulation, one
 *            round to nearest even at the end.
 *
 * The base product runs on the tcgen05 tensor cores (bf16 in, fp32 in tensor
 * memory); the low-rank expand is fused into its epilogue.  Results are
 * deterministic: the same inputs give the same bits on every call. */
MLORA_API mlora_status mlora_linear(const mlora_bf16 *x, int M, int K, const mlora_bf16 *W, int N,
                          const mlora_bf16 *A_stack, const mlora_bf16 *B_stack, int n_adapters, int r_max,
                          const int32_t *rank_of, const int32_t *adapter_idx, const int32_t *seg_offsets,
                          float scale, int mode, mlora_bf16 *y, void *workspace, size_t ws_bytes,
                          mlora_stream stream);

/* The same layer for several projections that read the same rows x, in one
 * launch of each kernel: q, k and v of an attention block, or gate and up of
 * its MLP ("Multi-LoRA Serving in Practice" lists q_proj, k_proj, v_proj,
 * o_proj, gate_proj, up_proj and down_proj as the usual LoRA targets).  The
 * pages define the layer per projection; fusing projections that share their
 * input is this library's layout, not the pages'.  Output slice s covers
 * output features [slice_end[s-1], slice_end[s]) (slice_end[-1] = 0):
 *
 *   y[m, n] = sum_k W[n, k] x[m, k]
 *             + [verify] scale * sum_{j<r} B_a[n, j] * sum_k A_{s,a}[j, k] x[m, k]
 *
 *   W        bf16 [N, K]   the projections' weights stacked along N
 *   slice_end   HOST int32 [n_slices], 1 <= n_slices <= MLORA_MAX_SLICES,
 *            increasing, each but the last a multiple of 128, the last == N
 *   A_stack  bf16 [n_slices, n_adapters, r_max, K]   each slice's own A
 *   B_stack  bf16 [n_adapters, N, r_max]   each adapter's B of every slice,
 *            stacked along N like W
 *   rank_of  int32 [n_adapters]: one rank per adapter for all its slices
 *   y        bf16 [M, N] out
 * Everything else as mlora_linear; with n_slices = 1 it is mlora_linear.  The
 * workspace must have mlora_linear_sliced_workspace_bytes(M, N, K, n_adapters,
 * n_slices) bytes; a plan from mlora_plan_segments on it serves any number of
 * slices.  Bad slice ends return MLORA_ERR_SHAPE. */
MLORA_API mlora_status mlora_linear_sliced(const mlora_bf16 *x, int M, int K, const mlora_bf16 *W, int N,
                                           int n_slices, const int32_t *slice_end, const mlora_bf16 *A_stack,
                                           const mlora_bf16 *B_stack, int n_adapters, int r_max,
                                           const int32_t *rank_of, const int32_t *adapter_idx,
                                           const int32_t *seg_offsets, float scale, int mode, mlora_bf16 *y,
                                           void *workspace, size_t ws_bytes, mlora_stream stream);

/* Which GEMM kernel a layer call of this shape runs on the current device
 * (the choice is made on the host from the sizes alone): 0 = the cluster
 * split-K kernel, 1 = the persistent stream-K kernel, -1 = sizes or mode
 * outside the supported ranges (or no CUDA device).  For observability and
 * profiling; the results of a call do not depend on it beyond fp32
 * summation order.  n_adapters and r_max matter in verify mode only. */
MLORA_API int mlora_linear_gemm_kernel(int M, int N, int K, int n_adapters, int r_max, int mode);

/* Test hook for the failure path of the stream-K GEMM's cross-CTA wait (no
 * counterpart on the pages).  With ns > 0, every later layer call that runs
 * the stream-K kernel (see mlora_linear_gemm_kernel) makes the owner of each
 * split tile wait up to ns nanoseconds on flag words that no CTA sets,
 * instead of on its contributors' flags: the wait gives up, the tile is
 * finished without the contributors' partial sums (wrong values) and
 * MLORA_DEV_TIMEOUT is raised in the workspace status word.  The
 * contributors' own flags stay set, so the caller must run
 * mlora_workspace_init before the workspace's next call.  ns = 0 (the default)
 * restores normal operation.  Process-wide; not for use while other threads
 * issue layer calls.  Nothing waits on a peer that cannot arrive, so no call
 * hangs or faults. */
MLORA_API void mlora_debug_set_flag_wait_ns(uint32_t ns);

/* Test hook for the draw's weights (no counterpart on the pages): the
 * kernels compute Q(f) = floor(f * 2^40) of a probability clamped to [0, 1]
 * from the bits of f with integer operations.  For the `count` fp32 bit
 * patterns first_bits, first_bits + 1, ... this adds to *mismatches (device
 * memory, caller-owned, caller-zeroed) the number whose Q differs from
 * CUDA's round-down conversion of the clamped f * 2^40.  Asynchronous on
 * `stream`.  MLORA_ERR_ARG when the range passes 2^32 or mismatches is NULL. */
MLORA_API mlora_status mlora_debug_q40_mismatches(uint32_t first_bits, uint32_t count,
                                                  unsigned long long *mismatches, mlora_stream stream);

/* Test hook for the probability expression (no counterpart on the pages):
 * the kernels compute e^d as 2^(d log2 e) with the PTX ex2.approx
 * instruction.  For the `count` fp32 bit patterns first_bits,
 * first_bits + 1, ... whose CUDA expf is a normal float, this raises
 * *max_rel_bits (device memory, caller-owned, caller-zeroed; the bit pattern
 * of a non-negative float) to the largest |e^d - expf(d)| / expf(d).
 * Asynchronous on `stream`.  MLORA_ERR_ARG when the range passes 2^32 or the
 * pointer is NULL. */
MLORA_API mlora_status mlora_debug_exp_max_rel_error(uint32_t first_bits, uint32_t count, unsigned int *max_rel_bits,
                                                     mlora_stream stream);

/* Which kernel writes the low-rank operand (the token windows of
 * bf16(scale * A_a x)) in later verify-mode layer calls (no counterpart on the
 * pages, which compute the per-adapter product without naming a kernel):
 *   MLORA_SHRINK_AUTO    the library's choice from the call's sizes (default);
 *   MLORA_SHRINK_WARP    warp items of 8 rank rows x 4 tokens (CUDA cores);
 *   MLORA_SHRINK_TENSOR  128-row tcgen05 tiles over 8 expand blocks' tokens.
 * The two differ only in fp32 summation order.  Process-wide; not for use
 * while other threads issue layer calls.  Returns MLORA_ERR_ARG for another
 * value.  mlora_shrink (the T output) always runs the warp items. */
#define MLORA_SHRINK_AUTO   0
#define MLORA_SHRINK_WARP   1
#define MLORA_SHRINK_TENSOR 2
MLORA_API mlora_status mlora_set_shrink_path(int path);

/* Allocation-free variant of mlora_linear.  The paper has no counterpart;
 * this is for callers that cannot allocate device memory for a workspace (a
 * plugin inside a host framework that owns every device buffer, or code
 * whose device memory budget is fixed at start-up and must not call
 * cudaMalloc).  Same arguments and results as mlora_linear, minus the plan
 * pointer and the workspace: the scratch (segment plan, low-rank activations
 * and status word) lives in one 512 KB array compiled into the library, which
 * every GPU that loads the library holds until the process exits.
 *   Limits: M <= 1024 rows and, in verify mode, n_adapters <= 256; larger
 *   sizes return MLORA_ERR_SHAPE and launch nothing.
 *   The first call on each device looks up the array's device address
 *   (cudaGetSymbolAddress) with that device current and keeps it; make that
 *   first call before any stream capture.
 *   It calls no allocating routine.  All calls share the array: calls whose
 *   work overlaps on the GPU (e.g. on two streams) race.  Device status bits
 *   (bad adapter index or rank) still select the same fallback but are not
 *   reported by this variant. */
MLORA_API mlora_status mlora_linear_noalloc(const mlora_bf16 *x, int M, int K, const mlora_bf16 *W, int N,
                                            const mlora_bf16 *A_stack, const mlora_bf16 *B_stack, int n_adapters,
                                            int r_max, const int32_t *rank_of, const int32_t *adapter_idx,
                                            float scale, int mode, mlora_bf16 *y, mlora_stream stream);

/* ------------------------------------------------------------------------- */
/* Accept / resample (steps a5-a6)                                            */
/* ------------------------------------------------------------------------- */

/* Speculative verification that keeps the target distribution (InvisibleLoRA
 * abstract: one LoRA-on pass verifies all proposals and preserves the output
 * distribution).  Per request b, with p = target, q = draft probabilities:
 *   1. keep draft x_i while (double)u_i * q_i(x_i) < p_i(x_i); n = first
 *      failing position (k if none fails);
 *   2. weights w(v) = max(0, Q(p_n(v)) - Q(q_n(v))) if n < k, else Q(p_k(v)),
 *      Q(f) = floor(f * 2^40);
 *   3. S = sum w, U = floor(u_k * 2^32), T = floor(U * S / 2^32); draw the
 *      smallest v whose running sum of w exceeds T.
 * Every decision is exact integer / exact float64 arithmetic, so results are
 * bit-reproducible.
 *
 * Launches: when V % 4 == 0 and p_target and q_draft are 16-byte aligned, a
 * streaming kernel (one CTA per SM, bulk copies through shared memory) and a
 * dependent draw kernel; otherwise one kernel with a CTA per (request,
 * 4096-entry chunk).  Both give the same tokens, status bits and counts.
 * All pointers are device memory owned by the caller; the call is
 * asynchronous on `stream`; workspace: mlora_accept_workspace_bytes(B, k, V).
 *
 *   p_target  fp32 [B, k+1, V]     q_draft  fp32 [B, k, V]
 *   draft_tok int32 [B, k]         uniforms fp32 [B, k+1] in [0, 1)
 *   out_tok   int32 [B, k+1] out:  kept drafts, the drawn token, then -1
 *   accepted  int32 [B] out:       n in [0, k]
 * B in [1, 32768], k in [1, 16], V in [1, 2^24].  Fallbacks: probability NaN/negative -> 0,
 * above 1 -> 1 (MLORA_DEV_BAD_PROB); uniform NaN/negative -> 0, >= 1 -> the
 * largest float below 1; a draft token outside [0, V) is rejected at its
 * position (MLORA_DEV_BAD_TOKEN); zero residual mass draws from p_n, and zero
 * mass there emits token 0 (MLORA_DEV_ZERO_MASS). */
MLORA_API mlora_status mlora_verify_accept(const float *p_target, const float *q_draft, const int32_t *draft_tok,
                                 const float *uniforms, int B, int k, int V, int32_t *out_tok, int32_t *accepted,
                                 void *workspace, size_t ws_bytes, mlora_stream stream);

/* The same step taking logits instead of probabilities: z_target [B, k+1, V]
 * are the LoRA-on pass's logits, z_draft [B, k, V] the LoRA-off passes'.  The
 * softmax is fused into the accept kernels: every probability they read is
 * e^(z - m) * R of its row, with the row statistics of mlora_softmax, so the
 * decisions are exactly those mlora_verify_accept takes on the probabilities
 * mlora_softmax writes for the same logits.  Everything else as
 * mlora_verify_accept; workspace mlora_accept_workspace_bytes(B, k, V).  The
 * pages give no formula for the distributions; the softmax of the logits at
 * temperature 1 is the plain reading of a language model's output. */
MLORA_API mlora_status mlora_verify_accept_logits(const float *z_target, const float *z_draft,
                                                  const int32_t *draft_tok, const float *uniforms, int B, int k, int V,
                                                  int32_t *out_tok, int32_t *accepted, void *workspace,
                                                  size_t ws_bytes, mlora_stream stream);

/* ------------------------------------------------------------------------- */
/* Softmax and the draft draw (the steps on either side of the accept step)  */
/* ------------------------------------------------------------------------- */

/* p[r, v] = e^(z[r, v] - m_r) * R_r for `rows` rows of V fp32 logits, with
 * m_r the row maximum, S_r the row's sum of e^(z - m_r) (accumulated in a
 * fixed order in fp32: the results are deterministic, and a row's values do
 * not depend on the other rows of the call) and R_r = 1/S_r rounded once.
 * e^d is computed as 2^(d log2 e) with the PTX ex2.approx instruction.  The
 * InvisibleLoRA abstract has both passes end in a distribution over the
 * vocabulary; the softmax of the logits is the plain reading.
 *   z, p   fp32 [rows, V] device (p may not alias z); rows in [1, 65536],
 *          V in [1, 2^24]; workspace mlora_softmax_workspace_bytes(rows, V). */
MLORA_API size_t mlora_softmax_workspace_bytes(int rows, int V);
MLORA_API mlora_status mlora_softmax(const float *z, int rows, int V, float *p, void *workspace, size_t ws_bytes,
                                     mlora_stream stream);

/* The draft token of each request from its LoRA-off logits (the InvisibleLoRA
 * abstract: the LoRA-off pass proposes the next token for every request):
 * q = softmax(z_draft[b]) as mlora_softmax computes it, then the exact integer
 * inverse CDF of Q(q) = floor(q * 2^40) with U = floor(uniforms[b] * 2^32),
 * the same draw the accept step uses for its residual.
 *   z_draft  fp32 [B, V] logits;  uniforms fp32 [B];  draft_tok int32 [B] out;
 *   q_out    fp32 [B, V] out, or NULL: the probabilities the draw used (what
 *            mlora_verify_accept takes as q; mlora_verify_accept_logits takes
 *            the logits instead).
 * Uniforms outside [0, 1) are clamped as in the accept step
 * (MLORA_DEV_BAD_PROB); a row of zero mass draws token 0 (MLORA_DEV_ZERO_MASS).
 * Workspace mlora_draft_sample_workspace_bytes(B, V). */
MLORA_API size_t mlora_draft_sample_workspace_bytes(int B, int V);
MLORA_API mlora_status mlora_draft_sample(const float *z_draft, int B, int V, const float *uniforms,
                                          int32_t *draft_tok, float *q_out, void *workspace, size_t ws_bytes,
                                          mlora_stream stream);

/* ------------------------------------------------------------------------- */
/* FP8 base weights for the draft pass                                        */
/* ------------------------------------------------------------------------- */

/* The "LoRA Inference" glossary lists quantizing the base weights to 8 bits
 * (INT8/FP8) among the serving optimisations that go with LoRA.  The
 * InvisibleLoRA draft pass runs the base model alone (LoRA off), so it can
 * read an E4M3 copy of W: half the bytes of the HBM-bound pass.  Drafts only
 * propose tokens; the LoRA-on verify pass (bf16 W) and the accept step decide
 * what is emitted, so the output distribution stays exact and only the
 * acceptance rate can change.  Format and rounding (a reading; the pages fix
 * neither): E4M3 (4 exponent bits, bias 7, 3 mantissa bits, largest finite
 * 448), round to nearest with ties to even, saturating at 448; one fp32 scale
 * per row, scale = amax / 448, code = E4M3(v / scale) (IEEE fp32 division);
 * a zero row gets scale 1 and +0 codes.  Inputs must be finite. */

/* Quantize bf16 rows src [R, K] (row-major) to E4M3 codes q [R, K] and fp32
 * scales [R]: W once, per output row, before the draft passes.  K % 16 == 0;
 * src and q 16-byte aligned.  Asynchronous on `stream`. */
MLORA_API mlora_status mlora_quantize_rows_fp8(const mlora_bf16 *src, int R, int K, uint8_t *q, float *scale,
                                               mlora_stream stream);

/* The draft (LoRA-off) layer on FP8 weights:
 *   y[m, n] = bf16_rn(x_scale[m] * w_scale[n] * sum_k Xq[m, k] * Wq[n, k])
 * with x quantized per token row into the workspace by the same rule, W8 and
 * w_scale from mlora_quantize_rows_fp8, products exact and sums in fp32 on
 * the tensor cores (kind::f8f6f4).  x bf16 [M, K], W8 uint8 [N, K], y bf16
 * [M, N]; 1 <= M <= 256, K % 16 == 0; x and W8 16-byte aligned.  flags: 0 or
 * MLORA_PREFETCH_WEIGHTS (W8 is constant: its first tiles may stream before
 * the preceding kernel ends).  Workspace: mlora_linear_fp8_workspace_bytes
 * (M, N, K), initialised once with mlora_workspace_init; calls sharing it
 * must not overlap.  MLORA_ERR_UNSUPPORTED if a CTA of the shape cannot be
 * resident on every SM at once. */
MLORA_API size_t mlora_linear_fp8_workspace_bytes(int M, int N, int K);
MLORA_API mlora_status mlora_linear_fp8(const mlora_bf16 *x, int M, int K, const uint8_t *W8, const float *w_scale,
                                        int N, mlora_bf16 *y, int flags, void *workspace, size_t ws_bytes,
                                        mlora_stream stream);

/* ------------------------------------------------------------------------- */
/* Hybrid KV cache                                                            */
/* ------------------------------------------------------------------------- */

/* The InvisibleLoRA abstract has one KV cache for both passes: the LoRA-off
 * drafter writes its speculative K/V entries into the cache of the LoRA-on
 * target, and the verification pass overwrites them, so the drafter reads
 * LoRA-conditioned K/V for the committed prefix and needs no cache of its
 * own.  The pages give no layout; this one is a paged cache:
 *   k_cache, v_cache  bf16 [num_blocks, block_size, H, D] each (caller-owned,
 *                     16-byte aligned for the vectorised copy, else a slower
 *                     word-by-word copy);
 *   block_table       int32 [B, max_blocks]: request b's position pos lives in
 *                     block block_table[b][pos / block_size] at offset
 *                     pos % block_size;
 *   seq_len           int32 [B]: request b's committed tokens (K/V in the cache
 *                     with LoRA-on values); negative = unused request slot.
 *
 * mlora_kv_write copies the K and V rows of one pass:
 *   y       bf16 [M, ld]: the fused q|k|v projection's output (mlora_linear
 *           or mlora_linear_sliced); K of row m = y[m, k_col : k_col + H*D],
 *           V = y[m, v_col : v_col + H*D], H heads of D contiguous values;
 *   rows_per_req  1 for a draft step (one row per request), k + 1 for the
 *           verify pass: row m is request m / rows_per_req at step
 *           t = m % rows_per_req (M <= B * rows_per_req);
 *   t0      the draft step (0 .. k-1) in the draft pass, 0 in the verify pass:
 *           row m goes to position seq_len[b] + t0 + t.
 * So in one decode cycle draft step t writes position L + t (L = seq_len[b]),
 * the verify pass writes L .. L + k over them, and mlora_kv_commit then sets
 * seq_len[b] = L + accepted[b] + 1 (the pending token and the kept drafts);
 * slots past it are stale and the next cycle overwrites them.
 * A slot outside [0, num_blocks) or past the table is not written and raises
 * MLORA_DEV_BAD_SLOT; rows of unused request slots are skipped.  Asynchronous
 * on `stream`; the workspace (any of this library's, at least
 * mlora_kv_workspace_bytes() bytes) holds only the status word.  Returns
 * MLORA_ERR_SHAPE for sizes outside the ranges (column ranges past ld,
 * M > B * rows_per_req, H*D > 2^20), MLORA_ERR_ARG for a null pointer (y may
 * be NULL when M = 0). */
MLORA_API size_t mlora_kv_workspace_bytes(void);
MLORA_API mlora_status mlora_kv_write(const void *y, int M, int ld, int k_col, int v_col, int H, int D,
                                      const int32_t *block_table, int B, int max_blocks, const int32_t *seq_len,
                                      int rows_per_req, int t0, void *k_cache, void *v_cache, int num_blocks,
                                      int block_size, void *workspace, size_t ws_bytes, mlora_stream stream);

/* seq_len[b] += accepted[b] + 1 for every used request slot (seq_len[b] >= 0);
 * accepted as the accept step writes it (0..k).  Asynchronous on `stream`. */
MLORA_API mlora_status mlora_kv_commit(const int32_t *accepted, int B, int32_t *seq_len, mlora_stream stream);

/* ------------------------------------------------------------------------- */
/* Run-time draft gate (host functions; no GPU needed)                        */
/* ------------------------------------------------------------------------- */

/* The InvisibleLoRA abstract has a run-time gate skip drafting on steps where
 * the adapter cost cannot repay a draft pass.  The cost model (a reading; the
 * pages give none) is speculative decoding's: with draft length k and each
 * draft kept with probability alpha, a decode cycle emits on average
 * E(alpha, k) = 1 + alpha + ... + alpha^k tokens per request. */

/* E(alpha, k) for alpha in [0, 1], k >= 0; 0 for arguments outside. */
MLORA_API double mlora_expected_tokens(double alpha, int k);

/* The draft length to use: t_cycle (HOST, [k_max + 1], entry 0 unused) holds
 * the measured time of a decode cycle with k drafts (k LoRA-off passes, the
 * LoRA-on pass over k + 1 rows per request, the accept step), t_plain the
 * time of one plain LoRA-on decode step of the same requests.  Returns the k
 * in [1, k_max] with the highest rate E(alpha, k) / t_cycle[k] if it beats
 * 1 / t_plain (the smallest such k on ties), else 0 (skip drafting); *gain
 * (optional) receives that best rate times t_plain.  Returns -1 for null
 * t_cycle, k_max outside [1, 64], a time that is not positive or alpha outside
 * [0, 1]. */
MLORA_API int mlora_draft_gate(const double *t_cycle, int k_max, double t_plain, double alpha, double *gain);

/* Maximum-likelihood acceptance rate from the kept-draft counts (HOST array
 * accepted[B], as mlora_verify_accept returns them, each clamped to [0, k]):
 * sum n / (sum n + number of requests with n < k); 0 when undefined. */
MLORA_API double mlora_estimate_acceptance(const int32_t *accepted, int B, int k);

/* ------------------------------------------------------------------------- */
/* Misc                                                                       */
/* ------------------------------------------------------------------------- */

MLORA_API const char *mlora_status_string(mlora_status s);

/* 1 if the current device can run the kernels (compute capability 10.3, the
 * only target the library is built for), else 0. */
MLORA_API int mlora_device_supported(void);

/* Number of kernels this library launched since load (all entry points). */
MLORA_API uint64_t mlora_launch_count(void);

#ifdef __cplusplus
}
#endif

#endif /* MLORA_H */
