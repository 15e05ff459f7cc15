// The hybrid KV cache (InvisibleLoRA abstract): one paged cache serves both
// passes.  The LoRA-off draft steps write their speculative K/V rows into the
// LoRA-on target's cache, the verify pass overwrites those slots with
// LoRA-conditioned rows, and the accept step's counts move each request's
// committed length past the kept drafts.
//
// Layout: K and V caches are [num_blocks, block_size, H*D] bf16; position pos
// of request b lives in block block_table[b * max_blocks + pos / block_size]
// at offset pos % block_size.  Row m of a pass belongs to request
// b = m / rows_per_req at step t = m % rows_per_req and goes to position
// seq_len[b] + t0 + t; its K and V come from the fused q|k|v projection's
// output row, columns [k_col, k_col + H*D) and [v_col, v_col + H*D).
//
// The copy is HBM-bound and tiny (2 * H*D * 2 bytes per row, a few MB per
// pass), so the kernel is latency-bound: one CTA per row, 16-byte pieces,
// every thread with at most a few pieces in flight; the slot is computed by
// every thread from two broadcast loads.  Slots outside the cache or the
// request's table are skipped and raise MLORA_DEV_BAD_SLOT; a request with a
// negative seq_len is an unused slot of the batch and is skipped silently.
#include "common.cuh"
#include "launch.h"

namespace mlora {

constexpr int KV_THREADS = 128;

__device__ __forceinline__ uint4 ldg_nc_v4(const uint16_t *p) {
  return __ldg(reinterpret_cast<const uint4 *>(p));
}

// VEC: every row segment starts on a 16-byte boundary and H*D is a multiple
// of 8 (checked on the host); otherwise one 16-bit word per thread and step.
template <bool VEC>
__global__ void __launch_bounds__(KV_THREADS)
    kv_write_kernel(const uint16_t *__restrict__ y, int M, long long ld, int k_col, int v_col, int HD,
                    const int32_t *__restrict__ block_table, int B, int max_blocks,
                    const int32_t *__restrict__ seq_len, int rows_per_req, int t0, uint16_t *__restrict__ kc,
                    uint16_t *__restrict__ vc, int num_blocks, int block_size, uint32_t *status) {
  grid_launch_dependents();
  grid_dependency_wait();  // y comes from the projection just before
  for (int m = blockIdx.x; m < M; m += gridDim.x) {
    const int b = m / rows_per_req, t = m - b * rows_per_req;
    if (b >= B) break;  // rows past the batch (the host keeps M <= B * rows_per_req)
    const int L = seq_len[b];
    if (L < 0) continue;  // unused request slot
    const long long pos = (long long)L + t0 + t;
    const long long j = pos / block_size;
    const int blk = j < max_blocks ? block_table[(size_t)b * max_blocks + j] : -1;
    if (blk < 0 || blk >= num_blocks) {
      if (threadIdx.x == 0) raise_status(status, MLORA_DEV_BAD_SLOT);
      continue;
    }
    const size_t dst = ((size_t)blk * block_size + (size_t)(pos - j * block_size)) * (size_t)HD;
    const uint16_t *src = y + (size_t)m * ld;
    if (VEC) {
      const int n8 = HD / 8;
      for (int c = threadIdx.x; c < 2 * n8; c += KV_THREADS) {
        const bool isv = c >= n8;
        const int e = (isv ? c - n8 : c) * 8;
        const uint4 v = ldg_nc_v4(src + (isv ? v_col : k_col) + e);
        *reinterpret_cast<uint4 *>((isv ? vc : kc) + dst + e) = v;
      }
    } else {
      for (int c = threadIdx.x; c < 2 * HD; c += KV_THREADS) {
        const bool isv = c >= HD;
        const int e = isv ? c - HD : c;
        (isv ? vc : kc)[dst + e] = src[(isv ? v_col : k_col) + e];
      }
    }
  }
}

// seq_len[b] += accepted[b] + 1 for every used request slot.
__global__ void __launch_bounds__(256)
    kv_commit_kernel(const int32_t *__restrict__ accepted, int B, int32_t *__restrict__ seq_len) {
  grid_launch_dependents();
  grid_dependency_wait();  // the counts come from the accept step just before
  const int b = blockIdx.x * blockDim.x + threadIdx.x;
  if (b < B) {
    const int L = seq_len[b];
    if (L >= 0) seq_len[b] = L + accepted[b] + 1;
  }
}

cudaError_t launch_kv_write(const KvWrite &a, int num_sms, cudaStream_t s) {
  if (a.M <= 0) return cudaSuccess;
  const int grid = a.M < num_sms * 16 ? a.M : num_sms * 16;
  auto aligned16 = [](const void *p) { return ((uintptr_t)p & 15u) == 0; };
  const bool vec = a.HD % 8 == 0 && a.ld % 8 == 0 && a.k_col % 8 == 0 && a.v_col % 8 == 0 && aligned16(a.y) &&
                   aligned16(a.k_cache) && aligned16(a.v_cache);
  if (vec)
    return launch_pdl(kv_write_kernel<true>, dim3((unsigned)grid), dim3(KV_THREADS), 0, s, a.y, a.M, (long long)a.ld,
                      a.k_col, a.v_col, a.HD, a.block_table, a.B, a.max_blocks, a.seq_len, a.rows_per_req, a.t0,
                      a.k_cache, a.v_cache, a.num_blocks, a.block_size, a.status);
  return launch_pdl(kv_write_kernel<false>, dim3((unsigned)grid), dim3(KV_THREADS), 0, s, a.y, a.M, (long long)a.ld,
                    a.k_col, a.v_col, a.HD, a.block_table, a.B, a.max_blocks, a.seq_len, a.rows_per_req, a.t0,
                    a.k_cache, a.v_cache, a.num_blocks, a.block_size, a.status);
}

cudaError_t launch_kv_commit(const int32_t *accepted, int B, int32_t *seq_len, cudaStream_t s) {
  if (B <= 0) return cudaSuccess;
  return launch_pdl(kv_commit_kernel, dim3((unsigned)((B + 255) / 256)), dim3(256), 0, s, accepted, B, seq_len);
}

}  // namespace mlora
