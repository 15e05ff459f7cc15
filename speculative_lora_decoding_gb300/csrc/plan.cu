// Step a1, the segment plan: a stable counting sort of token rows by adapter.
//
// The InvisibleLoRA abstract observes that requests are partitioned across the
// active adapters, and "Multi-LoRA Serving in Practice" (section "4. Batching:
// Heterogeneous LoRAs Break 'Neat' Batches") asks to aggregate requests of one
// adapter.  The plan gives, per adapter, the sorted positions of its rows; the
// shrink kernel reads each adapter's A once per group and the GEMM epilogue
// keeps each adapter's B row in registers across its group.
//
// One CTA of 256 threads: histogram in shared memory, block-wide scans for
// the offsets, the active-adapter list, the shrink work list and the expand
// blocks with their token windows (see common.cuh), then a
// warp-sequential ranking (match_any within a warp, warps in order) that
// keeps rows of one bucket in increasing row order, and finally the shrink
// work items written out in full, so that a shrink CTA finds its adapter,
// rank rows and token rows with one load.
#include "common.cuh"
#include "launch.h"

namespace mlora {

constexpr int PLAN_THREADS = 256;

__device__ __forceinline__ int warp_incl_scan(int v) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    int t = __shfl_up_sync(0xffffffffu, v, o);
    if (lane >= o) v += t;
  }
  return v;
}

// Exclusive scan over the block; every thread calls it.  sh: 33 ints.
__device__ int block_excl_scan(int v, int *sh, int *total) {
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  const int inc = warp_incl_scan(v);
  if (lane == 31) sh[w] = inc;
  block_sync();
  if (w == 0) {
    const int s = (lane < (int)(blockDim.x >> 5)) ? sh[lane] : 0;
    const int si = warp_incl_scan(s);
    sh[lane] = si - s;
    if (lane == 31) sh[32] = si;
  }
  block_sync();
  const int res = sh[w] + inc - v;
  *total = sh[32];
  block_sync();
  return res;
}

__device__ __forceinline__ int bucket_of(int a, int n_ad) { return (a >= 0 && a < n_ad) ? a : n_ad; }

__global__ void __launch_bounds__(PLAN_THREADS, 1)
    plan_kernel(const int32_t *__restrict__ adapter_idx, int M, const int32_t *__restrict__ rank_of, int n_ad,
                int r_max, int32_t *__restrict__ plan, uint32_t *status) {
  grid_launch_dependents();
  grid_dependency_wait();
  extern __shared__ int sh_dyn[];
  int *cnt = sh_dyn;                 // [n_ad + 1]: counts, then bucket offsets
  int *running = sh_dyn + n_ad + 1;  // [n_ad + 1]
  __shared__ int scan_sh[33];
  __shared__ uint32_t flags;
  __shared__ int max_rank;
  __shared__ int partial_block;  // an active rank reads padding columns in a 16-wide block

  const PlanLayout L = plan_layout(M, n_ad);
  const int tid = threadIdx.x;
  const int nb = n_ad + 1;
  if (tid == 0) {
    flags = 0;
    max_rank = 0;
    partial_block = 0;
  }
  for (int b = tid; b < nb; b += PLAN_THREADS) {
    cnt[b] = 0;
    running[b] = 0;
  }
  block_sync();

  // Validated ranks.
  for (int a = tid; a < n_ad; a += PLAN_THREADS) {
    int r = rank_of[a];
    if (r < 0 || r > r_max) {
      atomicOr(&flags, MLORA_DEV_BAD_RANK);
      r = 0;
    }
    plan[L.rank_eff + a] = r;
  }
  // Histogram and validated adapter per row.
  for (int m = tid; m < M; m += PLAN_THREADS) {
    const int a = adapter_idx[m];
    if (a < -1 || a >= n_ad) atomicOr(&flags, MLORA_DEV_BAD_ADAPTER);
    const int b = bucket_of(a, n_ad);
    plan[L.row_adapter + m] = (b < n_ad) ? b : -1;
    atomicAdd(&cnt[b], 1);
  }
  block_sync();

  // Bucket offsets: exclusive scan of counts, each thread owning a contiguous run.
  const int per = (nb + PLAN_THREADS - 1) / PLAN_THREADS;
  const int b0 = min(tid * per, nb), b1 = min(b0 + per, nb);
  {
    int local = 0;
    for (int b = b0; b < b1; ++b) local += cnt[b];
    int total;
    int off = block_excl_scan(local, scan_sh, &total);
    for (int b = b0; b < b1; ++b) {
      const int c = cnt[b];
      plan[L.seg_offsets + b] = off;
      running[b] = c;  // keep the count; `cnt` turns into offsets below
      cnt[b] = off;
      off += c;
    }
    if (tid == 0) plan[L.seg_offsets + nb] = total;
  }
  block_sync();

  // Active adapters (rows > 0), the shrink work list and the expand blocks
  // over them.  Adapter a's rows sit at sorted positions [s0, s1) = [cnt[a],
  // cnt[a] + running[a]); its token window is [w0, w1) = [s0 & ~15,
  // (s1 + 15) & ~15), one copy per 16-rank block in the operand buffer.
  {
    const int a0 = min(tid * per, n_ad), a1 = min(a0 + per, n_ad);
    int nact = 0, nitems = 0, rmax = 0, nsl = 0, nwin = 0;
    for (int a = a0; a < a1; ++a) {
      const int c = running[a];
      if (c > 0) {
        ++nact;
        const int r = plan[L.rank_eff + a];
        rmax = max(rmax, r);
        // A 16-wide block of B columns past the rank but inside r_max holds
        // caller padding (possibly NaN); past r_max it reads as zero.
        if ((r % 16) != 0 && r != r_max) partial_block = 1;
        nitems += ((r + SHRINK_J - 1) / SHRINK_J) * ((c + SHRINK_TOK - 1) / SHRINK_TOK);
        const int nblk = (r + 15) / 16;
        const int w0 = cnt[a] & ~15, w1 = (cnt[a] + c + 15) & ~15;
        nsl += nblk;
        nwin += nblk * (w1 - w0);
      }
    }
    if (rmax > 0) atomicMax(&max_rank, rmax);
    int tot_act, tot_items, tot_sl, tot_win;
    int pa = block_excl_scan(nact, scan_sh, &tot_act);
    int pi = block_excl_scan(nitems, scan_sh, &tot_items);
    int ps = block_excl_scan(nsl, scan_sh, &tot_sl);
    int pw = block_excl_scan(nwin, scan_sh, &tot_win);
    for (int a = a0; a < a1; ++a) {
      const int c = running[a];
      if (c > 0) {
        const int r = plan[L.rank_eff + a];
        const int w0 = cnt[a] & ~15, W = ((cnt[a] + c + 15) & ~15) - w0;
        plan[L.active + pa] = a;
        plan[L.item_off + pa] = pi;
        plan[L.slice_off + a] = ps;
        for (int j = 0; j * 16 < r; ++j) {
          int4 *rec = reinterpret_cast<int4 *>(plan + L.slices + (size_t)(ps + j) * EXP_WORDS);
          rec[0] = make_int4(a, 16 * j, min(16, r - 16 * j), pw + j * W);
          rec[1] = make_int4(w0, W, 0, 0);
        }
        ++pa;
        pi += ((r + SHRINK_J - 1) / SHRINK_J) * ((c + SHRINK_TOK - 1) / SHRINK_TOK);
        ps += (r + 15) / 16;
        pw += ((r + 15) / 16) * W;
      }
    }
    if (tid == 0) {
      plan[L.item_off + tot_act] = tot_items;
      plan[L.hdr + 0] = tot_act;
      plan[L.hdr + 1] = tot_items;
      plan[L.hdr + 2] = M;
      plan[L.hdr + 4] = tot_sl;
      plan[L.hdr + 6] = tot_win;
    }
  }
  block_sync();
  if (tid == 0) plan[L.hdr + 5] = partial_block ? 0 : 1;
  block_sync();
  if (tid == 0) plan[L.hdr + 3] = max_rank;
  block_sync();
  for (int b = tid; b < nb; b += PLAN_THREADS) running[b] = 0;
  block_sync();

  // Stable ranks: rows in chunks of PLAN_THREADS; within a warp lanes with
  // the same bucket are ranked by lane order, warps take their turn in order.
  const int lane = tid & 31, warp = tid >> 5;
  for (int base = 0; base < M; base += PLAN_THREADS) {
    const int m = base + tid;
    const int b = (m < M) ? bucket_of(adapter_idx[m], n_ad) : -1 - lane - 2 * PLAN_THREADS;
    const unsigned mask = __match_any_sync(0xffffffffu, b);
    const int leader = __ffs(mask) - 1;
    const int rank_in_warp = __popc(mask & ((1u << lane) - 1u));
    int basev = 0;
    for (int w = 0; w < PLAN_THREADS / 32; ++w) {
      if (warp == w && m < M && lane == leader) {
        basev = running[b];
        running[b] = basev + __popc(mask);
      }
      block_sync();
    }
    basev = __shfl_sync(0xffffffffu, basev, leader);
    if (m < M) plan[L.perm + cnt[b] + basev + rank_in_warp] = m;
  }
  block_sync();

  // Shrink work items, one record each: the item's adapter comes from a
  // binary search of the item offsets (copied to shared memory).
  const int n_active = plan[L.hdr + 0];
  const int total_items = plan[L.hdr + 1];
  int *ioff = running;  // reuse: [n_active + 1] item offsets
  for (int i = tid; i <= n_active; i += PLAN_THREADS) ioff[i] = plan[L.item_off + i];
  block_sync();
  for (int it = tid; it < total_items; it += PLAN_THREADS) {
    int lo = 0, hi = n_active;
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (ioff[mid] <= it) lo = mid; else hi = mid;
    }
    const int a = plan[L.active + lo];
    const int r = plan[L.rank_eff + a];
    const int s0 = plan[L.seg_offsets + a];
    const int c = plan[L.seg_offsets + a + 1] - s0;
    const int local = it - ioff[lo];
    const int nj = (r + SHRINK_J - 1) / SHRINK_J;
    const int j0 = (local % nj) * SHRINK_J;
    const int t0 = (local / nj) * SHRINK_TOK;
    const int ntok = min(SHRINK_TOK, c - t0);
    const int nrow = min(SHRINK_J, r - j0);
    int rows[SHRINK_TOK];
#pragma unroll
    for (int t = 0; t < SHRINK_TOK; ++t) rows[t] = (t < ntok) ? plan[L.perm + s0 + t0 + t] : 0;
    int4 *rec = reinterpret_cast<int4 *>(plan + L.items + (size_t)it * ITEM_WORDS);
    rec[0] = make_int4(a, j0 | (nrow << 8) | (ntok << 16), s0 + t0, plan[L.slice_off + a]);
    rec[1] = make_int4(rows[0], rows[1], rows[2], rows[3]);
  }
  block_sync();
  if (tid == 0 && flags) raise_status(status, flags);
}

cudaError_t launch_plan(const int32_t *adapter_idx, int M, const int32_t *rank_of, int n_ad, int r_max,
                        int32_t *plan, uint32_t *status, cudaStream_t s) {
  const size_t smem = 2 * (size_t)(n_ad + 1) * sizeof(int);  // <= 32.8 KB for n_ad <= 4096
  cudaError_t e = launch_pdl(plan_kernel, dim3(1), dim3(PLAN_THREADS), smem, s, adapter_idx, M, rank_of, n_ad, r_max,
                             plan, status);
  return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace mlora
