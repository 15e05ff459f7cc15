// Step a2 on the tensor cores, for the verify pass: the low-rank operand of
// the windowed expand, bf16(scale * A_a x) on each adapter's token window.
//
// The pages call each adapter's low-rank product "a small, GPU-inefficient
// operation" (InvisibleLoRA, abstract) because requests are spread over many
// adapters.  Here the token rows are already in adapter-sorted order (x_sorted),
// so the expand blocks (adapter a, 16-rank block; see common.cuh) of
// consecutive adapters cover consecutive token windows.  A unit takes 8
// consecutive blocks: their 128 rank rows of A (one 16-row TMA box each) are
// the MMA's M side, the union of their windows (up to 256 sorted token rows
// per pass) its N side, so each A row is read once for all the unit's
// tokens:
//
//   D[16 i + j, c] = sum_k A_{a_i}[j0_i + j, k] x_sorted[r0 + c, k]
//
// and the window entry of block i at token position p = r0 + c is
// bf16(scale * D[16 i + j, c]) if p is one of a_i's rows and j < rank
// columns of the block, else 0 (the other adapters' rows that the 16-row
// rounding of the window takes in).  Entries of D for other (block, token)
// pairs are computed and dropped: at most 8x the useful MMA work, a few
// GFLOP per call, while the bytes (A once, x once per unit) are what bound it.
//
// Split-K over a thread-block cluster of C CTAs (C = 1..16, the one that
// minimises waves x k-blocks per CTA for the clusters that fit at once): each
// CTA runs its contiguous share of the K loop into tensor memory, stages D in
// its idle ring, and after a cluster barrier CTA r adds the C copies of
// half-blocks (8 rank rows) [16 r / C, 16 (r + 1) / C) in rank order
// (deterministic) and writes their window rows.
//
// Per stage the A rows of blocks adjacent in A (consecutive adapters of rank
// r_max, the blocks of one adapter) arrive as one box of up to 128 rows, the
// token rows as one box of up to 256.  Measured on GB300, a CTA's copies of A
// stream at 20-35 GB/s whatever the ring depth (2 or 4 stages), L2 residency
// or cache hints, so the tiles pay off only where the warp items re-read A
// often and enough units fill the SMs: see shrink_on_tensor_cores.
//
// Warp roles as in the GEMMs: warp 0 issues the TMA loads, warp 1 owns
// tensor memory and issues tcgen05.mma, warps 2..5 stage; all six reduce.
#include "common.cuh"
#include "launch.h"

namespace mlora {

constexpr int SQ_THREADS = 192;
constexpr int SQ_BLOCKS = 8;                  // expand blocks per unit: 8 x 16 = 128 rank rows (MMA M)
constexpr int SQ_BK = 64;                     // K per stage (128 bytes of bf16)
constexpr int SQ_NMAX = 256;                  // token columns per pass (MMA N)
constexpr int SQ_XBOX = 64;                   // token rows per TMA box
constexpr int SQ_ABYTES = 128 * SQ_BK * 2;    // 16 KB: the unit's A rows of one stage
constexpr int SQ_STAGE = SQ_ABYTES + SQ_NMAX * SQ_BK * 2;  // + 32 KB of token rows
constexpr int SQ_STAGES = 4;
constexpr size_t SQ_SMEM = 1024 + (size_t)SQ_STAGES * SQ_STAGE + 512;
static_assert((size_t)SQ_STAGES * SQ_STAGE >= (size_t)128 * SQ_NMAX * 4, "D is staged in the ring");

__device__ __forceinline__ uint32_t ld_dsmem_u32(uint32_t caddr) {
  uint32_t v;
  asm volatile("ld.shared::cluster.u32 %0, [%1];" : "=r"(v) : "r"(caddr) : "memory");
  return v;
}

// Tensor maps of A (boxes of 16, 32, 64 and 128 rows: a run of blocks whose
// rank rows are adjacent in A, as for consecutive adapters of rank r_max or
// the blocks of one adapter, takes one box) and of the sorted token rows
// (boxes of 64, 128 and 256 rows).  Fewer, larger boxes per stage.
struct SqMaps {
  CUtensorMap a[4];
  CUtensorMap x[3];
};

struct SqArgs {
  int M, K, n_ad, r_max, n_slices, kblocks, groups, C;
  float scale;
  size_t tw_slice;   // bf16 elements of one slice's window buffer
  long long tw_rows; // window rows of one slice
  const int32_t *plan;
  uint16_t *tw;
  uint32_t *status;
};

__global__ void __launch_bounds__(SQ_THREADS, 1)
    shrink_mma_kernel(const __grid_constant__ SqMaps maps, const SqArgs args) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t *ring = align_smem_1024(smem_raw);
  uint8_t *tail = ring + (size_t)SQ_STAGES * SQ_STAGE;  // 512 bytes: barriers and the unit's records
  uint64_t *full = reinterpret_cast<uint64_t *>(tail);
  uint64_t *empty = full + SQ_STAGES;
  uint64_t *acc_full = empty + SQ_STAGES;
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(tail + 72);
  int *abort_flag = reinterpret_cast<int *>(tail + 76);
  int *zero_word = reinterpret_cast<int *>(tail + 80);
  int *acc_ready = reinterpret_cast<int *>(tail + 84);  // the MMA warp's verdict on the accumulator, per pass
  uint64_t *drain = reinterpret_cast<uint64_t *>(tail + 88);
  int4 *rec = reinterpret_cast<int4 *>(tail + 96);  // per block: {a, j0, rank columns (0: skip), win}, {w0, W, s0, s1}
  int *span = reinterpret_cast<int *>(tail + 96 + 2 * SQ_BLOCKS * 16);  // first row, end row of the windows

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int C = args.C;
  const uint32_t rank = C > 1 ? cluster_ctarank() : 0u;
  const int unit = blockIdx.x / C;
  const int slice = unit / args.groups, grp = unit - slice * args.groups;
  const PlanLayout L = plan_layout(args.M, args.n_ad);

  // The plan comes from a kernel earlier in the stream, x_sorted from the
  // gather just before; let the next kernel launch only after that (it reads
  // x_sorted too and relies on it being complete).
  grid_dependency_wait();
  grid_launch_dependents();
  const int ns = min(args.plan[L.hdr + 4], max_expand_slices(args.M, args.n_ad));  // a corrupt count reads no further
  const int b0 = grp * SQ_BLOCKS;
  if (b0 >= ns) return;  // the whole cluster leaves: every CTA reads the same ns
  const int nb = min(SQ_BLOCKS, ns - b0);

  if (threadIdx.x == 0) {
    for (int q = 0; q < SQ_STAGES; ++q) {
      mbar_init(&full[q], 1);
      mbar_init(&empty[q], 1);
    }
    mbar_init(acc_full, 1);
    mbar_init(drain, 1);
    *abort_flag = 0;
    *zero_word = 0;
    fence_mbar_init();
  }
  if (threadIdx.x < 32) {
    // The unit's block records, checked (a record out of range: the plan was
    // overwritten or made for other sizes; the block is dropped and
    // MLORA_DEV_BAD_PLAN raised); lane i takes block i.
    int lo = 1 << 30, hi = 0;
    if (lane < nb) {
      const int32_t *e = args.plan + L.slices + (size_t)(b0 + lane) * EXP_WORDS;
      const int a = e[0], j0 = e[1], rc = e[2], win = e[3], w0 = e[4], W = e[5];
      bool valid = (unsigned)a < (unsigned)args.n_ad && (j0 & 15) == 0 && j0 >= 0 && j0 < args.r_max && rc >= 1 &&
                   rc <= 16 && win >= 0 && w0 >= 0 && (w0 & 15) == 0 && W >= 0 && (W & 15) == 0 &&
                   (long long)win + W <= args.tw_rows && w0 + W <= ((args.M + 15) & ~15);
      const int s0 = valid ? args.plan[L.seg_offsets + a] : 0, s1 = valid ? args.plan[L.seg_offsets + a + 1] : 0;
      valid = valid && s0 >= 0 && s0 <= s1 && s1 <= args.M;
      if (!valid) raise_status(args.status, MLORA_DEV_BAD_PLAN);
      rec[2 * lane] = make_int4(a, j0, valid ? rc : 0, win);
      rec[2 * lane + 1] = make_int4(w0, W, s0, s1);  // the window, then the adapter's sorted rows [s0, s1)
      if (valid && W > 0) {
        lo = w0;
        hi = w0 + W;
      }
    } else if (lane < SQ_BLOCKS) {
      rec[2 * lane] = make_int4(0, 0, 0, 0);
      rec[2 * lane + 1] = make_int4(0, 0, 0, 0);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      lo = min(lo, __shfl_xor_sync(0xffffffffu, lo, o));
      hi = max(hi, __shfl_xor_sync(0xffffffffu, hi, o));
    }
    if (lane == 0) {
      span[0] = lo;
      span[1] = hi;
    }
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, SQ_NMAX);
    tmem_relinquish();
  }
  tc_fence_before_sync();
  block_sync();
  tc_fence_after_sync();
  const uint32_t tmem_base = *tmem_slot;
  volatile int *ab = abort_flag;
  volatile int *never = zero_word;
  const int r_lo = span[0], r_hi = span[1];
  const int kb_lo = (int)((long long)rank * args.kblocks / C), kb_hi = (int)((long long)(rank + 1) * args.kblocks / C);
  int stage = 0, issued = 0;
  uint32_t phase = 0, acc_phase = 0;
  bool ok = true;
  const uint32_t ring0 = smem_addr(ring);
  const float scale = args.scale;
  uint16_t *tw = args.tw + (size_t)slice * args.tw_slice;
  const int a_row0 = slice * args.n_ad;  // first A row of this slice, in adapters
  bool mma_any = false;

  // Passes of up to SQ_NMAX token columns over the windows' union; every CTA
  // of the cluster computes the same count, so all meet at the same cluster
  // barriers (an aborted CTA still takes part in them).
  const int n_pass = r_hi > r_lo ? (r_hi - r_lo + SQ_NMAX - 1) / SQ_NMAX : 0;
  for (int pass = 0; pass < n_pass; ++pass) {
    const int pr0 = r_lo + pass * SQ_NMAX;
    const int nt = min(SQ_NMAX, r_hi - pr0);
    const int n16 = (nt + 15) & ~15;
    const int nxb = (n16 + SQ_XBOX - 1) / SQ_XBOX;
    // Blocks whose window meets this pass's columns: only their A rows are
    // loaded (the rows of D of the others are left unused).
    uint32_t need = 0;
#pragma unroll
    for (int i = 0; i < SQ_BLOCKS; ++i) {
      const int4 r0 = rec[2 * i], r1 = rec[2 * i + 1];
      if (r0.z > 0 && r1.x < pr0 + nt && r1.x + r1.y > pr0) need |= 1u << i;
    }
    const uint32_t tx = (uint32_t)__popc(need) * (16 * SQ_BK * 2) + (uint32_t)nxb * (SQ_XBOX * SQ_BK * 2);

    if (warp == 0) {
      // -------------------------------------------------------- producer
      if (lane == 0 && ok && !*ab) {
        const uint64_t pol_a = policy_evict_first();  // each A row is read by one cluster only
        const uint64_t pol_x = policy_evict_last();   // the GEMM reads the token rows next
        for (int kb = kb_lo; kb < kb_hi; ++kb) {
          if (!mbar_wait_bounded(&empty[stage], phase ^ 1u, ab)) {
            *ab = 1;
            raise_status(args.status, MLORA_DEV_TIMEOUT);
            ok = false;
            break;
          }
          uint8_t *st = ring + (size_t)stage * SQ_STAGE;
          mbar_arrive_expect_tx(&full[stage], tx);
          // A: runs of needed blocks with adjacent rows, split into boxes of
          // 8, 4, 2 or 1 blocks; the box of blocks [i, i + n) lands at 2 KB x i.
#pragma unroll 1
          for (int i = 0; i < SQ_BLOCKS;) {
            if (!((need >> i) & 1u)) {
              ++i;
              continue;
            }
            const int row = (a_row0 + rec[2 * i].x) * args.r_max + rec[2 * i].y;
            int run = 1;
            while (i + run < SQ_BLOCKS && ((need >> (i + run)) & 1u) &&
                   (a_row0 + rec[2 * (i + run)].x) * args.r_max + rec[2 * (i + run)].y == row + 16 * run)
              ++run;
            const int lg = run >= 8 ? 3 : run >= 4 ? 2 : run >= 2 ? 1 : 0;
            tma_load_2d(st + i * (16 * SQ_BK * 2), &maps.a[lg], &full[stage], kb * SQ_BK, row, pol_a);
            i += 1 << lg;
          }
          // Token rows: 64-row units as one box of 256, 128 + 64, 128 or 64 rows.
          uint8_t *xs = st + SQ_ABYTES;
          if (nxb == 4) {
            tma_load_2d(xs, &maps.x[2], &full[stage], kb * SQ_BK, pr0, pol_x);
          } else {
            if (nxb >= 2) tma_load_2d(xs, &maps.x[1], &full[stage], kb * SQ_BK, pr0, pol_x);
            if (nxb != 2)
              tma_load_2d(xs + (nxb - 1) * (SQ_XBOX * SQ_BK * 2), &maps.x[0], &full[stage], kb * SQ_BK,
                          pr0 + (nxb - 1) * SQ_XBOX, pol_x);
          }
          ++issued;
          if (++stage == SQ_STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
      stage = __shfl_sync(0xffffffffu, stage, 0);
      phase = __shfl_sync(0xffffffffu, phase, 0);
      issued = __shfl_sync(0xffffffffu, issued, 0);
    } else if (warp == 1) {
      // -------------------------------------------------------- MMA issuer
      if (lane == 0 && ok && !*ab) {
        const uint32_t idesc = idesc_bf16_f32(128, n16);
        for (int kb = kb_lo; kb < kb_hi; ++kb) {
          if (!mbar_wait_bounded(&full[stage], phase, ab)) {
            *ab = 1;
            raise_status(args.status, MLORA_DEV_TIMEOUT);
            ok = false;
            break;
          }
          tc_fence_after_sync();
          const uint32_t a_addr = ring0 + (uint32_t)stage * SQ_STAGE;
          const uint64_t ad = smem_desc_kmajor_sw128(a_addr);
          const uint64_t bd = smem_desc_kmajor_sw128(a_addr + SQ_ABYTES);
#pragma unroll
          for (int kk = 0; kk < SQ_BK / 16; ++kk)
            mma_bf16_ss(tmem_base, ad + 2 * kk, bd + 2 * kk, idesc, (kb > kb_lo || kk > 0) ? 1u : 0u);
          mma_any = true;
          mma_commit(&empty[stage]);
          if (++stage == SQ_STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (ok) mma_commit(acc_full);
      }
      ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
      mma_any = __shfl_sync(0xffffffffu, mma_any ? 1 : 0, 0) != 0;
      stage = __shfl_sync(0xffffffffu, stage, 0);
      phase = __shfl_sync(0xffffffffu, phase, 0);
      // The accumulator handoff: this warp waits for the last MMA, then
      // releases the staging warps through named barrier 1, so that they
      // sleep in hardware instead of polling an mbarrier during the K loop.
      // It arrives in every pass, aborted or not.
      if (lane == 0) {
        const bool ready = ok && !*ab && mbar_wait_bounded(acc_full, acc_phase, ab);
        if (ok && !ready && !*ab) {
          *ab = 1;
          raise_status(args.status, MLORA_DEV_TIMEOUT);
        }
        *reinterpret_cast<volatile int *>(acc_ready) = ready ? 1 : 0;
      }
      __syncwarp();
      tc_fence_before_sync();
      named_bar_arrive(1, 160);
    } else {
      // -------------------------------------------------------- stage D
      // Warp w reads tensor-memory lanes 32 (w % 4) .. + 31 (rows of D) and
      // writes them transposed, Dt[c][row] (fp32, 128 rows per column), into
      // the ring, which no copy or MMA of this pass touches any more.
      named_bar_sync(1, 160);
      tc_fence_after_sync();
      const bool have = *reinterpret_cast<volatile int *>(acc_ready) != 0;
      if (have) {
        const int quad = warp & 3, row = quad * 32 + lane;
        const uint32_t taddr = tmem_base + ((uint32_t)(quad * 32) << 16);
        float *Dt = reinterpret_cast<float *>(ring);
        for (int c0 = 0; c0 < n16; c0 += 16) {
          uint32_t r[16];
          tmem_ld_x16(taddr + (uint32_t)c0, r);
          tmem_ld_wait();
#pragma unroll
          for (int e = 0; e < 16; ++e) Dt[(c0 + e) * 128 + row] = __uint_as_float(r[e]);
        }
      }
      tc_fence_before_sync();
    }
    acc_phase ^= 1u;
    __syncwarp();
    if (C > 1) cluster_sync_all(); else block_sync();  // every CTA's D is staged

    // ---------------------------------------------------------- reduction
    // CTA `rank` owns half-blocks (8 rank rows of one block) [16 rank / C,
    // 16 (rank + 1) / C): it adds the C staged copies of their rows in rank
    // order, scales, rounds to bf16 and writes the window rows of this pass
    // (16 bytes: one swizzled half of a window row).  Nothing is written if
    // any CTA of the cluster gave up.
    {
      const int hb_lo = (int)(rank * 16u / (uint32_t)C), hb_hi = (int)((rank + 1u) * 16u / (uint32_t)C);
      uint32_t peer[16];
      bool any_abort = C == 1 && *ab;
#pragma unroll
      for (int q = 0; q < 16; ++q) {
        peer[q] = 0u;
        if (q < C && C > 1) {
          peer[q] = map_to_rank(ring0, (uint32_t)q);
          any_abort |= ld_dsmem_u32(map_to_rank(smem_addr(abort_flag), (uint32_t)q)) != 0u;
        }
      }
      const int items = any_abort ? 0 : (hb_hi - hb_lo) * nt;
      for (int it = threadIdx.x; it < items; it += SQ_THREADS) {
        const int q_hb = it / nt;
        const int c = it - q_hb * nt, hb = hb_lo + q_hb;
        const int bi = hb >> 1, h = hb & 1;
        const int4 r0 = rec[2 * bi], r1 = rec[2 * bi + 1];
        const int p = pr0 + c;
        if (r0.z == 0 || p < r1.x || p >= r1.x + r1.y) continue;
        const bool member = p >= r1.z && p < r1.w;
        const int live = member ? max(0, min(8, r0.z - 8 * h)) : 0;  // entries of this half with a value
        float v[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) v[e] = 0.f;
        if (live > 0) {
          const uint32_t off = (uint32_t)((c * 128 + 16 * bi + 8 * h) * 4);
          if (C == 1) {
            const float4 lo = *reinterpret_cast<const float4 *>(ring + off);
            const float4 hi = *reinterpret_cast<const float4 *>(ring + off + 16);
            v[0] = lo.x, v[1] = lo.y, v[2] = lo.z, v[3] = lo.w, v[4] = hi.x, v[5] = hi.y, v[6] = hi.z, v[7] = hi.w;
          } else {
#pragma unroll
            for (int q = 0; q < 16; ++q) {
              if (q < C) {
                const float4 lo = ld_dsmem_f32x4(peer[q] + off), hi = ld_dsmem_f32x4(peer[q] + off + 16);
                v[0] += lo.x, v[1] += lo.y, v[2] += lo.z, v[3] += lo.w;
                v[4] += hi.x, v[5] += hi.y, v[6] += hi.z, v[7] += hi.w;
              }
            }
          }
        }
        uint32_t o[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const uint32_t lo = 2 * e < live ? float_to_bf16_bits(scale * v[2 * e]) : 0u;
          const uint32_t hi = 2 * e + 1 < live ? float_to_bf16_bits(scale * v[2 * e + 1]) : 0u;
          o[e] = lo | (hi << 16);
        }
        const int i = p - r1.x;
        uint16_t *dst = tw + (size_t)(r0.w + i) * 16 + 8 * (h ^ ((i >> 2) & 1));
        *reinterpret_cast<uint4 *>(dst) = make_uint4(o[0], o[1], o[2], o[3]);
      }
    }
    // Generic-proxy accesses to the ring are ordered before the next pass's
    // copies into it; the peers have read this CTA's staged D after the barrier.
    fence_proxy_async_smem();
    __syncwarp();
    if (C > 1) cluster_sync_all(); else block_sync();
  }

  // Teardown: this CTA's own copies land and its MMAs finish before shared
  // and tensor memory go away (only an abort leaves copies in flight).
  if (warp == 0 && lane == 0 && *ab) {
    const int n = issued < SQ_STAGES ? issued : SQ_STAGES;
    for (int i = issued - n; i < issued; ++i)
      mbar_wait_bounded(&full[i % SQ_STAGES], (uint32_t)((i / SQ_STAGES) & 1), never);
  }
  if (warp == 1 && lane == 0 && mma_any) {
    mma_commit(drain);
    mbar_wait_bounded(drain, 0u, never);
  }
  tc_fence_before_sync();
  block_sync();
  tc_fence_after_sync();
  if (warp == 1) tmem_dealloc(tmem_base, SQ_NMAX);
}

// ---------------------------------------------------------------------------
// Host side
// ---------------------------------------------------------------------------
constexpr int SQ_MAX_CLUSTER = 16;

typedef CUresult (*SqEncodeFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                               const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                               CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static SqEncodeFn sq_encode_fn() {
  static SqEncodeFn fn = nullptr;
  if (!fn) {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<SqEncodeFn>(p);
  }
  return fn;
}

// Row-major bf16 [rows, cols] in boxes of box_rows x 64 columns, 128-byte
// swizzle; out-of-range elements read as zero.
static bool sq_map(CUtensorMap *map, const void *base, long long rows, int cols, int box_rows) {
  SqEncodeFn fn = sq_encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)cols * 2};
  cuuint32_t box[2] = {(cuuint32_t)SQ_BK, (cuuint32_t)box_rows};
  cuuint32_t estr[2] = {1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

static bool sq_attributes() {
  static int done[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return false;
  if (dev < 64 && done[dev]) return true;
  if (cudaFuncSetAttribute(shrink_mma_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)SQ_SMEM) !=
      cudaSuccess)
    return false;
  if (cudaFuncSetAttribute(shrink_mma_kernel, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) != cudaSuccess)
    return false;
  if (dev < 64) done[dev] = 1;
  return true;
}

// Clusters of C CTAs (one per SM) that can be resident at once.
static int sq_max_clusters(int C) {
  struct Entry {
    int dev, C, n;
  };
  static Entry cache[64];
  static int ncache = 0;
  int dev = 0;
  cudaGetDevice(&dev);
  for (int i = 0; i < ncache; ++i)
    if (cache[i].dev == dev && cache[i].C == C) return cache[i].n;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(C * 16, 1, 1);
  cfg.blockDim = dim3(SQ_THREADS, 1, 1);
  cfg.dynamicSmemBytes = SQ_SMEM;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = C;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, shrink_mma_kernel, &cfg) != cudaSuccess) {
    cudaGetLastError();
    n = 0;
  }
  if (ncache < 64) cache[ncache++] = {dev, C, n};
  return n;
}

// Units (slice, 8 consecutive expand blocks) for M rows: at most
// ceil(r_max / 16) blocks for each of min(M, n_ad) active adapters.
static int sq_groups(int M, int n_ad, int r_max) {
  const long long blocks = (long long)((r_max + 15) / 16) * (M < n_ad ? M : n_ad);
  return (int)((blocks + SQ_BLOCKS - 1) / SQ_BLOCKS);
}

// Cluster size: the C (1..16, at most the k-blocks) that minimises waves x
// (k-blocks per CTA + a fixed cost per pass, more with a cluster reduction).
static int sq_cluster(int units, int kblocks, int num_sms) {
  int bestC = 1;
  double best = 1e30;
  for (int C = 1; C <= SQ_MAX_CLUSTER && C <= kblocks; ++C) {
    const int clusters = C == 1 ? num_sms : sq_max_clusters(C);
    if (clusters <= 0) continue;
    const long long waves = (units + clusters - 1) / clusters;
    const double kper = (double)((kblocks + C - 1) / C);
    const double cost = (double)waves * (kper + 4.0 + (C > 1 ? 2.0 + 0.25 * C : 0.0));
    if (cost < best - 1e-9) {
      best = cost;
      bestC = C;
    }
  }
  return bestC;
}

cudaError_t launch_shrink_mma(const uint16_t *xs, int M, int K, const uint16_t *A, int n_ad, int r_max,
                              const int32_t *plan, uint16_t *tw, float scale, int n_slices, int num_sms,
                              uint32_t *status, cudaStream_t s) {
  if (M <= 0 || n_ad <= 0 || n_slices <= 0) return cudaSuccess;
  if (!sq_attributes()) return cudaErrorInvalidValue;
  SqMaps maps;
  for (int i = 0; i < 4; ++i)
    if (!sq_map(&maps.a[i], A, (long long)n_slices * n_ad * r_max, K, 16 << i)) return cudaErrorInvalidValue;
  for (int i = 0; i < 3; ++i)
    if (!sq_map(&maps.x[i], xs, M, K, SQ_XBOX << i)) return cudaErrorInvalidValue;
  SqArgs a;
  a.M = M;
  a.K = K;
  a.n_ad = n_ad;
  a.r_max = r_max;
  a.n_slices = n_slices;
  a.kblocks = (K + SQ_BK - 1) / SQ_BK;
  a.groups = sq_groups(M, n_ad, r_max);
  a.C = sq_cluster(n_slices * a.groups, a.kblocks, num_sms);
  a.scale = scale;
  a.tw_rows = (long long)max_window_rows(M, n_ad);
  a.tw_slice = max_window_rows(M, n_ad) * 16;
  a.plan = plan;
  a.tw = tw;
  a.status = status;

  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(n_slices * a.groups * a.C), 1, 1);
  cfg.blockDim = dim3(SQ_THREADS, 1, 1);
  cfg.dynamicSmemBytes = SQ_SMEM;
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  int na = 0;
  attr[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[na].val.programmaticStreamSerializationAllowed = 1;
  ++na;
  if (a.C > 1) {
    attr[na].id = cudaLaunchAttributeClusterDimension;
    attr[na].val.clusterDim.x = a.C;
    attr[na].val.clusterDim.y = 1;
    attr[na].val.clusterDim.z = 1;
    ++na;
  }
  cfg.attrs = attr;
  cfg.numAttrs = na;
  cudaError_t e = cudaLaunchKernelEx(&cfg, shrink_mma_kernel, maps, a);
  note_launch();
  return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace mlora
