// Steps a3 + a4 as a persistent stream-K kernel: the base GEMM acc = x W^T on
// the tcgen05 tensor cores with the low-rank expand added by tensor-core MMAs
// (verify mode), for batches of up to 1024 token rows:
//
//   draft  (LoRA off): y[m, n] = bf16(acc[m, n])
//   verify (LoRA on):  y[perm[c], n] = bf16(acc[c, n] + sum_blocks B_a[n, block] . Twin[c, :])
//
// In verify mode the token rows come in adapter-sorted order (column c is row
// perm[c]) and each expand block (adapter a, 16-rank block) adds its MMA over
// a's token window only (expand.cuh), where the window holds scale * T on a's
// rows and 0 elsewhere ("output = W·x + scale · B(A·x)", "Multi-LoRA Serving
// in Practice", section "Core Principle: Shared Base Model, Per-Request
// Adapter Selection").
//
// Work split.  The token rows form up to four groups of at most 256 (Mb
// rows each); every group gets the same number of CTAs (at most one per SM
// in all), and a unit is a tile of 128 W rows with the CTAs' token group.
// Within a group the (tile, 64-wide k-block) pairs are cut into one
// contiguous, equal share per CTA, so every SM streams the same number of
// bytes whatever the tile count (no partial last wave), and CTA j of every
// group streams the same W k-blocks at about the same time: a W tile comes
// from DRAM once and serves the other groups from L2.  A CTA's share is a sequence of segments: the tail of a unit begun
// by the CTA before it, whole units, and the head of a unit that the CTAs
// after it finish.  The CTA that holds a unit's first k-block owns the unit
// and adds the expand MMAs.  A split unit is finished by its participants
// together: each publishes its segment's fp32 partial sums and counts itself
// in on the unit's arrival word; those whose shares end inside the unit (the
// owner, and the CTAs whose whole share lies in it) then each add up every
// partial for an equal slice of the unit's token columns and store y.
// A CTA waits at most once, in its last segment, after publishing all its
// earlier segments, and all CTAs are resident at once, so the waits always
// end; every wait is bounded nevertheless.  Partials are added in CTA order:
// results are deterministic.
//
// Residency: the waits above end only if every CTA of the grid is resident at
// once.  The host launches one CTA per SM only when the occupancy query says
// a CTA fits on every SM; each wait is bounded in any case, and a wait that
// gives up raises MLORA_DEV_TIMEOUT.
//
// Warp roles: warp 0 issues the TMA loads of W and x tiles (128-byte swizzle)
// and of the expand operands into a ring of stages that runs across segment
// boundaries; warp 1 owns tensor memory, issues tcgen05.mma from one thread
// into two accumulators used alternately, and zeroes B columns past an
// adapter's rank in shared memory before an expand MMA reads them; warps 2..5
// drain one accumulator while the MMAs fill the other.
#include "common.cuh"
#include "expand.cuh"
#include "launch.h"

namespace mlora {

constexpr int SK_THREADS = 192;
constexpr int SK_BN = 128;                       // W rows per tile (MMA M)
constexpr int SK_BK = 64;                        // K per stage: 128 bytes of bf16 (128 E4M3 values)
constexpr int SK_WTILE = SK_BN * SK_BK * 2;      // 16 KB
constexpr int SK_CHUNK = 32;                     // accumulator columns per tensor-memory load
constexpr size_t SK_SMEM_LIMIT = 220 * 1024;     // leaves room for a co-resident shrink CTA
constexpr int SK_MAX_STAGES = 8;
constexpr int SK_CACHE_BLOCKS = 256;             // expand block records kept in shared memory (8 KB)
constexpr int SK_YROW = 40;                      // bf16 per token row of an epilogue warp's y staging (32 + pad)
constexpr int SK_YSTAGE = 4 * 32 * SK_YROW * 2;  // staging of the four epilogue warps (y, partial sums): 10 KB
static_assert(4 * 16 * 36 * 4 <= SK_YSTAGE, "16 columns of a warp's fp32 partial sums fit its staging block");
// Alignment slack, barriers, the expand stage records, the cached block
// records, the y staging.
constexpr size_t SK_SMEM_FIXED =
    1024 + 256 + expand_smem_bytes(SK_MAX_STAGES) + SK_CACHE_BLOCKS * EXP_WORDS * 4 + SK_YSTAGE;
constexpr int SK_MIN_SHARE = 8;                  // k-blocks per CTA at least
constexpr int SK_MAX_PARTIALS = 8;               // contributors per tile besides its owner, at most
constexpr int SK_GROUP_ROWS = 256;               // token rows of a group: two accumulators fit in tensor memory
constexpr int SK_MAX_GROUPS = 4;                 // token groups of a call (M <= 1024)
struct SkArgs {
  int M, N, K, Mb, kblocks, total, P, stages, cols;
  int n_tg;  // token groups; CTAs [g Pg, (g + 1) Pg) serve group g (token rows [g Mb, +Mb))
  int Pg;    // CTAs per token group; total = (tile, k-block) pairs of one group
  int mode, prefetch_w, after_shrink;
  int sorted;  // verify mode: x in adapter-sorted order, token windows present
  int n_slices, slice_end[MLORA_MAX_SLICES];
  size_t tw_slice;  // bf16 elements of one slice's window buffer
  int n_ad;
  int vec_y;  // N % 8 == 0 and y 16-byte aligned: 16-byte stores of 8 outputs
  uint32_t test_flag_wait_ns;  // nonzero: owners poll never-set flags for this long (a test of the timeout path)
  uint16_t *y;
  const uint16_t *tw;  // token windows of the expand blocks, rows in the 32-byte-swizzled order
  const int32_t *plan;
  uint32_t *status;
  float *partials;  // [P][2][Mb][128]: a CTA's partial sums of its first and of a later split segment, token-major
  uint32_t *flags;  // [P] arrivals and [P] finished reducers of the split tile owned by CTA i (zero between calls)
  const float *w_scale;  // E4M3 operands: per W row and per token row scales of the codes
  const float *x_scale;
};

// Shares within a token group's CTAs: local CTA i holds linear k-blocks
// [sk_begin(i), sk_begin(i + 1)) of the group's (tile, k-block) pairs.
__device__ __forceinline__ int sk_begin(const SkArgs &a, int i) { return (int)((long long)i * a.total / a.Pg); }

// The local CTA whose share holds linear k-block g.
__device__ __forceinline__ int sk_cta_of(const SkArgs &a, int g) {
  int i = (int)((long long)g * a.Pg / a.total);
  while (i + 1 < a.Pg && sk_begin(a, i + 1) <= g) ++i;
  while (i > 0 && sk_begin(a, i) > g) --i;
  return i;
}

__device__ __forceinline__ int sk_slice_of(const SkArgs &a, int n0) {
  int s = 0;
#pragma unroll
  for (int i = 0; i + 1 < MLORA_MAX_SLICES; ++i)
    if (i + 1 < a.n_slices && n0 >= a.slice_end[i]) s = i + 1;
  return s;
}

// The expand operands' tensor maps: B_stack [n_ad][N][r_max] as a 2-D view
// [n_ad N, r_max] (one 16-rank block of 128 rows per box), and as 3-D maps
// {r_max, N, n_ad} whose boxes take the same block of 1, 2, 4 or 8
// consecutive adapters at once.
struct SkBMaps {
  CUtensorMap b2;
  CUtensorMap b3[4];
};

// A CTA's expand plan, built once from the cached block records: the blocks
// whose windows meet the CTA's token group, in plan order, E[k] = {adapter,
// j0 | rank columns << 8, first window row, first accumulator column | rows
// << 16}, and their packing into ring stages, D[s] = {first block, blocks,
// window bytes, last}.  Only the W tile (the B rows) changes from one owned
// unit to the next, so each unit replays the plan.  Built in place over the
// cached records (entry k, 16 bytes, never overtakes record k, 32 bytes).
// Returns the stage count (at least 1, an empty stage when no block meets
// the group: the MMA warp runs an owned unit's stages until `last`).
__device__ __forceinline__ int sk_expand_plan(int32_t *cache, int ns, int m0, int mcols, int n_ad, long long tw_rows,
                                              int stage_bytes, int lane, uint32_t *status) {
  int4 *E = reinterpret_cast<int4 *>(cache);
  int4 *D = reinterpret_cast<int4 *>(cache) + SK_CACHE_BLOCKS;
  int ne = 0;
  for (int c0 = 0; c0 < ns; c0 += 32) {
    int4 ent = make_int4(0, 0, 0, 0);
    bool keep = false;
    if (c0 + lane < ns) {
      const int4 e0 = reinterpret_cast<const int4 *>(cache)[(size_t)(c0 + lane) * 2];
      const int4 e1 = reinterpret_cast<const int4 *>(cache)[(size_t)(c0 + lane) * 2 + 1];
      const int w0 = e1.x, W = e1.y;
      const bool valid = (unsigned)e0.x < (unsigned)n_ad && (e0.y & 15) == 0 && (unsigned)e0.y < 64u &&
                         e0.z >= 1 && e0.z <= 16 && e0.w >= 0 && w0 >= 0 && (w0 & 15) == 0 && W >= 0 &&
                         (W & 15) == 0 && (long long)e0.w + W <= tw_rows;
      if (!valid) raise_status(status, MLORA_DEV_BAD_PLAN);
      const int cs = max(w0, m0), ce = min(w0 + W, m0 + mcols);
      keep = valid && ce > cs;
      if (keep) ent = make_int4(e0.x, e0.y | (e0.z << 8), e0.w + (cs - w0), (cs - m0) | ((ce - cs) << 16));
    }
    const uint32_t kb = __ballot_sync(0xffffffffu, keep);
    __syncwarp();  // every lane has read its record before any entry is written
    if (keep) E[ne + __popc(kb & ((1u << lane) - 1u))] = ent;
    ne += __popc(kb);
    __syncwarp();
  }
  int nst = 0;
  if (lane == 0) {
    for (int k = 0; k < ne;) {
      int cnt = 0, tbytes = 0;
      while (k + cnt < ne && cnt < EXP_MAX_PER_STAGE) {
        const int rows = E[k + cnt].w >> 16;  // <= 286: a block and its window always fit a stage
        if ((cnt + 1) * EXP_B_TILE + tbytes + rows * 32 > stage_bytes) break;
        tbytes += rows * 32;
        ++cnt;
      }
      D[nst++] = make_int4(k, cnt, tbytes, 0);
      k += cnt;
    }
    if (nst == 0) D[nst++] = make_int4(0, 0, 0, 0);
    D[nst - 1].w = 1;
  }
  nst = __shfl_sync(0xffffffffu, nst, 0);
  __syncwarp();
  return nst;
}

// Stages [s_begin, s_end) of one owned unit's expand from the plan (producer
// warp, all lanes):
// per stage, lane c describes block c in the stage record, lane 0 arms the
// barrier, then each lane that starts a run of consecutive adapters (same
// 16-rank block) loads their B tiles with 3-D boxes, and each lane that
// starts a run of back-to-back windows copies them with one bulk copy.
__device__ __forceinline__ bool sk_expand_issue(const int32_t *cache, int s_begin, int s_end, const SkBMaps &bm, int n0,
                                                const uint16_t *tw, uint8_t *ring, int stage_bytes, int S,
                                                uint64_t *full, uint64_t *empty, ExpandStage *meta, int &stage,
                                                uint32_t &phase, int &issued, volatile int *abort, uint64_t pol,
                                                int lane) {
  const int4 *E = reinterpret_cast<const int4 *>(cache);
  const int4 *D = reinterpret_cast<const int4 *>(cache) + SK_CACHE_BLOCKS;
  for (int s = s_begin; s < s_end; ++s) {
    const int4 dsc = D[s];
    // Every lane tests the barrier itself: a lane that waits behind another
    // lane's suspended wait (and a shuffle) measured about 0.5 us a stage.
    if (!__all_sync(0xffffffffu, mbar_wait_bounded(&empty[stage], phase ^ 1u, abort))) return false;
    uint8_t *st = ring + (size_t)stage * stage_bytes;
    ExpandStage &m = meta[stage];
    const int cnt = dsc.y;
    const bool mine = lane < cnt;
    const int4 e = mine ? E[dsc.x + lane] : make_int4(0, 0, 0, 0);
    const int rows = e.w >> 16;
    int incl = rows * 32;  // window bytes of blocks 0..lane
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int v = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += v;
    }
    const int toff = cnt * EXP_B_TILE + incl - rows * 32;
    if (mine) m.blk[lane] = make_int4(lane * EXP_B_TILE, toff, e.w & 0xFFFF, rows | (((e.y >> 8) & 0xFF) << 16));
    if (lane == 0) {
      m.count = cnt;
      m.last = dsc.w;
    }
    __syncwarp();
    // The arrival releases the record; the copies complete the phase.
    if (lane == 0) mbar_arrive_expect_tx(&full[stage], (uint32_t)(cnt * EXP_B_TILE + dsc.z));
    __syncwarp();
    const int pa = __shfl_up_sync(0xffffffffu, e.x, 1), py = __shfl_up_sync(0xffffffffu, e.y, 1);
    const int pz = __shfl_up_sync(0xffffffffu, e.z, 1), pr = __shfl_up_sync(0xffffffffu, rows, 1);
    const bool b_start = mine && (lane == 0 || e.x != pa + 1 || (e.y & 0xFF) != (py & 0xFF));
    const bool w_start = mine && (lane == 0 || e.z != pz + pr);
    const uint32_t bs = __ballot_sync(0xffffffffu, b_start) | (cnt < 32 ? (1u << cnt) : 0u);
    const uint32_t ws = __ballot_sync(0xffffffffu, w_start) | (cnt < 32 ? (1u << cnt) : 0u);
    const uint32_t above = lane < 31 ? ~((2u << lane) - 1u) : 0u;  // lanes after this one
    if (b_start) {
      const int len = __ffs(bs & above) - 1 - lane;
      for (int o = 0; o < len;) {
        const int lg = len - o >= 8 ? 3 : len - o >= 4 ? 2 : len - o >= 2 ? 1 : 0;
        tma_load_3d(st + (lane + o) * EXP_B_TILE, &bm.b3[lg], &full[stage], e.y & 0xFF, n0, e.x + o, pol);
        o += 1 << lg;
      }
    }
    const int wend = __ffs(ws & above) - 1;  // first lane after this one's window run
    const int wlast = __shfl_sync(0xffffffffu, incl, max(0, (w_start ? wend : lane + 1) - 1));
    if (w_start) bulk_load(st + toff, tw + (size_t)e.z * 16, (uint32_t)(wlast - (incl - rows * 32)), &full[stage]);
    ++issued;
    if (++stage == S) {
      stage = 0;
      phase ^= 1u;
    }
  }
  return true;
}

// F8: W and x are E4M3 codes (draft mode only): 128 values per 128-byte
// k-block row, kind::f8f6f4 MMAs, and the epilogue applies the row scales,
// y = bf16(acc * w_scale[n] * x_scale[m]).
template <bool F8>
__global__ void __launch_bounds__(SK_THREADS, 1)
    gemm_sk_kernel(const __grid_constant__ CUtensorMap tmap_w, const __grid_constant__ CUtensorMap tmap_x,
                   const __grid_constant__ SkBMaps bm, const SkArgs args) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t *ring = align_smem_1024(smem_raw);
  const int S = args.stages;
  const int stage_bytes = SK_WTILE + args.Mb * SK_BK * 2;
  constexpr int KBE = F8 ? 2 * SK_BK : SK_BK;  // values per k-block (the TMA coordinate unit)
  // Expand records (one per stage) and the producer's staged plan records.
  ExpandStage *meta = reinterpret_cast<ExpandStage *>(ring + (size_t)S * stage_bytes);
  int4 *chunk = reinterpret_cast<int4 *>(meta + S);
  uint64_t *full = reinterpret_cast<uint64_t *>(ring + (size_t)S * stage_bytes + expand_smem_bytes(S));
  uint64_t *empty = full + S;
  uint64_t *acc_full = empty + S;     // [2]: MMA commit -> epilogue
  uint64_t *acc_empty = acc_full + 2; // [2]: epilogue warps -> MMA issuer
  uint64_t *drain = acc_empty + 2;
  uint64_t *fix_bar = drain + 1;      // other participants' partial sums copied into the ring (reducers)
  uint64_t *epi_done = fix_bar + 1;   // every epilogue warp is done with tensor memory
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(epi_done + 1);
  int *abort_flag = reinterpret_cast<int *>(tmem_slot + 1);
  int *zero_word = abort_flag + 1;    // stays 0: for waits that only a time limit may end
  // The plan's expand block records, copied once per CTA (verify mode): every
  // owned unit scans them, so the scans read shared memory, not L2.
  int32_t *blk_cache = reinterpret_cast<int32_t *>(ring + (size_t)S * stage_bytes + expand_smem_bytes(S) + 256);
  // Per epilogue warp, its 32 W rows x 32 token columns of y in bf16, token-major.
  uint16_t *ystage = reinterpret_cast<uint16_t *>(blk_cache + SK_CACHE_BLOCKS * EXP_WORDS);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int cta = blockIdx.x;
  const int KB = args.kblocks;
  // Token group of this CTA and its index among the group's CTAs: CTA j of
  // every group streams the same W k-blocks at about the same time, so a W
  // tile read from DRAM for one group serves the others from L2.
  const int grp = cta / args.Pg, lc = cta - grp * args.Pg, cbase = grp * args.Pg;
  const int m0 = grp * args.Mb;
  const int g0 = sk_begin(args, lc), g1 = sk_begin(args, lc + 1);
  const bool tc = !F8 && args.sorted != 0 && args.mode == MLORA_VERIFY;
  const PlanLayout L = plan_layout(args.M, args.n_ad);

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&acc_full[b], 1);
      mbar_init(&acc_empty[b], 4);  // one arrival per epilogue warp
    }
    mbar_init(drain, 1);
    mbar_init(fix_bar, 1);
    mbar_init(epi_done, 4);
    *abort_flag = 0;
    *zero_word = 0;
    fence_mbar_init();
    grid_launch_dependents();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tmap_w);
    tma_prefetch_desc(&tmap_x);
    if (tc) {
      tma_prefetch_desc(&bm.b2);
      for (int q = 0; q < 4; ++q) tma_prefetch_desc(&bm.b3[q]);
    }
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, 2 * args.cols);
    tmem_relinquish();
  }
  tc_fence_before_sync();
  block_sync();
  tc_fence_after_sync();
  const uint32_t tmem_base = *tmem_slot;
  volatile int *ab = abort_flag;
  volatile int *never = zero_word;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    // The whole warp runs the loop and keeps the same ring position; lane 0
    // issues the k-blocks' copies, and at an owned tile's expand point the
    // lanes issue the expand stages from the plan.
    const uint64_t pol_w = policy_evict_first();
    const uint64_t pol_x = policy_evict_last();
    const uint32_t tx = (uint32_t)stage_bytes;
    int stage = 0, issued = 0, i = 0, early = 0, ns = -1, nst = 0;
    bool cached = false;
    uint32_t phase = 0;
    bool ok = true;
    bool waited = !args.after_shrink;
    if (lane == 0) {
      // With static weights the first ring of W tiles is requested before the
      // wait for the preceding kernel; x always comes after it.  (Not with the
      // expand: its operands would take ring stages between those k-blocks.)
      if (args.prefetch_w && !args.after_shrink && !tc) {
        for (int g = g0; g < g1 && early < S; ++g, ++early) {
          const int u = g / KB, kb = g - u * KB;
          mbar_arrive_expect_tx(&full[early], tx);
          tma_load_2d(ring + (size_t)early * stage_bytes, &tmap_w, &full[early], kb * KBE, u * SK_BN, pol_w);
        }
      }
      if (waited) grid_dependency_wait();
    }
    early = __shfl_sync(0xffffffffu, early, 0);
    // k-blocks [from, to) of unit u, all lanes: every lane waits for each
    // slot itself (a lane that waits alone while the others stand at a
    // shuffle measured about 0.5 us a wait), lane 0 issues the copies.  An
    // owned unit's k-block stages are marked in their record (count -1): the
    // MMA warp reads the kind of each of its stages.
    auto issue_kblocks = [&](int u, int from, int to) {
      const int w_row = u * SK_BN, x_row = m0;
      for (int kb = from; kb < to; ++kb, ++i) {
        uint8_t *st = ring + (size_t)stage * stage_bytes;
        if (i >= early) {
          if (!__all_sync(0xffffffffu, mbar_wait_bounded(&empty[stage], phase ^ 1u, ab))) {
            ok = false;
            break;
          }
          if (lane == 0) {
            if (tc) meta[stage].count = -1;
            mbar_arrive_expect_tx(&full[stage], tx);
            tma_load_2d(st, &tmap_w, &full[stage], kb * KBE, w_row, pol_w);
          }
        }
        if (lane == 0) tma_load_2d(st + SK_WTILE, &tmap_x, &full[stage], kb * KBE, x_row, pol_x);
        ++issued;
        if (++stage == S) {
          stage = 0;
          phase ^= 1u;
        }
      }
    };
    for (int g = g0; g < g1 && ok;) {
      const int u = g / KB, kb0 = g - u * KB, kb1 = min(KB, g1 - u * KB);
      const int t = u;
      const uint16_t *tws = args.tw + (size_t)sk_slice_of(args, t * SK_BN) * args.tw_slice;
      if (!(tc && kb0 == 0)) {
        issue_kblocks(u, kb0, kb1);
      } else {
        // An owned unit (verify mode): the expand operands go into the ring
        // before the unit's last S k-blocks, so that they land while those
        // stream; the first owned unit waits there for the kernels that wrote
        // the plan and the windows, while its first k-blocks stream.
        const int ins = max(kb0, kb1 - 1 - S);
        const int split = ins + 1;
        issue_kblocks(u, kb0, split);
        if (ok) {
          if (!waited) {
            grid_dependency_wait();  // the token windows come from the shrink kernel just before
            waited = true;
          }
          if (ns < 0) ns = args.plan[L.hdr + 4];
          // Also with no blocks at all (an empty stage flagged `last`): the MMA
          // warp runs every owned unit's stages until `last`.
          if (!cached && ns <= SK_CACHE_BLOCKS) {
            const int4 *src = reinterpret_cast<const int4 *>(args.plan + L.slices);
            for (int q = lane; q < ns * (EXP_WORDS / 4); q += 32) reinterpret_cast<int4 *>(blk_cache)[q] = src[q];
            __syncwarp();
            nst = sk_expand_plan(blk_cache, ns, m0, args.Mb, args.n_ad, (long long)(args.tw_slice / 16),
                                 stage_bytes, lane, args.status);
            cached = true;
          }
          if (cached)
            ok = sk_expand_issue(blk_cache, 0, nst, bm, t * SK_BN, tws, ring, stage_bytes, S, full, empty, meta,
                                 stage, phase, issued, ab, pol_w, lane);
          else
            ok = expand_produce(args.plan + L.slices, 0, ns, m0, args.Mb, t * SK_BN, args.N, &bm.b2, tws, ring,
                                stage_bytes, S, full, empty, meta, chunk, stage, phase, issued, ab, pol_w, lane,
                                args.n_ad, (long long)(args.tw_slice / 16), args.status);
        }
        if (ok) issue_kblocks(u, split, kb1);
      }
      g = u * KB + kb1;
    }
    if (lane == 0) {
      if (!ok) {
        *reinterpret_cast<volatile int *>(abort_flag) = 1;
        raise_status(args.status, MLORA_DEV_TIMEOUT);
      }
      if (*ab) {
        // Let this CTA's own copies land before shared memory goes away.
        const int n = issued < S ? issued : S;
        for (int k = issued - n; k < issued; ++k) {
          mbar_wait_bounded(&full[k % S], (uint32_t)((k / S) & 1), never);
        }
        for (int k = issued; k < early; ++k) {
          mbar_wait_bounded(&full[k], 0u, never);  // W half only: never completes, bounded
        }
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    const uint32_t idesc = F8 ? idesc_e4m3_f32(SK_BN, args.Mb) : idesc_bf16_f32(SK_BN, args.Mb);
    const uint32_t ring0 = smem_addr(ring);
    const uint32_t sbytes = (uint32_t)stage_bytes;
    int stage = 0, seg = 0;
    uint32_t phase = 0;
    bool ok = true, issued_any = false;
    for (int g = g0; g < g1 && ok; ++seg) {
      const int u = g / KB, kb0 = g - u * KB, kb1 = min(KB, g1 - u * KB);
      const int buf = seg & 1;
      const uint32_t acc = tmem_base + (uint32_t)(buf * args.cols);
      // The whole warp runs the segment's stages (every lane tests each
      // barrier itself), lane 0 issues the MMAs.  An owned unit (verify
      // mode) has its expand stages among its k-blocks wherever the producer
      // put them: each stage's record says which it is (count < 0: a
      // k-block), and the unit's stages end with its last k-block and the
      // expand stage flagged `last`, in either order.
      const bool expand_here = tc && kb0 == 0;
      if (seg >= 2 && ok)  // the accumulator's previous use (segment seg - 2) must be drained
        ok = __all_sync(0xffffffffu, mbar_wait_bounded(&acc_empty[buf], (uint32_t)(((seg >> 1) - 1) & 1), ab));
      tc_fence_after_sync();
      int kb = kb0;
      bool seen_last = !expand_here;
      while (ok && (kb < kb1 || !seen_last)) {
        if (!__all_sync(0xffffffffu, mbar_wait_bounded(&full[stage], phase, ab))) {
          ok = false;
          break;
        }
        tc_fence_after_sync();
        if (!expand_here || meta[stage].count < 0) {
          if (lane == 0) {
            const uint32_t a_addr = ring0 + (uint32_t)stage * sbytes;
            const uint64_t ad = smem_desc_kmajor_sw128(a_addr);
            const uint64_t bd = smem_desc_kmajor_sw128(a_addr + SK_WTILE);
            const uint32_t first = kb > kb0 ? 1u : 0u;
#pragma unroll
            for (int kk = 0; kk < SK_BK / 16; ++kk) {  // 32 bytes of K per instruction
              if (F8)
                mma_e4m3_ss(acc, ad + 2 * kk, bd + 2 * kk, idesc, kk > 0 ? 1u : first);
              else
                mma_bf16_ss(acc, ad + 2 * kk, bd + 2 * kk, idesc, kk > 0 ? 1u : first);
            }
            mma_commit(&empty[stage]);
          }
          ++kb;
        } else {
          seen_last = meta[stage].last != 0;
          expand_stage_mma(ring + (size_t)stage * stage_bytes, meta[stage], acc, &empty[stage], lane);
        }
        issued_any = true;
        __syncwarp();
        if (++stage == S) {
          stage = 0;
          phase ^= 1u;
        }
      }
      if (lane == 0 && ok) mma_commit(&acc_full[buf]);
      __syncwarp();
      g = u * KB + kb1;
    }
    issued_any = __shfl_sync(0xffffffffu, issued_any ? 1 : 0, 0) != 0 || issued_any;
    if (lane == 0 && !ok) {
      *reinterpret_cast<volatile int *>(abort_flag) = 1;
      raise_status(args.status, MLORA_DEV_TIMEOUT);
      if (issued_any) {
        // Wait for this thread's MMAs before tensor memory is freed.
        mma_commit(drain);
        mbar_wait_bounded(drain, 0, never);
      }
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ epilogue
    // Warp w reads tensor-memory lanes 32*(w%4)..+31: tile rows.
    const int quad = warp & 3, et = threadIdx.x - 64;
    const int row = quad * 32 + lane;
    const int32_t *perm = tc ? args.plan + L.perm : nullptr;  // output row of each accumulator column
    const uint32_t lane_off = (uint32_t)(quad * 32) << 16;
    grid_dependency_wait();  // y and the flags may still be in use by the preceding kernel
    int seg = 0;
    for (int g = g0; g < g1; ++seg) {
      const int u = g / KB, kb0 = g - u * KB, kb1 = min(KB, g1 - u * KB);
      const int t = u;
      const int gcols = min(args.Mb, args.M - m0);  // token columns of this unit
      const int buf = seg & 1;
      // All 128 threads agree on the outcome before any of them branches, so
      // the named barriers below are always reached by every thread.
      const bool ready = named_bar_and(1, 128, mbar_wait_bounded(&acc_full[buf], (uint32_t)((seg >> 1) & 1), ab));
      if (!ready) {
        if (et == 0) {
          *reinterpret_cast<volatile int *>(abort_flag) = 1;
          raise_status(args.status, MLORA_DEV_TIMEOUT);
        }
        __syncwarp();
        break;
      }
      tc_fence_after_sync();
      const uint32_t acc = tmem_base + (uint32_t)(buf * args.cols) + lane_off;
      const int nchunks = (gcols + SK_CHUNK - 1) / SK_CHUNK;
      const int n = t * SK_BN + row;
      // y for accumulator columns [cb, min(cb + 32, c_end)) from v: column c
      // is token position m0 + c, output row perm[m0 + c] with sorted rows
      // (lane j fetches it), else m0 + c.  An entry out of range (a plan
      // overwritten or made for other sizes) skips the store and raises
      // MLORA_DEV_BAD_PLAN.
      auto store_y = [&](int cb, int c_end, const float (&v)[SK_CHUNK]) {
        const int myc = m0 + cb + lane;
        int myrow = myc;
        if (perm) {
          myrow = myc < args.M ? __ldg(perm + myc) : -1;
          if (myc < args.M && (unsigned)myrow >= (unsigned)args.M) {
            raise_status(args.status, MLORA_DEV_BAD_PLAN);
            myrow = -1;
          }
        }
        uint16_t *yn = args.y + n;
        float wsn = 1.f, myxs = 1.f;  // E4M3: the scales of this thread's W row and of lane's token row
        if (F8) {
          wsn = n < args.N ? __ldg(args.w_scale + n) : 0.f;
          myxs = myc < args.M ? __ldg(args.x_scale + myc) : 0.f;
        }
        if (args.vec_y) {
          // Through shared memory: lane l writes its W row's 32 outputs as
          // column l of the warp's token-major block, then owns token
          // column l and stores its 32 outputs (this warp's 32 W rows) as
          // four 16-byte pieces.  The rows are padded to 80 bytes, so
          // neither side has bank conflicts.
          uint16_t *sy = ystage + (size_t)(quad * 32) * SK_YROW;
#pragma unroll
          for (int j = 0; j < SK_CHUNK; ++j) {
            const float xs = F8 ? __shfl_sync(0xffffffffu, myxs, j) : 1.f;
            sy[j * SK_YROW + lane] = float_to_bf16_bits(F8 ? v[j] * wsn * xs : v[j]);
          }
          __syncwarp();
          const int nb = t * SK_BN + quad * 32;  // first W row of this warp
          if (cb + lane < c_end && myrow >= 0) {
            const uint4 *src = reinterpret_cast<const uint4 *>(sy + lane * SK_YROW);
            uint16_t *dst = args.y + (size_t)myrow * args.N + nb;
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              if (nb + 8 * q + 8 <= args.N) {
                reinterpret_cast<uint4 *>(dst)[q] = src[q];
              } else {
                for (int e = 0; e < 8; ++e)
                  if (nb + 8 * q + e < args.N) dst[8 * q + e] = sy[lane * SK_YROW + 8 * q + e];
              }
            }
          }
          __syncwarp();  // the block is rewritten by the next chunk
          return;
        }
#pragma unroll
        for (int j = 0; j < SK_CHUNK; ++j) {
          const int orow = __shfl_sync(0xffffffffu, myrow, j);
          const float xs = F8 ? __shfl_sync(0xffffffffu, myxs, j) : 1.f;
          if (n < args.N && cb + j < c_end && orow >= 0)
            yn[(size_t)orow * args.N] = float_to_bf16_bits(F8 ? v[j] * wsn * xs : v[j]);
        }
      };
      if (kb0 == 0 && kb1 == KB) {
        // A whole unit: round once and store y straight from tensor memory.
        for (int cb = 0; cb < gcols; cb += SK_CHUNK) {
          uint32_t r[32];
          tmem_ld_x32(acc + cb, r);
          tmem_ld_wait();
          float v[SK_CHUNK];
#pragma unroll
          for (int j = 0; j < SK_CHUNK; ++j) v[j] = __uint_as_float(r[j]);
          store_y(cb, gcols, v);
        }
        tc_fence_before_sync();
        __syncwarp();
        if (lane == 0) mbar_arrive(&acc_empty[buf]);
      } else {
        // A split tile.  Every participant (the CTAs first..last holding its
        // k-blocks) publishes its fp32 partial sums, then counts itself in on
        // the tile's arrival word.  The participants whose shares end inside
        // the tile (all but a last one that continues past it) then reduce
        // it together: each takes an equal slice of the token columns, adds
        // every participant's partial for them in CTA order and stores y.
        // Only a CTA's last segment can reduce, and it publishes every
        // earlier split segment first, so all arrivals come before any wait;
        // all CTAs are resident at once, so the waits end (and are bounded).
        const int first = cbase + sk_cta_of(args, u * KB), last = cbase + sk_cta_of(args, (u + 1) * KB - 1);
        const int npart = last - first + 1;
        const int r_last = sk_begin(args, last - cbase + 1) <= (u + 1) * KB ? last : last - 1;
        const bool reducer = sk_begin(args, lc + 1) <= (u + 1) * KB;
        // Partial slot: 0 for a CTA's first segment, 1 for a later one.
        auto part_of = [&](int pc) {
          return args.partials + ((size_t)pc * 2 + (sk_begin(args, pc - cbase) >= u * KB ? 0 : 1)) * args.Mb * SK_BN;
        };
        // A reducer adds its own sums straight from tensor memory; it writes
        // them out only when other reducers need them.
        const int nred = r_last - first + 1;
        const bool publish = !reducer || nred > 1;
        if (publish) {
          // Through the warp's staging block, 16 columns at a time: each
          // column's 32 rows (this warp's) as 36 floats, so that lane l
          // stores rows 4 (l % 8) .. + 3 of column l / 8 + 4 q as one
          // 16-byte piece (no bank conflicts on either side).
          float *part = part_of(cta);
          float *sp = reinterpret_cast<float *>(ystage) + (size_t)quad * 16 * (32 + 4);
          for (int ch = 0; ch < nchunks; ++ch) {
            uint32_t r[32];
            tmem_ld_x32(acc + ch * SK_CHUNK, r);
            tmem_ld_wait();
#pragma unroll
            for (int h = 0; h < SK_CHUNK; h += 16) {
#pragma unroll
              for (int j = 0; j < 16; ++j) sp[j * 36 + lane] = __uint_as_float(r[h + j]);
              __syncwarp();
#pragma unroll
              for (int q = 0; q < 4; ++q) {
                const int jc = (lane >> 3) + 4 * q, col = ch * SK_CHUNK + h + jc;
                if (col < gcols)
                  *reinterpret_cast<float4 *>(part + (size_t)col * SK_BN + quad * 32 + 4 * (lane & 7)) =
                      *reinterpret_cast<const float4 *>(sp + jc * 36 + 4 * (lane & 7));
              }
              __syncwarp();  // the block is rewritten by the next half
            }
          }
        }
        if (!reducer) {
          tc_fence_before_sync();
          __syncwarp();
          if (lane == 0) mbar_arrive(&acc_empty[buf]);  // the accumulator is free: the partial holds it
        }
        named_bar_sync(1, 128);
        if (et == 0) {
          __threadfence();  // after the barrier: covers the partial sums every thread stored
          atomic_add_release_gpu(&args.flags[first], 1u);
        }
        __syncwarp();
        if (reducer) {
          bool have = true;
          if (et == 0) {
            // The timeout test polls a word past the grid's, which no CTA
            // sets, for test_flag_wait_ns instead of the tile's arrivals.
            const bool probe = args.test_flag_wait_ns != 0;
            const uint64_t limit = probe ? (uint64_t)args.test_flag_wait_ns : WAIT_LIMIT_NS;
            const uint32_t *word = &args.flags[probe ? 2 * args.P + first : first];
            bool seen = ld_acquire_gpu(word) >= (uint32_t)npart;
            if (!seen) {
              const uint64_t t0 = global_timer_ns();
              while (!(seen = ld_acquire_gpu(word) >= (uint32_t)npart)) {
                if (global_timer_ns() - t0 > limit) break;
                sleep_ns(32);
              }
            }
            if (!seen) {
              have = false;
              raise_status(args.status, MLORA_DEV_TIMEOUT);
            }
            fence_proxy_async_global();  // the bulk copies below read what generic stores wrote
          }
          __syncwarp();  // warps reach a barrier converged (bar.* counts whole warps)
          have = named_bar_and(1, 128, have);
          const int ri = cta - first;
          const int per = ((gcols + nred - 1) / nred + SK_CHUNK - 1) / SK_CHUNK * SK_CHUNK;
          const int c0 = ri * per, c1 = min(gcols, c0 + per);
          // The other participants' partials for the slice come into the
          // stage ring (idle in a CTA's last segment: every load landed and
          // every MMA that read it completed) with bulk copies, in rounds of
          // columns that fit it; this CTA's own sums come from tensor memory.
          const int nother = npart - 1;
          const size_t ring_bytes = (size_t)S * stage_bytes;
          int round_cols = (int)(ring_bytes / ((size_t)nother * SK_BN * 4)) / SK_CHUNK * SK_CHUNK;
          if (round_cols < SK_CHUNK) {  // excluded by the host's bound on participants
            if (have && et == 0) raise_status(args.status, MLORA_DEV_TIMEOUT);
            have = false;
          }
          const float *ringf = reinterpret_cast<const float *>(ring);
          uint32_t fix_phase = 0;
          for (int q0 = c0; have && q0 < c1; q0 += round_cols) {
            const int q1 = min(c1, q0 + round_cols), qn = q1 - q0;
            if (et == 0) {
              const uint32_t bytes = (uint32_t)qn * SK_BN * 4;
              mbar_arrive_expect_tx(fix_bar, bytes * (uint32_t)nother);
              int o = 0;
              for (int pc = first; pc <= last; ++pc)
                if (pc != cta) bulk_load(ring + (size_t)(o++) * qn * SK_BN * 4, part_of(pc) + (size_t)q0 * SK_BN, bytes,
                                         fix_bar);
            }
            __syncwarp();
            // Not cut short by the abort flag: the copies must land before
            // shared memory is reused or released.
            const bool landed = named_bar_and(1, 128, mbar_wait_bounded(fix_bar, fix_phase, never));
            fix_phase ^= 1u;
            if (!landed) {
              if (et == 0) raise_status(args.status, MLORA_DEV_TIMEOUT);
              have = false;
              break;
            }
            for (int cb = q0; cb < q1; cb += SK_CHUNK) {
              uint32_t r[32];
              tmem_ld_x32(acc + cb, r);
              tmem_ld_wait();
              float v[SK_CHUNK];
#pragma unroll
              for (int j = 0; j < SK_CHUNK; ++j) v[j] = 0.f;
              int o = 0;
              for (int pc = first; pc <= last; ++pc) {
                if (pc == cta) {
#pragma unroll
                  for (int j = 0; j < SK_CHUNK; ++j) v[j] += __uint_as_float(r[j]);
                  continue;
                }
                // Sixteen independent loads, then their sums.  Columns past
                // q1 read other bytes of the ring (inside it: qn <=
                // round_cols) and are never stored.
                const float *pp = ringf + ((size_t)(o++) * qn + (cb - q0)) * SK_BN + row;
#pragma unroll
                for (int h = 0; h < SK_CHUNK; h += 16) {
                  float t[16];
#pragma unroll
                  for (int j = 0; j < 16; ++j) t[j] = pp[(h + j) * SK_BN];
#pragma unroll
                  for (int j = 0; j < 16; ++j) v[h + j] += t[j];
                }
              }
              store_y(cb, q1, v);
            }
            named_bar_sync(1, 128);  // the ring is refilled only after every thread read it
          }
          tc_fence_before_sync();
          __syncwarp();
          if (lane == 0) mbar_arrive(&acc_empty[buf]);
          // The last reducer to finish puts the tile's words back to zero.
          named_bar_sync(1, 128);
          if (et == 0) {
            const uint32_t prev = atomicAdd(&args.flags[args.P + first], 1u);
            if (prev == (uint32_t)(nred - 1)) {
              args.flags[first] = 0u;
              args.flags[args.P + first] = 0u;
            }
          }
          __syncwarp();
        }
      }
      g = u * KB + kb1;
    }
    tc_fence_before_sync();
    __syncwarp();
    if (lane == 0) mbar_arrive(epi_done);
  }

  // Tensor memory is released only once every epilogue warp has finished
  // reading it (an mbarrier, so that the release does not rest on a CTA
  // barrier reached by warps whose lanes took different paths).
  if (warp == 1) {
    if (lane == 0) {
      if (!mbar_wait_bounded(epi_done, 0u, never)) raise_status(args.status, MLORA_DEV_TIMEOUT);
    }
    __syncwarp();
  }
  tc_fence_before_sync();
  block_sync();
  if (warp == 1) {
    tc_fence_after_sync();
    tmem_dealloc(tmem_base, 2 * args.cols);
  }
}

// One CTA of this shared-memory size fits on an SM (so a grid of one CTA per
// SM is resident at once on an otherwise idle GPU).  Cached per device.
template <bool F8>
static bool sk_resident(size_t smem) {
  static int attr_done[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return false;
  if (!attr_done[dev]) {
    if (cudaFuncSetAttribute(gemm_sk_kernel<F8>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)SK_SMEM_LIMIT) !=
        cudaSuccess) {
      cudaGetLastError();
      return false;
    }
    attr_done[dev] = 1;
  }
  int n = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, gemm_sk_kernel<F8>, SK_THREADS, smem) != cudaSuccess) {
    cudaGetLastError();
    return false;
  }
  return n >= 1;
}

// Token groups of M rows: as few as keep a group within SK_GROUP_ROWS, of
// equal size rounded up to 16 (the MMA's N granularity).
static void sk_groups(int M, int *n_tg, int *Mb) {
  const int g = (M + SK_GROUP_ROWS - 1) / SK_GROUP_ROWS;
  *n_tg = g;
  *Mb = ((M + g - 1) / g + 15) / 16 * 16;
}

SkShape sk_shape(int M, int N, int K, int num_sms, bool f8) {
  SkShape s = {};
  s.ok = false;
  if (M < 1 || M > SK_GROUP_ROWS * SK_MAX_GROUPS || num_sms <= 0) return s;
  sk_groups(M, &s.n_tg, &s.Mb);
  int cols = 32;
  while (cols < s.Mb) cols <<= 1;
  s.cols = cols;
  const int stage_bytes = SK_WTILE + s.Mb * SK_BK * 2;
  int st = (int)((SK_SMEM_LIMIT - SK_SMEM_FIXED) / stage_bytes);
  s.stages = st > SK_MAX_STAGES ? SK_MAX_STAGES : st;
  if (s.stages < 2) return s;
  s.n_tiles = (N + SK_BN - 1) / SK_BN;
  const int kbe = f8 ? 2 * SK_BK : SK_BK;  // values per 128-byte k-block row
  s.kblocks = (K + kbe - 1) / kbe;
  s.total = s.n_tiles * s.kblocks;  // (tile, k-block) pairs of one token group
  // Shares of at least ceil(kblocks / SK_MAX_PARTIALS) k-blocks: a unit then
  // meets at most SK_MAX_PARTIALS + 1 CTAs.
  int share = (s.kblocks + SK_MAX_PARTIALS - 1) / SK_MAX_PARTIALS;
  if (share < SK_MIN_SHARE) share = SK_MIN_SHARE;
  // The same number of CTAs for each token group, all resident at once.
  int Pg = s.total / share;
  if (Pg > num_sms / s.n_tg) Pg = num_sms / s.n_tg;
  if (Pg < 1) Pg = 1;
  s.Pg = Pg;
  s.P = Pg * s.n_tg;
  s.smem_bytes = SK_SMEM_FIXED + (size_t)s.stages * stage_bytes;
  s.ok = f8 ? sk_resident<true>(s.smem_bytes) : sk_resident<false>(s.smem_bytes);
  return s;
}

size_t sk_partial_bytes(int M, int num_sms) {
  if (M < 1 || M > SK_GROUP_ROWS * SK_MAX_GROUPS) return 0;
  int n_tg = 0, Mb = 0;
  sk_groups(M, &n_tg, &Mb);
  return (size_t)num_sms * 2 * Mb * SK_BN * sizeof(float);
}

typedef CUresult (*SkEncodeFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                               const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                               CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static SkEncodeFn sk_encode_fn() {
  static SkEncodeFn fn = nullptr;
  if (!fn) {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<SkEncodeFn>(p);
  }
  return fn;
}

// Row-major bf16 [rows, cols] read in boxes of box_rows x box_cols (64 columns
// with 128-byte swizzling, or 16 with 32-byte swizzling); out of range reads 0.
// bytes1: one-byte elements (E4M3 codes), boxes of 128 columns, 128-byte swizzle.
static bool sk_map(CUtensorMap *map, const void *base, long long rows, int cols, int box_rows, int box_cols,
                   bool bytes1 = false) {
  SkEncodeFn fn = sk_encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)cols * (bytes1 ? 1 : 2)};
  cuuint32_t box[2] = {(cuuint32_t)box_cols, (cuuint32_t)box_rows};
  cuuint32_t estr[2] = {1, 1};
  const CUtensorMapSwizzle sw = box_cols == 16 ? CU_TENSOR_MAP_SWIZZLE_32B : CU_TENSOR_MAP_SWIZZLE_128B;
  return fn(map, bytes1 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2,
            const_cast<void *>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// B_stack [n_ad][N][r_max] bf16 as a 3-D map {r_max, N, n_ad}: boxes of 16
// ranks x 128 rows x `depth` consecutive adapters, 32-byte swizzle (each
// adapter's 128 x 16 tile lands as with the 2-D view); out of range reads 0.
static bool sk_map_b3(CUtensorMap *map, const void *base, int n_ad, int N, int r_max, int depth) {
  SkEncodeFn fn = sk_encode_fn();
  if (!fn) return false;
  cuuint64_t dims[3] = {(cuuint64_t)r_max, (cuuint64_t)N, (cuuint64_t)n_ad};
  cuuint64_t strides[2] = {(cuuint64_t)r_max * 2, (cuuint64_t)N * r_max * 2};
  cuuint32_t box[3] = {16, (cuuint32_t)SK_BN, (cuuint32_t)depth};
  cuuint32_t estr[3] = {1, 1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_32B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

cudaError_t launch_gemm_sk(const GemmLaunch &g, const SkShape &sh, float *partials, uint32_t *flags, cudaStream_t s,
                           int *err_code) {
  *err_code = 0;
  if (!sh.ok) return cudaErrorInvalidValue;  // sk_shape set the kernel's attributes when it said ok
  CUtensorMap tw, tx;
  if (!sk_map(&tw, g.W, g.N, g.K, SK_BN, SK_BK) || !sk_map(&tx, g.x, g.M, g.K, sh.Mb, SK_BK)) {
    *err_code = 1;
    return cudaErrorInvalidValue;
  }
  const int sorted = (g.mode == MLORA_VERIFY && g.tw != nullptr) ? 1 : 0;
  SkBMaps bm;
  bm.b2 = tw;
  for (int q = 0; q < 4; ++q) bm.b3[q] = tw;
  if (sorted) {
    bool mapped = sk_map(&bm.b2, g.B_stack, (long long)g.n_ad * g.N, g.r_max, SK_BN, 16);
    // A run of consecutive adapters never exceeds n_ad: deeper boxes than
    // that are never used (a copy of the one-adapter map stands in).
    for (int q = 0; q < 4 && mapped; ++q)
      mapped = (1 << q) <= g.n_ad ? sk_map_b3(&bm.b3[q], g.B_stack, g.n_ad, g.N, g.r_max, 1 << q)
                                  : (bm.b3[q] = bm.b3[0], true);
    if (!mapped) {
      *err_code = 1;
      return cudaErrorInvalidValue;
    }
  }
  SkArgs a;
  a.M = g.M;
  a.N = g.N;
  a.K = g.K;
  a.Mb = sh.Mb;
  a.n_tg = sh.n_tg;
  a.kblocks = sh.kblocks;
  a.total = sh.total;
  a.P = sh.P;
  a.Pg = sh.Pg;
  a.stages = sh.stages;
  a.cols = sh.cols;
  a.mode = g.mode;
  a.prefetch_w = g.prefetch_w;
  a.after_shrink = g.after_shrink;
  a.sorted = sorted;
  a.n_slices = g.n_slices;
  for (int i = 0; i < MLORA_MAX_SLICES; ++i) a.slice_end[i] = i < g.n_slices ? g.slice_end[i] : g.N;
  a.tw_slice = max_window_rows(g.M, g.n_ad) * 16;
  a.test_flag_wait_ns = g.test_flag_wait_ns;
  a.n_ad = g.n_ad;
  a.y = g.y;
  a.vec_y = (g.N % 8 == 0 && (reinterpret_cast<uintptr_t>(g.y) & 15) == 0) ? 1 : 0;
  a.tw = g.tw;
  a.plan = g.plan;
  a.status = g.status;
  a.partials = partials;
  a.flags = flags;
  a.w_scale = nullptr;
  a.x_scale = nullptr;
  cudaError_t e = launch_pdl(gemm_sk_kernel<false>, dim3(sh.P), dim3(SK_THREADS), sh.smem_bytes, s, tw, tx, bm, a);
  return e != cudaSuccess ? e : cudaGetLastError();
}

cudaError_t launch_gemm_sk_f8(const F8Launch &g, const SkShape &sh, float *partials, uint32_t *flags, cudaStream_t s,
                              int *err_code) {
  *err_code = 0;
  if (!sh.ok) return cudaErrorInvalidValue;
  CUtensorMap tw, tx;
  if (!sk_map(&tw, g.W8, g.N, g.K, SK_BN, 2 * SK_BK, true) || !sk_map(&tx, g.x8, g.M, g.K, sh.Mb, 2 * SK_BK, true)) {
    *err_code = 1;
    return cudaErrorInvalidValue;
  }
  SkArgs a = {};
  a.M = g.M;
  a.N = g.N;
  a.K = g.K;
  a.Mb = sh.Mb;
  a.n_tg = sh.n_tg;
  a.kblocks = sh.kblocks;
  a.total = sh.total;
  a.P = sh.P;
  a.Pg = sh.Pg;
  a.stages = sh.stages;
  a.cols = sh.cols;
  a.mode = MLORA_DRAFT;
  a.prefetch_w = g.prefetch_w;
  a.after_shrink = 0;
  a.sorted = 0;
  a.n_slices = 1;
  for (int i = 0; i < MLORA_MAX_SLICES; ++i) a.slice_end[i] = g.N;
  a.y = g.y;
  a.vec_y = (g.N % 8 == 0 && (reinterpret_cast<uintptr_t>(g.y) & 15) == 0) ? 1 : 0;
  a.status = g.status;
  a.partials = partials;
  a.flags = flags;
  a.w_scale = g.w_scale;
  a.x_scale = g.x_scale;
  SkBMaps bm;  // no expand in the E4M3 draft pass: placeholders
  bm.b2 = tw;
  for (int q = 0; q < 4; ++q) bm.b3[q] = tw;
  cudaError_t e = launch_pdl(gemm_sk_kernel<true>, dim3(sh.P), dim3(SK_THREADS), sh.smem_bytes, s, tw, tx, bm, a);
  return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace mlora
