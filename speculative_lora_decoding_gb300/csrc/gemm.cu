// Steps a3 + a4: the base GEMM acc = x W^T on the tcgen05 tensor cores and
// the low-rank expand fused into its epilogue:
//
//   draft  (LoRA off): y[m, n] = bf16(acc[m, n])
//   verify (LoRA on):  y[m, n] = bf16(acc[m, n] + scale * sum_{j<r} T[m, j] B_a[n, j]),  a = adapter of row m
//
// ("output = W·x + scale · B(A·x)", "Multi-LoRA Serving in Practice", section
// "Core Principle: Shared Base Model, Per-Request Adapter Selection"; the two
// modes are the LoRA-off draft pass and LoRA-on verify pass of the
// InvisibleLoRA abstract.)
//
// Design for sm_103a:
//  * Operands swapped: 128 rows of W form the MMA's M side, the (few) token
//    rows its N side (16..256 per instruction, two instructions for up to 512
//    tokens).  Decode batches are small, so this keeps the tensor-core tile
//    full while W streams through exactly once.
//  * A unit is 128 W rows x up to 512 tokens.  When there are too few units
//    to cover the SMs, the C CTAs of one thread-block cluster split the unit's
//    K range (split-K).  Their fp32 accumulators meet in distributed shared
//    memory: each CTA copies its accumulator, 32 columns at a time, out of
//    tensor memory into its own shared memory, and then sums rows
//    [rank*128/C, (rank+1)*128/C) over all C CTAs in rank order.  The
//    reduction stays on chip, runs on all C CTAs at once and is deterministic.
//  * Warp roles: warp 0 issues TMA loads of W and x tiles (128-byte swizzle)
//    into a ring of shared-memory stages; warp 1 owns tensor memory and issues
//    tcgen05.mma from one thread; warps 2..5 drain the accumulator with
//    tcgen05.ld and run the epilogue.
//  * Programmatic dependent launch: the prologue (barriers, tensor memory,
//    descriptor prefetch) runs while the previous kernel in the stream
//    finishes; activations, T and the plan are read only after
//    griddepcontrol.wait.  With MLORA_PREFETCH_WEIGHTS the first ring of W
//    tiles is requested before that wait too.
//  * Every mbarrier wait is bounded; on expiry the CTA raises
//    MLORA_DEV_TIMEOUT, drains its own copies and MMAs, still takes part in
//    every cluster barrier, frees its tensor memory and returns.
#include "common.cuh"
#include "launch.h"

namespace mlora {

constexpr int GEMM_THREADS = 192;
constexpr int BLOCK_N = 128;                          // W rows per unit (MMA M)
constexpr int BLOCK_K = 64;                           // K per stage: 128 bytes of bf16
constexpr int W_TILE_BYTES = BLOCK_N * BLOCK_K * 2;   // 16 KB
constexpr int MAX_MB = 512;
constexpr int CHUNK = 32;                             // accumulator columns per reduction round
constexpr int RED_BYTES = 2 * CHUNK * BLOCK_N * 4;    // double-buffered reduction tile, 32 KB
constexpr int MAX_CLUSTER = 16;
constexpr size_t SMEM_LIMIT = 227 * 1024;
constexpr size_t SMEM_FIXED = 1024 + 256;             // alignment slack + barriers

struct GemmArgs {
  int M, N, K;
  int Mb, nsub, sub_n, n_tgroups, kblocks, C, stages, tmem_cols, red_bytes;
  int mode, prefetch_w;
  float scale;
  uint16_t *y;
  const uint16_t *B_stack;
  int r_max, n_ad;
  const float *T;
  const int32_t *plan;
  uint32_t *status;
};

struct SmemPtrs {
  uint8_t *stage0;
  float *red;
  uint64_t *full, *empty, *tfull, *drain;
  uint32_t *tmem_slot;
  int *abort_flag;
};

__device__ __forceinline__ SmemPtrs carve_smem(uint8_t *base, int stages, int stage_bytes, int red_bytes) {
  SmemPtrs p;
  p.stage0 = base;
  p.red = reinterpret_cast<float *>(base + (size_t)stages * stage_bytes);
  uint64_t *bars = reinterpret_cast<uint64_t *>(base + (size_t)stages * stage_bytes + red_bytes);
  p.full = bars;
  p.empty = bars + stages;
  p.tfull = bars + 2 * stages;
  p.drain = bars + 2 * stages + 1;
  uint32_t *w = reinterpret_cast<uint32_t *>(bars + 2 * stages + 2);
  p.tmem_slot = w;
  p.abort_flag = reinterpret_cast<int *>(w + 1);
  return p;
}

__device__ __forceinline__ void signal_abort(SmemPtrs &sp, uint32_t *status) {
  *reinterpret_cast<volatile int *>(sp.abort_flag) = 1;
  raise_status(status, MLORA_DEV_TIMEOUT);
}

__device__ __forceinline__ void unpack_bf16x2(uint32_t w, float &lo, float &hi) {
  lo = __uint_as_float(w << 16);
  hi = __uint_as_float(w & 0xFFFF0000u);
}

// B_a[n, 0:64] as packed bf16 pairs; entries at or past rank r are zeroed
// (the padding is never used, even if it holds NaN).
__device__ __forceinline__ void load_brow(const GemmArgs &a, int ad, int n, int r, uint32_t (&bp)[32]) {
#pragma unroll
  for (int i = 0; i < 32; ++i) bp[i] = 0u;
  if (r <= 0 || n >= a.N) return;
  const uint4 *brow = reinterpret_cast<const uint4 *>(a.B_stack + ((size_t)ad * a.N + n) * a.r_max);
#pragma unroll
  for (int q = 0; q < 8; ++q) {
    if (q * 8 < r) {
      const uint4 v = __ldg(brow + q);
      bp[4 * q + 0] = v.x;
      bp[4 * q + 1] = v.y;
      bp[4 * q + 2] = v.z;
      bp[4 * q + 3] = v.w;
    }
  }
#pragma unroll
  for (int e = 0; e < 32; ++e) {
    if (2 * e >= r) bp[e] &= 0xFFFF0000u;
    if (2 * e + 1 >= r) bp[e] &= 0x0000FFFFu;
  }
}

// sum_{j < r} T[m, j] * B[j], fp32, j in increasing order.
__device__ __forceinline__ float lowrank_dot(const float *T, int m, const uint32_t (&bp)[32], int r) {
  const float4 *trow = reinterpret_cast<const float4 *>(T + (size_t)m * T_STRIDE);
  float dot = 0.f;
#pragma unroll
  for (int q = 0; q < 8; ++q) {
    if (q * 8 < r) {
      const float4 t0 = __ldg(trow + 2 * q), t1 = __ldg(trow + 2 * q + 1);
      float b0, b1, b2, b3, b4, b5, b6, b7;
      unpack_bf16x2(bp[4 * q + 0], b0, b1);
      unpack_bf16x2(bp[4 * q + 1], b2, b3);
      unpack_bf16x2(bp[4 * q + 2], b4, b5);
      unpack_bf16x2(bp[4 * q + 3], b6, b7);
      dot = fmaf(t0.x, b0, dot);
      dot = fmaf(t0.y, b1, dot);
      dot = fmaf(t0.z, b2, dot);
      dot = fmaf(t0.w, b3, dot);
      dot = fmaf(t1.x, b4, dot);
      dot = fmaf(t1.y, b5, dot);
      dot = fmaf(t1.z, b6, dot);
      dot = fmaf(t1.w, b7, dot);
    }
  }
  return dot;
}

__global__ void __launch_bounds__(GEMM_THREADS, 1)
    gemm_kernel(const __grid_constant__ CUtensorMap tmap_w, const __grid_constant__ CUtensorMap tmap_x,
                const GemmArgs args) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
  const int S = args.stages;
  const int stage_bytes = W_TILE_BYTES + args.Mb * BLOCK_K * 2;
  SmemPtrs sp = carve_smem(smem, S, stage_bytes, args.red_bytes);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int C = args.C;
  const int rank = (int)blockIdx.x;          // K slice; equals the rank in the cluster (cluster spans x)
  const int u = (int)blockIdx.y;
  const int n_tile = u / args.n_tgroups, g = u % args.n_tgroups;
  const int m0 = g * args.Mb;
  const int mcount = min(args.Mb, args.M - m0);
  const int kb_lo = (int)((long long)rank * args.kblocks / C);
  const int kb_hi = (int)((long long)(rank + 1) * args.kblocks / C);

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(&sp.full[s], 1);
      mbar_init(&sp.empty[s], 1);
    }
    mbar_init(sp.tfull, 1);
    mbar_init(sp.drain, 1);
    *sp.abort_flag = 0;
    fence_mbar_init();
    grid_launch_dependents();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tmap_w);
    tma_prefetch_desc(&tmap_x);
  }
  if (warp == 1) {
    tmem_alloc(sp.tmem_slot, args.tmem_cols);
    tmem_relinquish();
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem_base = *sp.tmem_slot;
  volatile int *abort_flag = sp.abort_flag;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      const uint64_t pol_w = policy_evict_first();
      const uint64_t pol_x = policy_evict_last();
      const int nkb = kb_hi - kb_lo;
      // With static weights, the first ring of W tiles is requested before the
      // wait for the preceding kernel; x always comes after it.
      const int early = args.prefetch_w ? min(nkb, S) : 0;
      for (int i = 0; i < early; ++i) {
        mbar_arrive_expect_tx(&sp.full[i], (uint32_t)stage_bytes);
        tma_load_2d(sp.stage0 + (size_t)i * stage_bytes, &tmap_w, &sp.full[i], (kb_lo + i) * BLOCK_K,
                    n_tile * BLOCK_N, pol_w);
      }
      grid_dependency_wait();
      int stage = 0;
      uint32_t phase = 0;
      int issued = 0;
      for (int i = 0; i < nkb; ++i) {
        const int kb = kb_lo + i;
        uint8_t *st = sp.stage0 + (size_t)stage * stage_bytes;
        if (i >= early) {
          if (!mbar_wait_bounded(&sp.empty[stage], phase ^ 1u, abort_flag)) {
            signal_abort(sp, args.status);
            break;
          }
          mbar_arrive_expect_tx(&sp.full[stage], (uint32_t)stage_bytes);
          tma_load_2d(st, &tmap_w, &sp.full[stage], kb * BLOCK_K, n_tile * BLOCK_N, pol_w);
        }
        for (int s = 0; s < args.nsub; ++s)
          tma_load_2d(st + W_TILE_BYTES + (size_t)s * args.sub_n * BLOCK_K * 2, &tmap_x, &sp.full[stage],
                      kb * BLOCK_K, m0 + s * args.sub_n, pol_x);
        ++issued;
        if (++stage == S) {
          stage = 0;
          phase ^= 1u;
        }
      }
      if (*abort_flag) {
        // Let this CTA's own copies land before shared memory goes away.
        const int n = issued < S ? issued : S;
        for (int i = issued - n; i < issued; ++i) {
          volatile int never = 0;
          mbar_wait_bounded(&sp.full[i % S], (uint32_t)((i / S) & 1), &never);
        }
        if (early > issued) {
          for (int i = issued; i < early; ++i) {
            volatile int never = 0;
            mbar_wait_bounded(&sp.full[i], 0u, &never);  // W half only: never completes, bounded
          }
        }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      const uint32_t idesc = idesc_bf16_f32(BLOCK_N, args.sub_n);
      int stage = 0;
      uint32_t phase = 0;
      bool issued_any = false, ok = true;
      for (int kb = kb_lo; kb < kb_hi; ++kb) {
        if (!mbar_wait_bounded(&sp.full[stage], phase, abort_flag)) {
          signal_abort(sp, args.status);
          ok = false;
          break;
        }
        tc_fence_after_sync();
        const uint32_t a_addr = smem_addr(sp.stage0 + (size_t)stage * stage_bytes);
        const uint32_t b_addr = a_addr + W_TILE_BYTES;
#pragma unroll
        for (int kk = 0; kk < BLOCK_K / 16; ++kk) {
          const uint64_t adesc = smem_desc_kmajor_sw128(a_addr + kk * 32);
          for (int s = 0; s < args.nsub; ++s) {
            const uint64_t bdesc = smem_desc_kmajor_sw128(b_addr + s * args.sub_n * BLOCK_K * 2 + kk * 32);
            mma_bf16_ss(tmem_base + (uint32_t)(s * args.sub_n), adesc, bdesc, idesc,
                        (kb > kb_lo || kk > 0) ? 1u : 0u);
          }
        }
        issued_any = true;
        mma_commit(&sp.empty[stage]);
        if (++stage == S) {
          stage = 0;
          phase ^= 1u;
        }
      }
      if (ok) {
        mma_commit(sp.tfull);
      } else if (issued_any) {
        // Wait for this thread's MMAs before tensor memory is freed.
        mma_commit(sp.drain);
        volatile int never = 0;
        mbar_wait_bounded(sp.drain, 0, &never);
      }
    }
  }

  // ------------------------------------------------------------ epilogue
  // Warps 2..5 read tensor memory (warp w may touch lanes 32*(w%4)..+31);
  // all six warps take part in every cluster barrier.
  __syncwarp();
  const bool epi = warp >= 2;
  const int quad = warp & 3;
  const int et = threadIdx.x - 64;
  const PlanLayout L = plan_layout(args.M, args.n_ad);
  bool have_acc = false;
  if (epi) {
    have_acc = mbar_wait_bounded(sp.tfull, 0, abort_flag);
    if (!have_acc) signal_abort(sp, args.status);
    tc_fence_after_sync();
    grid_dependency_wait();  // the plan and T come from kernels earlier in the stream
  }
  const uint32_t taddr = tmem_base + ((uint32_t)(quad * 32) << 16);
  const int nchunks = (mcount + CHUNK - 1) / CHUNK;

  const bool verify = args.mode == MLORA_VERIFY;

  if (C == 1) {
    if (epi && have_acc) {
      const int n = n_tile * BLOCK_N + quad * 32 + lane;
      if (!verify) {
        for (int ch = 0; ch < nchunks; ++ch) {
          uint32_t r[32];
          tmem_ld_x32(taddr + ch * CHUNK, r);
          tmem_ld_wait();
          if (n < args.N) {
#pragma unroll
            for (int j = 0; j < CHUNK; ++j) {
              const int col = ch * CHUNK + j;
              if (col < mcount) args.y[(size_t)(m0 + col) * args.N + n] = float_to_bf16_bits(__uint_as_float(r[j]));
            }
          }
        }
      } else {
        // Walk the plan's buckets: one B row load per (adapter, output row),
        // accumulator columns fetched from tensor memory eight at a time.
        const int32_t *plan = args.plan;
        const int n_active = plan[L.hdr + 0];
        for (int ai = 0; ai <= n_active; ++ai) {
          const int b = (ai < n_active) ? plan[L.active + ai] : args.n_ad;
          const int s0 = plan[L.seg_offsets + b], s1 = plan[L.seg_offsets + b + 1];
          if (s0 == s1) continue;
          const int r = (b < args.n_ad) ? plan[L.rank_eff + b] : 0;
          uint32_t bp[32];
          load_brow(args, b, n, r, bp);
          for (int i = s0; i < s1; i += 8) {
            int mm[8];
            uint32_t own[8];
#pragma unroll
            for (int j = 0; j < 8; ++j) {
              mm[j] = (i + j < s1) ? plan[L.perm + i + j] : -1;
              own[j] = 0u;
              if (mm[j] >= m0 && mm[j] < m0 + mcount) tmem_ld_x1(taddr + (uint32_t)(mm[j] - m0), own[j]);
            }
            tmem_ld_wait();
#pragma unroll
            for (int j = 0; j < 8; ++j) {
              if (mm[j] < m0 || mm[j] >= m0 + mcount) continue;
              float v = __uint_as_float(own[j]);
              if (r > 0) v = fmaf(args.scale, lowrank_dot(args.T, mm[j], bp, r), v);
              if (n < args.N) args.y[(size_t)mm[j] * args.N + n] = float_to_bf16_bits(v);
            }
          }
        }
      }
    }
    tc_fence_before_sync();
    __syncthreads();
  } else {
    const int r0 = rank * BLOCK_N / C, r1 = (rank + 1) * BLOCK_N / C, R = r1 - r0;
    const uint32_t red_local = smem_addr(sp.red);
    // Verify mode keeps the reduced rows, column-major [Mb][R], in the stage
    // ring (free once the last MMA has completed) for the bucket walk below.
    float *fin = reinterpret_cast<float *>(sp.stage0);
    uint32_t peer[MAX_CLUSTER];
#pragma unroll
    for (int p = 0; p < MAX_CLUSTER; ++p) peer[p] = (p < C) ? map_to_rank(red_local, (uint32_t)p) : 0u;
    for (int ch = 0; ch < nchunks; ++ch) {
      const int buf = ch & 1;
      float *red = sp.red + buf * CHUNK * BLOCK_N;
      if (epi) {
        uint32_t r[32];
        if (have_acc) {
          tmem_ld_x32(taddr + ch * CHUNK, r);
          tmem_ld_wait();
        } else {
#pragma unroll
          for (int j = 0; j < 32; ++j) r[j] = 0u;
        }
#pragma unroll
        for (int j = 0; j < CHUNK; ++j) red[j * BLOCK_N + quad * 32 + lane] = __uint_as_float(r[j]);
      }
      cluster_sync_all();
      if (epi) {
        for (int e = et; e < R * CHUNK; e += 128) {
          const int i = e % R, c = e / R;
          const int col = ch * CHUNK + c;
          if (col >= mcount) continue;
          const uint32_t off = (uint32_t)((buf * CHUNK * BLOCK_N + c * BLOCK_N + r0 + i) * 4);
          float w[MAX_CLUSTER];
#pragma unroll
          for (int p = 0; p < MAX_CLUSTER; ++p)
            if (p < C) w[p] = ld_dsmem_f32(peer[p] + off);
          float v = w[0];
#pragma unroll
          for (int p = 1; p < MAX_CLUSTER; ++p)
            if (p < C) v += w[p];
          const int n = n_tile * BLOCK_N + r0 + i;
          if (verify) {
            fin[col * R + i] = v;
          } else if (n < args.N) {
            args.y[(size_t)(m0 + col) * args.N + n] = float_to_bf16_bits(v);
          }
        }
      }
    }
    if (verify && epi) {
      named_bar_sync(1, 128);
      // Threads split as (row i, column phase): 128 / R threads share a row.
      const int P = 128 / R;
      const int i = et % R, sub = et / R;
      const int n = n_tile * BLOCK_N + r0 + i;
      const int32_t *plan = args.plan;
      const int n_active = plan[L.hdr + 0];
      if (sub < P) {
        for (int ai = 0; ai <= n_active; ++ai) {
          const int b = (ai < n_active) ? plan[L.active + ai] : args.n_ad;
          const int s0 = plan[L.seg_offsets + b], s1 = plan[L.seg_offsets + b + 1];
          if (s0 == s1) continue;
          const int r = (b < args.n_ad) ? plan[L.rank_eff + b] : 0;
          uint32_t bp[32];
          load_brow(args, b, n, r, bp);
          for (int idx = s0 + sub; idx < s1; idx += P) {
            const int m = plan[L.perm + idx];
            if (m < m0 || m >= m0 + mcount) continue;
            float v = fin[(m - m0) * R + i];
            if (r > 0) v = fmaf(args.scale, lowrank_dot(args.T, m, bp, r), v);
            if (n < args.N) args.y[(size_t)m * args.N + n] = float_to_bf16_bits(v);
          }
        }
      }
    }
    tc_fence_before_sync();
    cluster_sync_all();  // no CTA leaves while a peer may still read its shared memory
  }
  if (warp == 1) {
    __syncwarp();
    tc_fence_after_sync();
    tmem_dealloc(tmem_base, args.tmem_cols);
  }
}

static int round_up_int(int v, int a) { return (v + a - 1) / a * a; }

static size_t smem_for(int Mb, int stages, int red_bytes) {
  return SMEM_FIXED + (size_t)stages * (W_TILE_BYTES + Mb * BLOCK_K * 2) + red_bytes;
}

static int stages_for(int Mb, int red_bytes) {
  const int stage_bytes = W_TILE_BYTES + Mb * BLOCK_K * 2;
  int s = (int)((SMEM_LIMIT - SMEM_FIXED - red_bytes) / stage_bytes);
  return s > 8 ? 8 : s;
}

// Clusters of size C that can be resident at once (one CTA per SM).
static int max_active_clusters(int C, size_t smem) {
  struct Entry {
    int dev, C;
    size_t smem;
    int n;
  };
  static Entry cache[64];
  static int ncache = 0;
  int dev = 0;
  cudaGetDevice(&dev);
  for (int i = 0; i < ncache; ++i)
    if (cache[i].dev == dev && cache[i].C == C && cache[i].smem == smem) return cache[i].n;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(C, MAX_CLUSTER, 1);
  cfg.blockDim = dim3(GEMM_THREADS, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = C;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, gemm_kernel, &cfg) != cudaSuccess) {
    cudaGetLastError();
    n = 0;
  }
  if (ncache < 64) cache[ncache++] = {dev, C, smem, n};
  return n;
}

static bool ensure_attributes() {
  static int done[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return false;
  if (dev < 64 && done[dev]) return true;
  if (cudaFuncSetAttribute(gemm_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)SMEM_LIMIT) != cudaSuccess)
    return false;
  if (cudaFuncSetAttribute(gemm_kernel, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) != cudaSuccess)
    return false;
  if (dev < 64) done[dev] = 1;
  return true;
}

GemmShape gemm_shape(int M, int N, int K, int num_sms) {
  GemmShape s;
  const int tg = (M + MAX_MB - 1) / MAX_MB;
  const int per = (M + tg - 1) / tg;
  int Mb = round_up_int(per, 16);
  int nsub = 1;
  if (Mb > 256) {
    Mb = round_up_int(per, 32);
    nsub = 2;
  }
  s.Mb = Mb;
  s.nsub = nsub;
  s.sub_n = Mb / nsub;
  s.n_tgroups = tg;
  s.n_units = ((N + BLOCK_N - 1) / BLOCK_N) * tg;
  s.kblocks = (K + BLOCK_K - 1) / BLOCK_K;
  int cols = 32;
  while (cols < Mb) cols <<= 1;
  s.tmem_cols = cols;
  s.nbuf = 1;
  s.total_iters = s.n_units * s.kblocks;
  // Split-K factor (a power of two, so each CTA owns 128 / C output rows):
  // minimise waves x (k-blocks per CTA + fixed cost), with a reduction cost
  // for C > 1; C = 1 needs no cluster.
  const bool attrs = ensure_attributes();
  int bestC = 1;
  double best = 1e30;
  for (int C = 1; C <= MAX_CLUSTER && C <= s.kblocks; C <<= 1) {  // powers of two: C divides 128 rows
    const int red = C > 1 ? RED_BYTES : 0;
    const int st = stages_for(Mb, red);
    if (st < 2) continue;
    int slots;
    if (C == 1) {
      slots = num_sms;
    } else {
      if (!attrs || num_sms <= 0) break;
      const int clusters = max_active_clusters(C, smem_for(Mb, st, red));
      if (clusters <= 0) continue;
      slots = clusters * C;
    }
    const long long ctas = (long long)s.n_units * C;
    const long long waves = (ctas + slots - 1) / slots;
    const double kper = (double)((s.kblocks + C - 1) / C);
    const double cost = (double)waves * (kper + 3.0 + (C > 1 ? 2.0 + 0.25 * C : 0.0));
    if (cost < best - 1e-9) {
      best = cost;
      bestC = C;
    }
  }
  s.C = bestC;
  s.red_bytes = bestC > 1 ? RED_BYTES : 0;
  s.stages = stages_for(Mb, s.red_bytes);
  s.grid = s.n_units * bestC;
  s.smem_bytes = smem_for(Mb, s.stages, s.red_bytes);
  s.partial_floats = 0;
  return s;
}

typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                   const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  if (!fn) {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  }
  return fn;
}

// Row-major bf16 matrix [rows, cols] read in boxes of box_rows x 64 with
// 128-byte swizzling; out-of-range elements read as zero.
static bool make_map(CUtensorMap *map, const void *base, int rows, int cols, int box_rows) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)cols * 2};
  cuuint32_t box[2] = {(cuuint32_t)BLOCK_K, (cuuint32_t)box_rows};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(base), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

cudaError_t launch_gemm(const GemmLaunch &g, const GemmShape &sh, cudaStream_t s, int *err_code) {
  *err_code = 0;
  CUtensorMap tw, tx;
  if (!make_map(&tw, g.W, g.N, g.K, BLOCK_N) || !make_map(&tx, g.x, g.M, g.K, sh.sub_n)) {
    *err_code = 1;
    return cudaErrorInvalidValue;
  }
  if (!ensure_attributes()) return cudaErrorInvalidValue;
  GemmArgs a;
  a.M = g.M;
  a.N = g.N;
  a.K = g.K;
  a.Mb = sh.Mb;
  a.nsub = sh.nsub;
  a.sub_n = sh.sub_n;
  a.n_tgroups = sh.n_tgroups;
  a.kblocks = sh.kblocks;
  a.C = sh.C;
  a.stages = sh.stages;
  a.tmem_cols = sh.tmem_cols;
  a.red_bytes = sh.red_bytes;
  a.mode = g.mode;
  a.prefetch_w = g.prefetch_w;
  a.scale = g.scale;
  a.y = g.y;
  a.B_stack = g.B_stack;
  a.r_max = g.r_max;
  a.n_ad = g.n_ad;
  a.T = g.T;
  a.plan = g.plan;
  a.status = g.status;

  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(sh.C, sh.n_units, 1);
  cfg.blockDim = dim3(GEMM_THREADS, 1, 1);
  cfg.dynamicSmemBytes = sh.smem_bytes;
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  int na = 0;
  attr[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[na].val.programmaticStreamSerializationAllowed = 1;
  ++na;
  if (sh.C > 1) {
    attr[na].id = cudaLaunchAttributeClusterDimension;
    attr[na].val.clusterDim.x = sh.C;
    attr[na].val.clusterDim.y = 1;
    attr[na].val.clusterDim.z = 1;
    ++na;
  }
  cfg.attrs = attr;
  cfg.numAttrs = na;
  cudaError_t e = cudaLaunchKernelEx(&cfg, gemm_kernel, tw, tx, a);
  note_launch();
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace mlora
