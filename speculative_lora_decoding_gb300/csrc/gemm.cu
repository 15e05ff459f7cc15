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
//    full while W streams through once.
//  * One CTA per SM, persistent over a linear (unit, k-block) iteration space
//    split evenly across the grid ("stream-K").  A unit is 128 W rows x up to
//    512 tokens.  Units shared by several CTAs are reduced by the last CTA to
//    arrive (an atomic counter per unit and epilogue warp, no spinning),
//    which sums the pieces in CTA order, so results are deterministic.
//  * Warp roles: warp 0 issues TMA loads of W and x tiles (128-byte swizzle)
//    into a ring of shared-memory stages; warp 1 owns tensor memory and issues
//    tcgen05.mma from one thread; warps 2..5 drain the fp32 accumulator from
//    tensor memory (tcgen05.ld) and run the epilogue.  Two accumulator buffers
//    when they fit let the next unit's MMAs overlap the epilogue.
//  * Every mbarrier wait is bounded; on expiry the CTA raises
//    MLORA_DEV_TIMEOUT, drains its own in-flight copies and MMAs, frees its
//    tensor memory and returns.
#include "common.cuh"
#include "launch.h"

namespace mlora {

constexpr int GEMM_THREADS = 192;
constexpr int BLOCK_N = 128;                          // W rows per unit (MMA M)
constexpr int BLOCK_K = 64;                           // K per stage: 128 bytes of bf16
constexpr int W_TILE_BYTES = BLOCK_N * BLOCK_K * 2;   // 16 KB
constexpr int MAX_MB = 512;
constexpr size_t SMEM_LIMIT = 227 * 1024;

struct GemmArgs {
  int M, N, K;
  int Mb, nsub, sub_n, n_tgroups, n_units, kblocks, total_iters, stages, nbuf, tmem_cols;
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

__device__ __forceinline__ long long iter_begin(int c, int G, long long total) { return (long long)c * total / G; }

// Largest CTA index whose range starts at or before iteration `it`.
__device__ __forceinline__ int cta_of_iter(long long it, int G, long long total) {
  return (int)(((it + 1) * (long long)G - 1) / total);
}

struct SmemPtrs {
  uint8_t *stage0;
  uint64_t *full, *empty, *tfull, *tempty, *drain;
  uint32_t *tmem_slot;
  int *abort_flag;
};

__device__ __forceinline__ SmemPtrs carve_smem(uint8_t *base, int stages, int stage_bytes) {
  SmemPtrs p;
  p.stage0 = base;
  uint64_t *bars = reinterpret_cast<uint64_t *>(base + (size_t)stages * stage_bytes);
  p.full = bars;
  p.empty = bars + stages;
  p.tfull = bars + 2 * stages;
  p.tempty = bars + 2 * stages + 2;
  p.drain = bars + 2 * stages + 4;
  uint32_t *w = reinterpret_cast<uint32_t *>(bars + 2 * stages + 5);
  p.tmem_slot = w;
  p.abort_flag = reinterpret_cast<int *>(w + 1);
  return p;
}

__device__ __forceinline__ void signal_abort(SmemPtrs &sp, uint32_t *status) {
  *reinterpret_cast<volatile int *>(sp.abort_flag) = 1;
  raise_status(status, MLORA_DEV_TIMEOUT);
}

// Unit pieces: value of (column col, row lane nl) of unit u summed over the
// CTAs that share it, in CTA order; `own` is this CTA's value.
struct PieceSum {
  const float *base;   // partials
  int Mb, c, c_lo, c_hi, u, kblocks, G;
  long long total;
  __device__ __forceinline__ const float *piece_ptr(int cc) const {
    const int first_unit = (int)(iter_begin(cc, G, total) / kblocks);
    const int slot = (u == first_unit) ? 0 : 1;
    return base + ((size_t)(cc * 2 + slot) * Mb) * BLOCK_N;
  }
};

__device__ __forceinline__ void unpack_bf16x2(uint32_t w, float &lo, float &hi) {
  lo = __uint_as_float(w << 16);
  hi = __uint_as_float(w & 0xFFFF0000u);
}

__global__ void __launch_bounds__(GEMM_THREADS, 1)
    gemm_kernel(const __grid_constant__ CUtensorMap tmap_w, const __grid_constant__ CUtensorMap tmap_x,
                const GemmArgs args) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
  const int S = args.stages;
  const int stage_bytes = W_TILE_BYTES + args.Mb * BLOCK_K * 2;
  SmemPtrs sp = carve_smem(smem, S, stage_bytes);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int G = gridDim.x, c = blockIdx.x;
  const long long total = args.total_iters;
  const long long it_begin = iter_begin(c, G, total), it_end = iter_begin(c + 1, G, total);
  const int kblocks = args.kblocks;

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(&sp.full[s], 1);
      mbar_init(&sp.empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&sp.tfull[b], 1);
      mbar_init(&sp.tempty[b], 4);
    }
    mbar_init(sp.drain, 1);
    *sp.abort_flag = 0;
    fence_mbar_init();
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
      const uint32_t tx_bytes = (uint32_t)stage_bytes;
      int stage = 0;
      uint32_t phase = 0;
      long long issued = 0;
      for (long long it = it_begin; it < it_end; ++it) {
        const int u = (int)(it / kblocks), kb = (int)(it % kblocks);
        const int n_tile = u / args.n_tgroups, g = u % args.n_tgroups;
        if (!mbar_wait_bounded(&sp.empty[stage], phase ^ 1u, abort_flag)) {
          signal_abort(sp, args.status);
          break;
        }
        mbar_arrive_expect_tx(&sp.full[stage], tx_bytes);
        uint8_t *st = sp.stage0 + (size_t)stage * stage_bytes;
        tma_load_2d(st, &tmap_w, &sp.full[stage], kb * BLOCK_K, n_tile * BLOCK_N, pol_w);
        for (int s = 0; s < args.nsub; ++s)
          tma_load_2d(st + W_TILE_BYTES + (size_t)s * args.sub_n * BLOCK_K * 2, &tmap_x, &sp.full[stage],
                      kb * BLOCK_K, g * args.Mb + s * args.sub_n, pol_x);
        ++issued;
        if (++stage == S) {
          stage = 0;
          phase ^= 1u;
        }
      }
      if (*abort_flag) {
        // Let this CTA's own copies land before shared memory goes away.
        const long long n = issued < S ? issued : S;
        for (long long i = issued - n; i < issued; ++i) {
          const int st = (int)(i % S);
          const uint32_t ph = (uint32_t)((i / S) & 1);
          volatile int never = 0;
          mbar_wait_bounded(&sp.full[st], ph, &never);
        }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      const uint32_t idesc = idesc_bf16_f32(BLOCK_N, args.sub_n);
      int stage = 0;
      uint32_t phase = 0;
      int seg = 0;
      bool issued_any = false;
      long long it = it_begin;
      while (it < it_end && !*abort_flag) {
        const int u = (int)(it / kblocks);
        const int kb0 = (int)(it % kblocks);
        const int kb1 = (int)min((long long)kblocks, kb0 + (it_end - it));
        const int buf = seg % args.nbuf, use = seg / args.nbuf;
        (void)u;
        if (!mbar_wait_bounded(&sp.tempty[buf], (uint32_t)(use & 1) ^ 1u, abort_flag)) {
          signal_abort(sp, args.status);
          break;
        }
        tc_fence_after_sync();
        const uint32_t d_base = tmem_base + (uint32_t)(buf * args.Mb);
        bool ok = true;
        for (int kb = kb0; kb < kb1; ++kb) {
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
              mma_bf16_ss(d_base + (uint32_t)(s * args.sub_n), adesc, bdesc, idesc, (kb > kb0 || kk > 0) ? 1u : 0u);
            }
          }
          issued_any = true;
          mma_commit(&sp.empty[stage]);
          if (++stage == S) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        mma_commit(&sp.tfull[buf]);
        it += kb1 - kb0;
        ++seg;
      }
      if (*abort_flag && issued_any) {
        // Wait for this thread's MMAs before tensor memory is freed.
        mma_commit(sp.drain);
        volatile int never = 0;
        mbar_wait_bounded(sp.drain, 0, &never);
      }
    }
  } else {
    // ------------------------------------------------------------ epilogue
    const int quad = warp & 3;               // tensor-memory lane quadrant this warp may read
    const int nl = quad * 32 + lane;         // W row within the unit
    const PlanLayout L = plan_layout(args.M, args.n_ad);
    const bool verify = args.mode == MLORA_VERIFY;
    int seg = 0;
    long long it = it_begin;
    while (it < it_end) {
      const int u = (int)(it / kblocks);
      const int kb0 = (int)(it % kblocks);
      const int kb1 = (int)min((long long)kblocks, kb0 + (it_end - it));
      const int buf = seg % args.nbuf, use = seg / args.nbuf;
      if (!mbar_wait_bounded(&sp.tfull[buf], (uint32_t)(use & 1), abort_flag)) {
        signal_abort(sp, args.status);
        break;
      }
      tc_fence_after_sync();
      const int n_tile = u / args.n_tgroups, g = u % args.n_tgroups;
      const int n = n_tile * BLOCK_N + nl;
      const int m0 = g * args.Mb;
      const int mcount = min(args.Mb, args.M - m0);
      const uint32_t taddr = tmem_base + ((uint32_t)(quad * 32) << 16) + (uint32_t)(buf * args.Mb);
      const bool split = !(kb0 == 0 && kb1 == kblocks);

      PieceSum ps;
      ps.base = args.partials;
      ps.Mb = args.Mb;
      ps.c = c;
      ps.u = u;
      ps.kblocks = kblocks;
      ps.G = G;
      ps.total = total;
      ps.c_lo = cta_of_iter((long long)u * kblocks, G, total);
      ps.c_hi = cta_of_iter((long long)u * kblocks + kblocks - 1, G, total);

      bool final_here = true;
      if (split) {
        // Publish this CTA's piece, then count arrivals.
        float *mine = const_cast<float *>(ps.piece_ptr(c));
        for (int col = 0; col < mcount; col += 16) {
          uint32_t r[16];
          tmem_ld_x16(taddr + col, r);
          tmem_ld_wait();
#pragma unroll
          for (int j = 0; j < 16; ++j) mine[(size_t)(col + j) * BLOCK_N + nl] = __uint_as_float(r[j]);
        }
        // Each epilogue warp counts its own 32 rows, so no CTA-wide barrier is needed.
        __threadfence();
        __syncwarp();
        uint32_t *ctr = &args.counters[(size_t)u * 4 + quad];
        int old = 0;
        if (lane == 0) old = (int)atomicAdd(ctr, 1u);
        old = __shfl_sync(0xffffffffu, old, 0);
        final_here = (old == ps.c_hi - ps.c_lo);
        if (final_here) {
          __threadfence();
          if (lane == 0) *ctr = 0u;
        }
      }

      if (final_here) {
        if (!verify) {
          for (int col = 0; col < mcount; col += 16) {
            uint32_t r[16];
            tmem_ld_x16(taddr + col, r);
            tmem_ld_wait();
            float v[16];
            if (!split) {
#pragma unroll
              for (int j = 0; j < 16; ++j) v[j] = __uint_as_float(r[j]);
            } else {
              for (int cc = ps.c_lo; cc <= ps.c_hi; ++cc) {
                float w[16];
                if (cc == c) {
#pragma unroll
                  for (int j = 0; j < 16; ++j) w[j] = __uint_as_float(r[j]);
                } else {
                  const float *pp = ps.piece_ptr(cc) + (size_t)col * BLOCK_N + nl;
#pragma unroll
                  for (int j = 0; j < 16; ++j) w[j] = __ldcg(pp + (size_t)j * BLOCK_N);
                }
                if (cc == ps.c_lo) {
#pragma unroll
                  for (int j = 0; j < 16; ++j) v[j] = w[j];
                } else {
#pragma unroll
                  for (int j = 0; j < 16; ++j) v[j] += w[j];
                }
              }
            }
            if (n < args.N) {
#pragma unroll
              for (int j = 0; j < 16; ++j)
                if (col + j < mcount) args.y[(size_t)(m0 + col + j) * args.N + n] = float_to_bf16_bits(v[j]);
            }
          }
        } else {
          // Verify: walk the plan's buckets so each adapter's B row stays in registers.
          const int32_t *plan = args.plan;
          const int n_active = plan[L.hdr + 0];
          for (int ai = 0; ai <= n_active; ++ai) {
            const int b = (ai < n_active) ? plan[L.active + ai] : args.n_ad;
            const int s0 = plan[L.seg_offsets + b], s1 = plan[L.seg_offsets + b + 1];
            if (s0 == s1) continue;
            const int r = (b < args.n_ad) ? plan[L.rank_eff + b] : 0;
            uint32_t bp[32];
#pragma unroll
            for (int i = 0; i < 32; ++i) bp[i] = 0u;
            if (r > 0 && n < args.N) {
              const uint16_t *brow = args.B_stack + ((size_t)b * args.N + n) * args.r_max;
#pragma unroll
              for (int q = 0; q < 8; ++q) {
                if (q * 8 < r) {
                  const uint4 v = __ldg(reinterpret_cast<const uint4 *>(brow) + q);
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
            for (int i = s0; i < s1; i += 4) {
              int mm[4];
              bool ok[4];
              uint32_t own[4];
#pragma unroll
              for (int j = 0; j < 4; ++j) {
                mm[j] = (i + j < s1) ? plan[L.perm + i + j] : -1;
                ok[j] = mm[j] >= m0 && mm[j] < m0 + mcount;
                own[j] = 0u;
                if (ok[j]) tmem_ld_x1(taddr + (uint32_t)(mm[j] - m0), own[j]);
              }
              tmem_ld_wait();
#pragma unroll
              for (int j = 0; j < 4; ++j) {
                if (!ok[j]) continue;
                const int col = mm[j] - m0;
                float v;
                if (!split) {
                  v = __uint_as_float(own[j]);
                } else {
                  v = 0.f;
                  for (int cc = ps.c_lo; cc <= ps.c_hi; ++cc) {
                    const float w = (cc == c) ? __uint_as_float(own[j])
                                              : __ldcg(ps.piece_ptr(cc) + (size_t)col * BLOCK_N + nl);
                    v = (cc == ps.c_lo) ? w : v + w;
                  }
                }
                if (r > 0) {
                  const float4 *trow = reinterpret_cast<const float4 *>(args.T + (size_t)mm[j] * T_STRIDE);
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
                  v = fmaf(args.scale, dot, v);
                }
                if (n < args.N) args.y[(size_t)mm[j] * args.N + n] = float_to_bf16_bits(v);
              }
            }
          }
        }
      }
      // Hand the accumulator buffer back to the MMA warp.
      tc_fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(&sp.tempty[buf]);
      it += kb1 - kb0;
      ++seg;
    }
  }

  tc_fence_before_sync();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after_sync();
    tmem_dealloc(tmem_base, args.tmem_cols);
  }
}

static int round_up_int(int v, int a) { return (v + a - 1) / a * a; }

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
  s.total_iters = s.n_units * s.kblocks;
  const int stage_bytes = W_TILE_BYTES + Mb * BLOCK_K * 2;
  const size_t fixed = 1024 + 256;
  int stages = (int)((SMEM_LIMIT - fixed) / stage_bytes);
  stages = stages > 8 ? 8 : stages;
  s.stages = stages;
  s.nbuf = (2 * Mb <= 512) ? 2 : 1;
  int cols = 32;
  while (cols < s.nbuf * Mb) cols <<= 1;
  s.tmem_cols = cols;
  const long long want = ((long long)s.total_iters + 3) / 4;
  s.grid = (int)(want < num_sms ? want : num_sms);
  if (s.grid < 1) s.grid = 1;
  s.smem_bytes = fixed + (size_t)stages * stage_bytes;
  s.partial_floats = (size_t)num_sms * 2 * Mb * BLOCK_N;
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
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  static int attr_done[64] = {0};
  if (dev < 64 && !attr_done[dev]) {
    e = cudaFuncSetAttribute(gemm_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)SMEM_LIMIT);
    if (e != cudaSuccess) return e;
    attr_done[dev] = 1;
  }
  GemmArgs a;
  a.M = g.M;
  a.N = g.N;
  a.K = g.K;
  a.Mb = sh.Mb;
  a.nsub = sh.nsub;
  a.sub_n = sh.sub_n;
  a.n_tgroups = sh.n_tgroups;
  a.n_units = sh.n_units;
  a.kblocks = sh.kblocks;
  a.total_iters = sh.total_iters;
  a.stages = sh.stages;
  a.nbuf = sh.nbuf;
  a.tmem_cols = sh.tmem_cols;
  a.mode = g.mode;
  a.scale = g.scale;
  a.y = g.y;
  a.B_stack = g.B_stack;
  a.r_max = g.r_max;
  a.n_ad = g.n_ad;
  a.T = g.T;
  a.plan = g.plan;
  a.partials = g.partials;
  a.counters = g.counters;
  a.status = g.status;
  gemm_kernel<<<sh.grid, GEMM_THREADS, sh.smem_bytes, s>>>(tw, tx, a);
  note_launch();
  return cudaGetLastError();
}

}  // namespace mlora
