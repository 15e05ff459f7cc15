// Steps a3 + a4, cluster split-K kernel: the base GEMM acc = x W^T on the
// tcgen05 tensor cores plus the low-rank expand:
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
//    memory: each CTA sums rows [rank*128/C, (rank+1)*128/C) over all C CTAs
//    in rank order.  The reduction stays on chip, runs on all C CTAs at once
//    and is deterministic.
//  * The verify expand (expand.cuh): the token rows come in adapter-sorted
//    order (x_sorted), so each adapter's rows are adjacent accumulator
//    columns; after the K loop one MMA per (adapter, 16-rank block) adds
//    B_a[n0:n0+128, block] x Twin^T over the adapter's token window only,
//    the blocks shared out over the cluster's CTAs, and the epilogue stores
//    column c to row perm[c].  Without the sorted rows (the allocation-free
//    entry point) the epilogue walks the plan's adapter buckets on the CUDA
//    cores instead.
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
#include "expand.cuh"
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
constexpr size_t SMEM_LIMIT = 220 * 1024;             // leaves room for a co-resident shrink CTA
constexpr int MAX_STAGES = 8;
constexpr size_t SMEM_FIXED = 1024 + 256 + expand_smem_bytes(MAX_STAGES);  // alignment slack, barriers, expand records

struct GemmArgs {
  int M, N, K;
  int Mb, nsub, sub_n, n_tgroups, kblocks, C, stages, tmem_cols, red_bytes;
  int mode, prefetch_w;
  int after_shrink;  // launched right after this library's shrink kernel: x and W are ready
  int sorted;        // verify mode with x in adapter-sorted order and the token windows (tensor-core expand)
  int n_slices;      // output slices: tile rows [slice_end[s-1], slice_end[s]) use T and windows of slice s
  int slice_end[MLORA_MAX_SLICES];
  size_t tw_slice;   // bf16 elements of one slice's window buffer
  float scale;
  uint16_t *y;
  const uint16_t *B_stack;
  const uint16_t *tw;  // token windows of the expand blocks, rows in the 32-byte-swizzled order
  int r_max, n_ad;
  const float *T;  // [n_slices][M][T_STRIDE]
  const int32_t *plan;
  uint32_t *status;
};

// Output slice of the tile starting at W row n0 (slice boundaries are
// multiples of the tile height, so a tile never straddles two).
__device__ __forceinline__ int slice_of(const GemmArgs &a, int n0) {
  int s = 0;
#pragma unroll
  for (int i = 0; i + 1 < MLORA_MAX_SLICES; ++i)
    if (i + 1 < a.n_slices && n0 >= a.slice_end[i]) s = i + 1;
  return s;
}

struct SmemPtrs {
  uint8_t *stage0;
  float *red;
  ExpandStage *meta;  // [stages] what an expand stage holds
  int4 *chunk;        // [EXP_CHUNK] the producer's staged plan records
  uint64_t *full, *empty, *tfull, *drain;
  uint32_t *tmem_slot;
  int *abort_flag;
  int *acc_ready;
  int *zero_word;  // stays 0: for waits that only a time limit may end
};

__device__ __forceinline__ SmemPtrs carve_smem(uint8_t *base, int stages, int stage_bytes, int red_bytes) {
  SmemPtrs p;
  p.stage0 = base;
  p.red = reinterpret_cast<float *>(base + (size_t)stages * stage_bytes);
  uint8_t *after = base + (size_t)stages * stage_bytes + red_bytes;
  p.meta = reinterpret_cast<ExpandStage *>(after);
  p.chunk = reinterpret_cast<int4 *>(after + (size_t)stages * sizeof(ExpandStage));
  uint64_t *bars = reinterpret_cast<uint64_t *>(after + expand_smem_bytes(stages));
  p.full = bars;
  p.empty = bars + stages;
  p.tfull = bars + 2 * stages;
  p.drain = bars + 2 * stages + 1;
  uint32_t *w = reinterpret_cast<uint32_t *>(bars + 2 * stages + 2);
  p.tmem_slot = w;
  p.abort_flag = reinterpret_cast<int *>(w + 1);
  p.acc_ready = reinterpret_cast<int *>(w + 2);
  p.zero_word = reinterpret_cast<int *>(w + 3);
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

// Accumulator columns [taddr, taddr + 32) of this warp's 32 lanes.
__device__ __forceinline__ void tmem_ld_acc_x32(uint32_t taddr, uint32_t (&r)[32]) {
  tmem_ld_x32(taddr, r);
  tmem_ld_wait();
}

// Tables the verify epilogue reads for every output: the plan's buckets
// (adapter, first and last sorted position, rank), its permutation and the
// rows of T.  Staged into shared memory (the freed stage ring) when the unit
// holds every token row and they fit; otherwise read from global memory.
struct VerifyTables {
  const int4 *bk;       // staged buckets, or nullptr
  const int32_t *perm;  // permutation
  const float *T;       // T rows: row m at T + (m - t_row0) * t_stride
  int t_row0, t_stride, nbk;
  size_t bytes;         // shared memory the staged tables occupy (0: not staged)
};

__device__ __forceinline__ VerifyTables stage_verify_tables(const GemmArgs &a, const PlanLayout &L, const float *Tu,
                                                            uint8_t *base, size_t avail, int m0, int mcount, int et) {
  const int32_t *plan = a.plan;
  const int n_active = plan[L.hdr + 0];
  const int rmax = plan[L.hdr + 3];
  const int rs = max(8, (rmax + 7) & ~7);
  VerifyTables v;
  v.bk = nullptr;
  v.perm = plan + L.perm;
  v.T = Tu;
  v.t_row0 = 0;
  v.t_stride = T_STRIDE;
  v.nbk = n_active + 1;
  v.bytes = 0;
  const size_t t_bytes = align_up((size_t)mcount * rs * 4, 16);
  const size_t p_bytes = align_up((size_t)a.M * 4, 16);
  const size_t need = t_bytes + p_bytes + (size_t)(n_active + 1) * 16;
  if (!(m0 == 0 && mcount == a.M) || need > avail) return v;
  float *sT = reinterpret_cast<float *>(base);
  int32_t *sp = reinterpret_cast<int32_t *>(base + t_bytes);
  int4 *sb = reinterpret_cast<int4 *>(base + t_bytes + p_bytes);
  // Four loads in flight per thread before their stores.
  const int nt = mcount * rs;
#pragma unroll 1
  for (int e0 = et; e0 < nt; e0 += 4 * 128) {
    float v[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const int e = e0 + k * 128;
      v[k] = e < nt ? Tu[(size_t)(m0 + e / rs) * T_STRIDE + e % rs] : 0.f;
    }
#pragma unroll
    for (int k = 0; k < 4; ++k)
      if (e0 + k * 128 < nt) sT[e0 + k * 128] = v[k];
  }
#pragma unroll 4
  for (int e = et; e < a.M; e += 128) sp[e] = plan[L.perm + e];
  for (int i = et; i <= n_active; i += 128) {
    const int b = (i < n_active) ? plan[L.active + i] : a.n_ad;
    const int r = (b < a.n_ad) ? plan[L.rank_eff + b] : 0;
    sb[i] = make_int4(b, plan[L.seg_offsets + b], plan[L.seg_offsets + b + 1], r);
  }
  named_bar_sync(1, 128);
  v.bk = sb;
  v.perm = sp;
  v.T = sT;
  v.t_row0 = m0;
  v.t_stride = rs;
  v.bytes = align_up(need, 16);
  return v;
}

__device__ __forceinline__ int4 bucket_at(const GemmArgs &a, const PlanLayout &L, const VerifyTables &v, int i) {
  if (v.bk) return v.bk[i];
  const int32_t *plan = a.plan;
  const int n_active = v.nbk - 1;
  const int b = (i < n_active) ? plan[L.active + i] : a.n_ad;
  const int r = (b < a.n_ad) ? plan[L.rank_eff + b] : 0;
  return make_int4(b, plan[L.seg_offsets + b], plan[L.seg_offsets + b + 1], r);
}

// The verify bucket walk.  Each thread owns one output row n and, for a group
// of buckets (adapter a, sorted positions [s0, s1), rank r), stages its masked
// rows B_a[n, 0:r] into shared memory (one 16-byte slot per 8 ranks,
// transposed so that lanes touch consecutive slots) in one round of loads,
// then finishes its share of each bucket's columns four at a time:
//   y[m, n] = bf16(acc[m, n] + scale * sum_{j<r} T[m, j] * B_a[n, j]).
// The value acc comes from tensor memory or, after a cluster reduction, from
// shared memory (fin, column-major [Mb][R]).
// The loops over rank chunks stay rolled to keep the code small.
template <bool FROM_TMEM>
__device__ __forceinline__ void verify_walk(const GemmArgs &a, const PlanLayout &L, const VerifyTables &vt, uint4 *Bs,
                                            int slot_cap, int et, int n, int m0, int mcount, int first, int step,
                                            uint32_t taddr, const float *fin, int R, int i_row) {
  int ai = 0;
  while (ai < vt.nbk) {
    // A group of buckets whose B rows fit the slots: stage them all in one
    // round of independent loads, then finish the group's columns.
    int aj = ai, used = 0;
    while (aj < vt.nbk) {
      const int nq = (bucket_at(a, L, vt, aj).w + 7) >> 3;
      if (aj > ai && used + nq > slot_cap) break;
      used += nq;
      ++aj;
    }
    // Staging walks the group's slots (bucket by bucket, 8 ranks per slot)
    // with a cursor, eight slots per batch: the batch's loads are all issued
    // before any of them is stored.
    {
      int cb = ai, cq = 0;
      int4 cbk = bucket_at(a, L, vt, cb);
#pragma unroll 1
      for (int base = 0; base < used; base += 8) {
        uint4 v[8];
        int qq[8], rr[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          v[k] = make_uint4(0u, 0u, 0u, 0u);
          qq[k] = 0;
          rr[k] = 0;
          if (base + k < used) {
            while (cq >= ((cbk.w + 7) >> 3)) {
              ++cb;
              cbk = bucket_at(a, L, vt, cb);
              cq = 0;
            }
            if (n < a.N && cbk.y < cbk.z)
              v[k] = __ldg(reinterpret_cast<const uint4 *>(a.B_stack + ((size_t)cbk.x * a.N + n) * a.r_max) + cq);
            qq[k] = cq;
            rr[k] = cbk.w;
            ++cq;
          }
        }
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          if (base + k < used) {
            uint32_t w[4] = {v[k].x, v[k].y, v[k].z, v[k].w};
            if (qq[k] * 8 + 8 > rr[k]) {
#pragma unroll
              for (int e = 0; e < 4; ++e) {
                if (qq[k] * 8 + 2 * e >= rr[k]) w[e] &= 0xFFFF0000u;
                if (qq[k] * 8 + 2 * e + 1 >= rr[k]) w[e] &= 0x0000FFFFu;
              }
            }
            Bs[(base + k) * 128 + et] = make_uint4(w[0], w[1], w[2], w[3]);
          }
        }
      }
    }
    int slot = 0;
#pragma unroll 1
    for (int b = ai; b < aj; ++b) {
      const int4 bk = bucket_at(a, L, vt, b);
      const int s0 = bk.y, s1 = bk.z, r = bk.w, nq = (r + 7) >> 3;
      const uint4 *bs = Bs + (size_t)slot * 128 + et;
      slot += nq;
#pragma unroll 1
      for (int i = s0 + first; i < s1; i += 4 * step) {
        int mm[4];
        float val[4];
#pragma unroll
        for (int jj = 0; jj < 4; ++jj) {
          const int idx = i + jj * step;
          int m = idx < s1 ? vt.perm[idx] : -1;
          if (m < m0 || m >= m0 + mcount) m = -1;
          mm[jj] = m;
          val[jj] = 0.f;
        }
        if (FROM_TMEM) {
          uint32_t own[4];
#pragma unroll
          for (int jj = 0; jj < 4; ++jj) {
            own[jj] = 0u;
            if (mm[jj] >= 0) tmem_ld_x1(taddr + (uint32_t)(mm[jj] - m0), own[jj]);
          }
          tmem_ld_wait();
#pragma unroll
          for (int jj = 0; jj < 4; ++jj) val[jj] = __uint_as_float(own[jj]);
        } else {
#pragma unroll
          for (int jj = 0; jj < 4; ++jj)
            if (mm[jj] >= 0) val[jj] = fin[(mm[jj] - m0) * R + i_row];
        }
        if (r > 0) {
          float dot[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll 1
          for (int q = 0; q < nq; ++q) {
            const uint4 bv = bs[q * 128];
            float b0, b1, b2, b3, b4, b5, b6, b7;
            unpack_bf16x2(bv.x, b0, b1);
            unpack_bf16x2(bv.y, b2, b3);
            unpack_bf16x2(bv.z, b4, b5);
            unpack_bf16x2(bv.w, b6, b7);
#pragma unroll
            for (int jj = 0; jj < 4; ++jj) {
              if (mm[jj] >= 0) {
                const float4 *trow =
                    reinterpret_cast<const float4 *>(vt.T + (size_t)(mm[jj] - vt.t_row0) * vt.t_stride) + 2 * q;
                const float4 t0 = trow[0], t1 = trow[1];
                float d = dot[jj];
                d = fmaf(t0.x, b0, d);
                d = fmaf(t0.y, b1, d);
                d = fmaf(t0.z, b2, d);
                d = fmaf(t0.w, b3, d);
                d = fmaf(t1.x, b4, d);
                d = fmaf(t1.y, b5, d);
                d = fmaf(t1.z, b6, d);
                d = fmaf(t1.w, b7, d);
                dot[jj] = d;
              }
            }
          }
#pragma unroll
          for (int jj = 0; jj < 4; ++jj) val[jj] = fmaf(a.scale, dot[jj], val[jj]);
        }
        if (n < a.N) {
#pragma unroll
          for (int jj = 0; jj < 4; ++jj)
            if (mm[jj] >= 0) a.y[(size_t)mm[jj] * a.N + n] = float_to_bf16_bits(val[jj]);
        }
      }
    }
    ai = aj;
  }
}

// Expand blocks of the tensor-core expand (verify mode with sorted rows), or
// -1 when the epilogue's bucket walk adds the low-rank term instead.
__device__ __forceinline__ int expand_blocks(const GemmArgs &a, const PlanLayout &L) {
  if (!a.sorted || a.mode != MLORA_VERIFY) return -1;
  return a.plan[L.hdr + 4];
}

// Split-K reduction through distributed shared memory: sums rows [r0, r0 + R)
// of columns [0, ncols) over the C_ peers' fp32 tiles laid out [column][128]
// at cluster addresses peer[p] (+ base), four rows per 16-byte load, eight
// loads in flight per thread (two rounds of DSMEM latency for C_ = 4 and 64
// columns).  Peers are added in rank order.  out(c, i, v) receives rows
// r0 + i .. r0 + i + 3 of column c.
template <int C_, class Out>
__device__ __forceinline__ void cluster_reduce_rows(const uint32_t *peer, uint32_t base, int r0, int R, int ncols,
                                                    int et, Out &&out) {
  constexpr int PG = C_ < 8 ? C_ : 8;  // peers per group of loads
  constexpr int NV = 8 / PG;           // units per round
  const int R4 = R / 4, total = ncols * R4;
#pragma unroll 1
  for (int e0 = et; e0 < total; e0 += 128 * NV) {
    float4 t[NV];
#pragma unroll
    for (int g0 = 0; g0 < C_; g0 += PG) {
      float4 w[NV][PG];
#pragma unroll
      for (int v = 0; v < NV; ++v) {
        const int e = e0 + v * 128;
        if (e < total) {
          const int c = e / R4, i4 = e - c * R4;
          const uint32_t off = base + (uint32_t)((c * BLOCK_N + r0 + 4 * i4) * 4);
#pragma unroll
          for (int p = 0; p < PG; ++p) w[v][p] = ld_dsmem_f32x4(peer[g0 + p] + off);
        }
      }
#pragma unroll
      for (int v = 0; v < NV; ++v) {
#pragma unroll
        for (int p = 0; p < PG; ++p) {
          if (g0 + p == 0) {
            t[v] = w[v][0];
          } else {
            t[v].x += w[v][p].x;
            t[v].y += w[v][p].y;
            t[v].z += w[v][p].z;
            t[v].w += w[v][p].w;
          }
        }
      }
    }
#pragma unroll
    for (int v = 0; v < NV; ++v) {
      const int e = e0 + v * 128;
      if (e < total) {
        const int c = e / R4;
        out(c, 4 * (e - c * R4), t[v]);
      }
    }
  }
}

template <class Out>
__device__ __forceinline__ void cluster_reduce_rows_c(int C, const uint32_t *peer, uint32_t base, int r0, int R,
                                                      int ncols, int et, Out &&out) {
  switch (C) {
    case 2: cluster_reduce_rows<2>(peer, base, r0, R, ncols, et, out); break;
    case 4: cluster_reduce_rows<4>(peer, base, r0, R, ncols, et, out); break;
    case 8: cluster_reduce_rows<8>(peer, base, r0, R, ncols, et, out); break;
    default: cluster_reduce_rows<16>(peer, base, r0, R, ncols, et, out); break;
  }
}

constexpr int Y_ROW = 40;  // bf16 per token row of an epilogue warp's y staging (32 + pad: no bank conflicts)

// Four bf16 outputs y[row, n .. n + 3] (columns past N dropped).
__device__ __forceinline__ void store_bf16x4(uint16_t *y, int N, size_t row, int n, float4 v) {
  uint16_t *dst = y + row * (size_t)N + n;
  if ((N & 3) == 0 && n + 3 < N) {
    const uint32_t lo = (uint32_t)float_to_bf16_bits(v.x) | ((uint32_t)float_to_bf16_bits(v.y) << 16);
    const uint32_t hi = (uint32_t)float_to_bf16_bits(v.z) | ((uint32_t)float_to_bf16_bits(v.w) << 16);
    *reinterpret_cast<uint2 *>(dst) = make_uint2(lo, hi);
  } else {
    const float f[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int j = 0; j < 4; ++j)
      if (n + j < N) dst[j] = float_to_bf16_bits(f[j]);
  }
}

// Shared memory allows one CTA per SM; the second block in the bounds caps
// registers (at 170) so that a shrink CTA still fits beside this one.
__global__ void __launch_bounds__(GEMM_THREADS, 2)
    gemm_kernel(const __grid_constant__ CUtensorMap tmap_w, const __grid_constant__ CUtensorMap tmap_x,
                const __grid_constant__ CUtensorMap tmap_b, const GemmArgs args) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = align_smem_1024(smem_raw);
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
  const int slice = slice_of(args, n_tile * BLOCK_N);
  const float *T_u = args.T + (size_t)slice * args.M * T_STRIDE;  // this tile's T

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(&sp.full[s], 1);
      mbar_init(&sp.empty[s], 1);
    }
    mbar_init(sp.tfull, 1);
    mbar_init(sp.drain, 1);
    *sp.abort_flag = 0;
    *sp.zero_word = 0;
    fence_mbar_init();
    grid_launch_dependents();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tmap_w);
    tma_prefetch_desc(&tmap_x);
    if (args.sorted) tma_prefetch_desc(&tmap_b);
  }
  if (warp == 1) {
    tmem_alloc(sp.tmem_slot, args.tmem_cols);
    tmem_relinquish();
  }
  tc_fence_before_sync();
  block_sync();
  tc_fence_after_sync();
  const uint32_t tmem_base = *sp.tmem_slot;
  volatile int *abort_flag = sp.abort_flag;

  // Expand blocks of this CTA, read from the plan after griddepcontrol.wait:
  // the cluster's CTAs share them out (the reduction adds every CTA's
  // accumulator, so any CTA may add any block), CTA `rank` taking blocks
  // [rank*ns/C, (rank+1)*ns/C).
  const PlanLayout L = plan_layout(args.M, args.n_ad);
  const bool sorted_verify = args.sorted && args.mode == MLORA_VERIFY;
  auto expand_range = [&](int &blo, int &bhi) {
    const int ns = expand_blocks(args, L);
    blo = ns > 0 ? (int)((long long)rank * ns / C) : 0;
    bhi = ns > 0 ? (int)((long long)(rank + 1) * ns / C) : 0;
  };

  // k-blocks before the expand: verify mode puts the expand's operand loads
  // into the ring before the last S k-blocks, so that they land while those
  // stream (the expand MMAs then add into the accumulator before the last
  // k-blocks do; the order of additions into it is free).  Not when the first
  // ring of W was requested early (those stages are already taken).
  const int nkb = kb_hi - kb_lo;
  const int early_n = (args.prefetch_w && !args.after_shrink) ? min(nkb, S) : 0;
  const int split = (sorted_verify && early_n == 0) ? max(1, nkb - S) : nkb;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    int stage = 0, issued = 0;
    uint32_t phase = 0;
    bool ok = true;
    const int early = early_n;
    const uint64_t pol_w = policy_evict_first();
    const uint64_t pol_x = policy_evict_last();
    // Loop constants in registers (the copies below are asm with memory
    // clobbers, after which kernel parameters would be re-read).
    const bool two = args.nsub == 2;
    const int w_row = n_tile * BLOCK_N, x_row1 = m0 + args.sub_n;
    const uint32_t x1_bytes = (uint32_t)(args.sub_n * BLOCK_K * 2);
    const uint32_t tx_bytes = (uint32_t)stage_bytes;
    // k-blocks [from, to) of this CTA's range, lane 0 only.
    auto issue = [&](int from, int to) {
      for (int i = from; i < to; ++i) {
        const int kb = kb_lo + i;
        uint8_t *st = sp.stage0 + (size_t)stage * stage_bytes;
        if (i >= early) {
          if (!mbar_wait_bounded(&sp.empty[stage], phase ^ 1u, abort_flag)) {
            signal_abort(sp, args.status);
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(&sp.full[stage], tx_bytes);
          tma_load_2d(st, &tmap_w, &sp.full[stage], kb * BLOCK_K, w_row, pol_w);
        }
        tma_load_2d(st + W_TILE_BYTES, &tmap_x, &sp.full[stage], kb * BLOCK_K, m0, pol_x);
        if (two) tma_load_2d(st + W_TILE_BYTES + x1_bytes, &tmap_x, &sp.full[stage], kb * BLOCK_K, x_row1, pol_x);
        ++issued;
        if (++stage == S) {
          stage = 0;
          phase ^= 1u;
        }
      }
    };
    auto sync_state = [&]() {
      ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
      stage = __shfl_sync(0xffffffffu, stage, 0);
      phase = __shfl_sync(0xffffffffu, phase, 0);
      issued = __shfl_sync(0xffffffffu, issued, 0);
      __syncwarp();
    };
    if (lane == 0) {
      // With static weights, the first ring of W tiles is requested before the
      // wait for the preceding kernel; x always comes after it.
      for (int i = 0; i < early; ++i) {
        mbar_arrive_expect_tx(&sp.full[i], tx_bytes);
        tma_load_2d(sp.stage0 + (size_t)i * stage_bytes, &tmap_w, &sp.full[i], (kb_lo + i) * BLOCK_K, w_row, pol_w);
      }
      // After this library's shrink kernel nothing the mainloop reads can
      // still be in flight (the shrink released this grid only after its own
      // predecessor had finished), so only the expand and the epilogue wait
      // for the shrink's output.
      if (!args.after_shrink) grid_dependency_wait();
      issue(0, split);
    }
    sync_state();
    if (ok && sorted_verify && !*abort_flag) {
      grid_dependency_wait();  // the plan and the token windows come from the kernels just before
      int blo = 0, bhi = 0;
      expand_range(blo, bhi);
      if (bhi > blo) {
        ok = expand_produce(args.plan + L.slices, blo, bhi, m0, args.Mb, n_tile * BLOCK_N, args.N, &tmap_b,
                            args.tw + (size_t)slice * args.tw_slice, sp.stage0, stage_bytes, S, sp.full, sp.empty,
                            sp.meta, sp.chunk, stage, phase, issued, abort_flag, pol_w, lane, args.n_ad,
                            (long long)(args.tw_slice / 16), args.status);
        if (!ok && lane == 0) signal_abort(sp, args.status);
      }
    }
    if (lane == 0 && ok && !*abort_flag) issue(split, nkb);
    sync_state();
    if (lane == 0 && *abort_flag) {
      // Let this CTA's own copies land before shared memory goes away.
      const int n = issued < S ? issued : S;
      for (int i = issued - n; i < issued; ++i) {
        mbar_wait_bounded(&sp.full[i % S], (uint32_t)((i / S) & 1), sp.zero_word);
      }
      if (early > issued) {
        for (int i = issued; i < early; ++i) {
          mbar_wait_bounded(&sp.full[i], 0u, sp.zero_word);  // W half only: never completes, bounded
        }
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    int stage = 0;
    uint32_t phase = 0;
    bool ok = true, issued_any = false;
    // Everything the loop needs is in registers before it starts: this one
    // thread issues every MMA of the CTA, so the issue path is kept to a few
    // integer adds per instruction (descriptor start addresses step by 32
    // bytes, i.e. 2 in the descriptor's 16-byte units, per 16-wide K step).
    const uint32_t idesc = idesc_bf16_f32(BLOCK_N, args.sub_n);
    const bool two = args.nsub == 2;
    const uint32_t d1 = tmem_base + (uint32_t)args.sub_n;
    const uint64_t x1_off = (uint64_t)((args.sub_n * BLOCK_K * 2) >> 4);
    const uint32_t ring0 = smem_addr(sp.stage0);
    const uint32_t sbytes = (uint32_t)stage_bytes;
    auto mma_kblocks = [&](int from, int to) {  // lane 0: k-blocks [kb_lo + from, kb_lo + to)
      for (int kb = kb_lo + from; kb < kb_lo + to; ++kb) {
        if (!mbar_wait_bounded(&sp.full[stage], phase, abort_flag)) {
          signal_abort(sp, args.status);
          ok = false;
          break;
        }
        tc_fence_after_sync();
        const uint32_t a_addr = ring0 + (uint32_t)stage * sbytes;
        const uint64_t ad = smem_desc_kmajor_sw128(a_addr);
        const uint64_t bd = smem_desc_kmajor_sw128(a_addr + W_TILE_BYTES);
        const uint32_t first = kb > kb_lo ? 1u : 0u;
#pragma unroll
        for (int kk = 0; kk < BLOCK_K / 16; ++kk) {
          const uint32_t accum = kk > 0 ? 1u : first;
          mma_bf16_ss(tmem_base, ad + 2 * kk, bd + 2 * kk, idesc, accum);
          if (two) mma_bf16_ss(d1, ad + 2 * kk, bd + x1_off + 2 * kk, idesc, accum);
        }
        issued_any = true;
        mma_commit(&sp.empty[stage]);
        if (++stage == S) {
          stage = 0;
          phase ^= 1u;
        }
      }
    };
    auto sync_state = [&]() {
      ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
      issued_any = __shfl_sync(0xffffffffu, issued_any ? 1 : 0, 0) != 0;
      stage = __shfl_sync(0xffffffffu, stage, 0);
      phase = __shfl_sync(0xffffffffu, phase, 0);
      __syncwarp();
    };
    if (lane == 0) mma_kblocks(0, split);
    sync_state();
    if (ok && sorted_verify) {
      grid_dependency_wait();  // the plan comes from a kernel earlier in the stream
      int blo = 0, bhi = 0;
      expand_range(blo, bhi);
      if (bhi > blo && !*abort_flag) {
        // The producer issues at least one expand stage whenever bhi > blo
        // and it has not given up.
        ok = expand_consume(sp.stage0, stage_bytes, S, sp.full, sp.empty, sp.meta, tmem_base, stage, phase,
                            abort_flag, lane);
        if (!ok && lane == 0) signal_abort(sp, args.status);
        issued_any = true;
      } else if (bhi > blo) {
        ok = false;  // the producer gave up before the expand
      }
    }
    if (lane == 0 && ok) mma_kblocks(split, nkb);
    sync_state();
    bool mma_ok = false;
    if (lane == 0) {
      if (ok) {
        mma_commit(sp.tfull);
      } else if (issued_any) {
        // Wait for this thread's MMAs before tensor memory is freed.
        mma_commit(sp.drain);
        mbar_wait_bounded(sp.drain, 0, sp.zero_word);
      }
      mma_ok = ok;
    }
    // Accumulator handoff: this thread waits for the last MMA, then the warp
    // releases the epilogue warps through named barrier 2, so they sleep in
    // hardware instead of polling while the mainloop runs.
    __syncwarp();
    if (lane == 0) {
      bool ready = mma_ok && mbar_wait_bounded(sp.tfull, 0, abort_flag);
      if (mma_ok && !ready) signal_abort(sp, args.status);
      *reinterpret_cast<volatile int *>(sp.acc_ready) = ready ? 1 : 0;
    }
    __syncwarp();
    tc_fence_before_sync();
    named_bar_arrive(2, 160);
  }

  // ------------------------------------------------------------ epilogue
  // Warps 2..5 read tensor memory (warp w may touch lanes 32*(w%4)..+31);
  // all six warps take part in every cluster barrier.
  __syncwarp();
  const bool epi = warp >= 2;
  const int quad = warp & 3;
  const int et = threadIdx.x - 64;
  bool have_acc = false;
  if (epi) {
    named_bar_sync(2, 160);  // released by the MMA warp once the accumulator is complete
    tc_fence_after_sync();
    have_acc = *reinterpret_cast<volatile int *>(sp.acc_ready) != 0;
    grid_dependency_wait();  // the plan and T come from kernels earlier in the stream
  }
  const uint32_t taddr = tmem_base + ((uint32_t)(quad * 32) << 16);
  const int nchunks = (mcount + CHUNK - 1) / CHUNK;

  // Verify work left for the epilogue: none once the tensor cores added it.
  const bool verify = args.mode == MLORA_VERIFY && !args.sorted;
  // Output row of accumulator column c: with sorted rows, perm[m0 + c].
  const int32_t *perm = args.sorted ? args.plan + L.perm : nullptr;
  // A permutation entry out of range (a plan overwritten or made for other
  // sizes) maps to -1: the store is skipped and MLORA_DEV_BAD_PLAN raised.
  auto out_row = [&](int c) -> long long {
    if (!perm) return (long long)(m0 + c);
    const int r = __ldg(perm + m0 + c);
    if ((unsigned)r < (unsigned)args.M) return r;
    raise_status(args.status, MLORA_DEV_BAD_PLAN);
    return -1;
  };

  if (C == 1) {
    if (epi && have_acc) {
      const int n = n_tile * BLOCK_N + quad * 32 + lane;
      if (!verify) {
        // With N % 8 == 0 and y 16-byte aligned, each warp's 32 W rows x 32
        // token columns go through a padded token-major block in the idle
        // stage ring, and lane j stores token column j's 32 outputs as four
        // 16-byte pieces; otherwise one two-byte store per output.
        const bool vec = (args.N & 7) == 0 && (reinterpret_cast<uintptr_t>(args.y) & 15) == 0;
        uint16_t *sy = reinterpret_cast<uint16_t *>(sp.stage0) + (size_t)quad * 32 * Y_ROW;
        const int nb = n_tile * BLOCK_N + quad * 32;
        for (int ch = 0; ch < nchunks; ++ch) {
          uint32_t r[32];
          tmem_ld_acc_x32(taddr + ch * CHUNK, r);
          // Lane j holds the output row of column ch * 32 + j.
          const int myc = ch * CHUNK + lane;
          const int myrow = myc < mcount ? (int)out_row(myc) : -1;
          if (vec) {
#pragma unroll
            for (int j = 0; j < CHUNK; ++j) sy[j * Y_ROW + lane] = float_to_bf16_bits(__uint_as_float(r[j]));
            __syncwarp();
            if (myrow >= 0) {
              const uint4 *src = reinterpret_cast<const uint4 *>(sy + lane * Y_ROW);
              uint16_t *dst = args.y + (size_t)myrow * args.N + nb;
#pragma unroll
              for (int q = 0; q < 4; ++q) {
                if (nb + 8 * q + 8 <= args.N) {
                  reinterpret_cast<uint4 *>(dst)[q] = src[q];
                } else {
                  for (int e = 0; e < 8; ++e)
                    if (nb + 8 * q + e < args.N) dst[8 * q + e] = sy[lane * Y_ROW + 8 * q + e];
                }
              }
            }
            __syncwarp();  // the block is rewritten by the next chunk
            continue;
          }
#pragma unroll
          for (int j = 0; j < CHUNK; ++j) {
            const int col = ch * CHUNK + j;
            const int row = __shfl_sync(0xffffffffu, myrow, j);
            if (n < args.N && col < mcount && row >= 0)
              args.y[(size_t)row * args.N + n] = float_to_bf16_bits(__uint_as_float(r[j]));
          }
        }
      } else {
        // Walk the plan's buckets (see verify_walk): the staged tables sit at
        // the start of the freed stage ring, the B-row slots after them.
        const size_t ring = (size_t)S * stage_bytes;
        const VerifyTables vt =
            stage_verify_tables(args, L, T_u, sp.stage0, ring - 8 * 128 * sizeof(uint4), m0, mcount, et);
        uint4 *Bs = reinterpret_cast<uint4 *>(sp.stage0 + vt.bytes);
        const int slot_cap = (int)((ring - vt.bytes) / (128 * sizeof(uint4)));
        verify_walk<true>(args, L, vt, Bs, slot_cap, et, n, m0, mcount, 0, 1, taddr, nullptr, 0, 0);
      }
    }
    tc_fence_before_sync();
    block_sync();
  } else {
    const int r0 = rank * BLOCK_N / C, r1 = (rank + 1) * BLOCK_N / C, R = r1 - r0;
    const size_t ring = (size_t)S * stage_bytes;
    // Verify mode keeps the reduced rows, column-major [Mb][R], in the stage
    // ring (free once the last MMA has completed) for the bucket walk below.
    float *fin = reinterpret_cast<float *>(sp.stage0);
    // One round when the whole accumulator fits the freed stage ring and no
    // bucket walk needs the ring afterwards; otherwise 32 columns at a time
    // through the double-buffered reduction tile.
    // (The epilogue writes whole 32-column chunks: round Mb up.)
    const bool oneshot = !verify && (size_t)((args.Mb + CHUNK - 1) / CHUNK * CHUNK) * BLOCK_N * 4 <= ring;
    if (oneshot) {
      float *acc_all = reinterpret_cast<float *>(sp.stage0);  // [Mb][128], one column of 128 rows after another
      const uint32_t ring_local = smem_addr(sp.stage0);
      uint32_t peer[MAX_CLUSTER];
#pragma unroll
      for (int p = 0; p < MAX_CLUSTER; ++p) peer[p] = (p < C) ? map_to_rank(ring_local, (uint32_t)p) : 0u;
      if (epi) {
        for (int ch = 0; ch < nchunks; ++ch) {
          uint32_t r[32];
          if (have_acc) {
            tmem_ld_acc_x32(taddr + ch * CHUNK, r);
          } else {
#pragma unroll
            for (int j = 0; j < 32; ++j) r[j] = 0u;
          }
#pragma unroll
          for (int j = 0; j < CHUNK; ++j) acc_all[(ch * CHUNK + j) * BLOCK_N + quad * 32 + lane] = __uint_as_float(r[j]);
        }
      }
      cluster_sync_all();
      if (epi)
        cluster_reduce_rows_c(C, peer, 0u, r0, R, mcount, et, [&](int c, int i, float4 v) {
          const long long row = out_row(c);
          if (row >= 0) store_bf16x4(args.y, args.N, (size_t)row, n_tile * BLOCK_N + r0 + i, v);
        });
    } else {
      const uint32_t red_local = smem_addr(sp.red);
      uint32_t peer[MAX_CLUSTER];
  #pragma unroll
      for (int p = 0; p < MAX_CLUSTER; ++p) peer[p] = (p < C) ? map_to_rank(red_local, (uint32_t)p) : 0u;
      for (int ch = 0; ch < nchunks; ++ch) {
        const int buf = ch & 1;
        float *red = sp.red + buf * CHUNK * BLOCK_N;
        if (epi) {
          uint32_t r[32];
          if (have_acc) {
            tmem_ld_acc_x32(taddr + ch * CHUNK, r);
          } else {
  #pragma unroll
            for (int j = 0; j < 32; ++j) r[j] = 0u;
          }
  #pragma unroll
          for (int j = 0; j < CHUNK; ++j) red[j * BLOCK_N + quad * 32 + lane] = __uint_as_float(r[j]);
        }
        cluster_sync_all();
        if (epi) {
          const int ncols = min(CHUNK, mcount - ch * CHUNK);
          cluster_reduce_rows_c(C, peer, (uint32_t)(buf * CHUNK * BLOCK_N * 4), r0, R, ncols, et,
                                [&](int c, int i, float4 v) {
                                  const int col = ch * CHUNK + c;
                                  if (verify) {
                                    *reinterpret_cast<float4 *>(&fin[col * R + i]) = v;
                                  } else {
                                    const long long row = out_row(col);
                                    if (row >= 0) store_bf16x4(args.y, args.N, (size_t)row, n_tile * BLOCK_N + r0 + i, v);
                                  }
                                });
        }
      }
    }
    if (verify && epi) {
      named_bar_sync(1, 128);
      // Stage ring after the reduction: fin, then the staged tables when
      // they fit, then the B-row slots.
      const size_t fin_bytes = align_up((size_t)args.Mb * R * 4, 16);
      const VerifyTables vt = stage_verify_tables(args, L, T_u, sp.stage0 + fin_bytes,
                                                  ring - fin_bytes - 8 * 128 * sizeof(uint4), m0, mcount, et);
      uint4 *Bs = reinterpret_cast<uint4 *>(sp.stage0 + fin_bytes + vt.bytes);
      const int slot_cap = (int)((ring - fin_bytes - vt.bytes) / (128 * sizeof(uint4)));
      // Threads split as (row i, column phase): P = floor(128 / R) threads
      // share a row; when R does not divide 128 the last 128 - P * R idle.
      const int P = 128 / R;
      const int i = et % R, sub = et / R;
      if (sub < P)
        verify_walk<false>(args, L, vt, Bs, slot_cap, et, n_tile * BLOCK_N + r0 + i, m0, mcount, sub, P, 0u, fin, R,
                           i);
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
  return s > MAX_STAGES ? MAX_STAGES : s;
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
  // Tensor-memory columns: a power of two >= 32 holding Mb fp32 columns.
  int cols = 32;
  while (cols < Mb) cols <<= 1;
  s.tmem_cols = cols;
  s.nbuf = 1;
  s.total_iters = s.n_units * s.kblocks;
  // Split-K factor C (CTA r of a cluster owns output rows [r*128/C,
  // (r+1)*128/C) in the reduction): minimise waves x (k-blocks per CTA +
  // fixed cost), with a reduction cost for C > 1; C = 1 needs no cluster.
  const bool attrs = ensure_attributes();
  int bestC = 1;
  double best = 1e30;
  // Powers of two only: measured, clusters of 3 ran slower than the
  // persistent stream-K kernel that takes those shapes instead.
  int bestW = 1;
  for (int C = 1; C <= MAX_CLUSTER && C <= s.kblocks; C <<= 1) {
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
      bestW = (int)waves;
    }
  }
  s.C = bestC;
  s.waves = bestW;
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

// Row-major bf16 matrix [rows, cols] read in boxes of box_rows x box_cols
// (64 columns with 128-byte swizzling, or 16 with 32-byte swizzling);
// out-of-range elements read as zero.
static bool make_map(CUtensorMap *map, const void *base, long long rows, int cols, int box_rows, int box_cols = BLOCK_K) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)cols * 2};
  cuuint32_t box[2] = {(cuuint32_t)box_cols, (cuuint32_t)box_rows};
  cuuint32_t estr[2] = {1, 1};
  const CUtensorMapSwizzle sw = box_cols == 16 ? CU_TENSOR_MAP_SWIZZLE_32B : CU_TENSOR_MAP_SWIZZLE_128B;
  CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(base), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

cudaError_t launch_gemm(const GemmLaunch &g, const GemmShape &sh, cudaStream_t s, int *err_code) {
  *err_code = 0;
  CUtensorMap tw, tx, tb;
  if (!make_map(&tw, g.W, g.N, g.K, BLOCK_N) || !make_map(&tx, g.x, g.M, g.K, sh.sub_n)) {
    *err_code = 1;
    return cudaErrorInvalidValue;
  }
  // Verify mode with the token windows: x is in adapter-sorted order and the
  // tensor cores add the low-rank term.
  const int sorted = (g.mode == MLORA_VERIFY && g.tw != nullptr) ? 1 : 0;
  tb = tw;
  if (sorted) {
    if (!make_map(&tb, g.B_stack, (long long)g.n_ad * g.N, g.r_max, BLOCK_N, 16)) {
      *err_code = 1;
      return cudaErrorInvalidValue;
    }
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
  a.after_shrink = g.after_shrink;
  a.sorted = sorted;
  a.n_slices = g.n_slices;
  for (int i = 0; i < MLORA_MAX_SLICES; ++i) a.slice_end[i] = i < g.n_slices ? g.slice_end[i] : g.N;
  a.tw_slice = max_window_rows(g.M, g.n_ad) * 16;
  a.scale = g.scale;
  a.y = g.y;
  a.B_stack = g.B_stack;
  a.tw = g.tw;
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
  cudaError_t e = cudaLaunchKernelEx(&cfg, gemm_kernel, tw, tx, tb, a);
  note_launch();
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace mlora
