// The low-rank expand on the tensor cores, shared by the two GEMM kernels
// (step a4 of "output = W·x + scale · B(A·x)", "Multi-LoRA Serving in
// Practice", section "Core Principle: Shared Base Model, Per-Request Adapter
// Selection").
//
// In verify mode the GEMM reads the token rows in adapter-sorted order, so the
// rows of adapter a are the adjacent accumulator columns [s0, s1).  For each
// expand block (a, 16-rank block j0) one MMA (two past 256 columns) adds
//
//   acc[n, w0:w0+W] += B_a[n0:n0+128, j0:j0+16] x Twin^T
//
// where Twin is the block's token window (W rows of 16 bf16, scale * T on a's
// rows and 0 on the neighbours the 16-row rounding takes in), written by the
// shrink kernel in the 32-byte-swizzled row order.  The MMA work is the
// window's, not the whole batch's: sum over blocks of 128 x 16 x W.
//
// The producer warp stages the plan's block records 32 at a time (one lane
// each), clips each window to the CTA's token columns and packs as many
// blocks as fit into a ring stage (B tiles first, 4 KB each, then the
// windows).  It describes the stage in an ExpandStage record before arming
// the stage's barrier; the MMA warp reads the record after the barrier
// completes, zeroes the B columns past the adapter's rank (they hold the
// caller's padding, possibly NaN, and NaN * 0 is NaN), and issues the MMAs.
// The final stage of a CTA's expand is flagged `last`.
#pragma once

#include "common.cuh"

namespace mlora {

constexpr int EXP_MAX_PER_STAGE = 16;  // expand blocks one ring stage carries at most
constexpr int EXP_CHUNK = 32;          // plan records the producer warp stages per round
constexpr int EXP_B_TILE = 128 * 32;   // one B tile: 128 rows x 16 bf16

// One ring stage filled with expand operands.
struct ExpandStage {
  int4 blk[EXP_MAX_PER_STAGE];  // {B tile offset, window offset (bytes in the stage),
                                //  first accumulator column, window rows | rank columns << 16}
  int count, last, pad0, pad1;
};

// Shared memory the expand needs besides the ring: one record per stage and
// the producer's staged plan records.
__host__ __device__ constexpr size_t expand_smem_bytes(int stages) {
  return (size_t)stages * sizeof(ExpandStage) + (size_t)EXP_CHUNK * 32;
}

// Zero logical columns [c0, 16) of a 128-row x 16-column bf16 tile written by
// TMA with 32-byte swizzling (row i at byte 32 i; its two 16-byte halves are
// swapped when bit 2 of i is set).  Each lane of the warp takes 4 rows.
__device__ __forceinline__ void zero_tail_columns_sw32(uint8_t *tile, int c0, int lane) {
#pragma unroll 1
  for (int q = 0; q < 4; ++q) {
    const int i = lane * 4 + q;
    uint8_t *row = tile + i * 32;
    const int flip = (i >> 2) & 1;
    for (int c = c0; c < 16; ++c) {
      const int chunk = (c >> 3) ^ flip;
      *reinterpret_cast<uint16_t *>(row + chunk * 16 + (c & 7) * 2) = 0;
    }
  }
}

// Producer side, called by all 32 lanes of the producer warp: issue the
// expand stages for plan blocks [blo, bhi) of the output tile starting at W
// row n0, with the windows clipped to token columns [m0, m0 + mcols).  Lane 0
// packs the stages and issues the copies; every lane waits for each stage's
// slot and keeps the same stage / phase / issued count.
// Returns false if a wait gave up.
// A record out of range (n_ad adapters, tw_rows rows in the window buffer)
// means the plan was overwritten or made for other sizes: the block is
// dropped and MLORA_DEV_BAD_PLAN raised.
__device__ __forceinline__ bool expand_produce(const int32_t *blocks, int blo, int bhi, int m0, int mcols, int n0,
                                               int N, const CUtensorMap *tmap_b, const uint16_t *tw, uint8_t *ring,
                                               int stage_bytes, int S, uint64_t *full, uint64_t *empty,
                                               ExpandStage *meta, int4 *chunk, int &stage, uint32_t &phase,
                                               int &issued, volatile int *abort, uint64_t pol, int lane, int n_ad,
                                               long long tw_rows, uint32_t *status) {
  bool ok = true;
  for (int c0 = blo; c0 < bhi && ok; c0 += EXP_CHUNK) {
    const int n = min(EXP_CHUNK, bhi - c0);
    const bool final_chunk = c0 + EXP_CHUNK >= bhi;
    if (lane < n) {
      const int4 e0 = *reinterpret_cast<const int4 *>(blocks + (size_t)(c0 + lane) * EXP_WORDS);
      const int4 e1 = *reinterpret_cast<const int4 *>(blocks + (size_t)(c0 + lane) * EXP_WORDS + 4);
      const int w0 = e1.x, W = e1.y;
      const bool valid = (unsigned)e0.x < (unsigned)n_ad && (e0.y & 15) == 0 && (unsigned)e0.y < 64u &&
                         e0.z >= 1 && e0.z <= 16 && e0.w >= 0 && w0 >= 0 && (w0 & 15) == 0 && W >= 0 &&
                         (W & 15) == 0 && (long long)e0.w + W <= tw_rows;
      if (!valid) raise_status(status, MLORA_DEV_BAD_PLAN);
      const int cs = max(w0, m0), ce = min(w0 + W, m0 + mcols);
      const int rows = (valid && ce > cs) ? ce - cs : 0;
      // {adapter, j0 | rank columns << 8, first window row, column | rows << 16}
      chunk[lane] = make_int4(e0.x, e0.y | (e0.z << 8), e0.w + (rows ? cs - w0 : 0), rows ? ((cs - m0) | (rows << 16)) : 0);
    }
    __syncwarp();
    // Lane 0 packs each stage; every lane waits for the stage's slot itself
    // (a lane that waits behind another's suspended wait and a shuffle
    // measured about 0.5 us a stage), so the loop stays warp-uniform.
    int i = 0;
    bool emitted = false;  // a stage of this chunk was issued
    while (true) {
      int sel[EXP_MAX_PER_STAGE];
      int cnt = 0, tbytes = 0, j = i;
      bool more = false;
      if (lane == 0) {
        while (j < n && cnt < EXP_MAX_PER_STAGE) {
          const int rows = chunk[j].w >> 16;
          if (rows == 0) {
            ++j;
            continue;
          }
          if ((cnt + 1) * EXP_B_TILE + tbytes + rows * 32 > stage_bytes) break;
          sel[cnt++] = j;
          tbytes += rows * 32;
          ++j;
        }
        for (int q = j; q < n; ++q) more |= (chunk[q].w >> 16) > 0;
      }
      cnt = __shfl_sync(0xffffffffu, cnt, 0);
      j = __shfl_sync(0xffffffffu, j, 0);
      more = __shfl_sync(0xffffffffu, more ? 1 : 0, 0) != 0;
      // The last chunk always issues a stage, so the MMA warp sees `last`.
      if (cnt == 0 && !(final_chunk && !emitted)) break;
      const bool last = final_chunk && !more;
      if (!__all_sync(0xffffffffu, mbar_wait_bounded(&empty[stage], phase ^ 1u, abort))) {
        ok = false;
        break;
      }
      if (lane == 0) {
        uint8_t *st = ring + (size_t)stage * stage_bytes;
        ExpandStage &m = meta[stage];
        int toff = cnt * EXP_B_TILE;
        for (int c = 0; c < cnt; ++c) {
          const int4 r = chunk[sel[c]];
          const int rows = r.w >> 16;
          m.blk[c] = make_int4(c * EXP_B_TILE, toff, r.w & 0xFFFF, rows | (((r.y >> 8) & 0xFF) << 16));
          toff += rows * 32;
        }
        m.count = cnt;
        m.last = last ? 1 : 0;
        // The arrival releases the record; the copies complete the phase.
        mbar_arrive_expect_tx(&full[stage], (uint32_t)(cnt * EXP_B_TILE + tbytes));
        for (int c = 0; c < cnt; ++c) {
          const int4 r = chunk[sel[c]];
          tma_load_2d(st + c * EXP_B_TILE, tmap_b, &full[stage], r.y & 0xFF, r.x * N + n0, pol);
        }
        // The windows of consecutive blocks usually sit back to back in the
        // window buffer (the plan lays them out in block order): one bulk
        // copy per run of contiguous windows, not one per block.
        for (int c = 0; c < cnt;) {
          const int4 r = chunk[sel[c]];
          int rows = r.w >> 16, e = c + 1;
          while (e < cnt && chunk[sel[e]].z == r.z + rows) rows += chunk[sel[e++]].w >> 16;
          bulk_load(st + m.blk[c].y, tw + (size_t)r.z * 16, (uint32_t)(rows * 32), &full[stage]);
          c = e;
        }
      }
      __syncwarp();
      emitted = true;
      ++issued;
      if (++stage == S) {
        stage = 0;
        phase ^= 1u;
      }
      i = j;
      if (!more) break;
    }
    __syncwarp();  // the chunk table is rewritten only after lane 0 has read it
  }
  return ok;
}

// The MMAs of one expand stage whose barrier has completed (all 32 lanes of
// the MMA warp): zero the B columns past each block's rank columns, then
// lane 0 issues one MMA per block (two past 256 window rows) into the
// accumulator columns of its window and commits the stage to `empty_bar`.
// acc is the tensor-memory address of the accumulator's column 0 (the CTA's
// first token column).
__device__ __forceinline__ void expand_stage_mma(uint8_t *st, const ExpandStage &m, uint32_t acc, uint64_t *empty_bar,
                                                 int lane) {
  const int cnt = m.count;
  bool zeroed = false;
  for (int c = 0; c < cnt; ++c) {
    const int cols = m.blk[c].w >> 16;
    if (cols < 16) {
      zero_tail_columns_sw32(st + m.blk[c].x, cols, lane);
      zeroed = true;
    }
  }
  if (zeroed) fence_proxy_async_smem();
  __syncwarp();
  if (lane == 0) {
    tc_fence_after_sync();
    const uint32_t base = smem_addr(st);
    for (int c = 0; c < cnt; ++c) {
      const int4 b = m.blk[c];
      const int rows = b.w & 0xFFFF;
      const uint64_t bd = smem_desc_kmajor_sw32(base + (uint32_t)b.x);
      for (int p = 0; p < rows; p += 256) {
        const int nn = min(256, rows - p);
        mma_bf16_ss(acc + (uint32_t)(b.z + p), bd, smem_desc_kmajor_sw32(base + (uint32_t)(b.y + p * 32)),
                    idesc_bf16_f32(128, nn), 1u);
      }
    }
    mma_commit(empty_bar);
  }
  __syncwarp();
}

// MMA side, called by all 32 lanes of the MMA warp after the producer has
// issued at least one expand stage: run stages until the one flagged `last`.
// Returns false if a wait gave up.
__device__ __forceinline__ bool expand_consume(uint8_t *ring, int stage_bytes, int S, uint64_t *full,
                                               uint64_t *empty, const ExpandStage *meta, uint32_t acc, int &stage,
                                               uint32_t &phase, volatile int *abort, int lane) {
  bool ok = true;
  while (true) {
    // Every lane tests the barrier itself (no lane waits behind another's
    // suspended wait); they agree on the outcome before going on.
    ok = __all_sync(0xffffffffu, mbar_wait_bounded(&full[stage], phase, abort));
    if (!ok) break;
    tc_fence_after_sync();
    const ExpandStage &m = meta[stage];
    const bool last = m.last != 0;
    expand_stage_mma(ring + (size_t)stage * stage_bytes, m, acc, &empty[stage], lane);
    if (++stage == S) {
      stage = 0;
      phase ^= 1u;
    }
    if (last) break;
  }
  return ok;
}

}  // namespace mlora
