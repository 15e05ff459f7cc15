// The steps on either side of the accept step: the softmax that turns a
// pass's logits into the distributions the accept step compares, and the draw
// of each request's draft token from the draft distribution q (the InvisibleLoRA
// abstract: a LoRA-off pass proposes the next token for every request, one
// LoRA-on pass verifies the proposals).
//
// One definition of a probability serves every kernel of the library (the
// functions of prob.cuh): p(v) = e^(z(v) - m) R, with m the row maximum and
// R = 1/S the reciprocal of the row sum below, rounded once per row.  The row
// statistics are built over 512-entry blocks: a lane takes the maximum of its
// 16 entries of the block, then the sum of e^(z - that maximum); the lanes'
// pairs are merged in a fixed tree (the maximum first, then the partial sums
// rescaled to it and added) into the block's pair, and a second kernel merges
// a row's block pairs the same way in a fixed order and stores (m, 1/S).
// Nothing depends on the grid or on the other rows of the call, so a row's
// statistics are the same in every call; because every entry of p is computed
// from them by the same expression, the probabilities the accept step derives
// from logits are bit-identical to the ones softmax_write writes.
//
// The draft draw uses the accept step's exact integer inverse CDF on
// Q(q(v)) = floor(q(v) * 2^40): S_w = sum of the weights, U = floor(u * 2^32),
// T = floor(U * S_w / 2^32), token = the smallest v whose running sum of
// weights exceeds T.  Each block's weight sum is kept (exact in uint64, so the
// order of the additions does not matter), the block holding T is found by a
// scan over them, then the token inside it by a warp scan.
//
// The kernels that read whole rows are streaming kernels: one warp per
// (row, 512-entry block) unit, each load instruction of a warp 512
// contiguous bytes, no barrier, atomic or fence between the warps (the merges
// run in the next kernel, ordered by the launch).
#include <algorithm>

#include "common.cuh"
#include "launch.h"
#include "prob.cuh"

namespace mlora {

constexpr int SM_BLOCK = 512;            // entries per (row, block) unit: 16 per lane
constexpr int UNIT_WARPS = 8;            // units per CTA of the streaming kernels
constexpr int ROW_WARPS = 4;             // rows per CTA of the per-row kernels
constexpr float SM_TWO_POW_32 = 4294967296.0f;

// The entries of block k a lane holds: lane l takes the block's four-entry
// groups 4 l + 128 j (j < 4), so that v[4 j + i] holds entry
// 512 k + 4 l + 128 j + i.
__device__ __forceinline__ int lane_entry(int k, int j, int i) {
  return SM_BLOCK * k + 4 * (threadIdx.x & 31) + 128 * j + i;
}

// Loads a lane's 16 entries of block k of `row`; entries at or past V read
// as `fill`.  vec: the row is 16-byte aligned and V a multiple of 4.  STREAM
// marks the lines evict-first (the last read of the row).
template <bool STREAM>
__device__ __forceinline__ void load_block(const float *row, int k, int V, bool vec, float fill, float (&v)[16]) {
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const int e = lane_entry(k, j, 0);
    if (vec) {
      float4 f = make_float4(fill, fill, fill, fill);
      if (e < V) {
        const float4 *p = reinterpret_cast<const float4 *>(row + e);
        f = STREAM ? __ldcs(p) : __ldg(p);
      }
      v[4 * j] = f.x, v[4 * j + 1] = f.y, v[4 * j + 2] = f.z, v[4 * j + 3] = f.w;
    } else {
#pragma unroll
      for (int i = 0; i < 4; ++i) v[4 * j + i] = e + i < V ? (STREAM ? __ldcs(row + e + i) : __ldg(row + e + i)) : fill;
    }
  }
}

// A partial sum s taken relative to the maximum m, rescaled to the maximum
// M >= m (nothing when m is -inf: every entry behind it is masked).
__device__ __forceinline__ float rescaled(float m, float s, float M) { return m == -INFINITY ? 0.f : s * exp_of(m - M); }

// (maximum, sum of e^(z - maximum)) of a lane's 16 entries, in index order.
__device__ __forceinline__ float2 lane_stats(const float (&v)[16]) {
  float m = v[0];
#pragma unroll
  for (int j = 1; j < 16; ++j) m = fmaxf(m, v[j]);
  float s = 0.f;
  if (m != -INFINITY) {
#pragma unroll
    for (int j = 0; j < 16; ++j) s += exp_of(v[j] - m);
  }
  return make_float2(m, s);
}

// Merge the warp's pairs: the maximum over the lanes, then each lane's sum
// rescaled to it and added in a fixed tree.  Valid in lane 0.
__device__ __forceinline__ float2 warp_merge(float m, float s) {
  float M = m;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
  float t = rescaled(m, s, M);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) t += __shfl_down_sync(0xffffffffu, t, o);
  return make_float2(M, t);
}

// part[r][k] = the pair of block k of row r, for the rows of two matrices
// taken as one: rows r < R1 are rows of z1, the others rows r - R1 of z2
// (R1 = all rows for one matrix).  Grid (rows, groups of UNIT_WARPS blocks);
// warp w of CTA (r, y) takes block k = UNIT_WARPS y + w.
__global__ void __launch_bounds__(UNIT_WARPS * 32)
    block_stats_kernel(const float *__restrict__ z1, int R1, const float *__restrict__ z2, int V, int nblk,
                       float2 *__restrict__ part) {
  grid_dependency_wait();
  grid_launch_dependents();
  const int r = blockIdx.x, k = blockIdx.y * UNIT_WARPS + (threadIdx.x >> 5);
  if (k >= nblk) return;
  const float *row = r < R1 ? z1 + (size_t)r * V : z2 + (size_t)(r - R1) * V;
  const bool vec = (V & 3) == 0 && (reinterpret_cast<uintptr_t>(r < R1 ? z1 : z2) & 15) == 0;
  float v[16];
  load_block<false>(row, k, V, vec, -INFINITY, v);
  const float2 t = lane_stats(v);
  const float2 w = warp_merge(t.x, t.y);
  if ((threadIdx.x & 31) == 0) part[(size_t)r * nblk + k] = w;
}

// A row's pair (m, 1/S) from its block pairs pr[0, nblk), by one warp: the
// maximum, then lane l adds the rescaled sums of blocks l, l + 32, ... in
// that order, the lanes' sums are added in a fixed tree, and the total's
// reciprocal is rounded once (IEEE).  Valid in lane 0.
__device__ __forceinline__ float2 merge_row(const float2 *pr, int nblk) {
  const int lane = threadIdx.x & 31;
  float M = -INFINITY;
  for (int k = lane; k < nblk; k += 32) M = fmaxf(M, pr[k].x);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
  float s = 0.f;
  for (int k = lane; k < nblk; k += 32) {
    const float2 p = pr[k];
    s += rescaled(p.x, p.y, M);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) s += __shfl_down_sync(0xffffffffu, s, o);
  return make_float2(M, __frcp_rn(s));
}

// stats[r] = merge_row of row r, one warp per row.
__global__ void __launch_bounds__(ROW_WARPS * 32)
    row_merge_kernel(const float2 *__restrict__ part, int R, int nblk, float2 *__restrict__ stats) {
  grid_dependency_wait();
  grid_launch_dependents();
  const int r = blockIdx.x * ROW_WARPS + (threadIdx.x >> 5);
  if (r >= R) return;
  const float2 st = merge_row(part + (size_t)r * nblk, nblk);
  if ((threadIdx.x & 31) == 0) stats[r] = st;
}

// p[r, v] = prob_from_logit(z[r, v], stats[r]), in the units of block_stats.
__global__ void __launch_bounds__(UNIT_WARPS * 32)
    softmax_write_kernel(const float *__restrict__ z, int V, int nblk, const float2 *__restrict__ stats,
                         float *__restrict__ p) {
  grid_dependency_wait();
  grid_launch_dependents();
  const int r = blockIdx.x, k = blockIdx.y * UNIT_WARPS + (threadIdx.x >> 5);
  if (k >= nblk) return;
  const bool vec = (V & 3) == 0 && (reinterpret_cast<uintptr_t>(z) & 15) == 0 &&
                   (reinterpret_cast<uintptr_t>(p) & 15) == 0;
  const float2 st = stats[r];
  float v[16];
  load_block<true>(z + (size_t)r * V, k, V, vec, 0.f, v);
  float *pr = p + (size_t)r * V;
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const int e = lane_entry(k, j, 0);
    if (vec) {
      if (e < V)
        __stcs(reinterpret_cast<float4 *>(pr + e), make_float4(prob_from_logit(v[4 * j], st), prob_from_logit(v[4 * j + 1], st),
                                                               prob_from_logit(v[4 * j + 2], st), prob_from_logit(v[4 * j + 3], st)));
    } else {
#pragma unroll
      for (int i = 0; i < 4; ++i)
        if (e + i < V) pr[e + i] = prob_from_logit(v[4 * j + i], st);
    }
  }
}

// Q(f) = floor(f * 2^40) of f clamped to [0, 1] (NaN to 0), in two parts,
// each from one float operation rounded down onto the integers of
// [2^23, 2^24], whose bit patterns are 0x4B000000 plus the integer:
//   h  = floor(c 2^23):          t1 = c 2^23 + 2^23 rounded down;
//   lo = floor((c 2^23 - h) 2^17): c 2^23 - h (exact, in [0, 1)) times 2^17
//                                  plus 2^23, rounded down;
// and Q = h 2^17 + lo.  q40_parts returns the two bit patterns; a sum of n
// of them, taken mod 2^32, less n * 0x4B000000 is the sum of the parts
// exactly as long as that sum is below 2^32.
constexpr uint32_t Q40_OFFSET = 0x4B000000u;  // the bit pattern of 2^23

__device__ __forceinline__ void q40_parts(float f, uint32_t &hb, uint32_t &lb) {
  const float c = fminf(fmaxf(f, 0.f), 1.f);
  const float t1 = __fmaf_rd(c, 8388608.0f, 8388608.0f);
  const float fr = __fmaf_rn(c, 8388608.0f, -(t1 - 8388608.0f));
  const float t2 = __fmaf_rd(fr, 131072.0f, 8388608.0f);
  hb = __float_as_uint(t1);
  lb = __float_as_uint(t2);
}

// Q from the parts' sums (offsets removed): h 2^17 + lo.
__device__ __forceinline__ uint64_t q40_join(uint32_t h, uint32_t lo) { return ((uint64_t)h << 17) + lo; }

__device__ __forceinline__ uint64_t q40(float f) {
  uint32_t hb, lb;
  q40_parts(f, hb, lb);
  return q40_join(hb - Q40_OFFSET, lb - Q40_OFFSET);
}

__device__ __forceinline__ uint64_t warp_sum_u64_sm(uint64_t v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

__device__ __forceinline__ uint64_t warp_incl_scan_u64_sm(uint64_t v) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint64_t t = __shfl_up_sync(0xffffffffu, v, o);
    if (lane >= o) v += t;
  }
  return v;
}

// Draft draw, first half: in the units of block_stats, the probabilities of
// block k of row b (written to q_out when it is given) and the block's exact
// weight sum blk[b][k] = sum of Q(q(v)).
__global__ void __launch_bounds__(UNIT_WARPS * 32)
    draw_weights_kernel(const float *__restrict__ z, int V, int nblk, const float2 *__restrict__ stats,
                        float *__restrict__ q_out, uint64_t *__restrict__ blk) {
  grid_dependency_wait();
  grid_launch_dependents();
  const int b = blockIdx.x, k = blockIdx.y * UNIT_WARPS + (threadIdx.x >> 5);
  if (k >= nblk) return;
  const bool vec = (V & 3) == 0 && (reinterpret_cast<uintptr_t>(z) & 15) == 0;
  const bool vec_q = (V & 3) == 0 && (reinterpret_cast<uintptr_t>(q_out) & 15) == 0;
  const float2 st = stats[b];
  float v[16];
  load_block<true>(z + (size_t)b * V, k, V, vec, 0.f, v);
  // The lane's 16 weights as sums of their parts' bit patterns (the h parts
  // sum below 2^27, the lo parts below 2^21).
  uint32_t sh = 0, sl = 0;
  if ((k + 1) * SM_BLOCK <= V) {  // every block but a row's last
#pragma unroll
    for (int j = 0; j < 16; ++j) {
      v[j] = prob_from_logit(v[j], st);
      uint32_t hb, lb;
      q40_parts(v[j], hb, lb);
      sh += hb, sl += lb;
    }
  } else {
#pragma unroll
    for (int j = 0; j < 16; ++j) {
      v[j] = lane_entry(k, j >> 2, j & 3) < V ? prob_from_logit(v[j], st) : 0.f;
      uint32_t hb, lb;
      q40_parts(v[j], hb, lb);
      sh += hb, sl += lb;
    }
  }
  uint64_t w = q40_join(sh - 16u * Q40_OFFSET, sl - 16u * Q40_OFFSET);
  if (q_out) {
    float *qr = q_out + (size_t)b * V;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int e = lane_entry(k, j, 0);
      if (vec_q) {
        if (e < V) *reinterpret_cast<float4 *>(qr + e) = make_float4(v[4 * j], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]);
      } else {
#pragma unroll
        for (int i = 0; i < 4; ++i)
          if (e + i < V) qr[e + i] = v[4 * j + i];
      }
    }
  }
  w = warp_sum_u64_sm(w);
  if ((threadIdx.x & 31) == 0) blk[(size_t)b * nblk + k] = w;
}

// Draft draw, second half, one warp per request b, three searches that each
// take one round of parallel loads: lane l sums a contiguous run of the
// blocks' weights and a warp scan finds the run that holds T; the warp scans
// that run 32 blocks at a time and finds the block; lane l recomputes the
// weights of 16 consecutive entries of the block (the same expression) and a
// last warp scan finds the token.
__global__ void __launch_bounds__(ROW_WARPS * 32)
    draw_token_kernel(const float *__restrict__ z, int B, int V, int nblk, const float2 *__restrict__ stats,
                      const uint64_t *__restrict__ blk, const float *__restrict__ u, int32_t *__restrict__ tok,
                      uint32_t *status) {
  grid_dependency_wait();
  grid_launch_dependents();
  const int b = blockIdx.x * ROW_WARPS + (threadIdx.x >> 5), lane = threadIdx.x & 31;
  if (b >= B) return;
  const uint64_t *bw = blk + (size_t)b * nblk;
  const int per = (nblk + 31) / 32;
  const int k0 = min(nblk, lane * per), k1 = min(nblk, k0 + per);
  uint64_t mine = 0;
  for (int k = k0; k < k1; ++k) mine += bw[k];
  const uint64_t inc = warp_incl_scan_u64_sm(mine);
  const uint64_t total = __shfl_sync(0xffffffffu, inc, 31);
  float uu = u[b];
  uint32_t fl = 0;
  if (!(uu >= 0.f)) {
    uu = 0.f;
    fl |= MLORA_DEV_BAD_PROB;
  } else if (uu >= 1.f) {
    uu = __uint_as_float(0x3F7FFFFFu);
    fl |= MLORA_DEV_BAD_PROB;
  }
  if (total == 0) fl |= MLORA_DEV_ZERO_MASS;
  const uint64_t U = __float2ull_rz(uu * SM_TWO_POW_32);
  const uint64_t T = total == 0 ? 0 : (__umul64hi(U, total) << 32) | ((U * total) >> 32);  // floor(U * S / 2^32) < S
  const uint32_t hit = __ballot_sync(0xffffffffu, total != 0 && inc - mine <= T && T < inc);
  int t = 0;
  if (hit) {
    const int src = __ffs(hit) - 1;
    uint64_t run = __shfl_sync(0xffffffffu, inc - mine, src);
    const int r0 = __shfl_sync(0xffffffffu, k0, src), r1 = __shfl_sync(0xffffffffu, k1, src);
    int kb = -1;
    uint64_t Tl = 0;
    for (int base = r0; base < r1 && kb < 0; base += 32) {
      const uint64_t w = base + lane < r1 ? bw[base + lane] : 0ull;
      const uint64_t c = warp_incl_scan_u64_sm(w);
      const uint32_t h = __ballot_sync(0xffffffffu, run + c - w <= T && T < run + c);
      if (h) {
        const int l = __ffs(h) - 1;
        kb = base + l;
        Tl = T - run - __shfl_sync(0xffffffffu, c - w, l);
      } else {
        run += __shfl_sync(0xffffffffu, c, 31);
      }
    }
    if (kb >= 0) {  // always, when the sums are consistent
      const float *row = z + (size_t)b * V;
      const float2 st = stats[b];
      const int v0 = kb * SM_BLOCK + 16 * lane;
      uint64_t mw = 0;
#pragma unroll
      for (int j = 0; j < 16; ++j)
        if (v0 + j < V) mw += q40(prob_from_logit(__ldg(row + v0 + j), st));
      const uint64_t inc2 = warp_incl_scan_u64_sm(mw);
      uint64_t run2 = inc2 - mw;
      const uint32_t hit2 = __ballot_sync(0xffffffffu, run2 <= Tl && Tl < run2 + mw);
      int found = -1;
      if (hit2 && lane == __ffs(hit2) - 1) {  // the lane's weights again, in order
        for (int j = 0; j < 16 && v0 + j < V; ++j) {
          run2 += q40(prob_from_logit(__ldg(row + v0 + j), st));
          if (Tl < run2) {
            found = v0 + j;
            break;
          }
        }
      }
      t = hit2 ? __shfl_sync(0xffffffffu, found, __ffs(hit2) - 1) : 0;
      if (t < 0) t = 0;  // unreachable when the sums are consistent
    }
  }
  if (lane == 0) {
    tok[b] = t;
    if (fl) raise_status(status, fl);
  }
}

// Test hook: counts the bit patterns first + i (i < count) whose q40 differs
// from CUDA's round-down conversion of the clamped f * 2^40.
__global__ void q40_check_kernel(uint32_t first, uint32_t count, unsigned long long *mismatches) {
  unsigned long long bad = 0;
  const uint32_t stride = gridDim.x * blockDim.x;
  for (uint32_t i = blockIdx.x * blockDim.x + threadIdx.x; i < count; i += stride) {
    const float f = __uint_as_float(first + i);
    const uint64_t ref = __float2ull_rd(fminf(fmaxf(f, 0.f), 1.f) * 1099511627776.0f);
    bad += q40(f) != ref;
    if (stride > count - i) break;  // the next i would wrap past 2^32
  }
  bad = warp_sum_u64_sm(bad);
  if ((threadIdx.x & 31) == 0 && bad) atomicAdd(mismatches, bad);
}

cudaError_t launch_q40_check(uint32_t first, uint32_t count, unsigned long long *mismatches, int num_sms,
                             cudaStream_t s) {
  q40_check_kernel<<<std::max(num_sms, 1) * 8, 256, 0, s>>>(first, count, mismatches);
  return cudaGetLastError();
}

// Test hook: the largest relative difference between exp_of(d) and CUDA's
// expf(d) over the bit patterns first + i (i < count), where expf(d) is a
// normal float; atomicMax on the bit pattern of the (non-negative) float.
__global__ void exp_check_kernel(uint32_t first, uint32_t count, unsigned int *max_rel_bits) {
  float worst = 0.f;
  const uint32_t stride = gridDim.x * blockDim.x;
  for (uint32_t i = blockIdx.x * blockDim.x + threadIdx.x; i < count; i += stride) {
    const float d = __uint_as_float(first + i);
    const float ref = expf(d);
    if (isfinite(d) && isfinite(ref) && ref >= 1.17549435e-38f) worst = fmaxf(worst, fabsf(exp_of(d) - ref) / ref);
    if (stride > count - i) break;  // the next i would wrap past 2^32
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) worst = fmaxf(worst, __shfl_xor_sync(0xffffffffu, worst, o));
  if ((threadIdx.x & 31) == 0 && worst > 0.f) atomicMax(max_rel_bits, __float_as_uint(worst));
}

cudaError_t launch_exp_check(uint32_t first, uint32_t count, unsigned int *max_rel_bits, int num_sms,
                             cudaStream_t s) {
  exp_check_kernel<<<std::max(num_sms, 1) * 8, 256, 0, s>>>(first, count, max_rel_bits);
  return cudaGetLastError();
}

static int blocks_of(int V) { return (V + SM_BLOCK - 1) / SM_BLOCK; }

// The grid of the streaming kernels: x = row, y = group of UNIT_WARPS blocks.
static dim3 unit_grid(int R, int nblk) { return dim3((unsigned)R, (unsigned)((nblk + UNIT_WARPS - 1) / UNIT_WARPS)); }

size_t row_stats_scratch_bytes(int R, int V) { return align_up((size_t)R * blocks_of(V) * sizeof(float2), 256); }

cudaError_t launch_row_stats(const float *z1, int R1, const float *z2, int R2, int V, float2 *stats, void *scratch,
                             cudaStream_t s) {
  const int nblk = blocks_of(V), R = R1 + R2;
  float2 *part = reinterpret_cast<float2 *>(scratch);
  cudaError_t e =
      launch_pdl(block_stats_kernel, unit_grid(R, nblk), dim3(UNIT_WARPS * 32), 0, s, z1, R1, z2, V, nblk, part);
  if (e != cudaSuccess) return e;
  e = launch_pdl(row_merge_kernel, dim3((unsigned)((R + ROW_WARPS - 1) / ROW_WARPS)), dim3(ROW_WARPS * 32), 0, s,
                 (const float2 *)part, R, nblk, stats);
  return e != cudaSuccess ? e : cudaGetLastError();
}

cudaError_t launch_softmax_write(const float *z, int R, int V, const float2 *stats, float *p, cudaStream_t s) {
  const int nblk = blocks_of(V);
  cudaError_t e = launch_pdl(softmax_write_kernel, unit_grid(R, nblk), dim3(UNIT_WARPS * 32), 0, s, z, V, nblk,
                             stats, p);
  return e != cudaSuccess ? e : cudaGetLastError();
}

static size_t draw_sums_bytes(int B, int V) { return align_up((size_t)B * blocks_of(V) * sizeof(uint64_t), 256); }

size_t draft_sample_scratch_bytes(int B, int V) { return draw_sums_bytes(B, V) + row_stats_scratch_bytes(B, V); }

cudaError_t launch_draft_sample(const float *z, int B, int V, const float *u, int32_t *tok, float2 *stats, float *q,
                                void *scratch, uint32_t *status, cudaStream_t s) {
  const int nblk = blocks_of(V);
  uint8_t *sc = static_cast<uint8_t *>(scratch);
  uint64_t *blk = reinterpret_cast<uint64_t *>(sc);
  cudaError_t e = launch_row_stats(z, B, nullptr, 0, V, stats, sc + draw_sums_bytes(B, V), s);
  if (e != cudaSuccess) return e;
  e = launch_pdl(draw_weights_kernel, unit_grid(B, nblk), dim3(UNIT_WARPS * 32), 0, s, z, V, nblk,
                 (const float2 *)stats, q, blk);
  if (e != cudaSuccess) return e;
  e = launch_pdl(draw_token_kernel, dim3((unsigned)((B + ROW_WARPS - 1) / ROW_WARPS)), dim3(ROW_WARPS * 32), 0, s, z,
                 B, V, nblk, (const float2 *)stats, (const uint64_t *)blk, u, tok, status);
  return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace mlora
