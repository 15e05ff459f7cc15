// Shared device helpers: workspace layout, status word, bounded waits and the
// hand-written inline-PTX wrappers for mbarrier, TMA (cp.async.bulk.tensor)
// and the fifth-generation tensor cores (tcgen05.*, tensor memory).
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/mlora.h"

namespace mlora {

// ---------------------------------------------------------------------------
// Workspace layout (bytes).  Header and counters sit at fixed offsets so that
// every operation can share one workspace; each kernel that bumps a counter
// puts it back to zero before it exits.
// ---------------------------------------------------------------------------
constexpr size_t WS_STATUS_OFF = 0;           // uint32 status bits
constexpr size_t WS_COUNTERS_OFF = 4096;      // uint32 [WS_MAX_COUNTERS]
constexpr size_t WS_MAX_COUNTERS = 65536;
constexpr size_t WS_SCRATCH_OFF = WS_COUNTERS_OFF + 4 * WS_MAX_COUNTERS;  // 266240
constexpr size_t WS_INIT_BYTES = WS_SCRATCH_OFF;

constexpr int T_STRIDE = 64;                  // row stride of the internal fp32 T buffer

__host__ __device__ constexpr size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

// Shrink work items: (adapter, block of SHRINK_J rank rows, chunk of SHRINK_TOK
// rows), one 32-byte record each: {adapter, j0 | nrow << 8 | ntok << 16,
// sorted position of the first token, first expand block of the adapter},
// then the four token rows (original row indices).
constexpr int SHRINK_J = 8;
constexpr int SHRINK_TOK = 4;
constexpr int ITEM_WORDS = 8;

// Upper bound on shrink items for M rows and n_ad adapters (rank <= 64).
__host__ __device__ inline size_t max_shrink_items(int M, int n_ad) {
  const int m_ad = M < n_ad ? M : n_ad;
  return (size_t)(64 / SHRINK_J) * ((M + SHRINK_TOK - 1) / SHRINK_TOK + m_ad);
}

// Upper bound on expand blocks, (adapter, 16-rank block) pairs: at most
// min(M, n_ad) active adapters of rank <= 64.
__host__ __device__ inline int max_expand_slices(int M, int n_ad) { return (M < n_ad ? M : n_ad) * 4; }

// Expand blocks and their token windows.  In verify mode the GEMM reads the
// token rows in adapter-sorted order, so the rows of adapter a occupy the
// contiguous sorted positions [s0, s1) and, in tensor memory, the
// accumulator columns of those positions.  The window of a is [w0, w0 + W)
// with w0 = s0 rounded down and w0 + W = s1 rounded up to 16 (the MMA's
// column granularity); each of its 16-rank blocks gets its own copy of the
// window in the low-rank operand buffer, W rows of 16 bf16: scale * T on
// a's rows, 0 on the rows of the neighbouring adapters the rounding takes
// in.  A block's record in the plan is EXP_WORDS int32:
//   {adapter, first rank j0, rank columns in the block (1..16),
//    first row of its window in the operand buffer, w0, W, 0, 0}.
constexpr int EXP_WORDS = 8;

// Rows of the operand buffer (per output slice): every active adapter has at
// most 4 blocks and a window of at most s_a + 30 rows.
__host__ __device__ inline size_t max_window_rows(int M, int n_ad) {
  const int m_ad = M < n_ad ? M : n_ad;
  return (size_t)4 * ((size_t)M + 32 * (size_t)m_ad);
}

// Plan layout inside scratch (int32 words), for M rows and n_ad adapters.
struct PlanLayout {
  size_t hdr;         // [0] n_active, [1] shrink items, [2] rows, [3] largest active rank,
                      // [4] expand blocks (adapter, 16-rank block) over the active adapters,
                      // [5] 1 if every active rank is a multiple of 16 or r_max,
                      // [6] window rows of one slice's operand buffer
  size_t seg_offsets; // [n_ad + 2]
  size_t perm;        // [M]
  size_t row_adapter; // [M]   validated adapter per row (-1: none)
  size_t rank_eff;    // [n_ad] validated ranks
  size_t active;      // [n_ad] adapters with rows, increasing
  size_t item_off;    // [n_ad + 1] prefix of shrink items over the active list
  size_t slice_off;   // [n_ad] first expand block of each adapter
  size_t slices;      // [max_expand_slices][EXP_WORDS] expand block records
  size_t items;       // [max_shrink_items][ITEM_WORDS], 16-byte aligned
  size_t words;       // total int32 words
};

__host__ __device__ inline PlanLayout plan_layout(int M, int n_ad) {
  PlanLayout L;
  size_t o = 0;
  L.hdr = o;          o += 16;
  L.seg_offsets = o;  o += align_up(n_ad + 2, 16);
  L.perm = o;         o += align_up(M, 16);
  L.row_adapter = o;  o += align_up(M, 16);
  L.rank_eff = o;     o += align_up(n_ad, 16);
  L.active = o;       o += align_up(n_ad, 16);
  L.item_off = o;     o += align_up(n_ad + 1, 16);
  L.slice_off = o;    o += align_up(n_ad, 16);
  L.slices = o;       o += align_up((size_t)max_expand_slices(M, n_ad) * EXP_WORDS, 16);
  L.items = o;        o += max_shrink_items(M, n_ad) * ITEM_WORDS;
  L.words = o;
  return L;
}

// ---------------------------------------------------------------------------
// Status word
// ---------------------------------------------------------------------------
__device__ __forceinline__ void raise_status(uint32_t *status, uint32_t bits) {
  if (status) atomicOr(status, bits);
}

// Bounded waits give up after this long and raise MLORA_DEV_TIMEOUT.
constexpr uint64_t WAIT_LIMIT_NS = 500ull * 1000ull * 1000ull;

__device__ __forceinline__ uint64_t global_timer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// ---------------------------------------------------------------------------
// Shared-memory addresses, mbarrier
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_addr(const void *p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// The first 1024-byte aligned byte of a dynamic shared-memory array (the
// 128-byte swizzle patterns repeat every 1024 bytes).  Offsetting the array
// itself keeps the pointer in the shared window for the compiler, so
// accesses through it are shared-memory instructions, not generic ones.
__device__ __forceinline__ uint8_t *align_smem_1024(uint8_t *smem_base) {
  return smem_base + ((1024u - (smem_addr(smem_base) & 1023u)) & 1023u);
}

__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}

// Test the phase; if it is not complete the thread may be suspended (it does
// not take issue slots) for up to MBAR_SUSPEND_NS or until the phase completes.
constexpr uint32_t MBAR_SUSPEND_NS = 20000;

__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity) {
  uint32_t done;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(done)
      : "r"(smem_addr(bar)), "r"(parity), "r"(MBAR_SUSPEND_NS)
      : "memory");
  return done != 0;
}

// Wait for the phase of `bar` with parity `parity` to complete.  Gives up
// (returns false) after WAIT_LIMIT_NS or as soon as *abort is set.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t *bar, uint32_t parity, volatile int *abort) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  while (true) {
    if (mbar_try_wait(bar, parity)) return true;
    if (*abort) return false;
    if (global_timer_ns() - t0 > WAIT_LIMIT_NS) return false;
  }
}

// ---------------------------------------------------------------------------
// TMA (tensor memory accelerator) loads
// ---------------------------------------------------------------------------
__device__ __forceinline__ void tma_prefetch_desc(const CUtensorMap *map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// Contiguous copy of `bytes` (a multiple of 16; both addresses 16-byte
// aligned) from global to shared memory; completion as transaction bytes.
__device__ __forceinline__ void bulk_load(void *smem_dst, const void *src, uint32_t bytes, uint64_t *bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                   smem_addr(smem_dst)),
               "l"(src), "r"(bytes), "r"(smem_addr(bar))
               : "memory");
}

// Generic-proxy accesses to global memory made visible (for example by an
// acquire) are ordered before this thread's later async-proxy (bulk copy)
// accesses.
__device__ __forceinline__ void fence_proxy_async_global() {
  asm volatile("fence.proxy.async.global;" ::: "memory");
}

// 2-D tiled load of the box at (c0 = inner coordinate, c1 = row) into shared
// memory; completion is signalled on `bar` as transaction bytes.
__device__ __forceinline__ void tma_load_2d(void *smem_dst, const CUtensorMap *map, uint64_t *bar, int c0, int c1,
                                            uint64_t cache_policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%3, %4}], [%2], %5;" ::"r"(smem_addr(smem_dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_addr(bar)), "r"(c0), "r"(c1), "l"(cache_policy)
      : "memory");
}

// 3-D tiled load of the box at (c0 = inner coordinate, c1, c2).
__device__ __forceinline__ void tma_load_3d(void *smem_dst, const CUtensorMap *map, uint64_t *bar, int c0, int c1,
                                            int c2, uint64_t cache_policy) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%3, %4, %5}], [%2], %6;" ::"r"(smem_addr(smem_dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_addr(bar)), "r"(c0), "r"(c1), "r"(c2), "l"(cache_policy)
      : "memory");
}

__device__ __forceinline__ uint64_t policy_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}

__device__ __forceinline__ uint64_t policy_evict_last() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
  return p;
}

// ---------------------------------------------------------------------------
// tcgen05: tensor memory and the fifth-generation MMA
// ---------------------------------------------------------------------------
__device__ __forceinline__ void tmem_alloc(uint32_t *smem_result, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_addr(smem_result)),
               "r"(ncols)
               : "memory");
}

__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}

__device__ __forceinline__ void tc_fence_before_sync() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}

__device__ __forceinline__ void tc_fence_after_sync() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// D[tmem] (+)= A[smem] * B[smem]^T, bf16 inputs, fp32 accumulator, one CTA.
__device__ __forceinline__ void mma_bf16_ss(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                            uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// D[tmem] (+)= A[smem] * B[smem]^T, E4M3 inputs (kind::f8f6f4, K = 32 per
// instruction: 32 bytes of each operand row, as kind::f16's 16 bf16), fp32
// accumulator, one CTA.
__device__ __forceinline__ void mma_e4m3_ss(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                            uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Arrive on `bar` once every tcgen05 operation this thread issued so far is done.
__device__ __forceinline__ void mma_commit(uint64_t *bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                   smem_addr(bar))
               : "memory");
}

// Shared-memory matrix descriptor for a K-major operand tile whose rows are
// 128 bytes (64 bf16) written by TMA with 128-byte swizzling: groups of 8 rows
// are 1024 bytes apart (stride byte offset), the leading byte offset is unused
// for this layout, descriptor version 1, swizzle mode 2 (128 B).
__device__ __forceinline__ uint64_t smem_desc_kmajor_sw128(uint32_t saddr) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr & 0x3FFFFu) >> 4);    // start address
  d |= (uint64_t)1 << 16;                       // leading byte offset (16 B, unused)
  d |= (uint64_t)(1024 >> 4) << 32;             // stride byte offset
  d |= (uint64_t)1 << 46;                       // descriptor version
  d |= (uint64_t)2 << 61;                       // 128-byte swizzle
  return d;
}

// Shared-memory matrix descriptor for a K-major operand tile whose rows are
// 32 bytes (16 bf16) written by TMA with 32-byte swizzling: groups of 8 rows
// are 256 bytes apart, descriptor version 1, swizzle mode 6 (32 B).  One MMA
// K step (16 bf16) spans the whole row.
__device__ __forceinline__ uint64_t smem_desc_kmajor_sw32(uint32_t saddr) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr & 0x3FFFFu) >> 4);
  d |= (uint64_t)1 << 16;
  d |= (uint64_t)(256 >> 4) << 32;
  d |= (uint64_t)1 << 46;
  d |= (uint64_t)6 << 61;
  return d;
}

// Instruction descriptor: kind::f16 with bf16 A and B, fp32 D, both operands
// K-major, shape M x N (M = 128, N % 16 == 0, 16 <= N <= 256).
__host__ __device__ constexpr uint32_t idesc_bf16_f32(int M, int N) {
  return (1u << 4)                          // D format: f32
         | (1u << 7)                        // A format: bf16
         | (1u << 10)                       // B format: bf16
         | ((uint32_t)(N >> 3) << 17)       // N / 8
         | ((uint32_t)(M >> 4) << 24);      // M / 16
}

// Instruction descriptor: kind::f8f6f4 with E4M3 A and B (format code 0),
// fp32 D, both operands K-major, shape M x N as for idesc_bf16_f32.
__host__ __device__ constexpr uint32_t idesc_e4m3_f32(int M, int N) {
  return (1u << 4)                          // D format: f32
         | (0u << 7)                        // A format: e4m3
         | (0u << 10)                       // B format: e4m3
         | ((uint32_t)(N >> 3) << 17)       // N / 8
         | ((uint32_t)(M >> 4) << 24);      // M / 16
}

// tensor memory -> registers: 32 lanes x 32 bit, repeated along columns.
__device__ __forceinline__ void tmem_ld_x1(uint32_t taddr, uint32_t &r0) {
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x1.b32 {%0}, [%1];" : "=r"(r0) : "r"(taddr));
}

__device__ __forceinline__ void tmem_ld_x16(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
}

__device__ __forceinline__ void tmem_ld_x32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
        "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
        "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
}

__device__ __forceinline__ void tmem_ld_wait() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

// ---------------------------------------------------------------------------
// Thread-block clusters: barrier and distributed shared memory
// ---------------------------------------------------------------------------
__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release;\n\tbarrier.cluster.wait.acquire;" ::: "memory");
}

__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

// Shared-memory address of the same variable in CTA `rank` of this cluster.
__device__ __forceinline__ uint32_t map_to_rank(uint32_t saddr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(saddr), "r"(rank));
  return r;
}

__device__ __forceinline__ float ld_dsmem_f32(uint32_t caddr) {
  float v;
  asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(caddr) : "memory");
  return v;
}

// 16 bytes from a peer CTA's shared memory (caddr 16-byte aligned).
__device__ __forceinline__ float4 ld_dsmem_f32x4(uint32_t caddr) {
  float4 v;
  asm volatile("ld.shared::cluster.v4.f32 {%0, %1, %2, %3}, [%4];"
               : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
               : "r"(caddr)
               : "memory");
  return v;
}

// Programmatic dependent launch: wait for the preceding grid's memory, and
// allow the next grid in the stream to begin launching.
__device__ __forceinline__ void grid_dependency_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void grid_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// CTA barrier reached by converged warps: bar.sync counts whole warps, so a
// warp whose lanes are still on different paths (one lane finishing a
// single-thread block) is first brought back together.
__device__ __forceinline__ void block_sync() {
  __syncwarp();
  __syncthreads();
}

// Named barrier over `nthreads` threads (ids 1..15; 0 is __syncthreads).
__device__ __forceinline__ void named_bar_sync(int id, int nthreads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

// Arrive on named barrier `id` without waiting (the waiters use bar.sync).
__device__ __forceinline__ void named_bar_arrive(int id, int nthreads) {
  asm volatile("bar.arrive %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

// Named barrier that also ANDs a predicate over its `nthreads` threads.
__device__ __forceinline__ bool named_bar_and(int id, int nthreads, bool pred) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.b32 p, %1, 0;\n\t"
      "bar.red.and.pred q, %2, %3, p;\n\t"
      "selp.u32 %0, 1, 0, q;\n\t}"
      : "=r"(r)
      : "r"((uint32_t)pred), "r"(id), "r"(nthreads)
      : "memory");
  return r != 0;
}

// Flags between CTAs of one grid: a release store after the data it
// publishes, an acquire load before the data is read.
__device__ __forceinline__ void st_release_gpu(uint32_t *p, uint32_t v) {
  asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

__device__ __forceinline__ void atomic_add_release_gpu(uint32_t *p, uint32_t v) {
  asm volatile("red.release.gpu.global.add.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

__device__ __forceinline__ uint32_t ld_acquire_gpu(const uint32_t *p) {
  uint32_t v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

// Shared-memory writes by threads become visible to the tensor cores (the
// async proxy) that read the same bytes as an MMA operand.
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void sleep_ns(uint32_t ns) { asm volatile("nanosleep.u32 %0;" ::"r"(ns)); }

__device__ __forceinline__ float bf16_bits_to_float(uint16_t b) { return __uint_as_float(((uint32_t)b) << 16); }

__device__ __forceinline__ uint16_t float_to_bf16_bits(float f) {
  return __bfloat16_as_ushort(__float2bfloat16_rn(f));
}

}  // namespace mlora
