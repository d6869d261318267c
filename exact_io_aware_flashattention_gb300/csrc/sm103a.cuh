// Inline-PTX building blocks for the sm_103a attention kernels: mbarriers with
// bounded waits, TMA tensor loads, tcgen05 (TMEM allocation, MMA, commit,
// TMEM loads/stores, fences) and the shared-memory / instruction descriptors
// the MMAs read.
//
// Shared-memory operand layout used everywhere: a tile of R rows whose
// contiguous dimension is split into 64-element (128-byte) column blocks, each
// block stored as R rows of 128 bytes with the 128-byte swizzle (16-byte chunk
// c of row r lives at chunk c ^ (r % 8)).  This is exactly what a TMA load
// with CU_TENSOR_MAP_SWIZZLE_128B and a {64, R} box writes.  Such a tile is
// read by tcgen05.mma either
//   * K-major  (rows = M or N, contiguous = K): 8-row groups 1024 B apart, a
//     16-element K step is a 32-byte advance inside the 128-byte row and the
//     next 64-element block starts R*128 bytes later; or
//   * MN-major (rows = K, contiguous = M or N): LBO = distance between the
//     64-element MN blocks (R*128 bytes), SBO = 1024 B between 8-row K groups,
//     a 16-element K step is a 2048-byte advance.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_bf16.h>

namespace fa {

// ---------------------------------------------------------------------------
// Device status words shared by all kernels of the library.
//   [0] first error code (0 = none), [1] flattened block index,
//   [2] wait-site id, [3] thread index,
//   [4] wait-site id of the first failed drain (0 = none), [5] its block.
// A drain is the wait, on a kernel's way out, for the TMA copies and MMAs it
// has already issued; if one gives up, work may still be in flight when the
// block exits, so the host treats the device as unusable from then on.
// ---------------------------------------------------------------------------
constexpr int kStatusWords = 8;

struct DevStatus {
  int* words;            // device pointer to kStatusWords ints
  unsigned long long timeout_ns;
};

constexpr int kErrDeviceTimeout = 8;   // == FA_ERR_DEVICE_TIMEOUT

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ unsigned long long globaltimer_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ void record_error(const DevStatus& st, int code, int site) {
  if (atomicCAS(st.words, 0, code) == 0) {
    st.words[1] = (int)(blockIdx.x + gridDim.x * (blockIdx.y + gridDim.y * blockIdx.z));
    st.words[2] = site;
    st.words[3] = (int)threadIdx.x;
  }
}

// ---------------------------------------------------------------------------
// mbarrier
// ---------------------------------------------------------------------------
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_fence_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// Wait until the phase with the given parity has completed.  Gives up after
// st.timeout_ns, or as soon as another thread of the CTA has raised *abort;
// records the failure in the status words and returns false.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, const DevStatus& st,
                                          volatile int* abort, int site) {
  const uint32_t a = smem_u32(bar);
  if (mbar_try_wait(a, parity)) return true;
  const unsigned long long t0 = globaltimer_ns();
  for (uint32_t it = 1;; ++it) {
    if (mbar_try_wait(a, parity)) return true;
    if ((it & 63u) == 0) {
      if (*abort) return false;
      if (globaltimer_ns() - t0 > st.timeout_ns) {
        record_error(st, kErrDeviceTimeout, site);
        *abort = 1;
        return false;
      }
    }
  }
}

// Warp-collective form: every lane polls the barrier (bounded) and the warp
// proceeds only if all lanes saw the phase complete, so lanes never split
// across a later .sync.aligned instruction or warp vote.  Polling from one
// lane while the others wait at a shuffle was measured 3-9 % slower in the
// forward and up to 2x slower in an MMA-issuing warp: the wake-up after the
// phase completes is on the critical path of every tile.
__device__ __forceinline__ bool mbar_wait_warp(uint64_t* bar, uint32_t parity, const DevStatus& st,
                                               volatile int* abort, int site) {
  return __all_sync(0xffffffffu, mbar_wait(bar, parity, st, abort, site));
}

// Bounded wait that ignores the abort flag, used on a block's way out to let
// the copies and MMAs it issued complete.  If it gives up, the site is
// recorded in words [4] / [5] (the host then refuses further launches on the
// device) and the block goes on to exit.
__device__ __forceinline__ bool mbar_wait_drain(uint64_t* bar, uint32_t parity, const DevStatus& st, int site) {
  const uint32_t a = smem_u32(bar);
  const unsigned long long t0 = globaltimer_ns();
  for (uint32_t it = 0;; ++it) {
    if (mbar_try_wait(a, parity)) return true;
    if ((it & 63u) == 63u && globaltimer_ns() - t0 > st.timeout_ns) {
      if (atomicCAS(st.words + 4, 0, site) == 0)
        st.words[5] = (int)(blockIdx.x + gridDim.x * (blockIdx.y + gridDim.y * blockIdx.z));
      return false;
    }
  }
}

// ---------------------------------------------------------------------------
// Proxy / thread-sync fences
// ---------------------------------------------------------------------------
// Make generic-proxy writes to shared memory visible to the async proxy
// (tcgen05.mma operand reads, TMA).
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// ---------------------------------------------------------------------------
// TMA
// ---------------------------------------------------------------------------
// A tensor map of rank R.  The rank is part of the type so that a tiled copy
// instruction of one dimensionality can only be given a map encoded with the
// same number of dimensions: a mismatch does not compile, instead of making
// the copy unit fail at run time.
template <int R>
struct TmaMap {
  CUtensorMap m;
};
using TmaMap3 = TmaMap<3>;
using TmaMap4 = TmaMap<4>;

template <int R>
__device__ __forceinline__ void tma_prefetch_desc(const TmaMap<R>* m) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&m->m)) : "memory");
}

// 4-D tiled load {c0 = innermost, ...} into shared memory; completion is
// reported as transaction bytes on *bar.
__device__ __forceinline__ void tma_load_4d(void* dst, const TmaMap4* m, uint64_t* bar, int c0, int c1,
                                            int c2, int c3) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4, %5}], [%6];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(m)), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(smem_u32(bar))
      : "memory");
}

__device__ __forceinline__ void tma_load_3d(void* dst, const TmaMap3* m, uint64_t* bar, int c0, int c1, int c2) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(m)), "r"(c0), "r"(c1), "r"(c2), "r"(smem_u32(bar))
      : "memory");
}

// Tiled 3-D reduce-add of a shared-memory box into global memory (the tensor
// map's element type and reduction), tracked by this thread's bulk group.
__device__ __forceinline__ void tma_reduce_add_3d(const TmaMap3* m, uint32_t ssrc, int c0, int c1, int c2) {
  asm volatile(
      "cp.reduce.async.bulk.tensor.3d.global.shared::cta.add.tile.bulk_group [%0, {%1, %2, %3}], [%4];" ::"l"(
          reinterpret_cast<uint64_t>(m)),
      "r"(c0), "r"(c1), "r"(c2), "r"(ssrc)
      : "memory");
}

// Tiled 4-D store of a shared-memory box to global memory, tracked by this
// thread's bulk group (rows outside the tensor are not written).
__device__ __forceinline__ void tma_store_4d(const TmaMap4* m, uint32_t ssrc, int c0, int c1, int c2, int c3) {
  asm volatile("cp.async.bulk.tensor.4d.global.shared::cta.tile.bulk_group [%0, {%1, %2, %3, %4}], [%5];" ::"l"(
                   reinterpret_cast<uint64_t>(m)),
               "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(ssrc)
               : "memory");
}
__device__ __forceinline__ void bulk_commit_group() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
// Wait until at most kPending of this thread's most recent bulk groups are
// still reading shared memory.
template <int kPending>
__device__ __forceinline__ void bulk_wait_read() {
  asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(kPending) : "memory");
}
// Wait until this thread's bulk groups have fully completed.
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

// ---------------------------------------------------------------------------
// tcgen05: tensor memory
// ---------------------------------------------------------------------------
// Executed by one full warp; writes the TMEM base address to *slot.
__device__ __forceinline__ void tmem_alloc(uint32_t* slot, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(slot)),
               "r"(ncols)
               : "memory");
}
// Per-thread register budget of the executing warpgroup (all four warps of
// the warpgroup must execute the same instruction).  An increase waits until
// the registers released by other warpgroups of the CTA cover it, so the
// shares must add up to the launch allocation.
template <int kRegs>
__device__ __forceinline__ void setmaxnreg_inc() {
  asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kRegs));
}
template <int kRegs>
__device__ __forceinline__ void setmaxnreg_dec() {
  asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kRegs));
}
__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}

// D[tmem] (+)= A[smem] * B[smem]^T, bf16 inputs, fp32 accumulate.
__device__ __forceinline__ void mma_bf16_ss(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                            uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// D[tmem] (+)= A[tmem] * B[smem]^T: A (M x 16 bf16 per instruction) read from
// tensor memory, lane m = row m, two bf16 per 32-bit column (lower half =
// lower k).
__device__ __forceinline__ void mma_bf16_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc,
                                            uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// The same two MMAs for a converged warp: every lane executes the call and
// elect.sync picks one lane (the lowest, lane 0 of a full warp) to issue.
__device__ __forceinline__ void mma_bf16_ss_warp(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                                 uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p, e;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "elect.sync _|e, 0xffffffff;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}
__device__ __forceinline__ void mma_bf16_ts_warp(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc,
                                                 uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p, e;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "elect.sync _|e, 0xffffffff;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Arrive (once) on *bar when every tcgen05 async operation issued so far by
// this thread has completed.
__device__ __forceinline__ void mma_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                   smem_u32(bar))
               : "memory");
}

// mma_commit from the lane elect.sync picks in a converged warp (the lane
// that issued the warp's MMAs).
__device__ __forceinline__ void mma_commit_warp(uint64_t* bar) {
  asm volatile(
      "{\n\t.reg .pred e;\n\t"
      "elect.sync _|e, 0xffffffff;\n\t"
      "@e tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n\t}" ::"r"(smem_u32(bar))
      : "memory");
}

// An MMA-issuing role run by one lane (kWarp = false) or by a whole converged
// warp (kWarp = true: every lane polls the barriers, the warp agrees on the
// outcome, and elect.sync picks the lane that issues each MMA and commit).
template <bool kWarp>
__device__ __forceinline__ bool issuer_wait(uint64_t* bar, uint32_t parity, const DevStatus& st, volatile int* abort,
                                            int site) {
  bool r = mbar_wait(bar, parity, st, abort, site);
  if constexpr (kWarp) r = __all_sync(0xffffffffu, r);
  return r;
}
template <bool kWarp>
__device__ __forceinline__ void issue_ss(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc, uint32_t acc) {
  if constexpr (kWarp) mma_bf16_ss_warp(d, a, b, idesc, acc); else mma_bf16_ss(d, a, b, idesc, acc);
}
template <bool kWarp>
__device__ __forceinline__ void issue_ts(uint32_t d, uint32_t a, uint64_t b, uint32_t idesc, uint32_t acc) {
  if constexpr (kWarp) mma_bf16_ts_warp(d, a, b, idesc, acc); else mma_bf16_ts(d, a, b, idesc, acc);
}
template <bool kWarp>
__device__ __forceinline__ void issue_commit(uint64_t* bar) {
  if constexpr (kWarp) mma_commit_warp(bar); else mma_commit(bar);
}

// 32 lanes x 32 consecutive 32-bit columns: thread t of the warp receives lane
// (taddr.lane + t), columns taddr.col .. +31.  The warp must own the lane
// quadrant (warp_id % 4).
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
      "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]),
        "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]),
        "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]),
        "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
}

__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
      "{%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, "
      "%17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]),
      "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]), "r"(r[16]),
      "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]),
      "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])
      : "memory");
}

// 32 lanes x 16 consecutive 32-bit columns.
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t* r) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
      "{%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]),
      "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
      : "memory");
}

__device__ __forceinline__ void tmem_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }
__device__ __forceinline__ void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// Registers written by tcgen05.ld are only valid after tcgen05.wait::ld.  This
// empty volatile asm, placed after the wait, makes every later use of the
// registers depend on a point after the wait.
template <int N>
__device__ __forceinline__ void reg_fence(uint32_t (&r)[N]) {
#pragma unroll
  for (int i = 0; i < N; ++i) asm volatile("" : "+r"(r[i]));
}

// ---------------------------------------------------------------------------
// Descriptors
// ---------------------------------------------------------------------------
// Shared-memory matrix descriptor, 128-byte swizzle.
__device__ __forceinline__ uint64_t sdesc_sw128(uint32_t saddr, uint32_t lbo_bytes, uint32_t sbo_bytes) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr & 0x3FFFFu) >> 4);
  d |= (uint64_t)((lbo_bytes >> 4) & 0x3FFFu) << 16;
  d |= (uint64_t)((sbo_bytes >> 4) & 0x3FFFu) << 32;
  d |= (uint64_t)1 << 46;  // descriptor version for tcgen05
  d |= (uint64_t)2 << 61;  // swizzle mode: 128 B
  return d;
}

// Instruction descriptor for kind::f16 with bf16 A/B and fp32 D.
__host__ __device__ constexpr uint32_t idesc_bf16(int M, int N, bool a_mn_major, bool b_mn_major) {
  return (1u << 4)                              // D: f32
         | (1u << 7)                            // A: bf16
         | (1u << 10)                           // B: bf16
         | ((a_mn_major ? 1u : 0u) << 15)       // A major-ness
         | ((b_mn_major ? 1u : 0u) << 16)       // B major-ness
         | ((uint32_t)(N >> 3) << 17)           // N / 8
         | ((uint32_t)(M >> 4) << 24);          // M / 16
}

// K-major operand: k16-th 16-element step of a tile with 64-element column
// blocks of `block_bytes` each.
__device__ __forceinline__ uint64_t desc_kmajor(uint32_t tile_addr, int k16, uint32_t block_bytes) {
  return sdesc_sw128(tile_addr + (uint32_t)(k16 >> 2) * block_bytes + (uint32_t)(k16 & 3) * 32u, 16u, 1024u);
}
// MN-major operand: k16-th 16-row step of a tile whose MN dimension is split
// into 64-element blocks `block_bytes` apart.
__device__ __forceinline__ uint64_t desc_mnmajor(uint32_t tile_addr, int k16, uint32_t block_bytes) {
  return sdesc_sw128(tile_addr + (uint32_t)k16 * 2048u, block_bytes, 1024u);
}
// Start-address offset (16-byte units) of k16 step `k16` inside a 128-byte
// swizzled operand tile: the descriptor of the step is the tile's k16 = 0
// descriptor plus this constant (the address field cannot overflow: shared
// memory addresses stay below 2^18).
__host__ __device__ constexpr uint64_t desc_step_kmajor(int k16, uint32_t block_bytes) {
  return (uint64_t)(((uint32_t)(k16 >> 2) * block_bytes + (uint32_t)(k16 & 3) * 32u) >> 4);
}
__host__ __device__ constexpr uint64_t desc_step_mnmajor(int k16) { return (uint64_t)((uint32_t)k16 * 2048u >> 4); }

// ---------------------------------------------------------------------------
// Math helpers
// ---------------------------------------------------------------------------
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Packed fp32 pairs (sm_100+ f32x2 arithmetic): one instruction, two lanes.
__device__ __forceinline__ uint64_t f2pack(float lo, float hi) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
__device__ __forceinline__ void f2unpack(uint64_t v, float& lo, float& hi) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
__device__ __forceinline__ uint64_t ffma2(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t d;
  asm("fma.rn.ftz.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}
__device__ __forceinline__ uint64_t fadd2(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("add.rn.ftz.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ uint64_t fmul2(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("mul.rn.ftz.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
// Three-input max.
__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}
// Two fp32 -> packed bf16x2 (round to nearest even), `lo` in the low half.
__device__ __forceinline__ uint32_t cvt_bf16x2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}


// 32-byte global store; `p` must be 32-byte aligned.
__device__ __forceinline__ void st_global_v8(void* p, const uint32_t* w) {
  asm volatile("st.global.v8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"l"(p), "r"(w[0]), "r"(w[1]), "r"(w[2]),
               "r"(w[3]), "r"(w[4]), "r"(w[5]), "r"(w[6]), "r"(w[7])
               : "memory");
}
__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
  asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c), "r"(d)
               : "memory");
}

// Byte offset of 16-byte chunk `c16` (0..7) of row `r` inside one 128-byte
// swizzled column block.
__device__ __forceinline__ uint32_t swz128(int r, int c16) {
  return (uint32_t)r * 128u + (uint32_t)((c16 ^ (r & 7)) << 4);
}

}  // namespace fa
