// Thin inline-PTX wrappers for the sm_103a features the attention kernels use:
// mbarriers, TMA tiled bulk copies, tcgen05 MMA with TMEM accumulators, TMEM
// loads/stores, and the shared-memory matrix / instruction descriptors of the
// 5th-generation tensor cores.  Every wait here is bounded: it gives up after a
// wall-clock limit, records an error code in a device word and returns false,
// so a lost arrival can never hang the GPU.
#pragma once
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

namespace fa {

// ---------------------------------------------------------------- error word
// Bits written into the device error word by a kernel that gave up waiting.
enum : uint32_t {
  kErrTimeoutTma = 1u << 0,       // a consumer waited too long for a TMA tile
  kErrTimeoutMma = 1u << 1,       // a waiter never saw a tensor-core commit
  kErrTimeoutSoftmax = 1u << 2,   // the MMA issuer never saw elementwise output
  kErrTimeoutRing = 1u << 3,      // the producer never got a free ring slot
  kErrTimeoutSync = 1u << 4,      // a warpgroup barrier never completed
  kErrSelfTest = 1u << 5,         // the failure-detection self-test's wait (expected to give up)
  kErrDebugCheck = 1u << 6,       // FA_DEBUG builds: a bounds, alignment or phase check failed
  kErrAborted = 1u << 31,         // set with the first failure: every later wait gives up at once
};

// What a failed FA_DEBUG check was about (err[1] = kDbgBase | kind when it is the
// first failure; err[3] then holds the offending value).
enum : uint32_t {
  kDbgBase = 0x100u,
  kDbgTmaCol = 1,      // TMA box column not a multiple of 64 or outside the head dimension
  kDbgTmaRow = 2,      // TMA box row outside [0, rows rounded up to 128)
  kDbgTmaPlane = 3,    // TMA box plane outside [0, planes)
  kDbgTmemCol = 4,     // TMEM access past the 512 allocated columns
  kDbgTmemLane = 5,    // TMEM lane quarter outside the 128 lanes
  kDbgBulk = 6,        // bulk copy source outside its row vector
  kDbgPhase = 7,       // an mbarrier ended the CTA with a phase count of the wrong parity
};

#ifdef FA_DEBUG
constexpr bool kDebug = true;
#else
constexpr bool kDebug = false;
#endif

// Device error record: [0] the bits above; [1] the code of the first failure;
// [2] its CTA index; [3] its barrier's shared-memory offset.

constexpr uint64_t kWaitLimitNs = 4000000000ull;  // 4 s of wall clock per wait
__device__ __forceinline__ uint64_t globaltimer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// ---------------------------------------------------------------- CTA order
// Linear CTA index -> (block, head) with heads taken in groups of G: every block of
// heads [g G, g G + G) comes before those of the next group, and inside a group the
// block index changes slowest (callers map a low block index to their heaviest
// block).  A bijection for any G >= 1.
__device__ __forceinline__ void grouped_tile(unsigned idx, int nheads, int nblocks, int G, int& blk, int& head) {
  G = max(1, min(G, nheads));
  const unsigned per = (unsigned)G * (unsigned)nblocks;
  const int g = (int)(idx / per);
  const unsigned rem = idx - (unsigned)g * per;
  const int g0 = g * G;
  const int gg = min(G, nheads - g0);
  blk = (int)(rem / (unsigned)gg);
  head = g0 + (int)(rem % (unsigned)gg);
}

// ---------------------------------------------------------------- mbarrier
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}
__device__ __forceinline__ uint32_t mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n"
      " mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
      " selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok;
}
// Wait for the phase with the given parity to complete.  Returns false (after
// recording `code` in the error record err[0..3]) if it did not complete within
// kWaitLimitNs, or at once if another wait of any CTA has already given up (the
// abort bit), so a failure ends the kernel quickly instead of hanging it.
// Records a wait that gave up: the first failure's code, CTA and barrier, then
// the abort bit that makes every other wait of the grid give up at once.  Out of
// line: it runs at most once per thread and keeps the hot wait loops small.
static __device__ __noinline__ void record_timeout(uint32_t* err, uint32_t code, uint32_t bar) {
  if (!err) return;
  if (atomicCAS(err + 1, 0u, code) == 0u) {
    err[2] = blockIdx.x;
    err[3] = bar;
  }
  atomicOr(err, code | kErrAborted);
}

// Records a failed FA_DEBUG check: the first failure's code, CTA and value, and
// the check bit.  It does not set the abort bit: the caller clamps the access to
// a safe value and the kernel runs on, so one launch reports every kind of slip.
static __device__ __noinline__ void record_check(uint32_t* err, uint32_t kind, uint32_t value) {
  if (!err) return;
  if (atomicCAS(err + 1, 0u, kDbgBase | kind) == 0u) {
    err[2] = blockIdx.x;
    err[3] = value;
  }
  atomicOr(err, kErrDebugCheck);
}

#ifdef FA_DEBUG
// Per-CTA context of the TMEM checks (debug builds only): the allocation's base
// address and the error record.  Each kernel sets them once, right after its
// TMEM allocation (debug_context).
static __shared__ uint32_t dbg_tmem_base;
static __shared__ uint32_t* dbg_err_ptr;
#endif

// The final drain of a CTA's tensor-core work passes honor_abort = false: it
// always waits (bounded) for the MMAs already issued before TMEM is released.
// `err` must point at the device error record.
__device__ __forceinline__ bool mbar_wait_for(uint32_t bar, uint32_t parity, uint32_t* err, uint32_t code,
                                              bool honor_abort, uint64_t limit_ns) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  for (uint32_t n = 0;; ++n) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((n & 63) == 63) {
      if (honor_abort && (*reinterpret_cast<volatile uint32_t*>(err) & kErrAborted)) return false;
      if (globaltimer_ns() - t0 > limit_ns) {
        record_timeout(err, code, bar);
        return false;
      }
    }
  }
}
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, uint32_t* err, uint32_t code,
                                          bool honor_abort = true) {
  return mbar_wait_for(bar, parity, err, code, honor_abort, kWaitLimitNs);
}

// Warp-uniform bounded wait: every lane waits, and every lane sees a failure if
// any lane's wait gave up, so a warp never splits between the two paths (a later
// warp-wide operation would otherwise wait for lanes that left).
__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, uint32_t* err, uint32_t code) {
  return __all_sync(0xffffffffu, mbar_wait(bar, parity, err, code));
}
// One arrival per warp (the barrier counts warps): __syncwarp orders every lane's
// earlier operations, fences included, before lane 0's arrive.  Arriving threads
// contend for one shared-memory word, so a warp arrives once, not 32 times.
__device__ __forceinline__ void warp_arrive(uint32_t bar) {
  __syncwarp();
  if ((threadIdx.x & 31) == 0) mbar_arrive(bar);
}

// A barrier among `count` threads built on an mbarrier, so that its wait is
// bounded like every other wait: each thread arrives, then waits for the phase.
struct SmemSync {
  uint32_t bar;
  uint32_t phase;
  __device__ __forceinline__ bool sync(uint32_t* err) {
    mbar_arrive(bar);
    const bool ok = mbar_wait(bar, phase, err, kErrTimeoutSync);
    phase ^= 1u;
    return ok;
  }
};

// ---------------------------------------------------------------- proxies / barriers
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
__device__ __forceinline__ void named_bar_sync(uint32_t id, uint32_t nthreads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

// ---------------------------------------------------------------- TMA
__device__ __forceinline__ void tma_prefetch_desc(const CUtensorMap* m) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(m)) : "memory");
}
// 3-D tiled load of one box into shared memory, completing `bar`'s transaction count.
__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap* m, uint32_t bar,
                                            int c0, int c1, int c2) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(m)), "r"(bar), "r"(c0), "r"(c1), "r"(c2)
      : "memory");
}
// Contiguous copy of `bytes` (a multiple of 16; both addresses 16-byte aligned)
// from global to shared memory, completing `bytes` transactions on `bar`.
__device__ __forceinline__ void bulk_load(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
               "l"(src), "r"(bytes), "r"(bar)
               : "memory");
}
// 3-D tiled store of one box from shared memory (rows outside the tensor are dropped).
__device__ __forceinline__ void tma_store_3d(const CUtensorMap* m, uint32_t src, int c0, int c1, int c2) {
  asm volatile(
      "cp.async.bulk.tensor.3d.global.shared::cta.tile.bulk_group [%0, {%2, %3, %4}], [%1];" ::"l"(
          reinterpret_cast<uint64_t>(m)),
      "r"(src), "r"(c0), "r"(c1), "r"(c2)
      : "memory");
}
__device__ __forceinline__ void tma_store_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
__device__ __forceinline__ void tma_store_wait_read0() {
  asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}
__device__ __forceinline__ void tma_store_wait0() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

// ---------------------------------------------------------------- tcgen05: TMEM
// FA_DEBUG builds: a TMEM address (lane quarter in bits 16-31, column in 0-15) and
// the columns an access spans, against the CTA's 512 allocated columns and 128
// lanes; a failure is recorded and the access goes to the allocation's base.
// Identity otherwise.
__device__ __forceinline__ uint32_t tm(uint32_t taddr, uint32_t ncols) {
#ifdef FA_DEBUG
  const uint32_t base = dbg_tmem_base;
  const uint32_t col = (taddr & 0xFFFFu) - (base & 0xFFFFu), lane = (taddr >> 16) - (base >> 16);
  if (col + ncols > 512u) {
    record_check(dbg_err_ptr, kDbgTmemCol, col);
    return base;
  }
  if (lane >= 128u || (lane & 31u)) {
    record_check(dbg_err_ptr, kDbgTmemLane, lane);
    return base;
  }
#endif
  return taddr;
}
// Sets the TMEM check context; every thread of the CTA calls it after reading the
// allocation's base (it synchronizes the CTA in FA_DEBUG builds, nothing otherwise).
__device__ __forceinline__ void debug_context(uint32_t tmem_base, uint32_t* err) {
#ifdef FA_DEBUG
  if (threadIdx.x == 0) {
    dbg_tmem_base = tmem_base;
    dbg_err_ptr = err;
  }
  __syncthreads();
#endif
}

__device__ __forceinline__ void tmem_alloc(uint32_t dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem), "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

__device__ __forceinline__ void tmem_ld_32x32b_x32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
               : "r"(tm(taddr, 32)));
}
__device__ __forceinline__ void tmem_st_32x32b_x32(uint32_t taddr, const uint32_t (&r)[32]) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32};"
               :: "r"(tm(taddr, 32)), "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]), "r"(r[16]), "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])
               : "memory");
}
__device__ __forceinline__ void tmem_st_32x32b_x16(uint32_t taddr, const uint32_t (&r)[16]) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16};"
               :: "r"(tm(taddr, 16)), "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
                  "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
               : "memory");
}
__device__ __forceinline__ void tmem_st_32x32b_x4(uint32_t taddr, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x4.b32 [%0], {%1, %2, %3, %4};" ::"r"(tm(taddr, 4)), "r"(a), "r"(b), "r"(c),
               "r"(d)
               : "memory");
}
__device__ __forceinline__ void tmem_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }
__device__ __forceinline__ void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }
// Ties the registers of a finished tcgen05.ld to program order after the wait,
// so no use of them can be scheduled before the data has arrived.
__device__ __forceinline__ void reg_fence32(uint32_t (&r)[32]) {
  asm volatile("" : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]), "+r"(r[6]), "+r"(r[7]), "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]), "+r"(r[12]), "+r"(r[13]), "+r"(r[14]), "+r"(r[15]), "+r"(r[16]), "+r"(r[17]), "+r"(r[18]), "+r"(r[19]), "+r"(r[20]), "+r"(r[21]), "+r"(r[22]), "+r"(r[23]), "+r"(r[24]), "+r"(r[25]), "+r"(r[26]), "+r"(r[27]), "+r"(r[28]), "+r"(r[29]), "+r"(r[30]), "+r"(r[31]) :: "memory");
}

// ---------------------------------------------------------------- tcgen05: MMA
// Accumulator columns an MMA writes: N, from bits 17-22 of the instruction descriptor.
__device__ __forceinline__ uint32_t idesc_n(uint32_t idesc) { return ((idesc >> 17) & 0x3Fu) << 3; }
// D[tmem] (+)= A[smem] * B[smem], kind::f16 (fp16 or bf16 inputs, fp32 accumulate).
__device__ __forceinline__ void mma_ss(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                       uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(tm(d_tmem, idesc_n(idesc))),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// D[tmem] (+)= A[tmem] * B[smem], kind::f16.  A (M x 16 per instruction) is read
// from TMEM: lane i holds row i, each 32-bit column two consecutive K elements.
__device__ __forceinline__ void mma_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc,
                                       uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n}\n" ::"r"(tm(d_tmem, idesc_n(idesc))),
      "r"(tm(a_tmem, 8)), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// The same MMAs with the shared-memory descriptors passed as (low, high) 32-bit
// halves.  The high half (stride, version, swizzle) is fixed per operand layout and
// the low half (start address, leading offset) advances by an immediate per K
// step, so issuing an MMA costs a couple of integer adds, not a descriptor build.
__device__ __forceinline__ void mma_ss_lohi(uint32_t d_tmem, uint32_t a_lo, uint32_t a_hi, uint32_t b_lo,
                                            uint32_t b_hi, uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n .reg .b64 a, b;\n setp.ne.b32 p, %6, 0;\n"
      " mov.b64 a, {%1, %2};\n mov.b64 b, {%3, %4};\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], a, b, %5, p;\n}\n" ::"r"(tm(d_tmem, idesc_n(idesc))),
      "r"(a_lo), "r"(a_hi), "r"(b_lo), "r"(b_hi), "r"(idesc), "r"(accumulate)
      : "memory");
}
__device__ __forceinline__ void mma_ts_lohi(uint32_t d_tmem, uint32_t a_tmem, uint32_t b_lo, uint32_t b_hi,
                                            uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n .reg .b64 b;\n setp.ne.b32 p, %5, 0;\n mov.b64 b, {%2, %3};\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], b, %4, p;\n}\n" ::"r"(tm(d_tmem, idesc_n(idesc))),
      "r"(tm(a_tmem, 8)), "r"(b_lo), "r"(b_hi), "r"(idesc), "r"(accumulate)
      : "memory");
}
// Low and high halves of the 128-byte-swizzle descriptor (see make_sdesc_sw128).
__host__ __device__ constexpr uint32_t sdesc_hi_sw128(uint32_t sbo_bytes) {
  return ((sbo_bytes >> 4) & 0x3FFFu) | (1u << 14) | (2u << 29);
}
__device__ __forceinline__ uint32_t sdesc_lo(uint32_t saddr, uint32_t lbo_bytes) {
  return ((saddr >> 4) & 0x3FFFu) | (((lbo_bytes >> 4) & 0x3FFFu) << 16);
}

// Arrive once on `bar` when every tcgen05 operation this thread issued so far has completed.
__device__ __forceinline__ void mma_commit(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
               : "memory");
}

// Instruction descriptor for kind::f16 with fp32 accumulation.
//   bits 4-5 accumulator format (1 = f32), 7-9 A format, 10-12 B format
//   (0 = f16, 1 = bf16), bit 15 A is MN-major, bit 16 B is MN-major,
//   bits 17-22 N/8, bits 24-28 M/16.
__host__ __device__ constexpr uint32_t make_idesc_f16(bool bf16, int M, int N, bool a_mn_major, bool b_mn_major) {
  return (1u << 4) | ((bf16 ? 1u : 0u) << 7) | ((bf16 ? 1u : 0u) << 10) | ((a_mn_major ? 1u : 0u) << 15) |
         ((b_mn_major ? 1u : 0u) << 16) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

// Shared-memory matrix descriptor, 128-byte swizzle (tiles are 1024-byte aligned).
//   bits 0-13 start >> 4, 16-29 leading byte offset >> 4, 32-45 stride byte
//   offset >> 4, bit 46 descriptor version 1, bits 61-63 swizzle (2 = 128 B).
// K-major operand: rows of 128 B along K, 8-row groups SBO apart (LBO unused).
// MN-major operand: 64 MN-elements per 128 B row, one row per K index, 8-row
//   K groups SBO apart, successive 64-element MN chunks LBO apart.
__device__ __forceinline__ uint64_t make_sdesc_sw128(uint32_t saddr, uint32_t lbo_bytes, uint32_t sbo_bytes) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr >> 4) & 0x3FFFu);
  d |= (uint64_t)((lbo_bytes >> 4) & 0x3FFFu) << 16;
  d |= (uint64_t)((sbo_bytes >> 4) & 0x3FFFu) << 32;
  d |= 1ull << 46;
  d |= 2ull << 61;
  return d;
}

// ---------------------------------------------------------------- math helpers
__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
// max(a, b, c) in one instruction.
__device__ __forceinline__ float max3f(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}
// (d0, d1) = (a0 * b + c, a1 * b + c) with one packed f32x2 FMA.
__device__ __forceinline__ void fma2(float a0, float a1, float b, float c, float& d0, float& d1) {
  asm("{\n .reg .b64 a, b, c, d;\n mov.b64 a, {%2, %3};\n mov.b64 b, {%4, %4};\n mov.b64 c, {%5, %5};\n"
      " fma.rn.f32x2 d, a, b, c;\n mov.b64 {%0, %1}, d;\n}\n"
      : "=f"(d0), "=f"(d1)
      : "f"(a0), "f"(a1), "f"(b), "f"(c));
}
// (d0, d1) = (a0 * b + c0, a1 * b + c1) with one packed f32x2 FMA.
__device__ __forceinline__ void fma2v(float a0, float a1, float b, float c0, float c1, float& d0, float& d1) {
  asm("{\n .reg .b64 a, b, c, d;\n mov.b64 a, {%2, %3};\n mov.b64 b, {%4, %4};\n mov.b64 c, {%5, %6};\n"
      " fma.rn.f32x2 d, a, b, c;\n mov.b64 {%0, %1}, d;\n}\n"
      : "=f"(d0), "=f"(d1)
      : "f"(a0), "f"(a1), "f"(b), "f"(c0), "f"(c1));
}
// (d0, d1) = (p0 * (a0 - b0), p1 * (a1 - b1)) with a packed f32x2 subtract and multiply.
__device__ __forceinline__ void submul2(float p0, float p1, float a0, float a1, float b0, float b1, float& d0,
                                        float& d1) {
  asm("{\n .reg .b64 p, a, b, d;\n mov.b64 p, {%2, %3};\n mov.b64 a, {%4, %5};\n mov.b64 b, {%6, %7};\n"
      " sub.f32x2 d, a, b;\n mul.f32x2 d, p, d;\n mov.b64 {%0, %1}, d;\n}\n"
      : "=f"(d0), "=f"(d1)
      : "f"(p0), "f"(p1), "f"(a0), "f"(a1), "f"(b0), "f"(b1));
}
// (d0, d1) += (a0, a1) with one packed f32x2 add.
__device__ __forceinline__ void add2(float& d0, float& d1, float a0, float a1) {
  asm("{\n .reg .b64 a, d;\n mov.b64 a, {%2, %3};\n mov.b64 d, {%0, %1};\n"
      " add.f32x2 d, d, a;\n mov.b64 {%0, %1}, d;\n}\n"
      : "+f"(d0), "+f"(d1)
      : "f"(a0), "f"(a1));
}
// Pack two fp32 values into one 32-bit word of 16-bit values (lo in bits 0-15), round to nearest even.
template <bool BF16>
__device__ __forceinline__ uint32_t pack2(float lo, float hi) {
  uint32_t r;
  if constexpr (BF16) {
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  } else {
    asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  }
  return r;
}
// Widen one stored 16-bit value to fp32 (exact).
template <bool BF16>
__device__ __forceinline__ float widen16(uint16_t x) {
  if constexpr (BF16) {
    return __uint_as_float((uint32_t)x << 16);
  } else {
    float y;
    asm("cvt.f32.f16 %0, %1;" : "=f"(y) : "h"(x));
    return y;
  }
}
__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
  asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c), "r"(d) : "memory");
}
__device__ __forceinline__ void ld_shared_v4(uint32_t addr, uint32_t& a, uint32_t& b, uint32_t& c, uint32_t& d) {
  asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];" : "=r"(a), "=r"(b), "=r"(c), "=r"(d) : "r"(addr) : "memory");
}

// Byte offset of the 16-byte chunk `c` (0..7) of row `r` inside a 128-byte-swizzled
// panel of 128-byte rows: the chunk index is XORed with the row's position in its
// 8-row group, the layout TMA writes with 128-byte swizzling.
__device__ __forceinline__ uint32_t sw128_offset(uint32_t r, uint32_t c) {
  return r * 128u + ((c ^ (r & 7u)) << 4);
}

// ---------------------------------------------------------------- FA_DEBUG checks
// Extents of a [planes, rows, cols] tensor as a TMA descriptor sees it.
struct Extent3 {
  int cols, rows, planes;
};
// In FA_DEBUG builds: checks a box origin against the tensor (column a multiple of
// 64 -- 128 bytes, so the 16-byte rule holds -- and inside the head dimension; row
// inside the rows rounded up to 256, the furthest any tile of these kernels
// starts: the forward's second 128-row sub-tile of a 256-row block; plane inside
// the planes), records a failure and clamps the origin to a valid one.  Compiles
// to nothing otherwise.
__device__ __forceinline__ void check_box(int& c0, int& c1, int& c2, const Extent3& e, uint32_t* err) {
  if constexpr (kDebug) {
    if (c0 < 0 || (c0 & 63) || c0 >= e.cols) { record_check(err, kDbgTmaCol, (uint32_t)c0); c0 = 0; }
    if (c1 < 0 || c1 >= (e.rows + 255) / 256 * 256) { record_check(err, kDbgTmaRow, (uint32_t)c1); c1 = 0; }
    if (c2 < 0 || c2 >= e.planes) { record_check(err, kDbgTmaPlane, (uint32_t)c2); c2 = 0; }
  }
}
__device__ __forceinline__ void tma_load_box(uint32_t dst, const CUtensorMap* m, uint32_t bar, int c0, int c1, int c2,
                                             const Extent3& e, uint32_t* err) {
  check_box(c0, c1, c2, e, err);
  tma_load_3d(dst, m, bar, c0, c1, c2);
}
__device__ __forceinline__ void tma_store_box(const CUtensorMap* m, uint32_t src, int c0, int c1, int c2,
                                              const Extent3& e, uint32_t* err) {
  check_box(c0, c1, c2, e, err);
  tma_store_3d(m, src, c0, c1, c2);
}
// In FA_DEBUG builds: a bulk copy of `bytes` from element `first` of a row vector
// of `count` floats must stay inside the vector and start 16-byte aligned; a
// failure is recorded and the copy starts at element 0 instead.
__device__ __forceinline__ void check_rows(long long& first, uint32_t bytes, long long count, uint32_t* err) {
  if constexpr (kDebug) {
    if (first < 0 || first + bytes / 4 > count || (first & 3)) {
      record_check(err, kDbgBulk, (uint32_t)first);
      first = 0;
    }
  }
}
__device__ __forceinline__ void bulk_load_rows(uint32_t dst, const float* vec, long long first, uint32_t bytes,
                                               long long count, uint32_t bar, uint32_t* err) {
  check_rows(first, bytes, count, err);
  bulk_load(dst, vec + first, bytes, bar);
}
// At CTA exit (all threads past the final barrier): an mbarrier that completed
// `phases` phases has current phase parity phases & 1.  A wrong count of
// arrivals or commits anywhere in the CTA's protocol shows up here.
__device__ __forceinline__ uint32_t mbar_test_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n"
      " mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n"
      " selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok;
}
// Indices i in [0, n) with i % m == s: the phases a barrier of stage s completes
// when n items go round a ring of m stages.
__device__ __forceinline__ uint32_t count_mod(int n, int s, int m) { return n > s ? (uint32_t)((n - 1 - s) / m + 1) : 0u; }
// True when no wait of the grid has given up (phase counts are only meaningful then).
__device__ __forceinline__ bool no_abort(const uint32_t* err) {
  return !(*reinterpret_cast<const volatile uint32_t*>(err) & kErrAborted);
}
__device__ __forceinline__ void check_phase(uint32_t bar, uint32_t phases, uint32_t* err, uint32_t id) {
  if constexpr (kDebug) {
    // test_wait.parity(p) is true once the phase with parity p has completed, i.e.
    // while the current phase's parity differs from p
    if (mbar_test_wait(bar, phases & 1u)) record_check(err, kDbgPhase, (id << 16) | (phases & 0xFFFFu));
  }
}

}  // namespace fa
