// la_tc_ptx.cuh -- thin inline-PTX wrappers for the sm_103a tensor-core path: mbarriers
// (with bounded waits), TMA tile loads, tcgen05 MMA / TMEM allocation / TMEM loads and
// stores, and the shared-memory and instruction descriptors of tcgen05.mma.
//
// Operand tiles.  Every bf16 operand tile lives in shared memory in the 128-byte swizzled
// layout that a TMA load with CU_TENSOR_MAP_SWIZZLE_128B and a 64-element-wide box
// produces: the tile's columns are split into blocks of 64 elements; a block stores its
// `rows` rows at 128 bytes each, and within a row the 16-byte chunk c sits at chunk
// position c ^ (row % 8).  Blocks follow each other at `rows * 128` bytes; every block is
// 1024-byte aligned.  The same bytes serve as a K-major operand (rows = M or N index,
// columns = K) or as an MN-major operand (rows = K index, columns = M or N).
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

namespace la {
namespace tc {

// A bounded mbarrier wait gives up after this many nanoseconds (every legitimate wait in
// the library's kernels is shorter than a whole kernel, far below this).  The test build
// (LA_TEST_HOOKS) shortens it to 5 ms so that a test can make a wait run out quickly; the
// drain of copies already in flight on the exit path keeps the long bound (kDrainNs).
#ifdef LA_TEST_HOOKS
constexpr uint64_t kWaitNs = 5000000ull;
#else
constexpr uint64_t kWaitNs = 2000000000ull;
#endif
constexpr uint64_t kDrainNs = 2000000000ull;

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// ---- mbarrier ---------------------------------------------------------------------------

__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

// Make barrier initialisation visible to the async proxy (TMA, tcgen05.commit).
__device__ __forceinline__ void fence_barrier_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
                 : "memory");
}


// One arrival of weight `count` (for a warp that arrives as a unit).
__device__ __forceinline__ void mbar_arrive_cnt(uint64_t *bar, uint32_t count) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

// Warp-wide arrival, called by all 32 lanes: the lanes synchronise (which orders their
// earlier memory operations before lane 0's release) and lane 0 arrives for all of them,
// so the barrier's expected count stays in threads.
__device__ __forceinline__ void mbar_arrive_warp(uint64_t *bar) {
    __syncwarp();
    if ((threadIdx.x & 31u) == 0u) mbar_arrive_cnt(bar, 32u);
}

// Non-blocking test: has the phase with the given parity completed?
__device__ __forceinline__ bool mbar_test(uint64_t *bar, uint32_t parity) {
    uint32_t done;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(done)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return done != 0;
}

// Test the phase; the thread may be suspended inside for up to kSuspendNs waiting for it,
// so that waiting warps do not spin on the issue slots.
constexpr uint32_t kSuspendNs = 200000u;
__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity) {
    uint32_t done;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(done)
        : "r"(smem_u32(bar)), "r"(parity), "r"(kSuspendNs)
        : "memory");
    return done != 0;
}

__device__ __forceinline__ uint64_t globaltimer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// Wait for the phase with the given parity to complete.  Gives up (returns false and
// raises *abort) after kWaitNs, or early once another thread raised *abort.
__device__ __forceinline__ bool mbar_wait(uint64_t *bar, uint32_t parity, volatile int *abort) {
    if (mbar_test(bar, parity)) return true;
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = globaltimer_ns();
    for (;;) {
        if (mbar_try_wait(bar, parity)) return true;
        if (*abort) return false;
        if (globaltimer_ns() - t0 > kWaitNs) {
            *abort = 1;
            return false;
        }
    }
}

// ---- async proxy fences -----------------------------------------------------------------

// Order this thread's generic-proxy shared-memory writes before later async-proxy reads
// (tcgen05.mma operands, TMA stores).
__device__ __forceinline__ void fence_proxy_async() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// ---- TMA --------------------------------------------------------------------------------


// Load one box of a 2-D tensor map at coordinates (x innermost, y) into shared memory,
// completing `bytes` transaction bytes on *bar.
__device__ __forceinline__ void tma_load_2d(void *dst, const CUtensorMap *map, uint64_t *bar, int x, int y) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%3, %4}], [%2];" ::"r"(
            smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(x), "r"(y)
        : "memory");
}

__device__ __forceinline__ void tma_load_3d(void *dst, const CUtensorMap *map, uint64_t *bar, int x, int y, int z) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(
            smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(x), "r"(y), "r"(z)
        : "memory");
}


__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
// Wait until every committed bulk group of this thread has finished reading shared memory.
__device__ __forceinline__ void bulk_wait_read() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }
// Wait until every committed bulk group of this thread has completed.
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

// ---- tcgen05: TMEM allocation -----------------------------------------------------------

// One full warp: allocate `ncols` TMEM columns (power of two >= 32); the base address is
// written to *dst (shared memory).
__device__ __forceinline__ void tmem_alloc(uint32_t *dst, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(dst)), "r"(ncols)
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

// ---- tcgen05: MMA -----------------------------------------------------------------------

// Instruction descriptor of kind::f16 with bf16 A and B and an fp32 accumulator.
// a_mn / b_mn: operand stored MN-major (else K-major).
__host__ __device__ constexpr uint32_t idesc_bf16(int M, int N, bool a_mn, bool b_mn) {
    return (1u << 4)                          // D format: f32
           | (1u << 7)                        // A format: bf16
           | (1u << 10)                       // B format: bf16
           | ((a_mn ? 1u : 0u) << 15)         // A major
           | ((b_mn ? 1u : 0u) << 16)         // B major
           | ((uint32_t)(N >> 3) << 17)       // N / 8
           | ((uint32_t)(M >> 4) << 24);      // M / 16
}

// Shared-memory matrix descriptor, 128-byte swizzle, sm_100-family version field.
__device__ __forceinline__ uint64_t sdesc(uint32_t saddr, uint32_t lbo_bytes, uint32_t sbo_bytes) {
    return (uint64_t)((saddr >> 4) & 0x3FFFu) | ((uint64_t)((lbo_bytes >> 4) & 0x3FFFu) << 16) |
           ((uint64_t)((sbo_bytes >> 4) & 0x3FFFu) << 32) | (1ull << 46) | (2ull << 61);
}

// Descriptor of a K-major operand taken from a swizzled tile with `rows` rows, starting at
// row `row0` (a multiple of 8), for the 16-element K step `kstep`.
__device__ __forceinline__ uint64_t desc_kmajor(uint32_t tile, int rows, int row0, int kstep) {
    const int k0 = kstep * 16;
    const uint32_t addr = tile + (uint32_t)(k0 / 64) * rows * 128u + (uint32_t)row0 * 128u + (uint32_t)(k0 % 64) * 2u;
    return sdesc(addr, 16u, 1024u);
}

// Descriptor of an MN-major operand taken from a swizzled tile whose rows are the K index
// (`rows` rows in all), starting at MN column `col0` (a multiple of 64), for K step `kstep`.
__device__ __forceinline__ uint64_t desc_mnmajor(uint32_t tile, int rows, int col0, int kstep) {
    const uint32_t addr = tile + (uint32_t)(col0 / 64) * rows * 128u + (uint32_t)(kstep * 16) * 128u;
    return sdesc(addr, (uint32_t)rows * 128u, 1024u);
}

// D[tmem] (+)= A * B, issued by one thread.
__device__ __forceinline__ void mma_bf16(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                         uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// The same MMA with the A operand kept in the collector buffer for the next MMA
// (`fill`), taken from it and kept (`use`), or taken from it and released (`lastuse`):
// consecutive MMAs that share A read it from shared memory once.  The A descriptor of the `lastuse` MMA must describe
// the same matrix as the `fill` before it, with the same major-ness.
__device__ __forceinline__ void mma_bf16_fill(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                              uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16.collector::a::fill [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

__device__ __forceinline__ void mma_bf16_use(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                             uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16.collector::a::use [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

__device__ __forceinline__ void mma_bf16_lastuse(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                                 uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16.collector::a::lastuse [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// ---- warp-collective issue ----------------------------------------------------------
// The *_w forms are called by all 32 lanes of a warp in warp-uniform control flow with
// warp-uniform arguments; lane 0, selected by a predicate inside the instruction block,
// issues the operation (always the same lane, so a commit covers the lane's MMAs).  Keeping the control flow uniform lets the compiler hold the
// descriptors and coordinates in uniform registers: measured on sm_103a, an MMA issued
// from inside a one-lane branch cost 80 cycles of issue alone and over 300 next to busy
// warps, against 47 and 60 for the warp-collective form.

#define LA_LANE0_MMA(QUAL)                                                        \
    asm volatile(                                                                 \
        "{\n\t.reg .pred p, e;\n\t.reg .u32 l;\n\t"                                 \
        "mov.u32 l, %%laneid;\n\tsetp.eq.u32 e, l, 0;\n\t"                            \
        "setp.ne.b32 p, %4, 0;\n\t"                                                 \
        "@e tcgen05.mma.cta_group::1.kind::f16" QUAL " [%0], %1, %2, %3, p;\n\t}" \
        ::"r"(d_tmem), "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)      \
        : "memory")

__device__ __forceinline__ void mma_bf16_w(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                           uint32_t accumulate) {
    LA_LANE0_MMA("");
}
__device__ __forceinline__ void mma_bf16_fill_w(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                                uint32_t accumulate) {
    LA_LANE0_MMA(".collector::a::fill");
}
__device__ __forceinline__ void mma_bf16_lastuse_w(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                                   uint32_t idesc, uint32_t accumulate) {
    LA_LANE0_MMA(".collector::a::lastuse");
}
#undef LA_LANE0_MMA

// Arrive once on *bar when every tcgen05 operation issued so far by the issuing lane is done.
__device__ __forceinline__ void mma_commit_w(uint64_t *bar) {
    asm volatile(
        "{\n\t.reg .pred e;\n\t.reg .u32 l;\n\tmov.u32 l, %%laneid;\n\tsetp.eq.u32 e, l, 0;\n\t"
        "@e tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n\t}" ::"r"(smem_u32(bar))
        : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx_w(uint64_t *bar, uint32_t bytes) {
    asm volatile(
        "{\n\t.reg .pred e;\n\t.reg .u32 l;\n\tmov.u32 l, %%laneid;\n\tsetp.eq.u32 e, l, 0;\n\t"
        "@e mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;\n\t}" ::"r"(smem_u32(bar)),
        "r"(bytes)
        : "memory");
}

// One arrival (count 1) on behalf of the warp.
__device__ __forceinline__ void mbar_arrive_w(uint64_t *bar) {
    __syncwarp();
    asm volatile(
        "{\n\t.reg .pred e;\n\t.reg .u32 l;\n\tmov.u32 l, %%laneid;\n\tsetp.eq.u32 e, l, 0;\n\t"
        "@e mbarrier.arrive.shared::cta.b64 _, [%0];\n\t}" ::"r"(smem_u32(bar))
        : "memory");
}


__device__ __forceinline__ void tma_load_4d_w(void *dst, const CUtensorMap *map, uint64_t *bar, int x, int y, int z,
                                              int w) {
    asm volatile(
        "{\n\t.reg .pred e;\n\t.reg .u32 l;\n\tmov.u32 l, %%laneid;\n\tsetp.eq.u32 e, l, 0;\n\t"
        "@e cp.async.bulk.tensor.4d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%3, %4, %5, %6}], "
        "[%2];\n\t}" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(x), "r"(y), "r"(z), "r"(w)
        : "memory");
}


__device__ __forceinline__ void tma_load_2d_w(void *dst, const CUtensorMap *map, uint64_t *bar, int x, int y) {
    asm volatile(
        "{\n\t.reg .pred e;\n\t.reg .u32 l;\n\tmov.u32 l, %%laneid;\n\tsetp.eq.u32 e, l, 0;\n\t"
        "@e cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%3, %4}], "
        "[%2];\n\t}" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(x), "r"(y)
        : "memory");
}

// Bring `bytes` (a multiple of 16) of global memory at p (16-byte aligned) into L2, from the
// calling thread, without waiting.
__device__ __forceinline__ void prefetch_l2_bulk(const void *p, uint32_t bytes) {
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p), "r"(bytes) : "memory");
}



// Store one box from shared memory (bulk-group completion) from lane 0.  Every lane then
// runs bulk_commit() and bulk_wait_read() / bulk_wait_all() (empty groups for the lanes
// that issued nothing) and __syncwarp(), so the warp waits for lane 0's copies.
__device__ __forceinline__ void tma_store_3d_w(const CUtensorMap *map, const void *src, int x, int y, int z) {
    asm volatile(
        "{\n\t.reg .pred e;\n\t.reg .u32 l;\n\tmov.u32 l, %%laneid;\n\tsetp.eq.u32 e, l, 0;\n\t"
        "@e cp.async.bulk.tensor.3d.global.shared::cta.bulk_group [%0, {%2, %3, %4}], [%1];\n\t}" ::"l"(
            reinterpret_cast<uint64_t>(map)),
        "r"(smem_u32(src)), "r"(x), "r"(y), "r"(z)
        : "memory");
}

// Store one box of a 2-D tensor map from shared memory from lane 0 (bulk-group completion;
// see tma_store_3d_w for the commit and wait that follow).
__device__ __forceinline__ void tma_store_2d_w(const CUtensorMap *map, const void *src, int x, int y) {
    asm volatile(
        "{\n\t.reg .pred e;\n\t.reg .u32 l;\n\tmov.u32 l, %%laneid;\n\tsetp.eq.u32 e, l, 0;\n\t"
        "@e cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%2, %3}], [%1];\n\t}" ::"l"(
            reinterpret_cast<uint64_t>(map)),
        "r"(smem_u32(src)), "r"(x), "r"(y)
        : "memory");
}

// Arrive once on *bar when every tcgen05 operation issued so far by this thread is done.
__device__ __forceinline__ void mma_commit(uint64_t *bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
                 : "memory");
}

// ---- tcgen05: TMEM <-> registers ----------------------------------------------------------

// Warp-wide: thread t gets TMEM lane (lane of taddr) + t, 16 consecutive 32-bit columns.
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float *v) {
    uint32_t r[16];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
        "%15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr));
#pragma unroll
    for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}

// Warp-wide: thread t gets TMEM lane (lane of taddr) + t, one 32-bit column.
__device__ __forceinline__ float tmem_ld1(uint32_t taddr) {
    uint32_t r;
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x1.b32 {%0}, [%1];" : "=r"(r) : "r"(taddr));
    return __uint_as_float(r);
}

// Warp-wide: thread t gets TMEM lane (lane of taddr) + t, two consecutive columns.
__device__ __forceinline__ void tmem_ld2(uint32_t taddr, float *v) {
    uint32_t r0, r1;
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x2.b32 {%0, %1}, [%2];" : "=r"(r0), "=r"(r1) : "r"(taddr));
    v[0] = __uint_as_float(r0);
    v[1] = __uint_as_float(r1);
}

// Warp-wide: thread t gets TMEM lane (lane of taddr) + t, four consecutive columns.
__device__ __forceinline__ void tmem_ld4(uint32_t taddr, float *v) {
    uint32_t r0, r1, r2, r3;
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x4.b32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(taddr));
    v[0] = __uint_as_float(r0);
    v[1] = __uint_as_float(r1);
    v[2] = __uint_as_float(r2);
    v[3] = __uint_as_float(r3);
}

// Warp-wide: thread t gets TMEM lane (lane of taddr) + t, 32 consecutive 32-bit columns.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float *v) {
    uint32_t r[32];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
        "%15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
          "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
          "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr));
#pragma unroll
    for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}


// Wait for this warp's TMEM loads, then pin the N loaded registers behind the wait: the
// empty asm "rewrites" each value, so no use of them can be scheduled before the wait.
template <int N>
__device__ __forceinline__ void tmem_wait_regs(float *v) {
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
    for (int i = 0; i < N; ++i) asm volatile("" : "+f"(v[i])::"memory");
}

// Warp-wide: thread t writes TMEM lane (lane of taddr) + t, 16 consecutive columns.
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const float *v) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
        "%15, %16};" ::"r"(taddr),
        "r"(__float_as_uint(v[0])), "r"(__float_as_uint(v[1])), "r"(__float_as_uint(v[2])),
        "r"(__float_as_uint(v[3])), "r"(__float_as_uint(v[4])), "r"(__float_as_uint(v[5])),
        "r"(__float_as_uint(v[6])), "r"(__float_as_uint(v[7])), "r"(__float_as_uint(v[8])),
        "r"(__float_as_uint(v[9])), "r"(__float_as_uint(v[10])), "r"(__float_as_uint(v[11])),
        "r"(__float_as_uint(v[12])), "r"(__float_as_uint(v[13])), "r"(__float_as_uint(v[14])),
        "r"(__float_as_uint(v[15]))
        : "memory");
}

// Zero two consecutive columns of this warp's 32 lanes.
__device__ __forceinline__ void tmem_zero2(uint32_t taddr) {
    asm volatile("tcgen05.st.sync.aligned.32x32b.x2.b32 [%0], {%1, %1};" ::"r"(taddr), "r"(0u) : "memory");
}

__device__ __forceinline__ void tmem_st_wait() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// ---- swizzled tile addressing (generic-proxy reads and writes by threads) ---------------

// Byte offset of element (row, col) in a swizzled bf16 tile with `rows` rows.
__host__ __device__ __forceinline__ uint32_t swz_offset(int rows, int row, int col) {
    const int blk = col >> 6, c = col & 63, chunk = c >> 3;
    return (uint32_t)blk * rows * 128u + (uint32_t)row * 128u + (uint32_t)((chunk ^ (row & 7)) << 4) +
           (uint32_t)(c & 7) * 2u;
}

// Byte offset of the 16-byte chunk holding columns [8*chunk16, 8*chunk16 + 8) of a row.
__host__ __device__ __forceinline__ uint32_t swz_chunk(int rows, int row, int chunk16) {
    const int blk = chunk16 >> 3, chunk = chunk16 & 7;
    return (uint32_t)blk * rows * 128u + (uint32_t)row * 128u + (uint32_t)((chunk ^ (row & 7)) << 4);
}

// Named barrier for a subset of warps (id 1..15; `threads` a multiple of 32).
__device__ __forceinline__ void named_barrier(int id, int threads) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(threads) : "memory");
}

}  // namespace tc
}  // namespace la
