// la_sm100.cuh -- thin inline-PTX wrappers for the Blackwell (sm_100a / sm_103a) features the
// chunked extend kernel uses: mbarriers with bounded waits, TMA tiled loads, and the 5th-generation
// tensor cores (tcgen05: TMEM allocation, MMA, commit, TMEM loads).
//
// Operand layouts follow the PTX ISA's canonical shared-memory matrix layouts with the 128-byte
// swizzle: an "atom" is 8 rows x 128 bytes (1024 bytes, 1024-byte aligned), 16-byte chunk c of
// row r stored at chunk position c ^ (r % 8).  TMA tiled loads with CU_TENSOR_MAP_SWIZZLE_128B
// produce exactly this layout for a box whose inner extent is 128 bytes.
#pragma once

#include <cuda_bf16.h>
#include <stdint.h>

namespace la {
namespace sm100 {

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// ---------------------------------------------------------------------------------------------
// mbarrier

__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
                 : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
                 "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
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

__device__ __forceinline__ uint64_t globaltimer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t));
    return t;
}

// Wait until the phase with the given parity has completed, for at most limit_ns nanoseconds.
// Returns false if the limit ran out.  Never spins forever.
__device__ __forceinline__ bool mbar_wait(uint64_t *bar, uint32_t parity, uint64_t limit_ns) {
    const uint32_t a = smem_u32(bar);
    if (mbar_try_wait(a, parity)) return true;
    const uint64_t t0 = globaltimer_ns();
    while (true) {
        if (mbar_try_wait(a, parity)) return true;
        if (globaltimer_ns() - t0 > limit_ns) return false;
    }
}

// ---------------------------------------------------------------------------------------------
// TMA (cp.async.bulk.tensor), no multicast

__device__ __forceinline__ void tma_prefetch_desc(const void *tmap) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(tmap)) : "memory");
}

// 2D tiled load of one box into shared memory; completion is signalled as transaction bytes on
// `bar`.  x is the inner (contiguous) coordinate in elements, y the row.
__device__ __forceinline__ void tma_load_2d(void *smem_dst, const void *tmap, uint64_t *bar, int x,
                                            int y) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %4}], [%2];" ::"r"(smem_u32(smem_dst)),
        "l"(reinterpret_cast<uint64_t>(tmap)), "r"(smem_u32(bar)), "r"(x), "r"(y)
        : "memory");
}

// Prefetch the cache line holding global address p into L2.
__device__ __forceinline__ void prefetch_l2(const void *p) {
    asm volatile("prefetch.global.L2 [%0];" ::"l"(__cvta_generic_to_global(p)) : "memory");
}

// 2D tiled store of one box from shared memory (128-byte swizzled, as the tensor map says) to
// global memory, tracked by this thread's bulk async-group.
__device__ __forceinline__ void tma_store_2d(const void *tmap, const void *smem_src, int x, int y) {
    asm volatile(
        "cp.async.bulk.tensor.2d.global.shared::cta.tile.bulk_group [%0, {%2, %3}], [%1];" ::"l"(
            reinterpret_cast<uint64_t>(tmap)),
        "r"(smem_u32(smem_src)), "r"(x), "r"(y)
        : "memory");
}

__device__ __forceinline__ void bulk_commit_group() {
    asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}

// Wait until every committed bulk store of this thread has finished reading shared memory.
__device__ __forceinline__ void bulk_wait_group_read0() {
    asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}

// Wait until every committed bulk store of this thread has completed.
__device__ __forceinline__ void bulk_wait_group0() {
    asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
}

// Make this thread's generic-proxy shared-memory writes visible to the async proxy (the tensor
// core reads operands through it).
__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// ---------------------------------------------------------------------------------------------
// tcgen05: tensor memory and MMA (cta_group::1)

__device__ __forceinline__ void tmem_alloc(uint32_t *smem_result, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(smem_result)),
                 "r"(ncols)
                 : "memory");
}

__device__ __forceinline__ void tmem_relinquish() {
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
                 : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}

__device__ __forceinline__ void tc_fence_after() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// Instruction descriptor for kind::f16 with bf16 A and B and an fp32 accumulator.
// Bits: [4,6) D format (1 = f32), [7,10) A format (1 = bf16), [10,13) B format (1 = bf16),
// 15 A major (0 = K-major, 1 = MN-major), 16 B major, [17,23) N >> 3, [24,29) M >> 4.
__host__ __device__ constexpr uint32_t idesc_bf16_f32(int M, int N, bool a_mn_major,
                                                       bool b_mn_major) {
    return (1u << 4) | (1u << 7) | (1u << 10) | ((a_mn_major ? 1u : 0u) << 15) |
           ((b_mn_major ? 1u : 0u) << 16) | ((uint32_t)(N >> 3) << 17) |
           ((uint32_t)(M >> 4) << 24);
}

// Shared-memory matrix descriptor, 128-byte swizzle.
// Bits: [0,14) start address >> 4, [16,30) leading-dimension byte offset >> 4,
// [32,46) stride-dimension byte offset >> 4, [46,49) fixed 0b001, [61,64) swizzle (2 = 128B).
// K-major operand: SBO = byte distance between 8-row groups, LBO unused.
// MN-major operand: LBO = byte distance between 64-element (128-byte) groups along M/N,
//                   SBO = byte distance between 8-row groups along K.
__device__ __forceinline__ uint64_t sdesc_sw128(uint32_t smem_addr, uint32_t lbo_bytes,
                                                uint32_t sbo_bytes) {
    uint64_t d = 0;
    d |= (uint64_t)((smem_addr & 0x3FFFFu) >> 4);
    d |= (uint64_t)((lbo_bytes >> 4) & 0x3FFFu) << 16;
    d |= (uint64_t)((sbo_bytes >> 4) & 0x3FFFu) << 32;
    d |= (uint64_t)1 << 46;
    d |= (uint64_t)2 << 61;
    return d;
}

// D[tmem] (+)= A[smem] * B[smem]; issued by one thread.
__device__ __forceinline__ void mma_bf16(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                         uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// Arrive once on `bar` when every MMA previously issued by this thread has completed.
__device__ __forceinline__ void mma_commit(uint64_t *bar) {
    asm volatile(
        "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
            smem_u32(bar))
        : "memory");
}

// Warp-collective TMEM load: thread t of the warp receives lane (taddr.lane + t), 32 consecutive
// 32-bit columns starting at taddr.col.  A warp may only access its own 32-lane quarter
// (warp_id % 4).
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
        "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
          "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]),
          "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
          "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]),
          "=r"(r[31])
        : "r"(taddr));
}

__device__ __forceinline__ void tmem_ld_wait() {
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// Wait for this thread's outstanding TMEM loads; the registers are in/out operands so that no
// use of them can be scheduled before the wait.
__device__ __forceinline__ void tmem_ld_wait_regs(uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.wait::ld.sync.aligned;"
        : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]), "+r"(r[6]),
          "+r"(r[7]), "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]), "+r"(r[12]),
          "+r"(r[13]), "+r"(r[14]), "+r"(r[15]), "+r"(r[16]), "+r"(r[17]), "+r"(r[18]),
          "+r"(r[19]), "+r"(r[20]), "+r"(r[21]), "+r"(r[22]), "+r"(r[23]), "+r"(r[24]),
          "+r"(r[25]), "+r"(r[26]), "+r"(r[27]), "+r"(r[28]), "+r"(r[29]), "+r"(r[30]),
          "+r"(r[31])
        :
        : "memory");
}

// Warp-collective TMEM store, the mirror of tmem_ld32: thread t of the warp writes lane
// (taddr.lane + t), 32 consecutive 32-bit columns.
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
        "{%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, "
        "%17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32};" ::"r"(
            taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
        "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]),
        "r"(r[15]), "r"(r[16]), "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]),
        "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]),
        "r"(r[29]), "r"(r[30]), "r"(r[31])
        : "memory");
}

__device__ __forceinline__ void tmem_st_wait() {
    asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// Pin two register blocks after a single wait (a second wait on no outstanding loads is free).
__device__ __forceinline__ void tmem_ld_wait_regs2(uint32_t (&a)[32], uint32_t (&b)[32]) {
    tmem_ld_wait_regs(a);
    tmem_ld_wait_regs(b);
}

// Byte offset of element (row, col) of a bf16 tile stored as 128-byte-swizzled atoms: column
// blocks of 64 elements lie block_stride bytes apart, rows 128 bytes apart within a block.
__device__ __forceinline__ uint32_t sw128_offset(int row, int col, uint32_t block_stride) {
    const int blk = col >> 6;
    const int c = (col & 63) >> 3;
    return (uint32_t)blk * block_stride + (uint32_t)row * 128u +
           ((uint32_t)(c ^ (row & 7)) << 4) + (uint32_t)(col & 7) * 2u;
}

// Pack two floats into a bf16x2 word (round to nearest even), low half = a.
__device__ __forceinline__ uint32_t pack_bf16x2(float a, float b) {
    __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<uint32_t *>(&h);
}

// lambda K as a bf16 pair hi + lo, by the error-free product transform in bf16 arithmetic:
// lambda = l1 + l2 with l1 = bf16(lambda) and l2 = bf16(lambda - l1); hi = bf16(l1 K), the fused
// e = l1 K - hi is exact (the 16-bit product minus its 8-bit rounding fits 8 bits), and
// lo = bf16(l2 K + e).  The pair carries lambda K to about 2^-17 relative in three bf16x2
// instructions per two values.
struct LamSplitBf {
    __nv_bfloat162 l1, l2;
};
__device__ __forceinline__ LamSplitBf lam_split_bf16(float lam) {
    const __nv_bfloat16 h = __float2bfloat16_rn(lam);
    return {__bfloat162bfloat162(h), __bfloat162bfloat162(__float2bfloat16_rn(lam - __bfloat162float(h)))};
}
__device__ __forceinline__ void bf16x8_lam_hilo_bf16(const uint4 x, const LamSplitBf &l, uint4 &hi,
                                                     uint4 &lo) {
    const uint32_t w[4] = {x.x, x.y, x.z, x.w};
    uint32_t hv[4], lv[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
        const __nv_bfloat162 k = *reinterpret_cast<const __nv_bfloat162 *>(&w[e]);
        const __nv_bfloat162 a = __hmul2(l.l1, k);
        const __nv_bfloat162 err = __hfma2(l.l1, k, __hneg2(a));
        const __nv_bfloat162 b = __hfma2(l.l2, k, err);
        hv[e] = *reinterpret_cast<const uint32_t *>(&a);
        lv[e] = *reinterpret_cast<const uint32_t *>(&b);
    }
    hi = make_uint4(hv[0], hv[1], hv[2], hv[3]);
    lo = make_uint4(lv[0], lv[1], lv[2], lv[3]);
}

}  // namespace sm100
}  // namespace la
