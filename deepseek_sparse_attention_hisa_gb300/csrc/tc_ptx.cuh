// Inline-PTX helpers for the sm_103a tensor-core path: tcgen05 (TMEM allocation, MMA,
// commit, TMEM loads), mbarriers with bounded waits, async-proxy fences and cp.async.
//
// Shared-memory operand layout used everywhere (the 128-byte swizzle):
//   an operand is stored in "atoms" of 8 rows x 128 bytes (1024 B, 1024-B aligned);
//   inside an atom, 16-byte unit u of row r lives at unit (u ^ (r % 8)).
//   K-major operand (rows = M or N, K contiguous): K is cut into chunks of 64 bf16
//     (128 B); chunk kc of row r sits at kc * chunk_bytes + r * 128.
//   MN-major operand (MN contiguous): the smem "row" is one k index holding 64 MN
//     elements; MN is cut into chunks of 64 with a stride of mn_chunk_bytes.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace hisa {
namespace tc {

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// byte offset of element (row, col) of a 128B-swizzled [rows x 64] bf16 chunk
__device__ __forceinline__ uint32_t sw128_offset(uint32_t row, uint32_t col_bf16) {
    const uint32_t unit = col_bf16 >> 3, e = col_bf16 & 7u;
    return row * 128u + (((unit ^ (row & 7u)) << 4) | (e << 1));
}

// ---- descriptors -------------------------------------------------------------
// Shared-memory matrix descriptor: start address, leading / stride byte offsets,
// descriptor version 1 (bit 46), 128-byte swizzle (layout type 2, bits 61-63).
__device__ __forceinline__ uint64_t smem_desc_sw128(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
    uint64_t d = 0;
    d |= (uint64_t)((saddr >> 4) & 0x3FFFu);
    d |= (uint64_t)((lbo >> 4) & 0x3FFFu) << 16;
    d |= (uint64_t)((sbo >> 4) & 0x3FFFu) << 32;
    d |= (uint64_t)1 << 46;
    d |= (uint64_t)2 << 61;
    return d;
}

// The start address is the low 14-bit field (address >> 4); shared memory is < 256 KiB,
// so moving a descriptor by a byte offset is an add of offset >> 4 with no carry out.
__device__ __forceinline__ uint64_t desc_add(uint64_t desc, uint32_t byte_offset) {
    return desc + (uint64_t)(byte_offset >> 4);
}

// Instruction descriptor, kind::f16: bf16 A and B, f32 accumulator.
// a_mn / b_mn select MN-major (transposed) operands.
__host__ __device__ constexpr uint32_t idesc_bf16_f32(int M, int N, int a_mn, int b_mn) {
    return (1u << 4)                       // D format: f32
           | (1u << 7)                     // A format: bf16
           | (1u << 10)                    // B format: bf16
           | ((uint32_t)a_mn << 15)        // A major-ness
           | ((uint32_t)b_mn << 16)        // B major-ness
           | ((uint32_t)(N >> 3) << 17)    // N / 8
           | ((uint32_t)(M >> 4) << 24);   // M / 16
}

// ---- TMEM --------------------------------------------------------------------
// Warp-wide: allocate ncols (power of two, 32..512) columns; the base address is
// written to *slot in shared memory.
__device__ __forceinline__ void tmem_alloc(uint32_t *slot, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;"
                 :: "r"(smem_u32(slot)), "r"(ncols) : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;"
                 :: "r"(taddr), "r"(ncols) : "memory");
}
__device__ __forceinline__ void fence_before_sync() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void fence_after_sync() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
// Make this thread's generic-proxy global writes visible to later async-proxy (TMA) reads.
__device__ __forceinline__ void fence_async_global() {
    asm volatile("fence.proxy.async.global;" ::: "memory");
}
// generic-proxy shared-memory writes -> visible to the async proxy (tensor core, TMA)
__device__ __forceinline__ void fence_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// One thread: D[tmem] (+)= A[smem] * B[smem]^T.
__device__ __forceinline__ void mma_bf16(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                         uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.u32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}"
        :: "r"(d_tmem), "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate) : "memory");
}

// Warp-wide: the whole warp passes the same (warp-uniform) operands and one lane,
// chosen by elect.sync, issues the MMA. Keeping the issue loop warp-uniform lets the
// descriptors live in uniform registers instead of being moved there per instruction.
__device__ __forceinline__ void mma_bf16_warp(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                              uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p, e;\n\t"
        "elect.sync _|e, 0xffffffff;\n\t"
        "setp.ne.u32 p, %4, 0;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}"
        :: "r"(d_tmem), "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate) : "memory");
}

// The same with A read from TMEM (a_tmem: its first column). Two bf16 per 32-bit column
// (the even element in the low half); a K step of 16 spans 8 columns. An M = 128 A operand
// holds row r in lane r, an M = 64 one row r in lane 32 (r / 16) + r % 16.
__device__ __forceinline__ void mma_bf16_tmem_a_warp(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc,
                                                     uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p, e;\n\t"
        "elect.sync _|e, 0xffffffff;\n\t"
        "setp.ne.u32 p, %4, 0;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}"
        :: "r"(d_tmem), "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate) : "memory");
}

// Warp-wide: one elected lane arranges an arrival (once) on mbar for when all MMAs this
// thread issued before have completed.
__device__ __forceinline__ void mma_commit_warp(uint64_t *mbar) {
    asm volatile(
        "{\n\t.reg .pred e;\n\telect.sync _|e, 0xffffffff;\n\t"
        "@e tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n\t}"
        :: "r"(smem_u32(mbar)) : "memory");
}

// Warp-wide: lane i of this warp's TMEM quadrant, 16 consecutive 32-bit columns.
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float (&v)[16]) {
    uint32_t r[16];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
        "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
          "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr));
#pragma unroll
    for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}
// 16 lanes x 2 halves: threads 0-15 read columns [c, c + 16) of TMEM lanes base + 0..15,
// threads 16-31 columns [c + 16, c + 32) of the same lanes (for M = 64 accumulators,
// whose rows live in lanes 0-15 of each 32-lane quadrant).
__device__ __forceinline__ void tmem_ld16_x2(uint32_t taddr, float (&v)[16]) {
    uint32_t r[16];
    asm volatile(
        "tcgen05.ld.sync.aligned.16x32bx2.x16.b32 "
        "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16], 16;"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
          "=r"(r[14]), "=r"(r[15])
        : "r"(taddr));
#pragma unroll
    for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}
__device__ __forceinline__ void tmem_ld_wait() {
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}
// Warp-wide: store 16 consecutive columns of this thread's lane.
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const float (&v)[16]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
        "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};"
        :: "r"(taddr), "r"(__float_as_uint(v[0])), "r"(__float_as_uint(v[1])),
           "r"(__float_as_uint(v[2])), "r"(__float_as_uint(v[3])), "r"(__float_as_uint(v[4])),
           "r"(__float_as_uint(v[5])), "r"(__float_as_uint(v[6])), "r"(__float_as_uint(v[7])),
           "r"(__float_as_uint(v[8])), "r"(__float_as_uint(v[9])), "r"(__float_as_uint(v[10])),
           "r"(__float_as_uint(v[11])), "r"(__float_as_uint(v[12])),
           "r"(__float_as_uint(v[13])), "r"(__float_as_uint(v[14])),
           "r"(__float_as_uint(v[15]))
        : "memory");
}
// Warp-wide: store 8 consecutive 32-bit columns of this thread's lane.
__device__ __forceinline__ void tmem_st8(uint32_t taddr, const uint32_t (&v)[8]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};"
        :: "r"(taddr), "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7])
        : "memory");
}
__device__ __forceinline__ void tmem_st_wait() {
    asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// ---- mbarriers -----------------------------------------------------------------
__device__ __forceinline__ void mbar_init(uint64_t *mbar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" :: "r"(smem_u32(mbar)), "r"(count)
                 : "memory");
}
__device__ __forceinline__ void mbar_fence_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t *mbar) {
    asm volatile("{\n\t.reg .b64 st;\n\tmbarrier.arrive.shared::cta.b64 st, [%0];\n\t}"
                 :: "r"(smem_u32(mbar)) : "memory");
}
__device__ __forceinline__ uint32_t mbar_try_wait(uint64_t *mbar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok) : "r"(smem_u32(mbar)), "r"(parity) : "memory");
    return ok;
}
// A waiter gives up after about kWaitCycles SM cycles (a quarter second at 2 GHz), far
// beyond any legitimate wait of these kernels, so a stuck pipeline ends promptly.
constexpr long long kWaitCycles = 1ll << 29;

// Bounded wait: returns false (and leaves the phase unconsumed) after `limit` polls or
// kWaitCycles cycles, so a kernel can record an error and exit instead of hanging.
__device__ __forceinline__ bool mbar_wait(uint64_t *mbar, uint32_t parity,
                                          uint32_t limit = (1u << 26)) {
    const long long t0 = clock64();
    for (uint32_t i = 0; i < limit; ++i) {
        if (mbar_try_wait(mbar, parity)) return true;
        if ((i & 255u) == 255u && clock64() - t0 > kWaitCycles) return false;
    }
    return false;
}

// The same, also giving up (every 256 polls) as soon as *abort is set.
__device__ __forceinline__ bool mbar_wait_abortable(uint64_t *mbar, uint32_t parity,
                                                    volatile int *abort) {
    const long long t0 = clock64();
    for (uint32_t i = 0; i < (1u << 26); ++i) {
        if (mbar_try_wait(mbar, parity)) return true;
        if ((i & 255u) == 255u && (*abort || clock64() - t0 > kWaitCycles)) return false;
    }
    return false;
}

// ---- TMA ------------------------------------------------------------------------
// Arrive on mbar and add `bytes` to the transaction count its current phase waits for.
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *mbar, uint32_t bytes) {
    asm volatile("{\n\t.reg .b64 st;\n\t"
                 "mbarrier.arrive.expect_tx.shared::cta.b64 st, [%0], %1;\n\t}"
                 :: "r"(smem_u32(mbar)), "r"(bytes) : "memory");
}
// One thread: load the box at element coordinates (x, y) of the 2-D tensor map `tmap`
// (a __grid_constant__ kernel parameter) into shared memory at dst; completion is
// counted in bytes on mbar. x * element size must be a multiple of 16 bytes.
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const void *tmap, int32_t x, int32_t y,
                                            uint64_t *mbar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes "
        "[%0], [%1, {%2, %3}], [%4];"
        :: "r"(dst), "l"(reinterpret_cast<uint64_t>(tmap)), "r"(x), "r"(y), "r"(smem_u32(mbar))
        : "memory");
}

// ---- cp.async (16-byte global -> shared copies) ---------------------------------
__device__ __forceinline__ void cp_async16(uint32_t saddr, const void *g) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" :: "r"(saddr), "l"(g) : "memory");
}
__device__ __forceinline__ void cp_async16_zfill(uint32_t saddr, const void *g, bool valid) {
    const uint32_t n = valid ? 16u : 0u;
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;"
                 :: "r"(saddr), "l"(g), "r"(n) : "memory");
}
// Arrive on mbar when all of this thread's prior cp.async copies have landed
// (counts as one arrival of the barrier's expected count).
__device__ __forceinline__ void cp_async_arrive(uint64_t *mbar) {
    asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" :: "r"(smem_u32(mbar))
                 : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() {
    asm volatile("cp.async.wait_all;" ::: "memory");
}

}  // namespace tc
}  // namespace hisa
