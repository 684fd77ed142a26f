// Pieces shared by the persistent indexer pipelines of the DeepSeek-V4 indexer shape
// (H_i = 64 heads x D_i = 128 dims): the q plane layout and its exact bf16 split, the split
// of f32 block means into three bf16 planes, and the bounded waits and named barriers the
// warp roles synchronise with ([HiSA issue] "HiSA decode path": scoring is f32 on the page).
#pragma once

#include "select_core.cuh"
#include "tc_ptx.cuh"

namespace hisa {
namespace pipe {

using namespace tc;

constexpr int kH = 64, kD = 128, kM = 128;                // heads, dims, rows per MMA tile
constexpr int kGroup = 128;                               // threads of each 4-warp role
constexpr uint32_t kQPlane = kH * kD * 2;                 // [64 heads x 128 dims] bf16, 16 KiB

struct Misc {
    uint32_t tmem;
    int abort;
};

__device__ __forceinline__ bool wait_bar(uint64_t *bar, uint32_t parity, volatile int *abort) {
    return mbar_wait_abortable(bar, parity, abort);
}

__device__ __forceinline__ bool wait_bar_warp(uint64_t *bar, uint32_t parity, volatile int *abort) {
    return __all_sync(0xffffffffu, wait_bar(bar, parity, abort));
}

__device__ __forceinline__ void named_sync(int id, int n) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(n) : "memory");
}

// True on every participating thread iff v is true on all of them (named barrier id).
__device__ __forceinline__ bool group_all(int id, int n, bool v) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.ne.u32 p, %1, 0;\n\t"
        "bar.red.and.pred q, %2, %3, p;\n\t"
        "selp.u32 %0, 1, 0, q;\n\t}"
        : "=r"(r)
        : "r"((uint32_t)v), "r"(id), "r"(n)
        : "memory");
    return r != 0u;
}

// Exact three-way split of 8 f32 values into bf16 planes, packed as 3 x uint4: each plane
// the bf16 rounding of what the planes before it left.
__device__ __forceinline__ void split3(const float (&x)[8], uint4 (&pl)[3]) {
    uint32_t w[3][4];
#pragma unroll
    for (int e = 0; e < 8; e += 2) {
        float r0 = x[e], r1 = x[e + 1];
#pragma unroll
        for (int k = 0; k < 3; ++k) {
            const __nv_bfloat162 b = __floats2bfloat162_rn(r0, r1);
            w[k][e / 2] = *reinterpret_cast<const uint32_t *>(&b);
            if (k < 2) {
                const float2 f = __bfloat1622float2(b);
                r0 -= f.x;
                r1 -= f.y;
            }
        }
    }
#pragma unroll
    for (int k = 0; k < 3; ++k) pl[k] = make_uint4(w[k][0], w[k][1], w[k][2], w[k][3]);
}

// Exact split by truncation of 16 f32 values (four float4) into three bf16 planes, two
// values per 32-bit word (the even one in the low half): hi = the top 8 significant bits,
// then the same of the (exact) remainder; the last remainder has at most 8 bits left.
__device__ __forceinline__ void split3_trunc16(const float4 (&a)[4], uint32_t (&pl)[3][8]) {
#pragma unroll
    for (int ch = 0; ch < 4; ++ch) {
        const float xs[4] = {a[ch].x, a[ch].y, a[ch].z, a[ch].w};
        uint32_t pk[3][4];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const uint32_t b0 = __float_as_uint(xs[q]) & 0xffff0000u;
            const float r1 = xs[q] - __uint_as_float(b0);
            const uint32_t b1 = __float_as_uint(r1) & 0xffff0000u;
            const float r2 = r1 - __uint_as_float(b1);
            pk[0][q] = b0;
            pk[1][q] = b1;
            pk[2][q] = __float_as_uint(r2);
        }
#pragma unroll
        for (int k = 0; k < 3; ++k) {
            pl[k][2 * ch] = __byte_perm(pk[k][0], pk[k][1], 0x7632);       // {hi(e0), hi(e1)}
            pl[k][2 * ch + 1] = __byte_perm(pk[k][2], pk[k][3], 0x7632);
        }
    }
}

// Byte offset of 16-byte unit u (dims 8u..8u+7) of head h of q plane `plane` when nq
// planes are stacked along N: per 64-dim chunk, plane 0's 64 heads, then plane 1's, ...
__device__ __forceinline__ uint32_t q_off(uint32_t plane, uint32_t h, uint32_t u, uint32_t nq) {
    return (u >> 3) * (nq * kH * 128u) + plane * (kH * 128u) + sw128_offset(h, (u & 7u) * 8u);
}


// One query row's q in a 4-warp builder group (128 threads, bt = thread index in the
// group): load() issues the global loads early so that they overlap the builder's waits,
// store() writes the q planes (three exact bf16 planes for f32 q, one for bf16 q) once
// the buffer is free. With HALVES (f32 q in a 22-warp CTA, where registers are short)
// only half of q is held in registers: the other half is prefetched into L2 by load() and
// read by store().
template <bool QBF16, bool HALVES>
struct QRegs {
    static constexpr int kQU = kH * 16 / kGroup;              // 16-byte q units per thread
    static constexpr int kHeld = (HALVES && !QBF16) ? kQU / 2 : kQU;
    static constexpr int NQ = QBF16 ? 1 : 3;
    float4 qf[QBF16 ? 1 : 2 * kHeld];
    uint4 qh[QBF16 ? kQU : 1];
    const float4 *q4 = nullptr;

    __device__ __forceinline__ void load(const void *q, int64_t row, int bt) {
        if (QBF16) {
            const uint4 *q16 = reinterpret_cast<const uint4 *>(
                reinterpret_cast<const __nv_bfloat16 *>(q) + row * kH * kD);
#pragma unroll
            for (int m = 0; m < kQU; ++m) qh[m] = __ldg(q16 + bt + m * kGroup);
        } else {
            q4 = reinterpret_cast<const float4 *>(reinterpret_cast<const float *>(q) + row * kH * kD);
#pragma unroll
            for (int m = 0; m < kHeld; ++m) {
                qf[2 * m] = __ldg(q4 + 2 * (bt + m * kGroup));
                qf[2 * m + 1] = __ldg(q4 + 2 * (bt + m * kGroup) + 1);
            }
#pragma unroll
            for (int m = kHeld; m < kQU; ++m)
                asm volatile("prefetch.global.L2 [%0];" ::"l"(q4 + 2 * (bt + m * kGroup)));
        }
    }

    // planes: the buffer of NQ planes in the layout q_off describes
    __device__ __forceinline__ void store(uint8_t *planes, int bt) {
        if (QBF16) {
#pragma unroll
            for (int m = 0; m < kQU; ++m) {
                const int u = bt + m * kGroup;
                *reinterpret_cast<uint4 *>(planes + q_off(0, u >> 4, u & 15, NQ)) = qh[m];
            }
            return;
        }
        auto put = [&](int m, const float4 &a, const float4 &b) {
            const int u = bt + m * kGroup;
            const float x[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
            uint4 pl[3];
            split3(x, pl);
#pragma unroll
            for (int k = 0; k < 3; ++k)
                *reinterpret_cast<uint4 *>(planes + q_off(k, u >> 4, u & 15, NQ)) = pl[k];
        };
#pragma unroll
        for (int m = 0; m < kHeld; ++m) put(m, qf[2 * m], qf[2 * m + 1]);
        if (kHeld < kQU) {
#pragma unroll
            for (int m = kHeld; m < kQU; ++m) {
                qf[2 * (m - kHeld)] = __ldg(q4 + 2 * (bt + m * kGroup));
                qf[2 * (m - kHeld) + 1] = __ldg(q4 + 2 * (bt + m * kGroup) + 1);
            }
#pragma unroll
            for (int m = kHeld; m < kQU; ++m) put(m, qf[2 * (m - kHeld)], qf[2 * (m - kHeld) + 1]);
        }
    }
};

// Block means ([HiSA issue] "HiSA decode path": the mean of each completed index block of
// pooled keys) of blocks [first, n) of one sequence, index_block 64 and D_i 128, from its
// bf16 keys (kv: the key array as 16-byte units, k0: the sequence's first pooled row) to f32
// rows means[base + beta], by a 4-warp group: thread bt owns dims 8 (bt / 8) .. + 7 of rows
// bt % 8 + 8 m; eight partial sums in row order, then the pairwise tree over the eight lanes
// of a dimension group.
__device__ __forceinline__ void append_block_means(const uint4 *kv, int64_t k0, int64_t first, int64_t n,
                                                   float *means, int64_t base, int bt) {
    const int k = bt & 7, gq = bt >> 3;
    for (int64_t beta = first; beta < n; ++beta) {
        const uint4 *src = kv + (k0 + beta * 64) * (kD / 8);
        uint4 u[8];
#pragma unroll
        for (int m = 0; m < 8; ++m) u[m] = __ldg(src + (8 * m + k) * (kD / 8) + gq);
        float ps[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) ps[e] = 0.f;
#pragma unroll
        for (int m = 0; m < 8; ++m) {
            const __nv_bfloat162 *h2 = reinterpret_cast<const __nv_bfloat162 *>(&u[m]);
#pragma unroll
            for (int e2 = 0; e2 < 4; ++e2) {
                const float2 f = __bfloat1622float2(h2[e2]);
                ps[2 * e2] += f.x;
                ps[2 * e2 + 1] += f.y;
            }
        }
#pragma unroll
        for (int off = 1; off < 8; off <<= 1)
#pragma unroll
            for (int e = 0; e < 8; ++e) ps[e] += __shfl_xor_sync(0xffffffffu, ps[e], off);
        if (k == 0) {
            float4 *dst = reinterpret_cast<float4 *>(means + (base + beta) * kD + gq * 8);
            dst[0] = make_float4(ps[0] / 64.f, ps[1] / 64.f, ps[2] / 64.f, ps[3] / 64.f);
            dst[1] = make_float4(ps[4] / 64.f, ps[5] / 64.f, ps[6] / 64.f, ps[7] / 64.f);
        }
    }
}

}  // namespace pipe
}  // namespace hisa
