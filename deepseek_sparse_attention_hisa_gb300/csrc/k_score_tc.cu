// Indexer scoring on the sm_103a tensor cores for the DeepSeek-V4 indexer shape
// (H_i = 64 heads, D_i = 128), with the top-k fused for the coarse and fine stages.
//
// score[row] = sum_h relu(q_h . row) * scale * w_h   ([HiSA issue] "Flat selection",
// "HiSA decode path": the coarse stage scores block means, the fine stage the rows of
// the kept blocks, the flat path every pooled row).
//
// Per tile of 128 scored rows: D[128 rows x 64 heads] = rows . q^T on tcgen05 (M = 128,
// N = 64, K = 128), f32 accumulators in TMEM (two buffers). Scoring is f32 on the page,
// so f32 operands are split exactly into three bf16 planes, x = x1 + x2 + x3 (each the
// bf16 rounding of what the previous planes leave over): bf16 products are exact in the
// f32 accumulator. bf16 keys need one plane; f32 q needs three (3 products per K step);
// f32 block means against f32 q use all nine plane pairs. The q planes are stacked along
// N (N = 64 * planes), so one MMA per rows plane and K step covers every q plane.
// The epilogue thread of TMEM lane r owns row r of the tile: it applies relu, the head
// weights and the head sum in registers, with no cross-thread reduction.
//
// Warp roles: 0 MMA issue + TMEM owner, 1-4 epilogue (warp w reads TMEM lanes
// 32*(w%4)..+31), 5-8 loaders (q planes; bf16 rows by TMA with the 128-byte swizzle,
// f32 rows through registers, split into planes). Coarse and fine CTAs own one
// query row and finish with block_topk over the scores held in shared memory; flat CTAs
// own a range of tiles of one query row and write scores to global memory.
// Waits are bounded; a timeout raises HISA_DEV_TIMEOUT and the CTA drains and exits.
#include "select_core.cuh"
#include "tc_ptx.cuh"

namespace hisa {
namespace {

using namespace tc;

// Two CTAs share an SM (one's set-up and select overlap the other's loads): 64-row tiles
// (M = 64: row r of a tile sits in TMEM lane r % 16 of quadrant r / 16), one 192-column
// accumulator (256 TMEM columns per CTA), about 100 KiB of shared memory.
constexpr int kH = 64, kD = 128, kTile = 64;
constexpr int kThreads = 288;                          // 9 warps
constexpr int kMmaWarp = 0, kLoadWarp0 = 5;               // epilogue: warps 1-4
constexpr int kLoaders = 128, kEpis = 128;
constexpr uint32_t kPlaneQ = kH * kD * 2;              // 16 KiB: [64 heads x 128 dims] bf16
constexpr uint32_t kPlaneRows = kTile * kD * 2;        // 16 KiB: [64 rows x 128 dims] bf16
constexpr int kSlots = 3;                              // bf16 row tiles in flight
constexpr uint32_t kOffQ = 0;
constexpr uint32_t kOffRows = kOffQ + 3 * kPlaneQ;     // 48 KiB: 3 slots, or 3 planes of 1 slot
constexpr uint32_t kOffW = kOffRows + 3 * kPlaneRows;
constexpr uint32_t kOffBlk = kOffW + kH * 4;
constexpr uint32_t kOffBar = kOffBlk + 64 * 4;
// barriers: full[3] empty[3] d_full d_free q_full drain
constexpr int kBarFull = 0, kBarEmpty = 3, kBarDFull = 6, kBarDFree = 7, kBarQ = 8,
              kBarDrain = 9, kNumBars = 10;
constexpr uint32_t kOffMisc = kOffBar + kNumBars * 8;
constexpr uint32_t kOffSc = kOffMisc + 64;             // scores of the fused select: n floats
constexpr int kMaxSel = 8192;                          // largest n a fused select holds
constexpr uint32_t kSmemFixed = kOffSc + 1024;         // + alignment slack
constexpr uint32_t kTmemCols = 256;                    // one accumulator of 64 * (q planes) columns

struct Misc {
    uint32_t tmem;
    int abort;
};

__device__ __forceinline__ bool wait_bar(uint64_t *bar, uint32_t parity, volatile int *abort) {
    return mbar_wait_abortable(bar, parity, abort);
}

// A wait taken by a whole warp; the result is made warp-uniform.
__device__ __forceinline__ bool wait_bar_warp(uint64_t *bar, uint32_t parity, volatile int *abort) {
    return __all_sync(0xffffffffu, wait_bar(bar, parity, abort));
}

// Exact three-way split of 8 f32 values into bf16 planes, packed as 3 x uint4.
__device__ __forceinline__ void split3(const float (&x)[8], uint4 (&pl)[3]) {
    uint32_t w[3][4];
#pragma unroll
    for (int e = 0; e < 8; e += 2) {
        float r0 = x[e], r1 = x[e + 1];
#pragma unroll
        for (int k = 0; k < 3; ++k) {
            const __nv_bfloat162 b = __floats2bfloat162_rn(r0, r1);
            w[k][e / 2] = *reinterpret_cast<const uint32_t *>(&b);
            const float2 f = __bfloat1622float2(b);
            r0 -= f.x;
            r1 -= f.y;
        }
    }
#pragma unroll
    for (int k = 0; k < 3; ++k) pl[k] = make_uint4(w[k][0], w[k][1], w[k][2], w[k][3]);
}

// Byte offset of unit u (dims 8u..8u+7) of head h of q plane `plane` when the nq planes
// are stacked along N: per 64-dim chunk, plane 0's 64 heads, then plane 1's, ... so one
// MMA with N = 64 * nq multiplies a row tile by every plane at once.
__device__ __forceinline__ uint32_t q_off(uint32_t plane, uint32_t h, uint32_t u, uint32_t nq) {
    return (u >> 3) * (nq * kH * 128u) + plane * (kH * 128u) + sw128_offset(h, (u & 7u) * 8u);
}

// Byte offset of the 16-byte unit u (dims 8u..8u+7) of row r in a K-major [rows x 128]
// bf16 operand of `rows` rows: two 64-dim chunks of rows*128 bytes.
__device__ __forceinline__ uint32_t unit_off(uint32_t r, uint32_t u, uint32_t rows) {
    return (u >> 3) * (rows * 128u) + sw128_offset(r, (u & 7u) * 8u);
}

}  // namespace
}  // namespace hisa

namespace hisa {
namespace {

template <int MODE, bool QBF16>
__global__ void __launch_bounds__(kThreads, 2) k_score_tc(const __grid_constant__ ScoreTcParams P) {
    constexpr int NQ = QBF16 ? 1 : 3;                    // q planes
    constexpr int NR = (MODE == kCoarse) ? 3 : 1;        // row planes
    const ScoreParams &p = P.s;
    // flat, and coarse / fine for a few long rows: CTAs own ranges of tiles of a row and
    // write its scores to p.out (selected by a later kernel); else one CTA per row selects
    const bool split = MODE == kFlat || P.tiles_per_cta > 0;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    __shared__ SelectShared<kThreads> sel_sh;
    __shared__ int s_state;
    const uint32_t raw = smem_u32(smem_raw);
    uint8_t *smem = smem_raw + (((raw + 1023u) & ~1023u) - raw);
    const uint32_t sbase = smem_u32(smem);
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + kOffBar);
    Misc *misc = reinterpret_cast<Misc *>(smem + kOffMisc);
    volatile int *abort = &misc->abort;
    float *sc = reinterpret_cast<float *>(smem + kOffSc);
    float *sw = reinterpret_cast<float *>(smem + kOffW);
    int *blk = reinterpret_cast<int *>(smem + kOffBlk);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int row = blockIdx.x;
    const int bq = row / p.L, j = row - bq * p.L;
    const int64_t k0 = p.key_off[bq];
    const int64_t Np = p.key_off[bq + 1] - k0;

    // ---- every independent global load first: kept blocks, q, weights, offsets ----
    constexpr int kQU = kH * 16 / kLoaders;                    // 16-byte q units per loader
    const int lt = tid - kLoadWarp0 * 32;                      // loader index (warps 5-8)
    float4 qf[QBF16 ? 1 : 2 * kQU];
    uint4 qh[QBF16 ? kQU : 1];
    float wv = 0.f;
    if (MODE == kFine)
        for (int e = tid; e < p.keep; e += kThreads) blk[e] = p.top_blk[(int64_t)row * p.keep + e];
    if (warp >= kLoadWarp0) {
        if (QBF16) {
            const uint4 *q16 = reinterpret_cast<const uint4 *>(
                reinterpret_cast<const __nv_bfloat16 *>(p.q) + (int64_t)row * kH * kD);
#pragma unroll
            for (int m = 0; m < kQU; ++m) qh[m] = __ldg(q16 + lt + m * kLoaders);
        } else {
            const float4 *q4 = reinterpret_cast<const float4 *>(
                reinterpret_cast<const float *>(p.q) + (int64_t)row * kH * kD);
#pragma unroll
            for (int m = 0; m < kQU; ++m) {
                qf[2 * m] = __ldg(q4 + 2 * (lt + m * kLoaders));
                qf[2 * m + 1] = __ldg(q4 + 2 * (lt + m * kLoaders) + 1);
            }
        }
        if (lt < kH) wv = __ldg(p.w + (int64_t)row * kH + lt);
    }
    __syncthreads();

    // ---- per-row validity (uniform over the CTA) and barrier set-up ----
    if (tid == 0) {
        int st = 0;
        const bool first = blockIdx.y == 0;
        if (!seq_ok(p.key_off, bq, p.Np_max, p.keys_rows)) {
            st = 1;
            if (first) flag(p.status, HISA_DEV_BAD_OFFSETS);
        } else if (MODE != kFlat && Np < (int64_t)p.b * p.keep) {
            st = 1;
            flag(p.status, HISA_DEV_GATE);
        } else if (MODE == kCoarse && (!means_ok(p.means_off, bq, Np / p.b, p.means_rows) ||
                                       (!split && Np / p.b > kMaxSel))) {
            st = 1;
            flag(p.status, HISA_DEV_BAD_OFFSETS);
        } else if (MODE == kFine) {
            for (int s = 1; s < p.keep; ++s) {     // insertion sort: candidates in ascending pos
                const int v = blk[s];
                int u = s;
                while (u > 0 && blk[u - 1] > v) { blk[u] = blk[u - 1]; --u; }
                blk[u] = v;
            }
            for (int s = 0; s < p.keep; ++s)
                if (blk[s] < 0 || (int64_t)blk[s] >= Np / p.b) st = 1;
            if (st) flag(p.status, HISA_DEV_BAD_BLOCK);
        }
        for (int b = 0; b < kNumBars; ++b) {
            uint32_t cnt = 1;
            if (b >= kBarFull && b < kBarFull + kSlots) cnt = MODE == kCoarse ? kLoaders : 1;
            if (b == kBarQ) cnt = kLoaders;
            if (b == kBarDFree) cnt = kEpis;
            mbar_init(&bars[b], cnt);
        }
        mbar_fence_init();
        misc->abort = 0;
        s_state = st;
    }
    __syncthreads();
    if (s_state) {
        if (MODE != kFlat && P.sel)
            for (int e = tid; e < P.k_sel; e += kThreads) P.sel[(int64_t)row * P.k_sel + e] = -1;
        return;
    }
    const int64_t n = MODE == kFlat ? Np : (MODE == kCoarse ? Np / p.b : (int64_t)p.keep * p.b);
    const int T_all = (int)((n + kTile - 1) / kTile);
    int t_begin = 0, t_end = T_all;
    if (split) {
        t_begin = (int)blockIdx.y * P.tiles_per_cta;
        t_end = t_begin + P.tiles_per_cta < T_all ? t_begin + P.tiles_per_cta : T_all;
        if (t_begin >= t_end) return;
    }
    const int T = t_end - t_begin;
    const int64_t V = p.causal ? visible_len((int64_t)p.t0[bq] + j, p.r, Np) : Np;

    // bf16 rows: one loader thread streams each 64-row tile as two TMA boxes (64 rows x
    // 64 dims, 128-byte swizzle). A fine tile is one kept block (index_block = 64); a flat
    // tile is 64 consecutive rows. Rows past Np or past the allocation are loaded as zeros
    // or never scored.
    auto issue_tile = [&](int i) {
        const int s = i % kSlots;
        const uint32_t slot = sbase + kOffRows + s * kPlaneRows;
        const int64_t c0 = (int64_t)(t_begin + i) * kTile;
        const int64_t y = MODE == kFine ? k0 + (int64_t)blk[c0 >> 6] * 64 : k0 + c0;
        mbar_arrive_expect_tx(&bars[kBarFull + s], 2u * 8192u);
#pragma unroll
        for (int ch = 0; ch < 2; ++ch)
            tma_load_2d(slot + ch * (kTile * 128), &P.keys_map, ch * 64, (int32_t)y, &bars[kBarFull + s]);
    };
    const int pre = MODE == kCoarse ? 0 : (T < kSlots ? T : kSlots);   // tiles issued up front
    if (MODE != kCoarse && warp >= kLoadWarp0 && lt == 0)
        for (int i = 0; i < pre; ++i) issue_tile(i);
    if (warp == kMmaWarp) {
        tmem_alloc(&misc->tmem, kTmemCols);
        tmem_relinquish();
    }
    if (warp >= kLoadWarp0) {
        // q planes from the registers loaded above
        if (QBF16) {
#pragma unroll
            for (int m = 0; m < kQU; ++m) {
                const int u = lt + m * kLoaders;
                *reinterpret_cast<uint4 *>(smem + kOffQ + q_off(0, u >> 4, u & 15, NQ)) = qh[m];
            }
        } else {
#pragma unroll
            for (int m = 0; m < kQU; ++m) {
                const int u = lt + m * kLoaders;
                const float x[8] = {qf[2 * m].x, qf[2 * m].y, qf[2 * m].z, qf[2 * m].w,
                                    qf[2 * m + 1].x, qf[2 * m + 1].y, qf[2 * m + 1].z, qf[2 * m + 1].w};
                uint4 pl[3];
                split3(x, pl);
#pragma unroll
                for (int k = 0; k < 3; ++k)
                    *reinterpret_cast<uint4 *>(smem + kOffQ + q_off(k, u >> 4, u & 15, NQ)) = pl[k];
            }
        }
        if (lt < kH) sw[lt] = wv * p.head_scale;
        fence_async_smem();
        mbar_arrive(&bars[kBarQ]);
    }
    fence_before_sync();
    __syncthreads();
    fence_after_sync();
    const uint32_t tmem = misc->tmem;
    bool ok = true;

    if (warp >= kLoadWarp0) {
        // ---------------- loaders ----------------
        const int uu = lt & 15, r0 = lt >> 4;             // unit uu of rows r0 + 8m
        if (MODE == kCoarse) {
            const float *means = reinterpret_cast<const float *>(p.rows) + p.means_off[bq] * kD;
            float4 reg[16];
            auto load_tile = [&](int ti) {
#pragma unroll
                for (int m = 0; m < 8; ++m) {
                    const int64_t c = (int64_t)ti * kTile + r0 + 8 * m;
                    if (c < n) {
                        const float4 *src = reinterpret_cast<const float4 *>(means + c * kD + uu * 8);
                        reg[2 * m] = __ldg(src);
                        reg[2 * m + 1] = __ldg(src + 1);
                    } else {
                        reg[2 * m] = reg[2 * m + 1] = make_float4(0.f, 0.f, 0.f, 0.f);
                    }
                }
            };
            load_tile(t_begin);
            for (int i = 0; i < T; ++i) {
                if (i >= 1 && !wait_bar(&bars[kBarEmpty], (i - 1) & 1, abort)) { ok = false; break; }
#pragma unroll
                for (int m = 0; m < 8; ++m) {
                    const float4 a = reg[2 * m], b = reg[2 * m + 1];
                    const float x[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
                    uint4 pl[3];
                    split3(x, pl);
                    const uint32_t off = unit_off(r0 + 8 * m, uu, kTile);
#pragma unroll
                    for (int k = 0; k < 3; ++k)
                        *reinterpret_cast<uint4 *>(smem + kOffRows + k * kPlaneRows + off) = pl[k];
                }
                fence_async_smem();
                mbar_arrive(&bars[kBarFull]);
                if (i + 1 < T) load_tile(t_begin + i + 1);
            }
        } else if (lt == 0) {
            int issued = pre;
            for (int i = pre; i < T; ++i) {
                if (!wait_bar(&bars[kBarEmpty + i % kSlots], ((i / kSlots) - 1) & 1, abort)) {
                    ok = false;
                    break;
                }
                issue_tile(i);
                ++issued;
            }
            if (!ok) {   // let the copies already in flight land before the CTA can exit
                for (int i = issued - 1; i >= 0 && i >= issued - kSlots; --i)
                    wait_bar(&bars[kBarFull + i % kSlots], (i / kSlots) & 1, abort);
            }
        }
    } else if (warp == kMmaWarp) {
        // ---------------- MMA issue (warp-uniform loop, one elected lane issues) -------
        // N = 64 * NQ: every q plane in one instruction; each rows plane is one MMA per
        // K step (the coarse stage's 3 x 3 plane pairs all accumulate, the smallest
        // ones below 2^-24 of the product included).
        const uint32_t idesc = idesc_bf16_f32(64, 64 * NQ, 0, 0);
        const uint64_t qd = smem_desc_sw128(sbase + kOffQ, 16, 1024);
        ok = wait_bar_warp(&bars[kBarQ], 0, abort);
        for (int i = 0; i < T && ok; ++i) {
            const int s = MODE == kCoarse ? 0 : i % kSlots;
            const uint32_t ph = MODE == kCoarse ? (uint32_t)(i & 1) : (uint32_t)((i / kSlots) & 1);
            if (!wait_bar_warp(&bars[kBarFull + s], ph, abort) ||
                (i >= 1 && !wait_bar_warp(&bars[kBarDFree], (i - 1) & 1, abort))) {
                ok = false;
                break;
            }
            fence_after_sync();
            const uint64_t rd = smem_desc_sw128(sbase + kOffRows + s * kPlaneRows, 16, 1024);
            const uint32_t d = tmem;
#pragma unroll
            for (int ks = 0; ks < kD / 16; ++ks) {
                const uint32_t ko = ks >> 2, kb = (ks & 3) * 32;
#pragma unroll
                for (int ra = 0; ra < NR; ++ra)
                    mma_bf16_warp(d, desc_add(rd, ra * kPlaneRows + ko * (kTile * 128) + kb),
                                  desc_add(qd, ko * (NQ * kH * 128) + kb), idesc,
                                  (ks > 0 || ra > 0) ? 1u : 0u);
            }
            mma_commit_warp(&bars[kBarEmpty + s]);
            mma_commit_warp(&bars[kBarDFull]);
        }
        mma_commit_warp(&bars[kBarDrain]);
        wait_bar_warp(&bars[kBarDrain], 0, abort);
    } else {
        // ---------------- epilogue: one row per thread ----------------
        const int quad = warp & 3;
        const int r = quad * 16 + lane;                 // valid for lane < 16 (M = 64 layout)
        ok = wait_bar(&bars[kBarQ], 0, abort);
        for (int i = 0; i < T && ok; ++i) {
            if (!wait_bar(&bars[kBarDFull], i & 1, abort)) { ok = false; break; }
            fence_after_sync();
            const uint32_t ta = tmem + ((uint32_t)(quad * 32) << 16);
            float acc = 0.f;
#pragma unroll
            for (int c = 0; c < 4; ++c) {           // 16 heads at a time: dot = sum over q planes
                float v[NQ][16];
#pragma unroll
                for (int qa = 0; qa < NQ; ++qa) tmem_ld16(ta + qa * 64 + c * 16, v[qa]);
                tmem_ld_wait();
#pragma unroll
                for (int q = 0; q < 16; ++q) {
                    float dot = v[0][q];
#pragma unroll
                    for (int qa = 1; qa < NQ; ++qa) dot += v[qa][q];
                    acc = fmaf(sw[c * 16 + q], fmaxf(dot, 0.f), acc);
                }
            }
            fence_before_sync();
            mbar_arrive(&bars[kBarDFree]);
            const int64_t cidx = (int64_t)(t_begin + i) * kTile + r;
            if (lane < 16 && cidx < n) {
                int64_t pos = cidx;
                if (MODE == kCoarse) pos = cidx * p.b;   // a block is eligible iff its first row is visible
                if (MODE == kFine) {
                    const uint32_t c32 = (uint32_t)cidx, b32 = (uint32_t)p.b, q32 = c32 / b32;
                    pos = (int64_t)blk[q32] * p.b + (c32 - q32 * b32);
                }
                const float score = pos < V ? acc : kNeg;
                if (!split) sc[cidx] = score;
                if (p.out) p.out[(int64_t)row * p.ld_out + cidx] = score;
            }
        }
    }
    if (!ok) {
        *abort = 1;
        flag(p.status, HISA_DEV_TIMEOUT);
    }
    fence_before_sync();
    __syncthreads();
    if (warp == kMmaWarp) {
        fence_after_sync();
        tmem_dealloc(tmem, kTmemCols);
    }
    if (!split) {
        int32_t *out = P.sel + (int64_t)row * P.k_sel;
        const int aborted = misc->abort;
        const int64_t kout = aborted ? 0 : (n < P.k_sel ? n : (int64_t)P.k_sel);
        // n <= kMaxSel <= kSmallMax scores in shared memory
        static_assert(kMaxSel <= kSmallMax, "fused select capacity");
        if (MODE == kFine) {
            const uint32_t b = (uint32_t)p.b;
            small_topk<kThreads, 0, 0>(
                sc, (int)n, (int)kout, out,
                [&](int64_t i) {
                    const uint32_t q32 = (uint32_t)i / b;
                    return (int32_t)((uint32_t)blk[q32] * b + ((uint32_t)i - q32 * b));
                },
                sel_sh, p.status);
        } else {
            small_topk<kThreads, 0, 0>(sc, (int)n, (int)kout, out, [](int64_t i) { return (int32_t)i; },
                                       sel_sh, p.status);
        }
        for (int64_t e = kout + tid; e < P.k_sel; e += kThreads) out[e] = -1;
    }
}

}  // namespace
}  // namespace hisa

namespace hisa {

int score_tc_split_ok(int mode, int H_i, int D_i, int rows_bf16, int b) {
    if (H_i != kH || D_i != kD) return 0;
    if (mode == kCoarse) return !rows_bf16;
    if (mode == kFine) return rows_bf16 && b == 64;
    return 0;
}

int score_tc_supported(int mode, int H_i, int D_i, int rows_bf16, int64_t n_max, int b) {
    if (H_i != kH || D_i != kD) return 0;
    if (mode == kCoarse) return !rows_bf16 && n_max <= kMaxSel;
    if (mode == kFine) return rows_bf16 && n_max <= kMaxSel && b == 64;
    return rows_bf16;
}

template <int MODE, bool QBF16>
static cudaError_t launch_t(const ScoreTcParams &p, dim3 grid, cudaStream_t s) {
    const cudaError_t attr = smem_attr_once<k_score_tc<MODE, QBF16>>((int)(kSmemFixed + kMaxSel * 4));
    if (attr != cudaSuccess) return attr;
    // the fused select keeps n scores in shared memory; split launches keep none
    const size_t smem = kSmemFixed + (p.tiles_per_cta > 0 ? 0 : (size_t)p.s.n_max * 4);
    k_score_tc<MODE, QBF16><<<grid, kThreads, smem, s>>>(p);
    return cudaGetLastError();
}

cudaError_t launch_score_tc(const ScoreTcParams &p_in, cudaStream_t s) {
    ScoreTcParams p = p_in;
    const int64_t rows = (int64_t)p.s.B * p.s.L;
    if (p.s.mode != kCoarse &&
        !encode_bf16_map(&p.keys_map, p.s.rows, (uint64_t)p.s.keys_rows, kD, 64, 64))
        return cudaErrorInvalidValue;
    dim3 grid((unsigned)rows, 1);
    const bool split = p.s.mode == kFlat || !p.sel;
    if (split) {
        const int64_t tiles = (p.s.n_max + kTile - 1) / kTile;
        if (tiles == 0) return cudaSuccess;
        int64_t tpc = (rows * tiles + kTargetCtas - 1) / kTargetCtas;
        if (tpc < 1) tpc = 1;
        if (tpc > tiles) tpc = tiles;
        p.tiles_per_cta = (int)tpc;
        grid.y = (unsigned)((tiles + tpc - 1) / tpc);
    }
    const bool qb = p.s.q_bf16 != 0;
    switch (p.s.mode) {
        case kFlat: return qb ? launch_t<kFlat, true>(p, grid, s) : launch_t<kFlat, false>(p, grid, s);
        case kCoarse:
            return qb ? launch_t<kCoarse, true>(p, grid, s) : launch_t<kCoarse, false>(p, grid, s);
        case kFine: return qb ? launch_t<kFine, true>(p, grid, s) : launch_t<kFine, false>(p, grid, s);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace hisa
