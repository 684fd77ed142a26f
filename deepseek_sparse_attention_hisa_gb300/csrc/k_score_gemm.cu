// Dense indexer scoring of many query rows of one sequence at once: the batched-prefill
// contraction L x Np x (H_i * D_i) of [HiSA issue] "Flat selection" (scores of every
// pooled row, NEG past V(t0 + j) when L > 1), for the DeepSeek-V4 indexer shape
// (H_i = 64, D_i = 128) with bf16 q and keys.
//
// A work unit is four consecutive query rows j0 .. j0 + 3 of one sequence. Their q (4 rows
// x 64 heads x 128 dims, bf16) stays in shared memory while every 128-key tile of the
// sequence streams past it: D[128 keys x 256] = keys . Q^T (M = 128, N = 4 x 64 = 256,
// K = 128) on tcgen05, f32 accumulators in TMEM (two buffers of 256 columns). bf16
// products are exact in the f32 accumulator, so the scores are f32 scoring of the bf16
// inputs. The epilogue thread of TMEM lane r owns key r of the tile: relu, head weights
// and the head sum in registers, then one coalesced store per row.
//
// One CTA per SM walks units blockIdx.x, blockIdx.x + gridDim.x, ... Warp 0 issues the
// MMAs and owns TMEM, warp 1 issues the TMA loads (q of a unit, then its key tiles into a
// four-slot ring), warps 2-9 form the epilogue (warp w reads TMEM lanes 32 (w % 4) ..
// + 31, for rows 2 ((w - 2) / 4) and 2 ((w - 2) / 4) + 1). Key tiles past the visible
// prefix of all four rows are not multiplied; their scores are written as NEG.
//
// The same kernel scores the coarse stage of many rows ([HiSA issue] "HiSA batched path":
// cscore over the block means, NEG for a block whose first row is not visible) with the
// f32 block means as the "keys": k_split_planes first splits each mean exactly into three
// bf16 planes (x = x1 + x2 + x3, truncation), and every 128-block tile is three key tiles
// (one per plane) whose products with the bf16 q accumulate in the same TMEM columns, so the
// scores are f32 scoring of the f32 means.
// Every wait is bounded; a timeout raises HISA_DEV_TIMEOUT, and the CTA drains and exits.
#include "hisa_internal.cuh"
#include "tc_ptx.cuh"

namespace hisa {
namespace {

using namespace tc;

constexpr int kH = 64, kD = 128, kM = 128, kRowsPerUnit = 4, kN = kRowsPerUnit * kH;
constexpr int kSlots = 4;
constexpr int kThreads = 320;                            // 10 warps
constexpr int kEpiThreads = 256;
constexpr int kBarEpi = 1;                               // named barrier of the epilogue
constexpr uint32_t kKeyTile = kM * kD * 2;               // 32 KiB
constexpr uint32_t kQBytes = kN * kD * 2;                // 64 KiB
constexpr uint32_t kOffQ = 0;
constexpr uint32_t kOffKeys = kOffQ + kQBytes;
constexpr uint32_t kOffW = kOffKeys + kSlots * kKeyTile;
constexpr uint32_t kOffBar = kOffW + kN * 4;
constexpr int kBarFull = 0, kBarEmpty = kSlots, kBarQFull = 2 * kSlots, kBarQEmpty = kBarQFull + 1,
              kBarAccFull = kBarQEmpty + 1, kBarAccEmpty = kBarAccFull + 2, kBarDrain = kBarAccEmpty + 2,
              kNumBars = kBarDrain + 1;
constexpr uint32_t kOffMisc = kOffBar + kNumBars * 8;
constexpr uint32_t kSmem = kOffMisc + 64 + 1024;         // + alignment slack

struct Misc {
    uint32_t tmem;
    int abort;
};

struct GemmParams {
    CUtensorMap keys_map;       // [keys_rows, 128] bf16, box 64 dims x 128 rows (coarse: the
                                // planes [3 * means_rows, 128], plane p of mean m at row
                                // p * means_rows + m)
    CUtensorMap q_map;          // [B * L * 64, 128] bf16, box 64 dims x 256 rows
    ScoreParams s;
    int units_per_seq;          // ceil(L / 4)
};

__device__ __forceinline__ bool wait_bar(uint64_t *bar, uint32_t parity, volatile int *abort) {
    return mbar_wait_abortable(bar, parity, abort);
}

__device__ __forceinline__ bool wait_bar_warp(uint64_t *bar, uint32_t parity, volatile int *abort) {
    return __all_sync(0xffffffffu, wait_bar(bar, parity, abort));
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

// What every role derives for a unit from the offsets alone. Flat: the scored rows are the
// sequence's pooled rows; coarse: its nb = floor(Np / b) block means.
struct Unit {
    int b, j0, rows;            // sequence, first row, rows of the unit in the sequence (<= 4)
    int64_t k0, Np;             // first scored row (pooled row / block-mean row), scored rows
    int64_t Np_seq;             // pooled rows of the sequence
    int T, Tv;                  // key tiles, tiles that reach into the visible prefix
    bool ok;
};

// Scored rows visible to the query row at position t: pooled rows p < V(t) (flat), blocks
// whose first row beta * b < V(t) (coarse).
template <int NP>
__device__ __forceinline__ int64_t visible_rows(const ScoreParams &p, int64_t t, int64_t Np, int64_t n) {
    const int64_t V = p.causal ? visible_len(t, p.r, Np) : Np;
    if (NP == 1) return V < n ? V : n;
    const int64_t vb = (V + p.b - 1) / p.b;
    return vb < n ? vb : n;
}

template <int NP>
__device__ __forceinline__ Unit unit_of(const ScoreParams &p, int units_per_seq, int u) {
    Unit x;
    x.b = u / units_per_seq;
    x.j0 = (u - x.b * units_per_seq) * kRowsPerUnit;
    x.rows = p.L - x.j0 < kRowsPerUnit ? p.L - x.j0 : kRowsPerUnit;
    x.ok = seq_ok(p.key_off, x.b, p.Np_max, p.keys_rows);
    x.Np_seq = x.ok ? p.key_off[x.b + 1] - p.key_off[x.b] : 0;
    if (NP == 1) {
        x.k0 = x.ok ? p.key_off[x.b] : 0;
        x.Np = x.Np_seq;
    } else {
        const int64_t nb = x.Np_seq / p.b;
        x.ok = x.ok && means_ok(p.means_off, x.b, nb, p.means_rows);
        x.k0 = x.ok ? p.means_off[x.b] : 0;
        x.Np = x.ok ? nb : 0;
    }
    x.T = (int)((x.Np + kM - 1) / kM);
    const int64_t Vl = visible_rows<NP>(p, (int64_t)(x.ok ? p.t0[x.b] : 0) + x.j0 + x.rows - 1,
                                        x.Np_seq, x.Np);
    x.Tv = (int)((Vl + kM - 1) / kM);
    return x;
}

// Three exact bf16 planes of each f32 block mean (truncation: x1 = the top 16 bits of x,
// x2 = the top 16 bits of x - x1, x3 = x - x1 - x2, which has at most 8 significant bits).
__global__ void k_split_planes(const float *means, int64_t n, __nv_bfloat16 *planes, int64_t plane_stride) {
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n;
         i += (int64_t)gridDim.x * blockDim.x) {
        const float x = means[i];
        const float x1 = __uint_as_float(__float_as_uint(x) & 0xffff0000u);
        const float r1 = x - x1;
        const float x2 = __uint_as_float(__float_as_uint(r1) & 0xffff0000u);
        const float x3 = r1 - x2;
        planes[i] = __float2bfloat16_rz(x1);
        planes[plane_stride + i] = __float2bfloat16_rz(x2);
        planes[2 * plane_stride + i] = __float2bfloat16_rz(x3);
    }
}

template <int NP>
__global__ void __launch_bounds__(kThreads, 1) k_score_gemm(const __grid_constant__ GemmParams P) {
    const ScoreParams &p = P.s;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    uint8_t *smem = smem_raw + (((raw + 1023u) & ~1023u) - raw);
    const uint32_t sbase = smem_u32(smem);
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + kOffBar);
    Misc *misc = reinterpret_cast<Misc *>(smem + kOffMisc);
    volatile int *abort = &misc->abort;
    float *sw = reinterpret_cast<float *>(smem + kOffW);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int units = p.B * P.units_per_seq;

    if (tid == 0) {
        for (int b = 0; b < kNumBars; ++b) {
            uint32_t cnt = 1;
            if (b == kBarAccEmpty || b == kBarAccEmpty + 1) cnt = kEpiThreads;
            mbar_init(&bars[b], cnt);
        }
        mbar_fence_init();
        misc->abort = 0;
    }
    if (warp == 0) {
        tmem_alloc(&misc->tmem, 512);
        tmem_relinquish();
    }
    fence_before_sync();
    __syncthreads();
    fence_after_sync();
    const uint32_t tmem = misc->tmem;
    grid_dep_wait();                                    // before the first global access
    bool ok = true;
    auto fail = [&]() {
        ok = false;
        *abort = 1;
    };

    if (warp == 1) {
        // ---------------- TMA producer ----------------
        if (lane == 0) {
            uint32_t g = 0;                                      // key tiles issued
            int i = 0;                                           // valid units so far
            for (int u = blockIdx.x; u < units && ok; u += gridDim.x) {
                const Unit x = unit_of<NP>(p, P.units_per_seq, u);
                if (!x.ok) {
                    if (x.j0 == 0) flag(p.status, HISA_DEV_BAD_OFFSETS);
                    continue;
                }
                if (i >= 1 && !wait_bar(&bars[kBarQEmpty], (i - 1) & 1, abort)) { fail(); break; }
                ++i;
                mbar_arrive_expect_tx(&bars[kBarQFull], kQBytes);
                const int32_t qy = (int32_t)(((int64_t)x.b * p.L + x.j0) * kH);
#pragma unroll
                for (int ch = 0; ch < 2; ++ch)
                    tma_load_2d(sbase + kOffQ + ch * (kN * 128), &P.q_map, ch * 64, qy, &bars[kBarQFull]);
                for (int t = 0; t < x.Tv * NP && ok; ++t, ++g) {   // coarse: plane t % 3 of tile t / 3
                    const uint32_t s = g % kSlots, use = g / kSlots;
                    if (use >= 1 && !wait_bar(&bars[kBarEmpty + s], (use - 1) & 1, abort)) { fail(); break; }
                    mbar_arrive_expect_tx(&bars[kBarFull + s], kKeyTile);
                    const int32_t y = (int32_t)((int64_t)(t % NP) * p.means_rows + x.k0 +
                                                (int64_t)(t / NP) * kM);
#pragma unroll
                    for (int ch = 0; ch < 2; ++ch)
                        tma_load_2d(sbase + kOffKeys + s * kKeyTile + ch * (kM * 128), &P.keys_map,
                                    ch * 64, y, &bars[kBarFull + s]);
                }
            }
            if (!ok) {   // let the copies in flight land before the CTA can exit
                for (uint32_t h = g > kSlots ? g - kSlots : 0; h < g; ++h)
                    mbar_wait(&bars[kBarFull + h % kSlots], (h / kSlots) & 1, 1u << 20);
                if (i >= 1) mbar_wait(&bars[kBarQFull], (i - 1) & 1, 1u << 20);
            }
        }
    } else if (warp == 0) {
        // ---------------- MMA issue (warp-uniform loop, one elected lane issues) ----------
        const uint32_t idesc = idesc_bf16_f32(kM, kN, 0, 0);
        const uint64_t qd = smem_desc_sw128(sbase + kOffQ, 16, 1024);
        uint32_t g = 0;
        int i = 0;
        uint32_t gs = 0;                                 // key slots consumed
        for (int u = blockIdx.x; u < units && ok; u += gridDim.x) {
            const Unit x = unit_of<NP>(p, P.units_per_seq, u);
            if (!x.ok) continue;
            if (!wait_bar_warp(&bars[kBarQFull], i & 1, abort)) { fail(); break; }
            fence_after_sync();
            for (int t = 0; t < x.Tv; ++t, ++g) {
                const uint32_t ab = g & 1;
                if (g >= 2 && !wait_bar_warp(&bars[kBarAccEmpty + ab], ((g >> 1) - 1) & 1, abort)) {
                    fail();
                    break;
                }
                const uint32_t d = tmem + ab * 256;
                bool good = true;
                for (int pl = 0; pl < NP; ++pl, ++gs) {          // the tile's planes, one slot each
                    const uint32_t s = gs % kSlots;
                    if (!wait_bar_warp(&bars[kBarFull + s], (gs / kSlots) & 1, abort)) { good = false; break; }
                    fence_after_sync();
                    const uint64_t kd = smem_desc_sw128(sbase + kOffKeys + s * kKeyTile, 16, 1024);
#pragma unroll
                    for (int ks = 0; ks < kD / 16; ++ks) {
                        const uint32_t ko = ks >> 2, kb = (ks & 3) * 32;
                        mma_bf16_warp(d, desc_add(kd, ko * (kM * 128) + kb), desc_add(qd, ko * (kN * 128) + kb),
                                      idesc, (ks > 0 || pl > 0) ? 1u : 0u);
                    }
                    mma_commit_warp(&bars[kBarEmpty + s]);
                }
                if (!good) { fail(); break; }
                mma_commit_warp(&bars[kBarAccFull + ab]);
            }
            if (!ok) break;
            mma_commit_warp(&bars[kBarQEmpty]);
            ++i;
        }
        mma_commit_warp(&bars[kBarDrain]);
        mbar_wait(&bars[kBarDrain], 0, 1u << 24);
    } else {
        // ---------------- epilogue: TMEM lane = key of the tile ----------------
        const int et = tid - 64;
        const int quad = warp & 3, half = (warp - 2) >> 2;       // rows 2 half, 2 half + 1
        const int key = quad * 32 + lane;
        uint32_t g = 0;
        for (int u = blockIdx.x; u < units; u += gridDim.x) {
            // every epilogue thread votes here, so that a timeout ends the loop for all of them
            if (!group_all(kBarEpi, kEpiThreads, ok)) { fail(); break; }
            const Unit x = unit_of<NP>(p, P.units_per_seq, u);
            if (!x.ok) continue;
            // weights of the unit's rows (w * H_i^-1/2 * D_i^-1/2), once the last unit is done
            {
                const int r = et >> 6, h = et & 63;
                sw[et] = r < x.rows ? __ldg(p.w + ((int64_t)x.b * p.L + x.j0 + r) * kH + h) * p.head_scale
                                    : 0.f;
            }
            asm volatile("bar.sync %0, %1;" ::"n"(kBarEpi), "n"(kEpiThreads) : "memory");
            int64_t V[2];
            float *orow[2];
#pragma unroll
            for (int rr = 0; rr < 2; ++rr) {
                const int r = 2 * half + rr;
                const int j = x.j0 + r;
                V[rr] = r < x.rows ? visible_rows<NP>(p, (int64_t)p.t0[x.b] + j, x.Np_seq, x.Np) : 0;
                orow[rr] = r < x.rows ? p.out + ((int64_t)x.b * p.L + j) * p.ld_out : nullptr;
            }
            for (int t = 0; t < x.T; ++t) {
                float sc[2] = {kNeg, kNeg};
                if (t < x.Tv) {
                    const uint32_t ab = g & 1;
                    if (!wait_bar(&bars[kBarAccFull + ab], (g >> 1) & 1, abort)) { fail(); break; }
                    fence_after_sync();
                    const uint32_t ta = tmem + ab * 256 + half * 128 + ((uint32_t)(quad * 32) << 16);
#pragma unroll
                    for (int rr = 0; rr < 2; ++rr) {
                        const float *wr = sw + (2 * half + rr) * kH;
                        float acc = 0.f;
#pragma unroll
                        for (int c = 0; c < 4; c += 2) {
                            float v0[16], v1[16];
                            tmem_ld16(ta + rr * 64 + c * 16, v0);
                            tmem_ld16(ta + rr * 64 + (c + 1) * 16, v1);
                            tmem_ld_wait();
#pragma unroll
                            for (int h = 0; h < 16; ++h) {
                                acc = fmaf(wr[c * 16 + h], fmaxf(v0[h], 0.f), acc);
                                acc = fmaf(wr[(c + 1) * 16 + h], fmaxf(v1[h], 0.f), acc);
                            }
                        }
                        sc[rr] = acc;
                    }
                    fence_before_sync();
                    mbar_arrive(&bars[kBarAccEmpty + ab]);
                    ++g;
                }
                const int64_t pos = (int64_t)t * kM + key;
                if (pos < x.Np) {
#pragma unroll
                    for (int rr = 0; rr < 2; ++rr)
                        if (orow[rr]) orow[rr][pos] = pos < V[rr] ? sc[rr] : kNeg;
                }
            }
        }
    }

    if (!ok) flag(p.status, HISA_DEV_TIMEOUT);
    fence_before_sync();
    __syncthreads();
    if (warp == 0) {
        fence_after_sync();
        tmem_dealloc(tmem, 512);
    }
}

bool encode_map_rows(CUtensorMap *map, const void *base, uint64_t rows, uint32_t box_rows) {
    return encode_bf16_map(map, base, rows, kD, 64, box_rows);
}

}  // namespace

int score_gemm_supported(int H_i, int D_i, int q_bf16, int rows_bf16, int B, int L) {
    return H_i == kH && D_i == kD && q_bf16 && rows_bf16 && L >= kRowsPerUnit &&
           (int64_t)B * L * kH < ((int64_t)1 << 31);
}

template <int NP>
cudaError_t launch_gemm_t(const ScoreParams &s, const void *key_rows, uint64_t n_key_rows,
                          cudaStream_t stream) {
    GemmParams P{};
    P.s = s;
    P.units_per_seq = (s.L + kRowsPerUnit - 1) / kRowsPerUnit;
    const int64_t units = (int64_t)s.B * P.units_per_seq;
    if (units == 0 || n_key_rows == 0) return cudaSuccess;
    if (!encode_map_rows(&P.keys_map, key_rows, n_key_rows, kM) ||
        !encode_map_rows(&P.q_map, s.q, (uint64_t)s.B * s.L * kH, kN))
        return cudaErrorInvalidValue;
    const cudaError_t attr = smem_attr_once<k_score_gemm<NP>>((int)kSmem);
    if (attr != cudaSuccess) return attr;
    const int sms = device_sm_count();
    if (sms <= 0) return cudaErrorInvalidDevice;
    const int grid = units < sms ? (int)units : sms;
    return launch_pdl(k_score_gemm<NP>, dim3(grid), dim3(kThreads), kSmem, stream, s.chained, P);
}

cudaError_t launch_score_gemm(const ScoreParams &s, cudaStream_t stream) {
    if (s.keys_rows == 0) return cudaSuccess;
    return launch_gemm_t<1>(s, s.rows, (uint64_t)s.keys_rows, stream);
}

size_t coarse_gemm_planes_bytes(int64_t means_rows) { return (size_t)means_rows * kD * 2 * 3; }

cudaError_t launch_coarse_gemm(const ScoreParams &s, void *planes, cudaStream_t stream) {
    if (s.means_rows == 0) return cudaSuccess;
    const int64_t n = s.means_rows * kD;
    const int64_t blocks = (n + 255) / 256 < 4096 ? (n + 255) / 256 : 4096;
    // the planes are this call's own scratch: nothing before the call writes them, and the
    // means are read after the previous kernel (the block-mean append) has completed
    cudaError_t e = launch_pdl(k_split_planes, dim3((unsigned)blocks), dim3(256), 0, stream, 0,
                               static_cast<const float *>(s.rows), n,
                               static_cast<__nv_bfloat16 *>(planes), n);
    if (e != cudaSuccess) return e;
    return launch_gemm_t<3>(s, planes, (uint64_t)(3 * s.means_rows), stream);
}

}  // namespace hisa
