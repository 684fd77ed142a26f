// Coarse and fine indexer stages of the DeepSeek-V4 indexer shape (H_i = 64, D_i = 128) as
// one persistent, warp-specialised tcgen05 pipeline per SM: score, then select, for a
// stream of query rows ([HiSA issue] "HiSA decode path" and "HiSA batched path": the
// coarse stage scores the block means and keeps the top Kb blocks, the fine stage scores
// the rows of the kept blocks and keeps the top k).
//
//   score[c] = sum_h relu(q_h . row_c) * w_h * H_i^-1/2 * D_i^-1/2, NEG past visibility.
//
// One CTA per SM walks the query rows blockIdx.x, blockIdx.x + gridDim.x, ... Its warps
// form a pipeline, so that one query's set-up and top-k overlap the next query's
// streaming and only the first set-up and the last top-k are exposed:
//   warp 0      MMA issue (one elected lane) and TMEM owner
//   warp 1      fine: TMA producer of the kept blocks' bf16 key tiles (a three-slot
//               ring); coarse: TMA of the f32 block means, [128 rows x 32 dims] boxes
//               into seven raw slots
//   warps 2-5   epilogue: TMEM -> relu, head weights, head sum -> scores in shared memory
//   warps 6-9   builders: per-query checks, kept blocks, head weights, q planes (two
//               q buffers, so the next query's are written while this one streams);
//               coarse, appending: the means of the newly completed blocks
//   warps 10-13 select: block top-k over the finished query's scores (named barrier 1)
//   warps 14-21 coarse: converters, f32 block means -> three bf16 planes in TMEM, where
//               they are the MMA's A operand (an eight-box ring)
//
// A tile is 128 scored rows, D = rows . q^T (M = 128, K = 128) in one of two TMEM
// accumulators (fine: [128 x 64 * q planes], coarse: [128 x 64]). Scoring is f32 on the page; f32 operands are split
// exactly into bf16 planes x = x1 + x2 + x3 (q: each plane the bf16 rounding of the
// remainder; block means: the remainder truncated to its top 8 significant bits, which is
// cheaper to form), so every bf16 product is exact in the f32 accumulator. The q planes
// are stacked along N. bf16 keys take one MMA per K step over all q planes. f32 block
// means take six of the nine plane products (x1 y1, x1 y2, x1 y3, x2 y1, x2 y2, x3 y1), one
// N = 64 MMA each, all accumulated into the same [128 x 64] accumulator:
// with |x2| < 2^-7 |x|, |x3| < 2^-14 |x|, |y2| <= 2^-8 |y| and |y3| <= 2^-16 |y|, the three
// left out (x2 y3, x3 y2, x3 y3) add up to less than 2^-21 of |x y|.
// Every wait is bounded; a timeout raises HISA_DEV_TIMEOUT, and the CTA drains and exits.
#include "pipe_common.cuh"

namespace hisa {
namespace {

using namespace tc;
using namespace pipe;

constexpr int kWarpMma = 0, kWarpTma = 1, kWarpEpi = 2, kWarpBld = 6, kWarpSel = 10, kWarpCvt = 14;
constexpr int kCvtWarps = 8, kCvtThreads = kCvtWarps * 32;  // coarse converters
constexpr int kBarSel = 1, kBarBld = 2;                   // named barriers (0 = __syncthreads)

template <int MODE>
constexpr int pipe_threads() { return MODE == kCoarse ? (kWarpCvt + kCvtWarps) * 32 : 14 * 32; }

// ---- shared memory (offsets from the 1024-aligned base) ----
constexpr uint32_t kOffQ = 0;                             // up to 3 planes, stacked along N
// two q buffers, so that the next query's planes are written while this one streams
template <int MODE>
constexpr int q_bufs() { return 2; }
// bytes of one q buffer: coarse keeps room for three planes, fine for its NQ planes (1 for
// bf16 q, 3 for f32 q), and the fine ring takes the rest: 5 key tiles with bf16 q, 3 with f32
template <int MODE, int NQ>
constexpr uint32_t q_span() { return MODE == kFine ? NQ * kQPlane : 3 * kQPlane; }
template <int MODE, int NQ>
constexpr uint32_t off_reg() { return q_bufs<MODE>() * q_span<MODE, NQ>(); }   // streaming region
template <int NQ>
constexpr int fine_slots() { return NQ == 1 ? 5 : 3; }
constexpr uint32_t kTileBytes = kM * kD * 2;              // fine: one [128 x 128] bf16 key tile
constexpr uint32_t kRawBytes = kM * 32 * 4;               // coarse: f32 means, 128 rows x 32 dims
constexpr int kRawSlots = 7;                              // coarse raw boxes in flight
// coarse TMEM: two [128 x 64] f32 accumulators in columns 0-127, then kASlots converted
// boxes, each three bf16 planes of 16 columns (the MMA's A operand, lane = tile row)
constexpr int kASlots = 8;
constexpr uint32_t kAColBase = 128, kABoxCols = 48;
static_assert(kAColBase + kASlots * kABoxCols <= 512, "coarse TMEM");
// coarse: kRawSlots raw f32 boxes; fine: the key tile ring
template <int MODE, int NQ>
constexpr uint32_t region_bytes() {
    return MODE == kCoarse ? kRawSlots * kRawBytes : fine_slots<NQ>() * kTileBytes;
}
// TMEM columns between the two accumulators
template <int MODE>
constexpr uint32_t acc_stride() { return MODE == kCoarse ? 64 : 256; }
constexpr uint32_t kOffReg = 2 * 3 * kQPlane;             // coarse streaming region
static_assert(off_reg<kCoarse, 1>() == kOffReg && off_reg<kCoarse, 3>() == kOffReg, "coarse layout");

struct QMeta {            // one query row, double-buffered
    int row;              // b * L + j
    int state;            // 0: score it; else its selection is all -1
    int n;                // scored rows: blocks (coarse) or candidates (fine)
    int T;                // tiles of kM rows
    int t_new;            // coarse, appending: the tile holding the first new block (T: none)
    long long base;       // first pooled row (fine) / first block-mean row (coarse)
    long long V;          // visible pooled rows of this query row
    int blk[64];          // kept blocks, ascending (fine)
    float w[kH];          // w_h * H_i^-1/2 * D_i^-1/2
};

// barriers
constexpr int kBarMetaFull = 0, kBarSlotFree = 2, kBarQFull = 4, kBarQEmpty = 6,
              kBarAccFull = 8, kBarAccEmpty = 10, kBarScFull = 12, kBarDrain = 14,
              kBarFull = 15,                // fine: its key slots; coarse: kASlots TMEM boxes, then kRawSlots raw
              kBarEmpty = kBarFull + kASlots + kRawSlots, kBarMeansReady = kBarEmpty + kASlots + kRawSlots,
              kNumBars = kBarMeansReady + 2;

template <int MODE, int NQ>
struct Layout {
    static constexpr uint32_t meta = off_reg<MODE, NQ>() + region_bytes<MODE, NQ>();
    static constexpr uint32_t bars = meta + 2 * sizeof(QMeta);
    static constexpr uint32_t misc = bars + kNumBars * 8;
    static constexpr uint32_t sc = (misc + 64 + 15) & ~15u;   // 2 x n_cap floats
    static constexpr uint32_t fixed = sc + 1024;                // + alignment slack
};

// Largest scored-row count one query may have: shared memory holds two score rows.
constexpr int kPipeMaxCoarse = 1024;
constexpr int kPipeMaxFine = 48 * 64;
static_assert(kPipeMaxFine <= kSmallMax && kPipeMaxCoarse <= kSmallMax, "select capacity");

// 227 KiB of shared memory per CTA: the layout, two score rows at capacity and the static
// select state (kept blocks and the select warps' SelectShared)
template <int MODE, int NQ>
constexpr bool fits() {
    constexpr int cap = MODE == kCoarse ? kPipeMaxCoarse : kPipeMaxFine;
    return Layout<MODE, NQ>::fixed + 2 * cap * 4 + sizeof(SelectShared<kGroup>) + 256 <=
           227 * 1024;
}
static_assert(fits<kCoarse, 1>() && fits<kCoarse, 3>() && fits<kFine, 1>() && fits<kFine, 3>(),
              "shared memory");
static_assert(fine_slots<1>() <= kASlots + kRawSlots && fine_slots<3>() <= kASlots + kRawSlots, "barriers");

}  // namespace
}  // namespace hisa

namespace hisa {
namespace {

// Candidate column -> absolute pooled id through the kept blocks (fine), or itself (coarse):
// named types, so that every select of a stage shares one instantiation of the select code.
struct FineIds {
    const int *blk;
    __device__ __forceinline__ int32_t operator()(int64_t c) const {
        return (int32_t)(blk[(int)c >> 6] * 64 + ((int)c & 63));
    }
};
struct OffsetIds {                        // coarse: block id = chunk start + column
    int off;
    __device__ __forceinline__ int32_t operator()(int64_t c) const { return (int32_t)(off + c); }
};


// Registers: 14 (fine) or 22 (coarse) warps spread over the SM's four 16K-register
// sub-partitions, so at most 128 or 88 registers per thread.
template <int MODE, bool QBF16>
__global__ void __launch_bounds__(pipe_threads<MODE>(), 1)
    k_score_pipe(const __grid_constant__ ScoreTcParams P) {
    constexpr int NQ = QBF16 ? 1 : 3;                       // q planes
    constexpr int kQB = q_bufs<MODE>();
    using Lay = Layout<MODE, NQ>;
    constexpr int kFineSlots = fine_slots<NQ>();
    const ScoreParams &p = P.s;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    __shared__ SelectShared<kGroup> sel_sh;             // the select warps' state
    __shared__ int s_blk_raw[64];                       // kept blocks as read (fine)
    const uint32_t raw = smem_u32(smem_raw);
    uint8_t *smem = smem_raw + (((raw + 1023u) & ~1023u) - raw);
    const uint32_t sbase = smem_u32(smem);
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + Lay::bars);
    QMeta *meta = reinterpret_cast<QMeta *>(smem + Lay::meta);
    Misc *misc = reinterpret_cast<Misc *>(smem + Lay::misc);
    volatile int *abort = &misc->abort;
    float *scb = reinterpret_cast<float *>(smem + Lay::sc);
    const int n_cap = (int)p.n_max;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    // coarse rows longer than kCoarseChunk blocks run as P.chunks virtual rows each
    const int nch = MODE == kCoarse && P.chunks > 1 ? P.chunks : 1;
    const int rows = p.B * p.L * nch;
    const int nql = (int)blockIdx.x < rows ? (rows - 1 - (int)blockIdx.x) / (int)gridDim.x + 1 : 0;

    // The first query's q, weights and offsets into L2 while the barriers and TMEM are set
    // up (a prefetch only warms L2, which every write reaches first, so it is safe whatever
    // the previous kernel writes).
    if (warp >= kWarpBld && warp < kWarpBld + 4 && nql > 0) {
        const int bt = tid - kWarpBld * 32;
        const int row = (int)blockIdx.x / nch, bq = row / p.L;
        const char *qrow = static_cast<const char *>(p.q) + (int64_t)row * kH * kD * (QBF16 ? 2 : 4);
        for (int o = bt * 128; o < kH * kD * (QBF16 ? 2 : 4); o += kGroup * 128)
            asm volatile("prefetch.global.L2 [%0];" ::"l"(qrow + o));
        if (bt < 2) asm volatile("prefetch.global.L2 [%0];" ::"l"(reinterpret_cast<const char *>(p.w + (int64_t)row * kH) + 128 * bt));
        if (bt == 2) asm volatile("prefetch.global.L2 [%0];" ::"l"(p.key_off + bq));
        if (bt == 3) asm volatile("prefetch.global.L2 [%0];" ::"l"(p.t0 + bq));
        if (MODE == kCoarse && bt == 4) asm volatile("prefetch.global.L2 [%0];" ::"l"(p.means_off + bq));
        if (MODE == kCoarse && bt == 5 && P.first_block)
            asm volatile("prefetch.global.L2 [%0];" ::"l"(P.first_block + bq));
    }

    if (tid == 0) {
        for (int b = 0; b < kNumBars; ++b) {
            uint32_t cnt = 1;
            if (b == kBarQFull || b == kBarQFull + 1 || b == kBarAccEmpty || b == kBarAccEmpty + 1 || b == kBarScFull ||
                b == kBarScFull + 1 || b == kBarMeansReady || b == kBarMeansReady + 1)
                cnt = kGroup;
            // coarse: Full / Empty + 0 .. kASlots - 1 guard the TMEM boxes, the next kRawSlots
            // the raw slots
            if (MODE == kCoarse && b >= kBarFull && b < kBarFull + kASlots) cnt = kCvtThreads;
            if (MODE == kCoarse && b >= kBarEmpty + kASlots && b < kBarEmpty + kASlots + kRawSlots)
                cnt = kCvtThreads;
            mbar_init(&bars[b], cnt);
        }
        mbar_fence_init();
        misc->abort = 0;
    }
    if (warp == kWarpMma) {
        tmem_alloc(&misc->tmem, 512);
        tmem_relinquish();
    }
    fence_before_sync();
    __syncthreads();
    fence_after_sync();
    const uint32_t tmem = misc->tmem;
    // coarse: before the first global access; fine: its builders wait before the first kept
    // blocks (the coarse output), so that q, w and the offsets load while the coarse stage ends
    if (MODE == kCoarse) grid_dep_wait();
    bool ok = true;
    auto fail = [&]() {
        ok = false;
        *abort = 1;
    };

    if (warp >= kWarpBld && warp < kWarpBld + 4) {
        // ---------------- builders: checks, kept blocks, weights, q planes ----------------
        const int bt = tid - kWarpBld * 32;
        for (int i = 0; i < nql; ++i) {
            const int qb = i & 1;
            const int vrow = (int)blockIdx.x + i * (int)gridDim.x;
            const int row = vrow / nch, chunk = vrow - row * nch;
            const int bq = row / p.L, j = row - bq * p.L;
            // this row's weights, offsets and position first (the row's checks and the loader's
            // first copies wait on them), then q, then the kept blocks: the loads overlap the
            // waits. With 22 warps (coarse, f32 q) only half of q is held in registers; the other
            // half is prefetched into L2 and read once the previous query's planes are free.
            const float wv = bt < kH ? __ldg(p.w + (int64_t)row * kH + bt) : 0.f;
            const int64_t k0 = p.key_off[bq], k1 = p.key_off[bq + 1];
            int64_t m0 = 0, m1 = 0, fb = 0;
            if (MODE == kCoarse) {
                m0 = p.means_off[bq];
                m1 = p.means_off[bq + 1];
                if (P.append_keys && P.first_block) fb = P.first_block[bq];
                fb = fb < 0 ? 0 : fb;
            }
            const int64_t t_row = p.causal ? (int64_t)p.t0[bq] + j : 0;
            QRegs<QBF16, MODE == kCoarse> qr;
            qr.load(p.q, row, bt);
            if (MODE == kFine && i == 0) {
                grid_dep_wait();
                // the fine form lets a chained successor (the combine) launch now: its CTAs
                // take each SM as this kernel's CTA there exits and load their first item's
                // q and local rows while the last selections finish
                grid_dep_trigger();
            }
            int bv = 0;
            if (MODE == kFine && bt < p.keep) bv = __ldg(p.top_blk + (int64_t)row * p.keep + bt);
            // meta slot qb is free once query i - 2 is selected
            const bool w1 = i < 2 || wait_bar(&bars[kBarSlotFree + qb], ((i >> 1) - 1) & 1, abort);
            if (!group_all(kBarBld, kGroup, w1)) { fail(); break; }
            QMeta &M = meta[qb];
            const int64_t Np = k1 - k0;
            if (MODE == kFine && bt < p.keep) s_blk_raw[bt] = bv;
            if (bt < kH) M.w[bt] = wv * p.head_scale;
            named_sync(kBarBld, kGroup);
            bool bad_blk = false;
            if (MODE == kFine && bt < p.keep) {
                // kept blocks in ascending order: each thread places its own by rank
                int rank = 0;
                for (int u = 0; u < p.keep; ++u) {
                    const int o = s_blk_raw[u];
                    rank += (o < bv || (o == bv && u < bt)) ? 1 : 0;
                }
                M.blk[rank] = bv;
                bad_blk = bv < 0 || (int64_t)bv >= Np / 64;
            }
            bad_blk = MODE == kFine && !group_all(kBarBld, kGroup, !bad_blk);
            bool w2 = true;
            if (bt == 0) {
                int st = 0;
                int64_t n = 0, base = k0;
                if (!seq_ok_v(k0, k1, p.Np_max, p.keys_rows)) {
                    st = 1;
                    flag(p.status, HISA_DEV_BAD_OFFSETS);
                } else if (Np < (int64_t)p.b * p.keep) {
                    st = 1;
                    flag(p.status, HISA_DEV_GATE);
                } else if (MODE == kCoarse) {
                    const int64_t nb = Np / p.b;
                    const int64_t c0 = (int64_t)chunk * kCoarseChunk;
                    n = nb - c0 < kCoarseChunk ? nb - c0 : kCoarseChunk;   // this chunk's blocks
                    base = m0 + c0;
                    if (!means_ok_v(m0, m1, nb, p.means_rows) || n > n_cap ||
                        nb > (int64_t)nch * kCoarseChunk) {
                        st = 1;
                        n = 0;
                        flag(p.status, HISA_DEV_BAD_OFFSETS);
                    } else if (n <= 0) {
                        st = 2;                           // a chunk past this row's blocks
                        n = 0;
                    }
                } else {
                    n = (int64_t)p.keep * 64;
                    if (bad_blk) {
                        st = 1;
                        flag(p.status, HISA_DEV_BAD_BLOCK);
                    }
                }
                M.row = row;
                M.state = st;
                M.n = (int)n;
                M.T = (int)((n + kM - 1) / kM);
                // the chunk's first new block (chunk-local), if it holds any
                const int64_t fbl = fb - (int64_t)chunk * kCoarseChunk;
                M.t_new = fbl < n ? (int)((fbl > 0 ? fbl : 0) / kM) : M.T;
                M.base = base;
                M.V = p.causal ? visible_len(t_row, p.r, Np) : Np;
                mbar_arrive(&bars[kBarMetaFull + qb]);
                // the q planes are free once the previous query's MMAs are done
                w2 = i < kQB || wait_bar(&bars[kBarQEmpty + i % kQB], (i / kQB - 1) & 1, abort);
            }
            if (!group_all(kBarBld, kGroup, w2)) { fail(); break; }
            const uint32_t qoff = kOffQ + (uint32_t)(i % kQB) * q_span<MODE, NQ>();
            qr.store(smem + qoff, bt);
            fence_async_smem();
            mbar_arrive(&bars[kBarQFull + i % kQB]);
            if (MODE == kCoarse && P.append_keys) {
                // block means of the newly completed blocks [first_block, nb)
                const QMeta &M = meta[qb];
                if (!M.state) {
                    // this chunk's new blocks, chunk-local: keys from block c0, means from base
                    const int64_t c0 = (int64_t)chunk * kCoarseChunk;
                    const int64_t fbl = fb - c0 > 0 ? fb - c0 : 0;
                    append_block_means(reinterpret_cast<const uint4 *>(P.append_keys), k0 + c0 * 64, fbl, M.n,
                                       const_cast<float *>(reinterpret_cast<const float *>(p.rows)), M.base, bt);
                    fence_async_global();               // the loader reads them by TMA
                }
                mbar_arrive(&bars[kBarMeansReady + qb]);
            }
        }
    }
    else if (MODE == kFine && warp == kWarpTma) {
        // ---------------- TMA producer: kept blocks, two per 128-row tile ----------------
        if (lane == 0) {
            uint32_t g = 0;                                    // tiles issued
            for (int i = 0; i < nql && ok; ++i) {
                const int qb = i & 1;
                if (!wait_bar(&bars[kBarMetaFull + qb], (i >> 1) & 1, abort)) { fail(); break; }
                const QMeta &M = meta[qb];
                if (M.state) continue;
                for (int t = 0; t < M.T; ++t, ++g) {
                    const uint32_t s = g % kFineSlots, use = g / kFineSlots;
                    if (use >= 1 && !wait_bar(&bars[kBarEmpty + s], (use - 1) & 1, abort)) {
                        fail();
                        break;
                    }
                    const int nblk = p.keep - 2 * t < 2 ? p.keep - 2 * t : 2;
                    const uint32_t slot = sbase + off_reg<MODE, NQ>() + s * kTileBytes;
                    mbar_arrive_expect_tx(&bars[kBarFull + s], (uint32_t)nblk * 16384u);
                    for (int hb = 0; hb < nblk; ++hb) {
                        const int32_t y = (int32_t)(M.base + (int64_t)M.blk[2 * t + hb] * 64);
#pragma unroll
                        for (int ch = 0; ch < 2; ++ch)
                            tma_load_2d(slot + ch * (kM * 128) + hb * (64 * 128), &P.keys_map, ch * 64, y,
                                        &bars[kBarFull + s]);
                    }
                }
            }
            if (!ok)   // let the copies in flight land before the CTA can exit
                for (uint32_t h = g > kFineSlots ? g - kFineSlots : 0; h < g; ++h)
                    mbar_wait(&bars[kBarFull + h % kFineSlots], (h / kFineSlots) & 1, 1u << 20);
        }
    } else if (MODE == kCoarse && warp == kWarpTma) {
        // ---------------- coarse loader: block means by TMA ----------------
        // Box v = one K quarter (32 dims) of one 128-row tile, a 128B-swizzled [128 rows x 32
        // dims] f32 box into raw slot v % kRawSlots; many small slots keep the bytes in flight
        // that the latency under load asks for. Rows past the allocation read as 0; rows past
        // the query's blocks are other data and never scored.
        if (lane == 0) {
            uint32_t u = 0;                                    // boxes issued
            for (int i = 0; i < nql && ok; ++i) {
                const int qb = i & 1;
                if (!wait_bar(&bars[kBarMetaFull + qb], (i >> 1) & 1, abort)) { fail(); break; }
                const QMeta &M = meta[qb];
                const int T = M.state ? 0 : M.T;
                // appended means: tiles from the one holding the first new block on wait for them
                const int t_new = P.append_keys ? M.t_new : T;
                for (int t = 0; t < T && ok; ++t) {
                    if (t == t_new && !wait_bar(&bars[kBarMeansReady + qb], (i >> 1) & 1, abort)) {
                        fail();
                        break;
                    }
                    for (int h = 0; h < 4; ++h, ++u) {
                        const uint32_t slot = u % kRawSlots, use = u / kRawSlots;
                        if (use >= 1 && !wait_bar(&bars[kBarEmpty + kASlots + slot], (use - 1) & 1, abort)) {
                            fail();
                            break;
                        }
                        mbar_arrive_expect_tx(&bars[kBarFull + kASlots + slot], kRawBytes);
                        const int32_t y = (int32_t)(M.base + (int64_t)t * kM);
                        tma_load_2d(sbase + kOffReg + slot * kRawBytes, &P.means_map, h * 32, y,
                                    &bars[kBarFull + kASlots + slot]);
                    }
                }
            }
            if (!ok)   // let the copies in flight land before the CTA can exit
                for (uint32_t v = u > kRawSlots ? u - kRawSlots : 0; v < u; ++v)
                    mbar_wait(&bars[kBarFull + kASlots + v % kRawSlots], (v / kRawSlots) & 1, 1u << 20);
        }
    } else if (warp == kWarpMma) {
        // ---------------- MMA issue (warp-uniform loop, one elected lane issues) ----------
        const uint32_t id_all = idesc_bf16_f32(kM, 64 * NQ, 0, 0);
        const uint32_t id_one = idesc_bf16_f32(kM, 64, 0, 0);

        uint32_t g = 0, gs = 0, u = 0;                       // tiles, fine slots, coarse boxes
        for (int i = 0; i < nql && ok; ++i) {
            const int qb = i & 1;
            if (!wait_bar_warp(&bars[kBarMetaFull + qb], (i >> 1) & 1, abort) ||
                !wait_bar_warp(&bars[kBarQFull + i % kQB], (i / kQB) & 1, abort)) {
                fail();
                break;
            }
            fence_after_sync();
            const uint64_t qd = smem_desc_sw128(sbase + kOffQ + (uint32_t)(i % kQB) * q_span<MODE, NQ>(), 16, 1024);
            const QMeta &M = meta[qb];
            const int T = M.state ? 0 : M.T;
            for (int t = 0; t < T; ++t, ++g) {
                const uint32_t ab = g & 1;
                if (g >= 2 && !wait_bar_warp(&bars[kBarAccEmpty + ab], ((g >> 1) - 1) & 1, abort)) {
                    fail();
                    break;
                }
                fence_after_sync();
                const uint32_t d = tmem + ab * acc_stride<MODE>();
                if (MODE == kFine) {
                    const uint32_t s = gs % kFineSlots;
                    if (!wait_bar_warp(&bars[kBarFull + s], (gs / kFineSlots) & 1, abort)) {
                        fail();
                        break;
                    }
                    fence_after_sync();
                    const uint64_t rd = smem_desc_sw128(sbase + off_reg<MODE, NQ>() + s * kTileBytes, 16, 1024);
#pragma unroll
                    for (int ks = 0; ks < kD / 16; ++ks) {
                        const uint32_t ko = ks >> 2, kb = (ks & 3) * 32;
                        mma_bf16_warp(d, desc_add(rd, ko * (kM * 128) + kb),
                                      desc_add(qd, ko * (NQ * kH * 128) + kb), id_all, ks > 0 ? 1u : 0u);
                    }
                    mma_commit_warp(&bars[kBarEmpty + s]);
                    ++gs;
                } else {
                    bool good = true;
                    for (int h = 0; h < 4; ++h, ++u) {           // the tile's four boxes
                        const uint32_t as = u % kASlots;
                        if (!wait_bar_warp(&bars[kBarFull + as], (u / kASlots) & 1, abort)) { good = false; break; }
                        fence_after_sync();
                        const uint32_t a0 = tmem + kAColBase + as * kABoxCols;
#pragma unroll
                        for (int kk = 0; kk < 2; ++kk) {
                            const uint32_t dim = h * 32 + kk * 16;
                            const uint64_t bq = desc_add(qd, (dim >> 6) * (NQ * kH * 128) + (dim & 63) * 2);
                            // rows plane ra against q plane qa, for ra + qa <= 2
#pragma unroll
                            for (int ra = 0; ra < 3; ++ra)
#pragma unroll
                                for (int qa = 0; qa < NQ && ra + qa <= 2; ++qa)
                                    mma_bf16_tmem_a_warp(d, a0 + ra * 16 + kk * 8, desc_add(bq, qa * (kH * 128)),
                                                         id_one, (h | kk | ra | qa) ? 1u : 0u);
                        }
                        mma_commit_warp(&bars[kBarEmpty + as]);
                    }
                    if (!good) { fail(); break; }
                }
                mma_commit_warp(&bars[kBarAccFull + ab]);
            }
            if (!ok) break;
            mma_commit_warp(&bars[kBarQEmpty + i % kQB]);
        }
        mma_commit_warp(&bars[kBarDrain]);
        mbar_wait(&bars[kBarDrain], 0, 1u << 24);
    } else if (warp >= kWarpEpi && warp < kWarpEpi + 4) {
        // ---------------- epilogue: TMEM lane = tile row ----------------
        const int quad = warp & 3;
        const int r = quad * 32 + lane;
        uint32_t g = 0;
        for (int i = 0; i < nql && ok; ++i) {
            const int qb = i & 1;
            const int vrow = (int)blockIdx.x + i * (int)gridDim.x;
            const int row = vrow / nch, c0 = (vrow - row * nch) * kCoarseChunk;
            if (!wait_bar(&bars[kBarMetaFull + qb], (i >> 1) & 1, abort) ||
                (i >= 2 && !wait_bar(&bars[kBarSlotFree + qb], ((i >> 1) - 1) & 1, abort))) {
                fail();
                break;
            }
            const QMeta &M = meta[qb];
            float *sc = scb + qb * n_cap;
            const int T = M.state ? 0 : M.T;
            for (int t = 0; t < T; ++t, ++g) {
                const uint32_t ab = g & 1;
                if (!wait_bar(&bars[kBarAccFull + ab], (g >> 1) & 1, abort)) { fail(); break; }
                fence_after_sync();
                const uint32_t ta = tmem + ab * acc_stride<MODE>() + ((uint32_t)(quad * 32) << 16);
                constexpr int NS = MODE == kCoarse ? 1 : NQ;   // column groups to sum
                float acc = 0.f;
#pragma unroll
                for (int c = 0; c < 4; ++c) {               // 16 heads at a time
                    float v[NS][16];
#pragma unroll
                    for (int qa = 0; qa < NS; ++qa) tmem_ld16(ta + qa * 64 + c * 16, v[qa]);
                    tmem_ld_wait();
#pragma unroll
                    for (int h = 0; h < 16; ++h) {
                        float dot = v[0][h];
#pragma unroll
                        for (int qa = 1; qa < NS; ++qa) dot += v[qa][h];
                        acc = fmaf(M.w[c * 16 + h], fmaxf(dot, 0.f), acc);
                    }
                }
                fence_before_sync();
                mbar_arrive(&bars[kBarAccEmpty + ab]);
                const int cidx = t * kM + r;
                if (cidx < M.n) {
                    // coarse: a block is eligible iff its first row is visible
                    const int64_t pos = MODE == kCoarse ? (int64_t)(c0 + cidx) * p.b
                                                        : (int64_t)M.blk[cidx >> 6] * 64 + (cidx & 63);
                    const float score = pos < M.V ? acc : kNeg;
                    sc[cidx] = score;
                    if (p.out) p.out[(int64_t)row * p.ld_out + c0 + cidx] = score;
                }
            }
            if (!ok) break;
            mbar_arrive(&bars[kBarScFull + qb]);
        }
    } else if (warp >= kWarpSel && warp < kWarpSel + 4) {
        // ---------------- select: top-k of a finished query, beside the next one's stream ----
        // The last query too: the select's code is then already in the SM's instruction cache
        // (a first run of a code path after the caches were flushed stalls on instruction
        // fetch; a CTA-wide select of the last query, a separate code path, took 4.7 us).
        const int st = tid - kWarpSel * 32;
        for (int i = 0; i < nql; ++i) {
            const int qb = i & 1;
            const int vrow = (int)blockIdx.x + i * (int)gridDim.x;
            const int row = vrow / nch, c0 = (vrow - row * nch) * kCoarseChunk;
            const bool w = wait_bar(&bars[kBarScFull + qb], (i >> 1) & 1, abort);
            if (!group_all(kBarSel, kGroup, w)) { fail(); break; }
            // coarse: the CTA's last scores are in, so its successor may launch during this
            // top-Kb (it waits for this grid before reading what it writes)
            if (MODE == kCoarse && i == nql - 1) grid_dep_trigger();
            const QMeta &M = meta[qb];
            const float *sc = scb + qb * n_cap;
            int32_t *out = nch > 1 ? P.chunk_ids + (int64_t)vrow * P.k_sel : P.sel + (int64_t)row * P.k_sel;
            const int64_t kout = M.state ? 0 : (M.n < P.k_sel ? M.n : P.k_sel);
            if (kout > 0) {
                if (MODE == kFine)
                    small_topk<kGroup, kBarSel, kWarpSel * 32>(sc, M.n, (int)kout, out, FineIds{M.blk}, sel_sh,
                                                              p.status);
                else
                    small_topk<kGroup, kBarSel, kWarpSel * 32>(sc, M.n, (int)kout, out, OffsetIds{c0}, sel_sh,
                                                              p.status);
            }
            for (int64_t e = kout + st; e < P.k_sel; e += kGroup) out[e] = -1;
            named_sync(kBarSel, kGroup);
            if (MODE == kCoarse && nch > 1) {            // the chunk's selected scores, for the merge
                if (st < kout) P.chunk_sc[(int64_t)vrow * P.k_sel + st] = sc[out[st] - c0];
                named_sync(kBarSel, kGroup);              // all reads of sc done before it is freed
            }
            if (st == 0) mbar_arrive(&bars[kBarSlotFree + qb]);
        }
    }
    else if (MODE == kCoarse && warp >= kWarpCvt && warp < kWarpCvt + kCvtWarps) {
        // ---------------- converters: f32 means -> three bf16 planes in TMEM ---------------
        // Box v (32 dims of a tile, raw slot v % kRawSlots) becomes TMEM box v % kASlots:
        // plane k in columns 16 k .. + 15, dims 2 c and 2 c + 1 in column c. TMEM lane = tile
        // row, so warp w converts rows 32 (w % 4) .. + 31 (its lane quadrant), dims 16 hf .. + 15,
        // hf = which of the quadrant's two converter warps it is. Each lane reads four 16-byte
        // pieces of its own swizzled row; eight consecutive rows cover all banks.
        const int quad = warp & 3, hf = (warp - kWarpCvt) >> 2;
        const int r = quad * 32 + lane;
        const uint32_t tlane = tmem + ((uint32_t)(quad * 32) << 16) + kAColBase + (uint32_t)hf * 8;
        uint32_t v = 0;                                        // boxes converted
        for (int i = 0; i < nql && ok; ++i) {
            const int qb = i & 1;
            if (!wait_bar(&bars[kBarMetaFull + qb], (i >> 1) & 1, abort)) { fail(); break; }
            const QMeta &M = meta[qb];
            const int nbox = M.state ? 0 : 4 * M.T;
            for (int e = 0; e < nbox; ++e, ++v) {
                const uint32_t slot = v % kRawSlots, as = v % kASlots;
                if (!wait_bar(&bars[kBarFull + kASlots + slot], (v / kRawSlots) & 1, abort) ||
                    (v >= kASlots && !wait_bar(&bars[kBarEmpty + as], (v / kASlots - 1) & 1, abort))) {
                    fail();
                    break;
                }
                const uint8_t *rowp = smem + kOffReg + slot * kRawBytes + r * 128;
                float4 a[4];
#pragma unroll
                for (int ch = 0; ch < 4; ++ch)
                    a[ch] = *reinterpret_cast<const float4 *>(rowp + (((4 * hf + ch) ^ (r & 7)) << 4));
                mbar_arrive(&bars[kBarEmpty + kASlots + slot]);
                uint32_t pl[3][8];
                split3_trunc16(a, pl);
                fence_after_sync();                    // after the wait for the MMAs that read the box
#pragma unroll
                for (int k = 0; k < 3; ++k) tmem_st8(tlane + as * kABoxCols + k * 16, pl[k]);
                tmem_st_wait();
                fence_before_sync();
                mbar_arrive(&bars[kBarFull + as]);
            }
        }
    }

    if (!ok) flag(p.status, HISA_DEV_TIMEOUT);
    fence_before_sync();
    __syncthreads();
    // coarse: every role of this CTA is done, the successor may take the SM once it exits.
    // (Triggered right after its wait instead, the fine grid launched while the coarse one
    // ran, and both pipeline kernels then streamed more slowly, as measured.)
    if (MODE == kCoarse) grid_dep_trigger();
    if (warp == kWarpMma) {
        fence_after_sync();
        tmem_dealloc(tmem, 512);
    }
}

}  // namespace

int score_pipe_supported(int mode, int H_i, int D_i, int rows_bf16, int64_t n_max, int b, int keep) {
    if (H_i != kH || D_i != kD || n_max < 1) return 0;
    if (mode == kCoarse) return !rows_bf16 && keep <= 64 && n_max <= (int64_t)kCoarseChunk * kCoarseMaxChunks;
    if (mode == kFine) return rows_bf16 && b == 64 && keep >= 1 && keep <= 48 && n_max <= kPipeMaxFine;
    return 0;
}

namespace {

template <int MODE, bool QBF16>
cudaError_t launch_pipe_t(const ScoreTcParams &p, cudaStream_t s) {
    constexpr int cap = MODE == kCoarse ? kPipeMaxCoarse : kPipeMaxFine;
    const cudaError_t attr =
        smem_attr_once<k_score_pipe<MODE, QBF16>>((int)(Layout<MODE, QBF16 ? 1 : 3>::fixed + 2 * cap * 4));
    if (p.s.n_max > cap) return cudaErrorInvalidValue;
    if (attr != cudaSuccess) return attr;
    const int rows = p.s.B * p.s.L * (MODE == kCoarse && p.chunks > 1 ? p.chunks : 1);
    const int sms = device_sm_count();
    if (sms <= 0) return cudaErrorInvalidDevice;
    const int grid = rows < sms ? rows : sms;
    const size_t smem = Layout<MODE, QBF16 ? 1 : 3>::fixed + 2 * (size_t)p.s.n_max * 4;
    // the coarse form waits for the previous grid before its first global access (before it
    // only warms L2 by prefetches), so it may always start while that grid ends
    const int chained = MODE == kCoarse ? 1 : p.s.chained;
    return launch_pdl(k_score_pipe<MODE, QBF16>, dim3(grid), dim3(pipe_threads<MODE>()), smem, s,
                      chained, p);
}

}  // namespace

cudaError_t launch_score_pipe_rows(const ScoreTcParams &p, cudaStream_t s);

namespace {

// The top keep blocks of each long coarse row from its chunks' top keep (id, score) pairs:
// by (score desc, id asc), -0.0 equal to +0.0, ids < 0 (chunks past the row, invalid rows)
// skipped; written in ascending id order, -1 past the candidates. One thread per candidate.
__global__ void __launch_bounds__(kCoarseMaxChunks * 64) k_coarse_merge(const int32_t *ids, const float *sc,
                                                                        int chunks, int keep, int32_t *top_blk) {
    __shared__ uint32_t s_key[kCoarseMaxChunks * 64];
    __shared__ int32_t s_id[kCoarseMaxChunks * 64];
    grid_dep_wait();                                 // the pairs are the previous grid's
    __shared__ int s_sel[kCoarseMaxChunks * 64];
    __shared__ int s_count;
    const int row = blockIdx.x, t = threadIdx.x, m = chunks * keep;
    const int32_t id = t < m ? ids[(int64_t)row * m + t] : -1;
    const uint32_t key = id >= 0 ? order_key(sc[(int64_t)row * m + t]) : 0u;
    s_key[t] = key;
    s_id[t] = id;
    if (t == 0) s_count = 0;
    __syncthreads();
    int rank = 0;
    if (id >= 0)
        for (int u = 0; u < m; ++u)
            rank += (s_id[u] >= 0 && (s_key[u] > key || (s_key[u] == key && s_id[u] < id))) ? 1 : 0;
    const int sel = id >= 0 && rank < keep;
    s_sel[t] = sel;
    if (sel) atomicAdd(&s_count, 1);
    __syncthreads();
    if (sel) {
        int pos = 0;
        for (int u = 0; u < m; ++u) pos += (s_sel[u] && s_id[u] < id) ? 1 : 0;
        top_blk[(int64_t)row * keep + pos] = id;
    }
    for (int e = s_count + t; e < keep; e += blockDim.x) top_blk[(int64_t)row * keep + e] = -1;
}

}  // namespace

cudaError_t launch_score_pipe(const ScoreTcParams &p_in, cudaStream_t s) {
    ScoreTcParams p = p_in;
    if (p.s.B * p.s.L == 0) return cudaSuccess;
    if (p.s.mode == kCoarse && p.chunks > 1) {
        // chunks of kCoarseChunk blocks, then the merge of their selections
        if (p.chunks > kCoarseMaxChunks || !p.chunk_ids || !p.chunk_sc || p.k_sel > 64)
            return cudaErrorInvalidValue;
        int32_t *sel = p.sel;
        p.s.n_max = kCoarseChunk;
        cudaError_t e = launch_score_pipe_rows(p, s);
        if (e != cudaSuccess) return e;
        // the merge waits before its first global access: a programmatic dependent
        return launch_pdl(k_coarse_merge, dim3((unsigned)(p.s.B * p.s.L)), dim3(kCoarseMaxChunks * 64), 0, s, 1,
                          static_cast<const int32_t *>(p.chunk_ids), static_cast<const float *>(p.chunk_sc),
                          p.chunks, p.k_sel, sel);
    }
    p.chunks = 1;
    return launch_score_pipe_rows(p, s);
}

cudaError_t launch_score_pipe_rows(const ScoreTcParams &p_in, cudaStream_t s) {
    ScoreTcParams p = p_in;
    if (p.s.mode == kFine &&
        !encode_bf16_map(&p.keys_map, p.s.rows, (uint64_t)p.s.keys_rows, kD, 64, 64))
        return cudaErrorInvalidValue;
    if (p.s.mode == kCoarse &&
        !encode_f32_map(&p.means_map, p.s.rows, (uint64_t)p.s.means_rows, kD, 32, kM))
        return cudaErrorInvalidValue;
    const bool qb = p.s.q_bf16 != 0;
    switch (p.s.mode) {
        case kCoarse: return qb ? launch_pipe_t<kCoarse, true>(p, s) : launch_pipe_t<kCoarse, false>(p, s);
        case kFine: return qb ? launch_pipe_t<kFine, true>(p, s) : launch_pipe_t<kFine, false>(p, s);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace hisa
