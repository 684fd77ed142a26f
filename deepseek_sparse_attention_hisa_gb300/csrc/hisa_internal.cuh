// Internal declarations shared by the kernel translation units of libhisa.
// Nothing here is part of the C ABI (see include/hisa.h).
#pragma once

#include <cuda.h>              // CUtensorMap (the encoder is fetched from the driver at run time)
#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include <atomic>

#include "../../include/hisa.h"

namespace hisa {

// ---- programmatic dependent launch ------------------------------------------------
// A call made with HISA_FLAG_CHAINED launches its kernels with programmatic stream
// serialization: the launch is prepared, and may start, while the previous kernel on the
// stream runs. grid_dep_wait() waits until the previous grid has completed and its writes
// are visible (without the attribute it returns at once: the kernel started after the
// previous work completed). Most kernels execute it before their first global-memory
// access. The scoring pipeline and the combine let their successor launch before they
// complete (grid_dep_trigger): the coarse form and the combine once every role of a CTA is
// done, the fine form right after its own wait (never before it, so that a successor never
// runs beside the kernel two back). The fine form reads q, w and the offsets before it
// waits and only the kept blocks (the coarse output) after; the combine waits before its
// first selected id (the fine output) and first output write, after its first item's q and
// local rows are on their way. The flag's contract (include/hisa.h) is that no such early-read input is written
// by the kernel just before the call.
__device__ __forceinline__ void grid_dep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void grid_dep_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                       cudaStream_t s, int chained, Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = chained ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, kernel, args...);
}

// SMs of the current device (cached per device; 0 if the runtime cannot tell).
int device_sm_count();

// cudaFuncSetAttribute(Kernel, MaxDynamicSharedMemorySize, bytes), made once per device
// (the attribute belongs to the device's context) and its result cached per device.
// Concurrent first calls may both set it, which is harmless.
template <auto Kernel>
cudaError_t smem_attr_once(int bytes) {
    static std::atomic<int> state[64];      // 0: not yet set; else 1 + the cudaError_t
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64)
        return cudaFuncSetAttribute(Kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    const int st = state[dev].load(std::memory_order_acquire);
    if (st != 0) return (cudaError_t)(st - 1);
    e = cudaFuncSetAttribute(Kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    state[dev].store(1 + (int)e, std::memory_order_release);
    return e;
}


constexpr float kNeg = -1e30f;            // selection mask value ([HiSA issue] "Flat selection")
constexpr size_t kStatusBytes = 256;      // status word region at the head of the workspace
constexpr int kTargetCtas = 304;          // 2 CTAs per SM on a 152-SM GB300
constexpr int kSmTarget = 152;            // one CTA per SM on a 152-SM GB300
constexpr int kMaxTopk = 2048;

enum ScoreMode : int { kFlat = 0, kCoarse = 1, kFine = 2 };

// ---------------------------------------------------------------------------
// device helpers
// ---------------------------------------------------------------------------
__device__ __forceinline__ float to_f32(float x) { return x; }
__device__ __forceinline__ float to_f32(__nv_bfloat16 x) { return __bfloat162float(x); }

__device__ __forceinline__ void flag(uint32_t *status, uint32_t bit) {
    if (status) atomicOr(status, bit);
}

// Visible pooled prefix V(t) = min(Np, floor((t+1)/r)).
__device__ __forceinline__ int64_t visible_len(int64_t t, int r, int64_t Np) {
    int64_t v = (t + 1) / r;
    if (t + 1 < 0) v = 0;
    return v < Np ? v : Np;
}

// Sequence b's pooled rows [off[b], off[b+1]) are usable iff they are ordered, fit Np_max
// and lie inside the allocation of `rows` rows.
__device__ __forceinline__ bool seq_ok_v(int64_t a, int64_t e, int64_t Np_max, int64_t rows) {
    return a >= 0 && e >= a && e - a <= Np_max && e <= rows;
}
__device__ __forceinline__ bool seq_ok(const int64_t *off, int b, int64_t Np_max, int64_t rows) {
    return seq_ok_v(off[b], off[b + 1], Np_max, rows);
}

// Sequence b's nb block-mean rows [moff[b], moff[b] + nb) fit its offsets and lie inside
// the rows allocated in the block-mean array.
__device__ __forceinline__ bool means_ok_v(int64_t a, int64_t e, int64_t nb, int64_t rows) {
    return a >= 0 && e - a >= nb && a + nb <= rows;
}
__device__ __forceinline__ bool means_ok(const int64_t *moff, int b, int64_t nb, int64_t rows) {
    return means_ok_v(moff[b], moff[b + 1], nb, rows);
}

// Orderable key of an f32 score: larger float -> larger key; -0.0 == +0.0.
__device__ __forceinline__ uint32_t order_key(float s) {
    uint32_t u = __float_as_uint(s);
    if ((u << 1) == 0u) u = 0u;
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// ---------------------------------------------------------------------------
// launch parameter blocks
// ---------------------------------------------------------------------------
struct ScoreParams {
    int mode;                 // ScoreMode
    int B, L, H_i, D_i, r, b, keep;
    int causal;               // apply the pooled causal mask (L > 1)
    const void *q;            // [B*L, H_i, D_i]
    int q_bf16;
    const float *w;           // [B*L, H_i] raw
    float head_scale;         // H_i^-1/2 * D_i^-1/2
    const void *rows;         // keys [sum Np, D_i] (flat / fine) or means [*, D_i] f32 (coarse)
    int rows_bf16;
    const int64_t *key_off;   // [B+1]
    const int64_t *means_off; // [B+1] (coarse)
    const int32_t *t0;        // [B]
    const int32_t *top_blk;   // [B*L, keep] (fine)
    float *out;               // [B*L, ld_out]
    int64_t ld_out;
    int64_t n_max;            // max scored rows per query row (grid.x extent)
    int64_t Np_max;
    int64_t keys_rows;        // rows allocated in the key array
    int64_t means_rows;       // rows allocated in the block-mean array (coarse)
    uint32_t *status;
    int chained;              // launch as a programmatic dependent (HISA_FLAG_CHAINED)
};

struct SelectParams {
    int mode;                 // ScoreMode: what a score column maps to
    int B, L, b, keep, k;
    const float *scores;      // [B*L, ld]
    int64_t ld;
    // flat rows longer than the shared-memory form holds: when work == scores (writable),
    // each chunk of those rows is reduced in place to its top k (score, id) pairs and one
    // CTA per row selects among them; null: one CTA per row selects over the whole row
    float *work;
    int smem_n;               // set by launch_select: scores its CTAs can hold in shared memory
    const int64_t *key_off;
    const int32_t *top_blk;   // fine: [B*L, keep]
    int32_t *out;             // [B*L, k]
    int64_t Np_max;
    int64_t keys_rows;        // rows allocated in the key array (the scored rows' bound)
    uint32_t *status;
};

struct MeansParams {
    int B, D_i, b;
    const void *keys;
    int keys_bf16;
    const int64_t *key_off;
    const int64_t *means_off;
    const int32_t *first_block;
    float *means;
    int64_t Np_max;
    int64_t keys_rows;
    int64_t means_rows;
    uint32_t *status;
    int chained;              // launch as a programmatic dependent (HISA_FLAG_CHAINED)
};

struct AttnParams {
    int B, L, H, Dh, window, W_max, r, k;
    int causal;
    int64_t Np_max;
    int64_t kv_rows;          // rows allocated in pooled_kv
    float scale;
    const void *q;            // [B*L, H, Dh]
    const void *local_kv;     // [B, W_max, Dh]
    const int32_t *local_len;
    const int32_t *local_pos0;
    const void *pooled_kv;    // [sum Np, Dh]
    const int64_t *kv_off;
    const int32_t *I;         // [B*L, k] or nullptr
    const float *sinks;       // [H]
    const int32_t *t0;
    void *out;                // [B*L, H, Dh] f32, or bf16 when out_bf16
    int out_bf16;
    float *part;              // split partials [B*L, nsplit, H, Dh + 2]
    int nsplit;
    int rows_per_split;       // multiple of the chunk size
    int kv_bf16;
    uint32_t *status;
    int chained;              // launch as a programmatic dependent (HISA_FLAG_CHAINED)
};

struct CompressParams {
    int B, D, C, r, overlap, rope_dims, b;
    int n_new_max;
    int k_bf16;
    float eps;
    double log_theta;         // ln(rope theta)
    const float *kv;          // [tok_rows, C] wkv(x)
    const float *gate;        // [tok_rows, C] wgate(x)
    const float *ape;         // [r, C]
    const float *norm_w;      // [D]
    const int64_t *tok_off;   // [B+1]
    const int32_t *p_first;   // [B]
    const int32_t *n_new;     // [B]
    void *keys;               // [keys_rows, D] out
    const int64_t *key_off;   // [B+1]
    float *means;             // [means_rows, D] out, or nullptr
    const int64_t *means_off; // [B+1]
    int64_t tok_rows, keys_rows, means_rows;
    uint32_t *status;
    int chained;
};

// Tensor-core scoring (H_i = 64, D_i = 128): `s` describes the rows and inputs; the
// coarse and fine modes also select (sel = top_blk or I, k_sel ids per query row); s.out
// is optional for them (the scores of every row) and required for the flat mode.
struct ScoreTcParams {
    CUtensorMap keys_map;     // bf16 keys [keys_rows, 128], box 64 dims x 64 rows, 128B swizzle
    CUtensorMap means_map;    // f32 block means [means_rows, 128], box 32 dims x 128 rows, 128B swizzle
    ScoreParams s;
    // coarse only: when append_keys is set, the kernel first writes the block means of blocks
    // [first_block[b], nb_b) from these bf16 keys (decode rows, index_block 64, D_i 128)
    const void *append_keys;
    const int32_t *first_block;
    int32_t *sel;
    int k_sel;
    int tiles_per_cta;        // flat: 128-row tiles per CTA (grid.y covers the row)
    // coarse rows of more than kCoarseChunk blocks: each query row is scored as `chunks`
    // chunks of kCoarseChunk blocks, each chunk's top-k_sel (id, score) pairs go to
    // chunk_ids / chunk_sc [rows * chunks, k_sel], and a merge writes sel
    int chunks;
    int32_t *chunk_ids;
    float *chunk_sc;
};
constexpr int kCoarseChunk = 1024;        // block means per chunk of a long coarse row
constexpr int kCoarseMaxChunks = 4;

// Encodes a 2-D bf16 tensor map over [rows, cols] (row-major) with a box of box_cols x
// box_rows and the 128-byte swizzle. Returns false if the driver has no encoder or
// rejects the map.
bool encode_f32_map(CUtensorMap *map, const void *base, uint64_t rows, uint64_t cols,
                    uint32_t box_cols, uint32_t box_rows);
bool encode_bf16_map(CUtensorMap *map, const void *base, uint64_t rows, uint64_t cols,
                     uint32_t box_cols, uint32_t box_rows);

// ---------------------------------------------------------------------------
// host launchers (one per kernel file); return the cudaGetLastError() of the launch
// ---------------------------------------------------------------------------
cudaError_t launch_scores_simt(const ScoreParams &p, cudaStream_t s);
cudaError_t launch_select(const SelectParams &p, int64_t n_max, cudaStream_t s);
// whether launch_select can take flat rows of up to ld scores and k ids in chunks
bool chunked_select_fits(int64_t ld, int k);
cudaError_t launch_block_means(const MeansParams &p, int64_t nb_max, cudaStream_t s);
cudaError_t launch_attend_simt(const AttnParams &p, cudaStream_t s);
cudaError_t launch_attend_combine(const AttnParams &p, cudaStream_t s);
cudaError_t launch_attend_tc(const AttnParams &p, cudaStream_t s);
int attend_simt_supported(int H, int Dh);
int attend_tc_supported(int H, int Dh, int kv_bf16);
int attend_chunk_rows();
cudaError_t launch_score_tc(const ScoreTcParams &p, cudaStream_t s);
int score_tc_supported(int mode, int H_i, int D_i, int rows_bf16, int64_t n_max, int b);
// coarse / fine rows split over CTAs (scores to memory, then launch_select): any n
int score_tc_split_ok(int mode, int H_i, int D_i, int rows_bf16, int b);
// Persistent coarse / fine scoring + select pipeline (one CTA per SM over all query rows).
cudaError_t launch_score_pipe(const ScoreTcParams &p, cudaStream_t s);
int score_pipe_supported(int mode, int H_i, int D_i, int rows_bf16, int64_t n_max, int b, int keep);
// Dense scoring of many query rows per sequence (batched prefill): flat scores to p.out.
cudaError_t launch_score_gemm(const ScoreParams &p, cudaStream_t s);
// Coarse scores of many bf16 query rows (batched prefill) as the same contraction over the
// f32 block means (p.rows) split into three exact bf16 planes held in `planes`
// (coarse_gemm_planes_bytes(p.means_rows) bytes); scores to p.out.
cudaError_t launch_coarse_gemm(const ScoreParams &p, void *planes, cudaStream_t s);
size_t coarse_gemm_planes_bytes(int64_t means_rows);
// The indexer compressor: new pooled rows and the block means they complete.
cudaError_t launch_compress(const CompressParams &p, cudaStream_t s);
int score_gemm_supported(int H_i, int D_i, int q_bf16, int rows_bf16, int B, int L);

}  // namespace hisa
