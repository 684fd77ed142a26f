// hisa_flat_topk_noalloc: the flat top-k selection for callers that cannot allocate
// device memory. Some hosts own every byte of device memory themselves (a serving
// runtime that hands all of it to its own pool at start-up, a plugin inside a framework
// that forbids allocations outside its allocator), and some run loops where cudaMalloc
// and cudaFree are too costly because they can synchronise the whole device. Such a
// caller cannot provide the score workspace hisa_flat_topk needs, so this entry point
// keeps that workspace in a fixed array in device memory that the library itself
// declares. The caller passes only inputs and outputs.
//
// The array lives in this translation unit. Every device that loads this code holds
// it until the process exits. In host code `g_flat_scratch` names a host-side stand-in
// of the symbol, not a device address: its device address is looked up once per device
// with cudaGetSymbolAddress, on the first call made while that device is current.
#include <mutex>

#include "hisa_internal.cuh"

using namespace hisa;

namespace {

static_assert(HISA_FLAT_NOALLOC_MAX_SCORES == (1 << 22), "header and library disagree");

// Status header (the same 256 bytes every workspace starts with) + the f32 flat
// scores of every query row, B * L * Np_max of them at most.
constexpr size_t kNoAllocBytes =
    (size_t)kStatusBytes + (size_t)HISA_FLAT_NOALLOC_MAX_SCORES * sizeof(float);

__device__ __align__(256) unsigned char g_flat_scratch[kNoAllocBytes];

constexpr int kMaxDevices = 64;
std::mutex g_mutex;
void *g_scratch_addr[kMaxDevices] = {};

// Device address of the array on the current device (looked up on first use).
hisa_status scratch_of_current_device(void **out) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) return HISA_ECUDA;
    if (dev < 0 || dev >= kMaxDevices) return HISA_EINVAL;
    std::lock_guard<std::mutex> lock(g_mutex);
    if (!g_scratch_addr[dev]) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_flat_scratch) != cudaSuccess || !p) return HISA_ECUDA;
        g_scratch_addr[dev] = p;
    }
    *out = g_scratch_addr[dev];
    return HISA_OK;
}

bool aligned_to(const void *p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

}  // namespace

extern "C" {

hisa_status hisa_flat_topk_noalloc(const hisa_index_desc *desc, const void *q, const float *w,
                                   const void *keys, const int64_t *key_off, const int32_t *t0,
                                   int32_t *I, uint32_t *dev_status, hisa_stream_t stream) {
    // Everything the host can check is checked before anything is enqueued.
    if (!desc) return HISA_EINVAL;
    const size_t need = hisa_workspace_bytes(HISA_OP_FLAT_TOPK, desc);
    if (need == 0)  // the descriptor itself is invalid: report hisa_flat_topk's verdict
        return hisa_flat_topk(desc, q, w, keys, key_off, t0, I, nullptr, 0, stream);
    if (need > kNoAllocBytes) return HISA_EWORKSPACE;
    if (!q || !w || !keys || !key_off || !t0 || !I) return HISA_EINVAL;
    if (!aligned_to(q, 16) || !aligned_to(keys, 16) || !aligned_to(w, 4)) return HISA_EINVAL;
    if (dev_status && !aligned_to(dev_status, 4)) return HISA_EINVAL;

    void *scratch = nullptr;
    hisa_status st = scratch_of_current_device(&scratch);
    if (st != HISA_OK) return st;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    // The array keeps the previous call's contents. Only the status word must start at
    // zero: every score a kernel reads is written earlier in the same call.
    if (cudaMemsetAsync(scratch, 0, kStatusBytes, s) != cudaSuccess) return HISA_ECUDA;
    st = hisa_flat_topk(desc, q, w, keys, key_off, t0, I, scratch, kNoAllocBytes, stream);
    if (st != HISA_OK) return st;
    if (dev_status &&
        cudaMemcpyAsync(dev_status, scratch, sizeof(uint32_t), cudaMemcpyDeviceToDevice, s) !=
            cudaSuccess)
        return HISA_ECUDA;
    return HISA_OK;
}

}  // extern "C"
