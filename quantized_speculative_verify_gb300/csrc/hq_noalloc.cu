// hq_noalloc.cu -- hq_verify_gemm for callers that cannot allocate device
// memory: the GEMM's scratch (error word, arrival counters, partial sums)
// comes from one file-scope device array instead of a caller workspace.
#include <cuda_runtime.h>

#include <mutex>

#include "hq_internal.cuh"

namespace {

// Shared by every call on a device; held until the process exits.
static __device__ __align__(256) uint8_t g_noalloc_scratch[HQ_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_setup_mutex;
void *g_scratch_ptr[kMaxDevices] = {};

// Device address of the array for the current device.  In host code the
// array's name is only a host-side stand-in, so the address is looked up
// once per device (with that device current) and cached.
int scratch_for_current_device(void **out) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return HQ_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_setup_mutex);
    if (!g_scratch_ptr[dev]) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) return HQ_ERR_CUDA;
        g_scratch_ptr[dev] = p;
    }
    *out = g_scratch_ptr[dev];
    return HQ_OK;
}

bool aligned(const void *p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

}  // namespace

extern "C" int hq_verify_gemm_noalloc(const hq_layer_desc *desc, const void *blob, const void *qop, const float *sx,
                                      int32_t M, float *Y, int32_t *partials, uint32_t flags, void *stream) {
    if (!desc || !hq::desc_valid(desc->K, desc->N, desc->group, desc->format)) return HQ_ERR_INVALID_ARG;
    if (M < 0 || M > HQ_MAX_M) return HQ_ERR_INVALID_ARG;
    if ((flags & ~(HQ_LAUNCH_PDL | HQ_LAUNCH_DETERMINISTIC)) != 0) return HQ_ERR_INVALID_ARG;
    if (M == 0) return HQ_OK;
    if (!blob || !qop || !sx || !Y) return HQ_ERR_INVALID_ARG;
    if (!aligned(blob, 16) || !aligned(qop, 16) || !aligned(sx, 4) || !aligned(Y, 4) ||
        (partials && !aligned(partials, 4)))
        return HQ_ERR_INVALID_ARG;
    const hq::Geom g = hq::make_geom(desc->K, desc->N, desc->group, desc->format);
    // The call needs exactly the workspace hq_verify_gemm would need.
    if (hq::ws_bytes(g) > (size_t)HQ_NOALLOC_SCRATCH_BYTES) return HQ_ERR_UNSUPPORTED;
    void *scratch = nullptr;
    const int st = scratch_for_current_device(&scratch);
    if (st != HQ_OK) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    // The previous call's contents stay in the array: clear the error word
    // and the n-block counters, which must start at zero.
    if (cudaMemsetAsync(scratch, 0, hq::ws_partial_offset(), s) != cudaSuccess) return HQ_ERR_CUDA;
    if (cudaMemsetAsync(static_cast<uint8_t *>(scratch) + hq::ws_counter_offset(), 0, hq::ws_counter_bytes(g), s) !=
        cudaSuccess)
        return HQ_ERR_CUDA;
    const cudaError_t e =
        hq::launch_verify_gemm(g, blob, static_cast<const uint8_t *>(qop), sx, M, Y, partials, scratch,
                               (flags & HQ_LAUNCH_PDL) != 0, (flags & HQ_LAUNCH_DETERMINISTIC) != 0, s);
    return e == cudaSuccess ? HQ_OK : HQ_ERR_CUDA;
}
