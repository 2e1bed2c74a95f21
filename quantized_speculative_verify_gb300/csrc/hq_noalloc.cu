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
// once per device (with that device current) and cached.  The first lookup
// also zero-fills the array (synchronously, on the legacy stream): the error
// word and the arrival counters must start at zero, and the kernels leave
// them at zero after every call that does not time out.  With create ==
// false a device whose array was never set up reports *out == NULL.
int scratch_for_current_device(void **out, bool create) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return HQ_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_setup_mutex);
    if (!g_scratch_ptr[dev] && create) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) return HQ_ERR_CUDA;
        if (cudaMemset(p, 0, HQ_NOALLOC_SCRATCH_BYTES) != cudaSuccess) return HQ_ERR_CUDA;
        if (cudaDeviceSynchronize() != cudaSuccess) return HQ_ERR_CUDA;
        g_scratch_ptr[dev] = p;
    }
    *out = g_scratch_ptr[dev];
    return HQ_OK;
}

bool aligned(const void *p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

}  // namespace

extern "C" int hq_verify_gemm_noalloc(const hq_layer_desc *desc, const void *blob, const void *qop, const float *sx,
                                      int32_t M, float *Y, int32_t *partials, uint32_t flags, void *stream) {
    if (!hq::desc_ok(desc)) return HQ_ERR_INVALID_ARG;
    if (M < 0 || M > HQ_MAX_M) return HQ_ERR_INVALID_ARG;
    if ((flags & ~(HQ_LAUNCH_PDL | HQ_LAUNCH_DETERMINISTIC | HQ_LAUNCH_EXACT_ORDER)) != 0) return HQ_ERR_INVALID_ARG;
    if (M == 0) return HQ_OK;
    if (!blob || !qop || !sx || !Y) return HQ_ERR_INVALID_ARG;
    if (!aligned(blob, 16) || !aligned(qop, 16) || !aligned(sx, 4) || !aligned(Y, 4) ||
        (partials && !aligned(partials, 4)))
        return HQ_ERR_INVALID_ARG;
    const hq::Geom g = hq::make_geom(desc->K, desc->N, desc->group, desc->format);
    // The call needs exactly the workspace hq_verify_gemm would need.
    if (hq::ws_bytes(g) > (size_t)HQ_NOALLOC_SCRATCH_BYTES) return HQ_ERR_UNSUPPORTED;
    void *scratch = nullptr;
    const int st = scratch_for_current_device(&scratch, true);
    if (st != HQ_OK) return st;
    const cudaError_t e =
        hq::launch_verify_gemm(g, blob, static_cast<const uint8_t *>(qop), sx, M, Y, partials, scratch, flags,
                               static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? HQ_OK : HQ_ERR_CUDA;
}

extern "C" int hq_noalloc_status(void *stream) {
    void *scratch = nullptr;
    const int st = scratch_for_current_device(&scratch, false);
    if (st != HQ_OK) return st;
    if (!scratch) return HQ_OK;  // no call has run on this device
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (cudaStreamSynchronize(s) != cudaSuccess) return HQ_ERR_CUDA;
    int v = 0;
    if (cudaMemcpy(&v, scratch, sizeof v, cudaMemcpyDeviceToHost) != cudaSuccess) return HQ_ERR_CUDA;
    if (v == 0) return HQ_OK;
    // A wait gave up: the error word and any counter the timed-out call left
    // behind go back to zero, so that the next call starts clean.
    if (cudaMemset(scratch, 0, hq::ws_partial_offset()) != cudaSuccess) return HQ_ERR_CUDA;
    if (cudaMemset(static_cast<uint8_t *>(scratch) + hq::ws_counter_offset(), 0,
                   (size_t)HQ_NOALLOC_SCRATCH_BYTES - hq::ws_counter_offset()) != cudaSuccess)
        return HQ_ERR_CUDA;
    if (cudaDeviceSynchronize() != cudaSuccess) return HQ_ERR_CUDA;
    return HQ_ERR_TIMEOUT;
}
