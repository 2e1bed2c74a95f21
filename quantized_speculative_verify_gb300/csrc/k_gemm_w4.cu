// k_gemm_w4.cu -- instances of the verify GEMM for the 4-bit asymmetric
// ("Medium") weight format.
#include "k_gemm.cuh"

namespace hq {
cudaError_t launch_gemm_w4(const GemmArgs &a, bool pdl, cudaStream_t s) { return launch_gemm_fmt<HQ_W4_ASYM>(a, pdl, s); }
}  // namespace hq
