// k_gemm_w8.cu -- instances of the verify GEMM for the 8-bit symmetric
// ("Large") weight format.
#include "k_gemm.cuh"

namespace hq {
cudaError_t launch_gemm_w8(const GemmArgs &a, bool pdl, cudaStream_t s) { return launch_gemm_fmt<HQ_W8_SYM>(a, pdl, s); }
}  // namespace hq
