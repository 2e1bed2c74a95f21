// k_gemm_rs.cu -- instances of the register-resident verify GEMM for 4-bit
// weights (fp16 row operand, up to 32 rows).
#include "k_gemm_rs.cuh"

namespace hq {
cudaError_t launch_gemm_w4_rs(const GemmArgs &a, bool pdl, cudaStream_t s) { return launch_gemm_rs<HQ_W4_ASYM>(a, pdl, s); }
}  // namespace hq
