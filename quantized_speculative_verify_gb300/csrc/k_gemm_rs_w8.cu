// k_gemm_rs_w8.cu -- instances of the register-resident verify GEMM for
// 8-bit weights (fp16 row operand, up to 32 rows).
#include "k_gemm_rs.cuh"

namespace hq {
cudaError_t launch_gemm_w8_rs(const GemmArgs &a, bool pdl, cudaStream_t s) { return launch_gemm_rs<HQ_W8_SYM>(a, pdl, s); }
}  // namespace hq
