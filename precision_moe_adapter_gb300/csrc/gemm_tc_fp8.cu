// gemm_tc_fp8.cu -- tcgen05 grouped GEMM instantiated for the fp8 weights.
#include "gemm_tc_host.cuh"

namespace pmoe {
bool launch_gemm_tc_fp8(const GemmArgs &g, int64_t P, DevErr *err, cudaStream_t st)
{
    return tc::launch_fmt<PMOE_W_FP8_B128_F32>(g, P, err, st);
}
}  // namespace pmoe
