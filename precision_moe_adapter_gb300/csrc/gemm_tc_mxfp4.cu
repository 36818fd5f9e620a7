// gemm_tc_mxfp4.cu -- tcgen05 grouped GEMM instantiated for the mxfp4 weights.
#include "gemm_tc_host.cuh"

namespace pmoe {
bool launch_gemm_tc_mxfp4(const GemmArgs &g, int64_t P, DevErr *err, cudaStream_t st)
{
    return tc::launch_fmt<PMOE_W_MXFP4_G32_E8M0>(g, P, err, st);
}
}  // namespace pmoe
