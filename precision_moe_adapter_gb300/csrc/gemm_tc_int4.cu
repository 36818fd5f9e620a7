// gemm_tc_int4.cu -- tcgen05 grouped GEMM instantiated for the int4 weights.
#include "gemm_tc_host.cuh"

namespace pmoe {
bool launch_gemm_tc_int4(const GemmArgs &g, int64_t P, DevErr *err, cudaStream_t st)
{
    return tc::launch_fmt<PMOE_W_INT4_G32_BF16>(g, P, err, st);
}
}  // namespace pmoe
