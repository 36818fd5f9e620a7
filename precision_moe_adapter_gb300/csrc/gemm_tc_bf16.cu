// gemm_tc_bf16.cu -- tcgen05 grouped GEMM instantiated for the bf16 weights.
#include "gemm_tc_host.cuh"

namespace pmoe {
bool launch_gemm_tc_bf16(const GemmArgs &g, int64_t P, DevErr *err, cudaStream_t st)
{
    return tc::launch_fmt<kFmtBF16>(g, P, err, st);
}
}  // namespace pmoe
