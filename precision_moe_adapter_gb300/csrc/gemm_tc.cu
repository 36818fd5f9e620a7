// gemm_tc.cu -- shared host helpers of the tcgen05 grouped GEMM: TMA
// descriptors (cuTensorMapEncodeTiled reached through the runtime's driver
// entry point, so the library does not link libcuda) and the dispatch by
// weight format.
#include <atomic>
#include <mutex>

#include "gemm_tc_host.cuh"

namespace pmoe {

bool launch_gemm_tc_int4(const GemmArgs &g, int64_t P, DevErr *err, cudaStream_t st);
bool launch_gemm_tc_mxfp4(const GemmArgs &g, int64_t P, DevErr *err, cudaStream_t st);
bool launch_gemm_tc_fp8(const GemmArgs &g, int64_t P, DevErr *err, cudaStream_t st);
bool launch_gemm_tc_bf16(const GemmArgs &g, int64_t P, DevErr *err, cudaStream_t st);

namespace tc {

typedef CUresult (*EncodeTiled)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static EncodeTiled encoder()
{
    static EncodeTiled fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = (EncodeTiled)p;
    });
    return fn;
}

// 16-bit row-major [rows][cols] tensor (BF16, or FP16: TMA copies the bits)
// as a 3-D map with one plane, box of box_rows rows x 64 columns (128 bytes:
// one swizzle row), 128-byte swizzle, zero fill out of bounds.
bool make_rows_tmap(CUtensorMap *m, const void *base, int64_t rows, int64_t cols, int box_rows)
{
    EncodeTiled enc = encoder();
    if (!enc) return false;
    cuuint64_t dims[3] = {(cuuint64_t)cols, (cuuint64_t)rows, 1};
    cuuint64_t strides[2] = {(cuuint64_t)cols * 2, (cuuint64_t)(rows > 0 ? rows : 1) * cols * 2};
    cuuint32_t box[3] = {(cuuint32_t)kBK, (cuuint32_t)box_rows, 1};
    cuuint32_t estr[3] = {1, 1, 1};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(base), dims, strides, box,
               estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool make_bytes_tmap(CUtensorMap *m, const void *base, int64_t rows, int64_t row_bytes,
                     int box_bytes, int box_rows, int swizzle_bytes, int l2_promote)
{
    EncodeTiled enc = encoder();
    if (!enc) return false;
    cuuint64_t dims[2] = {(cuuint64_t)row_bytes, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)row_bytes};
    cuuint32_t box[2] = {(cuuint32_t)box_bytes, (cuuint32_t)box_rows};
    cuuint32_t estr[2] = {1, 1};
    const CUtensorMapSwizzle swz = swizzle_bytes == 128  ? CU_TENSOR_MAP_SWIZZLE_128B
                                   : swizzle_bytes == 64 ? CU_TENSOR_MAP_SWIZZLE_64B
                                                         : CU_TENSOR_MAP_SWIZZLE_NONE;
    const CUtensorMapL2promotion pro = l2_promote == 256  ? CU_TENSOR_MAP_L2_PROMOTION_L2_256B
                                       : l2_promote == 128 ? CU_TENSOR_MAP_L2_PROMOTION_L2_128B
                                       : l2_promote == 64  ? CU_TENSOR_MAP_L2_PROMOTION_L2_64B
                                                           : CU_TENSOR_MAP_L2_PROMOTION_NONE;
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void *>(base), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, swz, pro, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool make_slots_tmap(CUtensorMap *m, const void *base, int64_t slots, int64_t rows, int64_t cols,
                     int64_t slot_bytes, int box_rows)
{
    EncodeTiled enc = encoder();
    if (!enc) return false;
    cuuint64_t dims[3] = {(cuuint64_t)cols, (cuuint64_t)rows, (cuuint64_t)slots};
    cuuint64_t strides[2] = {(cuuint64_t)cols * 2, (cuuint64_t)slot_bytes};
    cuuint32_t box[3] = {(cuuint32_t)kBK, (cuuint32_t)box_rows, 1};
    cuuint32_t estr[3] = {1, 1, 1};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(base), dims, strides, box,
               estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// One-shot test hook (pmoe_debug_expire_gemm_wait): the wait limit of the
// next grouped-GEMM launch, 0 when none is armed.
static std::atomic<uint64_t> g_expire_wait_ns{0};

void take_wait_hook(uint64_t &wait_ns, int &skip_item)
{
    const uint64_t v = g_expire_wait_ns.exchange(0);
    wait_ns = v ? v : kWaitNs;
    skip_item = v ? 0 : -1;
}

bool arm_wait_hook(uint64_t wait_ns)
{
    if (wait_ns < 100000ull || wait_ns > kWaitNs) return false;
    g_expire_wait_ns.store(wait_ns);
    return true;
}

int num_sms()
{
    static int n = 0;
    if (!n) {
        int dev = 0;
        cudaGetDevice(&dev);
        cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
        if (n <= 0) n = 1;
    }
    return n;
}

}  // namespace tc

int gemm_num_sms() { return tc::num_sms(); }

bool launch_gemm_tc(const GemmArgs &g, int64_t P, DevErr *err, cudaStream_t st)
{
    switch (g.fmt) {
    case PMOE_W_INT4_G32_BF16: return launch_gemm_tc_int4(g, P, err, st);
    case PMOE_W_MXFP4_G32_E8M0: return launch_gemm_tc_mxfp4(g, P, err, st);
    case PMOE_W_FP8_B128_F32: return launch_gemm_tc_fp8(g, P, err, st);
    case kFmtBF16: return launch_gemm_tc_bf16(g, P, err, st);
    }
    return false;
}

}  // namespace pmoe

extern "C" pmoe_status pmoe_debug_expire_gemm_wait(uint64_t wait_ns)
{
    return pmoe::tc::arm_wait_hook(wait_ns) ? PMOE_OK : PMOE_ERR_INVALID_ARG;
}
