// permute_noalloc.cu -- moe_permute without a caller workspace.
//
// Some callers cannot hand the library a workspace: a framework operator or
// plugin whose enqueue hook only receives its input and output tensors, or
// code that runs where allocating is not allowed (inside an allocator
// callback, or in a memory-capped inference process that has reserved
// every byte).  For them the grouping step keeps its per-block histogram in
// one fixed buffer of device memory that is part of the library image, so
// the call allocates nothing, neither on the device nor through a library
// that allocates behind the caller's back.
//
// The buffer is shared by every call in the process on a given device:
// calls that may overlap (two streams, or two host threads) race on it and
// must be ordered by the caller.  Nothing in it has to start at zero: each
// call overwrites the part it reads.  Its device address is looked up once
// per device, on the first call there.
#include <mutex>

#include "common.cuh"
#include "launch.h"

namespace pmoe {

constexpr size_t kNoAllocScratchBytes = PMOE_PERMUTE_NOALLOC_SCRATCH_BYTES;
static_assert(kNoAllocScratchBytes % 256 == 0, "whole 256-byte lines");

static __device__ __align__(256) int32_t g_permute_scratch[kNoAllocScratchBytes / sizeof(int32_t)];

namespace {
constexpr int kMaxDevices = 64;
std::mutex g_setup_mu;
int32_t *g_scratch_addr[kMaxDevices];   // per device, set by the first call there

// Device address of the scratch on the current device (nullptr on failure).
int32_t *scratch_on_current_device()
{
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
    std::lock_guard<std::mutex> lk(g_setup_mu);
    if (!g_scratch_addr[dev]) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_permute_scratch) != cudaSuccess || !p) return nullptr;
        g_scratch_addr[dev] = (int32_t *)p;
    }
    return g_scratch_addr[dev];
}
}  // namespace

// Bytes of the per-block histogram for P pairs and E experts, in 64-bit
// arithmetic (the same layout as permute_ws_bytes, whose int argument the
// caller's T*k is never narrowed into before this check).
size_t permute_noalloc_need_bytes(int64_t P, int E)
{
    const int64_t blocks = P > 0 ? (P + 1023) / 1024 : 1;
    return (size_t)blocks * (size_t)(E > 0 ? E : 0) * sizeof(int32_t);
}

}  // namespace pmoe

extern "C" pmoe_status moe_permute_noalloc(pmoe_dims dims, const int32_t *idx,
                                           const pmoe_routing *out, cudaStream_t stream)
{
    using namespace pmoe;
    if (!dims_ok(dims) || !out) return PMOE_ERR_INVALID_ARG;
    if ((dims.T > 0 && (!idx || !out->perm || !out->inv_perm)) || !out->counts ||
        !out->offsets || !out->active || !out->num_active)
        return PMOE_ERR_INVALID_ARG;
    // the per-block histogram must fit the fixed buffer (and T*k an int)
    const int64_t P = (int64_t)dims.T * dims.k;
    if (P > INT32_MAX || permute_noalloc_need_bytes(P, dims.E) > kNoAllocScratchBytes)
        return PMOE_ERR_WORKSPACE;
    int32_t *hist = scratch_on_current_device();
    if (!hist) return PMOE_ERR_CUDA;
    // no error word: an expert id outside [0, E) shows only in the outputs
    launch_permute((int)P, dims.E, idx, out->counts, out->offsets, out->perm,
                   out->inv_perm, out->active, out->num_active, hist, nullptr, stream);
    return cudaPeekAtLastError() == cudaSuccess ? PMOE_OK : PMOE_ERR_CUDA;
}
