// sv_verify_greedy_noalloc: greedy verification for callers that may not
// allocate device memory.
//
// Some callers cannot call cudaMalloc: a plugin whose host framework owns all
// device memory through its own caching pool (a direct cudaMalloc would fail
// once that pool has reserved the GPU, or would fragment it), or a decode
// loop that pre-reserves every buffer before serving starts and must not
// allocate on the latency path.  This entry point takes inputs and outputs
// only; its scratch (the per-segment argmax partials of sv_verify_greedy)
// lives in a fixed array compiled into the library.
//
// The array is a file-scope __device__ object: every GPU that loads the
// library holds SV_NOALLOC_SCRATCH_BYTES of it until the process exits.  In
// host code its name is only a stand-in, so every call looks up the array's
// device address on the current device with cudaGetSymbolAddress (no
// allocation, and no address kept across calls that a device reset could
// invalidate) and hands that address to the kernels.
#include <cuda_runtime.h>

#include "specverify.h"

namespace {

static __device__ __align__(256) unsigned char g_greedy_scratch[SV_NOALLOC_SCRATCH_BYTES];

// device address of the scratch array on the current device
int scratch_address(void** out)
{
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) {
        (void)cudaGetLastError();
        return SV_ERR_DEVICE;
    }
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_greedy_scratch) != cudaSuccess || p == nullptr) {
        (void)cudaGetLastError();  // leave no sticky launch error behind
        return SV_ERR_DEVICE;
    }
    *out = p;
    return SV_OK;
}

}  // namespace

extern "C" int sv_verify_greedy_noalloc(sv_rows target, int32_t R, int32_t k, int32_t branches,
                                        const int32_t* draft, int32_t* accept_len, int32_t* tokens,
                                        int32_t* branch, int32_t* status, sv_stream_t stream)
{
    // sv_verify_greedy's own argument checks, in its order: without a workspace it stops at
    // the workspace check, after every argument check and before anything is launched
    const int pre = sv_verify_greedy(target, R, k, branches, draft, accept_len, tokens, branch, status,
                                     nullptr, 0, stream);
    if (pre != SV_ERR_WORKSPACE) return pre;  // an argument error, or SV_OK for R == 0
    const size_t need = sv_verify_greedy_workspace(R, k, branches, target.width);
    if (need == 0) return SV_ERR_INVALID_ARG;
    if (need > SV_NOALLOC_SCRATCH_BYTES) return SV_ERR_LIMIT;  // batch too large for the fixed array
    void* scratch = nullptr;
    if (int rc = scratch_address(&scratch)) return rc;
    // Every scratch slot the kernels read is written earlier in the same call,
    // so nothing has to be cleared between calls.
    return sv_verify_greedy(target, R, k, branches, draft, accept_len, tokens, branch, status,
                            scratch, SV_NOALLOC_SCRATCH_BYTES, stream);
}
