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
// host code its name is only a stand-in, so the device address is fetched
// with cudaGetSymbolAddress once per device (on the first call made with that
// device current) and that address is what the kernels receive.
#include <mutex>

#include <cuda_runtime.h>

#include "specverify.h"

namespace {

constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_greedy_scratch[SV_NOALLOC_SCRATCH_BYTES];

std::mutex g_scratch_mu;
void* g_scratch_addr[kMaxDevices] = {};

// device address of the scratch array on the current device
int scratch_address(void** out)
{
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return SV_ERR_DEVICE;
    std::lock_guard<std::mutex> lock(g_scratch_mu);
    if (g_scratch_addr[dev] == nullptr) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_greedy_scratch) != cudaSuccess || p == nullptr) {
            (void)cudaGetLastError();  // leave no sticky launch error behind
            return SV_ERR_DEVICE;
        }
        g_scratch_addr[dev] = p;
    }
    *out = g_scratch_addr[dev];
    return SV_OK;
}

}  // namespace

extern "C" int sv_verify_greedy_noalloc(sv_rows target, int32_t R, int32_t k, int32_t branches,
                                        const int32_t* draft, int32_t* accept_len, int32_t* tokens,
                                        int32_t* branch, int32_t* status, sv_stream_t stream)
{
    if (R < 0 || k < 0 || branches < 1 || branches > SV_MAX_BRANCHES || (branches >= 2 && k < 1) ||
        target.width < 1)
        return SV_ERR_INVALID_ARG;
    if (k > SV_MAX_K) return SV_ERR_LIMIT;
    if (R == 0) return SV_OK;
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
