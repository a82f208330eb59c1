// sv_selftest_wait_timeout: runs out one bounded shared-memory barrier wait on
// purpose, with the same wait routine every kernel of the library uses, so that
// a test can see the timeout path work without any fault.
//
// One warp; lane 0 sets up two barriers.  Barrier `done` receives a 16-byte
// bulk copy (which it expects) and completes.  Barrier `never` expects 16
// transaction bytes that no copy delivers, so its wait gives up after
// `limit_cycles` and the kernel records SV_ST_TIMEOUT.  The only copy issued
// has landed before the kernel exits, so nothing is in flight afterwards.
#include <cuda_runtime.h>

#include "specverify.h"
#include "sv_device.cuh"

namespace {

__global__ void __launch_bounds__(32) wait_timeout_kernel(const uint4* src, int32_t* status, long long limit)
{
    __shared__ __align__(16) uint4 dst;
    __shared__ __align__(8) uint64_t done, never;
    if (threadIdx.x != 0) return;
    sv::mbar_init(&done, 1);
    sv::mbar_init(&never, 1);
    sv::fence_barrier_init();
    sv::mbar_arrive_expect_tx(&never, 16u);  // bytes that never come
    sv::mbar_arrive_expect_tx(&done, 16u);
    sv::bulk_copy_g2s(&dst, src, 16u, &done, sv::l2_policy_evict_first());
    int32_t st = 0;
    if (!sv::mbar_wait_bounded(&done, 0, limit)) st |= SV_ST_TIMEOUT;  // the copy lands: no timeout expected
    const bool copied = st == 0 && dst.x == src->x && dst.w == src->w;
    if (!sv::mbar_wait_bounded(&never, 0, limit)) st |= SV_ST_TIMEOUT;
    // the copy that was issued has landed (or the wait for it already gave up)
    status[0] = st;
    status[1] = copied ? 1 : 0;
}

}  // namespace

extern "C" int sv_selftest_wait_timeout(const void* src16, int32_t* status, int64_t limit_cycles, sv_stream_t stream)
{
    if (src16 == nullptr || status == nullptr || limit_cycles < 1) return SV_ERR_INVALID_ARG;
    if (reinterpret_cast<uintptr_t>(src16) % 16 != 0 || reinterpret_cast<uintptr_t>(status) % 4 != 0)
        return SV_ERR_ALIGN;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return SV_ERR_DEVICE;
    wait_timeout_kernel<<<1, 32, 0, reinterpret_cast<cudaStream_t>(stream)>>>(static_cast<const uint4*>(src16), status,
                                                                            static_cast<long long>(limit_cycles));
    return cudaGetLastError() == cudaSuccess ? SV_OK : SV_ERR_LAUNCH;
}
