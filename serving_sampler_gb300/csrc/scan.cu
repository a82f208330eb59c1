// Accept-length scan over caller-given accept flags and the commit
// ("Decode Before You Hear ...", method step 4: the accepted prefix ends at
// the first failure; "speculative decoding for Omni models", section 3: a
// draft counts only if every earlier draft was accepted).  One warp per
// request: a ballot over 32 positions at a time finds the first zero flag.
#include "sv_device.cuh"
#include "sv_internal.h"

namespace sv {

constexpr int kScanWarps = 8;

__global__ void __launch_bounds__(kScanWarps * 32)
    accept_scan_kernel(const uint8_t* __restrict__ accept, const int32_t* __restrict__ draft,
                       const int32_t* __restrict__ fix, int32_t R, int32_t k,
                       int32_t* __restrict__ accept_len, int32_t* __restrict__ tokens)
{
    const int lane = threadIdx.x & 31;
    const int64_t r = static_cast<int64_t>(blockIdx.x) * kScanWarps + (threadIdx.x >> 5);
    if (r >= R) return;
    int32_t n = k;
    for (int32_t j0 = 0; j0 < k; j0 += 32) {
        const int32_t j = j0 + lane;
        const unsigned m = __ballot_sync(0xffffffffu, j < k && accept[r * k + j] == 0);
        if (m) {
            n = j0 + __ffs(m) - 1;
            break;
        }
    }
    const int32_t f = fix[r * (k + 1) + n];
    for (int32_t j = lane; j <= k; j += 32)
        tokens[r * (k + 1) + j] = j < n ? draft[r * k + j] : (j == n ? f : -1);
    if (lane == 0) accept_len[r] = n;
}

cudaError_t launch_accept_scan(const uint8_t* accept, const int32_t* draft, const int32_t* fix,
                               int32_t R, int32_t k, int32_t* accept_len, int32_t* tokens,
                               cudaStream_t stream)
{
    const unsigned blocks = static_cast<unsigned>((R + kScanWarps - 1) / kScanWarps);
    accept_scan_kernel<<<blocks, kScanWarps * 32, 0, stream>>>(accept, draft, fix, R, k,
                                                              accept_len, tokens);
    return cudaGetLastError();
}

}  // namespace sv
