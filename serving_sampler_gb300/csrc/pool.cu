// Hypothesis pool ("Decode Before You Hear ...", method steps 3 and 5): each
// request keeps every draft of its session in a device-resident pool, and
// while the output continues, the longest n-gram of the pool that matches the
// emitted suffix supplies its continuation as the next drafts.
//
// Layout: a request's pool is int32 [Lp], its drafts in insertion order, each
// followed by -1; pool_len[r] entries are in use.  Because the separators are
// negative and the suffix's padding is negative, a match never crosses a
// draft boundary or runs past the emitted output.
//
// Lookup: one CTA per request scans every end position p once.  A position
// is a candidate when pool[p] equals the newest emitted token and pool[p + 1]
// is a token; only candidates walk backwards, so the scan reads the pool
// about once (two coalesced loads per position, the second an L1 hit).  The
// best (length, p) is one 32-bit key, length << 24 | p, so the longest match
// and then the latest position win a plain maximum.
#include "sv_device.cuh"
#include "sv_internal.h"

namespace sv {

constexpr int kPoolThreads = 256;
static_assert(SV_MAX_NGRAM < 128 && SV_MAX_POOL <= (1 << 24), "key layout: length << 24 | position");

__global__ void __launch_bounds__(kPoolThreads)
    pool_append_kernel(int32_t* __restrict__ pool, int32_t* __restrict__ pool_len, int32_t Lp,
                       const int32_t* __restrict__ drafts, int32_t k, int32_t* __restrict__ status)
{
    __shared__ int32_t s_len;
    const int64_t r = blockIdx.x;
    const int32_t* D = drafts + r * k;
    if (threadIdx.x == 0) s_len = k;
    __syncthreads();
    for (int32_t i = threadIdx.x; i < k; i += kPoolThreads)
        if (D[i] < 0) atomicMin(&s_len, i);
    __syncthreads();
    const int32_t L = s_len;
    const int32_t used = pool_len[r];
    const bool fits = L > 0 && used >= 0 && used <= Lp && static_cast<int64_t>(used) + L + 1 <= Lp;
    if (fits) {
        int32_t* P = pool + r * Lp + used;
        for (int32_t i = threadIdx.x; i < L; i += kPoolThreads) P[i] = D[i];
        if (threadIdx.x == 0) P[L] = -1;
    }
    __syncthreads();  // every thread has read pool_len[r]
    if (threadIdx.x == 0) {
        if (fits) pool_len[r] = used + L + 1;
        if (status != nullptr) status[r] = (L > 0 && !fits) ? SV_ST_POOL_FULL : 0;
    }
}

__global__ void __launch_bounds__(kPoolThreads)
    pool_lookup_kernel(const int32_t* __restrict__ pool, const int32_t* __restrict__ pool_len, int32_t Lp,
                       const int32_t* __restrict__ suffix, int32_t N, int32_t gamma,
                       int32_t* __restrict__ match_len, int32_t* __restrict__ cont)
{
    __shared__ int32_t s_suf[SV_MAX_NGRAM];
    __shared__ uint32_t s_best;
    __shared__ int32_t s_end;
    const int64_t r = blockIdx.x;
    const int32_t* P = pool + r * Lp;
    const int32_t len = min(max(pool_len[r], 0), Lp);
    for (int32_t i = threadIdx.x; i < N; i += kPoolThreads) s_suf[i] = suffix[r * N + i];
    if (threadIdx.x == 0) {
        s_best = 0u;
        s_end = gamma;
    }
    __syncthreads();

    const int32_t last = N > 0 ? s_suf[N - 1] : -1;
    uint32_t best = 0u;
    if (last >= 0) {
        for (int32_t p = threadIdx.x; p + 1 < len; p += kPoolThreads) {
            const int32_t v = __ldg(P + p), next = __ldg(P + p + 1);
            if (v != last || next < 0) continue;
            int32_t n = 1;
            while (n < N && n <= p) {
                const int32_t a = __ldg(P + p - n), b = s_suf[N - 1 - n];
                if (a < 0 || a != b) break;  // b < 0 with a >= 0 also breaks here
                ++n;
            }
            best = max(best, (static_cast<uint32_t>(n) << 24) | static_cast<uint32_t>(p));
        }
    }
    best = __reduce_max_sync(0xffffffffu, best);
    if ((threadIdx.x & 31) == 0) atomicMax(&s_best, best);
    __syncthreads();
    best = s_best;
    const int32_t n = static_cast<int32_t>(best >> 24);
    const int32_t from = static_cast<int32_t>(best & 0xFFFFFFu) + 1;  // continuation start when n > 0

    // the continuation ends at the draft's separator, the pool's end or gamma
    for (int32_t i = threadIdx.x; i < gamma; i += kPoolThreads)
        if (n == 0 || from + i >= len || __ldg(P + from + i) < 0) atomicMin(&s_end, i);
    __syncthreads();
    const int32_t end = s_end;
    for (int32_t i = threadIdx.x; i < gamma; i += kPoolThreads)
        cont[r * gamma + i] = i < end ? __ldg(P + from + i) : -1;
    if (threadIdx.x == 0) match_len[r] = n;
}

// The emitted suffix after a verify step: one warp per request reads the old
// suffix and the step's committed tokens (its n accepted drafts and the
// correction) into registers, then writes the last N of the concatenation.
constexpr int kSuffixWarps = 8;

__global__ void __launch_bounds__(kSuffixWarps * 32)
    suffix_append_kernel(int32_t* __restrict__ suffix, int32_t N, int32_t R, const int32_t* __restrict__ tokens,
                         const int32_t* __restrict__ accept_len, int32_t k)
{
    const int lane = threadIdx.x & 31;
    const int64_t r = static_cast<int64_t>(blockIdx.x) * kSuffixWarps + (threadIdx.x >> 5);
    if (r >= R) return;
    const int32_t n = min(max(accept_len[r], 0), k);
    const int32_t shift = n + 1;  // tokens committed by the step
    int32_t* S = suffix + r * N;
    const int32_t* tk = tokens + r * (k + 1);
    // new[i] = old[i + shift] while that lies in the old suffix, else tokens[i + shift - N]
    int32_t val[SV_MAX_NGRAM / 32];
#pragma unroll
    for (int h = 0; h < SV_MAX_NGRAM / 32; ++h) {
        const int32_t i = lane + 32 * h;
        const int32_t src = i + shift;
        val[h] = i < N ? (src < N ? S[src] : tk[src - N]) : 0;
    }
    __syncwarp();  // every lane has read the old suffix before any lane overwrites it
#pragma unroll
    for (int h = 0; h < SV_MAX_NGRAM / 32; ++h) {
        const int32_t i = lane + 32 * h;
        if (i < N) S[i] = val[h];
    }
}

cudaError_t launch_suffix_append(int32_t* suffix, int32_t N, int32_t R, const int32_t* tokens,
                                 const int32_t* accept_len, int32_t k, cudaStream_t stream)
{
    const unsigned blocks = static_cast<unsigned>((R + kSuffixWarps - 1) / kSuffixWarps);
    suffix_append_kernel<<<blocks, kSuffixWarps * 32, 0, stream>>>(suffix, N, R, tokens, accept_len, k);
    return cudaGetLastError();
}

cudaError_t launch_pool_append(int32_t* pool, int32_t* pool_len, int32_t Lp, const int32_t* drafts,
                               int32_t k, int32_t R, int32_t* status, cudaStream_t stream)
{
    pool_append_kernel<<<static_cast<unsigned>(R), kPoolThreads, 0, stream>>>(pool, pool_len, Lp, drafts, k,
                                                                               status);
    return cudaGetLastError();
}

cudaError_t launch_pool_lookup(const int32_t* pool, const int32_t* pool_len, int32_t Lp, const int32_t* suffix,
                               int32_t N, int32_t R, int32_t gamma, int32_t* match_len, int32_t* cont,
                               cudaStream_t stream)
{
    pool_lookup_kernel<<<static_cast<unsigned>(R), kPoolThreads, 0, stream>>>(pool, pool_len, Lp, suffix, N,
                                                                               gamma, match_len, cont);
    return cudaGetLastError();
}

}  // namespace sv
