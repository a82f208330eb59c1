// Greedy verification ("Decode Before You Hear: Speculative Listening ...",
// method steps 2 and 4): argmax of every target row, then per request the
// first draft position whose token differs from the row's argmax, the branch
// choice and the commit.
//
// Kernel 1 (argmax_segments_kernel) streams each row segment from HBM into
// shared memory with 1-D bulk copies (TMA) in 8 KB chunks, one mbarrier per
// chunk, and reduces (max, first index) while later chunks are in flight.
// The inner step takes the NaN-propagating max of 8 bf16 values with three
// packed max instructions and keeps (max, vector start) with two selects;
// the first index inside the winning vector is found once per segment.  Only
// a vector holding a NaN leaves the straight-line path.
// Kernel 2 (greedy_finalize_kernel) merges the segment results of each row
// and runs the per-request scan, one CTA per request; it is launched as a
// programmatic dependent of kernel 1 so its launch overlaps kernel 1.
#include <algorithm>
#include <cfloat>
#include <climits>

#include "sv_device.cuh"
#include "sv_internal.h"

namespace sv {

constexpr int kArgThreads = 128;
constexpr uint32_t kChunkBytes = 8192;
constexpr uint32_t kSegMaxBytes = 32768;
constexpr uint32_t kSegMinBytes = 4096;
constexpr int kSmemHeader = 128;  // chunk barriers live here
constexpr int64_t kTargetUnits = 4096;

SegPlan plan_segments(int64_t rows, int32_t width, int esize)
{
    const int vec = 16 / esize;
    const int64_t bytes = (int64_t)width * esize;
    int64_t nseg = (bytes + kSegMaxBytes - 1) / kSegMaxBytes;
    if (rows > 0 && rows * nseg < kTargetUnits) {
        // small batches: cut rows finer so the grid still covers every SM
        const int64_t want = (kTargetUnits + rows - 1) / rows;
        const int64_t cap = (bytes + kSegMinBytes - 1) / kSegMinBytes;
        nseg = std::max<int64_t>(nseg, std::min(want, cap));
    }
    if (nseg < 1) nseg = 1;
    int64_t seg_len = (width + nseg - 1) / nseg;
    seg_len = (seg_len + vec - 1) / vec * vec;
    if (seg_len < 1) seg_len = vec;
    nseg = (width + seg_len - 1) / seg_len;
    if (nseg < 1) nseg = 1;
    return SegPlan{(int32_t)nseg, (int32_t)seg_len};
}

template <int DT>
__device__ __forceinline__ float load_one(const char* p, int32_t e)
{
    if constexpr (DT == SV_BF16) {
        const uint16_t h = reinterpret_cast<const uint16_t*>(p)[e];
        return __uint_as_float(static_cast<uint32_t>(h) << 16);
    } else {
        return reinterpret_cast<const float*>(p)[e];
    }
}

// Running state of one thread: the largest value seen and the first index of
// the 16-byte vector (or single tail element) where it was first seen.  The
// exact index inside that vector is resolved once per segment, so the hot
// loop has no divergent branch: a new maximum is taken with two selects.
struct VecMax {
    float v;
    int32_t x;
};

__device__ __forceinline__ void vecmax_take(VecMax& st, float vm, int32_t x)
{
    const bool up = vm > st.v;
    st.v = up ? vm : st.v;
    st.x = up ? x : st.x;
}

__device__ __forceinline__ void scalar_take(VecMax& st, uint32_t& flags, float f, int32_t x)
{
    if (f != f) {
        flags |= kFlagNaN;
        return;
    }
    vecmax_take(st, f, x);
}

// one 16-byte vector of 8 bf16 or 4 fp32 values whose first index is x
template <int DT>
__device__ __forceinline__ void vec_take(VecMax& st, uint32_t& flags, uint4 q, int32_t x)
{
    float vm;
    if constexpr (DT == SV_BF16) {
        const uint32_t m = bmax2_nan(bmax2_nan(q.x, q.y), bmax2_nan(q.z, q.w));
        vm = fmax_nan(bf16_lo(m), bf16_hi(m));
    } else {
        vm = fmax_nan(fmax_nan(__uint_as_float(q.x), __uint_as_float(q.y)),
                      fmax_nan(__uint_as_float(q.z), __uint_as_float(q.w)));
    }
    if (vm != vm) {  // rare: a NaN in the vector; take the max of the others
        flags |= kFlagNaN;
        const uint32_t w[4] = {q.x, q.y, q.z, q.w};
        vm = -INFINITY;
        if constexpr (DT == SV_BF16) {
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                const float f = (e & 1) ? bf16_hi(w[e >> 1]) : bf16_lo(w[e >> 1]);
                vm = f > vm ? f : vm;
            }
        } else {
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const float f = __uint_as_float(w[e]);
                vm = f > vm ? f : vm;
            }
        }
    }
    vecmax_take(st, vm, x);
}

template <int DT>
__global__ void __launch_bounds__(kArgThreads)
    argmax_segments_kernel(const char* __restrict__ base, int64_t row_stride_bytes, int32_t V,
                           int32_t seg_len, int32_t nseg, int use_bulk,
                           ArgPartial* __restrict__ out)
{
    extern __shared__ __align__(128) unsigned char smem[];
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem);
    unsigned char* buf = smem + kSmemHeader;
    constexpr int ES = DT == SV_BF16 ? 2 : 4;
    constexpr int VEC = 16 / ES;

    // the finalize kernel may be scheduled now; it waits for this grid anyway
    pdl_launch_dependents();

    const int64_t unit = blockIdx.x;
    const int64_t row = unit / nseg;
    const int32_t seg = static_cast<int32_t>(unit - row * nseg);
    const int32_t x0 = seg * seg_len;
    const int32_t len = max(0, min(V, x0 + seg_len) - x0);
    const char* src = base + row * row_stride_bytes + static_cast<int64_t>(x0) * ES;

    VecMax st{-INFINITY, INT32_MAX};
    uint32_t flags = 0;
    int32_t nbulk = 0;
    if (use_bulk) {
        const uint32_t bulk_bytes = static_cast<uint32_t>(len * ES) & ~15u;
        nbulk = static_cast<int32_t>(bulk_bytes / ES);
        const int nch = static_cast<int>((bulk_bytes + kChunkBytes - 1) / kChunkBytes);
        if (threadIdx.x == 0) {
            for (int c = 0; c < nch; ++c) mbar_init(&bars[c], 1);
            fence_barrier_init();
        }
        __syncthreads();
        if (threadIdx.x == 0) {
            const uint64_t pol = l2_policy_evict_first();
            for (int c = 0; c < nch; ++c) {
                const uint32_t off = c * kChunkBytes;
                const uint32_t nb = min(kChunkBytes, bulk_bytes - off);
                mbar_arrive_expect_tx(&bars[c], nb);
                bulk_copy_g2s(buf + off, src + off, nb, &bars[c], pol);
            }
        }
        bool ok = true;
        for (int c = 0; c < nch; ++c) {
            if (!mbar_wait_bounded(&bars[c], 0)) {
                ok = false;
                break;
            }
            const uint32_t off = c * kChunkBytes;
            const uint32_t nb = min(kChunkBytes, bulk_bytes - off);
            const uint4* vp = reinterpret_cast<const uint4*>(buf + off);
            const int nv = static_cast<int>(nb / 16);
            const int32_t xc = x0 + static_cast<int32_t>(off / ES);
#pragma unroll 4
            for (int t = threadIdx.x; t < nv; t += kArgThreads) vec_take<DT>(st, flags, vp[t], xc + t * VEC);
        }
        if (!ok) {
            flags |= kFlagTimeout;
            // let copies still in flight land (bounded) before the CTA exits
            for (int c = 0; c < nch; ++c) (void)mbar_wait_bounded(&bars[c], 0);
        }
    }
    // the sub-16-byte tail, or the whole segment when bulk copies are off;
    // every thread still visits its elements in ascending order
    for (int32_t e = nbulk + threadIdx.x; e < len; e += kArgThreads)
        scalar_take(st, flags, load_one<DT>(src, e), x0 + e);

    // block reduction of (value, first vector start) and flags
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        const float ov = __shfl_xor_sync(0xffffffffu, st.v, o);
        const int32_t ox = __shfl_xor_sync(0xffffffffu, st.x, o);
        if (ov > st.v || (ov == st.v && ox < st.x)) st = VecMax{ov, ox};
    }
    flags = __reduce_or_sync(0xffffffffu, flags);
    __shared__ VecMax wbest[kArgThreads / 32];
    __shared__ uint32_t wflags[kArgThreads / 32];
    const int warp = threadIdx.x >> 5;
    if ((threadIdx.x & 31) == 0) {
        wbest[warp] = st;
        wflags[warp] = flags;
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        VecMax b = wbest[0];
        uint32_t f = wflags[0];
        for (int w = 1; w < kArgThreads / 32; ++w) {
            if (wbest[w].v > b.v || (wbest[w].v == b.v && wbest[w].x < b.x)) b = wbest[w];
            f |= wflags[w];
        }
        // the first element equal to the maximum, inside the winning vector
        int32_t idx = INT32_MAX;
        if (b.x != INT32_MAX) {
            for (int e = 0; e < VEC; ++e) {
                const int32_t le = b.x - x0 + e;
                if (le >= len) break;
                float f2;
                if (le < nbulk) {
                    if constexpr (DT == SV_BF16)
                        f2 = __uint_as_float(static_cast<uint32_t>(reinterpret_cast<const uint16_t*>(buf)[le]) << 16);
                    else
                        f2 = reinterpret_cast<const float*>(buf)[le];
                } else {
                    f2 = load_one<DT>(src, le);
                }
                if (f2 == b.v) {
                    idx = b.x + e;
                    break;
                }
            }
        }
        out[unit] = ArgPartial{b.v, idx, f, 0u};
    }
}

constexpr int kFinThreads = 256;

__device__ __forceinline__ int32_t branch_row(int32_t b, int32_t j, int32_t k)
{
    return j == 0 ? 0 : b * k + j;
}

// One CTA per request: every thread merges the segment results of some rows
// (independent loads, several in flight), then warp 0 runs the scan.
__global__ void __launch_bounds__(kFinThreads)
    greedy_finalize_kernel(const ArgPartial* __restrict__ part, int32_t nseg, int32_t R, int32_t k,
                           int32_t branches, int32_t V, const int32_t* __restrict__ draft,
                           int32_t* __restrict__ accept_len, int32_t* __restrict__ tokens,
                           int32_t* __restrict__ branch_out, int32_t* __restrict__ status)
{
    pdl_wait_primary();
    extern __shared__ int32_t fin_amax[];
    __shared__ uint32_t st_shared;
    const int64_t r = blockIdx.x;
    const int32_t rpr = branches == 1 ? k + 1 : 2 * k + 1;
    if (threadIdx.x == 0) st_shared = 0;
    __syncthreads();
    uint32_t st = 0;
    for (int32_t i = threadIdx.x; i < rpr; i += kFinThreads) {
        const ArgPartial* p = part + (r * rpr + i) * nseg;
        ArgMax best{-INFINITY, INT32_MAX};
        uint32_t fl = 0;
#pragma unroll 8
        for (int32_t s = 0; s < nseg; ++s) {
            const ArgPartial q = p[s];
            fl |= q.flags;
            if (argmax_better(q.v, q.i, best)) best = ArgMax{q.v, q.i};
        }
        fin_amax[i] = best.i == INT32_MAX ? 0 : best.i;
        if ((fl & kFlagNaN) || isinf(best.v)) st |= SV_ST_BAD_LOGITS;
        if (fl & kFlagTimeout) st |= SV_ST_TIMEOUT;
    }
    if (st) atomicOr(&st_shared, st);
    __syncthreads();
    if (threadIdx.x >= 32) return;
    const int lane = threadIdx.x;
    const int32_t* amax = fin_amax;
    st = 0;
    int32_t best_b = 0, best_n = 0;
    bool any = false;
    for (int32_t b = 0; b < branches; ++b) {
        const int32_t* d = draft + (r * branches + b) * k;
        for (int32_t j = lane; j < k; j += 32)
            if (d[j] < 0 || d[j] >= V) st |= SV_ST_TOKEN_RANGE;
        int32_t n = k;
        for (int32_t j0 = 0; j0 < k; j0 += 32) {
            const int32_t j = j0 + lane;
            const bool mism = j < k && d[j] != amax[branch_row(b, j, k)];
            const unsigned m = __ballot_sync(0xffffffffu, mism);
            if (m) {
                n = j0 + __ffs(m) - 1;
                break;
            }
        }
        const bool viable = (k == 0) || (n >= 1);
        if (viable && (!any || n > best_n)) {
            best_b = b;
            best_n = n;
            any = true;
        }
    }
    if (!any) {
        best_b = 0;
        best_n = 0;
    }
    const int32_t* d = draft + (r * branches + best_b) * k;
    const int32_t fix = amax[branch_row(best_b, best_n, k)];
    for (int32_t j = lane; j <= k; j += 32)
        tokens[r * (k + 1) + j] = j < best_n ? d[j] : (j == best_n ? fix : -1);
    st = __reduce_or_sync(0xffffffffu, st) | st_shared;
    if (lane == 0) {
        accept_len[r] = best_n;
        if (branch_out) branch_out[r] = best_b;
        if (status) status[r] = static_cast<int32_t>(st);
    }
}

size_t greedy_workspace_bytes(int64_t R, int32_t k, int32_t branches, int32_t V)
{
    const int64_t rows = R * (branches == 2 ? 2 * (int64_t)k + 1 : (int64_t)k + 1);
    int64_t nseg = 1;
    for (int es : {2, 4}) nseg = std::max<int64_t>(nseg, plan_segments(rows, V, es).nseg);
    return static_cast<size_t>(rows * nseg) * sizeof(ArgPartial) + 256;
}

template <int DT>
static cudaError_t launch_argmax(const Rows& t, int64_t rows, const SegPlan& plan, ArgPartial* out,
                                 cudaStream_t stream)
{
    const int64_t units = rows * plan.nseg;
    const size_t smem = kSmemHeader + (t.bulk_ok ? static_cast<size_t>(plan.seg_len) * t.esize : 0);
    cudaError_t e = cudaFuncSetAttribute(argmax_segments_kernel<DT>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(kSmemHeader + kSegMaxBytes));
    if (e != cudaSuccess) return e;
    argmax_segments_kernel<DT><<<static_cast<unsigned>(units), kArgThreads, smem, stream>>>(
        t.data, t.stride * t.esize, t.width, plan.seg_len, plan.nseg, t.bulk_ok ? 1 : 0, out);
    return cudaGetLastError();
}

cudaError_t launch_verify_greedy(const Rows& target, int32_t R, int32_t k, int32_t branches,
                                 const int32_t* draft, int32_t* accept_len, int32_t* tokens,
                                 int32_t* branch, int32_t* status, void* workspace,
                                 cudaStream_t stream)
{
    const int64_t rows = static_cast<int64_t>(R) * (branches == 2 ? 2 * k + 1 : k + 1);
    const SegPlan plan = plan_segments(rows, target.width, target.esize);
    ArgPartial* part = reinterpret_cast<ArgPartial*>(workspace);
    cudaError_t e = target.dtype == SV_BF16 ? launch_argmax<SV_BF16>(target, rows, plan, part, stream)
                                            : launch_argmax<SV_F32>(target, rows, plan, part, stream);
    if (e != cudaSuccess) return e;

    const int32_t rpr = branches == 2 ? 2 * k + 1 : k + 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(R));
    cfg.blockDim = dim3(kFinThreads);
    cfg.dynamicSmemBytes = static_cast<size_t>(rpr) * sizeof(int32_t);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, greedy_finalize_kernel, static_cast<const ArgPartial*>(part),
                              plan.nseg, R, k, branches, target.width, draft, accept_len, tokens,
                              branch, status);
}

}  // namespace sv
