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
// and runs the per-request scan and branch choice (one main branch, or up to
// eight branches sharing the first row), one CTA per request; it is launched
// as a programmatic dependent of kernel 1 so its launch overlaps kernel 1.
// With the top-2 output, kernel 1 also keeps each thread's two first
// (value, position) pairs and kernel 2 merges them into every row's argmax and
// runner-up id.  Modality inference reuses kernel 1 on full-vocabulary rows,
// then maps each row's argmax to its vocabulary partition
// (modality_finalize_kernel).
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

// ---- argmax and runner-up: the two first ids in (value descending, id
// ascending) order, NaN read as -inf --------------------------------------
// A thread keeps its two first (value, position) pairs, a position being the
// start of a 16-byte vector (bulk part) or an exact id (tail).  Per vector it
// takes the vector's two largest values with packed max / min instructions and
// merges them with selects; the exact ids are resolved once per segment.
struct Top2 {
    float v1;
    int32_t x1;  // INT32_MAX: none
    float v2;
    int32_t x2;
};

__device__ __forceinline__ uint32_t bmin2(uint32_t a, uint32_t b)
{
    uint32_t d;
    asm("min.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}

// the two largest values W1 >= W2 of a vector (a duplicated maximum gives W1 == W2); W1 is
// NaN when the vector holds a NaN
template <int DT>
__device__ __forceinline__ void vec_top2_vals(uint4 q, float& W1, float& W2)
{
    if constexpr (DT == SV_BF16) {
        const uint32_t T1 = bmax2_nan(q.x, q.y), T2 = bmin2(q.x, q.y);
        const uint32_t U1 = bmax2_nan(q.z, q.w), U2 = bmin2(q.z, q.w);
        const uint32_t V1 = bmax2_nan(T1, U1), V2 = bmax2_nan(bmin2(T1, U1), bmax2_nan(T2, U2));
        const float a = bf16_lo(V1), b = bf16_hi(V1);
        W1 = fmax_nan(a, b);
        W2 = fmaxf(fminf(a, b), fmaxf(bf16_lo(V2), bf16_hi(V2)));
    } else {
        const float a = __uint_as_float(q.x), b = __uint_as_float(q.y);
        const float c = __uint_as_float(q.z), d = __uint_as_float(q.w);
        const float T1 = fmax_nan(a, b), U1 = fmax_nan(c, d);
        W1 = fmax_nan(T1, U1);
        W2 = fmaxf(fminf(T1, U1), fmaxf(fminf(a, b), fminf(c, d)));
    }
}

// a vector at position xv, after every position the thread has taken: equal values keep the
// earlier pair
__device__ __forceinline__ void top2_take_vec(Top2& s, float W1, float W2, int32_t xv)
{
    const bool e1 = s.x1 == INT32_MAX, e2 = s.x2 == INT32_MAX;
    const bool up1 = e1 || W1 > s.v1;
    const bool sec = e1 || W2 > s.v1;  // with up1: the vector's second value beats the old first
    const bool up2 = e2 || W1 > s.v2;  // without up1: the vector's first value beats the old second
    const float nv2 = up1 ? (sec ? W2 : s.v1) : (up2 ? W1 : s.v2);
    const int32_t nx2 = up1 ? (sec ? xv : s.x1) : (up2 ? xv : s.x2);
    s.v1 = up1 ? W1 : s.v1;
    s.x1 = up1 ? xv : s.x1;
    s.v2 = nv2;
    s.x2 = nx2;
}

__device__ __forceinline__ void top2_take_one(Top2& s, float f, int32_t x)
{
    if (s.x1 == INT32_MAX || f > s.v1) {
        s.v2 = s.v1;
        s.x2 = s.x1;
        s.v1 = f;
        s.x1 = x;
    } else if (s.x2 == INT32_MAX || f > s.v2) {
        s.v2 = f;
        s.x2 = x;
    }
}

template <int DT>
__device__ __forceinline__ void vec_take2(Top2& st, uint32_t& flags, uint4 q, int32_t x)
{
    float W1, W2;
    vec_top2_vals<DT>(q, W1, W2);
    if (W1 != W1) {  // rare: a NaN in the vector, read as -inf
        flags |= kFlagNaN;
        if constexpr (DT == SV_BF16) {
            q = make_uint4(bf16x2_nan_to_ninf(q.x), bf16x2_nan_to_ninf(q.y), bf16x2_nan_to_ninf(q.z),
                           bf16x2_nan_to_ninf(q.w));
        } else {
            const uint32_t ninf = 0xFF800000u;
            q.x = __uint_as_float(q.x) != __uint_as_float(q.x) ? ninf : q.x;
            q.y = __uint_as_float(q.y) != __uint_as_float(q.y) ? ninf : q.y;
            q.z = __uint_as_float(q.z) != __uint_as_float(q.z) ? ninf : q.z;
            q.w = __uint_as_float(q.w) != __uint_as_float(q.w) ? ninf : q.w;
        }
        vec_top2_vals<DT>(q, W1, W2);
    }
    top2_take_vec(st, W1, W2, x);
}

// (value, id) pairs: does (v, i) come before (w, j)?  INT32_MAX ids (none) come last
__device__ __forceinline__ bool ranks_before(float v, int32_t i, float w, int32_t j)
{
    if (i == INT32_MAX) return false;
    if (j == INT32_MAX) return true;
    return v > w || (v == w && i < j);
}

// the two first of two sorted pairs
__device__ __forceinline__ Top2 top2_merge(const Top2& a, const Top2& b)
{
    Top2 r;
    if (ranks_before(a.v1, a.x1, b.v1, b.x1)) {
        r.v1 = a.v1;
        r.x1 = a.x1;
        const bool t = ranks_before(a.v2, a.x2, b.v1, b.x1);
        r.v2 = t ? a.v2 : b.v1;
        r.x2 = t ? a.x2 : b.x1;
    } else {
        r.v1 = b.v1;
        r.x1 = b.x1;
        const bool t = ranks_before(a.v1, a.x1, b.v2, b.x2);
        r.v2 = t ? a.v1 : b.v2;
        r.x2 = t ? a.x1 : b.x2;
    }
    return r;
}

__device__ __forceinline__ Top2 top2_shfl(const Top2& s, int o)
{
    return Top2{__shfl_xor_sync(0xffffffffu, s.v1, o), __shfl_xor_sync(0xffffffffu, s.x1, o),
                __shfl_xor_sync(0xffffffffu, s.v2, o), __shfl_xor_sync(0xffffffffu, s.x2, o)};
}

template <int DT, bool TOP2>
__global__ void __launch_bounds__(kArgThreads)
    argmax_segments_kernel(const char* __restrict__ base, int64_t row_stride_bytes, int32_t V,
                           int32_t seg_len, int32_t nseg, int use_bulk,
                           void* __restrict__ out_raw)
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
    Top2 s2{-INFINITY, INT32_MAX, -INFINITY, INT32_MAX};
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
            for (int t = threadIdx.x; t < nv; t += kArgThreads) {
                if constexpr (TOP2)
                    vec_take2<DT>(s2, flags, vp[t], xc + t * VEC);
                else
                    vec_take<DT>(st, flags, vp[t], xc + t * VEC);
            }
        }
        if (!ok) {
            flags |= kFlagTimeout;
            // let copies still in flight land (bounded) before the CTA exits
            for (int c = 0; c < nch; ++c) (void)mbar_wait_bounded(&bars[c], 0);
        }
    }
    // the sub-16-byte tail, or the whole segment when bulk copies are off;
    // every thread still visits its elements in ascending order
    for (int32_t e = nbulk + threadIdx.x; e < len; e += kArgThreads) {
        if constexpr (TOP2) {
            float f = load_one<DT>(src, e);
            if (f != f) {
                flags |= kFlagNaN;
                f = -INFINITY;
            }
            top2_take_one(s2, f, x0 + e);
        } else {
            scalar_take(st, flags, load_one<DT>(src, e), x0 + e);
        }
    }
    if constexpr (TOP2) {
        // exact ids: a bulk position is a vector start, resolved from shared memory
        auto value_at = [&](int32_t x) -> float {
            const int32_t le = x - x0;
            float f;
            if constexpr (DT == SV_BF16)
                f = __uint_as_float(static_cast<uint32_t>(reinterpret_cast<const uint16_t*>(buf)[le]) << 16);
            else
                f = reinterpret_cast<const float*>(buf)[le];
            return f != f ? -INFINITY : f;
        };
        const int32_t xb = x0 + nbulk;  // positions below are vector starts
        int32_t i1 = s2.x1, i2 = s2.x2;
        if (s2.x1 != INT32_MAX && s2.x1 < xb) {
            for (int e = 0; e < VEC; ++e)
                if (value_at(s2.x1 + e) == s2.v1) {
                    i1 = s2.x1 + e;
                    break;
                }
        }
        if (s2.x2 != INT32_MAX && s2.x2 < xb) {
            // the second value of the first pair's own vector skips that pair's id
            const int32_t skip = s2.x2 == s2.x1 ? i1 : INT32_MAX;
            for (int e = 0; e < VEC; ++e)
                if (s2.x2 + e != skip && value_at(s2.x2 + e) == s2.v2) {
                    i2 = s2.x2 + e;
                    break;
                }
        }
        Top2 r{s2.v1, i1, s2.v2, i2};
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) r = top2_merge(r, top2_shfl(r, o));
        flags = __reduce_or_sync(0xffffffffu, flags);
        __shared__ Top2 wtop[kArgThreads / 32];
        __shared__ uint32_t wfl2[kArgThreads / 32];
        const int warp2 = threadIdx.x >> 5;
        if ((threadIdx.x & 31) == 0) {
            wtop[warp2] = r;
            wfl2[warp2] = flags;
        }
        __syncthreads();
        if (threadIdx.x == 0) {
            Top2 b = wtop[0];
            uint32_t f = wfl2[0];
            for (int w = 1; w < kArgThreads / 32; ++w) {
                b = top2_merge(b, wtop[w]);
                f |= wfl2[w];
            }
            static_cast<Top2Partial*>(out_raw)[unit] = Top2Partial{b.v1, b.x1, b.v2, b.x2, f, {0u, 0u, 0u}};
        }
        return;
    }
    ArgPartial* out = static_cast<ArgPartial*>(out_raw);

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
// (independent loads, several in flight), then warp 0 runs the scan.  With
// TOP2 the segments hold the two first ids, and every row's pair is written.
template <bool TOP2>
__global__ void __launch_bounds__(kFinThreads)
    greedy_finalize_kernel(const void* __restrict__ part_raw, int32_t nseg, int32_t R, int32_t k,
                           int32_t branches, int32_t V, const int32_t* __restrict__ draft,
                           int32_t* __restrict__ accept_len, int32_t* __restrict__ tokens,
                           int32_t* __restrict__ branch_out, int32_t* __restrict__ status,
                           int32_t* __restrict__ top2)
{
    pdl_wait_primary();
    extern __shared__ int32_t fin_amax[];
    __shared__ uint32_t st_shared;
    const int64_t r = blockIdx.x;
    const int32_t rpr = 1 + branches * k;
    if (threadIdx.x == 0) st_shared = 0;
    __syncthreads();
    uint32_t st = 0;
    for (int32_t i = threadIdx.x; i < rpr; i += kFinThreads) {
        ArgMax best{-INFINITY, INT32_MAX};
        uint32_t fl = 0;
        if constexpr (TOP2) {
            const Top2Partial* p = static_cast<const Top2Partial*>(part_raw) + (r * rpr + i) * nseg;
            Top2 b{-INFINITY, INT32_MAX, -INFINITY, INT32_MAX};
            for (int32_t s = 0; s < nseg; ++s) {
                const Top2Partial q = p[s];
                fl |= q.flags;
                b = top2_merge(b, Top2{q.v1, q.i1, q.v2, q.i2});
            }
            best = ArgMax{b.v1, b.x1};
            top2[2 * (r * rpr + i)] = b.x1 == INT32_MAX ? 0 : b.x1;
            top2[2 * (r * rpr + i) + 1] = b.x2 == INT32_MAX ? -1 : b.x2;
        } else {
            const ArgPartial* p = static_cast<const ArgPartial*>(part_raw) + (r * rpr + i) * nseg;
#pragma unroll 8
            for (int32_t s = 0; s < nseg; ++s) {
                const ArgPartial q = p[s];
                fl |= q.flags;
                if (argmax_better(q.v, q.i, best)) best = ArgMax{q.v, q.i};
            }
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

// One thread per row: the row's argmax from its segment results, then the
// partition holding it (the text part or an audio codebook) and that
// partition's id range, the phase mask of the next step.
__global__ void __launch_bounds__(kFinThreads)
    modality_finalize_kernel(const ArgPartial* __restrict__ part, int32_t nseg, int64_t rows, PartTable pt,
                             int32_t* __restrict__ amax, int32_t* __restrict__ part_out,
                             int32_t* __restrict__ mask_lo, int32_t* __restrict__ mask_hi,
                             int32_t* __restrict__ status)
{
    pdl_wait_primary();
    const int64_t row = static_cast<int64_t>(blockIdx.x) * kFinThreads + threadIdx.x;
    if (row >= rows) return;
    const ArgPartial* p = part + row * nseg;
    ArgMax best{-INFINITY, INT32_MAX};
    uint32_t fl = 0;
    for (int32_t s = 0; s < nseg; ++s) {
        const ArgPartial q = p[s];
        fl |= q.flags;
        if (argmax_better(q.v, q.i, best)) best = ArgMax{q.v, q.i};
    }
    const int32_t a = best.i == INT32_MAX ? 0 : best.i;
    int32_t pi = -1;
    for (int32_t q = 0; q < pt.P; ++q)  // ascending starts: the first range holding a
        if (pt.start[q] <= a && a < pt.start[q + 1]) {
            pi = q;
            break;
        }
    if (amax) amax[row] = a;
    part_out[row] = pi;
    if (mask_lo) mask_lo[row] = pi < 0 ? 0 : pt.start[pi];
    if (mask_hi) mask_hi[row] = pi < 0 ? 0 : pt.start[pi + 1];
    if (status) {
        uint32_t st = 0;
        if ((fl & kFlagNaN) || isinf(best.v)) st |= SV_ST_BAD_LOGITS;
        if (fl & kFlagTimeout) st |= SV_ST_TIMEOUT;
        status[row] = static_cast<int32_t>(st);
    }
}

size_t greedy_workspace_bytes(int64_t R, int32_t k, int32_t branches, int32_t V, bool top2)
{
    const int64_t rows = R * (1 + static_cast<int64_t>(branches) * k);
    int64_t nseg = 1;
    for (int es : {2, 4}) nseg = std::max<int64_t>(nseg, plan_segments(rows, V, es).nseg);
    return static_cast<size_t>(rows * nseg) * (top2 ? sizeof(Top2Partial) : sizeof(ArgPartial)) + 256;
}

template <int DT, bool TOP2>
static cudaError_t launch_argmax(const Rows& t, int64_t rows, const SegPlan& plan, void* out, cudaStream_t stream)
{
    const int64_t units = rows * plan.nseg;
    const size_t smem = kSmemHeader + (t.bulk_ok ? static_cast<size_t>(plan.seg_len) * t.esize : 0);
    cudaError_t e = cudaFuncSetAttribute(argmax_segments_kernel<DT, TOP2>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(kSmemHeader + kSegMaxBytes));
    if (e != cudaSuccess) return e;
    argmax_segments_kernel<DT, TOP2><<<static_cast<unsigned>(units), kArgThreads, smem, stream>>>(
        t.data, t.stride * t.esize, t.width, plan.seg_len, plan.nseg, t.bulk_ok ? 1 : 0, out);
    return cudaGetLastError();
}

cudaError_t launch_verify_greedy(const Rows& target, int32_t R, int32_t k, int32_t branches,
                                 const int32_t* draft, int32_t* accept_len, int32_t* tokens,
                                 int32_t* branch, int32_t* status, void* workspace,
                                 cudaStream_t stream, int32_t* top2)
{
    const int64_t rows = static_cast<int64_t>(R) * (1 + static_cast<int64_t>(branches) * k);
    const SegPlan plan = plan_segments(rows, target.width, target.esize);
    void* part = workspace;
    const bool bf = target.dtype == SV_BF16;
    cudaError_t e = top2 ? (bf ? launch_argmax<SV_BF16, true>(target, rows, plan, part, stream)
                               : launch_argmax<SV_F32, true>(target, rows, plan, part, stream))
                         : (bf ? launch_argmax<SV_BF16, false>(target, rows, plan, part, stream)
                               : launch_argmax<SV_F32, false>(target, rows, plan, part, stream));
    if (e != cudaSuccess) return e;

    const int32_t rpr = 1 + branches * k;
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
    if (top2)
        return cudaLaunchKernelEx(&cfg, greedy_finalize_kernel<true>, static_cast<const void*>(part), plan.nseg,
                                  R, k, branches, target.width, draft, accept_len, tokens, branch, status, top2);
    return cudaLaunchKernelEx(&cfg, greedy_finalize_kernel<false>, static_cast<const void*>(part), plan.nseg, R,
                              k, branches, target.width, draft, accept_len, tokens, branch, status, top2);
}

size_t modality_workspace_bytes(int64_t rows, int32_t V)
{
    int64_t nseg = 1;
    for (int es : {2, 4}) nseg = std::max<int64_t>(nseg, plan_segments(rows, V, es).nseg);
    return static_cast<size_t>(rows * nseg) * sizeof(ArgPartial) + 256;
}

cudaError_t launch_infer_modality(const Rows& rows, int64_t nrows, const PartTable& pt, int32_t* amax,
                                  int32_t* part, int32_t* mask_lo, int32_t* mask_hi, int32_t* status,
                                  void* workspace, cudaStream_t stream)
{
    const SegPlan plan = plan_segments(nrows, rows.width, rows.esize);
    cudaError_t e = rows.dtype == SV_BF16 ? launch_argmax<SV_BF16, false>(rows, nrows, plan, workspace, stream)
                                          : launch_argmax<SV_F32, false>(rows, nrows, plan, workspace, stream);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>((nrows + kFinThreads - 1) / kFinThreads));
    cfg.blockDim = dim3(kFinThreads);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, modality_finalize_kernel, static_cast<const ArgPartial*>(workspace), plan.nseg,
                              nrows, pt, amax, part, mask_lo, mask_hi, status);
}

}  // namespace sv
