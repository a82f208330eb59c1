// Speculative sampling with a truncated draft vocabulary ("speculative
// decoding for Omni models", sections 2 and 4).
//
// Three kernels per call:
//   d2t_plan_kernel    one CTA: a bitmap of the d2t image over the target
//                      vocabulary, per-word prefix counts, and the support
//                      sorted by target id (xs[pos], js[pos]).  Every later
//                      pass visits the support in row order, so no pass
//                      gathers at random from a 300 KB target row.
//   sample_rows_kernel persistent CTAs, one (request, position) unit at a
//                      time.  The draft row y_j streams through a ring of
//                      bulk-copied 16 KB stages into a resident buffer Y
//                      while its max / sum-exp at T are taken; then the
//                      target row z_j streams through the same ring: max,
//                      sum-exp, argmax, NaN/inf flags, and z at the support
//                      positions (G[pos]).  A second pass over G and Y gives
//                      TV over the full vocabulary, p(x_j), q(x_j) and the
//                      accept test u_j < p/q.
//   race_commit_kernel RC CTAs per request: the accept-length scan, then the
//                      exponential race argmin E_x / w_x on the one selected
//                      row (residual max(0, p - q) at the first rejection, or
//                      p at the bonus row), Philox uniforms per element, CTA
//                      results merged with a 64-bit atomicMin; the last CTA
//                      of the request commits the tokens.
// Temperature scaling works in log2 units: with c = log2(e) / T,
// p(x) = 2^(z_x c - M) / S where M = max_x z_x c and S = sum 2^(z c - M).
#include <algorithm>
#include <cfloat>
#include <climits>

#include "sv_device.cuh"
#include "sv_internal.h"

namespace sv {

namespace {

constexpr int kPlanThreads = 1024;
constexpr int32_t kChunkElems = 2048;  // ids per bulk-copied chunk of the bf16 fast path (4 KB)
constexpr int kRowThreads = 512;
constexpr uint32_t kStageBytes = 16384;
constexpr int kStages = 4;
constexpr int kRowHeader = 128;
constexpr uint32_t kSmemBudget = 220 * 1024;
constexpr int kRaceThreads = 256;
constexpr int32_t kRaceSeg = 8192;  // elements of the race row per CTA
constexpr int32_t kMaxPlanWords = 25600;  // d2t mode supports V <= 819,200
constexpr float kLog2e = 1.4426950408889634f;

enum : uint32_t { kFlagAllNegInf = 8u, kFlagDraftBad = 16u, kFlagOffSupport = 32u };

struct D2tPlan {
    uint32_t* bitmap;  // [nw] support bits over target ids
    int32_t* prefix;   // [nw + 1] set bits before each word
    int32_t* xs;       // [Vd] support target ids, ascending
    int32_t* js;       // [Vd] the draft id of xs[pos]
    uint32_t* pairs;   // [Vd] (draft id << 16) | (xs & (kChunkElems - 1)), ascending xs (Vd <= 65535)
    int32_t* chunk;    // [V / kChunkElems + 2] support rank at every multiple of kChunkElems
    int32_t* x_of_j;   // [Vd] target id of every draft id (a copy of d2t)
    int32_t* header;   // [0] V, [1] Vd the plan was built for, [2] d2t out of range or repeated
    int32_t nw;
};

struct RowStat {
    float m, s;       // target: max of z c, sum 2^(z c - m)
    float mq, sq;     // draft row (sampling positions < k)
    float zx;         // z at the draft token
    float p, q;       // p(x_j), q(x_j)
    int32_t amax;     // raw argmax of the target row
    uint32_t flags;   // kFlag* of the target and draft rows
    int32_t accept;   // accept decision of position j
    int32_t rx;       // target id of the largest residual p - q on the support (-1: none)
    float rv;         // that residual
    float bkey;       // race key of the candidate bx_c if this row is raced (+inf: no bound)
    int32_t bxc;      // the candidate (-1: none)
};

struct RaceSlot {
    unsigned long long best;  // (key bits << 32) | x, minimum over the race CTAs
    unsigned int count;       // race CTAs done
    unsigned int pad;
};

struct SampleArgs {
    const char* tbase;
    int64_t tstride;  // bytes
    int32_t V;
    const char* dbase;
    int64_t dstride;  // bytes
    int32_t Vd;
    int identity;     // d2t == NULL
    int tbulk, dbulk; // rows 16-byte aligned
    D2tPlan plan;
    int32_t R, k;
    const int32_t* draft;
    const uint64_t* seeds;
    const float* temp;
    float* tv;
    float* pd;
    float* qd;
    int32_t* accept_len;
    int32_t* tokens;
    int32_t* status;
    RowStat* stats;
    RaceSlot* race;
    char* gslots;        // global-memory Y / G buffers when they do not fit in shared memory
    int64_t gslot_bytes;
    int smem_mode;
    int32_t race_ctas;   // CTAs per request in the race
    int32_t race_seg;    // elements per race CTA
};

__host__ __device__ inline int64_t align256(int64_t b) { return (b + 255) / 256 * 256; }

template <int DT>
__device__ __forceinline__ float ld_elem(const char* p, int64_t e)
{
    if constexpr (DT == SV_BF16) {
        const uint16_t h = reinterpret_cast<const uint16_t*>(p)[e];
        return __uint_as_float(static_cast<uint32_t>(h) << 16);
    } else {
        return reinterpret_cast<const float*>(p)[e];
    }
}

template <int DT>
__device__ __forceinline__ void st_elem(char* p, int64_t e, float v)
{
    if constexpr (DT == SV_BF16) {
        reinterpret_cast<uint16_t*>(p)[e] = static_cast<uint16_t>(__float_as_uint(v) >> 16);
    } else {
        reinterpret_cast<float*>(p)[e] = v;
    }
}

// number of support ids below x (x in [0, V])
__device__ __forceinline__ int32_t support_rank(const D2tPlan& pl, int32_t x)
{
    const int32_t w = x >> 5, b = x & 31;
    int32_t r = pl.prefix[w];
    if (b) r += __popc(pl.bitmap[w] & ((1u << b) - 1u));
    return r;
}

__device__ __forceinline__ bool in_support(const D2tPlan& pl, int32_t x)
{
    return (pl.bitmap[x >> 5] >> (x & 31)) & 1u;
}

// ---- block reductions (kRowThreads or kRaceThreads, any multiple of 32) ----
template <int NT>
__device__ __forceinline__ float block_sum(float v, float* scratch)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    const int w = threadIdx.x >> 5;
    __syncthreads();
    if ((threadIdx.x & 31) == 0) scratch[w] = v;
    __syncthreads();
    float t = 0.f;
    for (int i = 0; i < NT / 32; ++i) t += scratch[i];
    return t;
}

template <int NT>
__device__ __forceinline__ float block_max(float v, float* scratch)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    const int w = threadIdx.x >> 5;
    __syncthreads();
    if ((threadIdx.x & 31) == 0) scratch[w] = v;
    __syncthreads();
    float t = -INFINITY;
    for (int i = 0; i < NT / 32; ++i) t = fmaxf(t, scratch[i]);
    return t;
}

template <int NT>
__device__ __forceinline__ uint32_t block_or(uint32_t v, uint32_t* scratch)
{
    v = __reduce_or_sync(0xffffffffu, v);
    const int w = threadIdx.x >> 5;
    __syncthreads();
    if ((threadIdx.x & 31) == 0) scratch[w] = v;
    __syncthreads();
    uint32_t t = 0;
    for (int i = 0; i < NT / 32; ++i) t |= scratch[i];
    return t;
}

// (value, first position) maximum over the block
template <int NT>
__device__ __forceinline__ void block_argmax(float& v, int32_t& x, float* sv, int32_t* sx)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        const float ov = __shfl_xor_sync(0xffffffffu, v, o);
        const int32_t ox = __shfl_xor_sync(0xffffffffu, x, o);
        if (ov > v || (ov == v && ox < x)) {
            v = ov;
            x = ox;
        }
    }
    const int w = threadIdx.x >> 5;
    __syncthreads();
    if ((threadIdx.x & 31) == 0) {
        sv[w] = v;
        sx[w] = x;
    }
    __syncthreads();
    v = sv[0];
    x = sx[0];
    for (int i = 1; i < NT / 32; ++i)
        if (sv[i] > v || (sv[i] == v && sx[i] < x)) {
            v = sv[i];
            x = sx[i];
        }
}

// ---- online (max, sum 2^(t - max)) over scaled logits t ----------------------
struct Lse {
    float m, s;
};

// target row: max, sum, and the sum over ids outside the d2t support
struct Lse3 {
    float m, s, so;
};

// values of one 16-byte vector, NaN replaced by -inf; returns the max and
// whether a NaN was seen
template <int DT>
__device__ __forceinline__ int unpack_vec(uint4 q, float* f)
{
    if constexpr (DT == SV_BF16) {
        const uint32_t w[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            f[2 * e] = bf16_lo(w[e]);
            f[2 * e + 1] = bf16_hi(w[e]);
        }
        return 8;
    } else {
        f[0] = __uint_as_float(q.x);
        f[1] = __uint_as_float(q.y);
        f[2] = __uint_as_float(q.z);
        f[3] = __uint_as_float(q.w);
        return 4;
    }
}

}  // namespace

// ---------------------------------------------------------------------------
// d2t plan
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(kPlanThreads)
    d2t_plan_kernel(const int32_t* __restrict__ d2t, int32_t Vd, int32_t V, D2tPlan pl)
{
    extern __shared__ uint32_t plan_smem[];
    uint32_t* bits = plan_smem;
    int32_t* pref = reinterpret_cast<int32_t*>(plan_smem + pl.nw);
    __shared__ int32_t warp_tot[kPlanThreads / 32];
    __shared__ int bad_any;
    const int tid = threadIdx.x;
    pdl_launch_dependents();  // the row kernel streams rows while the plan is built
    if (tid == 0) bad_any = 0;
    for (int32_t w = tid; w < pl.nw; w += kPlanThreads) bits[w] = 0u;
    __syncthreads();
    int bad = 0;
    for (int32_t j = tid; j < Vd; j += kPlanThreads) {
        const int32_t x = d2t[j];
        if (x < 0 || x >= V) {
            bad = 1;
            continue;
        }
        const uint32_t bit = 1u << (x & 31);
        if (atomicOr(&bits[x >> 5], bit) & bit) bad = 1;
    }
    if (bad) atomicOr(&bad_any, 1);
    __syncthreads();
    // exclusive prefix of popcounts, each thread owning a contiguous block of words
    const int32_t per = (pl.nw + kPlanThreads - 1) / kPlanThreads;
    const int32_t w0 = min(pl.nw, tid * per), w1 = min(pl.nw, w0 + per);
    int32_t local = 0;
    for (int32_t w = w0; w < w1; ++w) local += __popc(bits[w]);
    int32_t incl = local;
    const int lane = tid & 31, warp = tid >> 5;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int32_t t = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += t;
    }
    if (lane == 31) warp_tot[warp] = incl;
    __syncthreads();
    int32_t before = 0;
    for (int i = 0; i < warp; ++i) before += warp_tot[i];
    int32_t run = before + incl - local;
    for (int32_t w = w0; w < w1; ++w) {
        pref[w] = run;
        run += __popc(bits[w]);
    }
    if (tid == kPlanThreads - 1) pref[pl.nw] = before + incl;  // total
    __syncthreads();
    for (int32_t w = tid; w < pl.nw; w += kPlanThreads) {
        pl.bitmap[w] = bits[w];
        pl.prefix[w] = pref[w];
    }
    for (int32_t j = tid; j < Vd; j += kPlanThreads) pl.x_of_j[j] = d2t[j];
    for (int32_t c = tid; c <= (V + kChunkElems - 1) / kChunkElems; c += kPlanThreads) {
        const int32_t x = min(V, c * kChunkElems);
        const int32_t w = x >> 5, b = x & 31;
        pl.chunk[c] = pref[w] + (b ? __popc(bits[w] & ((1u << b) - 1u)) : 0);
    }
    if (tid == 0) {
        pl.prefix[pl.nw] = pref[pl.nw];
        pl.header[0] = V;
        pl.header[1] = Vd;
        pl.header[2] = bad_any;
    }
    for (int32_t j = tid; j < Vd; j += kPlanThreads) {
        const int32_t x = d2t[j];
        if (x < 0 || x >= V) continue;
        const int32_t w = x >> 5, b = x & 31;
        const int32_t pos = pref[w] + (b ? __popc(bits[w] & ((1u << b) - 1u)) : 0);
        if (pos >= 0 && pos < Vd) {
            pl.xs[pos] = x;
            pl.js[pos] = j;
            pl.pairs[pos] = (static_cast<uint32_t>(j) << 16) | static_cast<uint32_t>(x & (kChunkElems - 1));
        }
    }
}

// ---------------------------------------------------------------------------
// row pass
// ---------------------------------------------------------------------------
namespace {

// One chunk of a row: bytes [off, off + nb) of the row, nb multiple of 16.
struct ChunkRef {
    const char* src;
    uint32_t nb;
};

__device__ __forceinline__ void issue_chunk(unsigned char* stage, uint64_t* bar, ChunkRef c, uint64_t pol,
                                            uint32_t& issued)
{
    ++issued;
    mbar_arrive_expect_tx(bar, c.nb);
    bulk_copy_g2s(stage, c.src, c.nb, bar, pol);
}

}  // namespace

template <int DT, int DD>
__global__ void __launch_bounds__(kRowThreads, 1) sample_rows_kernel(SampleArgs A)
{
    extern __shared__ __align__(128) unsigned char smem[];
    uint64_t* full = reinterpret_cast<uint64_t*>(smem);
    unsigned char* ring = smem + kRowHeader;
    constexpr int ET = DT == SV_BF16 ? 2 : 4;
    constexpr int ED = DD == SV_BF16 ? 2 : 4;
    constexpr int VT = 16 / ET;
    constexpr int VD = 16 / ED;
    __shared__ float red_f[kRowThreads / 32];
    __shared__ int32_t red_i[kRowThreads / 32];
    __shared__ uint32_t red_u[kRowThreads / 32];
    __shared__ float zx_shared;
    const int tid = threadIdx.x;

    pdl_launch_dependents();

    // resident buffers of the draft row (Y, draft dtype) and of the target
    // logits at the support positions (G, target dtype)
    char* Y;
    char* G;
    if (A.smem_mode) {
        Y = reinterpret_cast<char*>(ring + kStages * kStageBytes);
        G = Y + align256(static_cast<int64_t>(A.Vd) * ED);
    } else {
        Y = A.gslots + static_cast<int64_t>(blockIdx.x) * A.gslot_bytes;
        G = Y + align256(static_cast<int64_t>(A.Vd) * ED);
    }

    if (tid == 0) {
        for (int s = 0; s < kStages; ++s) mbar_init(&full[s], 1);
        fence_barrier_init();
    }
    __syncthreads();
    const uint64_t pol = l2_policy_evict_first();
    uint32_t gchunk = 0;   // chunks consumed by this CTA so far (stage / parity)
    uint32_t gissued = 0;  // chunks issued (thread 0 only)
    bool plan_ready = A.identity != 0;
    uint32_t timeout = 0;

    const int64_t units = static_cast<int64_t>(A.R) * (A.k + 1);
    for (int64_t unit = blockIdx.x; unit < units; unit += gridDim.x) {
        const int32_t r = static_cast<int32_t>(unit / (A.k + 1));
        const int32_t j = static_cast<int32_t>(unit - static_cast<int64_t>(r) * (A.k + 1));
        const float T = A.temp[r];
        const bool sampling = T > 0.f;
        const bool has_draft = sampling && j < A.k;
        const float c = sampling ? kLog2e / T : 0.f;
        const char* trow = A.tbase + unit * A.tstride;
        const char* drow = has_draft ? A.dbase + (static_cast<int64_t>(r) * A.k + j) * A.dstride : nullptr;
        const int32_t xj = has_draft ? A.draft[static_cast<int64_t>(r) * A.k + j] : -1;

        if (j == 0 && tid == 0) {
            A.race[r].best = ~0ull;
            A.race[r].count = 0u;
        }
        // chunk list: draft bulk chunks, then target bulk chunks
        const uint32_t dbulk = has_draft && A.dbulk ? (static_cast<uint32_t>(A.Vd) * ED) & ~15u : 0u;
        const uint32_t tbulk = A.tbulk ? (static_cast<uint32_t>(A.V) * ET) & ~15u : 0u;
        const uint32_t nd = (dbulk + kStageBytes - 1) / kStageBytes;
        const uint32_t nt = (tbulk + kStageBytes - 1) / kStageBytes;
        const uint32_t nchunks = nd + nt;
        auto chunk_ref = [&](uint32_t i) -> ChunkRef {
            if (i < nd) return ChunkRef{drow + i * kStageBytes, min(kStageBytes, dbulk - i * kStageBytes)};
            const uint32_t t = i - nd;
            return ChunkRef{trow + t * kStageBytes, min(kStageBytes, tbulk - t * kStageBytes)};
        };
        if (tid == 0) zx_shared = NAN;
        __syncthreads();  // every thread is done with the ring of the previous unit
        if (tid == 0) {
            for (uint32_t i = 0; i < nchunks && i < kStages; ++i)
                issue_chunk(ring + ((gchunk + i) % kStages) * kStageBytes, &full[(gchunk + i) % kStages],
                            chunk_ref(i), pol, gissued);
        }

        Lse dl{-INFINITY, 0.f};
        uint32_t dflags = 0;
        // ---- draft row: max / sum-exp, copy into Y --------------------------
        if (has_draft) {
            for (uint32_t i = 0; i < nd; ++i) {
                const uint32_t g = gchunk + i, s = g % kStages;
                if (!timeout && !mbar_wait_bounded(&full[s], (g / kStages) & 1u)) timeout = 1;
                const ChunkRef cr = chunk_ref(i);
                const uint4* vp = reinterpret_cast<const uint4*>(ring + s * kStageBytes);
                const int nv = static_cast<int>(cr.nb / 16);
                const int32_t e0 = static_cast<int32_t>(i * kStageBytes / ED);
                for (int v = tid; v < nv; v += kRowThreads) {
                    const uint4 q = vp[v];
                    *reinterpret_cast<uint4*>(Y + (static_cast<int64_t>(e0) + v * VD) * ED) = q;
                    float f[8];
                    const int n = unpack_vec<DD>(q, f);
                    float mx = -INFINITY;
                    for (int e = 0; e < n; ++e) {
                        if (f[e] != f[e]) {
                            dflags |= kFlagNaN;
                            f[e] = -INFINITY;
                        }
                        if (f[e] == INFINITY) dflags |= kFlagPosInf;
                        mx = fmaxf(mx, f[e]);
                    }
                    const float mt = mx * c;
                    if (mt > -INFINITY) {
                        if (mt > dl.m) {
                            dl.s = dl.m == -INFINITY ? 0.f : dl.s * exp2f(dl.m - mt);
                            dl.m = mt;
                        }
                        float acc = 0.f;
                        for (int e = 0; e < n; ++e) acc += exp2f(fmaf(f[e], c, -dl.m));
                        dl.s += acc;
                    }
                }
                __syncthreads();
                if (tid == 0 && i + kStages < nchunks) {
                    const uint32_t g2 = gchunk + i + kStages;
                    issue_chunk(ring + (g2 % kStages) * kStageBytes, &full[g2 % kStages], chunk_ref(i + kStages), pol, gissued);
                }
            }
            // unaligned draft rows, or the sub-16-byte tail
            for (int32_t e = static_cast<int32_t>(dbulk / ED) + tid; e < A.Vd; e += kRowThreads) {
                float f = ld_elem<DD>(drow, e);
                st_elem<DD>(Y, e, f);
                if (f != f) {
                    dflags |= kFlagNaN;
                    f = -INFINITY;
                }
                if (f == INFINITY) dflags |= kFlagPosInf;
                const float t = f * c;
                if (t > -INFINITY) {
                    if (t > dl.m) {
                        dl.s = dl.m == -INFINITY ? 0.f : dl.s * exp2f(dl.m - t);
                        dl.m = t;
                    }
                    dl.s += exp2f(t - dl.m);
                }
            }
        }

        // ---- target row -------------------------------------------------
        if (has_draft && !plan_ready) {
            pdl_wait_primary();  // the d2t plan is complete
            plan_ready = true;
        }
        Lse3 tl{-INFINITY, 0.f, 0.f};
        const bool track_off = has_draft && !A.identity;
        float bv = -INFINITY;  // argmax: value and the first index of its vector
        int32_t bx = INT32_MAX;
        uint32_t tflags = 0;
        for (uint32_t i = nd; i < nchunks; ++i) {
            const uint32_t g = gchunk + i, s = g % kStages;
            if (!timeout && !mbar_wait_bounded(&full[s], (g / kStages) & 1u)) timeout = 1;
            const ChunkRef cr = chunk_ref(i);
            const unsigned char* st = ring + s * kStageBytes;
            const uint4* vp = reinterpret_cast<const uint4*>(st);
            const int nv = static_cast<int>(cr.nb / 16);
            const int32_t x0 = static_cast<int32_t>((i - nd) * kStageBytes / ET);
            for (int v = tid; v < nv; v += kRowThreads) {
                float f[8];
                const int n = unpack_vec<DT>(vp[v], f);
                float mx = -INFINITY;
                for (int e = 0; e < n; ++e) {
                    if (f[e] != f[e]) {
                        tflags |= kFlagNaN;
                        f[e] = -INFINITY;
                    }
                    mx = fmaxf(mx, f[e]);
                }
                const bool up = mx > bv;
                bv = up ? mx : bv;
                bx = up ? x0 + v * VT : bx;
                if (sampling) {
                    const float mt = mx * c;
                    if (mt > -INFINITY) {
                        if (mt > tl.m) {
                            const float sc = tl.m == -INFINITY ? 0.f : exp2f(tl.m - mt);
                            tl.s *= sc;
                            tl.so *= sc;
                            tl.m = mt;
                        }
                        float acc = 0.f, acc_off = 0.f;
                        if (track_off) {
                            // support bits of the n ids of this vector (n divides 32)
                            const int32_t x = x0 + v * VT;
                            const uint32_t bits = A.plan.bitmap[x >> 5] >> (x & 31);
                            for (int e = 0; e < n; ++e) {
                                const float ex = exp2f(fmaf(f[e], c, -tl.m));
                                acc += ex;
                                acc_off += ((bits >> e) & 1u) ? 0.f : ex;
                            }
                        } else {
                            for (int e = 0; e < n; ++e) acc += exp2f(fmaf(f[e], c, -tl.m));
                        }
                        tl.s += acc;
                        tl.so += acc_off;
                    }
                }
            }
            const int32_t ne = static_cast<int32_t>(cr.nb / ET);
            if (has_draft) {
                // the support positions inside this chunk, in ascending order
                if (A.identity) {
                    for (int32_t e = tid; e < ne; e += kRowThreads) {
                        if constexpr (DT == SV_BF16)
                            reinterpret_cast<uint16_t*>(G)[x0 + e] = reinterpret_cast<const uint16_t*>(st)[e];
                        else
                            reinterpret_cast<float*>(G)[x0 + e] = reinterpret_cast<const float*>(st)[e];
                    }
                } else {
                    const int32_t p0 = support_rank(A.plan, x0), p1 = support_rank(A.plan, x0 + ne);
                    for (int32_t p = p0 + tid; p < p1; p += kRowThreads) {
                        const int32_t le = A.plan.xs[p] - x0;
                        if (le >= 0 && le < ne) {
                            if constexpr (DT == SV_BF16)
                                reinterpret_cast<uint16_t*>(G)[p] = reinterpret_cast<const uint16_t*>(st)[le];
                            else
                                reinterpret_cast<float*>(G)[p] = reinterpret_cast<const float*>(st)[le];
                        }
                    }
                }
                if (xj >= x0 && xj < x0 + ne && tid == 0)
                    zx_shared = ld_elem<DT>(reinterpret_cast<const char*>(st), xj - x0);
            }
            __syncthreads();
            if (tid == 0 && i + kStages < nchunks) {
                const uint32_t g2 = gchunk + i + kStages;
                issue_chunk(ring + (g2 % kStages) * kStageBytes, &full[g2 % kStages], chunk_ref(i + kStages), pol, gissued);
            }
        }
        gchunk += nchunks;
        // unaligned target rows, or the sub-16-byte tail
        const int32_t tb0 = static_cast<int32_t>(tbulk / ET);
        for (int32_t e = tb0 + tid; e < A.V; e += kRowThreads) {
            float f = ld_elem<DT>(trow, e);
            if (f != f) {
                tflags |= kFlagNaN;
                f = -INFINITY;
            }
            if (f > bv) {
                bv = f;
                bx = e;
            }
            if (sampling) {
                const float t = f * c;
                if (t > -INFINITY) {
                    if (t > tl.m) {
                        const float sc = tl.m == -INFINITY ? 0.f : exp2f(tl.m - t);
                        tl.s *= sc;
                        tl.so *= sc;
                        tl.m = t;
                    }
                    const float ex = exp2f(fmaf(f, c, -tl.m));
                    tl.s += ex;
                    if (track_off && !in_support(A.plan, e)) tl.so += ex;
                }
            }
            if (has_draft) {
                if (A.identity) {
                    st_elem<DT>(G, e, f);
                } else if (in_support(A.plan, e)) {
                    st_elem<DT>(G, support_rank(A.plan, e), f);
                }
                if (e == xj) zx_shared = f;
            }
        }

        // ---- reductions ---------------------------------------------------
        block_argmax<kRowThreads>(bv, bx, red_f, red_i);
        const uint32_t fl_t = block_or<kRowThreads>(tflags, red_u);
        const uint32_t fl_d = block_or<kRowThreads>(dflags, red_u);
        int32_t amax = 0;
        if (bx != INT32_MAX) {
            amax = bx;
            // first element equal to the maximum inside the winning vector
            for (int e = 0; e < VT; ++e) {
                const int32_t x = bx + e;
                if (x >= A.V) break;
                if (ld_elem<DT>(trow, x) == bv) {
                    amax = x;
                    break;
                }
            }
        }
        Lse T2{-INFINITY, 0.f}, D2{-INFINITY, 0.f};
        float s_off = 0.f;  // target mass outside the d2t support, unnormalised
        if (sampling) {
            const float M = block_max<kRowThreads>(tl.m, red_f);
            const float sc = (tl.m == -INFINITY || M == -INFINITY) ? 0.f : exp2f(tl.m - M);
            T2 = Lse{M, block_sum<kRowThreads>(tl.s * sc, red_f)};
            if (track_off) s_off = block_sum<kRowThreads>(tl.so * sc, red_f);
        }
        if (has_draft) {
            const float M = block_max<kRowThreads>(dl.m, red_f);
            const float part = dl.m == -INFINITY ? 0.f : dl.s * exp2f(dl.m - M);
            D2 = Lse{M, block_sum<kRowThreads>(M == -INFINITY ? 0.f : part, red_f)};
        }
        uint32_t flags = 0;
        if (fl_t & kFlagNaN) flags |= kFlagNaN;
        if (bv == INFINITY) flags |= kFlagPosInf;
        if (bv == -INFINITY) flags |= kFlagAllNegInf;
        if (has_draft && ((fl_d & (kFlagNaN | kFlagPosInf)) || D2.m == -INFINITY)) flags |= kFlagDraftBad;
        if (timeout) flags |= kFlagTimeout;

        // ---- TV over the full vocabulary, p(x_j), q(x_j), accept -------------
        float tvv = NAN, pj = NAN, qj = NAN;
        int32_t acc = 0;
        if (has_draft) {
            __syncthreads();  // G and Y complete
            const float invS = 1.f / T2.s, invSq = 1.f / D2.s;
            float a_abs = 0.f;
            const int32_t nsup = A.identity ? A.V : A.plan.prefix[A.plan.nw];
            for (int32_t p = tid; p < nsup; p += kRowThreads) {
                const int32_t jd = A.identity ? p : A.plan.js[p];
                if (jd < 0 || jd >= A.Vd) continue;
                float z = ld_elem<DT>(G, p);
                float y = ld_elem<DD>(Y, jd);
                z = z != z ? -INFINITY : z;
                y = y != y ? -INFINITY : y;
                const float pp = exp2f(fmaf(z, c, -T2.m)) * invS;
                const float qq = exp2f(fmaf(y, c, -D2.m)) * invSq;
                a_abs += fabsf(pp - qq);
            }
            a_abs = block_sum<kRowThreads>(a_abs, red_f);
            // TV over the full vocabulary: the support terms plus p's mass off the
            // support, summed directly (1 - sum_support p would cancel)
            tvv = 0.5f * (a_abs + s_off * invS);
            if (tid == 0) {
                const bool in_range = xj >= 0 && xj < A.V;
                float zx = zx_shared;
                zx = zx != zx ? -INFINITY : zx;
                pj = in_range ? exp2f(fmaf(zx, c, -T2.m)) * invS : 0.f;
                qj = 0.f;
                if (in_range && (A.identity || in_support(A.plan, xj))) {
                    const int32_t jd = A.identity ? xj : A.plan.js[support_rank(A.plan, xj)];
                    if (jd >= 0 && jd < A.Vd) {
                        float y = ld_elem<DD>(Y, jd);
                        y = y != y ? -INFINITY : y;
                        qj = exp2f(fmaf(y, c, -D2.m)) * invSq;
                    }
                }
                if (qj > 0.f) {
                    const uint4 w = philox_block(philox_key(A.seeds[r]), 0u, static_cast<uint32_t>(j), kTagAccept);
                    const float u = uniform_from_word(w.x);
                    acc = u < __fdiv_rn(pj, qj) ? 1 : 0;
                } else if (in_range) {
                    flags |= kFlagOffSupport;
                }
            }
        }
        if (tid == 0) {
            RowStat rs;
            rs.m = T2.m;
            rs.s = T2.s;
            rs.mq = D2.m;
            rs.sq = D2.s;
            rs.zx = zx_shared;
            rs.p = pj;
            rs.q = qj;
            rs.amax = amax;
            rs.flags = flags;
            rs.accept = acc;
            rs.rx = -1;
            rs.rv = 0.f;
            rs.bkey = INFINITY;
            rs.bxc = -1;
            A.stats[unit] = rs;
            if (j < A.k) {
                const int64_t o = static_cast<int64_t>(r) * A.k + j;
                if (A.tv) A.tv[o] = tvv;
                if (A.pd) A.pd[o] = pj;
                if (A.qd) A.qd[o] = qj;
            }
        }
    }
    // Completion of this grid must imply completion of the plan kernel, which
    // the race kernel reads after waiting on this grid only.
    if (!plan_ready) pdl_wait_primary();
    if (timeout && tid == 0) {
        // give copies that may still be in flight a bounded chance to land
        for (uint32_t g = gissued > kStages ? gissued - kStages : 0; g < gissued; ++g)
            (void)mbar_wait_bounded(&full[g % kStages], (g / kStages) & 1u);
    }
}

// ---------------------------------------------------------------------------
// row pass, fast path: bf16 target and draft rows, d2t vocabulary <= 32768
// ---------------------------------------------------------------------------
// Every warp streams its own share of a row: chunks of kChunkElems ids,
// chunk c going to warp c % kFastWarps, through a private two-stage ring of
// bulk copies that the warp's lane 0 issues one chunk ahead.  Each stage also
// receives the chunk's support entries as packed (draft id, offset) pairs,
// so the warp scatters the support logits to G[draft id] from shared memory.
// Warps never wait for each other inside a row; only the row's reductions
// and the TV pass (over G and the L2-resident draft row, in draft-id order)
// synchronise the CTA, and each warp has already issued its first chunk of
// the next row before they start.
namespace {

constexpr int kFastWarps = 12;
constexpr int kFastThreads = 32 * kFastWarps;
constexpr uint32_t kFastData = kChunkElems * 2;  // 4 KB of bf16 per stage
constexpr uint32_t kFastPairCap = 512;           // staged support entries per stage
constexpr uint32_t kFastStage = kFastData + kFastPairCap * 4;
constexpr int kFastHeader = 256;
constexpr int32_t kFastMaxVd = 32768;

__device__ __forceinline__ float ex2(float x)
{
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// two fp32 values in one 64-bit register, for the packed f32x2 instructions
__device__ __forceinline__ unsigned long long pack2(float lo, float hi)
{
    unsigned long long r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
    return r;
}
__device__ __forceinline__ void unpack2(unsigned long long v, float& lo, float& hi)
{
    asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
__device__ __forceinline__ unsigned long long fma2(unsigned long long a, unsigned long long b, unsigned long long c)
{
    unsigned long long r;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(a), "l"(b), "l"(c));
    return r;
}
__device__ __forceinline__ unsigned long long add2(unsigned long long a, unsigned long long b)
{
    unsigned long long r;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
    return r;
}

// the bf16x2 word w as two fp32 values (exact) in one 64-bit register
__device__ __forceinline__ unsigned long long bf16x2_to_f32x2(uint32_t w)
{
    return pack2(bf16_lo(w), bf16_hi(w));
}

// sum over the 8 bf16 values z of a vector of 2^(z c - m): packed fp32x2
// arguments, eight independent MUFU operations, a tree of packed adds
__device__ __forceinline__ float exp_sum8(uint4 q, unsigned long long c2, unsigned long long nm2)
{
    const unsigned long long t0 = fma2(bf16x2_to_f32x2(q.x), c2, nm2);
    const unsigned long long t1 = fma2(bf16x2_to_f32x2(q.y), c2, nm2);
    const unsigned long long t2 = fma2(bf16x2_to_f32x2(q.z), c2, nm2);
    const unsigned long long t3 = fma2(bf16x2_to_f32x2(q.w), c2, nm2);
    float a0, a1, a2, a3, a4, a5, a6, a7;
    unpack2(t0, a0, a1);
    unpack2(t1, a2, a3);
    unpack2(t2, a4, a5);
    unpack2(t3, a6, a7);
    const unsigned long long e0 = pack2(ex2(a0), ex2(a1)), e1 = pack2(ex2(a2), ex2(a3));
    const unsigned long long e2 = pack2(ex2(a4), ex2(a5)), e3 = pack2(ex2(a6), ex2(a7));
    float lo, hi;
    unpack2(add2(add2(e0, e1), add2(e2, e3)), lo, hi);
    return lo + hi;
}

// 16-byte read-only global load
__device__ __forceinline__ uint4 ld_nc_v4(const uint4* p)
{
    uint4 v;
    asm volatile("ld.global.nc.v4.u32 {%0, %1, %2, %3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(p));
    return v;
}

// order this thread's generic-proxy accesses to shared memory before later
// bulk copies (async proxy) into the same bytes
__device__ __forceinline__ void fence_proxy_async_smem()
{
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// replace NaN halves of a bf16x2 word by -inf
__device__ __forceinline__ uint32_t bf16x2_nan_to_ninf(uint32_t w)
{
    uint32_t lo = w & 0xFFFFu, hi = w >> 16;
    if ((lo & 0x7FFFu) > 0x7F80u) lo = 0xFF80u;
    if ((hi & 0x7FFFu) > 0x7F80u) hi = 0xFF80u;
    return lo | (hi << 16);
}

struct WarpRec {
    float bv;
    int32_t bx;
    uint32_t tfl, dfl;
    float tm, dm;
};

struct FastUnit {
    int32_t r, j;
    bool sampling, has_draft;
    const char* trow;
    const char* drow;
    int32_t nd, nt;  // draft / target chunks of the row
};

__device__ __forceinline__ FastUnit fast_unit(const SampleArgs& A, int64_t unit)
{
    FastUnit u;
    u.r = static_cast<int32_t>(unit / (A.k + 1));
    u.j = static_cast<int32_t>(unit - static_cast<int64_t>(u.r) * (A.k + 1));
    const float T = A.temp[u.r];
    u.sampling = T > 0.f;
    u.has_draft = u.sampling && u.j < A.k;
    u.trow = A.tbase + unit * A.tstride;
    u.drow = u.has_draft ? A.dbase + (static_cast<int64_t>(u.r) * A.k + u.j) * A.dstride : nullptr;
    u.nd = u.has_draft ? (A.Vd + kChunkElems - 1) / kChunkElems : 0;
    u.nt = (A.V + kChunkElems - 1) / kChunkElems;
    return u;
}

// chunks of warp w in a row: draft chunks w, w + W, ... then target chunks w, w + W, ...
__device__ __forceinline__ int32_t warp_chunks(int32_t n, int w)
{
    return n > w ? (n - w + kFastWarps - 1) / kFastWarps : 0;
}

// issue the i-th chunk of warp w of unit u into `stage` (lane 0 only)
__device__ __forceinline__ void issue_warp_chunk(const SampleArgs& A, const FastUnit& u, int w, int32_t i,
                                                 unsigned char* stage, uint64_t* bar, uint64_t pol_t,
                                                 uint64_t pol_d, bool plan_ok)
{
    const int32_t ndw = warp_chunks(u.nd, w);
    if (i < ndw) {
        const int32_t c = w + i * kFastWarps;
        const uint32_t off = static_cast<uint32_t>(c) * kFastData;
        const uint32_t nb = min(kFastData, static_cast<uint32_t>(A.Vd) * 2 - off);
        mbar_arrive_expect_tx(bar, nb);
        bulk_copy_g2s(stage, u.drow + off, nb, bar, pol_d);
        return;
    }
    const int32_t c = w + (i - ndw) * kFastWarps;
    const uint32_t off = static_cast<uint32_t>(c) * kFastData;
    const uint32_t nb = min(kFastData, static_cast<uint32_t>(A.V) * 2 - off);
    uint32_t pb = 0;
    int32_t p0a = 0;
    if (u.has_draft && plan_ok) {
        const int32_t p0 = A.plan.chunk[c], p1 = A.plan.chunk[c + 1];
        p0a = p0 & ~3;
        if (p1 > p0) pb = min(kFastPairCap * 4, static_cast<uint32_t>((p1 - p0a) * 4 + 15) & ~15u);
    }
    mbar_arrive_expect_tx(bar, nb + pb);
    bulk_copy_g2s(stage, u.trow + off, nb, bar, pol_t);
    if (pb) bulk_copy_g2s(stage + kFastData, A.plan.pairs + p0a, pb, bar, pol_d);
}

}  // namespace

__global__ void __launch_bounds__(kFastThreads, 1) sample_rows_fast_kernel(SampleArgs A)
{
    extern __shared__ __align__(128) unsigned char smem[];
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem);  // [warp][2]
    unsigned char* ring = smem + kFastHeader;
    uint16_t* G = reinterpret_cast<uint16_t*>(ring + kFastWarps * 2 * kFastStage);
    __shared__ float zx_shared;
    __shared__ int32_t rx_shared;
    __shared__ float rv_shared;
    __shared__ WarpRec wrec[kFastWarps];
    __shared__ float wsum[kFastWarps][2];
    __shared__ float wtv[kFastWarps], wrv[kFastWarps];
    __shared__ int32_t wrj[kFastWarps];
    __shared__ int32_t amax_shared;
    const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;

    pdl_wait_primary();  // a plan built in the same call must be complete
    pdl_launch_dependents();
    if (tid == 0) {
        for (int i = 0; i < 2 * kFastWarps; ++i) mbar_init(&bars[i], 1);
        fence_barrier_init();
    }
    __syncthreads();
    // a plan for other sizes, or built from a d2t with repeated / out-of-range ids, is not
    // trusted for shared-memory indexing (the race kernel reports SV_ST_BAD_D2T)
    const bool plan_ok = A.plan.header[0] == A.V && A.plan.header[1] == A.Vd && A.plan.header[2] == 0;
    const uint64_t pol_t = l2_policy_evict_first();
    uint64_t pol_d;
    asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(pol_d));
    unsigned char* wst = ring + w * 2 * kFastStage;  // this warp's two stages
    uint64_t* wbar = bars + 2 * w;
    uint32_t gi = 0;  // chunks this warp has consumed so far (stage = gi & 1)
    uint32_t timeout = 0;
    bool prefetched = false;

    const int64_t units = static_cast<int64_t>(A.R) * (A.k + 1);
    for (int64_t unit = blockIdx.x; unit < units; unit += gridDim.x) {
        const FastUnit u = fast_unit(A, unit);
        const float T = A.temp[u.r];
        const float c = u.sampling ? kLog2e / T : 0.f;
        const unsigned long long c2 = pack2(c, c);
        const int32_t xj = u.has_draft ? A.draft[static_cast<int64_t>(u.r) * A.k + u.j] : -1;
        const int32_t ndw = warp_chunks(u.nd, w), ntw = warp_chunks(u.nt, w);
        const int32_t nw_chunks = ndw + ntw;
        if (u.j == 0 && tid == 0) {
            A.race[u.r].best = ~0ull;
            A.race[u.r].count = 0u;
        }
        if (tid == 0) zx_shared = NAN;
        __syncthreads();  // G, zx and the exchange arrays of the previous row are no longer read
        if (lane == 0 && !prefetched && nw_chunks > 0)
            issue_warp_chunk(A, u, w, 0, wst + (gi & 1) * kFastStage, &wbar[gi & 1], pol_t, pol_d, plan_ok);

        float dm = -INFINITY, ds = 0.f, tm = -INFINITY, ts = 0.f, bv = -INFINITY;
        int32_t bx = INT32_MAX;
        uint32_t dflags = 0, tflags = 0;
        for (int32_t i = 0; i < nw_chunks; ++i, ++gi) {
            const uint32_t s = gi & 1;
            if (lane == 0 && i + 1 < nw_chunks) {
                fence_proxy_async_smem();
                issue_warp_chunk(A, u, w, i + 1, wst + (s ^ 1) * kFastStage, &wbar[s ^ 1], pol_t, pol_d, plan_ok);
            }
            if (!timeout && !mbar_wait_bounded(&wbar[s], (gi >> 1) & 1u)) timeout = 1;
            const unsigned char* st = wst + s * kFastStage;
            const uint4* vp = reinterpret_cast<const uint4*>(st);
            const bool is_draft = i < ndw;
            const int32_t cidx = w + (is_draft ? i : i - ndw) * kFastWarps;
            const uint32_t off = static_cast<uint32_t>(cidx) * kFastData;
            const uint32_t nb = min(kFastData, static_cast<uint32_t>(is_draft ? A.Vd : A.V) * 2 - off);
            const int nv = static_cast<int>(nb / 16);
            const int32_t x0 = static_cast<int32_t>(off / 2);
            // all 8 vectors of this lane first (independent loads and max trees), one update of
            // the running max, then 64 independent exps
            constexpr int kVL = kChunkElems / 8 / 32;  // vectors per lane per chunk
            uint4 q[kVL];
            float vmx[kVL];
            bool nan_seen = false;
#pragma unroll
            for (int e = 0; e < kVL; ++e) {
                const int v = lane + 32 * e;
                q[e] = v < nv ? vp[v] : make_uint4(0xFF80FF80u, 0xFF80FF80u, 0xFF80FF80u, 0xFF80FF80u);
                const uint32_t m2 = bmax2_nan(bmax2_nan(q[e].x, q[e].y), bmax2_nan(q[e].z, q[e].w));
                vmx[e] = fmax_nan(bf16_lo(m2), bf16_hi(m2));
                nan_seen |= vmx[e] != vmx[e];
            }
            if (nan_seen) {  // rare: NaN logits read as -inf
                (is_draft ? dflags : tflags) |= kFlagNaN;
#pragma unroll
                for (int e = 0; e < kVL; ++e) {
                    q[e] = make_uint4(bf16x2_nan_to_ninf(q[e].x), bf16x2_nan_to_ninf(q[e].y),
                                      bf16x2_nan_to_ninf(q[e].z), bf16x2_nan_to_ninf(q[e].w));
                    const uint32_t m3 = bmax2_nan(bmax2_nan(q[e].x, q[e].y), bmax2_nan(q[e].z, q[e].w));
                    vmx[e] = fmaxf(bf16_lo(m3), bf16_hi(m3));
                }
            }
            float lm = vmx[0];
#pragma unroll
            for (int e = 1; e < kVL; ++e) lm = fmaxf(lm, vmx[e]);
            if (!is_draft) {
#pragma unroll
                for (int e = 0; e < kVL; ++e) {  // ascending vector starts: strict > keeps the first
                    const bool up = vmx[e] > bv;
                    bv = up ? vmx[e] : bv;
                    bx = up ? x0 + (lane + 32 * e) * 8 : bx;
                }
            } else if (lm == INFINITY) {
                dflags |= kFlagPosInf;
            }
            if (is_draft || u.sampling) {
                float& rm = is_draft ? dm : tm;
                float& rs_ = is_draft ? ds : ts;
                const float mt = lm * c;
                if (mt > rm) {
                    rs_ = rm == -INFINITY ? 0.f : rs_ * ex2(rm - mt);
                    rm = mt;
                }
                if (rm > -INFINITY) {
                    const unsigned long long nm2 = pack2(-rm, -rm);
                    float acc8[kVL];
#pragma unroll
                    for (int e = 0; e < kVL; ++e) acc8[e] = exp_sum8(q[e], c2, nm2);
#pragma unroll
                    for (int e = 1; e < kVL; ++e) acc8[0] += acc8[e];
                    rs_ += acc8[0];
                }
            }
            if (!is_draft && u.has_draft) {
                // support entries of this chunk: G[draft id] = z at the chunk offset
                const uint16_t* zs = reinterpret_cast<const uint16_t*>(st);
                const uint32_t* pr = reinterpret_cast<const uint32_t*>(st + kFastData);
                const int32_t p0 = plan_ok ? A.plan.chunk[cidx] : 0;
                const int32_t cnt = plan_ok ? A.plan.chunk[cidx + 1] - p0 : 0;
                const int32_t base = p0 & 3;
                const int32_t staged = min(cnt, static_cast<int32_t>(kFastPairCap) - base);
#pragma unroll 4
                for (int32_t e = lane; e < staged; e += 32) {
                    const uint32_t pe = pr[base + e];
                    G[pe >> 16] = zs[pe & (kChunkElems - 1)];
                }
                for (int32_t e = max(staged, 0) + lane; e < cnt; e += 32) {  // beyond the staged entries
                    const uint32_t pe = A.plan.pairs[p0 + e];
                    G[pe >> 16] = zs[pe & (kChunkElems - 1)];
                }
                if (lane == 0 && xj >= x0 && xj < x0 + static_cast<int32_t>(nb / 2))
                    zx_shared = __uint_as_float(static_cast<uint32_t>(zs[xj - x0]) << 16);
            }
            __syncwarp();
        }
        // first chunk of this warp's next row, in flight during the reductions below
        prefetched = false;
        if (unit + gridDim.x < units) {
            const FastUnit un = fast_unit(A, unit + gridDim.x);
            if (warp_chunks(un.nd, w) + warp_chunks(un.nt, w) > 0) {
                if (lane == 0) {
                    fence_proxy_async_smem();
                    issue_warp_chunk(A, un, w, 0, wst + (gi & 1) * kFastStage, &wbar[gi & 1], pol_t, pol_d, plan_ok);
                }
                prefetched = true;
            }
        }

        // ---- reductions: two exchanges through shared memory ----
        const float my_bv = bv, my_tm = tm, my_ts = ts, my_dm = dm, my_ds = ds;
        const int32_t my_bx = bx;
        uint32_t tfl = tflags | (timeout ? kFlagTimeout : 0u);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
            const int32_t ox = __shfl_xor_sync(0xffffffffu, bx, o);
            if (ov > bv || (ov == bv && ox < bx)) {
                bv = ov;
                bx = ox;
            }
            tm = fmaxf(tm, __shfl_xor_sync(0xffffffffu, tm, o));
            dm = fmaxf(dm, __shfl_xor_sync(0xffffffffu, dm, o));
        }
        tfl = __reduce_or_sync(0xffffffffu, tfl);
        dflags = __reduce_or_sync(0xffffffffu, dflags);
        if (lane == 0) wrec[w] = WarpRec{bv, bx, tfl, dflags, tm, dm};
        __syncthreads();
        float BV = wrec[0].bv, M = wrec[0].tm, Mq = wrec[0].dm;
        int32_t BX = wrec[0].bx;
        uint32_t FLT = wrec[0].tfl, FLD = wrec[0].dfl;
        for (int i = 1; i < kFastWarps; ++i) {
            const WarpRec rec = wrec[i];
            if (rec.bv > BV || (rec.bv == BV && rec.bx < BX)) {
                BV = rec.bv;
                BX = rec.bx;
            }
            M = fmaxf(M, rec.tm);
            Mq = fmaxf(Mq, rec.dm);
            FLT |= rec.tfl;
            FLD |= rec.dfl;
        }
        // the thread that saw the winning vector finds the first equal element in it
        if (my_bx == BX && my_bv == BV && BX != INT32_MAX) {
            int32_t idx = BX;
            for (int e = 0; e < 8; ++e) {
                const int32_t x = BX + e;
                if (x >= A.V) break;
                if (ld_elem<SV_BF16>(u.trow, x) == BV) {
                    idx = x;
                    break;
                }
            }
            amax_shared = idx;
        }
        if (tid == 0 && BX == INT32_MAX) amax_shared = 0;
        float S = 0.f, Sq = 0.f;
        {
            float part_t = 0.f, part_d = 0.f;
            if (u.sampling && my_tm > -INFINITY && M > -INFINITY) part_t = my_ts * ex2(my_tm - M);
            if (u.has_draft && my_dm > -INFINITY && Mq > -INFINITY) part_d = my_ds * ex2(my_dm - Mq);
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) {
                part_t += __shfl_xor_sync(0xffffffffu, part_t, o);
                part_d += __shfl_xor_sync(0xffffffffu, part_d, o);
            }
            if (lane == 0) {
                wsum[w][0] = part_t;
                wsum[w][1] = part_d;
            }
            __syncthreads();
            for (int i = 0; i < kFastWarps; ++i) {
                S += wsum[i][0];
                Sq += wsum[i][1];
            }
        }
        if (!u.sampling) M = -INFINITY;
        if (!u.has_draft) Mq = -INFINITY;
        uint32_t flags = 0;
        if (FLT & kFlagNaN) flags |= kFlagNaN;
        if (FLT & kFlagTimeout) flags |= kFlagTimeout;
        if (BV == INFINITY) flags |= kFlagPosInf;
        if (BV == -INFINITY) flags |= kFlagAllNegInf;
        if (u.has_draft && ((FLD & (kFlagNaN | kFlagPosInf)) || Mq == -INFINITY)) flags |= kFlagDraftBad;

        // ---- TV = sum over the support of max(0, q - p); p(x_j), q(x_j), accept ----
        float tvv = NAN, pj = NAN, qj = NAN;
        int32_t acc = 0;
        if (u.has_draft) {
            const float invS = 1.f / S, invSq = 1.f / Sq;
            float a = 0.f;
            float rbest = 0.f;  // largest residual p - q seen and its draft id
            int32_t rj = -1;
            const int32_t nv8 = A.Vd / 8;
            const uint4* yv = reinterpret_cast<const uint4*>(u.drow);
            const uint4* gv = reinterpret_cast<const uint4*>(G);
            for (int32_t v = tid; v < nv8; v += kFastThreads) {
                const uint4 gq = gv[v];
                const uint4 yq = ld_nc_v4(yv + v);
                const uint32_t gw[4] = {gq.x, gq.y, gq.z, gq.w};
                const uint32_t yw[4] = {yq.x, yq.y, yq.z, yq.w};
                float d[8];
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    d[2 * e] = ex2(fmaf(bf16_lo(yw[e]), c, -Mq)) * invSq - ex2(fmaf(bf16_lo(gw[e]), c, -M)) * invS;
                    d[2 * e + 1] = ex2(fmaf(bf16_hi(yw[e]), c, -Mq)) * invSq - ex2(fmaf(bf16_hi(gw[e]), c, -M)) * invS;
                }
                // d = q - p: TV sums its positive part; the most negative d is the largest residual p - q
                float dmin = d[0];
                int emin = 0;
#pragma unroll
                for (int e = 1; e < 8; ++e) {
                    const bool lt = d[e] < dmin;
                    dmin = lt ? d[e] : dmin;
                    emin = lt ? e : emin;
                }
                if (-dmin > rbest) {
                    rbest = -dmin;
                    rj = v * 8 + emin;
                }
                a += ((fmaxf(d[0], 0.f) + fmaxf(d[1], 0.f)) + (fmaxf(d[2], 0.f) + fmaxf(d[3], 0.f))) +
                     ((fmaxf(d[4], 0.f) + fmaxf(d[5], 0.f)) + (fmaxf(d[6], 0.f) + fmaxf(d[7], 0.f)));
            }
            for (int32_t jd = nv8 * 8 + tid; jd < A.Vd; jd += kFastThreads) {
                const float pp = ex2(fmaf(__uint_as_float(static_cast<uint32_t>(G[jd]) << 16), c, -M)) * invS;
                const float qq = ex2(fmaf(ld_elem<SV_BF16>(u.drow, jd), c, -Mq)) * invSq;
                a += fmaxf(qq - pp, 0.f);
            }
            // one exchange: the TV sum and the largest support residual
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) {
                a += __shfl_xor_sync(0xffffffffu, a, o);
                const float ov = __shfl_xor_sync(0xffffffffu, rbest, o);
                const int32_t oj = __shfl_xor_sync(0xffffffffu, rj, o);
                if (ov > rbest || (ov == rbest && oj < rj)) {
                    rbest = ov;
                    rj = oj;
                }
            }
            if (lane == 0) {
                wtv[w] = a;
                wrv[w] = rbest;
                wrj[w] = rj;
            }
            __syncthreads();
            if (tid == 0) {
                tvv = 0.f;
                float nrv = 0.f;
                int32_t nrj = -1;
                for (int i = 0; i < kFastWarps; ++i) {
                    tvv += wtv[i];
                    if (wrv[i] > nrv || (wrv[i] == nrv && wrj[i] < nrj)) {
                        nrv = wrv[i];
                        nrj = wrj[i];
                    }
                }
                rx_shared = (plan_ok && nrj >= 0 && nrj < A.Vd && nrv > 0.f) ? A.plan.x_of_j[nrj] : -1;
                rv_shared = nrv;
                const bool in_range = xj >= 0 && xj < A.V;
                float zx = zx_shared;
                zx = zx != zx ? -INFINITY : zx;
                pj = in_range ? ex2(fmaf(zx, c, -M)) * invS : 0.f;
                qj = 0.f;
                if (in_range && in_support(A.plan, xj)) {
                    const int32_t jd = A.plan.js[support_rank(A.plan, xj)];
                    if (jd >= 0 && jd < A.Vd) {
                        float y = ld_elem<SV_BF16>(u.drow, jd);
                        y = y != y ? -INFINITY : y;
                        qj = ex2(fmaf(y, c, -Mq)) * invSq;
                    }
                }
                if (qj > 0.f) {
                    const uint4 w4 = philox_block(philox_key(A.seeds[u.r]), 0u, static_cast<uint32_t>(u.j), kTagAccept);
                    acc = uniform_from_word(w4.x) < __fdiv_rn(pj, qj) ? 1 : 0;
                } else if (in_range) {
                    flags |= kFlagOffSupport;
                }
            }
        } else {
            __syncthreads();  // amax_shared is visible to thread 0
        }
        if (tid == 0) {
            const int32_t amax = amax_shared;
            RowStat rs;
            rs.m = M;
            rs.s = S;
            rs.mq = Mq;
            rs.sq = Sq;
            rs.zx = zx_shared;
            rs.p = pj;
            rs.q = qj;
            rs.amax = amax;
            rs.flags = flags;
            rs.accept = acc;
            rs.rx = u.has_draft ? rx_shared : -1;
            rs.rv = u.has_draft ? rv_shared : 0.f;
            // a bound for the race on this row, should it be the selected one: the key of
            // the argmax, and for a residual race also of the largest support residual
            rs.bkey = INFINITY;
            rs.bxc = -1;
            if (u.sampling && !(flags & (kFlagNaN | kFlagPosInf | kFlagAllNegInf | kFlagDraftBad)) && S > 0.f) {
                const PhiloxKey key = philox_key(A.seeds[u.r]);
                const bool residual = u.j < A.k;
                const uint32_t tag = residual ? kTagResidual : kTagBonus;
                auto key_of = [&](int32_t x, float wt) -> float {
                    if (!(wt > 0.f)) return INFINITY;
                    const uint4 w4 = philox_block(key, static_cast<uint32_t>(x >> 2), static_cast<uint32_t>(u.j), tag);
                    const uint32_t wd = (x & 3) == 0 ? w4.x : ((x & 3) == 1 ? w4.y : ((x & 3) == 2 ? w4.z : w4.w));
                    return __fdiv_rn(-log1pf(-one_minus_uniform_from_word(wd)), wt);
                };
                float wa = ex2(fmaf(BV, c, -M)) * (1.f / S);
                if (residual && in_support(A.plan, amax)) {
                    const int32_t jd = A.plan.js[support_rank(A.plan, amax)];
                    if (jd >= 0 && jd < A.Vd) {
                        float y = ld_elem<SV_BF16>(u.drow, jd);
                        y = y != y ? -INFINITY : y;
                        wa -= ex2(fmaf(y, c, -Mq)) * (1.f / Sq);
                    }
                }
                rs.bkey = key_of(amax, wa);
                rs.bxc = rs.bkey < INFINITY ? amax : -1;
                if (residual && rs.rx >= 0) {
                    const float kr = key_of(rs.rx, rs.rv);
                    if (kr < rs.bkey) {
                        rs.bkey = kr;
                        rs.bxc = rs.rx;
                    }
                }
            }
            A.stats[unit] = rs;
            if (u.j < A.k) {
                const int64_t o = static_cast<int64_t>(u.r) * A.k + u.j;
                if (A.tv) A.tv[o] = tvv;
                if (A.pd) A.pd[o] = pj;
                if (A.qd) A.qd[o] = qj;
            }
        }
    }
    if (timeout && lane == 0) {
        // give this warp's copies that may still be in flight a bounded chance to land
        (void)mbar_wait_bounded(&wbar[gi & 1], (gi >> 1) & 1u);
        (void)mbar_wait_bounded(&wbar[(gi + 1) & 1], ((gi + 1) >> 1) & 1u);
    }
}

// ---------------------------------------------------------------------------
// scan + race + commit
// ---------------------------------------------------------------------------
namespace {

__device__ __forceinline__ unsigned long long pack_key(float key, int32_t x)
{
    return (static_cast<unsigned long long>(__float_as_uint(key)) << 32) | static_cast<uint32_t>(x);
}

}  // namespace

// E_x = -ln u_x >= -ln(1 - 2^-24) for every uniform of the library, so an
// element whose weight w satisfies best * w below this cannot have a key
// E_x / w_x below `best`.  The constant is taken a little low on purpose.
constexpr float kMinE = 5.9e-8f;

template <int DT>
__device__ __forceinline__ void load4(const char* row, int32_t x, bool vec_ok, float* z)
{
    if constexpr (DT == SV_BF16) {
        if (vec_ok) {
            const uint2 v = *reinterpret_cast<const uint2*>(row + static_cast<int64_t>(x) * 2);
            z[0] = bf16_lo(v.x);
            z[1] = bf16_hi(v.x);
            z[2] = bf16_lo(v.y);
            z[3] = bf16_hi(v.y);
            return;
        }
    } else {
        if (vec_ok) {
            const float4 v = *reinterpret_cast<const float4*>(row + static_cast<int64_t>(x) * 4);
            z[0] = v.x;
            z[1] = v.y;
            z[2] = v.z;
            z[3] = v.w;
            return;
        }
    }
#pragma unroll
    for (int e = 0; e < 4; ++e) z[e] = ld_elem<DT>(row, x + e);
}

// q(x) of the draft row (0 off the support): the residual weight needs it only for the
// few elements whose target weight alone could still win the race
template <int DD>
__device__ __forceinline__ float draft_q(const SampleArgs& A, const char* drow, int32_t x, float c, float mq,
                                         float invSq)
{
    int32_t jd = x;
    if (!A.identity) {
        if (!in_support(A.plan, x)) return 0.f;
        jd = A.plan.js[support_rank(A.plan, x)];
    }
    if (jd < 0 || jd >= A.Vd) return 0.f;
    float y = ld_elem<DD>(drow, jd);
    y = y != y ? -INFINITY : y;
    return ex2(fmaf(y, c, -mq)) * invSq;
}

// the race over row elements [x0, x1): this thread's best (key, x), starting from the
// bound `best`.  w_x = p(x) - q(x) (residual) or p(x) (bonus).  Since E_x >= v_x = 1 - u_x
// and w_x <= p(x), an element with v_x >= best * p(x) cannot win; the row's loads of a
// batch are issued together, Philox runs only for groups some element of which passes
// on p, and q is looked up only for elements that pass on p.
constexpr int kRaceBatch = 8;  // groups of 4 elements per thread in flight
template <int DT, int DD>
__device__ __forceinline__ void race_range(const SampleArgs& A, const char* trow, const char* drow, int32_t x0,
                                           int32_t x1, float c, const RowStat& rs, bool residual, PhiloxKey key,
                                           uint32_t row, uint32_t tag, bool vec_ok, float& best, int32_t& bx)
{
    const int32_t g0 = x0 >> 2, g1 = (x1 + 3) >> 2;
    const float invS = 1.f / rs.s, invSq = residual ? 1.f / rs.sq : 0.f;
    for (int32_t gb = g0 + static_cast<int32_t>(threadIdx.x); gb < g1; gb += kRaceBatch * kRaceThreads) {
        float z[kRaceBatch][4];
#pragma unroll
        for (int i = 0; i < kRaceBatch; ++i) {
            const int32_t g = gb + i * kRaceThreads, xb = 4 * g;
            if (g < g1 && xb >= x0 && xb + 4 <= x1) {
                load4<DT>(trow, xb, vec_ok, z[i]);
            } else {
#pragma unroll
                for (int e = 0; e < 4; ++e)
                    z[i][e] = (g < g1 && xb + e >= x0 && xb + e < x1) ? ld_elem<DT>(trow, xb + e) : -INFINITY;
            }
        }
#pragma unroll
        for (int i = 0; i < kRaceBatch; ++i) {
            const int32_t g = gb + i * kRaceThreads, xb = 4 * g;
            float w[4], wmax = 0.f;
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const float zz = z[i][e] != z[i][e] ? -INFINITY : z[i][e];
                w[e] = ex2(fmaf(zz, c, -rs.m)) * invS;
                wmax = fmaxf(wmax, w[e]);
            }
            if (!(best * wmax >= kMinE)) continue;  // no element of the group can beat `best`
            const uint4 w4 = philox_block(key, static_cast<uint32_t>(g), row, tag);
            const uint32_t words[4] = {w4.x, w4.y, w4.z, w4.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                float wt = w[e];
                if (!(wt > 0.f)) continue;
                const float v = one_minus_uniform_from_word(words[e]);
                if (!(v < best * wt)) continue;  // E >= v and w <= p
                const int32_t x = xb + e;
                if (residual) {
                    wt -= draft_q<DD>(A, drow, x, c, rs.mq, invSq);
                    if (!(wt > 0.f) || !(v < best * wt)) continue;
                }
                const float k2 = __fdiv_rn(-log1pf(-v), wt);
                if (k2 < best || (k2 == best && x < bx)) {
                    best = k2;
                    bx = x;
                }
            }
        }
    }
}

// the race key of one element (or +inf when its weight is not positive)
template <int DT, int DD>
__device__ __forceinline__ float single_key(const SampleArgs& A, const char* trow, const char* drow, int32_t x,
                                            float c, const RowStat& rs, bool residual, PhiloxKey key, uint32_t row,
                                            uint32_t tag)
{
    float z = ld_elem<DT>(trow, x);
    z = z != z ? -INFINITY : z;
    float w = ex2(fmaf(z, c, -rs.m)) * (1.f / rs.s);
    if (residual) {
        int32_t jd = -1;
        if (A.identity) {
            jd = x;
        } else if (in_support(A.plan, x)) {
            jd = A.plan.js[support_rank(A.plan, x)];
        }
        if (jd >= 0 && jd < A.Vd) {
            float y = ld_elem<DD>(drow, jd);
            y = y != y ? -INFINITY : y;
            w -= ex2(fmaf(y, c, -rs.mq)) * (1.f / rs.sq);
        }
    }
    if (!(w > 0.f)) return INFINITY;
    const uint4 w4 = philox_block(key, static_cast<uint32_t>(x >> 2), row, tag);
    const uint32_t wd = (x & 3) == 0 ? w4.x : ((x & 3) == 1 ? w4.y : ((x & 3) == 2 ? w4.z : w4.w));
    return __fdiv_rn(-log1pf(-one_minus_uniform_from_word(wd)), w);
}

template <int DT, int DD>
__global__ void __launch_bounds__(kRaceThreads) race_commit_kernel(SampleArgs A)
{
    pdl_wait_primary();
    __shared__ float red_f[kRaceThreads / 32];
    __shared__ int32_t red_i[kRaceThreads / 32];
    __shared__ int last_cta;
    __shared__ int32_t n_shared;
    __shared__ uint32_t fl_shared;
    const int tid = threadIdx.x, lane = tid & 31;
    const int32_t r = static_cast<int32_t>(blockIdx.x / A.race_ctas);
    const int32_t rc = static_cast<int32_t>(blockIdx.x - static_cast<int64_t>(r) * A.race_ctas);
    const int32_t k = A.k;
    const RowStat* st = A.stats + static_cast<int64_t>(r) * (k + 1);
    const int32_t* d = A.draft + static_cast<int64_t>(r) * k;
    const float T = A.temp[r];

    // request-level decisions (warp 0, ballots), identical in every CTA of the request
    if (tid < 32) {
        uint32_t fl = 0;
        for (int32_t j = lane; j <= k; j += 32) fl |= st[j].flags;
        fl = __reduce_or_sync(0xffffffffu, fl);
        const bool bad_rows = (fl & (kFlagNaN | kFlagPosInf | kFlagAllNegInf | kFlagDraftBad)) != 0;
        const bool greedy = !(T > 0.f) || bad_rows;
        int32_t n = k;
        for (int32_t j0 = 0; j0 < k; j0 += 32) {
            const int32_t j = j0 + lane;
            const bool fail = j < k && (greedy ? d[j] != st[j].amax : st[j].accept == 0);
            const unsigned m = __ballot_sync(0xffffffffu, fail);
            if (m) {
                n = j0 + __ffs(m) - 1;
                break;
            }
        }
        if (lane == 0) {
            n_shared = n;
            fl_shared = fl;
        }
    }
    __syncthreads();
    const int32_t n = n_shared;
    const uint32_t fl = fl_shared;
    const bool bad_rows = (fl & (kFlagNaN | kFlagPosInf | kFlagAllNegInf | kFlagDraftBad)) != 0;
    const bool greedy = !(T > 0.f) || bad_rows;
    int32_t token = -1;
    uint32_t status = 0;
    if (greedy) {
        if (rc != 0) return;
        token = st[n].amax;
    } else {
        const bool residual = n < k;
        const RowStat rs = st[n];
        const float c = kLog2e / T;
        const int32_t x0 = rc * A.race_seg, x1 = min(A.V, x0 + A.race_seg);
        const char* trow = A.tbase + (static_cast<int64_t>(r) * (k + 1) + n) * A.tstride;
        const char* drow = residual ? A.dbase + (static_cast<int64_t>(r) * k + n) * A.dstride : nullptr;
        const PhiloxKey key = philox_key(A.seeds[r]);
        const uint32_t tag = residual ? kTagResidual : kTagBonus;
        // start from the row's precomputed bound; the CTA holding its element keeps it as a candidate
        const int32_t cand_x = rs.bxc;
        float best = rs.bkey;
        int32_t bx = (tid == 0 && cand_x >= x0 && cand_x < x1 && best < INFINITY) ? cand_x : INT32_MAX;
        race_range<DT, DD>(A, trow, drow, x0, x1, c, rs, residual, key, static_cast<uint32_t>(n), tag,
                           A.tbulk != 0, best, bx);
        // (key, lowest x) minimum over the CTA; threads without a candidate carry (inf, INT32_MAX)
        float nb = bx == INT32_MAX ? -INFINITY : -best;
        int32_t nx = bx;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            const float ov = __shfl_xor_sync(0xffffffffu, nb, o);
            const int32_t ox = __shfl_xor_sync(0xffffffffu, nx, o);
            if (ov > nb || (ov == nb && ox < nx)) {
                nb = ov;
                nx = ox;
            }
        }
        if (lane == 0) {
            red_f[tid >> 5] = nb;
            red_i[tid >> 5] = nx;
        }
        __syncthreads();
        if (tid == 0) {
            for (int i = 1; i < kRaceThreads / 32; ++i)
                if (red_f[i] > nb || (red_f[i] == nb && red_i[i] < nx)) {
                    nb = red_f[i];
                    nx = red_i[i];
                }
            RaceSlot* slot = A.race + r;
            if (nx != INT32_MAX) atomicMin(&slot->best, pack_key(-nb, nx));
            __threadfence();
            const unsigned prev = atomicAdd(&slot->count, 1u);
            last_cta = prev == static_cast<unsigned>(A.race_ctas - 1);
        }
        __syncthreads();
        if (!last_cta) return;
        __threadfence();
        const unsigned long long packed = atomicOr(&A.race[r].best, 0ull);
        if (packed != ~0ull) {
            token = static_cast<int32_t>(packed & 0xffffffffull);
        } else {
            // no positive residual weight: draw the correction from p (rare)
            status |= SV_ST_RESIDUAL_ZERO;
            float b2 = INFINITY;
            int32_t x2 = INT32_MAX;
            race_range<DT, DD>(A, trow, drow, 0, A.V, c, rs, false, key, static_cast<uint32_t>(n), kTagResidual,
                               A.tbulk != 0, b2, x2);
            float nb2 = x2 == INT32_MAX ? -INFINITY : -b2;
            block_argmax<kRaceThreads>(nb2, x2, red_f, red_i);
            token = x2 == INT32_MAX ? 0 : x2;
        }
        if (residual && (rs.flags & kFlagOffSupport)) status |= SV_ST_OFF_SUPPORT;
    }
    // ---- commit (one CTA per request) ------------------------------------
    for (int32_t j = tid; j < k; j += kRaceThreads)
        if (d[j] < 0 || d[j] >= A.V) status |= SV_ST_TOKEN_RANGE;
    if (fl & kFlagTimeout) status |= SV_ST_TIMEOUT;
    if (bad_rows) status |= SV_ST_BAD_LOGITS;
    if (T < 0.f || T != T) status |= SV_ST_BAD_TEMP;
    if (!A.identity && (A.plan.header[2] != 0 || A.plan.header[0] != A.V || A.plan.header[1] != A.Vd))
        status |= SV_ST_BAD_D2T;
    int32_t* out = A.tokens + static_cast<int64_t>(r) * (k + 1);
    for (int32_t j = tid; j <= k; j += kRaceThreads) out[j] = j < n ? d[j] : (j == n ? token : -1);
    if (greedy) {
        // no sampling statistics for greedily verified requests
        for (int32_t j = tid; j < k; j += kRaceThreads) {
            const int64_t o = static_cast<int64_t>(r) * k + j;
            if (A.tv) A.tv[o] = NAN;
            if (A.pd) A.pd[o] = NAN;
            if (A.qd) A.qd[o] = NAN;
        }
    }
    status = block_or<kRaceThreads>(status, reinterpret_cast<uint32_t*>(red_i));
    if (tid == 0) {
        A.accept_len[r] = n;
        if (A.status) A.status[r] = static_cast<int32_t>(status);
    }
}

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------
namespace {

struct PlanLayout {
    int64_t header, bitmap, prefix, xs, js, pairs, chunk, x_of_j, total;
};

PlanLayout plan_layout(int32_t V, int32_t Vd)
{
    PlanLayout L{};
    const int64_t nw = (V + 31) / 32;
    int64_t off = 0;
    auto take = [&](int64_t bytes) {
        const int64_t o = off;
        off += align256(bytes + 16);  // 16 bytes of slack: bulk copies round up to 16
        return o;
    };
    L.header = take(16);
    L.bitmap = take(nw * 4);
    L.prefix = take((nw + 1) * 4);
    L.xs = take(static_cast<int64_t>(Vd) * 4);
    L.js = take(static_cast<int64_t>(Vd) * 4);
    L.pairs = take(static_cast<int64_t>(Vd) * 4);
    L.chunk = take((static_cast<int64_t>(V) / kChunkElems + 2) * 4);
    L.x_of_j = take(static_cast<int64_t>(Vd) * 4);
    L.total = off;
    return L;
}

D2tPlan plan_view(void* base, int32_t V, int32_t Vd)
{
    const PlanLayout L = plan_layout(V, Vd);
    char* b = static_cast<char*>(base);
    D2tPlan pl{};
    pl.header = reinterpret_cast<int32_t*>(b + L.header);
    pl.bitmap = reinterpret_cast<uint32_t*>(b + L.bitmap);
    pl.prefix = reinterpret_cast<int32_t*>(b + L.prefix);
    pl.xs = reinterpret_cast<int32_t*>(b + L.xs);
    pl.js = reinterpret_cast<int32_t*>(b + L.js);
    pl.pairs = reinterpret_cast<uint32_t*>(b + L.pairs);
    pl.chunk = reinterpret_cast<int32_t*>(b + L.chunk);
    pl.x_of_j = reinterpret_cast<int32_t*>(b + L.x_of_j);
    pl.nw = (V + 31) / 32;
    return pl;
}

struct SampleLayout {
    int64_t plan, stats, race, gslots;
    int64_t gslot_bytes;
    int64_t total;
    int smem_mode;
    size_t smem_bytes;
    int grid;
};

SampleLayout sample_layout(int64_t R, int32_t k, int32_t V, int32_t Vd, int et, int ed, int sms, bool own_plan)
{
    SampleLayout L{};
    int64_t off = 0;
    auto take = [&](int64_t bytes) {
        const int64_t o = off;
        off += align256(bytes);
        return o;
    };
    L.plan = take(own_plan ? plan_layout(V, Vd).total : 0);
    L.stats = take(R * (k + 1) * static_cast<int64_t>(sizeof(RowStat)));
    L.race = take(R * static_cast<int64_t>(sizeof(RaceSlot)));
    const int64_t units = R * (k + 1);
    L.grid = static_cast<int>(std::max<int64_t>(1, std::min<int64_t>(units, sms > 0 ? sms : 148)));
    const int64_t resident = align256(static_cast<int64_t>(Vd) * ed) + align256(static_cast<int64_t>(Vd) * et);
    const size_t ring = kRowHeader + static_cast<size_t>(kStages) * kStageBytes;
    L.smem_mode = ring + resident <= kSmemBudget ? 1 : 0;
    L.smem_bytes = ring + (L.smem_mode ? resident : 0);
    L.gslot_bytes = L.smem_mode ? 0 : resident;
    L.gslots = take(L.smem_mode ? 0 : L.gslot_bytes * L.grid);
    L.total = off + 256;
    return L;
}

size_t fast_smem_bytes(int32_t Vd)
{
    return static_cast<size_t>(kFastHeader + 2 * kFastWarps * static_cast<int64_t>(kFastStage) +
                               align256(static_cast<int64_t>(Vd) * 2));
}

bool fast_path_ok(const Rows& t, const Rows& d, bool identity)
{
    return !identity && t.dtype == SV_BF16 && d.dtype == SV_BF16 && t.bulk_ok && d.bulk_ok && d.data != nullptr &&
           t.width % 8 == 0 && d.width % 8 == 0 && d.width <= kFastMaxVd && fast_smem_bytes(d.width) <= 227 * 1024;
}

}  // namespace

size_t d2t_plan_bytes(int32_t V, int32_t Vd) { return static_cast<size_t>(plan_layout(V, Vd).total); }

cudaError_t launch_d2t_plan_build(const int32_t* d2t, int32_t Vd, int32_t V, void* plan, cudaStream_t stream)
{
    const D2tPlan pl = plan_view(plan, V, Vd);
    const size_t psmem = static_cast<size_t>(2 * pl.nw + 1) * 4;
    cudaError_t e = cudaFuncSetAttribute(d2t_plan_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(psmem));
    if (e != cudaSuccess) return e;
    d2t_plan_kernel<<<1, kPlanThreads, psmem, stream>>>(d2t, Vd, V, pl);
    return cudaGetLastError();
}

size_t sample_workspace_bytes(int64_t R, int32_t k, int32_t V, int32_t Vd)
{
    const int sms = device_sm_count();
    int64_t best = 0;
    for (int et : {2, 4})
        for (int ed : {2, 4}) best = std::max(best, sample_layout(R, k, V, Vd, et, ed, sms, true).total);
    return static_cast<size_t>(best);
}

template <int DT, int DD>
static cudaError_t launch_sample_t(const Rows& t, const Rows& d, const int32_t* d2t, const void* prebuilt,
                                   int32_t R, int32_t k, const int32_t* draft, const uint64_t* seeds,
                                   const float* temperature, int32_t* accept_len, int32_t* tokens, float* tv,
                                   float* p_draft, float* q_draft, int32_t* status, void* workspace,
                                   cudaStream_t stream)
{
    const int sms = device_sm_count();
    const bool identity = d2t == nullptr && prebuilt == nullptr;
    const bool own_plan = !identity && prebuilt == nullptr;
    const SampleLayout L = sample_layout(R, k, t.width, d.width, t.esize, d.esize, sms, own_plan);
    char* ws = static_cast<char*>(workspace);
    SampleArgs A{};
    A.tbase = t.data;
    A.tstride = t.stride * t.esize;
    A.V = t.width;
    A.dbase = d.data;
    A.dstride = d.stride * d.esize;
    A.Vd = d.width;
    A.identity = identity;
    A.tbulk = t.bulk_ok;
    A.dbulk = d.bulk_ok && d.data != nullptr;
    if (!identity) A.plan = plan_view(own_plan ? ws + L.plan : const_cast<void*>(prebuilt), t.width, d.width);
    A.R = R;
    A.k = k;
    A.draft = draft;
    A.seeds = seeds;
    A.temp = temperature;
    A.tv = tv;
    A.pd = p_draft;
    A.qd = q_draft;
    A.accept_len = accept_len;
    A.tokens = tokens;
    A.status = status;
    A.stats = reinterpret_cast<RowStat*>(ws + L.stats);
    A.race = reinterpret_cast<RaceSlot*>(ws + L.race);
    A.gslots = ws + L.gslots;
    A.gslot_bytes = L.gslot_bytes;
    A.smem_mode = L.smem_mode;
    A.race_seg = kRaceSeg;
    A.race_ctas = (t.width + kRaceSeg - 1) / kRaceSeg;

    cudaError_t e;
    if (own_plan) {
        if ((e = launch_d2t_plan_build(d2t, d.width, t.width, ws + L.plan, stream)) != cudaSuccess) return e;
    }
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = own_plan ? 1 : 0;
    if (fast_path_ok(t, d, identity)) {
        const size_t smem = fast_smem_bytes(d.width);
        e = cudaFuncSetAttribute(sample_rows_fast_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 static_cast<int>(smem));
        if (e != cudaSuccess) return e;
        cfg.gridDim = dim3(static_cast<unsigned>(L.grid));
        cfg.blockDim = dim3(kFastThreads);
        cfg.dynamicSmemBytes = smem;
        e = cudaLaunchKernelEx(&cfg, sample_rows_fast_kernel, A);
    } else {
        e = cudaFuncSetAttribute(sample_rows_kernel<DT, DD>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 static_cast<int>(L.smem_bytes));
        if (e != cudaSuccess) return e;
        cfg.gridDim = dim3(static_cast<unsigned>(L.grid));
        cfg.blockDim = dim3(kRowThreads);
        cfg.dynamicSmemBytes = L.smem_bytes;
        e = cudaLaunchKernelEx(&cfg, sample_rows_kernel<DT, DD>, A);
    }
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg2 = {};
    cfg2.gridDim = dim3(static_cast<unsigned>(static_cast<int64_t>(R) * A.race_ctas));
    cfg2.blockDim = dim3(kRaceThreads);
    cfg2.dynamicSmemBytes = 0;
    cfg2.stream = stream;
    cfg2.attrs = attr;
    cfg2.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg2, race_commit_kernel<DT, DD>, A);
}

cudaError_t launch_verify_sample(const Rows& target, const Rows& draft_logits, const int32_t* d2t,
                                 const void* d2t_plan, int32_t R, int32_t k, const int32_t* draft,
                                 const uint64_t* seeds, const float* temperature, int32_t* accept_len,
                                 int32_t* tokens, float* tv, float* p_draft, float* q_draft, int32_t* status,
                                 void* workspace, cudaStream_t stream)
{
    const bool tb = target.dtype == SV_BF16, db = draft_logits.dtype == SV_BF16;
#define SV_SAMPLE_CALL(A_, B_)                                                                            \
    launch_sample_t<A_, B_>(target, draft_logits, d2t, d2t_plan, R, k, draft, seeds, temperature, accept_len, \
                            tokens, tv, p_draft, q_draft, status, workspace, stream)
    if (tb && db) return SV_SAMPLE_CALL(SV_BF16, SV_BF16);
    if (tb && !db) return SV_SAMPLE_CALL(SV_BF16, SV_F32);
    if (!tb && db) return SV_SAMPLE_CALL(SV_F32, SV_BF16);
    return SV_SAMPLE_CALL(SV_F32, SV_F32);
#undef SV_SAMPLE_CALL
}

int32_t sample_max_plan_width() { return kMaxPlanWords * 32; }

}  // namespace sv
