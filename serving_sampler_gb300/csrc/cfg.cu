// Classifier-free-guidance merge per RVQ codebook, then verification ("An
// Efficient vLLM-Based Inference Pipeline for Unified Audio Understanding and
// Generation", paired CFG co-scheduling: per codebook the conditional and
// unconditional logits are merged linearly with weight w; Figure 1 text: each
// codebook samples from its own partition of the vocabulary).  Sampling rules
// follow "speculative decoding for Omni models", section 2.
//
// cfg_rows_warp_kernel  one warp per (request, frame j, codebook s) row.  The
//                  row's codebook slice of cond and uncond is merged in fp32 as
//                  fmaf(w, c - u, u) (packed fp32 pairs, the same roundings);
//                  pass 1 takes the merged row's argmax and online max /
//                  sum-exp at T and the draft row's; pass 2 (the slices again,
//                  from L2) TV = sum max(0, q - p) and p, q at the drafted id;
//                  then the accept test (Philox row j * S + s).
// cfg_race_kernel  one CTA per (request, codebook): the first frame n with a
//                  rejected codebook, then for codebook s its draft if its own
//                  test passed, else the exponential race over the codebook's
//                  ids of the residual at frame n (or of p at the bonus frame
//                  k), its weights rebuilt from the inputs.  Codebook 0 also
//                  writes accept_len.
#include <algorithm>
#include <cfloat>
#include <climits>

#include "sv_device.cuh"
#include "sv_internal.h"

namespace sv {

namespace {

constexpr int32_t kCfgMaxW = 16384;  // widest codebook

enum : uint32_t { kCfgBad = 1u, kCfgOffSupport = 2u };

struct CfgStat {
    float m, s;     // merged row: max of m c, sum 2^(m c - max)
    float mq, sq;   // draft row
    int32_t amax;   // argmax of the merged row (local id)
    uint32_t flags; // kCfgBad: NaN / +inf / all -inf in the merged or draft row
    int32_t accept; // accept decision (sampling)
    float pad;
};

struct CfgArgs {
    const char* cbase;
    const char* ubase;
    int64_t stride;  // bytes, shared by cond and uncond
    const char* dbase;
    int64_t dstride;
    int cvec, dvec;  // 16-byte loads allowed for cond/uncond slices and for draft rows
    CfgShape shape;
    int32_t R, k;
    const int32_t* draft;
    const uint64_t* seeds;
    const float* temp;
    int32_t* accept_len;
    int32_t* tokens;
    float* tv;
    int32_t* status;
    CfgStat* stats;
};



__device__ __forceinline__ float wsum(float v)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

}  // namespace

// One warp per (request, frame j, codebook s) row, four rows per CTA, no block
// barrier.  Pass 1 streams the row's codebook slices of cond, uncond and the
// draft row in batches of 32 ids per lane (the next batch's loads in flight
// while one is reduced): merged logits fmaf(w, c - u, u), argmax, NaN / +inf
// flags, and online max / sum-exp at T of the merged and the draft row.
// Pass 2 reads the slices again (from L2) for TV = sum max(0, q - p) and p, q
// at the drafted id.
constexpr int kCfgWarpRows = 4;

// one 8-id group of a row as raw 16-byte words (bf16: 1, fp32: 2); -inf beyond W
template <int DT>
struct Grp {
    static constexpr int kWords = DT == SV_BF16 ? 1 : 2;
    uint4 q[kWords];
};

template <int DT>
__device__ __forceinline__ void ld_grp(const char* p, int32_t e0, int32_t W, bool vec, Grp<DT>& g)
{
    if (vec && e0 + 8 <= W) {
#pragma unroll
        for (int h = 0; h < Grp<DT>::kWords; ++h)
            g.q[h] = ld_nc_v4(reinterpret_cast<const uint4*>(p + static_cast<int64_t>(e0) * (DT == SV_BF16 ? 2 : 4)) + h);
        return;
    }
    uint32_t wv[4 * Grp<DT>::kWords];
    if constexpr (DT == SV_BF16) {
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const uint32_t lo = e0 + 2 * i < W ? reinterpret_cast<const uint16_t*>(p)[e0 + 2 * i] : 0xFF80u;
            const uint32_t hi = e0 + 2 * i + 1 < W ? reinterpret_cast<const uint16_t*>(p)[e0 + 2 * i + 1] : 0xFF80u;
            wv[i] = lo | (hi << 16);
        }
    } else {
#pragma unroll
        for (int i = 0; i < 8; ++i)
            wv[i] = e0 + i < W ? reinterpret_cast<const uint32_t*>(p)[e0 + i] : 0xFF800000u;
    }
#pragma unroll
    for (int h = 0; h < Grp<DT>::kWords; ++h) g.q[h] = make_uint4(wv[4 * h], wv[4 * h + 1], wv[4 * h + 2], wv[4 * h + 3]);
}

// ids 2h, 2h + 1 of a group as an fp32 pair (h = 0..3)
template <int DT>
__device__ __forceinline__ unsigned long long grp_pair(const Grp<DT>& g, int h)
{
    if constexpr (DT == SV_BF16) {
        const uint32_t w = h == 0 ? g.q[0].x : h == 1 ? g.q[0].y : h == 2 ? g.q[0].z : g.q[0].w;
        return bf16x2_to_f32x2(w);
    } else {
        const uint4& q = g.q[h >> 1];
        return (h & 1) ? pack2(__uint_as_float(q.z), __uint_as_float(q.w))
                       : pack2(__uint_as_float(q.x), __uint_as_float(q.y));
    }
}

// element e of a row, widened exactly to fp32
template <int DT>
__device__ __forceinline__ float row_value(const char* p, int32_t e)
{
    if constexpr (DT == SV_BF16)
        return __uint_as_float(static_cast<uint32_t>(reinterpret_cast<const uint16_t*>(p)[e]) << 16);
    else
        return reinterpret_cast<const float*>(p)[e];
}

template <int DT, int DD>
__global__ void __launch_bounds__(32 * kCfgWarpRows, 4) cfg_rows_warp_kernel(CfgArgs A)
{
    constexpr int kG = 2;      // groups of 8 ids per lane and batch
    constexpr int kP = 4 * kG; // fp32 pairs per lane and batch
    pdl_launch_dependents();
    const int lane = threadIdx.x & 31;
    const int32_t S = A.shape.S, W = A.shape.W, k = A.k;
    const int64_t units = static_cast<int64_t>(A.R) * (k + 1) * S;
    const int64_t unit = static_cast<int64_t>(blockIdx.x) * kCfgWarpRows + (threadIdx.x >> 5);
    if (unit >= units) return;  // whole warps only
    const int32_t s = static_cast<int32_t>(unit % S);
    const int64_t rj = unit / S;
    const int32_t j = static_cast<int32_t>(rj % (k + 1));
    const int32_t r = static_cast<int32_t>(rj / (k + 1));
    const float T = A.temp[r];
    // NULL draft rows select greedy verification when there are drafts; with k = 0 the bonus
    // follows the temperature alone
    const bool sampling = T > 0.f && (A.dbase != nullptr || k == 0);
    const bool has_draft = sampling && j < k;
    const float c = sampling ? temp_scale(T) : 0.f;
    const unsigned long long w2 = pack2(A.shape.w, A.shape.w), c2 = pack2(c, c);
    const int64_t off = unit * A.stride + static_cast<int64_t>(A.shape.data_off[s]) * (DT == SV_BF16 ? 2 : 4);
    const char* cp = A.cbase + off;
    const char* up = A.ubase + off;
    const char* dp = has_draft ? A.dbase + ((static_cast<int64_t>(r) * k + j) * S + s) * A.dstride : nullptr;
    const bool cvec = A.cvec != 0, dvec = A.dvec != 0;
    const int32_t ngroups = (W + 7) / 8;
    const int32_t nb = (ngroups + 32 * kG - 1) / (32 * kG);

    Grp<DT> cg[kG], ug[kG];
    Grp<DD> yg[kG];
    auto load = [&](int32_t b) {
#pragma unroll
        for (int i = 0; i < kG; ++i) {
            const int32_t e0 = 8 * (lane + 32 * (kG * b + i));
            ld_grp<DT>(cp, e0, W, cvec, cg[i]);
            ld_grp<DT>(up, e0, W, cvec, ug[i]);
            if (dp) ld_grp<DD>(dp, e0, W, dvec, yg[i]);
        }
    };
    // merged pairs fmaf(w, c - u, u) (the same two roundings as the scalar form); ids at or
    // beyond W (only in the last batch) read -inf
    auto merge = [&](int32_t b, unsigned long long* m2) {
#pragma unroll
        for (int i = 0; i < kG; ++i)
#pragma unroll
            for (int h = 0; h < 4; ++h) {
                const unsigned long long u2 = grp_pair<DT>(ug[i], h);
                m2[4 * i + h] = fma2(w2, sub2(grp_pair<DT>(cg[i], h), u2), u2);
            }
        if (8 * 32 * kG * (b + 1) > W) {  // the tail batch
#pragma unroll
            for (int i = 0; i < kG; ++i)
#pragma unroll
                for (int h = 0; h < 4; ++h) {
                    const int32_t x = 8 * (lane + 32 * (kG * b + i)) + 2 * h;
                    float lo, hi;
                    unpack2(m2[4 * i + h], lo, hi);
                    m2[4 * i + h] = pack2(x < W ? lo : -INFINITY, x + 1 < W ? hi : -INFINITY);
                }
        }
    };

    // ---- pass 1 ----
    float bv = -INFINITY;  // argmax value (NaN-propagating per batch; a NaN row is flagged)
    int32_t bx = INT32_MAX;
    float ymx = -INFINITY;
    bool nan_seen = false;
    float tm = -INFINITY, dm = -INFINITY;                  // running maxima (log2 units)
    unsigned long long ts2 = 0ull, ds2 = 0ull;             // running sums (pairs)
    load(0);
    for (int32_t b = 0; b < nb; ++b) {
        unsigned long long m2[kP], y2[kP];
        merge(b, m2);
#pragma unroll
        for (int i = 0; i < kG; ++i)
#pragma unroll
            for (int h = 0; h < 4; ++h) y2[4 * i + h] = dp ? grp_pair<DD>(yg[i], h) : pack2(-INFINITY, -INFINITY);
        if (b + 1 < nb) load(b + 1);
        float lm = -INFINITY, ly = -INFINITY;
#pragma unroll
        for (int p = 0; p < kP; ++p) {
            float lo, hi;
            unpack2(m2[p], lo, hi);
            lm = fmax_nan(lm, fmax_nan(lo, hi));
            unpack2(y2[p], lo, hi);
            ly = fmax_nan(ly, fmax_nan(lo, hi));
        }
        if (lm != lm) {  // rare: NaN logits, which the argmax reads as -inf (the row is flagged)
            nan_seen = true;
            lm = -INFINITY;
#pragma unroll
            for (int p = 0; p < kP; ++p) {
                float lo, hi;
                unpack2(m2[p], lo, hi);
                lm = fmaxf(lm, fmaxf(lo, hi));
            }
        }
        if (lm > bv) {  // the first id of the batch holding its maximum (ids ascend in the lane)
#pragma unroll
            for (int p = kP - 1; p >= 0; --p) {
                float lo, hi;
                unpack2(m2[p], lo, hi);
                const int32_t x = 8 * (lane + 32 * (kG * b + p / 4)) + 2 * (p % 4);
                if (hi == lm) bx = x + 1;
                if (lo == lm) bx = x;
            }
            bv = lm;
        }
        ymx = fmax_nan(ymx, ly);
        if (sampling && !nan_seen) {
            const float mt = lm * c;
            if (mt > tm) {
                const float sc = tm == -INFINITY ? 0.f : ex2(tm - mt);
                ts2 = mul2(ts2, pack2(sc, sc));
                tm = mt;
            }
            if (tm > -INFINITY && tm < INFINITY) {
                const unsigned long long nm2 = pack2(-tm, -tm);
#pragma unroll
                for (int p = 0; p < kP; ++p) {
                    float a0, a1;
                    unpack2(fma2(m2[p], c2, nm2), a0, a1);
                    ts2 = add2(ts2, pack2(ex2(a0), ex2(a1)));
                }
            }
        }
        if (has_draft && !(ly != ly)) {
            const float yt = ly * c;
            if (yt > dm) {
                const float sc = dm == -INFINITY ? 0.f : ex2(dm - yt);
                ds2 = mul2(ds2, pack2(sc, sc));
                dm = yt;
            }
            if (dm > -INFINITY && dm < INFINITY) {
                const unsigned long long nd2 = pack2(-dm, -dm);
#pragma unroll
                for (int p = 0; p < kP; ++p) {
                    float a0, a1;
                    unpack2(fma2(y2[p], c2, nd2), a0, a1);
                    ds2 = add2(ds2, pack2(ex2(a0), ex2(a1)));
                }
            }
        }
    }
    float ts, ds;
    {
        float a0, a1;
        unpack2(ts2, a0, a1);
        ts = a0 + a1;
        unpack2(ds2, a0, a1);
        ds = a0 + a1;
    }
    // warp reductions
    const float my_tm = tm, my_dm = dm;
    bool bad_l = nan_seen || bv == INFINITY || (has_draft && (ymx != ymx || ymx == INFINITY));
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
        ymx = fmaxf(ymx, __shfl_xor_sync(0xffffffffu, ymx, o));
    }
    bool bad = __any_sync(0xffffffffu, bad_l) || bv == -INFINITY;
    if (has_draft) bad = bad || dm == -INFINITY;
    float sm = (my_tm > -INFINITY && tm > -INFINITY) ? ts * ex2(my_tm - tm) : 0.f;
    float sq = (my_dm > -INFINITY && dm > -INFINITY) ? ds * ex2(my_dm - dm) : 0.f;
    sm = wsum(sm);
    sq = wsum(sq);
    CfgStat st{};
    st.amax = bx == INT32_MAX ? 0 : bx;
    st.m = -INFINITY;
    st.mq = -INFINITY;
    float tvv = NAN;
    if (sampling && !bad) {
        st.m = tm;
        st.s = sm;
        if (has_draft) {
            st.mq = dm;
            st.sq = sq;
            // ---- pass 2: TV and p, q at the drafted id ----
            const int32_t xl = A.draft[(static_cast<int64_t>(r) * k + j) * S + s] - A.shape.id_base[s];
            const unsigned long long nm2 = pack2(-tm, -tm), nd2 = pack2(-dm, -dm);
            const unsigned long long iS2 = pack2(1.f / sm, 1.f / sm), iQ2 = pack2(1.f / sq, 1.f / sq);
            unsigned long long t2 = 0ull;
            load(0);
            for (int32_t b = 0; b < nb; ++b) {
                unsigned long long m2[kP], y2[kP];
                merge(b, m2);
#pragma unroll
                for (int i = 0; i < kG; ++i)
#pragma unroll
                    for (int h = 0; h < 4; ++h) y2[4 * i + h] = grp_pair<DD>(yg[i], h);
                if (b + 1 < nb) load(b + 1);
#pragma unroll
                for (int p = 0; p < kP; ++p) {
                    float a0, a1, b0, b1;
                    unpack2(fma2(m2[p], c2, nm2), a0, a1);
                    unpack2(fma2(y2[p], c2, nd2), b0, b1);
                    const unsigned long long p2 = mul2(pack2(ex2(a0), ex2(a1)), iS2);
                    const unsigned long long q2 = mul2(pack2(ex2(b0), ex2(b1)), iQ2);
                    float d0, d1;
                    unpack2(sub2(q2, p2), d0, d1);
                    // ids beyond W hold p = 0 and q of a -inf logit = 0
                    t2 = add2(t2, pack2(fmaxf(d0, 0.f), fmaxf(d1, 0.f)));
                }
            }
            float t;
            {
                float a0, a1;
                unpack2(t2, a0, a1);
                t = a0 + a1;
            }
            t = wsum(t);
            // p and q at the drafted id, with the pass's own operations on that id's inputs
            float pxl = 0.f, qxl = 0.f;
            if (xl >= 0 && xl < W) {
                const float cx = row_value<DT>(cp, xl), ux = row_value<DT>(up, xl), yx = row_value<DD>(dp, xl);
                const float mx = fmaf(A.shape.w, cx - ux, ux);
                pxl = ex2(fmaf(mx, c, -tm)) * (1.f / sm);
                qxl = ex2(fmaf(yx, c, -dm)) * (1.f / sq);
            }
            tvv = t;
            int32_t acc_ok = 0;
            if (xl >= 0 && xl < W) {
                if (qxl > 0.f) {
                    const uint4 w4 = philox_block(philox_key(A.seeds[r]), 0u, static_cast<uint32_t>(j * S + s),
                                                  kTagAccept);
                    acc_ok = uniform_from_word(w4.x) < __fdiv_rn(pxl, qxl) ? 1 : 0;
                } else {
                    st.flags |= kCfgOffSupport;
                }
            }
            st.accept = acc_ok;
        }
    }
    if (bad) st.flags |= kCfgBad;
    if (lane == 0) {
        A.stats[unit] = st;
        if (A.tv && j < k) A.tv[(static_cast<int64_t>(r) * k + j) * S + s] = tvv;
        if (A.status && j == 0 && s == 0) A.status[r] = 0;  // the race kernel ORs the codebooks' bits
    }
}

// One CTA of kCfgRaceThreads per (request, codebook): warp 0 finds the first frame
// n with a rejected codebook (or, greedy, a mismatching one); then codebook s's
// token at frame n: its draft if its own test passed, else the exponential race
// over the codebook's W ids of the residual max(0, p - q) at frame n (p at the
// bonus frame k).  The weights are rebuilt from the inputs into shared memory;
// the key of the heaviest id bounds the minimum key B, so a Philox block is
// generated only when one of its ids has B w >= 2^-24 and a logarithm is taken
// only when 1 - u <= B w (both widened against fp32 rounding).  Codebook 0
// writes accept_len; the codebooks' status bits meet in an atomic OR on a
// status word the row pass zeroed.
constexpr int kCfgRaceThreads = 128;
constexpr float kCfgRaceSlack = 1.0f + 1.0f / 1024.0f;
constexpr float kCfgRaceMinGap = 5.9604645e-8f;  // 2^-24: the smallest 1 - u

template <int DT, int DD>
__global__ void __launch_bounds__(kCfgRaceThreads) cfg_race_kernel(CfgArgs A)
{
    pdl_wait_primary();
    extern __shared__ __align__(16) float wbuf[];  // the race weights, W rounded up to 8
    __shared__ float hv_s[kCfgRaceThreads / 32];
    __shared__ int32_t hx_s[kCfgRaceThreads / 32];
    __shared__ unsigned long long kb_s[kCfgRaceThreads / 32];
    __shared__ float bound_s;
    __shared__ int32_t n_s;
    __shared__ uint32_t fl_s;
    const int tid = threadIdx.x, lane = tid & 31, wq = tid >> 5;
    const int32_t S = A.shape.S, W = A.shape.W, k = A.k;
    const int32_t r = static_cast<int32_t>(blockIdx.x / S);
    const int32_t s = static_cast<int32_t>(blockIdx.x - static_cast<int64_t>(r) * S);
    const float T = A.temp[r];
    const CfgStat* st = A.stats + static_cast<int64_t>(r) * (k + 1) * S;
    const int32_t* d = A.draft + static_cast<int64_t>(r) * k * S;

    // ---- the request's decisions (warp 0) ----
    if (wq == 0) {
        uint32_t fl = 0;
        for (int32_t i = lane; i < (k + 1) * S; i += 32) fl |= st[i].flags;
        fl = __reduce_or_sync(0xffffffffu, fl);
        const bool bad0 = (fl & kCfgBad) != 0;
        const bool greedy0 = !(T > 0.f) || (A.dbase == nullptr && k > 0) || bad0;
        uint32_t nf = static_cast<uint32_t>(k);
        for (int32_t i = lane; i < k * S; i += 32) {
            const int32_t q = i % S;
            const bool ok = greedy0 ? (d[i] - A.shape.id_base[q] == st[i].amax) : st[i].accept != 0;
            if (!ok) nf = min(nf, static_cast<uint32_t>(i / S));
        }
        nf = __reduce_min_sync(0xffffffffu, nf);
        if (lane == 0) {
            n_s = static_cast<int32_t>(nf);
            fl_s = fl;
        }
    }
    __syncthreads();
    const int32_t n = n_s;
    const bool bad = (fl_s & kCfgBad) != 0;
    const bool greedy = !(T > 0.f) || (A.dbase == nullptr && k > 0) || bad;

    int32_t tok_local = 0;
    uint32_t status = 0;
    const CfgStat sn = st[n * S + s];
    if (greedy) {
        tok_local = sn.amax;
    } else if (n < k && sn.accept) {
        tok_local = d[n * S + s] - A.shape.id_base[s];
    } else {
        const bool residual = n < k;
        const float c = temp_scale(T);
        const unsigned long long w2 = pack2(A.shape.w, A.shape.w), c2 = pack2(c, c);
        const unsigned long long nm2 = pack2(-sn.m, -sn.m), nd2 = pack2(-sn.mq, -sn.mq);
        const unsigned long long iS2 = pack2(1.f / sn.s, 1.f / sn.s);
        const unsigned long long iQ2 = residual ? pack2(1.f / sn.sq, 1.f / sn.sq) : 0ull;
        const int64_t row = (static_cast<int64_t>(r) * (k + 1) + n) * S + s;
        const int64_t off = row * A.stride + static_cast<int64_t>(A.shape.data_off[s]) * (DT == SV_BF16 ? 2 : 4);
        const char* cp = A.cbase + off;
        const char* up = A.ubase + off;
        const char* dp = residual ? A.dbase + ((static_cast<int64_t>(r) * k + n) * S + s) * A.dstride : nullptr;
        const bool cvec = A.cvec != 0, dvec = A.dvec != 0;
        const PhiloxKey key = philox_key(A.seeds[r]);
        const uint32_t prow = static_cast<uint32_t>(n * S + s);
        const uint32_t tag = residual ? kTagResidual : kTagBonus;
        const int32_t ngroups = (W + 7) / 8;
        for (int pass = 0; pass < 2; ++pass) {  // pass 1: no residual mass, draw from p
            const bool wres = residual && pass == 0;
            // ---- weights into shared memory; every thread's heaviest id ----
            float hw = 0.f;
            int32_t hx = INT32_MAX;
            for (int32_t g = tid; g < ngroups; g += kCfgRaceThreads) {
                const int32_t e0 = 8 * g;
                Grp<DT> cg, ug;
                Grp<DD> yg;
                ld_grp<DT>(cp, e0, W, cvec, cg);
                ld_grp<DT>(up, e0, W, cvec, ug);
                if (wres) ld_grp<DD>(dp, e0, W, dvec, yg);
                float wt[8];
#pragma unroll
                for (int h = 0; h < 4; ++h) {
                    const unsigned long long u2 = grp_pair<DT>(ug, h);
                    const unsigned long long m2 = fma2(w2, sub2(grp_pair<DT>(cg, h), u2), u2);
                    float a0, a1;
                    unpack2(fma2(m2, c2, nm2), a0, a1);
                    unsigned long long p2 = mul2(pack2(ex2(a0), ex2(a1)), iS2);
                    if (wres) {
                        float b0, b1;
                        unpack2(fma2(grp_pair<DD>(yg, h), c2, nd2), b0, b1);
                        p2 = sub2(p2, mul2(pack2(ex2(b0), ex2(b1)), iQ2));
                    }
                    unpack2(p2, wt[2 * h], wt[2 * h + 1]);
                }
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    wt[e] = (e0 + e < W && wt[e] > 0.f) ? wt[e] : 0.f;  // NaN never wins
                    if (wt[e] > hw) {  // ascending ids within the thread
                        hw = wt[e];
                        hx = e0 + e;
                    }
                }
                reinterpret_cast<float4*>(wbuf + e0)[0] = make_float4(wt[0], wt[1], wt[2], wt[3]);
                reinterpret_cast<float4*>(wbuf + e0)[1] = make_float4(wt[4], wt[5], wt[6], wt[7]);
            }
            // ---- the heaviest id of the row and its key: the bound B ----
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) {
                const float ov = __shfl_xor_sync(0xffffffffu, hw, o);
                const int32_t ox = __shfl_xor_sync(0xffffffffu, hx, o);
                if (ov > hw || (ov == hw && ox < hx)) {
                    hw = ov;
                    hx = ox;
                }
            }
            if (lane == 0) {
                hv_s[wq] = hw;
                hx_s[wq] = hx;
            }
            __syncthreads();
            if (tid == 0) {
                float bw = 0.f;
                int32_t bx = INT32_MAX;
                for (int i = 0; i < kCfgRaceThreads / 32; ++i)
                    if (hv_s[i] > bw || (hv_s[i] == bw && hx_s[i] < bx)) {
                        bw = hv_s[i];
                        bx = hx_s[i];
                    }
                float b = INFINITY;
                if (bw > 0.f && bx != INT32_MAX) {
                    const uint4 w4 = philox_block(key, static_cast<uint32_t>(bx) >> 2, prow, tag);
                    const uint32_t wd = (bx & 3) == 0 ? w4.x : (bx & 3) == 1 ? w4.y : (bx & 3) == 2 ? w4.z : w4.w;
                    b = __fdiv_rn(-log1pf(-one_minus_uniform_from_word(wd)), bw);
                }
                bound_s = b;
            }
            __syncthreads();
            const float B = bound_s;
            if (!(B < INFINITY)) {  // no weight anywhere (block-uniform)
                if (!residual || pass == 1) break;
                status |= SV_ST_RESIDUAL_ZERO;
                __syncthreads();  // wbuf and the shared arrays are written again
                continue;
            }
            // ---- the race: blocks of four ids, one Philox block each when one of them can win ----
            const float bs = B * kCfgRaceSlack;
            float best = INFINITY;
            int32_t bx = INT32_MAX;
            for (int32_t b4 = tid; 4 * b4 < W; b4 += kCfgRaceThreads) {
                const float4 wv = reinterpret_cast<const float4*>(wbuf)[b4];
                const float w4v[4] = {wv.x, wv.y, wv.z, wv.w};
                bool need = false;
#pragma unroll
                for (int e = 0; e < 4; ++e) need |= w4v[e] * bs >= kCfgRaceMinGap;
                if (!need) continue;
                const uint4 u4 = philox_block(key, static_cast<uint32_t>(b4), prow, tag);
                const uint32_t words[4] = {u4.x, u4.y, u4.z, u4.w};
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const float w = w4v[e];
                    if (!(w > 0.f)) continue;
                    const float om = one_minus_uniform_from_word(words[e]);
                    if (!(om <= w * bs)) continue;
                    const float kx = __fdiv_rn(-log1pf(-om), w);
                    if (kx < best) {  // ascending ids within the thread
                        best = kx;
                        bx = 4 * b4 + e;
                    }
                }
            }
            unsigned long long pk = bx == INT32_MAX ? ~0ull
                                                     : (static_cast<unsigned long long>(__float_as_uint(best)) << 32) |
                                                           static_cast<uint32_t>(bx);
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) {
                const unsigned long long ov = __shfl_xor_sync(0xffffffffu, pk, o);
                pk = ov < pk ? ov : pk;
            }
            if (lane == 0) kb_s[wq] = pk;
            __syncthreads();
            unsigned long long m = ~0ull;
            for (int i = 0; i < kCfgRaceThreads / 32; ++i) m = kb_s[i] < m ? kb_s[i] : m;
            tok_local = m == ~0ull ? 0 : static_cast<int32_t>(m & 0xFFFFFFFFu);
            break;
        }
        if (residual && (sn.flags & kCfgOffSupport)) status |= SV_ST_OFF_SUPPORT;
    }
    if (wq != 0) return;
    // ---- codebook s's tokens for every frame; status ----
    int32_t* out = A.tokens + static_cast<int64_t>(r) * (k + 1) * S;
    for (int32_t j = lane; j <= k; j += 32)
        out[j * S + s] = j < n ? d[j * S + s] : (j == n ? A.shape.id_base[s] + tok_local : -1);
    if (greedy && A.tv) {
        for (int32_t j = lane; j < k; j += 32) A.tv[(static_cast<int64_t>(r) * k + j) * S + s] = NAN;
    }
    uint32_t st_bits = status;
    for (int32_t j = lane; j < k; j += 32) {
        const int32_t l = d[j * S + s] - A.shape.id_base[s];
        if (l < 0 || l >= W) st_bits |= SV_ST_TOKEN_RANGE;
    }
    st_bits = __reduce_or_sync(0xffffffffu, st_bits);
    if (lane == 0) {
        if (s == 0) {
            if (bad) st_bits |= SV_ST_BAD_LOGITS;
            if (T < 0.f || T != T) st_bits |= SV_ST_BAD_TEMP;
            A.accept_len[r] = n;
        }
        if (A.status && st_bits) atomicOr(reinterpret_cast<unsigned int*>(A.status + r), st_bits);
    }
}

static int64_t cfg_stats_bytes(int64_t R, int32_t k, int32_t S)
{
    return (R * (k + 1) * S * static_cast<int64_t>(sizeof(CfgStat)) + 255) / 256 * 256;
}

size_t cfg_workspace_bytes(int64_t R, int32_t k, int32_t S, int32_t W)
{
    (void)W;
    return static_cast<size_t>(cfg_stats_bytes(R, k, S) + 256);
}

template <int DT, int DD>
static cudaError_t launch_cfg_t(const CfgArgs& A, int32_t R, int32_t k, cudaStream_t stream)
{
    cudaError_t e;
    const int64_t units = static_cast<int64_t>(R) * (k + 1) * A.shape.S;
    cfg_rows_warp_kernel<DT, DD>
        <<<static_cast<unsigned>((units + kCfgWarpRows - 1) / kCfgWarpRows), 32 * kCfgWarpRows, 0, stream>>>(A);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    const size_t wsmem = static_cast<size_t>((A.shape.W + 7) / 8) * 8 * sizeof(float);
    e = cudaFuncSetAttribute(cfg_race_kernel<DT, DD>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(wsmem));
    if (e != cudaSuccess) return e;
    cfg.gridDim = dim3(static_cast<unsigned>(static_cast<int64_t>(R) * A.shape.S));
    cfg.blockDim = dim3(kCfgRaceThreads);
    cfg.dynamicSmemBytes = wsmem;
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, cfg_race_kernel<DT, DD>, A);
}

cudaError_t launch_cfg_merge_sample(const Rows& cond, const Rows& uncond, const CfgShape& shape,
                                    const Rows* draft_logits, int32_t R, int32_t k,
                                    const int32_t* draft, const uint64_t* seeds,
                                    const float* temperature, int32_t* accept_len,
                                    int32_t* tokens, float* tv, int32_t* status, void* workspace,
                                    cudaStream_t stream)
{
    if (shape.W > kCfgMaxW) return cudaErrorInvalidValue;
    CfgArgs A{};
    A.cbase = cond.data;
    A.ubase = uncond.data;
    A.stride = cond.stride * cond.esize;
    A.dbase = draft_logits ? draft_logits->data : nullptr;
    A.dstride = draft_logits ? draft_logits->stride * draft_logits->esize : 0;
    // 16-byte loads: every slice start and the width in 16-byte units
    bool cvec = cond.bulk_ok && uncond.bulk_ok && (static_cast<int64_t>(shape.W) * cond.esize) % 16 == 0;
    for (int q = 0; q < shape.S; ++q) cvec = cvec && (static_cast<int64_t>(shape.data_off[q]) * cond.esize) % 16 == 0;
    A.cvec = cvec;
    A.dvec = draft_logits && draft_logits->bulk_ok && (static_cast<int64_t>(shape.W) * draft_logits->esize) % 16 == 0;
    A.shape = shape;
    A.R = R;
    A.k = k;
    A.draft = draft;
    A.seeds = seeds;
    A.temp = temperature;
    A.accept_len = accept_len;
    A.tokens = tokens;
    A.tv = tv;
    A.status = status;
    A.stats = static_cast<CfgStat*>(workspace);
    const bool cb = cond.dtype == SV_BF16;
    const bool db = draft_logits == nullptr || draft_logits->dtype == SV_BF16;
    if (cb && db) return launch_cfg_t<SV_BF16, SV_BF16>(A, R, k, stream);
    if (cb) return launch_cfg_t<SV_BF16, SV_F32>(A, R, k, stream);
    if (db) return launch_cfg_t<SV_F32, SV_BF16>(A, R, k, stream);
    return launch_cfg_t<SV_F32, SV_F32>(A, R, k, stream);
}

int32_t cfg_max_width() { return kCfgMaxW; }

}  // namespace sv
