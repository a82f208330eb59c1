// Classifier-free-guidance merge per RVQ codebook, then verification ("An
// Efficient vLLM-Based Inference Pipeline for Unified Audio Understanding and
// Generation", paired CFG co-scheduling: per codebook the conditional and
// unconditional logits are merged linearly with weight w; Figure 1 text: each
// codebook samples from its own partition of the vocabulary).  Sampling rules
// follow "speculative decoding for Omni models", section 2.
//
// cfg_rows_kernel  one CTA per (request, frame j, codebook s) row.  The row's
//                  codebook slice of cond and uncond is merged in fp32 as
//                  fmaf(w, c - u, u) into shared memory; the CTA takes the
//                  merged row's argmax, max and sum-exp at T, the draft row's
//                  max and sum-exp, TV = sum max(0, q - p), p and q at the
//                  drafted id, and the accept test (Philox row j * S + s).
// cfg_race_kernel  one CTA per (request, codebook): the first frame n with a
//                  rejected codebook, then for codebook s: its draft if its
//                  own test passed, else the residual race at frame n (or the
//                  bonus race at frame k), the merged row rebuilt from the
//                  inputs.  Codebook 0 also writes accept_len and status.
#include <algorithm>
#include <cfloat>
#include <climits>

#include "sv_device.cuh"
#include "sv_internal.h"

namespace sv {

namespace {

constexpr int kCfgThreads = 256;
constexpr float kLog2eC = 1.4426950408889634f;
constexpr int32_t kCfgMaxW = 16384;  // two fp32 rows of W in shared memory

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
    int esize;
    const char* dbase;
    int64_t dstride;
    int desize;
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

__device__ __forceinline__ float load_any(const char* p, int64_t e, int esize)
{
    if (esize == 2) return __uint_as_float(static_cast<uint32_t>(reinterpret_cast<const uint16_t*>(p)[e]) << 16);
    return reinterpret_cast<const float*>(p)[e];
}

// merged logit, fp32: d = c - u (one rounding), fmaf(w, d, u) (one rounding)
__device__ __forceinline__ float merge_one(float c, float u, float w)
{
    return __fmaf_rn(w, __fsub_rn(c, u), u);
}

template <int NT>
__device__ __forceinline__ float bsum(float v, float* sc)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    __syncthreads();
    if ((threadIdx.x & 31) == 0) sc[threadIdx.x >> 5] = v;
    __syncthreads();
    float t = 0.f;
    for (int i = 0; i < NT / 32; ++i) t += sc[i];
    return t;
}

template <int NT>
__device__ __forceinline__ float bmax(float v, float* sc)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    __syncthreads();
    if ((threadIdx.x & 31) == 0) sc[threadIdx.x >> 5] = v;
    __syncthreads();
    float t = -INFINITY;
    for (int i = 0; i < NT / 32; ++i) t = fmaxf(t, sc[i]);
    return t;
}

template <int NT>
__device__ __forceinline__ uint32_t bor(uint32_t v, uint32_t* sc)
{
    v = __reduce_or_sync(0xffffffffu, v);
    __syncthreads();
    if ((threadIdx.x & 31) == 0) sc[threadIdx.x >> 5] = v;
    __syncthreads();
    uint32_t t = 0;
    for (int i = 0; i < NT / 32; ++i) t |= sc[i];
    return t;
}

// (max value, lowest index) over the block
template <int NT>
__device__ __forceinline__ void bargmax(float& v, int32_t& x, float* sv, int32_t* sx)
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
    __syncthreads();
    if ((threadIdx.x & 31) == 0) {
        sv[threadIdx.x >> 5] = v;
        sx[threadIdx.x >> 5] = x;
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

// merge the codebook slice of one row into m[0..W); returns NaN / +inf flags
__device__ __forceinline__ uint32_t merge_row(const CfgArgs& A, int64_t row, int32_t s, float* m)
{
    const int32_t W = A.shape.W;
    const char* c = A.cbase + row * A.stride + static_cast<int64_t>(A.shape.data_off[s]) * A.esize;
    const char* u = A.ubase + row * A.stride + static_cast<int64_t>(A.shape.data_off[s]) * A.esize;
    uint32_t bad = 0;
    for (int32_t l = threadIdx.x; l < W; l += kCfgThreads) {
        const float v = merge_one(load_any(c, l, A.esize), load_any(u, l, A.esize), A.shape.w);
        if (v != v || v == INFINITY) bad = 1;
        m[l] = v != v ? -INFINITY : v;
    }
    return bad;
}

}  // namespace

__global__ void __launch_bounds__(kCfgThreads) cfg_rows_kernel(CfgArgs A)
{
    extern __shared__ __align__(16) float cfg_smem[];
    __shared__ float rf[kCfgThreads / 32];
    __shared__ int32_t ri[kCfgThreads / 32];
    __shared__ uint32_t ru[kCfgThreads / 32];
    pdl_launch_dependents();
    const int32_t S = A.shape.S, W = A.shape.W, k = A.k;
    const int64_t unit = blockIdx.x;  // ((r * (k + 1)) + j) * S + s
    const int32_t s = static_cast<int32_t>(unit % S);
    const int64_t rj = unit / S;
    const int32_t j = static_cast<int32_t>(rj % (k + 1));
    const int32_t r = static_cast<int32_t>(rj / (k + 1));
    const float T = A.temp[r];
    const bool sampling = T > 0.f && A.dbase != nullptr;
    const bool has_draft = sampling && j < k;
    const float c = sampling ? kLog2eC / T : 0.f;
    float* m = cfg_smem;
    float* y = cfg_smem + W;

    uint32_t bad = merge_row(A, unit, s, m);
    __syncthreads();
    float bv = -INFINITY;
    int32_t bx = INT32_MAX;
    float mx = -INFINITY;
    for (int32_t l = threadIdx.x; l < W; l += kCfgThreads) {
        const float v = m[l];
        if (v > bv) {
            bv = v;
            bx = l;
        }
    }
    bargmax<kCfgThreads>(bv, bx, rf, ri);
    mx = bv;
    CfgStat st{};
    st.amax = bx == INT32_MAX ? 0 : bx;
    st.m = -INFINITY;
    st.mq = -INFINITY;
    if (bv == -INFINITY) bad = 1;
    if (sampling) {
        const float M = mx * c;
        float acc = 0.f;
        if (M > -INFINITY && M < INFINITY)
            for (int32_t l = threadIdx.x; l < W; l += kCfgThreads) acc += exp2f(fmaf(m[l], c, -M));
        st.m = M;
        st.s = bsum<kCfgThreads>(acc, rf);
    }
    float tvv = NAN;
    if (has_draft) {
        const char* d = A.dbase + (((static_cast<int64_t>(r) * k + j) * S) + s) * A.dstride;
        float dm = -INFINITY;
        for (int32_t l = threadIdx.x; l < W; l += kCfgThreads) {
            float v = load_any(d, l, A.desize);
            if (v != v || v == INFINITY) bad = 1;
            v = v != v ? -INFINITY : v;
            y[l] = v;
            dm = fmaxf(dm, v);
        }
        dm = bmax<kCfgThreads>(dm, rf);
        const float Mq = dm * c;
        float acc = 0.f;
        if (Mq > -INFINITY && Mq < INFINITY)
            for (int32_t l = threadIdx.x; l < W; l += kCfgThreads) acc += exp2f(fmaf(y[l], c, -Mq));
        const float Sq = bsum<kCfgThreads>(acc, rf);
        st.mq = Mq;
        st.sq = Sq;
        if (dm == -INFINITY) bad = 1;
        // TV = sum max(0, q - p) (= 1/2 sum |p - q| since both sum to 1)
        const float invS = 1.f / st.s, invSq = 1.f / Sq;
        float a = 0.f;
        for (int32_t l = threadIdx.x; l < W; l += kCfgThreads) {
            const float p = exp2f(fmaf(m[l], c, -st.m)) * invS;
            const float q = exp2f(fmaf(y[l], c, -Mq)) * invSq;
            a += fmaxf(q - p, 0.f);
        }
        tvv = bsum<kCfgThreads>(a, rf);
        const int32_t xl = A.draft[(static_cast<int64_t>(r) * k + j) * S + s] - A.shape.id_base[s];
        int32_t acc_ok = 0;
        uint32_t off = 0;
        if (xl >= 0 && xl < W) {
            const float p = exp2f(fmaf(m[xl], c, -st.m)) * invS;
            const float q = exp2f(fmaf(y[xl], c, -Mq)) * invSq;
            if (q > 0.f) {
                const uint4 w = philox_block(philox_key(A.seeds[r]), 0u, static_cast<uint32_t>(j * S + s), kTagAccept);
                acc_ok = uniform_from_word(w.x) < __fdiv_rn(p, q) ? 1 : 0;
            } else {
                off = kCfgOffSupport;
            }
        }
        st.accept = acc_ok;
        st.flags |= off;
    }
    bad = bor<kCfgThreads>(bad, ru);
    if (bad) st.flags |= kCfgBad;
    if (threadIdx.x == 0) {
        A.stats[unit] = st;
        if (A.tv && j < k) A.tv[(static_cast<int64_t>(r) * k + j) * S + s] = tvv;
    }
}

__global__ void __launch_bounds__(kCfgThreads) cfg_race_kernel(CfgArgs A)
{
    pdl_wait_primary();
    extern __shared__ __align__(16) float cfg_smem[];
    __shared__ float rf[kCfgThreads / 32];
    __shared__ int32_t ri[kCfgThreads / 32];
    __shared__ uint32_t ru[kCfgThreads / 32];
    const int32_t S = A.shape.S, W = A.shape.W, k = A.k;
    const int32_t r = static_cast<int32_t>(blockIdx.x / S);
    const int32_t s = static_cast<int32_t>(blockIdx.x - static_cast<int64_t>(r) * S);
    const float T = A.temp[r];
    const CfgStat* st = A.stats + static_cast<int64_t>(r) * (k + 1) * S;
    const int32_t* d = A.draft + static_cast<int64_t>(r) * k * S;

    uint32_t fl = 0;
    for (int32_t i = threadIdx.x; i < (k + 1) * S; i += kCfgThreads) fl |= st[i].flags;
    fl = bor<kCfgThreads>(fl, ru);
    const bool bad = (fl & kCfgBad) != 0;
    const bool greedy = !(T > 0.f) || A.dbase == nullptr || bad;
    // first frame with a failing codebook
    int32_t n = k;
    for (int32_t j = 0; j < k && n == k; ++j) {
        bool all = true;
        for (int32_t q = 0; q < S; ++q) {
            const bool ok = greedy ? (d[j * S + q] - A.shape.id_base[q] == st[j * S + q].amax)
                                   : st[j * S + q].accept != 0;
            all = all && ok;
        }
        if (!all) n = j;
    }
    int32_t tok_local;
    uint32_t status = 0;
    const CfgStat& sn = st[n * S + s];
    if (greedy) {
        tok_local = sn.amax;
    } else if (n < k && sn.accept) {
        tok_local = d[n * S + s] - A.shape.id_base[s];
    } else {
        // race at frame n: residual max(0, p - q) or the bonus p
        const bool residual = n < k;
        const float c = kLog2eC / T;
        float* m = cfg_smem;
        float* y = cfg_smem + W;
        merge_row(A, (static_cast<int64_t>(r) * (k + 1) + n) * S + s, s, m);
        if (residual) {
            const char* dr = A.dbase + ((static_cast<int64_t>(r) * k + n) * S + s) * A.dstride;
            for (int32_t l = threadIdx.x; l < W; l += kCfgThreads) {
                float v = load_any(dr, l, A.desize);
                y[l] = v != v ? -INFINITY : v;
            }
        }
        __syncthreads();
        const float invS = 1.f / sn.s, invSq = residual ? 1.f / sn.sq : 0.f;
        const PhiloxKey key = philox_key(A.seeds[r]);
        const uint32_t row = static_cast<uint32_t>(n * S + s);
        const uint32_t tag = residual ? kTagResidual : kTagBonus;
        float best = INFINITY;
        int32_t bx = INT32_MAX;
        for (int32_t g = threadIdx.x; g < (W + 3) / 4; g += kCfgThreads) {
            const uint4 w4 = philox_block(key, static_cast<uint32_t>(g), row, tag);
            const uint32_t words[4] = {w4.x, w4.y, w4.z, w4.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int32_t l = 4 * g + e;
                if (l >= W) break;
                float wt = exp2f(fmaf(m[l], c, -sn.m)) * invS;
                if (residual) wt -= exp2f(fmaf(y[l], c, -sn.mq)) * invSq;
                if (!(wt > 0.f)) continue;
                const float v = one_minus_uniform_from_word(words[e]);
                if (!(v < best * wt)) continue;
                const float key2 = __fdiv_rn(-log1pf(-v), wt);
                if (key2 < best) {
                    best = key2;
                    bx = l;
                }
            }
        }
        float nb = -best;
        bargmax<kCfgThreads>(nb, bx, rf, ri);
        if (bx == INT32_MAX) {
            // no positive residual: draw from p with the same uniforms
            status |= SV_ST_RESIDUAL_ZERO;
            best = INFINITY;
            bx = INT32_MAX;
            for (int32_t g = threadIdx.x; g < (W + 3) / 4; g += kCfgThreads) {
                const uint4 w4 = philox_block(key, static_cast<uint32_t>(g), row, tag);
                const uint32_t words[4] = {w4.x, w4.y, w4.z, w4.w};
                for (int e = 0; e < 4; ++e) {
                    const int32_t l = 4 * g + e;
                    if (l >= W) break;
                    const float wt = exp2f(fmaf(m[l], c, -sn.m)) * invS;
                    if (!(wt > 0.f)) continue;
                    const float key2 = __fdiv_rn(-log1pf(-one_minus_uniform_from_word(words[e])), wt);
                    if (key2 < best) {
                        best = key2;
                        bx = l;
                    }
                }
            }
            nb = -best;
            bargmax<kCfgThreads>(nb, bx, rf, ri);
        }
        tok_local = bx == INT32_MAX ? 0 : bx;
        if (residual && (sn.flags & kCfgOffSupport)) status |= SV_ST_OFF_SUPPORT;
    }
    // tokens of codebook s for every frame
    int32_t* out = A.tokens + static_cast<int64_t>(r) * (k + 1) * S;
    for (int32_t j = threadIdx.x; j <= k; j += kCfgThreads)
        out[j * S + s] = j < n ? d[j * S + s] : (j == n ? A.shape.id_base[s] + tok_local : -1);
    if (greedy && A.tv) {
        for (int32_t j = threadIdx.x; j < k; j += kCfgThreads) A.tv[(static_cast<int64_t>(r) * k + j) * S + s] = NAN;
    }
    // request-level status: the OR over codebooks goes through an atomic on status
    uint32_t st_bits = status;
    for (int32_t j = threadIdx.x; j < k; j += kCfgThreads) {
        const int32_t l = d[j * S + s] - A.shape.id_base[s];
        if (l < 0 || l >= W) st_bits |= SV_ST_TOKEN_RANGE;
    }
    st_bits = bor<kCfgThreads>(st_bits, ru);
    if (s == 0) {
        if (bad) st_bits |= SV_ST_BAD_LOGITS;
        if (T < 0.f || T != T) st_bits |= SV_ST_BAD_TEMP;
    }
    if (threadIdx.x == 0) {
        if (s == 0) A.accept_len[r] = n;
        if (A.status) atomicOr(reinterpret_cast<unsigned int*>(A.status + r), st_bits);
    }
}

__global__ void cfg_clear_status_kernel(int32_t* status, int32_t R)
{
    const int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    if (i < R) status[i] = 0;
}

size_t cfg_workspace_bytes(int64_t R, int32_t k, int32_t S, int32_t W)
{
    (void)W;
    return static_cast<size_t>(R * (k + 1) * S) * sizeof(CfgStat) + 256;
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
    A.esize = cond.esize;
    A.dbase = draft_logits ? draft_logits->data : nullptr;
    A.dstride = draft_logits ? draft_logits->stride * draft_logits->esize : 0;
    A.desize = draft_logits ? draft_logits->esize : 4;
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
    const size_t smem = static_cast<size_t>(shape.W) * 2 * sizeof(float);
    cudaError_t e;
    for (const void* f : {reinterpret_cast<const void*>(cfg_rows_kernel), reinterpret_cast<const void*>(cfg_race_kernel)}) {
        e = cudaFuncSetAttribute(f, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
        if (e != cudaSuccess) return e;
    }
    if (status) {
        cfg_clear_status_kernel<<<static_cast<unsigned>((R + 255) / 256), 256, 0, stream>>>(status, R);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
    }
    const int64_t units = static_cast<int64_t>(R) * (k + 1) * shape.S;
    cfg_rows_kernel<<<static_cast<unsigned>(units), kCfgThreads, smem, stream>>>(A);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(static_cast<int64_t>(R) * shape.S));
    cfg.blockDim = dim3(kCfgThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, cfg_race_kernel, A);
}

int32_t cfg_max_width() { return kCfgMaxW; }

}  // namespace sv
