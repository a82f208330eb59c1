// Speculative sampling with a truncated draft vocabulary ("speculative
// decoding for Omni models", sections 2 and 4).
//
// The d2t plan (built once per draft model, or in the call):
//   d2t_plan_kernel    one CTA: a bitmap of the d2t image over the target
//                      vocabulary, per-word prefix counts, the support sorted
//                      by target id (xs[pos], js[pos]), the target id -> draft
//                      id map and the support rank at every chunk start.
//   d2t_group_kernel   one warp per 2048-id chunk: the chunk's support entries
//                      grouped for the shared-memory scatter of the row pass.
// Two kernels per call:
//   sample_rows_fast_kernel (target and draft rows of one dtype, bf16 or fp32,
//                      with a d2t map) or sample_rows_kernel (the general
//                      path): persistent CTAs, one (request, position)
//                      unit at a time.  The draft and target rows stream
//                      through bulk-copied shared-memory stages: max, sum-exp
//                      at T, argmax, NaN/inf flags and z at the support
//                      positions (G); the fast pass also records, per
//                      2048-id group, the lane holding the group's maximum.
//                      A second pass over G and the draft row gives TV over
//                      the full vocabulary, p(x_j), q(x_j) and the accept test
//                      u_j < p/q.
//   race_rows_kernel   the selected rows laid end to end in parts over one
//                      wave of CTAs: the accept-length scan, then on the one
//                      selected row (residual max(0, p - q) at the first
//                      rejection, or p at the bonus row) the exponential race
//                      over every id with Philox uniforms, pruned by a bound on
//                      the row's minimum key; then the commit.
// Temperature scaling works in log2 units: with c = log2(e) / T,
// p(x) = 2^(z_x c - M) / S where M = max_x z_x c and S = sum 2^(z c - M).
#include <algorithm>
#include <numeric>
#include <cfloat>
#include <climits>

#include "sv_device.cuh"
#include "sv_internal.h"

namespace sv {

namespace {

constexpr int kPlanThreads = 1024;
constexpr int32_t kChunkElems = 2048;  // ids per bulk-copied chunk of the fast path (4 KB bf16, 8 KB fp32)
constexpr int kRowThreads = 512;
constexpr uint32_t kStageBytes = 16384;
constexpr int kStages = 4;
constexpr int kRowHeader = 128;
constexpr uint32_t kSmemBudget = 220 * 1024;
constexpr int32_t kMaxPlanWords = 25600;  // d2t mode supports V <= 819,200

enum : uint32_t { kFlagAllNegInf = 8u, kFlagDraftBad = 16u, kFlagOffSupport = 32u };

struct D2tPlan {
    uint32_t* bitmap;  // [nw] support bits over target ids
    int32_t* prefix;   // [nw + 1] set bits before each word
    int32_t* xs;       // [Vd] support target ids, ascending
    int32_t* js;       // [Vd] the draft id of xs[pos]
    uint32_t* pairs;   // per chunk c of kChunkElems target ids, from c * 4096: its support entries
                       // (2 draft id << 16) | 2 (x & (kChunkElems - 1)) in bank-spread groups of 32
                       // (see d2t_group_kernel); empty slots hold (2 Vd << 16), a spare G slot
    int32_t* chunk;    // [V / kChunkElems + 2] support rank at every multiple of kChunkElems
    int32_t* pcount;   // [V / kChunkElems + 2] slots of every chunk in pairs (from c * kMaxGroups * 32)
    uint16_t* jmap;    // [V] draft id of every target id, 0xFFFF off the support
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
    // per request, reset by the row pass: the race's bound (fp32 bits), its packed (key, id)
    // minimum and the count of finished work items
    unsigned int* race_bound;
    unsigned long long* race_best;
    unsigned int* race_done;
    // per target row and group of the fast row pass (2048 bf16 or 1024 fp32 ids): the first
    // lane holding the group's largest logit, whose ids seed the race's bound; NULL without it
    uint8_t* clane;
    int32_t ngroups;
    char* gslots;        // global-memory Y / G buffers when they do not fit in shared memory
    int64_t gslot_bytes;
    int smem_mode;
};

__host__ __device__ inline int64_t align256(int64_t b) { return (b + 255) / 256 * 256; }

// The row passes take their units (request r, position j) in position-major order, L = j R + r;
// a persistent CTA takes L, L + grid, ...  Position-major order ends with the cheaper bonus rows
// (measured faster on the d2t workload, 85 against 93 us), and the host picks a grid coprime to
// 6, so that a CTA's requests change parity and residue mod 3 from unit to unit (batches that
// alternate greedy and sampled requests would otherwise split into greedy-only and sampled-only
// CTAs).
__device__ __forceinline__ void unit_rj(const SampleArgs& A, int64_t L, int32_t& r, int32_t& j)
{
    j = static_cast<int32_t>(L / A.R);
    r = static_cast<int32_t>(L - static_cast<int64_t>(j) * A.R);
}

// the race's per-request board for this call: the row pass resets it, the race
// kernel (launched after the row pass has completed) uses it
__device__ __forceinline__ void reset_race_board(const SampleArgs& A)
{
    for (int32_t r = blockIdx.x * blockDim.x + threadIdx.x; r < A.R; r += gridDim.x * blockDim.x) {
        A.race_bound[r] = 0x7F800000u;  // +inf
        A.race_best[r] = ~0ull;
        A.race_done[r] = 0u;
    }
}

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

// ---- block reductions (NT a multiple of 32, at most 1024 threads) ----
// Each warp reduces with shuffles, lane 0 leaves the warp's value in scratch,
// and every warp then reduces the NT / 32 values lane-parallel, so all threads
// return the same result.
template <int NT>
__device__ __forceinline__ float block_sum(float v, float* scratch)
{
    static_assert(NT % 32 == 0 && NT <= 1024, "block size");
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
    __syncthreads();
    if (lane == 0) scratch[w] = v;
    __syncthreads();
    float t = lane < NT / 32 ? scratch[lane] : 0.f;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) t += __shfl_xor_sync(0xffffffffu, t, o);
    return t;
}

template <int NT>
__device__ __forceinline__ float block_max(float v, float* scratch)
{
    static_assert(NT % 32 == 0 && NT <= 1024, "block size");
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
    __syncthreads();
    if (lane == 0) scratch[w] = v;
    __syncthreads();
    float t = lane < NT / 32 ? scratch[lane] : -INFINITY;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) t = fmaxf(t, __shfl_xor_sync(0xffffffffu, t, o));
    return t;
}

template <int NT>
__device__ __forceinline__ uint32_t block_or(uint32_t v, uint32_t* scratch)
{
    static_assert(NT % 32 == 0 && NT <= 1024, "block size");
    v = __reduce_or_sync(0xffffffffu, v);
    const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
    __syncthreads();
    if (lane == 0) scratch[w] = v;
    __syncthreads();
    return __reduce_or_sync(0xffffffffu, lane < NT / 32 ? scratch[lane] : 0u);
}

// (value, position) pairs: the larger value, the lower position among equal values
__device__ __forceinline__ void warp_argmax(float& v, int32_t& x)
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
}

// (value, first position) maximum over the block
template <int NT>
__device__ __forceinline__ void block_argmax(float& v, int32_t& x, float* sv, int32_t* sx)
{
    static_assert(NT % 32 == 0 && NT <= 1024, "block size");
    warp_argmax(v, x);
    const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
    __syncthreads();
    if (lane == 0) {
        sv[w] = v;
        sx[w] = x;
    }
    __syncthreads();
    v = lane < NT / 32 ? sv[lane] : -INFINITY;
    x = lane < NT / 32 ? sx[lane] : INT32_MAX;
    warp_argmax(v, x);
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
    for (int32_t x = tid; x < V; x += kPlanThreads) pl.jmap[x] = 0xFFFFu;
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
    const int32_t nch = (V + kChunkElems - 1) / kChunkElems;
    for (int32_t c = tid; c <= nch; c += kPlanThreads) {
        const int32_t x = min(V, c * kChunkElems);
        const int32_t w = x >> 5, b = x & 31;
        const int32_t rk = pref[w] + (b ? __popc(bits[w] & ((1u << b) - 1u)) : 0);
        pl.chunk[c] = rk;
    }
    __syncthreads();
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
        pl.jmap[x] = static_cast<uint16_t>(j);
        if (pos >= 0 && pos < Vd) {
            pl.xs[pos] = x;
            pl.js[pos] = j;
        }
    }
}

// ---------------------------------------------------------------------------
// support entries of every chunk, grouped for the row pass's scatter
// ---------------------------------------------------------------------------
// The row pass moves each support logit z[x] of a chunk (shared-memory stage)
// to G[draft id] (shared memory) with one 2-byte load and one 2-byte store per
// entry, 32 entries per warp instruction.  Entries are grouped here so that no
// bank is hit more than twice by one instruction, neither by the loads
// (bank (x & 2047) >> 1 mod 32) nor by the stores (bank j >> 1 mod 32): first
// fit over the chunk's entries in ascending x.  Group g of chunk c occupies
// slots c * kMaxGroups * 32 + 128 (g / 4) + 4 pos + (g % 4), pos = 0..31,
// which is the layout the row pass reads as one 16-byte word per lane for four
// groups; an entry is (2 j << 16) | 2 (x mod 2048), the byte offsets of the
// store and of the load (used by the row pass only, where j < 32768); slots
// without an entry hold (2 Vd << 16); pcount[c] = 32 x the groups rounded up to
// 4.  One CTA of one warp per chunk.
namespace {
constexpr int kMaxGroups = 128;  // 128 x 32 slots >= the 2048 entries a chunk can have
constexpr int kPadSlots = 512;   // slots of every chunk that hold an entry or padding (the row pass's registers)
constexpr int kBankCap = 2;
struct GroupState {
    uint8_t r[kMaxGroups][32];  // loads per bank
    uint8_t w[kMaxGroups][32];  // stores per bank
    uint8_t n[kMaxGroups];      // entries
};
}  // namespace

__global__ void __launch_bounds__(32) d2t_group_kernel(int32_t Vd, int32_t V, D2tPlan pl)
{
    extern __shared__ __align__(16) unsigned char group_smem[];
    GroupState& gs = *reinterpret_cast<GroupState*>(group_smem);
    uint16_t* slot_of = reinterpret_cast<uint16_t*>(group_smem + sizeof(GroupState));  // per entry
    const int lane = threadIdx.x;
    const int32_t c = blockIdx.x;
    for (int i = lane; i < kMaxGroups * 32 / 16; i += 32) {
        reinterpret_cast<uint4*>(gs.r)[i] = make_uint4(0u, 0u, 0u, 0u);
        reinterpret_cast<uint4*>(gs.w)[i] = make_uint4(0u, 0u, 0u, 0u);
    }
    for (int i = lane; i < kMaxGroups; i += 32) gs.n[i] = 0;
    __syncwarp();
    const int32_t p0 = min(max(pl.chunk[c], 0), Vd), p1 = min(max(pl.chunk[c + 1], p0), min(Vd, p0 + kChunkElems));
    int32_t ng = 0;
    for (int32_t p = p0; p < p1; ++p) {
        const int32_t x = pl.xs[p], j = pl.js[p];
        if (lane == 0) slot_of[p - p0] = 0xFFFFu;
        if (x < c * kChunkElems || x >= min(V, (c + 1) * kChunkElems) || j < 0 || j >= Vd) continue;
        const uint32_t xo = static_cast<uint32_t>(x - c * kChunkElems);
        const int rb = (xo >> 1) & 31, wb = (j >> 1) & 31;
        int g = -1;
        for (int s0 = 0; s0 < kMaxGroups && g < 0; s0 += 32) {  // first group with room
            const int gg = s0 + lane;
            const bool fit = gs.n[gg] < 32 && gs.r[gg][rb] < kBankCap && gs.w[gg][wb] < kBankCap;
            const unsigned m = __ballot_sync(0xffffffffu, fit);
            if (m) g = s0 + __ffs(m) - 1;
        }
        for (int s0 = 0; s0 < kMaxGroups && g < 0; s0 += 32) {  // no bank room: any group with room
            const unsigned m = __ballot_sync(0xffffffffu, gs.n[s0 + lane] < 32);
            if (m) g = s0 + __ffs(m) - 1;
        }
        if (lane == 0) {
            const int pos = gs.n[g];
            gs.n[g] = static_cast<uint8_t>(pos + 1);
            ++gs.r[g][rb];
            ++gs.w[g][wb];
            slot_of[p - p0] = static_cast<uint16_t>(128 * (g >> 2) + 4 * pos + (g & 3));
        }
        ng = max(ng, g + 1);
        __syncwarp();
    }
    const int32_t nslots = 32 * ((ng + 3) & ~3);
    uint32_t* out = pl.pairs + static_cast<int64_t>(c) * kMaxGroups * 32;
    for (int32_t i = lane; i < max(nslots, kPadSlots); i += 32) out[i] = static_cast<uint32_t>(2 * Vd) << 16;
    __syncwarp();
    for (int32_t p = p0 + lane; p < p1; p += 32) {
        const uint32_t sl = slot_of[p - p0];
        if (sl != 0xFFFFu)
            out[sl] = (static_cast<uint32_t>(2 * pl.js[p]) << 16) | static_cast<uint32_t>(2 * (pl.xs[p] - c * kChunkElems));
    }
    if (lane == 0) pl.pcount[c] = nslots;
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
    reset_race_board(A);

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
    for (int64_t L = blockIdx.x; L < units; L += gridDim.x) {
        int32_t r, j;
        unit_rj(A, L, r, j);
        const int64_t unit = static_cast<int64_t>(r) * (A.k + 1) + j;  // the row of (r, j)
        const float T = A.temp[r];
        const bool sampling = T > 0.f;
        const bool has_draft = sampling && j < A.k;
        const float c = sampling ? temp_scale(T) : 0.f;
        const char* trow = A.tbase + unit * A.tstride;
        const char* drow = has_draft ? A.dbase + (static_cast<int64_t>(r) * A.k + j) * A.dstride : nullptr;
        const int32_t xj = has_draft ? A.draft[static_cast<int64_t>(r) * A.k + j] : -1;

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
                            dl.s = dl.m == -INFINITY ? 0.f : dl.s * ex2(dl.m - mt);
                            dl.m = mt;
                        }
                        float acc = 0.f;
                        for (int e = 0; e < n; ++e) acc += ex2(fmaf(f[e], c, -dl.m));
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
                const float t = f * c;  // a candidate reference; the term itself as every other term
                if (t > -INFINITY) {
                    if (t > dl.m) {
                        dl.s = dl.m == -INFINITY ? 0.f : dl.s * ex2(dl.m - t);
                        dl.m = t;
                    }
                    dl.s += ex2(fmaf(f, c, -dl.m));
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
                            const float sc = tl.m == -INFINITY ? 0.f : ex2(tl.m - mt);
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
                                const float ex = ex2(fmaf(f[e], c, -tl.m));
                                acc += ex;
                                acc_off += ((bits >> e) & 1u) ? 0.f : ex;
                            }
                        } else {
                            for (int e = 0; e < n; ++e) acc += ex2(fmaf(f[e], c, -tl.m));
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
                        const float sc = tl.m == -INFINITY ? 0.f : ex2(tl.m - t);
                        tl.s *= sc;
                        tl.so *= sc;
                        tl.m = t;
                    }
                    const float ex = ex2(fmaf(f, c, -tl.m));
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
            const float sc = (tl.m == -INFINITY || M == -INFINITY) ? 0.f : ex2(tl.m - M);
            T2 = Lse{M, block_sum<kRowThreads>(tl.s * sc, red_f)};
            if (track_off) s_off = block_sum<kRowThreads>(tl.so * sc, red_f);
        }
        if (has_draft) {
            const float M = block_max<kRowThreads>(dl.m, red_f);
            const float part = dl.m == -INFINITY ? 0.f : dl.s * ex2(dl.m - M);
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
                const float pp = ex2(fmaf(z, c, -T2.m)) * invS;
                const float qq = ex2(fmaf(y, c, -D2.m)) * invSq;
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
                pj = in_range ? ex2(fmaf(zx, c, -T2.m)) * invS : 0.f;
                qj = 0.f;
                if (in_range && (A.identity || in_support(A.plan, xj))) {
                    const int32_t jd = A.identity ? xj : A.plan.js[support_rank(A.plan, xj)];
                    if (jd >= 0 && jd < A.Vd) {
                        float y = ld_elem<DD>(Y, jd);
                        y = y != y ? -INFINITY : y;
                        qj = ex2(fmaf(y, c, -D2.m)) * invSq;
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
// row pass, fast path: bf16 or fp32 target and draft rows, d2t vocabulary < 32768
// ---------------------------------------------------------------------------
// Two warp roles.  Each stream warp pulls its own share of a target row
// through a private ring of bulk-copied stages, one 2048-id chunk per stage:
// chunk s of a (request, position) unit belongs to stream warp (s + rot) % kStreamWarps,
// rot a hash of the request's seed and the position: a row's chunk count is rarely a
// multiple of the warp count, and varying which warps take the extra chunks evens the
// warps' shares over a CTA's units.  rot depends on the request's own inputs only, so
// the summation order, and with it every output bit of the row pass, does not depend on
// the request's place in the batch or on the launch geometry.  The warp's lane 0 refills a stage the moment
// it is read, with the warp's next chunk of this unit or of the CTA's next one.
// The support entries of a target chunk, packed (draft id, offset) pairs of the
// plan, come from L2 into registers while the chunk's maxima and exponentials
// are taken; the warp then scatters the support logits to G[draft id] from
// shared memory.
//
// The TV warps read the draft row of unit n themselves (its maximum, sum and
// flags) while the stream warps read the target row, then finish unit n (merge
// of the stream warps' records, the TV pass over G and the L2-resident draft
// row, p and q at the draft token, the accept test).  G, the warp records and
// the draft-token slots live in kNG buffers taken by unit in turn, handed over
// by two mbarriers per buffer (full: the stream warps are done with it; freed:
// the TV warps are).  bf16: two stages of 4 KB per stream warp and two buffers,
// so the TV warps finish unit n while the stream warps read unit n + 1.  fp32:
// one 8 KB stage per stream warp and one buffer (the 128 KB support image).
namespace {

constexpr int kStreamWarps = 12;                 // warps that stream the rows
constexpr int kTvWarps = 4;                      // warps that finish a unit: reductions, TV, accept test
constexpr int kFastWarps = kStreamWarps + kTvWarps;
constexpr int kFastThreads = 32 * kFastWarps;
constexpr int kTvThreads = 32 * kTvWarps;
constexpr int kPairRegs = 4;                     // uint4 groups of support entries per lane and chunk
static_assert(kPairRegs * 4 * 32 == kPadSlots, "the plan pads every chunk to the slots the registers hold");
constexpr int kFastHeader = 512;                 // the stage mbarriers, then the unit handoffs
constexpr int32_t kFastMaxVd = 32768;
constexpr int kHV = 8;                           // 16-byte vectors per lane taken together

template <int DT>
struct FastCfg {
    static constexpr int kElem = DT == SV_BF16 ? 2 : 4;
    static constexpr int kStages = DT == SV_BF16 ? 2 : 1;       // per stream warp
    static constexpr int kNG = DT == SV_BF16 ? 2 : 1;           // unit buffers
    static constexpr uint32_t kStageBytes = kChunkElems * kElem;
    static constexpr int kEPV = 16 / kElem;                     // elements per 16-byte vector
    static constexpr int kVPL = kChunkElems / kEPV / 32;        // vectors per lane and chunk
    static constexpr int kHalves = kVPL / kHV;
    static_assert((kStreamWarps * kStages + 2 * kNG) * 8 <= kFastHeader, "mbarriers fit the header");
};

__device__ __forceinline__ uint4 ninf_vec(int elem)
{
    return elem == 2 ? make_uint4(0xFF80FF80u, 0xFF80FF80u, 0xFF80FF80u, 0xFF80FF80u)
                     : make_uint4(0xFF800000u, 0xFF800000u, 0xFF800000u, 0xFF800000u);
}

// NaN-propagating maximum of one vector
template <int DT>
__device__ __forceinline__ float vec_max(uint4 q)
{
    if constexpr (DT == SV_BF16) {
        const uint32_t m = bmax2_nan(bmax2_nan(q.x, q.y), bmax2_nan(q.z, q.w));
        return fmax_nan(bf16_lo(m), bf16_hi(m));
    } else {
        return fmax_nan(fmax_nan(__uint_as_float(q.x), __uint_as_float(q.y)),
                        fmax_nan(__uint_as_float(q.z), __uint_as_float(q.w)));
    }
}

// NaN-propagating maximum of kHV vectors (bf16: one packed tree, widened once)
template <int DT>
__device__ __forceinline__ float group_max(const uint4 (&qv)[kHV])
{
    if constexpr (DT == SV_BF16) {
        uint32_t m2 = bmax2_nan(bmax2_nan(qv[0].x, qv[0].y), bmax2_nan(qv[0].z, qv[0].w));
#pragma unroll
        for (int e = 1; e < kHV; ++e)
            m2 = bmax2_nan(m2, bmax2_nan(bmax2_nan(qv[e].x, qv[e].y), bmax2_nan(qv[e].z, qv[e].w)));
        return fmax_nan(bf16_lo(m2), bf16_hi(m2));
    } else {
        float m = vec_max<DT>(qv[0]);
#pragma unroll
        for (int e = 1; e < kHV; ++e) m = fmax_nan(m, vec_max<DT>(qv[e]));
        return m;
    }
}

template <int DT>
__device__ __forceinline__ uint4 nan_to_ninf(uint4 q)
{
    if constexpr (DT == SV_BF16) {
        return make_uint4(bf16x2_nan_to_ninf(q.x), bf16x2_nan_to_ninf(q.y), bf16x2_nan_to_ninf(q.z),
                          bf16x2_nan_to_ninf(q.w));
    } else {
        auto f = [](uint32_t w) { return __uint_as_float(w) != __uint_as_float(w) ? 0xFF800000u : w; };
        return make_uint4(f(q.x), f(q.y), f(q.z), f(q.w));
    }
}

// the elements 2h and 2h + 1 of a vector as an fp32 pair (h < kEPV / 2), exact
template <int DT>
__device__ __forceinline__ unsigned long long vec_pair(uint4 q, int h)
{
    if constexpr (DT == SV_BF16) {
        return bf16x2_to_f32x2(h == 0 ? q.x : h == 1 ? q.y : h == 2 ? q.z : q.w);
    } else {
        return h == 0 ? pack2(__uint_as_float(q.x), __uint_as_float(q.y))
                      : pack2(__uint_as_float(q.z), __uint_as_float(q.w));
    }
}

// element t of a vector (t < kEPV)
template <int DT>
__device__ __forceinline__ float vec_elem(uint4 q, int t)
{
    const uint32_t w[4] = {q.x, q.y, q.z, q.w};
    if constexpr (DT == SV_BF16) return (t & 1) ? bf16_hi(w[t >> 1]) : bf16_lo(w[t >> 1]);
    else return __uint_as_float(w[t]);
}

// sum over the elements z of a vector of 2^(z c - m): packed fp32x2 arguments,
// independent MUFU operations, a tree of packed adds
template <int DT>
__device__ __forceinline__ float exp_sum_vec(uint4 q, unsigned long long c2, unsigned long long nm2)
{
    constexpr int kP = FastCfg<DT>::kEPV / 2;
    unsigned long long e[kP];
#pragma unroll
    for (int h = 0; h < kP; ++h) {
        float a0, a1;
        unpack2(fma2(vec_pair<DT>(q, h), c2, nm2), a0, a1);
        e[h] = pack2(ex2(a0), ex2(a1));
    }
    unsigned long long s2 = e[0];
#pragma unroll
    for (int h = 1; h < kP; ++h) s2 = add2(s2, e[h]);
    float lo, hi;
    unpack2(s2, lo, hi);
    return lo + hi;
}

// offset among the lane's kHV vectors (numbered lane + 32 e, kEPV elements each) of the
// first element equal to wm; every lane takes part
template <int DT>
__device__ __forceinline__ uint32_t first_max_offset(const uint4 (&qv)[kHV], float wm, int lane)
{
    constexpr int kEPV = FastCfg<DT>::kEPV;
    int ef = kHV;
#pragma unroll
    for (int e = kHV - 1; e >= 0; --e)
        if (vec_max<DT>(qv[e]) == wm) ef = e;
    uint32_t key = 0xFFFFFFFFu;
    if (ef < kHV) {
        uint4 v = qv[0];
#pragma unroll
        for (int e = 1; e < kHV; ++e)
            if (ef == e) v = qv[e];
        int first = kEPV - 1;
#pragma unroll
        for (int t = kEPV - 1; t >= 0; --t)
            if (vec_elem<DT>(v, t) == wm) first = t;
        key = static_cast<uint32_t>((lane + 32 * ef) * kEPV + first);
    }
    return __reduce_min_sync(0xffffffffu, key);
}

// shared-memory 32-bit accesses at 32-bit shared addresses
__device__ __forceinline__ uint32_t lds_u32(uint32_t addr)
{
    uint32_t v;
    asm("ld.shared.u32 %0, [%1];" : "=r"(v) : "r"(addr));
    return v;
}
__device__ __forceinline__ void sts_u32(uint32_t addr, uint32_t v)
{
    asm volatile("st.shared.u32 [%0], %1;" ::"r"(addr), "r"(v));
}

// G[draft id] = the chunk's logit at an entry's offset; a pair holds (2 draft id, 2 offset)
template <int DT>
__device__ __forceinline__ void scatter4(uint32_t zs_a, uint32_t g_a, uint4 pq)
{
    const uint32_t pe[4] = {pq.x, pq.y, pq.z, pq.w};
    uint32_t zv[4];
    if constexpr (DT == SV_BF16) {
#pragma unroll
        for (int e = 0; e < 4; ++e) zv[e] = lds_u16(zs_a + (pe[e] & 0xFFFFu));
#pragma unroll
        for (int e = 0; e < 4; ++e) sts_u16(g_a + (pe[e] >> 16), zv[e]);
    } else {
#pragma unroll
        for (int e = 0; e < 4; ++e) zv[e] = lds_u32(zs_a + 2 * (pe[e] & 0xFFFFu));
#pragma unroll
        for (int e = 0; e < 4; ++e) sts_u32(g_a + ((pe[e] >> 15) & ~3u), zv[e]);
    }
}

// element e of a row held in bytes (global or shared)
template <int DT>
__device__ __forceinline__ float row_elem(const void* row, int32_t e)
{
    if constexpr (DT == SV_BF16)
        return __uint_as_float(static_cast<uint32_t>(reinterpret_cast<const uint16_t*>(row)[e]) << 16);
    else
        return reinterpret_cast<const float*>(row)[e];
}

// this lane's register groups of the first kPadSlots (padded) support entries of a chunk
__device__ __forceinline__ void load_pairs(const SampleArgs& A, int32_t p0, int lane, uint4* pg)
{
#pragma unroll
    for (int t = 0; t < kPairRegs; ++t) pg[t] = ld_nc_v4(reinterpret_cast<const uint4*>(A.plan.pairs + p0 + 4 * (lane + 32 * t)));
}

// 16-byte read-only global load with an L2 cache policy
__device__ __forceinline__ uint4 ld_nc_v4_hint(const uint4* p, uint64_t pol)
{
    uint4 v;
    asm volatile("ld.global.nc.L2::cache_hint.v4.u32 {%0, %1, %2, %3}, [%4], %5;"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p), "l"(pol));
    return v;
}

// order this thread's generic-proxy accesses to shared memory before later
// bulk copies (async proxy) into the same bytes
__device__ __forceinline__ void fence_proxy_async_smem()
{
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

struct WarpRec {
    float bv;     // max of the target logits
    int32_t bx;   // its first id
    uint32_t tfl; // flags of the target row
    float tm;     // reference maximum (log2 units) of the target sum
    float ts;     // the sum
};

struct DraftRec {  // a TV warp's share of the draft row
    float m, s;    // reference maximum (log2 units) and sum
    uint32_t fl;   // flags
};

struct FastUnit {
    int32_t r, j;
    int64_t row;    // r (k + 1) + j, the unit's row of the statistics
    int32_t rot;    // chunk s goes to stream warp (s + rot) mod kStreamWarps
    bool sampling, has_draft;
    const char* trow;
    const char* drow;
    int32_t n;      // target chunks of the unit
};

__device__ __forceinline__ FastUnit fast_unit(const SampleArgs& A, int64_t unit, float T)
{
    FastUnit u;
    unit_rj(A, unit, u.r, u.j);  // R * (k + 1) < 2^31 (checked by the caller)
    u.row = static_cast<int64_t>(u.r) * (A.k + 1) + u.j;
    u.sampling = T > 0.f;
    u.has_draft = u.sampling && u.j < A.k;
    u.trow = A.tbase + u.row * A.tstride;
    u.drow = u.has_draft ? A.dbase + (static_cast<int64_t>(u.r) * A.k + u.j) * A.dstride : nullptr;
    u.n = (A.V + kChunkElems - 1) / kChunkElems;
    const uint64_t sd = A.seeds[u.r];
    u.rot = static_cast<int32_t>(((static_cast<uint32_t>(sd) ^ static_cast<uint32_t>(sd >> 32)) * 0x9E3779B1u >> 16) %
                                 kStreamWarps + u.j) % kStreamWarps;
    return u;
}

// the first chunk of stream warp w in a unit whose chunk s goes to warp (s + rot) mod W
__device__ __forceinline__ int32_t warp_first(int32_t rot, int w)
{
    return (w + kStreamWarps - rot) % kStreamWarps;
}

// chunks of a stream warp whose first chunk is q0 in a unit of n chunks: q0, q0 + W, ...
__device__ __forceinline__ int32_t warp_chunks(int32_t n, int32_t q0)
{
    return n > q0 ? (n - q0 + kStreamWarps - 1) / kStreamWarps : 0;
}

__device__ __forceinline__ float unit_temp(const SampleArgs& A, int64_t unit)
{
    return A.temp[static_cast<int32_t>(unit % A.R)];
}

// issue chunk q of unit u into `stage` (lane 0 only)
template <int DT>
__device__ __forceinline__ void issue_seq(const SampleArgs& A, const FastUnit& u, int32_t q, unsigned char* stage,
                                          uint64_t* bar, uint64_t pol_t)
{
    constexpr uint32_t kSB = FastCfg<DT>::kStageBytes;
    const uint32_t off = static_cast<uint32_t>(q) * kSB;
    const uint32_t nb = min(kSB, static_cast<uint32_t>(A.V) * FastCfg<DT>::kElem - off);
    mbar_arrive_expect_tx(bar, nb);
    bulk_copy_g2s(stage, u.trow + off, nb, bar, pol_t);
}

// The producer side of a warp's ring: the next chunk to issue (unit, index in
// the warp's list) and the temperature of the unit after it, loaded a unit
// ahead.  Every lane keeps the same copy; lane 0 issues.
struct Producer {
    int64_t unit;
    int32_t i, cnt, q0;
    FastUnit u;
    float t_next;
    uint32_t issued;
};

__device__ __forceinline__ void producer_enter(const SampleArgs& A, Producer& P, int w, int64_t units, float T)
{
    while (P.unit < units) {
        P.u = fast_unit(A, P.unit, T);
        P.q0 = warp_first(P.u.rot, w);
        P.cnt = warp_chunks(P.u.n, P.q0);
        P.i = 0;
        const int64_t nx = P.unit + gridDim.x;
        P.t_next = nx < units ? unit_temp(A, nx) : 0.f;
        if (P.cnt > 0) return;
        P.unit = nx;
        T = P.t_next;
    }
}

// issue the warp's next chunk if a stage is free
template <int DT>
__device__ __forceinline__ void producer_step(const SampleArgs& A, Producer& P, uint32_t consumed, int w, int lane,
                                              int64_t units, unsigned char* wst, uint64_t* wbar, uint64_t pol_t)
{
    constexpr uint32_t kS = FastCfg<DT>::kStages;
    if (P.unit >= units || P.issued - consumed >= kS) return;
    const uint32_t sidx = P.issued % kS;
    if (lane == 0) issue_seq<DT>(A, P.u, P.q0 + P.i * kStreamWarps, wst + sidx * FastCfg<DT>::kStageBytes, &wbar[sidx], pol_t);
    ++P.issued;
    if (++P.i == P.cnt) {
        P.unit += gridDim.x;
        producer_enter(A, P, w, units, P.t_next);
    }
}

}  // namespace

__device__ __forceinline__ void mbar_arrive(uint64_t* bar)
{
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}

// barrier 1 over the TV warps only
__device__ __forceinline__ void tv_bar_sync()
{
    asm volatile("bar.sync 1, %0;" ::"n"(kTvThreads) : "memory");
}

template <int DT>
__global__ void __launch_bounds__(kFastThreads, 1) sample_rows_fast_kernel(SampleArgs A)
{
    using Cfg = FastCfg<DT>;
    constexpr int kNG = Cfg::kNG, kS = Cfg::kStages, kE = Cfg::kElem, kEPV = Cfg::kEPV, kVPL = Cfg::kVPL;
    constexpr uint32_t kSB = Cfg::kStageBytes;
    extern __shared__ __align__(128) unsigned char smem[];
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem);  // [stream warp][stage]
    uint64_t* full = bars + kStreamWarps * kS;           // [buffer]: records, G and draft-token slots written
    uint64_t* freed = full + kNG;                         // [buffer]: the TV warps are done with them
    unsigned char* ring = smem + kFastHeader;
    const uint32_t gbytes = static_cast<uint32_t>(align256((static_cast<int64_t>(A.Vd) + 8) * kE));
    unsigned char* gbase = ring + kStreamWarps * kS * kSB;  // G of buffer 0 (then of buffer 1)
    int32_t* ctab = reinterpret_cast<int32_t*>(gbase + kNG * gbytes);
    __shared__ WarpRec wrec[kNG][kStreamWarps];
    __shared__ float zx_s[kNG];      // target logit of the draft token
    __shared__ int32_t jdx_s[kNG];   // its draft id (-1: off the support)
    __shared__ WarpRec merged;     // TV warps: the unit's merged record
    __shared__ DraftRec drec[kTvWarps];  // TV warps: their shares of the draft row
    __shared__ float wtv[kTvWarps];
    const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
    const int32_t nchunks_t = (A.V + kChunkElems - 1) / kChunkElems;

    pdl_wait_primary();  // a plan built in the same call must be complete
    pdl_launch_dependents();
    reset_race_board(A);
    if (tid == 0) {
        for (int i = 0; i < kS * kStreamWarps; ++i) mbar_init(&bars[i], 1);
        for (int b = 0; b < kNG; ++b) {
            mbar_init(&full[b], kStreamWarps * 32);
            mbar_init(&freed[b], kTvThreads);
        }
        fence_barrier_init();
    }
    if (tid < kNG) {
        zx_s[tid] = NAN;
        jdx_s[tid] = -1;
    }
    // a plan for other sizes, or built from a d2t with repeated / out-of-range ids, is not
    // trusted for shared-memory indexing (the race kernel reports SV_ST_BAD_D2T)
    const bool plan_ok = A.plan.header[0] == A.V && A.plan.header[1] == A.Vd && A.plan.header[2] == 0;
    for (int32_t c = tid; c <= nchunks_t; c += kFastThreads) ctab[c] = plan_ok && c < nchunks_t ? A.plan.pcount[c] : 0;
    __syncthreads();
    const int64_t units = static_cast<int64_t>(A.R) * (A.k + 1);

    if (w < kStreamWarps) {
        // ================= stream warps =================
        const uint64_t pol_t = l2_policy_evict_first();
        unsigned char* wst = ring + w * kS * kSB;  // this warp's stages
        uint64_t* wbar = bars + kS * w;
        uint32_t consumed = 0;  // chunks this warp has read so far (stage = consumed % kS)
        uint32_t timeout = 0;

        Producer P;
        P.unit = blockIdx.x;
        P.issued = 0;
        producer_enter(A, P, w, units, P.unit < units ? unit_temp(A, P.unit) : 0.f);
        for (int i = 0; i < kS; ++i)
            producer_step<DT>(A, P, consumed, w, lane, units, wst, wbar, pol_t);

        int64_t unit = blockIdx.x;
        float T = unit < units ? unit_temp(A, unit) : 0.f;
        for (uint32_t n = 0; unit < units; unit += gridDim.x, ++n) {
            const uint32_t b = n % kNG;
            const FastUnit u = fast_unit(A, unit, T);
            const int64_t un = unit + gridDim.x;
            const float T_next = un < units ? unit_temp(A, un) : 0.f;  // for the next unit, loaded early
            const float c = u.sampling ? temp_scale(T) : 0.f;
            const unsigned long long c2 = pack2(c, c);
            const int32_t xj = u.has_draft ? A.draft[static_cast<int64_t>(u.r) * A.k + u.j] : -1;
            const int32_t q0 = warp_first(u.rot, w);
            const int32_t nw_chunks = warp_chunks(u.n, q0);
            unsigned char* G = gbase + b * gbytes;
            // the TV warps are done with this buffer's previous unit
            if (n >= kNG && !timeout && !mbar_wait_bounded(&freed[b], ((n / kNG) + 1) & 1u)) timeout = 1;

            float tm = -INFINITY, ts = 0.f, bv = -INFINITY;
            int32_t bx = INT32_MAX;
            uint32_t tflags = 0;
            uint4 pg[kPairRegs];  // support entries of the target chunk pg_for (-1: none)
            int32_t pg_for = -1;
            for (int32_t i = 0; i < nw_chunks; ++i) {
                const uint32_t sidx = consumed % kS;
                if (!timeout && !mbar_wait_bounded(&wbar[sidx], (consumed / kS) & 1u)) timeout = 1;
                const unsigned char* st = wst + sidx * kSB;
                const uint4* vp = reinterpret_cast<const uint4*>(st);
                const int32_t q = q0 + i * kStreamWarps;
                const int32_t cidx = q;  // target chunk
                const uint32_t off = static_cast<uint32_t>(cidx) * kSB;
                const uint32_t nb = min(kSB, static_cast<uint32_t>(A.V) * kE - off);
                const int nv = static_cast<int>(nb / 16);
                const int32_t x0 = static_cast<int32_t>(off / kE);
                // support entries of a target chunk: this lane's groups of four packed pairs, from
                // L2 while the maxima and exponentials below run
                const bool scatter = u.has_draft && plan_ok;
                int32_t p0 = 0, p1 = 0;
                if (scatter) {
                    p0 = cidx * (kMaxGroups * 32);  // the chunk's slots: whole groups of four
                    p1 = p0 + ctab[cidx];
                    if (pg_for != cidx) load_pairs(A, p0, lane, pg);  // not prefetched
                }
                if (nv < kVPL * 32) {
                    // the row's last chunk: -inf beyond its end, so that every lane reads whole
                    // vectors; the fence orders these writes before the next bulk copy here
                    for (int v = nv + lane; v < kVPL * 32; v += 32) const_cast<uint4*>(vp)[v] = ninf_vec(kE);
                    fence_proxy_async_smem();
                    __syncwarp();
                }
#pragma unroll
                for (int h = 0; h < Cfg::kHalves; ++h) {
                    uint4 qv[kHV];
#pragma unroll
                    for (int e = 0; e < kHV; ++e) qv[e] = vp[lane + 32 * (kHV * h + e)];
                    // one NaN-propagating max tree over the lane's vectors
                    float lm = group_max<DT>(qv);
                    if (lm != lm) {  // rare: NaN logits read as -inf
                        tflags |= kFlagNaN;
                        lm = -INFINITY;
#pragma unroll
                        for (int e = 0; e < kHV; ++e) {
                            qv[e] = nan_to_ninf<DT>(qv[e]);
                            lm = fmaxf(lm, vec_max<DT>(qv[e]));
                        }
                    }
                    // Each lane sums its exponentials against its own maximum lr, so that they do
                    // not wait for the warp maximum; the lane's sum is then moved to the warp's
                    // running reference tm (the running maximum of z c) with one more exponential.
                    const float lr = lm > -INFINITY ? lm * c : 0.f;
                    float acc = 0.f;
                    if (u.sampling) {
                        const unsigned long long nl2 = pack2(-lr, -lr);
                        float ae[kHV];
#pragma unroll
                        for (int e = 0; e < kHV; ++e) ae[e] = exp_sum_vec<DT>(qv[e], c2, nl2);
                        acc = ((ae[0] + ae[1]) + (ae[2] + ae[3])) + ((ae[4] + ae[5]) + (ae[6] + ae[7]));
                    }
                    const float wm = warp_max(lm);
                    if (u.sampling && A.clane) {  // the first lane holding the group's maximum
                        const unsigned hold = __ballot_sync(0xffffffffu, lm == wm);
                        if (lane == 0)
                            A.clane[u.row * A.ngroups + cidx * Cfg::kHalves + h] = static_cast<uint8_t>(__ffs(hold) - 1);
                    }
                    if (wm > bv) {  // warp-uniform, rare after the first chunks
                        bx = x0 + kHV * 32 * kEPV * h + static_cast<int32_t>(first_max_offset<DT>(qv, wm, lane));
                        bv = wm;
                    }
                    if (u.sampling) {
                        const float mt = wm * c;
                        if (mt > tm) {  // warp-uniform
                            const float sc = tm == -INFINITY ? 0.f : ex2(tm - mt);
                            ts *= sc;
                            tm = mt;
                        }
                        ts += lm > -INFINITY ? acc * ex2(lr - tm) : 0.f;
                    }
                }
                if (scatter) {
                    // G[draft id] = z at the chunk offset for every entry of the lane's groups; a
                    // padding entry writes the spare slot G[Vd], which nothing reads
                    const uint32_t zs_a = smem_addr(st), g_a = smem_addr(G);
                    const bool here = xj >= x0 && xj < x0 + static_cast<int32_t>(nb / kE);
#pragma unroll
                    for (int t = 0; t < kPairRegs; ++t)  // every chunk has kPadSlots entries or padding
                        scatter4<DT>(zs_a, g_a, pg[t]);
                    // groups beyond this lane's registers (chunks denser than 512 entries)
                    for (int32_t g = p0 + 4 * 32 * kPairRegs + 4 * lane; g < p1; g += 4 * 32)
                        scatter4<DT>(zs_a, g_a, ld_nc_v4(reinterpret_cast<const uint4*>(A.plan.pairs + g)));
                    if (here) {  // the draft token: its logit and its draft id (from the registers)
                        const uint32_t xoff = static_cast<uint32_t>(xj - x0);
                        if (lane == 0) zx_s[b] = row_elem<DT>(st, static_cast<int32_t>(xoff));
#pragma unroll
                        for (int t = 0; t < kPairRegs; ++t) {
                            const uint32_t pe[4] = {pg[t].x, pg[t].y, pg[t].z, pg[t].w};
#pragma unroll
                            for (int e = 0; e < 4; ++e)
                                if ((pe[e] & 0xFFFFu) == 2 * xoff && static_cast<int32_t>(pe[e] >> 17) < A.Vd)
                                    jdx_s[b] = static_cast<int32_t>(pe[e] >> 17);
                        }
                        for (int32_t g = p0 + 4 * 32 * kPairRegs + lane; g < p1; g += 32) {  // beyond the registers
                            const uint32_t pe = A.plan.pairs[g];
                            if ((pe & 0xFFFFu) == 2 * xoff && static_cast<int32_t>(pe >> 17) < A.Vd)
                                jdx_s[b] = static_cast<int32_t>(pe >> 17);
                        }
                    }
                }
                {
                    // the support entries of this warp's next chunk, if it is a target chunk of this
                    // unit: in flight until that chunk's scatter
                    const int32_t qn = q + kStreamWarps;
                    pg_for = -1;
                    if (u.has_draft && plan_ok && qn < u.n) {
                        pg_for = qn;
                        load_pairs(A, pg_for * (kMaxGroups * 32), lane, pg);
                    }
                }
                // the stage is read: refill it with this warp's next chunk
                __syncwarp();
                ++consumed;
                if (lane == 0) fence_proxy_async_smem();
                producer_step<DT>(A, P, consumed, w, lane, units, wst, wbar, pol_t);
            }
            T = T_next;

            // this warp's record of the unit; every lane then signals the TV warps
            const uint32_t tfl = __reduce_or_sync(0xffffffffu, tflags | (timeout ? kFlagTimeout : 0u));
            float tsw = ts;
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) tsw += __shfl_xor_sync(0xffffffffu, tsw, o);
            if (lane == 0) wrec[b][w] = WarpRec{bv, bx, tfl, tm, tsw};
            mbar_arrive(&full[b]);
        }
        if (timeout && lane == 0) {
            // give this warp's copies that may still be in flight a bounded chance to land
            for (uint32_t g = consumed; g < P.issued; ++g)
                (void)mbar_wait_bounded(&wbar[g % kS], (g / kS) & 1u);
        }
        return;
    }

    // ================= TV warps =================
    const int ttid = tid - kStreamWarps * 32, tw = w - kStreamWarps;
    uint32_t tto = 0;  // a wait of these warps gave up
    uint64_t pol_keep;  // the draft rows stay in L2 between the two passes over them
    asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(pol_keep));
    int64_t unit = blockIdx.x;
    for (uint32_t n = 0; unit < units; unit += gridDim.x, ++n) {
        const uint32_t b = n % kNG;
        const float T = unit_temp(A, unit);
        const FastUnit u = fast_unit(A, unit, T);
        const float c = u.sampling ? temp_scale(T) : 0.f;
        const int32_t xj = u.has_draft ? A.draft[static_cast<int64_t>(u.r) * A.k + u.j] : -1;
        const uint64_t seed = (u.has_draft && ttid == 0) ? A.seeds[u.r] : 0ull;  // for the accept test
        const unsigned char* G = gbase + b * gbytes;

        const int32_t nv8 = u.has_draft ? A.Vd / kEPV : 0;  // draft-row vectors (Vd % 8 == 0 on this path)
        const uint4* yv = reinterpret_cast<const uint4*>(u.drow);
        {
            // ---- the draft row, read by these warps (from HBM, kept in L2 for the TV pass)
            // while the stream warps read the target row: maximum, sum at T, flags.  Each
            // thread sums a batch against the batch maximum and moves it to its running
            // reference. ----
            constexpr int kDraftBatch = kHV;
            const unsigned long long c2 = pack2(c, c);
            float rm = -INFINITY, rs = 0.f;
            uint32_t fl = 0;
#pragma unroll 1
            for (int32_t v0 = ttid; v0 < nv8; v0 += kTvThreads * kDraftBatch) {
                uint4 yb[kDraftBatch];
#pragma unroll
                for (int i = 0; i < kDraftBatch; ++i) {
                    const int32_t v = v0 + i * kTvThreads;
                    yb[i] = v < nv8 ? ld_nc_v4_hint(yv + v, pol_keep) : ninf_vec(kE);
                }
                float lm = group_max<DT>(yb);
                if (lm != lm) {  // rare: NaN logits, flagged (the request is verified greedily)
                    fl |= kFlagNaN;
                    lm = -INFINITY;
#pragma unroll
                    for (int i = 0; i < kDraftBatch; ++i) {
                        yb[i] = nan_to_ninf<DT>(yb[i]);
                        lm = fmaxf(lm, vec_max<DT>(yb[i]));
                    }
                }
                if (lm == INFINITY) fl |= kFlagPosInf;
                if (lm > -INFINITY && lm < INFINITY) {
                    const float lr = lm * c;
                    const unsigned long long nl2 = pack2(-lr, -lr);
                    float ae[kDraftBatch];
#pragma unroll
                    for (int i = 0; i < kDraftBatch; ++i) ae[i] = exp_sum_vec<DT>(yb[i], c2, nl2);
                    const float acc = ((ae[0] + ae[1]) + (ae[2] + ae[3])) + ((ae[4] + ae[5]) + (ae[6] + ae[7]));
                    if (lr > rm) {
                        rs *= rm == -INFINITY ? 0.f : ex2(rm - lr);
                        rm = lr;
                    }
                    rs += acc * ex2(lr - rm);
                }
            }
            float wm = rm;
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) wm = fmaxf(wm, __shfl_xor_sync(0xffffffffu, wm, o));
            float ws = rm > -INFINITY ? rs * ex2(rm - wm) : 0.f;
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) ws += __shfl_xor_sync(0xffffffffu, ws, o);
            fl = __reduce_or_sync(0xffffffffu, fl);
            if (lane == 0) drec[tw] = DraftRec{wm, ws, fl};
        }

        // the first batch of the TV pass's draft-row loads, in flight while the stream warps
        // finish the unit
        constexpr int kTvIter = (kFastMaxVd / kEPV + kTvThreads - 1) / kTvThreads;
        constexpr int kTvBatch = 8;  // draft-row loads in flight per thread
        uint4 yq[kTvBatch];
#pragma unroll
        for (int i = 0; i < kTvBatch; ++i) {
            const int32_t v = ttid + i * kTvThreads;
            if (v < nv8) yq[i] = ld_nc_v4(yv + v);
        }
        if (!tto && !mbar_wait_bounded(&full[b], (n / kNG) & 1u)) tto = 1;

        // ---- merge the stream warps' records: max, first argmax, reference maxima, sums ----
        if (tw == 0) {
            WarpRec rec = lane < kStreamWarps ? wrec[b][lane] : WarpRec{-INFINITY, INT32_MAX, 0u, -INFINITY, 0.f};
            float mbv = rec.bv, mtm = rec.tm;
            int32_t mbx = rec.bx;
            uint32_t ftl = rec.tfl;
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) {
                const float ov = __shfl_xor_sync(0xffffffffu, mbv, o);
                const int32_t ox = __shfl_xor_sync(0xffffffffu, mbx, o);
                if (ov > mbv || (ov == mbv && ox < mbx)) {
                    mbv = ov;
                    mbx = ox;
                }
                mtm = fmaxf(mtm, __shfl_xor_sync(0xffffffffu, mtm, o));
            }
            ftl = __reduce_or_sync(0xffffffffu, ftl);
            float st = (rec.tm > -INFINITY && mtm > -INFINITY) ? rec.ts * ex2(rec.tm - mtm) : 0.f;
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) st += __shfl_xor_sync(0xffffffffu, st, o);
            if (lane == 0) merged = WarpRec{mbv, mbx, ftl, mtm, st};
        }
        tv_bar_sync();  // merged and the TV warps' draft shares are written
        const float BV = merged.bv;
        float M = merged.tm;
        const float S = merged.ts;
        const uint32_t FLT = merged.tfl;
        float Mq = -INFINITY, Sq = 0.f;
        uint32_t FLD = 0;
#pragma unroll
        for (int i = 0; i < kTvWarps; ++i) {
            Mq = fmaxf(Mq, drec[i].m);
            FLD |= drec[i].fl;
        }
#pragma unroll
        for (int i = 0; i < kTvWarps; ++i)
            if (drec[i].m > -INFINITY) Sq += drec[i].s * ex2(drec[i].m - Mq);
        const int32_t amax = merged.bx == INT32_MAX ? 0 : merged.bx;
        if (!u.sampling) M = -INFINITY;
        if (!u.has_draft) Mq = -INFINITY;
        uint32_t flags = 0;
        if (FLT & kFlagNaN) flags |= kFlagNaN;
        if ((FLT & kFlagTimeout) || tto) flags |= kFlagTimeout;
        if (BV == INFINITY) flags |= kFlagPosInf;
        if (BV == -INFINITY) flags |= kFlagAllNegInf;
        if (u.has_draft && ((FLD & (kFlagNaN | kFlagPosInf)) || Mq == -INFINITY)) flags |= kFlagDraftBad;

        // ---- TV = sum over the support of max(0, q - p); p(x_j), q(x_j), accept ----
        // G (z at every draft id) and the L2-resident draft row, in draft-id order; every
        // thread issues a batch of draft-row loads before its arithmetic
        float tvv = NAN, pj = NAN, qj = NAN;
        int32_t acc = 0;
        const float invS = 1.f / S, invSq = 1.f / Sq;
        const int32_t jdx = jdx_s[b];
        if (u.has_draft) {
            const unsigned long long c2m = pack2(c, c), nM = pack2(-M, -M), nMq = pack2(-Mq, -Mq);
            const unsigned long long niS = pack2(-invS, -invS), iSq = pack2(invSq, invSq);
            const uint4* gv = reinterpret_cast<const uint4*>(G);
            float a = 0.f;
#pragma unroll 1
            for (int b0 = 0; b0 < kTvIter && b0 * kTvThreads < nv8; b0 += kTvBatch) {
#pragma unroll
                for (int i = 0; i < kTvBatch; ++i) {
                    const int32_t v = ttid + (b0 + i) * kTvThreads;
                    if (v >= nv8) break;
                    const uint4 yqi = yq[i];
                    const uint4 gq = gv[v];
                    float dv[kEPV];
#pragma unroll
                    for (int e = 0; e < kEPV / 2; ++e) {
                        // q and p of two ids at once: q - p = 2^(y c - Mq) / Sq - 2^(z c - M) / S
                        const unsigned long long ty = fma2(vec_pair<DT>(yqi, e), c2m, nMq);
                        const unsigned long long tz = fma2(vec_pair<DT>(gq, e), c2m, nM);
                        float y0, y1, z0, z1;
                        unpack2(ty, y0, y1);
                        unpack2(tz, z0, z1);
                        const unsigned long long eq = pack2(ex2(y0), ex2(y1));
                        const unsigned long long np = mul2(pack2(ex2(z0), ex2(z1)), niS);
                        unpack2(fma2(eq, iSq, np), dv[2 * e], dv[2 * e + 1]);
                    }
                    float pv[kEPV];
#pragma unroll
                    for (int e = 0; e < kEPV; ++e) pv[e] = fmaxf(dv[e], 0.f);
                    if constexpr (kEPV == 8)
                        a += ((pv[0] + pv[1]) + (pv[2] + pv[3])) + ((pv[4] + pv[5]) + (pv[6] + pv[7]));
                    else
                        a += (pv[0] + pv[1]) + (pv[2] + pv[3]);
                }
                // the next batch of draft-row loads
#pragma unroll
                for (int i = 0; i < kTvBatch; ++i) {
                    const int32_t v = ttid + (b0 + kTvBatch + i) * kTvThreads;
                    if (v < nv8) yq[i] = ld_nc_v4(yv + v);
                }
            }
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) a += __shfl_xor_sync(0xffffffffu, a, o);
            if (lane == 0) wtv[tw] = a;
        }
        tv_bar_sync();  // wtv is written; G, jdx and merged are no longer read
        if (ttid == 0) {
            const float zraw = zx_s[b];
            if (u.has_draft) {
                tvv = 0.f;
                for (int i = 0; i < kTvWarps; ++i) tvv += wtv[i];
                const bool in_range = xj >= 0 && xj < A.V;
                const float zx = zraw != zraw ? -INFINITY : zraw;
                pj = in_range ? ex2(fmaf(zx, c, -M)) * invS : 0.f;
                if (in_range && jdx >= 0) {  // q at the draft id, as the TV pass takes it
                    qj = ex2(fmaf(row_elem<DT>(u.drow, jdx), c, -Mq)) * invSq;
                } else {
                    qj = 0.f;
                }
                if (qj > 0.f) {
                    const uint4 w4 = philox_block(philox_key(seed), 0u, static_cast<uint32_t>(u.j), kTagAccept);
                    acc = uniform_from_word(w4.x) < __fdiv_rn(pj, qj) ? 1 : 0;
                } else if (in_range) {
                    flags |= kFlagOffSupport;
                }
            }
            RowStat rs;
            rs.m = M;
            rs.s = S;
            rs.mq = Mq;
            rs.sq = Sq;
            rs.zx = zraw;
            rs.p = pj;
            rs.q = qj;
            rs.amax = amax;
            rs.flags = flags;
            rs.accept = acc;
            A.stats[u.row] = rs;
            if (u.j < A.k) {
                const int64_t o = static_cast<int64_t>(u.r) * A.k + u.j;
                if (A.tv) A.tv[o] = tvv;
                if (A.pd) A.pd[o] = pj;
                if (A.qd) A.qd[o] = qj;
            }
            zx_s[b] = NAN;  // fresh draft-token slots for the buffer's next unit
            jdx_s[b] = -1;
        }
        mbar_arrive(&freed[b]);
    }
}
// ---------------------------------------------------------------------------
// scan + race + commit
// ---------------------------------------------------------------------------
// The correction token is a draw from w / sum(w), w = max(0, p - q) on the
// first rejected row (p on the bonus row), taken as one exponential race over
// the whole row: argmin over the ids with w_x > 0 of E_x / w_x, E_x = -ln u_x,
// u_x the Philox uniform of id x (counter (x >> 2, row, tag, 0), word x & 3).
//
// race_rows_kernel: the selected rows, each a fixed part cost followed by its
// ids, are cut into equal shares over one wave of CTAs (two per SM); a request
// with T <= 0 (verified greedily whatever its rows hold) takes only the cost of
// its decisions and commit.  The parts of a request meet in a packed 64-bit
// (key, id) minimum and the part that finishes last commits.  Warp 0 scans the accept flags for n.  Each warp
// streams 256-id steps of its part (the next step's loads in flight) and
// keeps a running minimum key; a bound B of the row's minimum key is shared
// through shared memory and, between the parts of a request, through the
// workspace, seeded with the exact keys of the largest logit of every group
// the part overlaps (lanes recorded by the fast row pass; else every lane's
// largest logit over the part).  An id can win only if
// 1 - u <= E <= B w (E = -ln u >= 1 - u) and 1 - u >= 2^-24, so it needs
// p B >= 2^-24: ids whose scaled logit t = z c - m is below
// lg2(S) - 24 - lg2(B) are skipped without an exponential, a Philox block is
// generated only when one of its four ids has B w >= 2^-24, and a logarithm
// is taken only when 1 - u <= B w.  Every test is widened by kRaceSlack
// against fp32 rounding, so no id that can win is skipped and the winner
// does not depend on which bound a warp saw.
namespace {

constexpr int kRaceThreads = 512;
constexpr int kRaceWarps = kRaceThreads / 32;
constexpr int32_t kRaceStep = 256;                // ids per warp step, eight per lane
// a part's fixed cost (decisions, seeds, setup) in ids of its race, measured on the sampling
// workload: parts are cut so that every CTA carries the same ids plus this cost per part
constexpr int64_t kRacePartIds = 16384;
constexpr int64_t kRaceGreedyIds = 2048;  // the same for a request verified greedily (T <= 0)
constexpr int64_t kRaceMinShare = 2LL * kRaceWarps * kRaceStep;  // at least two steps per warp
constexpr uint32_t kRaceSmemRow = 96 * 1024;      // draft rows up to this size are staged in shared memory
constexpr float kRaceSlack = 1.0f + 1.0f / 1024.0f;
constexpr float kRaceMinGap = 5.9604645e-8f;      // 2^-24: the smallest 1 - u
constexpr unsigned long long kNoKey = ~0ull;

// (key bits, id) packed so that the unsigned minimum is the lowest key, then the lowest id;
// keys are positive, so their bits order like the keys
__device__ __forceinline__ unsigned long long pack_key(float key, int32_t id)
{
    return (static_cast<unsigned long long>(__float_as_uint(key)) << 32) | static_cast<uint32_t>(id);
}

__device__ __forceinline__ unsigned long long warp_min_u64(unsigned long long v)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        const unsigned long long ov = __shfl_xor_sync(0xffffffffu, v, o);
        v = ov < v ? ov : v;
    }
    return v;
}

// the key E_x / w of an id from its uniform's complement 1 - u
__device__ __forceinline__ float race_key(float om, float w) { return __fdiv_rn(-log1pf(-om), w); }

__device__ __forceinline__ uint32_t word_of(uint4 w4, int e)
{
    return e == 0 ? w4.x : e == 1 ? w4.y : e == 2 ? w4.z : w4.w;
}

// the lowest scaled logit t = z c - m an id can have and still win against bound B
__device__ __forceinline__ float race_t_floor(float B, float S)
{
    if (!(B < INFINITY)) return -INFINITY;
    return __log2f(S) - 24.0f - __log2f(B * kRaceSlack) - 1e-3f;
}

// What a race over one row needs.
struct RaceRow {
    const char* trow;
    const char* drow;     // the draft row (residual weights only)
    const uint16_t* ysm;  // the draft row in shared memory (bf16), or NULL
    const float* ysmf;    // the draft row in shared memory (fp32), or NULL
    float c, m, S, invS, mq, invSq;
    PhiloxKey key;
    uint32_t row, tag;
    unsigned int* bound_g;  // the request's bound shared by the CTAs of its parts (fp32 bits), or NULL
};

// the largest of four target logits (NaN ignored), from their raw 16-byte words
template <int DT>
__device__ __forceinline__ float max4(const uint4* zq, int h)
{
    if constexpr (DT == SV_BF16) {
        const uint32_t a = h == 0 ? zq[0].x : zq[0].z, b = h == 0 ? zq[0].y : zq[0].w;
        uint32_t m;
        asm("max.bf16x2 %0, %1, %2;" : "=r"(m) : "r"(a), "r"(b));
        return fmaxf(bf16_lo(m), bf16_hi(m));
    } else {
        const uint4 q = zq[h];
        return fmaxf(fmaxf(__uint_as_float(q.x), __uint_as_float(q.y)), fmaxf(__uint_as_float(q.z), __uint_as_float(q.w)));
    }
}

// the raw words of the eight target logits of ids [x, x + 8) (-inf at and past x_end, plain loads
// at a ragged or unaligned end).  Read-only loads the compiler may batch and hoist.
template <int DT>
__device__ __forceinline__ void load_z8(const SampleArgs& A, const RaceRow& Rr, int32_t x, int32_t x_end, uint4* zq)
{
    constexpr int ZW = DT == SV_BF16 ? 1 : 2;
    if (x + 8 <= x_end && A.tbulk) {
#pragma unroll
        for (int h = 0; h < ZW; ++h)
            zq[h] = __ldg(reinterpret_cast<const uint4*>(Rr.trow + static_cast<int64_t>(x) * (2 * ZW)) + h);
        return;
    }
    uint32_t wv[4 * ZW];
#pragma unroll
    for (int e = 0; e < 8; ++e) {
        const bool ok = x + e < x_end;
        if constexpr (DT == SV_BF16) {
            const uint32_t h16 = ok ? __ldg(reinterpret_cast<const uint16_t*>(Rr.trow) + x + e) : 0xFF80u;
            if (e & 1) wv[e >> 1] |= h16 << 16;
            else wv[e >> 1] = h16;
        } else {
            wv[e] = ok ? __ldg(reinterpret_cast<const uint32_t*>(Rr.trow) + x + e) : 0xFF800000u;
        }
    }
#pragma unroll
    for (int h = 0; h < ZW; ++h) zq[h] = make_uint4(wv[4 * h], wv[4 * h + 1], wv[4 * h + 2], wv[4 * h + 3]);
}

template <int DT>
__device__ __forceinline__ float z_of(const uint4* zq, int e)
{
    if constexpr (DT == SV_BF16) {
        const uint32_t ww = (e >> 1) == 0 ? zq[0].x : (e >> 1) == 1 ? zq[0].y : (e >> 1) == 2 ? zq[0].z : zq[0].w;
        return (e & 1) ? bf16_hi(ww) : bf16_lo(ww);
    } else {
        const uint4 q = zq[e >> 2];
        const int t = e & 3;
        return __uint_as_float(t == 0 ? q.x : t == 1 ? q.y : t == 2 ? q.z : q.w);
    }
}

// where the residual weights read the draft row: the identity map (draft logit x of the draft
// row), the d2t map through a copy of the row in shared memory, or the d2t map from global memory
enum { kYIdentity = 0, kYShared = 1, kYGlobal = 2 };

// q at target id x (residual weights); jm is its draft id (0xFFFF: off the support).  The rows
// a race runs on hold no NaN (a request with one is verified greedily).
template <int DD, int YM>
__device__ __forceinline__ float q_at(const SampleArgs& A, const RaceRow& Rr, int32_t x, uint32_t jm)
{
    float v;
    if constexpr (YM == kYIdentity) {
        v = x < A.Vd ? ld_elem<DD>(Rr.drow, x) : -INFINITY;
    } else {
        const bool on = jm < static_cast<uint32_t>(A.Vd);
        const uint32_t j = on ? jm : 0u;
        if constexpr (YM == kYShared) {
            if constexpr (DD == SV_BF16) v = __uint_as_float(static_cast<uint32_t>(Rr.ysm[j]) << 16);
            else v = Rr.ysmf[j];
        } else {
            v = ld_elem<DD>(Rr.drow, j);
        }
        v = on ? v : -INFINITY;
    }
    return ex2(fmaf(v, Rr.c, -Rr.mq)) * Rr.invSq;
}

// the weight of id x: p, or max(0, p - q) with resid
template <int DT, int DD, int YM>
__device__ __forceinline__ float weight_at(const SampleArgs& A, const RaceRow& Rr, int32_t x, bool resid)
{
    const float z = ld_elem<DT>(Rr.trow, x);
    float w = ex2(fmaf(z, Rr.c, -Rr.m)) * Rr.invS;
    if (resid) {
        const uint32_t jm = YM == kYIdentity ? 0u : A.plan.jmap[x];
        w = fmaxf(w - q_at<DD, YM>(A, Rr, x, jm), 0.f);
    }
    return w;
}

// the key of id x with weight w; +inf when w is not positive
__device__ __forceinline__ float key_of(const RaceRow& Rr, int32_t x, float w)
{
    if (!(w > 0.f)) return INFINITY;
    const uint4 w4 = philox_block(Rr.key, static_cast<uint32_t>(x) >> 2, Rr.row, Rr.tag);
    return race_key(one_minus_uniform_from_word(word_of(w4, x & 3)), w);
}

// Pass 1 of the race over ids [x_lo, x_hi), one warp (steps warp, warp + nwarps, ...): every lane
// finds the id of its largest target logit (packed maxima, no exponential) and takes that id's
// exact key; the warp's smallest lowers the CTA's shared bound (fp32 bits in *bound_s).
template <int DT, int DD, int YM>
__device__ void race_seed_pass(const SampleArgs& A, const RaceRow& Rr, int32_t x_lo, int32_t x_hi, bool resid,
                               unsigned int* bound_s, int warp, int nwarps)
{
    constexpr int ZW = DT == SV_BF16 ? 1 : 2;
    constexpr int kBatch = 4;  // steps whose loads are in flight together
    const int lane = threadIdx.x & 31;
    float zb = -INFINITY;
    int32_t xb = -1;
    const int32_t step = kRaceStep * nwarps;
    for (int32_t x0 = x_lo + kRaceStep * warp; x0 < x_hi; x0 += kBatch * step) {
        uint4 zq[kBatch][ZW];
#pragma unroll
        for (int b = 0; b < kBatch; ++b) load_z8<DT>(A, Rr, x0 + b * step + 8 * lane, x_hi, zq[b]);
#pragma unroll
        for (int b = 0; b < kBatch; ++b) {
            const float m = fmaxf(max4<DT>(zq[b], 0), max4<DT>(zq[b], 1));
            if (m > zb) {  // ids ascend within the lane: the first of equal maxima
                zb = m;
                const int32_t x = x0 + b * step + 8 * lane;
#pragma unroll
                for (int e = 7; e >= 0; --e)
                    if (z_of<DT>(zq[b], e) == m) xb = x + e;
            }
        }
    }
    float kb = xb >= 0 ? key_of(Rr, xb, weight_at<DT, DD, YM>(A, Rr, xb, resid)) : INFINITY;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) kb = fminf(kb, __shfl_xor_sync(0xffffffffu, kb, o));
    if (lane == 0 && kb < INFINITY) {
        atomicMin(bound_s, __float_as_uint(kb));
        if (Rr.bound_g) atomicMin(Rr.bound_g, __float_as_uint(kb));
    }
}

// Pass 1 from the row pass's group records (fast row pass only): the groups that overlap the part,
// one per lane; each reads the eight 16-byte vectors of the lane that held its largest logit (the
// group may reach past the part: any id's key bounds the row's minimum) and takes the exact key
// of their first id of the largest value; the warp's smallest lowers the CTA's bound and the
// request's.
template <int DT, int DD, int YM>
__device__ void race_seed_groups(const SampleArgs& A, const RaceRow& Rr, int64_t srow, int32_t x_lo, int32_t x_hi,
                                 bool resid, unsigned int* bound_s, int warp, int nwarps)
{
    constexpr int kEPV = FastCfg<DT>::kEPV, kE = FastCfg<DT>::kElem;
    constexpr int32_t kG = kHV * 32 * kEPV;  // ids per group
    const int lane = threadIdx.x & 31;
    const int32_t g1 = (x_hi + kG - 1) / kG;
    float kb = INFINITY;
    for (int32_t g = x_lo / kG + 32 * warp + lane; g < g1; g += 32 * nwarps) {
        const int32_t L = A.clane[srow * A.ngroups + g];
        const int32_t xg = g * kG + kEPV * L;  // the lane's first id; its vectors follow every 32 kEPV ids
        uint4 v[kHV];
#pragma unroll
        for (int e = 0; e < kHV; ++e) {
            const int32_t x = xg + 32 * kEPV * e;
            v[e] = x < A.V ? __ldg(reinterpret_cast<const uint4*>(Rr.trow + static_cast<int64_t>(x) * kE)) : ninf_vec(kE);
        }
        float zb = -INFINITY;
        int32_t xb = -1;
#pragma unroll
        for (int e = 0; e < kHV; ++e)
#pragma unroll
            for (int t = 0; t < kEPV; ++t) {
                const float z = vec_elem<DT>(v[e], t);
                if (z > zb) {  // ids ascend: the first of equal maxima
                    zb = z;
                    xb = xg + 32 * kEPV * e + t;
                }
            }
        if (xb >= 0) kb = fminf(kb, key_of(Rr, xb, weight_at<DT, DD, YM>(A, Rr, xb, resid)));
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) kb = fminf(kb, __shfl_xor_sync(0xffffffffu, kb, o));
    if (lane == 0 && kb < INFINITY) {
        atomicMin(bound_s, __float_as_uint(kb));
        if (Rr.bound_g) atomicMin(Rr.bound_g, __float_as_uint(kb));
    }
}

// A queued block of four ids of pass 2: its first id and its raw target logits.
struct RaceQ {
    int32_t x[2 * 32];
    uint4 z[2 * 32];   // bf16: the first 8 bytes; fp32: all 16
};

// the full test of one queued block: weights (the block's draft ids read here, for the blocks
// that reach the queue only), the Philox block when one of its ids can win, keys where
// 1 - u <= B w (w = 0 never passes); updates the lane's running minimum (blocks reach a lane out
// of id order, so equal keys compare ids)
template <int DT, int DD, int YM>
__device__ __forceinline__ void race_block(const SampleArgs& A, const RaceRow& Rr, bool resid, int32_t x,
                                           uint4 zq, float tfl, float bs, float& best, int32_t& bx)
{
    uint2 jq = make_uint2(0u, 0u);  // four 16-bit draft ids (x is a multiple of four)
    if constexpr (YM != kYIdentity) {
        if (resid) jq = __ldg(reinterpret_cast<const uint2*>(A.plan.jmap + x));
    }
    float w[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
        float z;
        if constexpr (DT == SV_BF16) {
            const uint32_t ww = e < 2 ? zq.x : zq.y;
            z = (e & 1) ? bf16_hi(ww) : bf16_lo(ww);
        } else {
            z = __uint_as_float(e == 0 ? zq.x : e == 1 ? zq.y : e == 2 ? zq.z : zq.w);
        }
        const float t = fmaf(z, Rr.c, -Rr.m);
        w[e] = t >= tfl ? ex2(t) * Rr.invS : 0.f;
    }
    if (resid) {
        const uint32_t jm[4] = {jq.x & 0xFFFFu, jq.x >> 16, jq.y & 0xFFFFu, jq.y >> 16};
#pragma unroll
        for (int e = 0; e < 4; ++e) w[e] = fmaxf(w[e] - q_at<DD, YM>(A, Rr, x + e, jm[e]), 0.f);
    }
    const float wmax = fmaxf(fmaxf(w[0], w[1]), fmaxf(w[2], w[3]));
    if (!(wmax * bs >= kRaceMinGap)) return;
    const uint4 w4 = philox_block(Rr.key, static_cast<uint32_t>(x) >> 2, Rr.row, Rr.tag);
#pragma unroll
    for (int e = 0; e < 4; ++e) {
        const float om = one_minus_uniform_from_word(word_of(w4, e));
        if (om <= w[e] * bs) {  // rare
            const float kx = race_key(om, w[e]);
            if (kx < best || (kx == best && x + e < bx)) {
                best = kx;
                bx = x + e;
            }
        }
    }
}

// Pass 2: the race over ids [x_lo, x_hi) by one warp, against the shared bound (refreshed after every
// step); returns the warp's packed (key, id) minimum to every lane.  Each lane tests its two blocks
// of four ids per step on their largest raw logit alone; the blocks that pass go to the warp's queue in shared memory,
// which the warp works off 32 blocks at a time, one per lane, so that the exponentials and the
// Philox rounds run with every lane busy.
template <int DT, int DD, int YM>
__device__ unsigned long long race_pass(const SampleArgs& A, const RaceRow& Rr, int32_t x_lo, int32_t x_hi,
                                        bool resid, unsigned int* bound_s, RaceQ& q, int warp, int nwarps)
{
    const int lane = threadIdx.x & 31;
    const unsigned lt = (1u << lane) - 1u;
    float best = INFINITY;  // this lane's running minimum and its id
    int32_t bx = INT32_MAX;
    float B = __uint_as_float(*reinterpret_cast<volatile unsigned int*>(bound_s));
    float tfl = race_t_floor(B, Rr.S);
    float zfl = tfl > -INFINITY ? (tfl + Rr.m) / Rr.c : -INFINITY;  // the same floor on raw logits
    uint32_t qh = 0, qn = 0;  // the queue's head and length (warp-uniform)
    constexpr int ZW = DT == SV_BF16 ? 1 : 2;
    const int32_t step = kRaceStep * nwarps;
    // a step's target logits are loaded while the step before it is tested
    uint4 zn[ZW];
    load_z8<DT>(A, Rr, x_lo + kRaceStep * warp + 8 * lane, x_hi, zn);
    for (int32_t xs = x_lo + kRaceStep * warp; xs < x_hi; xs += step) {
        uint4 zq[ZW];
#pragma unroll
        for (int i = 0; i < ZW; ++i) zq[i] = zn[i];
        if (xs + step < x_hi) load_z8<DT>(A, Rr, xs + step + 8 * lane, x_hi, zn);
        // the bound the request's other parts have reached (read now, used at the step's end)
        const unsigned int gb = Rr.bound_g ? *reinterpret_cast<volatile unsigned int*>(Rr.bound_g) : 0x7F800000u;
        const int32_t x = xs + 8 * lane;
        // the blocks that can hold a winner join the queue (at most 31 + 32 entries at a time)
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const bool pass = max4<DT>(zq, h) >= zfl;  // false past the end (-inf)
            const unsigned bal = __ballot_sync(0xffffffffu, pass);
            if (pass) {
                const uint32_t s = (qh + qn + __popc(bal & lt)) & 63u;
                q.x[s] = x + 4 * h;
                if constexpr (DT == SV_BF16)
                    q.z[s] = h == 0 ? make_uint4(zq[0].x, zq[0].y, 0u, 0u) : make_uint4(zq[0].z, zq[0].w, 0u, 0u);
                else
                    q.z[s] = zq[h];
            }
            qn += __popc(bal);
            __syncwarp();
            if (qn >= 32) {  // warp-uniform
                const uint32_t s = (qh + lane) & 63u;
                race_block<DT, DD, YM>(A, Rr, resid, q.x[s], q.z[s], tfl, B * kRaceSlack, best, bx);
                qh = (qh + 32) & 63u;
                qn -= 32;
                __syncwarp();
            }
        }
        // a lower key lowers this lane's bound and the shared ones; the shared bounds lower this lane's
        const float sb = fminf(__uint_as_float(*reinterpret_cast<volatile unsigned int*>(bound_s)), __uint_as_float(gb));
        if (best < sb) {
            atomicMin(bound_s, __float_as_uint(best));
            if (Rr.bound_g) atomicMin(Rr.bound_g, __float_as_uint(best));
        }
        const float nb = fminf(fminf(best, sb), B);
        if (nb < B) {
            B = nb;
            tfl = race_t_floor(B, Rr.S);
            zfl = tfl > -INFINITY ? (tfl + Rr.m) / Rr.c : -INFINITY;
        }
    }
    if (lane < qn) {  // the queue's rest
        const uint32_t s = (qh + lane) & 63u;
        race_block<DT, DD, YM>(A, Rr, resid, q.x[s], q.z[s], tfl, B * kRaceSlack, best, bx);
    }
    __syncwarp();
    return warp_min_u64(bx == INT32_MAX ? kNoKey : pack_key(best, bx));
}

// a request's length on the partition line: its part cost, then its row's ids padded to whole
// steps; a request with T <= 0 (NaN included) is verified greedily and races nothing
__device__ __forceinline__ int64_t race_line_len(float T, int64_t Vp)
{
    return T > 0.f ? kRacePartIds + Vp : kRaceGreedyIds;
}

}  // namespace

template <int DT, int DD, int YM>
__global__ void __launch_bounds__(kRaceThreads, 2) race_rows_kernel(SampleArgs A)
{
    extern __shared__ __align__(16) unsigned char ysm_raw[];  // the selected draft row (d2t residual rows)
    __shared__ int32_t n_s, last_s;
    __shared__ uint32_t fl_s;
    __shared__ unsigned int bound_s;
    __shared__ unsigned long long wbest_s[kRaceWarps];
    __shared__ unsigned long long best_s;
    __shared__ uint32_t red_u[kRaceWarps];
    __shared__ long long line_s[kRaceWarps];  // the partition line's per-warp sums, then their prefix
    __shared__ long long p0_s;                // where the request holding this CTA's first position starts
    __shared__ int32_t r0_s;                  // that request
    __shared__ RaceQ queue_s[kRaceWarps];     // every warp's queue of blocks for pass 2
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int32_t k = A.k;
    const int64_t Vp = (static_cast<int64_t>(A.V) + kRaceStep - 1) / kRaceStep * kRaceStep;
    // ---- the partition line, from the inputs alone (taken while the row pass ends): thread t sums
    // the lengths of a contiguous run of requests, a block scan gives every run's start ----
    const int32_t per = (A.R + kRaceThreads - 1) / kRaceThreads;
    const int32_t ra = min(A.R, tid * per), rb = min(A.R, ra + per);
    long long run = 0;
    for (int32_t r = ra; r < rb; ++r) run += race_line_len(A.temp[r], Vp);
    long long incl = run;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const long long v = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += v;
    }
    if (lane == 31) line_s[warp] = incl;
    __syncthreads();
    if (warp == 0) {
        long long v = lane < kRaceWarps ? line_s[lane] : 0;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const long long u = __shfl_up_sync(0xffffffffu, v, o);
            if (lane >= o) v += u;
        }
        if (lane < kRaceWarps) line_s[lane] = v;
    }
    __syncthreads();
    const int64_t L = line_s[kRaceWarps - 1];
    // equal shares over the grid, each at least two steps per warp and a whole number of steps
    int64_t share = max(kRaceMinShare, (L + gridDim.x - 1) / gridDim.x);
    share = (share + kRaceStep - 1) / kRaceStep * kRaceStep;
    const int64_t g_lo = static_cast<int64_t>(blockIdx.x) * share, g_hi = min(L, g_lo + share);
    if (g_lo >= L) return;  // nothing on the line for this CTA (block-uniform)
    {
        int64_t pos = incl - run + (warp > 0 ? line_s[warp - 1] : 0);  // where this thread's run starts
        for (int32_t r = ra; r < rb; ++r) {
            const int64_t len = race_line_len(A.temp[r], Vp);
            if (pos <= g_lo && g_lo < pos + len) {
                r0_s = r;
                p0_s = pos;
            }
            pos += len;
        }
    }
    __syncthreads();
    pdl_wait_primary();
    int64_t pos = p0_s;
    for (int32_t r = r0_s; r < A.R && pos < g_hi; ++r) {
        const float T = A.temp[r];
        const int64_t len = race_line_len(T, Vp);
        const int64_t start = pos;
        pos += len;
        int32_t x_lo = 0, x_hi = 0, parts = 1;
        if (T > 0.f) {
            const int64_t ids0 = start + kRacePartIds;  // where the row's ids start
            x_lo = static_cast<int32_t>(g_lo > ids0 ? g_lo - ids0 : 0);
            x_hi = static_cast<int32_t>(min(Vp, g_hi - ids0));
            if (x_hi <= x_lo) continue;  // this share holds only the row's part cost (block-uniform)
            // the CTAs that share request r's row
            parts = static_cast<int32_t>((ids0 + Vp - 1) / share - ids0 / share + 1);
        } else if (start < g_lo) {
            continue;  // a greedily verified request is committed by the CTA holding its start
        }
        const bool first = x_lo == 0;  // this CTA holds the row's first part (commits a greedy request)
        const RowStat* st = A.stats + static_cast<int64_t>(r) * (k + 1);
        const int32_t* d = A.draft + static_cast<int64_t>(r) * k;
        // ---- the request's decisions (warp 0, ballots) ----
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
                n_s = n;
                fl_s = fl;
                bound_s = 0x7F800000u;  // +inf
            }
        }
        __syncthreads();
        const int32_t n = n_s;
        const uint32_t fl = fl_s;
        const bool bad_rows = (fl & (kFlagNaN | kFlagPosInf | kFlagAllNegInf | kFlagDraftBad)) != 0;
        const bool greedy = !(T > 0.f) || bad_rows;
        const bool residual = n < k;
        uint32_t status = 0;
        int32_t token = -1;
        bool commit = true;
        if (greedy) {
            commit = first;  // block-uniform
            token = st[n].amax;
        } else {
            const RowStat rs = st[n];
            RaceRow Rr;
            Rr.trow = A.tbase + (static_cast<int64_t>(r) * (k + 1) + n) * A.tstride;
            Rr.drow = residual ? A.dbase + (static_cast<int64_t>(r) * k + n) * A.dstride : nullptr;
            Rr.ysm = nullptr;
            Rr.ysmf = nullptr;
            Rr.c = temp_scale(T);
            Rr.m = rs.m;
            Rr.S = rs.s;
            Rr.invS = 1.f / rs.s;
            Rr.mq = rs.mq;
            Rr.invSq = residual ? 1.f / rs.sq : 0.f;
            Rr.key = philox_key(A.seeds[r]);
            Rr.row = static_cast<uint32_t>(n);
            Rr.tag = residual ? kTagResidual : kTagBonus;
            Rr.bound_g = parts > 1 ? A.race_bound + r : nullptr;
            constexpr int ED = DD == SV_BF16 ? 2 : 4;
            // the selected draft row into shared memory, for the d2t gathers of the residual weights
            const uint32_t ybytes = static_cast<uint32_t>(A.Vd) * ED;
            if (YM == kYShared && residual) {  // the launch checked that the row fits, aligned
                const uint4* src = reinterpret_cast<const uint4*>(Rr.drow);
                uint4* dst = reinterpret_cast<uint4*>(ysm_raw);
                constexpr int kY = 4;  // loads in flight per thread
                for (uint32_t i0 = tid; i0 < ybytes / 16; i0 += kY * kRaceThreads) {
                    uint4 v[kY];
#pragma unroll
                    for (int b = 0; b < kY; ++b)
                        if (i0 + b * kRaceThreads < ybytes / 16) v[b] = __ldg(src + i0 + b * kRaceThreads);
#pragma unroll
                    for (int b = 0; b < kY; ++b)
                        if (i0 + b * kRaceThreads < ybytes / 16) dst[i0 + b * kRaceThreads] = v[b];
                }
                if (DD == SV_BF16) Rr.ysm = reinterpret_cast<const uint16_t*>(ysm_raw);
                else Rr.ysmf = reinterpret_cast<const float*>(ysm_raw);
            }
            __syncthreads();
            const int32_t xe = min(x_hi, A.V);
            // pass 1 sets the bound from the keys of the groups' largest logits (the lanes the fast
            // row pass recorded; else from every lane's largest logit over the part); pass 2 is
            // the pruned race
            if (A.clane) {
                if (tid == 0 && A.tbulk) {  // the part's ids into L2 while the seeds are taken
                    constexpr int ET = DT == SV_BF16 ? 2 : 4;
                    for (int32_t x = x_lo; x < xe; x += 16384) {
                        const uint32_t pb = static_cast<uint32_t>((min(xe, x + 16384) - x) * ET) & ~15u;
                        const char* pa = Rr.trow + static_cast<int64_t>(x) * ET;
                        if (pb) asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(pa), "r"(pb) : "memory");
                    }
                }
                race_seed_groups<DT, DD, YM>(A, Rr, static_cast<int64_t>(r) * (k + 1) + n, x_lo, xe, residual,
                                             &bound_s, warp, kRaceWarps);
            } else {
                race_seed_pass<DT, DD, YM>(A, Rr, x_lo, xe, residual, &bound_s, warp, kRaceWarps);
            }
            __syncthreads();
            unsigned long long mine =
                race_pass<DT, DD, YM>(A, Rr, x_lo, xe, residual, &bound_s, queue_s[warp], warp, kRaceWarps);
            if (lane == 0) wbest_s[warp] = mine;
            __syncthreads();
            if (tid == 0) {
                unsigned long long b = kNoKey;
                for (int i = 0; i < kRaceWarps; ++i) b = wbest_s[i] < b ? wbest_s[i] : b;
                last_s = 1;
                if (parts > 1) {
                    if (b != kNoKey) atomicMin(A.race_best + r, b);
                    __threadfence();
                    last_s = atomicAdd(A.race_done + r, 1u) == static_cast<unsigned int>(parts - 1);
                    if (last_s) {
                        __threadfence();
                        b = atomicOr(A.race_best + r, 0ull);
                    }
                }
                best_s = b;
            }
            __syncthreads();
            commit = last_s != 0;  // block-uniform
            unsigned long long best = best_s;
            if (commit && best == kNoKey && residual) {
                // no residual mass anywhere: the correction is drawn from p (same row and tag)
                status |= SV_ST_RESIDUAL_ZERO;
                __syncthreads();
                if (tid == 0) bound_s = 0x7F800000u;
                __syncthreads();
                Rr.bound_g = nullptr;  // the bound of the residual race says nothing about p's
                race_seed_pass<DT, DD, YM>(A, Rr, 0, A.V, false, &bound_s, warp, kRaceWarps);
                __syncthreads();
                mine = race_pass<DT, DD, YM>(A, Rr, 0, A.V, false, &bound_s, queue_s[warp], warp, kRaceWarps);
                if (lane == 0) wbest_s[warp] = mine;
                __syncthreads();
                for (int i = 0; i < kRaceWarps; ++i) best = wbest_s[i] < best ? wbest_s[i] : best;
            }
            token = best == kNoKey ? 0 : static_cast<int32_t>(best & 0xFFFFFFFFu);
            if (residual && (rs.flags & kFlagOffSupport)) status |= SV_ST_OFF_SUPPORT;
        }
        if (commit) {
            // ---- commit (one CTA per request) ----
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
            status = block_or<kRaceThreads>(status, red_u);
            if (tid == 0) {
                A.accept_len[r] = n;
                if (A.status) A.status[r] = static_cast<int32_t>(status);
            }
        }
        __syncthreads();  // the shared state is written again by the next part
    }
}

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------
namespace {

struct PlanLayout {
    int64_t header, bitmap, prefix, xs, js, pairs, chunk, pcount, jmap, total;
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
    const int64_t nch = (static_cast<int64_t>(V) + kChunkElems - 1) / kChunkElems;
    L.pairs = take(nch * kMaxGroups * 32 * 4);
    L.chunk = take((static_cast<int64_t>(V) / kChunkElems + 2) * 4);
    L.pcount = take((static_cast<int64_t>(V) / kChunkElems + 2) * 4);
    L.jmap = take((static_cast<int64_t>(V) + 8) * 2);
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
    pl.pcount = reinterpret_cast<int32_t*>(b + L.pcount);
    pl.jmap = reinterpret_cast<uint16_t*>(b + L.jmap);
    pl.nw = (V + 31) / 32;
    return pl;
}

struct SampleLayout {
    int64_t plan, stats, rbound, rbest, rdone, clane, gslots;
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
    L.rbound = take(R * 4);
    L.rbest = take(R * 8);
    L.rdone = take(R * 4);
    // the fast row pass's group records: one byte per group of 2048 (bf16) or 1024 (fp32) ids
    L.clane = take(R * (k + 1) * ((static_cast<int64_t>(V) + kChunkElems - 1) / kChunkElems) * 2);
    const int64_t units = R * (k + 1);
    // one CTA per unit while they fit one per SM; else the largest grid within one CTA per SM that
    // is coprime to 6 (see unit_rj)
    int64_t g = std::max<int64_t>(1, std::min<int64_t>(units, sms > 0 ? sms : 148));
    if (g < units)
        while (g > 1 && std::gcd<int64_t>(g, 6) != 1) --g;
    L.grid = static_cast<int>(g);
    const int64_t resident = align256(static_cast<int64_t>(Vd) * ed) + align256(static_cast<int64_t>(Vd) * et);
    const size_t ring = kRowHeader + static_cast<size_t>(kStages) * kStageBytes;
    L.smem_mode = ring + resident <= kSmemBudget ? 1 : 0;
    L.smem_bytes = ring + (L.smem_mode ? resident : 0);
    L.gslot_bytes = L.smem_mode ? 0 : resident;
    L.gslots = take(L.smem_mode ? 0 : L.gslot_bytes * L.grid);
    L.total = off + 256;
    return L;
}

// the opt-in shared memory of a CTA (227 KB) less room for the kernel's static arrays
constexpr size_t kFastSmemLimit = 227 * 1024 - 1024;

template <int DT>
size_t fast_smem_bytes(int32_t V, int32_t Vd)
{
    using Cfg = FastCfg<DT>;
    return static_cast<size_t>(kFastHeader + kStreamWarps * Cfg::kStages * static_cast<int64_t>(Cfg::kStageBytes) +
                               Cfg::kNG * align256((static_cast<int64_t>(Vd) + 8) * Cfg::kElem) +
                               (static_cast<int64_t>(V + kChunkElems - 1) / kChunkElems + 1) * 4);
}

size_t fast_smem_bytes(const Rows& t, const Rows& d)
{
    return t.dtype == SV_BF16 ? fast_smem_bytes<SV_BF16>(t.width, d.width) : fast_smem_bytes<SV_F32>(t.width, d.width);
}

// the fast row pass: bf16 target and draft rows, or fp32 target and draft rows, with a d2t map
bool fast_path_ok(const Rows& t, const Rows& d, bool identity)
{
    return !identity && t.dtype == d.dtype && t.bulk_ok && d.bulk_ok && d.data != nullptr && t.width % 8 == 0 &&
           d.width % 8 == 0 && d.width < kFastMaxVd &&  // 2 Vd fits 16 bits
           fast_smem_bytes(t, d) <= kFastSmemLimit;
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
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    const size_t gsmem = sizeof(GroupState) + kChunkElems * 2;
    const int32_t nch = (V + kChunkElems - 1) / kChunkElems;
    d2t_group_kernel<<<nch, 32, gsmem, stream>>>(Vd, V, pl);
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
    const bool fast = fast_path_ok(t, d, identity);
    A.race_bound = reinterpret_cast<unsigned int*>(ws + L.rbound);
    A.race_best = reinterpret_cast<unsigned long long*>(ws + L.rbest);
    A.race_done = reinterpret_cast<unsigned int*>(ws + L.rdone);
    if (fast) {
        A.clane = reinterpret_cast<uint8_t*>(ws + L.clane);
        A.ngroups = ((t.width + kChunkElems - 1) / kChunkElems) * (t.dtype == SV_BF16 ? FastCfg<SV_BF16>::kHalves
                                                                                    : FastCfg<SV_F32>::kHalves);
    }
    A.gslots = ws + L.gslots;
    A.gslot_bytes = L.gslot_bytes;
    A.smem_mode = L.smem_mode;


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
    if (fast) {
        const size_t smem = fast_smem_bytes(t, d);
        auto* kern = t.dtype == SV_BF16 ? sample_rows_fast_kernel<SV_BF16> : sample_rows_fast_kernel<SV_F32>;
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
        if (e != cudaSuccess) return e;
        cfg.gridDim = dim3(static_cast<unsigned>(L.grid));
        cfg.blockDim = dim3(kFastThreads);
        cfg.dynamicSmemBytes = smem;
        e = cudaLaunchKernelEx(&cfg, kern, A);
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
    // the race: one wave of CTAs (two per SM), or fewer when even the longest partition line (every
    // request sampled) gives no CTA beyond the first ones a full minimum share; the kernel cuts the
    // line itself from the temperatures
    const int64_t slots = 2LL * (sms > 0 ? sms : 148);
    const int64_t Vp = (static_cast<int64_t>(t.width) + kRaceStep - 1) / kRaceStep * kRaceStep;
    const int64_t line_max = static_cast<int64_t>(R) * (kRacePartIds + Vp);
    const int64_t rgrid = std::max<int64_t>(1, std::min<int64_t>(slots, (line_max + kRaceMinShare - 1) / kRaceMinShare));
    const uint32_t ybytes = static_cast<uint32_t>(d.width) * d.esize;
    const bool yshared = !identity && A.dbulk && ybytes <= kRaceSmemRow && ybytes % 16 == 0;
    const size_t race_smem = yshared ? ybytes : 0;
    auto* race = identity ? race_rows_kernel<DT, DD, kYIdentity>
                          : (yshared ? race_rows_kernel<DT, DD, kYShared> : race_rows_kernel<DT, DD, kYGlobal>);
    e = cudaFuncSetAttribute(race, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(race_smem));
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg2 = {};
    cfg2.gridDim = dim3(static_cast<unsigned>(rgrid));
    cfg2.blockDim = dim3(kRaceThreads);
    cfg2.dynamicSmemBytes = race_smem;
    cfg2.stream = stream;
    cfg2.attrs = attr;
    cfg2.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg2, race, A);
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
