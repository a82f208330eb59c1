// The C ABI of specverify: argument checks, then the kernel launchers.
// Declarations and the contract of every call are in include/specverify.h.
#include <algorithm>
#include <cstdint>
#include <cuda_runtime.h>

#include "specverify.h"
#include "sv_internal.h"

namespace sv {

int device_sm_count()
{
    int dev = 0, n = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    return n;
}

static bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// Validate a logit matrix with `rows` rows; `min_stride` is the smallest
// legal row stride (the width, or offset + width for CFG partitions).
static int check_rows(const sv_rows& m, int64_t rows, int64_t min_stride, Rows* out)
{
    if (m.dtype != SV_BF16 && m.dtype != SV_F32) return SV_ERR_DTYPE;
    if (m.width < 1 || m.width > SV_MAX_WIDTH) return SV_ERR_SHAPE;
    if (rows > 1 && m.row_stride < min_stride) return SV_ERR_SHAPE;
    if (m.row_stride < 0) return SV_ERR_SHAPE;
    if (rows > 0 && m.data == nullptr) return SV_ERR_INVALID_ARG;
    const int es = m.dtype == SV_BF16 ? 2 : 4;
    if (!aligned(m.data, es)) return SV_ERR_ALIGN;
    out->data = static_cast<const char*>(m.data);
    out->dtype = m.dtype;
    out->esize = es;
    out->width = m.width;
    out->stride = rows > 1 ? m.row_stride : std::max<int64_t>(m.row_stride, min_stride);
    out->bulk_ok = aligned(m.data, 16) && ((out->stride * es) % 16 == 0);
    return SV_OK;
}

static int check_workspace(const void* ws, size_t bytes, size_t need)
{
    if (ws == nullptr || bytes < need || !aligned(ws, 256)) return SV_ERR_WORKSPACE;
    return SV_OK;
}

static int launched(cudaError_t e) { return e == cudaSuccess ? SV_OK : SV_ERR_LAUNCH; }

static bool have_device()
{
    int dev = 0;
    return cudaGetDevice(&dev) == cudaSuccess;
}

}  // namespace sv

using namespace sv;

extern "C" {

const char* sv_status_string(int code)
{
    switch (code) {
        case SV_OK: return "ok";
        case SV_ERR_INVALID_ARG: return "invalid argument";
        case SV_ERR_DTYPE: return "unsupported logit dtype";
        case SV_ERR_SHAPE: return "inconsistent width, row stride or offsets";
        case SV_ERR_LIMIT: return "size above a documented limit";
        case SV_ERR_LAUNCH: return "CUDA launch failed";
        case SV_ERR_WORKSPACE: return "workspace missing, too small or not 256-byte aligned";
        case SV_ERR_ALIGN: return "pointer not aligned to its element size";
        case SV_ERR_DEVICE: return "no usable CUDA device";
        default: return "unknown status";
    }
}

size_t sv_verify_greedy_workspace(int32_t R, int32_t k, int32_t branches, int32_t V)
{
    if (R < 0 || k < 0 || V < 1 || branches < 1 || branches > SV_MAX_BRANCHES) return 0;
    return greedy_workspace_bytes(R, k, branches, V);
}

int sv_verify_greedy(sv_rows target, int32_t R, int32_t k, int32_t branches, const int32_t* draft,
                     int32_t* accept_len, int32_t* tokens, int32_t* branch, int32_t* status,
                     void* workspace, size_t workspace_bytes, sv_stream_t stream)
{
    if (R < 0 || k < 0) return SV_ERR_INVALID_ARG;
    if (branches < 1 || (branches >= 2 && k < 1)) return SV_ERR_INVALID_ARG;
    if (branches > SV_MAX_BRANCHES) return SV_ERR_LIMIT;
    if (k > SV_MAX_K) return SV_ERR_LIMIT;
    if (R == 0) return SV_OK;
    if ((k > 0 && draft == nullptr) || accept_len == nullptr || tokens == nullptr)
        return SV_ERR_INVALID_ARG;
    if (!aligned(draft, 4) || !aligned(accept_len, 4) || !aligned(tokens, 4) ||
        !aligned(branch, 4) || !aligned(status, 4))
        return SV_ERR_ALIGN;
    const int64_t rows = static_cast<int64_t>(R) * (1 + static_cast<int64_t>(branches) * k);
    Rows t{};
    if (int rc = check_rows(target, rows, target.width, &t)) return rc;
    const SegPlan plan = plan_segments(rows, t.width, t.esize);
    if (rows * plan.nseg > INT32_MAX) return SV_ERR_LIMIT;
    if (int rc = check_workspace(workspace, workspace_bytes,
                                 greedy_workspace_bytes(R, k, branches, t.width)))
        return rc;
    if (!have_device()) return SV_ERR_DEVICE;
    return launched(launch_verify_greedy(t, R, k, branches, draft, accept_len, tokens, branch,
                                         status, workspace, stream));
}

size_t sv_verify_greedy_top2_workspace(int32_t R, int32_t k, int32_t branches, int32_t V)
{
    if (R < 0 || k < 0 || V < 1 || branches < 1 || branches > SV_MAX_BRANCHES) return 0;
    return greedy_workspace_bytes(R, k, branches, V, true);
}

int sv_verify_greedy_top2(sv_rows target, int32_t R, int32_t k, int32_t branches, const int32_t* draft,
                          int32_t* accept_len, int32_t* tokens, int32_t* branch, int32_t* status,
                          int32_t* top2, void* workspace, size_t workspace_bytes, sv_stream_t stream)
{
    if (R < 0 || k < 0) return SV_ERR_INVALID_ARG;
    if (branches < 1 || (branches >= 2 && k < 1)) return SV_ERR_INVALID_ARG;
    if (branches > SV_MAX_BRANCHES) return SV_ERR_LIMIT;
    if (k > SV_MAX_K) return SV_ERR_LIMIT;
    if (R == 0) return SV_OK;
    if ((k > 0 && draft == nullptr) || accept_len == nullptr || tokens == nullptr || top2 == nullptr)
        return SV_ERR_INVALID_ARG;
    if (!aligned(draft, 4) || !aligned(accept_len, 4) || !aligned(tokens, 4) ||
        !aligned(branch, 4) || !aligned(status, 4) || !aligned(top2, 4))
        return SV_ERR_ALIGN;
    const int64_t rows = static_cast<int64_t>(R) * (1 + static_cast<int64_t>(branches) * k);
    Rows t{};
    if (int rc = check_rows(target, rows, target.width, &t)) return rc;
    const SegPlan plan = plan_segments(rows, t.width, t.esize);
    if (rows * plan.nseg > INT32_MAX) return SV_ERR_LIMIT;
    if (int rc = check_workspace(workspace, workspace_bytes,
                                 greedy_workspace_bytes(R, k, branches, t.width, true)))
        return rc;
    if (!have_device()) return SV_ERR_DEVICE;
    return launched(launch_verify_greedy(t, R, k, branches, draft, accept_len, tokens, branch,
                                         status, workspace, stream, top2));
}

size_t sv_infer_modality_workspace(int32_t N, int32_t V)
{
    if (N < 0 || V < 1) return 0;
    return modality_workspace_bytes(N, V);
}

int sv_infer_modality(sv_rows logits, int32_t N, const int32_t* part_start, int32_t P, int32_t* amax,
                      int32_t* part, int32_t* mask_lo, int32_t* mask_hi, int32_t* status, void* workspace,
                      size_t workspace_bytes, sv_stream_t stream)
{
    if (N < 0 || P < 1 || part_start == nullptr) return SV_ERR_INVALID_ARG;
    if (P > kMaxParts) return SV_ERR_LIMIT;
    for (int32_t p = 0; p < P; ++p)
        if (part_start[p] > part_start[p + 1]) return SV_ERR_INVALID_ARG;
    if (N == 0) return SV_OK;
    if (part == nullptr) return SV_ERR_INVALID_ARG;
    if (!aligned(amax, 4) || !aligned(part, 4) || !aligned(mask_lo, 4) || !aligned(mask_hi, 4) ||
        !aligned(status, 4))
        return SV_ERR_ALIGN;
    Rows t{};
    if (int rc = check_rows(logits, N, logits.width, &t)) return rc;
    const SegPlan plan = plan_segments(N, t.width, t.esize);
    if (static_cast<int64_t>(N) * plan.nseg > INT32_MAX) return SV_ERR_LIMIT;
    if (int rc = check_workspace(workspace, workspace_bytes, modality_workspace_bytes(N, t.width))) return rc;
    if (!have_device()) return SV_ERR_DEVICE;
    PartTable pt{};
    pt.P = P;
    for (int32_t p = 0; p <= P; ++p) pt.start[p] = part_start[p];
    return launched(launch_infer_modality(t, N, pt, amax, part, mask_lo, mask_hi, status, workspace, stream));
}

size_t sv_verify_sample_workspace(int32_t R, int32_t k, int32_t V, int32_t Vd)
{
    if (R < 0 || k < 0 || V < 1 || Vd < 1) return 0;
    return sample_workspace_bytes(R, k, V, Vd);
}

int sv_verify_sample(sv_rows target, sv_rows draft_logits, const int32_t* d2t, const void* d2t_plan,
                     int32_t R, int32_t k, const int32_t* draft, const uint64_t* seeds,
                     const float* temperature, int32_t* accept_len, int32_t* tokens, float* tv,
                     float* p_draft, float* q_draft, int32_t* status, void* workspace,
                     size_t workspace_bytes, sv_stream_t stream)
{
    if (R < 0 || k < 0) return SV_ERR_INVALID_ARG;
    if (k > SV_MAX_K) return SV_ERR_LIMIT;
    if (static_cast<int64_t>(R) * (k + 1) > INT32_MAX) return SV_ERR_LIMIT;
    if (R == 0) return SV_OK;
    if ((k > 0 && draft == nullptr) || seeds == nullptr || temperature == nullptr ||
        accept_len == nullptr || tokens == nullptr)
        return SV_ERR_INVALID_ARG;
    if (!aligned(draft, 4) || !aligned(seeds, 8) || !aligned(temperature, 4) ||
        !aligned(accept_len, 4) || !aligned(tokens, 4) || !aligned(tv, 4) ||
        !aligned(p_draft, 4) || !aligned(q_draft, 4) || !aligned(status, 4) || !aligned(d2t, 4))
        return SV_ERR_ALIGN;
    if (!aligned(d2t_plan, 256)) return SV_ERR_WORKSPACE;
    Rows t{}, d{};
    if (int rc = check_rows(target, static_cast<int64_t>(R) * (k + 1), target.width, &t)) return rc;
    const int64_t drows = static_cast<int64_t>(R) * k;
    if (drows > 0) {
        if (int rc = check_rows(draft_logits, drows, draft_logits.width, &d)) return rc;
    } else {
        d = Rows{nullptr, SV_F32, 4, draft_logits.width > 0 ? draft_logits.width : t.width, 0, false};
    }
    const bool mapped = d2t != nullptr || d2t_plan != nullptr;
    if (!mapped && d.width != t.width) return SV_ERR_SHAPE;
    if (t.width > sample_max_plan_width()) return SV_ERR_LIMIT;  // the race keeps one sum per 2048 ids
    if (int rc = check_workspace(workspace, workspace_bytes,
                                 sample_workspace_bytes(R, k, t.width, d.width)))
        return rc;
    if (!have_device()) return SV_ERR_DEVICE;
    return launched(launch_verify_sample(t, d, d2t, d2t_plan, R, k, draft, seeds, temperature, accept_len,
                                         tokens, tv, p_draft, q_draft, status, workspace, stream));
}

size_t sv_d2t_plan_bytes(int32_t V, int32_t Vd)
{
    if (V < 1 || Vd < 1) return 0;
    return d2t_plan_bytes(V, Vd);
}

int sv_d2t_plan_build(const int32_t* d2t, int32_t Vd, int32_t V, void* plan, size_t plan_bytes,
                      sv_stream_t stream)
{
    if (V < 1 || Vd < 1 || d2t == nullptr) return SV_ERR_INVALID_ARG;
    if (V > sample_max_plan_width() || Vd > 65535) return SV_ERR_LIMIT;
    if (!aligned(d2t, 4)) return SV_ERR_ALIGN;
    if (int rc = check_workspace(plan, plan_bytes, d2t_plan_bytes(V, Vd))) return rc;
    if (!have_device()) return SV_ERR_DEVICE;
    return launched(launch_d2t_plan_build(d2t, Vd, V, plan, stream));
}

size_t sv_cfg_merge_sample_workspace(int32_t R, int32_t k, int32_t S, int32_t W)
{
    if (R < 0 || k < 0 || S < 1 || S > SV_MAX_S || W < 1) return 0;
    return cfg_workspace_bytes(R, k, S, W);
}

int sv_cfg_merge_sample(sv_rows cond, sv_rows uncond, const int32_t* cb_id_base,
                        const int32_t* cb_data_offset, int32_t S, float w, sv_rows draft_logits,
                        int32_t R, int32_t k, const int32_t* draft, const uint64_t* seeds,
                        const float* temperature, int32_t* accept_len, int32_t* tokens, float* tv,
                        int32_t* status, void* workspace, size_t workspace_bytes,
                        sv_stream_t stream)
{
    if (R < 0 || k < 0 || S < 1) return SV_ERR_INVALID_ARG;
    if (k > SV_MAX_K || S > SV_MAX_S) return SV_ERR_LIMIT;
    if (cb_id_base == nullptr) return SV_ERR_INVALID_ARG;
    if (cond.width > cfg_max_width()) return SV_ERR_LIMIT;
    if (cond.width != uncond.width || cond.dtype != uncond.dtype ||
        cond.row_stride != uncond.row_stride)
        return SV_ERR_SHAPE;
    if (R == 0) return SV_OK;
    if ((k > 0 && draft == nullptr) || seeds == nullptr || temperature == nullptr ||
        accept_len == nullptr || tokens == nullptr)
        return SV_ERR_INVALID_ARG;
    if (!aligned(draft, 4) || !aligned(seeds, 8) || !aligned(temperature, 4) ||
        !aligned(accept_len, 4) || !aligned(tokens, 4) || !aligned(tv, 4) || !aligned(status, 4))
        return SV_ERR_ALIGN;
    CfgShape shape{};
    shape.S = S;
    shape.W = cond.width;
    shape.w = w;
    int64_t max_end = cond.width;
    for (int s = 0; s < S; ++s) {
        shape.id_base[s] = cb_id_base[s];
        shape.data_off[s] = cb_data_offset ? cb_data_offset[s] : 0;
        if (shape.data_off[s] < 0) return SV_ERR_SHAPE;
        max_end = std::max<int64_t>(max_end, static_cast<int64_t>(shape.data_off[s]) + cond.width);
    }
    const int64_t rows = static_cast<int64_t>(R) * (k + 1) * S;
    Rows c{}, u{}, d{};
    if (int rc = check_rows(cond, rows, max_end, &c)) return rc;
    if (int rc = check_rows(uncond, rows, max_end, &u)) return rc;
    const Rows* dp = nullptr;
    if (draft_logits.data != nullptr && k > 0) {
        if (draft_logits.width != cond.width) return SV_ERR_SHAPE;
        if (int rc = check_rows(draft_logits, static_cast<int64_t>(R) * k * S, draft_logits.width, &d))
            return rc;
        dp = &d;
    }
    if (int rc = check_workspace(workspace, workspace_bytes, cfg_workspace_bytes(R, k, S, cond.width)))
        return rc;
    if (!have_device()) return SV_ERR_DEVICE;
    return launched(launch_cfg_merge_sample(c, u, shape, dp, R, k, draft, seeds, temperature,
                                            accept_len, tokens, tv, status, workspace, stream));
}

int sv_pool_append(int32_t* pool, int32_t* pool_len, int32_t Lp, const int32_t* drafts, int32_t k,
                   int32_t R, int32_t* status, sv_stream_t stream)
{
    if (R < 0 || k < 0 || Lp < 0) return SV_ERR_INVALID_ARG;
    if (k > SV_MAX_K || Lp > SV_MAX_POOL) return SV_ERR_LIMIT;
    if (R == 0) return SV_OK;
    if (pool_len == nullptr || (k > 0 && drafts == nullptr) || (Lp > 0 && pool == nullptr))
        return SV_ERR_INVALID_ARG;
    if (!aligned(pool, 4) || !aligned(pool_len, 4) || !aligned(drafts, 4) || !aligned(status, 4))
        return SV_ERR_ALIGN;
    if (!have_device()) return SV_ERR_DEVICE;
    return launched(launch_pool_append(pool, pool_len, Lp, drafts, k, R, status, stream));
}

int sv_pool_lookup(const int32_t* pool, const int32_t* pool_len, int32_t Lp, const int32_t* suffix,
                   int32_t N, int32_t R, int32_t gamma, int32_t* match_len, int32_t* cont,
                   sv_stream_t stream)
{
    if (R < 0 || N < 0 || gamma < 0 || Lp < 0) return SV_ERR_INVALID_ARG;
    if (N > SV_MAX_NGRAM || gamma > SV_MAX_K || Lp > SV_MAX_POOL) return SV_ERR_LIMIT;
    if (R == 0) return SV_OK;
    if (pool_len == nullptr || match_len == nullptr || (Lp > 0 && pool == nullptr) ||
        (N > 0 && suffix == nullptr) || (gamma > 0 && cont == nullptr))
        return SV_ERR_INVALID_ARG;
    if (!aligned(pool, 4) || !aligned(pool_len, 4) || !aligned(suffix, 4) || !aligned(match_len, 4) ||
        !aligned(cont, 4))
        return SV_ERR_ALIGN;
    if (!have_device()) return SV_ERR_DEVICE;
    return launched(launch_pool_lookup(pool, pool_len, Lp, suffix, N, R, gamma, match_len, cont, stream));
}

int sv_suffix_append(int32_t* suffix, int32_t N, int32_t R, const int32_t* tokens, const int32_t* accept_len,
                     int32_t k, sv_stream_t stream)
{
    if (R < 0 || N < 0 || k < 0) return SV_ERR_INVALID_ARG;
    if (N > SV_MAX_NGRAM || k > SV_MAX_K) return SV_ERR_LIMIT;
    if (R == 0 || N == 0) return SV_OK;
    if (suffix == nullptr || tokens == nullptr || accept_len == nullptr) return SV_ERR_INVALID_ARG;
    if (!aligned(suffix, 4) || !aligned(tokens, 4) || !aligned(accept_len, 4)) return SV_ERR_ALIGN;
    if (!have_device()) return SV_ERR_DEVICE;
    return launched(launch_suffix_append(suffix, N, R, tokens, accept_len, k, stream));
}

int sv_accept_scan(const uint8_t* accept, const int32_t* draft, const int32_t* fix, int32_t R,
                   int32_t k, int32_t* accept_len, int32_t* tokens, sv_stream_t stream)
{
    if (R < 0 || k < 0) return SV_ERR_INVALID_ARG;
    if (k > SV_MAX_K) return SV_ERR_LIMIT;
    if (R == 0) return SV_OK;
    if ((k > 0 && (accept == nullptr || draft == nullptr)) || fix == nullptr ||
        accept_len == nullptr || tokens == nullptr)
        return SV_ERR_INVALID_ARG;
    if (!aligned(draft, 4) || !aligned(fix, 4) || !aligned(accept_len, 4) || !aligned(tokens, 4))
        return SV_ERR_ALIGN;
    if (!have_device()) return SV_ERR_DEVICE;
    return launched(launch_accept_scan(accept, draft, fix, R, k, accept_len, tokens, stream));
}

}  // extern "C"
