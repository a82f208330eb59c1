// Host-side interfaces between the C ABI (api.cu) and the kernel launchers.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>

#include "specverify.h"

namespace sv {

// A validated logit matrix.
struct Rows {
    const char* data;
    int dtype;       // SV_BF16 / SV_F32
    int esize;       // bytes per element
    int32_t width;   // entries per row
    int64_t stride;  // elements between row starts
    bool bulk_ok;    // every row start is 16-byte aligned: bulk copies allowed
};

// Rows of a matrix are cut into `nseg` segments of `seg_len` elements (the
// last one may be shorter); one CTA streams one segment.
struct SegPlan {
    int32_t nseg;
    int32_t seg_len;
};
SegPlan plan_segments(int64_t rows, int32_t width, int esize);

// Per-segment argmax result (16 bytes).
struct ArgPartial {
    float v;
    int32_t i;
    uint32_t flags;
    uint32_t pad;
};

// a segment's two first ids (value descending, id ascending; INT32_MAX: none)
struct Top2Partial {
    float v1;
    int32_t i1;
    float v2;
    int32_t i2;
    uint32_t flags;
    uint32_t pad[3];
};

size_t greedy_workspace_bytes(int64_t R, int32_t k, int32_t branches, int32_t V, bool top2 = false);
// vocabulary partitions: [start[p], start[p + 1]) for p < P
constexpr int kMaxParts = SV_MAX_PARTS;
struct PartTable {
    int32_t P;
    int32_t start[kMaxParts + 1];
};
size_t modality_workspace_bytes(int64_t rows, int32_t V);
cudaError_t launch_infer_modality(const Rows& rows, int64_t nrows, const PartTable& pt, int32_t* amax,
                                  int32_t* part, int32_t* mask_lo, int32_t* mask_hi, int32_t* status,
                                  void* workspace, cudaStream_t stream);

// top2 != NULL: also the argmax and runner-up id of every row ([rows, 2])
cudaError_t launch_verify_greedy(const Rows& target, int32_t R, int32_t k, int32_t branches,
                                 const int32_t* draft, int32_t* accept_len, int32_t* tokens,
                                 int32_t* branch, int32_t* status, void* workspace,
                                 cudaStream_t stream, int32_t* top2 = nullptr);

cudaError_t launch_pool_append(int32_t* pool, int32_t* pool_len, int32_t Lp, const int32_t* drafts,
                               int32_t k, int32_t R, int32_t* status, cudaStream_t stream);
cudaError_t launch_pool_lookup(const int32_t* pool, const int32_t* pool_len, int32_t Lp, const int32_t* suffix,
                               int32_t N, int32_t R, int32_t gamma, int32_t* match_len, int32_t* cont,
                               cudaStream_t stream);

cudaError_t launch_suffix_append(int32_t* suffix, int32_t N, int32_t R, const int32_t* tokens,
                                 const int32_t* accept_len, int32_t k, cudaStream_t stream);

cudaError_t launch_accept_scan(const uint8_t* accept, const int32_t* draft, const int32_t* fix,
                               int32_t R, int32_t k, int32_t* accept_len, int32_t* tokens,
                               cudaStream_t stream);

size_t sample_workspace_bytes(int64_t R, int32_t k, int32_t V, int32_t Vd);
cudaError_t launch_verify_sample(const Rows& target, const Rows& draft_logits, const int32_t* d2t,
                                 const void* d2t_plan, int32_t R, int32_t k, const int32_t* draft,
                                 const uint64_t* seeds, const float* temperature, int32_t* accept_len,
                                 int32_t* tokens, float* tv, float* p_draft, float* q_draft, int32_t* status,
                                 void* workspace, cudaStream_t stream);
size_t d2t_plan_bytes(int32_t V, int32_t Vd);
cudaError_t launch_d2t_plan_build(const int32_t* d2t, int32_t Vd, int32_t V, void* plan, cudaStream_t stream);

// largest target vocabulary accepted together with a d2t map
int32_t sample_max_plan_width();

struct CfgShape {
    int32_t S, W;
    float w;
    int32_t id_base[SV_MAX_S];
    int32_t data_off[SV_MAX_S];
};
size_t cfg_workspace_bytes(int64_t R, int32_t k, int32_t S, int32_t W);
// widest codebook accepted by sv_cfg_merge_sample
int32_t cfg_max_width();
cudaError_t launch_cfg_merge_sample(const Rows& cond, const Rows& uncond, const CfgShape& shape,
                                    const Rows* draft_logits, int32_t R, int32_t k,
                                    const int32_t* draft, const uint64_t* seeds,
                                    const float* temperature, int32_t* accept_len,
                                    int32_t* tokens, float* tv, int32_t* status, void* workspace,
                                    cudaStream_t stream);

// number of SMs of the current device
int device_sm_count();

}  // namespace sv
