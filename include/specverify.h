/*
 * specverify -- speculative-decoding verify-and-sample on one GPU (sm_103a).
 *
 * The library turns the target model's logit rows for a block of draft
 * positions into committed tokens and accept lengths.  Three modes:
 *
 *   greedy verification  -- "Decode Before You Hear: Speculative Listening for
 *       Chunk-Interleaved Full-Duplex Speech Language Models" (digest), section
 *       "method steps", step 4 (accept the prefix before the first draft token
 *       that differs from argmax p_i, then commit argmax p_{n+1}) and step 2
 *       (a runner-up branch verified in the same forward pass);
 *   speculative sampling -- "speculative decoding for Omni models" (blog),
 *       section 2 (accept with probability min(1, p/q), resample from
 *       norm(max(0, p - q)) on rejection, bonus token from p when every draft
 *       is accepted, TV = 1/2 sum |p - q|) and section 4 (truncated draft
 *       vocabulary mapped by d2t; ids outside it have q = 0);
 *   CFG merge per codebook -- "An Efficient vLLM-Based Inference Pipeline for
 *       Unified Audio Understanding and Generation" (digest), paired CFG
 *       co-scheduling section and Figure 1 text (the conditional and
 *       unconditional logits of each codebook are merged linearly with w > 1,
 *       then one token per codebook is sampled from the audio partition).
 *
 * Conventions shared by every call
 *  - Pointers are DEVICE pointers unless a comment says HOST.  The caller owns
 *    every buffer; the library allocates and frees nothing.
 *  - Every call is asynchronous on `stream` (a cudaStream_t; NULL = the legacy
 *    default stream).  The return value reports host-side argument checks and
 *    the launch status only; per-request data problems are reported in the
 *    device-written `status` array (bits SV_ST_*), never by a trap.
 *  - Results are a pure function of the inputs: they do not depend on the
 *    batch size, the position of a request in the batch or the launch
 *    geometry (every sum is taken in an order fixed by the request's own
 *    inputs).  Random draws come from Philox4x32-10 keyed by the request's
 *    seed, so a call repeated on the same inputs gives the same bits.
 *  - Ties in an argmax or in the sampler go to the lowest index.  NaN logits
 *    read as -inf.
 *  - Workspace: calls that take one need at least the number of bytes the
 *    matching *_workspace function returns, 256-byte aligned.  Its contents on
 *    entry do not matter; calls sharing one workspace must not overlap.
 *  - The library keeps no state between calls and is thread-safe.
 */
#ifndef SPECVERIFY_H
#define SPECVERIFY_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

struct CUstream_st;
typedef struct CUstream_st* sv_stream_t; /* same type as cudaStream_t */

/* return codes */
enum {
    SV_OK = 0,
    SV_ERR_INVALID_ARG = -1, /* NULL where a buffer is required, negative size, bad enum */
    SV_ERR_DTYPE = -2,       /* logit dtype is neither SV_BF16 nor SV_F32 */
    SV_ERR_SHAPE = -3,       /* width / row_stride / offsets inconsistent */
    SV_ERR_LIMIT = -4,       /* k, S or a size above the documented limits */
    SV_ERR_LAUNCH = -5,      /* the CUDA launch failed (see cudaGetLastError) */
    SV_ERR_WORKSPACE = -6,   /* workspace NULL, too small or not 256-byte aligned */
    SV_ERR_ALIGN = -7,       /* a pointer is not aligned to its element size */
    SV_ERR_DEVICE = -8       /* no usable CUDA device */
};

/* logit element types */
enum { SV_BF16 = 0, SV_F32 = 1 };

/* per-request status bits, written to status[r] (0 = nothing to report) */
enum {
    SV_ST_TOKEN_RANGE = 1,    /* a draft token is outside the vocabulary: it never matches */
    SV_ST_BAD_LOGITS = 2,     /* a row holds NaN or +inf or is all -inf (sampling: greedy used) */
    SV_ST_OFF_SUPPORT = 4,    /* a tested draft token has q = 0: rejected */
    SV_ST_RESIDUAL_ZERO = 8,  /* max(0, p - q) had no mass: the correction was drawn from p */
    SV_ST_BAD_TEMP = 16,      /* temperature negative or NaN: greedy verification used */
    SV_ST_BAD_D2T = 32,       /* d2t holds an id outside [0, V) or a repeated id */
    SV_ST_TIMEOUT = 64,       /* a bounded device wait gave up; the request's outputs are invalid */
    SV_ST_POOL_FULL = 128     /* sv_pool_append: the draft did not fit in the pool; nothing inserted */
};

/* limits */
#define SV_MAX_K 256       /* drafts per request (per branch) */
#define SV_MAX_S 16        /* codebooks per CFG frame */
#define SV_MAX_PARTS 64    /* vocabulary partitions of sv_infer_modality */
#define SV_MAX_BRANCHES 8  /* draft branches sharing the first row (sv_verify_greedy) */
#define SV_MAX_NGRAM 64     /* emitted-suffix tokens matched by sv_pool_lookup */
#define SV_MAX_POOL (1 << 24) /* pool capacity per request (tokens and separators) */
#define SV_MAX_WIDTH (1 << 30)

/* A matrix of logit rows: row i, entry x is at data + (i * row_stride + x)
 * elements.  `data` must be aligned to the element size.  Rows whose start
 * is 16-byte aligned (data 16-byte aligned and row_stride * element size a
 * multiple of 16) take the bulk-copy path; other layouts are accepted and
 * read with plain loads. */
typedef struct sv_rows {
    const void* data;
    int32_t dtype;      /* SV_BF16 or SV_F32 */
    int32_t width;      /* entries per row: V, Vd or W */
    int64_t row_stride; /* elements between consecutive row starts, >= width */
} sv_rows;

/* Human-readable text for a return code. */
const char* sv_status_string(int code);

/* ------------------------------------------------------------------------
 * sv_verify_greedy -- greedy verification with optional further branches.
 * Source: "Decode Before You Hear ..." method steps 2 and 4 (a runner-up
 * branch beside the main draft); more branches are tree drafts whose first
 * tokens differ.
 *
 *   target      rows of raw target logits, width V: 1 + branches * k rows per
 *               request laid out as [p_1 | branch 0 p_2..p_{k+1} | branch 1
 *               p_2..p_{k+1} | ...] (row p_1 is shared by every branch; with
 *               one branch, the k + 1 rows of positions 1..k and the row after
 *               the last draft; with two, [p_1 | main | runner]).  Request r's
 *               rows start at row r * rows_per_request.
 *   R           requests (>= 0; 0 is a no-op).
 *   k           drafts per branch, 0 <= k <= SV_MAX_K (k >= 1 with 2+ branches).
 *   branches    1 <= branches <= SV_MAX_BRANCHES.
 *   draft       int32 [R, branches, k] target ids.
 *   accept_len  int32 [R] out: accepted drafts n in [0, k].
 *   tokens      int32 [R, k + 1] out: the n accepted drafts then the
 *               correction argmax p_{n+1}; remaining entries -1.
 *   branch      int32 [R] out or NULL: the branch whose tokens were taken.
 *   status      int32 [R] out or NULL: SV_ST_* bits.
 * argmax is over raw logits (temperature cannot change it).  A branch is
 * viable when its first draft equals argmax p_1; among viable branches the
 * longer accepted prefix wins, ties to the lower branch; with none viable
 * n = 0 and branch 0.
 * ---------------------------------------------------------------------- */
size_t sv_verify_greedy_workspace(int32_t R, int32_t k, int32_t branches, int32_t V);
int sv_verify_greedy(sv_rows target, int32_t R, int32_t k, int32_t branches,
                     const int32_t* draft, int32_t* accept_len, int32_t* tokens,
                     int32_t* branch, int32_t* status, void* workspace,
                     size_t workspace_bytes, sv_stream_t stream);

/* ------------------------------------------------------------------------
 * sv_verify_greedy_top2 -- sv_verify_greedy that also returns, fused into the
 * same pass over the rows, the argmax and the runner-up id of every row.
 * Source: "Decode Before You Hear ..." method step 2: the runner-up branch
 * starts from the second-best token of the verified row.
 *
 *   top2        int32 [R * rows_per_request, 2] out: per row, in row order,
 *               the first two ids when ids are ordered by logit (descending),
 *               then by id (ascending), NaN read as -inf; the first equals the
 *               argmax of sv_verify_greedy; the second is -1 when V == 1.
 * Every other argument, output and limit is that of sv_verify_greedy; the
 * workspace is sized by sv_verify_greedy_top2_workspace.
 * ---------------------------------------------------------------------- */
size_t sv_verify_greedy_top2_workspace(int32_t R, int32_t k, int32_t branches, int32_t V);
int sv_verify_greedy_top2(sv_rows target, int32_t R, int32_t k, int32_t branches,
                          const int32_t* draft, int32_t* accept_len, int32_t* tokens,
                          int32_t* branch, int32_t* status, int32_t* top2, void* workspace,
                          size_t workspace_bytes, sv_stream_t stream);

/* ------------------------------------------------------------------------
 * sv_infer_modality -- the modality of each row of full-vocabulary logits and
 * the phase mask of its next step.
 * Source: "An Efficient vLLM-Based Inference Pipeline ..." phase management and
 * Figure 1 text: the vocabulary is split into a text part and S audio
 * sub-vocabularies; since continuous batching flattens the requests' tokens,
 * the current modality is inferred from the partition that holds the maximum
 * of the unmasked output distribution.
 *
 *   logits      N rows of raw logits over the full vocabulary, width V.
 *   part_start  HOST int32 [P + 1], ascending: partition p is the id range
 *               [part_start[p], part_start[p + 1]) (e.g. the text part, then
 *               the S codebooks); ids outside every range belong to none.
 *   P           partitions, 1 <= P <= SV_MAX_PARTS.
 *   amax        int32 [N] out or NULL: argmax of the row (NaN read as -inf,
 *               lowest id among equal maxima).
 *   part        int32 [N] out: the partition holding the argmax, -1 for none.
 *   mask_lo, mask_hi  int32 [N] out or NULL: that partition's id range, the
 *               vocabulary mask of the row's next step (0, 0 for none).
 *   status      int32 [N] out or NULL: SV_ST_BAD_LOGITS for NaN or +-inf maxima.
 * The workspace is sized by sv_infer_modality_workspace(N, V).
 * ---------------------------------------------------------------------- */
size_t sv_infer_modality_workspace(int32_t N, int32_t V);
int sv_infer_modality(sv_rows logits, int32_t N, const int32_t* part_start, int32_t P,
                      int32_t* amax, int32_t* part, int32_t* mask_lo, int32_t* mask_hi,
                      int32_t* status, void* workspace, size_t workspace_bytes,
                      sv_stream_t stream);

/* ------------------------------------------------------------------------
 * sv_verify_greedy_noalloc -- sv_verify_greedy without a workspace argument.
 * The source pages have no counterpart; this is a convenience for callers
 * that cannot allocate device memory: a plugin whose host framework owns all
 * GPU memory through its own caching pool, or a serving loop that reserves
 * every buffer up front and must not allocate while decoding.
 *
 * Arguments, outputs and results are those of sv_verify_greedy.  The scratch
 * lives in a fixed device array of SV_NOALLOC_SCRATCH_BYTES compiled into the
 * library; every GPU that loads the library keeps it until the process exits.
 *  - Argument errors are those of sv_verify_greedy, checked in its order.
 *    Batches whose workspace (sv_verify_greedy_workspace) exceeds that size
 *    are then rejected with SV_ERR_LIMIT before anything is launched.
 *  - Every call looks up the array's device address on the current device
 *    (cudaGetSymbolAddress with that device current).  The first call on a
 *    device may also load the library's device code: make that first call
 *    before any stream capture.
 *  - All calls share the one array.  Calls that overlap on the GPU (other
 *    streams, other host threads) race on it and give wrong results;
 *    serialise them.  The array keeps the last call's contents, which no
 *    later call depends on.
 *  - Calls no cudaMalloc, cudaFree or other allocating routine.
 * ---------------------------------------------------------------------- */
#define SV_NOALLOC_SCRATCH_BYTES (8u << 20)
int sv_verify_greedy_noalloc(sv_rows target, int32_t R, int32_t k, int32_t branches,
                             const int32_t* draft, int32_t* accept_len, int32_t* tokens,
                             int32_t* branch, int32_t* status, sv_stream_t stream);

/* ------------------------------------------------------------------------
 * sv_verify_sample -- speculative sampling with a truncated draft vocabulary.
 * Source: "speculative decoding for Omni models", sections 2 and 4.
 *
 *   target        target logits, width V, k + 1 rows per request (positions
 *                 0..k-1 then the bonus row k).
 *   draft_logits  draft-model logits, width Vd, k rows per request.  Read only
 *                 for requests with temperature > 0.
 *   d2t           int32 [Vd]: draft id -> target id, injective; NULL means the
 *                 identity (then Vd must equal V).  Target ids outside the
 *                 image of d2t have q = 0.
 *   d2t_plan      NULL, or the plan sv_d2t_plan_build made from this d2t
 *                 (then d2t may be NULL): skips building it in the call.
 *   draft         int32 [R, k] draft tokens as TARGET ids.
 *   seeds         uint64 [R] Philox key of each request.
 *   temperature   float [R]; T > 0 samples, T <= 0 verifies greedily.  T = +inf
 *                 weighs every finite logit the same; the kernels scale logits
 *                 by log2(e)/T in fp32, so T below ~1e-7 with logits near 100
 *                 is outside their range.
 *   accept_len    int32 [R] out; tokens int32 [R, k + 1] out (-1 padded).
 *   tv, p_draft, q_draft  float [R, k] out or NULL: TV(p_j, q_j) over the
 *                 full target vocabulary, p_j(x_j) and q_j(x_j) for every
 *                 position j (also after the first rejection); NaN for
 *                 greedy requests.
 *   status        int32 [R] out or NULL.
 * Definition: p_j = softmax(z_j / T), q_j = softmax(y_j / T) pushed through
 * d2t.  Position j is accepted when q_j(x_j) > 0 and u_j < p_j(x_j)/q_j(x_j)
 * with u_j the Philox uniform (counter (0, j, 0, 0), word 0).  n = leading
 * accepts.  n < k: the correction is drawn from r = max(0, p_n - q_n) (all
 * of p_n if r has no mass, status bit 8); n == k: the bonus is drawn from
 * p_k.  The draw is a two-level exponential race: ids are cut into chunks of
 * 2048; the chunk c = argmin E_c / W_c over the chunk sums W_c of the
 * weights, E_c = -ln u_c with u_c from counter (c >> 2, row, tag, 0) word
 * c & 3 (tag 3 correction, 4 bonus); then the id = argmin E_x / w_x over
 * that chunk, u_x from counter (x >> 2, row, tag, 0) word x & 3 (tag 1
 * correction, 2 bonus); row is n (or k).  A uniform from word w is
 * (2 * (w >> 9) + 1) * 2^-24.
 * Limits: V <= 819,200 (SV_ERR_LIMIT above).
 * ---------------------------------------------------------------------- */
size_t sv_verify_sample_workspace(int32_t R, int32_t k, int32_t V, int32_t Vd);
int sv_verify_sample(sv_rows target, sv_rows draft_logits, const int32_t* d2t,
                     const void* d2t_plan, int32_t R, int32_t k, const int32_t* draft,
                     const uint64_t* seeds, const float* temperature, int32_t* accept_len,
                     int32_t* tokens, float* tv, float* p_draft, float* q_draft,
                     int32_t* status, void* workspace, size_t workspace_bytes,
                     sv_stream_t stream);

/* ------------------------------------------------------------------------
 * sv_d2t_plan_build -- prepare a truncated-vocabulary map once.
 * Source: "speculative decoding for Omni models", section 4 (d2t maps the
 * draft vocabulary into the target vocabulary).  The map is a constant of
 * the draft model, so its device-side form (a support bitmap over target
 * ids, per-word prefix counts, the support sorted by target id with its
 * draft ids) can be built once and passed to every sv_verify_sample call as
 * `d2t_plan`.  With d2t_plan == NULL and d2t != NULL, sv_verify_sample
 * builds the same plan in its workspace on every call.
 *
 *   d2t         int32 [Vd] draft id -> target id.
 *   plan        device buffer of at least sv_d2t_plan_bytes(V, Vd) bytes,
 *               256-byte aligned, owned by the caller; valid for this (V, Vd)
 *               until d2t changes.  A plan whose (V, Vd) differ from the
 *               call's, or a d2t with ids out of range or repeated, makes
 *               sv_verify_sample report SV_ST_BAD_D2T.
 * Limits: V <= 819,200.
 * ---------------------------------------------------------------------- */
size_t sv_d2t_plan_bytes(int32_t V, int32_t Vd);
int sv_d2t_plan_build(const int32_t* d2t, int32_t Vd, int32_t V, void* plan, size_t plan_bytes,
                      sv_stream_t stream);

/* ------------------------------------------------------------------------
 * sv_cfg_merge_sample -- CFG merge per RVQ codebook, then verification.
 * Source: "An Efficient vLLM-Based Inference Pipeline ..." paired CFG
 * co-scheduling and Figure 1 text; sampling rules as in sv_verify_sample.
 *
 *   cond, uncond    logit rows sharing dtype and row_stride; row
 *                   (r * (k + 1) + j) * S + s holds frame j, codebook s of
 *                   request r.  `width` is W, the codebook size.
 *   cb_id_base      HOST int32 [S]: absolute vocabulary id of entry 0 of
 *                   codebook s (the audio partition: the phase mask).
 *   cb_data_offset  HOST int32 [S] or NULL (all 0): element offset of codebook
 *                   s inside its row; offset + W <= row_stride.
 *   S               codebooks, 1 <= S <= SV_MAX_S;  w  CFG weight;  W <= 16384.
 *   draft_logits    draft rows, width W, row (r * k + j) * S + s; data == NULL
 *                   selects greedy verification on the merged logits when k > 0
 *                   (with k = 0 there are no draft rows: a request with T > 0
 *                   draws its bonus from p, as in sv_verify_sample).
 *   draft           int32 [R, k, S] absolute ids.
 *   seeds, temperature  as in sv_verify_sample.
 *   accept_len      int32 [R] out: accepted FRAMES.
 *   tokens          int32 [R, k + 1, S] out: absolute ids, -1 padded.
 *   tv              float [R, k, S] out or NULL;  status int32 [R] out or NULL.
 * The merge is m = u + w (c - u) evaluated in fp32 as d = c - u then
 * fmaf(w, d, u).  A frame is accepted when all S codebooks pass; at the
 * first rejected frame n each codebook keeps its draft if its own test
 * passed, else takes its residual sample (Philox row n * S + s); uniforms of
 * (frame j, codebook s) use Philox row j * S + s.  The residual and bonus
 * draws are the two-level race of sv_verify_sample with 256-id chunks.
 * ---------------------------------------------------------------------- */
size_t sv_cfg_merge_sample_workspace(int32_t R, int32_t k, int32_t S, int32_t W);
int sv_cfg_merge_sample(sv_rows cond, sv_rows uncond, const int32_t* cb_id_base,
                        const int32_t* cb_data_offset, int32_t S, float w,
                        sv_rows draft_logits, int32_t R, int32_t k, const int32_t* draft,
                        const uint64_t* seeds, const float* temperature,
                        int32_t* accept_len, int32_t* tokens, float* tv, int32_t* status,
                        void* workspace, size_t workspace_bytes, sv_stream_t stream);

/* ------------------------------------------------------------------------
 * sv_pool_append / sv_pool_lookup -- the hypothesis pool.
 * Source: "Decode Before You Hear ..." method steps 3 and 5 and the tool-call
 * case study (Figure 6 (b)): every draft of the session enters a pool indexed
 * by n-grams; while the output is unfinished, each later forward first takes
 * the longest n-gram of the pool that matches the emitted suffix and feeds
 * its continuation in as drafts.
 *
 * Pool layout, kept on the device by the caller:
 *   pool        int32 [R, Lp]: request r's drafts in insertion order, each
 *               followed by -1.  Entries at or beyond pool_len[r] are unused
 *               and never read.
 *   pool_len    int32 [R]: entries in use (start a session with 0).  Values
 *               outside [0, Lp] read as a full pool (append) or are clamped
 *               to [0, Lp] (lookup).
 *   Lp          capacity per request, 0 <= Lp <= SV_MAX_POOL.
 *
 * sv_pool_append inserts drafts int32 [R, k] (k <= SV_MAX_K; a negative id
 * ends a draft early, an empty draft inserts nothing).  A draft of L tokens
 * needs L + 1 free entries; when they are not there nothing of it is written
 * and status[r] (int32 [R] out or NULL) gets SV_ST_POOL_FULL.  drafts must
 * not overlap the pool.  Call it once per branch to insert several drafts.
 *
 * sv_pool_lookup:
 *   suffix      int32 [R, N]: the last N emitted tokens, oldest first,
 *               right-aligned; -1 on the left where the output is shorter.
 *               0 <= N <= SV_MAX_NGRAM.
 *   gamma       continuation tokens wanted, 0 <= gamma <= SV_MAX_K.
 *   match_len   int32 [R] out: length n of the match, 0 for none.
 *   cont        int32 [R, gamma] out: the continuation, -1 padded.
 * A match of length n >= 1 ends at pool position p when pool[p-n+1 .. p]
 * equals the last n suffix tokens (none negative, so it lies inside one
 * draft) and pool[p+1] is a token (not a separator).  The longest match
 * wins, then the latest p (the most recently inserted draft).  The
 * continuation is pool[p+1 ..] up to gamma tokens or that draft's end.
 * ---------------------------------------------------------------------- */
int sv_pool_append(int32_t* pool, int32_t* pool_len, int32_t Lp, const int32_t* drafts, int32_t k,
                   int32_t R, int32_t* status, sv_stream_t stream);
int sv_pool_lookup(const int32_t* pool, const int32_t* pool_len, int32_t Lp, const int32_t* suffix,
                   int32_t N, int32_t R, int32_t gamma, int32_t* match_len, int32_t* cont,
                   sv_stream_t stream);

/* sv_suffix_append: the emitted suffix after a verify step, on the device.
 *   suffix      int32 [R, N] in/out, as sv_pool_lookup takes it (oldest first,
 *               -1 on the left where the output is shorter), 0 <= N <= SV_MAX_NGRAM.
 *   tokens      int32 [R, k + 1]: a verify call's tokens; the step committed
 *               tokens[r, 0 .. n], n = accept_len[r] clamped to [0, k].
 *   accept_len  int32 [R].
 * The new suffix is the last N tokens of the old suffix followed by the committed
 * tokens.  tokens and accept_len must not overlap suffix. */
int sv_suffix_append(int32_t* suffix, int32_t N, int32_t R, const int32_t* tokens, const int32_t* accept_len,
                     int32_t k, sv_stream_t stream);

/* ------------------------------------------------------------------------
 * sv_accept_scan -- accept length and commit from caller-given accept flags.
 * Source: "Decode Before You Hear ..." step 4 (the accepted prefix stops at
 * the first failure); "speculative decoding for Omni models" section 3
 * (draft i counts only when drafts 1..i-1 were accepted).
 *
 *   accept      uint8 [R, k], nonzero = accepted.
 *   draft       int32 [R, k].
 *   fix         int32 [R, k + 1]: the token to commit when the chain stops
 *               at position j (j = k: every draft accepted).
 *   accept_len  int32 [R] out;  tokens int32 [R, k + 1] out (-1 padded).
 * ---------------------------------------------------------------------- */
int sv_accept_scan(const uint8_t* accept, const int32_t* draft, const int32_t* fix, int32_t R,
                   int32_t k, int32_t* accept_len, int32_t* tokens, sv_stream_t stream);

/* ------------------------------------------------------------------------
 * sv_selftest_wait_timeout -- a self-test of the library's bounded waits; the
 * source pages have no counterpart.  Every wait of the library on a
 * shared-memory barrier gives up after a time limit and reports
 * SV_ST_TIMEOUT instead of hanging; this call makes one such wait run out on
 * purpose, with the same wait routine and a caller-chosen limit, so a test can
 * check that the timeout path works without any fault.
 *
 *   src16         16 readable, 16-byte aligned device bytes (copied once).
 *   status        int32 [2] out (device): [0] SV_ST_TIMEOUT when the wait
 *                 that cannot complete gave up (the expected result); [1] 1
 *                 when the copy that was issued landed intact.
 *   limit_cycles  the wait's limit in SM cycles (>= 1).
 * Launches one warp on `stream`; nothing is in flight when it exits.
 * ---------------------------------------------------------------------- */
int sv_selftest_wait_timeout(const void* src16, int32_t* status, int64_t limit_cycles, sv_stream_t stream);

#ifdef __cplusplus
}
#endif
#endif /* SPECVERIFY_H */
