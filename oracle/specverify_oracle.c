/*
 * specverify oracle -- a plain, slow, fp64 CPU statement of the speculative
 * verify-and-sample step.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path may call, link or
 * load this file: only the tests, the smoke check and the CPU-baseline leg of
 * the benchmark use it.  It shares no code, header, table or helper with the
 * CUDA library; the only thing both sides see is the seeded synthetic input.
 *
 * Sources followed (page title, section):
 *  [P1] "Decode Before You Hear: Speculative Listening for Chunk-Interleaved
 *       Full-Duplex Speech Language Models" (digest), section "method steps",
 *       step 4: the accepted prefix length n is the index of the first draft
 *       token that differs from argmax p_i (or gamma when none differs); the
 *       correction argmax p_{n+1} is committed, so every pass commits >= 1
 *       token.  Step 2: a runner-up branch whose first token is the best
 *       token other than the main draft's first token, verified in the same
 *       forward pass.  Steps 3 and 5: every draft of the session goes into a
 *       pool indexed by n-grams; while the output continues, the longest
 *       n-gram of the pool matching the emitted suffix supplies its
 *       continuation (the tool-call case study, Figure 6 (b)).
 *  [P3] "speculative decoding for Omni models" (blog), section 2 "why it is
 *       lossless": accept draft x_i with probability min(1, p(x_i)/q(x_i));
 *       on rejection resample from norm(max(0, p - q)) and drop the rest;
 *       if all k drafts are accepted draw one extra token from p.  TV(p,q) =
 *       1/2 sum |p - q| and the single-position acceptance is 1 - TV.
 *       Section 4: a truncated draft vocabulary is mapped into the target
 *       vocabulary by d2t; target ids outside the image have q = 0 and are
 *       always rejected; TV must be taken over the full target vocabulary.
 *  [P2] "An Efficient vLLM-Based Inference Pipeline for Unified Audio
 *       Understanding and Generation" (digest), section on paired CFG
 *       co-scheduling: per codebook, the conditional and unconditional
 *       logits are merged linearly with a weight w > 1 before one token per
 *       codebook is sampled; only the audio partition of the vocabulary is
 *       sampled (Figure 1 text: the vocabulary is split into a text part and
 *       S audio sub-vocabularies).
 *
 * Readings where the pages are silent (each is listed in the design notes):
 *  - softmax with temperature T: p = softmax(z / T); the draft uses the same T.
 *  - T <= 0 (or NaN) selects greedy verification for that request.
 *  - argmax and the sampler break ties toward the lowest index.
 *  - the accept test is the strict comparison u < p/q with u in (0,1).
 *  - the sampler is an exponential race over the whole row: the token is
 *    argmin_x E_x / w_x over the ids with w_x > 0, E_x = -ln u_x, u_x the
 *    Philox4x32-10 uniform of id x keyed by the request seed and counted by
 *    (x >> 2, row, tag, 0), word x & 3; tags 0 accept, 1 residual, 2 bonus.
 *    P(argmin = x) = w_x / sum w, which is the draw from norm(w) the blog
 *    asks for.  The same race serves the full target vocabulary and the CFG
 *    codebook rows.
 *  - the uniform from a 32-bit word r is (2 * (r >> 9) + 1) * 2^-24.
 *  - NaN logits count as -inf.  A sampling request with a NaN, +inf or
 *    all -inf row is verified greedily and flagged (status bit 2).
 *  - CFG merge: m = u + w * (c - u), evaluated in fp32 as d = c - u (one
 *    rounding) then fmaf(w, d, u) (one rounding); greedy CFG compares these
 *    fp32 values, sampling widens them exactly to fp64.
 *  - a CFG frame is accepted when all S codebooks are accepted; at the first
 *    rejected frame each codebook keeps its draft if its own test passed,
 *    else draws its own residual sample.
 *  - hypothesis pool: drafts are stored in insertion order with -1
 *    separators; a match lies inside one draft and must have a token after
 *    it; the longest match wins, then the most recently inserted.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

enum { OR_BF16 = 0, OR_F32 = 1 };

enum {
    OR_ST_TOKEN_RANGE = 1,   /* a draft token outside the vocabulary */
    OR_ST_BAD_LOGITS = 2,    /* NaN / +inf / all -inf row */
    OR_ST_OFF_SUPPORT = 4,   /* draft token has q = 0 */
    OR_ST_RESIDUAL_ZERO = 8, /* residual mass was 0, sampled from p instead */
    OR_ST_BAD_TEMP = 16,     /* temperature negative or NaN: greedy used */
    OR_ST_BAD_D2T = 32       /* d2t entry out of range or repeated */
};

enum { TAG_ACCEPT = 0, TAG_RESIDUAL = 1, TAG_BONUS = 2 };

/* ------------------------------------------------------------------ */
/* Philox4x32-10, from Salmon, Moraes, Dror, Shaw, "Parallel Random    */
/* Numbers: As Easy as 1, 2, 3" (SC'11): ten rounds of two 32x32->64    */
/* multiplies, the high halves xor-ed with the other two counter words */
/* and the round key; the key is bumped by the Weyl constants between  */
/* rounds.                                                              */
/* ------------------------------------------------------------------ */
#define PHILOX_MUL_A 0xD2511F53u
#define PHILOX_MUL_B 0xCD9E8D57u
#define PHILOX_WEYL_A 0x9E3779B9u
#define PHILOX_WEYL_B 0xBB67AE85u

void or_philox4x32_10(const uint32_t ctr_in[4], const uint32_t key_in[2], uint32_t out[4])
{
    uint32_t c0 = ctr_in[0], c1 = ctr_in[1], c2 = ctr_in[2], c3 = ctr_in[3];
    uint32_t k0 = key_in[0], k1 = key_in[1];
    for (int round = 0; round < 10; ++round) {
        if (round > 0) {
            k0 += PHILOX_WEYL_A;
            k1 += PHILOX_WEYL_B;
        }
        uint64_t prod_a = (uint64_t)PHILOX_MUL_A * (uint64_t)c0;
        uint64_t prod_b = (uint64_t)PHILOX_MUL_B * (uint64_t)c2;
        uint32_t hi_a = (uint32_t)(prod_a >> 32), lo_a = (uint32_t)prod_a;
        uint32_t hi_b = (uint32_t)(prod_b >> 32), lo_b = (uint32_t)prod_b;
        uint32_t n0 = hi_b ^ c1 ^ k0;
        uint32_t n1 = lo_b;
        uint32_t n2 = hi_a ^ c3 ^ k1;
        uint32_t n3 = lo_a;
        c0 = n0; c1 = n1; c2 = n2; c3 = n3;
    }
    out[0] = c0; out[1] = c1; out[2] = c2; out[3] = c3;
}

/* uniform in (0,1): odd multiples of 2^-24, exact in fp32 and fp64 */
double or_uniform_from_word(uint32_t r)
{
    return ldexp(2.0 * (double)(r >> 9) + 1.0, -24);
}

/* the uniform for element x of (seed, row, tag) */
double or_uniform(uint64_t seed, uint32_t row, uint32_t tag, uint32_t x)
{
    uint32_t ctr[4] = { x >> 2, row, tag, 0u };
    uint32_t key[2] = { (uint32_t)(seed & 0xffffffffu), (uint32_t)(seed >> 32) };
    uint32_t out[4];
    or_philox4x32_10(ctr, key, out);
    return or_uniform_from_word(out[x & 3u]);
}

/* ------------------------------------------------------------------ */
/* element access                                                      */
/* ------------------------------------------------------------------ */
static double load_elem(const void* base, int dtype, int64_t idx)
{
    if (dtype == OR_BF16) {
        uint32_t bits = (uint32_t)((const uint16_t*)base)[idx] << 16;
        float f;
        memcpy(&f, &bits, sizeof f);
        return (double)f;
    }
    return (double)((const float*)base)[idx];
}

static float load_elem_f32(const void* base, int dtype, int64_t idx)
{
    if (dtype == OR_BF16) {
        uint32_t bits = (uint32_t)((const uint16_t*)base)[idx] << 16;
        float f;
        memcpy(&f, &bits, sizeof f);
        return f;
    }
    return ((const float*)base)[idx];
}

/* a row is "bad" for sampling when it holds NaN or +inf, or is all -inf */
static int row_is_bad(const double* z, int32_t n)
{
    int any_finite = 0;
    for (int32_t x = 0; x < n; ++x) {
        if (isnan(z[x]) || (isinf(z[x]) && z[x] > 0)) return 1;
        if (!isinf(z[x])) any_finite = 1;
    }
    return !any_finite;
}

/* argmax with NaN read as -inf, lowest index among equal maxima */
static int32_t argmax_row(const double* z, int32_t n)
{
    int32_t best = 0;
    double best_v = -INFINITY;
    for (int32_t x = 0; x < n; ++x) {
        double v = isnan(z[x]) ? -INFINITY : z[x];
        if (v > best_v) {
            best_v = v;
            best = x;
        }
    }
    return best;
}

/* the two ids ranked first when ids are ordered by value (descending), then
 * by id (ascending), NaN read as -inf: the argmax and the runner-up of a row
 * ([SL] "method steps", step 2: the runner-up branch starts from the second-best
 * token of the verified row).  second = -1 for a one-id row. */
static void top2_row(const double* z, int32_t n, int32_t* first, int32_t* second)
{
    int32_t a = -1, b = -1;
    double av = -INFINITY, bv = -INFINITY;
    for (int32_t x = 0; x < n; ++x) {  /* ascending ids: an equal value never displaces */
        double v = isnan(z[x]) ? -INFINITY : z[x];
        if (a < 0 || v > av) {
            b = a;
            bv = av;
            a = x;
            av = v;
        } else if (b < 0 || v > bv) {
            b = x;
            bv = v;
        }
    }
    *first = a < 0 ? 0 : a;
    *second = b;
}

int or_top2_rows(const void* rows, int dtype, int64_t row_stride, int64_t nrows, int32_t V,
                 int32_t* top2)
{
    if (V < 1 || nrows < 0) return -1;
    double* z = (double*)malloc(sizeof(double) * (size_t)V);
    for (int64_t r = 0; r < nrows; ++r) {
        for (int32_t x = 0; x < V; ++x) z[x] = load_elem(rows, dtype, r * row_stride + x);
        top2_row(z, V, &top2[2 * r], &top2[2 * r + 1]);
    }
    free(z);
    return 0;
}

/* modality of a row of the full vocabulary ("An Efficient vLLM-Based
 * Inference Pipeline ..." phase management: the vocabulary is split into a
 * text part and S audio sub-vocabularies, and the current modality is the
 * partition holding the maximum of the unmasked distribution): per row the
 * argmax (NaN read as -inf, lowest id), the partition p with
 * part_start[p] <= argmax < part_start[p + 1] (-1 when none), and that
 * partition's id range [lo, hi) as the phase mask of the next step (0, 0
 * when none).  part_start holds P + 1 ascending ids. */
int or_infer_modality(const void* rows, int dtype, int64_t row_stride, int64_t nrows, int32_t V,
                      const int32_t* part_start, int32_t P, int32_t* amax, int32_t* part,
                      int32_t* mask_lo, int32_t* mask_hi)
{
    if (V < 1 || nrows < 0 || P < 1) return -1;
    for (int32_t p = 0; p < P; ++p)
        if (part_start[p] > part_start[p + 1]) return -1;
    double* z = (double*)malloc(sizeof(double) * (size_t)V);
    for (int64_t r = 0; r < nrows; ++r) {
        for (int32_t x = 0; x < V; ++x) z[x] = load_elem(rows, dtype, r * row_stride + x);
        const int32_t a = argmax_row(z, V);
        int32_t pi = -1;
        for (int32_t p = 0; p < P; ++p)
            if (part_start[p] <= a && a < part_start[p + 1]) {
                pi = p;
                break;
            }
        amax[r] = a;
        part[r] = pi;
        mask_lo[r] = pi < 0 ? 0 : part_start[pi];
        mask_hi[r] = pi < 0 ? 0 : part_start[pi + 1];
    }
    free(z);
    return 0;
}

/* p = softmax(z / T) in fp64; NaN read as -inf.  Caller ensures the row
 * is not bad. */
static void softmax_T(const double* z, int32_t n, double T, double* p)
{
    double m = -INFINITY;
    for (int32_t x = 0; x < n; ++x) {
        double t = isnan(z[x]) ? -INFINITY : z[x] / T;
        p[x] = t;
        if (t > m) m = t;
    }
    double s = 0.0;
    for (int32_t x = 0; x < n; ++x) {
        p[x] = exp(p[x] - m);
        s += p[x];
    }
    for (int32_t x = 0; x < n; ++x) p[x] /= s;
}

/* exponential race over the weights w[x0..x1) >= 0: argmin_{w_x > 0} E_x / w_x
 * with E_x = -ln u_x, u_x the uniform of the absolute id x.  Returns -1 if
 * every weight is 0.  *margin receives (key2 - key1) / key1 for the two
 * smallest keys (INFINITY if only one). */
static int32_t race_span(const double* w, int32_t x0, int32_t x1, uint64_t seed, uint32_t row,
                         uint32_t tag, double* margin)
{
    int32_t arg = -1;
    double best = INFINITY, second = INFINITY;
    for (int32_t x = x0; x < x1; ++x) {
        if (!(w[x] > 0.0)) continue;
        double e = -log(or_uniform(seed, row, tag, (uint32_t)x));
        double key = e / w[x];
        if (key < best) {
            second = best;
            best = key;
            arg = x;
        } else if (key < second) {
            second = key;
        }
    }
    if (margin) *margin = (arg >= 0 && isfinite(second)) ? (second - best) / best : INFINITY;
    return arg;
}

int32_t or_race(const double* w, int32_t n, uint64_t seed, uint32_t row, uint32_t tag,
                double* margin)
{
    return race_span(w, 0, n, seed, row, tag, margin);
}

/* ------------------------------------------------------------------ */
/* hypothesis pool ([SL] "method steps" 3 and 5: every draft of the      */
/* session goes into a pool indexed by n-grams; while the output         */
/* continues, the longest n-gram of the pool matching the emitted suffix */
/* supplies its continuation as the next drafts).                        */
/* A request's pool is int32 [Lp]: its drafts in insertion order, each   */
/* followed by -1; pool_len[r] entries are in use.                       */
/* ------------------------------------------------------------------ */

/* append: draft r is drafts[r, 0 .. L) with L the first index holding a */
/* negative id (k if none).  L == 0 inserts nothing.  When pool_len + L  */
/* + 1 exceeds Lp (or pool_len is outside [0, Lp]) nothing is inserted   */
/* and status bit 128 is set.                                            */
int or_pool_append(int32_t* pool, int32_t* pool_len, int32_t Lp, const int32_t* drafts, int32_t k,
                   int32_t R, int32_t* status)
{
    if (Lp < 0 || k < 0 || R < 0) return -1;
    for (int32_t r = 0; r < R; ++r) {
        const int32_t* D = drafts + (int64_t)r * k;
        int32_t L = 0;
        while (L < k && D[L] >= 0) ++L;
        status[r] = 0;
        if (L == 0) continue;
        const int32_t used = pool_len[r];
        if (used < 0 || used > Lp || (int64_t)used + L + 1 > Lp) {
            status[r] = 128;
            continue;
        }
        int32_t* P = pool + (int64_t)r * Lp;
        for (int32_t i = 0; i < L; ++i) P[used + i] = D[i];
        P[used + L] = -1;
        pool_len[r] = used + L + 1;
    }
    return 0;
}

/* lookup: suffix [R, N] holds the last N emitted tokens, -1 where the   */
/* output is shorter (left side).  A match of length n >= 1 ends at pool */
/* position p when pool[p - n + 1 .. p] equals the last n suffix tokens  */
/* (all >= 0, so inside one draft) and pool[p + 1] >= 0 (a continuation */
/* exists), with p + 1 < len, len = pool_len[r] clamped to [0, Lp].  The */
/* longest match wins, the latest p among equal lengths; the             */
/* continuation is pool[p + 1 ..] up to gamma tokens or the draft's end, */
/* -1 padded.  match_len 0: no continuation.                             */
int or_pool_lookup(const int32_t* pool, const int32_t* pool_len, int32_t Lp, const int32_t* suffix,
                   int32_t N, int32_t R, int32_t gamma, int32_t* match_len, int32_t* cont)
{
    if (Lp < 0 || N < 0 || R < 0 || gamma < 0) return -1;
    for (int32_t r = 0; r < R; ++r) {
        const int32_t* P = pool + (int64_t)r * Lp;
        const int32_t* S = suffix + (int64_t)r * N;
        int32_t len = pool_len[r];
        if (len < 0) len = 0;
        if (len > Lp) len = Lp;
        int32_t best_n = 0, best_p = -1;
        for (int32_t p = 0; p + 1 < len; ++p) {
            if (P[p + 1] < 0) continue;  /* no continuation after p */
            int32_t n = 0;
            while (n < N && p - n >= 0 && P[p - n] >= 0 && S[N - 1 - n] >= 0 && P[p - n] == S[N - 1 - n]) ++n;
            if (n > 0 && n >= best_n) {  /* ascending p: the latest among equal lengths */
                best_n = n;
                best_p = p;
            }
        }
        match_len[r] = best_n;
        int32_t* out = cont + (int64_t)r * gamma;
        int32_t i = 0;
        if (best_p >= 0)
            for (; i < gamma && best_p + 1 + i < len && P[best_p + 1 + i] >= 0; ++i) out[i] = P[best_p + 1 + i];
        for (; i < gamma; ++i) out[i] = -1;
    }
    return 0;
}

/* suffix update after a verify step: the tokens a step commits are its  */
/* n accepted drafts and the correction, tokens[r, 0 .. n] with n =      */
/* accept_len[r] (clamped to [0, k]); the emitted suffix [R, N] (oldest  */
/* first, -1 on the left where the output is shorter) becomes the last N */
/* tokens of the old suffix followed by them.                            */
int or_suffix_append(int32_t* suffix, int32_t N, int32_t R, const int32_t* tokens, const int32_t* accept_len,
                     int32_t k)
{
    if (N < 0 || R < 0 || k < 0) return -1;
    int32_t* all = (int32_t*)malloc(sizeof(int32_t) * (size_t)(N + k + 1));
    for (int32_t r = 0; r < R; ++r) {
        int32_t n = accept_len[r];
        if (n < 0) n = 0;
        if (n > k) n = k;
        int32_t m = 0;
        for (int32_t i = 0; i < N; ++i) all[m++] = suffix[(int64_t)r * N + i];
        for (int32_t j = 0; j <= n; ++j) all[m++] = tokens[(int64_t)r * (k + 1) + j];
        for (int32_t i = 0; i < N; ++i) suffix[(int64_t)r * N + i] = all[m - N + i];
    }
    free(all);
    return 0;
}

/* ------------------------------------------------------------------ */
/* accept-length scan over caller-given accept flags ([P1] step 4,      */
/* [P3] section 3: draft i counts only if drafts 0..i-1 were accepted)  */
/* ------------------------------------------------------------------ */
int or_accept_scan(const uint8_t* accept, const int32_t* draft, const int32_t* fix, int32_t R,
                   int32_t k, int32_t* accept_len, int32_t* tokens)
{
    for (int32_t r = 0; r < R; ++r) {
        int32_t n = 0;
        while (n < k && accept[(int64_t)r * k + n]) ++n;
        int32_t* out = tokens + (int64_t)r * (k + 1);
        for (int32_t j = 0; j <= k; ++j) out[j] = -1;
        for (int32_t j = 0; j < n; ++j) out[j] = draft[(int64_t)r * k + j];
        out[n] = fix[(int64_t)r * (k + 1) + n];
        accept_len[r] = n;
    }
    return 0;
}

/* ------------------------------------------------------------------ */
/* greedy verification ([P1] step 4, with the step-2 runner-up branch)  */
/* target rows per request: 1 + branches * k: p_1 shared, then each    */
/* branch's p_2..p_{k+1} ([p_1 | main | runner | ...]; branches == 1:   */
/* k + 1 rows).  More than two branches are tree drafts whose first    */
/* tokens differ.                                                      */
/* ------------------------------------------------------------------ */
static int64_t branch_row(int32_t b, int32_t j, int32_t k)
{
    return j == 0 ? 0 : (int64_t)b * k + j;
}

int or_verify_greedy(const void* target, int dtype, int64_t row_stride, int32_t V, int32_t R,
                     int32_t k, int32_t branches, const int32_t* draft, int32_t* accept_len,
                     int32_t* tokens, int32_t* branch_out, int32_t* status)
{
    if (branches < 1 || branches > 8 || k < 0 || (branches >= 2 && k < 1)) return -1;
    const int32_t rows_per_req = 1 + branches * k;
    double* z = (double*)malloc(sizeof(double) * (size_t)(V > 0 ? V : 1));
    int32_t* amax = (int32_t*)malloc(sizeof(int32_t) * (size_t)rows_per_req);
    for (int32_t r = 0; r < R; ++r) {
        int32_t st = 0;
        for (int32_t i = 0; i < rows_per_req; ++i) {
            int64_t row = (int64_t)r * rows_per_req + i;
            for (int32_t x = 0; x < V; ++x) z[x] = load_elem(target, dtype, row * row_stride + x);
            if (row_is_bad(z, V)) st |= OR_ST_BAD_LOGITS;
            amax[i] = argmax_row(z, V);
        }
        int32_t best_b = 0, best_n = 0, any_viable = 0;
        for (int32_t b = 0; b < branches; ++b) {
            const int32_t* d = draft + ((int64_t)r * branches + b) * k;
            int32_t n = 0;
            for (int32_t j = 0; j < k; ++j)
                if (d[j] < 0 || d[j] >= V) st |= OR_ST_TOKEN_RANGE;
            while (n < k && d[n] == amax[branch_row(b, n, k)]) ++n;
            int viable = (k == 0) || (n >= 1);
            if (viable && (!any_viable || n > best_n)) {
                best_b = b;
                best_n = n;
                any_viable = 1;
            }
        }
        if (!any_viable) {
            best_b = 0;
            best_n = 0;
        }
        const int32_t* d = draft + ((int64_t)r * branches + best_b) * k;
        int32_t* out = tokens + (int64_t)r * (k + 1);
        for (int32_t j = 0; j <= k; ++j) out[j] = -1;
        for (int32_t j = 0; j < best_n; ++j) out[j] = d[j];
        out[best_n] = amax[branch_row(best_b, best_n, k)];
        accept_len[r] = best_n;
        if (branch_out) branch_out[r] = best_b;
        if (status) status[r] = st;
    }
    free(z);
    free(amax);
    return 0;
}

/* ------------------------------------------------------------------ */
/* speculative sampling ([P3] section 2) with a truncated draft         */
/* vocabulary ([P3] section 4).                                         */
/* target rows per request: k + 1 (positions 0..k-1, bonus row k);      */
/* draft rows per request: k, each over Vd draft ids; d2t maps draft id */
/* -> target id (NULL: identity, Vd == V).                              */
/* Optional outputs (NULL to skip): tv, p_draft, q_draft [R,k];         */
/* accept_margin [R,k] = |u - p/q| (INFINITY where no test was made);   */
/* race_margin [R] (INFINITY for greedy requests).                      */
/* ------------------------------------------------------------------ */
int or_verify_sample(const void* target, int t_dtype, int64_t t_stride, int32_t V,
                     const void* draft_logits, int d_dtype, int64_t d_stride, int32_t Vd,
                     const int32_t* d2t, int32_t R, int32_t k, const int32_t* draft,
                     const uint64_t* seeds, const float* temperature, int32_t* accept_len,
                     int32_t* tokens, double* tv, double* p_draft, double* q_draft,
                     int32_t* status, double* accept_margin, double* race_margin)
{
    if (k < 0 || V < 1 || Vd < 1) return -1;
    if (!d2t && Vd != V) return -1;
    /* t2d: target id -> draft id, -1 off the draft support */
    int32_t* t2d = (int32_t*)malloc(sizeof(int32_t) * (size_t)V);
    int bad_d2t = 0;
    for (int32_t x = 0; x < V; ++x) t2d[x] = d2t ? -1 : x;
    if (d2t) {
        for (int32_t jd = 0; jd < Vd; ++jd) {
            int32_t x = d2t[jd];
            if (x < 0 || x >= V || t2d[x] >= 0) {
                bad_d2t = 1;
                continue;
            }
            t2d[x] = jd;
        }
    }
    double* z = (double*)malloc(sizeof(double) * (size_t)V);
    double* y = (double*)malloc(sizeof(double) * (size_t)Vd);
    double* p = (double*)malloc(sizeof(double) * (size_t)V);
    double* qt = (double*)malloc(sizeof(double) * (size_t)Vd);
    double* qx = (double*)malloc(sizeof(double) * (size_t)V); /* q in target space */
    double* w = (double*)malloc(sizeof(double) * (size_t)V);
    int32_t* amax = (int32_t*)malloc(sizeof(int32_t) * (size_t)(k + 1));

    for (int32_t r = 0; r < R; ++r) {
        int32_t st = bad_d2t ? OR_ST_BAD_D2T : 0;
        const double T = (double)temperature[r];
        const int32_t* d = draft + (int64_t)r * k;
        int32_t* out = tokens + (int64_t)r * (k + 1);
        for (int32_t j = 0; j <= k; ++j) out[j] = -1;
        for (int32_t j = 0; j < k; ++j) {
            if (d[j] < 0 || d[j] >= V) st |= OR_ST_TOKEN_RANGE;
            if (tv) tv[(int64_t)r * k + j] = NAN;
            if (p_draft) p_draft[(int64_t)r * k + j] = NAN;
            if (q_draft) q_draft[(int64_t)r * k + j] = NAN;
            if (accept_margin) accept_margin[(int64_t)r * k + j] = INFINITY;
        }
        if (race_margin) race_margin[r] = INFINITY;

        /* validity of every row the request uses, and raw argmaxes */
        int greedy = !(T > 0.0);
        if (T < 0.0 || isnan(T)) st |= OR_ST_BAD_TEMP;
        for (int32_t j = 0; j <= k; ++j) {
            int64_t row = (int64_t)r * (k + 1) + j;
            for (int32_t x = 0; x < V; ++x) z[x] = load_elem(target, t_dtype, row * t_stride + x);
            amax[j] = argmax_row(z, V);
            if (row_is_bad(z, V)) st |= OR_ST_BAD_LOGITS;
        }
        if (!greedy) {
            for (int32_t j = 0; j < k; ++j) {
                int64_t row = (int64_t)r * k + j;
                for (int32_t jd = 0; jd < Vd; ++jd)
                    y[jd] = load_elem(draft_logits, d_dtype, row * d_stride + jd);
                if (row_is_bad(y, Vd)) st |= OR_ST_BAD_LOGITS;
            }
        }
        if (st & OR_ST_BAD_LOGITS) greedy = 1;

        if (greedy) {
            int32_t n = 0;
            while (n < k && d[n] == amax[n]) ++n;
            for (int32_t j = 0; j < n; ++j) out[j] = d[j];
            out[n] = amax[n];
            accept_len[r] = n;
            if (status) status[r] = st;
            continue;
        }

        /* sampling: positions in order until the first rejection */
        int32_t n = k;
        for (int32_t j = 0; j < k; ++j) {
            int64_t trow = (int64_t)r * (k + 1) + j;
            int64_t drow = (int64_t)r * k + j;
            for (int32_t x = 0; x < V; ++x) z[x] = load_elem(target, t_dtype, trow * t_stride + x);
            for (int32_t jd = 0; jd < Vd; ++jd)
                y[jd] = load_elem(draft_logits, d_dtype, drow * d_stride + jd);
            softmax_T(z, V, T, p);
            softmax_T(y, Vd, T, qt);
            for (int32_t x = 0; x < V; ++x) qx[x] = t2d[x] >= 0 ? qt[t2d[x]] : 0.0;
            /* TV over the full target vocabulary */
            double acc = 0.0;
            for (int32_t x = 0; x < V; ++x) acc += fabs(p[x] - qx[x]);
            const int32_t xj = d[j];
            const double pd = (xj >= 0 && xj < V) ? p[xj] : 0.0;
            const double qd = (xj >= 0 && xj < V) ? qx[xj] : 0.0;
            if (tv) tv[drow] = 0.5 * acc;
            if (p_draft) p_draft[drow] = pd;
            if (q_draft) q_draft[drow] = qd;
            if (n < k) continue; /* statistics only, the chain already stopped */
            int accepted = 0;
            if (qd > 0.0) {
                double u = or_uniform(seeds[r], (uint32_t)j, TAG_ACCEPT, 0u);
                accepted = u < pd / qd;
                if (accept_margin) accept_margin[drow] = fabs(u - pd / qd);
            } else if (xj >= 0 && xj < V) {
                st |= OR_ST_OFF_SUPPORT;
            }
            if (!accepted) {
                /* residual max(0, p - q) on this row */
                n = j;
                double mass = 0.0;
                for (int32_t x = 0; x < V; ++x) {
                    w[x] = p[x] - qx[x] > 0.0 ? p[x] - qx[x] : 0.0;
                    mass += w[x];
                }
                double mg;
                int32_t tok;
                if (mass > 0.0) {
                    tok = or_race(w, V, seeds[r], (uint32_t)j, TAG_RESIDUAL, &mg);
                } else {
                    st |= OR_ST_RESIDUAL_ZERO;
                    tok = or_race(p, V, seeds[r], (uint32_t)j, TAG_RESIDUAL, &mg);
                }
                out[n] = tok;
                if (race_margin) race_margin[r] = mg;
            }
        }
        if (n == k) {
            /* every draft accepted: bonus token from p on row k */
            int64_t trow = (int64_t)r * (k + 1) + k;
            for (int32_t x = 0; x < V; ++x) z[x] = load_elem(target, t_dtype, trow * t_stride + x);
            softmax_T(z, V, T, p);
            double mg;
            out[k] = or_race(p, V, seeds[r], (uint32_t)k, TAG_BONUS, &mg);
            if (race_margin) race_margin[r] = mg;
        }
        for (int32_t j = 0; j < n; ++j) out[j] = d[j];
        accept_len[r] = n;
        if (status) status[r] = st;
    }
    free(t2d); free(z); free(y); free(p); free(qt); free(qx); free(w); free(amax);
    return 0;
}

/* ------------------------------------------------------------------ */
/* CFG merge per codebook, then verify ([P2] paired CFG; [P3] sec. 2).  */
/* Row (r, frame j, codebook s) is row (r * (k + 1) + j) * S + s of     */
/* cond / uncond; its codebook slice starts at element cb_data_offset[s]*/
/* and has W entries; local id l is absolute id cb_id_base[s] + l.      */
/* Draft logit rows: (r * k + j) * S + s, W entries from element 0.     */
/* T <= 0, or draft_logits == NULL with k > 0: greedy on the merged logits. */
/* Optional: tv [R,k,S], accept_margin [R,k,S], race_margin [R,S].      */
/* ------------------------------------------------------------------ */
static void merged_row(const void* cond, const void* uncond, int dtype, int64_t stride,
                       int64_t row, int32_t off, int32_t W, float wgt, float* m)
{
    for (int32_t l = 0; l < W; ++l) {
        float c = load_elem_f32(cond, dtype, row * stride + off + l);
        float u = load_elem_f32(uncond, dtype, row * stride + off + l);
        float dlt = c - u;        /* one fp32 rounding */
        m[l] = fmaf(wgt, dlt, u); /* one fp32 rounding */
    }
}

int or_cfg_merge_sample(const void* cond, const void* uncond, int dtype, int64_t stride,
                        const int32_t* cb_id_base, const int32_t* cb_data_offset, int32_t S,
                        int32_t W, float wgt, const void* draft_logits, int d_dtype,
                        int64_t d_stride, int32_t R, int32_t k, const int32_t* draft,
                        const uint64_t* seeds, const float* temperature, int32_t* accept_len,
                        int32_t* tokens, double* tv, int32_t* status, double* accept_margin,
                        double* race_margin)
{
    if (S < 1 || W < 1 || k < 0) return -1;
    float* m = (float*)malloc(sizeof(float) * (size_t)W);
    double* zd = (double*)malloc(sizeof(double) * (size_t)W);
    double* y = (double*)malloc(sizeof(double) * (size_t)W);
    double* p = (double*)malloc(sizeof(double) * (size_t)W);
    double* q = (double*)malloc(sizeof(double) * (size_t)W);
    double* w = (double*)malloc(sizeof(double) * (size_t)W);
    int32_t* amax = (int32_t*)malloc(sizeof(int32_t) * (size_t)(k + 1) * S);
    uint8_t* acc = (uint8_t*)malloc((size_t)(k > 0 ? k : 1) * S);

    for (int32_t r = 0; r < R; ++r) {
        int32_t st = 0;
        const double T = (double)temperature[r];
        /* NULL draft logits select greedy verification when there are draft rows; with k = 0
           the bonus follows the temperature alone (drawn from p when T > 0) */
        int greedy = !(T > 0.0) || (draft_logits == NULL && k > 0);
        if (T < 0.0 || isnan(T)) st |= OR_ST_BAD_TEMP;
        const int32_t* d = draft + (int64_t)r * k * S;
        int32_t* out = tokens + (int64_t)r * (k + 1) * S;
        for (int64_t i = 0; i < (int64_t)(k + 1) * S; ++i) out[i] = -1;
        for (int64_t i = 0; i < (int64_t)k * S; ++i) {
            if (tv) tv[(int64_t)r * k * S + i] = NAN;
            if (accept_margin) accept_margin[(int64_t)r * k * S + i] = INFINITY;
        }
        for (int32_t s = 0; s < S; ++s)
            if (race_margin) race_margin[(int64_t)r * S + s] = INFINITY;
        for (int32_t j = 0; j < k; ++j)
            for (int32_t s = 0; s < S; ++s) {
                int32_t l = d[j * S + s] - cb_id_base[s];
                if (l < 0 || l >= W) st |= OR_ST_TOKEN_RANGE;
            }
        /* merged argmaxes and row validity */
        for (int32_t j = 0; j <= k; ++j)
            for (int32_t s = 0; s < S; ++s) {
                int64_t row = ((int64_t)r * (k + 1) + j) * S + s;
                merged_row(cond, uncond, dtype, stride, row, cb_data_offset[s], W, wgt, m);
                for (int32_t l = 0; l < W; ++l) zd[l] = (double)m[l];
                amax[j * S + s] = argmax_row(zd, W);
                if (row_is_bad(zd, W)) st |= OR_ST_BAD_LOGITS;
            }
        if (!greedy) {
            for (int32_t j = 0; j < k; ++j)
                for (int32_t s = 0; s < S; ++s) {
                    int64_t row = ((int64_t)r * k + j) * S + s;
                    for (int32_t l = 0; l < W; ++l)
                        y[l] = load_elem(draft_logits, d_dtype, row * d_stride + l);
                    if (row_is_bad(y, W)) st |= OR_ST_BAD_LOGITS;
                }
        }
        if (st & OR_ST_BAD_LOGITS) greedy = 1;

        if (greedy) {
            int32_t n = 0;
            while (n < k) {
                int all = 1;
                for (int32_t s = 0; s < S; ++s)
                    if (d[n * S + s] - cb_id_base[s] != amax[n * S + s]) all = 0;
                if (!all) break;
                ++n;
            }
            for (int32_t j = 0; j < n; ++j)
                for (int32_t s = 0; s < S; ++s) out[j * S + s] = d[j * S + s];
            for (int32_t s = 0; s < S; ++s) out[n * S + s] = cb_id_base[s] + amax[n * S + s];
            accept_len[r] = n;
            if (status) status[r] = st;
            continue;
        }

        /* every (frame, codebook) test and TV; the chain stops at the first
         * frame with a rejected codebook */
        int32_t n = k;
        for (int32_t j = 0; j < k; ++j) {
            int frame_ok = 1;
            for (int32_t s = 0; s < S; ++s) {
                int64_t row = ((int64_t)r * (k + 1) + j) * S + s;
                int64_t drow = ((int64_t)r * k + j) * S + s;
                merged_row(cond, uncond, dtype, stride, row, cb_data_offset[s], W, wgt, m);
                for (int32_t l = 0; l < W; ++l) zd[l] = (double)m[l];
                for (int32_t l = 0; l < W; ++l)
                    y[l] = load_elem(draft_logits, d_dtype, drow * d_stride + l);
                softmax_T(zd, W, T, p);
                softmax_T(y, W, T, q);
                double a = 0.0;
                for (int32_t l = 0; l < W; ++l) a += fabs(p[l] - q[l]);
                if (tv) tv[drow] = 0.5 * a;
                int32_t l = d[j * S + s] - cb_id_base[s];
                int ok = 0;
                if (l >= 0 && l < W && q[l] > 0.0) {
                    uint32_t urow = (uint32_t)(j * S + s);
                    double u = or_uniform(seeds[r], urow, TAG_ACCEPT, 0u);
                    ok = u < p[l] / q[l];
                    if (accept_margin && j <= n) accept_margin[drow] = fabs(u - p[l] / q[l]);
                }
                acc[j * S + s] = (uint8_t)ok;
                if (!ok) frame_ok = 0;
            }
            if (!frame_ok && n == k) n = j;
        }
        for (int32_t j = 0; j < n; ++j)
            for (int32_t s = 0; s < S; ++s) out[j * S + s] = d[j * S + s];
        for (int32_t s = 0; s < S; ++s) {
            int64_t row = ((int64_t)r * (k + 1) + n) * S + s;
            uint32_t urow = (uint32_t)(n * S + s);
            merged_row(cond, uncond, dtype, stride, row, cb_data_offset[s], W, wgt, m);
            for (int32_t l = 0; l < W; ++l) zd[l] = (double)m[l];
            softmax_T(zd, W, T, p);
            double mg = INFINITY;
            int32_t tok;
            if (n == k) {
                tok = or_race(p, W, seeds[r], urow, TAG_BONUS, &mg);
            } else if (acc[n * S + s]) {
                tok = d[n * S + s] - cb_id_base[s];
            } else {
                int64_t drow = ((int64_t)r * k + n) * S + s;
                for (int32_t l = 0; l < W; ++l)
                    y[l] = load_elem(draft_logits, d_dtype, drow * d_stride + l);
                softmax_T(y, W, T, q);
                double mass = 0.0;
                for (int32_t l = 0; l < W; ++l) {
                    w[l] = p[l] - q[l] > 0.0 ? p[l] - q[l] : 0.0;
                    mass += w[l];
                }
                int32_t ld = d[n * S + s] - cb_id_base[s];
                if (!(ld >= 0 && ld < W && q[ld] > 0.0) && ld >= 0 && ld < W)
                    st |= OR_ST_OFF_SUPPORT;
                if (mass > 0.0) {
                    tok = or_race(w, W, seeds[r], urow, TAG_RESIDUAL, &mg);
                } else {
                    st |= OR_ST_RESIDUAL_ZERO;
                    tok = or_race(p, W, seeds[r], urow, TAG_RESIDUAL, &mg);
                }
            }
            out[n * S + s] = cb_id_base[s] + tok;
            if (race_margin) race_margin[(int64_t)r * S + s] = mg;
        }
        accept_len[r] = n;
        if (status) status[r] = st;
    }
    free(m); free(zd); free(y); free(p); free(q); free(w); free(amax); free(acc);
    return 0;
}
