/*
 * oracle.c -- plain CPU oracle for DGQ KV-cache compression and INT8 paged decode
 * attention.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the tests, the smoke check and the benchmark's CPU
 * baseline load this library; the product path (libdgq.so) never does, and this file
 * shares no code, header, table or constant with it.  It is deliberately slow and
 * single-threaded: every step is written out in the order the sources give it, one
 * IEEE-754 operation at a time, so that it can be checked against them by eye.
 * Build flags: -O2 -ffp-contract=off (no FMA contraction; no fast-math).
 *
 * Sources (cited by title and section):
 *   [DGQ]   "DeepSeek KV-cache dynamic group quantisation (DGQ)" article, pptc.cn news 101026
 *           §2.2  per-head variance curve along L, 16-token windows, jump detection,
 *                 3-5 segments, independent min/max INT8 per segment, segment ids
 *           §3.2  length-aware n_groups rule inside compress()
 *           §3.3  storage formula (INT8 body + per-token segment marker)
 *   [PAGED] "DeepSeek-V4 high-concurrency KV-cache bottleneck" article (deepseek.csdn.net),
 *           "PagedAttention implementation" section: logical blocks mapped to scattered
 *           physical blocks through a block table.
 *   Where the articles leave a step open, the readings below are the plainest ones the
 *   rest supports; each is marked READING.
 *
 * Parity pins (tests/test_oracle_*.py check this file against them):
 *   n_groups       closed-form table of the [DGQ] §3.2 rule at its edges
 *   variance       fp64 variance within the fp32 error bound; constant rows -> 0
 *   window means   fp64 mean within bound; exact for partial windows of equal values
 *   boundaries     planted variance steps recovered exactly; brute force over all
 *                  k-subsets of windows on tiny inputs
 *   seg min/max    brute-force numpy min/max over each segment slice
 *   codes          min -> 0, max -> 255, |dequant - x| <= scale/2 (+fp32 slack),
 *                  monotone in x; one segment == textbook per-tensor asymmetric uint8
 *   paging         gather through the block table reproduces the unpaged codes;
 *                  bytes written == 1 B/element + one 128-byte record per (request, head)
 *   attention      numpy fp64 brute force; two-key closed form; uniform average for
 *                  equal keys; invariance under any permutation of physical blocks
 *   settings       max_groups = 1 gives one segment; a cap gives the top jumps of the uncapped
 *                  rule; a floor above every window mean gives one segment; planted quiet /
 *                  loud regions give boundaries only at loud transitions; brute force over
 *                  the candidate subsets on tiny inputs
 *   comparisons    fixed-64 groups: two-valued groups round-trip exactly, error <= scale/2;
 *                  symmetric INT8: values on the k * max/127 grid round-trip exactly; E4M3: the
 *                  format's own numbers round-trip, ties go to the even mantissa, 448 caps
 *   unquantised    attention over the raw bf16 rows equals the paged attention over a
 *                  cache whose values are all exactly representable; numpy fp64 brute force
 *   append         a first token alone: its min -> 0, max -> 255; in-range values give
 *                  the codes compress gives them when the segment keeps its min/max;
 *                  out-of-range values clamp to 0 / 255; flat segments give 0
 *   re-segmentation trigger bits against the closed form of the length rule at every length
 *                  edge; a re-segmented request equals a fresh compress of its grown history,
 *                  the others equal the plain append; steps to 2048 and 16384 change the count
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define OR_D 128        /* head dimension handled here */
#define OR_WIN 16       /* window length, [DGQ] §2.2 "win_size=16" */
#define OR_MAX_SEG 5    /* at most five segments, [DGQ] §2.2 / §3.2 */

/* One segment record per (request, KV head): 128 bytes. */
typedef struct {
    int32_t n_seg;               /* number of segments (0 only when seq_len == 0) */
    int32_t seq_len;             /* tokens compressed */
    int32_t start[OR_MAX_SEG];   /* first token of each segment; unused entries = seq_len */
    float k_min[OR_MAX_SEG];
    float k_scale[OR_MAX_SEG];
    float v_min[OR_MAX_SEG];
    float v_scale[OR_MAX_SEG];
    float k_inv_last;            /* 255/(max-min) of the last segment, K and V (0 when flat) */
    float v_inv_last;
    int32_t pad[3];
} oracle_seg;

static float bf16_to_float(uint16_t h)
{
    uint32_t b = (uint32_t)h << 16;
    float f;
    memcpy(&f, &b, sizeof f);
    return f;
}

/* ---------------------------------------------------------------------------------
 * a1. n_groups, [DGQ] §3.2 compress(): "if seq_len < 2048: 2; elif < 16384: 3; else
 * min(5, int(log2(seq_len / 1024)) + 2)".  The extracted text lost the comparison
 * operators; READING: strict "<" as the thresholds 2048 / 16384 suggest, int() = floor
 * (the argument is >= 16 there, so truncation and floor agree).
 * -------------------------------------------------------------------------------*/
int32_t oracle_ngroups(int32_t L)
{
    if (L < 2048) return 2;
    if (L < 16384) return 3;
    int32_t g = (int32_t)floor(log2((double)L / 1024.0)) + 2;
    return g < 5 ? g : 5;
}

/* Balanced pairwise sum of n = 2^k fp32 values: sum(left half) + sum(right half).
 * READING: [DGQ] fixes neither the precision nor the order of the variance sums; the
 * oracle fixes fp32 and this tree, so that a GPU reduction can reproduce it bit for bit
 * (the segment boundaries are integer decisions taken on these sums). */
static float pairwise_sum(const float *a, int n)
{
    if (n == 1) return a[0];
    return pairwise_sum(a, n / 2) + pairwise_sum(a + n / 2, n / 2);
}

/* a2. Per-token variance of K over the head dimension, [DGQ] §2.2 ("for each head,
 * compute the variance curve along the L dimension").  READING: population variance
 * (divide by D), two-pass (mean first), of K only, as the article analyses K. */
float oracle_token_variance(const uint16_t *k_row)
{
    float x[OR_D], e[OR_D];
    for (int d = 0; d < OR_D; ++d) x[d] = bf16_to_float(k_row[d]);
    float mean = pairwise_sum(x, OR_D) / (float)OR_D;
    for (int d = 0; d < OR_D; ++d) {
        float dev = x[d] - mean;
        e[d] = dev * dev;
    }
    return pairwise_sum(e, OR_D) / (float)OR_D;
}

/* a3. Window means of the variance curve, [DGQ] §2.2 (window of 16 tokens).
 * READING: non-overlapping windows [16w, 16w+16); the last, partial, window is kept
 * and averaged over its own token count (its sum is taken over the 16-slot tree with
 * +0 in the empty slots, which adds nothing). */
void oracle_window_means(const float *var, int32_t L, float *means)
{
    int32_t W = (L + OR_WIN - 1) / OR_WIN;
    for (int32_t w = 0; w < W; ++w) {
        float slot[OR_WIN];
        int32_t cnt = L - w * OR_WIN;
        if (cnt > OR_WIN) cnt = OR_WIN;
        for (int32_t i = 0; i < OR_WIN; ++i) slot[i] = i < cnt ? var[w * OR_WIN + i] : 0.0f;
        means[w] = pairwise_sum(slot, OR_WIN) / (float)cnt;
    }
}

/* a4. Segment starts from the largest jumps between adjacent window means, [DGQ] §2.2
 * ("detect abrupt changes of the variance ... cut the sequence into 3-5 segments") with
 * the segment count from the §3.2 rule.
 * READINGS: jump_w = |m[w+1] - m[w]| between windows w and w+1; the n_groups-1 largest
 * jumps are taken (ties to the earlier window); a boundary after window w starts a
 * segment at token 16(w+1); the count is capped by the W-1 available jumps; zero jumps
 * are still used when fewer nonzero ones exist.  Returns n_seg, writes n_seg starts. */
/* Group-selection settings, [DGQ] section 5.3 (tuning switches of its vLLM integration):
 * max_groups caps the number of segments (the article's VLLM_DGQ_MAX_GROUPS; 5 leaves the
 * length rule alone) and min_var is a variance floor (its VLLM_DGQ_MIN_VAR: "tokens whose
 * variance is below the threshold go into the same group").  READING of the floor: a window
 * whose mean variance is below min_var is quiet, and no boundary is placed between two quiet
 * windows (a jump between a quiet and a louder window is still a candidate); when fewer
 * candidates than boundaries exist, the pair gets fewer segments.  min_var = 0 changes
 * nothing (window means are >= 0). */
int32_t oracle_boundaries_ex(const float *means, int32_t W, int32_t L, int32_t max_groups, float min_var,
                             int32_t *start)
{
    int32_t k = oracle_ngroups(L);
    if (k > max_groups) k = max_groups;
    if (k > W) k = W;
    k -= 1;
    int32_t chosen[OR_MAX_SEG];
    for (int32_t s = 0; s < k; ++s) {
        int32_t best = -1;
        float best_jump = 0.0f;
        for (int32_t w = 0; w + 1 < W; ++w) {
            int taken = 0;
            for (int32_t c = 0; c < s; ++c)
                if (chosen[c] == w) taken = 1;
            if (taken) continue;
            if (!(means[w] >= min_var || means[w + 1] >= min_var)) continue; /* both quiet */
            float jump = fabsf(means[w + 1] - means[w]);
            /* READING: two adjacent windows whose fp32 variance overflowed (both means +inf)
             * have no defined jump (inf - inf is NaN); such a pair of windows is no candidate,
             * like two quiet windows, and a pair left with fewer candidates gets fewer segments.
             * An overflowed window next to a finite one gives an infinite jump, which is one. */
            if (jump != jump) continue;
            if (best < 0 || jump > best_jump) { /* strict: earlier window wins ties */
                best = w;
                best_jump = jump;
            }
        }
        if (best < 0) { /* no candidate left */
            k = s;
            break;
        }
        chosen[s] = best;
    }
    /* starts: 0 followed by the chosen cut tokens in ascending order */
    start[0] = 0;
    for (int32_t s = 0; s < k; ++s) start[s + 1] = OR_WIN * (chosen[s] + 1);
    for (int32_t i = 2; i <= k; ++i) {
        int32_t v = start[i], j = i - 1;
        while (j >= 1 && start[j] > v) {
            start[j + 1] = start[j];
            --j;
        }
        start[j + 1] = v;
    }
    return k + 1;
}

int32_t oracle_boundaries(const float *means, int32_t W, int32_t L, int32_t *start)
{
    return oracle_boundaries_ex(means, W, L, OR_MAX_SEG, 0.0f, start);
}

/* a5. fp32 min and max over all tokens x D of one segment, [DGQ] §2.2 ("each segment
 * computes its own min/max").  READING: -0.0 results are stored as +0.0. */
static void segment_min_max(const uint16_t *x, int64_t row_stride, int32_t t0, int32_t t1,
                            float *mn, float *mx)
{
    float lo = INFINITY, hi = -INFINITY;
    for (int32_t t = t0; t < t1; ++t)
        for (int d = 0; d < OR_D; ++d) {
            float v = bf16_to_float(x[(int64_t)t * row_stride + d]);
            if (v < lo) lo = v;
            if (v > hi) hi = v;
        }
    if (lo == 0.0f) lo = 0.0f;
    if (hi == 0.0f) hi = 0.0f;
    *mn = lo;
    *mx = hi;
}

/* Affine uint8 parameters of one segment: scale = (max-min)/255 for dequantisation and,
 * as a separate IEEE division, inv = 255/(max-min) for encoding.  A flat segment
 * (max == min) gets scale = inv = 0, so every code is 0 and decodes to min. */
static void segment_affine(float mn, float mx, float *scale, float *inv)
{
    float r = mx - mn;
    if (r == 0.0f) {
        *scale = 0.0f;
        *inv = 0.0f;
    } else {
        *scale = r / 255.0f;
        *inv = 255.0f / r;
    }
}

/* a6. One code: q = rint((x - min) * inv), round-half-even, kept in [0, 255]. */
uint8_t oracle_encode(float x, float mn, float inv)
{
    float u = (x - mn) * inv;
    float q = rintf(u);
    if (q < 0.0f) q = 0.0f;
    if (q > 255.0f) q = 255.0f;
    return (uint8_t)q;
}

/* Compress one (request, KV head): L rows of K and V (bf16, rows `row_stride` elements
 * apart).  Fills the record and, when non-null, the unpaged codes [L, 128]. */
void oracle_compress_pair_ex(const uint16_t *k, const uint16_t *v, int64_t row_stride, int32_t L,
                             int32_t max_groups, float min_var, oracle_seg *rec, uint8_t *k_codes,
                             uint8_t *v_codes)
{
    memset(rec, 0, sizeof *rec);
    rec->seq_len = L;
    for (int i = 0; i < OR_MAX_SEG; ++i) rec->start[i] = L;
    if (L <= 0) return;

    int32_t W = (L + OR_WIN - 1) / OR_WIN;
    float *var = (float *)malloc(sizeof(float) * (size_t)L);
    float *means = (float *)malloc(sizeof(float) * (size_t)W);
    float k_inv[OR_MAX_SEG], v_inv[OR_MAX_SEG];

    for (int32_t t = 0; t < L; ++t) var[t] = oracle_token_variance(k + (int64_t)t * row_stride);
    oracle_window_means(var, L, means);
    /* READING: one segmentation per (request, KV head), derived from K and shared by K
     * and V (the article derives the segments from K, and its storage formula counts a
     * single marker bit per layer x head x token), with separate min/scale for K and V. */
    int32_t n = oracle_boundaries_ex(means, W, L, max_groups, min_var, rec->start);
    rec->n_seg = n;

    for (int32_t s = 0; s < n; ++s) {
        int32_t t0 = rec->start[s], t1 = s + 1 < n ? rec->start[s + 1] : L;
        float mn, mx;
        segment_min_max(k, row_stride, t0, t1, &mn, &mx);
        rec->k_min[s] = mn;
        segment_affine(mn, mx, &rec->k_scale[s], &k_inv[s]);
        segment_min_max(v, row_stride, t0, t1, &mn, &mx);
        rec->v_min[s] = mn;
        segment_affine(mn, mx, &rec->v_scale[s], &v_inv[s]);
    }
    rec->k_inv_last = k_inv[n - 1];
    rec->v_inv_last = v_inv[n - 1];

    if (k_codes || v_codes) {
        int32_t s = 0;
        for (int32_t t = 0; t < L; ++t) {
            while (s + 1 < n && rec->start[s + 1] <= t) ++s;
            for (int d = 0; d < OR_D; ++d) {
                if (k_codes)
                    k_codes[(int64_t)t * OR_D + d] = oracle_encode(
                        bf16_to_float(k[(int64_t)t * row_stride + d]), rec->k_min[s], k_inv[s]);
                if (v_codes)
                    v_codes[(int64_t)t * OR_D + d] = oracle_encode(
                        bf16_to_float(v[(int64_t)t * row_stride + d]), rec->v_min[s], v_inv[s]);
            }
        }
    }
    free(var);
    free(means);
}

/* Independent V segmentation (a group-selection variant; the article derives its segments from
 * K only, [DGQ] section 2.2).  READING: V is segmented by the same rule applied to V's own
 * per-token variance (a2-a4 on V), and each tensor is encoded with its own segments (a5-a6).
 * One tensor x of one (request, KV head): its starts, per-segment min / scale / inverse and codes
 * (unpaged [L, 128], when non-null).  Returns the number of segments (0 when L == 0). */
static int32_t encode_own_segments(const uint16_t *x, int64_t row_stride, int32_t L, int32_t max_groups,
                                   float min_var, int32_t *start, float *mn, float *scale, float *inv,
                                   uint8_t *codes)
{
    for (int i = 0; i < OR_MAX_SEG; ++i) {
        start[i] = L;
        mn[i] = scale[i] = inv[i] = 0.0f;
    }
    if (L <= 0) return 0;
    int32_t W = (L + OR_WIN - 1) / OR_WIN;
    float *var = (float *)malloc(sizeof(float) * (size_t)L);
    float *means = (float *)malloc(sizeof(float) * (size_t)W);
    for (int32_t t = 0; t < L; ++t) var[t] = oracle_token_variance(x + (int64_t)t * row_stride);
    oracle_window_means(var, L, means);
    int32_t n = oracle_boundaries_ex(means, W, L, max_groups, min_var, start);
    for (int32_t s = 0; s < n; ++s) {
        int32_t t0 = start[s], t1 = s + 1 < n ? start[s + 1] : L;
        float mx;
        segment_min_max(x, row_stride, t0, t1, &mn[s], &mx);
        segment_affine(mn[s], mx, &scale[s], &inv[s]);
    }
    if (codes) {
        int32_t s = 0;
        for (int32_t t = 0; t < L; ++t) {
            while (s + 1 < n && start[s + 1] <= t) ++s;
            for (int d = 0; d < OR_D; ++d)
                codes[(int64_t)t * OR_D + d] = oracle_encode(bf16_to_float(x[(int64_t)t * row_stride + d]), mn[s],
                                                             inv[s]);
        }
    }
    free(var);
    free(means);
    return n;
}

/* One (request, KV head) with independent segmentations: k_rec holds K's segments (start,
 * k_min, k_scale, k_inv_last; V fields 0), v_rec V's (start, v_min, v_scale, v_inv_last; K fields
 * 0); both carry n_seg of their own tensor and seq_len = L. */
void oracle_compress_pair_split(const uint16_t *k, const uint16_t *v, int64_t row_stride, int32_t L,
                                int32_t max_groups, float min_var, oracle_seg *k_rec, oracle_seg *v_rec,
                                uint8_t *k_codes, uint8_t *v_codes)
{
    float inv[OR_MAX_SEG], sc[OR_MAX_SEG], mn[OR_MAX_SEG];
    memset(k_rec, 0, sizeof *k_rec);
    memset(v_rec, 0, sizeof *v_rec);
    k_rec->seq_len = v_rec->seq_len = L;
    int32_t n = encode_own_segments(k, row_stride, L, max_groups, min_var, k_rec->start, mn, sc, inv, k_codes);
    k_rec->n_seg = n;
    for (int i = 0; i < OR_MAX_SEG; ++i) {
        k_rec->k_min[i] = mn[i];
        k_rec->k_scale[i] = sc[i];
    }
    k_rec->k_inv_last = n > 0 ? inv[n - 1] : 0.0f;
    n = encode_own_segments(v, row_stride, L, max_groups, min_var, v_rec->start, mn, sc, inv, v_codes);
    v_rec->n_seg = n;
    for (int i = 0; i < OR_MAX_SEG; ++i) {
        v_rec->v_min[i] = mn[i];
        v_rec->v_scale[i] = sc[i];
    }
    v_rec->v_inv_last = n > 0 ? inv[n - 1] : 0.0f;
    if (L <= 0) {  /* as the shared path: an empty pair's starts are all 0 */
        for (int i = 0; i < OR_MAX_SEG; ++i) k_rec->start[i] = v_rec->start[i] = 0;
    }
}

/* One layer with independent segmentations (pools as oracle_compress_ex; two record tables). */
void oracle_compress_split(const uint16_t *k, const uint16_t *v, const int32_t *cu_seqlens, int32_t B, int32_t Hkv,
                           int32_t bs, const int32_t *block_tables, int32_t max_blocks, int32_t max_groups,
                           float min_var, uint8_t *k_pool, uint8_t *v_pool, oracle_seg *k_table, oracle_seg *v_table)
{
    for (int32_t b = 0; b < B; ++b) {
        int32_t L = cu_seqlens[b + 1] - cu_seqlens[b];
        for (int32_t h = 0; h < Hkv; ++h) {
            const int64_t row0 = ((int64_t)cu_seqlens[b] * Hkv + h) * OR_D;
            uint8_t *kc = (uint8_t *)malloc((size_t)(L > 0 ? L : 1) * OR_D);
            uint8_t *vc = (uint8_t *)malloc((size_t)(L > 0 ? L : 1) * OR_D);
            oracle_compress_pair_split(k + row0, v + row0, (int64_t)Hkv * OR_D, L, max_groups, min_var,
                                       &k_table[(int64_t)b * Hkv + h], &v_table[(int64_t)b * Hkv + h], kc, vc);
            for (int32_t t = 0; t < L; ++t) {
                int64_t blk = block_tables[(int64_t)b * max_blocks + t / bs];
                int64_t dst = ((blk * Hkv + h) * bs + t % bs) * OR_D;
                memcpy(k_pool + dst, kc + (int64_t)t * OR_D, OR_D);
                memcpy(v_pool + dst, vc + (int64_t)t * OR_D, OR_D);
            }
            free(kc);
            free(vc);
        }
    }
}

/* a2-a7 for one layer of a batch.  K and V are packed variable-length [T, Hkv, 128]
 * with request b on rows cu_seqlens[b] .. cu_seqlens[b+1]).  Token t of request b, head h
 * is stored at pool[block_tables[b][t / bs]][h][t % bs][0..128), [PAGED]
 * "PagedAttention implementation" (logical block -> physical block).  Slots past the
 * sequence end in its last block are left untouched.  Pools are [num_blocks, Hkv, bs, 128]
 * uint8, the record table [B, Hkv]. */
void oracle_compress_pair(const uint16_t *k, const uint16_t *v, int64_t row_stride, int32_t L,
                          oracle_seg *rec, uint8_t *k_codes, uint8_t *v_codes)
{
    oracle_compress_pair_ex(k, v, row_stride, L, OR_MAX_SEG, 0.0f, rec, k_codes, v_codes);
}

void oracle_compress_ex(const uint16_t *k, const uint16_t *v, const int32_t *cu_seqlens,
                        int32_t B, int32_t Hkv, int32_t bs, const int32_t *block_tables,
                        int32_t max_blocks, int32_t max_groups, float min_var, uint8_t *k_pool,
                        uint8_t *v_pool, oracle_seg *table)
{
    for (int32_t b = 0; b < B; ++b) {
        int32_t L = cu_seqlens[b + 1] - cu_seqlens[b];
        for (int32_t h = 0; h < Hkv; ++h) {
            const int64_t row0 = ((int64_t)cu_seqlens[b] * Hkv + h) * OR_D;
            uint8_t *kc = (uint8_t *)malloc((size_t)(L > 0 ? L : 1) * OR_D);
            uint8_t *vc = (uint8_t *)malloc((size_t)(L > 0 ? L : 1) * OR_D);
            oracle_seg *rec = &table[(int64_t)b * Hkv + h];
            oracle_compress_pair_ex(k + row0, v + row0, (int64_t)Hkv * OR_D, L, max_groups, min_var, rec, kc,
                                    vc);
            for (int32_t t = 0; t < L; ++t) {
                int64_t blk = block_tables[(int64_t)b * max_blocks + t / bs];
                int64_t dst = ((blk * Hkv + h) * bs + t % bs) * OR_D;
                memcpy(k_pool + dst, kc + (int64_t)t * OR_D, OR_D);
                memcpy(v_pool + dst, vc + (int64_t)t * OR_D, OR_D);
            }
            free(kc);
            free(vc);
        }
    }
}

void oracle_compress(const uint16_t *k, const uint16_t *v, const int32_t *cu_seqlens,
                     int32_t B, int32_t Hkv, int32_t bs, const int32_t *block_tables,
                     int32_t max_blocks, uint8_t *k_pool, uint8_t *v_pool, oracle_seg *table)
{
    oracle_compress_ex(k, v, cu_seqlens, B, Hkv, bs, block_tables, max_blocks, OR_MAX_SEG, 0.0f, k_pool, v_pool,
                       table);
}

/* Decode-step append for one layer: request b's new key and value (one token per
 * (request, KV head), bf16 [B, Hkv, 128]) go into the cache at position L = the record's
 * seq_len.  [DGQ] section 2.2 analyses the cache as each new token is generated, but says
 * nothing about how a token generated after compression is encoded.  READING: the token
 * joins the last segment and is encoded with that segment's min and 255/(max-min), the
 * same two IEEE steps as a6, its codes held to [0, 255] (values outside the segment's
 * range clamp; the segment's parameters, and so every code already stored, stay as they
 * are).  The boundaries are not revisited: that needs the bf16 history, which the cache no
 * longer holds.  A request with no token yet (n_seg == 0) gets a first segment made of the
 * new token alone (a5 over one token).  The record's seq_len, and every start[] entry past
 * the last segment, become L + 1.  A pair whose slot L has no block-table column
 * (L / bs >= max_blocks) is left untouched and counted; the return value is that count. */
int32_t oracle_append(const uint16_t *k_new, const uint16_t *v_new, int32_t B, int32_t Hkv, int32_t bs,
                      const int32_t *block_tables, int32_t max_blocks, uint8_t *k_pool, uint8_t *v_pool,
                      oracle_seg *table)
{
    int32_t skipped = 0;
    for (int32_t b = 0; b < B; ++b) {
        for (int32_t h = 0; h < Hkv; ++h) {
            oracle_seg *rec = &table[(int64_t)b * Hkv + h];
            const int32_t L = rec->seq_len;
            if (L / bs >= max_blocks) {
                ++skipped;
                continue;
            }
            const uint16_t *kx = k_new + ((int64_t)b * Hkv + h) * OR_D;
            const uint16_t *vx = v_new + ((int64_t)b * Hkv + h) * OR_D;
            if (rec->n_seg == 0) {
                float mn, mx;
                segment_min_max(kx, OR_D, 0, 1, &mn, &mx);
                rec->k_min[0] = mn;
                segment_affine(mn, mx, &rec->k_scale[0], &rec->k_inv_last);
                segment_min_max(vx, OR_D, 0, 1, &mn, &mx);
                rec->v_min[0] = mn;
                segment_affine(mn, mx, &rec->v_scale[0], &rec->v_inv_last);
                rec->n_seg = 1;
                rec->start[0] = 0;
            }
            const int32_t s = rec->n_seg - 1;
            const int64_t blk = block_tables[(int64_t)b * max_blocks + L / bs];
            const int64_t dst = ((blk * Hkv + h) * bs + L % bs) * OR_D;
            for (int d = 0; d < OR_D; ++d) {
                k_pool[dst + d] = oracle_encode(bf16_to_float(kx[d]), rec->k_min[s], rec->k_inv_last);
                v_pool[dst + d] = oracle_encode(bf16_to_float(vx[d]), rec->v_min[s], rec->v_inv_last);
            }
            rec->seq_len = L + 1;
            for (int32_t i = rec->n_seg; i < OR_MAX_SEG; ++i) rec->start[i] = L + 1;
        }
    }
    return skipped;
}

/* Decode-step append with independent V segmentation: as oracle_append, each tensor with its own
 * record (K: k_table's K fields; V: v_table's V fields; a record with n_seg == 0 gets a first
 * segment made of the new token's own values of that tensor).  The slot is taken from K's
 * record (both records of a pair hold the same seq_len).  Returns the pairs skipped for want of
 * a block-table column. */
static void append_tensor(const uint16_t *x, oracle_seg *rec, int which_v, int32_t L, uint8_t *dst)
{
    float *mn0 = which_v ? rec->v_min : rec->k_min;
    float *sc0 = which_v ? rec->v_scale : rec->k_scale;
    float *inv = which_v ? &rec->v_inv_last : &rec->k_inv_last;
    if (rec->n_seg == 0) {
        float mn, mx;
        segment_min_max(x, OR_D, 0, 1, &mn, &mx);
        mn0[0] = mn;
        segment_affine(mn, mx, &sc0[0], inv);
        rec->n_seg = 1;
        rec->start[0] = 0;
    }
    const int32_t s = rec->n_seg - 1;
    for (int d = 0; d < OR_D; ++d) dst[d] = oracle_encode(bf16_to_float(x[d]), mn0[s], *inv);
    rec->seq_len = L + 1;
    for (int32_t i = rec->n_seg; i < OR_MAX_SEG; ++i) rec->start[i] = L + 1;
}

int32_t oracle_append_split(const uint16_t *k_new, const uint16_t *v_new, int32_t B, int32_t Hkv, int32_t bs,
                            const int32_t *block_tables, int32_t max_blocks, uint8_t *k_pool, uint8_t *v_pool,
                            oracle_seg *k_table, oracle_seg *v_table)
{
    int32_t skipped = 0;
    for (int32_t b = 0; b < B; ++b) {
        for (int32_t h = 0; h < Hkv; ++h) {
            oracle_seg *kr = &k_table[(int64_t)b * Hkv + h], *vr = &v_table[(int64_t)b * Hkv + h];
            const int32_t L = kr->seq_len;
            if (L / bs >= max_blocks) {
                ++skipped;
                continue;
            }
            const int64_t blk = block_tables[(int64_t)b * max_blocks + L / bs];
            const int64_t dst = ((blk * Hkv + h) * bs + L % bs) * OR_D;
            append_tensor(k_new + ((int64_t)b * Hkv + h) * OR_D, kr, 0, L, k_pool + dst);
            append_tensor(v_new + ((int64_t)b * Hkv + h) * OR_D, vr, 1, L, v_pool + dst);
        }
    }
    return skipped;
}

/* Re-segmentation triggers of a decode-step append, [DGQ] section 2.2 (the variance curve is
 * analysed in real time as each new token is generated; segments come from jumps between
 * 16-token window means) and section 3.2 (the segment count follows the length).  READING:
 * appending token L -- the cache grows from L to L + 1 tokens -- completes a window when L + 1 is
 * a multiple of 16 (a new window mean, hence a new candidate jump, exists: bit 1), and changes the
 * segment count when n_groups(L + 1) != n_groups(L) (bit 2; by the rule this happens at
 * L + 1 = 2048 and 16384, both also window ends).  A partial window adds no mean the segmentation
 * of complete windows lacks, so no other length triggers. */
int32_t oracle_resegment_flags(int32_t L)
{
    int32_t f = 0;
    if ((L + 1) % OR_WIN == 0) f |= 1;
    if (oracle_ngroups(L + 1) != oracle_ngroups(L)) f |= 2;
    return f;
}

/* One decode step with re-segmentation: oracle_append of the step's token, then every request
 * with a pair whose trigger bits (oracle_resegment_flags of its length before the append) meet
 * `mask` is compressed again from its bf16 history -- oracle_compress_pair_ex over its L + 1
 * tokens: new boundaries, new segment parameters, every code re-encoded and scattered through
 * the block table.  READING: the INT8 cache cannot be re-segmented from its own codes (the
 * segment extremes and the variance need the original values), so a re-segmentation redoes the
 * method's compression of the whole request from the bf16 K/V a serving engine keeps (its bf16
 * paged cache); [DGQ] section 2.2 gives no incremental form.
 * k_hist, v_hist: packed [T, Hkv, 128] bf16, request b's L + 1 tokens on rows hist_cu[b] ..
 * hist_cu[b + 1] - 1 (the last of them is the step's token).  flags_out [B, Hkv]: every pair's
 * trigger bits.  Returns the pairs the append skipped for want of a block-table column. */
int32_t oracle_append_resegment(const uint16_t *k_new, const uint16_t *v_new, int32_t B, int32_t Hkv, int32_t bs,
                                const int32_t *block_tables, int32_t max_blocks, uint8_t *k_pool, uint8_t *v_pool,
                                oracle_seg *table, const uint16_t *k_hist, const uint16_t *v_hist,
                                const int32_t *hist_cu, int32_t mask, int32_t max_groups, float min_var,
                                int32_t *flags_out)
{
    for (int64_t p = 0; p < (int64_t)B * Hkv; ++p) flags_out[p] = oracle_resegment_flags(table[p].seq_len);
    const int32_t skipped = oracle_append(k_new, v_new, B, Hkv, bs, block_tables, max_blocks, k_pool, v_pool, table);
    for (int32_t b = 0; b < B; ++b) {
        int redo = 0;
        for (int32_t h = 0; h < Hkv; ++h)
            if (flags_out[(int64_t)b * Hkv + h] & mask) redo = 1;
        if (!redo) continue;
        /* the request's history, compressed as one request of its own */
        const int32_t cu[2] = {0, hist_cu[b + 1] - hist_cu[b]};
        const int64_t row0 = (int64_t)hist_cu[b] * Hkv * OR_D;
        oracle_compress_ex(k_hist + row0, v_hist + row0, cu, 1, Hkv, bs, block_tables + (int64_t)b * max_blocks,
                           max_blocks, max_groups, min_var, k_pool, v_pool, table + (int64_t)b * Hkv);
    }
    return skipped;
}

/* Dequantised value of one code, in fp64: min + q * scale. */
static double dequant(uint8_t q, float mn, float scale)
{
    return (double)mn + (double)q * (double)scale;
}

static int32_t segment_of(const oracle_seg *rec, int32_t t)
{
    int32_t s = 0;
    for (int32_t i = 1; i < rec->n_seg; ++i)
        if (rec->start[i] <= t) s = i;
    return s;
}

/* Dequantise one (request, KV head) back to an fp64 [L, 128] array (test helper). */
void oracle_dequant_pair(const uint8_t *pool, const oracle_seg *table, const int32_t *block_tables,
                         int32_t b, int32_t h, int32_t Hkv, int32_t bs, int32_t max_blocks,
                         int32_t L, int which_v, double *out)
{
    const oracle_seg *rec = &table[(int64_t)b * Hkv + h];
    for (int32_t t = 0; t < L; ++t) {
        int32_t s = segment_of(rec, t);
        float mn = which_v ? rec->v_min[s] : rec->k_min[s];
        float sc = which_v ? rec->v_scale[s] : rec->k_scale[s];
        int64_t blk = block_tables[(int64_t)b * max_blocks + t / bs];
        const uint8_t *row = pool + ((blk * Hkv + h) * bs + t % bs) * OR_D;
        for (int d = 0; d < OR_D; ++d) out[(int64_t)t * OR_D + d] = dequant(row[d], mn, sc);
    }
}

/* a8-a10. Decode-step attention in fp64 over the dequantised paged cache plus the
 * current step's own bf16 key/value.
 * q [B, Hq, 128], k_new / v_new [B, Hkv, 128] (bf16 bits); out [B, Hq, 128] fp64.
 * Query head hq reads KV head hq / (Hq / Hkv) (grouped-query attention, consecutive
 * query heads share a KV head).  Scores are q.k / sqrt(128); softmax over the L cached
 * positions and the current one; output = sum_t p_t v_t.
 * READINGS: the cached tokens are exactly positions 0..L-1 (no mask, keys already
 * rotary-embedded), the current token at position L is attended unquantised and is not
 * part of the cache. */
void oracle_paged_decode_attn(const uint16_t *q, const uint16_t *k_new, const uint16_t *v_new,
                              const uint8_t *k_pool, const uint8_t *v_pool,
                              const oracle_seg *table, const int32_t *block_tables,
                              const int32_t *seq_lens, int32_t B, int32_t Hq, int32_t Hkv,
                              int32_t bs, int32_t max_blocks, double *out)
{
    const int32_t G = Hq / Hkv;
    const double inv_sqrt_d = 1.0 / sqrt((double)OR_D);
    for (int32_t b = 0; b < B; ++b) {
        const int32_t L = seq_lens[b];
        double *s = (double *)malloc(sizeof(double) * (size_t)(L + 1));
        for (int32_t hq = 0; hq < Hq; ++hq) {
            const int32_t h = hq / G;
            const oracle_seg *rec = &table[(int64_t)b * Hkv + h];
            const uint16_t *qv = q + ((int64_t)b * Hq + hq) * OR_D;
            for (int32_t t = 0; t < L; ++t) {
                int32_t sg = segment_of(rec, t);
                int64_t blk = block_tables[(int64_t)b * max_blocks + t / bs];
                const uint8_t *kr = k_pool + ((blk * Hkv + h) * bs + t % bs) * OR_D;
                double acc = 0.0;
                for (int d = 0; d < OR_D; ++d)
                    acc += (double)bf16_to_float(qv[d]) * dequant(kr[d], rec->k_min[sg], rec->k_scale[sg]);
                s[t] = acc * inv_sqrt_d;
            }
            {
                const uint16_t *kn = k_new + ((int64_t)b * Hkv + h) * OR_D;
                double acc = 0.0;
                for (int d = 0; d < OR_D; ++d)
                    acc += (double)bf16_to_float(qv[d]) * (double)bf16_to_float(kn[d]);
                s[L] = acc * inv_sqrt_d;
            }
            double m = s[0];
            for (int32_t t = 1; t <= L; ++t)
                if (s[t] > m) m = s[t];
            double l = 0.0;
            for (int32_t t = 0; t <= L; ++t) {
                s[t] = exp(s[t] - m);
                l += s[t];
            }
            double o[OR_D];
            for (int d = 0; d < OR_D; ++d) o[d] = 0.0;
            for (int32_t t = 0; t < L; ++t) {
                int32_t sg = segment_of(rec, t);
                int64_t blk = block_tables[(int64_t)b * max_blocks + t / bs];
                const uint8_t *vr = v_pool + ((blk * Hkv + h) * bs + t % bs) * OR_D;
                for (int d = 0; d < OR_D; ++d)
                    o[d] += s[t] * dequant(vr[d], rec->v_min[sg], rec->v_scale[sg]);
            }
            {
                const uint16_t *vn = v_new + ((int64_t)b * Hkv + h) * OR_D;
                for (int d = 0; d < OR_D; ++d) o[d] += s[L] * (double)bf16_to_float(vn[d]);
            }
            double *dst = out + ((int64_t)b * Hq + hq) * OR_D;
            for (int d = 0; d < OR_D; ++d) dst[d] = o[d] / l;
        }
        free(s);
    }
}

/* Fidelity context: the same decode-step attention (a8-a10 in fp64) over the original,
 * unquantised bf16 keys and values, packed [T, Hkv, 128] with request b on rows
 * cu_seqlens[b] .. cu_seqlens[b] + seq_lens[b] - 1.  Comparing it with the attention over the
 * compressed cache shows the error the INT8 encoding itself introduces. */
void oracle_decode_attn_unquantised(const uint16_t *q, const uint16_t *k_new, const uint16_t *v_new,
                                    const uint16_t *k, const uint16_t *v, const int32_t *cu_seqlens,
                                    const int32_t *seq_lens, int32_t B, int32_t Hq, int32_t Hkv, double *out)
{
    const int32_t G = Hq / Hkv;
    const double inv_sqrt_d = 1.0 / sqrt((double)OR_D);
    for (int32_t b = 0; b < B; ++b) {
        const int32_t L = seq_lens[b];
        double *s = (double *)malloc(sizeof(double) * (size_t)(L + 1));
        for (int32_t hq = 0; hq < Hq; ++hq) {
            const int32_t h = hq / G;
            const uint16_t *qv = q + ((int64_t)b * Hq + hq) * OR_D;
            for (int32_t t = 0; t <= L; ++t) {
                const uint16_t *kr = t < L ? k + (((int64_t)cu_seqlens[b] + t) * Hkv + h) * OR_D
                                           : k_new + ((int64_t)b * Hkv + h) * OR_D;
                double acc = 0.0;
                for (int d = 0; d < OR_D; ++d) acc += (double)bf16_to_float(qv[d]) * (double)bf16_to_float(kr[d]);
                s[t] = acc * inv_sqrt_d;
            }
            double m = s[0];
            for (int32_t t = 1; t <= L; ++t)
                if (s[t] > m) m = s[t];
            double l = 0.0;
            for (int32_t t = 0; t <= L; ++t) {
                s[t] = exp(s[t] - m);
                l += s[t];
            }
            double o[OR_D];
            for (int d = 0; d < OR_D; ++d) o[d] = 0.0;
            for (int32_t t = 0; t <= L; ++t) {
                const uint16_t *vr = t < L ? v + (((int64_t)cu_seqlens[b] + t) * Hkv + h) * OR_D
                                           : v_new + ((int64_t)b * Hkv + h) * OR_D;
                for (int d = 0; d < OR_D; ++d) o[d] += s[t] * (double)bf16_to_float(vr[d]);
            }
            double *dst = out + ((int64_t)b * Hq + hq) * OR_D;
            for (int d = 0; d < OR_D; ++d) dst[d] = o[d] / l;
        }
        free(s);
    }
}

/* ---- comparison quantisers (fidelity context) --------------------------------------------
 * Each returns the dequantised fp64 values of one (request, head) pair [L, 128] (rows
 * `row_stride` elements apart in x), so that attention over them can be compared with DGQ's.
 *   fixed 64-dim groups ([DGQ] section 2.2: "traditional group quantisation cuts the cache into
 *     fixed blocks of e.g. 64 dimensions, each with its own min/max, INT8"): per token and per
 *     64-element half, the DGQ affine code (a5-a6 over that group) and its dequantisation;
 *   symmetric INT8 ("DeepSeek-V4" article, FP8+FP16 section: scale = max|k| / 127, k / scale
 *     held to [-128, 127]): READING: per (request, head) tensor, round-half-even to an integer
 *     (the printed snippet omits the rounding), dequantised as q * scale;
 *   FP8 E4M3 ([DGQ] section 2.3 table): each value rounded half-even to the nearest E4M3 number
 *     (3 mantissa bits, exponent bias 7, largest 448, subnormal step 2^-9), saturating. */
void oracle_dequant_fixed64(const uint16_t *x, int64_t row_stride, int32_t L, double *out)
{
    for (int32_t t = 0; t < L; ++t)
        for (int g = 0; g < 2; ++g) {
            float mn = INFINITY, mx = -INFINITY;
            for (int d = 64 * g; d < 64 * g + 64; ++d) {
                float v = bf16_to_float(x[(int64_t)t * row_stride + d]);
                if (v < mn) mn = v;
                if (v > mx) mx = v;
            }
            if (mn == 0.0f) mn = 0.0f;
            if (mx == 0.0f) mx = 0.0f;
            float scale, inv;
            segment_affine(mn, mx, &scale, &inv);
            for (int d = 64 * g; d < 64 * g + 64; ++d) {
                uint8_t q = oracle_encode(bf16_to_float(x[(int64_t)t * row_stride + d]), mn, inv);
                out[(int64_t)t * OR_D + d] = dequant(q, mn, scale);
            }
        }
}

void oracle_dequant_sym_int8(const uint16_t *x, int64_t row_stride, int32_t L, double *out)
{
    float amax = 0.0f;
    for (int32_t t = 0; t < L; ++t)
        for (int d = 0; d < OR_D; ++d) {
            float v = fabsf(bf16_to_float(x[(int64_t)t * row_stride + d]));
            if (v > amax) amax = v;
        }
    const float scale = amax / 127.0f;
    for (int32_t t = 0; t < L; ++t)
        for (int d = 0; d < OR_D; ++d) {
            float v = bf16_to_float(x[(int64_t)t * row_stride + d]);
            float q = scale > 0.0f ? rintf(v / scale) : 0.0f;
            if (q < -128.0f) q = -128.0f;
            if (q > 127.0f) q = 127.0f;
            out[(int64_t)t * OR_D + d] = (double)q * (double)scale;
        }
}

static double round_e4m3(double v)
{
    const double a = fabs(v);
    if (a == 0.0) return 0.0;
    int e;
    frexp(a, &e);                       /* a = m * 2^e, 0.5 <= m < 1: leading bit at 2^(e-1) */
    int lead = e - 1;
    if (lead < -6) lead = -6;           /* subnormals share the step of the smallest normal */
    const double quantum = ldexp(1.0, lead - 3);
    double r = nearbyint(a / quantum) * quantum;  /* half-even (default rounding mode) */
    if (r > 448.0) r = 448.0;           /* saturate to the largest finite E4M3 value */
    return v < 0.0 ? -r : r;
}

void oracle_dequant_fp8_e4m3(const uint16_t *x, int64_t row_stride, int32_t L, double *out)
{
    for (int32_t t = 0; t < L; ++t)
        for (int d = 0; d < OR_D; ++d)
            out[(int64_t)t * OR_D + d] = round_e4m3((double)bf16_to_float(x[(int64_t)t * row_stride + d]));
}

/* Decode attention (a9-a10 in fp64) of one request over dense fp64 keys/values [L, Hkv, 128]
 * plus the current token's bf16 key/value: the comparison quantisers' counterpart of
 * oracle_paged_decode_attn. */
void oracle_decode_attn_dense(const uint16_t *q, const uint16_t *k_new, const uint16_t *v_new, const double *kd,
                              const double *vd, int32_t L, int32_t Hq, int32_t Hkv, double *out)
{
    const int32_t G = Hq / Hkv;
    const double inv_sqrt_d = 1.0 / sqrt((double)OR_D);
    double *s = (double *)malloc(sizeof(double) * (size_t)(L + 1));
    for (int32_t hq = 0; hq < Hq; ++hq) {
        const int32_t h = hq / G;
        const uint16_t *qv = q + (int64_t)hq * OR_D;
        for (int32_t t = 0; t <= L; ++t) {
            double acc = 0.0;
            for (int d = 0; d < OR_D; ++d) {
                const double kv = t < L ? kd[((int64_t)t * Hkv + h) * OR_D + d]
                                        : (double)bf16_to_float(k_new[(int64_t)h * OR_D + d]);
                acc += (double)bf16_to_float(qv[d]) * kv;
            }
            s[t] = acc * inv_sqrt_d;
        }
        double m = s[0];
        for (int32_t t = 1; t <= L; ++t)
            if (s[t] > m) m = s[t];
        double l = 0.0;
        for (int32_t t = 0; t <= L; ++t) {
            s[t] = exp(s[t] - m);
            l += s[t];
        }
        for (int d = 0; d < OR_D; ++d) {
            double o = 0.0;
            for (int32_t t = 0; t <= L; ++t) {
                const double vv = t < L ? vd[((int64_t)t * Hkv + h) * OR_D + d]
                                        : (double)bf16_to_float(v_new[(int64_t)h * OR_D + d]);
                o += s[t] * vv;
            }
            out[(int64_t)hq * OR_D + d] = o / l;
        }
    }
    free(s);
}

/* Algorithmic bytes one compress call writes for a request of L tokens and Hkv heads:
 * 1 byte per K and per V element plus one 128-byte record per head ([DGQ] §3.3 gives the
 * INT8 body at 1 byte per element; the record replaces its per-token marker bits). */
int64_t oracle_compress_bytes_written(int32_t L, int32_t Hkv)
{
    return 2LL * L * Hkv * OR_D + (int64_t)sizeof(oracle_seg) * Hkv;
}
