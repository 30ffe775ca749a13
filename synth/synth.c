/*
 * synth.c -- host side of the seeded synthetic-input generator (libsynth.so).
 *
 * Builds the per-(layer, request, head) variance spans and fills bf16 tensors with
 * the Gaussian stream defined in synth_core.h.  Shapes and value distributions follow
 * the workloads the DGQ page analyses: K/V whose standard deviation is piecewise
 * constant along the sequence, with magnitudes 0.03 .. 0.47 as in the page's own
 * example of low- and high-variance tokens ("DeepSeek dynamic group quantisation"
 * page, section 2.2).  Nothing here computes any part of the DGQ method.
 *
 * Span rules (which tensor positions get which sigma):
 *   SYNTH_RULE_SET3  : 3 spans, each sigma drawn from {0.03, 0.15, 0.47}
 *   SYNTH_RULE_U     : 3..5 spans, each sigma uniform in [0.03, 0.5]
 *   SYNTH_RULE_PERM5 : 5 spans, sigmas a random order of {0.03, 0.08, 0.15, 0.3, 0.47}
 * The k-1 cut points are uniform over token positions 1..L-1 (duplicates allowed, so
 * a span may be empty); K and V of the same (layer, request, head) share the spans.
 */
#include "synth_core.h"

#include <stdint.h>
#include <stddef.h>

#define SYNTH_MAX_SPANS 5

enum { SYNTH_RULE_SET3 = 0, SYNTH_RULE_U = 1, SYNTH_RULE_PERM5 = 2 };

uint64_t synth_hash_c(uint64_t key, uint64_t ctr) { return synth_hash(key, ctr); }

uint64_t synth_key_c(uint64_t seed, uint32_t stream, uint32_t layer, uint32_t req,
                     uint32_t head)
{
    return synth_key(seed, stream, layer, req, head);
}

float synth_normal_c(uint64_t key, uint64_t ctr)
{
    return synth_normal_from_hash(synth_hash(key, ctr));
}

uint16_t synth_bf16_c(float x) { return synth_bf16(x); }

/* Span table of one (layer, request, head); returns the number of spans. */
int32_t synth_spans(uint64_t seed, uint32_t layer, uint32_t req, uint32_t head,
                    int32_t L, int32_t rule, int32_t *start, float *sigma)
{
    static const float set3[3] = {0.03f, 0.15f, 0.47f};
    static const float set5[5] = {0.03f, 0.08f, 0.15f, 0.3f, 0.47f};
    uint64_t key = synth_key(seed, SYNTH_STREAM_SPAN, layer, req, head);
    int32_t n;
    if (rule == SYNTH_RULE_SET3)
        n = 3;
    else if (rule == SYNTH_RULE_U)
        n = 3 + (int32_t)(synth_hash(key, 0) % 3u);
    else
        n = 5;

    start[0] = 0;
    for (int32_t i = 1; i < n; ++i)
        start[i] = (L >= 2) ? 1 + (int32_t)(synth_hash(key, (uint64_t)i) % (uint64_t)(L - 1)) : 0;
    /* insertion sort of the cut points */
    for (int32_t i = 2; i < n; ++i) {
        int32_t v = start[i], j = i - 1;
        while (j >= 1 && start[j] > v) {
            start[j + 1] = start[j];
            --j;
        }
        start[j + 1] = v;
    }

    if (rule == SYNTH_RULE_SET3) {
        for (int32_t i = 0; i < n; ++i)
            sigma[i] = set3[synth_hash(key, 100u + (uint64_t)i) % 3u];
    } else if (rule == SYNTH_RULE_U) {
        for (int32_t i = 0; i < n; ++i) {
            float u = (float)(uint32_t)(synth_hash(key, 100u + (uint64_t)i) >> 40) * 0x1p-24f;
            sigma[i] = 0.03f + 0.47f * u;
        }
    } else {
        float s[5];
        for (int32_t i = 0; i < 5; ++i) s[i] = set5[i];
        for (int32_t i = 4; i > 0; --i) { /* Fisher-Yates */
            int32_t j = (int32_t)(synth_hash(key, 200u + (uint64_t)i) % (uint64_t)(i + 1));
            float t = s[i];
            s[i] = s[j];
            s[j] = t;
        }
        for (int32_t i = 0; i < 5; ++i) sigma[i] = s[i];
    }
    for (int32_t i = n; i < SYNTH_MAX_SPANS; ++i) {
        start[i] = L;
        sigma[i] = 0.0f;
    }
    return n;
}

static float span_sigma_at(int32_t t, int32_t n, const int32_t *start, const float *sigma)
{
    int32_t s = 0;
    for (int32_t i = 1; i < n; ++i)
        if (start[i] <= t) s = i;
    return sigma[s];
}

/* K or V of one (layer, request, head): L rows of D bf16 values, rows `row_stride`
 * elements apart. Element (t, d) is draw number t*D + d of the pair's stream. */
void synth_fill_pair(uint64_t seed, uint32_t stream, uint32_t layer, uint32_t req,
                     uint32_t head, int32_t L, int32_t D, int32_t n_spans,
                     const int32_t *start, const float *sigma, uint16_t *out,
                     int64_t row_stride)
{
    uint64_t key = synth_key(seed, stream, layer, req, head);
    for (int32_t t = 0; t < L; ++t) {
        float sg = span_sigma_at(t, n_spans, start, sigma);
        for (int32_t d = 0; d < D; ++d)
            out[(int64_t)t * row_stride + d] =
                synth_gauss_bf16(key, (uint64_t)t * (uint64_t)D + (uint64_t)d, sg);
    }
}

/* Whole layer of packed variable-length K or V, [T, H, D], request b owning rows
 * cu_seqlens[b] .. cu_seqlens[b+1]; span tables are [B*H] counts, [B*H*5] starts and
 * sigmas, indexed b*H + h. */
void synth_fill_layer(uint64_t seed, uint32_t stream, uint32_t layer, int32_t B, int32_t H,
                      int32_t D, const int32_t *cu_seqlens, const int32_t *span_n,
                      const int32_t *span_start, const float *span_sigma, uint16_t *out)
{
    for (int32_t b = 0; b < B; ++b) {
        int32_t L = cu_seqlens[b + 1] - cu_seqlens[b];
        for (int32_t h = 0; h < H; ++h) {
            int64_t p = (int64_t)b * H + h;
            synth_fill_pair(seed, stream, layer, (uint32_t)b, (uint32_t)h, L, D, span_n[p],
                            span_start + p * SYNTH_MAX_SPANS, span_sigma + p * SYNTH_MAX_SPANS,
                            out + ((int64_t)cu_seqlens[b] * H + h) * D, (int64_t)H * D);
        }
    }
}

/* One vector per (request, head) with constant sigma: out is [B, H, D]. */
void synth_fill_heads(uint64_t seed, uint32_t stream, uint32_t layer, int32_t B, int32_t H,
                      int32_t D, float sigma, uint16_t *out)
{
    for (int32_t b = 0; b < B; ++b)
        for (int32_t h = 0; h < H; ++h) {
            uint64_t key = synth_key(seed, stream, layer, (uint32_t)b, (uint32_t)h);
            for (int32_t d = 0; d < D; ++d)
                out[((int64_t)b * H + h) * D + d] = synth_gauss_bf16(key, (uint64_t)d, sigma);
        }
}

/* Uniform random bytes for one (layer, block, head) code tile (decode-only tests that
 * need a cache without going through compression). */
void synth_fill_bytes(uint64_t seed, uint32_t stream, uint32_t layer, int64_t n, uint8_t *out)
{
    uint64_t key = synth_key(seed, stream, layer, 0, 0);
    for (int64_t i = 0; i < n; ++i)
        out[i] = (uint8_t)(synth_hash(key, (uint64_t)i) >> 56);
}

/* Random permutation of 0..n-1 (Fisher-Yates driven by the SplitMix64 stream). */
void synth_permutation(uint64_t seed, uint32_t stream, int64_t n, int32_t *out)
{
    uint64_t key = synth_key(seed, stream, 0, 0, 0);
    for (int64_t i = 0; i < n; ++i) out[i] = (int32_t)i;
    for (int64_t i = n - 1; i > 0; --i) {
        int64_t j = (int64_t)(synth_hash(key, (uint64_t)i) % (uint64_t)(i + 1));
        int32_t t = out[i];
        out[i] = out[j];
        out[j] = t;
    }
}
