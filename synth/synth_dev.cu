/*
 * synth_dev.cu -- device side of the seeded synthetic-input generator (libsynth_dev.so).
 *
 * Fills device buffers with exactly the bits synth.c produces on the host (same
 * synth_core.h, compiled with -fmad=false), so full-size benchmark inputs can be made
 * on the GPU while the CPU oracle regenerates any slice it checks from the host
 * library.  Test and bench infrastructure only; holds none of the DGQ method.
 */
#include "synth_core.h"

#include <cuda_runtime.h>
#include <stdint.h>

#define SYNTH_MAX_SPANS 5

/* One thread per 8 consecutive elements of one (token, head) row (D % 8 == 0). */
__global__ void synth_layer_kernel(uint64_t seed, uint32_t stream, uint32_t layer, int32_t B,
                                   int32_t H, int32_t D, const int32_t *__restrict__ cu_seqlens,
                                   const int32_t *__restrict__ span_n,
                                   const int32_t *__restrict__ span_start,
                                   const float *__restrict__ span_sigma, int64_t total_rows,
                                   uint16_t *__restrict__ out)
{
    const int32_t groups = D / 8;
    int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= total_rows * groups) return;
    int64_t row = i / groups; /* row = t_glob * H + h */
    int32_t g = (int32_t)(i % groups);
    int64_t tg = row / H;
    int32_t h = (int32_t)(row % H);
    int32_t lo = 0, hi = B - 1; /* request owning global token tg */
    while (lo < hi) {
        int32_t mid = (lo + hi + 1) >> 1;
        if (cu_seqlens[mid] <= tg) lo = mid;
        else hi = mid - 1;
    }
    int32_t b = lo;
    int32_t t = (int32_t)(tg - cu_seqlens[b]);
    int64_t p = (int64_t)b * H + h;
    int32_t n = span_n[p];
    int32_t s = 0;
    for (int32_t k = 1; k < n; ++k)
        if (span_start[p * SYNTH_MAX_SPANS + k] <= t) s = k;
    float sg = span_sigma[p * SYNTH_MAX_SPANS + s];
    uint64_t key = synth_key(seed, stream, layer, (uint32_t)b, (uint32_t)h);
    uint16_t v[8];
#pragma unroll
    for (int j = 0; j < 8; ++j)
        v[j] = synth_gauss_bf16(key, (uint64_t)t * (uint64_t)D + (uint64_t)(g * 8 + j), sg);
    uint4 w;
    w.x = (uint32_t)v[0] | ((uint32_t)v[1] << 16);
    w.y = (uint32_t)v[2] | ((uint32_t)v[3] << 16);
    w.z = (uint32_t)v[4] | ((uint32_t)v[5] << 16);
    w.w = (uint32_t)v[6] | ((uint32_t)v[7] << 16);
    *reinterpret_cast<uint4 *>(out + row * D + g * 8) = w;
}

__global__ void synth_heads_kernel(uint64_t seed, uint32_t stream, uint32_t layer, int32_t B,
                                   int32_t H, int32_t D, float sigma, uint16_t *__restrict__ out)
{
    int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= (int64_t)B * H * D) return;
    int32_t d = (int32_t)(i % D);
    int64_t bh = i / D;
    int32_t h = (int32_t)(bh % H);
    int32_t b = (int32_t)(bh / H);
    uint64_t key = synth_key(seed, stream, layer, (uint32_t)b, (uint32_t)h);
    out[i] = synth_gauss_bf16(key, (uint64_t)d, sigma);
}

__global__ void synth_bytes_kernel(uint64_t seed, uint32_t stream, uint32_t layer, int64_t n,
                                   uint8_t *__restrict__ out)
{
    int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= n) return;
    uint64_t key = synth_key(seed, stream, layer, 0, 0);
    out[i] = (uint8_t)(synth_hash(key, (uint64_t)i) >> 56);
}

extern "C" {

/* All pointers are device pointers; span tables as in synth_fill_layer (host). */
int synth_dev_fill_layer(uint64_t seed, uint32_t stream, uint32_t layer, int32_t B, int32_t H,
                         int32_t D, const int32_t *cu_seqlens, const int32_t *span_n,
                         const int32_t *span_start, const float *span_sigma, int64_t total_tokens,
                         uint16_t *out, void *stream_ptr)
{
    if (D % 8 != 0 || B <= 0 || H <= 0) return -1;
    int64_t rows = total_tokens * H;
    int64_t threads = rows * (D / 8);
    if (threads == 0) return 0;
    int64_t blocks = (threads + 255) / 256;
    synth_layer_kernel<<<(unsigned)blocks, 256, 0, (cudaStream_t)stream_ptr>>>(
        seed, stream, layer, B, H, D, cu_seqlens, span_n, span_start, span_sigma, rows, out);
    return (int)cudaGetLastError();
}

int synth_dev_fill_heads(uint64_t seed, uint32_t stream, uint32_t layer, int32_t B, int32_t H,
                         int32_t D, float sigma, uint16_t *out, void *stream_ptr)
{
    int64_t n = (int64_t)B * H * D;
    if (n == 0) return 0;
    synth_heads_kernel<<<(unsigned)((n + 255) / 256), 256, 0, (cudaStream_t)stream_ptr>>>(
        seed, stream, layer, B, H, D, sigma, out);
    return (int)cudaGetLastError();
}

int synth_dev_fill_bytes(uint64_t seed, uint32_t stream, uint32_t layer, int64_t n, uint8_t *out,
                         void *stream_ptr)
{
    if (n == 0) return 0;
    synth_bytes_kernel<<<(unsigned)((n + 255) / 256), 256, 0, (cudaStream_t)stream_ptr>>>(
        seed, stream, layer, n, out);
    return (int)cudaGetLastError();
}

} /* extern "C" */
