/*
 * synth_core.h -- seeded synthetic inputs for the DGQ KV-cache tests and bench.
 *
 * This module generates K/V/Q tensors; it holds none of the DGQ method's arithmetic
 * (no variance, no segmentation, no quantisation, no attention).  It is compiled
 * twice from this one header: as C by gcc for the host library (libsynth.so) and as
 * CUDA by nvcc for the device filler (libsynth_dev.so).  Both builds must produce
 * identical bits, so every floating-point step below is a single IEEE-754 binary32
 * operation (+, -, *, /, sqrt) compiled without FMA contraction
 * (gcc -ffp-contract=off, nvcc -fmad=false), and the transcendental functions are
 * written out here as short polynomials instead of calling a math library.
 *
 * Generator (published definitions):
 *   - SplitMix64 (Steele, Lea & Flood, "Fast splittable pseudorandom number
 *     generators", OOPSLA 2014; finaliser constants as in Vigna's splitmix64.c),
 *     used in counter form: output n of a stream with state s is mix(s + (n+1)*gamma).
 *   - Box-Muller (Box & Muller, 1958): n = sqrt(-2 ln u1) * cos(2 pi u2).
 *     ln is evaluated as e*ln2 + 2*atanh((m-1)/(m+1)) with the atanh Taylor series
 *     to s^11; cos(2 pi x) by quadrant folding and the cosine Taylor series to
 *     theta^12.  Both are accurate to a few 1e-7 relative, which is ample for
 *     synthetic data; what matters is that host and device agree bit for bit.
 *   - bf16 from fp32 by round-to-nearest-even on the bit pattern.
 */
#ifndef SYNTH_CORE_H
#define SYNTH_CORE_H

#include <stdint.h>
#if !defined(__CUDA_ARCH__)
#include <math.h>
#endif

#if defined(__CUDACC__)
#define SYNTH_FN static __host__ __device__ __forceinline__
#else
#define SYNTH_FN static inline
#endif

#define SYNTH_GAMMA 0x9E3779B97F4A7C15ULL

/* Streams: independent tensors drawn for one (layer, request, head). */
enum {
    SYNTH_STREAM_K = 1,
    SYNTH_STREAM_V = 2,
    SYNTH_STREAM_Q = 3,
    SYNTH_STREAM_KNEW = 4,
    SYNTH_STREAM_VNEW = 5,
    SYNTH_STREAM_SPAN = 6,
    SYNTH_STREAM_CODES = 7,
    SYNTH_STREAM_META = 8
};

SYNTH_FN uint64_t synth_mix(uint64_t z)
{
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
    return z ^ (z >> 31);
}

/* Output number `ctr` of the SplitMix64 stream whose state starts at `key`. */
SYNTH_FN uint64_t synth_hash(uint64_t key, uint64_t ctr)
{
    return synth_mix(key + (ctr + 1ULL) * SYNTH_GAMMA);
}

SYNTH_FN uint64_t synth_key(uint64_t seed, uint32_t stream, uint32_t layer,
                            uint32_t req, uint32_t head)
{
    uint64_t k = synth_hash(seed, stream);
    k = synth_hash(k, layer);
    k = synth_hash(k, req);
    return synth_hash(k, head);
}

SYNTH_FN float synth_f32_from_bits(uint32_t b)
{
    union { uint32_t u; float f; } c;
    c.u = b;
    return c.f;
}

SYNTH_FN uint32_t synth_bits_from_f32(float f)
{
    union { uint32_t u; float f; } c;
    c.f = f;
    return c.u;
}

/* Natural log for x in [2^-24, 1] (x is always k * 2^-24, k >= 1, here). */
SYNTH_FN float synth_ln(float x)
{
    uint32_t b = synth_bits_from_f32(x);
    int e = (int)((b >> 23) & 0xFFu) - 127;
    float m = synth_f32_from_bits((b & 0x7FFFFFu) | 0x3F800000u); /* [1, 2) */
    if (m > 1.41421354f) {
        m = m * 0.5f;
        e += 1;
    }
    float s = (m - 1.0f) / (m + 1.0f); /* |s| <= 0.1716 */
    float s2 = s * s;
    float p = 0x1.745d18p-4f;          /* 1/11 */
    p = p * s2 + 0x1.c71c72p-4f;       /* 1/9  */
    p = p * s2 + 0x1.24924ap-3f;       /* 1/7  */
    p = p * s2 + 0x1.99999ap-3f;       /* 1/5  */
    p = p * s2 + 0x1.555556p-2f;       /* 1/3  */
    p = p * s2 + 1.0f;
    float lnm = (2.0f * s) * p;
    return (float)e * 0x1.62e430p-1f + lnm; /* ln 2 */
}

/* cos(2*pi*x) for x in [0, 1). */
SYNTH_FN float synth_cos2pi(float x)
{
    float y = x > 0.5f ? 1.0f - x : x; /* cos is even and 1-periodic: y in [0, 0.5] */
    float sign = 1.0f;
    if (y > 0.25f) { /* cos(2 pi y) = -cos(2 pi (0.5 - y)) */
        y = 0.5f - y;
        sign = -1.0f;
    }
    float t = y * 0x1.921fb6p+2f; /* 2*pi*y in [0, pi/2] */
    float t2 = t * t;
    float p = 0x1.1ee9ecp-29f;          /*  1/12! */
    p = p * t2 - 0x1.27e4fcp-22f;       /* -1/10! */
    p = p * t2 + 0x1.a01a02p-16f;       /*  1/8!  */
    p = p * t2 - 0x1.6c16c2p-10f;       /* -1/6!  */
    p = p * t2 + 0x1.555556p-5f;        /*  1/4!  */
    p = p * t2 - 0.5f;
    p = p * t2 + 1.0f;
    return sign * p;
}

/* One N(0,1) deviate from one 64-bit hash (Box-Muller, cosine branch). */
SYNTH_FN float synth_normal_from_hash(uint64_t h)
{
    float u1 = (float)((uint32_t)(h >> 40) + 1u) * 0x1p-24f;     /* (0, 1] */
    float u2 = (float)((uint32_t)(h >> 16) & 0xFFFFFFu) * 0x1p-24f; /* [0, 1) */
    float r = -2.0f * synth_ln(u1);
#if defined(__CUDA_ARCH__)
    r = __fsqrt_rn(r);
#else
    r = sqrtf(r);
#endif
    return r * synth_cos2pi(u2);
}

/* fp32 -> bf16 bit pattern, round to nearest even (inputs are finite). */
SYNTH_FN uint16_t synth_bf16(float f)
{
    uint32_t b = synth_bits_from_f32(f);
    uint32_t lsb = (b >> 16) & 1u;
    b += 0x7FFFu + lsb;
    return (uint16_t)(b >> 16);
}

/* Element `ctr` of a Gaussian tensor stream with standard deviation sigma, as bf16. */
SYNTH_FN uint16_t synth_gauss_bf16(uint64_t key, uint64_t ctr, float sigma)
{
    return synth_bf16(sigma * synth_normal_from_hash(synth_hash(key, ctr)));
}

#endif /* SYNTH_CORE_H */
