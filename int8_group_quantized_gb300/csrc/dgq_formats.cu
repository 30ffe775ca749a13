// dgq_formats.cu -- the comparison encodings written into the same paged cache layout as DGQ
// (sm_103a): fixed 64-value groups, symmetric per-(request, head) INT8 and FP8 E4M3.
//
// Method:
//  * fixed groups: "DeepSeek KV-cache dynamic group quantisation (DGQ)" article, section 2.2
//    (the traditional scheme it replaces: fixed blocks of 64 dimensions, each with its own
//    min/max INT8 parameters), encoded with the DGQ quantiser's own steps on each group;
//  * symmetric INT8: "DeepSeek-V4 high-concurrency KV-cache bottleneck" article, FP8+FP16
//    scheme section (scale = max|k| / 127, k / scale held to [-128, 127]; rounded half-even);
//  * FP8 E4M3: the DGQ article's section 2.3 format table (E4M3 row): each value rounded to
//    the nearest E4M3 number, saturating at +-448.
// Token t of request b, head h goes to pool[block_tables[b][t / bs]][h][t % bs] ("PagedAttention
// implementation" section of the DeepSeek-V4 article).
//
// GPU design: memory-bound codecs.  A CTA takes 256 tokens of one (request, head) pair, one warp
// per token row at a time (lane i holds values 4i .. 4i+3 of the K row and of the V row: 8-byte
// loads, 4-byte code stores, both coalesced per row), four rows in flight per warp.  The
// symmetric format first reduces max|x| per pair (one order-preserving integer atomic per CTA
// and tensor), then encodes.  The first CTA of each pair writes its record.  Compiled with
// -fmad=false; every step that decides a code is a single IEEE operation.
#include "dgq_device.cuh"
#include "dgq.h"
#include "dgq_launch.h"

#include <cuda_fp8.h>
#include <stdint.h>

namespace dgq {

constexpr int kFmtWarps = 8;
constexpr int kFmtTokens = 256;   // tokens per CTA
constexpr int kFmtUnroll = 4;     // rows in flight per warp

struct FormatArgs {
    const uint2 *k;  // [T, Hkv, 32] groups of four bf16
    const uint2 *v;
    int32_t T;
    const int32_t *cu;
    const int32_t *bt;
    uint8_t *kpool, *vpool;
    float4 *kpar, *vpar;  // fixed groups: [num_blocks * Hkv * bs] (min0, scale0, min1, scale1)
    dgq_seg_record *table;
    uint32_t *amax;       // symmetric: [pairs][2] bit patterns of max|x| (K, V)
    WsHeader *hdr;
    int32_t B, Hkv, bs, max_blocks, num_blocks;
};

__device__ __forceinline__ float fb_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float fb_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// min/max over the 16 lanes of a half row (lanes 0-15: values 0..63; 16-31: 64..127); -0 as +0
__device__ __forceinline__ void half_min_max(const float (&x)[4], float &mn, float &mx)
{
    mn = fminf(fminf(x[0], x[1]), fminf(x[2], x[3]));
    mx = fmaxf(fmaxf(x[0], x[1]), fmaxf(x[2], x[3]));
#pragma unroll
    for (int o = 8; o; o >>= 1) {
        mn = fminf(mn, __shfl_xor_sync(0xffffffffu, mn, o));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    }
    if (mn == 0.0f) mn = 0.0f;
    if (mx == 0.0f) mx = 0.0f;
}

// Four affine codes rint((x - mn) * inv) (x >= mn, so 0 <= u < 255.5 and the 1.5 * 2^23 add
// rounds half-even and leaves the code in the low byte), packed little-endian.
__device__ __forceinline__ uint32_t affine4(const float (&x)[4], float mn, float inv)
{
    uint32_t c = 0;
#pragma unroll
    for (int e = 0; e < 4; ++e) {
        const float u = __fmul_rn(__fsub_rn(x[e], mn), inv);
        c |= (__float_as_uint(__fadd_rn(u, 12582912.0f)) & 0xFFu) << (8 * e);
    }
    return c;
}

// Four symmetric codes rint(x / s) held to [-128, 127], stored as q + 128.
__device__ __forceinline__ uint32_t sym4(const float (&x)[4], float s)
{
    uint32_t c = 0;
#pragma unroll
    for (int e = 0; e < 4; ++e) {
        float q = s > 0.0f ? rintf(__fdiv_rn(x[e], s)) : 0.0f;
        q = fminf(fmaxf(q, -128.0f), 127.0f);
        c |= ((uint32_t)((int32_t)q + 128) & 0xFFu) << (8 * e);
    }
    return c;
}

// Four E4M3 bytes, round-half-even with saturation to the largest finite value.
__device__ __forceinline__ uint32_t e4m3x4(const float (&x)[4])
{
    const uint32_t lo = __nv_cvt_float2_to_fp8x2(make_float2(x[0], x[1]), __NV_SATFINITE, __NV_E4M3);
    const uint32_t hi = __nv_cvt_float2_to_fp8x2(make_float2(x[2], x[3]), __NV_SATFINITE, __NV_E4M3);
    return (lo & 0xFFFFu) | (hi << 16);
}

__device__ __forceinline__ void load4(const uint2 w, float (&x)[4])
{
    x[0] = fb_lo(w.x);
    x[1] = fb_hi(w.x);
    x[2] = fb_lo(w.y);
    x[3] = fb_hi(w.y);
}

// the pair and token range of this CTA; false when the CTA has no tokens (or a bad length)
struct FmtTile {
    int32_t b, h, L, row0, t0, t1;
};

__device__ __forceinline__ bool fmt_tile(const FormatArgs &a, FmtTile &ft)
{
    const int32_t pair = blockIdx.x;
    ft.b = pair / a.Hkv;
    ft.h = pair - ft.b * a.Hkv;
    const int32_t c0 = __ldg(a.cu + ft.b), c1 = __ldg(a.cu + ft.b + 1);
    ft.L = c1 - c0;
    ft.row0 = c0;
    ft.t0 = blockIdx.y * kFmtTokens;
    ft.t1 = min(ft.t0 + kFmtTokens, ft.L);
    if (ft.L < 0 || c0 < 0 || c1 > a.T || (int64_t)ft.L > (int64_t)a.max_blocks * a.bs) {
        if (threadIdx.x == 0 && blockIdx.y == 0) record_error(a.hdr, kErrBadLength);
        return false;
    }
    return ft.t0 < ft.t1;
}

// max |x| of each pair's K and V (symmetric format, first pass)
__global__ void __launch_bounds__(kFmtWarps * 32) sym_amax_kernel(FormatArgs a)
{
    FmtTile ft;
    if (!fmt_tile(a, ft)) return;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    float km = 0.0f, vm = 0.0f;
    for (int32_t t = ft.t0 + warp; t < ft.t1; t += kFmtWarps * kFmtUnroll) {
        uint2 kw[kFmtUnroll], vw[kFmtUnroll];
#pragma unroll
        for (int u = 0; u < kFmtUnroll; ++u) {
            const int32_t tt = t + u * kFmtWarps;
            const int64_t row = ((int64_t)(ft.row0 + tt) * a.Hkv + ft.h) * 32 + lane;
            kw[u] = tt < ft.t1 ? __ldcs(a.k + row) : make_uint2(0u, 0u);
            vw[u] = tt < ft.t1 ? __ldcs(a.v + row) : make_uint2(0u, 0u);
        }
#pragma unroll
        for (int u = 0; u < kFmtUnroll; ++u) {
            float x[4], y[4];
            load4(kw[u], x);
            load4(vw[u], y);
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                km = fmaxf(km, fabsf(x[e]));
                vm = fmaxf(vm, fabsf(y[e]));
            }
        }
    }
#pragma unroll
    for (int o = 16; o; o >>= 1) {
        km = fmaxf(km, __shfl_xor_sync(0xffffffffu, km, o));
        vm = fmaxf(vm, __shfl_xor_sync(0xffffffffu, vm, o));
    }
    __shared__ float s_m[kFmtWarps][2];
    if (lane == 0) {
        s_m[warp][0] = km;
        s_m[warp][1] = vm;
    }
    __syncthreads();
    if (threadIdx.x < 2) {
        float m = 0.0f;
        for (int w = 0; w < kFmtWarps; ++w) m = fmaxf(m, s_m[w][threadIdx.x]);
        // non-negative floats order like their bit patterns
        atomicMax(a.amax + 2 * (int64_t)blockIdx.x + threadIdx.x, __float_as_uint(m));
    }
}

template <int Fmt>
__global__ void __launch_bounds__(kFmtWarps * 32) format_encode_kernel(FormatArgs a)
{
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int32_t pair = blockIdx.x;
    float ks = 0.0f, vs = 0.0f;  // symmetric scales
    if (Fmt == DGQ_FORMAT_SYM_INT8) {
        ks = __fdiv_rn(__uint_as_float(__ldcg(a.amax + 2 * (int64_t)pair)), 127.0f);
        vs = __fdiv_rn(__uint_as_float(__ldcg(a.amax + 2 * (int64_t)pair + 1)), 127.0f);
    }
    FmtTile ft;
    const bool any = fmt_tile(a, ft);
    if (blockIdx.y == 0 && warp == 0) {  // the pair's record, lane i writing word i
        const int32_t L = max(ft.L, 0);
        uint32_t w = 0u;
        const bool sym = Fmt == DGQ_FORMAT_SYM_INT8;
        const float kmin = ks > 0.0f ? -128.0f * ks : 0.0f, vmin = vs > 0.0f ? -128.0f * vs : 0.0f;
        if (lane == 0) w = L > 0 ? 1u : 0u;                       // n_seg
        if (lane == 1) w = (uint32_t)L;                           // seq_len
        if (lane >= 3 && lane <= 6) w = (uint32_t)L;              // start[1..4]
        if (L > 0) {
            if (lane == 7) w = __float_as_uint(sym ? kmin : 0.0f);    // k_min[0]
            if (lane == 12) w = __float_as_uint(sym ? ks : 1.0f);     // k_scale[0]
            if (lane == 17) w = __float_as_uint(sym ? vmin : 0.0f);   // v_min[0]
            if (lane == 22) w = __float_as_uint(sym ? vs : 1.0f);     // v_scale[0]
        }
        reinterpret_cast<uint32_t *>(a.table + pair)[lane] = w;
    }
    if (!any) return;
    for (int32_t t = ft.t0 + warp; t < ft.t1; t += kFmtWarps * kFmtUnroll) {
        uint2 kw[kFmtUnroll], vw[kFmtUnroll];
#pragma unroll
        for (int u = 0; u < kFmtUnroll; ++u) {
            const int32_t tt = t + u * kFmtWarps;
            const int64_t row = ((int64_t)(ft.row0 + tt) * a.Hkv + ft.h) * 32 + lane;
            kw[u] = tt < ft.t1 ? __ldcs(a.k + row) : make_uint2(0u, 0u);
            vw[u] = tt < ft.t1 ? __ldcs(a.v + row) : make_uint2(0u, 0u);
        }
#pragma unroll
        for (int u = 0; u < kFmtUnroll; ++u) {
            const int32_t tt = t + u * kFmtWarps;
            if (tt >= ft.t1) break;  // warp-uniform
            const int32_t blk = __ldg(a.bt + (int64_t)ft.b * a.max_blocks + tt / a.bs);
            if ((uint32_t)blk >= (uint32_t)a.num_blocks) {  // not a block of the pools: skipped
                if (lane == 0) record_error(a.hdr, kErrBadBlock);
                continue;
            }
            const int64_t slot = ((int64_t)blk * a.Hkv + ft.h) * a.bs + tt % a.bs;
            float x[4], y[4];
            load4(kw[u], x);
            load4(vw[u], y);
            uint32_t kc, vc;
            if (Fmt == DGQ_FORMAT_FIXED64) {
                float kmn, kmx, vmn, vmx, ksc, kinv, vsc, vinv;
                half_min_max(x, kmn, kmx);
                half_min_max(y, vmn, vmx);
                const float kr = __fsub_rn(kmx, kmn), vr = __fsub_rn(vmx, vmn);
                ksc = kr == 0.0f ? 0.0f : __fdiv_rn(kr, 255.0f);
                kinv = kr == 0.0f ? 0.0f : __fdiv_rn(255.0f, kr);
                vsc = vr == 0.0f ? 0.0f : __fdiv_rn(vr, 255.0f);
                vinv = vr == 0.0f ? 0.0f : __fdiv_rn(255.0f, vr);
                kc = affine4(x, kmn, kinv);
                vc = affine4(y, vmn, vinv);
                // lane 0 stores both halves' parameters (lane 16 holds the second half's)
                const float kmn1 = __shfl_sync(0xffffffffu, kmn, 16), ksc1 = __shfl_sync(0xffffffffu, ksc, 16);
                const float vmn1 = __shfl_sync(0xffffffffu, vmn, 16), vsc1 = __shfl_sync(0xffffffffu, vsc, 16);
                if (lane == 0) {
                    __stcs(a.kpar + slot, make_float4(kmn, ksc, kmn1, ksc1));
                    __stcs(a.vpar + slot, make_float4(vmn, vsc, vmn1, vsc1));
                }
            } else if (Fmt == DGQ_FORMAT_SYM_INT8) {
                kc = sym4(x, ks);
                vc = sym4(y, vs);
            } else {
                kc = e4m3x4(x);
                vc = e4m3x4(y);
            }
            __stcs(reinterpret_cast<uint32_t *>(a.kpool + slot * kD) + lane, kc);
            __stcs(reinterpret_cast<uint32_t *>(a.vpool + slot * kD) + lane, vc);
        }
    }
}

size_t format_workspace_bytes(int32_t B, int32_t Hkv)
{
    return sizeof(WsHeader) + (((size_t)B * Hkv * 8 + 255) & ~(size_t)255);
}

cudaError_t launch_format_encode(int32_t fmt, const void *k, const void *v, int32_t T, const int32_t *cu, int32_t B,
                                 int32_t max_seqlen, int32_t Hkv, int32_t bs, const int32_t *bt, int32_t max_blocks,
                                 uint8_t *kpool, uint8_t *vpool, int32_t num_blocks, float *kpar, float *vpar,
                                 dgq_seg_record *table, void *ws, cudaStream_t stream)
{
    FormatArgs a;
    a.k = static_cast<const uint2 *>(k);
    a.v = static_cast<const uint2 *>(v);
    a.T = T;
    a.cu = cu;
    a.bt = bt;
    a.kpool = kpool;
    a.vpool = vpool;
    a.kpar = reinterpret_cast<float4 *>(kpar);
    a.vpar = reinterpret_cast<float4 *>(vpar);
    a.table = table;
    a.hdr = static_cast<WsHeader *>(ws);
    a.amax = reinterpret_cast<uint32_t *>(static_cast<uint8_t *>(ws) + sizeof(WsHeader));
    a.B = B;
    a.Hkv = Hkv;
    a.bs = bs;
    a.max_blocks = max_blocks;
    a.num_blocks = num_blocks;
    const dim3 grid((unsigned)(B * Hkv), (unsigned)max(1, (max_seqlen + kFmtTokens - 1) / kFmtTokens));
    const dim3 block(kFmtWarps * 32);
    if (fmt == DGQ_FORMAT_SYM_INT8) {
        cudaError_t e = cudaMemsetAsync(a.amax, 0, (size_t)B * Hkv * 8, stream);
        if (e != cudaSuccess) return e;
        sym_amax_kernel<<<grid, block, 0, stream>>>(a);
        format_encode_kernel<DGQ_FORMAT_SYM_INT8><<<grid, block, 0, stream>>>(a);
    } else if (fmt == DGQ_FORMAT_FIXED64) {
        format_encode_kernel<DGQ_FORMAT_FIXED64><<<grid, block, 0, stream>>>(a);
    } else {
        format_encode_kernel<DGQ_FORMAT_FP8_E4M3><<<grid, block, 0, stream>>>(a);
    }
    return cudaGetLastError();
}

}  // namespace dgq
