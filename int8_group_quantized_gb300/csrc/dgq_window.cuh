// dgq_window.cuh -- per-window arithmetic shared by the two compress kernels: window statistics
// (balanced fp32 sums of the per-token variance, K/V extremes), segment parameters and the
// quantiser, all in the exact IEEE steps the method fixes.  Included by dgq_compress.cu and
// dgq_compress_cluster.cu, both compiled with -fmad=false.
#pragma once

#include "dgq_device.cuh"
#include "dgq.h"
#include "dgq_launch.h"

#include <cuda_bf16.h>
#include <stdint.h>

namespace dgq {

constexpr int kTileBytes = kWin * kD * 2;  // 16 tokens x 128 bf16 = 4 KB
constexpr int kWinBytes = 2 * kTileBytes;  // K tile + V tile

// Quantisation parameters of one pair as the segmentation warp publishes them.
struct alignas(16) PairParams {
    float k_min[kMaxSeg], k_inv[kMaxSeg], v_min[kMaxSeg], v_inv[kMaxSeg];
    int32_t start[kMaxSeg];
    int32_t n_seg;
    int32_t pad[6];
};
static_assert(sizeof(PairParams) == 128, "PairParams is 128 bytes");


// ---- warp reductions ------------------------------------------------------------------------

__device__ __forceinline__ float warp_min(float v)
{
#pragma unroll
    for (int o = 16; o; o >>= 1) v = fminf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}

__device__ __forceinline__ float warp_max(float v)
{
#pragma unroll
    for (int o = 16; o; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}

__device__ __forceinline__ float canon_zero(float x) { return x == 0.0f ? 0.0f : x; }

// ---- packed fp32 pairs ----------------------------------------------------------------------
//
// sm_100-class GPUs execute fp32 add/sub/mul/fma on register pairs (f32x2); each half is an
// ordinary IEEE operation with round-to-nearest-even.  Measured on this GPU: a packed multiply
// whose result feeds a packed add is contracted into a fused multiply-add by the assembler,
// even with explicit rounding, which would change the rounding.  So products that feed packed
// sums here are scalar __fmul_rn, and the one packed product (the quantiser's) feeds a packed
// fused multiply-add by one, which the assembler leaves alone (checked on near-tie inputs).
__device__ __forceinline__ uint64_t f2_pack(uint32_t lo_bits, uint32_t hi_bits)
{
    uint64_t r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "r"(lo_bits), "r"(hi_bits));
    return r;
}
__device__ __forceinline__ void f2_unpack(uint64_t v, uint32_t &lo_bits, uint32_t &hi_bits)
{
    asm("mov.b64 {%0, %1}, %2;" : "=r"(lo_bits), "=r"(hi_bits) : "l"(v));
}
__device__ __forceinline__ uint64_t f2_add(uint64_t a, uint64_t b)
{
    uint64_t r;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
    return r;
}
__device__ __forceinline__ uint64_t f2_mul(uint64_t a, uint64_t b)
{
    uint64_t r;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
    return r;
}
__device__ __forceinline__ uint64_t f2_fma(uint64_t a, uint64_t b, uint64_t c)
{
    uint64_t r;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(a), "l"(b), "l"(c));
    return r;
}
__device__ __forceinline__ uint32_t f2u(float x) { return __float_as_uint(x); }

// ---- mixed bf16 / fp32 arithmetic -----------------------------------------------------------
//
// sm_100-class GPUs add and subtract a bf16 operand to or from an fp32 one directly: the bf16
// value is widened exactly and the fp32 result rounded once (round-to-nearest-even), the same
// IEEE operation as widening first, without the unpacking instruction.

// x - c for the two bf16 of a word (low half to d_lo).
__device__ __forceinline__ void bf2_sub(uint32_t w, float c, float &d_lo, float &d_hi)
{
    asm("{\n.reg .b16 lo, hi;\nmov.b32 {lo, hi}, %2;\nsub.rn.f32.bf16 %0, lo, %3;\nsub.rn.f32.bf16 %1, hi, %3;\n}"
        : "=f"(d_lo), "=f"(d_hi)
        : "r"(w), "f"(c));
}
// x_lo + x_hi of the two bf16 of a word, in fp32 (one rounding).
__device__ __forceinline__ float bf2_sum(uint32_t w)
{
    float r;
    asm("{\n.reg .b16 lo, hi;\nmov.b32 {lo, hi}, %1;\nadd.rn.f32.bf16 %0, hi, %2;\n}"
        : "=f"(r)
        : "r"(w), "f"(__uint_as_float(w << 16)));
    return r;
}

// ---- window tiles ----------------------------------------------------------------------------
//
// K and V come either as packed rows [T, Hkv, 128] bf16 -- a tensor map views each as 4-D (64
// elements, 2 halves, Hkv, T) -- or from a bf16 paged cache [blocks, Hkv, bs, 128] addressed
// through a block table -- then a 5-D map (64, 2, bs, Hkv, blocks) and the window's block.
// One copy per tensor brings the tile of a window -- 16 tokens of one head -- into shared memory
// as 32 rows of 128 bytes (row 2t + half) with the 128-byte swizzle: 16-byte chunk c of row r sits
// at chunk position c ^ (r & 7) (the tile starts on a 1024-byte boundary).  Packed rows at or
// past T are filled with zeros; rows of a partial window past its request's end hold other
// tokens (the next request's, or the rest of the block), and every reader masks them.  With this
// layout the statistics' row reads (eight lanes on eight consecutive rows) and the quantiser's
// chunk reads (eight lanes on one row) each touch eight distinct 16-byte bank groups per
// quarter-warp.
struct TileSource {
    CUtensorMap k, v;
    const int32_t *bt;  // paged source: [B, max_blocks] block table; null for packed rows
    int32_t max_blocks, num_blocks, bs;
};

// Byte offset of 16-byte chunk `chunk` (0..15) of token t in a tile.
__device__ __forceinline__ uint32_t tile_off(int t, int chunk)
{
    const int r = 2 * t + (chunk >> 3);
    return (uint32_t)(r * 128 + (((chunk & 7) ^ (r & 7)) << 4));
}

// Lane 0's copies of the window of tokens t0 .. t0+15 of request b (rows from c0 when packed),
// head h: K tile at dst, V tile at dst + kTileBytes, both completing on `bar` (one arrival,
// kWinBytes of transactions).  `pol`: the copies' L2 eviction policy.  A paged source's block id
// outside the cache is flagged in `hdr` and block 0 read instead (the copies always complete).
// (Fetching the source block one window ahead measured no faster: the copy is not waiting on it.)
__device__ __forceinline__ void load_window(uint32_t dst, uint64_t *bar, const TileSource &s, int32_t b, int32_t h,
                                            int32_t c0, int32_t t0, uint64_t pol, WsHeader *hdr)
{
    if (s.bt == nullptr) {
        mbar_arrive_expect_tx(bar, kWinBytes);
        tma_load_4d_hint(dst, &s.k, 0, 0, h, c0 + t0, smem_u32(bar), pol);
        tma_load_4d_hint(dst + kTileBytes, &s.v, 0, 0, h, c0 + t0, smem_u32(bar), pol);
    } else {
        int32_t blk = __ldg(s.bt + (int64_t)b * s.max_blocks + pow2_div(t0, s.bs));
        if ((uint32_t)blk >= (uint32_t)s.num_blocks) {
            record_error(hdr, kErrBadBlock);
            blk = 0;
        }
        mbar_arrive_expect_tx(bar, kWinBytes);
        tma_load_5d_hint(dst, &s.k, 0, 0, pow2_mod(t0, s.bs), h, blk, smem_u32(bar), pol);
        tma_load_5d_hint(dst + kTileBytes, &s.v, 0, 0, pow2_mod(t0, s.bs), h, blk, smem_u32(bar), pol);
    }
}

// Host: the tensor maps of a call's source; false if the driver refuses them.
inline bool encode_tile_source(const SourceDesc &d, int32_t Hkv, int32_t bs, TileSource *s)
{
    const PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
    if (!enc) return false;
    s->bt = d.bt;
    s->max_blocks = d.max_blocks;
    s->num_blocks = d.num_blocks;
    s->bs = bs;
    const void *src[2] = {d.k, d.v};
    CUtensorMap *dst[2] = {&s->k, &s->v};
    for (int i = 0; i < 2; ++i) {
        CUresult r;
        if (d.bt == nullptr) {
            const cuuint64_t dims[4] = {64, 2, (cuuint64_t)Hkv, (cuuint64_t)(d.T > 0 ? d.T : 1)};
            const cuuint64_t strides[3] = {128, 256, (cuuint64_t)Hkv * 256};  // bytes, dimensions 1..3
            const cuuint32_t box[4] = {64, 2, 1, kWin};
            const cuuint32_t estr[4] = {1, 1, 1, 1};
            r = enc(dst[i], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void *>(src[i]), dims, strides, box,
                    estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
        } else {
            const cuuint64_t dims[5] = {64, 2, (cuuint64_t)bs, (cuuint64_t)Hkv, (cuuint64_t)d.num_blocks};
            const cuuint64_t strides[4] = {128, 256, (cuuint64_t)bs * 256, (cuuint64_t)Hkv * bs * 256};
            const cuuint32_t box[5] = {64, 2, kWin, 1, 1};
            const cuuint32_t estr[5] = {1, 1, 1, 1, 1};
            r = enc(dst[i], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 5, const_cast<void *>(src[i]), dims, strides, box,
                    estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
        }
        if (r != CUDA_SUCCESS) return false;
    }
    return true;
}

// ---- statistics of one window (one warp, tile in shared memory) --------------------------
//
// Lane (t, hh) = (lane >> 1, lane & 1) takes elements [64 hh, 64 hh + 64) of token t (tile row
// 2t + hh).  Its 64-element sum is a balanced tree whose two 32-element halves run side by side
// in the two fp32 lanes of packed registers; one shuffle adds the other half-row.  This is the
// balanced pairwise order over the 128 elements, identical in both lanes of the token.

struct WinStats {
    float mean, kmn, kmx, vmn, vmx;
};

// Balanced sum of the 64 values of half-row hh of token t of a K tile: word i holds elements
// 2i, 2i+1 (bf16).  In each packed register the low half belongs to elements [0, 32), the
// high half to [32, 64).  With `squares`, `centre` is subtracted and the difference squared
// first.  The words are read again from shared memory for each pass (cheap)
// instead of being held in registers across both.
template <bool squares>
__device__ __forceinline__ float sum64(uint32_t kt, int t, int hh, float centre, __nv_bfloat162 &mn2,
                                       __nv_bfloat162 &mx2)
{
    // leaf pair i (i < 16) packs elements (2i, 32 + 2i) and (2i+1, 33 + 2i); leaves 4j..4j+3 come
    // from chunks j and j + 4 of the half-row and are reduced to node j at once.  The first
    // pass also takes the min/max of the K values (on packed bf16 pairs: exact).
    uint64_t node[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const uint4 qa = ld_shared_v4(kt + tile_off(t, hh * 8 + j));
        const uint4 qb = ld_shared_v4(kt + tile_off(t, hh * 8 + j + 4));
        const uint32_t wa[4] = {qa.x, qa.y, qa.z, qa.w};
        const uint32_t wb[4] = {qb.x, qb.y, qb.z, qb.w};
        uint64_t l[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            if (!squares) {
                const __nv_bfloat162 xa = *reinterpret_cast<const __nv_bfloat162 *>(wa + e);
                const __nv_bfloat162 xb = *reinterpret_cast<const __nv_bfloat162 *>(wb + e);
                mn2 = __hmin2(mn2, __hmin2(xa, xb));
                mx2 = __hmax2(mx2, __hmax2(xa, xb));
            }
            if (squares) {  // (x - mean)^2: mixed-precision difference, scalar squares, packed sum
                float da0, da1, db0, db1;
                bf2_sub(wa[e], centre, da0, da1);
                bf2_sub(wb[e], centre, db0, db1);
                l[e] = f2_add(f2_pack(f2u(__fmul_rn(da0, da0)), f2u(__fmul_rn(db0, db0))),
                              f2_pack(f2u(__fmul_rn(da1, da1)), f2u(__fmul_rn(db1, db1))));
            } else {  // x_2i + x_2i+1: the two halves of a word
                l[e] = f2_pack(f2u(bf2_sum(wa[e])), f2u(bf2_sum(wb[e])));
            }
        }
        node[j] = f2_add(f2_add(l[0], l[1]), f2_add(l[2], l[3]));
    }
    const uint64_t r = f2_add(f2_add(node[0], node[1]), f2_add(node[2], node[3]));
    uint32_t lo, hi;
    f2_unpack(r, lo, hi);
    return __fadd_rn(__uint_as_float(lo), __uint_as_float(hi));
}

__device__ __forceinline__ WinStats window_stats(uint32_t kt, uint32_t vt, int32_t cnt)
{
    const int lane = threadIdx.x & 31;
    const int t = lane >> 1, hh = lane & 1;
    const bool ok = t < cnt;  // rows past the request end hold other data: masked
    __nv_bfloat162 kmn2 = __float2bfloat162_rn(INFINITY), kmx2 = __float2bfloat162_rn(-INFINITY);
    __nv_bfloat162 vmn2 = kmn2, vmx2 = kmx2;
    float s = sum64<false>(kt, t, hh, 0, kmn2, kmx2);
    s = __fadd_rn(s, __shfl_xor_sync(0xffffffffu, s, 1));
    const float mean = __fmul_rn(s, 0.0078125f);  // exact /128
    float e = sum64<true>(kt, t, hh, mean, kmn2, kmx2);
    e = __fadd_rn(e, __shfl_xor_sync(0xffffffffu, e, 1));
#pragma unroll 2
    for (int j = 0; j < 8; ++j) {
        const uint4 r = ld_shared_v4(vt + tile_off(t, hh * 8 + j));
        const uint32_t vw[4] = {r.x, r.y, r.z, r.w};
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const __nv_bfloat162 vx = *reinterpret_cast<const __nv_bfloat162 *>(vw + q);
            vmn2 = __hmin2(vmn2, vx);
            vmx2 = __hmax2(vmx2, vx);
        }
    }
    float var = __fmul_rn(e, 0.0078125f);
    var = ok ? var : 0.0f;
    // window mean: balanced tree over the 16 tokens (lanes 2t and 2t + 1 hold the same value)
#pragma unroll
    for (int o = 2; o <= 16; o <<= 1) var = __fadd_rn(var, __shfl_xor_sync(0xffffffffu, var, o));
    WinStats res;
    res.mean = __fdiv_rn(var, (float)cnt);
    const float kn = ok ? fminf(__low2float(kmn2), __high2float(kmn2)) : INFINITY;
    const float kx = ok ? fmaxf(__low2float(kmx2), __high2float(kmx2)) : -INFINITY;
    const float vn = ok ? fminf(__low2float(vmn2), __high2float(vmn2)) : INFINITY;
    const float vx = ok ? fmaxf(__low2float(vmx2), __high2float(vmx2)) : -INFINITY;
    res.kmn = warp_min(kn);
    res.kmx = warp_max(kx);
    res.vmn = warp_min(vn);
    res.vmx = warp_max(vx);
    return res;
}

// ---- quantisation -----------------------------------------------------------------------

// Eight codes from eight bf16 values: rint((x - min) * inv).  The difference is the mixed
// bf16 - fp32 subtraction (one rounding), the product a packed fp32 pair (one rounding each).
// The rounding to an integer adds 1.5 * 2^23, which rounds u to an integer (round-to-nearest-
// even) and leaves it in the low mantissa bits: 0 <= u <= 255 * (1 + 2^-22) < 255.5 because
// x >= min, so the low byte is the code.  The add is written as the packed fused multiply-add
// u * 1 + 1.5 * 2^23, which is the rounded sum itself: measured on this GPU, a plain packed add
// whose operand comes from a packed product is contracted with it into one fused multiply-add
// by the assembler (one rounding instead of two: a different code whenever the rounded product
// is a tie), and a fused multiply-add by one is not.
__device__ __forceinline__ uint2 encode8(const uint4 &q, float mn, uint64_t inv2)
{
    const uint32_t wv[4] = {q.x, q.y, q.z, q.w};
    const uint64_t one2 = f2_pack(0x3F800000u, 0x3F800000u), mag2 = f2_pack(0x4B400000u, 0x4B400000u);
    uint32_t c[8];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
        float d0, d1;
        bf2_sub(wv[e], mn, d0, d1);
        f2_unpack(f2_fma(f2_mul(f2_pack(f2u(d0), f2u(d1)), inv2), one2, mag2), c[2 * e], c[2 * e + 1]);
    }
    const uint32_t lo = __byte_perm(__byte_perm(c[0], c[1], 0x0040), __byte_perm(c[2], c[3], 0x0040), 0x5410);
    const uint32_t hi = __byte_perm(__byte_perm(c[4], c[5], 0x0040), __byte_perm(c[6], c[7], 0x0040), 0x5410);
    return make_uint2(lo, hi);
}

// Quantisation parameters of one pair held by a warp: lane i < 5 holds segment i's
// (start, k_min, k_inv, v_min, v_inv).
struct PairCache {
    int32_t start;
    float kmn, kinv, vmn, vinv;
};

__device__ __forceinline__ PairCache load_params(const PairParams *pp)
{
    const int lane = threadIdx.x & 31;
    const int i = lane < kMaxSeg ? lane : 0;
    PairCache pc;
    pc.start = __ldcg(pp->start + i);
    pc.kmn = __ldcg(pp->k_min + i);
    pc.kinv = __ldcg(pp->k_inv + i);
    pc.vmn = __ldcg(pp->v_min + i);
    pc.vinv = __ldcg(pp->v_inv + i);
    return pc;
}

// Codes of one window tile, written straight to their slots in the physical block.
__device__ __forceinline__ void window_quant(uint8_t *kpool, uint8_t *vpool, int32_t Hkv, int32_t bs, int32_t h,
                                             int32_t t0, int32_t cnt, int32_t blk, uint32_t kt, uint32_t vt,
                                             const PairCache &pc)
{
    const int lane = threadIdx.x & 31;
    const int half = lane >> 4, sub = lane & 15;
    // segment of the window: how many of starts 1..4 (lanes 1..4) lie at or before t0
    const unsigned ballot = __ballot_sync(0xffffffffu, lane >= 1 && lane < kMaxSeg && pc.start <= t0);
    const int s = __popc(ballot);
    const float kmn = __shfl_sync(0xffffffffu, pc.kmn, s), kinv = __shfl_sync(0xffffffffu, pc.kinv, s);
    const float vmn = __shfl_sync(0xffffffffu, pc.vmn, s), vinv = __shfl_sync(0xffffffffu, pc.vinv, s);
    const int64_t dst0 = (((int64_t)blk * Hkv + h) * bs + pow2_mod(t0, bs)) * kD + sub * 8;
    const uint64_t kinv2 = f2_pack(__float_as_uint(kinv), __float_as_uint(kinv));
    const uint64_t vinv2 = f2_pack(__float_as_uint(vinv), __float_as_uint(vinv));
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const int tt = 2 * i + half;
        if (tt < cnt) {
            const uint4 kq = ld_shared_v4(kt + tile_off(tt, sub));
            const uint4 vq = ld_shared_v4(vt + tile_off(tt, sub));
            __stcs(reinterpret_cast<uint2 *>(kpool + dst0 + tt * kD), encode8(kq, kmn, kinv2));
            __stcs(reinterpret_cast<uint2 *>(vpool + dst0 + tt * kD), encode8(vq, vmn, vinv2));
        }
    }
}

// ---- segment parameters ------------------------------------------------------------------

// Record and quantiser parameters of a pair from its segment starts (pair-local windows, `cut`,
// ascending, k of them) and the per-segment fp32 extremes.
__device__ __forceinline__ void make_params(int32_t L, int k, const int32_t (&cut)[4], const float (&kmn)[kMaxSeg],
                                            const float (&kmx)[kMaxSeg], const float (&vmn)[kMaxSeg],
                                            const float (&vmx)[kMaxSeg], dgq_seg_record &rec, PairParams &pp)
{
    const int32_t n = k + 1;
#pragma unroll
    for (int i = 0; i < kMaxSeg; ++i) {
        rec.start[i] = i == 0 ? 0 : (i <= k ? kWin * cut[i - 1] : L);
        pp.start[i] = rec.start[i];
        if (i < n) {
            const float kn = canon_zero(kmn[i]), kx = canon_zero(kmx[i]);
            const float vn = canon_zero(vmn[i]), vx = canon_zero(vmx[i]);
            const float kr = __fsub_rn(kx, kn), vr = __fsub_rn(vx, vn);
            rec.k_min[i] = kn;
            rec.v_min[i] = vn;
            rec.k_scale[i] = kr == 0.0f ? 0.0f : __fdiv_rn(kr, 255.0f);
            rec.v_scale[i] = vr == 0.0f ? 0.0f : __fdiv_rn(vr, 255.0f);
            pp.k_min[i] = kn;
            pp.v_min[i] = vn;
            pp.k_inv[i] = kr == 0.0f ? 0.0f : __fdiv_rn(255.0f, kr);
            pp.v_inv[i] = vr == 0.0f ? 0.0f : __fdiv_rn(255.0f, vr);
        } else {
            rec.k_min[i] = rec.k_scale[i] = rec.v_min[i] = rec.v_scale[i] = 0.0f;
            pp.k_min[i] = pp.k_inv[i] = pp.v_min[i] = pp.v_inv[i] = 0.0f;
        }
    }
    rec.n_seg = n;
    rec.seq_len = L;
    rec.k_inv_last = rec.v_inv_last = 0.0f;  // the encoder's factors of segment n - 1 = k
#pragma unroll
    for (int i = 0; i < kMaxSeg; ++i) {
        if (i == k) {
            rec.k_inv_last = pp.k_inv[i];
            rec.v_inv_last = pp.v_inv[i];
        }
    }
    rec.pad[0] = rec.pad[1] = rec.pad[2] = 0;
    pp.n_seg = n;
#pragma unroll
    for (int i = 0; i < 6; ++i) pp.pad[i] = 0;
}

// Segmentation of a pair of at most 256 windows held by one warp, lane i owning windows
// 8i .. 8i+7 (means m[], extremes mm[] as K min, K max, V min, V max; unused slots hold the
// identities).  At most k boundaries; a jump between two windows whose means are both below
// min_var is no candidate.  Returns the number of boundaries placed and fills the segment
// starts and the per-segment extremes, identical in every lane.
__device__ __forceinline__ int segment_small(int32_t W, int k, float min_var, const float (&m)[8],
                                             const float4 (&mm)[8], int32_t (&cut)[4], float (&kmn)[kMaxSeg],
                                             float (&kmx)[kMaxSeg], float (&vmn)[kMaxSeg], float (&vmx)[kMaxSeg])
{
    const int lane = threadIdx.x & 31;
    // per-lane top-k of (jump desc, window asc); the jump of window w < W-1 is |m[w+1] - m[w]|
    float cj[4] = {-1.0f, -1.0f, -1.0f, -1.0f};
    int32_t cw[4] = {INT32_MAX, INT32_MAX, INT32_MAX, INT32_MAX};
    const float mnext = __shfl_down_sync(0xffffffffu, m[0], 1);  // first mean of the next lane
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const int32_t w = 8 * lane + i;
        if (k == 0 || w + 1 >= W) continue;
        const float mn1 = i < 7 ? m[i + 1] : mnext;
        if (!(m[i] >= min_var || mn1 >= min_var)) continue;  // two quiet windows stay together
        const float j = fabsf(__fsub_rn(mn1, m[i]));
        // a lane meets its windows in increasing order: an equal jump keeps the earlier window first
        if (j > cj[3]) {
            cj[3] = j;
            cw[3] = w;
#pragma unroll
            for (int s = 3; s > 0; --s) {
                if (cj[s] > cj[s - 1]) {
                    const float tj = cj[s]; cj[s] = cj[s - 1]; cj[s - 1] = tj;
                    const int32_t tw = cw[s]; cw[s] = cw[s - 1]; cw[s - 1] = tw;
                }
            }
        }
    }
    // k rounds of warp arg-best; the winning lane pops its head
#pragma unroll
    for (int s = 0; s < 4; ++s) cut[s] = INT32_MAX;
    for (int r = 0; r < k; ++r) {
        const float bj = cj[0];
        const int32_t bw = cw[0];
        float j = bj;
        int32_t wv = bw;
#pragma unroll
        for (int o = 16; o; o >>= 1) {
            const float oj = __shfl_xor_sync(0xffffffffu, j, o);
            const int32_t ow = __shfl_xor_sync(0xffffffffu, wv, o);
            if (oj > j || (oj == j && ow < wv)) {
                j = oj;
                wv = ow;
            }
        }
        if (j < 0.0f) {  // no candidate left (same in every lane)
            k = r;
            break;
        }
        if (bw == wv) {  // a window sits in one lane only
            cj[0] = cj[1]; cj[1] = cj[2]; cj[2] = cj[3]; cj[3] = -1.0f;
            cw[0] = cw[1]; cw[1] = cw[2]; cw[2] = cw[3]; cw[3] = INT32_MAX;
        }
        int32_t c = wv + 1;  // insertion into the sorted list of starts
#pragma unroll
        for (int s = 0; s < 4; ++s) {
            if (c < cut[s]) {
                const int32_t t = cut[s];
                cut[s] = c;
                c = t;
            }
        }
    }
#pragma unroll
    for (int s = 0; s < kMaxSeg; ++s) {
        kmn[s] = INFINITY; kmx[s] = -INFINITY; vmn[s] = INFINITY; vmx[s] = -INFINITY;
    }
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const int32_t w = 8 * lane + i;
        if (w >= W) continue;
        const int sg = (w >= cut[0]) + (w >= cut[1]) + (w >= cut[2]) + (w >= cut[3]);
#pragma unroll
        for (int s = 0; s < kMaxSeg; ++s) {
            if (s == sg) {
                kmn[s] = fminf(kmn[s], mm[i].x); kmx[s] = fmaxf(kmx[s], mm[i].y);
                vmn[s] = fminf(vmn[s], mm[i].z); vmx[s] = fmaxf(vmx[s], mm[i].w);
            }
        }
    }
#pragma unroll
    for (int s = 0; s < kMaxSeg; ++s) {
        kmn[s] = warp_min(kmn[s]); kmx[s] = warp_max(kmx[s]);
        vmn[s] = warp_min(vmn[s]); vmx[s] = warp_max(vmx[s]);
    }
    return k;
}

}  // namespace dgq
