// dgq_attn.cu -- decode-step GQA attention over the DGQ INT8 paged cache (sm_103a).
//
// Method: scores q . x_K / sqrt(D) over the cached tokens, whose keys/values are
// dequantised per segment (x = min + q * scale, segment looked up per token: "DeepSeek
// KV-cache dynamic group quantisation (DGQ)" article, section 2.2; dequantisation on the
// GPU: section 3.2), gathered through the block table ("PagedAttention implementation",
// DeepSeek-V4 KV-cache article), plus the current token's own bf16 key/value.
//
// GPU design.
//  * Work: every (request, KV head) pair is cut into 16-token tiles (a tile never crosses a
//    block, since block sizes are multiples of 16, nor a segment, since segment starts are);
//    all tiles of all pairs form one flat list and each persistent CTA takes a contiguous
//    slice of it, so mixed lengths and a single long request balance alike.  The slices are
//    equal in cost, a pair costing its tiles plus a fixed charge for the end of a piece
//    (measured on this GPU: with slices equal in tiles, CTAs over many short pairs ran up to
//    16% longer than the mean and set the kernel's time).  The four warps of a CTA take every
//    fourth tile of the slice and combine their softmax states in shared memory wherever the
//    slice crosses from one pair to the next.  A CTA's part of a pair is a "piece".  A pair
//    inside one CTA is finished there; the pieces of a pair shared by several CTAs go to a
//    small combine kernel chained with programmatic dependent launch, which folds them in a
//    fixed order (bitwise reproducible on a given GPU) with the current token.
//    The next pieces' record, query rows and current key/value are staged in shared memory by
//    bulk copies while the current piece streams, so a piece boundary waits on no global load.
//  * Loads: each warp copies its tiles' K and V rows with cp.async (whole 128-byte rows, four
//    rows per instruction) into its own shared-memory ring, three tiles deep, with the 16-byte
//    columns of row i XOR-permuted by i % 8 so the fragment reads hit distinct banks.  Measured
//    on this GPU: three CTAs per SM at depth 3 stream faster than two at depth 4 to 6; the
//    per-copy issue cost of TMA caps single-tile copies of 2 KB blocks at 2-4 TB/s, while
//    per-thread 16-byte copies stream at the HBM rate.  Block ids come 32 tiles ahead from one
//    coalesced load per warp.
//  * Math: codes become fp16 (1024 + q) with byte permutes, and the GQA query group multiplies
//    them on the tensor cores (mma.sync m16n8k16, fp32 accumulate): S^T = Q . K^T and
//    O^T += V^T . P^T.  The affine dequantisation is folded out of the inner loop: for a tile
//    inside segment s,
//      q . x_K = k_scale[s] * (q . (1024 + c)) + (k_min[s] - 1024 k_scale[s]) * sum(q),
//      sum_t p_t x_V = v_scale[s] * sum_t p_t (1024 + c_t) + (v_min[s] - 1024 v_scale[s]) sum p.
//  * Online softmax in the log2 domain with lazy rescaling (the running max moves only when a
//    tile's max exceeds it by more than 8, so p <= 256 stays exact enough in fp16).
//  * The comparison encodings run through the same kernel, instantiated per code format: the
//    symmetric INT8 cache is a one-segment affine cache (the path above); FP8 E4M3 codes are
//    converted to fp16 exactly (E4M3 values are fp16 values); fixed 64-value groups are
//    dequantised to fp16 in registers, code * scale + min per (token, half row), from per-token
//    parameters copied into the ring beside each tile.  Both of the latter feed the tensor
//    cores the decoded values themselves, so their per-tile fold is the identity.
#include "dgq_device.cuh"
#include "dgq.h"
#include "dgq_launch.h"

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>
#include <stdint.h>

namespace dgq {

constexpr int kTile = 16;                          // tokens per tile
constexpr int kWarpsPerCta = 4;
constexpr int kAttnThreads = kWarpsPerCta * 32;
constexpr int kMaxCtasPerSm = 3;
constexpr int kDepth = 3;                          // tiles in flight per warp (3 CTAs of 4 warps fit per SM)
constexpr int kTileBytes = kTile * kD;            // 16 rows of 128 codes = 2 KB
constexpr int kTileSmem = 2 * kTileBytes;          // K tile + V tile
constexpr int kParBytes = kTile * 16;              // fixed groups: a tile's (min0, scale0, min1, scale1) per token

// Code formats of the decode kernel's instances.
enum : int { kDecAffine = 0, kDecFp8 = 1, kDecFixed = 2, kDecSplitV = 3 };

// Bytes of one ring stage: the K and V tiles, and for fixed groups their K and V parameters.
template <int Fmt>
__host__ __device__ constexpr int stage_bytes() { return kTileSmem + (Fmt == kDecFixed ? 2 * kParBytes : 0); }
constexpr int kPartStride = 132;                   // floats per (piece, head) partial: m, l, pad, pad, O[128]
constexpr int32_t kMaxGroup = 8;                   // largest query-head group the entry points accept
constexpr float kLog2eOverSqrtD = 0.12751743074570180f;  // log2(e) / sqrt(128)
constexpr float kLazyRescale = 8.0f;               // log2 units
constexpr int32_t kPieceCost = 10;                 // tile times a piece's end costs a CTA (measured)

struct AttnArgs {
    const uint16_t *q;
    const uint16_t *knew;
    const uint16_t *vnew;
    const uint8_t *kpool;
    const uint8_t *vpool;
    const dgq_seg_record *table;
    const dgq_seg_record *vtable;  // independent V segmentation: V's records (K's are in `table`)
    const float4 *kpar;  // fixed groups: per-slot (min0, scale0, min1, scale1) of K and of V
    const float4 *vpar;
    const int32_t *bt;
    const int32_t *seq_lens;
    uint16_t *out;
    WsHeader *hdr;
    int2 *pair_info;  // per pair: first and last CTA holding a piece of it
    int32_t *held;    // per CTA of the main kernel: 1 when its slice holds tiles
    float *part;
    int32_t B, Hq, Hkv, G, bs, max_blocks, num_blocks;
};

// Token order inside each 8-column n-tile: column n holds token tau(n).  With it, the K row a
// lane supplies to S^T and the V rows it supplies to O^T cover the tokens whose scores it holds.
__device__ __forceinline__ int tau(int n) { return (n >> 1) + ((n & 1) << 2); }

__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) { return __byte_perm(a, b, sel); }

__device__ __forceinline__ uint32_t bf16x2_to_f16x2(uint32_t w)
{
    __half2 h = __floats2half2_rn(bf16lo_to_f32(w), bf16hi_to_f32(w));
    return *reinterpret_cast<uint32_t *>(&h);
}

__device__ __forceinline__ uint32_t f32x2_to_f16x2(float lo, float hi)
{
    __half2 h = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&h);
}

__device__ __forceinline__ float f16lo(uint32_t w) { return __low2float(*reinterpret_cast<const __half2 *>(&w)); }
__device__ __forceinline__ float f16hi(uint32_t w) { return __high2float(*reinterpret_cast<const __half2 *>(&w)); }

__device__ __forceinline__ void mma16816(float *c, uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3, uint32_t b0,
                                         uint32_t b1)
{
    asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t word(const uint4 &v, int i)
{
    return i == 0 ? v.x : (i == 1 ? v.y : (i == 2 ? v.z : v.w));
}

// Two codes as the fp16 pair the tensor cores take, from bytes 0-1 (Hi = false) or 2-3 of w:
// 1024 + code for the affine formats (the offset is folded out per tile); the E4M3 values
// themselves; for fixed groups code * scale + min (per-lane scale and min pairs sc2, mn2; the
// code is recovered exactly as (1024 + code) - 1024, then one rounded fp16 multiply-add).
template <int Fmt, bool Hi>
__device__ __forceinline__ uint32_t codes2(uint32_t w, uint32_t sc2, uint32_t mn2)
{
    if constexpr (Fmt == kDecFp8) {
        const __half2_raw h = __nv_cvt_fp8x2_to_halfraw2((__nv_fp8x2_storage_t)(Hi ? (w >> 16) : (w & 0xFFFFu)),
                                                         __NV_E4M3);
        return (uint32_t)h.x | ((uint32_t)h.y << 16);
    } else {
        const uint32_t x = prmt(w, 0x64646464u, Hi ? 0x4342 : 0x4140);
        if constexpr (Fmt == kDecFixed) {
            const __half2 c = __hsub2(*reinterpret_cast<const __half2 *>(&x), __half2(__half_raw{0x6400}, __half_raw{0x6400}));
            const __half2 y = __hfma2(c, *reinterpret_cast<const __half2 *>(&sc2), *reinterpret_cast<const __half2 *>(&mn2));
            return *reinterpret_cast<const uint32_t *>(&y);
        } else {
            (void)sc2;
            (void)mn2;
            return x;
        }
    }
}

// 8-byte shared-memory load by 32-bit shared address (volatile: stays after the copy wait)
__device__ __forceinline__ uint2 ld_shared_v2(uint32_t addr)
{
    uint2 v;
    asm volatile("ld.shared.v2.u32 {%0, %1}, [%2];" : "=r"(v.x), "=r"(v.y) : "r"(addr));
    return v;
}

__device__ __forceinline__ uint32_t half2_bits(float lo, float hi)
{
    const __half2 h = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<const uint32_t *>(&h);
}

// 2^x on the MUFU unit (flush-to-zero); arguments here are <= 8 or -inf.
__device__ __forceinline__ float ex2(float x)
{
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

__device__ __forceinline__ void cp_async16(uint32_t dst, const void *src)
{
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }

// ---- the flat tile list ---------------------------------------------------------------------

struct TileLoc {
    int32_t b, h, j, ntl, L;  // request, head, tile within the pair, tiles in the pair, length
};

__device__ __forceinline__ int32_t tiles_of(int32_t L) { return max(1, (L + kTile - 1) / kTile); }

__device__ __forceinline__ TileLoc locate_tile(int32_t x, const int32_t *s_tpre, const int32_t *s_len, int32_t B)
{
    int32_t lo = 0, hi = B - 1;
    while (lo < hi) {
        const int32_t mid = (lo + hi + 1) >> 1;
        if (s_tpre[mid] <= x) lo = mid;
        else hi = mid - 1;
    }
    TileLoc c;
    c.b = lo;
    c.L = s_len[lo];
    c.ntl = tiles_of(c.L);
    const int32_t off = x - s_tpre[lo];
    c.h = off / c.ntl;
    c.j = off - c.h * c.ntl;
    return c;
}

__device__ __forceinline__ void advance(TileLoc &c, const int32_t *s_len, int32_t Hkv)
{
    if (++c.j == c.ntl) {
        c.j = 0;
        if (++c.h == Hkv) {
            c.h = 0;
            ++c.b;
            c.L = s_len[c.b];
            c.ntl = tiles_of(c.L);
        }
    }
}

// The CTAs split the flat tile list evenly by cost, not by tiles: each pair costs its tiles plus
// kPieceCost, what the end of a piece (the warps' wait for the piece's last tile, the merge, the
// staging of the next piece) takes in tile times of a CTA.  Pair p's tiles sit at cost positions
// x + kPieceCost (p + 1) (x its flat tile index) and CTA c of n takes the tiles whose positions
// fall in [C c / n, C (c + 1) / n), C = T + kPieceCost * pairs.

// Tiles whose cost position is below q (q in [0, C]); s_tpre: tile prefix over requests [B + 1].
__device__ __forceinline__ int32_t tile_at(int64_t q, const int32_t *s_tpre, const int32_t *s_len, int32_t B,
                                           int32_t Hkv)
{
    const int64_t kh = (int64_t)kPieceCost * Hkv;
    int32_t lo = 0, hi = B;  // the last request whose cost range starts at or below q (B: the end)
    while (lo < hi) {
        const int32_t mid = (lo + hi + 1) >> 1;
        if (s_tpre[mid] + kh * mid <= q) lo = mid;
        else hi = mid - 1;
    }
    if (lo == B) return s_tpre[B];
    const int32_t ntl = tiles_of(s_len[lo]);
    const int32_t r = (int32_t)(q - (s_tpre[lo] + kh * lo));  // < Hkv * (ntl + kPieceCost)
    const int32_t u = ntl + kPieceCost;
    const int32_t h = r / u;
    const int32_t j = r - h * u - kPieceCost;  // < ntl
    return s_tpre[lo] + h * ntl + max(0, j);
}

// Workspace header word: 1 when every CTA of the main kernel holds tiles.  That is so when each
// CTA's cost range is longer than kPieceCost: runs of positions without a tile are at most
// kPieceCost long.
constexpr int kHdrAllHeld = 0;

// CTA holding flat tile x of pair p
__device__ __forceinline__ int32_t owner(int32_t x, int32_t p, int64_t C, int32_t n)
{
    const int64_t pos = (int64_t)x + (int64_t)kPieceCost * (p + 1);
    return (int32_t)(((pos + 1) * n - 1) / C);
}

// Final softmax merge with the current token: (O + p_new v_new) / (L + p_new), where (M, L, O)
// are the cached tokens' max, sum and weighted value sum relative to M (log2 domain).
__device__ __forceinline__ float finish(float M, float L, float O, float s_new, float v_new)
{
    const float Mf = fmaxf(M, s_new);
    const float wo = (M == -INFINITY) ? 0.0f : ex2(M - Mf);
    const float wn = ex2(s_new - Mf);
    return fmaf(O, wo, wn * v_new) / fmaf(L, wo, wn);
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi)
{
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&v);
}

// q . k_new over 128 dims for one query head (every lane gets the sum), log2 domain
__device__ __forceinline__ float score_new(const uint16_t *qrow, const uint16_t *krow, int lane)
{
    const uint2 qv = __ldg(reinterpret_cast<const uint2 *>(qrow) + lane);
    const uint2 kv = __ldg(reinterpret_cast<const uint2 *>(krow) + lane);
    float acc = bf16lo_to_f32(qv.x) * bf16lo_to_f32(kv.x);
    acc = fmaf(bf16hi_to_f32(qv.x), bf16hi_to_f32(kv.x), acc);
    acc = fmaf(bf16lo_to_f32(qv.y), bf16lo_to_f32(kv.y), acc);
    acc = fmaf(bf16hi_to_f32(qv.y), bf16hi_to_f32(kv.y), acc);
#pragma unroll
    for (int o = 16; o; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
    return acc * kLog2eOverSqrtD;
}

// One pair's slice of this CTA: request b, KV head h, its tiles in the flat list start at fp.
struct Piece {
    int32_t b, h, ntl, L, fp;
};

__device__ __forceinline__ void next_piece(Piece &pz, const int32_t *s_tpre, const int32_t *s_len, int32_t B,
                                           int32_t Hkv)
{
    if (++pz.h == Hkv) {
        pz.h = 0;
        if (++pz.b >= B) {
            pz.fp = INT32_MAX;
            return;
        }
        pz.L = s_len[pz.b];
        pz.ntl = tiles_of(pz.L);
    }
    pz.fp = s_tpre[pz.b] + pz.h * pz.ntl;
}

// Per-piece data staged in shared memory ahead of use: the segment record, the current token's
// key and value and the group's query rows.
constexpr int kPbRec = 0, kPbKnew = 128, kPbVnew = 384, kPbQ = 640, kPbRecV = kPbQ + 8 * 256;

// Bytes of one piece's staging buffer (plus V's own record with independent V segmentation).
template <int Fmt>
__host__ __device__ constexpr int piece_bytes() { return kPbRecV + (Fmt == kDecSplitV ? 128 : 0); }


template <int Fmt>
__global__ void __launch_bounds__(kAttnThreads, kMaxCtasPerSm) attn_kernel(AttnArgs a)
{
    constexpr int kStage = stage_bytes<Fmt>();
    constexpr int kWarpSmem = kDepth * kStage;
    constexpr int kPieceBytes = piece_bytes<Fmt>();
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = align_smem_1024(smem_raw);
    uint8_t *pbuf = smem + kWarpsPerCta * kWarpSmem;                                 // [2][kPieceBytes]
    uint64_t *pbar = reinterpret_cast<uint64_t *>(pbuf + 2 * kPieceBytes);          // [2]
    float *s_comb = reinterpret_cast<float *>(pbar + 2);                           // [4][G][132]
    float *s_snew = s_comb + kWarpsPerCta * a.G * kPartStride;                       // [8]
    int32_t *s_tpre = reinterpret_cast<int32_t *>(s_snew + 8);                       // [B+1]
    int32_t *s_len = s_tpre + a.B + 1;                                               // [B]
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int32_t B = a.B, Hkv = a.Hkv, G = a.G;

    pdl_launch_dependents();  // the combine kernel may be scheduled while this one runs
    if (tid == 0) {
        mbar_init(&pbar[0], 1);
        mbar_init(&pbar[1], 1);
        fence_barrier_init();
    }
    for (int i = tid; i < B; i += kAttnThreads) {
        int32_t L = __ldg(a.seq_lens + i);
        if (L < 0 || L > a.max_blocks * a.bs) {  // beyond the block table's row: flagged, clamped
            record_error(a.hdr, kErrBadLength);
            L = L < 0 ? 0 : a.max_blocks * a.bs;
        }
        s_len[i] = L;
    }
    __syncthreads();
    if (warp == 0) {  // exclusive scan of Hkv * tiles_of(L_b)
        int32_t carry = 0;
        for (int base = 0; base < B; base += 32) {
            const int i = base + lane;
            const int32_t v = i < B ? Hkv * tiles_of(s_len[i]) : 0;
            int32_t x = v;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int32_t y = __shfl_up_sync(0xffffffffu, x, o);
                if (lane >= o) x += y;
            }
            if (i < B) s_tpre[i] = carry + x - v;
            carry += __shfl_sync(0xffffffffu, x, 31);
        }
        if (lane == 0) s_tpre[B] = carry;
    }
    __syncthreads();

    const int32_t T = s_tpre[B];
    const int64_t C = (int64_t)T + (int64_t)kPieceCost * B * Hkv;  // total cost
    const int32_t ncta = gridDim.x, cta = blockIdx.x;
    const int32_t c0 = tile_at(C * cta / ncta, s_tpre, s_len, B, Hkv);
    const int32_t c1 = tile_at(C * (cta + 1) / ncta, s_tpre, s_len, B, Hkv);
    if (tid == 0) a.held[cta] = c0 < c1 ? 1 : 0;  // read by the merge kernels
    if (cta == 0 && tid == 0) a.hdr->pad[kHdrAllHeld] = C / ncta > kPieceCost ? 1u : 0u;
    if (c0 >= c1) return;  // the whole CTA: no barrier follows for it

    const int r = lane >> 2, cq = lane & 3;
    const int tr = tau(r);
    const bool gvalid = r < G;  // this lane's softmax head (rows of S^T)
    const uint32_t ring = smem_u32(smem) + warp * kWarpSmem;
    const int per_blk = a.bs / kTile;  // tiles per block
    const uint32_t nthr = kAttnThreads;

    // ---- pieces of this CTA's slice, and the staging of their data two pieces ahead
    Piece cur;
    {
        const TileLoc c = locate_tile(c0, s_tpre, s_len, B);
        cur.b = c.b; cur.h = c.h; cur.ntl = c.ntl; cur.L = c.L;
        cur.fp = s_tpre[c.b] + c.h * c.ntl;
    }
    auto stage_piece = [&](const Piece &pz, int buf) {  // thread 0 only
        uint8_t *dst = pbuf + buf * kPieceBytes;
        mbar_arrive_expect_tx(&pbar[buf], (uint32_t)(kPbQ + 256 * G + (Fmt == kDecSplitV ? 128 : 0)));
        bulk_load(dst + kPbRec, a.table + (int64_t)pz.b * Hkv + pz.h, 128, &pbar[buf]);
        if constexpr (Fmt == kDecSplitV) bulk_load(dst + kPbRecV, a.vtable + (int64_t)pz.b * Hkv + pz.h, 128, &pbar[buf]);
        bulk_load(dst + kPbKnew, a.knew + ((int64_t)pz.b * Hkv + pz.h) * kD, 256, &pbar[buf]);
        bulk_load(dst + kPbVnew, a.vnew + ((int64_t)pz.b * Hkv + pz.h) * kD, 256, &pbar[buf]);
        bulk_load(dst + kPbQ, a.q + ((int64_t)pz.b * a.Hq + pz.h * G) * kD, (uint32_t)(256 * G), &pbar[buf]);
    };
    Piece ahead = cur;  // the next piece to stage
    if (tid == 0) {
        stage_piece(ahead, 0);
        next_piece(ahead, s_tpre, s_len, B, Hkv);
        if (ahead.fp < c1) stage_piece(ahead, 1);
    } else {
        next_piece(ahead, s_tpre, s_len, B, Hkv);
    }
    next_piece(ahead, s_tpre, s_len, B, Hkv);  // ahead = piece 2

    // This warp's tiles: x = xw0 + 4k, k = 0 .. nmine-1, inside the CTA's slice [c0, c1).
    const int32_t xw0 = c0 + warp;
    const int32_t nmine = c1 > xw0 ? (c1 - xw0 + kWarpsPerCta - 1) / kWarpsPerCta : 0;

    // ---- block ids, 32 tiles ahead: lane l of a batch holds the block of this warp's tile kbase + l
    auto fetch_batch = [&](int32_t kbase) -> int32_t {
        const int32_t k = kbase + lane;
        int32_t blk = 0;
        if (k < nmine) {
            const TileLoc c = locate_tile(xw0 + kWarpsPerCta * k, s_tpre, s_len, B);
            if (c.L > 0) blk = __ldg(a.bt + (int64_t)c.b * a.max_blocks + pow2_div(c.j, per_blk));
            if ((uint32_t)blk >= (uint32_t)a.num_blocks) {  // not a block of the pools: flagged,
                record_error(a.hdr, kErrBadBlock);          // and block 0 read instead
                blk = 0;
            }
        }
        return blk;
    };
    int32_t kb = 0;
    int32_t bq_cur = fetch_batch(0), bq_next = fetch_batch(32);

    // ---- copies of one tile into ring stage `st`; the issue point runs kDepth tiles ahead of the
    // compute point and always lies in the two fetched batches
    TileLoc ic;
    if (nmine > 0) ic = locate_tile(xw0, s_tpre, s_len, B);
    int32_t kn = 0;  // next of this warp's tiles to issue
    auto issue = [&](int st) {
        if (kn - kb >= 32) {
            kb += 32;
            bq_cur = bq_next;
            bq_next = fetch_batch(kb + 32);
        }
        const int32_t blk = __shfl_sync(0xffffffffu, bq_cur, (kn - kb) & 31);
        if (kn < nmine && ic.L > 0) {
            const int64_t row0 = ((int64_t)blk * Hkv + ic.h) * a.bs + pow2_mod(ic.j, per_blk) * kTile;
            const uint8_t *kp = a.kpool + row0 * kD;
            const uint8_t *vp = a.vpool + row0 * kD;
            // whole 128-byte rows: lane l copies 16-byte column l % 8 of rows 4i + l / 8, stored
            // at column (l % 8) ^ (row % 8) so the fragment reads below hit 8 distinct columns
            const uint32_t dst = ring + st * kStage;
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int row = 4 * i + (lane >> 3), col = lane & 7;
                const uint32_t off = row * kD + ((col ^ (row & 7)) << 4);
                cp_async16(dst + off, kp + row * kD + col * 16);
                cp_async16(dst + kTileBytes + off, vp + row * kD + col * 16);
            }
            if constexpr (Fmt == kDecFixed) {  // lanes 0-15: K parameters of token lane; 16-31: V
                const float4 *src = (lane < 16 ? a.kpar : a.vpar) + row0 + (lane & 15);
                cp_async16(dst + kTileSmem + lane * 16, src);
            }
        }
        cp_async_commit();
        if (kn < nmine) {
            if (kn + 1 < nmine)
                for (int i = 0; i < kWarpsPerCta; ++i) advance(ic, s_len, Hkv);
            ++kn;
        }
    };
#pragma unroll
    for (int k = 0; k < kDepth; ++k) issue(k);

    uint32_t qa0[8], qa2[8];
    float o[8][4];
    int32_t kc = 0;  // next of this warp's tiles to compute

    for (int32_t n = 0; cur.fp < c1; ++n) {
        const int buf = n & 1;
        const int32_t p = cur.b * Hkv + cur.h;
        const int32_t pe = min(cur.fp + cur.ntl, c1);  // end of this piece
        const uint8_t *pb = pbuf + buf * kPieceBytes;
        if (!mbar_wait_bounded(&pbar[buf], (uint32_t)(n >> 1) & 1u)) record_error(a.hdr, kErrFullWait);

        // piece start (per warp): record word, Q fragments of head g = r, state
        const uint32_t recw = reinterpret_cast<const uint32_t *>(pb + kPbRec)[lane];
        const uint32_t recw_v = Fmt == kDecSplitV ? reinterpret_cast<const uint32_t *>(pb + kPbRecV)[lane] : 0u;
        float qsum;
        {
            float qs = 0.0f;
            if (gvalid) {  // columns d = 16cq + 64(jj/4) + 4(jj%4) + {0,1 | 2,3}
                const uint32_t qrow = smem_u32(pb + kPbQ) + r * 256;
#pragma unroll
                for (int half = 0; half < 2; ++half) {
                    const uint4 u0 = ld_shared_v4(qrow + 32 * cq + 128 * half);
                    const uint4 u1 = ld_shared_v4(qrow + 32 * cq + 128 * half + 16);
                    const uint32_t wv[8] = {u0.x, u0.y, u0.z, u0.w, u1.x, u1.y, u1.z, u1.w};
#pragma unroll
                    for (int m = 0; m < 4; ++m) {
                        const uint32_t h0 = bf16x2_to_f16x2(wv[2 * m]), h1 = bf16x2_to_f16x2(wv[2 * m + 1]);
                        qa0[4 * half + m] = h0;
                        qa2[4 * half + m] = h1;
                        qs += (f16lo(h0) + f16hi(h0)) + (f16lo(h1) + f16hi(h1));
                    }
                }
            } else {
#pragma unroll
                for (int jj = 0; jj < 8; ++jj) qa0[jj] = qa2[jj] = 0u;
            }
            qs += __shfl_xor_sync(0xffffffffu, qs, 1);
            qs += __shfl_xor_sync(0xffffffffu, qs, 2);
            qsum = qs;
        }
        int seg = -1, vseg = -1;
        float ak = 0.f, bk = 0.f, cv = 0.f;
        bool vflat = false;
        float m_run = -INFINITY, l_run = 0.f, bsum = 0.f, sigma = 1.0f;
#pragma unroll
        for (int i = 0; i < 8; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.0f;

        // this warp's tiles of the piece
        for (; kc < nmine && xw0 + kWarpsPerCta * kc < pe; ++kc) {
            const int32_t j = xw0 + kWarpsPerCta * kc - cur.fp;  // tile within the pair
            const int st = kc % kDepth;
            cp_async_wait<kDepth - 1>();  // this lane's copies of the tile have landed ...
            __syncwarp();                  // ... and, after the warp meets, every lane's
            const int32_t tok0 = j * kTile;
            const int32_t valid = min(kTile, cur.L - tok0);
            if (valid > 0) {
                // segment constants (record words: start 2..6, k_min 7.., k_scale 12.., v_min 17.., v_scale 22..)
                // (independent V segmentation: K's segment sgk from `recw`, V's sgv from `recw_v`)
                int sgk = 0, sgv = 0, sg = 0;
                if constexpr (Fmt == kDecAffine) {
                    sg = __popc(__ballot_sync(0xffffffffu, lane >= 3 && lane <= 6 && (int32_t)recw <= tok0));
                    sgk = sgv = sg;
                } else if constexpr (Fmt == kDecSplitV) {
                    sgk = __popc(__ballot_sync(0xffffffffu, lane >= 3 && lane <= 6 && (int32_t)recw <= tok0));
                    sgv = __popc(__ballot_sync(0xffffffffu, lane >= 3 && lane <= 6 && (int32_t)recw_v <= tok0));
                    sg = sgk * 8 + sgv;
                }
                if ((Fmt == kDecFp8 || Fmt == kDecFixed) && sg != seg) {  // decoded values: identity fold
                    seg = sg;
                    vflat = false;
                    ak = kLog2eOverSqrtD;
                    bk = 0.0f;
                    cv = 0.0f;
                } else if (sg != seg) {
                    seg = sg;
                    const uint32_t vw = Fmt == kDecSplitV ? recw_v : recw;
                    const float kmin = __uint_as_float(__shfl_sync(0xffffffffu, recw, 7 + sgk));
                    const float kscale = __uint_as_float(__shfl_sync(0xffffffffu, recw, 12 + sgk));
                    const float vmin = __uint_as_float(__shfl_sync(0xffffffffu, vw, 17 + sgv));
                    const float vsc = __uint_as_float(__shfl_sync(0xffffffffu, vw, 22 + sgv));
                    // a flat V segment (scale 0) decodes to v_min whatever its codes: it only feeds bsum
                    vflat = !(vsc > 0.0f);
                    ak = kscale * kLog2eOverSqrtD;
                    bk = (kmin - 1024.0f * kscale) * qsum * kLog2eOverSqrtD;
                    cv = vflat ? vmin : vmin - 1024.0f * vsc;
                    if (!vflat && sgv != vseg) {
                        if (vseg >= 0) {  // keep sigma * o invariant across the change of V scale
                            const float ratio = sigma / vsc;
#pragma unroll
                            for (int i = 0; i < 8; ++i)
#pragma unroll
                                for (int e = 0; e < 4; ++e) o[i][e] *= ratio;
                        }
                        sigma = vsc;
                        vseg = sgv;
                    }
                }

                const uint32_t tile = ring + st * kStage;
                // fixed groups: this lane's K rows tau(r), 8 + tau(r) (columns cq < 4: values 0-63;
                // cq + 4: 64-127) and V rows cq, cq + 4, cq + 8, cq + 12 (column tau(r): half tau(r) / 4)
                uint32_t ksc[2][2] = {{0u, 0u}, {0u, 0u}}, kmn[2][2] = {{0u, 0u}, {0u, 0u}};
                uint32_t vsc_ab = 0u, vmn_ab = 0u, vsc_cd = 0u, vmn_cd = 0u;
                if constexpr (Fmt == kDecFixed) {
                    const uint32_t kpb = tile + kTileSmem, vpb = kpb + kParBytes;
#pragma unroll
                    for (int n = 0; n < 2; ++n) {
                        const uint4 pw = ld_shared_v4(kpb + (8 * n + tr) * 16);
                        kmn[n][0] = half2_bits(__uint_as_float(pw.x), __uint_as_float(pw.x));
                        ksc[n][0] = half2_bits(__uint_as_float(pw.y), __uint_as_float(pw.y));
                        kmn[n][1] = half2_bits(__uint_as_float(pw.z), __uint_as_float(pw.z));
                        ksc[n][1] = half2_bits(__uint_as_float(pw.w), __uint_as_float(pw.w));
                    }
                    const uint32_t hv = (uint32_t)(tr >> 2) * 8;
                    uint2 pa = ld_shared_v2(vpb + cq * 16 + hv), pb_ = ld_shared_v2(vpb + (cq + 4) * 16 + hv);
                    uint2 pc = ld_shared_v2(vpb + (cq + 8) * 16 + hv), pd = ld_shared_v2(vpb + (cq + 12) * 16 + hv);
                    if (valid < kTile) {  // slots past the end hold anything (NaN parameters too): their
                        const uint2 z2 = make_uint2(0u, 0u);  // values become 0, so 0-weight rows add 0
                        if (cq >= valid) pa = z2;
                        if (cq + 4 >= valid) pb_ = z2;
                        if (cq + 8 >= valid) pc = z2;
                        if (cq + 12 >= valid) pd = z2;
                    }
                    vmn_ab = half2_bits(__uint_as_float(pa.x), __uint_as_float(pb_.x));
                    vsc_ab = half2_bits(__uint_as_float(pa.y), __uint_as_float(pb_.y));
                    vmn_cd = half2_bits(__uint_as_float(pc.x), __uint_as_float(pd.x));
                    vsc_cd = half2_bits(__uint_as_float(pc.y), __uint_as_float(pd.y));
                }
                // S^T = Q K^T: two n-tiles of 8 tokens x 8 k-steps, four accumulator chains;
                // this lane supplies rows tau(r) and 8 + tau(r), columns cq and cq + 4
                const uint32_t kr0 = tile + tr * kD, kr1 = tile + (8 + tr) * kD;
                const uint4 k0 = ld_shared_v4(kr0 + ((cq ^ tr) << 4)), k1 = ld_shared_v4(kr0 + (((cq + 4) ^ tr) << 4));
                const uint4 k2 = ld_shared_v4(kr1 + ((cq ^ tr) << 4)), k3 = ld_shared_v4(kr1 + (((cq + 4) ^ tr) << 4));
                float sa[2][4], sb[2][4];
#pragma unroll
                for (int e = 0; e < 4; ++e) sa[0][e] = sa[1][e] = sb[0][e] = sb[1][e] = 0.0f;
#pragma unroll
                for (int jj = 0; jj < 8; jj += 2) {
                    const uint4 &lo0 = jj < 4 ? k0 : k1;  // n-tile 0: row tau(r), columns cq | cq + 4
                    const uint4 &lo1 = jj < 4 ? k2 : k3;  // n-tile 1: row 8 + tau(r)
                    const int hf = jj < 4 ? 0 : 1;        // which 64-value half these columns are in
                    const uint32_t w00 = word(lo0, jj & 3), w01 = word(lo0, (jj + 1) & 3);
                    const uint32_t w10 = word(lo1, jj & 3), w11 = word(lo1, (jj + 1) & 3);
                    const uint32_t s0 = ksc[0][hf], m0 = kmn[0][hf], s1 = ksc[1][hf], m1 = kmn[1][hf];
                    mma16816(sa[0], qa0[jj], 0u, qa2[jj], 0u, codes2<Fmt, false>(w00, s0, m0), codes2<Fmt, true>(w00, s0, m0));
                    mma16816(sa[1], qa0[jj], 0u, qa2[jj], 0u, codes2<Fmt, false>(w10, s1, m1), codes2<Fmt, true>(w10, s1, m1));
                    mma16816(sb[0], qa0[jj + 1], 0u, qa2[jj + 1], 0u, codes2<Fmt, false>(w01, s0, m0),
                             codes2<Fmt, true>(w01, s0, m0));
                    mma16816(sb[1], qa0[jj + 1], 0u, qa2[jj + 1], 0u, codes2<Fmt, false>(w11, s1, m1),
                             codes2<Fmt, true>(w11, s1, m1));
                }
                // lane scores for head r: tokens cq, cq+4 (n-tile 0) and 8+cq, 12+cq (n-tile 1)
                float z[4];
                z[0] = (cq < valid) ? fmaf(ak, sa[0][0] + sb[0][0], bk) : -INFINITY;
                z[1] = (cq + 4 < valid) ? fmaf(ak, sa[0][1] + sb[0][1], bk) : -INFINITY;
                z[2] = (cq + 8 < valid) ? fmaf(ak, sa[1][0] + sb[1][0], bk) : -INFINITY;
                z[3] = (cq + 12 < valid) ? fmaf(ak, sa[1][1] + sb[1][1], bk) : -INFINITY;
                float mt = fmaxf(fmaxf(z[0], z[1]), fmaxf(z[2], z[3]));
                mt = fmaxf(mt, __shfl_xor_sync(0xffffffffu, mt, 1));
                mt = fmaxf(mt, __shfl_xor_sync(0xffffffffu, mt, 2));
                const bool need = gvalid && (mt > m_run + kLazyRescale);
                float alpha = 1.0f;
                if (need) {
                    alpha = (m_run == -INFINITY) ? 0.0f : ex2(m_run - mt);
                    m_run = mt;
                    l_run *= alpha;
                    bsum *= alpha;
                }
                if (__any_sync(0xffffffffu, need)) {
                    const float a0 = __shfl_sync(0xffffffffu, alpha, 8 * cq);      // head 2cq
                    const float a1 = __shfl_sync(0xffffffffu, alpha, 8 * cq + 4);  // head 2cq+1
#pragma unroll
                    for (int i = 0; i < 8; ++i) {
                        o[i][0] *= a0;
                        o[i][2] *= a0;
                        o[i][1] *= a1;
                        o[i][3] *= a1;
                    }
                }
                float pr[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) pr[e] = gvalid ? ex2(z[e] - m_run) : 0.0f;
                // the tensor cores see p rounded to fp16; the sums use the same rounded weights so
                // the 1024 offset of the codes cancels exactly against bsum
                const uint32_t pb0 = f32x2_to_f16x2(pr[0], pr[1]);
                const uint32_t pb1 = f32x2_to_f16x2(pr[2], pr[3]);
                const float psum = (f16lo(pb0) + f16hi(pb0)) + (f16lo(pb1) + f16hi(pb1));
                l_run += psum;
                bsum = fmaf(cv, psum, bsum);

                // O^T += V^T P^T: rows (d) 16*tr + 2i (+1), k = tokens cq, cq+4, 8+cq, 12+cq
                if (!vflat) {
                    // rows cq, cq + 4, cq + 8, cq + 12, column tau(r)
                    const uint32_t vt = tile + kTileBytes;  // rows cq + 4i, column tau(r)
                    uint4 va = ld_shared_v4(vt + cq * kD + ((tr ^ cq) << 4));
                    uint4 vb = ld_shared_v4(vt + (cq + 4) * kD + ((tr ^ (cq + 4)) << 4));
                    uint4 vc = ld_shared_v4(vt + (cq + 8) * kD + ((tr ^ cq) << 4));
                    uint4 vd = ld_shared_v4(vt + (cq + 12) * kD + ((tr ^ (cq + 4)) << 4));
                    if constexpr (Fmt == kDecFp8) {
                        // slots past the end hold any byte, E4M3 NaN patterns too (0 * NaN would
                        // reach the sums): their codes become +0
                        if (valid < kTile) {
                            const uint4 z4 = make_uint4(0u, 0u, 0u, 0u);
                            if (cq >= valid) va = z4;
                            if (cq + 4 >= valid) vb = z4;
                            if (cq + 8 >= valid) vc = z4;
                            if (cq + 12 >= valid) vd = z4;
                        }
                    }
#pragma unroll
                    for (int wi = 0; wi < 4; ++wi) {
                        const uint32_t xab01 = prmt(word(va, wi), word(vb, wi), 0x5140);
                        const uint32_t xab23 = prmt(word(va, wi), word(vb, wi), 0x7362);
                        const uint32_t xcd01 = prmt(word(vc, wi), word(vd, wi), 0x5140);
                        const uint32_t xcd23 = prmt(word(vc, wi), word(vd, wi), 0x7362);
                        mma16816(o[2 * wi], codes2<Fmt, false>(xab01, vsc_ab, vmn_ab),
                                 codes2<Fmt, true>(xab01, vsc_ab, vmn_ab), codes2<Fmt, false>(xcd01, vsc_cd, vmn_cd),
                                 codes2<Fmt, true>(xcd01, vsc_cd, vmn_cd), pb0, pb1);
                        mma16816(o[2 * wi + 1], codes2<Fmt, false>(xab23, vsc_ab, vmn_ab),
                                 codes2<Fmt, true>(xab23, vsc_ab, vmn_ab), codes2<Fmt, false>(xcd23, vsc_cd, vmn_cd),
                                 codes2<Fmt, true>(xcd23, vsc_cd, vmn_cd), pb0, pb1);
                    }
                }
            }
            issue(st);  // refill this stage kDepth tiles ahead (its reads above are complete)
        }

        // ================================================ end of the piece: combine the four warps
        {
            float l = l_run, bs_ = bsum;
            l += __shfl_xor_sync(0xffffffffu, l, 1);
            l += __shfl_xor_sync(0xffffffffu, l, 2);
            bs_ += __shfl_xor_sync(0xffffffffu, bs_, 1);
            bs_ += __shfl_xor_sync(0xffffffffu, bs_, 2);
            float *cw = s_comb + warp * G * kPartStride;
            if (gvalid && cq == 0) {
                cw[r * kPartStride + 0] = m_run;
                cw[r * kPartStride + 1] = l;
            }
            const int g0 = 2 * cq, g1 = 2 * cq + 1;
            const float b0 = __shfl_sync(0xffffffffu, bs_, 8 * cq), b1 = __shfl_sync(0xffffffffu, bs_, 8 * cq + 4);
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const int d = 16 * tr + 2 * i;
                if (g0 < G)
                    *reinterpret_cast<float2 *>(cw + g0 * kPartStride + 4 + d) =
                        make_float2(fmaf(sigma, o[i][0], b0), fmaf(sigma, o[i][2], b0));
                if (g1 < G)
                    *reinterpret_cast<float2 *>(cw + g1 * kPartStride + 4 + d) =
                        make_float2(fmaf(sigma, o[i][1], b1), fmaf(sigma, o[i][3], b1));
            }
            // the current token's score s_new = q . k_new (log2 domain), one warp per head
            for (int g = warp; g < G; g += kWarpsPerCta) {
                const uint2 qv = reinterpret_cast<const uint2 *>(pb + kPbQ + g * 256)[lane];
                const uint2 kv = reinterpret_cast<const uint2 *>(pb + kPbKnew)[lane];
                float acc = bf16lo_to_f32(qv.x) * bf16lo_to_f32(kv.x);
                acc = fmaf(bf16hi_to_f32(qv.x), bf16hi_to_f32(kv.x), acc);
                acc = fmaf(bf16lo_to_f32(qv.y), bf16lo_to_f32(kv.y), acc);
                acc = fmaf(bf16hi_to_f32(qv.y), bf16hi_to_f32(kv.y), acc);
#pragma unroll
                for (int off = 16; off; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
                if (lane == 0) s_snew[g] = acc * kLog2eOverSqrtD;
            }
        }
        named_bar_sync(1, nthr);

        const int d = tid;  // thread d owns output column d
        const float vn = bf16lo_to_f32((uint32_t)reinterpret_cast<const uint16_t *>(pb + kPbVnew)[d]);
        uint16_t *orow = a.out + ((int64_t)cur.b * a.Hq + cur.h * G) * kD + d;
        // CTAs holding the pair's first and last tiles (this CTA unless the pair leaves its slice;
        // the division only for such pairs)
        const int32_t cfirst = cur.fp >= c0 ? cta : owner(cur.fp, p, C, ncta);
        const int32_t clast = cur.fp + cur.ntl <= c1 ? cta : owner(cur.fp + cur.ntl - 1, p, C, ncta);
        for (int g = 0; g < G; ++g) {
            float M = -INFINITY, L = 0.0f, O = 0.0f;
#pragma unroll
            for (int ww = 0; ww < kWarpsPerCta; ++ww) M = fmaxf(M, s_comb[(ww * G + g) * kPartStride]);
            if (M != -INFINITY) {
#pragma unroll
                for (int ww = 0; ww < kWarpsPerCta; ++ww) {
                    const float *cw = s_comb + (ww * G + g) * kPartStride;
                    if (cw[0] != -INFINITY) {
                        const float f = ex2(cw[0] - M);
                        L = fmaf(cw[1], f, L);
                        O = fmaf(cw[4 + d], f, O);
                    }
                }
            }
            if (cfirst == clast) {
                __nv_bfloat16 ob = __float2bfloat16_rn(finish(M, L, O, s_snew[g], vn));
                orow[g * kD] = *reinterpret_cast<uint16_t *>(&ob);
            } else {  // this CTA's piece at slot p + cta (unique per piece); merged by the combine kernel
                float *dst = a.part + ((int64_t)(p + cta) * G + g) * kPartStride;
                __stcg(dst + 4 + d, O);
                if (d == 0) __stcg(reinterpret_cast<float2 *>(dst), make_float2(M, L));
            }
        }
        if (tid == 0 && cur.fp >= c0) a.pair_info[p] = make_int2(cfirst, clast);  // first piece of the pair
        named_bar_sync(1, nthr);  // the piece buffer, s_comb and s_snew are free again
        if (tid == 0 && ahead.fp < c1) stage_piece(ahead, buf);
        next_piece(ahead, s_tpre, s_len, B, Hkv);
        next_piece(cur, s_tpre, s_len, B, Hkv);
    }
    cp_async_wait<0>();  // no copy may still target shared memory when the CTA exits
}

// Merge of the pieces of every pair that several CTAs share, after the main kernel
// (programmatic dependent launch).  One item per (pair, query head); a grid of at most 4 CTAs
// per SM walks the items (at 128 registers a thread the slot arrays below stay in registers),
// and these small CTAs can already be resident while the main kernel runs.  The pieces are
// folded in a fixed order and the current token is added last, as in the single-piece path:
// the warp merge folds an item's pieces in CTA order, kCombineSlots loads in flight per round;
// the block merge gives warp w the pieces of CTAs cfirst + w, + 4, ... (in that order,
// kCombineSlots per round) and then folds the four warps' states in warp order.
constexpr int kCombineWarps = 4;
constexpr int kCombineSlots = 8;    // pieces one warp keeps in flight per round
constexpr int kCombineCtasPerSm = 4;  // 128 registers a thread: the slot arrays stay in registers
// combine_kernel reads the current value and writes the output with one thread per dimension
static_assert(kCombineWarps * 32 == kD, "the block merge has exactly one thread per head dimension");

__global__ void __launch_bounds__(kCombineWarps * 32, kCombineCtasPerSm) combine_kernel(AttnArgs a)
{
    const int32_t G = a.G, Hkv = a.Hkv;
    const int32_t items = a.B * Hkv * G;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    __shared__ float s_m[kCombineWarps], s_l[kCombineWarps];
    __shared__ float4 s_o[kCombineWarps][32];
    __shared__ float s_sn;
    if (blockIdx.x == 0 && tid == 0) a.hdr->path = kPathBlockMerge;  // which merge ran (tests read it)

    bool waited = false;
    for (int32_t item = blockIdx.x; item < items; item += gridDim.x) {
        const int32_t p = item / G, g = item - p * G;
        const int32_t b = p / Hkv, h = p - b * Hkv;
        // inputs of this call (not written by the main kernel): loaded before the wait
        const uint2 qv = __ldg(reinterpret_cast<const uint2 *>(a.q + ((int64_t)b * a.Hq + h * G + g) * kD) + lane);
        const uint2 kv = __ldg(reinterpret_cast<const uint2 *>(a.knew + ((int64_t)b * Hkv + h) * kD) + lane);
        const float vn = bf16lo_to_f32((uint32_t)__ldg(a.vnew + ((int64_t)b * Hkv + h) * kD + tid));
        if (!waited) {
            pdl_wait_primary();
            waited = true;
        }
        const int2 info = __ldcg(a.pair_info + p);
        const int32_t cfirst = info.x, clast = info.y;
        if (cfirst == clast) continue;  // finished inside the main kernel
        const bool all_held = __ldcg(&a.hdr->pad[kHdrAllHeld]) != 0;  // no slot is empty

        // warp w folds slots cfirst + w, + 4, ...: per slot its (m, l) and this lane's 4 columns of O
        float m_w = -INFINITY, l_w = 0.0f;
        float4 o_w = make_float4(0.f, 0.f, 0.f, 0.f);
        for (int32_t base = cfirst + warp; base <= clast; base += kCombineWarps * kCombineSlots) {
            float mm[kCombineSlots], ll[kCombineSlots];
            float4 oo[kCombineSlots];
#pragma unroll
            for (int i = 0; i < kCombineSlots; ++i) {
                const int32_t cc = base + i * kCombineWarps;
                mm[i] = -INFINITY;
                ll[i] = 0.0f;
                oo[i] = make_float4(0.f, 0.f, 0.f, 0.f);
                if (cc <= clast) {
                    const float *src = a.part + ((int64_t)(p + cc) * G + g) * kPartStride;
                    const float2 ml = __ldcg(reinterpret_cast<const float2 *>(src));
                    mm[i] = ml.x;
                    ll[i] = ml.y;
                    oo[i] = __ldcg(reinterpret_cast<const float4 *>(src + 4) + lane);
                }
            }
            // the slot of a CTA whose slice is empty holds stale data (no piece of this call
            // writes it): dropped
            if (!all_held) {
#pragma unroll
                for (int i = 0; i < kCombineSlots; ++i) {
                    const int32_t cc = base + i * kCombineWarps;
                    if (cc <= clast && __ldcg(a.held + cc) == 0) {
                        mm[i] = -INFINITY;
                        ll[i] = 0.0f;
                        oo[i] = make_float4(0.f, 0.f, 0.f, 0.f);
                    }
                }
            }
#pragma unroll
            for (int i = 0; i < kCombineSlots; ++i) {  // in slot order: online fold
                const float M = fmaxf(m_w, mm[i]);
                if (M == -INFINITY) continue;
                const float fo = m_w == -INFINITY ? 0.0f : ex2(m_w - M);
                const float fn = mm[i] == -INFINITY ? 0.0f : ex2(mm[i] - M);
                l_w = l_w * fo + ll[i] * fn;
                o_w.x = o_w.x * fo + oo[i].x * fn;
                o_w.y = o_w.y * fo + oo[i].y * fn;
                o_w.z = o_w.z * fo + oo[i].z * fn;
                o_w.w = o_w.w * fo + oo[i].w * fn;
                m_w = M;
            }
        }
        if (lane == 0) {
            s_m[warp] = m_w;
            s_l[warp] = l_w;
        }
        s_o[warp][lane] = o_w;
        if (warp == 0) {  // the current token's score
            float acc = bf16lo_to_f32(qv.x) * bf16lo_to_f32(kv.x);
            acc = fmaf(bf16hi_to_f32(qv.x), bf16hi_to_f32(kv.x), acc);
            acc = fmaf(bf16lo_to_f32(qv.y), bf16lo_to_f32(kv.y), acc);
            acc = fmaf(bf16hi_to_f32(qv.y), bf16hi_to_f32(kv.y), acc);
#pragma unroll
            for (int off = 16; off; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
            if (lane == 0) s_sn = acc * kLog2eOverSqrtD;
        }
        __syncthreads();
        {  // thread d: fold the warps in order, then the current token
            const int d = tid;
            float M = -INFINITY, L = 0.0f, O = 0.0f;
            for (int w = 0; w < kCombineWarps; ++w) {
                const float mw = s_m[w];
                const float Mn = fmaxf(M, mw);
                if (Mn == -INFINITY) continue;
                const float fo = M == -INFINITY ? 0.0f : ex2(M - Mn);
                const float fn = mw == -INFINITY ? 0.0f : ex2(mw - Mn);
                const float ow = reinterpret_cast<const float *>(&s_o[w][d >> 2])[d & 3];
                L = L * fo + s_l[w] * fn;
                O = O * fo + ow * fn;
                M = Mn;
            }
            __nv_bfloat16 ob = __float2bfloat16_rn(finish(M, L, O, s_sn, vn));
            a.out[((int64_t)b * a.Hq + h * G + g) * kD + d] = *reinterpret_cast<uint16_t *>(&ob);
        }
        __syncthreads();  // shared memory is reused by the next item
    }
    if (!waited) pdl_wait_primary();
}

// The same merge with one warp per (pair, query head) item, for calls whose pairs are split over
// few CTAs: the warp folds the pieces in CTA order (kCombineSlots in flight), adds the current
// token and writes its four columns per lane; no shared memory and no block barrier.
__global__ void __launch_bounds__(kCombineWarps * 32, kCombineCtasPerSm) combine_warp_kernel(AttnArgs a)
{
    const int32_t G = a.G, Hkv = a.Hkv;
    const int32_t items = a.B * Hkv * G;
    const int lane = threadIdx.x & 31;
    const int32_t nw = gridDim.x * kCombineWarps;
    if (blockIdx.x == 0 && threadIdx.x == 0) a.hdr->path = kPathWarpMerge;  // which merge ran (tests read it)
    bool waited = false;
    for (int32_t item = blockIdx.x * kCombineWarps + (threadIdx.x >> 5); item < items; item += nw) {
        const int32_t p = item / G, g = item - p * G;
        const int32_t b = p / Hkv, h = p - b * Hkv;
        // inputs of this call (not written by the main kernel): loaded before the wait
        const uint2 qv = __ldg(reinterpret_cast<const uint2 *>(a.q + ((int64_t)b * a.Hq + h * G + g) * kD) + lane);
        const uint2 kv = __ldg(reinterpret_cast<const uint2 *>(a.knew + ((int64_t)b * Hkv + h) * kD) + lane);
        const uint2 vv = __ldg(reinterpret_cast<const uint2 *>(a.vnew + ((int64_t)b * Hkv + h) * kD) + lane);
        if (!waited) {
            pdl_wait_primary();
            waited = true;
        }
        const int2 info = __ldcg(a.pair_info + p);
        const int32_t cfirst = info.x, clast = info.y;
        if (cfirst == clast) continue;  // finished inside the main kernel
        const bool all_held = __ldcg(&a.hdr->pad[kHdrAllHeld]) != 0;  // no slot is empty
        float M = -INFINITY, L = 0.0f;
        float4 O = make_float4(0.f, 0.f, 0.f, 0.f);
        for (int32_t base = cfirst; base <= clast; base += kCombineSlots) {
            float mm[kCombineSlots], ll[kCombineSlots];
            float4 oo[kCombineSlots];
#pragma unroll
            for (int i = 0; i < kCombineSlots; ++i) {
                const int32_t cc = base + i;
                mm[i] = -INFINITY;
                ll[i] = 0.0f;
                oo[i] = make_float4(0.f, 0.f, 0.f, 0.f);
                if (cc <= clast) {
                    const float *src = a.part + ((int64_t)(p + cc) * G + g) * kPartStride;
                    const float2 ml = __ldcg(reinterpret_cast<const float2 *>(src));
                    mm[i] = ml.x;
                    ll[i] = ml.y;
                    oo[i] = __ldcg(reinterpret_cast<const float4 *>(src + 4) + lane);
                }
            }
            // the slot of a CTA whose slice is empty holds stale data (no piece of this call
            // writes it): dropped
            if (!all_held) {
#pragma unroll
                for (int i = 0; i < kCombineSlots; ++i) {
                    const int32_t cc = base + i;
                    if (cc <= clast && __ldcg(a.held + cc) == 0) {
                        mm[i] = -INFINITY;
                        ll[i] = 0.0f;
                        oo[i] = make_float4(0.f, 0.f, 0.f, 0.f);
                    }
                }
            }
#pragma unroll
            for (int i = 0; i < kCombineSlots; ++i) {  // in CTA order: online fold
                const float Mn = fmaxf(M, mm[i]);
                if (Mn == -INFINITY) continue;
                const float fo = M == -INFINITY ? 0.0f : ex2(M - Mn);
                const float fn = mm[i] == -INFINITY ? 0.0f : ex2(mm[i] - Mn);
                L = L * fo + ll[i] * fn;
                O.x = O.x * fo + oo[i].x * fn;
                O.y = O.y * fo + oo[i].y * fn;
                O.z = O.z * fo + oo[i].z * fn;
                O.w = O.w * fo + oo[i].w * fn;
                M = Mn;
            }
        }
        // the current token's score, then this lane's columns 4 lane .. 4 lane + 3
        float acc = bf16lo_to_f32(qv.x) * bf16lo_to_f32(kv.x);
        acc = fmaf(bf16hi_to_f32(qv.x), bf16hi_to_f32(kv.x), acc);
        acc = fmaf(bf16lo_to_f32(qv.y), bf16lo_to_f32(kv.y), acc);
        acc = fmaf(bf16hi_to_f32(qv.y), bf16hi_to_f32(kv.y), acc);
#pragma unroll
        for (int off = 16; off; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
        const float sn = acc * kLog2eOverSqrtD;
        uint2 res;
        res.x = pack_bf16x2(finish(M, L, O.x, sn, bf16lo_to_f32(vv.x)), finish(M, L, O.y, sn, bf16hi_to_f32(vv.x)));
        res.y = pack_bf16x2(finish(M, L, O.z, sn, bf16lo_to_f32(vv.y)), finish(M, L, O.w, sn, bf16hi_to_f32(vv.y)));
        reinterpret_cast<uint2 *>(a.out + ((int64_t)b * a.Hq + h * G + g) * kD)[lane] = res;
    }
    if (!waited) pdl_wait_primary();
}

}  // namespace dgq

// ---- host launcher ---------------------------------------------------------------------------

namespace dgq {

size_t attn_smem_bytes(int dec, int32_t B, int32_t G)
{
    const int stage = dec == kDecFixed ? stage_bytes<kDecFixed>() : stage_bytes<kDecAffine>();
    const int piece = dec == kDecSplitV ? piece_bytes<kDecSplitV>() : piece_bytes<kDecAffine>();
    return 1024 + (size_t)kWarpsPerCta * kDepth * stage + 2 * (size_t)piece + 16 + (size_t)kWarpsPerCta * G * kPartStride * 4 +
           8 * 4 + (size_t)(2 * B + 1) * 4;
}

int attn_max_ctas(int nsm) { return nsm * kMaxCtasPerSm; }

AttnLayout attn_layout(int32_t batch, int32_t Hq, int32_t Hkv, int nsm)
{
    AttnLayout l;
    const size_t P = (size_t)batch * Hkv;
    const size_t G = (size_t)(Hq / Hkv);
    size_t off = sizeof(WsHeader);
    l.off_count = off;  // per-pair piece range (int2)
    off = (off + P * 8 + 255) & ~size_t(255);
    l.off_held = off;  // per CTA of the main kernel (int32)
    off = (off + (size_t)attn_max_ctas(nsm) * 4 + 255) & ~size_t(255);
    l.off_part = off;
    off += (P + (size_t)attn_max_ctas(nsm)) * G * kPartStride * 4;
    l.total = (off + 255) & ~size_t(255);
    return l;
}

cudaError_t launch_attn(int32_t format, const void *q, const void *knew, const void *vnew, const uint8_t *kpool,
                        const uint8_t *vpool, const dgq_seg_record *table, const dgq_seg_record *vtable,
                        const float *kpar, const float *vpar,
                        const int32_t *bt, const int32_t *seq_lens, int32_t max_seqlen, int32_t B, int32_t Hq,
                        int32_t Hkv, int32_t bs, int32_t max_blocks, int32_t num_blocks, void *out, void *ws, int nsm,
                        bool *map_failed, cudaStream_t stream)
{
    *map_failed = false;
    const int32_t G = Hq / Hkv;
    AttnLayout l = attn_layout(B, Hq, Hkv, nsm);
    char *base = static_cast<char *>(ws);
    AttnArgs a;
    a.q = static_cast<const uint16_t *>(q);
    a.knew = static_cast<const uint16_t *>(knew);
    a.vnew = static_cast<const uint16_t *>(vnew);
    a.kpool = kpool;
    a.vpool = vpool;
    a.table = table;
    a.vtable = vtable;
    a.kpar = reinterpret_cast<const float4 *>(kpar);
    a.vpar = reinterpret_cast<const float4 *>(vpar);
    a.bt = bt;
    a.seq_lens = seq_lens;
    a.out = static_cast<uint16_t *>(out);
    a.hdr = reinterpret_cast<WsHeader *>(base);
    a.pair_info = reinterpret_cast<int2 *>(base + l.off_count);
    a.held = reinterpret_cast<int32_t *>(base + l.off_held);
    a.part = reinterpret_cast<float *>(base + l.off_part);
    a.B = B;
    a.Hq = Hq;
    a.Hkv = Hkv;
    a.G = G;
    a.bs = bs;
    a.max_blocks = max_blocks;
    a.num_blocks = num_blocks;

    // the kernel instance for the code format (the symmetric INT8 cache is an affine one)
    const int dec = vtable != nullptr ? kDecSplitV
                                      : (format == DGQ_FORMAT_FP8_E4M3 ? kDecFp8
                                                                       : (format == DGQ_FORMAT_FIXED64 ? kDecFixed
                                                                                                       : kDecAffine));
    void (*kern)(AttnArgs) = dec == kDecFp8 ? attn_kernel<kDecFp8>
                             : dec == kDecFixed ? attn_kernel<kDecFixed>
                             : dec == kDecSplitV ? attn_kernel<kDecSplitV>
                                                 : attn_kernel<kDecAffine>;

    // per-device launch shape, computed once per (instance, device, shared-memory size) and host
    // thread; the kernel's shared-memory limit is raised once per device and host thread to what
    // the largest call needs (every thread sets the same value, so none lowers it under another)
    static thread_local int limit_dev[4] = {-1, -1, -1, -1};
    static thread_local int cached_dev[4] = {-1, -1, -1, -1};
    static thread_local size_t cached_smem[4] = {0, 0, 0, 0};
    static thread_local int cached_occ[4] = {0, 0, 0, 0};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const size_t smem = attn_smem_bytes(dec, B, G);
    if (dev != limit_dev[dec]) {
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)attn_smem_bytes(dec, kMaxCallBatch, kMaxGroup));
        if (e != cudaSuccess) return e;
        limit_dev[dec] = dev;
    }
    if (dev != cached_dev[dec] || smem != cached_smem[dec]) {
        int occ = 0;
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, kern, kAttnThreads, smem);
        if (e != cudaSuccess) return e;
        if (occ < 1) return cudaErrorInvalidConfiguration;
        cached_dev[dec] = dev;
        cached_smem[dec] = smem;
        cached_occ[dec] = occ > kMaxCtasPerSm ? kMaxCtasPerSm : occ;
    }
    // upper bound on tiles (every request at max_seqlen): no more CTAs than tiles
    const int64_t tiles = (int64_t)B * Hkv * (max_seqlen > 0 ? (max_seqlen + kTile - 1) / kTile : 1);
    int64_t grid = (int64_t)nsm * cached_occ[dec];
    if (grid > tiles) grid = tiles;
    if (grid < 1) grid = 1;
    kern<<<(unsigned)grid, kAttnThreads, smem, stream>>>(a);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;

    // merge of shared pairs, chained with programmatic dependent launch
    cudaLaunchConfig_t cfg = {};
    const int64_t items = (int64_t)B * Hkv * G;
    // pairs split over few CTAs (at least one pair per two CTAs): one warp per item; otherwise
    // the four warps of a CTA share an item's pieces
    const bool warp_merge = (int64_t)B * Hkv * 2 >= grid;
    const int64_t per_cta = warp_merge ? kCombineWarps : 1;
    const int64_t cneed = (items + per_cta - 1) / per_cta;
    const int64_t cgrid = cneed < (int64_t)nsm * kCombineCtasPerSm ? cneed : (int64_t)nsm * kCombineCtasPerSm;
    cfg.gridDim = dim3((unsigned)cgrid);
    cfg.blockDim = dim3(kCombineWarps * 32);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return warp_merge ? cudaLaunchKernelEx(&cfg, combine_warp_kernel, a) : cudaLaunchKernelEx(&cfg, combine_kernel, a);
}

}  // namespace dgq
