// dgq_compress.cu -- DGQ encode of one layer into the paged INT8 cache (sm_103a).
//
// Method ("DeepSeek KV-cache dynamic group quantisation (DGQ)" article, sections 2.2, 3.2):
// per (request, KV head) the per-token variance of K over D, its mean over 16-token
// windows, the n_groups-1 largest jumps between adjacent window means as segment
// boundaries, per-segment fp32 min/max of K and V, and uint8 codes
// q = rint((x - min) * (255 / (max - min))).  Codes go to the physical block named by the
// block table ("PagedAttention implementation", DeepSeek-V4 KV-cache article).
//
// GPU design: one persistent cooperative kernel.  The flat space of all 16-token windows
// of all (request, head) pairs is cut into super-groups of ~32 MB of bf16 K+V.  Every CTA
// walks the super-groups in order; for super-group i it first computes window statistics
// (variance mean, K/V min/max) for its share of super-group i, then quantises its share
// of the pairs that were completed in super-group i-1.  The warp that finishes the last
// window of a pair segments that pair (no waiting) and publishes a per-pair flag; a
// quantising warp waits on that flag (bounded).  The second read of K/V therefore trails
// the first by about two super-groups (~64 MB), so it is served from the 126 MB L2.
// All windows stay within one block (bs is a multiple of 16) and within one segment
// (boundaries sit on window edges), so a warp's quantisation of a window needs one block
// id and one (min, inv) pair per tensor.
//
// Bit-exactness: every fp32 step that feeds a code or a boundary is a single IEEE
// operation via __fadd_rn / __fsub_rn / __fmul_rn / __fdiv_rn, in the pairwise order the
// oracle fixes (this file is also compiled with -fmad=false).
#include "dgq_device.cuh"
#include "dgq.h"
#include "dgq_launch.h"

#include <cuda_bf16.h>

#include <stdint.h>

namespace dgq {

// Per-(request, head) quantisation parameters published by the segmenting warp.
struct PairParams {
    float k_min[kMaxSeg], k_inv[kMaxSeg], v_min[kMaxSeg], v_inv[kMaxSeg];
    int32_t start[kMaxSeg];
    int32_t n_seg;
    int32_t pad[6];
};
static_assert(sizeof(PairParams) == 128, "PairParams is 128 bytes");

struct CompressArgs {
    const uint16_t *k;
    const uint16_t *v;
    const int32_t *cu;
    const int32_t *bt;
    uint8_t *kpool;
    uint8_t *vpool;
    dgq_seg_record *table;
    WsHeader *hdr;
    uint32_t *pair_count;
    uint32_t *pair_flag;
    PairParams *params;
    float *win_mean;
    float4 *win_mm;
    int32_t B, Hkv, bs, max_blocks;
    int32_t wps;  // windows per super-group
};

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;

__device__ __forceinline__ int32_t ngroups(int32_t L)
{
    if (L < 2048) return 2;
    if (L < 16384) return 3;
    // floor(log2(L / 1024)) = floor(log2(L)) - 10 for integer L >= 1024
    int32_t g = (31 - __clz(L)) - 10 + 2;
    return g < 5 ? g : 5;
}

// ---- window decomposition ------------------------------------------------------------------

struct WinLoc {
    int32_t b, h, wi, W, L;  // request, head, window within the pair, windows in pair, length
};

// s_wpre[b] = Hkv * (windows of requests 0..b-1); s_cu = cu_seqlens copy.
__device__ __forceinline__ WinLoc locate(int32_t w, const int32_t *s_wpre, const int32_t *s_cu, int32_t B,
                                         int32_t Hkv)
{
    int32_t lo = 0, hi = B - 1;
    while (lo < hi) {
        int32_t mid = (lo + hi + 1) >> 1;
        if (s_wpre[mid] <= w) lo = mid;
        else hi = mid - 1;
    }
    WinLoc r;
    r.b = lo;
    r.L = s_cu[lo + 1] - s_cu[lo];
    r.W = (r.L + kWin - 1) / kWin;
    int32_t off = w - s_wpre[lo];
    r.h = off / r.W;
    r.wi = off - r.h * r.W;
    return r;
}

// first window of the pair containing window w, and one past its last window
__device__ __forceinline__ void pair_span(int32_t w, const int32_t *s_wpre, const int32_t *s_cu, int32_t B,
                                          int32_t Hkv, int32_t *first, int32_t *end)
{
    WinLoc l = locate(w, s_wpre, s_cu, B, Hkv);
    *first = w - l.wi;
    *end = *first + l.W;
}

// ---- canonical fp32 sums ---------------------------------------------------------------------

// In-lane balanced tree over 8 values, then butterfly over the 16 lanes of a half-warp
// (xor 1, 2, 4, 8): lane i holds elements [8i, 8i+8) of a 128-element row, so the result
// is sum(left 64) + sum(right 64) recursively, identical in every lane.
__device__ __forceinline__ float tree8(const float *x)
{
    float a = __fadd_rn(x[0], x[1]), b = __fadd_rn(x[2], x[3]);
    float c = __fadd_rn(x[4], x[5]), d = __fadd_rn(x[6], x[7]);
    return __fadd_rn(__fadd_rn(a, b), __fadd_rn(c, d));
}

__device__ __forceinline__ float halfwarp_tree(float s)
{
#pragma unroll
    for (int o = 1; o <= 8; o <<= 1) s = __fadd_rn(s, __shfl_xor_sync(0xffffffffu, s, o));
    return s;
}

__device__ __forceinline__ void unpack8(const uint4 &q, float *x)
{
    x[0] = bf16lo_to_f32(q.x); x[1] = bf16hi_to_f32(q.x);
    x[2] = bf16lo_to_f32(q.y); x[3] = bf16hi_to_f32(q.y);
    x[4] = bf16lo_to_f32(q.z); x[5] = bf16hi_to_f32(q.z);
    x[6] = bf16lo_to_f32(q.w); x[7] = bf16hi_to_f32(q.w);
}

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

// ---- segmentation of one pair (one warp, after its last window's statistics) -------------

__device__ __noinline__ void segment_pair(const CompressArgs &a, int32_t p, int32_t b, int32_t h, int32_t L,
                                          int32_t W, int32_t wbase, uint32_t target)
{
    const int lane = threadIdx.x & 31;
    const int32_t k = min(ngroups(L), W) - 1;  // boundaries to place (0..4)

    // per-lane top-k of (jump desc, window asc) over this lane's windows
    float cj[4] = {-1.0f, -1.0f, -1.0f, -1.0f};
    int32_t cw[4] = {INT32_MAX, INT32_MAX, INT32_MAX, INT32_MAX};
    if (k > 0) {
        for (int32_t w = lane; w + 1 < W; w += 32) {
            float m0 = __ldcg(a.win_mean + wbase + w);
            float m1 = __ldcg(a.win_mean + wbase + w + 1);
            float j = fabsf(__fsub_rn(m1, m0));
            // insert; windows arrive in increasing order, so equal jumps keep the earlier one
            if (j > cj[3]) {
                cj[3] = j; cw[3] = w;
#pragma unroll
                for (int s = 3; s > 0; --s) {
                    if (cj[s] > cj[s - 1]) {
                        float tj = cj[s]; cj[s] = cj[s - 1]; cj[s - 1] = tj;
                        int32_t tw = cw[s]; cw[s] = cw[s - 1]; cw[s - 1] = tw;
                    }
                }
            }
        }
    }
    // k rounds of warp arg-best; the winning lane advances its list
    int32_t cut[4] = {INT32_MAX, INT32_MAX, INT32_MAX, INT32_MAX};  // first window of segments 1..k
    for (int r = 0; r < k; ++r) {
        const float bj = cj[0];
        const int32_t bw = cw[0];
        // select (jump desc, window asc)
        float j = bj;
        int32_t wv = bw;
#pragma unroll
        for (int o = 16; o; o >>= 1) {
            float oj = __shfl_xor_sync(0xffffffffu, j, o);
            int32_t ow = __shfl_xor_sync(0xffffffffu, wv, o);
            if (oj > j || (oj == j && ow < wv)) {
                j = oj;
                wv = ow;
            }
        }
        if (bw == wv) {  // windows are unique, so exactly one lane matches: pop its head
            cj[0] = cj[1]; cj[1] = cj[2]; cj[2] = cj[3]; cj[3] = -1.0f;
            cw[0] = cw[1]; cw[1] = cw[2]; cw[2] = cw[3]; cw[3] = INT32_MAX;
        }
        // insertion into the sorted cut list
        int32_t c = wv + 1;
#pragma unroll
        for (int s = 0; s < 4; ++s) {
            if (c < cut[s]) {
                int32_t t = cut[s];
                cut[s] = c;
                c = t;
            }
        }
    }

    // per-segment fp32 min/max from the window min/max
    float kmn[kMaxSeg], kmx[kMaxSeg], vmn[kMaxSeg], vmx[kMaxSeg];
#pragma unroll
    for (int s = 0; s < kMaxSeg; ++s) {
        kmn[s] = INFINITY; kmx[s] = -INFINITY; vmn[s] = INFINITY; vmx[s] = -INFINITY;
    }
    for (int32_t w = lane; w < W; w += 32) {
        float4 mm = __ldcg(a.win_mm + wbase + w);
        int s = (w >= cut[0]) + (w >= cut[1]) + (w >= cut[2]) + (w >= cut[3]);
#pragma unroll
        for (int i = 0; i < kMaxSeg; ++i) {
            if (s == i) {
                kmn[i] = fminf(kmn[i], mm.x); kmx[i] = fmaxf(kmx[i], mm.y);
                vmn[i] = fminf(vmn[i], mm.z); vmx[i] = fmaxf(vmx[i], mm.w);
            }
        }
    }
#pragma unroll
    for (int i = 0; i < kMaxSeg; ++i) {
        kmn[i] = warp_min(kmn[i]); kmx[i] = warp_max(kmx[i]);
        vmn[i] = warp_min(vmn[i]); vmx[i] = warp_max(vmx[i]);
    }

    if (lane == 0) {
        const int32_t n = k + 1;
        dgq_seg_record rec;
        PairParams pp;
#pragma unroll
        for (int i = 0; i < kMaxSeg; ++i) {
            rec.start[i] = i == 0 ? 0 : (i <= k ? kWin * cut[i - 1] : L);
            rec.pad[i] = 0;
            pp.start[i] = rec.start[i];
            if (i < n) {
                float kn = canon_zero(kmn[i]), kx = canon_zero(kmx[i]);
                float vn = canon_zero(vmn[i]), vx = canon_zero(vmx[i]);
                float kr = __fsub_rn(kx, kn), vr = __fsub_rn(vx, vn);
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
        pp.n_seg = n;
#pragma unroll
        for (int i = 0; i < 6; ++i) pp.pad[i] = 0;
        a.table[p] = rec;
        const uint32_t *src = reinterpret_cast<const uint32_t *>(&pp);
        uint32_t *dst = reinterpret_cast<uint32_t *>(a.params + p);
#pragma unroll
        for (int i = 0; i < 32; ++i) __stcg(dst + i, src[i]);
        a.pair_count[p] = 0;  // nobody else touches the counter in this call
        __threadfence();
        st_release_gpu(a.pair_flag + p, target);
    }
    __syncwarp();
}

// ---- statistics of one window (one warp) -----------------------------------------------

__device__ __forceinline__ void window_stats(const CompressArgs &a, int32_t w, const WinLoc &loc,
                                             const int32_t *s_cu, uint32_t target)
{
    const int lane = threadIdx.x & 31;
    const int half = lane >> 4, sub = lane & 15;
    const int32_t t0 = loc.wi * kWin;
    const int32_t cnt = min(kWin, loc.L - t0);
    const int64_t row0 = ((int64_t)(s_cu[loc.b] + t0) * a.Hkv + loc.h) * kD + sub * 8;
    const int64_t rstride = (int64_t)a.Hkv * kD;

    uint4 kq[8], vq[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        int tt = 2 * i + half;
        if (tt < cnt) {
            kq[i] = __ldg(reinterpret_cast<const uint4 *>(a.k + row0 + tt * rstride));
            vq[i] = __ldg(reinterpret_cast<const uint4 *>(a.v + row0 + tt * rstride));
        }
    }
    // min/max on packed bf16 pairs (exact: bf16 -> fp32 widening preserves order)
    __nv_bfloat162 kmn2 = __float2bfloat162_rn(INFINITY), kmx2 = __float2bfloat162_rn(-INFINITY);
    __nv_bfloat162 vmn2 = kmn2, vmx2 = kmx2;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        if ((2 * i + half) < cnt) {
            const uint32_t *kw = reinterpret_cast<const uint32_t *>(&kq[i]);
            const uint32_t *vw = reinterpret_cast<const uint32_t *>(&vq[i]);
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                __nv_bfloat162 kx = *reinterpret_cast<const __nv_bfloat162 *>(kw + j);
                __nv_bfloat162 vx = *reinterpret_cast<const __nv_bfloat162 *>(vw + j);
                kmn2 = __hmin2(kmn2, kx); kmx2 = __hmax2(kmx2, kx);
                vmn2 = __hmin2(vmn2, vx); vmx2 = __hmax2(vmx2, vx);
            }
        }
    }
    float var[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const bool ok = (2 * i + half) < cnt;
        float x[8];
        unpack8(ok ? kq[i] : make_uint4(0, 0, 0, 0), x);
        float mean = __fmul_rn(halfwarp_tree(tree8(x)), 0.0078125f);  // exact /128
        float e[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            float d = __fsub_rn(x[j], mean);
            e[j] = __fmul_rn(d, d);
        }
        float v = __fmul_rn(halfwarp_tree(tree8(e)), 0.0078125f);
        var[i] = ok ? v : 0.0f;
    }
    float kmn = fminf(__low2float(kmn2), __high2float(kmn2));
    float kmx = fmaxf(__low2float(kmx2), __high2float(kmx2));
    float vmn = fminf(__low2float(vmn2), __high2float(vmn2));
    float vmx = fmaxf(__low2float(vmx2), __high2float(vmx2));
    // window mean: tokens 2i (lower half-warp) and 2i+1 (upper) pair up first
    float s[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) s[i] = __fadd_rn(var[i], __shfl_xor_sync(0xffffffffu, var[i], 16));
    float sum16 = __fadd_rn(__fadd_rn(__fadd_rn(s[0], s[1]), __fadd_rn(s[2], s[3])),
                            __fadd_rn(__fadd_rn(s[4], s[5]), __fadd_rn(s[6], s[7])));
    float mean_w = __fdiv_rn(sum16, (float)cnt);
    kmn = warp_min(kmn); kmx = warp_max(kmx);
    vmn = warp_min(vmn); vmx = warp_max(vmx);

    int last = 0;
    const int32_t p = loc.b * a.Hkv + loc.h;
    if (lane == 0) {
        __stcg(a.win_mean + w, mean_w);
        __stcg(a.win_mm + w, make_float4(kmn, kmx, vmn, vmx));
        __threadfence();
        uint32_t old = atomicAdd(a.pair_count + p, 1u);
        last = (old == (uint32_t)loc.W - 1u);
        if (last) __threadfence();
    }
    last = __shfl_sync(0xffffffffu, last, 0);
    if (last) segment_pair(a, p, loc.b, loc.h, loc.L, loc.W, w - loc.wi, target);
}

// ---- quantise one window (one warp) ----------------------------------------------------

__device__ __forceinline__ uint32_t code_bits(float x, float mn, float inv)
{
    // rint((x - min) * inv) for 0 <= u < 2^22: adding 1.5 * 2^23 rounds u to an integer
    // (round-to-nearest-even) and leaves that integer in the low mantissa bits.  x >= min
    // makes u >= 0, and u <= 255 * (1 + 2^-22) < 255.5, so the low byte is the code.
    float u = __fmul_rn(__fsub_rn(x, mn), inv);
    return __float_as_uint(__fadd_rn(u, 12582912.0f));
}

__device__ __forceinline__ uint2 encode8(const uint4 &q, float mn, float inv)
{
    float x[8];
    unpack8(q, x);
    uint32_t c[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) c[j] = code_bits(x[j], mn, inv);
    uint32_t lo = __byte_perm(__byte_perm(c[0], c[1], 0x0040), __byte_perm(c[2], c[3], 0x0040), 0x5410);
    uint32_t hi = __byte_perm(__byte_perm(c[4], c[5], 0x0040), __byte_perm(c[6], c[7], 0x0040), 0x5410);
    return make_uint2(lo, hi);
}

__device__ __forceinline__ void window_quant(const CompressArgs &a, int32_t w, const WinLoc &loc,
                                             const int32_t *s_cu, uint32_t target)
{
    const int lane = threadIdx.x & 31;
    const int32_t p = loc.b * a.Hkv + loc.h;
    int ok = 1;
    if (lane == 0) {
        uint32_t it = 0;
        while (ld_acquire_gpu(a.pair_flag + p) != target) {
            if (++it >= kSpinLimit) {
                record_error(a.hdr, kErrFlagWait);
                ok = 0;
                break;
            }
            __nanosleep(64);
        }
    }
    ok = __shfl_sync(0xffffffffu, ok, 0);
    if (!ok) return;
    (void)ld_acquire_gpu(a.pair_flag + p);  // every lane acquires the published parameters

    const int half = lane >> 4, sub = lane & 15;
    const int32_t t0 = loc.wi * kWin;
    const int32_t cnt = min(kWin, loc.L - t0);
    const PairParams *pp = a.params + p;
    int s = 0;
#pragma unroll
    for (int i = 1; i < kMaxSeg; ++i) s += (t0 >= __ldcg(pp->start + i));
    const float kmn = __ldcg(pp->k_min + s), kinv = __ldcg(pp->k_inv + s);
    const float vmn = __ldcg(pp->v_min + s), vinv = __ldcg(pp->v_inv + s);

    const int64_t row0 = ((int64_t)(s_cu[loc.b] + t0) * a.Hkv + loc.h) * kD + sub * 8;
    const int64_t rstride = (int64_t)a.Hkv * kD;
    const int64_t blk = __ldg(a.bt + (int64_t)loc.b * a.max_blocks + t0 / a.bs);
    const int64_t dst0 = ((blk * a.Hkv + loc.h) * a.bs + (t0 % a.bs)) * kD + sub * 8;

    uint4 kq[8], vq[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        int tt = 2 * i + half;
        if (tt < cnt) {
            kq[i] = __ldcs(reinterpret_cast<const uint4 *>(a.k + row0 + tt * rstride));
            vq[i] = __ldcs(reinterpret_cast<const uint4 *>(a.v + row0 + tt * rstride));
        }
    }
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        int tt = 2 * i + half;
        if (tt < cnt) {
            __stcs(reinterpret_cast<uint2 *>(a.kpool + dst0 + tt * kD), encode8(kq[i], kmn, kinv));
            __stcs(reinterpret_cast<uint2 *>(a.vpool + dst0 + tt * kD), encode8(vq[i], vmn, vinv));
        }
    }
}

// ---- the kernel ---------------------------------------------------------------------------

__global__ void __launch_bounds__(kThreads, 1) compress_kernel(CompressArgs a)
{
    extern __shared__ int32_t smem[];
    int32_t *s_cu = smem;              // [B+1]
    int32_t *s_wpre = smem + a.B + 1;  // [B+1]
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int B = a.B;

    for (int i = tid; i <= B; i += kThreads) s_cu[i] = __ldg(a.cu + i);
    __syncthreads();
    // exclusive scan of Hkv * ceil(L_b / 16) (single warp; B is small)
    if (warp == 0) {
        int32_t carry = 0;
        for (int base = 0; base < B; base += 32) {
            int i = base + lane;
            int32_t v = 0;
            if (i < B) v = a.Hkv * ((s_cu[i + 1] - s_cu[i] + kWin - 1) / kWin);
            int32_t x = v;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                int32_t y = __shfl_up_sync(0xffffffffu, x, o);
                if (lane >= o) x += y;
            }
            if (i < B) s_wpre[i] = carry + x - v;
            carry += __shfl_sync(0xffffffffu, x, 31);
        }
        if (lane == 0) s_wpre[B] = carry;
    }
    __syncthreads();

    const int32_t Wtot = s_wpre[B];
    const uint32_t target = *reinterpret_cast<volatile uint32_t *>(&a.hdr->epoch) + 1u;
    const int32_t ncta = gridDim.x, cta = blockIdx.x;

    // empty requests: a record with n_seg = 0
    for (int32_t b = cta; b < B; b += ncta) {
        if (s_cu[b + 1] == s_cu[b]) {
            for (int32_t h = tid; h < a.Hkv; h += kThreads) {
                dgq_seg_record rec = {};
                a.table[(int64_t)b * a.Hkv + h] = rec;
            }
        }
    }

    const int32_t wps = a.wps;
    const int32_t nsg = (Wtot + wps - 1) / wps;
    for (int32_t i = 0; i <= nsg; ++i) {
        if (i < nsg) {  // statistics of super-group i, this CTA's contiguous share
            int32_t lo = i * wps, len = min(wps, Wtot - lo);
            int32_t w0 = lo + (int32_t)(((int64_t)len * cta) / ncta);
            int32_t w1 = lo + (int32_t)(((int64_t)len * (cta + 1)) / ncta);
            for (int32_t w = w0 + warp; w < w1; w += kWarps) {
                WinLoc loc = locate(w, s_wpre, s_cu, B, a.Hkv);
                window_stats(a, w, loc, s_cu, target);
            }
        }
        if (i >= 1) {  // quantise the pairs whose last window lies in super-group i-1
            // Those pairs form one contiguous run of windows: from the start of the pair
            // holding the super-group's first window (if that pair ends inside it) to the end
            // of the pair holding its last window (if that pair ends exactly there; else to
            // that pair's start).
            const int32_t A = (i - 1) * wps, Z = min(i * wps, Wtot) - 1;
            int32_t fA, eA, fZ, eZ;
            pair_span(A, s_wpre, s_cu, B, a.Hkv, &fA, &eA);
            pair_span(Z, s_wpre, s_cu, B, a.Hkv, &fZ, &eZ);
            const int32_t q0 = fA;
            const int32_t q1 = (eZ - 1 == Z) ? eZ : fZ;
            int32_t len = q1 - q0;
            if (len > 0) {
                int32_t w0 = q0 + (int32_t)(((int64_t)len * cta) / ncta);
                int32_t w1 = q0 + (int32_t)(((int64_t)len * (cta + 1)) / ncta);
                for (int32_t w = w0 + warp; w < w1; w += kWarps) {
                    WinLoc loc = locate(w, s_wpre, s_cu, B, a.Hkv);
                    window_quant(a, w, loc, s_cu, target);
                }
            }
        }
    }

    __syncthreads();
    if (tid == 0) {
        __threadfence();
        uint32_t old = atomicAdd(&a.hdr->done_ctas, 1u);
        if (old == (uint32_t)ncta - 1u) {  // last CTA of the call: advance the epoch
            a.hdr->done_ctas = 0;
            a.hdr->epoch = target;
            __threadfence();
        }
    }
}

}  // namespace dgq

// ---- host launcher (called from dgq_host.cpp after argument checks) ---------------------

namespace dgq {


static inline size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

CompressLayout compress_layout(int32_t batch, int32_t max_seqlen, int32_t Hkv)
{
    CompressLayout l;
    size_t P = (size_t)batch * Hkv;
    size_t Wmax = P * (size_t)((max_seqlen + kWin - 1) / kWin);
    size_t off = sizeof(WsHeader);
    l.off_count = off; off = align256(off + P * 4);
    l.off_flag = off; off = align256(off + P * 4);
    l.off_params = off; off = align256(off + P * sizeof(PairParams));
    l.off_mean = off; off = align256(off + Wmax * 4);
    l.off_mm = off; off = align256(off + Wmax * 16);
    l.total = off;
    return l;
}

cudaError_t launch_compress(const void *k, const void *v, const int32_t *cu, int32_t B, int32_t max_seqlen,
                            int32_t Hkv, int32_t bs, const int32_t *bt, int32_t max_blocks, uint8_t *kpool,
                            uint8_t *vpool, dgq_seg_record *table, void *ws, cudaStream_t stream)
{
    CompressLayout l = compress_layout(B, max_seqlen, Hkv);
    char *base = static_cast<char *>(ws);
    CompressArgs a;
    a.k = static_cast<const uint16_t *>(k);
    a.v = static_cast<const uint16_t *>(v);
    a.cu = cu;
    a.bt = bt;
    a.kpool = kpool;
    a.vpool = vpool;
    a.table = table;
    a.hdr = reinterpret_cast<WsHeader *>(base);
    a.pair_count = reinterpret_cast<uint32_t *>(base + l.off_count);
    a.pair_flag = reinterpret_cast<uint32_t *>(base + l.off_flag);
    a.params = reinterpret_cast<PairParams *>(base + l.off_params);
    a.win_mean = reinterpret_cast<float *>(base + l.off_mean);
    a.win_mm = reinterpret_cast<float4 *>(base + l.off_mm);
    a.B = B;
    a.Hkv = Hkv;
    a.bs = bs;
    a.max_blocks = max_blocks;
    a.wps = 4096;  // 4096 windows x 16 tokens x 512 B (K+V bf16) = 32 MB per super-group

    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    int nsm = 0;
    e = cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    size_t smem = (size_t)(2 * (B + 1)) * sizeof(int32_t);
    if (smem > 48 * 1024) {
        e = cudaFuncSetAttribute(compress_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
    }
    int occ = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, compress_kernel, kThreads, smem);
    if (e != cudaSuccess) return e;
    if (occ < 1) return cudaErrorInvalidConfiguration;
    if (occ > 2) occ = 2;
    dim3 grid(nsm * occ), block(kThreads);
    void *args[] = {&a};
    return cudaLaunchCooperativeKernel((const void *)compress_kernel, grid, block, args, smem, stream);
}

}  // namespace dgq
