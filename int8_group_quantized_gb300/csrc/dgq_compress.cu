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

constexpr int kCWarps = 8;                          // consumer warps (plus one TMA producer warp)
constexpr int kThreads = (kCWarps + 1) * 32;
constexpr int kCStages = 16;                        // shared-memory ring of window tiles
constexpr int kTileBytes = kWin * kD * 2;           // 16 tokens x 128 bf16 = 4 KB
constexpr int kCStageBytes = 2 * kTileBytes;        // K tile + V tile

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

// ---- statistics of one window (one warp, tile in shared memory) --------------------------
//
// Lane (half, sub) reads 8 consecutive bf16 of token 2i + half in pass i, so each half-warp
// covers one 128-element row and the half-warp butterfly reproduces the pairwise order.

struct WinStats {
    float mean, kmn, kmx, vmn, vmx;
};

__device__ __forceinline__ WinStats window_stats(uint32_t kt, uint32_t vt, int32_t cnt)
{
    const int lane = threadIdx.x & 31;
    const int half = lane >> 4, sub = lane & 15;
    __nv_bfloat162 kmn2 = __float2bfloat162_rn(INFINITY), kmx2 = __float2bfloat162_rn(-INFINITY);
    __nv_bfloat162 vmn2 = kmn2, vmx2 = kmx2;
    float var[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const int tt = 2 * i + half;
        const bool ok = tt < cnt;
        const uint4 kq = ld_shared_v4(kt + tt * (kD * 2) + sub * 16);
        const uint4 vq = ld_shared_v4(vt + tt * (kD * 2) + sub * 16);
        if (ok) {  // min/max on packed bf16 pairs (exact: widening to fp32 preserves order)
            const uint32_t kw[4] = {kq.x, kq.y, kq.z, kq.w};
            const uint32_t vw[4] = {vq.x, vq.y, vq.z, vq.w};
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const __nv_bfloat162 kx = *reinterpret_cast<const __nv_bfloat162 *>(kw + j);
                const __nv_bfloat162 vx = *reinterpret_cast<const __nv_bfloat162 *>(vw + j);
                kmn2 = __hmin2(kmn2, kx); kmx2 = __hmax2(kmx2, kx);
                vmn2 = __hmin2(vmn2, vx); vmx2 = __hmax2(vmx2, vx);
            }
        }
        float x[8];
        unpack8(kq, x);
        const float mean = __fmul_rn(halfwarp_tree(tree8(x)), 0.0078125f);  // exact /128
        float e[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const float d = __fsub_rn(x[j], mean);
            e[j] = __fmul_rn(d, d);
        }
        const float v = __fmul_rn(halfwarp_tree(tree8(e)), 0.0078125f);
        var[i] = ok ? v : 0.0f;
    }
    // window mean: tokens 2i (lower half-warp) and 2i+1 (upper) pair up first
    float s[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) s[i] = __fadd_rn(var[i], __shfl_xor_sync(0xffffffffu, var[i], 16));
    const float sum16 = __fadd_rn(__fadd_rn(__fadd_rn(s[0], s[1]), __fadd_rn(s[2], s[3])),
                                  __fadd_rn(__fadd_rn(s[4], s[5]), __fadd_rn(s[6], s[7])));
    WinStats r;
    r.mean = __fdiv_rn(sum16, (float)cnt);
    r.kmn = warp_min(fminf(__low2float(kmn2), __high2float(kmn2)));
    r.kmx = warp_max(fmaxf(__low2float(kmx2), __high2float(kmx2)));
    r.vmn = warp_min(fminf(__low2float(vmn2), __high2float(vmn2)));
    r.vmx = warp_max(fmaxf(__low2float(vmx2), __high2float(vmx2)));
    return r;
}

// ---- quantisation -----------------------------------------------------------------------

__device__ __forceinline__ uint32_t code_bits(float x, float mn, float inv)
{
    // rint((x - min) * inv) for 0 <= u < 2^22: adding 1.5 * 2^23 rounds u to an integer
    // (round-to-nearest-even) and leaves that integer in the low mantissa bits.  x >= min
    // makes u >= 0, and u <= 255 * (1 + 2^-22) < 255.5, so the low byte is the code.
    const float u = __fmul_rn(__fsub_rn(x, mn), inv);
    return __float_as_uint(__fadd_rn(u, 12582912.0f));
}

__device__ __forceinline__ uint2 encode8(const uint4 &q, float mn, float inv)
{
    float x[8];
    unpack8(q, x);
    uint32_t c[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) c[j] = code_bits(x[j], mn, inv);
    const uint32_t lo = __byte_perm(__byte_perm(c[0], c[1], 0x0040), __byte_perm(c[2], c[3], 0x0040), 0x5410);
    const uint32_t hi = __byte_perm(__byte_perm(c[4], c[5], 0x0040), __byte_perm(c[6], c[7], 0x0040), 0x5410);
    return make_uint2(lo, hi);
}

// Quantisation parameters of one pair, read once per run of windows of that pair: lane i < 5
// holds segment i's (start, k_min, k_inv, v_min, v_inv).
struct PairCache {
    int32_t p;
    int32_t start;
    float kmn, kinv, vmn, vinv;
};

// Wait (bounded) for the pair's segmentation; false if the wait timed out.
__device__ __forceinline__ bool load_pair(const CompressArgs &a, int32_t p, uint32_t target, PairCache &pc)
{
    const int lane = threadIdx.x & 31;
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
    if (!ok) return false;
    (void)ld_acquire_gpu(a.pair_flag + p);  // every lane acquires the published parameters
    const PairParams *pp = a.params + p;
    const int i = lane < kMaxSeg ? lane : 0;
    pc.p = p;
    pc.start = __ldcg(pp->start + i);
    pc.kmn = __ldcg(pp->k_min + i);
    pc.kinv = __ldcg(pp->k_inv + i);
    pc.vmn = __ldcg(pp->v_min + i);
    pc.vinv = __ldcg(pp->v_inv + i);
    return true;
}

// Codes of one window tile, written straight to its slots in the physical block.
__device__ __forceinline__ void window_quant(const CompressArgs &a, const WinLoc &loc, uint32_t kt, uint32_t vt,
                                             const PairCache &pc, int64_t blk)
{
    const int lane = threadIdx.x & 31;
    const int half = lane >> 4, sub = lane & 15;
    const int32_t t0 = loc.wi * kWin;
    const int32_t cnt = min(kWin, loc.L - t0);
    // segment of the window: number of starts 1..4 at or before t0 (lanes 1..4 hold them)
    const unsigned ballot = __ballot_sync(0xffffffffu, lane >= 1 && lane < kMaxSeg && pc.start <= t0);
    const int s = __popc(ballot);
    const float kmn = __shfl_sync(0xffffffffu, pc.kmn, s), kinv = __shfl_sync(0xffffffffu, pc.kinv, s);
    const float vmn = __shfl_sync(0xffffffffu, pc.vmn, s), vinv = __shfl_sync(0xffffffffu, pc.vinv, s);
    const int64_t dst0 = ((blk * a.Hkv + loc.h) * a.bs + (t0 % a.bs)) * kD + sub * 8;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const int tt = 2 * i + half;
        if (tt < cnt) {
            const uint4 kq = ld_shared_v4(kt + tt * (kD * 2) + sub * 16);
            const uint4 vq = ld_shared_v4(vt + tt * (kD * 2) + sub * 16);
            __stcs(reinterpret_cast<uint2 *>(a.kpool + dst0 + tt * kD), encode8(kq, kmn, kinv));
            __stcs(reinterpret_cast<uint2 *>(a.vpool + dst0 + tt * kD), encode8(vq, vmn, vinv));
        }
    }
}

// ---- the kernel ---------------------------------------------------------------------------

// Per-warp pending arrivals: windows of one pair counted locally and published with one fence.
struct Pending {
    int32_t p, cnt, b, h, L, W, wbase;
};

__device__ __forceinline__ void flush_pending(const CompressArgs &a, Pending &pd, uint32_t target)
{
    if (pd.cnt == 0) return;
    const int lane = threadIdx.x & 31;
    int last = 0;
    if (lane == 0) {
        __threadfence();  // this warp's window statistics before the arrival count
        const uint32_t old = atomicAdd(a.pair_count + pd.p, (uint32_t)pd.cnt);
        last = (old + (uint32_t)pd.cnt == (uint32_t)pd.W);
        if (last) __threadfence();
    }
    last = __shfl_sync(0xffffffffu, last, 0);
    if (last) segment_pair(a, pd.p, pd.b, pd.h, pd.L, pd.W, pd.wbase, target);
    pd.cnt = 0;
    pd.p = -1;
}

__global__ void __launch_bounds__(kThreads, 1)
    compress_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV, CompressArgs a)
{
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = align_smem_1024(smem_raw);
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + kCStages * kCStageBytes);
    uint64_t *empty = full + kCStages;
    int32_t *s_cu = reinterpret_cast<int32_t *>(empty + kCStages);  // [B+1]
    int32_t *s_wpre = s_cu + a.B + 1;                                // [B+1]
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int B = a.B;

    if (tid == 0) {
        for (int s = 0; s < kCStages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        fence_barrier_init();
    }
    for (int i = tid; i <= B; i += kThreads) s_cu[i] = __ldg(a.cu + i);
    __syncthreads();
    // exclusive scan of Hkv * ceil(L_b / 16) (single warp; B is small)
    if (warp == 0) {
        int32_t carry = 0;
        for (int base = 0; base < B; base += 32) {
            const int i = base + lane;
            int32_t v = 0;
            if (i < B) v = a.Hkv * ((s_cu[i + 1] - s_cu[i] + kWin - 1) / kWin);
            int32_t x = v;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int32_t y = __shfl_up_sync(0xffffffffu, x, o);
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

    // The work list of this CTA, identical for the producer and the consumers: for each
    // super-group i, the statistics of its share of super-group i, then the quantisation of its
    // share of the pairs that end in super-group i-1.  Item k uses stage k % kCStages and is
    // processed by consumer warp k % kCWarps.
    const int32_t wps = a.wps;
    const int32_t nsg = (Wtot + wps - 1) / wps;
    auto ranges = [&](int32_t i, int32_t &s0, int32_t &s1, int32_t &q0, int32_t &q1) {
        s0 = s1 = q0 = q1 = 0;
        if (i < nsg) {
            const int32_t lo = i * wps, len = min(wps, Wtot - lo);
            s0 = lo + (int32_t)(((int64_t)len * cta) / ncta);
            s1 = lo + (int32_t)(((int64_t)len * (cta + 1)) / ncta);
        }
        if (i >= 1) {
            // pairs whose last window lies in super-group i-1: from the start of the pair holding
            // its first window to the end of the pair holding its last window (or that pair's
            // start, if it ends later)
            const int32_t A = (i - 1) * wps, Z = min(i * wps, Wtot) - 1;
            int32_t fA, eA, fZ, eZ;
            pair_span(A, s_wpre, s_cu, B, a.Hkv, &fA, &eA);
            pair_span(Z, s_wpre, s_cu, B, a.Hkv, &fZ, &eZ);
            const int32_t lo = fA, hi = (eZ - 1 == Z) ? eZ : fZ;
            if (hi > lo) {
                q0 = lo + (int32_t)(((int64_t)(hi - lo) * cta) / ncta);
                q1 = lo + (int32_t)(((int64_t)(hi - lo) * (cta + 1)) / ncta);
            }
        }
    };

    if (warp == kCWarps) {
        // ---------------------------------------------------------------- TMA producer
        if (lane == 0) {
            prefetch_tensormap(&tmK);
            prefetch_tensormap(&tmV);
            const uint64_t pol_first = make_policy_evict_first();
            uint32_t k = 0;
            bool abort = false;
            for (int32_t i = 0; i <= nsg && !abort; ++i) {
                int32_t s0, s1, q0, q1;
                ranges(i, s0, s1, q0, q1);
                for (int part = 0; part < 2 && !abort; ++part) {
                    const int32_t w0 = part ? q0 : s0, w1 = part ? q1 : s1;
                    for (int32_t w = w0; w < w1; ++w, ++k) {
                        const int stage = k % kCStages;
                        const uint32_t use = k / kCStages;
                        if (use > 0 && !mbar_wait_bounded(&empty[stage], (use - 1) & 1)) {
                            record_error(a.hdr, kErrEmptyWait);
                            abort = true;
                            break;
                        }
                        const WinLoc loc = locate(w, s_wpre, s_cu, B, a.Hkv);
                        const int32_t row = s_cu[loc.b] + loc.wi * kWin;
                        uint8_t *dst = smem + stage * kCStageBytes;
                        mbar_arrive_expect_tx(&full[stage], kCStageBytes);
                        // first read: normal priority, so the tile stays in L2 for its second read;
                        // second read (quantisation) is the last use: evict first
                        if (part) {
                            tma_load_3d_hint(dst, &tmK, 0, loc.h, row, &full[stage], pol_first);
                            tma_load_3d_hint(dst + kTileBytes, &tmV, 0, loc.h, row, &full[stage], pol_first);
                        } else {
                            tma_load_3d(dst, &tmK, 0, loc.h, row, &full[stage]);
                            tma_load_3d(dst + kTileBytes, &tmV, 0, loc.h, row, &full[stage]);
                        }
                    }
                }
            }
        }
    } else {
        // ---------------------------------------------------------------- consumers
        Pending pd;
        pd.p = -1;
        pd.cnt = 0;
        PairCache pc;
        pc.p = -1;
        bool pc_ok = false;
        uint32_t k = 0;
        for (int32_t i = 0; i <= nsg; ++i) {
            int32_t s0, s1, q0, q1;
            ranges(i, s0, s1, q0, q1);
            for (int part = 0; part < 2; ++part) {
                const int32_t w0 = part ? q0 : s0, w1 = part ? q1 : s1;
                for (int32_t w = w0; w < w1; ++w, ++k) {
                    if ((int)(k % kCWarps) != warp) continue;
                    const int stage = k % kCStages;
                    const uint32_t use = k / kCStages;
                    const WinLoc loc = locate(w, s_wpre, s_cu, B, a.Hkv);
                    int64_t blk = 0;
                    if (part == 1) {  // block id and pair parameters, before waiting for the tile
                        blk = __ldg(a.bt + (int64_t)loc.b * a.max_blocks + (loc.wi * kWin) / a.bs);
                        const int32_t p = loc.b * a.Hkv + loc.h;
                        if (p != pc.p) pc_ok = load_pair(a, p, target, pc);
                    }
                    if (!mbar_wait_bounded(&full[stage], use & 1)) {
                        record_error(a.hdr, kErrFullWait);
                        continue;  // no data: skip the window (the call reports the error)
                    }
                    const uint32_t kt = smem_u32(smem) + stage * kCStageBytes;
                    const uint32_t vt = kt + kTileBytes;
                    if (part == 0) {
                        const int32_t cnt = min(kWin, loc.L - loc.wi * kWin);
                        const WinStats st = window_stats(kt, vt, cnt);
                        const int32_t p = loc.b * a.Hkv + loc.h;
                        if (lane == 0) {
                            __stcg(a.win_mean + w, st.mean);
                            __stcg(a.win_mm + w, make_float4(st.kmn, st.kmx, st.vmn, st.vmx));
                        }
                        __syncwarp();
                        if (lane == 0) mbar_arrive(&empty[stage]);
                        if (p != pd.p) {
                            flush_pending(a, pd, target);
                            pd.p = p; pd.b = loc.b; pd.h = loc.h; pd.L = loc.L; pd.W = loc.W;
                            pd.wbase = w - loc.wi;
                        }
                        ++pd.cnt;
                    } else {
                        if (pc_ok) window_quant(a, loc, kt, vt, pc, blk);
                        __syncwarp();
                        if (lane == 0) mbar_arrive(&empty[stage]);
                    }
                }
                if (part == 0) flush_pending(a, pd, target);  // before any wait on a flag
            }
        }
    }

    __syncthreads();
    if (tid == 0) {
        __threadfence();
        const uint32_t old = atomicAdd(&a.hdr->done_ctas, 1u);
        if (old == (uint32_t)ncta - 1u) {  // last CTA of the call: advance the epoch
            a.hdr->done_ctas = 0;
            a.hdr->epoch = target;
            __threadfence();
        }
    }
}

}  // namespace dgq

// ---- host launcher (called from dgq_host.cu after argument checks) ---------------------

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

size_t compress_smem_bytes(int32_t B)
{
    return 1024 + (size_t)kCStages * kCStageBytes + 2 * kCStages * 8 + (size_t)(2 * (B + 1)) * 4;
}

// 3-D map over a packed [T, Hkv, 128] bf16 tensor; box = 16 tokens of one head (4 KB).
static bool make_kv_map(CUtensorMap *map, const void *base, int32_t T, int32_t Hkv)
{
    auto fn = tensor_map_encoder();
    if (!fn) return false;
    cuuint64_t dims[3] = {(cuuint64_t)kD, (cuuint64_t)Hkv, (cuuint64_t)T};
    cuuint64_t strides[2] = {(cuuint64_t)kD * 2, (cuuint64_t)Hkv * kD * 2};
    cuuint32_t box[3] = {(cuuint32_t)kD, 1, (cuuint32_t)kWin};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT16, 3, const_cast<void *>(base), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

cudaError_t launch_compress(const void *k, const void *v, const int32_t *cu, int32_t B, int32_t T,
                            int32_t max_seqlen, int32_t Hkv, int32_t bs, const int32_t *bt, int32_t max_blocks,
                            uint8_t *kpool, uint8_t *vpool, dgq_seg_record *table, void *ws, bool *map_failed,
                            cudaStream_t stream)
{
    *map_failed = false;
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

    CUtensorMap mk, mv;
    const int32_t Tmap = T > 0 ? T : 1;
    if (!make_kv_map(&mk, k, Tmap, Hkv) || !make_kv_map(&mv, v, Tmap, Hkv)) {
        *map_failed = true;
        return cudaErrorInvalidValue;
    }
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    int nsm = 0;
    e = cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    const size_t smem = compress_smem_bytes(B);
    e = cudaFuncSetAttribute(compress_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    int occ = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, compress_kernel, kThreads, smem);
    if (e != cudaSuccess) return e;
    if (occ < 1) return cudaErrorInvalidConfiguration;
    dim3 grid(nsm), block(kThreads);  // one CTA per SM; every CTA is resident (cooperative launch)
    void *args[] = {&mk, &mv, &a};
    return cudaLaunchCooperativeKernel((const void *)compress_kernel, grid, block, args, smem, stream);
}

}  // namespace dgq
