// dgq_prefill.cu -- DGQ compression in two phases for chunked prefill (sm_103a): the window
// statistics of each prefill chunk are taken as soon as the chunk's bf16 K/V are in the paged
// cache (while they are still in L2), and one finishing call segments every (request, head) from
// the accumulated statistics and writes the codes in a single pass over the bf16 cache.
//
// Method ("DeepSeek KV-cache dynamic group quantisation (DGQ)" article, sections 2.2 and 3.2):
// the same per-token variance, 16-token window means, n_groups-1 largest jumps, per-segment
// min/max and codes as dgq_compress -- a window's statistics depend only on its own 16 tokens,
// so computing them chunk by chunk changes nothing.  The paged bf16 source follows the
// "PagedAttention implementation" section of the DeepSeek-V4 KV-cache article; the point of the
// split is that K/V do not travel from HBM twice (the DeepSeek-V4 article's chunked-prefill
// remark; DGQ section 3.2 on keeping compression inside the inference pipeline).
//
// GPU design.
//  * Statistics and codes: sixteen warps per SM stream the windows of the call (a flat list over
//    (request, head, window)) through one shared-memory slot each, one TMA tile copy per tensor
//    and window (the 5-D paged tile map of dgq_window.cuh), and run the shared window arithmetic
//    (window_stats / window_quant) on them.  Measured on this GPU: 16 warps with one window in
//    flight each beat 8 or 12 warps with two (the statistics of an L2-resident chunk are bound
//    by the latency of the window arithmetic, not by bandwidth).
//  * Segmentation: one CTA of eight warps per (request, head): every thread keeps the top four
//    jumps (descending, earlier window first) of its strided share of the windows, each warp
//    reduces its lanes' lists to its own top k, warp 0 merges the eight lists, and the CTA
//    reduces the per-segment extremes; the record and the quantiser parameters follow from
//    make_params.  Compiled with -fmad=false.
#include "dgq_device.cuh"
#include "dgq.h"
#include "dgq_launch.h"
#include "dgq_window.cuh"

#include <stdint.h>

namespace dgq {

constexpr int kPfWarps = 16;                      // worker warps per CTA (statistics and codes)
constexpr int kPfSlots = 1;                       // windows in flight per warp
constexpr int kPfThreads = kPfWarps * 32;
constexpr int kPfRingBytes = kPfWarps * kPfSlots * kWinBytes;
constexpr int kSegThreads = 256;                  // segmentation CTA (one per pair)
constexpr int kStatFloats = 8;  // per window: K mean variance, k min, k max, v min, v max, V mean variance, 0, 0

struct PrefillArgs {
    TileSource src;
    const int32_t *begin;  // statistics: first token of each request's chunk (a multiple of 16)
    const int32_t *end;    // statistics: one past its last token; codes: the request's length
    const int32_t *bt;     // codes: destination block table
    uint8_t *kpool, *vpool;
    float *stats;          // [B, Hkv, max_windows, 8]
    dgq_seg_record *table;
    dgq_seg_record *vtable;  // independent V segmentation: V's records (null: one shared segmentation)
    PairParams *params;    // [2][B * Hkv] quantiser parameters (workspace): K's (or shared), V's
    const int32_t *sel;    // finish: per-pair flags selecting the requests to encode (null: all)
    int32_t sel_mask;
    WsHeader *hdr;
    int32_t B, Hkv, bs, max_windows, max_blocks, num_blocks, max_seqlen;
    int32_t max_groups;
    float min_var;
};

// Whether the finish encodes request b: always without selection flags, else when a flag of one
// of its pairs meets the mask.
__device__ __forceinline__ bool pf_selected(const PrefillArgs &a, int32_t b)
{
    if (a.sel == nullptr) return true;
    int32_t any = 0;
    for (int32_t h = 0; h < a.Hkv; ++h) any |= __ldg(a.sel + (int64_t)b * a.Hkv + h);
    return (any & a.sel_mask) != 0;
}

// Windows of request b in this call: [w0, w1).  Statistics: the chunk's windows; codes: all of
// the request's (none when the finish does not select it).  A range that the call's sizes cannot
// hold is flagged and dropped.
__device__ __forceinline__ void pf_range(const PrefillArgs &a, bool quant, int32_t b, int32_t &w0, int32_t &w1)
{
    w0 = w1 = 0;
    if (quant && !pf_selected(a, b)) return;
    const int32_t t0 = quant ? 0 : __ldg(a.begin + b), t1 = __ldg(a.end + b);
    if (t0 < 0 || t1 < t0 || t1 > a.max_seqlen || (t0 & (kWin - 1)) != 0) {
        if (t1 != t0) record_error(a.hdr, kErrBadLength);
        return;
    }
    w0 = t0 / kWin;
    w1 = (t1 + kWin - 1) / kWin;
}

// Mean variance of the tokens of a V tile, in the same balanced order as K's (window_stats).
__device__ __forceinline__ float tile_var_mean(uint32_t tile, int32_t cnt)
{
    const int lane = threadIdx.x & 31;
    const int t = lane >> 1, hh = lane & 1;
    __nv_bfloat162 mn2 = __float2bfloat162_rn(INFINITY), mx2 = __float2bfloat162_rn(-INFINITY);
    float s = sum64<false>(tile, t, hh, 0, mn2, mx2);
    s = __fadd_rn(s, __shfl_xor_sync(0xffffffffu, s, 1));
    const float mean = __fmul_rn(s, 0.0078125f);  // exact /128
    float e = sum64<true>(tile, t, hh, mean, mn2, mx2);
    e = __fadd_rn(e, __shfl_xor_sync(0xffffffffu, e, 1));
    float var = __fmul_rn(e, 0.0078125f);
    var = t < cnt ? var : 0.0f;
#pragma unroll
    for (int o = 2; o <= 16; o <<= 1) var = __fadd_rn(var, __shfl_xor_sync(0xffffffffu, var, o));
    return __fdiv_rn(var, (float)cnt);
}

// Codes of one window tile when K and V have their own segments: as window_quant, with K's
// segment looked up in pk and V's in pv.
__device__ __forceinline__ void window_quant_split(uint8_t *kpool, uint8_t *vpool, int32_t Hkv, int32_t bs,
                                                   int32_t h, int32_t t0, int32_t cnt, int32_t blk, uint32_t kt,
                                                   uint32_t vt, const PairCache &pk, const PairCache &pv)
{
    const int lane = threadIdx.x & 31;
    const int half = lane >> 4, sub = lane & 15;
    const int sk = __popc(__ballot_sync(0xffffffffu, lane >= 1 && lane < kMaxSeg && pk.start <= t0));
    const int sv = __popc(__ballot_sync(0xffffffffu, lane >= 1 && lane < kMaxSeg && pv.start <= t0));
    const float kmn = __shfl_sync(0xffffffffu, pk.kmn, sk), kinv = __shfl_sync(0xffffffffu, pk.kinv, sk);
    const float vmn = __shfl_sync(0xffffffffu, pv.vmn, sv), vinv = __shfl_sync(0xffffffffu, pv.vinv, sv);
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

// Statistics (quant == false) or codes (quant == true) of every window of the call; `split`:
// statistics also take V's mean variance, codes use K's and V's own segments.
template <bool quant, bool split>
__global__ void __launch_bounds__(kPfThreads, 1) prefill_window_kernel(const __grid_constant__ PrefillArgs a)
{
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = align_smem_1024(smem_raw);
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + kPfRingBytes);  // [kPfWarps][kPfSlots]
    int32_t *s_pre = reinterpret_cast<int32_t *>(full + kPfSlots * kPfWarps);  // [B + 1] window prefix
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int32_t B = a.B, Hkv = a.Hkv;

    if (tid < kPfSlots * kPfWarps) mbar_init(&full[tid], 1);
    if (tid == 0) fence_barrier_init();
    if (warp == 0) {  // exclusive scan of Hkv * (windows of request b)
        int32_t carry = 0;
        for (int base = 0; base < B; base += 32) {
            const int i = base + lane;
            int32_t v = 0;
            if (i < B) {
                int32_t w0, w1;
                pf_range(a, quant, i, w0, w1);
                v = Hkv * (w1 - w0);
            }
            int32_t x = v;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int32_t y = __shfl_up_sync(0xffffffffu, x, o);
                if (lane >= o) x += y;
            }
            if (i < B) s_pre[i] = carry + x - v;
            carry += __shfl_sync(0xffffffffu, x, 31);
        }
        if (lane == 0) s_pre[B] = carry;
    }
    __syncthreads();
    const int32_t total = s_pre[B];
    const int32_t nwarps = gridDim.x * kPfWarps;
    const uint32_t ring = smem_u32(smem) + warp * kPfSlots * kWinBytes;
    uint64_t *bars = full + kPfSlots * warp;
    const uint64_t pol = quant ? make_policy_evict_first() : make_policy_evict_normal();

    struct Loc {
        int32_t b, h, w, t1;
    };
    auto locate = [&](int32_t x) -> Loc {
        int32_t lo = 0, hi = B - 1;
        while (lo < hi) {
            const int32_t mid = (lo + hi + 1) >> 1;
            if (s_pre[mid] <= x) lo = mid;
            else hi = mid - 1;
        }
        int32_t w0, w1;
        pf_range(a, quant, lo, w0, w1);
        const int32_t off = x - s_pre[lo], n = w1 - w0;
        Loc l;
        l.b = lo;
        l.h = off / n;
        l.w = w0 + (off - l.h * n);
        l.t1 = __ldg(a.end + lo);
        return l;
    };
    auto issue = [&](int32_t x, int slot) {
        if (x < total && lane == 0) {
            const Loc l = locate(x);
            fence_proxy_async_smem();  // the slot's earlier reads come before the copy
            load_window(ring + slot * kWinBytes, bars + slot, a.src, l.b, l.h, 0, l.w * kWin, pol, a.hdr);
        }
    };

    const int32_t nw = nwarps;
    int32_t x = blockIdx.x * kPfWarps + warp;
#pragma unroll
    for (int k = 0; k < kPfSlots; ++k) issue(x + k * nw, k);
    uint32_t phase = 0;  // bit s: parity of ring slot s's next completion
    int slot = 0;
    bool failed = false;
    for (; x < total; x += nw, slot = slot + 1 == kPfSlots ? 0 : slot + 1) {
        const Loc l = locate(x);
        if (!mbar_wait_bounded(bars + slot, (phase >> slot) & 1u)) {  // the copy never completed
            if (lane == 0) record_error(a.hdr, kErrBarrierWait);
            failed = true;
            break;
        }
        phase ^= 1u << slot;
        const uint32_t kt = ring + slot * kWinBytes, vt = kt + kTileBytes;
        const int32_t t0 = l.w * kWin, cnt = min(kWin, l.t1 - t0);
        const int64_t pair = (int64_t)l.b * Hkv + l.h;
        if (!quant) {
            const WinStats s = window_stats(kt, vt, cnt);
            const float vmean = split ? tile_var_mean(vt, cnt) : 0.0f;
            if (lane == 0) {
                float4 *dst = reinterpret_cast<float4 *>(a.stats + (pair * a.max_windows + l.w) * kStatFloats);
                __stcg(dst, make_float4(s.mean, s.kmn, s.kmx, s.vmn));
                __stcg(dst + 1, make_float4(s.vmx, vmean, 0.0f, 0.0f));
            }
        } else {
            const PairCache pc = load_params(a.params + pair);
            int32_t blk = -1;
            if (pow2_div(t0, a.bs) < a.max_blocks) blk = __ldg(a.bt + (int64_t)l.b * a.max_blocks + pow2_div(t0, a.bs));
            if ((uint32_t)blk < (uint32_t)a.num_blocks) {
                if (split)
                    window_quant_split(a.kpool, a.vpool, Hkv, a.bs, l.h, t0, cnt, blk, kt, vt, pc,
                                       load_params(a.params + (int64_t)a.B * Hkv + pair));
                else
                    window_quant(a.kpool, a.vpool, Hkv, a.bs, l.h, t0, cnt, blk, kt, vt, pc);
            } else if (lane == 0) {  // not a block of the pools: flagged, nothing written
                record_error(a.hdr, kErrBadBlock);
            }
        }
        __syncwarp();  // the slot's reads are done before it is refilled
        issue(x + kPfSlots * nw, slot);
    }
    // A normal exit leaves no copy in flight (windows past the end are never issued).  After a
    // timed-out wait, wait again (bounded) for this slot's copy and those of the next windows, so
    // that no copy still targets shared memory when the CTA exits.
    if (failed) {
        for (int k = 0; k < kPfSlots; ++k) {
            const int sl = (slot + k) % kPfSlots;
            if (x + k * nw < total) mbar_wait_bounded(bars + sl, (phase >> sl) & 1u);
        }
    }
}

// Boundaries of one pair, chosen by the whole CTA from the window means at float `slot` of each
// window's statistics: at most k of them (the k largest jumps |m[w+1] - m[w]|, descending, the
// earlier window first on ties; none between two windows below min_var).  Every thread keeps
// the top four of its strided share of the windows, each warp reduces its lanes' lists to its
// own top four, and warp 0 merges the warps' lists.  Returns the number placed; cut[] holds
// the starts in windows, ascending (INT32_MAX past the last), in every thread.
__device__ int cta_boundaries(const float *st, int32_t W, int k, float min_var, int slot, int32_t (&cut)[4])
{
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    __shared__ float s_cj[kSegThreads / 32][4];
    __shared__ int32_t s_cw[kSegThreads / 32][4];
    __shared__ int32_t s_cut[4];
    __shared__ int s_k;
    float cj[4] = {-1.0f, -1.0f, -1.0f, -1.0f};
    int32_t cw[4] = {INT32_MAX, INT32_MAX, INT32_MAX, INT32_MAX};
    if (k > 0) {
        for (int32_t w = tid; w + 1 < W; w += kSegThreads) {
            const float m0 = __ldcg(st + (int64_t)w * kStatFloats + slot);
            const float m1 = __ldcg(st + (int64_t)(w + 1) * kStatFloats + slot);
            if (!(m0 >= min_var || m1 >= min_var)) continue;  // two quiet windows stay together
            const float j = fabsf(__fsub_rn(m1, m0));
            if (j > cj[3]) {  // windows arrive in increasing order: an equal jump keeps the earlier
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
    }
    for (int r = 0; r < 4; ++r) {  // each warp: four rounds of arg-best over the lanes' list heads
        float j = cj[0];
        int32_t wv = cw[0];
#pragma unroll
        for (int o = 16; o; o >>= 1) {
            const float oj = __shfl_xor_sync(0xffffffffu, j, o);
            const int32_t ow = __shfl_xor_sync(0xffffffffu, wv, o);
            if (oj > j || (oj == j && ow < wv)) {
                j = oj;
                wv = ow;
            }
        }
        if (lane == 0) {
            s_cj[warp][r] = j;
            s_cw[warp][r] = wv;
        }
        if (cw[0] == wv && j >= 0.0f) {  // the winner pops its head (a window sits in one thread)
            cj[0] = cj[1]; cj[1] = cj[2]; cj[2] = cj[3]; cj[3] = -1.0f;
            cw[0] = cw[1]; cw[1] = cw[2]; cw[2] = cw[3]; cw[3] = INT32_MAX;
        }
    }
    __syncthreads();
    if (warp == 0) {  // merge: one candidate per lane, k rounds of arg-best
        float mj = s_cj[lane >> 2][lane & 3];
        int32_t mw = s_cw[lane >> 2][lane & 3];
        int32_t c4[4] = {INT32_MAX, INT32_MAX, INT32_MAX, INT32_MAX};
        int kk = k < 0 ? 0 : k;
        for (int r = 0; r < kk; ++r) {
            float j = mj;
            int32_t wv = mw;
#pragma unroll
            for (int o = 16; o; o >>= 1) {
                const float oj = __shfl_xor_sync(0xffffffffu, j, o);
                const int32_t ow = __shfl_xor_sync(0xffffffffu, wv, o);
                if (oj > j || (oj == j && ow < wv)) {
                    j = oj;
                    wv = ow;
                }
            }
            if (j < 0.0f) {  // no candidate left
                kk = r;
                break;
            }
            if (mw == wv) {
                mj = -1.0f;
                mw = INT32_MAX;
            }
            int32_t c = wv + 1;  // insertion into the sorted list of starts (in windows)
#pragma unroll
            for (int s = 0; s < 4; ++s) {
                if (c < c4[s]) {
                    const int32_t t = c4[s];
                    c4[s] = c;
                    c = t;
                }
            }
        }
        if (lane == 0) {
#pragma unroll
            for (int s = 0; s < 4; ++s) s_cut[s] = c4[s];
            s_k = k < 0 ? -1 : kk;
        }
    }
    __syncthreads();
#pragma unroll
    for (int s = 0; s < 4; ++s) cut[s] = s_cut[s];
    const int res = s_k;
    __syncthreads();  // the shared lists may be reused by the next call
    return res;
}

// Per-segment extremes of one pair under cut[] (exact in any order), reduced over the CTA:
// floats lo_slot (minima) and lo_slot + 1 (maxima) of each window's statistics.
__device__ void cta_extremes(const float *st, int32_t W, const int32_t (&cut)[4], int lo_slot, float (&mn)[kMaxSeg],
                             float (&mx)[kMaxSeg])
{
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    __shared__ float s_mm[kSegThreads / 32][2][kMaxSeg];
#pragma unroll
    for (int s = 0; s < kMaxSeg; ++s) {
        mn[s] = INFINITY;
        mx[s] = -INFINITY;
    }
    for (int32_t w = tid; w < W; w += kSegThreads) {
        const float lo = __ldcg(st + (int64_t)w * kStatFloats + lo_slot);
        const float hi = __ldcg(st + (int64_t)w * kStatFloats + lo_slot + 1);
        const int sg = (w >= cut[0]) + (w >= cut[1]) + (w >= cut[2]) + (w >= cut[3]);
#pragma unroll
        for (int s = 0; s < kMaxSeg; ++s) {
            if (s == sg) {
                mn[s] = fminf(mn[s], lo);
                mx[s] = fmaxf(mx[s], hi);
            }
        }
    }
#pragma unroll
    for (int s = 0; s < kMaxSeg; ++s) {
        mn[s] = warp_min(mn[s]);
        mx[s] = warp_max(mx[s]);
    }
    if (lane == 0) {
#pragma unroll
        for (int s = 0; s < kMaxSeg; ++s) {
            s_mm[warp][0][s] = mn[s];
            s_mm[warp][1][s] = mx[s];
        }
    }
    __syncthreads();
#pragma unroll
    for (int s = 0; s < kMaxSeg; ++s) {
        for (int w = 0; w < kSegThreads / 32; ++w) {
            mn[s] = fminf(mn[s], s_mm[w][0][s]);
            mx[s] = fmaxf(mx[s], s_mm[w][1][s]);
        }
    }
    __syncthreads();
}

// Segmentation of pair blockIdx.x from its window statistics: record(s) and quantiser parameters.
__global__ void __launch_bounds__(kSegThreads) prefill_segment_kernel(const __grid_constant__ PrefillArgs a)
{
    const int tid = threadIdx.x;
    const int32_t pair = blockIdx.x, b = pair / a.Hkv;
    const int64_t P = (int64_t)a.B * a.Hkv;
    if (!pf_selected(a, b)) return;  // a request the call does not select keeps its record
    int32_t L = __ldg(a.end + b);
    if (L < 0 || L > a.max_seqlen) {
        if (tid == 0) record_error(a.hdr, kErrBadLength);
        L = 0;
    }
    const int32_t W = (L + kWin - 1) / kWin;
    const int k0 = L == 0 ? -1 : min(min(ngroups(L), a.max_groups), W) - 1;  // boundaries to place
    const float *st = a.stats + (int64_t)pair * a.max_windows * kStatFloats;

    int32_t cut[4];
    const int k = cta_boundaries(st, W, k0, a.min_var, 0, cut);  // from K's variance
    float kmn[kMaxSeg], kmx[kMaxSeg], vmn[kMaxSeg], vmx[kMaxSeg];
    cta_extremes(st, W, cut, 1, kmn, kmx);
    if (a.vtable == nullptr) {  // one segmentation, shared by K and V
        cta_extremes(st, W, cut, 3, vmn, vmx);
        if (tid == 0) {
            dgq_seg_record rec = {};
            PairParams pp = {};
            if (k >= 0) make_params(L, k, cut, kmn, kmx, vmn, vmx, rec, pp);
            a.table[pair] = rec;
            a.params[pair] = pp;
        }
        return;
    }
    // independent V segmentation: V's boundaries from V's variance, each record keeps its tensor's
    // fields (the other tensor's are 0)
    int32_t vcut[4];
    const int kv = cta_boundaries(st, W, k0, a.min_var, 5, vcut);
    cta_extremes(st, W, vcut, 3, vmn, vmx);
    if (tid == 0) {
        dgq_seg_record rk = {}, rv = {};
        PairParams pk = {}, pv = {};
        if (k >= 0) {
            make_params(L, k, cut, kmn, kmx, kmn, kmx, rk, pk);
            make_params(L, kv, vcut, vmn, vmx, vmn, vmx, rv, pv);
#pragma unroll
            for (int s = 0; s < kMaxSeg; ++s) {
                rk.v_min[s] = rk.v_scale[s] = 0.0f;
                rv.k_min[s] = rv.k_scale[s] = 0.0f;
            }
            rk.v_inv_last = 0.0f;
            rv.k_inv_last = 0.0f;
        }
        a.table[pair] = rk;
        a.vtable[pair] = rv;
        a.params[pair] = pk;
        a.params[P + pair] = pv;
    }
}

size_t prefill_workspace_bytes(int32_t B, int32_t Hkv)
{
    return sizeof(WsHeader) + 2 * (size_t)B * Hkv * sizeof(PairParams);
}

static size_t prefill_smem(int32_t B) { return 1024 + kPfRingBytes + 8 * kPfSlots * kPfWarps + 4 * ((size_t)B + 1); }

template <bool quant, bool split>
static cudaError_t launch_windows(const PrefillArgs &a, int nsm, cudaStream_t stream)
{
    // the shared-memory limit is raised once per device, to what the largest batch needs
    static thread_local int ready_dev = -1;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev != ready_dev) {
        e = cudaFuncSetAttribute(prefill_window_kernel<quant, split>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)prefill_smem(kMaxCallBatch));
        if (e != cudaSuccess) return e;
        ready_dev = dev;
    }
    prefill_window_kernel<quant, split><<<nsm, kPfThreads, prefill_smem(a.B), stream>>>(a);
    return cudaGetLastError();
}

static bool prefill_args(const SourceDesc &src, int32_t B, int32_t max_seqlen, int32_t Hkv, int32_t bs,
                         float *stats, int32_t max_windows, void *ws, PrefillArgs &a)
{
    if (!encode_tile_source(src, Hkv, bs, &a.src)) return false;
    a.begin = a.end = a.bt = nullptr;
    a.kpool = a.vpool = nullptr;
    a.stats = stats;
    a.table = a.vtable = nullptr;
    a.hdr = static_cast<WsHeader *>(ws);
    a.params = reinterpret_cast<PairParams *>(static_cast<uint8_t *>(ws) + sizeof(WsHeader));
    a.sel = nullptr;
    a.sel_mask = 0;
    a.B = B;
    a.Hkv = Hkv;
    a.bs = bs;
    a.max_windows = max_windows;
    a.max_blocks = a.num_blocks = 0;
    a.max_seqlen = max_seqlen;
    a.max_groups = kMaxSeg;
    a.min_var = 0.0f;
    return true;
}

cudaError_t launch_prefill_stats(const SourceDesc &src, const int32_t *begin, const int32_t *end, int32_t B,
                                 int32_t max_seqlen, int32_t Hkv, int32_t bs, float *stats, int32_t max_windows,
                                 bool v_variance, void *ws, int nsm, bool *map_failed, cudaStream_t stream)
{
    PrefillArgs a;
    *map_failed = !prefill_args(src, B, max_seqlen, Hkv, bs, stats, max_windows, ws, a);
    if (*map_failed) return cudaErrorInvalidValue;
    a.begin = begin;
    a.end = end;
    return v_variance ? launch_windows<false, true>(a, nsm, stream) : launch_windows<false, false>(a, nsm, stream);
}

cudaError_t launch_prefill_finish(const SourceDesc &src, const int32_t *seq_lens, int32_t B, int32_t max_seqlen,
                                  int32_t Hkv, int32_t bs, const float *stats, int32_t max_windows,
                                  const int32_t *bt, int32_t max_blocks, uint8_t *kpool, uint8_t *vpool,
                                  int32_t num_blocks, dgq_seg_record *table, dgq_seg_record *vtable,
                                  GroupSettings gs, const int32_t *sel, int32_t sel_mask, void *ws, int nsm,
                                  bool *map_failed, cudaStream_t stream)
{
    PrefillArgs a;
    *map_failed = !prefill_args(src, B, max_seqlen, Hkv, bs, const_cast<float *>(stats), max_windows, ws, a);
    if (*map_failed) return cudaErrorInvalidValue;
    a.sel = sel;
    a.sel_mask = sel_mask;
    a.end = seq_lens;
    a.bt = bt;
    a.max_blocks = max_blocks;
    a.kpool = kpool;
    a.vpool = vpool;
    a.num_blocks = num_blocks;
    a.table = table;
    a.vtable = vtable;
    a.max_groups = gs.max_groups;
    a.min_var = gs.min_var;
    prefill_segment_kernel<<<(unsigned)(B * Hkv), kSegThreads, 0, stream>>>(a);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    return vtable ? launch_windows<true, true>(a, nsm, stream) : launch_windows<true, false>(a, nsm, stream);
}

}  // namespace dgq
