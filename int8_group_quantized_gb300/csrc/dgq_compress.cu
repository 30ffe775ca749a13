// dgq_compress.cu -- DGQ encode of one layer into the paged INT8 cache (sm_103a).
//
// Method ("DeepSeek KV-cache dynamic group quantisation (DGQ)" article, sections 2.2, 3.2):
// per (request, KV head) the per-token variance of K over D, its mean over 16-token
// windows, the n_groups-1 largest jumps between adjacent window means as segment
// boundaries, per-segment fp32 min/max of K and V, and uint8 codes
// q = rint((x - min) * (255 / (max - min))).  Codes go to the physical block named by the
// block table ("PagedAttention implementation", DeepSeek-V4 KV-cache article).
//
// GPU design: one persistent cooperative kernel, one CTA per SM: 10 worker warps, an
// arrival warp and a segmentation warp.
//  * The flat list of all 16-token windows of all (request, head) pairs, in (request, head,
//    window) order, is cut into chunks of 128-256 MB of bf16 K+V (at least four of the call's
//    longest pairs; see kChunkMax).  Workers
//    compute window statistics (variance mean; K and V min/max, also folded into aggregates
//    of 64 windows with exact order-preserving integer atomics) for their CTA's share of
//    each chunk.  Quantisation range m holds the pairs whose last window lies in chunk m; it
//    needs the statistics of chunks 0..m of every CTA: one grid barrier per chunk.
//  * The barrier is split.  A CTA publishes its progress once its workers have finished a
//    chunk's statistics (one release store per CTA and chunk, to a word of its own, so CTAs
//    may run several chunks apart), and only waits for the other CTAs when it is about to
//    quantise range m.  Meanwhile its workers keep computing statistics of later chunks, up
//    to a lead of 512-768 MB past their quantisation position, so that they keep streaming
//    while a range is segmented; within that lead a worker takes statistics before
//    quantisation.  Measured on this GPU with quantisation first (one 131072-token request; 64
//    requests of 128-32768 tokens): 64 MB chunks with a 128 MB lead took 340 / 790 us per layer,
//    256 MB chunks with a 768 MB lead 232 / 655 us, 128 MB chunks with a 512 MB lead 251 / 629 us
//    (long pairs want the larger chunks, shorter ones the smaller); with statistics first the
//    chosen rule takes 235 / 601 us, and smaller chunks or leads stay slower.  Most second reads come from
//    DRAM rather than L2 (they carry an evict-first hint); fewer segmentation stalls matter
//    more here than L2 reuse.
//  * Under full HBM load every dependent round trip through L2 costs microseconds, so all
//    global synchronisation lives in two control warps: the arrival warp publishes the CTA's
//    progress; the segmentation warp polls the progress words of all CTAs and segments every
//    pair that overlaps its CTA's share of a range (a pair shared by several CTAs is
//    segmented by each; the result is the same bits).  Parameters go to a per-CTA slice of the workspace; workers learn of them
//    through shared-memory flags with CTA-scope release/acquire and never wait on global
//    memory themselves.
//  * Each worker streams its windows (every 10th window of its CTA's share) through a
//    private two-window shared-memory ring, one TMA tile copy per window and tensor.  Windows never cross a
//    block (block sizes are multiples of 16) nor a segment (boundaries sit on window
//    edges), so quantising a window needs one block id and one (min, inv) pair per tensor.
//
// Bit-exactness: every fp32 step that feeds a code or a boundary is a single IEEE
// operation via __fadd_rn / __fsub_rn / __fmul_rn / __fdiv_rn, in the pairwise order the
// oracle fixes (this file is also compiled with -fmad=false).  Min and max are exact in any
// order.
#include "dgq_device.cuh"
#include "dgq.h"
#include "dgq_launch.h"
#include "dgq_window.cuh"

#include <cuda_bf16.h>

#include <stdint.h>

namespace dgq {

constexpr int kAgg = 64;        // windows per min/max aggregate
constexpr int kWorkers = 10;    // worker warps per CTA (plus an arrival warp and a segmentation warp)
constexpr int kThreads = (kWorkers + 2) * 32;
constexpr int kRing = 2;                   // windows in flight per worker
static_assert(kRing == 2, "the worker loop alternates two ring slots");
constexpr int kRingBytes = kWorkers * kRing * kWinBytes;
// Windows per chunk, chosen per call: at least four of the call's longest pairs, between 16384
// and kChunkMax (128 to 256 MB of K+V); statistics may lead quantisation by max(65536 windows,
// three chunks).  Measured per layer with quantisation first (one 131072-token request / 64
// requests of 128-32768 tokens, us): 256 MB chunks with a 768 MB lead 232 / 655; 128 MB with
// 512 MB 251 / 629; 128 MB with 384 MB 260 / 643; 192 MB with 576 MB 282 / 640; 512 MB with 1 GB
// 271 / 690.  With statistics first, 128 MB chunks with a 384 MB lead took 267 / 618, with a
// 256 MB lead 282 / 654, and 64 MB chunks 370-379 / 716-733.
constexpr int32_t kChunkMax = 32768;
constexpr int32_t kChunkMin = 16384;
constexpr int kMaxSms = 256;               // largest grid the workspace layout provides for

struct CompressArgs {
    TileSource src;  // where the K and V window tiles come from
    const int32_t *cu;
    const int32_t *bt;
    uint8_t *kpool;
    uint8_t *vpool;
    dgq_seg_record *table;
    WsHeader *hdr;
    PairParams *params;  // [ncta][2][cap]: per-CTA slices, double-buffered by range parity
    uint32_t *prog;      // [ncta]: chunks whose statistics the CTA has published
    float *win_mean;
    float4 *win_mm;
    uint4 *agg;  // per 64 flat windows: ~enc(k min), enc(k max), ~enc(v min), enc(v max); 0 = empty
    int32_t B, Hkv, bs, max_blocks, cap;
    int32_t max_seqlen, num_blocks;  // for the device-side checks of lengths and block ids
    int32_t chunk, ahead;  // windows per chunk; statistics' lead over quantisation, in windows
    int32_t max_groups;  // group-selection settings
    float min_var;
};

// ---- window decomposition ------------------------------------------------------------------

struct WinLoc {
    int32_t b, h, wi, W, L, c0;  // request, head, window in pair, windows in pair, length, cu[b]
};

// s_wpre[b] = Hkv * (windows of requests 0..b-1).
__device__ __forceinline__ WinLoc locate(int32_t w, const int32_t *s_wpre, const int32_t *cu, int32_t B)
{
    int32_t lo = 0, hi = B - 1;
    while (lo < hi) {
        const int32_t mid = (lo + hi + 1) >> 1;
        if (s_wpre[mid] <= w) lo = mid;
        else hi = mid - 1;
    }
    WinLoc r;
    r.b = lo;
    r.c0 = __ldg(cu + lo);
    r.L = __ldg(cu + lo + 1) - r.c0;
    r.W = (r.L + kWin - 1) / kWin;
    const int32_t off = w - s_wpre[lo];
    r.h = off / r.W;
    r.wi = off - r.h * r.W;
    return r;
}

// Move a location n windows forward (the target window must exist); returns how many pair
// boundaries were crossed.
__device__ __forceinline__ int32_t step_loc(WinLoc &l, int32_t n, const int32_t *cu, int32_t Hkv)
{
    int32_t crossed = 0;
    l.wi += n;
    while (l.wi >= l.W) {
        l.wi -= l.W;
        ++crossed;
        if (++l.h == Hkv) {
            l.h = 0;
            do {  // next non-empty request
                l.c0 += l.L;
                ++l.b;
                l.L = __ldg(cu + l.b + 1) - l.c0;
            } while (l.L == 0);
            l.W = (l.L + kWin - 1) / kWin;
        }
    }
    return crossed;
}

// Order-preserving map of fp32 (finite, or infinite) onto uint32, so that an integer max
// atomic gives the exact fp32 max in any order; every value maps above 0, the empty mark.
__device__ __forceinline__ uint32_t ord_enc(float x)
{
    const uint32_t u = __float_as_uint(x);
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
__device__ __forceinline__ float ord_dec(uint32_t e)
{
    return __uint_as_float((e & 0x80000000u) ? (e & 0x7FFFFFFFu) : ~e);
}

// ---- segmentation of one pair (one warp; all of the pair's statistics are visible) ---------

// kFloor: the variance floor is set (a.min_var > 0); without it every jump is a candidate and
// the test is compiled out of the candidate loops, which are on the critical path of long pairs.
template <bool kFloor>
__device__ __noinline__ void segment_pair(const CompressArgs &a, int32_t p, int32_t L, int32_t W, int32_t wbase,
                                          PairParams *dst, bool write_record)
{
    const int lane = threadIdx.x & 31;
    int32_t k = min(min(ngroups(L), a.max_groups), W) - 1;  // boundaries to place (0..4)

    // (1) per-lane top-k of (jump desc, window asc); the jump of window w < W-1 is
    // |m[w+1] - m[w]|.  A pair of at most 256 windows is read in one round (lane i holds windows
    // 8i .. 8i+7 with their means and extremes); a longer one reads aligned quads of the flat
    // mean array, eight quads in flight per lane, and takes its extremes from aggregates below.
    float cj[4] = {-1.0f, -1.0f, -1.0f, -1.0f};
    int32_t cw[4] = {INT32_MAX, INT32_MAX, INT32_MAX, INT32_MAX};
    const bool small = W <= 8 * 32;
    float4 smm[8];  // small pairs: extremes of this lane's windows
    if (small) {
        float m[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const int32_t w = 8 * lane + i;
            m[i] = 0.0f;
            smm[i] = make_float4(INFINITY, -INFINITY, INFINITY, -INFINITY);
            if (w < W) {
                m[i] = __ldcg(a.win_mean + wbase + w);
                smm[i] = __ldcg(a.win_mm + wbase + w);
            }
        }
        const float mnext = __shfl_down_sync(0xffffffffu, m[0], 1);  // first mean of the next lane
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const int32_t w = 8 * lane + i;
            if (k == 0 || w + 1 >= W) continue;
            const float mn1 = i < 7 ? m[i + 1] : mnext;
            if (kFloor && !(m[i] >= a.min_var || mn1 >= a.min_var)) continue;  // two quiet windows stay together
            const float j = fabsf(__fsub_rn(mn1, m[i]));
            // a lane meets its windows in increasing order, so an equal jump keeps the earlier
            // window ahead of it
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
    } else if (k > 0) {
        const int32_t q0 = wbase >> 2, q1 = (wbase + W - 1) >> 2;
        const float4 *mq = reinterpret_cast<const float4 *>(a.win_mean);
        for (int32_t qb = q0 + lane; qb <= q1; qb += 32 * 8) {
            float4 mv[8];
            float nx[8];
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                const int32_t q = qb + 32 * u;
                mv[u] = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
                nx[u] = 0.0f;
                if (q <= q1) {
                    mv[u] = __ldcg(mq + q);
                    if (4 * q + 4 < wbase + W) nx[u] = __ldcg(a.win_mean + 4 * q + 4);
                }
            }
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                const int32_t q = qb + 32 * u;
                const float m5[5] = {mv[u].x, mv[u].y, mv[u].z, mv[u].w, nx[u]};
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int32_t w = 4 * q + e - wbase;  // window within the pair
                    if (q > q1 || w < 0 || w + 1 >= W) continue;
                    if (kFloor && !(m5[e] >= a.min_var || m5[e + 1] >= a.min_var)) continue;  // two quiet windows
                    const float j = fabsf(__fsub_rn(m5[e + 1], m5[e]));
                    // a lane meets its windows in increasing order, so an equal jump keeps the
                    // earlier window ahead of it
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
            }
        }
    }
    // k rounds of warp arg-best; the winning lane pops its head
    int32_t cut[4] = {INT32_MAX, INT32_MAX, INT32_MAX, INT32_MAX};  // first window of segments 1..k
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
        if (bw == wv) {  // a window sits in one lane only, so exactly one lane matches
            cj[0] = cj[1]; cj[1] = cj[2]; cj[2] = cj[3]; cj[3] = -1.0f;
            cw[0] = cw[1]; cw[1] = cw[2]; cw[2] = cw[3]; cw[3] = INT32_MAX;
        }
        int32_t c = wv + 1;  // insertion into the sorted cut list
#pragma unroll
        for (int s = 0; s < 4; ++s) {
            if (c < cut[s]) {
                const int32_t t = cut[s];
                cut[s] = c;
                c = t;
            }
        }
    }

    float kmn[kMaxSeg], kmx[kMaxSeg], vmn[kMaxSeg], vmx[kMaxSeg];
#pragma unroll
    for (int s = 0; s < kMaxSeg; ++s) {
        kmn[s] = INFINITY; kmx[s] = -INFINITY; vmn[s] = INFINITY; vmx[s] = -INFINITY;
    }
    if (small) {  // extremes of the windows held in registers
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const int32_t w = 8 * lane + i;
            if (w >= W) continue;
            const int sg = (w >= cut[0]) + (w >= cut[1]) + (w >= cut[2]) + (w >= cut[3]);
#pragma unroll
            for (int s = 0; s < kMaxSeg; ++s) {
                if (s == sg) {
                    kmn[s] = fminf(kmn[s], smm[i].x); kmx[s] = fmaxf(kmx[s], smm[i].y);
                    vmn[s] = fminf(vmn[s], smm[i].z); vmx[s] = fmaxf(vmx[s], smm[i].w);
                }
            }
        }
    } else {
        // (2) per-segment fp32 min/max: whole 64-window aggregates inside the segment, single
        // windows at its two ragged ends.  The runs of all segments are walked as one list so that
        // every load of a round is issued before any is used.
        int32_t rsrc[3 * kMaxSeg], rlen[3 * kMaxSeg], roff[3 * kMaxSeg];
        int32_t total = 0;
#pragma unroll
        for (int s = 0; s < kMaxSeg; ++s) {
            rsrc[3 * s] = rsrc[3 * s + 1] = rsrc[3 * s + 2] = 0;
            rlen[3 * s] = rlen[3 * s + 1] = rlen[3 * s + 2] = 0;
            if (s <= k) {
                const int32_t sw = s == 0 ? 0 : cut[s - 1];
                const int32_t ew = s < k ? cut[s] : W;
                const int32_t f0 = wbase + sw, f1 = wbase + ew;             // flat windows [f0, f1)
                const int32_t a0 = (f0 + kAgg - 1) / kAgg, a1 = f1 / kAgg;  // aggregates [a0, a1) inside
                const bool whole = a0 < a1;
                rsrc[3 * s] = a0;                          // aggregates
                rlen[3 * s] = whole ? a1 - a0 : 0;
                rsrc[3 * s + 1] = f0;                      // head windows [f0, e0)
                rlen[3 * s + 1] = (whole ? a0 * kAgg : f1) - f0;
                rsrc[3 * s + 2] = whole ? a1 * kAgg : f1;  // tail windows [e1, f1)
                rlen[3 * s + 2] = whole ? f1 - a1 * kAgg : 0;
            }
        }
#pragma unroll
        for (int r = 0; r < 3 * kMaxSeg; ++r) {
            roff[r] = total;
            total += rlen[r];
        }
        constexpr int kItems = 4;  // loads per lane per round
        for (int32_t base = 0; base < total; base += 32 * kItems) {
            uint4 v[kItems];
            int rr[kItems];
#pragma unroll
            for (int u = 0; u < kItems; ++u) {
                const int32_t idx = base + lane + 32 * u;
                rr[u] = -1;
                int32_t src = 0;
#pragma unroll
                for (int r = 0; r < 3 * kMaxSeg; ++r) {
                    if (idx >= roff[r] && idx < roff[r] + rlen[r]) {
                        rr[u] = r;
                        src = rsrc[r] + idx - roff[r];
                    }
                }
                if (rr[u] >= 0)
                    v[u] = (rr[u] % 3 == 0) ? __ldcg(a.agg + src) : __ldcg(reinterpret_cast<const uint4 *>(a.win_mm + src));
            }
#pragma unroll
            for (int u = 0; u < kItems; ++u) {
                if (rr[u] < 0) continue;
                float kn, kx, vn, vx;
                if (rr[u] % 3 == 0) {
                    kn = ord_dec(~v[u].x); kx = ord_dec(v[u].y); vn = ord_dec(~v[u].z); vx = ord_dec(v[u].w);
                } else {
                    kn = __uint_as_float(v[u].x); kx = __uint_as_float(v[u].y);
                    vn = __uint_as_float(v[u].z); vx = __uint_as_float(v[u].w);
                }
                const int sg = rr[u] / 3;
#pragma unroll
                for (int s = 0; s < kMaxSeg; ++s) {
                    if (s == sg) {
                        kmn[s] = fminf(kmn[s], kn); kmx[s] = fmaxf(kmx[s], kx);
                        vmn[s] = fminf(vmn[s], vn); vmx[s] = fmaxf(vmx[s], vx);
                    }
                }
            }
        }
    }
#pragma unroll
    for (int s = 0; s < kMaxSeg; ++s) {
        kmn[s] = warp_min(kmn[s]); kmx[s] = warp_max(kmx[s]);
        vmn[s] = warp_min(vmn[s]); vmx[s] = warp_max(vmx[s]);
    }

    if (lane == 0) {
        const int32_t n = k + 1;
        dgq_seg_record rec;
        PairParams pp;
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
        if (write_record) a.table[p] = rec;
        const uint4 *src = reinterpret_cast<const uint4 *>(&pp);
        uint4 *d = reinterpret_cast<uint4 *>(dst);
#pragma unroll
        for (int i = 0; i < 8; ++i) __stcg(d + i, src[i]);
    }
    __syncwarp();
}

// ---- the kernel ---------------------------------------------------------------------------

// A warp's position in one of its two item sequences (statistics of chunk m, or
// quantisation of range m): window w of the CTA's share [.., end), its location, and (for
// quantisation) the ordinal of its pair among the pairs of the share.  w < 0: sequence over.
struct Cursor {
    int32_t m, w, end, slot;
    WinLoc loc;
};

// One window in flight in a worker's ring.
struct Item {
    int32_t kind;    // 0 statistics, 1 quantisation; after an error 2 (quantisation) or 3
                     // (statistics): nothing to compute
    int32_t m, slot;
    int32_t next_m;  // chunk / range of the worker's next item of the same kind (M if none)
    int32_t w;       // flat window index
    int32_t cnt;     // tokens in the window
    int32_t t0;      // first token of the window within its pair
    int32_t h;       // KV head
    int32_t blk;     // physical block holding the window (quantisation)
    PairCache pc;
};

// shared-memory control words
struct CtaCtl {
    int32_t stats_done[kWorkers];  // per worker: first chunk whose statistics are not all done
    int32_t quant_done[kWorkers];  // per worker: first range whose quantisation is not all done
    int32_t ready[2];              // range m's parameters are published when ready[m & 1] >= m + 1
    int32_t abort;
    int32_t last;
    int32_t pad[4];
    uint64_t full[kWorkers][kRing];  // a worker's ring slot holds its window
};

__global__ void __launch_bounds__(kThreads, 1) compress_kernel(const __grid_constant__ CompressArgs a)
{
    extern __shared__ __align__(16) uint8_t smem_raw[];
    uint8_t *smem = align_smem_1024(smem_raw);  // window tiles start on 1024-byte boundaries
    CtaCtl *ctl = reinterpret_cast<CtaCtl *>(smem + kRingBytes);
    int32_t *s_wpre = reinterpret_cast<int32_t *>(smem + kRingBytes + sizeof(CtaCtl));  // [B+1]
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int B = a.B;

    if (warp == 0) {  // exclusive scan of Hkv * ceil(L_b / 16)
        int32_t carry = 0;
        bool bad = false;  // a length outside [0, max_seqlen]: the workspace was sized for less
        for (int base = 0; base < B; base += 32) {
            const int i = base + lane;
            int32_t v = 0;
            if (i < B) {
                const int32_t L = __ldg(a.cu + i + 1) - __ldg(a.cu + i);
                bad |= L < 0 || L > a.max_seqlen;
                v = a.Hkv * ((max(0, min(L, a.max_seqlen)) + kWin - 1) / kWin);
            }
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
        bad = __any_sync(0xffffffffu, bad);
        if (lane == 0) {
            ctl->last = bad ? 1 : 0;  // read after the barrier below, reset before any other use
            if (bad) record_error(a.hdr, kErrBadLength);
        }
    }
    if (tid >= 32 && tid < 32 + kWorkers) {
        ctl->stats_done[tid - 32] = 0;
        ctl->quant_done[tid - 32] = 0;
    }
    if (tid == 32) {
        ctl->ready[0] = ctl->ready[1] = 0;
        ctl->abort = 0;
        for (int w = 0; w < kWorkers; ++w)
            for (int r = 0; r < kRing; ++r) mbar_init(&ctl->full[w][r], 1);
        fence_barrier_init();
    }
    __syncthreads();

    // every CTA read the same lengths: all leave here together, before any grid-wide step
    if (ctl->last) return;
    __syncthreads();  // the check above is read by every thread before the word is reused
    if (tid == 0) ctl->last = 0;
    const int32_t Wtot = s_wpre[B];
    if (blockIdx.x == 0 && tid == 0) a.hdr->path = kPathGrid;
    const int32_t chunk = a.chunk;
    const int32_t M = (Wtot + chunk - 1) / chunk;  // chunks (and quantisation ranges)
    const int32_t ncta = gridDim.x, cta = blockIdx.x;

    // empty requests: a record with n_seg = 0
    for (int32_t b = cta; b < B; b += ncta) {
        if (__ldg(a.cu + b + 1) == __ldg(a.cu + b)) {
            for (int32_t h = tid; h < a.Hkv; h += kThreads) {
                dgq_seg_record rec = {};
                a.table[(int64_t)b * a.Hkv + h] = rec;
            }
        }
    }

    // end of the pairs completed by chunk m (the first window of the pair holding window
    // min((m+1) chunk, Wtot), or Wtot)
    auto qend = [&](int32_t m) -> int32_t {
        const int32_t E = (int32_t)min((int64_t)(m + 1) * chunk, (int64_t)Wtot);
        if (E >= Wtot) return Wtot;
        return E - locate(E, s_wpre, a.cu, B).wi;
    };
    auto split = [&](int32_t lo0, int32_t hi0, int32_t &lo, int32_t &hi) {
        const int64_t n = hi0 - lo0;
        lo = lo0 + (int32_t)((n * cta) / ncta);
        hi = lo0 + (int32_t)((n * (cta + 1)) / ncta);
    };
    // this CTA's share of chunk m's statistics / of range m's quantisation
    auto stats_share = [&](int32_t m, int32_t &lo, int32_t &hi) {
        split(m * chunk, (int32_t)min((int64_t)(m + 1) * chunk, (int64_t)Wtot), lo, hi);
    };
    auto quant_share = [&](int32_t m, int32_t &lo, int32_t &hi) {
        split(m == 0 ? 0 : qend(m - 1), qend(m), lo, hi);
    };
    auto slice = [&](int32_t m) { return a.params + ((int64_t)cta * 2 + (m & 1)) * a.cap; };

    // bounded wait helper for the control warps: false while waiting may go on; true (after
    // recording the error and telling the CTA to skip dependent work) once the limit is reached
    auto give_up = [&](uint32_t &spins) -> bool {
        if (++spins < kSpinLimit) {
            __nanosleep(128);
            return false;
        }
        if (lane == 0) {
            record_error(a.hdr, kErrBarrierWait);
            st_release_cta_shared(&ctl->abort, 1);
        }
        return true;
    };

    if (warp == kWorkers) {
        // ================================================================ arrival warp
        // Publish the CTA's progress as soon as every worker has finished a chunk's statistics.
        int32_t ma = 0;
        uint32_t spins = 0;
        while (ma < M) {
            int32_t d = INT32_MAX;
            if (lane == 0)
                for (int i = 0; i < kWorkers; ++i) d = min(d, ld_acquire_cta_shared(ctl->stats_done + i));
            d = __shfl_sync(0xffffffffu, d, 0);
            if (d > ma) {
                ma = d < M ? d : M;
                // the workers' window statistics (acquired above) before the progress word
                if (lane == 0) st_release_gpu(a.prog + cta, (uint32_t)ma);
                spins = 0;
            } else if (give_up(spins)) {
                break;
            }
        }
    } else if (warp == kWorkers + 1) {
        // ================================================================ segmentation warp
        // Per range: wait until every CTA has published chunks 0..m (and no worker still uses
        // the parameter slice of range m-2), segment the pairs overlapping this CTA's share,
        // and let the workers quantise the range.
        for (int32_t ms = 0; ms < M; ++ms) {
            int32_t qlo, qhi;
            quant_share(ms, qlo, qhi);
            if (qlo < qhi) {
                uint32_t spins = 0;
                bool ok = true;
                while (true) {
                    int32_t d = INT32_MAX;
                    if (lane == 0)
                        for (int i = 0; i < kWorkers; ++i) d = min(d, ld_acquire_cta_shared(ctl->quant_done + i));
                    d = __shfl_sync(0xffffffffu, d, 0);
                    uint32_t done = 0;
                    if (d >= ms - 1) {  // all progress words in one round of relaxed loads
                        uint32_t pv[kMaxSms / 32];
#pragma unroll
                        for (int j = 0; j < kMaxSms / 32; ++j)
                            pv[j] = lane + 32 * j < ncta ? ld_relaxed_gpu(a.prog + lane + 32 * j) : 0xffffffffu;
                        done = 0xffffffffu;
#pragma unroll
                        for (int j = 0; j < kMaxSms / 32; ++j) done = min(done, pv[j]);
                        done = __reduce_min_sync(0xffffffffu, done);
                    }
                    if (d >= ms - 1 && done >= (uint32_t)(ms + 1)) break;
                    if (give_up(spins)) {
                        ok = false;
                        break;
                    }
                }
                if (!ok) break;
                __threadfence();  // with the relaxed loads above: acquire of every CTA's progress
                __syncwarp();
                PairParams *out = slice(ms);
                WinLoc l = locate(qlo, s_wpre, a.cu, B);
                int32_t w = qlo, slot = 0;
                while (true) {
                    const int32_t wbase = w - l.wi;
                    if (a.min_var > 0.0f)
                        segment_pair<true>(a, l.b * a.Hkv + l.h, l.L, l.W, wbase, out + slot, wbase >= qlo);
                    else
                        segment_pair<false>(a, l.b * a.Hkv + l.h, l.L, l.W, wbase, out + slot, wbase >= qlo);
                    ++slot;
                    w = wbase + l.W;
                    if (w >= qhi) break;
                    step_loc(l, l.W - l.wi, a.cu, a.Hkv);
                }
                __syncwarp();
            }
            if (lane == 0) {
                __threadfence_block();
                st_release_cta_shared(ctl->ready + (ms & 1), ms + 1);
            }
        }
    } else {
        // ================================================================ worker warps
        const uint32_t ring = smem_u32(smem) + warp * (kRing * kWinBytes);
        uint64_t *full = ctl->full[warp];
        const uint64_t pol_stats = make_policy_evict_normal();
        const uint64_t pol_quant = make_policy_evict_first();  // second read: last use

        auto seek = [&](Cursor &c, bool quant) {
            for (; c.m < M; ++c.m) {
                int32_t lo, hi;
                if (quant) quant_share(c.m, lo, hi);
                else stats_share(c.m, lo, hi);
                if (lo + warp < hi) {
                    c.w = lo + warp;
                    c.end = hi;
                    if (quant) {
                        c.loc = locate(lo, s_wpre, a.cu, B);
                        c.slot = step_loc(c.loc, warp, a.cu, a.Hkv);
                    } else {
                        c.loc = locate(c.w, s_wpre, a.cu, B);
                        c.slot = 0;
                    }
                    return;
                }
            }
            c.w = -1;
        };
        auto advance = [&](Cursor &c, bool quant) {
            c.w += kWorkers;
            if (c.w < c.end) {
                c.slot += step_loc(c.loc, kWorkers, a.cu, a.Hkv);
                return;
            }
            ++c.m;
            seek(c, quant);
        };

        Cursor sc, qc;
        sc.m = 0;
        qc.m = 0;
        seek(sc, false);
        seek(qc, true);
        if (lane == 0) {
            st_release_cta_shared(ctl->stats_done + warp, sc.w >= 0 ? sc.m : M);
            st_release_cta_shared(ctl->quant_done + warp, qc.w >= 0 ? qc.m : M);
        }

        int32_t cur_m = -1, cur_slot = -1;  // parameters currently held in `params`
        PairCache params = {0, 0.0f, 0.0f, 0.0f, 0.0f};

        // Choose the next item and start its copy into ring slot `slot`; false when nothing may
        // start now.
        auto try_issue = [&](Item &it, int slot) -> bool {
            it.slot = slot;
            const bool aborted = *reinterpret_cast<volatile int32_t *>(&ctl->abort) != 0;
            // statistics first, as long as the lead allows: quantisation waits for ranges whose
            // segmentation needs every CTA's statistics, so letting statistics stream keeps the
            // later ranges' segmentation ahead of the workers (measured on the mixed batch: 613
            // against 645 us per layer with quantisation first; the long request unchanged)
            const bool stats_ok = sc.w >= 0 && (qc.w < 0 || sc.m <= qc.m || sc.w < qc.w + a.ahead);
            if (qc.w >= 0 &&
                (aborted || (!stats_ok && ld_acquire_cta_shared(ctl->ready + (qc.m & 1)) >= qc.m + 1))) {
                it.kind = aborted ? 2 : 1;
                it.m = qc.m;
                if (!aborted) {
                    if (qc.m != cur_m || qc.slot != cur_slot) {
                        params = load_params(slice(qc.m) + qc.slot);
                        cur_m = qc.m;
                        cur_slot = qc.slot;
                    }
                    it.pc = params;
                    it.blk = __ldg(a.bt + (int64_t)qc.loc.b * a.max_blocks + pow2_div(qc.loc.wi * kWin, a.bs));
                    it.h = qc.loc.h;
                }
            } else if (stats_ok) {
                it.kind = 0;
                it.w = sc.w;
                it.m = sc.m;
            } else {
                return false;
            }
            const WinLoc &l = it.kind == 0 ? sc.loc : qc.loc;
            it.t0 = l.wi * kWin;
            it.cnt = min(kWin, l.L - it.t0);
            if (it.kind != 2 && lane == 0) {
                fence_proxy_async_smem();  // the slot's earlier reads come before the copy
                load_window(ring + slot * kWinBytes, full + slot, a.src, l.b, l.h, l.c0, it.t0,
                            it.kind == 1 ? pol_quant : pol_stats, a.hdr);
            }
            if (it.kind == 0) {
                advance(sc, false);
                it.next_m = sc.w >= 0 ? sc.m : M;
            } else {
                advance(qc, true);
                it.next_m = qc.w >= 0 ? qc.m : M;
            }
            return true;
        };

        uint32_t phase = 0;  // bit s: parity of ring slot s's next completion
        // Wait for the window in ring slot `slot` and compute on it.
        auto process = [&](Item &it, int slot) {
            if (it.kind != 2) {
                if (!mbar_wait_bounded(full + slot, (phase >> slot) & 1u)) {
                    record_error(a.hdr, kErrBarrierWait);
                    if (lane == 0) st_release_cta_shared(&ctl->abort, 1);
                    it.kind = it.kind == 0 ? 3 : 2;  // skip the arithmetic, keep the progress
                }
                phase ^= 1u << slot;
            }
            const uint32_t kt = ring + slot * kWinBytes, vt = kt + kTileBytes;
            if (it.kind == 0) {
                const WinStats s = window_stats(kt, vt, it.cnt);
                if (lane == 0) {
                    __stcg(a.win_mean + it.w, s.mean);
                    __stcg(a.win_mm + it.w, make_float4(s.kmn, s.kmx, s.vmn, s.vmx));
                    uint32_t *g = reinterpret_cast<uint32_t *>(a.agg + it.w / kAgg);
                    atomicMax(g + 0, ~ord_enc(s.kmn));
                    atomicMax(g + 1, ord_enc(s.kmx));
                    atomicMax(g + 2, ~ord_enc(s.vmn));
                    atomicMax(g + 3, ord_enc(s.vmx));
                }
            } else if (it.kind == 1) {
                if ((uint32_t)it.blk < (uint32_t)a.num_blocks)
                    window_quant(a.kpool, a.vpool, a.Hkv, a.bs, it.h, it.t0, it.cnt, it.blk, kt, vt, it.pc);
                else if (lane == 0)  // not a block of the pools: flagged, nothing written
                    record_error(a.hdr, kErrBadBlock);
            }
            __syncwarp();  // the slot's reads are done before it is refilled
            if (lane == 0 && it.next_m != it.m) {
                if (it.kind == 0 || it.kind == 3) st_release_cta_shared(ctl->stats_done + warp, it.next_m);
                else st_release_cta_shared(ctl->quant_done + warp, it.next_m);
            }
        };

        // Windows in flight, oldest first: slots are used in turn, so the slot of the next copy
        // is always the one the oldest window frees.  One inlined copy of process() (the window
        // arithmetic is long): two copies measured a third more instruction-fetch stalls.
        Item f0, f1;
        int nin = 0, next_slot = 0;
        uint32_t spins = 0;
        while (true) {
            if (nin == 0 && try_issue(f0, next_slot)) {
                nin = 1;
                next_slot ^= 1;
            }
            if (nin == 1 && try_issue(f1, next_slot)) {
                nin = 2;
                next_slot ^= 1;
            }
            if (nin > 0) {
                spins = 0;
                process(f0, f0.slot);
                f0 = f1;
                --nin;
                continue;
            }
            if (sc.w < 0 && qc.w < 0) break;
            // blocked on the parameters of range qc.m
            if (++spins >= kSpinLimit) {
                record_error(a.hdr, kErrBarrierWait);
                if (lane == 0) st_release_cta_shared(&ctl->abort, 1);
                spins = 0;
            }
            __nanosleep(64);
        }
    }

    __syncthreads();
    if (tid == 0) {
        __threadfence();
        const uint32_t old = atomicAdd(&a.hdr->done_ctas, 1u);
        ctl->last = (old == (uint32_t)ncta - 1u);  // last CTA of the call
    }
    __syncthreads();
    if (ctl->last) {
        __threadfence();
        // clear the min/max aggregates and the progress words for the next call
        const int32_t nagg = (Wtot + kAgg - 1) / kAgg;
        for (int32_t i = tid; i < nagg; i += kThreads) a.agg[i] = make_uint4(0, 0, 0, 0);
        for (int32_t i = tid; i < ncta; i += kThreads) a.prog[i] = 0;
        if (tid == 0) a.hdr->done_ctas = 0;
        __threadfence();
    }
}

}  // namespace dgq

// ---- host launcher (called from dgq_host.cu after argument checks) ---------------------

namespace dgq {

static inline size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

// Pairs that can overlap one CTA's share of a quantisation range: a range holds at most
// kChunkMax + (windows of the longest pair) - 1 windows, and a share of n windows overlaps at
// most n + 1 pairs.
static int32_t params_cap(int32_t max_seqlen, int nsm)
{
    const int64_t wpair = (max_seqlen + kWin - 1) / kWin;
    return (int32_t)((kChunkMax + wpair + nsm - 1) / nsm + 2);
}

// The layout does not depend on the SM count: nsm * params_cap(.., nsm) is at most
// kChunkMax + wpair + 3 * nsm pairs for any nsm <= kMaxSms.
CompressLayout compress_layout(int32_t batch, int32_t max_seqlen, int32_t Hkv)
{
    CompressLayout l;
    const size_t P = (size_t)batch * Hkv;
    const size_t wpair = (size_t)((max_seqlen + kWin - 1) / kWin);
    const size_t Wmax = P * wpair;
    size_t off = sizeof(WsHeader);
    l.off_prog = off; off = align256(off + kMaxSms * 4);
    l.off_params = off; off = align256(off + 2 * (kChunkMax + wpair + 3 * kMaxSms) * sizeof(PairParams));
    l.off_mean = off; off = align256(off + (Wmax + 4) * 4);  // +4: quad reads past the end
    l.off_mm = off; off = align256(off + Wmax * 16);
    l.off_agg = off; off = align256(off + (Wmax / kAgg + 1) * 16);
    l.total = off;
    return l;
}

// + 1024: slack to start the rings on a 1024-byte boundary
static size_t compress_smem_bytes(int32_t B)
{
    return 1024 + (size_t)kRingBytes + sizeof(CtaCtl) + (size_t)(B + 1) * 4;
}

cudaError_t launch_compress(const SourceDesc &src, const int32_t *cu, int32_t B,
                            int32_t max_seqlen, int32_t Hkv, int32_t bs, const int32_t *bt, int32_t max_blocks,
                            uint8_t *kpool, uint8_t *vpool, int32_t num_blocks, dgq_seg_record *table, void *ws,
                            GroupSettings gs, int nsm, cudaStream_t stream)
{
    if (nsm > kMaxSms) return cudaErrorInvalidConfiguration;
    const CompressLayout l = compress_layout(B, max_seqlen, Hkv);
    char *base = static_cast<char *>(ws);
    CompressArgs a;
    if (!encode_tile_source(src, Hkv, bs, &a.src)) return cudaErrorInvalidValue;
    a.cu = cu;
    a.bt = bt;
    a.kpool = kpool;
    a.vpool = vpool;
    a.table = table;
    a.hdr = reinterpret_cast<WsHeader *>(base);
    a.prog = reinterpret_cast<uint32_t *>(base + l.off_prog);
    a.params = reinterpret_cast<PairParams *>(base + l.off_params);
    a.win_mean = reinterpret_cast<float *>(base + l.off_mean);
    a.win_mm = reinterpret_cast<float4 *>(base + l.off_mm);
    a.agg = reinterpret_cast<uint4 *>(base + l.off_agg);
    a.B = B;
    a.Hkv = Hkv;
    a.bs = bs;
    a.max_blocks = max_blocks;
    a.cap = params_cap(max_seqlen, nsm);
    a.max_seqlen = max_seqlen;
    a.num_blocks = num_blocks;
    a.max_groups = gs.max_groups;
    {
        const int32_t wpair = (max_seqlen + kWin - 1) / kWin;
        a.chunk = 4 * wpair > kChunkMin ? (4 * wpair < kChunkMax ? 4 * wpair : kChunkMax) : kChunkMin;
        a.ahead = 3 * a.chunk > 65536 ? 3 * a.chunk : 65536;
    }
    a.min_var = gs.min_var;

    // per-device launch set-up, done once per (device, shared-memory size) and host thread; the
    // kernel's shared-memory limit is raised to what the largest call needs (the same value from
    // every host thread, so none lowers it under another)
    static thread_local int cached_dev = -1;
    static thread_local size_t cached_smem = 0;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const size_t smem = compress_smem_bytes(B);
    if (dev != cached_dev || smem != cached_smem) {
        e = cudaFuncSetAttribute(compress_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)compress_smem_bytes(kMaxCallBatch));
        if (e != cudaSuccess) return e;
        int occ = 0;
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, compress_kernel, kThreads, smem);
        if (e != cudaSuccess) return e;
        if (occ < 1) return cudaErrorInvalidConfiguration;
        cached_dev = dev;
        cached_smem = smem;
    }
    dim3 grid(nsm), block(kThreads);  // one CTA per SM, all resident (cooperative launch)
    void *args[] = {&a};
    return cudaLaunchCooperativeKernel((const void *)compress_kernel, grid, block, args, smem, stream);
}

}  // namespace dgq
