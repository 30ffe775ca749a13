// dgq_compress_cluster.cu -- DGQ encode of one layer for requests of at most 4096 tokens
// (sm_103a), on thread-block clusters.
//
// Method: as in dgq_compress.cu ("DeepSeek KV-cache dynamic group quantisation (DGQ)" article,
// sections 2.2, 3.2; paged storage per "PagedAttention implementation", DeepSeek-V4 KV-cache
// article).  Same arithmetic (dgq_window.cuh), same outputs bit for bit.
//
// GPU design.  When every (request, KV head) pair is short (at most 256 windows, 1 MB of bf16
// K+V), a pair's segmentation needs no grid-wide step: clusters of kCl CTAs take whole pairs
// round-robin, and the kCl CTAs of a cluster split each pair's windows.
//  * Workers (per-warp two-window rings filled by TMA, as in the grid-wide kernel) compute
//    window statistics and send them straight into the shared memory of the pair's owner CTA
//    (owners rotate through the cluster) with asynchronous remote stores that complete bytes on
//    the owner's mbarrier (st.async ... mbarrier::complete_tx); the owner arms that barrier with
//    the pair's byte count.  Every worker also arrives on that barrier once it is done with the
//    pair's statistics (even with no window of the pair), so a phase completes only after every
//    worker has moved past the pair and so has taken the parameters of the pair that last used
//    the slot; that arrival is relaxed, as it publishes no data.  Measured on this GPU, a
//    cluster-scope release arrive per worker and pair (the data in the worker's own shared
//    memory) waited for the worker's outstanding code stores and cost 5-6% of the kernel.
//  * The owner's segmentation warp reads the pair's statistics from its own shared memory,
//    segments the pair, writes the record, stores the quantiser parameters into every CTA of
//    the cluster and arrives on each CTA's "ready" mbarrier.  No step goes through L2 or a grid
//    barrier.
//  * Workers quantise a pair once its parameters are ready, re-reading its K/V (read a few
//    microseconds earlier, so from L2; the re-read carries an evict-first hint and takes the
//    CTA's windows in the reverse of their first-read order), and meanwhile
//    compute statistics of the next pair (kSlots - 1 later pairs; with clusters of 2 at most two
//    windows per worker of it, see stats_ahead): a cluster holds at most kSlots pairs (2 MB)
//    between first read and re-read, the whole GPU about 70 MB.
//  * Twelve workers and one segmentation warp per CTA (127 registers a thread): measured on
//    this GPU, 12 workers with 2 pair slots took 104 us per layer of the Llama-3-8B batch-32
//    workload where 10 workers with 3 slots took 120 us.
//  * Clusters of 4 or 2 CTAs (not 8: measured on this GPU, only 15 clusters of 8 CTAs fit at
//    once, 120 of 152 SMs; 36 of 4, 144 SMs; 76 of 2, all 152).  Measured per layer: the
//    Llama-3-8B batch (256 pairs of 128 windows) 105 us with clusters of 4 and 118 us with
//    clusters of 2 (the last round of pairs leaves more of the GPU idle); the MHA batch (3200
//    pairs of 16-128 windows) 743 us with 4 and 639 us with 2 (more, smaller clusters; each CTA
//    gets a larger share of a short pair).  Calls with at least kManyPairs pairs take clusters
//    of 2.
// Every wait is bounded; a timeout records an error in the workspace header and the CTA skips
// dependent work.
#include "dgq_device.cuh"
#include "dgq.h"
#include "dgq_launch.h"
#include "dgq_window.cuh"

#include <stdint.h>

namespace dgq {

constexpr int32_t kManyPairs = 1024;                     // from this many pairs on: clusters of 2
constexpr int kCWorkers = 12;                            // worker warps per CTA (plus a segmentation warp)
constexpr int kCThreads = (kCWorkers + 1) * 32;
constexpr int kCRing = 2;                                // windows in flight per worker
static_assert(kCRing == 2, "the worker loop alternates two ring slots");
constexpr int kCRingBytes = kCWorkers * kCRing * kWinBytes;
constexpr int kSlots = 2;                                // pairs a cluster holds at once
constexpr int32_t kClusterMaxWin = 256;                  // pairs of at most 256 windows (4096 tokens)

// Statistics of the next pair run at most this many windows per worker ahead of the pair being
// quantised.  Clusters of 2 (calls with many pairs, mostly short: DRAM-bound) keep the read-ahead
// short so that more of the quantisation's re-read still finds its windows in L2 (measured on the
// MHA batch, per layer: 579 us without a cap, 561 with 2 windows, 566 with 3, 595 with 1).
// Clusters of 4 (few long pairs: latency-bound) need the read-ahead to cover segmentation and
// take no cap (2 windows measured 13% slower on the Llama-shaped batch).
template <int kCl>
__host__ __device__ constexpr int32_t stats_ahead() { return kCl == 2 ? 2 : kClusterMaxWin; }
static_assert(kClusterMaxWin == 8 * 32, "segment_small holds 8 windows per lane");

struct ClusterArgs {
    TileSource src;  // where the K and V window tiles come from
    const int32_t *cu;
    const int32_t *bt;
    uint8_t *kpool;
    uint8_t *vpool;
    dgq_seg_record *table;
    WsHeader *hdr;
    int32_t B, Hkv, bs, max_blocks;
    int32_t max_groups;  // group-selection settings
    float min_var;
    int32_t max_seqlen, num_blocks;  // for the device-side checks of lengths and block ids
};

struct ClusterSmem {
    float mean[kSlots][kClusterMaxWin];  // owner side: statistics of every window of an owned pair
    float4 mm[kSlots][kClusterMaxWin];
    PairParams par[kSlots];
    uint64_t stats_done[kSlots];  // owner side: the pair's statistics have all landed (byte count)
    uint64_t ready[kSlots];       // parameters of the slot's pair are in par[]
    uint64_t full[kCWorkers][kCRing];  // a worker's ring slot holds its window
    int32_t abort;
    int32_t pad[3];
};

// ---- cluster helpers (inline PTX) ------------------------------------------------------------

__device__ __forceinline__ uint32_t cluster_rank()
{
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}
__device__ __forceinline__ uint32_t cluster_id()
{
    uint32_t r;
    asm volatile("mov.u32 %0, %%clusterid.x;" : "=r"(r));
    return r;
}
__device__ __forceinline__ uint32_t cluster_count()
{
    uint32_t r;
    asm volatile("mov.u32 %0, %%nclusterid.x;" : "=r"(r));
    return r;
}
// shared-memory address of the same variable in CTA `rank` of the cluster
__device__ __forceinline__ uint32_t map_rank(const void *p, uint32_t rank)
{
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(smem_u32(p)), "r"(rank));
    return r;
}
__device__ __forceinline__ bool try_wait_cluster(uint64_t *bar, uint32_t parity)
{
    uint32_t ok;
    asm volatile(
        "{\n.reg .pred p;\nmbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\nselp.u32 %0, 1, 0, p;\n}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}
// non-blocking test (try_wait may suspend the thread for a while when the phase is open)
__device__ __forceinline__ bool test_wait_cluster(uint64_t *bar, uint32_t parity)
{
    uint32_t ok;
    asm volatile(
        "{\n.reg .pred p;\nmbarrier.test_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\nselp.u32 %0, 1, 0, p;\n}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}
// Asynchronous stores into another CTA's shared memory, each completing its bytes on an mbarrier
// of that CTA (both addresses from mapa).  They need no fence: the owner observes them through
// the barrier's phase.
__device__ __forceinline__ void st_async_f32(uint32_t addr, float v, uint32_t bar)
{
    asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.b32 [%0], %1, [%2];" ::"r"(addr),
                 "r"(__float_as_uint(v)), "r"(bar)
                 : "memory");
}
__device__ __forceinline__ void st_async_f4(uint32_t addr, float4 v, uint32_t bar)
{
    asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.v4.b32 [%0], {%1, %2, %3, %4}, [%5];" ::"r"(
                     addr),
                 "r"(__float_as_uint(v.x)), "r"(__float_as_uint(v.y)), "r"(__float_as_uint(v.z)),
                 "r"(__float_as_uint(v.w)), "r"(bar)
                 : "memory");
}
// Arrival without release on another CTA's mbarrier: a worker tells the owner that it is done
// with a pair's statistics (its data travel by st.async and complete on their own).
__device__ __forceinline__ void remote_arrive_relaxed(uint32_t bar)
{
    asm volatile("mbarrier.arrive.relaxed.cluster.shared::cluster.b64 _, [%0];" ::"r"(bar) : "memory");
}
// Arrival on another CTA's mbarrier that also announces bytes still to come by st.async (no
// release: the bytes themselves complete the phase).
__device__ __forceinline__ void remote_arrive_expect_tx(uint32_t bar, uint32_t bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.relaxed.cluster.shared::cluster.b64 _, [%0], %1;" ::"r"(bar),
                 "r"(bytes)
                 : "memory");
}
// The owner arms its statistics barrier: its own arrival and the bytes to expect (no release:
// it publishes nothing).
__device__ __forceinline__ void arm_expect_tx(uint64_t *bar, uint32_t bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.relaxed.cta.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
                 : "memory");
}
constexpr uint32_t kStatBytes = 4 + 16;  // per window: mean (fp32) and extremes (float4)

__device__ __forceinline__ void cluster_sync_all()
{
    asm volatile("barrier.cluster.arrive.release.aligned;\nbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// Quantiser parameters of one pair from this CTA's shared memory: lane i < 5 gets segment i's.
__device__ __forceinline__ PairCache load_params_smem(const PairParams *pp)
{
    const int lane = threadIdx.x & 31;
    const int i = lane < kMaxSeg ? lane : 0;
    PairCache pc;
    pc.start = pp->start[i];
    pc.kmn = pp->k_min[i];
    pc.kinv = pp->k_inv[i];
    pc.vmn = pp->v_min[i];
    pc.vinv = pp->v_inv[i];
    return pc;
}

// Windows [lo, hi) of a pair of W windows held by CTA `r` of a cluster of kCl CTAs.
template <int kCl>
__device__ __forceinline__ void cta_range(int32_t W, int32_t r, int32_t &lo, int32_t &hi)
{
    lo = (W * r) / kCl;
    hi = (W * (r + 1)) / kCl;
}

// ---- the kernel ---------------------------------------------------------------------------

// A worker's position in the cluster's pair sequence j = 0, 1, ... (pair p = cluster + j *
// clusters) for one of its two item sequences: window i of its CTA's range [lo, hi).
struct PairCursor {
    int32_t j, i, lo, hi;
    int32_t L, c0, h, b;
};

struct CItem {
    int32_t kind;  // 0 statistics, 1 quantisation, 2 nothing to do (after an error)
    int32_t j, idx, cnt, t0, h, blk, slot;
    bool last;     // statistics: the worker's last window of pair j
    PairCache pc;
};

template <int kCl>
__global__ void __launch_bounds__(kCThreads, 1) compress_cluster_kernel(const __grid_constant__ ClusterArgs a)
{
    extern __shared__ __align__(16) uint8_t smem_raw[];
    uint8_t *smem = align_smem_1024(smem_raw);  // window tiles start on 1024-byte boundaries
    ClusterSmem *cs = reinterpret_cast<ClusterSmem *>(smem + kCRingBytes);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int32_t rank = (int32_t)cluster_rank();
    const int32_t clu = (int32_t)cluster_id(), ncl = (int32_t)cluster_count();
    const int32_t P = a.B * a.Hkv;
    const int32_t nj = clu < P ? (P - clu + ncl - 1) / ncl : 0;  // pairs of this cluster

    if (tid == 0) {
        for (int s = 0; s < kSlots; ++s) {
            // every worker of the cluster and the owner arrive; the workers' bytes complete too
            mbar_init(&cs->stats_done[s], kCl * kCWorkers + 1);
            mbar_init(&cs->ready[s], 1);
        }
        for (int w = 0; w < kCWorkers; ++w)
            for (int r = 0; r < kCRing; ++r) mbar_init(&cs->full[w][r], 1);
        cs->abort = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    cluster_sync_all();  // every CTA's barriers exist before any remote arrive
    if (blockIdx.x == 0 && tid == 0) a.hdr->path = kPathClusterWhole;

    // Request offsets of the cluster's pairs, fetched 32 pairs at a time (lane i: pair jb + i) so
    // that a warp moving to its next pair does not wait for two dependent global loads.
    struct PairGeo {
        int32_t jb, c0, L;
    };
    auto geo_fetch = [&](PairGeo &g, int32_t jb) {
        g.jb = jb;
        g.c0 = 0;
        g.L = 0;
        if (jb + lane < nj) {
            const int32_t b = (clu + (jb + lane) * ncl) / a.Hkv;
            g.c0 = __ldg(a.cu + b);
            g.L = __ldg(a.cu + b + 1) - g.c0;
        }
    };
    auto pair_of = [&](int32_t j, PairCursor &c, PairGeo &g) {
        if (j - g.jb >= 32) geo_fetch(g, j);  // pairs are visited in increasing order
        const int32_t p = clu + j * ncl;
        c.b = p / a.Hkv;
        c.h = p - c.b * a.Hkv;
        c.c0 = __shfl_sync(0xffffffffu, g.c0, j - g.jb);
        c.L = __shfl_sync(0xffffffffu, g.L, j - g.jb);
        if (c.L < 0 || c.L > a.max_seqlen) {  // longer than the call's sizes allow: flagged, skipped
            if (lane == 0) record_error(a.hdr, kErrBadLength);
            c.L = 0;
        }
        cta_range<kCl>((c.L + kWin - 1) / kWin, rank, c.lo, c.hi);
    };
    auto aborted = [&]() { return *reinterpret_cast<volatile int32_t *>(&cs->abort) != 0; };

    if (warp == kCWorkers) {
        // ================================================================ segmentation warp
        // Pairs j = rank, rank + kCl, ... are owned by this CTA.
        PairGeo geo;
        geo_fetch(geo, 0);
        for (int32_t q = 0; q * kCl + rank < nj; ++q) {
            const int32_t j = q * kCl + rank;
            const int32_t qs = q % kSlots;
            PairCursor pc;
            pair_of(j, pc, geo);
            const int32_t W = (pc.L + kWin - 1) / kWin;
            if (lane == 0) arm_expect_tx(&cs->stats_done[qs], (uint32_t)W * kStatBytes);
            bool ok = true;
            for (uint32_t it = 0; !try_wait_cluster(&cs->stats_done[qs], (uint32_t)(q / kSlots) & 1u);) {
                if (++it >= kSpinLimit || aborted()) {
                    ok = false;
                    break;
                }
                __nanosleep(32);
            }
            if (!ok) {
                if (lane == 0) {
                    record_error(a.hdr, kErrBarrierWait);
                    st_release_cta_shared(&cs->abort, 1);
                }
                break;
            }
            const int32_t p = clu + j * ncl;
            const int slot = j % kSlots;
            dgq_seg_record rec = {};
            PairParams pp = {};
            if (W > 0) {
                // the pair's window statistics, sent here by the cluster's workers; lane i holds
                // windows 8i .. 8i+7
                float m[8];
                float4 mm[8];
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    const int32_t w = 8 * lane + i;
                    m[i] = 0.0f;
                    mm[i] = make_float4(INFINITY, -INFINITY, INFINITY, -INFINITY);
                    if (w < W) {
                        m[i] = cs->mean[qs][w];
                        mm[i] = cs->mm[qs][w];
                    }
                }
                int k = min(min(ngroups(pc.L), a.max_groups), W) - 1;
                int32_t cut[4];
                float kmn[kMaxSeg], kmx[kMaxSeg], vmn[kMaxSeg], vmx[kMaxSeg];
                k = segment_small(W, k, a.min_var, m, mm, cut, kmn, kmx, vmn, vmx);
                make_params(pc.L, k, cut, kmn, kmx, vmn, vmx, rec, pp);  // same values in every lane
            }
            if (lane == 0) a.table[p] = rec;
            // parameters into every CTA of the cluster (lane r < kCl serves CTA r): the arrival on
            // its "ready" barrier announces 128 bytes, which the asynchronous stores complete
            if (lane < kCl) {
                const uint4 *src = reinterpret_cast<const uint4 *>(&pp);
                const uint32_t dst = map_rank(&cs->par[slot], (uint32_t)lane);
                const uint32_t bar = map_rank(&cs->ready[slot], (uint32_t)lane);
                remote_arrive_expect_tx(bar, (uint32_t)sizeof(PairParams));
#pragma unroll
                for (int i = 0; i < 8; ++i)
                    st_async_f4(dst + 16 * i, make_float4(__uint_as_float(src[i].x), __uint_as_float(src[i].y),
                                                          __uint_as_float(src[i].z), __uint_as_float(src[i].w)),
                                bar);
            }
            __syncwarp();
        }
    } else {
        // ================================================================ worker warps
        const uint32_t ring = smem_u32(smem) + warp * (kCRing * kWinBytes);
        uint64_t *full = cs->full[warp];
        const uint64_t pol_stats = make_policy_evict_normal();
        const uint64_t pol_quant = make_policy_evict_first();  // second read: last use

        // position a cursor on pair j (windows lo + warp, + kCWorkers, ...); i >= hi: none here
        PairGeo sgeo, qgeo;  // one per cursor
        geo_fetch(sgeo, 0);
        qgeo = sgeo;
        auto start_pair = [&](PairCursor &c, PairGeo &g, int32_t j) {
            c.j = j;
            if (j < nj) {
                pair_of(j, c, g);
                c.i = c.lo + warp;
            }
        };
        // the arrival a worker owes pair j's owner once it is done with pair j's statistics
        auto arrive_stats = [&](int32_t j) {
            if (lane == 0) {
                const int32_t q = j / kCl;
                remote_arrive_relaxed(map_rank(&cs->stats_done[q % kSlots], (uint32_t)(j % kCl)));
            }
        };

        PairCursor sc, qc;
        start_pair(sc, sgeo, 0);
        start_pair(qc, qgeo, 0);
        int32_t pc_j = -1;
        PairCache params = {0, 0.0f, 0.0f, 0.0f, 0.0f};

        // Choose the next item and start its copy into ring slot `slot`; false when nothing may
        // start now.
        auto try_issue = [&](CItem &it, int slot) -> bool {
            it.slot = slot;
            // quantisation: pairs whose parameters are ready (pairs with no window here are passed
            // once ready, so that their statistics slot may be reused)
            while (qc.j < nj) {
                const bool ab = aborted();
                if (!ab && !test_wait_cluster(&cs->ready[qc.j % kSlots], (uint32_t)(qc.j / kSlots) & 1u)) break;
                if (qc.i >= qc.hi) {
                    start_pair(qc, qgeo, qc.j + 1);
                    continue;
                }
                it.kind = ab ? 2 : 1;
                it.j = qc.j;
                // the CTA's windows of the pair are re-read last-read first, while they are the
                // likeliest still to be in L2 (measured 1.4% faster on the MHA batch)
                it.t0 = (qc.lo + qc.hi - 1 - qc.i) * kWin;
                it.cnt = min(kWin, qc.L - it.t0);
                it.h = qc.h;
                if (!ab) {
                    if (pc_j != qc.j) {
                        params = load_params_smem(&cs->par[qc.j % kSlots]);
                        pc_j = qc.j;
                    }
                    it.pc = params;
                    it.blk = __ldg(a.bt + (int64_t)qc.b * a.max_blocks + pow2_div(it.t0, a.bs));
                    if (lane == 0) {
                        fence_proxy_async_smem();  // the slot's earlier reads come before the copy
                        load_window(ring + slot * kWinBytes, full + slot, a.src, qc.b, qc.h, qc.c0, it.t0,
                                    pol_quant, a.hdr);
                    }
                }
                qc.i += kCWorkers;
                return true;
            }
            // statistics: at most kSlots - 1 pairs past the oldest pair still to quantise
            while (sc.j < nj && sc.j < qc.j + kSlots) {
                if (sc.i >= sc.hi) {  // nothing (more) of this pair for this worker
                    if (sc.i == sc.lo + warp) arrive_stats(sc.j);  // it had no window at all
                    start_pair(sc, sgeo, sc.j + 1);
                    continue;
                }
                if (sc.j > qc.j && sc.i >= sc.lo + warp + stats_ahead<kCl>() * kCWorkers)
                    return false;  // far enough ahead: quantisation of pair qc.j comes first
                it.kind = 0;
                it.j = sc.j;
                it.idx = sc.i;  // window within the pair
                it.t0 = sc.i * kWin;
                it.cnt = min(kWin, sc.L - it.t0);
                it.last = sc.i + kCWorkers >= sc.hi;
                if (lane == 0) {
                    fence_proxy_async_smem();
                    load_window(ring + slot * kWinBytes, full + slot, a.src, sc.b, sc.h, sc.c0, it.t0, pol_stats,
                                a.hdr);
                }
                sc.i += kCWorkers;
                return true;
            }
            return false;
        };

        uint32_t phase = 0;  // bit s: parity of ring slot s's next completion
        // Wait for the window in ring slot `slot` and compute on it.
        auto process = [&](CItem &it, int slot) {
            if (it.kind != 2) {
                if (!mbar_wait_bounded(full + slot, (phase >> slot) & 1u)) {
                    if (lane == 0) {
                        record_error(a.hdr, kErrBarrierWait);
                        st_release_cta_shared(&cs->abort, 1);
                    }
                    it.kind = 2;
                }
                phase ^= 1u << slot;
            }
            const uint32_t kt = ring + slot * kWinBytes, vt = kt + kTileBytes;
            if (it.kind == 0) {
                const WinStats s = window_stats(kt, vt, it.cnt);
                if (lane == 0) {  // into the owner's shared memory, completing bytes on its barrier
                    const uint32_t owner = (uint32_t)(it.j % kCl);
                    const int qs = (it.j / kCl) % kSlots;
                    const uint32_t bar = map_rank(&cs->stats_done[qs], owner);
                    st_async_f32(map_rank(&cs->mean[qs][it.idx], owner), s.mean, bar);
                    st_async_f4(map_rank(&cs->mm[qs][it.idx], owner), make_float4(s.kmn, s.kmx, s.vmn, s.vmx), bar);
                }
                if (it.last) arrive_stats(it.j);
            } else if (it.kind == 1) {
                if ((uint32_t)it.blk < (uint32_t)a.num_blocks)
                    window_quant(a.kpool, a.vpool, a.Hkv, a.bs, it.h, it.t0, it.cnt, it.blk, kt, vt, it.pc);
                else if (lane == 0)  // not a block of the pools: flagged, nothing written
                    record_error(a.hdr, kErrBadBlock);
            }
            __syncwarp();  // the slot's reads are done before it is refilled
        };

        // Windows in flight, oldest first: slots are used in turn, so the slot of the next copy
        // is always the one the oldest window frees.  One inlined copy of process() (the window
        // arithmetic is long): two copies measured a third more instruction-fetch stalls.
        CItem f0, f1;
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
            if (sc.j >= nj && qc.j >= nj) break;
            if (++spins >= kSpinLimit) {  // waiting for parameters that never came
                if (lane == 0) {
                    record_error(a.hdr, kErrBarrierWait);
                    st_release_cta_shared(&cs->abort, 1);
                }
                spins = 0;
            }
            __nanosleep(32);
        }
    }
    cluster_sync_all();  // no CTA leaves while others may still reach its shared memory
}

// ---- host launcher -------------------------------------------------------------------------

int32_t cluster_compress_max_seqlen() { return kClusterMaxWin * kWin; }

template <int kCl>
static cudaError_t launch_cluster_size(const ClusterArgs &a, cudaStream_t stream)
{
    const size_t smem = 1024 + (size_t)kCRingBytes + sizeof(ClusterSmem);  // + alignment slack
    static thread_local int cached_dev = -1, cached_clusters = 0;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = kCl;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.blockDim = dim3(kCThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (dev != cached_dev) {
        e = cudaFuncSetAttribute(compress_cluster_kernel<kCl>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
        int nsm = 0;
        e = cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev);
        if (e != cudaSuccess) return e;
        cfg.gridDim = dim3((unsigned)(nsm / kCl * kCl));
        int nclusters = 0;  // clusters that fit on the GPU at once (GPC boundaries)
        e = cudaOccupancyMaxActiveClusters(&nclusters, compress_cluster_kernel<kCl>, &cfg);
        if (e != cudaSuccess) return e;
        if (nclusters < 1) return cudaErrorInvalidConfiguration;
        cached_dev = dev;
        cached_clusters = nclusters;
    }
    cfg.gridDim = dim3((unsigned)(cached_clusters * kCl));  // one wave: every cluster resident
    return cudaLaunchKernelEx(&cfg, compress_cluster_kernel<kCl>, a);
}

cudaError_t launch_compress_cluster(const SourceDesc &src, const int32_t *cu, int32_t B,
                                    int32_t max_seqlen, int32_t Hkv, int32_t bs, const int32_t *bt,
                                    int32_t max_blocks, uint8_t *kpool, uint8_t *vpool, int32_t num_blocks,
                                    dgq_seg_record *table, void *ws, GroupSettings gs, cudaStream_t stream)
{
    ClusterArgs a;
    if (!encode_tile_source(src, Hkv, bs, &a.src)) return cudaErrorInvalidValue;
    a.cu = cu;
    a.bt = bt;
    a.kpool = kpool;
    a.vpool = vpool;
    a.table = table;
    a.hdr = static_cast<WsHeader *>(ws);
    a.B = B;
    a.Hkv = Hkv;
    a.bs = bs;
    a.max_blocks = max_blocks;
    a.max_groups = gs.max_groups;
    a.min_var = gs.min_var;
    a.max_seqlen = max_seqlen;
    a.num_blocks = num_blocks;
    return (int64_t)B * Hkv >= kManyPairs ? launch_cluster_size<2>(a, stream) : launch_cluster_size<4>(a, stream);
}

}  // namespace dgq
