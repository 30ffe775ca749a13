// dgq_attn.cu -- decode-step GQA attention over the DGQ INT8 paged cache (sm_103a).
//
// Method: scores q . x_K / sqrt(D) over the cached tokens, whose keys/values are
// dequantised per segment (x = min + q * scale, segment looked up per token: "DeepSeek
// KV-cache dynamic group quantisation (DGQ)" article, section 2.2; dequantisation on the
// GPU: section 3.2), gathered through the block table ("PagedAttention implementation",
// DeepSeek-V4 KV-cache article), plus the current token's own bf16 key/value.
//
// GPU design.
//  * Work space: every (request, KV head) pair is cut into 64-token chunks; all chunks of
//    all pairs form one flat list, and each persistent CTA takes an equal contiguous slice
//    of it (a pair may span several CTAs, a CTA may cover several pairs).  A CTA's run of
//    chunks of one pair is a "piece"; pieces are merged per pair by the CTA that finishes
//    last, in CTA order (fixed, so results are bitwise reproducible on a given GPU).
//  * Pipeline: one producer warp issues TMA tiled copies (128-byte swizzle) of the uint8 K
//    and V blocks of each chunk into a 6-stage shared-memory ring (mbarrier complete_tx);
//    four consumer warps each take 16 tokens of a stage.
//  * Math: codes become fp16 (1024 + q) with one byte-permute per two codes, and the GQA
//    query group multiplies them on the tensor cores (mma.sync m16n8k16, fp32 accumulate):
//    S^T = Q . K^T (16 x 8 tokens per mma) and O^T += V^T . P^T.  The affine dequantisation
//    is folded out of the inner loop: for a tile inside segment s,
//      q . x_K = k_scale[s] * (q . (1024 + c)) + (k_min[s] - 1024 k_scale[s]) * sum(q),
//      sum_t p_t x_V = v_scale[s] * sum_t p_t (1024 + c_t) + (v_min[s] - 1024 v_scale[s]) sum p.
//    Segment starts are multiples of 16, so a 16-token tile never straddles two segments.
//  * Online softmax in the log2 domain with lazy rescaling (the running max moves only when
//    a tile's max exceeds it by more than 8, so p <= 256 stays exact enough in fp16).
#include "dgq_device.cuh"
#include "dgq.h"
#include "dgq_launch.h"

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <stdint.h>

namespace dgq {

constexpr int kChunk = 64;                      // tokens per pipeline stage
constexpr int kStages = 6;
constexpr int kConsumerWarps = 4;
constexpr int kAttnThreads = (kConsumerWarps + 1) * 32;
constexpr int kStageBytes = kChunk * kD;        // 8 KB per tensor per stage
constexpr int kPartStride = 132;                // floats per (piece, head) partial: m, l, O[128], pad
constexpr float kLog2eOverSqrtD = 0.12751743074570180f;  // log2(e) / sqrt(128)
constexpr float kLazyRescale = 8.0f;            // log2 units

struct AttnArgs {
    const uint16_t *q;
    const uint16_t *knew;
    const uint16_t *vnew;
    const dgq_seg_record *table;
    const int32_t *bt;
    const int32_t *seq_lens;
    uint16_t *out;
    WsHeader *hdr;
    uint32_t *pair_count;
    float *part;
    int32_t B, Hq, Hkv, G, bs, max_blocks;
};

// token order inside each 8-column n-tile: column n holds token kTau[n]; it keeps the rows a
// quarter-warp reads at the same time in different halves of the 128-byte swizzle pattern.
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
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint4 lds128(uint32_t addr) { return ld_shared_v4(addr); }

__device__ __forceinline__ uint32_t word(const uint4 &v, int i)
{
    return i == 0 ? v.x : (i == 1 ? v.y : (i == 2 ? v.z : v.w));
}

struct ChunkLoc {
    int32_t b, h, j, nch, L;
};

// Step a chunk cursor to the next chunk of the flat list (pairs in (request, head) order).
__device__ __forceinline__ void advance(ChunkLoc &c, const int32_t *s_len, int32_t Hkv)
{
    if (++c.j == c.nch) {
        c.j = 0;
        if (++c.h == Hkv) {
            c.h = 0;
            ++c.b;
            c.L = s_len[c.b];
            c.nch = max(1, (c.L + 63) / 64);
        }
    }
}

// 2^x on the MUFU unit (flush-to-zero); arguments here are <= 8 or -inf.
__device__ __forceinline__ float ex2(float x)
{
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

__device__ __forceinline__ ChunkLoc locate_chunk(int32_t x, const int32_t *s_cpre, const int32_t *s_len, int32_t B,
                                                 int32_t Hkv)
{
    int32_t lo = 0, hi = B - 1;
    while (lo < hi) {
        int32_t mid = (lo + hi + 1) >> 1;
        if (s_cpre[mid] <= x) lo = mid;
        else hi = mid - 1;
    }
    ChunkLoc c;
    c.b = lo;
    c.nch = (s_cpre[lo + 1] - s_cpre[lo]) / Hkv;
    int32_t off = x - s_cpre[lo];
    c.h = off / c.nch;
    c.j = off - c.h * c.nch;
    c.L = s_len[lo];
    return c;
}

// CTA owning flat chunk x when C chunks are split evenly over n CTAs
__device__ __forceinline__ int32_t owner(int32_t x, int32_t C, int32_t n)
{
    return (int32_t)((((int64_t)x + 1) * n - 1) / C);
}

// whether CTA c owns at least one chunk (with fewer chunks than CTAs, some own none)
__device__ __forceinline__ bool owns_chunks(int32_t c, int32_t C, int32_t n)
{
    return ((int64_t)(c + 1) * C) / n > ((int64_t)c * C) / n;
}

// Final softmax merge with the current token: (O + p_new v_new) / (L + p_new), where (M, L, O)
// are the cached tokens' max, sum and weighted value sum relative to M (log2 domain).
__device__ __forceinline__ uint16_t finish(float M, float L, float O, float s_new, float v_new)
{
    const float Mf = fmaxf(M, s_new);
    const float wo = (M == -INFINITY) ? 0.0f : exp2f(M - Mf);
    const float wn = exp2f(s_new - Mf);
    const float o = fmaf(O, wo, wn * v_new) / fmaf(L, wo, wn);
    __nv_bfloat16 ob = __float2bfloat16_rn(o);
    return *reinterpret_cast<uint16_t *>(&ob);
}

// Per-warp online-softmax state of the current piece.
struct WarpState {
    float m;      // running max (log2 domain) of head g = lane/4
    float l;      // partial sum of p over this lane's tokens
    float bsum;   // partial sum of (v_min - 1024 sigma) * p
    float sigma;  // V scale of the current (non-flat) segment: O = sigma * o + bsum
    int seg;      // current segment (-1 before the first tile)
    float o[8][4];
};

__global__ void __launch_bounds__(kAttnThreads, 2)
    attn_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV, AttnArgs a)
{
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = align_smem_1024(smem_raw);
    uint8_t *sK = smem;
    uint8_t *sV = smem + kStages * kStageBytes;
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + 2 * kStages * kStageBytes);
    uint64_t *empty = full + kStages;
    volatile int32_t *s_flag = reinterpret_cast<volatile int32_t *>(empty + kStages);  // [0] abort [1] last
    float *s_snew = reinterpret_cast<float *>(const_cast<int32_t *>(s_flag) + 4);      // [8]
    dgq_seg_record *s_rec = reinterpret_cast<dgq_seg_record *>(s_snew + 8);
    float *s_comb = reinterpret_cast<float *>(s_rec + 1);                               // [4][G][132]
    int32_t *s_cpre = reinterpret_cast<int32_t *>(s_comb + kConsumerWarps * a.G * kPartStride);  // [B+1]
    int32_t *s_len = s_cpre + (a.B + 1);                                                         // [B]

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int32_t B = a.B, Hkv = a.Hkv, G = a.G;

    if (tid == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], kConsumerWarps);
        }
        s_flag[0] = 0;
        s_flag[1] = 0;
        fence_barrier_init();
    }
    if (warp == 0) {  // exclusive scan of Hkv * max(1, ceil(L_b / 64))
        int32_t carry = 0;
        for (int base = 0; base < B; base += 32) {
            int i = base + lane;
            int32_t v = 0;
            if (i < B) {
                int32_t L = __ldg(a.seq_lens + i);
                s_len[i] = L;
                v = Hkv * max(1, (L + kChunk - 1) / kChunk);
            }
            int32_t x = v;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                int32_t y = __shfl_up_sync(0xffffffffu, x, o);
                if (lane >= o) x += y;
            }
            if (i < B) s_cpre[i] = carry + x - v;
            carry += __shfl_sync(0xffffffffu, x, 31);
        }
        if (lane == 0) s_cpre[B] = carry;
    }
    __syncthreads();

    const int32_t C = s_cpre[B];
    const int32_t ncta = gridDim.x, cta = blockIdx.x;
    const int32_t cbeg = (int32_t)(((int64_t)C * cta) / ncta);
    const int32_t cend = (int32_t)(((int64_t)C * (cta + 1)) / ncta);

    // ------------------------------------------------------------------ producer warp
    if (warp == kConsumerWarps) {
        if (lane == 0) {
            prefetch_tensormap(&tmK);
            prefetch_tensormap(&tmV);
            // Block ids of the next chunk are loaded one chunk ahead, so the table lookups overlap
            // the wait for a free stage instead of sitting between the wait and the copies.
            const int per_chunk = kChunk / a.bs;  // 1, 2 or 4 blocks
            auto fetch = [&](const ChunkLoc &c, int32_t *dst) {
                const int32_t nt = min(kChunk, c.L - kChunk * c.j);
                const int nblk = nt > 0 ? (nt + a.bs - 1) / a.bs : 0;
                const int32_t *btrow = a.bt + (int64_t)c.b * a.max_blocks + per_chunk * c.j;
#pragma unroll
                for (int i = 0; i < 4; ++i)
                    if (i < nblk) dst[i] = __ldg(btrow + i);
            };
            if (cbeg < cend) {
                ChunkLoc cur = locate_chunk(cbeg, s_cpre, s_len, B, Hkv);
                int32_t nxt[4] = {0, 0, 0, 0};
                fetch(cur, nxt);
                uint32_t it = 0;
                for (int32_t x = cbeg; x < cend; ++x) {
                    const ChunkLoc c = cur;
                    int32_t blk[4] = {nxt[0], nxt[1], nxt[2], nxt[3]};
                    if (x + 1 < cend) {
                        advance(cur, s_len, Hkv);
                        fetch(cur, nxt);
                    }
                    const int32_t nt = min(kChunk, c.L - kChunk * c.j);
                    if (nt <= 0) continue;
                    const int stage = it % kStages;
                    const uint32_t use = it / kStages;
                    if (use > 0 && !mbar_wait_bounded(&empty[stage], (use - 1) & 1)) {
                        record_error(a.hdr, kErrEmptyWait);
                        s_flag[0] = 1;
                        break;
                    }
                    if (s_flag[0]) break;
                    const int nblk = (nt + a.bs - 1) / a.bs;
                    mbar_arrive_expect_tx(&full[stage], (uint32_t)(nblk * a.bs * kD * 2));
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        if (i < nblk) {
                            const int32_t y = (blk[i] * Hkv + c.h) * a.bs;
                            tma_load_2d(sK + stage * kStageBytes + i * a.bs * kD, &tmK, 0, y, &full[stage]);
                            tma_load_2d(sV + stage * kStageBytes + i * a.bs * kD, &tmV, 0, y, &full[stage]);
                        }
                    }
                    ++it;
                }
            }
        }
        return;
    }

    // ------------------------------------------------------------------ consumer warps
    const int w = warp;                 // 0..3: tokens [16w, 16w+16) of each chunk
    const int r = lane >> 2, cq = lane & 3;
    const int tr = tau(r);              // 16-byte column (of 8) this lane reads from V rows
    const bool gvalid = r < G;          // this lane's softmax head
    const int ctid = tid;               // 0..127
    const uint32_t M64 = 0x64646464u;

    uint32_t qa0[8], qa2[8];
    float qsum = 0.0f;
    WarpState st;
    uint32_t it = 0;

    ChunkLoc cur;
    if (cbeg < cend) cur = locate_chunk(cbeg, s_cpre, s_len, B, Hkv);
    for (int32_t x = cbeg; x < cend; ++x) {
        const ChunkLoc c = cur;
        if (x + 1 < cend) advance(cur, s_len, Hkv);
        const int32_t p = c.b * Hkv + c.h;
        const bool first = (x == cbeg) || (c.j == 0);
        const bool last = (x == cend - 1) || (c.j == c.nch - 1);

        if (first) {
            named_bar_sync(1, kConsumerWarps * 32);
            if (ctid < 32) reinterpret_cast<uint32_t *>(s_rec)[ctid] = __ldg(reinterpret_cast<const uint32_t *>(a.table + p) + ctid);
            // Q fragments: head g = r, columns d = 16cq + 64(jj/4) + 4(jj%4) + {0,1 | 2,3}
            float qs = 0.0f;
            if (gvalid) {
                const uint16_t *qrow = a.q + ((int64_t)c.b * a.Hq + c.h * G + r) * kD;
#pragma unroll
                for (int half = 0; half < 2; ++half) {
                    const uint4 *src = reinterpret_cast<const uint4 *>(qrow + 16 * cq + 64 * half);
                    uint4 u0 = __ldg(src), u1 = __ldg(src + 1);
                    uint32_t wv[8] = {u0.x, u0.y, u0.z, u0.w, u1.x, u1.y, u1.z, u1.w};
#pragma unroll
                    for (int m = 0; m < 4; ++m) {
                        uint32_t h0 = bf16x2_to_f16x2(wv[2 * m]), h1 = bf16x2_to_f16x2(wv[2 * m + 1]);
                        qa0[4 * half + m] = h0;
                        qa2[4 * half + m] = h1;
                        qs += f16lo(h0) + f16hi(h0) + f16lo(h1) + f16hi(h1);
                    }
                }
            } else {
#pragma unroll
                for (int jj = 0; jj < 8; ++jj) qa0[jj] = qa2[jj] = 0u;
            }
            qs += __shfl_xor_sync(0xffffffffu, qs, 1);
            qs += __shfl_xor_sync(0xffffffffu, qs, 2);
            qsum = qs;
            st.m = -INFINITY;
            st.l = 0.0f;
            st.bsum = 0.0f;
            st.sigma = 1.0f;
            st.seg = -1;
#pragma unroll
            for (int i = 0; i < 8; ++i) st.o[i][0] = st.o[i][1] = st.o[i][2] = st.o[i][3] = 0.0f;
            named_bar_sync(1, kConsumerWarps * 32);
        }

        const int32_t nt = min(kChunk, c.L - kChunk * c.j);
        if (nt > 0 && !s_flag[0]) {
            const int stage = it % kStages;
            const uint32_t use = it / kStages;
            bool ok = mbar_wait_bounded(&full[stage], use & 1);
            if (!ok) {
                record_error(a.hdr, kErrFullWait);
                s_flag[0] = 1;
            }
            const int32_t t0 = kChunk * c.j + 16 * w;
            const int32_t valid = min(16, c.L - t0);
            if (ok && valid > 0) {
                const uint32_t kt = smem_u32(sK) + stage * kStageBytes + w * 2048;
                const uint32_t vt = smem_u32(sV) + stage * kStageBytes + w * 2048;
                // ---- segment of this tile
                const int sg = (t0 >= s_rec->start[1]) + (t0 >= s_rec->start[2]) + (t0 >= s_rec->start[3]) +
                               (t0 >= s_rec->start[4]);
                const float kscale = s_rec->k_scale[sg], kmin = s_rec->k_min[sg];
                const float vscale = s_rec->v_scale[sg], vmin = s_rec->v_min[sg];
                // A flat V segment (scale 0) decodes to v_min whatever its codes: it only feeds bsum.
                const bool vflat = !(vscale > 0.0f);
                if (!vflat && sg != st.seg) {
                    if (st.seg >= 0) {  // keep sigma * o invariant across the change of scale
                        const float ratio = st.sigma / vscale;
#pragma unroll
                        for (int i = 0; i < 8; ++i)
#pragma unroll
                            for (int e = 0; e < 4; ++e) st.o[i][e] *= ratio;
                    }
                    st.sigma = vscale;
                    st.seg = sg;
                }
                const float ak = kscale * kLog2eOverSqrtD;
                const float bk = (kmin - 1024.0f * kscale) * qsum * kLog2eOverSqrtD;
                const float cv = vflat ? vmin : vmin - 1024.0f * vscale;

                // ---- S^T = Q K^T: two n-tiles of 8 tokens, 8 k-steps of 16 columns
                // four independent accumulator chains (two n-tiles x even/odd k-steps)
                float sacc[2][4], sacc2[2][4];
                uint4 klo[2], khi[2];
#pragma unroll
                for (int nt2 = 0; nt2 < 2; ++nt2) {
                    const int row = nt2 * 8 + tr;  // token row this lane supplies (n = r)
                    const uint32_t rp = kt + row * kD;
                    klo[nt2] = lds128(rp + ((cq ^ (row & 7)) << 4));
                    khi[nt2] = lds128(rp + (((cq + 4) ^ (row & 7)) << 4));
#pragma unroll
                    for (int e = 0; e < 4; ++e) sacc[nt2][e] = sacc2[nt2][e] = 0.0f;
                }
#pragma unroll
                for (int jj = 0; jj < 8; jj += 2) {
#pragma unroll
                    for (int nt2 = 0; nt2 < 2; ++nt2) {
                        const uint32_t w0 = word(jj < 4 ? klo[nt2] : khi[nt2], jj & 3);
                        const uint32_t w1 = word(jj < 4 ? klo[nt2] : khi[nt2], (jj + 1) & 3);
                        mma16816(sacc[nt2], qa0[jj], 0u, qa2[jj], 0u, prmt(w0, M64, 0x4140), prmt(w0, M64, 0x4342));
                        mma16816(sacc2[nt2], qa0[jj + 1], 0u, qa2[jj + 1], 0u, prmt(w1, M64, 0x4140),
                                 prmt(w1, M64, 0x4342));
                    }
                }
#pragma unroll
                for (int nt2 = 0; nt2 < 2; ++nt2) {
                    sacc[nt2][0] += sacc2[nt2][0];
                    sacc[nt2][1] += sacc2[nt2][1];
                }
                // lane scores for head r: tokens cq, cq+4 (tile 0) and 8+cq, 12+cq (tile 1)
                float z[4];
                z[0] = (cq < valid) ? fmaf(ak, sacc[0][0], bk) : -INFINITY;
                z[1] = (cq + 4 < valid) ? fmaf(ak, sacc[0][1], bk) : -INFINITY;
                z[2] = (cq + 8 < valid) ? fmaf(ak, sacc[1][0], bk) : -INFINITY;
                z[3] = (cq + 12 < valid) ? fmaf(ak, sacc[1][1], bk) : -INFINITY;
                float mt = fmaxf(fmaxf(z[0], z[1]), fmaxf(z[2], z[3]));
                mt = fmaxf(mt, __shfl_xor_sync(0xffffffffu, mt, 1));
                mt = fmaxf(mt, __shfl_xor_sync(0xffffffffu, mt, 2));
                const bool need = gvalid && (mt > st.m + kLazyRescale);
                float alpha = 1.0f;
                if (need) {
                    alpha = (st.m == -INFINITY) ? 0.0f : ex2(st.m - mt);
                    st.m = mt;
                    st.l *= alpha;
                    st.bsum *= alpha;
                }
                if (__any_sync(0xffffffffu, need)) {
                    const float a0 = __shfl_sync(0xffffffffu, alpha, 8 * cq);      // head 2cq
                    const float a1 = __shfl_sync(0xffffffffu, alpha, 8 * cq + 4);  // head 2cq+1
#pragma unroll
                    for (int i = 0; i < 8; ++i) {
                        st.o[i][0] *= a0;
                        st.o[i][2] *= a0;
                        st.o[i][1] *= a1;
                        st.o[i][3] *= a1;
                    }
                }
                float pr[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) pr[e] = gvalid ? ex2(z[e] - st.m) : 0.0f;
                // the tensor cores see p rounded to fp16; the sums use the same rounded weights so
                // the 1024 offset of the codes cancels exactly against bsum
                const uint32_t pb0 = f32x2_to_f16x2(pr[0], pr[1]);
                const uint32_t pb1 = f32x2_to_f16x2(pr[2], pr[3]);
                const float psum = (f16lo(pb0) + f16hi(pb0)) + (f16lo(pb1) + f16hi(pb1));
                st.l += psum;
                st.bsum = fmaf(cv, psum, st.bsum);

                // ---- O^T += V^T P^T: rows (d) 16*tr + 2i (+1), k = tokens cq, cq+4, 8+cq, 12+cq
                if (!vflat) {
                const uint4 va = lds128(vt + cq * kD + ((tr ^ cq) << 4));
                const uint4 vb = lds128(vt + (cq + 4) * kD + ((tr ^ (cq + 4)) << 4));
                const uint4 vc = lds128(vt + (cq + 8) * kD + ((tr ^ cq) << 4));
                const uint4 vd = lds128(vt + (cq + 12) * kD + ((tr ^ (cq + 4)) << 4));
#pragma unroll
                for (int wi = 0; wi < 4; ++wi) {
                    const uint32_t xab01 = prmt(word(va, wi), word(vb, wi), 0x5140);
                    const uint32_t xab23 = prmt(word(va, wi), word(vb, wi), 0x7362);
                    const uint32_t xcd01 = prmt(word(vc, wi), word(vd, wi), 0x5140);
                    const uint32_t xcd23 = prmt(word(vc, wi), word(vd, wi), 0x7362);
                    mma16816(st.o[2 * wi], prmt(xab01, M64, 0x4140), prmt(xab01, M64, 0x4342),
                             prmt(xcd01, M64, 0x4140), prmt(xcd01, M64, 0x4342), pb0, pb1);
                    mma16816(st.o[2 * wi + 1], prmt(xab23, M64, 0x4140), prmt(xab23, M64, 0x4342),
                             prmt(xcd23, M64, 0x4140), prmt(xcd23, M64, 0x4342), pb0, pb1);
                }
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty[stage]);
            ++it;
        }

        if (!last) continue;

        // ================================================================ end of a piece
        // reduce the per-lane partial sums of head r over its four lanes
        float l = st.l, bsum = st.bsum;
        l += __shfl_xor_sync(0xffffffffu, l, 1);
        l += __shfl_xor_sync(0xffffffffu, l, 2);
        bsum += __shfl_xor_sync(0xffffffffu, bsum, 1);
        bsum += __shfl_xor_sync(0xffffffffu, bsum, 2);
        {
            float *cw = s_comb + w * G * kPartStride;
            if (gvalid && cq == 0) {
                cw[r * kPartStride + 0] = st.m;
                cw[r * kPartStride + 1] = l;
            }
            const float b0 = __shfl_sync(0xffffffffu, bsum, 8 * cq);
            const float b1 = __shfl_sync(0xffffffffu, bsum, 8 * cq + 4);
            const int g0 = 2 * cq, g1 = 2 * cq + 1;
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const int d = 16 * tr + 2 * i;
                if (g0 < G) {
                    cw[g0 * kPartStride + 2 + d] = fmaf(st.sigma, st.o[i][0], b0);
                    cw[g0 * kPartStride + 3 + d] = fmaf(st.sigma, st.o[i][2], b0);
                }
                if (g1 < G) {
                    cw[g1 * kPartStride + 2 + d] = fmaf(st.sigma, st.o[i][1], b1);
                    cw[g1 * kPartStride + 3 + d] = fmaf(st.sigma, st.o[i][3], b1);
                }
            }
        }
        named_bar_sync(1, kConsumerWarps * 32);

        // the current token's score s_new = q . k_new / sqrt(D) (log2 domain), one warp per head
        for (int g = w; g < G; g += kConsumerWarps) {
            const uint16_t *qrow = a.q + ((int64_t)c.b * a.Hq + c.h * G + g) * kD;
            const uint16_t *krow = a.knew + ((int64_t)c.b * Hkv + c.h) * kD;
            float acc = 0.0f;
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int dd = lane + 32 * i;
                acc = fmaf(__uint_as_float((uint32_t)__ldg(qrow + dd) << 16),
                           __uint_as_float((uint32_t)__ldg(krow + dd) << 16), acc);
            }
#pragma unroll
            for (int o = 16; o; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
            if (lane == 0) s_snew[g] = acc * kLog2eOverSqrtD;
        }
        named_bar_sync(1, kConsumerWarps * 32);

        // combine the four warps (thread ctid owns column d = ctid), then either finish the
        // pair here (it has a single piece) or publish this piece
        const int d = ctid;
        const float vn = __uint_as_float((uint32_t)__ldg(a.vnew + ((int64_t)c.b * Hkv + c.h) * kD + d) << 16);
        uint16_t *orow = a.out + ((int64_t)c.b * a.Hq + c.h * G) * kD + d;
        const int32_t first_chunk = s_cpre[c.b] + c.h * c.nch;
        const int32_t cfirst = owner(first_chunk, C, ncta);
        const int32_t clast = owner(first_chunk + c.nch - 1, C, ncta);
        for (int g = 0; g < G; ++g) {
            float M = -INFINITY;
#pragma unroll
            for (int ww = 0; ww < kConsumerWarps; ++ww) M = fmaxf(M, s_comb[(ww * G + g) * kPartStride]);
            float Ls = 0.0f, Os = 0.0f;
            if (M != -INFINITY) {
#pragma unroll
                for (int ww = 0; ww < kConsumerWarps; ++ww) {
                    const float *cw = s_comb + (ww * G + g) * kPartStride;
                    const float mw = cw[0];
                    if (mw != -INFINITY) {
                        const float f = exp2f(mw - M);
                        Ls = fmaf(cw[1], f, Ls);
                        Os = fmaf(cw[2 + d], f, Os);
                    }
                }
            }
            if (cfirst == clast) {
                orow[g * kD] = finish(M, Ls, Os, s_snew[g], vn);
            } else {
                float *dst = a.part + ((int64_t)(p + cta) * G + g) * kPartStride;
                __stcg(dst + 2 + d, Os);
                if (d == 0) {
                    __stcg(dst + 0, M);
                    __stcg(dst + 1, Ls);
                }
            }
        }
        if (cfirst != clast) {
            // the last piece to arrive merges all pieces of the pair in CTA order
            __threadfence();
            named_bar_sync(1, kConsumerWarps * 32);
            if (ctid == 0) {
                uint32_t pieces = 0;  // CTAs holding a piece of this pair
                for (int32_t cc = cfirst; cc <= clast; ++cc) pieces += owns_chunks(cc, C, ncta) ? 1u : 0u;
                const uint32_t old = atomicAdd(a.pair_count + p, 1u);
                const bool is_last = old + 1u == pieces;
                if (is_last) {
                    __threadfence();
                    a.pair_count[p] = 0;
                }
                s_flag[1] = is_last ? 1 : 0;
            }
            named_bar_sync(1, kConsumerWarps * 32);
            if (s_flag[1]) {
                for (int g = 0; g < G; ++g) {
                    float M = -INFINITY;
                    for (int32_t cc = cfirst; cc <= clast; ++cc)
                        if (owns_chunks(cc, C, ncta))
                            M = fmaxf(M, __ldcg(a.part + ((int64_t)(p + cc) * G + g) * kPartStride));
                    float Ls = 0.0f, Os = 0.0f;
                    if (M != -INFINITY) {
                        for (int32_t cc = cfirst; cc <= clast; ++cc) {
                            if (!owns_chunks(cc, C, ncta)) continue;
                            const float *src = a.part + ((int64_t)(p + cc) * G + g) * kPartStride;
                            const float mc = __ldcg(src);
                            if (mc != -INFINITY) {
                                const float f = exp2f(mc - M);
                                Ls = fmaf(__ldcg(src + 1), f, Ls);
                                Os = fmaf(__ldcg(src + 2 + d), f, Os);
                            }
                        }
                    }
                    orow[g * kD] = finish(M, Ls, Os, s_snew[g], vn);
                }
            }
        }
        named_bar_sync(1, kConsumerWarps * 32);
    }
}

}  // namespace dgq

// ---- host launcher ---------------------------------------------------------------------------

namespace dgq {

// 2-D map over a pool [num_blocks * Hkv * bs rows, 128 bytes], box = one (block, head) tile.
static bool make_pool_map(CUtensorMap *map, const uint8_t *pool, int64_t rows, int32_t bs)
{
    auto fn = tensor_map_encoder();
    if (!fn) return false;
    cuuint64_t dims[2] = {(cuuint64_t)kD, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)kD};
    cuuint32_t box[2] = {(cuuint32_t)kD, (cuuint32_t)bs};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<uint8_t *>(pool), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

size_t attn_smem_bytes(int32_t B, int32_t G)
{
    return 1024 + 2 * kStages * kStageBytes + 2 * kStages * 8 + 16 + 32 + sizeof(dgq_seg_record) +
           (size_t)kConsumerWarps * G * kPartStride * 4 + (size_t)(2 * B + 1) * 4;
}

int attn_max_ctas(int nsm) { return nsm * 3; }


AttnLayout attn_layout(int32_t batch, int32_t Hq, int32_t Hkv, int nsm)
{
    AttnLayout l;
    size_t P = (size_t)batch * Hkv;
    size_t G = (size_t)(Hq / Hkv);
    size_t off = sizeof(WsHeader);
    l.off_count = off;
    off = (off + P * 4 + 255) & ~size_t(255);
    l.off_part = off;
    off += (P + (size_t)attn_max_ctas(nsm)) * G * kPartStride * 4;
    l.total = (off + 255) & ~size_t(255);
    return l;
}

cudaError_t launch_attn(const void *q, const void *knew, const void *vnew, const uint8_t *kpool, const uint8_t *vpool,
                        const dgq_seg_record *table, const int32_t *bt, const int32_t *seq_lens, int32_t max_seqlen,
                        int32_t B, int32_t Hq, int32_t Hkv, int32_t bs, int32_t max_blocks, int32_t num_blocks,
                        void *out, void *ws, int nsm, bool *map_failed, cudaStream_t stream)
{
    *map_failed = false;
    CUtensorMap mk, mv;
    const int64_t rows = (int64_t)num_blocks * Hkv * bs;
    if (!make_pool_map(&mk, kpool, rows, bs) || !make_pool_map(&mv, vpool, rows, bs)) {
        *map_failed = true;
        return cudaErrorInvalidValue;
    }
    const int32_t G = Hq / Hkv;
    AttnLayout l = attn_layout(B, Hq, Hkv, nsm);
    char *base = static_cast<char *>(ws);
    AttnArgs a;
    a.q = static_cast<const uint16_t *>(q);
    a.knew = static_cast<const uint16_t *>(knew);
    a.vnew = static_cast<const uint16_t *>(vnew);
    a.table = table;
    a.bt = bt;
    a.seq_lens = seq_lens;
    a.out = static_cast<uint16_t *>(out);
    a.hdr = reinterpret_cast<WsHeader *>(base);
    a.pair_count = reinterpret_cast<uint32_t *>(base + l.off_count);
    a.part = reinterpret_cast<float *>(base + l.off_part);
    a.B = B;
    a.Hq = Hq;
    a.Hkv = Hkv;
    a.G = G;
    a.bs = bs;
    a.max_blocks = max_blocks;

    const size_t smem = attn_smem_bytes(B, G);
    cudaError_t e = cudaFuncSetAttribute(attn_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    int occ = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, attn_kernel, kAttnThreads, smem);
    if (e != cudaSuccess) return e;
    if (occ < 1) return cudaErrorInvalidConfiguration;
    if (occ > 3) occ = 3;
    // upper bound on chunks: every request at max_seqlen
    const int64_t cmax = (int64_t)B * Hkv * (int64_t)((max_seqlen + kChunk - 1) / kChunk > 0 ? (max_seqlen + kChunk - 1) / kChunk : 1);
    int64_t grid = (int64_t)nsm * occ;
    if (grid > cmax) grid = cmax;
    if (grid < 1) grid = 1;
    attn_kernel<<<(unsigned)grid, kAttnThreads, smem, stream>>>(mk, mv, a);
    return cudaGetLastError();
}

}  // namespace dgq
