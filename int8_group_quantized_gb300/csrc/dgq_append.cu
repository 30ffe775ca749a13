// dgq_append.cu -- decode-step append: each (request, KV head)'s new key and value encoded
// into the INT8 paged cache at position L = seq_len (sm_103a).
//
// Method: the new token joins the last segment of its record and is encoded with that
// segment's min and 255/(max-min) in the two IEEE steps of the compress quantiser ("DeepSeek
// KV-cache dynamic group quantisation (DGQ)" article, section 2.2: independent min/max INT8
// per segment), its codes held to [0, 255]; a request with no token yet gets a first segment
// made of the new token alone.  Token L goes to pool[block_tables[b][L / bs]][h][L % bs]
// ("PagedAttention implementation" section of the DeepSeek-V4 KV-cache article).
//
// GPU design: one warp per (request, head) pair, 8 pairs per CTA.  Lane i reads word i of the
// 128-byte record and elements 4i .. 4i+3 of the new K and V rows, writes their four codes
// as one 32-bit store, and writes word i of the updated record back.  The launch is a
// programmatic dependent one: it starts while the previous kernel drains and waits for it
// (griddepcontrol.wait) before touching the records.  Compiled with -fmad=false.
#include "dgq_device.cuh"
#include "dgq.h"
#include "dgq_launch.h"

#include <stdint.h>

namespace dgq {

constexpr int kAppendPairsPerCta = 8;

// word offsets in dgq_seg_record
constexpr int kWN = 0, kWLen = 1, kWStart = 2, kWKMin = 7, kWKScale = 12, kWVMin = 17, kWVScale = 22,
              kWKInv = 27, kWVInv = 28;
static_assert(sizeof(dgq_seg_record) == 32 * 4, "one record word per lane");

struct AppendArgs {
    const uint2 *k_new;  // [B * Hkv * 32] groups of four bf16
    const uint2 *v_new;
    const int32_t *bt;
    uint8_t *kpool;
    uint8_t *vpool;
    uint32_t *table;     // records as words
    uint32_t *vtable;    // independent V segmentation: V's records (null otherwise)
    int32_t *flags;      // re-segmentation bits per pair (null: not reported)
    WsHeader *hdr;
    int32_t pairs, Hkv, bs, max_blocks, num_blocks;
};

// Re-segmentation bits of appending token L: a 16-token window completed, or the length reached a
// threshold of the n_groups rule.
__device__ __forceinline__ int32_t reseg_bits(int32_t L)
{
    return (((L + 1) % kWin == 0) ? DGQ_RESEG_WINDOW : 0) | (ngroups(L + 1) != ngroups(L) ? DGQ_RESEG_NGROUPS : 0);
}

__device__ __forceinline__ float bf_lo_f(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf_hi_f(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// min/max of the 128 values of a row held four per lane; -0 stored as +0
__device__ __forceinline__ void row_min_max(const float (&x)[4], float &mn, float &mx)
{
    mn = fminf(fminf(x[0], x[1]), fminf(x[2], x[3]));
    mx = fmaxf(fmaxf(x[0], x[1]), fmaxf(x[2], x[3]));
#pragma unroll
    for (int o = 16; o; o >>= 1) {
        mn = fminf(mn, __shfl_xor_sync(0xffffffffu, mn, o));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    }
    if (mn == 0.0f) mn = 0.0f;
    if (mx == 0.0f) mx = 0.0f;
}

// scale = (max - min) / 255 and inv = 255 / (max - min), both 0 for a flat row
__device__ __forceinline__ void affine(float mn, float mx, float &scale, float &inv)
{
    const float r = __fsub_rn(mx, mn);
    scale = r == 0.0f ? 0.0f : __fdiv_rn(r, 255.0f);
    inv = r == 0.0f ? 0.0f : __fdiv_rn(255.0f, r);
}

// Four codes min(max(rint((x - mn) * inv), 0), 255), packed little-endian.  Clamping u to
// [0, 255] before rounding gives the same integers (rint is monotone and the bounds are
// integers) and keeps the 1.5 * 2^23 rounding add exact.
__device__ __forceinline__ uint32_t encode4(const float (&x)[4], float mn, float inv)
{
    uint32_t c[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
        float u = __fmul_rn(__fsub_rn(x[e], mn), inv);
        u = fminf(fmaxf(u, 0.0f), 255.0f);
        c[e] = __float_as_uint(__fadd_rn(u, 12582912.0f)) & 0xFFu;
    }
    return c[0] | (c[1] << 8) | (c[2] << 16) | (c[3] << 24);
}

__global__ void __launch_bounds__(kAppendPairsPerCta * 32) append_kernel(AppendArgs a)
{
    pdl_wait_primary();  // records and pools as the previous kernel in the stream left them
    const int lane = threadIdx.x & 31;
    const int32_t pair = blockIdx.x * kAppendPairsPerCta + (threadIdx.x >> 5);
    if (pair >= a.pairs) return;
    const int32_t b = pair / a.Hkv, h = pair - b * a.Hkv;
    uint32_t *rec = a.table + (int64_t)pair * 32;
    const uint32_t w = rec[lane];
    const int32_t n_seg = (int32_t)__shfl_sync(0xffffffffu, w, kWN);
    const int32_t L = (int32_t)__shfl_sync(0xffffffffu, w, kWLen);
    if (L < 0 || L / a.bs >= a.max_blocks) {  // the block table has no column for slot L
        if (lane == 0) {
            record_error(a.hdr, kErrNoBlock);
            if (a.flags) a.flags[pair] = 0;
        }
        return;
    }
    const int32_t blk = __ldg(a.bt + (int64_t)b * a.max_blocks + L / a.bs);
    if ((uint32_t)blk >= (uint32_t)a.num_blocks) {  // not a block of the pools: flagged, untouched
        if (lane == 0) {
            record_error(a.hdr, kErrBadBlock);
            if (a.flags) a.flags[pair] = 0;
        }
        return;
    }
    if (a.flags && lane == 0) a.flags[pair] = reseg_bits(L);
    const uint2 kw = __ldg(a.k_new + (int64_t)pair * 32 + lane);
    const uint2 vw = __ldg(a.v_new + (int64_t)pair * 32 + lane);
    const float kx[4] = {bf_lo_f(kw.x), bf_hi_f(kw.x), bf_lo_f(kw.y), bf_hi_f(kw.y)};
    const float vx[4] = {bf_lo_f(vw.x), bf_hi_f(vw.x), bf_lo_f(vw.y), bf_hi_f(vw.y)};

    float kmn, kinv, vmn, vinv, kscale = 0.0f, vscale = 0.0f, kmx, vmx;
    if (n_seg == 0) {  // the first token: a segment of its own
        row_min_max(kx, kmn, kmx);
        row_min_max(vx, vmn, vmx);
        affine(kmn, kmx, kscale, kinv);
        affine(vmn, vmx, vscale, vinv);
    } else {
        const int s = n_seg - 1;
        kmn = __uint_as_float(__shfl_sync(0xffffffffu, w, kWKMin + s));
        vmn = __uint_as_float(__shfl_sync(0xffffffffu, w, kWVMin + s));
        kinv = __uint_as_float(__shfl_sync(0xffffffffu, w, kWKInv));
        vinv = __uint_as_float(__shfl_sync(0xffffffffu, w, kWVInv));
    }
    const int64_t dst = (((int64_t)blk * a.Hkv + h) * a.bs + L % a.bs) * kD + lane * 4;
    *reinterpret_cast<uint32_t *>(a.kpool + dst) = encode4(kx, kmn, kinv);
    *reinterpret_cast<uint32_t *>(a.vpool + dst) = encode4(vx, vmn, vinv);

    // the record: seq_len L + 1, start entries past the last segment L + 1, and for a first
    // token its segment's parameters
    const int32_t n_new = n_seg == 0 ? 1 : n_seg;
    uint32_t nw = w;
    if (lane == kWN) nw = (uint32_t)n_new;
    if (lane == kWLen) nw = (uint32_t)(L + 1);
    if (lane >= kWStart && lane < kWStart + kMaxSeg) {
        const int i = lane - kWStart;
        if (i >= n_new) nw = (uint32_t)(L + 1);
        else if (n_seg == 0) nw = 0u;  // start[0]
    }
    if (n_seg == 0) {
        if (lane == kWKMin) nw = __float_as_uint(kmn);
        if (lane == kWKScale) nw = __float_as_uint(kscale);
        if (lane == kWVMin) nw = __float_as_uint(vmn);
        if (lane == kWVScale) nw = __float_as_uint(vscale);
        if (lane == kWKInv) nw = __float_as_uint(kinv);
        if (lane == kWVInv) nw = __float_as_uint(vinv);
    }
    rec[lane] = nw;
}

// One tensor's new row (four values per lane) into slot `dst` with its own record, of which this
// lane holds word w; returns the lane's updated record word.  As append_kernel, for the fields of
// one tensor (K: k_min / k_scale / k_inv_last; V: the V fields).
__device__ __forceinline__ uint32_t append_one(const float (&x)[4], uint32_t w, bool is_v, uint8_t *pool,
                                               int64_t dst, int32_t L)
{
    const int lane = threadIdx.x & 31;
    const int wmin = is_v ? kWVMin : kWKMin, wscale = is_v ? kWVScale : kWKScale, winv = is_v ? kWVInv : kWKInv;
    const int32_t n_seg = (int32_t)__shfl_sync(0xffffffffu, w, kWN);
    float mn, inv, scale = 0.0f, mx;
    if (n_seg == 0) {  // the first token: a segment of its own
        row_min_max(x, mn, mx);
        affine(mn, mx, scale, inv);
    } else {
        mn = __uint_as_float(__shfl_sync(0xffffffffu, w, wmin + n_seg - 1));
        inv = __uint_as_float(__shfl_sync(0xffffffffu, w, winv));
    }
    *reinterpret_cast<uint32_t *>(pool + dst) = encode4(x, mn, inv);
    const int32_t n_new = n_seg == 0 ? 1 : n_seg;
    uint32_t nw = w;
    if (lane == kWN) nw = (uint32_t)n_new;
    if (lane == kWLen) nw = (uint32_t)(L + 1);
    if (lane >= kWStart && lane < kWStart + kMaxSeg) {
        const int i = lane - kWStart;
        if (i >= n_new) nw = (uint32_t)(L + 1);
        else if (n_seg == 0) nw = 0u;  // start[0]
    }
    if (n_seg == 0) {
        if (lane == wmin) nw = __float_as_uint(mn);
        if (lane == wscale) nw = __float_as_uint(scale);
        if (lane == winv) nw = __float_as_uint(inv);
    }
    return nw;
}

// Append with independent V segmentation: K's and V's codes each from their own record.
__global__ void __launch_bounds__(kAppendPairsPerCta * 32) append_split_kernel(AppendArgs a)
{
    pdl_wait_primary();  // records and pools as the previous kernel in the stream left them
    const int lane = threadIdx.x & 31;
    const int32_t pair = blockIdx.x * kAppendPairsPerCta + (threadIdx.x >> 5);
    if (pair >= a.pairs) return;
    const int32_t b = pair / a.Hkv, h = pair - b * a.Hkv;
    uint32_t *krec = a.table + (int64_t)pair * 32, *vrec = a.vtable + (int64_t)pair * 32;
    const uint32_t wk = krec[lane], wv = vrec[lane];
    const int32_t L = (int32_t)__shfl_sync(0xffffffffu, wk, kWLen);
    int err = kErrNone;
    int32_t blk = -1;
    if (L != (int32_t)__shfl_sync(0xffffffffu, wv, kWLen)) {  // the two records disagree: untouched
        err = kErrBadLength;
    } else if (L < 0 || L / a.bs >= a.max_blocks) {  // the block table has no column for slot L
        err = kErrNoBlock;
    } else {
        blk = __ldg(a.bt + (int64_t)b * a.max_blocks + L / a.bs);
        if ((uint32_t)blk >= (uint32_t)a.num_blocks) err = kErrBadBlock;  // not a block of the pools
    }
    if (a.flags && lane == 0) a.flags[pair] = err == kErrNone ? reseg_bits(L) : 0;
    if (err != kErrNone) {  // flagged, untouched
        if (lane == 0) record_error(a.hdr, err);
        return;
    }
    const uint2 kw = __ldg(a.k_new + (int64_t)pair * 32 + lane);
    const uint2 vw = __ldg(a.v_new + (int64_t)pair * 32 + lane);
    const float kx[4] = {bf_lo_f(kw.x), bf_hi_f(kw.x), bf_lo_f(kw.y), bf_hi_f(kw.y)};
    const float vx[4] = {bf_lo_f(vw.x), bf_hi_f(vw.x), bf_lo_f(vw.y), bf_hi_f(vw.y)};
    const int64_t dst = (((int64_t)blk * a.Hkv + h) * a.bs + L % a.bs) * kD + lane * 4;
    const uint32_t nk = append_one(kx, wk, false, a.kpool, dst, L);
    const uint32_t nv = append_one(vx, wv, true, a.vpool, dst, L);
    krec[lane] = nk;
    vrec[lane] = nv;
}

cudaError_t launch_append(const void *k_new, const void *v_new, int32_t B, int32_t Hkv, int32_t bs,
                          const int32_t *bt, int32_t max_blocks, uint8_t *kpool, uint8_t *vpool, int32_t num_blocks,
                          dgq_seg_record *table, dgq_seg_record *vtable, int32_t *flags, void *ws,
                          cudaStream_t stream)
{
    AppendArgs a;
    a.flags = flags;
    a.k_new = static_cast<const uint2 *>(k_new);
    a.v_new = static_cast<const uint2 *>(v_new);
    a.bt = bt;
    a.kpool = kpool;
    a.vpool = vpool;
    a.table = reinterpret_cast<uint32_t *>(table);
    a.vtable = reinterpret_cast<uint32_t *>(vtable);
    a.hdr = static_cast<WsHeader *>(ws);
    a.pairs = B * Hkv;
    a.Hkv = Hkv;
    a.bs = bs;
    a.max_blocks = max_blocks;
    a.num_blocks = num_blocks;
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.gridDim = dim3((unsigned)((a.pairs + kAppendPairsPerCta - 1) / kAppendPairsPerCta));
    cfg.blockDim = dim3(kAppendPairsPerCta * 32);
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return vtable ? cudaLaunchKernelEx(&cfg, append_split_kernel, a) : cudaLaunchKernelEx(&cfg, append_kernel, a);
}

}  // namespace dgq
