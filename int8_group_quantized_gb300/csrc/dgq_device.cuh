// dgq_device.cuh -- small sm_103a device helpers shared by the DGQ kernels: memory-ordering
// primitives, mbarrier and TMA wrappers in inline PTX, bounded waits, and the workspace
// header layout.  No DGQ arithmetic lives here.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace dgq {

constexpr int kD = 128;     // head dimension
constexpr int kWin = 16;    // variance window (tokens)
constexpr int kMaxSeg = 5;  // segments per (request, KV head)

// n_groups(L), the length rule of the DGQ article (section 3.2): 2 below 2048 tokens, 3 below
// 16384, else min(5, floor(log2(L / 1024)) + 2), which is 5 for every L >= 16384.
__device__ __forceinline__ int32_t ngroups(int32_t L)
{
    if (L < 2048) return 2;
    if (L < 16384) return 3;
    // floor(log2(L / 1024)) = floor(log2(L)) - 10 for integer L >= 1024
    const int32_t g = (31 - __clz(L)) - 10 + 2;
    return g < 5 ? g : 5;
}

// Block sizes are powers of two (16, 32 or 64 tokens, checked on the host), so the block and the
// slot of a token index t >= 0 come from a shift and a mask instead of an integer division.
__device__ __forceinline__ int32_t pow2_div(int32_t t, int32_t n) { return t >> (__ffs(n) - 1); }
__device__ __forceinline__ int32_t pow2_mod(int32_t t, int32_t n) { return t & (n - 1); }

// Every workspace starts with this 256-byte header.
struct WsHeader {
    uint32_t error;        // first device-side error code (0 = none)
    uint32_t path;         // which kernel path the last call took (kPath*), for tests
    uint32_t done_ctas;    // CTAs finished in the current call (compress)
    uint32_t pad[61];
};
static_assert(sizeof(WsHeader) == 256, "workspace header must be 256 bytes");

// Device-side error codes written to WsHeader::error.
enum : uint32_t {
    kErrNone = 0,
    kErrBarrierWait = 1,    // compress: a chunk barrier never completed, or a worker waited
                            // too long for its CTA's segmentation
    kErrFullWait = 2,       // decode: a TMA stage never completed
    kErrEmptyWait = 3,      // decode: consumers never released a stage
    kErrNoBlock = 4,        // append: a pair's next slot has no block-table column
    kErrBadBlock = 5,       // a block-table entry outside [0, num_blocks): its window/tile skipped
    kErrBadLength = 6,      // a request length outside what the call's sizes allow: clamped or skipped
};

// WsHeader::path values
enum : uint32_t { kPathGrid = 1, kPathClusterWhole = 2, kPathBlockMerge = 3, kPathWarpMerge = 4 };

// Upper bound on spin iterations of any wait (each iteration sleeps or polls ~tens of ns;
// ~2^26 iterations is seconds, far beyond any legitimate wait).
constexpr uint32_t kSpinLimit = 1u << 26;

__device__ __forceinline__ void record_error(WsHeader *hdr, uint32_t code)
{
    atomicCAS(&hdr->error, 0u, code);
}

__device__ __forceinline__ uint32_t ld_acquire_gpu(const uint32_t *p)
{
    uint32_t v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ uint32_t ld_relaxed_gpu(const uint32_t *p)
{
    uint32_t v;
    asm volatile("ld.relaxed.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ int32_t ld_acquire_cta_shared(const int32_t *p)
{
    int32_t v;
    asm volatile("ld.acquire.cta.shared::cta.b32 %0, [%1];"
                 : "=r"(v)
                 : "r"(static_cast<uint32_t>(__cvta_generic_to_shared(p)))
                 : "memory");
    return v;
}

__device__ __forceinline__ void st_release_cta_shared(int32_t *p, int32_t v)
{
    asm volatile("st.release.cta.shared::cta.b32 [%0], %1;" ::"r"(static_cast<uint32_t>(__cvta_generic_to_shared(p))),
                 "r"(v)
                 : "memory");
}

__device__ __forceinline__ void st_release_gpu(uint32_t *p, uint32_t v)
{
    asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

__device__ __forceinline__ uint32_t atom_add_acq_rel_gpu(uint32_t *p, uint32_t v)
{
    uint32_t old;
    asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
    return old;
}

// ---- mbarrier ------------------------------------------------------------------------------

__device__ __forceinline__ uint32_t smem_u32(const void *p)
{
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// The dynamic shared-memory base rounded up to 1024 bytes by pointer arithmetic (an integer
// round trip would hide from the compiler that the result is a shared-memory address).
__device__ __forceinline__ uint8_t *align_smem_1024(uint8_t *raw)
{
    return raw + ((1024u - (smem_u32(raw) & 1023u)) & 1023u);
}

// 16-byte shared-memory load by 32-bit shared address.  volatile keeps it after the mbarrier
// wait that made the data visible.
__device__ __forceinline__ uint4 ld_shared_v4(uint32_t addr)
{
    uint4 v;
    asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(addr));
    return v;
}

__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t *bar)
{
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity)
{
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// Bounded wait for the phase with the given parity; false when the bound was hit.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t *bar, uint32_t parity)
{
    for (uint32_t i = 0; i < kSpinLimit; ++i)
        if (mbar_try_wait(bar, parity)) return true;
    return false;
}

__device__ __forceinline__ void fence_barrier_init()
{
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

// ---- TMA (tiled tensor copy, global -> shared, completion on an mbarrier) -----------------

__device__ __forceinline__ void tma_load_2d(void *smem_dst, const CUtensorMap *map, int32_t x, int32_t y,
                                            uint64_t *bar)
{
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3}], [%4];" ::"r"(smem_u32(smem_dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_u32(bar))
        : "memory");
}

__device__ __forceinline__ void tma_load_3d(void *smem_dst, const CUtensorMap *map, int32_t x, int32_t y, int32_t z,
                                            uint64_t *bar)
{
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(smem_u32(smem_dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(smem_u32(bar))
        : "memory");
}

// Same, with an L2 eviction-priority policy (from make_policy_*) attached to the copy.
__device__ __forceinline__ void tma_load_3d_hint(void *smem_dst, const CUtensorMap *map, int32_t x, int32_t y,
                                                 int32_t z, uint64_t *bar, uint64_t policy)
{
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1, {%2, %3, %4}], [%5], %6;" ::"r"(smem_u32(smem_dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(smem_u32(bar)), "l"(policy)
        : "memory");
}

// 4-D tile copy to a 32-bit shared address, with an L2 eviction-priority policy.
__device__ __forceinline__ void tma_load_4d_hint(uint32_t dst, const CUtensorMap *map, int32_t c0, int32_t c1,
                                                 int32_t c2, int32_t c3, uint32_t bar, uint64_t policy)
{
    asm volatile(
        "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1, {%2, %3, %4, %5}], [%6], %7;" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(bar), "l"(policy)
        : "memory");
}

// 5-D tile copy to a 32-bit shared address, with an L2 eviction-priority policy.
__device__ __forceinline__ void tma_load_5d_hint(uint32_t dst, const CUtensorMap *map, int32_t c0, int32_t c1,
                                                 int32_t c2, int32_t c3, int32_t c4, uint32_t bar, uint64_t policy)
{
    asm volatile(
        "cp.async.bulk.tensor.5d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1, {%2, %3, %4, %5, %6}], [%7], %8;" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(c4), "r"(bar), "l"(policy)
        : "memory");
}

// Orders this thread's earlier shared-memory accesses before later async-proxy (TMA) ones.
__device__ __forceinline__ void fence_proxy_async_smem()
{
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ uint64_t make_policy_evict_first()
{
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}

__device__ __forceinline__ uint64_t make_policy_evict_normal()
{
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_normal.b64 %0, 1.0;" : "=l"(p));
    return p;
}

__device__ __forceinline__ uint64_t make_policy_evict_last()
{
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
    return p;
}

// 1-D bulk copy global -> shared (16-byte aligned addresses, size a multiple of 16), completing
// on an mbarrier (the caller has announced the bytes with mbar_arrive_expect_tx).
__device__ __forceinline__ void bulk_load(void *smem_dst, const void *src, uint32_t bytes, uint64_t *bar)
{
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                     smem_u32(smem_dst)),
                 "l"(src), "r"(bytes), "r"(smem_u32(bar))
                 : "memory");
}

// Programmatic dependent launch: let the next kernel in the stream be scheduled early / wait for
// the previous kernel's completion (and the visibility of its memory) before going on.
__device__ __forceinline__ void pdl_launch_dependents() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
__device__ __forceinline__ void pdl_wait_primary() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

__device__ __forceinline__ void prefetch_tensormap(const CUtensorMap *map)
{
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// Named barrier among `count` threads (ids 1..15; 0 is __syncthreads).
__device__ __forceinline__ void named_bar_sync(uint32_t id, uint32_t count)
{
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}

// ---- bf16 bit helpers ------------------------------------------------------------------------

__device__ __forceinline__ float bf16lo_to_f32(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16hi_to_f32(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

}  // namespace dgq
