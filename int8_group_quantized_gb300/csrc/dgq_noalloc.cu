// dgq_noalloc.cu -- decode attention for callers that cannot allocate device memory.
//
// dgq_paged_decode_attn needs a caller-provided workspace (split-K partials, per-pair piece
// ranges and a small header).  Some callers have no way to provide one: code that runs
// where cudaMalloc is not allowed or not wanted (for example inside a serving engine that
// hands each operator only the buffers it pre-planned, or a plugin running under an
// allocator that forbids new device allocations mid-step).  This file gives them one entry
// point whose workspace is a fixed array in the library's own device memory.
//
// The array is a file-scope __device__ variable: every GPU that loads the library holds
// DGQ_NOALLOC_SCRATCH_BYTES of it until the process exits.  Host code cannot use the
// variable's name as a device address, so the first call on each device looks the address
// up (cudaGetSymbolAddress) with that device current and caches it; nothing here calls
// cudaMalloc, cudaFree or any allocating routine.
#include <cuda_runtime.h>

#include <mutex>
#include <stddef.h>
#include <stdint.h>

#include "dgq.h"

namespace {

static __device__ __align__(256) unsigned char g_attn_scratch[DGQ_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
constexpr size_t kHeaderBytes = 256;  // the workspace header: must hold zeros when a call starts

std::mutex g_mu;
void *g_scratch_dev[kMaxDevices];  // device address of g_attn_scratch, per device (null until set up)

// Device address of the scratch array on the current device (set up on first use).
dgq_status scratch_address(void **out)
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return DGQ_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDevices) return DGQ_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lock(g_mu);
    if (!g_scratch_dev[dev]) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_attn_scratch) != cudaSuccess || !p) return DGQ_ERR_CUDA;
        g_scratch_dev[dev] = p;
    }
    *out = g_scratch_dev[dev];
    return DGQ_OK;
}

}  // namespace

extern "C" dgq_status dgq_paged_decode_attn_noalloc(const void *q_bf16, const void *k_new_bf16,
                                                    const void *v_new_bf16, const uint8_t *k_pool,
                                                    const uint8_t *v_pool, const dgq_seg_record *seg_table,
                                                    const int32_t *block_tables_dev, const int32_t *seq_lens_dev,
                                                    int32_t max_seqlen, int32_t batch, int32_t num_q_heads,
                                                    int32_t num_kv_heads, int32_t head_dim, int32_t block_size,
                                                    int32_t max_blocks_per_seq, int32_t num_blocks, void *out_bf16,
                                                    void *cuda_stream)
{
    // Shapes the workspace query rejects fall through to the regular entry point, which
    // reports the precise argument error.
    const size_t need = dgq_attn_workspace_size(batch, num_q_heads, num_kv_heads, max_seqlen);
    if (need > (size_t)DGQ_NOALLOC_SCRATCH_BYTES) return DGQ_ERR_SCRATCH_LIMIT;
    void *scratch = nullptr;
    const dgq_status st = scratch_address(&scratch);
    if (st != DGQ_OK) return st;
    // The previous call left the scratch ready, but a call that failed part-way may not have:
    // clear the header (error word and launch counters) so that every call starts clean.
    if (need > 0 &&
        cudaMemsetAsync(scratch, 0, kHeaderBytes, static_cast<cudaStream_t>(cuda_stream)) != cudaSuccess)
        return DGQ_ERR_CUDA;
    return dgq_paged_decode_attn(q_bf16, k_new_bf16, v_new_bf16, k_pool, v_pool, seg_table, block_tables_dev,
                                 seq_lens_dev, max_seqlen, batch, num_q_heads, num_kv_heads, head_dim, block_size,
                                 max_blocks_per_seq, num_blocks, out_bf16, scratch,
                                 (size_t)DGQ_NOALLOC_SCRATCH_BYTES, cuda_stream);
}
