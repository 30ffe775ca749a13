// dgq_host.cu -- the C ABI of libdgq.so: argument checks, workspace sizing, launch,
// device error read-back, and the host block pool.  Every check runs before any launch.
#include "dgq.h"

#include <cuda_runtime.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#include <vector>

#include "dgq_launch.h"

static_assert(sizeof(dgq_seg_record) == 128, "dgq_seg_record must be 128 bytes");

namespace dgq {
PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder()
{
    static thread_local PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    if (!fn) {
        cudaDriverEntryPointQueryResult q;
        void *p = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    }
    return fn;
}
}  // namespace dgq

namespace {

constexpr int32_t kMaxBatch = dgq::kMaxCallBatch;  // per-call limit (the kernels keep per-request prefixes on chip)

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bool block_size_ok(int32_t bs) { return bs == 16 || bs == 32 || bs == 64; }

int device_sm_count(int *nsm)
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return -1;
    if (cudaDeviceGetAttribute(nsm, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return -1;
    return 0;
}

}  // namespace

extern "C" {

const char *dgq_status_str(dgq_status s)
{
    switch (s) {
    case DGQ_OK: return "ok";
    case DGQ_ERR_INVALID_ARG: return "invalid argument";
    case DGQ_ERR_UNSUPPORTED: return "unsupported shape";
    case DGQ_ERR_WORKSPACE: return "workspace too small or missing";
    case DGQ_ERR_CUDA: return "CUDA error";
    case DGQ_ERR_POOL_EXHAUSTED: return "block pool exhausted";
    case DGQ_ERR_DEVICE: return "device-side wait timed out";
    case DGQ_ERR_SCRATCH_LIMIT: return "problem too large for the fixed no-allocation scratch array";
    }
    return "unknown status";
}

size_t dgq_compress_workspace_size(int32_t batch, int32_t max_seqlen, int32_t num_kv_heads)
{
    if (batch <= 0 || max_seqlen < 0 || num_kv_heads <= 0) return 0;
    return dgq::compress_layout(batch, max_seqlen, num_kv_heads).total;
}

dgq_status dgq_compress(const void *k_bf16, const void *v_bf16, int32_t total_tokens, const int32_t *cu_seqlens_dev,
                        int32_t batch, int32_t max_seqlen, int32_t num_kv_heads, int32_t head_dim, int32_t block_size,
                        const int32_t *block_tables_dev, int32_t max_blocks_per_seq, uint8_t *k_pool,
                        uint8_t *v_pool, int32_t num_blocks, dgq_seg_record *seg_table, void *workspace,
                        size_t workspace_bytes, void *cuda_stream)
{
    return dgq_compress_ex(k_bf16, v_bf16, total_tokens, cu_seqlens_dev, batch, max_seqlen, num_kv_heads, head_dim,
                           block_size, block_tables_dev, max_blocks_per_seq, k_pool, v_pool, num_blocks, seg_table,
                           workspace, workspace_bytes, nullptr, cuda_stream);
}

namespace {

// Checks and launch shared by the packed and the paged-source entry points.
dgq_status compress_impl(const dgq::SourceDesc &src, const int32_t *cu_seqlens_dev, int32_t batch,
                         int32_t max_seqlen, int32_t num_kv_heads, int32_t head_dim, int32_t block_size,
                         const int32_t *block_tables_dev, int32_t max_blocks_per_seq, uint8_t *k_pool,
                         uint8_t *v_pool, int32_t num_blocks, dgq_seg_record *seg_table, void *workspace,
                         size_t workspace_bytes, const dgq_compress_options *options, void *cuda_stream)
{
    dgq::GroupSettings gs = {DGQ_MAX_SEG, 0.0f};
    if (options) {
        if (options->max_groups < 1 || options->max_groups > DGQ_MAX_SEG || !(options->min_var >= 0.0f) ||
            !(options->min_var <= 3.4e38f))
            return DGQ_ERR_INVALID_ARG;
        gs.max_groups = options->max_groups;
        gs.min_var = options->min_var;
    }
    if (head_dim != DGQ_HEAD_DIM || !block_size_ok(block_size)) return DGQ_ERR_UNSUPPORTED;
    if (batch <= 0 || batch > kMaxBatch || max_seqlen < 0 || num_kv_heads <= 0 || num_blocks <= 0 ||
        max_blocks_per_seq <= 0)
        return DGQ_ERR_INVALID_ARG;
    if ((int64_t)max_seqlen > (int64_t)max_blocks_per_seq * block_size) return DGQ_ERR_INVALID_ARG;
    if (src.bt == nullptr && src.T < 0) return DGQ_ERR_INVALID_ARG;
    if (src.bt != nullptr &&
        (src.num_blocks <= 0 || src.max_blocks <= 0 || (int64_t)max_seqlen > (int64_t)src.max_blocks * block_size ||
         !aligned16(src.bt)))
        return DGQ_ERR_INVALID_ARG;
    // flat window index and pool row index are 32-bit on the device
    const int64_t windows = (int64_t)batch * num_kv_heads * ((max_seqlen + DGQ_WINDOW - 1) / DGQ_WINDOW);
    if (windows >= INT32_MAX || (int64_t)num_blocks * num_kv_heads * block_size >= INT32_MAX)
        return DGQ_ERR_UNSUPPORTED;
    if (!src.k || !src.v || !cu_seqlens_dev || !block_tables_dev || !k_pool || !v_pool || !seg_table)
        return DGQ_ERR_INVALID_ARG;
    if (!aligned16(src.k) || !aligned16(src.v) || !aligned16(k_pool) || !aligned16(v_pool) ||
        !aligned16(seg_table) || !aligned16(cu_seqlens_dev) || !aligned16(block_tables_dev))
        return DGQ_ERR_INVALID_ARG;
    if (!workspace || !aligned16(workspace) ||
        workspace_bytes < dgq_compress_workspace_size(batch, max_seqlen, num_kv_heads))
        return DGQ_ERR_WORKSPACE;
    int nsm = 0;
    if (device_sm_count(&nsm) != 0) return DGQ_ERR_CUDA;
    const cudaStream_t stream = static_cast<cudaStream_t>(cuda_stream);
    const cudaError_t e =
        max_seqlen <= dgq::cluster_compress_max_seqlen()
            ? dgq::launch_compress_cluster(src, cu_seqlens_dev, batch, max_seqlen, num_kv_heads, block_size,
                                           block_tables_dev, max_blocks_per_seq, k_pool, v_pool, num_blocks,
                                           seg_table, workspace, gs, stream)
            : dgq::launch_compress(src, cu_seqlens_dev, batch, max_seqlen, num_kv_heads, block_size,
                                   block_tables_dev, max_blocks_per_seq, k_pool, v_pool, num_blocks, seg_table,
                                   workspace, gs, nsm, stream);
    return e == cudaSuccess ? DGQ_OK : DGQ_ERR_CUDA;
}

}  // namespace

dgq_status dgq_compress_ex(const void *k_bf16, const void *v_bf16, int32_t total_tokens,
                           const int32_t *cu_seqlens_dev, int32_t batch, int32_t max_seqlen, int32_t num_kv_heads,
                           int32_t head_dim, int32_t block_size, const int32_t *block_tables_dev,
                           int32_t max_blocks_per_seq, uint8_t *k_pool, uint8_t *v_pool, int32_t num_blocks,
                           dgq_seg_record *seg_table, void *workspace, size_t workspace_bytes,
                           const dgq_compress_options *options, void *cuda_stream)
{
    const dgq::SourceDesc src = {k_bf16, v_bf16, total_tokens, nullptr, 0, 0};
    return compress_impl(src, cu_seqlens_dev, batch, max_seqlen, num_kv_heads, head_dim, block_size,
                         block_tables_dev, max_blocks_per_seq, k_pool, v_pool, num_blocks, seg_table, workspace,
                         workspace_bytes, options, cuda_stream);
}

dgq_status dgq_compress_paged(const void *k_src_bf16, const void *v_src_bf16, int32_t num_src_blocks,
                              const int32_t *src_block_tables_dev, int32_t max_src_blocks_per_seq,
                              const int32_t *cu_seqlens_dev, int32_t batch, int32_t max_seqlen,
                              int32_t num_kv_heads, int32_t head_dim, int32_t block_size,
                              const int32_t *block_tables_dev, int32_t max_blocks_per_seq, uint8_t *k_pool,
                              uint8_t *v_pool, int32_t num_blocks, dgq_seg_record *seg_table, void *workspace,
                              size_t workspace_bytes, const dgq_compress_options *options, void *cuda_stream)
{
    if (!src_block_tables_dev) return DGQ_ERR_INVALID_ARG;
    const dgq::SourceDesc src = {k_src_bf16, v_src_bf16, 0, src_block_tables_dev, max_src_blocks_per_seq,
                                 num_src_blocks};
    return compress_impl(src, cu_seqlens_dev, batch, max_seqlen, num_kv_heads, head_dim, block_size,
                         block_tables_dev, max_blocks_per_seq, k_pool, v_pool, num_blocks, seg_table, workspace,
                         workspace_bytes, options, cuda_stream);
}

size_t dgq_append_workspace_size(void) { return 256; }  // the workspace header alone

namespace {
dgq_status append_impl(const void *k_new_bf16, const void *v_new_bf16, int32_t batch, int32_t num_kv_heads,
                       int32_t head_dim, int32_t block_size, const int32_t *block_tables_dev,
                       int32_t max_blocks_per_seq, uint8_t *k_pool, uint8_t *v_pool, int32_t num_blocks,
                       dgq_seg_record *seg_table, dgq_seg_record *v_seg_table, int32_t *flags, void *workspace,
                       size_t workspace_bytes, void *cuda_stream);
}  // namespace

dgq_status dgq_append_ex(const void *k_new_bf16, const void *v_new_bf16, int32_t batch, int32_t num_kv_heads,
                         int32_t head_dim, int32_t block_size, const int32_t *block_tables_dev,
                         int32_t max_blocks_per_seq, uint8_t *k_pool, uint8_t *v_pool, int32_t num_blocks,
                         dgq_seg_record *seg_table, int32_t *resegment_flags, void *workspace,
                         size_t workspace_bytes, void *cuda_stream)
{
    if (resegment_flags && !aligned16(resegment_flags)) return DGQ_ERR_INVALID_ARG;
    return append_impl(k_new_bf16, v_new_bf16, batch, num_kv_heads, head_dim, block_size, block_tables_dev,
                       max_blocks_per_seq, k_pool, v_pool, num_blocks, seg_table, nullptr, resegment_flags,
                       workspace, workspace_bytes, cuda_stream);
}

dgq_status dgq_append(const void *k_new_bf16, const void *v_new_bf16, int32_t batch, int32_t num_kv_heads,
                      int32_t head_dim, int32_t block_size, const int32_t *block_tables_dev,
                      int32_t max_blocks_per_seq, uint8_t *k_pool, uint8_t *v_pool, int32_t num_blocks,
                      dgq_seg_record *seg_table, void *workspace, size_t workspace_bytes, void *cuda_stream)
{
    return append_impl(k_new_bf16, v_new_bf16, batch, num_kv_heads, head_dim, block_size, block_tables_dev,
                       max_blocks_per_seq, k_pool, v_pool, num_blocks, seg_table, nullptr, nullptr, workspace,
                       workspace_bytes, cuda_stream);
}

dgq_status dgq_append_split(const void *k_new_bf16, const void *v_new_bf16, int32_t batch, int32_t num_kv_heads,
                            int32_t head_dim, int32_t block_size, const int32_t *block_tables_dev,
                            int32_t max_blocks_per_seq, uint8_t *k_pool, uint8_t *v_pool, int32_t num_blocks,
                            dgq_seg_record *k_seg_table, dgq_seg_record *v_seg_table, void *workspace,
                            size_t workspace_bytes, void *cuda_stream)
{
    if (!v_seg_table || !aligned16(v_seg_table)) return DGQ_ERR_INVALID_ARG;
    return append_impl(k_new_bf16, v_new_bf16, batch, num_kv_heads, head_dim, block_size, block_tables_dev,
                       max_blocks_per_seq, k_pool, v_pool, num_blocks, k_seg_table, v_seg_table, nullptr,
                       workspace, workspace_bytes, cuda_stream);
}

namespace {
dgq_status append_impl(const void *k_new_bf16, const void *v_new_bf16, int32_t batch, int32_t num_kv_heads,
                       int32_t head_dim, int32_t block_size, const int32_t *block_tables_dev,
                       int32_t max_blocks_per_seq, uint8_t *k_pool, uint8_t *v_pool, int32_t num_blocks,
                       dgq_seg_record *seg_table, dgq_seg_record *v_seg_table, int32_t *flags, void *workspace,
                       size_t workspace_bytes, void *cuda_stream)
{
    if (head_dim != DGQ_HEAD_DIM || !block_size_ok(block_size)) return DGQ_ERR_UNSUPPORTED;
    if (batch <= 0 || batch > kMaxBatch || num_kv_heads <= 0 || num_blocks <= 0 || max_blocks_per_seq <= 0)
        return DGQ_ERR_INVALID_ARG;
    if ((int64_t)num_blocks * num_kv_heads * block_size >= INT32_MAX) return DGQ_ERR_UNSUPPORTED;
    if (!k_new_bf16 || !v_new_bf16 || !block_tables_dev || !k_pool || !v_pool || !seg_table)
        return DGQ_ERR_INVALID_ARG;
    if (!aligned16(k_new_bf16) || !aligned16(v_new_bf16) || !aligned16(block_tables_dev) || !aligned16(k_pool) ||
        !aligned16(v_pool) || !aligned16(seg_table))
        return DGQ_ERR_INVALID_ARG;
    if (!workspace || !aligned16(workspace) || workspace_bytes < dgq_append_workspace_size())
        return DGQ_ERR_WORKSPACE;
    const cudaError_t e = dgq::launch_append(k_new_bf16, v_new_bf16, batch, num_kv_heads, block_size,
                                             block_tables_dev, max_blocks_per_seq, k_pool, v_pool, num_blocks,
                                             seg_table, v_seg_table, flags, workspace,
                                             static_cast<cudaStream_t>(cuda_stream));
    return e == cudaSuccess ? DGQ_OK : DGQ_ERR_CUDA;
}
}  // namespace

size_t dgq_attn_workspace_size(int32_t batch, int32_t num_q_heads, int32_t num_kv_heads, int32_t max_seqlen)
{
    (void)max_seqlen;
    if (batch <= 0 || num_q_heads <= 0 || num_kv_heads <= 0 || num_q_heads % num_kv_heads) return 0;
    int nsm = 0;
    if (device_sm_count(&nsm) != 0) return 0;
    return dgq::attn_layout(batch, num_q_heads, num_kv_heads, nsm).total;
}

dgq_status dgq_paged_decode_attn(const void *q_bf16, const void *k_new_bf16, const void *v_new_bf16,
                                 const uint8_t *k_pool, const uint8_t *v_pool, const dgq_seg_record *seg_table,
                                 const int32_t *block_tables_dev, const int32_t *seq_lens_dev, int32_t max_seqlen,
                                 int32_t batch, int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim,
                                 int32_t block_size, int32_t max_blocks_per_seq, int32_t num_blocks, void *out_bf16,
                                 void *workspace, size_t workspace_bytes, void *cuda_stream)
{
    return dgq_paged_decode_attn_format(DGQ_FORMAT_DGQ, q_bf16, k_new_bf16, v_new_bf16, k_pool, v_pool, seg_table,
                                        nullptr, nullptr, block_tables_dev, seq_lens_dev, max_seqlen, batch,
                                        num_q_heads, num_kv_heads, head_dim, block_size, max_blocks_per_seq,
                                        num_blocks, out_bf16, workspace, workspace_bytes, cuda_stream);
}

namespace {
dgq_status attn_impl(int32_t format, const void *q_bf16, const void *k_new_bf16, const void *v_new_bf16,
                     const uint8_t *k_pool, const uint8_t *v_pool, const dgq_seg_record *seg_table,
                     const dgq_seg_record *v_seg_table, const float *k_group_params, const float *v_group_params,
                     const int32_t *block_tables_dev, const int32_t *seq_lens_dev, int32_t max_seqlen, int32_t batch,
                     int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim, int32_t block_size,
                     int32_t max_blocks_per_seq, int32_t num_blocks, void *out_bf16, void *workspace,
                     size_t workspace_bytes, void *cuda_stream);
}  // namespace

dgq_status dgq_paged_decode_attn_split(const void *q_bf16, const void *k_new_bf16, const void *v_new_bf16,
                                       const uint8_t *k_pool, const uint8_t *v_pool, const dgq_seg_record *k_seg_table,
                                       const dgq_seg_record *v_seg_table, const int32_t *block_tables_dev,
                                       const int32_t *seq_lens_dev, int32_t max_seqlen, int32_t batch,
                                       int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim, int32_t block_size,
                                       int32_t max_blocks_per_seq, int32_t num_blocks, void *out_bf16,
                                       void *workspace, size_t workspace_bytes, void *cuda_stream)
{
    if (!v_seg_table || !aligned16(v_seg_table)) return DGQ_ERR_INVALID_ARG;
    return attn_impl(DGQ_FORMAT_DGQ, q_bf16, k_new_bf16, v_new_bf16, k_pool, v_pool, k_seg_table, v_seg_table,
                     nullptr, nullptr, block_tables_dev, seq_lens_dev, max_seqlen, batch, num_q_heads, num_kv_heads,
                     head_dim, block_size, max_blocks_per_seq, num_blocks, out_bf16, workspace, workspace_bytes,
                     cuda_stream);
}

dgq_status dgq_paged_decode_attn_format(int32_t format, const void *q_bf16, const void *k_new_bf16,
                                        const void *v_new_bf16, const uint8_t *k_pool, const uint8_t *v_pool,
                                        const dgq_seg_record *seg_table, const float *k_group_params,
                                        const float *v_group_params, const int32_t *block_tables_dev,
                                        const int32_t *seq_lens_dev, int32_t max_seqlen, int32_t batch,
                                        int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim,
                                        int32_t block_size, int32_t max_blocks_per_seq, int32_t num_blocks,
                                        void *out_bf16, void *workspace, size_t workspace_bytes, void *cuda_stream)
{
    return attn_impl(format, q_bf16, k_new_bf16, v_new_bf16, k_pool, v_pool, seg_table, nullptr, k_group_params,
                     v_group_params, block_tables_dev, seq_lens_dev, max_seqlen, batch, num_q_heads, num_kv_heads,
                     head_dim, block_size, max_blocks_per_seq, num_blocks, out_bf16, workspace, workspace_bytes,
                     cuda_stream);
}

namespace {
dgq_status attn_impl(int32_t format, const void *q_bf16, const void *k_new_bf16, const void *v_new_bf16,
                     const uint8_t *k_pool, const uint8_t *v_pool, const dgq_seg_record *seg_table,
                     const dgq_seg_record *v_seg_table, const float *k_group_params, const float *v_group_params,
                     const int32_t *block_tables_dev, const int32_t *seq_lens_dev, int32_t max_seqlen, int32_t batch,
                     int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim, int32_t block_size,
                     int32_t max_blocks_per_seq, int32_t num_blocks, void *out_bf16, void *workspace,
                     size_t workspace_bytes, void *cuda_stream)
{
    if (format != DGQ_FORMAT_DGQ && format != DGQ_FORMAT_FIXED64 && format != DGQ_FORMAT_SYM_INT8 &&
        format != DGQ_FORMAT_FP8_E4M3)
        return DGQ_ERR_INVALID_ARG;
    if (format == DGQ_FORMAT_FIXED64 && (!k_group_params || !v_group_params || !aligned16(k_group_params) ||
                                         !aligned16(v_group_params)))
        return DGQ_ERR_INVALID_ARG;
    if (head_dim != DGQ_HEAD_DIM || !block_size_ok(block_size)) return DGQ_ERR_UNSUPPORTED;
    if (batch <= 0 || batch > kMaxBatch || max_seqlen < 0 || num_q_heads <= 0 || num_kv_heads <= 0 ||
        num_blocks <= 0 || max_blocks_per_seq <= 0)
        return DGQ_ERR_INVALID_ARG;
    if (num_q_heads % num_kv_heads) return DGQ_ERR_INVALID_ARG;
    const int32_t G = num_q_heads / num_kv_heads;
    if (G != 1 && G != 2 && G != 4 && G != 8) return DGQ_ERR_UNSUPPORTED;
    if ((int64_t)max_seqlen > (int64_t)max_blocks_per_seq * block_size) return DGQ_ERR_INVALID_ARG;
    const int64_t chunks = (int64_t)batch * num_kv_heads * ((max_seqlen + 63) / 64 + 1);
    if (chunks >= INT32_MAX || (int64_t)num_blocks * num_kv_heads * block_size >= INT32_MAX)
        return DGQ_ERR_UNSUPPORTED;
    if (!q_bf16 || !k_new_bf16 || !v_new_bf16 || !k_pool || !v_pool || !seg_table || !block_tables_dev ||
        !seq_lens_dev || !out_bf16)
        return DGQ_ERR_INVALID_ARG;
    if (!aligned16(q_bf16) || !aligned16(k_new_bf16) || !aligned16(v_new_bf16) || !aligned16(k_pool) ||
        !aligned16(v_pool) || !aligned16(seg_table) || !aligned16(out_bf16) || !aligned16(block_tables_dev) ||
        !aligned16(seq_lens_dev))
        return DGQ_ERR_INVALID_ARG;
    int nsm = 0;
    if (device_sm_count(&nsm) != 0) return DGQ_ERR_CUDA;
    if (!workspace || !aligned16(workspace) ||
        workspace_bytes < dgq::attn_layout(batch, num_q_heads, num_kv_heads, nsm).total)
        return DGQ_ERR_WORKSPACE;
    bool map_failed = false;
    cudaError_t e = dgq::launch_attn(format, q_bf16, k_new_bf16, v_new_bf16, k_pool, v_pool, seg_table,
                                     v_seg_table, k_group_params, v_group_params, block_tables_dev, seq_lens_dev,
                                     max_seqlen, batch, num_q_heads, num_kv_heads, block_size, max_blocks_per_seq,
                                     num_blocks, out_bf16, workspace, nsm, &map_failed,
                                     static_cast<cudaStream_t>(cuda_stream));
    if (map_failed) return DGQ_ERR_INVALID_ARG;
    return e == cudaSuccess ? DGQ_OK : DGQ_ERR_CUDA;
}
}  // namespace

size_t dgq_prefill_workspace_size(int32_t batch, int32_t num_kv_heads)
{
    if (batch <= 0 || num_kv_heads <= 0) return 0;
    return dgq::prefill_workspace_bytes(batch, num_kv_heads);
}

namespace {

// Checks shared by the two prefill calls (source, sizes, statistics array, workspace).
dgq_status prefill_checks(const void *k_src, const void *v_src, int32_t num_src_blocks, const int32_t *src_bt,
                          int32_t max_src_blocks, int32_t batch, int32_t max_seqlen, int32_t num_kv_heads,
                          int32_t head_dim, int32_t block_size, const void *stats, int32_t max_windows,
                          const void *workspace, size_t workspace_bytes)
{
    if (head_dim != DGQ_HEAD_DIM || !block_size_ok(block_size)) return DGQ_ERR_UNSUPPORTED;
    if (batch <= 0 || batch > kMaxBatch || max_seqlen < 0 || num_kv_heads <= 0 || num_src_blocks <= 0 ||
        max_src_blocks <= 0)
        return DGQ_ERR_INVALID_ARG;
    if ((int64_t)max_seqlen > (int64_t)max_src_blocks * block_size) return DGQ_ERR_INVALID_ARG;
    if (max_windows < (max_seqlen + DGQ_WINDOW - 1) / DGQ_WINDOW || max_windows <= 0) return DGQ_ERR_INVALID_ARG;
    const int64_t windows = (int64_t)batch * num_kv_heads * max_windows;
    if (windows >= INT32_MAX || (int64_t)num_src_blocks * num_kv_heads * block_size >= INT32_MAX)
        return DGQ_ERR_UNSUPPORTED;
    if (!k_src || !v_src || !src_bt || !stats) return DGQ_ERR_INVALID_ARG;
    if (!aligned16(k_src) || !aligned16(v_src) || !aligned16(src_bt) || !aligned16(stats))
        return DGQ_ERR_INVALID_ARG;
    if (!workspace || !aligned16(workspace) || workspace_bytes < dgq::prefill_workspace_bytes(batch, num_kv_heads))
        return DGQ_ERR_WORKSPACE;
    return DGQ_OK;
}

}  // namespace

dgq_status dgq_prefill_chunk_stats(const void *k_src_bf16, const void *v_src_bf16, int32_t num_src_blocks,
                                   const int32_t *src_block_tables_dev, int32_t max_src_blocks_per_seq,
                                   const int32_t *chunk_begin_dev, const int32_t *chunk_end_dev, int32_t batch,
                                   int32_t max_seqlen, int32_t num_kv_heads, int32_t head_dim, int32_t block_size,
                                   float *window_stats, int32_t max_windows, int32_t flags, void *workspace,
                                   size_t workspace_bytes, void *cuda_stream)
{
    if (flags & ~DGQ_PREFILL_V_VARIANCE) return DGQ_ERR_INVALID_ARG;
    dgq_status st = prefill_checks(k_src_bf16, v_src_bf16, num_src_blocks, src_block_tables_dev,
                                   max_src_blocks_per_seq, batch, max_seqlen, num_kv_heads, head_dim, block_size,
                                   window_stats, max_windows, workspace, workspace_bytes);
    if (st != DGQ_OK) return st;
    if (!chunk_begin_dev || !chunk_end_dev || !aligned16(chunk_begin_dev) || !aligned16(chunk_end_dev))
        return DGQ_ERR_INVALID_ARG;
    int nsm = 0;
    if (device_sm_count(&nsm) != 0) return DGQ_ERR_CUDA;
    const dgq::SourceDesc src = {k_src_bf16, v_src_bf16, 0, src_block_tables_dev, max_src_blocks_per_seq,
                                 num_src_blocks};
    bool map_failed = false;
    const cudaError_t e = dgq::launch_prefill_stats(src, chunk_begin_dev, chunk_end_dev, batch, max_seqlen,
                                                    num_kv_heads, block_size, window_stats, max_windows,
                                                    (flags & DGQ_PREFILL_V_VARIANCE) != 0, workspace, nsm,
                                                    &map_failed, static_cast<cudaStream_t>(cuda_stream));
    if (map_failed) return DGQ_ERR_INVALID_ARG;
    return e == cudaSuccess ? DGQ_OK : DGQ_ERR_CUDA;
}

dgq_status dgq_prefill_finish(const void *k_src_bf16, const void *v_src_bf16, int32_t num_src_blocks,
                              const int32_t *src_block_tables_dev, int32_t max_src_blocks_per_seq,
                              const int32_t *seq_lens_dev, int32_t batch, int32_t max_seqlen, int32_t num_kv_heads,
                              int32_t head_dim, int32_t block_size, const float *window_stats, int32_t max_windows,
                              const int32_t *block_tables_dev, int32_t max_blocks_per_seq, uint8_t *k_pool,
                              uint8_t *v_pool, int32_t num_blocks, dgq_seg_record *seg_table,
                              dgq_seg_record *v_seg_table, const dgq_compress_options *options, void *workspace,
                              size_t workspace_bytes, void *cuda_stream)
{
    return dgq_prefill_finish_ex(k_src_bf16, v_src_bf16, num_src_blocks, src_block_tables_dev,
                                 max_src_blocks_per_seq, seq_lens_dev, batch, max_seqlen, num_kv_heads, head_dim,
                                 block_size, window_stats, max_windows, block_tables_dev, max_blocks_per_seq, k_pool,
                                 v_pool, num_blocks, seg_table, v_seg_table, options, nullptr, 0, workspace,
                                 workspace_bytes, cuda_stream);
}

dgq_status dgq_prefill_finish_ex(const void *k_src_bf16, const void *v_src_bf16, int32_t num_src_blocks,
                                 const int32_t *src_block_tables_dev, int32_t max_src_blocks_per_seq,
                                 const int32_t *seq_lens_dev, int32_t batch, int32_t max_seqlen,
                                 int32_t num_kv_heads, int32_t head_dim, int32_t block_size,
                                 const float *window_stats, int32_t max_windows, const int32_t *block_tables_dev,
                                 int32_t max_blocks_per_seq, uint8_t *k_pool, uint8_t *v_pool, int32_t num_blocks,
                                 dgq_seg_record *seg_table, dgq_seg_record *v_seg_table,
                                 const dgq_compress_options *options, const int32_t *pair_flags,
                                 int32_t flag_mask, void *workspace, size_t workspace_bytes, void *cuda_stream)
{
    if (v_seg_table && !aligned16(v_seg_table)) return DGQ_ERR_INVALID_ARG;
    if (pair_flags && !aligned16(pair_flags)) return DGQ_ERR_INVALID_ARG;
    dgq::GroupSettings gs = {DGQ_MAX_SEG, 0.0f};
    if (options) {
        if (options->max_groups < 1 || options->max_groups > DGQ_MAX_SEG || !(options->min_var >= 0.0f) ||
            !(options->min_var <= 3.4e38f))
            return DGQ_ERR_INVALID_ARG;
        gs.max_groups = options->max_groups;
        gs.min_var = options->min_var;
    }
    dgq_status st = prefill_checks(k_src_bf16, v_src_bf16, num_src_blocks, src_block_tables_dev,
                                   max_src_blocks_per_seq, batch, max_seqlen, num_kv_heads, head_dim, block_size,
                                   window_stats, max_windows, workspace, workspace_bytes);
    if (st != DGQ_OK) return st;
    if (num_blocks <= 0 || max_blocks_per_seq <= 0 ||
        (int64_t)max_seqlen > (int64_t)max_blocks_per_seq * block_size ||
        (int64_t)num_blocks * num_kv_heads * block_size >= INT32_MAX)
        return DGQ_ERR_INVALID_ARG;
    if (!seq_lens_dev || !block_tables_dev || !k_pool || !v_pool || !seg_table) return DGQ_ERR_INVALID_ARG;
    if (!aligned16(seq_lens_dev) || !aligned16(block_tables_dev) || !aligned16(k_pool) || !aligned16(v_pool) ||
        !aligned16(seg_table))
        return DGQ_ERR_INVALID_ARG;
    int nsm = 0;
    if (device_sm_count(&nsm) != 0) return DGQ_ERR_CUDA;
    const dgq::SourceDesc src = {k_src_bf16, v_src_bf16, 0, src_block_tables_dev, max_src_blocks_per_seq,
                                 num_src_blocks};
    bool map_failed = false;
    const cudaError_t e = dgq::launch_prefill_finish(
        src, seq_lens_dev, batch, max_seqlen, num_kv_heads, block_size, window_stats, max_windows, block_tables_dev,
        max_blocks_per_seq, k_pool, v_pool, num_blocks, seg_table, v_seg_table, gs, pair_flags, flag_mask,
        workspace, nsm, &map_failed, static_cast<cudaStream_t>(cuda_stream));
    if (map_failed) return DGQ_ERR_INVALID_ARG;
    return e == cudaSuccess ? DGQ_OK : DGQ_ERR_CUDA;
}

size_t dgq_encode_format_workspace_size(int32_t batch, int32_t num_kv_heads)
{
    if (batch <= 0 || num_kv_heads <= 0) return 0;
    return dgq::format_workspace_bytes(batch, num_kv_heads);
}

dgq_status dgq_encode_format(int32_t format, const void *k_bf16, const void *v_bf16, int32_t total_tokens,
                             const int32_t *cu_seqlens_dev, int32_t batch, int32_t max_seqlen, int32_t num_kv_heads,
                             int32_t head_dim, int32_t block_size, const int32_t *block_tables_dev,
                             int32_t max_blocks_per_seq, uint8_t *k_pool, uint8_t *v_pool, int32_t num_blocks,
                             dgq_seg_record *seg_table, float *k_group_params, float *v_group_params,
                             void *workspace, size_t workspace_bytes, void *cuda_stream)
{
    if (format != DGQ_FORMAT_FIXED64 && format != DGQ_FORMAT_SYM_INT8 && format != DGQ_FORMAT_FP8_E4M3)
        return DGQ_ERR_INVALID_ARG;
    if (format == DGQ_FORMAT_FIXED64 && (!k_group_params || !v_group_params || !aligned16(k_group_params) ||
                                         !aligned16(v_group_params)))
        return DGQ_ERR_INVALID_ARG;
    if (head_dim != DGQ_HEAD_DIM || !block_size_ok(block_size)) return DGQ_ERR_UNSUPPORTED;
    if (batch <= 0 || batch > kMaxBatch || max_seqlen < 0 || total_tokens < 0 || num_kv_heads <= 0 ||
        num_blocks <= 0 || max_blocks_per_seq <= 0)
        return DGQ_ERR_INVALID_ARG;
    if ((int64_t)max_seqlen > (int64_t)max_blocks_per_seq * block_size) return DGQ_ERR_INVALID_ARG;
    // grid: one CTA column per (request, head) pair, one row per 256 tokens
    if ((int64_t)batch * num_kv_heads >= INT32_MAX || (max_seqlen + 255) / 256 > 65535 ||
        (int64_t)num_blocks * num_kv_heads * block_size >= INT32_MAX)
        return DGQ_ERR_UNSUPPORTED;
    if (!k_bf16 || !v_bf16 || !cu_seqlens_dev || !block_tables_dev || !k_pool || !v_pool || !seg_table)
        return DGQ_ERR_INVALID_ARG;
    if (!aligned16(k_bf16) || !aligned16(v_bf16) || !aligned16(k_pool) || !aligned16(v_pool) ||
        !aligned16(seg_table) || !aligned16(cu_seqlens_dev) || !aligned16(block_tables_dev))
        return DGQ_ERR_INVALID_ARG;
    if (!workspace || !aligned16(workspace) || workspace_bytes < dgq::format_workspace_bytes(batch, num_kv_heads))
        return DGQ_ERR_WORKSPACE;
    const cudaError_t e = dgq::launch_format_encode(
        format, k_bf16, v_bf16, total_tokens, cu_seqlens_dev, batch, max_seqlen, num_kv_heads, block_size,
        block_tables_dev, max_blocks_per_seq, k_pool, v_pool, num_blocks, k_group_params, v_group_params, seg_table,
        workspace, static_cast<cudaStream_t>(cuda_stream));
    return e == cudaSuccess ? DGQ_OK : DGQ_ERR_CUDA;
}

dgq_status dgq_workspace_init(void *workspace, size_t workspace_bytes, void *cuda_stream)
{
    if (!workspace || workspace_bytes == 0) return DGQ_ERR_INVALID_ARG;
    cudaError_t e = cudaMemsetAsync(workspace, 0, workspace_bytes, static_cast<cudaStream_t>(cuda_stream));
    return e == cudaSuccess ? DGQ_OK : DGQ_ERR_CUDA;
}

dgq_status dgq_workspace_error(const void *workspace, void *cuda_stream, int32_t *device_error)
{
    if (!workspace || !device_error) return DGQ_ERR_INVALID_ARG;
    uint32_t word = 0;
    cudaStream_t s = static_cast<cudaStream_t>(cuda_stream);
    if (cudaMemcpyAsync(&word, workspace, sizeof(word), cudaMemcpyDeviceToHost, s) != cudaSuccess)
        return DGQ_ERR_CUDA;
    if (cudaStreamSynchronize(s) != cudaSuccess) return DGQ_ERR_CUDA;
    *device_error = (int32_t)word;
    return word ? DGQ_ERR_DEVICE : DGQ_OK;
}

// ---- host block pool --------------------------------------------------------------------

struct dgq_pool {
    int32_t num_blocks;
    std::vector<int32_t> free_list;  // stack of free ids
    std::vector<uint8_t> is_free;
};

dgq_pool *dgq_pool_create(int32_t num_blocks)
{
    if (num_blocks <= 0) return nullptr;
    dgq_pool *p = new (std::nothrow) dgq_pool;
    if (!p) return nullptr;
    p->num_blocks = num_blocks;
    p->free_list.resize(num_blocks);
    p->is_free.assign(num_blocks, 1);
    for (int32_t i = 0; i < num_blocks; ++i) p->free_list[i] = num_blocks - 1 - i;  // pops 0, 1, 2, ...
    return p;
}

void dgq_pool_destroy(dgq_pool *pool) { delete pool; }

dgq_status dgq_pool_alloc(dgq_pool *pool, int32_t n, int32_t *out_ids)
{
    if (!pool || n < 0 || (n > 0 && !out_ids)) return DGQ_ERR_INVALID_ARG;
    if ((size_t)n > pool->free_list.size()) return DGQ_ERR_POOL_EXHAUSTED;
    for (int32_t i = 0; i < n; ++i) {
        int32_t id = pool->free_list.back();
        pool->free_list.pop_back();
        pool->is_free[id] = 0;
        out_ids[i] = id;
    }
    return DGQ_OK;
}

dgq_status dgq_pool_free(dgq_pool *pool, const int32_t *ids, int32_t n)
{
    if (!pool || n < 0 || (n > 0 && !ids)) return DGQ_ERR_INVALID_ARG;
    std::vector<uint8_t> seen;
    for (int32_t i = 0; i < n; ++i) {  // validate all first: nothing is freed on error
        int32_t id = ids[i];
        if (id < 0 || id >= pool->num_blocks || pool->is_free[id]) return DGQ_ERR_INVALID_ARG;
        if (seen.empty()) seen.assign(pool->num_blocks, 0);
        if (seen[id]) return DGQ_ERR_INVALID_ARG;
        seen[id] = 1;
    }
    for (int32_t i = 0; i < n; ++i) {
        pool->is_free[ids[i]] = 1;
        pool->free_list.push_back(ids[i]);
    }
    return DGQ_OK;
}

int32_t dgq_pool_num_free(const dgq_pool *pool) { return pool ? (int32_t)pool->free_list.size() : -1; }

dgq_status dgq_pool_alloc_table_row(dgq_pool *pool, int32_t len, int32_t block_size, int32_t *table, int32_t row,
                                    int32_t max_blocks_per_seq)
{
    if (!pool || !table || len < 0 || row < 0 || max_blocks_per_seq <= 0 || block_size <= 0)
        return DGQ_ERR_INVALID_ARG;
    const int32_t n = (len + block_size - 1) / block_size;
    if (n > max_blocks_per_seq) return DGQ_ERR_INVALID_ARG;
    int32_t *dst = table + (int64_t)row * max_blocks_per_seq;
    dgq_status s = dgq_pool_alloc(pool, n, dst);
    if (s != DGQ_OK) return s;
    for (int32_t i = n; i < max_blocks_per_seq; ++i) dst[i] = 0;
    return DGQ_OK;
}

}  // extern "C"
