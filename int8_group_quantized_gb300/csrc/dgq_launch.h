// dgq_launch.h -- internal declarations shared by the host ABI and the kernel translation units.
#pragma once

#include <cuda_runtime.h>
#include <cudaTypedefs.h>
#include <stddef.h>
#include <stdint.h>

#include "dgq.h"

namespace dgq {

// Requests per call the entry points accept (the kernels keep per-request prefixes on chip).  A
// kernel's dynamic shared-memory limit is a property of the kernel shared by every host thread, so
// the launchers raise it once, to what a call of this many requests needs, and never lower it.
constexpr int32_t kMaxCallBatch = 8192;

// Group-selection settings passed to both compress kernels (see dgq_compress_options).
struct GroupSettings {
    int32_t max_groups;
    float min_var;
};

// Where compress reads K and V: packed rows [T, Hkv, 128] (bt == null) or a bf16 paged cache
// [num_blocks, Hkv, bs, 128] with its [B, max_blocks] block table.
struct SourceDesc {
    const void *k, *v;
    int32_t T;
    const int32_t *bt;
    int32_t max_blocks, num_blocks;
};

struct CompressLayout {
    size_t off_prog, off_params, off_mean, off_mm, off_agg, total;
};
CompressLayout compress_layout(int32_t batch, int32_t max_seqlen, int32_t Hkv);
cudaError_t launch_compress(const SourceDesc &src, const int32_t *cu, int32_t B,
                            int32_t max_seqlen, int32_t Hkv, int32_t bs, const int32_t *bt, int32_t max_blocks,
                            uint8_t *kpool, uint8_t *vpool, int32_t num_blocks, dgq_seg_record *table, void *ws,
                            GroupSettings gs, int nsm, cudaStream_t stream);

// Compression of calls whose requests are all at most cluster_compress_max_seqlen() tokens:
// pairs segmented inside thread-block clusters (no grid-wide step, no workspace beyond the
// header).
int32_t cluster_compress_max_seqlen();
cudaError_t launch_compress_cluster(const SourceDesc &src, const int32_t *cu, int32_t B,
                                    int32_t max_seqlen, int32_t Hkv, int32_t bs, const int32_t *bt,
                                    int32_t max_blocks, uint8_t *kpool, uint8_t *vpool, int32_t num_blocks,
                                    dgq_seg_record *table, void *ws, GroupSettings gs, cudaStream_t stream);

struct AttnLayout {
    size_t off_count, off_held, off_part, total;
};
AttnLayout attn_layout(int32_t batch, int32_t Hq, int32_t Hkv, int nsm);
// format: a dgq_format (DGQ and SYM_INT8 decode through the records; kpar / vpar are read for
// FIXED64 only).  vtable non-null (DGQ only): independent V segmentation, V's records there.
cudaError_t launch_attn(int32_t format, const void *q, const void *knew, const void *vnew, const uint8_t *kpool,
                        const uint8_t *vpool, const dgq_seg_record *table, const dgq_seg_record *vtable,
                        const float *kpar, const float *vpar,
                        const int32_t *bt, const int32_t *seq_lens, int32_t max_seqlen, int32_t B, int32_t Hq,
                        int32_t Hkv, int32_t bs, int32_t max_blocks, int32_t num_blocks, void *out, void *ws, int nsm,
                        bool *map_failed, cudaStream_t stream);

// Comparison encodings (FIXED64, SYM_INT8, FP8_E4M3) of packed rows into the paged cache.
size_t format_workspace_bytes(int32_t B, int32_t Hkv);
cudaError_t launch_format_encode(int32_t format, const void *k, const void *v, int32_t T, const int32_t *cu, int32_t B,
                                 int32_t max_seqlen, int32_t Hkv, int32_t bs, const int32_t *bt, int32_t max_blocks,
                                 uint8_t *kpool, uint8_t *vpool, int32_t num_blocks, float *kpar, float *vpar,
                                 dgq_seg_record *table, void *ws, cudaStream_t stream);

cudaError_t launch_append(const void *k_new, const void *v_new, int32_t B, int32_t Hkv, int32_t bs,
                          const int32_t *bt, int32_t max_blocks, uint8_t *kpool, uint8_t *vpool, int32_t num_blocks,
                          dgq_seg_record *table, dgq_seg_record *vtable, int32_t *flags, void *ws,
                          cudaStream_t stream);

// Compression in two phases for chunked prefill: window statistics of each request's chunk
// [begin, end) from a bf16 paged cache, then segmentation and codes for whole requests.
size_t prefill_workspace_bytes(int32_t B, int32_t Hkv);
cudaError_t launch_prefill_stats(const SourceDesc &src, const int32_t *begin, const int32_t *end, int32_t B,
                                 int32_t max_seqlen, int32_t Hkv, int32_t bs, float *stats, int32_t max_windows,
                                 bool v_variance, void *ws, int nsm, bool *map_failed, cudaStream_t stream);
// vtable non-null: independent V segmentation (V's records there)
cudaError_t launch_prefill_finish(const SourceDesc &src, const int32_t *seq_lens, int32_t B, int32_t max_seqlen,
                                  int32_t Hkv, int32_t bs, const float *stats, int32_t max_windows,
                                  const int32_t *bt, int32_t max_blocks, uint8_t *kpool, uint8_t *vpool,
                                  int32_t num_blocks, dgq_seg_record *table, dgq_seg_record *vtable,
                                  GroupSettings gs, const int32_t *sel, int32_t sel_mask, void *ws, int nsm,
                                  bool *map_failed, cudaStream_t stream);

// cuTensorMapEncodeTiled from the driver (through the runtime's entry-point query), or null.
PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder();

}  // namespace dgq
