/*
 * dgq.h -- C ABI of libdgq.so: an LLM decoder's KV cache compressed to INT8 by dynamic
 * group quantisation (DGQ), stored in fixed-size paged blocks, and read by decode-step
 * attention.  sm_103a (GB300) only.
 *
 * Sources, cited by title and section:
 *   [DGQ]   "DeepSeek KV-cache dynamic group quantisation (DGQ)" article (pptc.cn news
 *           101026): section 2.2 (per-head variance curve along L, 16-token windows,
 *           boundaries at abrupt variance changes, 3-5 segments, independent min/max INT8
 *           per segment, per-token segment id used at decode), section 3.2 (length-aware
 *           n_groups in compress(); decompress is the hot part and belongs in CUDA),
 *           section 3.3 (storage formula).
 *   [PAGED] "DeepSeek-V4 high-concurrency KV-cache bottleneck" article (deepseek.csdn.net),
 *           "PagedAttention implementation" section (logical blocks mapped to scattered
 *           physical blocks via a page table with a free list) and its modified forward()
 *           that passes block_tables to paged_attention().
 *
 * Conventions for every call below:
 *   - Head dimension D is 128; block_size (tokens per physical block) is 16, 32 or 64.
 *   - Device pointers are raw CUDA device addresses; the caller owns every buffer.  The
 *     library allocates no device memory.  Pointers must be 16-byte aligned.
 *   - `cuda_stream` is a cudaStream_t passed as void* (NULL = legacy default stream).
 *     Calls enqueue work on it and return without synchronising.
 *   - All argument checks happen on the host, before any launch; a failed check launches
 *     nothing and returns a negative dgq_status.  Block-table entries and sequence lengths
 *     live on the device and are trusted (each entry < num_blocks; seq_lens[b] <=
 *     max_seqlen).
 *   - A workspace is a caller-owned device buffer of at least the queried size.  It must be
 *     zero-filled before its first use (dgq_workspace_init); every call leaves it ready for
 *     the next one.  Calls that share a workspace must be ordered on one stream.  Device-side
 *     failures (a wait that timed out) are recorded in the workspace and read with
 *     dgq_workspace_error.
 *   - bf16 values are IEEE bfloat16 bit patterns; fp32 is IEEE binary32.
 *   - Host threads: each launcher keeps the launch shape of its kernel (occupancy, shared-memory
 *     limit) for the device it last ran on, per host thread; host threads share no library
 *     state, so calls from several threads at once are safe (each on its own stream and
 *     workspace, as above), on any number of devices.
 *   - CUDA graphs: every compute call (compress, decode, append, the prefill calls, the
 *     comparison formats) enqueues only kernel launches and workspace memsets on its stream,
 *     with no host synchronisation, so it may be captured into a graph on a capturing stream;
 *     a replay does what the call does.  Make one call on the device and host thread first
 *     (outside the capture) so that the launcher's per-device setup is done; the decode merge's
 *     programmatic dependent launch becomes a programmatic edge of the graph.
 *     dgq_workspace_error reads the workspace back and synchronises: not inside a capture.
 */
#ifndef DGQ_H
#define DGQ_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define DGQ_HEAD_DIM 128
#define DGQ_WINDOW 16   /* variance-smoothing window, [DGQ] section 2.2 */
#define DGQ_MAX_SEG 5   /* segments per (request, KV head), [DGQ] sections 2.2 and 3.2 */

typedef enum dgq_status {
    DGQ_OK = 0,
    DGQ_ERR_INVALID_ARG = -1,    /* null pointer, bad size, misaligned pointer */
    DGQ_ERR_UNSUPPORTED = -2,    /* shape outside what the kernels handle (D, block size, G) */
    DGQ_ERR_WORKSPACE = -3,      /* workspace missing or smaller than the queried size */
    DGQ_ERR_CUDA = -4,           /* a CUDA runtime call or launch failed */
    DGQ_ERR_POOL_EXHAUSTED = -5, /* block pool has fewer free blocks than requested */
    DGQ_ERR_DEVICE = -6,         /* a device-side wait timed out (see dgq_workspace_error) */
    DGQ_ERR_SCRATCH_LIMIT = -7   /* the problem needs more scratch than the library's fixed array */
} dgq_status;

/*
 * Segment record of one (request, KV head): exactly 128 bytes.
 * [DGQ] section 2.2 keeps one segment id per token and looks up the segment's min/max at
 * decode; here the id is implicit: token t belongs to segment s = max{i : start[i] <= t}.
 * Dequantised value of code q in segment s: x = min[s] + q * scale[s] (fp32 values; the
 * decode kernel evaluates it in fp32).  Entries i >= n_seg hold start = seq_len, min =
 * scale = 0.  A record with seq_len == 0 has n_seg == 0.
 */
typedef struct dgq_seg_record {
    int32_t n_seg;              /* 1..5 (0 when seq_len == 0) */
    int32_t seq_len;            /* tokens compressed into the cache for this (request, head) */
    int32_t start[DGQ_MAX_SEG]; /* start[0] = 0, ascending, multiples of 16 */
    float k_min[DGQ_MAX_SEG];
    float k_scale[DGQ_MAX_SEG]; /* (max - min) / 255, or 0 for a flat segment */
    float v_min[DGQ_MAX_SEG];
    float v_scale[DGQ_MAX_SEG];
    float k_inv_last;           /* 255 / (max - min) of the last segment (0 if flat or n_seg == 0): */
    float v_inv_last;           /*   the encoder's factor, kept so that dgq_append encodes alike */
    int32_t pad[3];             /* zero */
} dgq_seg_record;

/* ---------------------------------------------------------------------------------------
 * dgq_compress -- DGQ encode of one layer for a batch of requests into a paged cache.
 *
 * Computes, per (request b, KV head h), [DGQ] section 2.2 / 3.2:
 *   1. per-token variance of K over D (fp32, population, mean first; the sums use the
 *      balanced pairwise order sum(left half) + sum(right half));
 *   2. the mean of that variance over each non-overlapping 16-token window (the last,
 *      partial, window averaged over its own token count);
 *   3. n_groups(L) = 2 if L < 2048, 3 if L < 16384, else min(5, floor(log2(L/1024)) + 2),
 *      and the n_groups-1 largest jumps |m[w+1] - m[w]| between adjacent window means
 *      (ties to the earlier window; at most W-1 of them), each starting a segment at
 *      token 16(w+1); one segmentation per (request, head), shared by K and V;
 *   4. fp32 min/max of K and of V over each segment (all tokens x D), scale = (max-min)/255,
 *      and codes q = rint((x - min) * (255 / (max - min))) (two rounded fp32 operations,
 *      round-half-even), 0 for a flat segment;
 *   5. stores the codes of token t at pool[block_tables[b][t / bs]][h][t % bs][0..128)
 *      ([PAGED] PagedAttention: logical block t / bs -> physical block), and the record.
 *
 * k_bf16, v_bf16   [T, Hkv, 128] bf16, device.  Packed variable length: request b owns
 *                  rows cu_seqlens[b] .. cu_seqlens[b+1]-1.
 * total_tokens     T, the number of rows the K and V buffers hold (>= cu_seqlens[batch]);
 *                  the kernels never read past row T.
 * cu_seqlens_dev   [batch+1] int32, device, non-decreasing, cu_seqlens[0] = 0.
 * max_seqlen       host upper bound on every request length (sizes the workspace).
 * block_tables_dev [batch, max_blocks_per_seq] int32, device.  The first ceil(L_b / bs)
 *                  entries of row b name distinct physical blocks < num_blocks; requests
 *                  of one call use disjoint blocks.  max_seqlen <= max_blocks_per_seq * bs.
 * k_pool, v_pool   [num_blocks, Hkv, block_size, 128] uint8, device; only the slots of
 *                  tokens 0..L_b-1 are written (the rest of a last block is untouched).
 * seg_table        [batch, Hkv] dgq_seg_record, device, written in full.
 * workspace        >= dgq_compress_workspace_size(batch, max_seqlen, num_kv_heads) bytes.
 * Inputs must be finite; requests may be empty (L = 0 writes a record with n_seg = 0).
 * Finite values large enough to overflow the fp32 variance (|x| beyond about 2^62) give a
 * window mean of +inf; the jump between two such adjacent windows is undefined (inf - inf) and
 * is no boundary candidate, and a pair left with fewer candidates gets fewer segments.
 * Kernel: when every request is at most 4096 tokens long, a non-cooperative kernel of
 * thread-block clusters that each segment whole (request, head) pairs; otherwise one
 * cooperative kernel with one block per SM, in which the whole GPU takes part (the call then
 * needs the GPU to itself for its duration, as any cooperative launch).
 */
dgq_status dgq_compress(const void *k_bf16, const void *v_bf16, int32_t total_tokens,
                        const int32_t *cu_seqlens_dev, int32_t batch, int32_t max_seqlen, int32_t num_kv_heads,
                        int32_t head_dim, int32_t block_size, const int32_t *block_tables_dev,
                        int32_t max_blocks_per_seq, uint8_t *k_pool, uint8_t *v_pool,
                        int32_t num_blocks, dgq_seg_record *seg_table, void *workspace,
                        size_t workspace_bytes, void *cuda_stream);

size_t dgq_compress_workspace_size(int32_t batch, int32_t max_seqlen, int32_t num_kv_heads);

/*
 * Group-selection settings, [DGQ] section 5.3 (tuning switches of the article's vLLM
 * integration: a maximum group count, and a variance threshold below which tokens share a
 * group).
 *   max_groups  1..5: at most this many segments per (request, KV head): n_groups becomes
 *               min(n_groups(L), max_groups).  5 leaves the length rule alone.
 *   min_var     >= 0, finite: a window whose mean variance is below min_var is quiet, and no
 *               boundary is placed between two quiet windows (a jump between a quiet and a
 *               louder window is still a candidate); with fewer candidates than boundaries the
 *               pair gets fewer segments.  0 changes nothing (window means are >= 0).
 */
typedef struct dgq_compress_options {
    int32_t max_groups;
    float min_var;
} dgq_compress_options;

/* dgq_compress with explicit settings; options == NULL is { 5, 0.0f }, i.e. dgq_compress.
 * Settings outside the ranges above: DGQ_ERR_INVALID_ARG. */
dgq_status dgq_compress_ex(const void *k_bf16, const void *v_bf16, int32_t total_tokens,
                           const int32_t *cu_seqlens_dev, int32_t batch, int32_t max_seqlen, int32_t num_kv_heads,
                           int32_t head_dim, int32_t block_size, const int32_t *block_tables_dev,
                           int32_t max_blocks_per_seq, uint8_t *k_pool, uint8_t *v_pool,
                           int32_t num_blocks, dgq_seg_record *seg_table, void *workspace,
                           size_t workspace_bytes, const dgq_compress_options *options, void *cuda_stream);

/* ---------------------------------------------------------------------------------------
 * dgq_compress_paged -- dgq_compress reading K and V straight from a bf16 paged cache (the
 * layout a serving engine keeps them in after prefill, [PAGED] "PagedAttention implementation"),
 * so they need not be gathered into packed rows first: one read of the bf16 cache per pass and
 * no extra copy.  Same computation and outputs as dgq_compress_ex on the gathered rows.
 *
 * k_src_bf16, v_src_bf16  [num_src_blocks, Hkv, block_size, 128] bf16, device: token t of
 *                         request b, head h is row src[src_block_tables[b][t / bs]][h][t % bs].
 * src_block_tables_dev    [batch, max_src_blocks_per_seq] int32, device; max_seqlen <=
 *                         max_src_blocks_per_seq * block_size.  An entry outside
 *                         [0, num_src_blocks) is flagged in the workspace (block 0 read instead).
 * cu_seqlens_dev          [batch+1] int32, device: lengths only (L_b = cu[b+1] - cu[b]); no
 *                         packed rows are read.
 * The destination (block_size, block tables, pools, records), workspace and options are those
 * of dgq_compress_ex; source and destination use the same block_size.
 */
dgq_status dgq_compress_paged(const void *k_src_bf16, const void *v_src_bf16, int32_t num_src_blocks,
                              const int32_t *src_block_tables_dev, int32_t max_src_blocks_per_seq,
                              const int32_t *cu_seqlens_dev, int32_t batch, int32_t max_seqlen,
                              int32_t num_kv_heads, int32_t head_dim, int32_t block_size,
                              const int32_t *block_tables_dev, int32_t max_blocks_per_seq, uint8_t *k_pool,
                              uint8_t *v_pool, int32_t num_blocks, dgq_seg_record *seg_table, void *workspace,
                              size_t workspace_bytes, const dgq_compress_options *options, void *cuda_stream);

/* ---------------------------------------------------------------------------------------
 * Compression in two phases, for chunked prefill.  dgq_compress_paged reads the bf16 cache
 * twice from HBM (statistics, then codes).  When prefill writes a long request chunk by chunk,
 * the statistics of each chunk can be taken right after the chunk is written, while it is
 * still in L2; the finishing call then reads the cache from HBM once, for the codes.  Results
 * are identical to dgq_compress_paged on the complete cache (a window's statistics depend on
 * its 16 tokens only; segmentation and codes need the whole request, so they wait for the end).
 * [DGQ] section 3.2 (compression inside the inference pipeline); [PAGED] chunked prefill into
 * the paged cache.
 *
 * window_stats     [batch, Hkv, max_windows, 8] fp32, device, caller-owned: per 16-token window
 *                  (K mean variance, K min, K max, V min, V max, V mean variance (0 unless
 *                  DGQ_PREFILL_V_VARIANCE), 2 zeros); max_windows >= ceil(max_seqlen / 16).
 *                  Written by dgq_prefill_chunk_stats, read by dgq_prefill_finish.
 *
 * Independent V segmentation (a group-selection variant; the method itself derives one
 * segmentation from K, [DGQ] section 2.2): V is segmented by the same rule applied to V's own
 * variance and encoded with its own segments.  Statistics taken with DGQ_PREFILL_V_VARIANCE and
 * a non-NULL v_seg_table in dgq_prefill_finish select it: seg_table then receives K's records
 * (V fields 0) and v_seg_table V's (start, n_seg, v_min, v_scale, v_inv_last; K fields 0); decode
 * with dgq_paged_decode_attn_split; append the decode steps' tokens with dgq_append_split.
 * workspace        >= dgq_prefill_workspace_size(batch, Hkv) bytes, zero-filled before first use.
 * The bf16 source (k_src, v_src, src block tables) is as for dgq_compress_paged.
 */
size_t dgq_prefill_workspace_size(int32_t batch, int32_t num_kv_heads);

#define DGQ_PREFILL_V_VARIANCE 1 /* dgq_prefill_chunk_stats flag: also V's mean variance per window */

/* Statistics of the windows of tokens [chunk_begin[b], chunk_end[b]) of every request b (device
 * arrays [batch] int32).  chunk_begin[b] is a multiple of 16; chunk_end[b] is a multiple of 16
 * unless the chunk is the request's last one (its partial last window is averaged over its own
 * tokens, as in dgq_compress); an empty range (begin == end) skips the request.  A range that is
 * not window-aligned or ends past max_seqlen is flagged in the workspace and skipped.  flags: 0 or
 * DGQ_PREFILL_V_VARIANCE (other bits: DGQ_ERR_INVALID_ARG). */
dgq_status dgq_prefill_chunk_stats(const void *k_src_bf16, const void *v_src_bf16, int32_t num_src_blocks,
                                   const int32_t *src_block_tables_dev, int32_t max_src_blocks_per_seq,
                                   const int32_t *chunk_begin_dev, const int32_t *chunk_end_dev, int32_t batch,
                                   int32_t max_seqlen, int32_t num_kv_heads, int32_t head_dim, int32_t block_size,
                                   float *window_stats, int32_t max_windows, int32_t flags, void *workspace,
                                   size_t workspace_bytes, void *cuda_stream);

/* Segmentation of every (request, head) from window_stats (every window of tokens
 * [0, seq_lens[b]) must have been written by earlier dgq_prefill_chunk_stats calls), then the
 * codes of all tokens from the bf16 cache into the INT8 pools and the records, as
 * dgq_compress_paged with the same options would write them.  v_seg_table: NULL for the method's
 * shared segmentation, else [batch, Hkv] records for independent V segmentation (above).  Two
 * launches. */
dgq_status dgq_prefill_finish(const void *k_src_bf16, const void *v_src_bf16, int32_t num_src_blocks,
                              const int32_t *src_block_tables_dev, int32_t max_src_blocks_per_seq,
                              const int32_t *seq_lens_dev, int32_t batch, int32_t max_seqlen, int32_t num_kv_heads,
                              int32_t head_dim, int32_t block_size, const float *window_stats, int32_t max_windows,
                              const int32_t *block_tables_dev, int32_t max_blocks_per_seq, uint8_t *k_pool,
                              uint8_t *v_pool, int32_t num_blocks, dgq_seg_record *seg_table,
                              dgq_seg_record *v_seg_table, const dgq_compress_options *options, void *workspace,
                              size_t workspace_bytes, void *cuda_stream);

/* dgq_prefill_finish restricted to the requests a re-segmentation selects: request b is segmented
 * and encoded when (pair_flags[b][h] & flag_mask) != 0 for some head h (pair_flags [batch, Hkv]
 * int32, device, e.g. as dgq_append_ex wrote them); the records, codes and window statistics of
 * every other request are left untouched.  pair_flags == NULL selects every request
 * (dgq_prefill_finish).  Other arguments as dgq_prefill_finish. */
dgq_status dgq_prefill_finish_ex(const void *k_src_bf16, const void *v_src_bf16, int32_t num_src_blocks,
                                 const int32_t *src_block_tables_dev, int32_t max_src_blocks_per_seq,
                                 const int32_t *seq_lens_dev, int32_t batch, int32_t max_seqlen,
                                 int32_t num_kv_heads, int32_t head_dim, int32_t block_size,
                                 const float *window_stats, int32_t max_windows, const int32_t *block_tables_dev,
                                 int32_t max_blocks_per_seq, uint8_t *k_pool, uint8_t *v_pool, int32_t num_blocks,
                                 dgq_seg_record *seg_table, dgq_seg_record *v_seg_table,
                                 const dgq_compress_options *options, const int32_t *pair_flags,
                                 int32_t flag_mask, void *workspace, size_t workspace_bytes, void *cuda_stream);

/* ---------------------------------------------------------------------------------------
 * dgq_paged_decode_attn -- one decode step of grouped-query attention over the INT8
 * paged cache plus the step's own (unquantised) key and value.
 *
 * For request b and query head hq (KV head h = hq / G, G = Hq / Hkv, consecutive query
 * heads share a KV head): scores s_t = q . x_K(t) / sqrt(128) for the cached tokens
 * t < L_b, where x_K(t) = k_min[s] + code * k_scale[s] from the record of (b, h) and the
 * codes gathered through the block table ([DGQ] section 2.2: segment lookup per token;
 * section 3.2: dequantisation on the GPU; [PAGED] paged_attention(q, k, v, block_tables)),
 * plus s_L = q . k_new / sqrt(128) for the current token; out = softmax(s) . [x_V ; v_new].
 * The softmax is computed online in fp32 over splits of the sequence that run on different
 * thread blocks and are merged in a fixed order (bitwise reproducible for a given GPU).
 *
 * q_bf16           [batch, Hq, 128] bf16, device, |q| < 65504.
 * k_new_bf16, v_new_bf16  [batch, Hkv, 128] bf16, device: the step's own key / value.
 * k_pool, v_pool, seg_table, block_tables_dev: as written by dgq_compress.
 * seq_lens_dev     [batch] int32, device: cached tokens per request (0 allowed); must not
 *                  exceed the record's seq_len.
 * out_bf16         [batch, Hq, 128] bf16, device.
 * Supported: Hq % Hkv == 0 with G = Hq / Hkv in {1, 2, 4, 8}.
 * workspace        >= dgq_attn_workspace_size(batch, Hq, Hkv, max_seqlen) bytes.
 */
dgq_status dgq_paged_decode_attn(const void *q_bf16, const void *k_new_bf16,
                                 const void *v_new_bf16, const uint8_t *k_pool,
                                 const uint8_t *v_pool, const dgq_seg_record *seg_table,
                                 const int32_t *block_tables_dev, const int32_t *seq_lens_dev,
                                 int32_t max_seqlen, int32_t batch, int32_t num_q_heads,
                                 int32_t num_kv_heads, int32_t head_dim, int32_t block_size,
                                 int32_t max_blocks_per_seq, int32_t num_blocks, void *out_bf16,
                                 void *workspace, size_t workspace_bytes, void *cuda_stream);

size_t dgq_attn_workspace_size(int32_t batch, int32_t num_q_heads, int32_t num_kv_heads,
                               int32_t max_seqlen);

/* dgq_paged_decode_attn over a cache with independent V segmentation (dgq_prefill_finish with a
 * v_seg_table): keys are dequantised with k_seg_table's segments and K parameters, values with
 * v_seg_table's segments and V parameters.  Same arguments otherwise. */
dgq_status dgq_paged_decode_attn_split(const void *q_bf16, const void *k_new_bf16, const void *v_new_bf16,
                                       const uint8_t *k_pool, const uint8_t *v_pool, const dgq_seg_record *k_seg_table,
                                       const dgq_seg_record *v_seg_table, const int32_t *block_tables_dev,
                                       const int32_t *seq_lens_dev, int32_t max_seqlen, int32_t batch,
                                       int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim, int32_t block_size,
                                       int32_t max_blocks_per_seq, int32_t num_blocks, void *out_bf16,
                                       void *workspace, size_t workspace_bytes, void *cuda_stream);

/* ---------------------------------------------------------------------------------------
 * dgq_paged_decode_attn_noalloc -- the same decode attention for callers that cannot
 * allocate device memory.  The source articles have no counterpart: this is a deployment
 * convenience of this library.
 *
 * Who needs it: code that must not call cudaMalloc (or any allocator) while it runs -- an
 * operator inside a serving engine that only receives the buffers it planned ahead, or a
 * plugin whose host framework forbids new device allocations during a step -- and so has no
 * workspace to pass.  Here the workspace is a fixed array that lives in the library's own
 * device memory: DGQ_NOALLOC_SCRATCH_BYTES on every GPU that loads the library, held until
 * the process exits.  Nothing is allocated by this call.
 *
 * Arguments, layouts and results are those of dgq_paged_decode_attn without the workspace.
 * Limits and behaviour:
 *   - a problem whose dgq_attn_workspace_size(batch, Hq, Hkv, max_seqlen) exceeds
 *     DGQ_NOALLOC_SCRATCH_BYTES is rejected with DGQ_ERR_SCRATCH_LIMIT before any launch;
 *   - the first call on a device looks up the array's device address (with that device
 *     current) and keeps it; make that first call before any stream capture;
 *   - every call on a device shares the one array, which keeps the previous call's contents:
 *     each call clears the array's 256-byte header on the stream before it launches, so calls
 *     issued in order on one stream are safe, while calls that overlap on the GPU (several
 *     streams at once) race and give wrong results;
 *   - no device-side error is reported: a wait that timed out, a block id outside the pool or
 *     a request longer than its block-table row is recorded in the array's header as in a
 *     workspace, but the next call clears that header and no call reads it, so this entry
 *     point returns DGQ_OK for them (the guarded accesses stay inside the caller's buffers as
 *     with the regular entry point); a caller that needs those checks uses
 *     dgq_paged_decode_attn with a workspace and dgq_workspace_error.
 */
#define DGQ_NOALLOC_SCRATCH_BYTES (8u << 20)

dgq_status dgq_paged_decode_attn_noalloc(const void *q_bf16, const void *k_new_bf16,
                                         const void *v_new_bf16, const uint8_t *k_pool,
                                         const uint8_t *v_pool, const dgq_seg_record *seg_table,
                                         const int32_t *block_tables_dev, const int32_t *seq_lens_dev,
                                         int32_t max_seqlen, int32_t batch, int32_t num_q_heads,
                                         int32_t num_kv_heads, int32_t head_dim, int32_t block_size,
                                         int32_t max_blocks_per_seq, int32_t num_blocks, void *out_bf16,
                                         void *cuda_stream);

/* ---------------------------------------------------------------------------------------
 * dgq_append -- one decode step's key and value of every (request b, KV head h) written into
 * the INT8 paged cache at position L = seg_table[b][h].seq_len.
 *
 * [DGQ] section 2.2 analyses the cache as each new token is generated but does not say how a
 * token that arrives after compression is encoded.  Reading taken here: the token joins the
 * last segment s = n_seg - 1 and each value x is encoded as q = min(max(rint((x - min[s]) *
 * inv), 0), 255) with inv = k_inv_last / v_inv_last of the record (the compress quantiser's
 * two IEEE steps; values outside the segment's range clamp, and the segment's min and scale,
 * hence every code already stored, stay as they are).  Boundaries are not revisited (that
 * needs the bf16 history): dgq_append_ex reports when a re-segmentation is due and
 * dgq_prefill_finish_ex performs it from the caller's bf16 history.  A record with n_seg == 0 gets a first
 * segment made of the new token alone (its min/max over the 128 values, as in compress).
 * The record's seq_len and its start entries past the last segment become L + 1.
 *
 * k_new_bf16, v_new_bf16  [batch, Hkv, 128] bf16, device.
 * block_tables_dev        [batch, max_blocks_per_seq] int32, device: column L / bs of row b
 *                         names the block that receives token L.  The caller adds a block
 *                         (e.g. from dgq_pool_alloc) when L is a multiple of block_size.
 * k_pool, v_pool          [num_blocks, Hkv, block_size, 128] uint8, device: slot L of every
 *                         pair is written, nothing else.
 * seg_table               [batch, Hkv] records, device, read and updated in place.
 * workspace               >= dgq_append_workspace_size() bytes, zero-filled before first use.
 *                         A pair whose slot has no column (L / bs >= max_blocks_per_seq) is
 *                         left untouched and flagged there (dgq_workspace_error).
 * The launch is programmatic-dependent: it may start while the previous kernel on the stream
 * finishes and waits for it before reading any record.
 */
dgq_status dgq_append(const void *k_new_bf16, const void *v_new_bf16, int32_t batch, int32_t num_kv_heads,
                      int32_t head_dim, int32_t block_size, const int32_t *block_tables_dev,
                      int32_t max_blocks_per_seq, uint8_t *k_pool, uint8_t *v_pool, int32_t num_blocks,
                      dgq_seg_record *seg_table, void *workspace, size_t workspace_bytes, void *cuda_stream);

size_t dgq_append_workspace_size(void);

/* ---------------------------------------------------------------------------------------
 * Re-segmentation after appends.  [DGQ] section 2.2 analyses the variance curve as each new
 * token is generated (segments come from jumps between 16-token window means) and section 3.2
 * ties the segment count to the length.  dgq_append keeps the boundaries; these two calls let a
 * caller that keeps the bf16 history (its bf16 paged cache) re-run the segmentation when it
 * changes:
 *   DGQ_RESEG_WINDOW   appending token L completed a 16-token window ((L + 1) % 16 == 0): a new
 *                      window mean, hence a new candidate jump, exists;
 *   DGQ_RESEG_NGROUPS  the length reached a threshold of the n_groups rule (L + 1 = 2048 or
 *                      16384; for every L >= 16384 the rule gives 5), so the segment count changes.
 * A step with re-segmentation: dgq_append_ex (flags per pair); the step's bf16 K/V written into
 * the bf16 paged history (the caller's own cache write); dgq_prefill_chunk_stats over the window
 * each flagged request just completed ([L + 1 - 16, L + 1); an empty range for the others); then
 * dgq_prefill_finish_ex with the flags, which segments and re-encodes exactly the flagged
 * requests from their whole bf16 history (records and every code), as dgq_compress_paged of the
 * L + 1 tokens would, and leaves every other request untouched.
 */
#define DGQ_RESEG_WINDOW 1
#define DGQ_RESEG_NGROUPS 2

/* dgq_append, and in resegment_flags ([batch, Hkv] int32, device, written for every pair; NULL:
 * none) each pair's DGQ_RESEG_* bits for the token it appended (0 for a pair left untouched). */
dgq_status dgq_append_ex(const void *k_new_bf16, const void *v_new_bf16, int32_t batch, int32_t num_kv_heads,
                         int32_t head_dim, int32_t block_size, const int32_t *block_tables_dev,
                         int32_t max_blocks_per_seq, uint8_t *k_pool, uint8_t *v_pool, int32_t num_blocks,
                         dgq_seg_record *seg_table, int32_t *resegment_flags, void *workspace,
                         size_t workspace_bytes, void *cuda_stream);

/* dgq_append for a cache with independent V segmentation (dgq_prefill_finish with a v_seg_table):
 * K's codes from k_seg_table's last K segment, V's from v_seg_table's last V segment, each record
 * updated for its own tensor (a record with n_seg == 0 gets a segment made of the new token's
 * values of that tensor).  Both records of a pair must hold the same seq_len; a pair whose two
 * records disagree is left untouched and flagged in the workspace.  Arguments as dgq_append. */
dgq_status dgq_append_split(const void *k_new_bf16, const void *v_new_bf16, int32_t batch, int32_t num_kv_heads,
                            int32_t head_dim, int32_t block_size, const int32_t *block_tables_dev,
                            int32_t max_blocks_per_seq, uint8_t *k_pool, uint8_t *v_pool, int32_t num_blocks,
                            dgq_seg_record *k_seg_table, dgq_seg_record *v_seg_table, void *workspace,
                            size_t workspace_bytes, void *cuda_stream);

/* ---------------------------------------------------------------------------------------
 * Comparison encodings: the same paged cache layout and the same decode kernel, with the
 * K/V codes produced by one of the quantisers DGQ is measured against, so that accuracy and
 * decode speed can be set side by side on one workload.  Sources:
 *   [DGQ] section 2.2: the traditional alternative cuts each vector into fixed groups of 64
 *         dimensions, each with its own min/max INT8 parameters;
 *   [DGQ] section 2.3: the FP8 (E4M3) comparison row of its format table;
 *   [PAGED] "FP8+FP16 scheme: technical details" section: symmetric INT8 with scale =
 *         max|k| / 127 and k / scale held to [-128, 127].
 *
 * DGQ_FORMAT_DGQ       the records and codes of dgq_compress (dgq_encode_format rejects it).
 * DGQ_FORMAT_FIXED64   per token and per 64-value half of each K and V row: min/max over the
 *                      64 values, scale = (max - min) / 255, codes rint((x - min) * (255 /
 *                      (max - min))) -- the DGQ quantiser (two IEEE steps, -0 min/max stored as
 *                      +0, 0 codes and scale for a flat group) on a fixed group.  The parameters
 *                      go to a side array [num_blocks, Hkv, block_size, 4] fp32 per tensor:
 *                      (min of values 0..63, its scale, min of values 64..127, its scale) in
 *                      the slot of the token's codes (16 B per token and head: 12.5% more bytes
 *                      than the codes).
 * DGQ_FORMAT_SYM_INT8  per (request, KV head) and tensor: s = amax / 127 (IEEE division; amax =
 *                      largest |x| over the pair), q = rint(x / s) (IEEE division, half-even)
 *                      held to [-128, 127], 0 when s == 0.  READING: the printed snippet has no
 *                      rounding step; round-half-even is taken.  Stored as the byte q + 128,
 *                      with a one-segment record (min = -128 s, scale = s), so the DGQ decode
 *                      path reads it unchanged.
 * DGQ_FORMAT_FP8_E4M3  every value rounded (half-even) to the nearest E4M3 number (bias 7,
 *                      3 mantissa bits, largest finite 448, subnormal step 2^-9), saturating to
 *                      +-448; stored as the E4M3 byte.
 * For FIXED64 and FP8_E4M3 the record of each pair holds n_seg = 1, seq_len = L and the identity
 * parameters (min 0, scale 1): the codes carry their own scale.  dgq_append supports only DGQ.
 */
typedef enum dgq_format {
    DGQ_FORMAT_DGQ = 0,
    DGQ_FORMAT_FIXED64 = 1,
    DGQ_FORMAT_SYM_INT8 = 2,
    DGQ_FORMAT_FP8_E4M3 = 3
} dgq_format;

/*
 * dgq_encode_format -- one layer's K/V of a batch of requests encoded into the paged cache in
 * a comparison format.  Arguments as for dgq_compress (packed rows, cu_seqlens, block tables,
 * pools, records), plus:
 * format            DGQ_FORMAT_FIXED64, DGQ_FORMAT_SYM_INT8 or DGQ_FORMAT_FP8_E4M3 (anything
 *                   else: DGQ_ERR_INVALID_ARG).
 * k_group_params, v_group_params  FIXED64 only: [num_blocks, Hkv, block_size, 4] fp32, device,
 *                   written for the slots of tokens 0..L_b-1; ignored (may be NULL) otherwise.
 * workspace         >= dgq_encode_format_workspace_size(batch, num_kv_heads) bytes, zero-filled
 *                   before first use (SYM_INT8 keeps its per-pair maxima there).
 * A block-table entry outside [0, num_blocks) is flagged in the workspace and its slots are
 * skipped.  Two or three launches, no cooperative launch.
 */
dgq_status dgq_encode_format(int32_t format, const void *k_bf16, const void *v_bf16, int32_t total_tokens,
                             const int32_t *cu_seqlens_dev, int32_t batch, int32_t max_seqlen,
                             int32_t num_kv_heads, int32_t head_dim, int32_t block_size,
                             const int32_t *block_tables_dev, int32_t max_blocks_per_seq, uint8_t *k_pool,
                             uint8_t *v_pool, int32_t num_blocks, dgq_seg_record *seg_table,
                             float *k_group_params, float *v_group_params, void *workspace,
                             size_t workspace_bytes, void *cuda_stream);

size_t dgq_encode_format_workspace_size(int32_t batch, int32_t num_kv_heads);

/*
 * dgq_paged_decode_attn_format -- dgq_paged_decode_attn over a cache written in `format`
 * (DGQ_FORMAT_DGQ and DGQ_FORMAT_SYM_INT8 are decoded through the records; FP8_E4M3 codes are
 * E4M3 values; FIXED64 codes are decoded with their per-token, per-half parameters, read from
 * k_group_params / v_group_params, which must be non-NULL for it).  Same kernel, tiling,
 * workspace and results layout as dgq_paged_decode_attn.
 */
dgq_status dgq_paged_decode_attn_format(int32_t format, const void *q_bf16, const void *k_new_bf16,
                                        const void *v_new_bf16, const uint8_t *k_pool, const uint8_t *v_pool,
                                        const dgq_seg_record *seg_table, const float *k_group_params,
                                        const float *v_group_params, const int32_t *block_tables_dev,
                                        const int32_t *seq_lens_dev, int32_t max_seqlen, int32_t batch,
                                        int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim,
                                        int32_t block_size, int32_t max_blocks_per_seq, int32_t num_blocks,
                                        void *out_bf16, void *workspace, size_t workspace_bytes,
                                        void *cuda_stream);

/* Zero-fill a workspace (cudaMemsetAsync on the stream). */
dgq_status dgq_workspace_init(void *workspace, size_t workspace_bytes, void *cuda_stream);

/* Synchronise the stream and read the device-side error word of a workspace into
 * *device_error (0 = none; otherwise an internal code naming the wait that timed out).
 * Returns DGQ_ERR_DEVICE when the word is non-zero.  The workspace must be re-initialised
 * after a device-side error. */
dgq_status dgq_workspace_error(const void *workspace, void *cuda_stream, int32_t *device_error);

/* ---------------------------------------------------------------------------------------
 * Host block bookkeeping ([PAGED] BlockTable: physical blocks handed out from a free list
 * and returned when a request ends).  Plain host memory; not thread-safe.
 */
typedef struct dgq_pool dgq_pool;

dgq_pool *dgq_pool_create(int32_t num_blocks);          /* NULL on bad size / no memory */
void dgq_pool_destroy(dgq_pool *pool);
/* Takes n blocks (all or nothing); ids in ascending order of availability. */
dgq_status dgq_pool_alloc(dgq_pool *pool, int32_t n, int32_t *out_ids);
/* Returns blocks; an id out of range or already free is DGQ_ERR_INVALID_ARG (nothing freed). */
dgq_status dgq_pool_free(dgq_pool *pool, const int32_t *ids, int32_t n);
int32_t dgq_pool_num_free(const dgq_pool *pool);
/* Fills row `row` of a host block table [*, max_blocks_per_seq] with blocks for `len`
 * tokens taken from the pool (ceil(len / block_size) of them); unused entries set to 0. */
dgq_status dgq_pool_alloc_table_row(dgq_pool *pool, int32_t len, int32_t block_size,
                                    int32_t *table, int32_t row, int32_t max_blocks_per_seq);

const char *dgq_status_str(dgq_status status);

#ifdef __cplusplus
}
#endif

#endif /* DGQ_H */
