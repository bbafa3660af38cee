/*
 * pkv.h -- C ABI of the paged-KV attention library for GB300 (sm_103a):
 * block-paged KV cache with asymmetric K/V head sizes (K 192 / V 128 with
 * GQA, and the MLA shape 576 / 512 where V is a prefix of K).
 *
 * Sources the operations follow (web pages, by title and section):
 *   - vLLM PR #64064 "ROCm AITER unified attention for MiMo-V2.6":
 *     "Details" -- reshape_and_cache_flash writes V with V's own head size
 *     and head stride; one packed (head_size + head_size_v) row per KV head,
 *     K first; "Tests" -- block sizes 16 and 64, two cache layouts, bf16 and
 *     fp8 caches, per-tensor and per-head scales; "Details" / "Known
 *     limitations" -- a backend that splits the page at head_size serves
 *     v <= k only.
 *   - vLLM PR #50371 "Enable 12-head MLA persistent decode": "Purpose" and
 *     "Test Plan" (12 query heads, one latent head, D 576 -> 512) and the
 *     discussion of split-KV with split selection from device-side sequence
 *     metadata (launch shape stays graph-stable).
 *   - Hugging Face model card "diffbot/MiMo-V2.6-Flash-MOPD-FP8KV-W4A8-2x-
 *     RTX-PRO-6000": "What the kernels do" (split-KV for the speculative
 *     verify step, FP8 E4M3 K/V converted in the kernel, a prefill attention
 *     kernel for the global layers) and "Update 2026-10-01" (a query row with
 *     no visible key is 0, not NaN, after the split-KV merge).
 *
 * Conventions shared by every call:
 *   - All tensor pointers are DEVICE pointers owned by the caller.  The
 *     library allocates no device memory and performs no host<->device
 *     synchronisation, except pkv_get_device_error, which says so.
 *   - Every call is asynchronous on `stream` (a cudaStream_t; NULL is the
 *     legacy default stream) and returns a status: PKV_OK (0) or a negative
 *     PKV_E* code.  Arguments are validated on the host before anything is
 *     launched; a rejected call launches nothing.  PKV_ECUDA means a launch
 *     failed; pkv_last_cuda_error() returns the cudaError_t value.
 *   - Stream order holds as for any kernel launch.  The kernels of
 *     pkv_kv_cache_write, pkv_paged_attn_decode(_fused, _noalloc) and
 *     pkv_splitkv_reduce(_sink) use programmatic dependent launch so that
 *     the next kernel can be placed while the current one finishes.  Each
 *     waits for everything ahead of it on the stream before it touches
 *     memory.  A caller's own kernel queued behind one of them sees that
 *     kernel's results as usual.  The exception is a kernel launched with
 *     the programmatic-stream-serialization attribute: it must wait
 *     (griddepcontrol.wait / cudaGridDependencySynchronize) before reading
 *     them, as that attribute requires.  PKV_PDL=0 in the environment
 *     (read once per process) launches them without the attribute.
 *   - bf16 tensors are IEEE bfloat16; fp8 is OCP FP8 E4M3 ("e4m3fn":
 *     saturating, max 448, no infinities).
 *   - Sequences: sequence b has q_len(b) = query_start_loc[b+1] -
 *     query_start_loc[b] query tokens and seq_lens[b] keys in total, the
 *     query tokens' own keys included (they are written to the cache first).
 *     Query i of the sequence sits at position seq_lens[b] - q_len(b) + i and
 *     attends to keys 0 .. that position (causal, bottom-right aligned).  Key
 *     j of sequence b lives in page block_table[b * max_blocks_per_seq +
 *     j / block_size] at offset j % block_size.  Only the first
 *     ceil(seq_lens[b] / block_size) entries of a block-table row are read.
 *   - Query head h reads KV head h / (num_q_heads / num_kv_heads).
 *   - Out-of-range slots or page ids met on the device are not dereferenced:
 *     the element is skipped (write) or read as zero (attention) and the
 *     device error word records PKV_EDEV_RANGE (see pkv_get_device_error).
 */
#ifndef PKV_H_
#define PKV_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st *pkv_stream_t; /* the same type as cudaStream_t */

/* status codes */
#define PKV_OK 0
#define PKV_EINVAL (-1)        /* null pointer, size or stride out of range */
#define PKV_EUNSUPPORTED (-2)  /* valid, but a shape / dtype this build lacks */
#define PKV_ECUDA (-3)         /* a CUDA launch or query failed */

/* device error word values (pkv_get_device_error) */
#define PKV_EDEV_NONE 0
#define PKV_EDEV_RANGE 1       /* slot or page id out of range: skipped */
#define PKV_EDEV_TIMEOUT 2     /* a bounded wait in a kernel gave up */

/* cache element types */
#define PKV_BF16 0
#define PKV_FP8_E4M3 1

/* cache layouts; R = row_elems */
#define PKV_NHD 0              /* [num_blocks][block_size][num_kv_heads][R] */
#define PKV_HND 1              /* [num_blocks][num_kv_heads][block_size][R] */

/* fp8 scale modes (bf16 caches take PKV_SCALE_NONE) */
#define PKV_SCALE_NONE 0
#define PKV_SCALE_TENSOR 1     /* k_scale[0], v_scale[0] */
#define PKV_SCALE_HEAD 2       /* k_scale[h], v_scale[h], h < num_kv_heads */

/*
 * One block-paged cache (vLLM PR #64064, "Details").  Every (slot, KV head)
 * owns one row of row_elems elements; K occupies [k_off, k_off + head_size)
 * and V occupies [v_off, v_off + head_size_v).  MiMo: row 320, K at 0 (192),
 * V at 192 (128).  MLA: row 576, K at 0 (576), V at 0 (512) -- V is a prefix
 * of K and is never written separately.
 */
typedef struct pkv_cache_desc {
    int dtype;        /* PKV_BF16 | PKV_FP8_E4M3 */
    int layout;       /* PKV_NHD | PKV_HND */
    int num_blocks;   /* pages in the cache */
    int block_size;   /* tokens per page, >= 1 */
    int num_kv_heads;
    int row_elems;    /* R */
    int k_off, head_size;
    int v_off, head_size_v;
    int scale_mode;   /* PKV_SCALE_* */
} pkv_cache_desc;

/*
 * pkv_kv_cache_write -- vLLM PR #64064, "Details" (the asymmetric branch of
 * reshape_and_cache_flash).
 *
 * For every token t < num_tokens with s = slot_mapping[t] >= 0, and every
 * KV head h: row = the (s / block_size, s % block_size, h) row of `cache`;
 *   row[k_off + i] = enc_k(key[t * key_tok_stride + h * key_head_stride + i])
 *                    for i < head_size,
 *   row[v_off + i] = enc_v(value[t * val_tok_stride + h * val_head_stride + i])
 *                    for i < head_size_v (skipped when value == NULL).
 * Strides are in elements.  A negative slot skips the token.  No other byte of
 * the cache is written.  enc is a bit copy for a bf16 cache; for an fp8 cache
 * it is E4M3(x / scale) with the division in IEEE binary32, round-to-nearest-
 * even and saturation to +-448 (NaN stays NaN).  key/value: bf16.  slot_mapping:
 * int64 [num_tokens].  k_scale / v_scale: device float32, [1] or
 * [num_kv_heads] by d->scale_mode (NULL for bf16 caches).  When V is a prefix
 * of K (value == NULL), read it back with v_scale equal to k_scale.
 * Errors: PKV_EINVAL for null pointers (key, slot_mapping, cache, d; scales
 * when required), negative sizes, K or V ranges outside the row, num_tokens <
 * 0; PKV_EUNSUPPORTED for an unknown dtype / layout / scale mode.
 */
int pkv_kv_cache_write(const void *key, int64_t key_tok_stride,
                       int64_t key_head_stride, const void *value,
                       int64_t val_tok_stride, int64_t val_head_stride,
                       const int64_t *slot_mapping, int num_tokens,
                       void *cache, const pkv_cache_desc *d,
                       const float *k_scale, const float *v_scale,
                       pkv_stream_t stream);

/*
 * pkv_paged_attn_prefill -- causal varlen attention of a batch of query
 * chunks over the paged cache (the prefill rows of the MiMo model card's
 * "What the kernels do"; semantics of vLLM PR #64064's unified attention).
 *
 * out[t][h][:] = sum_j softmax_j(softmax_scale * q[t][h] . K_j) * V_j over the
 * keys j the query token sees (see the sequence conventions above).  q: bf16
 * [num_tokens][num_q_heads][head_size]; out: bf16
 * [num_tokens][num_q_heads][head_size_v]; block_table: int32
 * [num_seqs][max_blocks_per_seq]; seq_lens: int32 [num_seqs];
 * query_start_loc: int32 [num_seqs + 1], non-decreasing, last = num_tokens.
 * seq_lens[b] >= q_len(b) is required for every row to see a key; a row that
 * sees none is written as 0.  The K and V of every visible key must already
 * be in the cache.  Keys past seq_lens[b] in the last page are never used,
 * whatever the cache holds there.
 * softmax_scale must be > 0.
 * FP8 E4M3 cache (the MiMo model card's production setting, "What the
 * kernels do": FP8 K/V converted in the kernel, Q.K^T kept in 16-bit, its
 * FP8 Q.K^T having had 7x the error): the E4M3 codes are widened exactly to
 * bf16 in shared memory between the TMA load and the tensor-core MMAs, and
 * k_scale / v_scale (as in the write: [1] or [num_kv_heads] by
 * d->scale_mode, positive) fold into the softmax scale and the output, so
 * out = softmax(scale * q (k_scale K)^T) (v_scale V) with Q.K^T the exact
 * products of bf16 q and the codes summed in f32.  No workspace: nothing
 * beyond the cache is read or written.  bf16 caches take NULL scales.
 * This build: head_size 192 and head_size_v 128, num_q_heads / num_kv_heads
 * dividing 128, block_size a power of two >= 8, K at a 64-element column
 * offset and V at a 16-byte one; otherwise PKV_EUNSUPPORTED.  PKV_EINVAL for null
 * pointers, softmax_scale <= 0 or inconsistent sizes, and when q, cache or
 * out is not device memory of the current device (pinned or mapped host
 * memory, managed memory, another GPU's memory): the kernel's tensor maps
 * and its K/V loads (for FP8 caches and rows that do not split into
 * 64-column slabs, multicast to the two CTAs of a cluster) cover this GPU's
 * own memory only.
 */
int pkv_paged_attn_prefill(const void *q, int num_q_heads, int num_tokens,
                           const void *cache, const pkv_cache_desc *d,
                           const int32_t *block_table, int max_blocks_per_seq,
                           const int32_t *seq_lens,
                           const int32_t *query_start_loc, int num_seqs,
                           float softmax_scale, const float *k_scale,
                           const float *v_scale, void *out,
                           pkv_stream_t stream);

/*
 * pkv_prefill_fp8_workspace_bytes -- size of the workspace that
 * pkv_paged_attn_prefill_fp8 needs: num_seqs * max_blocks_per_seq pages of
 * block_size * num_kv_heads * row_elems bf16 elements (rounded up to 256
 * bytes), then num_seqs * max_blocks_per_seq int32 block-table entries.
 * Returns 0 for an invalid descriptor or sizes.
 */
size_t pkv_prefill_fp8_workspace_bytes(int num_seqs, int max_blocks_per_seq,
                                       const pkv_cache_desc *d);

/*
 * pkv_paged_attn_prefill_fp8 -- the prefill over an FP8 E4M3 cache in two
 * passes, for callers that can give it a workspace: the same result as
 * pkv_paged_attn_prefill on the FP8 cache (which widens the codes inside
 * the kernel and needs no workspace), faster, because the tensor-core MMAs
 * then read bf16 slabs that no widening step in shared memory competes
 * with.  Two passes on `stream`:
 *   1. every page a sequence uses (block_table[b][j], j < ceil(seq_lens[b] /
 *      block_size)) is copied into the workspace as its E4M3 codes widened
 *      to bf16 (exact), with a remapped block table;
 *   2. the tcgen05 prefill of pkv_paged_attn_prefill runs on those pages,
 *      with k_scale folded into the softmax scale and v_scale into the
 *      output, per KV head (SCALE_HEAD) or per tensor.
 * Q.K^T is exact products of bf16 q and E4M3 codes summed in f32.  The
 * result is out = softmax(scale * q (k_scale K)^T) (v_scale V) as in
 * pkv_paged_attn_prefill, with the attention sink of
 * pkv_paged_attn_prefill_sink when sinks is not NULL.
 * cache: FP8 E4M3 (d->dtype PKV_FP8_E4M3); k_scale / v_scale as in the
 * decode (positive).  workspace: device memory of at least
 * pkv_prefill_fp8_workspace_bytes(num_seqs, max_blocks_per_seq, d) bytes,
 * 256-byte aligned, overwritten by the call; overlapping calls must not
 * share it.  An out-of-range page id is skipped (read as zeros) and
 * recorded as PKV_EDEV_RANGE.  Status codes as in pkv_paged_attn_prefill;
 * PKV_EINVAL also for a non-FP8 cache, a missing, misaligned or too small
 * workspace, or a q, cache, workspace or out that is not device memory of
 * the current device (checked before the first pass is launched).
 */
int pkv_paged_attn_prefill_fp8(const void *q, int num_q_heads, int num_tokens,
                               const void *cache, const pkv_cache_desc *d,
                               const int32_t *block_table, int max_blocks_per_seq,
                               const int32_t *seq_lens,
                               const int32_t *query_start_loc, int num_seqs,
                               float softmax_scale, const float *k_scale,
                               const float *v_scale, const float *sinks,
                               void *workspace, size_t workspace_bytes, void *out,
                               pkv_stream_t stream);

/*
 * pkv_paged_attn_prefill_sink -- pkv_paged_attn_prefill with an attention
 * sink: one extra logit per query head in every row's softmax denominator,
 * with no value vector (MiMo model card, "Update 2026-10-01": the vision
 * encoder's sink, vLLM #58235):
 *   out = sum_j exp(s_j) V_j / (exp(sinks[h]) + sum_j exp(s_j)),
 * s_j = softmax_scale * q.k_j over the row's visible keys, h the row's query
 * head.  sinks: float32 [num_q_heads], device memory; a sink of -inf is no
 * sink; NULL gives pkv_paged_attn_prefill's result.  Other arguments,
 * layouts, status codes and supported shapes (bf16 and FP8 caches) as in
 * pkv_paged_attn_prefill.
 */
int pkv_paged_attn_prefill_sink(const void *q, int num_q_heads, int num_tokens,
                                const void *cache, const pkv_cache_desc *d,
                                const int32_t *block_table, int max_blocks_per_seq,
                                const int32_t *seq_lens,
                                const int32_t *query_start_loc, int num_seqs,
                                float softmax_scale, const float *k_scale,
                                const float *v_scale, const float *sinks,
                                void *out, pkv_stream_t stream);

/*
 * pkv_paged_attn_decode -- split-KV decode and speculative verify (q_len 1
 * .. max_query_len) over the paged cache: the verify-step split-KV of the
 * MiMo model card's "What the kernels do", the 12-head MLA decode of vLLM
 * PR #50371 ("Purpose"), split selection from device-side sequence lengths
 * with a graph-stable launch shape (vLLM PR #50371 discussion).
 *
 * The P = ceil(seq_lens[b] / block_size) pages of sequence b are cut into
 * num_splits segments of pps = ceil(P / num_splits) pages; segment s covers
 * pages [s * pps, min((s + 1) * pps, P)).  For every query row (t, h) and
 * segment s, over the keys of the segment that the row sees:
 *   partial_lse[s][t][h]  = log(sum_j exp(softmax_scale * q . K_j))  (natural
 *                           log; -inf when the segment has no such key),
 *   partial_o[s][t][h][:] = sum_j softmax_j * V_j  (normalised within the
 *                           segment; left unwritten when partial_lse is -inf).
 * K and V are dequantised with k_scale / v_scale for fp8 caches.  Merge the
 * segments with pkv_splitkv_reduce.  partial_o: float32
 * [num_splits][num_tokens][num_q_heads][head_size_v]; partial_lse: float32
 * [num_splits][num_tokens][num_q_heads]; both 4-byte aligned (PKV_EINVAL
 * otherwise).  Other arguments as in prefill.
 * A sequence with seq_lens[b] == 0 (a padded row) gives -inf everywhere; its
 * block-table row is never read.  max_query_len bounds q_len(b) for the
 * launch shape (1 .. 64).
 * This build: head_size / head_size_v 192 / 128 (bf16 or fp8 cache) or
 * 576 / 512 (bf16 or fp8 cache); otherwise PKV_EUNSUPPORTED.
 */
int pkv_paged_attn_decode(const void *q, int num_q_heads, int num_tokens,
                          const void *cache, const pkv_cache_desc *d,
                          const int32_t *block_table, int max_blocks_per_seq,
                          const int32_t *seq_lens,
                          const int32_t *query_start_loc, int num_seqs,
                          int max_query_len, float softmax_scale,
                          const float *k_scale, const float *v_scale,
                          int num_splits, float *partial_o,
                          float *partial_lse, pkv_stream_t stream);

/*
 * pkv_paged_attn_decode_balanced -- pkv_paged_attn_decode with the segments
 * chosen on the device from seq_lens so that every work range carries the
 * same number of pages (split selection from device-side sequence metadata
 * under a fixed launch shape, vLLM PR #50371 discussion).
 *
 * Segmentation ("balanced ranges"): with P_b = ceil(seq_lens[b] /
 * block_size), the pages of all sequences are laid end to end in sequence
 * order (sequence b from global page G_b = P_0 + ... + P_{b-1}, Ptot pages
 * in all) and cut into ranges of R pages,
 *   R = max(ceil(Ptot / W), Rmin, 1),  W = num_ranges,
 *   Rmin = Ptot if max_splits == 1, else floor(max(Pmax - 2, 0) /
 *          (max_splits - 1)) + 1  (Pmax = max_b P_b),
 * so that no sequence meets more than max_splits ranges.  Segment s of
 * sequence b is the part of the sequence inside range floor(G_b / R) + s
 * (its pages [max(G_b, rR), min(G_b + P_b, (r + 1)R)) - G_b); segments past
 * the sequence's last range are empty.  partial_o / partial_lse hold
 * max_splits segments per row and mean what they mean in
 * pkv_paged_attn_decode (an empty segment: lse -inf, o unwritten), so
 * pkv_splitkv_reduce(_sink) with num_splits = max_splits merges them.  The
 * launch runs one CTA per (range, block of KV heads) up to the resident
 * CTAs of the device and each CTA streams its ranges' pages, so the work is
 * even whatever the mix of sequence lengths.
 * num_ranges: W >= 1, or 0 for pkv_decode_balanced_ranges(d) (one
 * (range, head block) per resident CTA of the current device).  seq_lens[b] <= max_blocks_per_seq
 * * block_size is required.  Other arguments, layouts and status codes as
 * in pkv_paged_attn_decode; PKV_EINVAL also for num_ranges < 0 or above
 * 2^24, or num_seqs * max_blocks_per_seq of 2^31 or more; PKV_EUNSUPPORTED
 * for more than 16384 sequences (use pkv_paged_attn_decode).  Up to 128
 * sequences, every CTA reads all lengths once; beyond, a CTA reads them in
 * chunks of 128 (their page counts first, then the chunk windows it needs),
 * a few more dependent reads before its first copy.
 */
int pkv_paged_attn_decode_balanced(const void *q, int num_q_heads, int num_tokens,
                                   const void *cache, const pkv_cache_desc *d,
                                   const int32_t *block_table, int max_blocks_per_seq,
                                   const int32_t *seq_lens,
                                   const int32_t *query_start_loc, int num_seqs,
                                   int max_query_len, float softmax_scale,
                                   const float *k_scale, const float *v_scale,
                                   int max_splits, int num_ranges, float *partial_o,
                                   float *partial_lse, pkv_stream_t stream);

/*
 * pkv_decode_balanced_ranges -- the range count W that
 * pkv_paged_attn_decode_balanced takes for num_ranges = 0 on the current
 * device: the decode kernel's resident CTAs (SMs x CTAs per SM of the
 * kernel form that serves this cache) divided by its blocks of KV heads
 * (the bf16 K192 / V128 form takes four KV heads per block when
 * num_kv_heads is a multiple of 4, the other forms one), at least 1.
 * Host-only; a negative status for an invalid or unsupported descriptor.
 */
int pkv_decode_balanced_ranges(const pkv_cache_desc *d);

/*
 * pkv_decode_workspace_bytes -- size of the workspace that
 * pkv_paged_attn_decode_fused needs for these sizes: one 32-bit counter per
 * (sequence, KV head, 16-row group of the head's q_len * G rows).  Returns
 * 0 for invalid sizes.
 */
size_t pkv_decode_workspace_bytes(int num_seqs, int num_q_heads,
                                  int num_kv_heads, int max_query_len);

/*
 * pkv_paged_attn_decode_fused -- pkv_paged_attn_decode and
 * pkv_splitkv_reduce in one launch (the fused split merge ranked next in
 * the scope of this library; the pages merge in a second stage, vLLM PR
 * #50371 discussion, "both stages").  Every work unit writes its segment's
 * partials as pkv_paged_attn_decode does, then counts itself done in the
 * workspace; the last unit of each (sequence, KV-head block, row group) to
 * finish merges all segments of its rows as pkv_splitkv_reduce does (0 and
 * lse -inf for a row with no visible key) into out (bf16 [num_tokens]
 * [num_q_heads][head_size_v]) and lse_out (float32 [num_tokens]
 * [num_q_heads], or NULL), and resets its counter.
 * workspace: device memory of at least pkv_decode_workspace_bytes(...)
 * (workspace_bytes gives its size), zero-filled by the caller before its
 * first use; every call leaves it zero again, so it can be reused without
 * clearing (after a call that ended with a device error -- see
 * pkv_get_device_error -- it must be zero-filled again).  Calls that overlap
 * in time must not share a workspace.
 * partial_o / partial_lse are scratch here (same shapes as in
 * pkv_paged_attn_decode).  For num_splits > 32 the merge runs as a second
 * launch on the same stream (same results, workspace untouched).  Other
 * arguments, sizes and status codes as in pkv_paged_attn_decode; PKV_EINVAL
 * also for a missing or too small workspace, a null out, partial_o not
 * 16-byte aligned, out not 8-byte aligned, or num_tokens * num_q_heads of
 * 2^31 or more (the merge reads the partials 16 bytes at a time).
 */
int pkv_paged_attn_decode_fused(const void *q, int num_q_heads, int num_tokens,
                                const void *cache, const pkv_cache_desc *d,
                                const int32_t *block_table, int max_blocks_per_seq,
                                const int32_t *seq_lens,
                                const int32_t *query_start_loc, int num_seqs,
                                int max_query_len, float softmax_scale,
                                const float *k_scale, const float *v_scale,
                                int num_splits, float *partial_o,
                                float *partial_lse, void *workspace,
                                size_t workspace_bytes, void *out, float *lse_out,
                                pkv_stream_t stream);

/*
 * pkv_paged_attn_decode_balanced_fused -- pkv_paged_attn_decode_balanced and
 * the split merge in one launch: every unit writes its segment's partials
 * and counts itself done in the workspace; the last unit of each (sequence,
 * KV-head block, 16-row group) to finish merges that sequence's segments (as
 * many as its ranges) as pkv_splitkv_reduce does into out (bf16
 * [num_tokens][num_q_heads][head_size_v]) and lse_out (float32
 * [num_tokens][num_q_heads], or NULL), and resets its counter; the rows of a
 * sequence with no key are written as 0 (lse -inf).  Segmentation, max_splits
 * and num_ranges as in pkv_paged_attn_decode_balanced; workspace rules,
 * partial_o / partial_lse (scratch here) and the fallback past 32 splits (a
 * second launch) as in pkv_paged_attn_decode_fused.  Status codes as in
 * those two calls; PKV_EINVAL also for num_ranges < 0.
 */
int pkv_paged_attn_decode_balanced_fused(
    const void *q, int num_q_heads, int num_tokens, const void *cache,
    const pkv_cache_desc *d, const int32_t *block_table, int max_blocks_per_seq,
    const int32_t *seq_lens, const int32_t *query_start_loc, int num_seqs,
    int max_query_len, float softmax_scale, const float *k_scale, const float *v_scale,
    int max_splits, int num_ranges, float *partial_o, float *partial_lse, void *workspace,
    size_t workspace_bytes, void *out, float *lse_out, pkv_stream_t stream);

/*
 * pkv_paged_attn_decode_fused_noalloc -- pkv_paged_attn_decode_fused
 * without a caller workspace.  The pages have no counterpart.  It serves
 * callers that cannot allocate device memory for the counters: a serving
 * engine that hands all free GPU memory to its KV-cache pool at start-up
 * and takes no further allocation during a step, or a plain C host program
 * that links only this library and has no allocator of its own.  Its
 * counters live in a fixed array of 65536 32-bit counters (256 KB) in this
 * library's own device memory, one array per device, held by every device
 * that loads the library until the process exits; nothing is allocated.
 * Set-up: the first call on a device looks up that device's array address
 * (cudaGetSymbolAddress, with the device current; a failure returns
 * PKV_ECUDA), so make that first call before any stream capture.  After
 * every argument has been checked, each call zero-fills, on `stream`, the
 * counters it is about to use (so a call after a device error needs no
 * clearing), then launches as pkv_paged_attn_decode_fused does.  All calls
 * on a device share that one array, which keeps the last call's contents:
 * calls that overlap in time (on different streams or host threads) race
 * on it and give wrong results, so serialise them.
 * PKV_EINVAL also when num_splits <= 32 (the merge runs inside the decode
 * kernel and uses the counters) and pkv_decode_workspace_bytes(num_seqs,
 * num_q_heads, d->num_kv_heads, max_query_len) exceeds 256 KB (more than
 * 65536 counters).  Past 32 splits the merge is a second launch that uses
 * no counter, so no size limit applies.  Other arguments, results and
 * status codes as in pkv_paged_attn_decode_fused.
 */
int pkv_paged_attn_decode_fused_noalloc(const void *q, int num_q_heads,
                                        int num_tokens, const void *cache,
                                        const pkv_cache_desc *d,
                                        const int32_t *block_table,
                                        int max_blocks_per_seq,
                                        const int32_t *seq_lens,
                                        const int32_t *query_start_loc,
                                        int num_seqs, int max_query_len,
                                        float softmax_scale, const float *k_scale,
                                        const float *v_scale, int num_splits,
                                        float *partial_o, float *partial_lse,
                                        void *out, float *lse_out,
                                        pkv_stream_t stream);

/*
 * pkv_splitkv_reduce -- the split-KV merge (MiMo model card, "What the
 * kernels do" and "Update 2026-10-01").
 *
 * For each row r < num_rows: M = max_s partial_lse[s][r].  If M is -inf, or
 * num_splits is 0, out[r][:] = 0 and lse_out[r] = -inf (never NaN).
 * Otherwise w_s = exp(partial_lse[s][r] - M) (segments at -inf are skipped:
 * their partial_o values never enter the sum and may be left unwritten, as
 * the decode leaves them), out[r][:] = sum_s w_s * partial_o[s][r][:]
 * / sum_s w_s, rounded to bf16, and lse_out[r] = M + log(sum_s w_s).
 * partial_o: float32 [num_splits][num_rows][head_size_v] (all of it must be
 * allocated); partial_lse: float32 [num_splits][num_rows]; out: bf16
 * [num_rows][head_size_v]; lse_out: float32 [num_rows] or NULL.  For the
 * decode call, num_rows = num_tokens * num_q_heads.  When head_size_v is a
 * multiple of 4, partial_o must be 16-byte aligned and out 8-byte aligned
 * (PKV_EINVAL otherwise).
 */
int pkv_splitkv_reduce(const float *partial_o, const float *partial_lse,
                       int num_splits, int num_rows, int head_size_v,
                       void *out, float *lse_out, pkv_stream_t stream);

/*
 * pkv_splitkv_reduce_sink -- pkv_splitkv_reduce with an attention sink: one
 * extra logit per query head in the softmax denominator, with no value
 * vector (MiMo model card, "Update 2026-10-01": the vision encoder's sink,
 * vLLM #58235).  Row r is (token r / num_q_heads, query head r %
 * num_q_heads), as in the decode's partials, and its sink is
 * sinks[r % num_q_heads].  The sink enters the merge once per row, as one
 * more segment with lse = sink and o = 0:
 *   M = max(sink, max_s lse_s); W = exp(sink - M) + sum_s exp(lse_s - M);
 *   out = sum_s exp(lse_s - M) o_s / W; lse_out = M + log(W).
 * A row whose segments are all empty is then 0 with lse = sink.  The decode
 * partials themselves carry no sink: pkv_paged_attn_decode followed by this
 * call gives sink attention.
 * sinks: float32 [num_q_heads], device memory, or NULL (then the result is
 * pkv_splitkv_reduce's); a sink of -inf is no sink.
 * PKV_EINVAL also when num_q_heads < 1 or num_rows is not a multiple of it.
 * Other arguments and status codes as in pkv_splitkv_reduce.
 */
int pkv_splitkv_reduce_sink(const float *partial_o, const float *partial_lse,
                            int num_splits, int num_rows, int head_size_v,
                            const float *sinks, int num_q_heads, void *out,
                            float *lse_out, pkv_stream_t stream);

/*
 * pkv_decode_suggest_splits -- a split count for the decode launch on the
 * current device: two work units per SM for a single sequence; for a batch
 * two to four per SM, preferring a unit count that divides evenly over the
 * SMs (a unit covers four KV heads when num_kv_heads is a multiple of 4, else
 * one); for sequences of up to max_seq_len keys, capped so that every segment
 * keeps at least 256 keys and one page.
 * Host-only; returns >= 1, or a negative status.
 */
int pkv_decode_suggest_splits(int num_seqs, int num_q_heads, int num_kv_heads,
                              int max_query_len, int max_seq_len,
                              int block_size);

/*
 * pkv_supports -- whether this build serves a K/V head-size pair for a cache
 * dtype in each call: bit 0 write, bit 1 prefill, bit 2 decode.
 * Mirrors the per-backend capability check of vLLM PR #64064 ("Details":
 * v <= k is what a page split at head_size can serve); 0 when v > k.
 */
int pkv_supports(int head_size, int head_size_v, int dtype);

/*
 * pkv_get_device_error -- reads and clears the library's device error word
 * (PKV_EDEV_*), ordering the read after all work queued on `stream`.  This
 * call synchronises `stream`.  Returns PKV_OK or PKV_ECUDA.
 */
int pkv_get_device_error(int *code, pkv_stream_t stream);

/*
 * pkv_selftest_bounded_wait -- checks, on the current device, the failure
 * path that every kernel of the library shares: a one-warp kernel waits on an
 * mbarrier that nothing arrives on, with the same bounded wait the kernels
 * use but a limit of `limit_us` microseconds (1 .. 2,000,000); the wait
 * gives up, records PKV_EDEV_TIMEOUT in the device error word and the kernel
 * returns, so the context stays usable.  Read the outcome with
 * pkv_get_device_error.  Not part of the attention path (the pages have no
 * counterpart); asynchronous on `stream`; PKV_EINVAL for a limit out of
 * range.
 */
int pkv_selftest_bounded_wait(int limit_us, pkv_stream_t stream);

/* The cudaError_t of the last PKV_ECUDA return on the calling thread. */
int pkv_last_cuda_error(void);

/* A static description of a status code. */
const char *pkv_status_string(int status);

#ifdef __cplusplus
}
#endif

#endif /* PKV_H_ */
