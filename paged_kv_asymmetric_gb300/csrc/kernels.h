// kernels.h -- internal launch interfaces between the C ABI (api.cu) and the
// kernels.  Not installed; the public interface is include/pkv.h.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "pkv.h"

namespace pkv {

struct WriteParams {
  const __nv_bfloat16* key;
  const __nv_bfloat16* value;
  int64_t key_tok_stride, key_head_stride;
  int64_t val_tok_stride, val_head_stride;
  const int64_t* slot_mapping;
  int num_tokens;
  int has_value;
  void* cache;
  int dtype, layout, num_blocks, block_size, num_kv_heads, row_elems;
  int k_off, head_size, v_off, head_size_v, scale_mode;
  const float* k_scale;
  const float* v_scale;
  int* err;
};

// Shared by the decode and prefill kernels.
struct AttnParams {
  const __nv_bfloat16* q;      // [T][Hq][dk]
  const void* cache;
  int dtype, layout, num_blocks, block_size, num_kv_heads, row_elems;
  int k_off, head_size, v_off, head_size_v, scale_mode;
  const int32_t* block_table;
  int max_blocks_per_seq;
  const int32_t* seq_lens;
  const int32_t* query_start_loc;
  int num_seqs;
  int num_tokens;
  int num_q_heads;
  int group;                   // Hq / Hkv
  int max_query_len;
  float softmax_scale;
  const float* k_scale;
  const float* v_scale;
  // decode: the segment count; with split_ranges = W > 0 the segments are
  // balanced ranges of the batch's pages (W ranges at most), else equal
  // shares of each sequence's pages
  int num_splits;
  int split_ranges;
  float* partial_o;            // [S][T][Hq][dv]
  float* partial_lse;          // [S][T][Hq]
  // prefill, and the fused decode's merged output
  __nv_bfloat16* out;          // [T][Hq][dv]
  int* err;
  // fused decode: counters of finished units per (sequence, KV-head block,
  // row group), the merged lse (nullable), and whether to merge in-kernel
  int* counters;
  float* lse_out;
  int fused;
  // prefill: one attention-sink logit per query head (nullable), an extra
  // term exp(sink) in each row's softmax denominator
  const float* sinks;
  // prefill over an FP8 cache, or over a bf16 cache of widened E4M3 codes:
  // k_scale is folded into the softmax scale and v_scale into the output,
  // per KV head (or per tensor)
  int fold_scales;
};

// The FP8 prefill's first pass: every page a sequence uses is copied from
// the FP8 cache into `pages` (bf16, the same page geometry) as its E4M3
// codes widened exactly to bf16, page j of sequence b to page
// b * max_blocks_per_seq + j, whose index goes to remap[b][j] (-1 for
// entries past the sequence's pages).  An out-of-range page id is recorded
// in err and its remap entry set to -1.
cudaError_t launch_fp8_pages_to_bf16(const uint8_t* cache, int64_t page_elems, int num_blocks,
                                     const int32_t* block_table, int max_blocks_per_seq,
                                     const int32_t* seq_lens, int num_seqs, int block_size,
                                     __nv_bfloat16* pages, int32_t* remap, int* err,
                                     int num_sms, cudaStream_t stream);

// The fused decode merges in-kernel up to this many splits (its per-row
// weights live in shared memory); beyond, the merge is a second launch.
constexpr int kFusedMaxSplits = 32;

cudaError_t launch_cache_write(const WriteParams& p, int num_sms,
                               cudaStream_t stream);

// Returns cudaErrorNotSupported for a shape without an instantiation.
cudaError_t launch_decode(const AttnParams& p, int num_sms, cudaStream_t stream);
// Resident CTAs per SM of the decode kernel form that serves p's shape, and
// its head blocks (KV heads / heads per unit).
int decode_ctas_per_sm(const AttnParams& p);
int decode_head_blocks(const AttnParams& p);
// Balanced ranges keep every sequence's first page, length and query range
// on chip for batches of up to kBalancedMaxSeqs sequences; larger batches
// keep a window of that many sequences and every chunk's first page, so at
// most kBalancedMaxSeqs chunks: kBalancedMaxSeqsWide sequences per launch.
constexpr int kBalancedMaxSeqs = 128;
constexpr int kBalancedMaxSeqsWide = kBalancedMaxSeqs * kBalancedMaxSeqs;
bool decode_supported(int head_size, int head_size_v, int dtype);

// sinks: nullable, one attention-sink logit per query head; row r takes
// sinks[r % num_q_heads].
cudaError_t launch_splitkv_reduce(const float* partial_o,
                                  const float* partial_lse, int num_splits,
                                  int num_rows, int head_size_v,
                                  __nv_bfloat16* out, float* lse_out,
                                  cudaStream_t stream, const float* sinks = nullptr,
                                  int num_q_heads = 1);

cudaError_t launch_prefill(const AttnParams& p, int num_sms,
                           cudaStream_t stream);

cudaError_t launch_bounded_wait_selftest(int* err, uint64_t limit_ns,
                                         cudaStream_t stream);
bool prefill_supported(int head_size, int head_size_v, int dtype);

}  // namespace pkv
