// api.cu -- the C ABI declared in include/pkv.h: host-side argument checks
// (everything is checked before anything is launched), the device error word
// and the launches.  No call allocates device memory or synchronises, except
// pkv_get_device_error.
#include <math.h>
#include <stdint.h>

#include <initializer_list>
#include <mutex>

#include "common.cuh"
#include "kernels.h"

namespace {

// The device error word (PKV_EDEV_*).  Kernels receive its address; host
// code reads it only through pkv_get_device_error.
__device__ int g_pkv_dev_error = 0;

thread_local int t_last_cuda_error = 0;

constexpr int kMaxDevices = 64;
std::mutex g_dev_mu;
int* g_err_ptr[kMaxDevices] = {nullptr};
int g_num_sms[kMaxDevices] = {0};

// Counters of pkv_paged_attn_decode_fused_noalloc: a fixed array in the
// library's device image instead of a caller workspace (one per device; all
// calls on a device share it).
constexpr int kNoAllocCounters = 65536;
static __device__ __align__(256) int g_noalloc_counters[kNoAllocCounters];
int* g_noalloc_ptr[kMaxDevices] = {nullptr};

int fail_cuda(cudaError_t e) {
  t_last_cuda_error = static_cast<int>(e);
  return PKV_ECUDA;
}

// Per-device constants: the device address of the error word and the SM
// count.  Resolved once per device, with that device current.
int device_info(int** err_ptr, int* num_sms) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return fail_cuda(e);
  if (dev < 0 || dev >= kMaxDevices) return fail_cuda(cudaErrorInvalidDevice);
  std::lock_guard<std::mutex> lock(g_dev_mu);
  if (g_err_ptr[dev] == nullptr) {
    void* ptr = nullptr;
    e = cudaGetSymbolAddress(&ptr, g_pkv_dev_error);
    if (e != cudaSuccess) return fail_cuda(e);
    int sms = 0;
    e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return fail_cuda(e);
    g_num_sms[dev] = sms;
    g_err_ptr[dev] = static_cast<int*>(ptr);
  }
  if (err_ptr) *err_ptr = g_err_ptr[dev];
  if (num_sms) *num_sms = g_num_sms[dev];
  return PKV_OK;
}

int check_desc(const pkv_cache_desc* d) {
  if (d == nullptr) return PKV_EINVAL;
  if (d->dtype != PKV_BF16 && d->dtype != PKV_FP8_E4M3) return PKV_EUNSUPPORTED;
  if (d->layout != PKV_NHD && d->layout != PKV_HND) return PKV_EUNSUPPORTED;
  if (d->scale_mode < PKV_SCALE_NONE || d->scale_mode > PKV_SCALE_HEAD)
    return PKV_EUNSUPPORTED;
  if (d->num_blocks < 1 || d->block_size < 1 || d->num_kv_heads < 1 ||
      d->row_elems < 1 || d->head_size < 1 || d->head_size_v < 1 ||
      d->k_off < 0 || d->v_off < 0)
    return PKV_EINVAL;
  if (static_cast<int64_t>(d->k_off) + d->head_size > d->row_elems ||
      static_cast<int64_t>(d->v_off) + d->head_size_v > d->row_elems)
    return PKV_EINVAL;
  if (d->dtype == PKV_BF16 && d->scale_mode != PKV_SCALE_NONE) return PKV_EINVAL;
  if (d->dtype == PKV_FP8_E4M3 && d->scale_mode == PKV_SCALE_NONE)
    return PKV_EINVAL;
  return PKV_OK;
}

int check_attn_common(const void* q, int num_q_heads, int num_tokens,
                      const void* cache, const pkv_cache_desc* d,
                      const int32_t* block_table, int max_blocks_per_seq,
                      const int32_t* seq_lens, const int32_t* qsl,
                      int num_seqs, float softmax_scale, const float* k_scale,
                      const float* v_scale) {
  int rc = check_desc(d);
  if (rc != PKV_OK) return rc;
  if (d->head_size_v > d->head_size) return PKV_EUNSUPPORTED;
  if (num_tokens < 0 || num_seqs < 0 || num_q_heads < 1) return PKV_EINVAL;
  if (num_q_heads % d->num_kv_heads != 0) return PKV_EINVAL;
  if (!isfinite(softmax_scale)) return PKV_EINVAL;
  if (num_tokens > 0 && q == nullptr) return PKV_EINVAL;
  if (cache == nullptr || qsl == nullptr) return PKV_EINVAL;
  if (num_seqs > 0 &&
      (block_table == nullptr || seq_lens == nullptr || max_blocks_per_seq < 1))
    return PKV_EINVAL;
  if (d->dtype == PKV_FP8_E4M3 && (k_scale == nullptr || v_scale == nullptr))
    return PKV_EINVAL;
  return PKV_OK;
}

pkv::AttnParams make_params(const void* q, int num_q_heads, int num_tokens,
                            const void* cache, const pkv_cache_desc* d,
                            const int32_t* block_table, int max_blocks_per_seq,
                            const int32_t* seq_lens, const int32_t* qsl,
                            int num_seqs, float softmax_scale,
                            const float* k_scale, const float* v_scale,
                            int* err) {
  pkv::AttnParams p{};
  p.q = static_cast<const __nv_bfloat16*>(q);
  p.cache = cache;
  p.dtype = d->dtype;
  p.layout = d->layout;
  p.num_blocks = d->num_blocks;
  p.block_size = d->block_size;
  p.num_kv_heads = d->num_kv_heads;
  p.row_elems = d->row_elems;
  p.k_off = d->k_off;
  p.head_size = d->head_size;
  p.v_off = d->v_off;
  p.head_size_v = d->head_size_v;
  p.scale_mode = d->scale_mode;
  p.block_table = block_table;
  p.max_blocks_per_seq = max_blocks_per_seq;
  p.seq_lens = seq_lens;
  p.query_start_loc = qsl;
  p.num_seqs = num_seqs;
  p.num_tokens = num_tokens;
  p.num_q_heads = num_q_heads;
  p.group = num_q_heads / d->num_kv_heads;
  p.softmax_scale = softmax_scale;
  p.k_scale = k_scale;
  p.v_scale = v_scale;
  p.err = err;
  return p;
}

bool aligned16(const void* p) {
  return (reinterpret_cast<uintptr_t>(p) & 15u) == 0;
}

// Whether every pointer is plain device memory of the current device.  The
// prefill's tensor maps and its TMA loads (cluster-multicast ones among
// them) must cover this GPU's own memory only: pinned or mapped host memory, managed memory and a
// peer GPU's memory are refused before any tensor map is encoded.
int check_local_device(std::initializer_list<const void*> ptrs) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return fail_cuda(e);
  for (const void* ptr : ptrs) {
    cudaPointerAttributes a{};
    e = cudaPointerGetAttributes(&a, ptr);
    if (e != cudaSuccess) {
      (void)cudaGetLastError();  // not a pointer CUDA knows: clear the error
      return PKV_EINVAL;
    }
    if (a.type != cudaMemoryTypeDevice || a.device != dev) return PKV_EINVAL;
  }
  return PKV_OK;
}

}  // namespace

extern "C" {

int pkv_kv_cache_write(const void* key, int64_t key_tok_stride,
                       int64_t key_head_stride, const void* value,
                       int64_t val_tok_stride, int64_t val_head_stride,
                       const int64_t* slot_mapping, int num_tokens, void* cache,
                       const pkv_cache_desc* d, const float* k_scale,
                       const float* v_scale, pkv_stream_t stream) {
  int rc = check_desc(d);
  if (rc != PKV_OK) return rc;
  if (num_tokens < 0) return PKV_EINVAL;
  if (num_tokens == 0) return PKV_OK;
  if (key == nullptr || slot_mapping == nullptr || cache == nullptr)
    return PKV_EINVAL;
  if (key_tok_stride < 0 || key_head_stride < 0 || val_tok_stride < 0 ||
      val_head_stride < 0)
    return PKV_EINVAL;
  if (d->dtype == PKV_FP8_E4M3 &&
      (k_scale == nullptr || (value != nullptr && v_scale == nullptr)))
    return PKV_EINVAL;
  int* err = nullptr;
  int sms = 0;
  rc = device_info(&err, &sms);
  if (rc != PKV_OK) return rc;
  pkv::WriteParams p{};
  p.key = static_cast<const __nv_bfloat16*>(key);
  p.value = static_cast<const __nv_bfloat16*>(value);
  p.key_tok_stride = key_tok_stride;
  p.key_head_stride = key_head_stride;
  p.val_tok_stride = val_tok_stride;
  p.val_head_stride = val_head_stride;
  p.slot_mapping = slot_mapping;
  p.num_tokens = num_tokens;
  p.has_value = value != nullptr;
  p.cache = cache;
  p.dtype = d->dtype;
  p.layout = d->layout;
  p.num_blocks = d->num_blocks;
  p.block_size = d->block_size;
  p.num_kv_heads = d->num_kv_heads;
  p.row_elems = d->row_elems;
  p.k_off = d->k_off;
  p.head_size = d->head_size;
  p.v_off = d->v_off;
  p.head_size_v = d->head_size_v;
  p.scale_mode = d->scale_mode;
  p.k_scale = k_scale;
  p.v_scale = value != nullptr ? v_scale : k_scale;
  p.err = err;
  cudaError_t e = pkv::launch_cache_write(p, sms, reinterpret_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? PKV_OK : fail_cuda(e);
}

namespace {

int prefill_impl(const void* q, int num_q_heads, int num_tokens, const void* cache,
                 const pkv_cache_desc* d, const int32_t* block_table,
                 int max_blocks_per_seq, const int32_t* seq_lens,
                 const int32_t* query_start_loc, int num_seqs, float softmax_scale,
                 const float* k_scale, const float* v_scale, const float* sinks,
                 void* out, pkv_stream_t stream, int fold_scale_mode = -1) {
  int rc = check_attn_common(q, num_q_heads, num_tokens, cache, d, block_table,
                             max_blocks_per_seq, seq_lens, query_start_loc,
                             num_seqs, softmax_scale, k_scale, v_scale);
  if (rc != PKV_OK) return rc;
  if (num_tokens > 0 && out == nullptr) return PKV_EINVAL;
  if (!(softmax_scale > 0.f)) return PKV_EINVAL;
  if (!pkv::prefill_supported(d->head_size, d->head_size_v, d->dtype))
    return PKV_EUNSUPPORTED;
  const int G = num_q_heads / d->num_kv_heads;
  if (128 % G != 0) return PKV_EUNSUPPORTED;
  const int bs = d->block_size;
  if (bs < 8 || (bs & (bs - 1)) != 0) return PKV_EUNSUPPORTED;
  // TMA tiles: 16-byte aligned base and row strides, 64-column K/V boxes
  // whose first byte sits on a 16-byte boundary
  const int esz = d->dtype == PKV_FP8_E4M3 ? 1 : 2;
  if (!aligned16(cache) || !aligned16(q) || (d->row_elems * esz) % 16 != 0 ||
      d->k_off % 64 != 0 || (d->v_off * esz) % 16 != 0)
    return PKV_EUNSUPPORTED;
  if (num_tokens == 0 || num_seqs == 0) return PKV_OK;
  // q and the cache are read through tensor maps (some K/V boxes multicast
  // to both CTAs of a cluster), out is written: all must be this GPU's memory
  rc = check_local_device({q, cache, out});
  if (rc != PKV_OK) return rc;
  int* err = nullptr;
  int sms = 0;
  rc = device_info(&err, &sms);
  if (rc != PKV_OK) return rc;
  pkv::AttnParams p = make_params(q, num_q_heads, num_tokens, cache, d,
                                  block_table, max_blocks_per_seq, seq_lens,
                                  query_start_loc, num_seqs, softmax_scale,
                                  k_scale, v_scale, err);
  p.out = static_cast<__nv_bfloat16*>(out);
  p.sinks = sinks;
  // FP8 cache: the E4M3 codes are widened to bf16 in the kernel, k_scale
  // folds into the softmax scale and v_scale into the output; the same fold
  // for a bf16 cache that holds widened E4M3 codes (the two-pass form)
  p.fold_scales = d->dtype == PKV_FP8_E4M3 ? 1 : 0;
  if (fold_scale_mode >= 0) {
    p.fold_scales = 1;
    p.scale_mode = fold_scale_mode;
  }
  cudaError_t e = pkv::launch_prefill(p, sms, reinterpret_cast<cudaStream_t>(stream));
  if (e == cudaErrorNotSupported) return PKV_EUNSUPPORTED;
  return e == cudaSuccess ? PKV_OK : fail_cuda(e);
}

}  // namespace

int pkv_paged_attn_prefill(const void* q, int num_q_heads, int num_tokens,
                           const void* cache, const pkv_cache_desc* d,
                           const int32_t* block_table, int max_blocks_per_seq,
                           const int32_t* seq_lens,
                           const int32_t* query_start_loc, int num_seqs,
                           float softmax_scale, const float* k_scale,
                           const float* v_scale, void* out,
                           pkv_stream_t stream) {
  return prefill_impl(q, num_q_heads, num_tokens, cache, d, block_table, max_blocks_per_seq,
                      seq_lens, query_start_loc, num_seqs, softmax_scale, k_scale, v_scale,
                      nullptr, out, stream);
}

namespace {

// The FP8 prefill's workspace: widened pages, then the remapped block table.
size_t fp8_pages_bytes(int num_seqs, int max_blocks_per_seq, const pkv_cache_desc* d) {
  const size_t page = static_cast<size_t>(d->block_size) * d->num_kv_heads * d->row_elems * 2;
  const size_t bytes = static_cast<size_t>(num_seqs) * max_blocks_per_seq * page;
  return (bytes + 255) & ~static_cast<size_t>(255);
}

}  // namespace

size_t pkv_prefill_fp8_workspace_bytes(int num_seqs, int max_blocks_per_seq,
                                       const pkv_cache_desc* d) {
  if (d == nullptr || check_desc(d) != PKV_OK || num_seqs < 0 || max_blocks_per_seq < 1)
    return 0;
  if (static_cast<int64_t>(num_seqs) * max_blocks_per_seq > (int64_t{1} << 31) - 1) return 0;
  return fp8_pages_bytes(num_seqs, max_blocks_per_seq, d) +
         static_cast<size_t>(num_seqs) * max_blocks_per_seq * sizeof(int32_t);
}

int pkv_paged_attn_prefill_fp8(const void* q, int num_q_heads, int num_tokens,
                               const void* cache, const pkv_cache_desc* d,
                               const int32_t* block_table, int max_blocks_per_seq,
                               const int32_t* seq_lens, const int32_t* query_start_loc,
                               int num_seqs, float softmax_scale, const float* k_scale,
                               const float* v_scale, const float* sinks, void* workspace,
                               size_t workspace_bytes, void* out, pkv_stream_t stream) {
  if (d == nullptr) return PKV_EINVAL;
  int rc = check_attn_common(q, num_q_heads, num_tokens, cache, d, block_table,
                             max_blocks_per_seq, seq_lens, query_start_loc, num_seqs,
                             softmax_scale, k_scale, v_scale);
  if (rc != PKV_OK) return rc;
  if (d->dtype != PKV_FP8_E4M3) return PKV_EINVAL;
  const size_t need = pkv_prefill_fp8_workspace_bytes(num_seqs, max_blocks_per_seq, d);
  if (need == 0 && num_seqs > 0) return PKV_EINVAL;
  if (num_tokens > 0 && (workspace == nullptr || workspace_bytes < need ||
                         (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0))
    return PKV_EINVAL;
  // the widened pages are an ordinary bf16 cache of num_seqs x max_blocks
  // pages (unscaled codes: the scales fold into the prefill)
  pkv_cache_desc wd = *d;
  wd.dtype = PKV_BF16;
  wd.scale_mode = PKV_SCALE_NONE;
  wd.num_blocks = num_seqs * max_blocks_per_seq;
  if (num_tokens == 0 || num_seqs == 0) return PKV_OK;
  if (wd.num_blocks < 1) return PKV_EINVAL;
  // every later check of the prefill, on the widened cache, before any launch
  if (!(softmax_scale > 0.f) || out == nullptr) return PKV_EINVAL;
  if (!pkv::prefill_supported(wd.head_size, wd.head_size_v, wd.dtype)) return PKV_EUNSUPPORTED;
  const int G = num_q_heads / d->num_kv_heads;
  if (128 % G != 0) return PKV_EUNSUPPORTED;
  const int bs = d->block_size;
  if (bs < 8 || (bs & (bs - 1)) != 0) return PKV_EUNSUPPORTED;
  if (!aligned16(cache) || !aligned16(q) || (d->row_elems * 2) % 16 != 0 ||
      d->k_off % 64 != 0 || d->v_off % 8 != 0)
    return PKV_EUNSUPPORTED;
  // the widened pages (workspace) and q are read through tensor maps by the
  // prefill: every buffer must be this GPU's memory, checked before the
  // first launch
  rc = check_local_device({q, cache, workspace, out});
  if (rc != PKV_OK) return rc;
  int* err = nullptr;
  int sms = 0;
  rc = device_info(&err, &sms);
  if (rc != PKV_OK) return rc;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  auto* pages = reinterpret_cast<__nv_bfloat16*>(ws);
  auto* remap = reinterpret_cast<int32_t*>(ws + fp8_pages_bytes(num_seqs, max_blocks_per_seq, d));
  const int64_t page_elems = static_cast<int64_t>(bs) * d->num_kv_heads * d->row_elems;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  cudaError_t e = pkv::launch_fp8_pages_to_bf16(
      static_cast<const uint8_t*>(cache), page_elems, d->num_blocks, block_table,
      max_blocks_per_seq, seq_lens, num_seqs, bs, pages, remap, err, sms, s);
  if (e != cudaSuccess) return fail_cuda(e);
  return prefill_impl(q, num_q_heads, num_tokens, pages, &wd, remap, max_blocks_per_seq,
                      seq_lens, query_start_loc, num_seqs, softmax_scale, k_scale, v_scale,
                      sinks, out, stream, /*fold_scale_mode=*/d->scale_mode);
}

int pkv_paged_attn_prefill_sink(const void* q, int num_q_heads, int num_tokens,
                                const void* cache, const pkv_cache_desc* d,
                                const int32_t* block_table, int max_blocks_per_seq,
                                const int32_t* seq_lens, const int32_t* query_start_loc,
                                int num_seqs, float softmax_scale, const float* k_scale,
                                const float* v_scale, const float* sinks, void* out,
                                pkv_stream_t stream) {
  return prefill_impl(q, num_q_heads, num_tokens, cache, d, block_table, max_blocks_per_seq,
                      seq_lens, query_start_loc, num_seqs, softmax_scale, k_scale, v_scale,
                      sinks, out, stream);
}

namespace {

// Checks of pkv_paged_attn_decode and its fused form, and the kernel
// parameters they share.  `launch` is false when there is nothing to do.
int decode_prepare(const void* q, int num_q_heads, int num_tokens, const void* cache,
                   const pkv_cache_desc* d, const int32_t* block_table,
                   int max_blocks_per_seq, const int32_t* seq_lens,
                   const int32_t* query_start_loc, int num_seqs, int max_query_len,
                   float softmax_scale, const float* k_scale, const float* v_scale,
                   int num_splits, float* partial_o, float* partial_lse,
                   pkv::AttnParams* p, int* sms, bool* launch) {
  *launch = false;
  int rc = check_attn_common(q, num_q_heads, num_tokens, cache, d, block_table,
                             max_blocks_per_seq, seq_lens, query_start_loc,
                             num_seqs, softmax_scale, k_scale, v_scale);
  if (rc != PKV_OK) return rc;
  if (max_query_len < 1 || max_query_len > 64) return PKV_EINVAL;
  if (num_splits < 1 || num_splits > 65535) return PKV_EINVAL;
  if (num_tokens > 0 && (partial_o == nullptr || partial_lse == nullptr))
    return PKV_EINVAL;
  if (((reinterpret_cast<uintptr_t>(partial_o) | reinterpret_cast<uintptr_t>(partial_lse)) &
       3u) != 0)
    return PKV_EINVAL;  // float stores
  if (!pkv::decode_supported(d->head_size, d->head_size_v, d->dtype))
    return PKV_EUNSUPPORTED;
  const int esz = d->dtype == PKV_FP8_E4M3 ? 1 : 2;
  const int lo = d->k_off < d->v_off ? d->k_off : d->v_off;
  const int hi_k = d->k_off + d->head_size, hi_v = d->v_off + d->head_size_v;
  const int span = (hi_k > hi_v ? hi_k : hi_v) - lo;
  const int max_span = d->head_size == 192 ? 320 : 576;
  // 16-byte cp.async pieces: the staged span, its start and the K / V starts
  // within it are whole pieces; rows and the cache base are 16-byte aligned.
  if (span > max_span || (span * esz) % 16 != 0 || (lo * esz) % 16 != 0 ||
      ((d->k_off - lo) * esz) % 16 != 0 || ((d->v_off - lo) * esz) % 16 != 0 ||
      (static_cast<int64_t>(d->row_elems) * esz) % 16 != 0 ||
      !aligned16(cache) || !aligned16(q))
    return PKV_EUNSUPPORTED;
  const int G = num_q_heads / d->num_kv_heads;
  const int64_t row_groups = (static_cast<int64_t>(max_query_len) * G + 15) / 16;
  if (row_groups * d->num_kv_heads > 65535 || num_seqs > 65535)
    return PKV_EINVAL;
  // work units (split x sequence x KV head x row group) are counted in int
  if (static_cast<int64_t>(num_splits) * num_seqs * d->num_kv_heads * row_groups >
      (int64_t{1} << 30))
    return PKV_EINVAL;
  // 16-key chunks are whole TMA boxes of one page (or two pages of 8)
  if (!(d->block_size % 16 == 0 || d->block_size == 8)) return PKV_EUNSUPPORTED;
  if (num_tokens == 0 || num_seqs == 0) return PKV_OK;
  int* err = nullptr;
  rc = device_info(&err, sms);
  if (rc != PKV_OK) return rc;
  *p = make_params(q, num_q_heads, num_tokens, cache, d, block_table,
                   max_blocks_per_seq, seq_lens, query_start_loc, num_seqs,
                   softmax_scale, k_scale, v_scale, err);
  p->max_query_len = max_query_len;
  p->num_splits = num_splits;
  p->partial_o = partial_o;
  p->partial_lse = partial_lse;
  *launch = true;
  return PKV_OK;
}

}  // namespace

int pkv_paged_attn_decode(const void* q, int num_q_heads, int num_tokens,
                          const void* cache, const pkv_cache_desc* d,
                          const int32_t* block_table, int max_blocks_per_seq,
                          const int32_t* seq_lens,
                          const int32_t* query_start_loc, int num_seqs,
                          int max_query_len, float softmax_scale,
                          const float* k_scale, const float* v_scale,
                          int num_splits, float* partial_o, float* partial_lse,
                          pkv_stream_t stream) {
  pkv::AttnParams p{};
  int sms = 0;
  bool launch = false;
  const int rc = decode_prepare(q, num_q_heads, num_tokens, cache, d, block_table,
                                max_blocks_per_seq, seq_lens, query_start_loc, num_seqs,
                                max_query_len, softmax_scale, k_scale, v_scale, num_splits,
                                partial_o, partial_lse, &p, &sms, &launch);
  if (rc != PKV_OK || !launch) return rc;
  cudaError_t e = pkv::launch_decode(p, sms, reinterpret_cast<cudaStream_t>(stream));
  if (e == cudaErrorNotSupported) return PKV_EUNSUPPORTED;
  return e == cudaSuccess ? PKV_OK : fail_cuda(e);
}

namespace {

// One (range, head block) item per resident CTA of the decode kernel.
int default_ranges(const pkv::AttnParams& p, int sms) {
  const int slots = pkv::decode_ctas_per_sm(p) * sms;
  const int hb = pkv::decode_head_blocks(p);
  return slots / hb > 0 ? slots / hb : 1;
}

}  // namespace

int pkv_paged_attn_decode_balanced(const void* q, int num_q_heads, int num_tokens,
                                   const void* cache, const pkv_cache_desc* d,
                                   const int32_t* block_table, int max_blocks_per_seq,
                                   const int32_t* seq_lens,
                                   const int32_t* query_start_loc, int num_seqs,
                                   int max_query_len, float softmax_scale,
                                   const float* k_scale, const float* v_scale,
                                   int max_splits, int num_ranges, float* partial_o,
                                   float* partial_lse, pkv_stream_t stream) {
  if (num_ranges < 0 || num_ranges > (1 << 24)) return PKV_EINVAL;
  // the batch's page line is counted in int
  if (static_cast<int64_t>(num_seqs) * max_blocks_per_seq > INT32_MAX) return PKV_EINVAL;
  if (num_seqs > pkv::kBalancedMaxSeqsWide) return PKV_EUNSUPPORTED;
  pkv::AttnParams p{};
  int sms = 0;
  bool launch = false;
  const int rc = decode_prepare(q, num_q_heads, num_tokens, cache, d, block_table,
                                max_blocks_per_seq, seq_lens, query_start_loc, num_seqs,
                                max_query_len, softmax_scale, k_scale, v_scale, max_splits,
                                partial_o, partial_lse, &p, &sms, &launch);
  if (rc != PKV_OK || !launch) return rc;
  p.split_ranges = num_ranges > 0 ? num_ranges : default_ranges(p, sms);
  // (range, head block) items are counted in int
  if (static_cast<int64_t>(p.split_ranges) * pkv::decode_head_blocks(p) > (int64_t{1} << 30))
    return PKV_EINVAL;
  cudaError_t e = pkv::launch_decode(p, sms, reinterpret_cast<cudaStream_t>(stream));
  if (e == cudaErrorNotSupported) return PKV_EUNSUPPORTED;
  return e == cudaSuccess ? PKV_OK : fail_cuda(e);
}

int pkv_decode_balanced_ranges(const pkv_cache_desc* d) {
  int rc = check_desc(d);
  if (rc != PKV_OK) return rc;
  if (!pkv::decode_supported(d->head_size, d->head_size_v, d->dtype)) return PKV_EUNSUPPORTED;
  int sms = 0;
  rc = device_info(nullptr, &sms);
  if (rc != PKV_OK) return rc;
  pkv::AttnParams p{};
  p.head_size = d->head_size;
  p.head_size_v = d->head_size_v;
  p.dtype = d->dtype;
  p.num_kv_heads = d->num_kv_heads;
  return default_ranges(p, sms);
}

int pkv_paged_attn_decode_balanced_fused(
    const void* q, int num_q_heads, int num_tokens, const void* cache,
    const pkv_cache_desc* d, const int32_t* block_table, int max_blocks_per_seq,
    const int32_t* seq_lens, const int32_t* query_start_loc, int num_seqs,
    int max_query_len, float softmax_scale, const float* k_scale, const float* v_scale,
    int max_splits, int num_ranges, float* partial_o, float* partial_lse, void* workspace,
    size_t workspace_bytes, void* out, float* lse_out, pkv_stream_t stream);

size_t pkv_decode_workspace_bytes(int num_seqs, int num_q_heads, int num_kv_heads,
                                  int max_query_len) {
  if (num_seqs < 0 || num_q_heads < 1 || num_kv_heads < 1 || max_query_len < 1 ||
      num_q_heads % num_kv_heads != 0)
    return 0;
  const int64_t G = num_q_heads / num_kv_heads;
  const int64_t rg = (static_cast<int64_t>(max_query_len) * G + 15) / 16;
  return static_cast<size_t>(num_seqs) * num_kv_heads * rg * sizeof(int);
}

namespace {

// The fused decode; with `clear`, the counters it uses are zeroed on the
// stream first (after every argument has been checked).  num_ranges >= 0:
// balanced ranges (0: the default count), else equal segments.
int decode_fused_impl(const void* q, int num_q_heads, int num_tokens, const void* cache,
                      const pkv_cache_desc* d, const int32_t* block_table,
                      int max_blocks_per_seq, const int32_t* seq_lens,
                      const int32_t* query_start_loc, int num_seqs, int max_query_len,
                      float softmax_scale, const float* k_scale, const float* v_scale,
                      int num_splits, float* partial_o, float* partial_lse, void* workspace,
                      size_t workspace_bytes, void* out, float* lse_out, pkv_stream_t stream,
                      bool clear, int num_ranges = -1) {
  const bool balanced = num_ranges >= 0;
  if (balanced) {
    if (num_ranges > (1 << 24)) return PKV_EINVAL;
    if (static_cast<int64_t>(num_seqs) * max_blocks_per_seq > INT32_MAX) return PKV_EINVAL;
    if (num_seqs > pkv::kBalancedMaxSeqsWide) return PKV_EUNSUPPORTED;
  }
  pkv::AttnParams p{};
  int sms = 0;
  bool launch = false;
  int rc = decode_prepare(q, num_q_heads, num_tokens, cache, d, block_table,
                          max_blocks_per_seq, seq_lens, query_start_loc, num_seqs,
                          max_query_len, softmax_scale, k_scale, v_scale, num_splits,
                          partial_o, partial_lse, &p, &sms, &launch);
  if (rc != PKV_OK) return rc;
  if (num_tokens > 0 && out == nullptr) return PKV_EINVAL;
  // the merge (in the kernel, or the second launch past 32 splits) reads the
  // partials 16 bytes at a time and stores 4 bf16 outputs at a time, and
  // counts rows in int
  if ((reinterpret_cast<uintptr_t>(out) & 7u) != 0) return PKV_EINVAL;
  if ((reinterpret_cast<uintptr_t>(partial_o) & 15u) != 0) return PKV_EINVAL;
  if (static_cast<int64_t>(num_tokens) * num_q_heads > INT32_MAX) return PKV_EINVAL;
  const size_t need = pkv_decode_workspace_bytes(num_seqs, num_q_heads, d->num_kv_heads,
                                                 max_query_len);
  if (num_tokens > 0 && (workspace == nullptr || workspace_bytes < need ||
                         (reinterpret_cast<uintptr_t>(workspace) & 3u) != 0))
    return PKV_EINVAL;
  if (!launch) return PKV_OK;
  if (balanced) {
    p.split_ranges = num_ranges > 0 ? num_ranges : default_ranges(p, sms);
    if (static_cast<int64_t>(p.split_ranges) * pkv::decode_head_blocks(p) > (int64_t{1} << 30))
      return PKV_EINVAL;
  }
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (clear && num_splits <= pkv::kFusedMaxSplits) {
    const cudaError_t e = cudaMemsetAsync(workspace, 0, need, s);
    if (e != cudaSuccess) return fail_cuda(e);
  }
  p.out = static_cast<__nv_bfloat16*>(out);
  p.lse_out = lse_out;
  if (num_splits <= pkv::kFusedMaxSplits) {
    p.counters = static_cast<int*>(workspace);
    p.fused = 1;
    cudaError_t e = pkv::launch_decode(p, sms, s);
    if (e == cudaErrorNotSupported) return PKV_EUNSUPPORTED;
    return e == cudaSuccess ? PKV_OK : fail_cuda(e);
  }
  cudaError_t e = pkv::launch_decode(p, sms, s);
  if (e == cudaErrorNotSupported) return PKV_EUNSUPPORTED;
  if (e == cudaSuccess)
    e = pkv::launch_splitkv_reduce(partial_o, partial_lse, num_splits,
                                   num_tokens * num_q_heads, d->head_size_v,
                                   p.out, lse_out, s);
  return e == cudaSuccess ? PKV_OK : fail_cuda(e);
}

}  // namespace

int pkv_paged_attn_decode_fused(const void* q, int num_q_heads, int num_tokens,
                                const void* cache, const pkv_cache_desc* d,
                                const int32_t* block_table, int max_blocks_per_seq,
                                const int32_t* seq_lens,
                                const int32_t* query_start_loc, int num_seqs,
                                int max_query_len, float softmax_scale,
                                const float* k_scale, const float* v_scale,
                                int num_splits, float* partial_o, float* partial_lse,
                                void* workspace, size_t workspace_bytes, void* out,
                                float* lse_out, pkv_stream_t stream) {
  return decode_fused_impl(q, num_q_heads, num_tokens, cache, d, block_table,
                           max_blocks_per_seq, seq_lens, query_start_loc, num_seqs,
                           max_query_len, softmax_scale, k_scale, v_scale, num_splits,
                           partial_o, partial_lse, workspace, workspace_bytes, out, lse_out,
                           stream, /*clear=*/false);
}

int pkv_paged_attn_decode_fused_noalloc(const void* q, int num_q_heads, int num_tokens,
                                        const void* cache, const pkv_cache_desc* d,
                                        const int32_t* block_table, int max_blocks_per_seq,
                                        const int32_t* seq_lens,
                                        const int32_t* query_start_loc, int num_seqs,
                                        int max_query_len, float softmax_scale,
                                        const float* k_scale, const float* v_scale,
                                        int num_splits, float* partial_o,
                                        float* partial_lse, void* out, float* lse_out,
                                        pkv_stream_t stream) {
  if (d == nullptr) return PKV_EINVAL;
  // The counters serve the in-kernel merge only (up to kFusedMaxSplits
  // splits); there the sizes must fit the fixed counter array.  Past it the
  // merge is a second launch that uses no counter, and any size is taken.
  const size_t array_bytes = sizeof(int) * static_cast<size_t>(kNoAllocCounters);
  const size_t need = pkv_decode_workspace_bytes(num_seqs, num_q_heads, d->num_kv_heads,
                                                 max_query_len);
  const bool in_kernel_merge = num_splits <= pkv::kFusedMaxSplits;
  if (in_kernel_merge && need > array_bytes) return PKV_EINVAL;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return fail_cuda(e);
  if (dev < 0 || dev >= kMaxDevices) return fail_cuda(cudaErrorInvalidDevice);
  int* counters = nullptr;
  {
    std::lock_guard<std::mutex> lock(g_dev_mu);
    if (g_noalloc_ptr[dev] == nullptr) {
      void* ptr = nullptr;
      e = cudaGetSymbolAddress(&ptr, g_noalloc_counters);
      if (e != cudaSuccess) return fail_cuda(e);
      g_noalloc_ptr[dev] = static_cast<int*>(ptr);
    }
    counters = g_noalloc_ptr[dev];
  }
  return decode_fused_impl(q, num_q_heads, num_tokens, cache, d, block_table,
                           max_blocks_per_seq, seq_lens, query_start_loc, num_seqs,
                           max_query_len, softmax_scale, k_scale, v_scale, num_splits,
                           partial_o, partial_lse, counters,
                           in_kernel_merge || need <= array_bytes ? array_bytes : need, out,
                           lse_out, stream, /*clear=*/true);
}

int pkv_paged_attn_decode_balanced_fused(
    const void* q, int num_q_heads, int num_tokens, const void* cache,
    const pkv_cache_desc* d, const int32_t* block_table, int max_blocks_per_seq,
    const int32_t* seq_lens, const int32_t* query_start_loc, int num_seqs,
    int max_query_len, float softmax_scale, const float* k_scale, const float* v_scale,
    int max_splits, int num_ranges, float* partial_o, float* partial_lse, void* workspace,
    size_t workspace_bytes, void* out, float* lse_out, pkv_stream_t stream) {
  if (num_ranges < 0) return PKV_EINVAL;
  return decode_fused_impl(q, num_q_heads, num_tokens, cache, d, block_table,
                           max_blocks_per_seq, seq_lens, query_start_loc, num_seqs,
                           max_query_len, softmax_scale, k_scale, v_scale, max_splits,
                           partial_o, partial_lse, workspace, workspace_bytes, out, lse_out,
                           stream, /*clear=*/false, num_ranges);
}

int pkv_splitkv_reduce(const float* partial_o, const float* partial_lse,
                       int num_splits, int num_rows, int head_size_v, void* out,
                       float* lse_out, pkv_stream_t stream) {
  if (num_splits < 0 || num_rows < 0 || head_size_v < 1) return PKV_EINVAL;
  if (num_rows == 0) return PKV_OK;
  if (out == nullptr) return PKV_EINVAL;
  if (num_splits > 0 && (partial_o == nullptr || partial_lse == nullptr))
    return PKV_EINVAL;
  if ((head_size_v & 3) == 0 &&
      ((reinterpret_cast<uintptr_t>(partial_o) & 15u) != 0 ||
       (reinterpret_cast<uintptr_t>(out) & 7u) != 0))
    return PKV_EINVAL;
  cudaError_t e = pkv::launch_splitkv_reduce(
      partial_o, partial_lse, num_splits, num_rows, head_size_v,
      static_cast<__nv_bfloat16*>(out), lse_out,
      reinterpret_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? PKV_OK : fail_cuda(e);
}

int pkv_splitkv_reduce_sink(const float* partial_o, const float* partial_lse,
                            int num_splits, int num_rows, int head_size_v,
                            const float* sinks, int num_q_heads, void* out, float* lse_out,
                            pkv_stream_t stream) {
  if (num_splits < 0 || num_rows < 0 || head_size_v < 1 || num_q_heads < 1)
    return PKV_EINVAL;
  if (num_rows % num_q_heads != 0) return PKV_EINVAL;
  if (num_rows == 0) return PKV_OK;
  if (out == nullptr) return PKV_EINVAL;
  if (num_splits > 0 && (partial_o == nullptr || partial_lse == nullptr))
    return PKV_EINVAL;
  if ((head_size_v & 3) == 0 &&
      ((reinterpret_cast<uintptr_t>(partial_o) & 15u) != 0 ||
       (reinterpret_cast<uintptr_t>(out) & 7u) != 0))
    return PKV_EINVAL;
  cudaError_t e = pkv::launch_splitkv_reduce(
      partial_o, partial_lse, num_splits, num_rows, head_size_v,
      static_cast<__nv_bfloat16*>(out), lse_out, reinterpret_cast<cudaStream_t>(stream),
      sinks, num_q_heads);
  return e == cudaSuccess ? PKV_OK : fail_cuda(e);
}

int pkv_decode_suggest_splits(int num_seqs, int num_q_heads, int num_kv_heads,
                              int max_query_len, int max_seq_len,
                              int block_size) {
  if (num_seqs < 1 || num_q_heads < 1 || num_kv_heads < 1 ||
      max_query_len < 1 || max_seq_len < 0 || block_size < 1 ||
      num_q_heads % num_kv_heads != 0)
    return PKV_EINVAL;
  int sms = 0;
  int rc = device_info(nullptr, &sms);
  if (rc != PKV_OK) return rc;
  const int64_t G = num_q_heads / num_kv_heads;
  // work units per split: the decode kernel takes KV heads four at a time
  // when the head count allows
  const int64_t head_units = num_kv_heads % 4 == 0 ? num_kv_heads / 4 : num_kv_heads;
  const int64_t units = static_cast<int64_t>(num_seqs) * head_units *
                        ((max_query_len * G + 15) / 16);
  // Two units per SM for a single sequence (its units are all alike; some
  // decode shapes run two CTAs per SM).  For a batch at least two per SM, and
  // among up to twice that many splits the count that would leave the fewest
  // SMs idle at the end if the units were alike (ceil(n / sms) * sms / n),
  // taking more splits only for a gain of more than 2 %.
  int64_t s = (2 * static_cast<int64_t>(sms) + units - 1) / units;
  if (num_seqs > 1) {
    const int64_t lo = (2 * static_cast<int64_t>(sms) + units - 1) / units;
    s = lo;
    int64_t best_num = 1, best_den = 1;  // imbalance of `s` as a fraction
    for (int64_t c = lo; c <= 2 * lo; ++c) {
      const int64_t n = c * units;
      const int64_t num = (n + sms - 1) / sms * sms;  // imbalance = num / n
      if (c == lo || num * best_den * 100 < best_num * n * 98) {
        s = c;
        best_num = num;
        best_den = n;
      }
    }
  }
  // and at least 256 keys, and one page, per segment
  const int64_t by_keys = max_seq_len / 256;
  if (s > by_keys) s = by_keys;
  const int64_t pages = (static_cast<int64_t>(max_seq_len) + block_size - 1) / block_size;
  if (s > pages) s = pages;
  if (s < 1) s = 1;
  if (s > 1024) s = 1024;
  return static_cast<int>(s);
}

int pkv_supports(int head_size, int head_size_v, int dtype) {
  if (head_size < 1 || head_size_v < 1 || head_size_v > head_size) return 0;
  if (dtype != PKV_BF16 && dtype != PKV_FP8_E4M3) return 0;
  int bits = 1;  // the write takes any K / V sizes
  if (pkv::prefill_supported(head_size, head_size_v, dtype)) bits |= 2;
  if (pkv::decode_supported(head_size, head_size_v, dtype)) bits |= 4;
  return bits;
}

int pkv_get_device_error(int* code, pkv_stream_t stream) {
  if (code == nullptr) return PKV_EINVAL;
  int* err = nullptr;
  int rc = device_info(&err, nullptr);
  if (rc != PKV_OK) return rc;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  int host = 0;
  cudaError_t e = cudaMemcpyAsync(&host, err, sizeof(int), cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess) e = cudaMemsetAsync(err, 0, sizeof(int), s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return fail_cuda(e);
  *code = host;
  return PKV_OK;
}

int pkv_selftest_bounded_wait(int limit_us, pkv_stream_t stream) {
  if (limit_us < 1 || limit_us > 2000000) return PKV_EINVAL;
  int* err = nullptr;
  int rc = device_info(&err, nullptr);
  if (rc != PKV_OK) return rc;
  const cudaError_t e = pkv::launch_bounded_wait_selftest(
      err, static_cast<uint64_t>(limit_us) * 1000u, reinterpret_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? PKV_OK : fail_cuda(e);
}

int pkv_last_cuda_error(void) { return t_last_cuda_error; }

const char* pkv_status_string(int status) {
  switch (status) {
    case PKV_OK: return "ok";
    case PKV_EINVAL: return "invalid argument";
    case PKV_EUNSUPPORTED: return "unsupported shape, dtype or layout";
    case PKV_ECUDA: return "CUDA error (see pkv_last_cuda_error)";
    default: return "unknown status";
  }
}

}  // extern "C"
