// tmap.h -- host-side construction of TMA tensor maps over the block-paged
// cache (and over row-major Q), shared by the prefill and decode launchers.
#pragma once

#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>

#include "pkv.h"

namespace pkv {

inline PFN_cuTensorMapEncodeTiled_v12000 tmap_encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000,
                                         cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
  });
  return fn;
}

// A 4-D map over the cache whose boxes are `box_cols` row elements wide (at
// most one swizzle span: 128 bytes, or 64 with swizzle64; rows land densely
// with no_swizzle) and `box_rows` token slots high, for one KV head of one
// page.  Coordinates: NHD (col,
// head, slot, page), HND (col, slot, head, page).  Columns past row_elems
// read as zero.
inline bool make_cache_tmap(CUtensorMap* map, const void* cache, int dtype,
                            int layout, int num_blocks, int block_size,
                            int num_kv_heads, int row_elems, int box_cols,
                            int box_rows, bool swizzle64 = false,
                            bool no_swizzle = false) {
  PFN_cuTensorMapEncodeTiled_v12000 encode = tmap_encode_fn();
  if (encode == nullptr) return false;
  const cuuint64_t e = dtype == PKV_FP8_E4M3 ? 1 : 2;
  const cuuint64_t R = static_cast<cuuint64_t>(row_elems);
  const cuuint64_t H = static_cast<cuuint64_t>(num_kv_heads);
  const cuuint64_t B = static_cast<cuuint64_t>(block_size);
  cuuint64_t dims[4], strides[3];
  cuuint32_t box[4];
  if (layout == PKV_NHD) {  // [blk][bs][H][R]
    dims[0] = R; dims[1] = H; dims[2] = B; dims[3] = static_cast<cuuint64_t>(num_blocks);
    strides[0] = R * e; strides[1] = H * R * e; strides[2] = B * H * R * e;
    box[0] = box_cols; box[1] = 1; box[2] = box_rows; box[3] = 1;
  } else {                  // [blk][H][bs][R]
    dims[0] = R; dims[1] = B; dims[2] = H; dims[3] = static_cast<cuuint64_t>(num_blocks);
    strides[0] = R * e; strides[1] = B * R * e; strides[2] = H * B * R * e;
    box[0] = box_cols; box[1] = box_rows; box[2] = 1; box[3] = 1;
  }
  const cuuint32_t es[4] = {1, 1, 1, 1};
  return encode(map,
                dtype == PKV_FP8_E4M3 ? CU_TENSOR_MAP_DATA_TYPE_UINT8
                                      : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16,
                4, const_cast<void*>(cache), dims, strides, box, es,
                CU_TENSOR_MAP_INTERLEAVE_NONE,
                no_swizzle ? CU_TENSOR_MAP_SWIZZLE_NONE
                           : swizzle64 ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_128B,
                CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// A 4-D map over the cache whose boxes hold `box_heads` consecutive KV heads
// x `box_rows` token slots x `box_cols` row elements, landing in shared memory
// as [head][slot][box_cols] (each head's slots contiguous).  Coordinates are
// (col, slot, head, page) for both layouts, so for NHD the strides do not
// increase (slot stride H*R*e > head stride R*e); the encoder accepts that and
// a layout check on GB300 confirmed every element of such boxes.
inline bool make_cache_tmap_heads(CUtensorMap* map, const void* cache, int dtype,
                                  int layout, int num_blocks, int block_size,
                                  int num_kv_heads, int row_elems, int box_cols,
                                  int box_rows, int box_heads) {
  PFN_cuTensorMapEncodeTiled_v12000 encode = tmap_encode_fn();
  if (encode == nullptr) return false;
  const cuuint64_t e = dtype == PKV_FP8_E4M3 ? 1 : 2;
  const cuuint64_t R = static_cast<cuuint64_t>(row_elems);
  const cuuint64_t H = static_cast<cuuint64_t>(num_kv_heads);
  const cuuint64_t B = static_cast<cuuint64_t>(block_size);
  const cuuint64_t dims[4] = {R, B, H, static_cast<cuuint64_t>(num_blocks)};
  cuuint64_t strides[3];
  if (layout == PKV_NHD) {  // [blk][bs][H][R]
    strides[0] = H * R * e; strides[1] = R * e; strides[2] = B * H * R * e;
  } else {                  // [blk][H][bs][R]
    strides[0] = R * e; strides[1] = B * R * e; strides[2] = H * B * R * e;
  }
  const cuuint32_t box[4] = {static_cast<cuuint32_t>(box_cols),
                             static_cast<cuuint32_t>(box_rows),
                             static_cast<cuuint32_t>(box_heads), 1};
  const cuuint32_t es[4] = {1, 1, 1, 1};
  return encode(map,
                dtype == PKV_FP8_E4M3 ? CU_TENSOR_MAP_DATA_TYPE_UINT8
                                      : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16,
                4, const_cast<void*>(cache), dims, strides, box, es,
                CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// A 5-D map over a bf16 cache whose rows split into 64-column slabs
// (row_elems a multiple of 64), for page-grouped loads: coordinates (col
// 0..63 of a slab, key 0..7 of an 8-key group, slab, group within the page,
// page), with the KV head folded into the slab index (NHD: a head's row is
// the next R / 64 slabs) or into the page index (HND: page * H + head).  A
// box of (64, 8, nslab, box_rows / 8, 1) holds the nslab slabs of
// box_rows keys of one page and head and lands in shared memory as
// [8-key group][slab][8 keys][128 bytes], 128-byte swizzled.  The strides do
// not increase (a key's stride exceeds a slab's), which the encoder accepts
// (the decode's head-block maps have the same property).
inline bool make_cache_tmap_groups(CUtensorMap* map, const void* cache, int layout,
                                   int num_blocks, int block_size, int num_kv_heads,
                                   int row_elems, int nslab, int box_rows) {
  PFN_cuTensorMapEncodeTiled_v12000 encode = tmap_encode_fn();
  if (encode == nullptr) return false;
  if (row_elems % 64 != 0 || block_size % 8 != 0 || box_rows % 8 != 0) return false;
  const cuuint64_t R = static_cast<cuuint64_t>(row_elems);
  const cuuint64_t H = static_cast<cuuint64_t>(num_kv_heads);
  const cuuint64_t B = static_cast<cuuint64_t>(block_size);
  const cuuint64_t NB = static_cast<cuuint64_t>(num_blocks);
  cuuint64_t dims[5], strides[4];
  dims[0] = 64;
  dims[1] = 8;
  dims[3] = B / 8;
  strides[1] = 128;
  if (layout == PKV_NHD) {  // [blk][bs][H][R]
    dims[2] = H * R / 64;
    dims[4] = NB;
    strides[0] = H * R * 2;
    strides[2] = 8 * H * R * 2;
    strides[3] = B * H * R * 2;
  } else {                  // [blk][H][bs][R]
    dims[2] = R / 64;
    dims[4] = NB * H;
    strides[0] = R * 2;
    strides[2] = 8 * R * 2;
    strides[3] = B * R * 2;
  }
  const cuuint32_t box[5] = {64, 8, static_cast<cuuint32_t>(nslab),
                             static_cast<cuuint32_t>(box_rows / 8), 1};
  const cuuint32_t es[5] = {1, 1, 1, 1, 1};
  return encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 5, const_cast<void*>(cache), dims,
                strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Sets the dynamic shared-memory limit of `fn` once per device.
template <class F>
inline cudaError_t ensure_smem_attr(F* fn, int bytes, int* done) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev >= 0 && dev < 64 && !done[dev]) {
    e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e != cudaSuccess) return e;
    done[dev] = 1;
  }
  return cudaSuccess;
}

}  // namespace pkv
