// write.cu -- the cache write (vLLM PR #64064, "Details": the asymmetric
// branch of reshape_and_cache_flash).  K and V of each token are scattered by
// slot_mapping into one packed row per KV head; V is read with its own token
// and head strides and written with its own length at its own offset.
//
// Layout of the work: one warp per token; a lane moves 16-byte pieces of the
// token's K and V rows (8 bf16 elements, or 16 for an fp8 cache so that
// every store is 16 bytes wide), all loads before all stores.  The kernel is
// bound by HBM bandwidth; its algorithmic traffic per token and KV head is
// the bf16 K and V read (2 * (dk + dv) bytes) plus the cache row written
// (e * (dk + dv)).
#include "common.cuh"
#include "kernels.h"

namespace pkv {

namespace {

__device__ __forceinline__ int64_t row_elem_offset(const WriteParams& p,
                                                   int64_t slot, int head) {
  int64_t blk = slot / p.block_size;
  int64_t off = slot - blk * p.block_size;
  if (p.layout == PKV_NHD)
    return ((blk * p.block_size + off) * p.num_kv_heads + head) *
           static_cast<int64_t>(p.row_elems);
  return ((blk * p.num_kv_heads + head) * p.block_size + off) *
         static_cast<int64_t>(p.row_elems);
}

__device__ __forceinline__ float scale_for(const float* s, int mode, int h) {
  return mode == PKV_SCALE_HEAD ? s[h] : s[0];
}

// E4M3 of x / s: IEEE binary32 division (round to nearest even), then the
// hardware conversion with round-to-nearest-even and saturation.
__device__ __forceinline__ uint16_t enc2(float a, float b, float s) {
  float2 v = make_float2(__fdiv_rn(a, s), __fdiv_rn(b, s));
  return static_cast<uint16_t>(
      __nv_cvt_float2_to_fp8x2(v, __NV_SATFINITE, __NV_E4M3));
}

// Vector path: one warp per token.  The token's slot and cache-row offsets
// are computed once; its K and V rows of all KV heads are pieces of EPT
// elements (16 bytes of bf16 source; EPT 8 for a bf16 cache, 16 for fp8 so
// that every store is 16 bytes wide), lane i taking pieces i, i + 32, ...;
// all of a lane's loads are issued before its stores, so a warp has the
// whole token (e.g. 4 heads x 640 bytes) in flight.
template <bool FP8, int EPT>
__global__ void __launch_bounds__(256)
    cache_write_vec_kernel(WriteParams p) {
  constexpr int PPL = 8;                      // pieces per lane per round
  constexpr int NV = EPT / 8;                 // 16-byte source loads per piece
  const int lane = threadIdx.x & 31;
  const int kp = p.head_size / EPT;          // pieces per K row
  const int vp = p.has_value ? p.head_size_v / EPT : 0;
  const int per_head = kp + vp;
  const int npieces = p.num_kv_heads * per_head;
  const int64_t nslots = static_cast<int64_t>(p.num_blocks) * p.block_size;
  const int64_t warps = static_cast<int64_t>(gridDim.x) * (blockDim.x >> 5);
  for (int64_t t = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
       t < p.num_tokens; t += warps) {
    const int64_t slot = __ldg(p.slot_mapping + t);
    if (slot < 0) continue;
    if (slot >= nslots) {
      if (lane == 0) set_dev_error(p.err, PKV_EDEV_RANGE);
      continue;
    }
    const int64_t blk = slot / p.block_size;
    const int off = static_cast<int>(slot - blk * p.block_size);
    for (int base = 0; base < npieces; base += 32 * PPL) {
      uint4 v[PPL][NV];
#pragma unroll
      for (int j = 0; j < PPL; ++j) {
        const int piece = base + lane + 32 * j;
        if (piece < npieces) {
          const int h = piece / per_head, q = piece - h * per_head;
          const bool is_k = q < kp;
          const int e0 = (is_k ? q : q - kp) * EPT;
          const __nv_bfloat16* src =
              is_k ? p.key + t * p.key_tok_stride + h * p.key_head_stride + e0
                   : p.value + t * p.val_tok_stride + h * p.val_head_stride + e0;
#pragma unroll
          for (int c = 0; c < NV; ++c) v[j][c] = __ldg(reinterpret_cast<const uint4*>(src) + c);
        }
      }
#pragma unroll
      for (int j = 0; j < PPL; ++j) {
        const int piece = base + lane + 32 * j;
        if (piece >= npieces) continue;
        const int h = piece / per_head, q = piece - h * per_head;
        const bool is_k = q < kp;
        const int e0 = (is_k ? q : q - kp) * EPT;
        const int64_t row = p.layout == PKV_NHD
                                ? (blk * p.block_size + off) * p.num_kv_heads + h
                                : (blk * p.num_kv_heads + h) * p.block_size + off;
        const int64_t dst = row * p.row_elems + (is_k ? p.k_off : p.v_off) + e0;
        if constexpr (!FP8) {
          *reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(p.cache) + dst) = v[j][0];
        } else {
          const float s = scale_for(is_k ? p.k_scale : p.v_scale, p.scale_mode, h);
          uint32_t w[EPT / 4];
#pragma unroll
          for (int c = 0; c < NV; ++c) {
            const uint32_t in[4] = {v[j][c].x, v[j][c].y, v[j][c].z, v[j][c].w};
#pragma unroll
            for (int k = 0; k < 2; ++k) {
              float2 f0 = __bfloat1622float2(
                  *reinterpret_cast<const __nv_bfloat162*>(&in[2 * k]));
              float2 f1 = __bfloat1622float2(
                  *reinterpret_cast<const __nv_bfloat162*>(&in[2 * k + 1]));
              w[2 * c + k] = static_cast<uint32_t>(enc2(f0.x, f0.y, s)) |
                             (static_cast<uint32_t>(enc2(f1.x, f1.y, s)) << 16);
            }
          }
          uint8_t* out = static_cast<uint8_t*>(p.cache) + dst;
          if constexpr (EPT == 16)
            *reinterpret_cast<uint4*>(out) = make_uint4(w[0], w[1], w[2], w[3]);
          else
            *reinterpret_cast<uint2*>(out) = make_uint2(w[0], w[1]);
        }
      }
    }
  }
}

// Element path for shapes or strides the vector path cannot take.
template <bool FP8>
__global__ void __launch_bounds__(256)
    cache_write_scalar_kernel(WriteParams p, int64_t total_items) {
  const int per_head = p.head_size + (p.has_value ? p.head_size_v : 0);
  const int64_t nslots = static_cast<int64_t>(p.num_blocks) * p.block_size;
  for (int64_t item = blockIdx.x * static_cast<int64_t>(blockDim.x) +
                      threadIdx.x;
       item < total_items; item += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    int64_t th = item / per_head;
    int e = static_cast<int>(item - th * per_head);
    int64_t t = th / p.num_kv_heads;
    int h = static_cast<int>(th - t * p.num_kv_heads);
    int64_t slot = __ldg(p.slot_mapping + t);
    if (slot < 0) continue;
    if (slot >= nslots) {
      set_dev_error(p.err, PKV_EDEV_RANGE);
      continue;
    }
    const bool is_k = e < p.head_size;
    const int i = is_k ? e : e - p.head_size;
    const __nv_bfloat16 x =
        is_k ? p.key[t * p.key_tok_stride + h * p.key_head_stride + i]
             : p.value[t * p.val_tok_stride + h * p.val_head_stride + i];
    const int64_t dst = row_elem_offset(p, slot, h) + (is_k ? p.k_off : p.v_off) + i;
    if constexpr (!FP8) {
      static_cast<__nv_bfloat16*>(p.cache)[dst] = x;
    } else {
      const float s = scale_for(is_k ? p.k_scale : p.v_scale, p.scale_mode, h);
      float y = __fdiv_rn(__bfloat162float(x), s);
      static_cast<uint8_t*>(p.cache)[dst] = static_cast<uint8_t>(
          __nv_cvt_float_to_fp8(y, __NV_SATFINITE, __NV_E4M3));
    }
  }
}

inline bool aligned(const void* p, int bytes) {
  return (reinterpret_cast<uintptr_t>(p) % bytes) == 0;
}

}  // namespace

cudaError_t launch_cache_write(const WriteParams& p, int num_sms,
                               cudaStream_t stream) {
  const bool fp8 = p.dtype == PKV_FP8_E4M3;
  const int esz = fp8 ? 1 : 2;
  // The vector path needs 16-byte aligned source pieces and destination
  // pieces of 16 (bf16) or 8/16 (fp8) bytes.
  auto vec_ok = [&](int ept) {
    bool ok = p.head_size % ept == 0 && aligned(p.key, 16) &&
              p.key_tok_stride % 8 == 0 && p.key_head_stride % 8 == 0 &&
              (p.k_off * esz) % (ept * esz) == 0 &&
              (p.row_elems * esz) % (ept * esz) == 0 &&
              aligned(p.cache, ept * esz);
    if (p.has_value)
      ok = ok && p.head_size_v % ept == 0 && aligned(p.value, 16) &&
           p.val_tok_stride % 8 == 0 && p.val_head_stride % 8 == 0 &&
           (p.v_off * esz) % (ept * esz) == 0;
    return ok;
  };
  const int64_t th = static_cast<int64_t>(p.num_tokens) * p.num_kv_heads;
  const int threads = 256;
  auto grid_for = [&](int64_t items) {
    int64_t blocks = (items + threads - 1) / threads;
    int64_t cap = static_cast<int64_t>(num_sms) * 16;  // grid-stride beyond
    return static_cast<unsigned>(blocks < cap ? (blocks > 0 ? blocks : 1) : cap);
  };
  // vector path: a warp per token, 8 warps per block, at most 16 blocks per
  // SM resident at a time (grid-stride beyond)
  const int64_t tok_blocks = (static_cast<int64_t>(p.num_tokens) + 7) / 8;
  const int64_t tok_cap = static_cast<int64_t>(num_sms) * 16;
  const unsigned vgrid = static_cast<unsigned>(
      tok_blocks < tok_cap ? (tok_blocks > 0 ? tok_blocks : 1) : tok_cap);
  if (!fp8 && vec_ok(8)) {
    cache_write_vec_kernel<false, 8><<<vgrid, threads, 0, stream>>>(p);
  } else if (fp8 && vec_ok(16)) {
    cache_write_vec_kernel<true, 16><<<vgrid, threads, 0, stream>>>(p);
  } else if (fp8 && vec_ok(8)) {
    cache_write_vec_kernel<true, 8><<<vgrid, threads, 0, stream>>>(p);
  } else {
    int64_t items = th * (p.head_size + (p.has_value ? p.head_size_v : 0));
    if (fp8)
      cache_write_scalar_kernel<true><<<grid_for(items), threads, 0, stream>>>(p, items);
    else
      cache_write_scalar_kernel<false><<<grid_for(items), threads, 0, stream>>>(p, items);
  }
  return cudaGetLastError();
}

}  // namespace pkv
