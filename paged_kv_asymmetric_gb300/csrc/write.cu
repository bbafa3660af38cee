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
#include "pdl.cuh"

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

// x / s rounded to nearest even in binary32, from y = RN(1 / s): Markstein's
// correction (P. Markstein, "Computation of elementary functions on the IBM
// RISC System/6000 processor", IBM J. Res. Dev. 34(1), 1990; the "Handbook
// of Floating-Point Arithmetic", Muller et al., gives it as a theorem): with
// q0 = RN(x y) within an ulp of x / s and the exact remainder r = x - q0 s
// (one FMA), RN(q0 + r y) is the correctly rounded quotient, barring
// overflow and underflow on the way.  The remainder is formed with the
// opposite sign, r' = q0 s - x, and the quotient as q0 - r' y: the same
// value, but a zero quotient keeps its sign (x = -0 gives -0 + -0, where
// q0 + r y would give +0; a q0 that underflowed to zero gives x y rounded
// with its own sign).  A non-finite q0 (x infinite or NaN) is passed through,
// as the division gives it.  A quotient in the binary32 subnormal range may
// differ from the division in its last bits, which no E4M3 code can see
// (they all encode as a signed zero).  Callers take this path only for
// scales within [2^-64, 2^64] whose reciprocal is finite and nonzero.
__device__ __forceinline__ float div_rn_by(float x, float s, float y) {
  const float q0 = x * y;
  const float rn = fmaf(q0, s, -x);
  const float q = fmaf(-rn, y, q0);
  return isfinite(q0) ? q : q0;
}

// E4M3 of x / s with the quotient from div_rn_by (y = RN(1 / s)).
__device__ __forceinline__ uint16_t enc2_by(float a, float b, float s, float y) {
  float2 v = make_float2(div_rn_by(a, s, y), div_rn_by(b, s, y));
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
  pdl_trigger();  // the next kernel of the step may start launching
  pdl_wait();     // every global access comes after the kernel ahead completes
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

// Token path: one warp per token, the token's pieces dealt to lanes as in
// the vector path, but with each lane's piece geometry (source and
// destination offsets, K or V, scale) computed once for all tokens, which
// takes at most 32 * PPL pieces per token.  A token's loads do not wait for
// its slot: they are issued first, and the slot decides the stores.  A warp
// that has more than one token (grid-stride) loads its next token's pieces
// and slot before it encodes and stores the current one, so the FP8 encode
// of one token overlaps the loads of the next.
// Loads of the next token are kept in registers beside the current ones
// (WR_PREFETCH) when a lane's pieces are at most 8 16-byte loads; the block
// count per SM is then the one whose register share holds both sets.
template <bool FP8, int EPT, int PPL>
constexpr bool WR_PREFETCH = PPL * (EPT / 8) <= 8;
template <bool FP8, int EPT, int PPL>
constexpr int WR_BLOCKS =
    WR_PREFETCH<FP8, EPT, PPL>
        ? (PPL * (EPT / 8) <= (FP8 ? 4 : 5) ? 3 : 2)
        : ((FP8 && PPL <= 3) ? 4 : (PPL <= (FP8 ? 4 : 8)) ? 3 : 1);

template <bool FP8, int EPT, int PPL>
__global__ void __launch_bounds__(256, (WR_BLOCKS<FP8, EPT, PPL>))
    cache_write_tok_kernel(WriteParams p) {
  pdl_trigger();  // the next kernel of the step may start launching
  pdl_wait();     // every global access comes after the kernel ahead completes
  constexpr int NV = EPT / 8;  // 16-byte source loads per piece
  const int lane = threadIdx.x & 31;
  const int kp = p.head_size / EPT;
  const int vp = p.has_value ? p.head_size_v / EPT : 0;
  const int per_head = kp + vp;
  const int npieces = p.num_kv_heads * per_head;
  const int64_t nslots = static_cast<int64_t>(p.num_blocks) * p.block_size;
  const int64_t R = p.row_elems;
  // offsets within one token's K / V rows and within one slot's rows (the
  // launcher checks that they fit in 32 bits)
  int32_t soff[PPL], doff[PPL];
  bool is_k[PPL], act[PPL];
  float sc[PPL], rc[PPL];  // fp8: the scale and its reciprocal RN(1 / s) (0: divide)
#pragma unroll
  for (int j = 0; j < PPL; ++j) {
    const int piece = lane + 32 * j;
    act[j] = piece < npieces;
    const int h = act[j] ? piece / per_head : 0;
    const int q = piece - h * per_head;
    is_k[j] = q < kp;
    const int e0 = (is_k[j] ? q : q - kp) * EPT;
    soff[j] = static_cast<int32_t>((is_k[j] ? h * p.key_head_stride : h * p.val_head_stride) + e0);
    doff[j] = static_cast<int32_t>((p.layout == PKV_NHD ? h * R : h * p.block_size * R) +
                                   (is_k[j] ? p.k_off : p.v_off) + e0);
    sc[j] = 1.f;
    rc[j] = 0.f;
    if constexpr (FP8) {
      sc[j] = scale_for(is_k[j] ? p.k_scale : p.v_scale, p.scale_mode, h);
      const float y = __frcp_rn(sc[j]);
      // the FMA-corrected product where the scale and its reciprocal are
      // finite and nonzero and the remainder cannot underflow; else divide
      rc[j] = (isfinite(sc[j]) && isfinite(y) && y != 0.f && fabsf(sc[j]) >= 0x1p-64f &&
               fabsf(sc[j]) <= 0x1p64f)
                  ? y
                  : 0.f;
    }
  }
  const int64_t warps = static_cast<int64_t>(gridDim.x) * (blockDim.x >> 5);
  // token t's slot and pieces, loaded into (slot, v)
  auto load = [&](int64_t t, int64_t& slot, uint4 (&v)[PPL][NV]) {
    slot = __ldg(p.slot_mapping + t);
    const __nv_bfloat16* kt = p.key + t * p.key_tok_stride;
    const __nv_bfloat16* vt = p.has_value ? p.value + t * p.val_tok_stride : kt;
#pragma unroll
    for (int j = 0; j < PPL; ++j)
      if (act[j]) {
        const uint4* src = reinterpret_cast<const uint4*>((is_k[j] ? kt : vt) + soff[j]);
#pragma unroll
        for (int c = 0; c < NV; ++c) v[j][c] = __ldg(src + c);
      }
  };
  constexpr bool kPrefetch = WR_PREFETCH<FP8, EPT, PPL>;
  int64_t t = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  int64_t next_slot = -1;
  uint4 nv[kPrefetch ? PPL : 1][NV];
  if (kPrefetch && t < p.num_tokens) load(t, next_slot, *reinterpret_cast<uint4(*)[PPL][NV]>(nv));
  for (; t < p.num_tokens; t += warps) {
    int64_t slot;
    uint4 v[PPL][NV];
    if constexpr (kPrefetch) {
      slot = next_slot;
#pragma unroll
      for (int j = 0; j < PPL; ++j)
#pragma unroll
        for (int c = 0; c < NV; ++c) v[j][c] = nv[j][c];
      if (t + warps < p.num_tokens)
        load(t + warps, next_slot, *reinterpret_cast<uint4(*)[PPL][NV]>(nv));
    } else {
      load(t, slot, v);
    }
    if (slot < 0) continue;
    if (slot >= nslots) {
      if (lane == 0) set_dev_error(p.err, PKV_EDEV_RANGE);
      continue;
    }
    const int64_t blk = slot / p.block_size;
    const int64_t off = slot - blk * p.block_size;
    const int64_t base = p.layout == PKV_NHD
                             ? slot * p.num_kv_heads * R
                             : (blk * p.num_kv_heads * p.block_size + off) * R;
#pragma unroll
    for (int j = 0; j < PPL; ++j) {
      if (!act[j]) continue;
      const int64_t dst = base + doff[j];
      if constexpr (!FP8) {
        *reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(p.cache) + dst) = v[j][0];
      } else {
        uint32_t w[EPT / 4];
#pragma unroll
        for (int c = 0; c < NV; ++c) {
          const uint32_t in[4] = {v[j][c].x, v[j][c].y, v[j][c].z, v[j][c].w};
#pragma unroll
          for (int k = 0; k < 2; ++k) {
            float2 f0 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&in[2 * k]));
            float2 f1 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&in[2 * k + 1]));
            if (rc[j] != 0.f)
              w[2 * c + k] = static_cast<uint32_t>(enc2_by(f0.x, f0.y, sc[j], rc[j])) |
                             (static_cast<uint32_t>(enc2_by(f1.x, f1.y, sc[j], rc[j])) << 16);
            else
              w[2 * c + k] = static_cast<uint32_t>(enc2(f0.x, f0.y, sc[j])) |
                             (static_cast<uint32_t>(enc2(f1.x, f1.y, sc[j])) << 16);
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

// Element path for shapes or strides the vector path cannot take.
template <bool FP8>
__global__ void __launch_bounds__(256)
    cache_write_scalar_kernel(WriteParams p, int64_t total_items) {
  pdl_trigger();  // the next kernel of the step may start launching
  pdl_wait();     // every global access comes after the kernel ahead completes
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

// The token path's launch: one warp per token (8 per block) when a warp
// keeps one token in registers; with the next token's loads kept as well,
// the resident blocks only (WR_BLOCKS per SM), each warp striding over
// tokens so that its loads run one token ahead.
template <bool FP8, int EPT, int PPL>
cudaError_t launch_tok(const WriteParams& p, int num_sms, cudaStream_t stream) {
  const int64_t blocks = (static_cast<int64_t>(p.num_tokens) + 7) / 8;
  int64_t cap = int64_t{1} << 30;
  if (WR_PREFETCH<FP8, EPT, PPL>) cap = static_cast<int64_t>(num_sms) * WR_BLOCKS<FP8, EPT, PPL>;
  const unsigned grid =
      static_cast<unsigned>(blocks < cap ? (blocks > 0 ? blocks : 1) : cap);
  return launch_pdl(cache_write_tok_kernel<FP8, EPT, PPL>, grid, 256, 0, stream, p);
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
  // token path: one warp per token, every token its own warp (the block
  // scheduler balances), when a token's pieces fit 32 x PPL lanes
  const int ept = fp8 ? (vec_ok(16) ? 16 : 8) : 8;
  const int pieces = p.num_kv_heads * (p.head_size / ept +
                                       (p.has_value ? p.head_size_v / ept : 0));
  // the token path keeps per-lane offsets in 32 bits: a token's K / V rows
  // and a slot's rows of all heads must span less than 2^31 elements
  const int64_t src_span = static_cast<int64_t>(p.num_kv_heads) *
      (p.key_head_stride > p.val_head_stride ? p.key_head_stride : p.val_head_stride) +
      p.head_size + p.head_size_v;
  const int64_t dst_span = static_cast<int64_t>(p.num_kv_heads) * p.block_size * p.row_elems;
  const bool tok = (fp8 ? vec_ok(ept) : vec_ok(8)) && pieces <= 512 &&
                   src_span < (int64_t{1} << 31) && dst_span < (int64_t{1} << 31);
  cudaError_t e = cudaSuccess;
  if (tok) {
    if (!fp8) {
      if (pieces <= 128) e = launch_tok<false, 8, 4>(p, num_sms, stream);
      else if (pieces <= 160) e = launch_tok<false, 8, 5>(p, num_sms, stream);
      else if (pieces <= 256) e = launch_tok<false, 8, 8>(p, num_sms, stream);
      else e = launch_tok<false, 8, 16>(p, num_sms, stream);
    } else if (ept == 16) {
      if (pieces <= 96) e = launch_tok<true, 16, 3>(p, num_sms, stream);
      else if (pieces <= 128) e = launch_tok<true, 16, 4>(p, num_sms, stream);
      else if (pieces <= 256) e = launch_tok<true, 16, 8>(p, num_sms, stream);
      else e = launch_tok<true, 16, 16>(p, num_sms, stream);
    } else {
      if (pieces <= 128) e = launch_tok<true, 8, 4>(p, num_sms, stream);
      else if (pieces <= 256) e = launch_tok<true, 8, 8>(p, num_sms, stream);
      else e = launch_tok<true, 8, 16>(p, num_sms, stream);
    }
  } else if (!fp8 && vec_ok(8)) {
    e = launch_pdl(cache_write_vec_kernel<false, 8>, vgrid, threads, 0, stream, p);
  } else if (fp8 && vec_ok(16)) {
    e = launch_pdl(cache_write_vec_kernel<true, 16>, vgrid, threads, 0, stream, p);
  } else if (fp8 && vec_ok(8)) {
    e = launch_pdl(cache_write_vec_kernel<true, 8>, vgrid, threads, 0, stream, p);
  } else {
    int64_t items = th * (p.head_size + (p.has_value ? p.head_size_v : 0));
    if (fp8)
      e = launch_pdl(cache_write_scalar_kernel<true>, grid_for(items), threads, 0, stream, p, items);
    else
      e = launch_pdl(cache_write_scalar_kernel<false>, grid_for(items), threads, 0, stream, p, items);
  }
  return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace pkv
