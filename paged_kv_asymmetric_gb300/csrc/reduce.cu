// reduce.cu -- the split-KV merge (MiMo-V2.6-Flash 2x RTX PRO 6000 model
// card, "What the kernels do" and "Update 2026-10-01"): each row's segment
// partials (o_s, lse_s) are combined with weights exp(lse_s - max lse); a row
// whose segments are all empty is written as 0 with lse -inf instead of the
// exp(-inf - -inf) = NaN the unclamped merge produces.  An attention sink
// (the same card's "Update 2026-10-01": one extra logit in the softmax
// denominator, vLLM #58235) joins the merge once per row as one more segment
// with lse = sink and no value: it enters the maximum and the weight sum.
//
// One warp per row: the split weights are recomputed by every lane from the
// (broadcast) lse values, and each lane accumulates four consecutive output
// columns per pass with 16-byte loads.  The kernel reads S * dv * 4 bytes per
// row and writes dv * 2; it is small next to the decode it follows.
#include <math.h>

#include "common.cuh"
#include "kernels.h"

namespace pkv {

namespace {

__global__ void __launch_bounds__(256)
    splitkv_reduce_kernel(const float* __restrict__ po,
                          const float* __restrict__ plse, int S, int rows,
                          int dv, __nv_bfloat16* __restrict__ out,
                          float* __restrict__ lse_out, const float* __restrict__ sinks,
                          int hq) {
  const int lane = threadIdx.x & 31;
  const int wpb = blockDim.x >> 5;
  const bool vec = (dv & 3) == 0;
  for (int r = blockIdx.x * wpb + (threadIdx.x >> 5); r < rows;
       r += gridDim.x * wpb) {
    float M = -INFINITY;
    for (int s = lane; s < S; s += 32)
      M = fmaxf(M, __ldg(plse + static_cast<int64_t>(s) * rows + r));
#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
      M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
    const float sink = sinks != nullptr ? __ldg(sinks + r % hq) : -INFINITY;
    M = fmaxf(M, sink);
    __nv_bfloat16* orow = out + static_cast<int64_t>(r) * dv;
    if (M == -INFINITY) {  // no segment saw a key: 0, never NaN
      for (int c = lane; c < dv; c += 32) orow[c] = __float2bfloat16_rn(0.f);
      if (lse_out != nullptr && lane == 0) lse_out[r] = -INFINITY;
      continue;
    }
    const float Ml2 = M * kLog2e;
    // the sink's weight (0 without a sink)
    const float wsink = sink == -INFINITY ? 0.f : fast_exp2(fmaf(sink, kLog2e, -Ml2));
    float W = 0.f;
    if (vec) {
      for (int c0 = 0; c0 < dv; c0 += 128) {
        const int c = c0 + 4 * lane;
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
        float wsum = wsink;
        for (int s = 0; s < S; ++s) {
          const float x = __ldg(plse + static_cast<int64_t>(s) * rows + r);
          if (x == -INFINITY) continue;  // empty segment: o_s is not read
          const float w = fast_exp2(fmaf(x, kLog2e, -Ml2));
          wsum += w;
          if (c < dv) {
            const float4 v = __ldg(reinterpret_cast<const float4*>(
                po + (static_cast<int64_t>(s) * rows + r) * dv + c));
            acc.x = fmaf(w, v.x, acc.x);
            acc.y = fmaf(w, v.y, acc.y);
            acc.z = fmaf(w, v.z, acc.z);
            acc.w = fmaf(w, v.w, acc.w);
          }
        }
        W = wsum;
        if (c < dv) {
          const float inv = 1.f / wsum;
          uint2 st;
          st.x = pack_bf16x2(acc.x * inv, acc.y * inv);
          st.y = pack_bf16x2(acc.z * inv, acc.w * inv);
          *reinterpret_cast<uint2*>(orow + c) = st;
        }
      }
    } else {
      for (int c = lane; c < dv; c += 32) {
        float acc = 0.f, wsum = wsink;
        for (int s = 0; s < S; ++s) {
          const float x = __ldg(plse + static_cast<int64_t>(s) * rows + r);
          if (x == -INFINITY) continue;
          const float w = fast_exp2(fmaf(x, kLog2e, -Ml2));
          wsum += w;
          acc = fmaf(w, __ldg(po + (static_cast<int64_t>(s) * rows + r) * dv + c),
                     acc);
        }
        W = wsum;
        orow[c] = __float2bfloat16_rn(acc / wsum);
      }
    }
    if (lse_out != nullptr && lane == 0) {
      lse_out[r] = M + fast_log2(W) * kLn2;
    }
  }
}

// One CTA per (row, block of columns) for dv % 4 == 0: the split maxima and
// weight sums are block reductions (repeated by each column block of a row:
// S values), and the threads form `ngrp` groups over the splits x `cols`
// lanes over 16-byte column pieces, so that a row with hundreds of splits is
// read by hundreds of loads in flight instead of one warp's serial walk.
// Rows are split into column blocks when there are too few rows to fill the
// GPU (e.g. one token of an MLA decode with 150+ splits).
template <int THREADS>
__global__ void __launch_bounds__(THREADS)
    splitkv_reduce_rows_kernel(const float* __restrict__ po,
                               const float* __restrict__ plse, int S, int rows,
                               int dv, __nv_bfloat16* __restrict__ out,
                               float* __restrict__ lse_out,
                               const float* __restrict__ sinks, int hq) {
  __shared__ float red[THREADS / 32];
  __shared__ float4 part[THREADS];
  const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
  const int r = blockIdx.x;
  const int ncb = gridDim.y;  // column blocks per row
  auto block_reduce = [&](float v, bool is_max) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float u = __shfl_xor_sync(0xffffffffu, v, o);
      v = is_max ? fmaxf(v, u) : v + u;
    }
    __syncthreads();
    if (lane == 0) red[wid] = v;
    __syncthreads();
    v = red[0];
#pragma unroll
    for (int w = 1; w < THREADS / 32; ++w) v = is_max ? fmaxf(v, red[w]) : v + red[w];
    return v;
  };
  float M = -INFINITY;
  for (int s = tid; s < S; s += THREADS)
    M = fmaxf(M, __ldg(plse + static_cast<int64_t>(s) * rows + r));
  M = block_reduce(M, true);
  const float sink = sinks != nullptr ? __ldg(sinks + r % hq) : -INFINITY;
  M = fmaxf(M, sink);
  __nv_bfloat16* orow = out + static_cast<int64_t>(r) * dv;
  const int dv4 = dv >> 2;
  const int cb4 = dv4 / ncb;  // 16-byte pieces of this block
  const int c4_lo = blockIdx.y * cb4;
  if (M == -INFINITY) {  // no segment saw a key: 0, never NaN
    for (int c = tid; c < 4 * cb4; c += THREADS) orow[4 * c4_lo + c] = __float2bfloat16_rn(0.f);
    if (lse_out != nullptr && tid == 0 && blockIdx.y == 0) lse_out[r] = -INFINITY;
    return;
  }
  const float Ml2 = M * kLog2e;
  float wsum = 0.f;
  for (int s = tid; s < S; s += THREADS) {
    const float x = __ldg(plse + static_cast<int64_t>(s) * rows + r);
    if (x != -INFINITY) wsum += fast_exp2(fmaf(x, kLog2e, -Ml2));
  }
  const float W = block_reduce(wsum, false) +
                  (sink == -INFINITY ? 0.f : fast_exp2(fmaf(sink, kLog2e, -Ml2)));
  const float inv = 1.f / W;
  const int cols = cb4 < THREADS ? cb4 : THREADS;
  const int ngrp = THREADS / cols;
  const int c = tid % cols, grp = tid / cols;
  for (int c0 = 0; c0 < cb4; c0 += cols) {
    const int c4 = c4_lo + c0 + c;
    const bool in = c0 + c < cb4;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    if (grp < ngrp && in) {
      // four splits per step, their loads independent of each other
      constexpr int U = 4;
      for (int s0 = grp; s0 < S; s0 += U * ngrp) {
        float w[U];
        float4 v[U];
#pragma unroll
        for (int k = 0; k < U; ++k) {
          const int s = s0 + k * ngrp;
          const float x = s < S ? __ldg(plse + static_cast<int64_t>(s) * rows + r)
                                : -INFINITY;
          // an empty segment's o_s is not read
          w[k] = x == -INFINITY ? 0.f : fast_exp2(fmaf(x, kLog2e, -Ml2));
          v[k] = w[k] != 0.f
                     ? __ldg(reinterpret_cast<const float4*>(
                                 po + (static_cast<int64_t>(s) * rows + r) * dv) + c4)
                     : make_float4(0.f, 0.f, 0.f, 0.f);
        }
#pragma unroll
        for (int k = 0; k < U; ++k) {
          acc.x = fmaf(w[k], v[k].x, acc.x);
          acc.y = fmaf(w[k], v[k].y, acc.y);
          acc.z = fmaf(w[k], v[k].z, acc.z);
          acc.w = fmaf(w[k], v[k].w, acc.w);
        }
      }
    }
    __syncthreads();
    part[tid] = acc;
    __syncthreads();
    if (grp == 0 && in) {
      for (int g2 = 1; g2 < ngrp; ++g2) {
        const float4 v = part[g2 * cols + c];
        acc.x += v.x; acc.y += v.y; acc.z += v.z; acc.w += v.w;
      }
      uint2 st;
      st.x = pack_bf16x2(acc.x * inv, acc.y * inv);
      st.y = pack_bf16x2(acc.z * inv, acc.w * inv);
      *reinterpret_cast<uint2*>(orow + 4 * c4) = st;
    }
  }
  if (lse_out != nullptr && tid == 0 && blockIdx.y == 0) lse_out[r] = M + fast_log2(W) * kLn2;
}

}  // namespace

cudaError_t launch_splitkv_reduce(const float* partial_o,
                                  const float* partial_lse, int num_splits,
                                  int num_rows, int head_size_v,
                                  __nv_bfloat16* out, float* lse_out,
                                  cudaStream_t stream, const float* sinks,
                                  int num_q_heads) {
  if (num_rows == 0) return cudaSuccess;
  if ((head_size_v & 3) == 0) {
    // column blocks (a power of two dividing dv/4, >= 8 pieces each) until
    // there are about 2 x 152 CTAs
    const int dv4 = head_size_v >> 2;
    int ncb = 1;
    while (static_cast<int64_t>(num_rows) * ncb < 304 && dv4 % (2 * ncb) == 0 &&
           dv4 / (2 * ncb) >= 8)
      ncb *= 2;
    splitkv_reduce_rows_kernel<512><<<dim3(num_rows, ncb), 512, 0, stream>>>(
        partial_o, partial_lse, num_splits, num_rows, head_size_v, out, lse_out, sinks,
        num_q_heads);
    return cudaGetLastError();
  }
  const int wpb = 8;
  int blocks = (num_rows + wpb - 1) / wpb;
  if (blocks > 65535) blocks = 65535;
  splitkv_reduce_kernel<<<blocks, 32 * wpb, 0, stream>>>(
      partial_o, partial_lse, num_splits, num_rows, head_size_v, out, lse_out, sinks,
      num_q_heads);
  return cudaGetLastError();
}

}  // namespace pkv
