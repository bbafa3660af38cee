// reduce.cu -- the split-KV merge (MiMo-V2.6-Flash 2x RTX PRO 6000 model
// card, "What the kernels do" and "Update 2026-10-01"): each row's segment
// partials (o_s, lse_s) are combined with weights exp(lse_s - max lse); a row
// whose segments are all empty is written as 0 with lse -inf instead of the
// exp(-inf - -inf) = NaN the unclamped merge produces.  An attention sink
// (the same card's "Update 2026-10-01": one extra logit in the softmax
// denominator, vLLM #58235) joins the merge once per row as one more segment
// with lse = sink and no value: it enters the maximum and the weight sum.
//
// Three forms.  The merge reads S * dv * 4 bytes per row and writes dv * 2,
// a few MB next to the decode it follows, so its time is memory latency and
// the number of dependent round trips, not bandwidth:
//  * up to 32 splits (dv % 4 == 0): one warp per (row, 128 columns); lane s
//    loads lse_s, and only the segments whose lse is finite have their
//    16-byte partials loaded, all in flight together: two round trips, and
//    no read of a partial the decode left unwritten (with balanced ranges
//    most of a row's split slots are empty);
//  * more splits: a CTA per (row, column block), the splits spread over
//    its threads;
//  * dv % 4 != 0: one warp per row, one column per lane.
#include <math.h>

#include "common.cuh"
#include "kernels.h"
#include "pdl.cuh"

namespace pkv {

namespace {

// dv % 4 != 0 (any split count): one warp per row, one column per lane.
__global__ void __launch_bounds__(256)
    splitkv_reduce_kernel(const float* __restrict__ po,
                          const float* __restrict__ plse, int S, int rows,
                          int dv, __nv_bfloat16* __restrict__ out,
                          float* __restrict__ lse_out, const float* __restrict__ sinks,
                          int hq) {
  pdl_trigger();  // the next kernel of the step may start launching
  pdl_wait();     // every global access comes after the kernel ahead completes
  const int lane = threadIdx.x & 31;
  const int wpb = blockDim.x >> 5;
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
    for (int c = lane; c < dv; c += 32) {
      float acc = 0.f, wsum = wsink;
      for (int s = 0; s < S; ++s) {
        const float x = __ldg(plse + static_cast<int64_t>(s) * rows + r);
        if (x == -INFINITY) continue;  // empty segment: o_s is not read
        const float w = fast_exp2(fmaf(x, kLog2e, -Ml2));
        wsum += w;
        acc = fmaf(w, __ldg(po + (static_cast<int64_t>(s) * rows + r) * dv + c), acc);
      }
      W = wsum;
      orow[c] = __float2bfloat16_rn(acc / wsum);
    }
    if (lse_out != nullptr && lane == 0) {
      lse_out[r] = M + fast_log2(W) * kLn2;
    }
  }
}

// Up to SB splits, dv % 4 == 0: warp g of the grid merges columns
// [128 * cb, 128 * cb + 128) of row g / ncb (cb = g % ncb).  Lane s loads
// lse_s; a ballot names the segments that saw a key, and only their
// partials are loaded (an empty segment's partial was never written, and
// reading it would cost HBM traffic for nothing).  A segment whose weight
// underflows to 0 is skipped by a select.  The weights pass from lane s to
// the others through shared memory.
template <int SB>
__global__ void __launch_bounds__(128)
    splitkv_reduce_warp4_kernel(const float* __restrict__ po,
                                const float* __restrict__ plse, int S, int rows,
                                int dv, __nv_bfloat16* __restrict__ out,
                                float* __restrict__ lse_out,
                                const float* __restrict__ sinks, int hq) {
  static_assert(SB >= 1 && SB <= 32, "one split per lane");
  pdl_trigger();  // the next kernel of the step may start launching
  pdl_wait();     // every global access comes after the kernel ahead completes
  __shared__ float wsh[4][SB];
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  const int dv4 = dv >> 2;
  const int ncb = (dv4 + 31) >> 5;
  const int64_t g = static_cast<int64_t>(blockIdx.x) * 4 + wid;
  if (g >= static_cast<int64_t>(rows) * ncb) return;  // whole warps; no CTA barrier below
  const int r = static_cast<int>(g / ncb);
  const int c4 = static_cast<int>(g - static_cast<int64_t>(r) * ncb) * 32 + lane;
  const bool in = c4 < dv4;
  const float x = lane < S ? __ldg(plse + static_cast<int64_t>(lane) * rows + r) : -INFINITY;
  // the segments with a visible key (bit s = segment s; none past S)
  const uint32_t live = __ballot_sync(0xffffffffu, x != -INFINITY);
  const float4* po4 = reinterpret_cast<const float4*>(po);
  float4 v[SB];
#pragma unroll
  for (int s = 0; s < SB; ++s)
    v[s] = (((live >> s) & 1u) && in)
               ? __ldg(po4 + (static_cast<int64_t>(s) * rows + r) * dv4 + c4)
               : make_float4(0.f, 0.f, 0.f, 0.f);
  float M = x;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
  const float sink = sinks != nullptr ? __ldg(sinks + r % hq) : -INFINITY;
  M = fmaxf(M, sink);
  __nv_bfloat16* orow = out + static_cast<int64_t>(r) * dv;
  const bool first = c4 == lane;  // column block 0 writes the row's lse
  if (M == -INFINITY) {  // no segment saw a key: 0, never NaN
    if (in) *reinterpret_cast<uint2*>(orow + 4 * c4) = make_uint2(0u, 0u);
    if (lse_out != nullptr && first && lane == 0) lse_out[r] = -INFINITY;
    return;
  }
  const float Ml2 = M * kLog2e;
  const float w = x == -INFINITY ? 0.f : fast_exp2(fmaf(x, kLog2e, -Ml2));
  float W = w;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) W += __shfl_xor_sync(0xffffffffu, W, o);
  W += sink == -INFINITY ? 0.f : fast_exp2(fmaf(sink, kLog2e, -Ml2));
  if (lane < SB) wsh[wid][lane] = w;
  __syncwarp();
  if (in) {
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int s = 0; s < SB; ++s) {
      const float ws = wsh[wid][s];
      const bool use = ws != 0.f;
      acc.x = use ? fmaf(ws, v[s].x, acc.x) : acc.x;
      acc.y = use ? fmaf(ws, v[s].y, acc.y) : acc.y;
      acc.z = use ? fmaf(ws, v[s].z, acc.z) : acc.z;
      acc.w = use ? fmaf(ws, v[s].w, acc.w) : acc.w;
    }
    const float inv = 1.f / W;
    *reinterpret_cast<uint2*>(orow + 4 * c4) =
        make_uint2(pack_bf16x2(acc.x * inv, acc.y * inv), pack_bf16x2(acc.z * inv, acc.w * inv));
  }
  if (lse_out != nullptr && first && lane == 0) lse_out[r] = M + fast_log2(W) * kLn2;
}

// More than 32 splits, dv % 4 == 0: one CTA per (row, block of columns).
// The threads form `ngrp` groups over the splits x `cols` lanes over 16-byte
// column pieces.  Each thread loads its splits' lse values and partials
// together (eight splits per step, all in flight) and keeps them relative to
// its own running maximum, rescaling when a later step raises it, as an
// online softmax does.  The CTA then takes the row maximum (the sink
// included), rescales each group's sums to it, and adds the groups through
// shared memory, so a row costs one round trip to memory.  Rows are split
// into column blocks when there are too few rows to fill the GPU (e.g. one
// token of an MLA decode with 300 splits).
template <int THREADS>
__global__ void __launch_bounds__(THREADS)
    splitkv_reduce_rows_kernel(const float* __restrict__ po,
                               const float* __restrict__ plse, int S, int rows,
                               int dv, __nv_bfloat16* __restrict__ out,
                               float* __restrict__ lse_out,
                               const float* __restrict__ sinks, int hq) {
  __shared__ float red[THREADS / 32];
  pdl_trigger();  // the next kernel of the step may start launching
  pdl_wait();     // every global access comes after the kernel ahead completes
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
  const float sink = sinks != nullptr ? __ldg(sinks + r % hq) : -INFINITY;
  __nv_bfloat16* orow = out + static_cast<int64_t>(r) * dv;
  const int dv4 = dv >> 2;
  const int cb4 = dv4 / ncb;  // 16-byte pieces of this block
  const int c4_lo = blockIdx.y * cb4;
  const int cols = cb4 < THREADS ? cb4 : THREADS;
  const int ngrp = THREADS / cols;
  const int c = tid % cols, grp = tid / cols;
  const bool grp_ok = grp < ngrp;  // the last THREADS % cols threads idle
  const float4* po4 = reinterpret_cast<const float4*>(po);
  for (int c0 = 0; c0 < cb4; c0 += cols) {
    const int c4 = c4_lo + c0 + c;
    const bool in = grp_ok && c0 + c < cb4;
    // this thread's splits grp, grp + ngrp, ...: weight sum and weighted
    // partials relative to their running maximum m
    float m = -INFINITY, ws = 0.f;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    constexpr int U = 8;
    for (int s0 = grp; s0 < S; s0 += U * ngrp) {
      float x[U];
      float4 v[U];
#pragma unroll
      for (int k = 0; k < U; ++k) {
        const int s = s0 + k * ngrp;
        x[k] = (grp_ok && s < S) ? __ldg(plse + static_cast<int64_t>(s) * rows + r) : -INFINITY;
        v[k] = (in && s < S) ? __ldg(po4 + (static_cast<int64_t>(s) * rows + r) * dv4 + c4)
                             : make_float4(0.f, 0.f, 0.f, 0.f);
      }
      float mb = m;
#pragma unroll
      for (int k = 0; k < U; ++k) mb = fmaxf(mb, x[k]);
      if (mb == -INFINITY) continue;  // no visible segment so far
      const float mbl2 = mb * kLog2e;
      const float f = m == -INFINITY ? 0.f : fast_exp2(fmaf(m, kLog2e, -mbl2));
      ws *= f;
      acc.x *= f; acc.y *= f; acc.z *= f; acc.w *= f;
#pragma unroll
      for (int k = 0; k < U; ++k) {
        // an empty segment (lse -inf) has weight 0 and its partial is skipped
        const float w = x[k] == -INFINITY ? 0.f : fast_exp2(fmaf(x[k], kLog2e, -mbl2));
        const bool use = w != 0.f;
        ws += w;
        acc.x = use ? fmaf(w, v[k].x, acc.x) : acc.x;
        acc.y = use ? fmaf(w, v[k].y, acc.y) : acc.y;
        acc.z = use ? fmaf(w, v[k].z, acc.z) : acc.z;
        acc.w = use ? fmaf(w, v[k].w, acc.w) : acc.w;
      }
      m = mb;
    }
    // the row maximum over all groups and the sink (uniform over the CTA)
    const float M = fmaxf(block_reduce(m, true), sink);
    if (M == -INFINITY) {  // no segment saw a key: 0, never NaN
      if (grp == 0 && in) *reinterpret_cast<uint2*>(orow + 4 * c4) = make_uint2(0u, 0u);
      if (lse_out != nullptr && tid == 0 && blockIdx.y == 0 && c0 == 0) lse_out[r] = -INFINITY;
      continue;
    }
    const float Ml2 = M * kLog2e;
    const float f = m == -INFINITY ? 0.f : fast_exp2(fmaf(m, kLog2e, -Ml2));
    acc.x *= f; acc.y *= f; acc.z *= f; acc.w *= f;
    // every lane of a group holds the group's weight sum: count it once
    const float W = block_reduce(c == 0 && grp_ok ? ws * f : 0.f, false) +
                    (sink == -INFINITY ? 0.f : fast_exp2(fmaf(sink, kLog2e, -Ml2)));
    part[tid] = acc;  // block_reduce ended with a barrier after its last write
    __syncthreads();
    if (grp == 0 && in) {
      for (int g2 = 1; g2 < ngrp; ++g2) {
        const float4 v = part[g2 * cols + c];
        acc.x += v.x; acc.y += v.y; acc.z += v.z; acc.w += v.w;
      }
      const float inv = 1.f / W;
      *reinterpret_cast<uint2*>(orow + 4 * c4) =
          make_uint2(pack_bf16x2(acc.x * inv, acc.y * inv), pack_bf16x2(acc.z * inv, acc.w * inv));
    }
    if (lse_out != nullptr && tid == 0 && blockIdx.y == 0 && c0 == 0)
      lse_out[r] = M + fast_log2(W) * kLn2;
    __syncthreads();  // part[] is read before the next pass writes it
  }
}

}  // namespace

cudaError_t launch_splitkv_reduce(const float* partial_o,
                                  const float* partial_lse, int num_splits,
                                  int num_rows, int head_size_v,
                                  __nv_bfloat16* out, float* lse_out,
                                  cudaStream_t stream, const float* sinks,
                                  int num_q_heads) {
  if (num_rows == 0) return cudaSuccess;
  if ((head_size_v & 3) == 0 && num_splits <= 32) {
    const int64_t warps = static_cast<int64_t>(num_rows) * ((head_size_v / 4 + 31) / 32);
    const int64_t blocks = (warps + 3) / 4;
    if (blocks > 0x7fffffff) return cudaErrorInvalidValue;
    const unsigned grid = static_cast<unsigned>(blocks);
    auto kernel = num_splits <= 8    ? splitkv_reduce_warp4_kernel<8>
                  : num_splits <= 16 ? splitkv_reduce_warp4_kernel<16>
                                     : splitkv_reduce_warp4_kernel<32>;
    return launch_pdl(kernel, grid, 128, 0, stream, partial_o, partial_lse, num_splits,
                      num_rows, head_size_v, out, lse_out, sinks, num_q_heads);
  }
  if ((head_size_v & 3) == 0) {
    // column blocks (a power of two dividing dv/4, >= 8 pieces each) until
    // there are about 2 x 152 CTAs
    const int dv4 = head_size_v >> 2;
    int ncb = 1;
    while (static_cast<int64_t>(num_rows) * ncb < 304 && dv4 % (2 * ncb) == 0 &&
           dv4 / (2 * ncb) >= 8)
      ncb *= 2;
    return launch_pdl(splitkv_reduce_rows_kernel<512>, dim3(num_rows, ncb), 512, 0, stream,
                      partial_o, partial_lse, num_splits, num_rows, head_size_v, out, lse_out,
                      sinks, num_q_heads);
  }
  const int wpb = 8;
  int blocks = (num_rows + wpb - 1) / wpb;
  if (blocks > 65535) blocks = 65535;
  return launch_pdl(splitkv_reduce_kernel, blocks, 32 * wpb, 0, stream, partial_o, partial_lse,
                    num_splits, num_rows, head_size_v, out, lse_out, sinks, num_q_heads);
}

}  // namespace pkv
