// dequant.cu -- the FP8 prefill's first pass: the pages a batch of sequences
// uses, from the FP8 cache into a bf16 workspace, as their E4M3 codes widened
// exactly to bf16 (an E4M3 value has 4 significant bits and an exponent
// within bf16's range).  The scales are not applied here: the prefill folds
// k_scale into its softmax scale and v_scale into its output, so Q.K^T runs
// on exact values, as the MiMo-V2.6 model card ("What the kernels do")
// wants the FP8 path's Q.K^T kept in 16-bit.
//
// A page is bs x H x R contiguous bytes in both layouts, so each one widens
// as a flat run.  Bound by HBM: per page e * bs * H * R bytes read and twice
// that written (plus one block-table entry each way).
#include "common.cuh"
#include "kernels.h"

namespace pkv {

namespace {

// One CTA per (sequence, block-table entry), grid-strided.  Each thread
// widens 16 codes per step: one 16-byte load, two 16-byte stores.
__global__ void __launch_bounds__(256)
    fp8_pages_to_bf16_kernel(const uint8_t* __restrict__ cache, int64_t page_elems,
                             int num_blocks, const int32_t* __restrict__ block_table,
                             int max_blocks, const int32_t* __restrict__ seq_lens,
                             int num_seqs, int bs, __nv_bfloat16* __restrict__ pages,
                             int32_t* __restrict__ remap, int* err) {
  const int64_t entries = static_cast<int64_t>(num_seqs) * max_blocks;
  for (int64_t e = blockIdx.x; e < entries; e += gridDim.x) {
    const int b = static_cast<int>(e / max_blocks);
    const int j = static_cast<int>(e - static_cast<int64_t>(b) * max_blocks);
    const int L = __ldg(seq_lens + b);
    const int np = (L + bs - 1) / bs;
    if (j >= np) {
      if (threadIdx.x == 0) remap[e] = -1;
      continue;
    }
    const int page = __ldg(block_table + e);
    if (page < 0 || page >= num_blocks) {
      if (threadIdx.x == 0) {
        remap[e] = -1;  // the prefill reads it as zeros and records the error too
        set_dev_error(err, PKV_EDEV_RANGE);
      }
      continue;
    }
    if (threadIdx.x == 0) remap[e] = static_cast<int32_t>(e);
    const uint4* src = reinterpret_cast<const uint4*>(cache + static_cast<int64_t>(page) * page_elems);
    uint4* dst = reinterpret_cast<uint4*>(pages + e * page_elems);
    const int64_t n16 = page_elems / 16;
    for (int64_t i = threadIdx.x; i < n16; i += blockDim.x) {
      const uint4 w = __ldg(src + i);
      const uint32_t in[4] = {w.x, w.y, w.z, w.w};
      uint32_t o[8];
#pragma unroll
      for (int k = 0; k < 4; ++k) {
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          // two codes -> f16x2 (exact) -> two floats -> bf16x2 (exact)
          const uint32_t f16 = e4m3x2_to_f16x2(static_cast<uint16_t>(in[k] >> (16 * h)));
          const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&f16));
          o[2 * k + h] = pack_bf16x2(f.x, f.y);
        }
      }
      dst[2 * i] = make_uint4(o[0], o[1], o[2], o[3]);
      dst[2 * i + 1] = make_uint4(o[4], o[5], o[6], o[7]);
    }
  }
}

}  // namespace

cudaError_t launch_fp8_pages_to_bf16(const uint8_t* cache, int64_t page_elems, int num_blocks,
                                     const int32_t* block_table, int max_blocks_per_seq,
                                     const int32_t* seq_lens, int num_seqs, int block_size,
                                     __nv_bfloat16* pages, int32_t* remap, int* err,
                                     int num_sms, cudaStream_t stream) {
  const int64_t entries = static_cast<int64_t>(num_seqs) * max_blocks_per_seq;
  if (entries == 0) return cudaSuccess;
  const int64_t cap = static_cast<int64_t>(num_sms) * 8;
  const unsigned grid = static_cast<unsigned>(entries < cap ? entries : cap);
  fp8_pages_to_bf16_kernel<<<grid, 256, 0, stream>>>(cache, page_elems, num_blocks,
                                                     block_table, max_blocks_per_seq,
                                                     seq_lens, num_seqs, block_size, pages,
                                                     remap, err);
  return cudaGetLastError();
}

}  // namespace pkv
