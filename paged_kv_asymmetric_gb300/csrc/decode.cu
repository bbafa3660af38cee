// decode.cu -- split-KV decode and speculative verify over the paged cache.
//
// What it computes (MiMo-V2.6-Flash 2x RTX PRO 6000 model card, "What the
// kernels do": split-KV also for the multi-token verify step, one program for
// the whole verify; vLLM PR #50371: 12-head MLA decode, D 576 / 512, split
// selection from device-side sequence lengths with a graph-stable launch):
// for every query row of a sequence and every page-aligned segment of its
// keys, the segment-normalised softmax(scale * q K^T) V and its log-sum-exp.
// pkv_splitkv_reduce merges the segments.
//
// GB300 design.  The path is bound by HBM bandwidth: every key's packed
// K|V row is read once per (sequence, KV head) and used by all q_len * G
// query rows of that KV head (G = Hq / Hkv).  One CTA handles (split, KV head,
// 16-row group, sequence); the rows are (query token, query head) pairs, so
// a 1+3-token verify with G = 4 fills exactly one m16 tile.  Those 16 rows
// are too few for tcgen05 (M >= 64), and the FP8 path needs its operands in
// registers for the E4M3 -> f16 conversion, so the contraction runs on the
// warp-level m16n8k16 MMA; at ~32 flop per byte (verify) it stays far below
// that unit's rate at full HBM bandwidth.
//
//  * Groups of WG warps stream disjoint 16-key chunks of the segment through
//    their own NSTAGE-deep cp.async ring in shared memory (zero-filled past
//    the last key, so garbage in a partly filled page never reaches the MMA).
//    Within a group, warp w owns a slice of the K dimension for Q.K^T
//    (partial scores summed through shared memory when WG > 1) and a slice of
//    V's columns for P.V.
//  * Rows of 16-byte chunks are XOR-swizzled so that the fragment loads below
//    are free of bank conflicts.
//  * bf16 cache: K fragments come straight from 16-byte shared loads (the
//    reduction index is permuted identically in Q and K, which leaves the dot
//    products unchanged), V fragments from ldmatrix.trans.
//  * fp8 cache: E4M3 codes are converted to f16 in registers (exact), K from
//    16-byte loads, V by byte-permuting four keys' 16-byte column runs into
//    k-pairs; the MMA runs in f16 with Q converted bf16 -> f16; k_scale is
//    folded into the softmax scale and v_scale into the output.
//  * Online softmax in registers with exp2; groups merge their (max, sum, O)
//    through shared memory at the end and write one partial per row.
#include <math.h>

#include "common.cuh"
#include "kernels.h"

namespace pkv {

namespace {

template <int DK_, int DV_, bool FP8_, int WG_, int NG_, int NSTAGE_, int SPAN_>
struct DecodeCfg {
  static constexpr int DK = DK_, DV = DV_, WG = WG_, NG = NG_;
  static constexpr int NSTAGE = NSTAGE_, SPAN = SPAN_;
  static constexpr bool FP8 = FP8_;
  static constexpr int ESZ = FP8 ? 1 : 2;
  static constexpr int PITCH = ((SPAN * ESZ + 127) / 128) * 128;  // bytes/row
  static constexpr int UNIT = FP8 ? 64 : 32;  // K elements per 16-byte load
  static constexpr int NU = DK / UNIT;
  static constexpr int UPW = (NU + WG - 1) / WG;  // K units per warp (max)
  static constexpr int QW = FP8 ? 8 : 4;  // Q words per unit per row
  static constexpr int DVS = DV / WG;     // V columns per warp
  static constexpr int NT = DVS / 8;      // n8 tiles per warp
  static constexpr int THREADS = 32 * WG * NG;
  static constexpr int STAGE_BYTES = 16 * PITCH;
  static constexpr int STAGING = NG * NSTAGE * STAGE_BYTES;
  static constexpr int DVP = DV + 4;      // padded merge row (floats)
  static constexpr int MERGE = NG * 16 * DVP * 4 + 2 * NG * 16 * 4;
  static constexpr int MAIN = STAGING > MERGE ? STAGING : MERGE;
  static constexpr int SBUF = WG > 1 ? NG * 2 * WG * 32 * 8 * 4 : 0;
  static constexpr int SMEM = MAIN + SBUF;
  static_assert(DK % UNIT == 0, "K head size must be a multiple of the unit");
  static_assert(DV % WG == 0 && DVS % (FP8 ? 128 : 16) == 0,
                "V slice per warp must be a multiple of 128 (fp8) / 16");
  static_assert(SMEM <= 227 * 1024, "shared memory budget");
};

// XOR pattern applied to the 16-byte chunk index of a staged row.  bf16: a
// 3-bit bit reversal (distinct over any 8 consecutive rows, and rows 2m,
// 2m+1 land in opposite halves of a 128-byte line).  fp8: rows 2m and 2m+1
// differ in bit 2 and rows {0,2,4,6} / {1,3,5,7} differ in bits 1-2.
template <bool FP8>
__device__ __forceinline__ int swz(int row) {
  if constexpr (FP8)
    return (((row >> 1) & 3) << 1) ^ ((row & 1) << 2);
  else
    return ((row & 1) << 2) | (row & 2) | ((row >> 2) & 1);
}

template <bool FP8>
__device__ __forceinline__ uint32_t chunk_addr(uint32_t stage, int pitch,
                                               int row, int chunk) {
  return stage + row * pitch + ((chunk ^ swz<FP8>(row)) << 4);
}

template <class C>
__global__ void __launch_bounds__(C::THREADS)
    decode_kernel(const AttnParams p) {
  extern __shared__ __align__(128) uint8_t smem[];
  constexpr bool FP8 = C::FP8;
  constexpr int WG = C::WG, NG = C::NG, NSTAGE = C::NSTAGE;

  const int split = blockIdx.x;
  const int b = blockIdx.z;
  const int g = blockIdx.y % p.num_kv_heads;
  const int rgrp = blockIdx.y / p.num_kv_heads;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int grp = warp / WG, wig = warp % WG;
  const int gr = lane >> 2, qd = lane & 3;
  const int G = p.group;

  const int qs = __ldg(p.query_start_loc + b);
  const int qlen = __ldg(p.query_start_loc + b + 1) - qs;
  const int L = __ldg(p.seq_lens + b);
  const int row0 = rgrp * 16;
  if (row0 >= qlen * G) return;
  const int nrows = min(16, qlen * G - row0);

  const int bs = p.block_size;
  const int P = (L + bs - 1) / bs;
  const int pps = (P + p.num_splits - 1) / p.num_splits;
  const int page_lo = min(split * pps, P);
  const int page_hi = min(page_lo + pps, P);
  const int klo = page_lo * bs;
  const int khi = min(page_hi * bs, L);
  // the CTA's last row belongs to its latest query token: it sees the most
  const int i_last = (row0 + nrows - 1) / G;
  const int kmax = min(khi, max(0, min(L, L - qlen + i_last + 1)));

  const int64_t T = p.num_tokens;
  if (kmax <= klo) {  // no key of this segment is visible to any row
    for (int r = threadIdx.x; r < nrows; r += blockDim.x) {
      const int rr = row0 + r;
      const int64_t t = qs + rr / G;
      const int h = g * G + rr % G;
      p.partial_lse[(split * T + t) * p.num_q_heads + h] = -INFINITY;
    }
    return;
  }

  // ---- per-row visibility (rows gr and gr + 8 of the 16-row tile) ----
  int vis_end[2];
#pragma unroll
  for (int k = 0; k < 2; ++k) {
    const int r = gr + 8 * k;
    if (r < nrows) {
      const int i = (row0 + r) / G;
      vis_end[k] = min(khi, max(0, min(L, L - qlen + i + 1)));
    } else {
      vis_end[k] = 0;
    }
  }

  // ---- Q fragments for this warp's K units ----
  uint32_t qa[C::UPW][2][C::QW];
#pragma unroll
  for (int uu = 0; uu < C::UPW; ++uu) {
    const int u = wig + uu * WG;
#pragma unroll
    for (int k = 0; k < 2; ++k) {
      const int r = gr + 8 * k;
      if (u < C::NU && r < nrows) {
        const int rr = row0 + r;
        const int64_t t = qs + rr / G;
        const int h = g * G + rr % G;
        const uint4* src = reinterpret_cast<const uint4*>(
            p.q + (t * p.num_q_heads + h) * C::DK + u * C::UNIT +
            qd * (C::UNIT / 4));
        if constexpr (!FP8) {
          const uint4 v = __ldg(src);
          qa[uu][k][0] = v.x; qa[uu][k][1] = v.y;
          qa[uu][k][2] = v.z; qa[uu][k][3] = v.w;
        } else {
          const uint4 v0 = __ldg(src), v1 = __ldg(src + 1);
          const uint32_t w[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
#pragma unroll
          for (int j = 0; j < 8; ++j) qa[uu][k][j] = bf16x2_to_f16x2(w[j]);
        }
      } else {
#pragma unroll
        for (int j = 0; j < C::QW; ++j) qa[uu][k][j] = 0u;
      }
    }
  }

  // ---- cache geometry ----
  const int lo = min(p.k_off, p.v_off);
  const int kc0 = (p.k_off - lo) * C::ESZ / 16;   // first K chunk in the span
  const int vc0 = (p.v_off - lo) * C::ESZ / 16;
  const int nch = (max(p.k_off + C::DK, p.v_off + C::DV) - lo) * C::ESZ / 16;
  const int64_t row_bytes = static_cast<int64_t>(p.row_elems) * C::ESZ;
  int64_t page_stride, tok_stride, head_stride;
  if (p.layout == PKV_NHD) {
    tok_stride = p.num_kv_heads * row_bytes;
    head_stride = row_bytes;
  } else {
    tok_stride = row_bytes;
    head_stride = static_cast<int64_t>(bs) * row_bytes;
  }
  page_stride = static_cast<int64_t>(bs) * p.num_kv_heads * row_bytes;
  const uint8_t* cache = static_cast<const uint8_t*>(p.cache);
  const int32_t* bt = p.block_table + static_cast<int64_t>(b) * p.max_blocks_per_seq;

  float qk_scale = p.softmax_scale * kLog2e;
  float v_mul = 1.f;
  if constexpr (FP8) {
    const int sidx = p.scale_mode == PKV_SCALE_HEAD ? g : 0;
    qk_scale *= __ldg(p.k_scale + sidx);
    v_mul = __ldg(p.v_scale + sidx);
  }

  const uint32_t stage0 = smem_u32(smem) + grp * NSTAGE * C::STAGE_BYTES;

  const int nchunks = (kmax - klo + 15) / 16;
  const int n_my = nchunks > grp ? (nchunks - grp + NG - 1) / NG : 0;

  // Issues the cp.async copies of the group's it-th chunk (16 keys).
  auto load_chunk = [&](int it) {
    if (it < n_my) {
      const int kb = klo + (grp + it * NG) * 16;
      const uint32_t dst_stage = stage0 + (it % NSTAGE) * C::STAGE_BYTES;
      // lanes 0..15 resolve one row's byte offset each; shared by shuffle
      int64_t my_off = -1;
      if (lane < 16) {
        const int key = kb + lane;
        if (key < kmax) {
          const int pg = __ldg(bt + key / bs);
          if (pg >= 0 && pg < p.num_blocks) {
            my_off = pg * page_stride + (key % bs) * tok_stride +
                     g * head_stride + static_cast<int64_t>(lo) * C::ESZ;
          } else {
            set_dev_error(p.err, PKV_EDEV_RANGE);
          }
        }
      }
      // the trip count is uniform across the warp (the shuffle needs all
      // lanes); lanes past the end only take part in the shuffle
      for (int base = wig * 32; base < 16 * nch; base += 32 * WG) {
        const int idx = base + lane;
        const int row = min(idx / nch, 15);
        const int ch = idx - row * nch;
        const int64_t off = __shfl_sync(0xffffffffu, my_off, row);
        if (idx < 16 * nch) {
          const uint8_t* src = off >= 0 ? cache + off + ch * 16 : cache;
          cp_async_16(chunk_addr<FP8>(dst_stage, C::PITCH, row, ch), src,
                      off >= 0 ? 16 : 0);
        }
      }
    }
    cp_async_commit();
  };

  auto group_sync = [&]() {
    if constexpr (WG == 1)
      __syncwarp();
    else
      named_barrier(1 + grp, 32 * WG);
  };

  float o[C::NT][4];
#pragma unroll
  for (int nt = 0; nt < C::NT; ++nt)
    o[nt][0] = o[nt][1] = o[nt][2] = o[nt][3] = 0.f;
  float m_run[2] = {-INFINITY, -INFINITY};
  float l_run[2] = {0.f, 0.f};
  float* sbuf = reinterpret_cast<float*>(smem + C::MAIN) +
                grp * 2 * WG * 32 * 8;

#pragma unroll
  for (int s = 0; s < NSTAGE - 1; ++s) load_chunk(s);

  for (int it = 0; it < n_my; ++it) {
    cp_async_wait<NSTAGE - 2>();
    group_sync();
    load_chunk(it + NSTAGE - 1);
    const uint32_t st = stage0 + (it % NSTAGE) * C::STAGE_BYTES;
    const int kb = klo + (grp + it * NG) * 16;

    // ---- S = Q K^T over this warp's K units (two n8 tiles of keys) ----
    float s[2][4];
#pragma unroll
    for (int t = 0; t < 2; ++t) s[t][0] = s[t][1] = s[t][2] = s[t][3] = 0.f;
#pragma unroll
    for (int uu = 0; uu < C::UPW; ++uu) {
      const int u = wig + uu * WG;
      if (u < C::NU) {
#pragma unroll
        for (int t = 0; t < 2; ++t) {
          const int row = 8 * t + gr;
          uint4 kw;
          asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];\n"
                       : "=r"(kw.x), "=r"(kw.y), "=r"(kw.z), "=r"(kw.w)
                       : "r"(chunk_addr<FP8>(st, C::PITCH, row,
                                             kc0 + 4 * u + qd)));
          if constexpr (!FP8) {
            const uint32_t a0[4] = {qa[uu][0][0], qa[uu][1][0], qa[uu][0][1],
                                    qa[uu][1][1]};
            const uint32_t a1[4] = {qa[uu][0][2], qa[uu][1][2], qa[uu][0][3],
                                    qa[uu][1][3]};
            mma_16816<false>(s[t], a0, kw.x, kw.y);
            mma_16816<false>(s[t], a1, kw.z, kw.w);
          } else {
            const uint32_t w[4] = {kw.x, kw.y, kw.z, kw.w};
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              const uint32_t a[4] = {qa[uu][0][2 * j], qa[uu][1][2 * j],
                                     qa[uu][0][2 * j + 1], qa[uu][1][2 * j + 1]};
              mma_16816<true>(s[t], a,
                              e4m3x2_to_f16x2(static_cast<uint16_t>(w[j])),
                              e4m3x2_to_f16x2(static_cast<uint16_t>(w[j] >> 16)));
            }
          }
        }
      }
    }
    if constexpr (WG > 1) {  // sum the K-slice partial scores of the group
      float* mine = sbuf + ((it & 1) * WG + wig) * 32 * 8 + lane * 8;
      *reinterpret_cast<float4*>(mine) = make_float4(s[0][0], s[0][1], s[0][2], s[0][3]);
      *reinterpret_cast<float4*>(mine + 4) = make_float4(s[1][0], s[1][1], s[1][2], s[1][3]);
      group_sync();
#pragma unroll
      for (int t = 0; t < 2; ++t) s[t][0] = s[t][1] = s[t][2] = s[t][3] = 0.f;
#pragma unroll
      for (int w2 = 0; w2 < WG; ++w2) {
        const float* src = sbuf + ((it & 1) * WG + w2) * 32 * 8 + lane * 8;
        const float4 x = *reinterpret_cast<const float4*>(src);
        const float4 y = *reinterpret_cast<const float4*>(src + 4);
        s[0][0] += x.x; s[0][1] += x.y; s[0][2] += x.z; s[0][3] += x.w;
        s[1][0] += y.x; s[1][1] += y.y; s[1][2] += y.z; s[1][3] += y.w;
      }
    }

    // ---- online softmax (rows gr, gr + 8), log2 domain ----
    float cmax[2] = {-INFINITY, -INFINITY};
#pragma unroll
    for (int t = 0; t < 2; ++t)
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int key = kb + 8 * t + 2 * qd + (e & 1);
        const int k = e >> 1;
        const float v = key < vis_end[k] ? s[t][e] * qk_scale : -INFINITY;
        s[t][e] = v;
        cmax[k] = fmaxf(cmax[k], v);
      }
    float alpha[2], base[2];
#pragma unroll
    for (int k = 0; k < 2; ++k) {
      cmax[k] = fmaxf(cmax[k], __shfl_xor_sync(0xffffffffu, cmax[k], 1));
      cmax[k] = fmaxf(cmax[k], __shfl_xor_sync(0xffffffffu, cmax[k], 2));
      const float mn = fmaxf(m_run[k], cmax[k]);
      base[k] = mn == -INFINITY ? 0.f : mn;
      alpha[k] = fast_exp2(m_run[k] - base[k]);
      m_run[k] = mn;
    }
    float psum[2] = {0.f, 0.f};
#pragma unroll
    for (int t = 0; t < 2; ++t)
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float pv = fast_exp2(s[t][e] - base[e >> 1]);
        s[t][e] = pv;
        psum[e >> 1] += pv;
      }
#pragma unroll
    for (int k = 0; k < 2; ++k) l_run[k] = l_run[k] * alpha[k] + psum[k];
#pragma unroll
    for (int nt = 0; nt < C::NT; ++nt) {
      o[nt][0] *= alpha[0]; o[nt][1] *= alpha[0];
      o[nt][2] *= alpha[1]; o[nt][3] *= alpha[1];
    }
    uint32_t pa[4];
    if constexpr (!FP8) {
      pa[0] = pack_bf16x2(s[0][0], s[0][1]);
      pa[1] = pack_bf16x2(s[0][2], s[0][3]);
      pa[2] = pack_bf16x2(s[1][0], s[1][1]);
      pa[3] = pack_bf16x2(s[1][2], s[1][3]);
    } else {
      pa[0] = pack_f16x2(s[0][0], s[0][1]);
      pa[1] = pack_f16x2(s[0][2], s[0][3]);
      pa[2] = pack_f16x2(s[1][0], s[1][1]);
      pa[3] = pack_f16x2(s[1][2], s[1][3]);
    }

    // ---- O += P V over this warp's V columns ----
    const int vcol0 = wig * C::DVS;  // first V column of the slice
    if constexpr (!FP8) {
#pragma unroll
      for (int np = 0; np < C::NT / 2; ++np) {
        const int m = lane >> 3;
        const int row = (m & 1) * 8 + (lane & 7);
        const int ch = vc0 + (vcol0 + 16 * np) / 8 + (m >> 1);
        uint32_t r[4];
        ldmatrix_x4_trans(r, chunk_addr<false>(st, C::PITCH, row, ch));
        mma_16816<false>(o[2 * np], pa, r[0], r[1]);
        mma_16816<false>(o[2 * np + 1], pa, r[2], r[3]);
      }
    } else {
#pragma unroll
      for (int vb = 0; vb < C::DVS / 128; ++vb) {
        const int ch = vc0 + (vcol0 + 128 * vb) / 16 + gr;
        uint32_t kw[4][4];
        const int rows[4] = {2 * qd, 2 * qd + 1, 2 * qd + 8, 2 * qd + 9};
#pragma unroll
        for (int k = 0; k < 4; ++k)
          asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];\n"
                       : "=r"(kw[k][0]), "=r"(kw[k][1]), "=r"(kw[k][2]),
                         "=r"(kw[k][3])
                       : "r"(chunk_addr<true>(st, C::PITCH, rows[k], ch)));
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          const int w = j >> 2, sel = j & 3;
          const uint32_t b0 = e4m3x2_to_f16x2(pick_bytes(kw[0][w], kw[1][w], sel));
          const uint32_t b1 = e4m3x2_to_f16x2(pick_bytes(kw[2][w], kw[3][w], sel));
          mma_16816<true>(o[16 * vb + j], pa, b0, b1);
        }
      }
    }
  }
#pragma unroll
  for (int k = 0; k < 2; ++k) {
    l_run[k] += __shfl_xor_sync(0xffffffffu, l_run[k], 1);
    l_run[k] += __shfl_xor_sync(0xffffffffu, l_run[k], 2);
  }

  // ---- merge the groups through shared memory ----
  cp_async_wait<0>();
  __syncthreads();
  float* so = reinterpret_cast<float*>(smem);           // [NG][16][DVP]
  float* sm = so + NG * 16 * C::DVP;                    // [NG][16]
  float* sl = sm + NG * 16;                             // [NG][16]
  const int vcol0 = wig * C::DVS;
#pragma unroll
  for (int nt = 0; nt < C::NT; ++nt)
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      int col;
      if constexpr (!FP8)
        col = vcol0 + 8 * nt + 2 * qd + e;
      else
        col = vcol0 + 128 * (nt / 16) + 16 * (2 * qd + e) + (nt % 16);
      so[(grp * 16 + gr) * C::DVP + col] = o[nt][e];
      so[(grp * 16 + gr + 8) * C::DVP + col] = o[nt][2 + e];
    }
  if (wig == 0 && qd == 0) {
    sm[grp * 16 + gr] = m_run[0];
    sm[grp * 16 + gr + 8] = m_run[1];
    sl[grp * 16 + gr] = l_run[0];
    sl[grp * 16 + gr + 8] = l_run[1];
  }
  __syncthreads();
  for (int idx = threadIdx.x; idx < nrows * C::DV; idx += C::THREADS) {
    const int r = idx / C::DV;
    const int c = idx - r * C::DV;
    const int rr = row0 + r;
    const int64_t t = qs + rr / G;
    const int h = g * G + rr % G;
    float M = -INFINITY;
#pragma unroll
    for (int q = 0; q < NG; ++q) M = fmaxf(M, sm[q * 16 + r]);
    const int64_t orow = (split * T + t) * p.num_q_heads + h;
    if (M == -INFINITY) {
      if (c == 0) p.partial_lse[orow] = -INFINITY;
      continue;
    }
    float lsum = 0.f, acc = 0.f;
#pragma unroll
    for (int q = 0; q < NG; ++q) {
      const float mq = sm[q * 16 + r];
      if (mq == -INFINITY) continue;
      const float w = fast_exp2(mq - M);
      lsum += w * sl[q * 16 + r];
      acc += w * so[(q * 16 + r) * C::DVP + c];
    }
    p.partial_o[orow * C::DV + c] = acc / lsum * v_mul;
    if (c == 0) p.partial_lse[orow] = (M + fast_log2(lsum)) * kLn2;
  }
}

template <class C>
cudaError_t launch_cfg(const AttnParams& p, cudaStream_t stream) {
  static int attr_set[64] = {0};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 64 && !attr_set[dev]) {
    e = cudaFuncSetAttribute(decode_kernel<C>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                             C::SMEM);
    if (e != cudaSuccess) return e;
    attr_set[dev] = 1;
  }
  const int row_groups = (p.max_query_len * p.group + 15) / 16;
  dim3 grid(p.num_splits, p.num_kv_heads * row_groups, p.num_seqs);
  decode_kernel<C><<<grid, C::THREADS, C::SMEM, stream>>>(p);
  return cudaGetLastError();
}

using CfgBf16_192 = DecodeCfg<192, 128, false, 1, 4, 2, 320>;
using CfgFp8_192 = DecodeCfg<192, 128, true, 1, 4, 3, 320>;
using CfgBf16_576 = DecodeCfg<576, 512, false, 4, 2, 2, 576>;
using CfgFp8_576 = DecodeCfg<576, 512, true, 4, 2, 3, 576>;

}  // namespace

bool decode_supported(int head_size, int head_size_v, int dtype) {
  (void)dtype;
  return (head_size == 192 && head_size_v == 128) ||
         (head_size == 576 && head_size_v == 512);
}

cudaError_t launch_decode(const AttnParams& p, cudaStream_t stream) {
  const bool fp8 = p.dtype == PKV_FP8_E4M3;
  if (p.head_size == 192 && p.head_size_v == 128)
    return fp8 ? launch_cfg<CfgFp8_192>(p, stream)
               : launch_cfg<CfgBf16_192>(p, stream);
  if (p.head_size == 576 && p.head_size_v == 512)
    return fp8 ? launch_cfg<CfgFp8_576>(p, stream)
               : launch_cfg<CfgBf16_576>(p, stream);
  return cudaErrorNotSupported;
}

}  // namespace pkv
