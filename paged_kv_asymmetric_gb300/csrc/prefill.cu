// prefill.cu -- causal varlen prefill attention over the block-paged cache on
// the 5th-generation tensor core (tcgen05 MMA, accumulators in tensor memory,
// operands staged by TMA).
//
// What it computes: for every query token t of a sequence and query head h,
// out[t][h] = softmax(scale * q K^T over the keys t sees) V, causal and
// bottom-right aligned (vLLM PR #64064: unified attention over the packed
// K|V page; MiMo-V2.6-Flash 2x RTX PRO 6000 model card, "What the kernels
// do": a prefill attention kernel for the global layers with wide tiles).
// K head 192, V head 128.
//
// GB300 design (prior art on the pages was an sm_120 mma.sync kernel; this is
// not a translation of it):
//  * Persistent CTAs, one per SM.  A work item is a 128-row query tile of one
//    KV head: 128 / G consecutive tokens x the G query heads that share the
//    KV head (GQA packing), so every K/V tile staged in shared memory serves
//    all G heads.  Items are taken longest-first (last query tile first).
//  * Warp roles: warp 0 issues TMA loads (Q tile as three 64-column slabs;
//    K and V pages as 64-column boxes of one page each into 128-key slabs of
//    a shared 8-slab ring), warp 1 issues tcgen05.mma from one thread, warps
//    4..7 run the softmax with one thread per query row.
//  * S = Q K^T (M 128, N 128 keys, K 192) goes to one of two tensor-memory
//    buffers, so the MMA of key tile j+1 runs while the softmax reads tile j.
//    P is written as bf16 to shared memory (128-byte swizzled, the layout the
//    MMA reads) and O += P V (two N = 64 halves) accumulates in tensor memory.
//  * Online softmax with a lazy rescale: the running maximum used as the
//    exponent base is only raised, and O and the running sum rescaled, when
//    a new row maximum exceeds it by more than 2^8; the result is the same
//    up to rounding because the final O / l uses the same base.
//  * Keys past the sequence end in the last tile are masked out of S, and the
//    corresponding V rows are zeroed in shared memory before the P V MMA
//    reads them, so whatever the cache holds there cannot produce NaN.
//  * Every mbarrier wait is bounded (2 s): on expiry the kernel records
//    PKV_EDEV_TIMEOUT, every role stops at its next wait, the MMA thread waits
//    (bounded) for its MMAs to drain, and tensor memory is freed before exit.
#include <math.h>

#include <mutex>

#include <cudaTypedefs.h>

#include "common.cuh"
#include "kernels.h"
#include "tc5.cuh"

namespace pkv {

namespace {

constexpr int DK = 192, DV = 128;
constexpr int BM = 128, BN = 128;
constexpr int SLAB = 128 * 64 * 2;  // one 128-row x 64-column bf16 slab
constexpr int KSLABS = DK / 64;     // 3
constexpr int VSLABS = DV / 64;     // 2
constexpr int NSLAB = 8;            // K/V ring
constexpr int Q_OFF = 0;
constexpr int RING_OFF = Q_OFF + KSLABS * SLAB;
constexpr int P_OFF = RING_OFF + NSLAB * SLAB;
constexpr int BAR_OFF = P_OFF + 2 * SLAB;
enum {
  B_QFULL = 0,
  B_QEMPTY,
  B_SFULL0,
  B_SFULL1,
  B_SFREE0,
  B_SFREE1,
  B_PFULL,
  B_ODONE,
  B_OFREE,
  B_FINAL,
  B_SLAB_FULL0,
  B_SLAB_EMPTY0 = B_SLAB_FULL0 + NSLAB,
  NBAR = B_SLAB_EMPTY0 + NSLAB
};
constexpr int MISC_OFF = BAR_OFF + NBAR * 8;  // tmem base, abort word
constexpr int SMEM_BYTES = MISC_OFF + 16 + 1024;  // + alignment slack
constexpr int THREADS = 256;
constexpr uint32_t TMEM_COLS = 512;
constexpr uint32_t TM_S0 = 0, TM_O = 256;  // S buffers at 0 and 128
constexpr float kRescaleThreshold = 8.0f;  // log2 units

static_assert(SMEM_BYTES <= 227 * 1024, "shared memory budget");

struct Item {
  int b, qt, g, q0, nq, L, qlen;
  int minpos, nkeys, ntiles;
};

// The idx-th work item (longest-first within each sequence), or false.
__device__ __forceinline__ bool get_item(const AttnParams& p, int TQ, int idx,
                                         Item& it) {
  int acc = 0;
  for (int b = 0; b < p.num_seqs; ++b) {
    const int qs = __ldg(p.query_start_loc + b);
    const int qlen = __ldg(p.query_start_loc + b + 1) - qs;
    const int nt = (qlen + TQ - 1) / TQ;
    const int cnt = nt * p.num_kv_heads;
    if (idx < acc + cnt) {
      const int j = idx - acc;
      it.b = b;
      it.qt = nt - 1 - j / p.num_kv_heads;
      it.g = j % p.num_kv_heads;
      it.q0 = qs + it.qt * TQ;
      it.nq = min(TQ, qlen - it.qt * TQ);
      it.L = __ldg(p.seq_lens + b);
      it.qlen = qlen;
      it.minpos = it.L - qlen + it.qt * TQ;
      const int maxpos = it.minpos + it.nq - 1;
      it.nkeys = max(0, min(maxpos + 1, it.L));
      it.ntiles = (it.nkeys + BN - 1) / BN;
      return true;
    }
    acc += cnt;
  }
  return false;
}

__global__ void __launch_bounds__(THREADS, 1)
    prefill_kernel(const __grid_constant__ CUtensorMap q_map,
                   const __grid_constant__ CUtensorMap kv_map,
                   const AttnParams p) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t sbase = (raw + 1023u) & ~1023u;
  uint8_t* smem = smem_raw + (sbase - raw);
  const uint32_t bar0 = sbase + BAR_OFF;
  auto bar = [&](int i) { return bar0 + 8u * static_cast<uint32_t>(i); };
  volatile uint32_t* tmem_slot = reinterpret_cast<volatile uint32_t*>(smem + MISC_OFF);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + MISC_OFF + 8);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int G = p.group;
  const int TQ = BM / G;

  if (threadIdx.x == 0) {
    for (int i = 0; i < NBAR; ++i) {
      uint32_t count = 1;
      if (i == B_SFREE0 || i == B_SFREE1 || i == B_PFULL || i == B_OFREE)
        count = 128;
      tc5::mbar_init(bar(i), count);
    }
    *abort_flag = 0;
    tc5::fence_mbar_init();
    tc5::prefetch_tmap(&q_map);
    tc5::prefetch_tmap(&kv_map);
  }
  if (warp == 1) {
    tc5::tmem_alloc(sbase + MISC_OFF, TMEM_COLS);
    tc5::tmem_relinquish();
  }
  tc5::tc_fence_before();
  __syncthreads();
  tc5::tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  const int bs = p.block_size;
  const int box_rows = bs < BN ? bs : BN;
  const int nbox = BN / box_rows;

  if (warp == 0) {
    // ------------------------------------------------ TMA producer ------
    // The whole warp runs this loop.  Lane i owns box i of a 128-key slab
    // (nbox <= 16 boxes, one page or part of one each): it loads that box's
    // page id two tiles ahead of use and issues the box's copy itself, so
    // page-table reads never sit between consecutive copies.
    uint32_t qi = 0, f = 0;
    bool ok = true;
    const int32_t* bt_row = nullptr;
    auto load_pid = [&](const Item& it, int kt) -> int {
      const int key0 = kt * BN + lane * box_rows;
      if (kt >= it.ntiles || lane >= nbox || key0 >= it.L) return -1;
      return __ldg(bt_row + key0 / bs);
    };
    auto fill_slab = [&](const Item& it, int kt, int col, int pid) -> bool {
      const uint32_t slot = f % NSLAB;
      bool w = true;
      if (lane == 0)
        w = tc5::mbar_wait(bar(B_SLAB_EMPTY0 + slot), ((f / NSLAB) & 1u) ^ 1u,
                           abort_flag, p.err);
      if (!__shfl_sync(0xffffffffu, w, 0)) return false;
      const int lim = it.L - kt * BN;  // keys of the tile inside the sequence
      const int nb = min(nbox, (lim + box_rows - 1) / box_rows);
      const uint32_t full = bar(B_SLAB_FULL0 + slot);
      if (lane == 0)
        tc5::mbar_arrive_expect_tx(full, static_cast<uint32_t>(nb * box_rows * 128));
      __syncwarp();
      if (lane < nb) {
        const int key0 = kt * BN + lane * box_rows;
        const int off = key0 % bs;
        int page = pid;
        if (page < 0 || page >= p.num_blocks) {
          set_dev_error(p.err, PKV_EDEV_RANGE);
          page = p.num_blocks;  // out-of-range box: TMA fills zeros
        }
        const uint32_t dst = sbase + RING_OFF + slot * SLAB + lane * box_rows * 128;
        if (p.layout == PKV_NHD)
          tc5::tma_load_4d(dst, &kv_map, col, it.g, off, page, full);
        else
          tc5::tma_load_4d(dst, &kv_map, col, off, it.g, page, full);
      }
      ++f;
      return true;
    };
    for (int idx = blockIdx.x; ok; idx += gridDim.x) {
      Item it;
      if (!get_item(p, TQ, idx, it)) break;
      if (it.ntiles == 0) continue;
      bt_row = p.block_table + static_cast<int64_t>(it.b) * p.max_blocks_per_seq;
      int pid0 = load_pid(it, 0), pid1 = load_pid(it, 1);
      bool w = true;
      if (lane == 0) {
        w = tc5::mbar_wait(bar(B_QEMPTY), (qi & 1u) ^ 1u, abort_flag, p.err);
        if (w) {
          tc5::mbar_arrive_expect_tx(bar(B_QFULL), KSLABS * SLAB);
          for (int c = 0; c < KSLABS; ++c)
            tc5::tma_load_3d(sbase + Q_OFF + c * SLAB, &q_map, 64 * c, it.g * G,
                             it.q0, bar(B_QFULL));
        }
      }
      if (!__shfl_sync(0xffffffffu, w, 0)) break;
      ++qi;
      for (int c = 0; c < KSLABS && ok; ++c) ok = fill_slab(it, 0, p.k_off + 64 * c, pid0);
      for (int j = 0; j < it.ntiles && ok; ++j) {
        const int pid2 = load_pid(it, j + 2);  // prefetch
        if (j + 1 < it.ntiles)
          for (int c = 0; c < KSLABS && ok; ++c)
            ok = fill_slab(it, j + 1, p.k_off + 64 * c, pid1);
        for (int h = 0; h < VSLABS && ok; ++h) ok = fill_slab(it, j, p.v_off + 64 * h, pid0);
        pid0 = pid1;
        pid1 = pid2;
      }
    }
    // Outstanding copies land before the CTA may exit (they all have on the
    // normal path; after an abort some may still be in flight).
    if (lane == 0) {
      for (uint32_t k = f > NSLAB ? f - NSLAB : 0; k < f; ++k)
        tc5::mbar_wait(bar(B_SLAB_FULL0 + k % NSLAB), (k / NSLAB) & 1u, abort_flag,
                       p.err, /*honor_abort=*/false);
      if (qi > 0)
        tc5::mbar_wait(bar(B_QFULL), (qi - 1) & 1u, abort_flag, p.err, false);
    }
    __syncwarp();
  } else if (warp == 1 && lane == 0) {
    // ------------------------------------------------ MMA issuer --------
    constexpr uint32_t idesc_s = tc5::idesc_bf16_f32(BM, BN, false);
    constexpr uint32_t idesc_pv = tc5::idesc_bf16_f32(BM, 64, true);
    uint32_t qi = 0, f = 0, sidx = 0, pvidx = 0;
    bool ok = true;
    auto issue_s = [&]() -> bool {
      const uint32_t buf = sidx & 1u;
      if (!tc5::mbar_wait(bar(B_SFREE0 + buf), ((sidx >> 1) & 1u) ^ 1u, abort_flag, p.err))
        return false;
      for (int c = 0; c < KSLABS; ++c) {
        const uint32_t slot = f % NSLAB;
        if (!tc5::mbar_wait(bar(B_SLAB_FULL0 + slot), (f / NSLAB) & 1u, abort_flag, p.err))
          return false;
        tc5::tc_fence_after();
        const uint32_t qa = sbase + Q_OFF + c * SLAB;
        const uint32_t ka = sbase + RING_OFF + slot * SLAB;
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
          tc5::mma_f16_ss(tmem + TM_S0 + buf * BN, tc5::sdesc_sw128(qa + 32 * kk, 16, 1024),
                          tc5::sdesc_sw128(ka + 32 * kk, 16, 1024), idesc_s,
                          (c | kk) != 0);
        tc5::mma_commit(bar(B_SLAB_EMPTY0 + slot));
        ++f;
      }
      tc5::mma_commit(bar(B_SFULL0 + buf));
      ++sidx;
      return true;
    };
    for (int idx = blockIdx.x; ok; idx += gridDim.x) {
      Item it;
      if (!get_item(p, TQ, idx, it)) break;
      if (it.ntiles == 0) continue;
      if (!tc5::mbar_wait(bar(B_QFULL), qi & 1u, abort_flag, p.err)) break;
      tc5::tc_fence_after();
      ok = issue_s();
      for (int j = 0; j < it.ntiles && ok; ++j) {
        if (j + 1 < it.ntiles) {
          ok = issue_s();
          if (!ok) break;
        } else {
          tc5::mma_commit(bar(B_QEMPTY));  // every S MMA of the item issued
        }
        const uint32_t v0 = f % NSLAB, v1 = (f + 1) % NSLAB;
        ok = tc5::mbar_wait(bar(B_SLAB_FULL0 + v0), (f / NSLAB) & 1u, abort_flag, p.err) &&
             tc5::mbar_wait(bar(B_SLAB_FULL0 + v1), ((f + 1) / NSLAB) & 1u, abort_flag, p.err) &&
             tc5::mbar_wait(bar(B_PFULL), pvidx & 1u, abort_flag, p.err);
        if (ok && j == 0)
          ok = tc5::mbar_wait(bar(B_OFREE), (qi & 1u) ^ 1u, abort_flag, p.err);
        if (!ok) break;
        tc5::tc_fence_after();
#pragma unroll
        for (int h = 0; h < VSLABS; ++h) {
          const uint32_t va = sbase + RING_OFF + (h == 0 ? v0 : v1) * SLAB;
#pragma unroll
          for (int kk = 0; kk < BN / 16; ++kk) {
            const uint32_t pa = sbase + P_OFF + (kk / 4) * SLAB + (kk % 4) * 32;
            tc5::mma_f16_ss(tmem + TM_O + 64 * h, tc5::sdesc_sw128(pa, 16, 1024),
                            tc5::sdesc_sw128(va + kk * 2048, SLAB, 1024), idesc_pv,
                            (j > 0 || kk > 0) ? 1u : 0u);
          }
        }
        tc5::mma_commit(bar(B_SLAB_EMPTY0 + v0));
        tc5::mma_commit(bar(B_SLAB_EMPTY0 + v1));
        f += 2;
        tc5::mma_commit(bar(B_ODONE));
        ++pvidx;
      }
      ++qi;
    }
    // drain: every MMA issued above has completed before TMEM is freed
    tc5::mma_commit(bar(B_FINAL));
    tc5::mbar_wait(bar(B_FINAL), 0, abort_flag, p.err, /*honor_abort=*/false);
  } else if (warp >= 4) {
    // ------------------------------------------------ softmax -----------
    const int r = threadIdx.x - 128;               // query row of the tile
    const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const float scale_log2 = p.softmax_scale * kLog2e;
    uint32_t sidx = 0, pvidx = 0, fbase = 0;
    uint8_t* psm = smem + P_OFF;
    // waits whose outcome is the same for the whole warp, so that the warp
    // stays converged for the warp-collective tensor-memory accesses
    auto wwait = [&](uint32_t b, uint32_t parity) {
      const bool r = tc5::mbar_wait(b, parity, abort_flag, p.err);
      return __all_sync(0xffffffffu, r);
    };
    for (int idx = blockIdx.x;; idx += gridDim.x) {
      Item it;
      if (!get_item(p, TQ, idx, it)) break;
      const int tr = r / G, hr = r % G;
      const bool valid = tr < it.nq;
      const int pos = it.minpos + tr;
      const int64_t orow =
          (static_cast<int64_t>(it.q0 + tr) * p.num_q_heads + it.g * G + hr) * DV;
      if (it.ntiles == 0) {
        if (valid) {
          uint4* dst = reinterpret_cast<uint4*>(p.out + orow);
#pragma unroll
          for (int c = 0; c < DV / 8; ++c) dst[c] = make_uint4(0, 0, 0, 0);
        }
        continue;
      }
      float m = -INFINITY, l = 0.f;
      bool ok = true;
      for (int j = 0; j < it.ntiles; ++j) {
        const uint32_t buf = sidx & 1u;
        if (!wwait(bar(B_SFULL0 + buf), (sidx >> 1) & 1u)) {
          ok = false;
          break;
        }
        tc5::tc_fence_after();
        float s[BN];
        {
          uint32_t v[BN / 32][32];
#pragma unroll
          for (int c = 0; c < BN / 32; ++c)
            tc5::tmem_ld_32x32b_x32(tmem + lane_off + TM_S0 + buf * BN + 32 * c, v[c]);
          tc5::tmem_wait_ld();
#pragma unroll
          for (int c = 0; c < BN / 32; ++c)
#pragma unroll
            for (int k = 0; k < 32; ++k) s[32 * c + k] = __uint_as_float(v[c][k]);
        }
        tc5::tc_fence_before();
        tc5::mbar_arrive(bar(B_SFREE0 + buf));
        ++sidx;

        const int kbase = j * BN;
        if (!valid || kbase + BN - 1 > pos) {
#pragma unroll
          for (int c = 0; c < BN; ++c)
            if (!valid || kbase + c > pos) s[c] = -INFINITY;
        }
        float mx = -INFINITY;
#pragma unroll
        for (int c = 0; c < BN; ++c) mx = fmaxf(mx, s[c]);
        const float mt = mx * scale_log2;
        const float m_new = fmaxf(m, mt);
        bool o_ready = false;  // PV of tile j-1 known complete
        // The rescale touches tensor memory with warp-collective loads and
        // stores, so the decision is taken per warp: when any row of the
        // warp needs a higher base, every row of the warp moves to its own
        // current maximum (alpha = 1 where that is unchanged).
        const bool need = j > 0 && m_new > m + kRescaleThreshold;
        if (j == 0) {
          m = m_new;
        } else if (__any_sync(0xffffffffu, need)) {
          if (!wwait(bar(B_ODONE), (pvidx - 1) & 1u)) {
            ok = false;
            break;
          }
          o_ready = true;
          tc5::tc_fence_after();
          const float alpha = m_new == -INFINITY ? 1.f : fast_exp2(m - m_new);
#pragma unroll
          for (int c = 0; c < DV / 32; ++c) {
            uint32_t v[32];
            tc5::tmem_ld_32x32b_x32(tmem + lane_off + TM_O + 32 * c, v);
            tc5::tmem_wait_ld();
#pragma unroll
            for (int k = 0; k < 32; ++k)
              v[k] = __float_as_uint(__uint_as_float(v[k]) * alpha);
            tc5::tmem_st_32x32b_x32(tmem + lane_off + TM_O + 32 * c, v);
          }
          tc5::tmem_wait_st();
          l *= alpha;
          m = m_new;
        }
        const float base = m == -INFINITY ? 0.f : m;
        uint32_t pk[BN / 2];
#pragma unroll
        for (int c = 0; c < BN / 2; ++c) {
          const float p0 = fast_exp2(fmaf(s[2 * c], scale_log2, -base));
          const float p1 = fast_exp2(fmaf(s[2 * c + 1], scale_log2, -base));
          l += p0 + p1;
          pk[c] = pack_bf16x2(p0, p1);
        }
        if (j > 0 && !o_ready) {  // P of tile j-1 still being read?
          if (!wwait(bar(B_ODONE), (pvidx - 1) & 1u)) {
            ok = false;
            break;
          }
        }
        // P row -> shared memory, K-major with the 128-byte swizzle
        {
          uint8_t* rowp = psm + (r >> 3) * 1024 + (r & 7) * 128;
#pragma unroll
          for (int sl = 0; sl < 2; ++sl)
#pragma unroll
            for (int ch = 0; ch < 8; ++ch) {
              const int w = sl * 32 + ch * 4;
              *reinterpret_cast<uint4*>(rowp + sl * SLAB + ((ch ^ (r & 7)) << 4)) =
                  make_uint4(pk[w], pk[w + 1], pk[w + 2], pk[w + 3]);
            }
        }
        if (kbase + BN > it.L) {
          // last tile: zero the V rows of keys past the sequence end
          const uint32_t vfill =
              fbase + 3u * static_cast<uint32_t>(min(j + 2, it.ntiles)) + 2u * j;
          for (int h = 0; h < VSLABS && ok; ++h) {
            const uint32_t fi = vfill + h;
            ok = wwait(bar(B_SLAB_FULL0 + fi % NSLAB), (fi / NSLAB) & 1u);
            if (ok && kbase + r >= it.L) {
              uint4* vrow = reinterpret_cast<uint4*>(smem + RING_OFF + (fi % NSLAB) * SLAB +
                                                     r * 128);
#pragma unroll
              for (int ch = 0; ch < 8; ++ch) vrow[ch] = make_uint4(0, 0, 0, 0);
            }
          }
          if (!ok) break;
        }
        tc5::fence_proxy_async_smem();
        tc5::tc_fence_before();
        tc5::mbar_arrive(bar(B_PFULL));
        ++pvidx;
      }
      if (!ok) break;
      // ---- epilogue: O / l -> bf16 ----
      if (!wwait(bar(B_ODONE), (pvidx - 1) & 1u)) break;
      tc5::tc_fence_after();
      const float inv = l > 0.f ? 1.f / l : 0.f;
      uint4 packed[DV / 8];
#pragma unroll
      for (int c = 0; c < DV / 32; ++c) {
        uint32_t v[32];
        tc5::tmem_ld_32x32b_x32(tmem + lane_off + TM_O + 32 * c, v);
        tc5::tmem_wait_ld();
#pragma unroll
        for (int k = 0; k < 4; ++k)
          packed[4 * c + k] = make_uint4(
              pack_bf16x2(__uint_as_float(v[8 * k + 0]) * inv, __uint_as_float(v[8 * k + 1]) * inv),
              pack_bf16x2(__uint_as_float(v[8 * k + 2]) * inv, __uint_as_float(v[8 * k + 3]) * inv),
              pack_bf16x2(__uint_as_float(v[8 * k + 4]) * inv, __uint_as_float(v[8 * k + 5]) * inv),
              pack_bf16x2(__uint_as_float(v[8 * k + 6]) * inv, __uint_as_float(v[8 * k + 7]) * inv));
      }
      tc5::tc_fence_before();
      tc5::mbar_arrive(bar(B_OFREE));
      if (valid) {
        uint4* dst = reinterpret_cast<uint4*>(p.out + orow);
#pragma unroll
        for (int c = 0; c < DV / 8; ++c) dst[c] = packed[c];
      }
      fbase += 5u * static_cast<uint32_t>(it.ntiles);
    }
  }

  tc5::tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc5::tc_fence_after();
    tc5::tmem_dealloc(tmem, TMEM_COLS);
  }
}

PFN_cuTensorMapEncodeTiled_v12000 get_encode_fn() {
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

}  // namespace

bool prefill_supported(int head_size, int head_size_v, int dtype) {
  return head_size == DK && head_size_v == DV && dtype == PKV_BF16;
}

cudaError_t launch_prefill(const AttnParams& p, int num_sms,
                           cudaStream_t stream) {
  if (!prefill_supported(p.head_size, p.head_size_v, p.dtype))
    return cudaErrorNotSupported;
  PFN_cuTensorMapEncodeTiled_v12000 encode = get_encode_fn();
  if (encode == nullptr) return cudaErrorNotSupported;
  const int G = p.group;
  const int TQ = BM / G;
  alignas(64) CUtensorMap q_map, kv_map;
  {
    const cuuint64_t dims[3] = {static_cast<cuuint64_t>(DK),
                                static_cast<cuuint64_t>(p.num_q_heads),
                                static_cast<cuuint64_t>(p.num_tokens)};
    const cuuint64_t strides[2] = {static_cast<cuuint64_t>(DK) * 2,
                                   static_cast<cuuint64_t>(p.num_q_heads) * DK * 2};
    const cuuint32_t box[3] = {64, static_cast<cuuint32_t>(G),
                               static_cast<cuuint32_t>(TQ)};
    const cuuint32_t es[3] = {1, 1, 1};
    if (encode(&q_map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3,
               const_cast<__nv_bfloat16*>(p.q), dims, strides, box, es,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
  }
  {
    const cuuint64_t R = static_cast<cuuint64_t>(p.row_elems);
    const cuuint64_t H = static_cast<cuuint64_t>(p.num_kv_heads);
    const cuuint64_t B = static_cast<cuuint64_t>(p.block_size);
    const cuuint32_t box_rows = static_cast<cuuint32_t>(p.block_size < BN ? p.block_size : BN);
    cuuint64_t dims[4], strides[3];
    cuuint32_t box[4];
    if (p.layout == PKV_NHD) {  // [blk][bs][H][R]: dims (R, H, bs, blk)
      dims[0] = R; dims[1] = H; dims[2] = B; dims[3] = p.num_blocks;
      strides[0] = R * 2; strides[1] = H * R * 2; strides[2] = B * H * R * 2;
      box[0] = 64; box[1] = 1; box[2] = box_rows; box[3] = 1;
    } else {                    // [blk][H][bs][R]: dims (R, bs, H, blk)
      dims[0] = R; dims[1] = B; dims[2] = H; dims[3] = p.num_blocks;
      strides[0] = R * 2; strides[1] = B * R * 2; strides[2] = H * B * R * 2;
      box[0] = 64; box[1] = box_rows; box[2] = 1; box[3] = 1;
    }
    const cuuint32_t es[4] = {1, 1, 1, 1};
    if (encode(&kv_map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(p.cache),
               dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
               CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
  }
  static int attr_set[64] = {0};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 64 && !attr_set[dev]) {
    e = cudaFuncSetAttribute(prefill_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             SMEM_BYTES);
    if (e != cudaSuccess) return e;
    attr_set[dev] = 1;
  }
  prefill_kernel<<<num_sms, THREADS, SMEM_BYTES, stream>>>(q_map, kv_map, p);
  return cudaGetLastError();
}

}  // namespace pkv
