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
// K|V row is read once per (sequence, KV head) and serves all q_len * G query
// rows of that KV head (G = Hq / Hkv).
//  * Work unit = (split, sequence, KV head, 16-row group); the rows are
//    (query token, query head) pairs, so a 1+3-token verify with G = 4 is one
//    m16 tile.  Persistent CTAs (one per SM) take units round-robin and keep
//    streaming across unit boundaries: loads for the next unit overlap the
//    end of the current one, and no CTA pays a cold start per unit.
//  * Warp 0 is the producer: it copies the unit's 16 query rows into a
//    double-buffered Q slot (cp.async, completion on an mbarrier) and each
//    16-key chunk of K|V rows into a ring slot with TMA boxes of 16 slots x
//    128 bytes of one page and KV head (one instruction per box, 128-byte
//    swizzle, columns past the row read as zero), page ids prefetched by all
//    lanes ahead of use.
//  * Consumer warps form NG groups of WG warps; chunk c (counted across
//    units) goes to group c % NG, and the ring has a multiple of NG slots, so
//    each slot is consumed by one group in order (no mbarrier phase can be
//    mistaken for the one two fills later).  Within a group, warp w owns a
//    slice of the K dimension for Q.K^T (partial scores summed through
//    shared memory when WG > 1) and a slice of V's columns for P.V.  16
//    rows are below tcgen05's M = 64, and the FP8 operands are converted in
//    registers, so the contraction runs on the warp-level m16n8k16 MMA
//    (~4-32 flop per byte here).
//  * bf16 cache: K and V fragments come from ldmatrix (.trans for V) on the
//    swizzled slot.  fp8 cache: E4M3 codes become f16 in registers (exact),
//    K through 16-byte loads with the reduction index permuted identically
//    in Q and K, V by byte-permuting four keys' 16-column runs into k-pairs;
//    the MMA runs in f16 with Q converted bf16 -> f16; k_scale is folded into
//    the softmax scale and v_scale into the output.
//  * Online softmax in registers with exp2.  The last chunk of a unit has its
//    rows past the last visible key zeroed in shared memory, so garbage in a
//    partly filled page cannot reach the MMA; the scores of those keys are
//    masked.  Groups merge (max, sum, O) through shared memory per unit.
//  * Every mbarrier wait is bounded; after a timeout the kernel records
//    PKV_EDEV_TIMEOUT, the waits of all roles return at once, every warp
//    still walks the same units (so named barriers stay matched), and the
//    producer waits (bounded) for its own copies before exit.
#include <math.h>

#include "common.cuh"
#include "kernels.h"
#include "tc5.cuh"
#include "tmap.h"

namespace pkv {

namespace {

template <int DK_, int DV_, bool FP8_, int WG_, int NG_, int NSLOT_, int NQ_,
          int SPAN_>
struct DecodeCfg {
  static constexpr int DK = DK_, DV = DV_, WG = WG_, NG = NG_;
  static constexpr int NSLOT = NSLOT_, NQ = NQ_, SPAN = SPAN_;
  static constexpr int MAXP = 128;  // page ids staged with a unit
  static constexpr bool FP8 = FP8_;
  static constexpr int ESZ = FP8 ? 1 : 2;
  static constexpr int SPAN_BYTES = SPAN * ESZ;
  static constexpr int NBOX = (SPAN_BYTES + 127) / 128;  // 128-byte column boxes
  static constexpr int BOX_COLS = 128 / ESZ;
  static constexpr int SLOT_BYTES = NBOX * 16 * 128;
  static constexpr int NCW = WG * NG;                      // consumer warps
  static constexpr int THREADS = 32 * (1 + NCW);
  static constexpr int QCH = DK * 2 / 16;                  // 16-byte Q pieces per row
  static constexpr int Q_BYTES = 16 * DK * 2;
  static constexpr int KSTEPS = DK / 16;
  static constexpr int KSW = KSTEPS / WG;                  // bf16: k-steps per warp
  static constexpr int NU = DK / 64;                       // fp8: 64-wide units
  static constexpr int UPW = (NU + WG - 1) / WG;
  static constexpr int DVS = DV / WG;                      // V columns per warp
  static constexpr int NT = DVS / 8;
  static constexpr int DVP = DV + 4;
  static constexpr int RING_OFF = 0;
  static constexpr int Q_OFF = RING_OFF + NSLOT * SLOT_BYTES;
  static constexpr int DESC_OFF = Q_OFF + NQ * Q_BYTES;
  static constexpr int DESC_BYTES = 64 + MAXP * 4;  // descriptor + page ids
  static constexpr int MERGE_OFF = DESC_OFF + NQ * DESC_BYTES;
  static constexpr int MERGE = NG > 1 ? NG * 16 * DVP * 4 + 2 * NG * 16 * 4 : 0;
  static constexpr int SBUF_OFF = MERGE_OFF + MERGE;
  static constexpr int SBUF = WG > 1 ? NG * 2 * WG * 32 * 8 * 4 : 0;
  static constexpr int BAR_OFF = SBUF_OFF + SBUF;
  static constexpr int NBAR = 2 * NSLOT + 2 * NQ;
  static constexpr int SMEM = BAR_OFF + NBAR * 8 + 16 + 1024;
  static_assert(DK % 64 == 0 && KSTEPS % WG == 0, "K slices");
  static_assert(DV % WG == 0 && DVS % (FP8 ? 128 : 16) == 0, "V slices");
  static_assert(QCH % 8 == 0, "Q rows in whole 128-byte groups");
  static_assert(SMEM <= 227 * 1024, "shared memory budget");
  static_assert(NSLOT % NG == 0, "each ring slot belongs to one consumer group");
};

// Address of the 16-byte piece `piece` (byte offset / 16 within the staged
// span) of key row `row` in a ring slot: TMA box piece/8 holds 16 rows x 128
// bytes, and the 128-byte swizzle permutes 16-byte pieces by the row index.
__device__ __forceinline__ uint32_t slot_piece(uint32_t slot, int row, int piece) {
  return slot + (piece >> 3) * 2048 + row * 128 + (((piece & 7) ^ (row & 7)) << 4);
}

// Q rows (bf16, DK wide) in a Q slot: rows of DK*2 bytes, 16-byte pieces
// swizzled within each 128-byte group by the row index.
template <int DK>
__device__ __forceinline__ uint32_t q_piece(uint32_t qslot, int row, int piece) {
  return qslot + row * (DK * 2) + ((piece & ~7) | ((piece & 7) ^ (row & 7))) * 16;
}

__device__ __forceinline__ void ldmatrix_x4(uint32_t (&r)[4], uint32_t saddr) {
  asm volatile(
      "ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];\n"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
      : "r"(saddr));
}

__device__ __forceinline__ uint4 lds128(uint32_t saddr) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "r"(saddr));
  return v;
}

__device__ __forceinline__ void cp_async_4(uint32_t dst, const void* src) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4;\n" ::"r"(dst), "l"(src));
}

// OR of `pred` over the `count` threads that meet at named barrier `id`;
// every participant gets the same answer.
__device__ __forceinline__ bool barrier_or(int id, int count, bool pred) {
  uint32_t r;
  asm volatile(
      "{\n .reg .pred p, q;\n setp.ne.u32 p, %1, 0;\n"
      " barrier.red.or.pred q, %2, %3, p;\n selp.u32 %0, 1, 0, q;\n}\n"
      : "=r"(r)
      : "r"(static_cast<uint32_t>(pred)), "r"(id), "r"(count)
      : "memory");
  return r != 0;
}

// A work unit; the producer stages it in shared memory as 16 ints followed
// by its page ids.
struct Unit {
  int b, g, s, row0, nrows, qs, qlen, L;
  int klo, khi, kmax, nch, page_lo, npages, pad0, pad1;
};
static_assert(sizeof(Unit) == 64, "descriptor size");

// Sequence of unit u: split-major order over (split, sequence, KV head, row
// group).
__device__ __forceinline__ int unit_seq(const AttnParams& p, int RG, int u) {
  const int per_split = p.num_seqs * p.num_kv_heads * RG;
  return (u % per_split) / (p.num_kv_heads * RG);
}

// Unit u's parameters from its sequence's query_start_loc pair and length.
__device__ __forceinline__ void unit_params(const AttnParams& p, int RG, int u,
                                            int q0, int q1, int L, Unit& un) {
  const int per_split = p.num_seqs * p.num_kv_heads * RG;
  un.s = u / per_split;
  int rem = u - un.s * per_split;
  un.b = rem / (p.num_kv_heads * RG);
  rem -= un.b * p.num_kv_heads * RG;
  un.g = rem % p.num_kv_heads;
  const int rg = rem / p.num_kv_heads;
  const int G = p.group;
  un.qs = q0;
  un.qlen = q1 - q0;
  un.L = L;
  un.row0 = rg * 16;
  un.nrows = max(0, min(16, un.qlen * G - un.row0));
  const int bs = p.block_size;
  const int P = (un.L + bs - 1) / bs;
  const int pps = (P + p.num_splits - 1) / p.num_splits;
  const int page_lo = min(un.s * pps, P);
  const int page_hi = min(page_lo + pps, P);
  un.klo = page_lo * bs;
  un.khi = min(page_hi * bs, un.L);
  un.kmax = un.klo;
  if (un.nrows > 0) {
    // the unit's last row belongs to its latest query token: it sees most
    const int i_last = (un.row0 + un.nrows - 1) / G;
    un.kmax = min(un.khi, max(0, min(un.L, un.L - un.qlen + i_last + 1)));
  }
  un.nch = un.kmax > un.klo ? (un.kmax - un.klo + 15) / 16 : 0;
  un.page_lo = page_lo;
  un.npages = page_hi - page_lo;
  un.pad0 = un.pad1 = 0;
}

template <class C>
__global__ void __launch_bounds__(C::THREADS, 1)
    decode_kernel(const __grid_constant__ CUtensorMap kv_map, const AttnParams p) {
  extern __shared__ uint8_t smem_raw[];
  constexpr bool FP8 = C::FP8;
  constexpr int WG = C::WG, NG = C::NG, NSLOT = C::NSLOT;
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t sbase = (raw + 1023u) & ~1023u;
  uint8_t* smem = smem_raw + (sbase - raw);
  const uint32_t bar0 = sbase + C::BAR_OFF;
  auto slot_full = [&](int i) { return bar0 + 8u * i; };
  auto slot_empty = [&](int i) { return bar0 + 8u * (NSLOT + i); };
  auto q_full = [&](int i) { return bar0 + 8u * (2 * NSLOT + i); };
  auto q_empty = [&](int i) { return bar0 + 8u * (2 * NSLOT + C::NQ + i); };
  auto desc_of = [&](int i) {
    return reinterpret_cast<Unit*>(smem + C::DESC_OFF + i * C::DESC_BYTES);
  };
  auto pages_of = [&](int i) {
    return reinterpret_cast<const int*>(smem + C::DESC_OFF + i * C::DESC_BYTES + 64);
  };
  volatile int* abort_flag =
      reinterpret_cast<volatile int*>(smem + C::BAR_OFF + C::NBAR * 8);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int G = p.group;
  const int RG = (p.max_query_len * G + 15) / 16;
  const int num_units = p.num_splits * p.num_seqs * p.num_kv_heads * RG;
  const int bs = p.block_size;
  const int box_rows = bs < 16 ? bs : 16;
  const int nrb = 16 / box_rows;  // row boxes per chunk
  const int lo = min(p.k_off, p.v_off);
  const int64_t T = p.num_tokens;

  if (threadIdx.x == 0) {
    for (int i = 0; i < NSLOT; ++i) {
      tc5::mbar_init(slot_full(i), 1);
      tc5::mbar_init(slot_empty(i), WG);
    }
    for (int i = 0; i < C::NQ; ++i) {
      tc5::mbar_init(q_full(i), 1);
      tc5::mbar_init(q_empty(i), C::NCW);
    }
    *abort_flag = 0;
    tc5::fence_mbar_init();
    tc5::prefetch_tmap(&kv_map);
  }
  __syncthreads();

  if (warp == 0) {
    // ------------------------------------------------ producer warp -----
    // Units are staged two ahead of the one whose chunks are being issued:
    // the unit's query rows, its page ids (block-table entries, copied
    // asynchronously) and a descriptor go to one of NQ slots, so that no
    // block-table or sequence-metadata read sits in front of a copy.
    uint32_t gc = 0;    // chunks issued
    uint32_t qs_n = 0;  // units staged
    uint32_t qi_n = 0;  // units issued
    const int my_units =
        static_cast<int>(blockIdx.x) < num_units
            ? (num_units - 1 - static_cast<int>(blockIdx.x)) / static_cast<int>(gridDim.x) + 1
            : 0;
    int pos = 0;                 // next position in this CTA's unit list
    int mq0 = 0, mq1 = 0, mL = 0;  // metadata of the unit at `pos`
    auto meta_load = [&](int ps) {
      if (ps < my_units) {
        const int b = unit_seq(p, RG, blockIdx.x + ps * gridDim.x);
        mq0 = __ldg(p.query_start_loc + b);
        mq1 = __ldg(p.query_start_loc + b + 1);
        mL = __ldg(p.seq_lens + b);
      }
    };
    meta_load(0);
    bool alive = true;
    auto stage_next = [&]() {
      while (pos < my_units) {
        Unit un;
        unit_params(p, RG, blockIdx.x + pos * gridDim.x, mq0, mq1, mL, un);
        ++pos;
        meta_load(pos);  // the next unit's metadata is in flight meanwhile
        if (un.nrows == 0) continue;
        if (un.nch == 0) {  // no key of this segment is visible to any row
          for (int r = lane; r < un.nrows; r += 32) {
            const int rr = un.row0 + r;
            const int64_t t = un.qs + rr / G;
            const int h = un.g * G + rr % G;
            p.partial_lse[(un.s * T + t) * p.num_q_heads + h] = -INFINITY;
          }
          continue;
        }
        const uint32_t qslot = qs_n % C::NQ;
        bool w = true;
        if (lane == 0)
          w = tc5::mbar_wait(q_empty(qslot), ((qs_n / C::NQ) & 1u) ^ 1u, abort_flag, p.err);
        if (!__shfl_sync(0xffffffffu, w, 0)) {
          alive = false;
          return;
        }
        const uint32_t qdst = sbase + C::Q_OFF + qslot * C::Q_BYTES;
        for (int i = lane; i < 16 * C::QCH; i += 32) {
          const int r = i / C::QCH, j = i - r * C::QCH;
          const bool valid = r < un.nrows;
          const int rr = un.row0 + r;
          const int64_t t = un.qs + rr / G;
          const int h = un.g * G + rr % G;
          const __nv_bfloat16* src =
              valid ? p.q + (t * p.num_q_heads + h) * C::DK + j * 8 : p.q;
          cp_async_16(q_piece<C::DK>(qdst, r, j), src, valid ? 16 : 0);
        }
        const int np = min(un.npages, C::MAXP);
        const int32_t* bt = p.block_table +
                            static_cast<int64_t>(un.b) * p.max_blocks_per_seq + un.page_lo;
        const uint32_t pdst = sbase + C::DESC_OFF + qslot * C::DESC_BYTES + 64;
        for (int i = lane; i < np; i += 32) cp_async_4(pdst + 4 * i, bt + i);
        if (lane == 0) *desc_of(qslot) = un;
        cp_async_commit();
        ++qs_n;
        return;
      }
    };
    stage_next();
    if (alive) stage_next();
    while (alive && qi_n < qs_n) {
      const uint32_t qslot = qi_n % C::NQ;
      // this unit's copies are complete once at most the newer unit's group
      // is still pending
      if (qs_n - qi_n >= 2)
        cp_async_wait<1>();
      else
        cp_async_wait<0>();
      __syncwarp();
      if (lane == 0) tc5::mbar_arrive(q_full(qslot));
      const Unit un = *desc_of(qslot);
      const int* pages = pages_of(qslot);
      const int32_t* bt = p.block_table + static_cast<int64_t>(un.b) * p.max_blocks_per_seq;
      // Chunks go out in batches of PB: lane i owns chunk i of the batch
      // (its slot wait, its transaction count, its page ids and its boxes),
      // so the fixed cost of getting a chunk under way is paid in parallel.
      constexpr int PB = C::NSLOT / 3 > 1 ? C::NSLOT / 3 : 1;
      for (int k0 = 0; k0 < un.nch; k0 += PB) {
        const int nbatch = min(PB, un.nch - k0);
        const bool mine = lane < nbatch;
        const uint32_t c = gc + lane;
        const uint32_t slot = c % NSLOT;
        bool w = true;
        if (mine)
          w = tc5::mbar_wait(slot_empty(slot), ((c / NSLOT) & 1u) ^ 1u, abort_flag, p.err);
        if (!__all_sync(0xffffffffu, w)) {
          alive = false;
          break;
        }
        if (mine) {
          const int kb = un.klo + (k0 + lane) * 16;
          const int nvr = min(nrb, (un.kmax - kb + box_rows - 1) / box_rows);
          tc5::mbar_arrive_expect_tx(slot_full(slot),
                                     static_cast<uint32_t>(nvr * C::NBOX * box_rows * 128));
          for (int rb = 0; rb < nvr; ++rb) {
            const int key0 = kb + rb * box_rows;
            const int pidx = key0 / bs - un.page_lo;
            int page = pidx < C::MAXP ? pages[pidx] : __ldg(bt + key0 / bs);
            if (page < 0 || page >= p.num_blocks) {
              set_dev_error(p.err, PKV_EDEV_RANGE);
              page = p.num_blocks;  // out-of-range box: TMA fills zeros
            }
            const uint32_t dst0 =
                sbase + C::RING_OFF + slot * C::SLOT_BYTES + rb * box_rows * 128;
#pragma unroll
            for (int cb = 0; cb < C::NBOX; ++cb) {
              const int col = lo + cb * C::BOX_COLS;
              if (p.layout == PKV_NHD)
                tc5::tma_load_4d(dst0 + cb * 2048, &kv_map, col, un.g, key0 % bs, page,
                                 slot_full(slot));
              else
                tc5::tma_load_4d(dst0 + cb * 2048, &kv_map, col, key0 % bs, un.g, page,
                                 slot_full(slot));
            }
          }
        }
        gc += nbatch;
      }
      ++qi_n;
      if (alive) stage_next();
    }
    if (alive) {  // end marker for the consumers
      const uint32_t qslot = qs_n % C::NQ;
      bool w = true;
      if (lane == 0) {
        w = tc5::mbar_wait(q_empty(qslot), ((qs_n / C::NQ) & 1u) ^ 1u, abort_flag, p.err);
        if (w) {
          desc_of(qslot)->nch = -1;
          tc5::mbar_arrive(q_full(qslot));
        }
      }
      __syncwarp();
    }
    // outstanding copies land before the CTA may exit
    if (lane == 0)
      for (uint32_t k = gc > NSLOT ? gc - NSLOT : 0; k < gc; ++k)
        tc5::mbar_wait(slot_full(k % NSLOT), (k / NSLOT) & 1u, abort_flag, p.err, false);
    cp_async_wait<0>();
    __syncwarp();
  } else {
    // ------------------------------------------------ consumer warps ----
    const int cw = warp - 1;
    const int grp = cw / WG, wig = cw % WG;
    const int gr = lane >> 2, qd = lane & 3;
    const int ctid = threadIdx.x - 32;  // consumer thread index
    uint32_t gc = 0, qc = 0;
    uint32_t xk = 0;  // chunks this group has processed: picks the exchange buffer
    float* sbuf = reinterpret_cast<float*>(smem + C::SBUF_OFF) + grp * 2 * WG * 32 * 8;
    auto group_sync = [&]() {
      if constexpr (WG == 1)
        __syncwarp();
      else
        named_barrier(2 + grp, 32 * WG);
    };
    auto wait_all = [&](uint32_t b, uint32_t parity) {
      const bool r = tc5::mbar_wait(b, parity, abort_flag, p.err);
      return __all_sync(0xffffffffu, r);
    };
    for (;;) {
      // ---- next staged unit: descriptor and Q fragments ----
      const uint32_t qslot = qc % C::NQ;
      wait_all(q_full(qslot), (qc / C::NQ) & 1u);
      // every consumer warp takes the same decision to stop after a timeout
      if (barrier_or(15, 32 * C::NCW, *abort_flag != 0)) break;
      const Unit un = *desc_of(qslot);
      if (un.nch < 0) break;
      const uint32_t qsrc = sbase + C::Q_OFF + qslot * C::Q_BYTES;
      uint32_t qa[FP8 ? C::UPW : C::KSW][FP8 ? 16 : 4];
      if constexpr (!FP8) {
#pragma unroll
        for (int kk = 0; kk < C::KSW; ++kk) {
          const int ks = wig * C::KSW + kk;
          const int m = lane >> 3;
          const int row = (m & 1) * 8 + (lane & 7);
          ldmatrix_x4(qa[kk], q_piece<C::DK>(qsrc, row, ks * 2 + (m >> 1)));
        }
      } else {
#pragma unroll
        for (int uu = 0; uu < C::UPW; ++uu) {
          const int un_ = wig + uu * WG;
          if (un_ < C::NU) {
#pragma unroll
            for (int k = 0; k < 2; ++k) {
              const int row = gr + 8 * k;
              const uint4 v0 = lds128(q_piece<C::DK>(qsrc, row, un_ * 8 + 2 * qd));
              const uint4 v1 = lds128(q_piece<C::DK>(qsrc, row, un_ * 8 + 2 * qd + 1));
              const uint32_t wv[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
#pragma unroll
              for (int j = 0; j < 8; ++j) qa[uu][k * 8 + j] = bf16x2_to_f16x2(wv[j]);
            }
          } else {
#pragma unroll
            for (int j = 0; j < 16; ++j) qa[uu][j] = 0u;
          }
        }
      }
      __syncwarp();
      if (lane == 0) tc5::mbar_arrive(q_empty(qslot));
      ++qc;

      // ---- per-row visibility, scales ----
      int vis_end[2];
#pragma unroll
      for (int k = 0; k < 2; ++k) {
        const int r = gr + 8 * k;
        if (r < un.nrows) {
          const int i = (un.row0 + r) / G;
          vis_end[k] = min(un.khi, max(0, min(un.L, un.L - un.qlen + i + 1)));
        } else {
          vis_end[k] = 0;
        }
      }
      float qk_scale = p.softmax_scale * kLog2e;
      float v_mul = 1.f;
      if constexpr (FP8) {
        const int sidx = p.scale_mode == PKV_SCALE_HEAD ? un.g : 0;
        qk_scale *= __ldg(p.k_scale + sidx);
        v_mul = __ldg(p.v_scale + sidx);
      }
      const int kc0 = (p.k_off - lo) * C::ESZ / 16;  // first K piece in the span
      const int vc0 = (p.v_off - lo) * C::ESZ / 16;
      const int vcol0 = wig * C::DVS;

      float o[C::NT][4];
#pragma unroll
      for (int nt = 0; nt < C::NT; ++nt) o[nt][0] = o[nt][1] = o[nt][2] = o[nt][3] = 0.f;
      float m_run[2] = {-INFINITY, -INFINITY};
      float l_run[2] = {0.f, 0.f};

      // Chunk c (counted over all units) belongs to group c % NG, and
      // NSLOT % NG == 0, so a ring slot is only ever consumed by one group,
      // in order: when a group waits for chunk c, the slot's previous chunk
      // c - NSLOT was its own and has completed, and the parity wait cannot
      // be satisfied by the phase of chunk c - 2 * NSLOT.
      const int k_first = static_cast<int>((grp + NG - static_cast<int>(gc % NG)) % NG);
      for (int k = k_first; k < un.nch; k += NG) {
        const uint32_t c = gc + k;
        const uint32_t slot = c % NSLOT;
        const uint32_t st = sbase + C::RING_OFF + slot * C::SLOT_BYTES;
        wait_all(slot_full(slot), (c / NSLOT) & 1u);
        const int kb = un.klo + k * 16;
        if (kb + 16 > un.kmax) {
          // rows past the last visible key: zero them before anyone reads
          const int r0 = un.kmax - kb;
          const int n = (16 - r0) * C::NBOX * 8;
          for (int i = wig * 32 + lane; i < n; i += 32 * WG) {
            const int row = r0 + i / (C::NBOX * 8);
            const int piece = i % (C::NBOX * 8);
            asm volatile("st.shared.v4.u32 [%0], {%1,%1,%1,%1};\n" ::"r"(
                             slot_piece(st, row, piece)),
                         "r"(0u)
                         : "memory");
          }
          tc5::fence_proxy_async_smem();
          group_sync();
        }

        // ---- S = Q K^T over this warp's K slice (two n8 tiles of keys) ----
        float s[2][4];
#pragma unroll
        for (int t = 0; t < 2; ++t) s[t][0] = s[t][1] = s[t][2] = s[t][3] = 0.f;
        if constexpr (!FP8) {
          float s2[2][4];
#pragma unroll
          for (int t = 0; t < 2; ++t) s2[t][0] = s2[t][1] = s2[t][2] = s2[t][3] = 0.f;
#pragma unroll
          for (int kk = 0; kk < C::KSW; ++kk) {
            const int ks = wig * C::KSW + kk;
            const int m = lane >> 3;
            const int row = (m >> 1) * 8 + (lane & 7);
            uint32_t kf[4];
            ldmatrix_x4(kf, slot_piece(st, row, kc0 + ks * 2 + (m & 1)));
            // two accumulator chains per tile for more independent MMAs
            if (kk & 1) {
              mma_16816<false>(s2[0], qa[kk], kf[0], kf[1]);
              mma_16816<false>(s2[1], qa[kk], kf[2], kf[3]);
            } else {
              mma_16816<false>(s[0], qa[kk], kf[0], kf[1]);
              mma_16816<false>(s[1], qa[kk], kf[2], kf[3]);
            }
          }
#pragma unroll
          for (int t = 0; t < 2; ++t)
#pragma unroll
            for (int e = 0; e < 4; ++e) s[t][e] += s2[t][e];
        } else {
#pragma unroll
          for (int uu = 0; uu < C::UPW; ++uu) {
            const int un_ = wig + uu * WG;
            if (un_ < C::NU) {
#pragma unroll
              for (int t = 0; t < 2; ++t) {
                const uint4 kw = lds128(slot_piece(st, 8 * t + gr, kc0 + 4 * un_ + qd));
                const uint32_t wv[4] = {kw.x, kw.y, kw.z, kw.w};
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                  const uint32_t a[4] = {qa[uu][2 * j], qa[uu][8 + 2 * j],
                                         qa[uu][2 * j + 1], qa[uu][8 + 2 * j + 1]};
                  mma_16816<true>(s[t], a, e4m3x2_to_f16x2(static_cast<uint16_t>(wv[j])),
                                  e4m3x2_to_f16x2(static_cast<uint16_t>(wv[j] >> 16)));
                }
              }
            }
          }
        }
        if constexpr (WG > 1) {  // sum the K-slice partial scores of the group
          const int buf = xk & 1u;
          float* mine = sbuf + (buf * WG + wig) * 32 * 8 + lane * 8;
          *reinterpret_cast<float4*>(mine) = make_float4(s[0][0], s[0][1], s[0][2], s[0][3]);
          *reinterpret_cast<float4*>(mine + 4) = make_float4(s[1][0], s[1][1], s[1][2], s[1][3]);
          group_sync();
#pragma unroll
          for (int t = 0; t < 2; ++t) s[t][0] = s[t][1] = s[t][2] = s[t][3] = 0.f;
#pragma unroll
          for (int w2 = 0; w2 < WG; ++w2) {
            const float* src = sbuf + (buf * WG + w2) * 32 * 8 + lane * 8;
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
            const int kr = e >> 1;
            const float v = key < vis_end[kr] ? s[t][e] * qk_scale : -INFINITY;
            s[t][e] = v;
            cmax[kr] = fmaxf(cmax[kr], v);
          }
        float alpha[2], base[2];
#pragma unroll
        for (int kr = 0; kr < 2; ++kr) {
          cmax[kr] = fmaxf(cmax[kr], __shfl_xor_sync(0xffffffffu, cmax[kr], 1));
          cmax[kr] = fmaxf(cmax[kr], __shfl_xor_sync(0xffffffffu, cmax[kr], 2));
          const float mn = fmaxf(m_run[kr], cmax[kr]);
          base[kr] = mn == -INFINITY ? 0.f : mn;
          alpha[kr] = fast_exp2(m_run[kr] - base[kr]);
          m_run[kr] = mn;
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
        for (int kr = 0; kr < 2; ++kr) l_run[kr] = l_run[kr] * alpha[kr] + psum[kr];
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
        if constexpr (!FP8) {
#pragma unroll
          for (int np = 0; np < C::NT / 2; ++np) {
            const int m = lane >> 3;
            const int row = (m & 1) * 8 + (lane & 7);
            uint32_t r[4];
            ldmatrix_x4_trans(r, slot_piece(st, row, vc0 + (vcol0 + 16 * np) / 8 + (m >> 1)));
            mma_16816<false>(o[2 * np], pa, r[0], r[1]);
            mma_16816<false>(o[2 * np + 1], pa, r[2], r[3]);
          }
        } else {
#pragma unroll
          for (int vb = 0; vb < C::DVS / 128; ++vb) {
            const int piece = vc0 + (vcol0 + 128 * vb) / 16 + gr;
            const int rows[4] = {2 * qd, 2 * qd + 1, 2 * qd + 8, 2 * qd + 9};
            uint32_t kw[4][4];
#pragma unroll
            for (int k4 = 0; k4 < 4; ++k4) {
              const uint4 v = lds128(slot_piece(st, rows[k4], piece));
              kw[k4][0] = v.x; kw[k4][1] = v.y; kw[k4][2] = v.z; kw[k4][3] = v.w;
            }
#pragma unroll
            for (int j = 0; j < 16; ++j) {
              const int wd = j >> 2, sel = j & 3;
              const uint32_t b0 = e4m3x2_to_f16x2(pick_bytes(kw[0][wd], kw[1][wd], sel));
              const uint32_t b1 = e4m3x2_to_f16x2(pick_bytes(kw[2][wd], kw[3][wd], sel));
              mma_16816<true>(o[16 * vb + j], pa, b0, b1);
            }
          }
        }
        __syncwarp();
        if (lane == 0) tc5::mbar_arrive(slot_empty(slot));
        ++xk;
      }
      gc += un.nch;
#pragma unroll
      for (int kr = 0; kr < 2; ++kr) {
        l_run[kr] += __shfl_xor_sync(0xffffffffu, l_run[kr], 1);
        l_run[kr] += __shfl_xor_sync(0xffffffffu, l_run[kr], 2);
      }
      auto col_of = [&](int nt, int e) {
        if constexpr (!FP8)
          return vcol0 + 8 * nt + 2 * qd + e;
        else
          return vcol0 + 128 * (nt / 16) + 16 * (2 * qd + e) + (nt % 16);
      };

      if constexpr (NG == 1) {
        // one group: every warp writes its own V columns of the partial
#pragma unroll
        for (int kr = 0; kr < 2; ++kr) {
          const int r = gr + 8 * kr;
          if (r >= un.nrows) continue;
          const int rr = un.row0 + r;
          const int64_t t = un.qs + rr / G;
          const int h = un.g * G + rr % G;
          const int64_t orow = (un.s * T + t) * p.num_q_heads + h;
          if (l_run[kr] > 0.f) {
            const float inv = v_mul / l_run[kr];
            float* dst = p.partial_o + orow * C::DV;
#pragma unroll
            for (int nt = 0; nt < C::NT; ++nt)
#pragma unroll
              for (int e = 0; e < 2; ++e) dst[col_of(nt, e)] = o[nt][2 * kr + e] * inv;
          }
          if (wig == 0 && qd == 0)
            p.partial_lse[orow] =
                l_run[kr] > 0.f ? (m_run[kr] + fast_log2(l_run[kr])) * kLn2 : -INFINITY;
        }
      } else {
        // ---- merge the groups through shared memory ----
        float* so = reinterpret_cast<float*>(smem + C::MERGE_OFF);  // [NG][16][DVP]
        float* sm = so + NG * 16 * C::DVP;                          // [NG][16]
        float* sl = sm + NG * 16;                                   // [NG][16]
        named_barrier(1, 32 * C::NCW);  // previous unit's merge reads done
#pragma unroll
        for (int nt = 0; nt < C::NT; ++nt)
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            so[(grp * 16 + gr) * C::DVP + col_of(nt, e)] = o[nt][e];
            so[(grp * 16 + gr + 8) * C::DVP + col_of(nt, e)] = o[nt][2 + e];
          }
        if (wig == 0 && qd == 0) {
          sm[grp * 16 + gr] = m_run[0];
          sm[grp * 16 + gr + 8] = m_run[1];
          sl[grp * 16 + gr] = l_run[0];
          sl[grp * 16 + gr + 8] = l_run[1];
        }
        named_barrier(1, 32 * C::NCW);
        for (int idx = ctid; idx < un.nrows * C::DV; idx += 32 * C::NCW) {
          const int r = idx / C::DV;
          const int cc = idx - r * C::DV;
          const int rr = un.row0 + r;
          const int64_t t = un.qs + rr / G;
          const int h = un.g * G + rr % G;
          float M = -INFINITY;
#pragma unroll
          for (int q = 0; q < NG; ++q) M = fmaxf(M, sm[q * 16 + r]);
          const int64_t orow = (un.s * T + t) * p.num_q_heads + h;
          if (M == -INFINITY) {
            if (cc == 0) p.partial_lse[orow] = -INFINITY;
            continue;
          }
          float lsum = 0.f, acc = 0.f;
#pragma unroll
          for (int q = 0; q < NG; ++q) {
            const float mq = sm[q * 16 + r];
            if (mq == -INFINITY) continue;
            const float wq = fast_exp2(mq - M);
            lsum += wq * sl[q * 16 + r];
            acc += wq * so[(q * 16 + r) * C::DVP + cc];
          }
          p.partial_o[orow * C::DV + cc] = acc / lsum * v_mul;
          if (cc == 0) p.partial_lse[orow] = (M + fast_log2(lsum)) * kLn2;
        }
      }
    }
  }
}

template <class C>
cudaError_t launch_cfg(const AttnParams& p, int num_sms, cudaStream_t stream) {
  static int attr_set[64] = {0};
  cudaError_t e = ensure_smem_attr(decode_kernel<C>, C::SMEM, attr_set);
  if (e != cudaSuccess) return e;
  alignas(64) CUtensorMap kv_map;
  const int box_rows = p.block_size < 16 ? p.block_size : 16;
  if (!make_cache_tmap(&kv_map, p.cache, p.dtype, p.layout, p.num_blocks,
                       p.block_size, p.num_kv_heads, p.row_elems, C::BOX_COLS,
                       box_rows))
    return cudaErrorInvalidValue;
  const int64_t RG = (static_cast<int64_t>(p.max_query_len) * p.group + 15) / 16;
  const int64_t units = static_cast<int64_t>(p.num_splits) * p.num_seqs * p.num_kv_heads * RG;
  const int grid = static_cast<int>(units < num_sms ? units : num_sms);
  decode_kernel<C><<<grid, C::THREADS, C::SMEM, stream>>>(kv_map, p);
  return cudaGetLastError();
}

// <DK, DV, fp8, warps per group, groups, ring slots, unit slots, staged span>
using CfgBf16_192 = DecodeCfg<192, 128, false, 1, 6, 12, 4, 320>;
using CfgFp8_192 = DecodeCfg<192, 128, true, 1, 6, 18, 4, 320>;
using CfgBf16_576 = DecodeCfg<576, 512, false, 4, 1, 7, 3, 576>;
using CfgFp8_576 = DecodeCfg<576, 512, true, 4, 1, 12, 3, 576>;

}  // namespace

bool decode_supported(int head_size, int head_size_v, int dtype) {
  (void)dtype;
  return (head_size == 192 && head_size_v == 128) ||
         (head_size == 576 && head_size_v == 512);
}

cudaError_t launch_decode(const AttnParams& p, int num_sms, cudaStream_t stream) {
  const bool fp8 = p.dtype == PKV_FP8_E4M3;
  if (p.head_size == 192 && p.head_size_v == 128)
    return fp8 ? launch_cfg<CfgFp8_192>(p, num_sms, stream)
               : launch_cfg<CfgBf16_192>(p, num_sms, stream);
  if (p.head_size == 576 && p.head_size_v == 512)
    return fp8 ? launch_cfg<CfgFp8_576>(p, num_sms, stream)
               : launch_cfg<CfgBf16_576>(p, num_sms, stream);
  return cudaErrorNotSupported;
}

}  // namespace pkv
