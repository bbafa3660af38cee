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
//  * Work unit = (split, sequence, block of HPC KV heads, 16-row group); a
//    row is a (query token, query head) pair of one KV head, so a 1+3-token
//    verify with G = 4 is one m16 tile per head.  Persistent CTAs (one per
//    SM) take units in alternating directions and keep streaming across unit
//    boundaries.
//  * Warp 0 is the producer: it stages each unit's query rows (cp.async,
//    completion on an mbarrier), page ids and a descriptor ahead of use, and
//    streams chunks of KPC keys x HPC heads into a ring with TMA boxes of up
//    to KPC rows x 128 bytes of one page and head (128-byte swizzle, columns
//    past the row read as zero), the boxes of a chunk issued by parallel
//    lanes.  Measured on GB300, the rate at which one SM can bring in pages
//    is set by the number of boxes and of chunk handshakes per byte, not by
//    DRAM: 10 KB chunks (16 keys of one head) top out near 3.1 TB/s, 40 KB
//    chunks (16 keys of four heads, or 64 keys of one) reach 6.6-7.3 TB/s.
//    So a chunk holds four heads where Hkv allows, or more keys per head.
//  * Consumer warps form groups of WG warps: group (h, n) handles head h of
//    the block in every chunk c with c % NG == n.  The ring has a multiple
//    of NG slots, so a slot is only consumed by the groups of one n, in fill
//    order (no mbarrier phase can be mistaken for the one two fills later).
//    Within a group, warp w owns a slice of the K dimension for Q.K^T
//    (partial scores summed through shared memory when WG > 1) and a slice
//    of V's columns for P.V.  16 rows are below tcgen05's M = 64, and the
//    FP8 operands are converted in registers, so the contraction runs on the
//    warp-level m16n8k16 MMA (~4-32 flop per byte here).
//  * bf16 cache: K and V fragments come from ldmatrix (.trans for V) on the
//    swizzled slot.  fp8 cache in the warp-MMA form (V before K in the row):
//    E4M3 codes become f16 in registers (exact), K through 16-byte loads with
//    the reduction index permuted identically in Q and K, V by byte-permuting
//    four keys' 16-column runs into k-pairs; the MMA runs in f16 with Q
//    converted bf16 -> f16; k_scale is folded into the softmax scale and
//    v_scale into the output.
//  * fp8 cache, K192 / V128 with K first: the tensor-core form (its branch
//    of the kernel describes it): 128-key chunks of one head; S^T = K Q^T on
//    tcgen05's 8-bit path with Q split exactly into two E4M3 terms, O^T +=
//    V^T P^T in f16, both accumulators in TMEM.
//  * Online softmax in registers with exp2.  The last chunk of a unit has its
//    rows past the last visible key zeroed in shared memory, so garbage in a
//    partly filled page cannot reach the MMA; the scores of those keys are
//    masked.  When NG > 1 the groups of a head combine (max, sum, O) in
//    registers through shared memory at the end of a unit.
//  * Every mbarrier wait is bounded; after a timeout the kernel records
//    PKV_EDEV_TIMEOUT, the waits of all roles return at once, every warp
//    still walks the same units (so named barriers stay matched), and the
//    producer waits (bounded) for its own copies before exit.
#include <math.h>

#include "common.cuh"
#include "kernels.h"
#include "pdl.cuh"
#include "tc5.cuh"
#include "tmap.h"

namespace pkv {

namespace {

template <int DK_, int DV_, bool FP8_, int HPC_, int WG_, int NG_, int KPC_,
          int NSLOT_, int NQ_, int SPAN_, bool NARROW_ = false, int CTAS_ = 1,
          bool TC_ = false>
struct DecodeCfg {
  static constexpr int CTAS = CTAS_;  // CTAs per SM
  // tensor-core form (fp8 cache, one head, 128-key chunks): one MMA-issuing
  // warp and four softmax warps, one key per thread; S^T and O^T in TMEM
  static constexpr bool TC = TC_;
  static constexpr int DK = DK_, DV = DV_, HPC = HPC_, WG = WG_, NG = NG_;
  static constexpr int KPC = KPC_, NSLOT = NSLOT_, NQ = NQ_, SPAN = SPAN_;
  // narrow: a head's rows fit in 8 and the MMAs run transposed (S^T = K Q^T)
  static constexpr bool NARROW = NARROW_;
  static constexpr int QROWS = NARROW ? 8 : 16;           // staged Q rows per head
  static constexpr int MAXP = 128;  // page ids staged with a unit
  static constexpr bool FP8 = FP8_;
  static constexpr int ESZ = FP8 ? 1 : 2;
  static constexpr int SPAN_BYTES = SPAN * ESZ;
  static constexpr int NBOX = (SPAN_BYTES + 127) / 128;  // 128-byte column boxes
  static constexpr int BOX_COLS = 128 / ESZ;
  // A ring slot is [column box][head][KPC rows][128 bytes]: one head's rows
  // of a 128-byte column slice are contiguous (CB_BYTES), the HPC heads of a
  // slice are adjacent (CB_STRIDE) so that one TMA box can bring them all.
  static constexpr int CB_BYTES = KPC * 128;
  static constexpr int CB_STRIDE = HPC * CB_BYTES;
  // tensor-core form: the third column box is 64 bytes wide (span bytes
  // 256..319, 64-byte swizzle), so a slot holds no padding
  static constexpr int SLOT_BYTES = TC ? 2 * CB_STRIDE + KPC * 64 : NBOX * CB_STRIDE;
  // bytes a chunk's boxes bring per key row of one head
  static constexpr int ROW_BYTES = TC ? 320 : NBOX * 128;
  static constexpr int NGRP = HPC * NG;                  // consumer groups
  static constexpr int SXW = TC ? 8 : 0;                 // softmax warps (TC)
  static constexpr int NCW = TC ? SXW + 1 : NGRP * WG;   // consumer warps
  // threads of the fused merge at the end of a unit
  static constexpr int FIN_THREADS = TC ? 32 * SXW : 32 * NCW;
  // arrivals that free a ring slot / a Q slot
  static constexpr int SLOT_EMPTY_N = TC ? SXW + 1 : HPC * WG;
  static constexpr int Q_EMPTY_N = TC ? SXW + 1 : NCW;
  static constexpr int THREADS = 32 * (1 + NCW);
  static constexpr int QCH = DK * 2 / 16;                // 16-byte Q pieces per row
  static constexpr int QH_BYTES = QROWS * DK * 2;        // one head's Q rows
  static constexpr int Q_BYTES = HPC * QH_BYTES;
  static constexpr int KSTEPS = DK / 16;
  // bf16: k-steps per warp, at most (warp w takes [w*KSTEPS/WG, (w+1)*KSTEPS/WG))
  static constexpr int KSW = (KSTEPS + WG - 1) / WG;
  static constexpr int NU = DK / 64;                       // fp8: 64-wide units
  static constexpr int UPW = (NU + WG - 1) / WG;
  static constexpr int DVS = DV / WG;                      // V columns per warp
  static constexpr int NT = DVS / 8;
  static constexpr int DVP = DV + 4;
  static constexpr int RING_OFF = 0;
  // tensor-core form: V converted to f16 ([64-column slab][KPC keys][128 B],
  // 128-byte swizzle) twice, P^T in f16 ([64-key atom][16 rows][128 B])
  // twice, and Q as two E4M3 terms stacked as 32 rows ([128-column atom][hi
  // rows 0..15, lo rows 16..31][128 B]) once
  static constexpr int V16_OFF = RING_OFF + NSLOT * SLOT_BYTES;
  static constexpr int V16_BYTES = TC ? (DV / 64) * KPC * 128 : 0;
  static constexpr int PT_OFF = V16_OFF + 2 * V16_BYTES;
  static constexpr int PT_BYTES = TC ? (KPC / 64) * 16 * 128 : 0;
  static constexpr int Q8_OFF = PT_OFF + 2 * PT_BYTES;
  static constexpr int Q8_BYTES = TC ? ((DK + 127) / 128) * 32 * 128 : 0;
  static constexpr int Q_OFF = Q8_OFF + Q8_BYTES;
  static constexpr int DESC_OFF = Q_OFF + NQ * Q_BYTES;
  static constexpr int DESC_BYTES = 64 + MAXP * 4;  // descriptor + page ids
  // Descriptor slots: two at least, so that staging unit n+1 (while unit n
  // is issued from its page list) never overwrites unit n's.
  static constexpr int ND = NQ > 2 ? NQ : 2;
  static constexpr int MAXSORT = 128;  // sequences ranked by length, at most
  static_assert(MAXSORT == kBalancedMaxSeqs, "balanced ranges take the ranked batch size");
  // the sequences' ranking (equal segments) or, for balanced ranges, every
  // sequence's first global page (MAXSORT + 1 entries, the last = all pages)
  static constexpr int ORDER_OFF = DESC_OFF + ND * DESC_BYTES;
  static constexpr int ORDER_BYTES = ((MAXSORT + 1) * 4 + 15) / 16 * 16;
  static constexpr int MERGE_OFF = ORDER_OFF + ORDER_BYTES;
  // every chunk class's (O, max, sum) per head and row, combined by all
  static constexpr int MROW = DVP + 2;
  static constexpr int MERGE = NG > 1 ? NG * HPC * 16 * MROW * 4 : 0;
  static constexpr int SBUF_OFF = MERGE_OFF + MERGE;
  static constexpr int SBUF_LANE = NARROW ? 4 : 8;  // partial scores per lane
  static constexpr int SBUF = WG > 1 ? NGRP * 2 * WG * 32 * SBUF_LANE * 4 : 0;
  // Fused merge: per (head, row) weights of up to kFusedMaxSplits splits and
  // a flag; it reuses the score-exchange or class-merge buffer (idle at the
  // end of a unit) when one is large enough.
  static constexpr int WBUF = HPC * 16 * kFusedMaxSplits * 4 + 16;
  static constexpr int WBUF_OFF = SBUF >= WBUF ? SBUF_OFF : MERGE >= WBUF ? MERGE_OFF
                                                                          : SBUF_OFF + SBUF;
  static constexpr int BAR_OFF = (SBUF >= WBUF || MERGE >= WBUF) ? SBUF_OFF + SBUF
                                                                 : SBUF_OFF + SBUF + WBUF;
  // tensor-core form: s_full[2], s_free[2], p_full[2], pv_done[2],
  // q8_full (+1 spare), and the MMA warp's drain barrier; then scratch:
  // per-row Q scales [2][16], the row reductions [4 warps][16], the row
  // sums [16] and the TMEM address
  static constexpr int NBAR_TC = TC ? 11 : 0;
  static constexpr int NBAR = 2 * NSLOT + 2 * NQ + NBAR_TC;
  static constexpr int TCS_OFF = BAR_OFF + NBAR * 8 + 16;
  static constexpr int TCS_BYTES = TC ? (2 * 16 + 4 * 16 + 16 + 4) * 4 : 0;
  static constexpr int SMEM = TCS_OFF + TCS_BYTES + 1024;
  static_assert(DK % 64 == 0, "K in 64-column units");
  // (also reads the warp-MMA form's sizes, which the other forms leave unused)
  static_assert(NU >= 1 && UPW >= 1 && NT >= 1, "warp-MMA form sizes");
  static_assert(DV % WG == 0 && DVS % (FP8 ? 128 : 16) == 0, "V slices");
  static_assert(QCH % 8 == 0, "Q rows in whole 128-byte groups");
  static_assert(KPC % 16 == 0 && KPC <= 256, "keys per chunk");
  static_assert(SMEM * CTAS <= 227 * 1024, "shared memory budget");
  static_assert(NSLOT % NG == 0, "each ring slot belongs to one chunk class");
  static_assert(NGRP + 2 <= 15, "named barrier ids");
  static_assert(!TC || (FP8 && HPC == 1 && NG == 1 && WG == 1 && KPC == 128 && DK == 192 &&
                         DV == 128 && !NARROW && CTAS == 1),
                "tensor-core form: fp8, one head, 128-key chunks, K 192 / V 128");
  static_assert(!NARROW || (!FP8 && NG == 1 && KSTEPS % WG == 0 && KSW % 2 == 0 &&
                             DVS % 16 == 0),
                "narrow form: bf16, one chunk class, k-step pairs, 16-column V tiles");
};

// Address of the 16-byte piece `piece` (byte offset / 16 within the staged
// span) of key row `row` of one head's part of a ring slot (`sub` = the slot
// + head * CB_BYTES): column slice piece/8 is CB_STRIDE further on, holding
// the head's rows x 128 bytes, and the 128-byte swizzle permutes 16-byte
// pieces by the row index.
template <int CB_STRIDE>
__device__ __forceinline__ uint32_t slot_piece(uint32_t sub, int row, int piece) {
  return sub + (piece >> 3) * CB_STRIDE + row * 128 + (((piece & 7) ^ (row & 7)) << 4);
}

// Transposes an 8x8 matrix of 16-bit values held in the MMA fragment layout
// (thread t: row t/4, columns 2(t%4) and 2(t%4)+1).
__device__ __forceinline__ uint32_t movmatrix_trans(uint32_t a) {
  uint32_t d;
  asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;\n" : "=r"(d) : "r"(a));
  return d;
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

// Rows of one TMA box: the largest power of two <= kpc that divides the
// block size, so that a chunk's boxes tile it and none straddles a page.
__host__ __device__ constexpr int box_rows_for(int bs, int kpc) {
  int r = kpc;
  while (r > 1 && bs % r != 0) r >>= 1;
  return r;
}

// A work unit; the producer stages it in shared memory as 16 ints followed
// by its page ids.
struct Unit {
  int b, hb, s, row0, nrows, qs, qlen, L;
  // nseg: the segments of the unit's sequence that units write (balanced
  // ranges; the fused merge counts to it), 0 for equal segments
  int klo, khi, kmax, nch, page_lo, npages, nseg, pad1;
};
static_assert(sizeof(Unit) == 64, "descriptor size");

// Units are numbered sequence-major, longest sequence first (when the
// sequences were ranked), then over (split, row group, head block); the
// CTAs take them in rounds, alternately forwards and backwards, so that
// every CTA's share of keys is about the same.
struct UnitShape {
  int S, HB, RG;  // splits, head blocks per sequence, 16-row groups per head
  __device__ int per_seq() const { return S * RG * HB; }
};

// A unit's parameters from its sequence b (query_start_loc pair q0, q1 and
// length L), head block, row group, segment s and the segment's pages
// [page_lo, page_hi) in the sequence's own page numbers.
template <int KPC>
__device__ __forceinline__ void unit_params_pages(const AttnParams& p, int b, int hb, int rg,
                                                  int s, int q0, int q1, int L, int page_lo,
                                                  int page_hi, Unit& un) {
  const int G = p.group;
  un.b = b;
  un.hb = hb;
  un.s = s;
  un.qs = q0;
  un.qlen = q1 - q0;
  un.L = L;
  un.row0 = rg * 16;
  un.nrows = max(0, min(16, un.qlen * G - un.row0));
  const int bs = p.block_size;
  un.klo = page_lo * bs;
  un.khi = min(page_hi * bs, un.L);
  un.kmax = un.klo;
  if (un.nrows > 0) {
    // the unit's last row belongs to its latest query token: it sees most
    const int i_last = (un.row0 + un.nrows - 1) / G;
    un.kmax = min(un.khi, max(0, min(un.L, un.L - un.qlen + i_last + 1)));
  }
  un.nch = un.kmax > un.klo ? (un.kmax - un.klo + KPC - 1) / KPC : 0;
  un.page_lo = page_lo;
  un.npages = page_hi - page_lo;
  un.nseg = un.pad1 = 0;
}

// Unit u's parameters under equal segments, for sequence b (the rank-u /
// per_seq sequence) with its query_start_loc pair and length: segment s of
// the sequence's P pages is [s * pps, min((s + 1) * pps, P)), pps =
// ceil(P / num_splits).
template <int KPC>
__device__ __forceinline__ void unit_params(const AttnParams& p, UnitShape us, int u, int b,
                                            int q0, int q1, int L, Unit& un) {
  const int rem = u % us.per_seq();
  const int hb = rem % us.HB;
  const int rg = (rem / us.HB) % us.RG;
  const int s = rem / (us.HB * us.RG);
  const int P = (L + p.block_size - 1) / p.block_size;
  const int pps = (P + p.num_splits - 1) / p.num_splits;
  const int page_lo = min(s * pps, P);
  const int page_hi = min(page_lo + pps, P);
  unit_params_pages<KPC>(p, b, hb, rg, s, q0, q1, L, page_lo, page_hi, un);
}

// The end of a unit in the fused decode, run by every consumer thread of
// the CTA (ctid = its index among them) once the unit's partials are
// written.  The unit counts itself done; the last unit of its (sequence,
// KV-head block, row group) merges the segments of its rows as
// pkv_splitkv_reduce does and puts the counter back to zero.  Ordering: a
// barrier, then one thread's fence before its atomic, publishes the CTA's
// partial writes; the last unit fences after its atomic and reads the
// partials with L1-bypassing loads.
template <class C>
__device__ __forceinline__ void fused_finish(const AttnParams& p, const Unit& un, int HB,
                                             int RG, uint8_t* smem, int ctid) {
  constexpr int NT = C::FIN_THREADS;
  float* wb = reinterpret_cast<float*>(smem + C::WBUF_OFF);
  volatile int* flag =
      reinterpret_cast<volatile int*>(smem + C::WBUF_OFF + C::HPC * 16 * kFusedMaxSplits * 4);
  // units that write the rows: every split (equal segments), or the
  // sequence's ranges (balanced)
  const int S = un.nseg > 0 ? un.nseg : p.num_splits;
  named_barrier(1, NT);  // the unit's partials are written
  if (ctid == 0) {
    __threadfence();
    const int key = (un.b * HB + un.hb) * RG + un.row0 / 16;
    const int last = atomicAdd(p.counters + key, 1) == S - 1;
    if (last) {
      p.counters[key] = 0;  // zero again for the next call
      __threadfence();
    }
    *flag = last;
  }
  named_barrier(1, NT);
  if (!*flag) return;
  const int64_t TH = static_cast<int64_t>(p.num_tokens) * p.num_q_heads;
  const int G = p.group;
  const int nr = C::HPC * un.nrows;
  auto row_of = [&](int h, int r) {
    const int rr = un.row0 + r;
    return (static_cast<int64_t>(un.qs) + rr / G) * p.num_q_heads + (un.hb * C::HPC + h) * G +
           rr % G;
  };
  // per row: the segments' weights exp(lse_s - M) / sum, and the merged lse
  for (int i = ctid; i < nr; i += NT) {
    const int h = i / un.nrows, r = i - h * un.nrows;
    const int64_t row = row_of(h, r);
    float* w = wb + i * kFusedMaxSplits;
    float M = -INFINITY;
    for (int s = 0; s < S; ++s) M = fmaxf(M, __ldcg(p.partial_lse + s * TH + row));
    if (M == -INFINITY) {  // no segment saw a key: 0, never NaN
      for (int s = 0; s < S; ++s) w[s] = 0.f;
      if (p.lse_out != nullptr) p.lse_out[row] = -INFINITY;
      continue;
    }
    const float Ml2 = M * kLog2e;
    float W = 0.f;
    for (int s = 0; s < S; ++s) {
      const float x = __ldcg(p.partial_lse + s * TH + row);
      const float e = x == -INFINITY ? 0.f : fast_exp2(fmaf(x, kLog2e, -Ml2));
      w[s] = e;
      W += e;
    }
    const float inv = 1.f / W;
    for (int s = 0; s < S; ++s) w[s] *= inv;
    if (p.lse_out != nullptr) p.lse_out[row] = M + fast_log2(W) * kLn2;
  }
  named_barrier(1, NT);
  constexpr int DV4 = C::DV / 4;
  for (int i = ctid; i < nr * DV4; i += NT) {
    const int hr = i / DV4, c4 = i - hr * DV4;
    const int h = hr / un.nrows, r = hr - h * un.nrows;
    const int64_t row = row_of(h, r);
    const float* w = wb + hr * kFusedMaxSplits;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int s = 0; s < S; ++s) {
      const float ws = w[s];
      if (ws == 0.f) continue;  // an empty segment's partial is not read
      const float4 v =
          __ldcg(reinterpret_cast<const float4*>(p.partial_o + (s * TH + row) * C::DV) + c4);
      acc.x = fmaf(ws, v.x, acc.x);
      acc.y = fmaf(ws, v.y, acc.y);
      acc.z = fmaf(ws, v.z, acc.z);
      acc.w = fmaf(ws, v.w, acc.w);
    }
    *reinterpret_cast<uint2*>(p.out + row * C::DV + 4 * c4) =
        make_uint2(pack_bf16x2(acc.x, acc.y), pack_bf16x2(acc.z, acc.w));
  }
  named_barrier(1, NT);  // the weights are read before the buffer is reused
}

// BAL: 0 equal segments; 1 balanced ranges (split_ranges > 0) over at most
// MAXSORT sequences; 2 balanced ranges over more (a window of sequences).
// Each unit list is its own instantiation, so that the code of one does not
// weigh on another's (the window's bookkeeping slowed the headline batch by
// 15 % when it was compiled into the same kernel).
template <class C, int BAL>
__global__ void __launch_bounds__(C::THREADS, C::CTAS)
    decode_kernel(const __grid_constant__ CUtensorMap kv_map,
                  const __grid_constant__ CUtensorMap kv_map64, const AttnParams p,
                  int head_boxes) {
  // the next kernel of the step may start launching; nothing here (TMEM
  // included) is touched before the kernel ahead has completed
  pdl_trigger();
  pdl_wait();
  extern __shared__ uint8_t smem_raw[];
  constexpr bool FP8 = C::FP8;
  constexpr int HPC = C::HPC, WG = C::WG, NG = C::NG, KPC = C::KPC, NSLOT = C::NSLOT;
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
  const UnitShape us{p.num_splits, p.num_kv_heads / HPC, (p.max_query_len * G + 15) / 16};
  const int num_units = p.num_seqs * us.per_seq();
  const int bs = p.block_size;
  const int box_rows = box_rows_for(bs, KPC);
  const int nrb = KPC / box_rows;  // row boxes per column box of a chunk
  const int lo = min(p.k_off, p.v_off);
  const int64_t T = p.num_tokens;

  if (threadIdx.x == 0) {
    for (int i = 0; i < NSLOT; ++i) {
      tc5::mbar_init(slot_full(i), 1);
      tc5::mbar_init(slot_empty(i), C::SLOT_EMPTY_N);  // every warp of one chunk class
    }
    for (int i = 0; i < C::NQ; ++i) {
      tc5::mbar_init(q_full(i), 1);
      tc5::mbar_init(q_empty(i), C::Q_EMPTY_N);
    }
    if constexpr (C::TC) {
      const int tcb = 2 * NSLOT + 2 * C::NQ;
      for (int i = 0; i < 2; ++i) {
        tc5::mbar_init(bar0 + 8u * (tcb + i), 1);      // s_full: MMA commit
        tc5::mbar_init(bar0 + 8u * (tcb + 2 + i), C::SXW);  // s_free: softmax warps
        tc5::mbar_init(bar0 + 8u * (tcb + 4 + i), C::SXW);  // p_full: softmax warps
        tc5::mbar_init(bar0 + 8u * (tcb + 6 + i), 1);       // pv_done: MMA commit
        tc5::mbar_init(bar0 + 8u * (tcb + 8 + i), C::SXW);  // q8_full: softmax warps
      }
      tc5::mbar_init(bar0 + 8u * (tcb + 10), 1);       // the MMA warp's drain
    }
    *abort_flag = 0;
    tc5::fence_mbar_init();
    tc5::prefetch_tmap(&kv_map);
    if constexpr (C::TC) tc5::prefetch_tmap(&kv_map64);
  }
  if constexpr (C::TC) {
    if (warp == C::SXW + 1) {  // 128 columns: S^T twice (32 each) and O^T (16)
      tc5::tmem_alloc(sbase + C::TCS_OFF + (2 * 16 + 4 * 16 + 16) * 4, 128);
      tc5::tmem_relinquish();
    }
  }
  // Q slots start as zeros: a unit stages only its valid rows, and the rows
  // past them (masked, never written out) only need to be finite.
  for (int i = threadIdx.x; i < C::NQ * C::Q_BYTES / 16; i += C::THREADS)
    reinterpret_cast<uint4*>(smem + C::Q_OFF)[i] = make_uint4(0, 0, 0, 0);
  __syncthreads();
  if constexpr (C::TC) tc5::tc_fence_after();

  if (warp == 0) {
    // ------------------------------------------------ producer warp -----
    // Units are staged two ahead of the one whose chunks are being issued:
    // the unit's query rows, its page ids (block-table entries, copied
    // asynchronously) and a descriptor go to one of NQ slots, so that no
    // block-table or sequence-metadata read sits in front of a copy.
    uint32_t gc = 0;    // chunks issued
    uint32_t qs_n = 0;  // units staged
    uint32_t qi_n = 0;  // units issued
    // the k-th unit of this CTA: rounds of gridDim.x units, dealt forwards
    // and backwards in turn
    auto unit_at = [&](int k) {
      const int r = (k & 1) ? static_cast<int>(gridDim.x - 1 - blockIdx.x)
                            : static_cast<int>(blockIdx.x);
      return k * static_cast<int>(gridDim.x) + r;
    };
    // Balanced ranges (split_ranges = W > 0, at most MAXSORT sequences): the
    // pages of all sequences laid end to end in sequence order, sequence b
    // from global page gst[b], cut into ranges of R pages.  A work item is
    // (range, head block); this CTA takes items blockIdx.x, blockIdx.x +
    // gridDim.x, ..., and a unit is one (piece of a sequence inside the
    // item's range, the item's head block, row group).  Items of one range
    // sit next to each other, so the CTAs that read the different heads of
    // the same pages run side by side.
    constexpr bool balanced = BAL != 0;
    int* gst = reinterpret_cast<int*>(smem + C::ORDER_OFF);  // [MAXSORT + 1]
    // query_start_loc[b] and seq_lens[b] of the lane registers (b uniform
    // over the warp; b == num_seqs gives the last query_start_loc entry)
    int L4_[4], Q4_[4], qend_ = 0;
    auto pick4 = [&](const int (&a)[4], int b) {
      const int t = b & 3;
      const int v = t == 0 ? a[0] : t == 1 ? a[1] : t == 2 ? a[2] : a[3];
      return __shfl_sync(0xffffffffu, v, (b >> 2) & 31);
    };
    auto seq_q = [&](int b) { return b >= p.num_seqs ? qend_ : pick4(Q4_, b); };
    auto seq_L = [&](int b) { return pick4(L4_, b); };
    int64_t bR = 1;     // pages per range
    int bnr = 0;        // ranges that hold pages
    // lane l holds the lengths and first query tokens of sequences 4l ..
    // 4l + 3 (balanced ranges), read with the lengths, so that no later
    // metadata read stands between the lengths and the first copy
    int (&L4)[4] = L4_;
    int (&Q4)[4] = Q4_;
    int& qend = qend_;
    L4[0] = L4[1] = L4[2] = L4[3] = 0;
    Q4[0] = Q4[1] = Q4[2] = Q4[3] = 0;
    // A batch of more than MAXSORT sequences (BAL == 2) holds a window
    // instead: the MAXSORT sequences of chunk wc (lane l: MAXSORT wc + 4l ..
    // + 3) with their first global pages in G4, gst[] then holding every
    // chunk's first global page and qend the first query token after the
    // window.
    int G4[4] = {0, 0, 0, 0};
    const int nb = p.num_seqs;
    constexpr bool wide = BAL == 2;
    constexpr int WIN = C::MAXSORT;
    const int nch = (nb + WIN - 1) / WIN;  // chunks (wide)
    int wc = -1;                           // the window's chunk (wide)
    auto npages = [&](int L) { return L > 0 ? (L + bs - 1) / bs : 0; };
    // the window of chunk c (warp-uniform c): lengths, first query tokens,
    // first global pages (gst[c] plus a warp scan inside the chunk)
    auto load_window = [&](int c) {
      wc = c;
      int lsum = 0;
#pragma unroll
      for (int t = 0; t < 4; ++t) {
        const int i = WIN * c + 4 * lane + t;
        L4[t] = i < nb ? __ldg(p.seq_lens + i) : 0;
        Q4[t] = i < nb ? __ldg(p.query_start_loc + i) : 0;
      }
      qend = __ldg(p.query_start_loc + min(WIN * c + WIN, nb));
#pragma unroll
      for (int t = 0; t < 4; ++t) lsum += npages(L4[t]);
      int incl = lsum;
#pragma unroll
      for (int d = 1; d < 32; d <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, incl, d);
        if (lane >= d) incl += y;
      }
      int g = gst[c] + incl - lsum;
#pragma unroll
      for (int t = 0; t < 4; ++t) {
        G4[t] = g;
        g += npages(L4[t]);
      }
    };
    // sequence b's first global page (0 <= b <= num_seqs; wide: b in the
    // window or the first sequence after it), length and first query token
    // (b == num_seqs, or past the window: the next first query token); b is
    // uniform over the warp
    auto gstart = [&](int b) -> int {
      if (!wide) return gst[b];
      const int i = b - WIN * wc;
      return (i >= WIN || b >= nb) ? gst[wc + 1] : pick4(G4, i);
    };
    auto seq_Lb = [&](int b) { return wide ? pick4(L4_, b - WIN * wc) : seq_L(b); };
    auto seq_qb = [&](int b) {
      if (!wide) return seq_q(b);
      const int i = b - WIN * wc;
      return (i >= WIN || b >= nb) ? qend_ : pick4(Q4_, i);
    };
    if constexpr (!wide) {
      if (balanced) {
        // lane l takes sequences 4l .. 4l + 3: their page counts, then a warp
        // scan of the lanes' sums gives every sequence's first global page
        const int nb = p.num_seqs;
        int P4[4], lsum = 0, lmax = 0;
        qend = __ldg(p.query_start_loc + nb);
#pragma unroll
        for (int t = 0; t < 4; ++t) {
          const int i = 4 * lane + t;
          L4[t] = i < nb ? __ldg(p.seq_lens + i) : 0;
          Q4[t] = i < nb ? __ldg(p.query_start_loc + i) : 0;
        }
#pragma unroll
        for (int t = 0; t < 4; ++t) {
          const int L = L4[t];
          P4[t] = L > 0 ? (L + bs - 1) / bs : 0;
          lsum += P4[t];
          lmax = max(lmax, P4[t]);
        }
        int incl = lsum;
#pragma unroll
        for (int d = 1; d < 32; d <<= 1) {
          const int y = __shfl_up_sync(0xffffffffu, incl, d);
          if (lane >= d) incl += y;
        }
        int g = incl - lsum;
#pragma unroll
        for (int t = 0; t < 4; ++t) {
          const int i = 4 * lane + t;
          if (i <= nb) gst[i] = g;
          g += P4[t];
        }
        if (lane == 31 && nb == C::MAXSORT) gst[nb] = g;  // the entry past a full batch
#pragma unroll
        for (int d = 16; d > 0; d >>= 1) lmax = max(lmax, __shfl_xor_sync(0xffffffffu, lmax, d));
        const int64_t Ptot = __shfl_sync(0xffffffffu, incl, 31);
        __syncwarp();
        // R = max(ceil(Ptot / W), Rmin, 1): Rmin keeps every sequence within
        // num_splits segments (one of P >= 2 pages meets at most
        // floor((P - 2) / R) + 2 ranges)
        const int64_t Rmin = p.num_splits == 1 ? Ptot
                                               : (lmax > 2 ? lmax - 2 : 0) / (p.num_splits - 1) + 1;
        bR = max(max((Ptot + p.split_ranges - 1) / p.split_ranges, Rmin), int64_t{1});
        bnr = static_cast<int>((Ptot + bR - 1) / bR);
        // segments past a sequence's last range hold no key: their lse is
        // -inf, written here for the sequences b = blockIdx.x (mod gridDim.x)
        for (int b = blockIdx.x; b < nb; b += gridDim.x) {
          const int nseg = gst[b + 1] > gst[b]
                               ? static_cast<int>((gst[b + 1] - 1) / bR - gst[b] / bR + 1)
                               : 0;
          const int q0 = seq_q(b);
          const int rows = (seq_q(b + 1) - q0) * p.num_q_heads;
          const int n = (p.num_splits - nseg) * rows;
          for (int i = lane; i < n; i += 32) {
            const int sg = nseg + i / rows, rr = i - (i / rows) * rows;
            p.partial_lse[(static_cast<int64_t>(sg) * T + q0) * p.num_q_heads + rr] = -INFINITY;
          }
          // fused merge: a sequence without keys has no unit to merge its
          // rows, so they are written here (0, lse -inf)
          if (p.fused && nseg == 0) {
            for (int i = lane; i < rows * (C::DV / 2); i += 32) {
              const int rr = i / (C::DV / 2), c2 = i - rr * (C::DV / 2);
              reinterpret_cast<uint32_t*>(p.out + (static_cast<int64_t>(q0) * p.num_q_heads + rr) *
                                                      C::DV)[c2] = 0u;
            }
            if (p.lse_out != nullptr)
              for (int i = lane; i < rows; i += 32)
                p.lse_out[static_cast<int64_t>(q0) * p.num_q_heads + i] = -INFINITY;
          }
        }
      }
    } else {
      if (balanced) {
        // every chunk's page count (the next chunk's lengths in flight while
        // one is summed): gst[c] = the chunk's first global page
        int lmax = 0;
        int cur[4], run = 0;
#pragma unroll
        for (int t = 0; t < 4; ++t) {
          const int i = 4 * lane + t;
          cur[t] = i < nb ? __ldg(p.seq_lens + i) : 0;
        }
        for (int c = 0; c < nch; ++c) {
          int nxt[4];
#pragma unroll
          for (int t = 0; t < 4; ++t) {
            const int i = WIN * (c + 1) + 4 * lane + t;
            nxt[t] = i < nb ? __ldg(p.seq_lens + i) : 0;
          }
          int sum = 0;
#pragma unroll
          for (int t = 0; t < 4; ++t) {
            const int P = npages(cur[t]);
            sum += P;
            lmax = max(lmax, P);
          }
#pragma unroll
          for (int d = 16; d > 0; d >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, d);
          if (lane == 0) gst[c] = run;
          run += sum;
#pragma unroll
          for (int t = 0; t < 4; ++t) cur[t] = nxt[t];
        }
        if (lane == 0) gst[nch] = run;
        const int64_t Ptot = run;
#pragma unroll
        for (int d = 16; d > 0; d >>= 1) lmax = max(lmax, __shfl_xor_sync(0xffffffffu, lmax, d));
        __syncwarp();
        // R = max(ceil(Ptot / W), Rmin, 1): Rmin keeps every sequence within
        // num_splits segments (one of P >= 2 pages meets at most
        // floor((P - 2) / R) + 2 ranges)
        const int64_t Rmin = p.num_splits == 1 ? Ptot
                                               : (lmax > 2 ? lmax - 2 : 0) / (p.num_splits - 1) + 1;
        bR = max(max((Ptot + p.split_ranges - 1) / p.split_ranges, Rmin), int64_t{1});
        bnr = static_cast<int>((Ptot + bR - 1) / bR);
        // segments past a sequence's last range hold no key: their lse is
        // -inf, written here for this CTA's block of consecutive sequences
        auto fill_seq = [&](int b) {
          const int g0 = gstart(b), g1 = gstart(b + 1);
          const int nseg = g1 > g0 ? static_cast<int>((g1 - 1) / bR - g0 / bR + 1) : 0;
          const int q0 = seq_qb(b);
          const int rows = (seq_qb(b + 1) - q0) * p.num_q_heads;
          const int n = (p.num_splits - nseg) * rows;
          for (int i = lane; i < n; i += 32) {
            const int sg = nseg + i / rows, rr = i - (i / rows) * rows;
            p.partial_lse[(static_cast<int64_t>(sg) * T + q0) * p.num_q_heads + rr] = -INFINITY;
          }
          // fused merge: a sequence without keys has no unit to merge its
          // rows, so they are written here (0, lse -inf)
          if (p.fused && nseg == 0) {
            for (int i = lane; i < rows * (C::DV / 2); i += 32) {
              const int rr = i / (C::DV / 2), c2 = i - rr * (C::DV / 2);
              reinterpret_cast<uint32_t*>(p.out + (static_cast<int64_t>(q0) * p.num_q_heads + rr) *
                                                      C::DV)[c2] = 0u;
            }
            if (p.lse_out != nullptr)
              for (int i = lane; i < rows; i += 32)
                p.lse_out[static_cast<int64_t>(q0) * p.num_q_heads + i] = -INFINITY;
          }
        };
        const int per = (nb + static_cast<int>(gridDim.x) - 1) / static_cast<int>(gridDim.x);
        const int b0 = static_cast<int>(blockIdx.x) * per, b1 = min(b0 + per, nb);
        for (int b = b0; b < b1; ++b) {
          if (b == b0 || b % WIN == 0) load_window(b / WIN);
          fill_seq(b);
        }
      }
    }
    // work item, sequence, row group of the piece, the piece's pages
    int bi = blockIdx.x, bb = -1, bj = 0, bplo = 0, bphi = 0;
    int bL = 0, bq0 = 0, bq1 = 0;  // the piece's sequence: length, query_start_loc pair
    // wide: the window that holds sequence b (warp-uniform b < num_seqs)
    auto window_for = [&](int b) {
      if (wide && b < nb && b / WIN != wc) load_window(b / WIN);
    };
    // moves (bi, bb) to the next piece of a sequence inside the range of one
    // of this CTA's items; false when there is none
    auto next_piece = [&]() -> bool {
      if constexpr (!wide) {
        for (;;) {
          if (bi >= bnr * us.HB) return false;
          const int64_t r0 = static_cast<int64_t>(bi / us.HB) * bR;
          const int64_t r1 = r0 + bR;
          if (bb < 0) {  // the sequence holding global page r0: gst[bb] <= r0 < gst[bb + 1]
            int lo = 0, hi = p.num_seqs - 1;
            while (lo < hi) {
              const int mid = (lo + hi) >> 1;
              if (gst[mid + 1] > r0) hi = mid; else lo = mid + 1;
            }
            bb = lo;
          } else {
            ++bb;
          }
          while (bb < p.num_seqs && gst[bb + 1] == gst[bb]) ++bb;  // no pages
          if (bb < p.num_seqs && gst[bb] < r1) {
            bplo = static_cast<int>(max(static_cast<int64_t>(gst[bb]), r0) - gst[bb]);
            bphi = static_cast<int>(min(static_cast<int64_t>(gst[bb + 1]), r1) - gst[bb]);
            bj = 0;
            bL = seq_L(bb);
            bq0 = seq_q(bb);
            bq1 = seq_q(bb + 1);
            return true;
          }
          bi += gridDim.x;
          bb = -1;
        }
      } else {
        for (;;) {
          if (bi >= bnr * us.HB) return false;
          const int64_t r0 = static_cast<int64_t>(bi / us.HB) * bR;
          const int64_t r1 = r0 + bR;
          if (bb < 0) {
            // the chunk holding global page r0, then the one sequence of its
            // window with pages around r0
            int lo = 0, hi = nch - 1;
            while (lo < hi) {
              const int mid = (lo + hi) >> 1;
              if (gst[mid + 1] > r0) hi = mid; else lo = mid + 1;
            }
            if (lo != wc) load_window(lo);
            int hit = -1;
#pragma unroll
            for (int t = 0; t < 4; ++t) {
              const int i = WIN * lo + 4 * lane + t;
              const int P = npages(L4[t]);
              if (i < nb && P > 0 && G4[t] <= r0 && r0 < G4[t] + P) hit = i;
            }
            const unsigned m = __ballot_sync(0xffffffffu, hit >= 0);
            bb = m ? __shfl_sync(0xffffffffu, hit, __ffs(m) - 1) : nb;
          } else {
            ++bb;
            window_for(bb);
          }
          while (bb < nb && gstart(bb + 1) == gstart(bb)) {  // no pages
            ++bb;
            window_for(bb);
          }
          if (bb < nb && gstart(bb) < r1) {
            const int g0 = gstart(bb), g1 = gstart(bb + 1);
            bplo = static_cast<int>(max(static_cast<int64_t>(g0), r0) - g0);
            bphi = static_cast<int>(min(static_cast<int64_t>(g1), r1) - g0);
            bj = 0;
            bL = seq_Lb(bb);
            bq0 = seq_qb(bb);
            bq1 = seq_qb(bb + 1);
            return true;
          }
          bi += gridDim.x;
          bb = -1;
        }
      }
    };
    bool bpiece = balanced && next_piece();
    // Sequences ranked by decreasing length (ties by index) when there are
    // few enough to rank here; otherwise in their own order.
    int* order = reinterpret_cast<int*>(smem + C::ORDER_OFF);
    const bool ranked = !balanced && p.num_seqs <= C::MAXSORT;
    if (ranked) {
      // lane l holds the lengths of sequences l, l + 32, l + 64, l + 96 and
      // counts, for each, the sequences that come before it
      static_assert(C::MAXSORT == 128, "four sequences per lane");
      const int nb = p.num_seqs, nu = (nb + 31) / 32;
      int v[4], rank[4];
      // the query_start_loc entries come with the lengths (lane l: sequences
      // l, l + 32, l + 64, l + 96, and the last entry), so that the first
      // unit's metadata needs no read of its own
      qend_ = __ldg(p.query_start_loc + nb);
#pragma unroll
      for (int t = 0; t < 4; ++t) {
        const int i = lane + 32 * t;
        v[t] = i < nb ? __ldg(p.seq_lens + i) : 0;
        Q4_[t] = i < nb ? __ldg(p.query_start_loc + i) : 0;
        L4_[t] = v[t];
        rank[t] = 0;
      }
      for (int u = 0; u < nu; ++u) {
        const int vu = u == 0 ? v[0] : u == 1 ? v[1] : u == 2 ? v[2] : v[3];
        for (int src = 0; src < 32; ++src) {
          const int lj = __shfl_sync(0xffffffffu, vu, src);
          const int j = src + 32 * u;
#pragma unroll
          for (int t = 0; t < 4; ++t) {
            const int i = lane + 32 * t;
            rank[t] += (j < nb) && (lj > v[t] || (lj == v[t] && j < i));
          }
        }
      }
#pragma unroll
      for (int t = 0; t < 4; ++t)
        if (lane + 32 * t < nb) order[rank[t]] = lane + 32 * t;
      __syncwarp();
    }
    auto seq_of = [&](int u) {
      const int r = u / us.per_seq();
      return ranked ? order[r] : r;
    };
    int pos = 0;                   // next position in this CTA's unit list
    int mb = 0, mq0 = 0, mq1 = 0, mL = 0;  // metadata of the unit at `pos`
    // sequence b's entry of a ranked batch's lane registers (lane b % 32,
    // register b / 32; b uniform over the warp)
    auto pick32 = [&](const int (&a)[4], int b) {
      const int t = (b >> 5) & 3;
      const int x = t == 0 ? a[0] : t == 1 ? a[1] : t == 2 ? a[2] : a[3];
      return __shfl_sync(0xffffffffu, x, b & 31);
    };
    auto meta_load = [&](int ps) {
      const int u = unit_at(ps);
      if (u < num_units) {
        mb = seq_of(u);
        if (ranked) {
          mq0 = pick32(Q4_, mb);
          mq1 = mb + 1 < p.num_seqs ? pick32(Q4_, mb + 1) : qend_;
          mL = pick32(L4_, mb);
        } else {
          mq0 = __ldg(p.query_start_loc + mb);
          mq1 = __ldg(p.query_start_loc + mb + 1);
          mL = __ldg(p.seq_lens + mb);
        }
      }
    };
    if (!balanced) meta_load(0);
    // the next unit of this CTA's list into `un`; false at the end
    auto next_unit = [&](Unit& un) -> bool {
      if (balanced) {
        if (!bpiece) return false;
        const int b = bb;
        const int g0 = gstart(b), g1 = gstart(b + 1);
        unit_params_pages<KPC>(p, b, bi % us.HB, bj, static_cast<int>(bi / us.HB - g0 / bR), bq0,
                               bq1, bL, bplo, bphi, un);
        un.nseg = static_cast<int>((g1 - 1) / bR - g0 / bR + 1);
        if (++bj == us.RG) bpiece = next_piece();
        if (un.s >= p.num_splits) {  // excluded by R >= Rmin; never written past the partials
          set_dev_error(p.err, PKV_EDEV_RANGE);
          un.nrows = 0;
        }
        return true;
      }
      if (unit_at(pos) >= num_units) return false;
      unit_params<KPC>(p, us, unit_at(pos), mb, mq0, mq1, mL, un);
      ++pos;
      meta_load(pos);  // the next unit's metadata is in flight meanwhile
      return true;
    };
    bool alive = true;
    auto stage_next = [&]() {
      Unit un;
      while (next_unit(un)) {
        if (un.nrows == 0) continue;
        if (un.nch == 0 && !p.fused) {  // no key of this segment is visible to any row
          for (int i = lane; i < HPC * un.nrows; i += 32) {
            const int h = i / un.nrows, r = i - h * un.nrows;
            const int rr = un.row0 + r;
            const int64_t t = un.qs + rr / G;
            const int qh = (un.hb * HPC + h) * G + rr % G;
            p.partial_lse[(un.s * T + t) * p.num_q_heads + qh] = -INFINITY;
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
        const int qn = min(un.nrows, C::QROWS) * C::QCH;  // pieces of one head's valid rows
        for (int i = lane; i < HPC * qn; i += 32) {
          const int h = i / qn, rj = i - h * qn;
          const int r = rj / C::QCH, j = rj - r * C::QCH;
          const int rr = un.row0 + r;
          const int64_t t = un.qs + rr / G;
          const int qh = (un.hb * HPC + h) * G + rr % G;
          cp_async_16(q_piece<C::DK>(qdst + h * C::QH_BYTES, r, j),
                      p.q + (t * p.num_q_heads + qh) * C::DK + j * 8, 16);
        }
        const int np = min(un.npages, C::MAXP);
        const int32_t* bt = p.block_table +
                            static_cast<int64_t>(un.b) * p.max_blocks_per_seq + un.page_lo;
        const uint32_t dslot = qs_n % C::ND;
        const uint32_t pdst = sbase + C::DESC_OFF + dslot * C::DESC_BYTES + 64;
        for (int i = lane; i < np; i += 32) cp_async_4(pdst + 4 * i, bt + i);
        if (lane == 0) *desc_of(dslot) = un;
        cp_async_commit();
        ++qs_n;
        return;
      }
    };
    // One unit is staged ahead: the next unit is staged while the ring is
    // full of the current one's chunks, so unit boundaries cost no wait.
    stage_next();
    while (alive && qi_n < qs_n) {
      const uint32_t qslot = qi_n % C::NQ;
      cp_async_wait<0>();  // this unit's rows and page ids (staged last)
      __syncwarp();
      if (lane == 0) tc5::mbar_arrive(q_full(qslot));
      const Unit un = *desc_of(qi_n % C::ND);
      const int* pages = pages_of(qi_n % C::ND);
      const int32_t* bt = p.block_table + static_cast<int64_t>(un.b) * p.max_blocks_per_seq;
      const int k_stage = min(un.nch, NSLOT) - 1;  // stage the next unit after this chunk
      for (int k = 0; k < un.nch; ++k) {
        const uint32_t slot = gc % NSLOT;
        bool w = true;
        if (lane == 0)
          w = tc5::mbar_wait(slot_empty(slot), ((gc / NSLOT) & 1u) ^ 1u, abort_flag, p.err);
        if (!__shfl_sync(0xffffffffu, w, 0)) {
          alive = false;
          break;
        }
        // the chunk's boxes, issued by parallel lanes: with head boxes one
        // per column slice (HPC heads x KPC rows), else one per head, column
        // slice and row box that holds visible keys
        const int kb = un.klo + k * KPC;
        const int nvr = min(nrb, (un.kmax - kb + box_rows - 1) / box_rows);
        const int per_head = C::NBOX * nvr;
        if (lane == 0)
          tc5::mbar_arrive_expect_tx(slot_full(slot),
                                     static_cast<uint32_t>(HPC * nvr * box_rows * C::ROW_BYTES));
        __syncwarp();
        const uint32_t st = sbase + C::RING_OFF + slot * C::SLOT_BYTES;
        const int nboxes = head_boxes ? C::NBOX : HPC * per_head;
        for (int i = lane; i < nboxes; i += 32) {
          const int h = head_boxes ? 0 : i / per_head;
          const int rem = head_boxes ? i : i - h * per_head;
          const int rb = rem / C::NBOX, cb = rem - rb * C::NBOX;
          const int key0 = kb + rb * box_rows;
          const int pidx = key0 / bs - un.page_lo;
          int page = pidx < C::MAXP ? pages[pidx] : __ldg(bt + key0 / bs);
          if (page < 0 || page >= p.num_blocks) {
            set_dev_error(p.err, PKV_EDEV_RANGE);
            page = p.num_blocks;  // out-of-range box: TMA fills zeros
          }
          const uint32_t dst = st + cb * C::CB_STRIDE + h * C::CB_BYTES +
                               rb * box_rows * (C::TC && cb == 2 ? 64 : 128);
          const int col = lo + cb * C::BOX_COLS;
          const int head = un.hb * HPC + h;
          if (C::TC && cb == 2) {  // the 64-byte third box
            if (p.layout == PKV_NHD)
              tc5::tma_load_4d(dst, &kv_map64, col, head, key0 % bs, page, slot_full(slot));
            else
              tc5::tma_load_4d(dst, &kv_map64, col, key0 % bs, head, page, slot_full(slot));
          } else if (head_boxes)  // (col, slot, head, page) in both layouts
            tc5::tma_load_4d(dst, &kv_map, col, key0 % bs, head, page, slot_full(slot));
          else if (p.layout == PKV_NHD)
            tc5::tma_load_4d(dst, &kv_map, col, head, key0 % bs, page, slot_full(slot));
          else
            tc5::tma_load_4d(dst, &kv_map, col, key0 % bs, head, page, slot_full(slot));
        }
        ++gc;
        if (k == k_stage && alive) stage_next();
      }
      // a unit without chunks (an empty segment staged for the fused merge)
      // stages the next one here
      if (alive && qs_n == qi_n + 1) stage_next();
      ++qi_n;
    }
    if (alive) {  // end marker for the consumers
      const uint32_t qslot = qs_n % C::NQ;
      bool w = true;
      if (lane == 0) {
        w = tc5::mbar_wait(q_empty(qslot), ((qs_n / C::NQ) & 1u) ^ 1u, abort_flag, p.err);
        if (w) {
          desc_of(qs_n % C::ND)->nch = -1;
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
  } else if constexpr (C::TC) {
    // ------------------------------ tensor-core form (fp8 cache) --------
    // Warps 1..SXW (softmax warps): warp w covers keys 32 (w % 4) .. + 31 of
    // every chunk -- TMEM lanes 32 (w % 4) .. + 31 of S^T, the lane quarter
    // the warp may touch -- and half hf = (w - 1) / 4 of the work on them:
    // query rows 8 hf .. 8 hf + 7 (S^T columns) and V columns 64 hf .. + 63.
    // Per chunk a thread scales and masks its key's scores, turns them into
    // f16 probabilities P^T in shared memory, and converts its key's V
    // columns from E4M3 to f16.  At the end of a unit it owns V column
    // 32 (w % 4) + lane of O^T for its 8 rows.  Warp SXW + 1 issues every
    // MMA: S^T = K Q^T on the 8-bit path straight from the ring (Q split
    // exactly into two E4M3 terms, stacked as N = 32: S^T columns 0..15 are
    // the hi products, 16..31 the lo ones), and O^T += V^T P^T in f16.
    constexpr int KCH = C::KPC;         // keys per chunk: the M of S^T
    constexpr int SXW = C::SXW;
    constexpr int NH = SXW / 4;         // halves of a key's work
    constexpr int RPT = 16 / NH;        // query rows per thread
    constexpr int VPT = C::DV / NH;     // V columns per thread
    constexpr int NSX = 32 * SXW;       // softmax threads
    constexpr int TCB = 2 * NSLOT + 2 * C::NQ;
    auto s_full = [&](uint32_t i) { return bar0 + 8u * (TCB + i); };
    auto s_free = [&](uint32_t i) { return bar0 + 8u * (TCB + 2 + i); };
    auto p_full = [&](uint32_t i) { return bar0 + 8u * (TCB + 4 + i); };
    auto pv_done = [&](uint32_t i) { return bar0 + 8u * (TCB + 6 + i); };
    auto q8_full = [&](uint32_t i) { return bar0 + 8u * (TCB + 8 + i); };
    const uint32_t fin_bar = bar0 + 8u * (TCB + 10);
    float* qscale = reinterpret_cast<float*>(smem + C::TCS_OFF);  // [2][16]
    float* red = qscale + 32;                                      // [4][16]
    float* lsum = red + 64;                                        // [16]
    const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(lsum + 16);
    auto v16_buf = [&](uint32_t i) { return sbase + C::V16_OFF + i * C::V16_BYTES; };
    auto pt_buf = [&](uint32_t i) { return sbase + C::PT_OFF + i * C::PT_BYTES; };
    const uint32_t q8 = sbase + C::Q8_OFF;
    constexpr uint32_t TM_O = 64;  // O^T columns; S^T buffers (32 wide) at 0 and 32
    if (warp == SXW + 1) {
      // ---------------------------------------------------- MMA warp ----
      if (lane == 0) {
        constexpr uint32_t ID_S = tc5::idesc_e4m3_f32(KCH, 32);
        constexpr uint32_t ID_PV = tc5::idesc_f16_f32(C::DV, 16, /*a_mn=*/true, false);
        uint32_t gc = 0, qc = 0;
        bool ok = true;
        for (;;) {
          const uint32_t qslot = qc % C::NQ;
          if (!tc5::mbar_wait(q_full(qslot), (qc / C::NQ) & 1u, abort_flag, p.err)) break;
          const Unit un = *desc_of(qc % C::ND);
          tc5::mbar_arrive(q_empty(qslot));
          const uint32_t u = qc++;
          if (un.nch < 0 || *abort_flag) break;
          if (!tc5::mbar_wait(q8_full(0), u & 1u, abort_flag, p.err)) break;
          for (int k = 0; k <= un.nch && ok; ++k) {
            if (k < un.nch) {  // S^T(c) = K(c) [Q_hi; Q_lo]^T, 6 k-steps of 32
              const uint32_t c = gc + k;
              const uint32_t slot = c % NSLOT;
              ok = tc5::mbar_wait(slot_full(slot), (c / NSLOT) & 1u, abort_flag, p.err) &&
                   tc5::mbar_wait(s_free(c & 1u), ((c >> 1) & 1u) ^ 1u, abort_flag, p.err);
              if (!ok) break;
              tc5::tc_fence_after();
              const uint32_t st = sbase + C::RING_OFF + slot * C::SLOT_BYTES;
#pragma unroll
              for (int ks = 0; ks < C::DK / 32; ++ks)
                tc5::mma_f8f6f4_ss(
                    tmem + 32u * (c & 1u),
                    tc5::sdesc_sw128(st + (ks >> 2) * C::CB_STRIDE + (ks & 3) * 32, 16, 1024),
                    tc5::sdesc_sw128(q8 + (ks >> 2) * 4096 + (ks & 3) * 32, 16, 1024), ID_S,
                    ks ? 1u : 0u);
              tc5::mma_commit(s_full(c & 1u));
              tc5::mma_commit(slot_empty(slot));
            }
            if (k > 0) {  // O^T += V^T(c-1) P^T(c-1), 16 keys per MMA
              const uint32_t c = gc + k - 1;
              ok = tc5::mbar_wait(p_full(c & 1u), (c >> 1) & 1u, abort_flag, p.err);
              if (!ok) break;
              tc5::tc_fence_after();
              const uint32_t pb = pt_buf(c & 1u);
              const uint32_t vb = v16_buf(c & 1u);
#pragma unroll
              for (int kk = 0; kk < KCH / 16; ++kk)
                tc5::mma_f16_ss(tmem + TM_O,
                                tc5::sdesc_sw128(vb + kk * 2048, KCH * 128, 1024),
                                tc5::sdesc_sw128(pb + (kk >> 2) * 2048 + (kk & 3) * 32, 16, 1024),
                                ID_PV, (k > 1 || kk > 0) ? 1u : 0u);
              tc5::mma_commit(pv_done(c & 1u));
            }
          }
          if (!ok) break;
          gc += un.nch;
        }
        // every MMA issued above has completed before TMEM is freed
        tc5::mma_commit(fin_bar);
        tc5::mbar_wait(fin_bar, 0, abort_flag, p.err, /*honor_abort=*/false);
      }
      __syncwarp();
    } else {
      // ------------------------------------------------ softmax warps ----
      constexpr float kTau = 8.f;  // P <= 2^8 between max updates (log2 units)
      const int quad = warp & 3;
      const int hf = (warp - 1) / 4;
      const int r0 = RPT * hf;            // my first query row
      const int kk = 32 * quad + lane;    // my key of a chunk / my column of O^T
      const int sxid = threadIdx.x - 32;
      const uint32_t tl = tmem + (static_cast<uint32_t>(32 * quad) << 16);
      const int vbyte0 = p.v_off - lo;    // V's first byte in the staged span
      uint32_t gc = 0, qc = 0;
      // reduce-scatter of RPT per-row values over the warp (max or sum): the
      // lane ends with row r0 + (lane / (32 / RPT)) over the warp's 32 keys
      auto warp_rows = [&](float (&v)[RPT], bool is_max) {
#pragma unroll
        for (int h = RPT / 2; h >= 1; h >>= 1) {
          const int m = (32 / RPT) * h;  // partner lane distance; its bit picks the half kept
          const bool up = (lane & m) != 0;
#pragma unroll
          for (int r = 0; r < h; ++r) {
            const float send = up ? v[r] : v[r + h];
            const float keep = up ? v[r + h] : v[r];
            const float got = __shfl_xor_sync(0xffffffffu, send, m);
            v[r] = is_max ? fmaxf(keep, got) : keep + got;
          }
        }
#pragma unroll
        for (int m = 16 / RPT; m >= 1; m >>= 1) {
          const float got = __shfl_xor_sync(0xffffffffu, v[0], m);
          v[0] = is_max ? fmaxf(v[0], got) : v[0] + got;
        }
        return v[0];
      };
      // The next staged unit: its descriptor, and its Q rows split into the
      // Q buffer with their scales (every S^T MMA of the previous unit has
      // completed: this thread has read all of their results).  False at the
      // end marker or after a timeout, the same in all softmax threads.
      auto fetch = [&](Unit& un, uint32_t& u) -> bool {
        const uint32_t qslot = qc % C::NQ;
        tc5::mbar_wait(q_full(qslot), (qc / C::NQ) & 1u, abort_flag, p.err);
        if (barrier_or(3, NSX, *abort_flag != 0)) return false;
        un = *desc_of(qc % C::ND);
        if (un.nch < 0) return false;
        u = qc++;
        if (sxid < 128) {
          // ---- Q rows -> hi + lo E4M3 terms, scaled by 2^e per row so that
          //      the row's largest |q| lands in [128, 256): for bf16 input the
          //      two terms hold q exactly (hi keeps 4 significant bits, the
          //      remainder has at most 4 more) wherever the remainder is
          //      within E4M3's range ----
          const uint32_t qsrc = sbase + C::Q_OFF + qslot * C::Q_BYTES;
          const int r = sxid >> 3, g = sxid & 7;  // row, piece group of 3 x 8 columns
          float x[24];
          float amax = 0.f;
#pragma unroll
          for (int j = 0; j < 3; ++j) {
            const uint4 v = lds128(q_piece<C::DK>(qsrc, r, g + 8 * j));
            const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
            for (int m = 0; m < 4; ++m) {
              const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w[m]));
              x[8 * j + 2 * m] = f.x;
              x[8 * j + 2 * m + 1] = f.y;
              amax = fmaxf(amax, fmaxf(fabsf(f.x), fabsf(f.y)));
            }
          }
          amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
          amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
          amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 4));
          int e = 0;
          if (amax > 0.f)
            e = min(7 - (static_cast<int>((__float_as_uint(amax) >> 23) & 0xffu) - 127), 126);
          const float sc = __uint_as_float(static_cast<uint32_t>(e + 127) << 23);  // 2^e
          if (g == 0) qscale[(u & 1u) * 16 + r] = __uint_as_float(static_cast<uint32_t>(127 - e) << 23);
          const uint32_t qb = q8;
#pragma unroll
          for (int j = 0; j < 3; ++j) {
            uint32_t hi[2], lo8[2];
#pragma unroll
            for (int m = 0; m < 4; ++m) {
              const float a = x[8 * j + 2 * m] * sc, b = x[8 * j + 2 * m + 1] * sc;
              const uint16_t h = static_cast<uint16_t>(
                  __nv_cvt_float2_to_fp8x2(make_float2(a, b), __NV_SATFINITE, __NV_E4M3));
              const uint32_t hf2 = e4m3x2_to_f16x2(h);
              const float2 hv = __half22float2(*reinterpret_cast<const __half2*>(&hf2));
              const uint16_t l = static_cast<uint16_t>(__nv_cvt_float2_to_fp8x2(
                  make_float2(a - hv.x, b - hv.y), __NV_SATFINITE, __NV_E4M3));
              if (m & 1) {
                hi[m >> 1] |= static_cast<uint32_t>(h) << 16;
                lo8[m >> 1] |= static_cast<uint32_t>(l) << 16;
              } else {
                hi[m >> 1] = h;
                lo8[m >> 1] = l;
              }
            }
            const int d0 = 8 * (g + 8 * j);  // first of this piece's 8 columns
            const uint32_t off = (d0 >> 7) * 4096 + r * 128 +
                                 ((((d0 & 127) >> 4) ^ (r & 7)) << 4) + (d0 & 15);
            asm volatile("st.shared.v2.u32 [%0], {%1,%2};\n" ::"r"(qb + off), "r"(hi[0]),
                         "r"(hi[1]) : "memory");
            asm volatile("st.shared.v2.u32 [%0], {%1,%2};\n" ::"r"(qb + 16 * 128 + off),
                         "r"(lo8[0]), "r"(lo8[1]) : "memory");
          }
          tc5::fence_proxy_async_smem();
        }
        __syncwarp();
        if (lane == 0) {
          tc5::mbar_arrive(q8_full(0));
          tc5::mbar_arrive(q_empty(qslot));
        }
        named_barrier(3, NSX);  // the row scales are visible
        return true;
      };
      Unit un;
      uint32_t u = 0;
      bool have = fetch(un, u);
      while (have) {
        const int kvh = un.hb;
        const int sidx = p.scale_mode == PKV_SCALE_HEAD ? kvh : 0;
        const float base_scale = p.softmax_scale * kLog2e * __ldg(p.k_scale + sidx);
        float qs[RPT], m_ref[RPT], l[RPT];
        int vis[RPT];
#pragma unroll
        for (int j = 0; j < RPT; ++j) {
          const int r = r0 + j;
          qs[j] = base_scale * qscale[(u & 1u) * 16 + r];
          m_ref[j] = -INFINITY;
          l[j] = 0.f;
          vis[j] = 0;
          if (r < un.nrows) {
            const int i = (un.row0 + r) / G;
            vis[j] = min(un.khi, max(0, min(un.L, un.L - un.qlen + i + 1)));
          }
        }
        for (int k = 0; k < un.nch; ++k) {
          const uint32_t c = gc + k;
          const uint32_t slot = c % NSLOT;
          const int key = un.klo + k * KCH + kk;
          // ---- my key's V columns, E4M3 -> f16, into [64-column slab][key]
          //      [128 B] of buffer c % 2 (zeros past the last key any row
          //      sees); its previous user PV(c - 2) has completed, and so has
          //      the P^T buffer's.  The ring slot is released right after. ----
          tc5::mbar_wait(slot_full(slot), (c / NSLOT) & 1u, abort_flag, p.err);
          if (c >= 2) tc5::mbar_wait(pv_done(c & 1u), ((c - 2) >> 1) & 1u, abort_flag, p.err);
          {
            const uint32_t st = sbase + C::RING_OFF + slot * C::SLOT_BYTES;
            const uint32_t vb = v16_buf(c & 1u);
            const bool valid = key < un.kmax;
#pragma unroll
            for (int i = 0; i < VPT / 16; ++i) {
              const int d0 = VPT * hf + 16 * i;  // first of these 16 V columns
              const int byte = vbyte0 + d0;
              uint4 w = make_uint4(0, 0, 0, 0);
              if (valid) {
                uint32_t a;
                if (byte < 256) {  // 128-byte rows, 128-byte swizzle
                  a = st + (byte >> 7) * C::CB_STRIDE + kk * 128 +
                      ((((byte & 127) >> 4) ^ (kk & 7)) << 4);
                } else {  // the third box: 64-byte rows, 64-byte swizzle
                  const uint32_t o = kk * 64 + (byte - 256);
                  a = st + 2 * C::CB_STRIDE + (o ^ (((o >> 7) & 3u) << 4));
                }
                w = lds128(a);
              }
              const uint32_t h[8] = {
                  e4m3x2_to_f16x2(static_cast<uint16_t>(w.x)), e4m3x2_to_f16x2(static_cast<uint16_t>(w.x >> 16)),
                  e4m3x2_to_f16x2(static_cast<uint16_t>(w.y)), e4m3x2_to_f16x2(static_cast<uint16_t>(w.y >> 16)),
                  e4m3x2_to_f16x2(static_cast<uint16_t>(w.z)), e4m3x2_to_f16x2(static_cast<uint16_t>(w.z >> 16)),
                  e4m3x2_to_f16x2(static_cast<uint16_t>(w.w)), e4m3x2_to_f16x2(static_cast<uint16_t>(w.w >> 16))};
              const uint32_t srow = vb + (d0 >> 6) * (KCH * 128) + kk * 128;
              const int pc0 = (d0 & 63) >> 3;
              asm volatile("st.shared.v4.u32 [%0], {%1,%2,%3,%4};\n" ::"r"(srow + ((pc0 ^ (kk & 7)) << 4)),
                           "r"(h[0]), "r"(h[1]), "r"(h[2]), "r"(h[3]) : "memory");
              asm volatile("st.shared.v4.u32 [%0], {%1,%2,%3,%4};\n" ::"r"(srow + (((pc0 + 1) ^ (kk & 7)) << 4)),
                           "r"(h[4]), "r"(h[5]), "r"(h[6]), "r"(h[7]) : "memory");
            }
          }
          __syncwarp();
          if (lane == 0) tc5::mbar_arrive(slot_empty(slot));
          // ---- my key's scores for my rows (log2 domain), masked ----
          tc5::mbar_wait(s_full(c & 1u), (c >> 1) & 1u, abort_flag, p.err);
          tc5::tc_fence_after();
          uint32_t sr[RPT], sl[RPT];
          tc5::tmem_ld_32x32b_x8(tl + 32u * (c & 1u) + r0, sr);
          tc5::tmem_ld_32x32b_x8(tl + 32u * (c & 1u) + 16 + r0, sl);
          tc5::tmem_wait_ld();
          tc5::tc_fence_before();
          __syncwarp();
          if (lane == 0) tc5::mbar_arrive(s_free(c & 1u));
          float x[RPT];
          bool need = false;
#pragma unroll
          for (int j = 0; j < RPT; ++j) {
            x[j] = key < vis[j] ? (__uint_as_float(sr[j]) + __uint_as_float(sl[j])) * qs[j]
                                : -INFINITY;
            need |= x[j] > m_ref[j] + kTau;
          }
          if (barrier_or(3, NSX, need)) {
            // a score passed its row's reference by more than kTau: take the
            // chunk's exact row maxima, move the references up and rescale
            // what was accumulated (O^T in TMEM, this thread's row sums)
            float v[RPT];
#pragma unroll
            for (int j = 0; j < RPT; ++j) v[j] = x[j];
            const float wm = warp_rows(v, true);
            if ((lane & (32 / RPT - 1)) == 0) red[quad * 16 + r0 + lane / (32 / RPT)] = wm;
            named_barrier(3, NSX);
            float alpha[RPT];
            bool rescale = false;
#pragma unroll
            for (int j = 0; j < RPT; ++j) {
              const int r = r0 + j;
              const float cm = fmaxf(fmaxf(red[r], red[16 + r]), fmaxf(red[32 + r], red[48 + r]));
              const float mn = fmaxf(m_ref[j], cm);
              alpha[j] = m_ref[j] == -INFINITY ? 1.f : fast_exp2(m_ref[j] - mn);
              rescale |= alpha[j] != 1.f;
              m_ref[j] = mn;
              l[j] *= alpha[j];
            }
            named_barrier(3, NSX);  // red[] is read before it is written again
            if (k > 0 && rescale) {
              const uint32_t cp = c - 1;
              tc5::mbar_wait(pv_done(cp & 1u), (cp >> 1) & 1u, abort_flag, p.err);
              tc5::tc_fence_after();
              uint32_t o[RPT];
              tc5::tmem_ld_32x32b_x8(tl + TM_O + r0, o);
              tc5::tmem_wait_ld();
#pragma unroll
              for (int j = 0; j < RPT; ++j) o[j] = __float_as_uint(__uint_as_float(o[j]) * alpha[j]);
              tc5::tmem_st_32x32b_x8(tl + TM_O + r0, o);
              tc5::tmem_wait_st();
              tc5::tc_fence_before();
            }
          }
          float pr[RPT];
#pragma unroll
          for (int j = 0; j < RPT; ++j) {
            pr[j] = fast_exp2(x[j] - (m_ref[j] == -INFINITY ? 0.f : m_ref[j]));
            l[j] += pr[j];
          }
          // ---- P^T (f16) for the B operand: [64-key atom][16 rows][128 B];
          //      lane pairs swap values so each store holds two keys.  The
          //      even lane of a pair stores row j, the odd lane row j + 4:
          //      rows 4 apart have complementary swizzled 16-byte chunks, so
          //      the warp's 32 stores hit 32 different banks ----
          {
            static_assert(RPT == 8, "P^T store pairs rows four apart");
            const uint32_t pb = pt_buf(c & 1u);
            const int k0 = kk & ~1;
            const bool odd = lane & 1;
            const uint32_t pbase = pb + (k0 >> 6) * 2048 + (k0 & 7) * 2;
            const int kc = (k0 & 63) >> 3;
#pragma unroll
            for (int j = 0; j < RPT / 2; ++j) {
              const float send = odd ? pr[j] : pr[j + RPT / 2];
              const float recv = __shfl_xor_sync(0xffffffffu, send, 1);
              const int r = r0 + j + (odd ? RPT / 2 : 0);
              const uint32_t val = odd ? pack_f16x2(recv, pr[j + RPT / 2]) : pack_f16x2(pr[j], recv);
              asm volatile("st.shared.b32 [%0], %1;\n" ::"r"(pbase + r * 128 + ((kc ^ (r & 7)) << 4)),
                           "r"(val) : "memory");
            }
          }
          tc5::fence_proxy_async_smem();  // V and P^T -> the tensor core
          __syncwarp();
          if (lane == 0) tc5::mbar_arrive(p_full(c & 1u));
        }
        gc += un.nch;
        // the next unit's Q first, so that its S^T MMAs can start while this
        // unit's last PV drains and its partials are written
        Unit nx;
        uint32_t u_next = 0;
        const bool have_next = fetch(nx, u_next);
        // ---- row sums over all keys of the unit, then the partials ----
        {
          float v[RPT];
#pragma unroll
          for (int j = 0; j < RPT; ++j) v[j] = l[j];
          const float ws = warp_rows(v, false);
          if ((lane & (32 / RPT - 1)) == 0) red[quad * 16 + r0 + lane / (32 / RPT)] = ws;
        }
        named_barrier(3, NSX);
        if (sxid < 16) lsum[sxid] = red[sxid] + red[16 + sxid] + red[32 + sxid] + red[48 + sxid];
        named_barrier(3, NSX);
        float L[RPT];
#pragma unroll
        for (int j = 0; j < RPT; ++j) L[j] = lsum[r0 + j];
        auto orow_of = [&](int r) {
          const int rr = un.row0 + r;
          const int64_t t = un.qs + rr / G;
          return (un.s * T + t) * p.num_q_heads + kvh * G + rr % G;
        };
        if (un.nch > 0) {
          const uint32_t cl = gc - 1;
          tc5::mbar_wait(pv_done(cl & 1u), (cl >> 1) & 1u, abort_flag, p.err);
          tc5::tc_fence_after();
          uint32_t o[RPT];
          tc5::tmem_ld_32x32b_x8(tl + TM_O + r0, o);
          tc5::tmem_wait_ld();
          tc5::tc_fence_before();
          const float vm = __ldg(p.v_scale + sidx);
#pragma unroll
          for (int j = 0; j < RPT; ++j)
            if (r0 + j < un.nrows && L[j] > 0.f)
              p.partial_o[orow_of(r0 + j) * C::DV + kk] = __uint_as_float(o[j]) * (vm / L[j]);
        }
        // the lse of row r: the thread of the first softmax warp's half
        // that holds it (lane r - r0), from its own row references
        if (quad == 1 && lane < RPT && r0 + lane < un.nrows) {
          float mr = 0.f, lr = 0.f;
#pragma unroll
          for (int j = 0; j < RPT; ++j)
            if (j == lane) {
              mr = m_ref[j];
              lr = L[j];
            }
          p.partial_lse[orow_of(r0 + lane)] = lr > 0.f ? (mr + fast_log2(lr)) * kLn2 : -INFINITY;
        }
        if (p.fused) fused_finish<C>(p, un, us.HB, us.RG, smem, sxid);
        un = nx;
        u = u_next;
        have = have_next;
      }
    }
    // TMEM is freed once the MMAs have drained and no warp reads it
    named_barrier(4, 32 * (SXW + 1));
    if (warp == SXW + 1) tc5::tmem_dealloc(tmem, 128);
  } else if constexpr (C::NARROW) {
    // --------------------------------------- consumer warps, narrow form --
    // A head's rows fit in 8 (q_len * G <= 8): S^T = K Q^T with the 16 keys
    // of a step as M and the rows as N = 8, then O^T += V^T P^T with V's
    // columns as M.  Half the MMAs of the row-major form, whose 16-row tiles
    // would be at least half padding; P^T reaches the B operand through two
    // in-register 8x8 transposes.
    const int cw = warp - 1;
    const int grp = cw / WG, wig = cw % WG;
    const int hg = grp;  // one chunk class: group = head of the block
    const int gr = lane >> 2, qd = lane & 3;
    uint32_t gc = 0, qc = 0;
    uint32_t xk = 0;  // 16-key steps processed: picks the exchange buffer
    float* sbuf = reinterpret_cast<float*>(smem + C::SBUF_OFF) + grp * 2 * WG * 32 * 4;
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
    constexpr int MT = C::DVS / 16;  // 16-column V tiles of this warp
    for (;;) {
      const uint32_t qslot = qc % C::NQ;
      wait_all(q_full(qslot), (qc / C::NQ) & 1u);
      // the warps that meet at named barriers take the same decision to stop
      // after a timeout: all consumer warps when units end in the fused
      // merge, else the warps of a group
      if (p.fused) {
        if (barrier_or(15, 32 * C::NCW, *abort_flag != 0)) break;
      } else if constexpr (WG > 1) {
        if (barrier_or(2 + grp, 32 * WG, *abort_flag != 0)) break;
      } else {
        if (__any_sync(0xffffffffu, *abort_flag != 0)) break;
      }
      const Unit un = *desc_of(qc % C::ND);
      if (un.nch < 0) break;
      const int kvh = un.hb * HPC + hg;
      const uint32_t qsrc = sbase + C::Q_OFF + qslot * C::Q_BYTES + hg * C::QH_BYTES;
      // Q^T fragments (B operand) of rows 0..7 over this warp's k-steps
      uint32_t qb[C::KSW][2];
#pragma unroll
      for (int kk = 0; kk < C::KSW; kk += 2) {
        const int ks = wig * C::KSW + kk;
        uint32_t r[4];
        ldmatrix_x4(r, q_piece<C::DK>(qsrc, lane & 7, 2 * ks + (lane >> 3)));
        qb[kk][0] = r[0];
        qb[kk][1] = r[1];
        qb[kk + 1][0] = r[2];
        qb[kk + 1][1] = r[3];
      }
      __syncwarp();
      if (lane == 0) tc5::mbar_arrive(q_empty(qslot));
      ++qc;

      // rows 2qd and 2qd + 1 of this thread: visibility
      int vis_end[2];
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        const int r = 2 * qd + j;
        if (r < un.nrows) {
          const int i = (un.row0 + r) / G;
          vis_end[j] = min(un.khi, max(0, min(un.L, un.L - un.qlen + i + 1)));
        } else {
          vis_end[j] = 0;
        }
      }
      const float qk_scale = p.softmax_scale * kLog2e;
      const int kc0 = (p.k_off - lo) * C::ESZ / 16;
      const int vc0 = (p.v_off - lo) * C::ESZ / 16;
      const int vcol0 = wig * C::DVS;

      float o[MT][4];  // O^T: V columns (gr, gr + 8 of each tile) x rows (2qd, 2qd + 1)
#pragma unroll
      for (int mt = 0; mt < MT; ++mt) o[mt][0] = o[mt][1] = o[mt][2] = o[mt][3] = 0.f;
      float m_run[2] = {-INFINITY, -INFINITY};
      float l_run[2] = {0.f, 0.f};

      for (int k = 0; k < un.nch; ++k) {
        const uint32_t c = gc + k;
        const uint32_t slot = c % NSLOT;
        const uint32_t st = sbase + C::RING_OFF + slot * C::SLOT_BYTES + hg * C::CB_BYTES;
        wait_all(slot_full(slot), (c / NSLOT) & 1u);
        const int kb = un.klo + k * KPC;
        if (kb + KPC > un.kmax) {
          // rows past the last visible key: zero them before anyone reads
          const int r0 = un.kmax - kb;
          const int n = (KPC - r0) * C::NBOX * 8;
          for (int i = wig * 32 + lane; i < n; i += 32 * WG) {
            const int row = r0 + i / (C::NBOX * 8);
            const int piece = i % (C::NBOX * 8);
            asm volatile("st.shared.v4.u32 [%0], {%1,%1,%1,%1};\n" ::"r"(
                             slot_piece<C::CB_STRIDE>(st, row, piece)),
                         "r"(0u)
                         : "memory");
          }
          tc5::fence_proxy_async_smem();
          group_sync();
        }
        const int nsteps = min(KPC / 16, (un.kmax - kb + 15) / 16);
        for (int ks16 = 0; ks16 < nsteps; ++ks16) {
          const int r16 = 16 * ks16;
          const int kb16 = kb + r16;
          // ---- S^T = K Q^T over this warp's K slice ----
          float s[4] = {0.f, 0.f, 0.f, 0.f}, s2[4] = {0.f, 0.f, 0.f, 0.f};
          const int mj = lane >> 3;  // the 8x8 matrix this lane addresses
#pragma unroll
          for (int kk = 0; kk < C::KSW; ++kk) {
            const int ks = wig * C::KSW + kk;
            uint32_t kf[4];
            ldmatrix_x4(kf, slot_piece<C::CB_STRIDE>(st, r16 + (lane & 7) + 8 * (mj & 1),
                                                    kc0 + 2 * ks + (mj >> 1)));
            if (kk & 1)
              mma_16816<false>(s2, kf, qb[kk][0], qb[kk][1]);
            else
              mma_16816<false>(s, kf, qb[kk][0], qb[kk][1]);
          }
#pragma unroll
          for (int e = 0; e < 4; ++e) s[e] += s2[e];
          if constexpr (WG > 1) {  // sum the K-slice partial scores of the group
            const int buf = xk & 1u;
            *reinterpret_cast<float4*>(sbuf + ((buf * WG + wig) * 32 + lane) * 4) =
                make_float4(s[0], s[1], s[2], s[3]);
            group_sync();
            s[0] = s[1] = s[2] = s[3] = 0.f;
#pragma unroll
            for (int w2 = 0; w2 < WG; ++w2) {
              const float4 x =
                  *reinterpret_cast<const float4*>(sbuf + ((buf * WG + w2) * 32 + lane) * 4);
              s[0] += x.x; s[1] += x.y; s[2] += x.z; s[3] += x.w;
            }
          }
          ++xk;

          // ---- online softmax over the keys (M) of rows 2qd + j ----
          // element e: key kb16 + gr + 8 * (e >> 1), row 2qd + (e & 1)
          float cmax[2] = {-INFINITY, -INFINITY};
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int key = kb16 + gr + 8 * (e >> 1);
            const int j = e & 1;
            const float v = key < vis_end[j] ? s[e] * qk_scale : -INFINITY;
            s[e] = v;
            cmax[j] = fmaxf(cmax[j], v);
          }
          float alpha[2], base[2];
#pragma unroll
          for (int j = 0; j < 2; ++j) {
            cmax[j] = fmaxf(cmax[j], __shfl_xor_sync(0xffffffffu, cmax[j], 4));
            cmax[j] = fmaxf(cmax[j], __shfl_xor_sync(0xffffffffu, cmax[j], 8));
            cmax[j] = fmaxf(cmax[j], __shfl_xor_sync(0xffffffffu, cmax[j], 16));
            const float mn = fmaxf(m_run[j], cmax[j]);
            base[j] = mn == -INFINITY ? 0.f : mn;
            alpha[j] = fast_exp2(m_run[j] - base[j]);
            m_run[j] = mn;
          }
          float pr[4];
#pragma unroll
          for (int e = 0; e < 4; ++e) pr[e] = fast_exp2(s[e] - base[e & 1]);
#pragma unroll
          for (int j = 0; j < 2; ++j) l_run[j] = l_run[j] * alpha[j] + (pr[j] + pr[j + 2]);
#pragma unroll
          for (int mt = 0; mt < MT; ++mt) {
            o[mt][0] *= alpha[0]; o[mt][1] *= alpha[1];
            o[mt][2] *= alpha[0]; o[mt][3] *= alpha[1];
          }
          // P^T as the B operand: keys 0-7 and 8-15, each an 8x8 transpose
          const uint32_t pb0 = movmatrix_trans(pack_bf16x2(pr[0], pr[1]));
          const uint32_t pb1 = movmatrix_trans(pack_bf16x2(pr[2], pr[3]));

          // ---- O^T += V^T P^T over this warp's V columns ----
#pragma unroll
          for (int mt = 0; mt < MT; ++mt) {
            uint32_t a[4];
            ldmatrix_x4_trans(a, slot_piece<C::CB_STRIDE>(
                                     st, r16 + (lane & 7) + 8 * (mj >> 1),
                                     vc0 + (vcol0 + 16 * mt) / 8 + (mj & 1)));
            mma_16816<false>(o[mt], a, pb0, pb1);
          }
        }
        __syncwarp();
        if (lane == 0) tc5::mbar_arrive(slot_empty(slot));
      }
      gc += un.nch;
      // row sums: over the 8 lanes that share qd
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        l_run[j] += __shfl_xor_sync(0xffffffffu, l_run[j], 4);
        l_run[j] += __shfl_xor_sync(0xffffffffu, l_run[j], 8);
        l_run[j] += __shfl_xor_sync(0xffffffffu, l_run[j], 16);
      }
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        const int r = 2 * qd + j;
        if (r >= un.nrows) continue;
        const int rr = un.row0 + r;
        const int64_t t = un.qs + rr / G;
        const int qh = kvh * G + rr % G;
        const int64_t orow = (un.s * T + t) * p.num_q_heads + qh;
        if (l_run[j] > 0.f) {
          const float inv = 1.f / l_run[j];
          float* dst = p.partial_o + orow * C::DV + vcol0;
#pragma unroll
          for (int mt = 0; mt < MT; ++mt) {
            dst[16 * mt + gr] = o[mt][j] * inv;
            dst[16 * mt + gr + 8] = o[mt][2 + j] * inv;
          }
        }
        if (wig == 0 && gr == 0)
          p.partial_lse[orow] =
              l_run[j] > 0.f ? (m_run[j] + fast_log2(l_run[j])) * kLn2 : -INFINITY;
      }
      if (p.fused) fused_finish<C>(p, un, us.HB, us.RG, smem, threadIdx.x - 32);
    }
  } else {
    // ------------------------------------------------ consumer warps ----
    const int cw = warp - 1;
    const int grp = cw / WG, wig = cw % WG;
    const int hg = grp % HPC;  // head of the block this group handles
    const int ng = grp / HPC;  // chunk class: chunks c with c % NG == ng
    const int gr = lane >> 2, qd = lane & 3;
    uint32_t gc = 0, qc = 0;
    uint32_t xk = 0;  // 16-key steps this group has processed: picks the exchange buffer
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
      // The warps that meet at named barriers take the same decision to stop
      // after a timeout: all consumer warps when the classes merge or units
      // end in the fused merge, else the warps of one group.
      if (NG > 1 || p.fused) {
        if (barrier_or(15, 32 * C::NCW, *abort_flag != 0)) break;
      } else if constexpr (WG > 1) {
        if (barrier_or(2 + grp, 32 * WG, *abort_flag != 0)) break;
      } else {
        if (__any_sync(0xffffffffu, *abort_flag != 0)) break;
      }
      const Unit un = *desc_of(qc % C::ND);
      if (un.nch < 0) break;
      const int kvh = un.hb * HPC + hg;  // this group's KV head
      const uint32_t qsrc = sbase + C::Q_OFF + qslot * C::Q_BYTES + hg * C::QH_BYTES;
      // this warp's k-steps of the bf16 path: [ks_lo, ks_lo + nks) (a
      // compile-time count when WG divides them)
      constexpr bool kEven = C::KSTEPS % WG == 0;
      const int ks_lo = kEven ? wig * C::KSW : wig * C::KSTEPS / WG;
      const int nks = kEven ? C::KSW : (wig + 1) * C::KSTEPS / WG - ks_lo;
      uint32_t qa[FP8 ? C::UPW : C::KSW][FP8 ? 16 : 4];
      if constexpr (!FP8) {
#pragma unroll
        for (int kk = 0; kk < C::KSW; ++kk) {
          const int ks = ks_lo + (kEven || kk < nks ? kk : 0);
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
        const int sidx = p.scale_mode == PKV_SCALE_HEAD ? kvh : 0;
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

      // Chunk c (counted over all units) belongs to class c % NG, and
      // NSLOT % NG == 0, so a ring slot is only ever consumed by one class,
      // in order: when a group waits for chunk c, the slot's previous chunk
      // c - NSLOT was its class's own and has completed, and the parity wait
      // cannot be satisfied by the phase of chunk c - 2 * NSLOT.
      const int k_first = static_cast<int>((ng + NG - static_cast<int>(gc % NG)) % NG);
      for (int k = k_first; k < un.nch; k += NG) {
        const uint32_t c = gc + k;
        const uint32_t slot = c % NSLOT;
        const uint32_t st = sbase + C::RING_OFF + slot * C::SLOT_BYTES + hg * C::CB_BYTES;
        wait_all(slot_full(slot), (c / NSLOT) & 1u);
        const int kb = un.klo + k * KPC;
        if (kb + KPC > un.kmax) {
          // rows past the last visible key: zero them before anyone reads
          const int r0 = un.kmax - kb;
          const int n = (KPC - r0) * C::NBOX * 8;
          for (int i = wig * 32 + lane; i < n; i += 32 * WG) {
            const int row = r0 + i / (C::NBOX * 8);
            const int piece = i % (C::NBOX * 8);
            asm volatile("st.shared.v4.u32 [%0], {%1,%1,%1,%1};\n" ::"r"(
                             slot_piece<C::CB_STRIDE>(st, row, piece)),
                         "r"(0u)
                         : "memory");
          }
          tc5::fence_proxy_async_smem();
          group_sync();
        }
        const int nsteps = min(KPC / 16, (un.kmax - kb + 15) / 16);
        for (int ks16 = 0; ks16 < nsteps; ++ks16) {
          const int r16 = 16 * ks16;  // first row of this 16-key step in the slot
          const int kb16 = kb + r16;

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
              if (!kEven && kk >= nks) break;
              const int ks = ks_lo + kk;
              const int m = lane >> 3;
              const int row = r16 + (m >> 1) * 8 + (lane & 7);
              uint32_t kf[4];
              ldmatrix_x4(kf, slot_piece<C::CB_STRIDE>(st, row, kc0 + ks * 2 + (m & 1)));
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
            // two accumulator chains per tile (j even / odd)
            float s2[2][4];
#pragma unroll
            for (int t = 0; t < 2; ++t) s2[t][0] = s2[t][1] = s2[t][2] = s2[t][3] = 0.f;
#pragma unroll
            for (int uu = 0; uu < C::UPW; ++uu) {
              const int un_ = wig + uu * WG;
              if (un_ < C::NU) {
                uint4 kw[2];
#pragma unroll
                for (int t = 0; t < 2; ++t)
                  kw[t] = lds128(slot_piece<C::CB_STRIDE>(st, r16 + 8 * t + gr, kc0 + 4 * un_ + qd));
#pragma unroll
                for (int t = 0; t < 2; ++t) {
                  const uint32_t wv[4] = {kw[t].x, kw[t].y, kw[t].z, kw[t].w};
#pragma unroll
                  for (int j = 0; j < 4; ++j) {
                    const uint32_t a[4] = {qa[uu][2 * j], qa[uu][8 + 2 * j],
                                           qa[uu][2 * j + 1], qa[uu][8 + 2 * j + 1]};
                    mma_16816<true>(j & 1 ? s2[t] : s[t], a,
                                    e4m3x2_to_f16x2(static_cast<uint16_t>(wv[j])),
                                    e4m3x2_to_f16x2(static_cast<uint16_t>(wv[j] >> 16)));
                  }
                }
              }
            }
#pragma unroll
            for (int t = 0; t < 2; ++t)
#pragma unroll
              for (int e = 0; e < 4; ++e) s[t][e] += s2[t][e];
          }
          if constexpr (WG > 1) {  // sum the K-slice partial scores of the group
            // a warp's block holds its two key tiles one after the other,
            // each as 32 lanes x 16 contiguous bytes, so every 16-byte store
            // and load of the warp is free of bank conflicts
            const int buf = xk & 1u;
            float* mine = sbuf + (buf * WG + wig) * 32 * 8 + lane * 4;
            *reinterpret_cast<float4*>(mine) = make_float4(s[0][0], s[0][1], s[0][2], s[0][3]);
            *reinterpret_cast<float4*>(mine + 128) = make_float4(s[1][0], s[1][1], s[1][2], s[1][3]);
            group_sync();
#pragma unroll
            for (int t = 0; t < 2; ++t) s[t][0] = s[t][1] = s[t][2] = s[t][3] = 0.f;
#pragma unroll
            for (int w2 = 0; w2 < WG; ++w2) {
              const float* src = sbuf + (buf * WG + w2) * 32 * 8 + lane * 4;
              const float4 x = *reinterpret_cast<const float4*>(src);
              const float4 y = *reinterpret_cast<const float4*>(src + 128);
              s[0][0] += x.x; s[0][1] += x.y; s[0][2] += x.z; s[0][3] += x.w;
              s[1][0] += y.x; s[1][1] += y.y; s[1][2] += y.z; s[1][3] += y.w;
            }
          }
          ++xk;

          // ---- online softmax (rows gr, gr + 8), log2 domain ----
          float cmax[2] = {-INFINITY, -INFINITY};
#pragma unroll
          for (int t = 0; t < 2; ++t)
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const int key = kb16 + 8 * t + 2 * qd + (e & 1);
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
              const int row = r16 + (m & 1) * 8 + (lane & 7);
              uint32_t r[4];
              ldmatrix_x4_trans(
                  r, slot_piece<C::CB_STRIDE>(st, row, vc0 + (vcol0 + 16 * np) / 8 + (m >> 1)));
              mma_16816<false>(o[2 * np], pa, r[0], r[1]);
              mma_16816<false>(o[2 * np + 1], pa, r[2], r[3]);
            }
          } else {
#pragma unroll
            for (int vb = 0; vb < C::DVS / 128; ++vb) {
              const int piece = vc0 + (vcol0 + 128 * vb) / 16 + gr;
              const int rows[4] = {r16 + 2 * qd, r16 + 2 * qd + 1, r16 + 2 * qd + 8,
                                   r16 + 2 * qd + 9};
              uint32_t kw[4][4];
#pragma unroll
              for (int k4 = 0; k4 < 4; ++k4) {
                const uint4 v = lds128(slot_piece<C::CB_STRIDE>(st, rows[k4], piece));
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
        }
        __syncwarp();
        if (lane == 0) tc5::mbar_arrive(slot_empty(slot));
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

      if constexpr (NG > 1) {
        // ---- every chunk class hands its (O, max, sum) of each row over;
        //      then all consumer threads combine the classes element-wise ----
        float* mo = reinterpret_cast<float*>(smem + C::MERGE_OFF);
        auto mrow = [&](int q, int h, int r) { return mo + ((q * HPC + h) * 16 + r) * C::MROW; };
        named_barrier(1, 32 * C::NCW);  // the previous unit's reads are done
#pragma unroll
        for (int kr = 0; kr < 2; ++kr) {
          float* b = mrow(ng, hg, gr + 8 * kr);
#pragma unroll
          for (int nt = 0; nt < C::NT; ++nt)
#pragma unroll
            for (int e = 0; e < 2; ++e) b[col_of(nt, e)] = o[nt][2 * kr + e];
          if (wig == 0 && qd == 0) {
            b[C::DVP] = m_run[kr];
            b[C::DVP + 1] = l_run[kr];
          }
        }
        named_barrier(1, 32 * C::NCW);
        const int ctid = threadIdx.x - 32;
        const int per_head = un.nrows * C::DV;
        for (int idx = ctid; idx < HPC * per_head; idx += 32 * C::NCW) {
          const int h = idx / per_head;
          const int rc = idx - h * per_head;
          const int r = rc / C::DV, cc = rc - r * C::DV;
          float M = -INFINITY;
#pragma unroll
          for (int q = 0; q < NG; ++q) M = fmaxf(M, mrow(q, h, r)[C::DVP]);
          const int rr = un.row0 + r;
          const int64_t t = un.qs + rr / G;
          const int kvh2 = un.hb * HPC + h;
          const int64_t orow = (un.s * T + t) * p.num_q_heads + kvh2 * G + rr % G;
          if (M == -INFINITY) {  // no class saw a key of this row
            if (cc == 0) p.partial_lse[orow] = -INFINITY;
            continue;
          }
          float l = 0.f, acc = 0.f;
#pragma unroll
          for (int q = 0; q < NG; ++q) {
            const float* b = mrow(q, h, r);
            const float wq = fast_exp2(b[C::DVP] - M);  // 0 for a class without keys
            l += wq * b[C::DVP + 1];
            acc += wq * b[cc];
          }
          float vm = 1.f;
          if constexpr (FP8)
            vm = __ldg(p.v_scale + (p.scale_mode == PKV_SCALE_HEAD ? kvh2 : 0));
          p.partial_o[orow * C::DV + cc] = acc / l * vm;
          if (cc == 0) p.partial_lse[orow] = (M + fast_log2(l)) * kLn2;
        }
      } else {
        // every warp writes its own V columns of the head's partial rows
#pragma unroll
        for (int kr = 0; kr < 2; ++kr) {
          const int r = gr + 8 * kr;
          if (r >= un.nrows) continue;
          const int rr = un.row0 + r;
          const int64_t t = un.qs + rr / G;
          const int qh = kvh * G + rr % G;
          const int64_t orow = (un.s * T + t) * p.num_q_heads + qh;
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
      }
      if (p.fused) fused_finish<C>(p, un, us.HB, us.RG, smem, threadIdx.x - 32);
    }
  }
}

template <class C>
cudaError_t launch_cfg(const AttnParams& p, int num_sms, cudaStream_t stream) {
  static int attr_set[3][64] = {{0}};
  const int bal = p.split_ranges <= 0 ? 0 : p.num_seqs <= kBalancedMaxSeqs ? 1 : 2;
  cudaError_t e = bal == 2   ? ensure_smem_attr(decode_kernel<C, 2>, C::SMEM, attr_set[2])
                  : bal == 1 ? ensure_smem_attr(decode_kernel<C, 1>, C::SMEM, attr_set[1])
                             : ensure_smem_attr(decode_kernel<C, 0>, C::SMEM, attr_set[0]);
  if (e != cudaSuccess) return e;
  alignas(64) CUtensorMap kv_map;
  const int box_rows = box_rows_for(p.block_size, C::KPC);
  // one box for all HPC heads of a column slice when a chunk's keys are one
  // box high (5 boxes per 16-key chunk of 4 heads instead of 20)
  const int head_boxes = C::HPC > 1 && box_rows == C::KPC ? 1 : 0;
  const bool ok =
      head_boxes ? make_cache_tmap_heads(&kv_map, p.cache, p.dtype, p.layout, p.num_blocks,
                                         p.block_size, p.num_kv_heads, p.row_elems,
                                         C::BOX_COLS, box_rows, C::HPC)
                 : make_cache_tmap(&kv_map, p.cache, p.dtype, p.layout, p.num_blocks,
                                   p.block_size, p.num_kv_heads, p.row_elems, C::BOX_COLS,
                                   box_rows);
  if (!ok) return cudaErrorInvalidValue;
  // tensor-core form: the third column box (span bytes 256..319) is 64 bytes
  // wide with a 64-byte swizzle
  alignas(64) CUtensorMap kv_map64 = kv_map;
  if (C::TC && !make_cache_tmap(&kv_map64, p.cache, p.dtype, p.layout, p.num_blocks,
                                p.block_size, p.num_kv_heads, p.row_elems, 64, box_rows,
                                /*swizzle64=*/true))
    return cudaErrorInvalidValue;
  const int64_t RG = (static_cast<int64_t>(p.max_query_len) * p.group + 15) / 16;
  // equal segments: one CTA per unit up to the resident slots; balanced
  // ranges: one CTA per (range, head block) up to the resident slots
  const int64_t units = p.split_ranges > 0
                            ? static_cast<int64_t>(p.split_ranges) * (p.num_kv_heads / C::HPC)
                            : static_cast<int64_t>(p.num_splits) * p.num_seqs *
                                  (p.num_kv_heads / C::HPC) * RG;
  const int64_t slots = static_cast<int64_t>(C::CTAS) * num_sms;
  const int grid = static_cast<int>(units < slots ? units : slots);
  e = bal == 2   ? launch_pdl(decode_kernel<C, 2>, grid, C::THREADS, C::SMEM, stream, kv_map,
                              kv_map64, p, head_boxes)
      : bal == 1 ? launch_pdl(decode_kernel<C, 1>, grid, C::THREADS, C::SMEM, stream, kv_map,
                              kv_map64, p, head_boxes)
                 : launch_pdl(decode_kernel<C, 0>, grid, C::THREADS, C::SMEM, stream, kv_map,
                              kv_map64, p, head_boxes);
  return e != cudaSuccess ? e : cudaGetLastError();
}

// <DK, DV, fp8, heads per chunk, warps per group, chunk classes, keys per
//  chunk, ring slots, unit slots, staged span>
// K192 / V128, bf16: four heads per chunk (40 KB of 16 keys) when Hkv
// allows, else one head with six chunk classes.
using CfgBf16_192x4 = DecodeCfg<192, 128, false, 4, 2, 1, 16, 4, 2, 320>;
// the same with a head's rows in 8 (q_len * G <= 8): transposed MMAs
using CfgBf16_192x4n = DecodeCfg<192, 128, false, 4, 2, 1, 16, 4, 2, 320, true>;
using CfgBf16_192x1 = DecodeCfg<192, 128, false, 1, 1, 6, 16, 12, 4, 320>;
// K192 / V128, fp8: one head, 64 keys per chunk (three 8 KB boxes at block
// 64), six chunk classes.
using CfgFp8_192 = DecodeCfg<192, 128, true, 1, 1, 6, 64, 6, 2, 320>;
// The same on the tensor cores: one head, 128 keys per chunk (40 KB),
// three ring slots; for rows whose K precedes V.
using CfgFp8_192tc = DecodeCfg<192, 128, true, 1, 1, 1, 128, 3, 2, 320, false, 1, true>;
// MLA 576 / 512: one latent head, 32 (bf16) or 64 (fp8) keys per chunk.
using CfgBf16_576 = DecodeCfg<576, 512, false, 1, 4, 1, 32, 2, 1, 576, false, 2>;
// the same with 16-key chunks in four ring slots, for short segments (a
// unit of a few pages): its stream fills sooner (MLA batch 1 at 100K, six
// pages a unit: 41.0 against 43.0 us), while long segments stream faster
// in 32-key chunks (batch 16: 356 against 389 us)
using CfgBf16_576s = DecodeCfg<576, 512, false, 1, 4, 1, 16, 4, 1, 576, false, 2>;
using CfgFp8_576 = DecodeCfg<576, 512, true, 1, 4, 1, 64, 4, 2, 576>;

}  // namespace

int decode_ctas_per_sm(const AttnParams& p) {
  if (p.head_size == 576 && p.head_size_v == 512)
    return p.dtype == PKV_FP8_E4M3 ? CfgFp8_576::CTAS : CfgBf16_576::CTAS;
  return 1;
}

namespace {
// Keys a segment holds at most, from what the host knows (the block-table
// width, and the segment count or, for balanced ranges, the range count):
// the MLA bf16 form takes 16-key chunks up to kShortSegKeys keys a unit.
constexpr int64_t kShortSegKeys = 1024;
bool short_segments(const AttnParams& p) {
  const int64_t mb = p.max_blocks_per_seq;
  const int64_t pages =
      p.split_ranges > 0
          ? (static_cast<int64_t>(p.num_seqs) * mb + p.split_ranges - 1) / p.split_ranges
          : (mb + p.num_splits - 1) / p.num_splits;
  return pages * p.block_size <= kShortSegKeys;
}
}  // namespace

int decode_head_blocks(const AttnParams& p) {
  // four KV heads per unit only in the bf16 K192 form with Hkv % 4 == 0
  if (p.head_size == 192 && p.dtype == PKV_BF16 && p.num_kv_heads % 4 == 0)
    return p.num_kv_heads / 4;
  return p.num_kv_heads;
}

bool decode_supported(int head_size, int head_size_v, int dtype) {
  (void)dtype;
  return (head_size == 192 && head_size_v == 128) ||
         (head_size == 576 && head_size_v == 512);
}

cudaError_t launch_decode(const AttnParams& p, int num_sms, cudaStream_t stream) {
  const bool fp8 = p.dtype == PKV_FP8_E4M3;
  if (p.head_size == 192 && p.head_size_v == 128) {
    if (fp8)
      return p.k_off <= p.v_off ? launch_cfg<CfgFp8_192tc>(p, num_sms, stream)
                                : launch_cfg<CfgFp8_192>(p, num_sms, stream);
    if (p.num_kv_heads % 4 != 0) return launch_cfg<CfgBf16_192x1>(p, num_sms, stream);
    return p.max_query_len * p.group <= 8 ? launch_cfg<CfgBf16_192x4n>(p, num_sms, stream)
                                          : launch_cfg<CfgBf16_192x4>(p, num_sms, stream);
  }
  if (p.head_size == 576 && p.head_size_v == 512)
    return fp8 ? launch_cfg<CfgFp8_576>(p, num_sms, stream)
               : short_segments(p) ? launch_cfg<CfgBf16_576s>(p, num_sms, stream)
                                   : launch_cfg<CfgBf16_576>(p, num_sms, stream);
  return cudaErrorNotSupported;
}

}  // namespace pkv
