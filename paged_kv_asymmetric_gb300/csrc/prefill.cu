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
//  * Persistent clusters of two CTAs, one CTA per SM.  A CTA's work item is
//    two 128-row query tiles of one KV head (tiles A and B); a tile is 128 / G
//    consecutive tokens x the G query heads that share the KV head (GQA
//    packing).  The two CTAs of a cluster take adjacent items of the same
//    sequence and KV head and walk the same key tiles: with slab fills each
//    K/V box is read from L2 once, by one of them, and multicast into both
//    shared memories, so a K/V tile feeds 4 x 128 query rows.  (Without this
//    the slab boxes alone ran at ~3.6 TB/s from L2 and bounded the kernel.)
//    Units are numbered longest-first and dealt to the clusters in
//    alternating directions.
//  * Warp roles: warp 0 issues TMA loads (the two Q tiles as 64-column slabs;
//    K and V pages as 64-column boxes of one page each into 128-key slabs of
//    an 8-slab ring, half of each slab's boxes per CTA, a slot refilled once
//    the MMAs of both CTAs have read it; or page-grouped boxes into part
//    slots, below; page ids prefetched two tiles ahead by all lanes),
//    warp 1 issues tcgen05.mma from one thread, warps 4..7 run the softmax
//    of tile A and warps 8..11 that of tile B, one thread per query row.
//  * Tensor memory holds S and O of both tiles (4 x 128 columns).  The
//    tensor core works on one tile while the softmax works on the other:
//    S_A(j) and S_B(j) = Q K_j^T (M 128, N 128, K 192, operands in shared
//    memory); the softmax turns S_X(j) into bf16 P and stores it over S_X's
//    first 64 columns in tensor memory; O_X += P V_j reads P straight from
//    tensor memory (A operand) and V_j from shared memory in one N = 128 MMA
//    per 16 keys (an N = 64 MMA costs as much time as an N = 128 one).
//    Issue order: S_A(0) S_B(0) | PV_A(j) S_A(j+1) PV_B(j) S_B(j+1) | ...
//    A commit after S_X(j+1) also covers PV_X(j), so when the softmax sees
//    S_X(j+1) ready, P_X(j) has been consumed and O_X is stable.
//  * bf16 caches whose rows split into 64-column slabs: page-grouped fills.
//    A key tile's K part (three slabs) and V part (two) are laid out as
//    [8-key group][slab][8 keys][128 B], so one 5-D TMA box per 16 keys of a
//    page brings all of a part's columns for them: 16 boxes per 128-key tile
//    instead of 40 at 16-key pages.  The ring holds fixed part slots: two K
//    slots taken by alternate tiles (a tile's K is loaded while the previous
//    one is still read) and a V slot of two 64-key halves with their own
//    barriers (the next tile's first half loads while the MMAs still read
//    the second, and P.V starts on the first half before the second lands).
//    The producer issues the K of tile j + 1 before the V of tile j, and each
//    CTA loads its own parts.  The MMAs step over a part's key groups at a
//    3 KB (K) or 2 KB (V) stride.  Other row layouts and FP8 caches fill one
//    64-column slab at a time into the 8-slab ring, multicast to both CTAs.
//  * Online softmax with a lazy rescale: the exponent base moves (and O and
//    the running sum are rescaled in place) only when a row maximum grows by
//    more than 2^8, decided per warp; the result is the same up to rounding.
//  * Keys past the sequence end in its last tile are masked out of S, and the
//    corresponding V rows are zeroed in shared memory before any P V MMA
//    reads them, so whatever the cache holds there cannot produce NaN.
//  * Every mbarrier wait is bounded (2 s): on expiry the kernel records
//    PKV_EDEV_TIMEOUT, every role stops at its next wait, copies and MMAs in
//    flight are waited for (bounded) and tensor memory is freed before exit.
#include <math.h>

#include "common.cuh"
#include "kernels.h"
#include "tc5.cuh"
#include "tmap.h"

namespace pkv {

namespace {

constexpr int DK = 192, DV = 128;
constexpr int BM = 128, BN = 128;
constexpr int SLAB = 128 * 64 * 2;  // one 128-row x 64-column bf16 slab
constexpr int KSLABS = DK / 64;     // 3
constexpr int VSLABS = DV / 64;     // 2
constexpr int NSLAB = 8;            // K/V ring
constexpr int Q_OFF = 0;            // tiles A and B: 2 x 3 slabs
constexpr int RING_OFF = Q_OFF + 2 * KSLABS * SLAB;
constexpr int BAR_OFF = RING_OFF + NSLAB * SLAB;
enum {
  B_QFULL = 0,
  B_QEMPTY,
  B_SFULL0,   // + tile
  B_PFULL0 = B_SFULL0 + 2,
  B_ODONE0 = B_PFULL0 + 2,
  B_OFREE0 = B_ODONE0 + 2,
  B_FINAL = B_OFREE0 + 2,
  B_SLAB_FULL0,
  B_SLAB_EMPTY0 = B_SLAB_FULL0 + NSLAB,
  // FP8 cache: a slab's E4M3 codes have been widened to bf16 in place
  B_SLAB_READY0 = B_SLAB_EMPTY0 + NSLAB,
  NBAR = B_SLAB_READY0 + NSLAB
};
constexpr int MISC_OFF = BAR_OFF + NBAR * 8;  // tmem base, abort word
constexpr int SMEM_BYTES = MISC_OFF + 16 + 1024;  // + alignment slack
constexpr int THREADS = 384;  // 4 control warps + 2 softmax warpgroups
// FP8 cache: one more warpgroup (warps 12..15) widens the E4M3 slabs
constexpr int THREADS_F8 = 512;
constexpr uint32_t TMEM_COLS = 512;
// tensor-memory columns: S and O of tile A, then of tile B
__device__ __forceinline__ uint32_t tm_s(int x) { return x ? 256u : 0u; }
__device__ __forceinline__ uint32_t tm_o(int x) { return x ? 384u : 128u; }
constexpr float kRescaleThreshold = 8.0f;  // log2 units

static_assert(SMEM_BYTES <= 227 * 1024, "shared memory budget");

// Ring fills of an item: five per key tile (K's three slabs, V's two), tile j
// taking fills fbase + 5j .. fbase + 5j + 4.  One N = 128 MMA reads both V
// slabs at a fixed stride, so they must sit in adjacent slots; in the one
// tile position in eight where they would straddle the end of the ring, the
// tile's V is filled before its K.
constexpr int FILLS_PER_TILE = KSLABS + VSLABS;
static_assert(FILLS_PER_TILE == 5 && NSLAB == 8, "fill pattern");
__device__ __forceinline__ bool v_first(uint32_t fbase, int j) {
  return (fbase + FILLS_PER_TILE * j + KSLABS) % NSLAB == NSLAB - 1;
}
__device__ __forceinline__ uint32_t k_fill(uint32_t fbase, int j, int c) {
  return fbase + FILLS_PER_TILE * j + (v_first(fbase, j) ? VSLABS : 0) + c;
}
__device__ __forceinline__ uint32_t v_fill(uint32_t fbase, int j, int h) {
  return fbase + FILLS_PER_TILE * j + (v_first(fbase, j) ? 0 : KSLABS) + h;
}

// Page-grouped fills use the ring as fixed part slots: K parts of tiles
// alternate between slabs 0..2 and 3..5 (a K part is loaded while the other
// is still read), and every tile's V part takes slabs 6..7, one slab per
// 64-key half with its own barriers (the next tile's first half loads while
// the MMAs still read the second, and P.V starts on the first half before
// the second lands).  Tile t (counted over the CTA's items) uses K slot
// t & 1, whose barriers are those of its first slab; a slot's n-th use is
// phase n & 1 (K: n = t >> 1; V: n = t).  Each CTA loads its own parts, so
// a slot is free once this CTA's MMAs have read it.
__device__ __forceinline__ uint32_t kslot_slab(uint32_t t) { return (t & 1u) * KSLABS; }
constexpr uint32_t VSLOT_SLAB = 2 * KSLABS;
static_assert(VSLOT_SLAB + VSLABS <= NSLAB, "three part slots in the ring");
constexpr uint32_t KGROUP = KSLABS * 1024;  // a K part's 8-key group stride
constexpr uint32_t VGROUP = VSLABS * 1024;  // and a V part's

struct Item {
  int b, g, L, qlen;
  int q0[2], nq[2], minpos[2];
  int nkeys, ntiles;
};

constexpr int CLUSTER = 2;          // CTAs sharing each K/V load
constexpr uint16_t CLUSTER_MASK = (1u << CLUSTER) - 1;

// The idx-th work unit, as seen by cluster rank `rank`.  A unit is query
// tiles 4u .. 4u + 3 of one sequence and KV head; rank r takes tiles 4u + 2r
// and 4u + 2r + 1 (its item), and both ranks walk the key tiles of the unit's
// last token, so that every K/V tile is loaded once for the pair (keys past a
// row's position are masked as usual).  Units are numbered longest-first
// within each sequence; false when idx is past the end.
__device__ __forceinline__ bool get_unit(const AttnParams& p, int TQ, int idx,
                                         int rank, Item& it) {
  int acc = 0;
  for (int b = 0; b < p.num_seqs; ++b) {
    const int qs = __ldg(p.query_start_loc + b);
    const int qlen = __ldg(p.query_start_loc + b + 1) - qs;
    const int ntq = (qlen + TQ - 1) / TQ;
    const int nu = (ntq + 2 * CLUSTER - 1) / (2 * CLUSTER);
    const int cnt = nu * p.num_kv_heads;
    if (idx < acc + cnt) {
      const int j = idx - acc;
      const int u = nu - 1 - j / p.num_kv_heads;
      it.b = b;
      it.g = j % p.num_kv_heads;
      it.L = __ldg(p.seq_lens + b);
      it.qlen = qlen;
      for (int x = 0; x < 2; ++x) {
        const int t0 = (2 * CLUSTER * u + 2 * rank + x) * TQ;
        it.q0[x] = qs + t0;
        it.nq[x] = max(0, min(TQ, qlen - t0));
        it.minpos[x] = it.L - qlen + t0;
      }
      const int tend = min(qlen, 2 * CLUSTER * (u + 1) * TQ);  // past the unit's last token
      it.nkeys = max(0, min(it.L - qlen + tend, it.L));
      it.ntiles = (it.nkeys + BN - 1) / BN;
      return true;
    }
    acc += cnt;
  }
  return false;
}

// FP8 cache: one ring slab's 128 key rows x 64 columns, landed by TMA as E4M3
// codes in the slab's upper half (row r at byte 8192 + 64 r), widened in
// place to the bf16 slab the MMAs read (row r at byte 128 r, 16-byte chunk c
// at chunk c ^ (r & 7): the 128-byte swizzle of the bf16 boxes).  An E4M3
// value has 4 significant bits and an exponent within bf16's range, so
// E4M3 -> f16 -> bf16 is exact (NaN stays NaN).  Run by the 64 threads of
// the widening warpgroup (ct = 0..127, named barrier kWidenBar).  Output row r
// covers the input of rows 2r - 128 and 2r - 127, so the rows go in three
// steps: rows 0..63 (their output lies below all input); rows 64..95 (over
// the input of rows 0..63, already read) while rows 96..127's input is read
// into registers; then rows 96..127.
constexpr int kWidenBar = 1;
constexpr int kWidenThreads = 128;

__device__ __forceinline__ uint4 widen8(uint2 w) {
  const uint32_t in[2] = {w.x, w.y};
  uint32_t o[4];
#pragma unroll
  for (int k = 0; k < 2; ++k)
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const uint32_t f16 = e4m3x2_to_f16x2(static_cast<uint16_t>(in[k] >> (16 * h)));
      const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&f16));
      o[2 * k + h] = pack_bf16x2(f.x, f.y);
    }
  return make_uint4(o[0], o[1], o[2], o[3]);
}

__device__ __forceinline__ void widen_slab(uint8_t* slab, int ct) {
  auto src = [&](int row, int c) {
    return *reinterpret_cast<const uint2*>(slab + 8192 + 64 * row + 8 * c);
  };
  auto dst = [&](int row, int c) {
    return reinterpret_cast<uint4*>(slab + 128 * row + 16 * (c ^ (row & 7)));
  };
  constexpr int kRows64 = 512 / kWidenThreads;  // 16-byte outputs per thread, rows 0..63
  constexpr int kRows32 = 256 / kWidenThreads;  // and per 32 rows
#pragma unroll
  for (int i = 0; i < kRows64; ++i) {  // rows 0..63
    const int q = ct + kWidenThreads * i;
    *dst(q >> 3, q & 7) = widen8(src(q >> 3, q & 7));
  }
  named_barrier(kWidenBar, kWidenThreads);
  uint2 hold[kRows32];
#pragma unroll
  for (int i = 0; i < kRows32; ++i) {  // rows 64..95; rows 96..127 read
    const int q = ct + kWidenThreads * i;
    *dst(64 + (q >> 3), q & 7) = widen8(src(64 + (q >> 3), q & 7));
    hold[i] = src(96 + (q >> 3), q & 7);
  }
  named_barrier(kWidenBar, kWidenThreads);
#pragma unroll
  for (int i = 0; i < kRows32; ++i) {  // rows 96..127
    const int q = ct + kWidenThreads * i;
    *dst(96 + (q >> 3), q & 7) = widen8(hold[i]);
  }
}

// The k-th unit of this cluster.  Units are numbered longest-first and dealt
// in rounds over the clusters, alternately forwards and backwards, so that
// every cluster's total work is about the same.
__device__ __forceinline__ int unit_index(int k) {
  const int ncl = static_cast<int>(tc5::num_clusters_x());
  const int cid = static_cast<int>(tc5::cluster_id_x());
  return k * ncl + ((k & 1) ? ncl - 1 - cid : cid);
}

// F8: the cache holds E4M3 codes; they are widened to bf16 in shared memory
// by warps 12..15 between the TMA fill and the MMAs (k_scale and v_scale
// fold into the softmax scale and the output, p.fold_scales).  PG (bf16
// only): page-grouped fills, kv_map bringing a page's K part and v_map its
// V part; otherwise kv_map brings one 64-column slab of a page (v_map is
// unused).
template <bool F8, bool PG>
__global__ void __launch_bounds__(F8 ? THREADS_F8 : THREADS, 1)
    prefill_kernel(const __grid_constant__ CUtensorMap q_map,
                   const __grid_constant__ CUtensorMap kv_map,
                   const __grid_constant__ CUtensorMap v_map,
                   const AttnParams p) {
  static_assert(!(F8 && PG), "page-grouped fills are for bf16 caches");
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t sbase = (raw + 1023u) & ~1023u;
  uint8_t* smem = smem_raw + (sbase - raw);
  const uint32_t bar0 = sbase + BAR_OFF;
  auto bar = [&](int i) { return bar0 + 8u * static_cast<uint32_t>(i); };
  volatile uint32_t* tmem_slot = reinterpret_cast<volatile uint32_t*>(smem + MISC_OFF);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + MISC_OFF + 8);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int rank = static_cast<int>(tc5::cluster_ctarank());
  const int G = p.group;
  const int TQ = BM / G;

  if (threadIdx.x == 0) {
    for (int i = 0; i < NBAR; ++i) {
      uint32_t count = 1;
      if ((i >= B_PFULL0 && i < B_PFULL0 + 2) || (i >= B_OFREE0 && i < B_OFREE0 + 2))
        count = 128;
      // one commit per CTA that reads the slab (page-grouped: this CTA's own)
      if (i >= B_SLAB_EMPTY0 && i < B_SLAB_EMPTY0 + NSLAB) count = PG ? 1 : CLUSTER;
      tc5::mbar_init(bar(i), count);
    }
    *abort_flag = 0;
    tc5::fence_mbar_init();
    tc5::prefetch_tmap(&q_map);
    tc5::prefetch_tmap(&kv_map);
    if (PG) tc5::prefetch_tmap(&v_map);
  }
  if (warp == 1) {
    tc5::tmem_alloc(sbase + MISC_OFF, TMEM_COLS);
    tc5::tmem_relinquish();
  }
  tc5::tc_fence_before();
  __syncthreads();
  // the peer's barriers are initialised before either CTA's first copy
  tc5::cluster_sync();
  tc5::tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  const int bs = p.block_size;
  // rows of a K/V box: a page, or 128 keys of it (slab fills) or 16 keys of
  // it (page-grouped fills: eight or more boxes a part in flight stream
  // faster than fewer larger ones, and a V part's two key halves each get
  // whole boxes)
  const int box_rows = PG ? (bs < 16 ? bs : 16) : (bs < BN ? bs : BN);
  const int nbox = BN / box_rows;

  // Registers: the bf16 block is launched with 384 x 168; the control
  // warpgroup (producer, MMA issuer, two idle warps) keeps 120 per thread and
  // the two softmax warpgroups take 192 (128 x 120 + 256 x 192 = 64,512),
  // enough to hold a whole S row per thread.  The FP8 block's split is given
  // with its widening warpgroup below.

  if (warp < 4) {
  if constexpr (F8)
    asm volatile("setmaxnreg.dec.sync.aligned.u32 104;\n" ::: "memory");
  else
    asm volatile("setmaxnreg.dec.sync.aligned.u32 120;\n" ::: "memory");
  if (warp == 0) {
    // ------------------------------------------------ TMA producer ------
    // Fill order per item: K_0, V_0, K_1, V_1, ...  Lane i owns box i of a
    // 128-key slab (nbox <= 16 boxes, one page or part of one each): it
    // loads that box's page id two tiles ahead and issues the box itself.
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
      constexpr int kRowBytes = F8 ? 64 : 128;  // one box row: 64 columns
      if (lane == 0)
        tc5::mbar_arrive_expect_tx(full, static_cast<uint32_t>(nb * box_rows * kRowBytes));
      __syncwarp();
      // each box is copied by one rank into both CTAs (ranks alternate)
      if (lane < nb && ((lane + static_cast<int>(f)) % CLUSTER) == rank) {
        const int key0 = kt * BN + lane * box_rows;
        const int off = key0 % bs;
        int page = pid;
        if (page < 0 || page >= p.num_blocks) {
          set_dev_error(p.err, PKV_EDEV_RANGE);
          page = p.num_blocks;  // out-of-range box: TMA fills zeros
        }
        const uint32_t dst = sbase + RING_OFF + slot * SLAB + (F8 ? 8192 : 0) +
                             lane * box_rows * kRowBytes;
        if (p.layout == PKV_NHD)
          tc5::tma_load_4d_mc(dst, &kv_map, col, it.g, off, page, full, CLUSTER_MASK);
        else
          tc5::tma_load_4d_mc(dst, &kv_map, col, off, it.g, page, full, CLUSTER_MASK);
      }
      ++f;
      return true;
    };
    // page-grouped fills: tile t's K part (kv_map, slot t & 1) or one 64-key
    // half of its V part (v_map, the V slot's slab for that half): one box
    // per 16 keys of a page (per page when pages are smaller), each CTA
    // loading its own, the slot's previous use read by this CTA's MMAs first
    uint32_t tk = 0, tv = 0;  // K parts and V parts (both halves) issued
    // vh: the 64-key half of a V part (its boxes and its slab)
    auto fill_part = [&](const Item& it, int kt, bool is_v, int pid, int vh) -> bool {
      const uint32_t t = is_v ? tv : tk;
      const uint32_t slab = is_v ? VSLOT_SLAB + vh : kslot_slab(t);
      const uint32_t use = is_v ? t : t >> 1;
      bool w = true;
      if (lane == 0)
        w = tc5::mbar_wait(bar(B_SLAB_EMPTY0 + slab), (use & 1u) ^ 1u, abort_flag, p.err);
      if (!__shfl_sync(0xffffffffu, w, 0)) return false;
      const int nsl = is_v ? VSLABS : KSLABS;
      const int lim = it.L - kt * BN;
      const int nb = min(nbox, (lim + box_rows - 1) / box_rows);
      // this fill's boxes: all of a K part, one half of a V part (none when
      // the sequence ends in the first half: the phase then completes
      // with no bytes)
      const int b0 = is_v ? vh * (nbox / 2) : 0;
      const int b1 = min(nb, is_v ? b0 + nbox / 2 : nbox);
      const uint32_t full = bar(B_SLAB_FULL0 + slab);
      if (lane == 0)
        tc5::mbar_arrive_expect_tx(
            full, static_cast<uint32_t>(max(0, b1 - b0) * box_rows * nsl * 128));
      __syncwarp();
      if (lane >= b0 && lane < b1) {
        const int key0 = kt * BN + lane * box_rows;
        const int off = key0 % bs;
        int page = pid;
        if (page < 0 || page >= p.num_blocks) {
          set_dev_error(p.err, PKV_EDEV_RANGE);
          page = p.num_blocks;  // out-of-range box: TMA fills zeros
        }
        const uint32_t dst = sbase + RING_OFF + (is_v ? VSLOT_SLAB : slab) * SLAB +
                             static_cast<uint32_t>(lane * box_rows * nsl * 128);
        int cs = (is_v ? p.v_off : p.k_off) / 64, pg = page;
        if (p.layout == PKV_NHD)
          cs += it.g * (p.row_elems / 64);
        else
          pg = page * p.num_kv_heads + it.g;
        tc5::tma_load_5d(dst, is_v ? &v_map : &kv_map, 0, 0, cs, off / 8, pg, full);
      }
      if (!is_v)
        ++tk;
      else if (vh == 1)
        ++tv;
      return true;
    };
    for (int k = 0; ok; ++k) {
      Item it;
      if (!get_unit(p, TQ, unit_index(k), rank, it)) break;
      if (it.ntiles == 0) continue;
      bt_row = p.block_table + static_cast<int64_t>(it.b) * p.max_blocks_per_seq;
      int pid0 = load_pid(it, 0), pid1 = load_pid(it, 1);
      bool w = true;
      if (lane == 0) {
        w = tc5::mbar_wait(bar(B_QEMPTY), (qi & 1u) ^ 1u, abort_flag, p.err);
        if (w) {
          tc5::mbar_arrive_expect_tx(bar(B_QFULL), 2 * KSLABS * SLAB);
          for (int x = 0; x < 2; ++x)
            for (int c = 0; c < KSLABS; ++c)
              tc5::tma_load_3d(sbase + Q_OFF + (x * KSLABS + c) * SLAB, &q_map, 64 * c,
                               it.g * G, it.q0[x], bar(B_QFULL));
        }
      }
      if (!__shfl_sync(0xffffffffu, w, 0)) break;
      ++qi;
      // page-grouped: K runs one tile ahead of V (K of tile j + 1 is issued
      // before V of tile j, as its slot frees earlier)
      if constexpr (PG) ok = fill_part(it, 0, false, pid0, 0);
      for (int j = 0; j < it.ntiles && ok; ++j) {
        const int pid2 = load_pid(it, j + 2);  // prefetch
        if constexpr (PG) {
          if (j + 1 < it.ntiles) ok = fill_part(it, j + 1, false, pid1, 0);
          if (ok) ok = fill_part(it, j, true, pid0, 0);
          if (ok) ok = fill_part(it, j, true, pid0, 1);
        } else {
          const bool vf = v_first(f, 0);
          for (int h = 0; h < VSLABS && ok && vf; ++h) ok = fill_slab(it, j, p.v_off + 64 * h, pid0);
          for (int c = 0; c < KSLABS && ok; ++c) ok = fill_slab(it, j, p.k_off + 64 * c, pid0);
          for (int h = 0; h < VSLABS && ok && !vf; ++h) ok = fill_slab(it, j, p.v_off + 64 * h, pid0);
        }
        pid0 = pid1;
        pid1 = pid2;
      }
    }
    // Outstanding copies land before the CTA may exit (they all have on the
    // normal path; after an abort some may still be in flight).
    if (lane == 0) {
      if constexpr (PG) {  // the last use of each part slot
        for (uint32_t t = tk > 2 ? tk - 2 : 0; t < tk; ++t)
          tc5::mbar_wait(bar(B_SLAB_FULL0 + kslot_slab(t)), (t >> 1) & 1u, abort_flag, p.err,
                         /*honor_abort=*/false);
        if (tv > 0)
          for (int h = 0; h < 2; ++h)
            tc5::mbar_wait(bar(B_SLAB_FULL0 + VSLOT_SLAB + h), (tv - 1) & 1u, abort_flag, p.err,
                           /*honor_abort=*/false);
      }
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
    constexpr uint32_t idesc_pv = tc5::idesc_bf16_f32(BM, DV, true);
    uint32_t qi = 0, fbase = 0;
    uint32_t pc[2] = {0, 0};  // P tiles consumed per query tile
    bool ok = true;
    auto wait = [&](int b, uint32_t parity) {
      if (ok) ok = tc5::mbar_wait(bar(b), parity, abort_flag, p.err);
      return ok;
    };
    auto slab_addr = [&](uint32_t fill) { return sbase + RING_OFF + (fill % NSLAB) * SLAB; };
    // a slot is free again once both CTAs' MMAs have read it
    auto release = [&](uint32_t slot) {
      tc5::mma_commit_mc(bar(B_SLAB_EMPTY0 + slot), CLUSTER_MASK);
    };
    auto wait_fill = [&](uint32_t fill) {
      return wait((F8 ? B_SLAB_READY0 : B_SLAB_FULL0) + fill % NSLAB, (fill / NSLAB) & 1u);
    };
    // S_x = Q_x K_j^T: K's slab c at address ka(c), 8-row groups kgs apart
    auto issue_s_at = [&](int x, uint32_t k0, uint32_t kstep, uint32_t kgs, bool ring) {
      tc5::tc_fence_after();
#pragma unroll
      for (int c = 0; c < KSLABS; ++c) {
        const uint32_t qa = sbase + Q_OFF + (x * KSLABS + c) * SLAB;
        // one slab a fill: slab c is fill k0 + c of the ring; page-grouped:
        // 1 KB on in every group of the part at k0
        const uint32_t ka = ring ? slab_addr(k0 + c) : k0 + kstep * c;
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
          tc5::mma_f16_ss(tmem + tm_s(x), tc5::sdesc_sw128(qa + 32 * kk, 16, 1024),
                          tc5::sdesc_sw128(ka + 32 * kk, 16, kgs), idesc_s,
                          (c | kk) != 0);
      }
      tc5::mma_commit(bar(B_SFULL0 + x));
    };
    // O_x += P_x V_j: N = 128 over V's two 64-column slabs (the leading byte
    // offset steps from one to the other: the next slab, or 1 KB on in a
    // page-grouped part), K = 16 keys (two 8-key groups) a step
    // (keys 16 k0 .. 16 k1 - 1 of the tile)
    auto issue_pv_at = [&](int x, uint32_t va, uint32_t lbo, uint32_t vgs, bool first, int k0,
                           int k1) {
      tc5::tc_fence_after();
#pragma unroll
      for (int kk = k0; kk < k1; ++kk)
        tc5::mma_f16_ts(tmem + tm_o(x), tmem + tm_s(x) + 8 * kk,
                        tc5::sdesc_sw128(va + kk * 2 * vgs, lbo, vgs), idesc_pv,
                        (!first || kk > 0) ? 1u : 0u);
    };
    uint32_t tcnt = 0;  // page-grouped: key tiles of the items so far
    for (int k = 0; ok; ++k) {
      Item it;
      if (!get_unit(p, TQ, unit_index(k), rank, it)) break;
      if (it.ntiles == 0) continue;
      const int n = it.ntiles;
      if (!wait(B_QFULL, qi & 1u)) break;
      if constexpr (PG) {
        // K parts in two alternating slots (tile t: slot t & 1), V parts in
        // one; each slot freed by this CTA's own commit
        const uint32_t t0 = tcnt;
        auto kwait = [&](uint32_t t) { return wait(B_SLAB_FULL0 + kslot_slab(t), (t >> 1) & 1u); };
        auto kaddr = [&](uint32_t t) { return sbase + RING_OFF + kslot_slab(t) * SLAB; };
        auto krelease = [&](uint32_t t) { tc5::mma_commit(bar(B_SLAB_EMPTY0 + kslot_slab(t))); };
        const uint32_t vaddr = sbase + RING_OFF + VSLOT_SLAB * SLAB;
        kwait(t0);
        if (!ok) break;
        issue_s_at(0, kaddr(t0), 1024u, KGROUP, false);
        issue_s_at(1, kaddr(t0), 1024u, KGROUP, false);
        if (n == 1) tc5::mma_commit(bar(B_QEMPTY));
        krelease(t0);
        for (int j = 0; j < n && ok; ++j) {
          const uint32_t t = t0 + static_cast<uint32_t>(j);
          for (int x = 0; x < 2 && ok; ++x) {
            if (x == 0) wait(B_SLAB_FULL0 + VSLOT_SLAB, t & 1u);  // V keys 0..63
            wait(B_PFULL0 + x, pc[x] & 1u);
            if (j == 0) wait(B_OFREE0 + x, (qi & 1u) ^ 1u);
            if (!ok) break;
            ++pc[x];
            issue_pv_at(x, vaddr, 1024u, VGROUP, j == 0, 0, BN / 32);
            // the first half is free once P.V_B has read it
            if (x == 1) tc5::mma_commit(bar(B_SLAB_EMPTY0 + VSLOT_SLAB));
            if (x == 0) wait(B_SLAB_FULL0 + VSLOT_SLAB + 1, t & 1u);  // V keys 64..127
            if (!ok) break;
            issue_pv_at(x, vaddr, 1024u, VGROUP, j == 0, BN / 32, BN / 16);
            if (j == n - 1) tc5::mma_commit(bar(B_ODONE0 + x));
            if (x == 1) tc5::mma_commit(bar(B_SLAB_EMPTY0 + VSLOT_SLAB + 1));
            if (j + 1 < n) {
              if (x == 0) kwait(t + 1);
              if (!ok) break;
              issue_s_at(x, kaddr(t + 1), 1024u, KGROUP, false);
              if (x == 1) {
                if (j + 2 == n) tc5::mma_commit(bar(B_QEMPTY));  // last S issued
                krelease(t + 1);
              }
            }
          }
        }
        tcnt += static_cast<uint32_t>(n);
        ++qi;
      } else {
      // S_A(0), S_B(0)
      for (int c = 0; c < KSLABS; ++c) wait_fill(k_fill(fbase, 0, c));
      if (!ok) break;
      issue_s_at(0, k_fill(fbase, 0, 0), 0u, 1024u, true);
      issue_s_at(1, k_fill(fbase, 0, 0), 0u, 1024u, true);
      if (n == 1) tc5::mma_commit(bar(B_QEMPTY));
      for (int c = 0; c < KSLABS; ++c)
        release(k_fill(fbase, 0, c) % NSLAB);
      for (int j = 0; j < n && ok; ++j) {
        for (int x = 0; x < 2 && ok; ++x) {
          if (x == 0)
            for (int h = 0; h < VSLABS; ++h) wait_fill(v_fill(fbase, j, h));
          wait(B_PFULL0 + x, pc[x] & 1u);
          if (j == 0) wait(B_OFREE0 + x, (qi & 1u) ^ 1u);
          if (!ok) break;
          ++pc[x];
          issue_pv_at(x, slab_addr(v_fill(fbase, j, 0)), static_cast<uint32_t>(SLAB), 1024u,
                      j == 0, 0, BN / 16);
          if (j == n - 1) tc5::mma_commit(bar(B_ODONE0 + x));
          if (x == 1)
            for (int h = 0; h < VSLABS; ++h)
              release(v_fill(fbase, j, h) % NSLAB);
          if (j + 1 < n) {
            if (x == 0)
              for (int c = 0; c < KSLABS; ++c) wait_fill(k_fill(fbase, j + 1, c));
            if (!ok) break;
            issue_s_at(x, k_fill(fbase, j + 1, 0), 0u, 1024u, true);
            if (x == 1) {
              if (j + 2 == n) tc5::mma_commit(bar(B_QEMPTY));  // last S issued
              for (int c = 0; c < KSLABS; ++c)
                release(k_fill(fbase, j + 1, c) % NSLAB);
            }
          }
        }
      }
      fbase += FILLS_PER_TILE * static_cast<uint32_t>(n);
      ++qi;
      }
    }
    // drain: every MMA issued above has completed before TMEM is freed
    tc5::mma_commit(bar(B_FINAL));
    tc5::mbar_wait(bar(B_FINAL), 0, abort_flag, p.err, /*honor_abort=*/false);
  }
  } else if (F8 && warp >= 12) {
    // Registers: the FP8 block is launched with 512 x 128; the control
    // warpgroup keeps 104, the widening warpgroup 40, and the two softmax
    // warpgroups take 184 (128 x 104 + 128 x 40 + 256 x 184 = 65,536).
    asm volatile("setmaxnreg.dec.sync.aligned.u32 40;\n" ::: "memory");
    // ------------------------------------------------ E4M3 widening -----
    // Warps 12..15 take the ring fills in the producer's order: wait for a
    // fill to land, widen it in place, make the bf16 rows visible to the
    // tensor core, and mark the slab ready.
    const int ct = threadIdx.x - 384;
    uint32_t f = 0;
    bool ok = true;
    for (int k = 0; ok; ++k) {
      Item it;
      if (!get_unit(p, TQ, unit_index(k), rank, it)) break;
      const uint32_t nf = FILLS_PER_TILE * static_cast<uint32_t>(it.ntiles);
      for (uint32_t i = 0; i < nf; ++i, ++f) {
        const uint32_t slot = f % NSLAB;
        const bool w = tc5::mbar_wait(bar(B_SLAB_FULL0 + slot), (f / NSLAB) & 1u, abort_flag,
                                      p.err);
        // all four warps take the same decision to stop
        if (barrier_or(kWidenBar, kWidenThreads, !w)) {
          ok = false;
          break;
        }
        widen_slab(smem + RING_OFF + slot * SLAB, ct);
        tc5::fence_proxy_async_smem();
        named_barrier(kWidenBar, kWidenThreads);
        if (ct == 0) tc5::mbar_arrive(bar(B_SLAB_READY0 + slot));
      }
    }
  } else {
    // bf16 block: 384 x 168 at launch, control 120, softmax 192
    // (128 x 120 + 256 x 192 = 64,512); FP8 block: softmax 184 (above)
    if constexpr (F8)
      asm volatile("setmaxnreg.inc.sync.aligned.u32 184;\n" ::: "memory");
    else
      asm volatile("setmaxnreg.inc.sync.aligned.u32 192;\n" ::: "memory");
    // ------------------------------------------------ softmax -----------
    // Warps 4..7 own query tile A, warps 8..11 tile B; one thread per row.
    const int x = (warp - 4) >> 2;                 // query tile of this warp
    const int r = (threadIdx.x - 128) & 127;       // its row of the tile
    const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const uint32_t ts = tmem + lane_off + tm_s(x), to = tmem + lane_off + tm_o(x);
    const float scale_log2_base = p.softmax_scale * kLog2e;
    uint32_t sc = 0;  // S tiles seen
    uint32_t items = 0, fbase = 0;
    uint32_t tcnt = 0;  // page-grouped: key tiles of the items so far
    // waits whose outcome is the same for the whole warp, so that the warp
    // stays converged for the warp-collective tensor-memory accesses
    auto wwait = [&](uint32_t b, uint32_t parity) {
      const bool rr = tc5::mbar_wait(b, parity, abort_flag, p.err);
      return __all_sync(0xffffffffu, rr);
    };
    for (int k = 0;; ++k) {
      Item it;
      if (!get_unit(p, TQ, unit_index(k), rank, it)) break;
      // FP8 caches (their codes widened to bf16): k_scale joins the softmax
      // scale and v_scale the output, for this item's KV head
      float scale_log2 = scale_log2_base, v_mul = 1.f;
      if (p.fold_scales) {
        const int si = p.scale_mode == PKV_SCALE_HEAD ? it.g : 0;
        scale_log2 *= __ldg(p.k_scale + si);
        v_mul = __ldg(p.v_scale + si);
      }
      const int tr = r / G, hr = r % G;
      const bool valid = tr < it.nq[x];
      const int pos = it.minpos[x] + tr;
      const int64_t orow =
          (static_cast<int64_t>(it.q0[x] + tr) * p.num_q_heads + it.g * G + hr) * DV;
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
      for (int j = 0; j < it.ntiles && ok; ++j) {
        const int kbase = j * BN;
        if (!wwait(bar(B_SFULL0 + x), sc & 1u)) {
          ok = false;
          break;
        }
        ++sc;
        tc5::tc_fence_after();
        const bool masked = !valid || kbase + BN - 1 > pos;
        float sv[BN];
        {
          uint32_t v[BN / 32][32];
#pragma unroll
          for (int c = 0; c < BN / 32; ++c) tc5::tmem_ld_32x32b_x32(ts + 32 * c, v[c]);
          tc5::tmem_wait_ld();
#pragma unroll
          for (int c = 0; c < BN / 32; ++c)
#pragma unroll
            for (int k = 0; k < 32; ++k) sv[32 * c + k] = __uint_as_float(v[c][k]);
        }
        if (masked) {
#pragma unroll
          for (int c = 0; c < BN; ++c)
            if (!valid || kbase + c > pos) sv[c] = -INFINITY;
        }
        float mx;
        {
          // eight chains of three-input maxima
          float mc[8];
#pragma unroll
          for (int k = 0; k < 8; ++k) mc[k] = sv[k];
#pragma unroll
          for (int c = 8; c < BN; c += 16)
#pragma unroll
            for (int k = 0; k < 8; ++k) mc[k] = fmax3(mc[k], sv[c + k], sv[c + 8 + k]);
          mx = fmax3(fmax3(mc[0], mc[1], mc[2]), fmax3(mc[3], mc[4], mc[5]),
                     fmaxf(mc[6], mc[7]));
        }
        const float m_new = fmaxf(m, mx * scale_log2);
        // The rescale touches O with warp-collective tensor-memory loads and
        // stores, so it is decided per warp; PV(j-1) has completed (the
        // commit behind S(j) covers it).  It runs after the exponentials,
        // once S is no longer held in registers, and before P is published,
        // so the next P.V MMA sees the rescaled O.
        const bool need = j > 0 && m_new > m + kRescaleThreshold;
        bool rescale = false;
        float alpha = 1.f;
        if (j == 0) {
          m = m_new;
        } else if (__any_sync(0xffffffffu, need)) {
          alpha = m_new == -INFINITY ? 1.f : fast_exp2(m - m_new);
          l *= alpha;
          m = m_new;
          rescale = true;
        }
        const float base = m == -INFINITY ? 0.f : m;
        // P (bf16) over the first 64 columns of S; the exponent arguments
        // and the running sums go two at a time (packed f32x2)
        const uint64_t sc2 = f2_pack(scale_log2, scale_log2);
        const uint64_t nb2 = f2_pack(-base, -base);
        uint64_t ls2[2] = {f2_pack(0.f, 0.f), f2_pack(0.f, 0.f)};
#pragma unroll
        for (int c = 0; c < BN / 32; ++c) {
          uint32_t pk[16];
#pragma unroll
          for (int k = 0; k < 16; ++k) {
            float a0, a1;
            f2_unpack(f2_fma(f2_pack(sv[32 * c + 2 * k], sv[32 * c + 2 * k + 1]), sc2, nb2),
                      a0, a1);
            const float p0 = fast_exp2(a0);
            const float p1 = fast_exp2(a1);
            ls2[k & 1] = f2_add(ls2[k & 1], f2_pack(p0, p1));
            pk[k] = pack_bf16x2(p0, p1);
          }
          tc5::tmem_st_32x32b_x16(ts + 16 * c, pk);
        }
        {
          float s0, s1, s2, s3;
          f2_unpack(ls2[0], s0, s1);
          f2_unpack(ls2[1], s2, s3);
          l += (s0 + s1) + (s2 + s3);
        }
        if (rescale) {  // warp-uniform
#pragma unroll
          for (int c = 0; c < DV / 32; ++c) {
            uint32_t v[32];
            tc5::tmem_ld_32x32b_x32(to + 32 * c, v);
            tc5::tmem_wait_ld();
#pragma unroll
            for (int k = 0; k < 32; ++k) v[k] = __float_as_uint(__uint_as_float(v[k]) * alpha);
            tc5::tmem_st_32x32b_x32(to + 32 * c, v);
          }
        }
        tc5::tmem_wait_st();
        bool zeroed = false;
        if (x == 0 && kbase + BN > it.L) {
          // last tile: zero the V rows of keys past the sequence end (one
          // slab a fill: row r of each V slab; page-grouped: key r's 8-key
          // group of the V slot holds its row of both slabs, 1 KB apart)
          const uint32_t tv = tcnt + static_cast<uint32_t>(j);  // page-grouped tile
          for (int h = 0; h < VSLABS && ok; ++h) {
            const uint32_t fi = v_fill(fbase, j, h);
            if constexpr (PG)  // the V half that holds this warp's 32 rows
              ok = h > 0 || wwait(bar(B_SLAB_FULL0 + VSLOT_SLAB + (r >> 6)), tv & 1u);
            else
              ok = wwait(bar((F8 ? B_SLAB_READY0 : B_SLAB_FULL0) + fi % NSLAB),
                         (fi / NSLAB) & 1u);
            if (ok && kbase + r >= it.L) {
              const uint32_t off =
                  PG ? VSLOT_SLAB * SLAB + (r >> 3) * VGROUP + h * 1024 + (r & 7) * 128
                     : (fi % NSLAB) * SLAB + r * 128;
              uint4* vrow = reinterpret_cast<uint4*>(smem + RING_OFF + off);
#pragma unroll
              for (int ch = 0; ch < 8; ++ch) vrow[ch] = make_uint4(0, 0, 0, 0);
            }
          }
          zeroed = true;
        }
        if (!ok) break;
        if (zeroed) tc5::fence_proxy_async_smem();
        tc5::tc_fence_before();
        tc5::mbar_arrive(bar(B_PFULL0 + x));
      }
      if (!ok) break;
      // ---- epilogue: O / l -> bf16 ----
      if (!wwait(bar(B_ODONE0 + x), items & 1u)) break;
      tc5::tc_fence_after();
      if (p.sinks != nullptr && valid && m != -INFINITY) {
        // the attention sink: one more logit in the denominator, no value
        const float sk = __ldg(p.sinks + it.g * G + hr);
        if (sk != -INFINITY) l += fast_exp2(fmaf(sk, kLog2e, -m));
      }
      const float inv = l > 0.f ? v_mul / l : 0.f;
      uint4* dst = reinterpret_cast<uint4*>(p.out + orow);
#pragma unroll
      for (int c = 0; c < DV / 32; ++c) {
        uint32_t v[32];
        tc5::tmem_ld_32x32b_x32(to + 32 * c, v);
        tc5::tmem_wait_ld();
        if (valid) {
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            auto o2 = [&](int i) {
              return pack_bf16x2(__uint_as_float(v[8 * k + i]) * inv,
                                 __uint_as_float(v[8 * k + i + 1]) * inv);
            };
            dst[4 * c + k] = make_uint4(o2(0), o2(2), o2(4), o2(6));
          }
        }
      }
      tc5::tc_fence_before();
      tc5::mbar_arrive(bar(B_OFREE0 + x));
      fbase += FILLS_PER_TILE * static_cast<uint32_t>(it.ntiles);
      tcnt += static_cast<uint32_t>(it.ntiles);
      ++items;
    }
  }

  tc5::tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc5::tc_fence_after();
    tc5::tmem_dealloc(tmem, TMEM_COLS);
  }
  // Neither CTA leaves while the other may still signal its barriers (the
  // MMA commits that free ring slots arrive in both CTAs).
  tc5::cluster_sync();
}

}  // namespace

bool prefill_supported(int head_size, int head_size_v, int dtype) {
  return head_size == DK && head_size_v == DV && (dtype == PKV_BF16 || dtype == PKV_FP8_E4M3);
}

cudaError_t launch_prefill(const AttnParams& p, int num_sms,
                           cudaStream_t stream) {
  if (!prefill_supported(p.head_size, p.head_size_v, p.dtype))
    return cudaErrorNotSupported;
  PFN_cuTensorMapEncodeTiled_v12000 encode = tmap_encode_fn();
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
  const int box_rows = p.block_size < BN ? p.block_size : BN;
  const bool f8 = p.dtype == PKV_FP8_E4M3;
  // bf16 rows that split into 64-column slabs: page-grouped boxes of up to
  // 16 keys (a page's three K slabs in one box, its two V slabs in another;
  // on the 32K causal prefill 3.83-3.89 ms at pages of 16 to 256 keys and
  // 4.26 ms at 8, against 4.21-5.73 ms for slab fills); other bf16 rows:
  // one 64-column box per slab in the MMAs' 128-byte swizzle; FP8: 64-column
  // boxes of E4M3 codes landing densely, widened in shared memory
  const bool pg = !f8 && p.row_elems % 64 == 0 && p.k_off % 64 == 0 && p.v_off % 64 == 0 &&
                  box_rows % 8 == 0;
  alignas(64) CUtensorMap v_map;
  if (pg) {
    const int pg_rows = p.block_size < 16 ? p.block_size : 16;  // as in the kernel
    if (!make_cache_tmap_groups(&kv_map, p.cache, p.layout, p.num_blocks, p.block_size,
                                p.num_kv_heads, p.row_elems, KSLABS, pg_rows) ||
        !make_cache_tmap_groups(&v_map, p.cache, p.layout, p.num_blocks, p.block_size,
                                p.num_kv_heads, p.row_elems, VSLABS, pg_rows))
      return cudaErrorInvalidValue;
  } else {
    if (!make_cache_tmap(&kv_map, p.cache, p.dtype, p.layout, p.num_blocks,
                         p.block_size, p.num_kv_heads, p.row_elems, 64, box_rows,
                         /*swizzle64=*/false, /*no_swizzle=*/f8))
      return cudaErrorInvalidValue;
    v_map = kv_map;  // unused
  }
  const int variant = f8 ? 1 : pg ? 2 : 0;
  auto kernel = f8 ? prefill_kernel<true, false>
                   : pg ? prefill_kernel<false, true> : prefill_kernel<false, false>;
  static int attr_set[3][64] = {{0}};
  cudaError_t e = ensure_smem_attr(kernel, SMEM_BYTES, attr_set[variant]);
  if (e != cudaSuccess) return e;
  // Persistent: as many CTA pairs (clusters) as can be resident at once.
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = CLUSTER;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(num_sms / CLUSTER * CLUSTER));
  cfg.blockDim = dim3(f8 ? THREADS_F8 : THREADS);
  cfg.dynamicSmemBytes = SMEM_BYTES;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int dev = 0;
  e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  static int max_clusters[3][64] = {{0}};
  int ncl = dev < 64 ? max_clusters[variant][dev] : 0;
  if (ncl == 0) {
    e = cudaOccupancyMaxActiveClusters(&ncl, kernel, &cfg);
    if (e != cudaSuccess) return e;
    if (ncl < 1) return cudaErrorNotSupported;
    if (dev < 64) max_clusters[variant][dev] = ncl;
  }
  if (ncl > num_sms / CLUSTER) ncl = num_sms / CLUSTER;
  cfg.gridDim = dim3(static_cast<unsigned>(ncl * CLUSTER));
  e = cudaLaunchKernelEx(&cfg, kernel, q_map, kv_map, v_map, p);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace pkv
