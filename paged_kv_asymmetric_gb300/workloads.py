"""Seeded synthetic workloads for paged-KV attention with asymmetric heads.

This module only draws inputs: sequence lengths, page placement, Q/K/V values
and (for FP8 caches) the per-head scales chosen from the drawn values.  It
holds none of the attention arithmetic, so both the CUDA path and the CPU
oracle can take their inputs from it.

The shapes follow the workloads the pages run: MiMo-V2.6's global attention
layers (16 query / 4 KV heads per rank, K 192 / V 128, block size 16 or 64,
vLLM PR #64064 "Validation" and "Details"; the MiMo-V2.6-Flash 2x RTX PRO 6000
model card, "Benchmarks": ~46K-token prompts, FP8 E4M3 KV cache, 1+3-token
speculative verify) and the Kimi K3 MLA decode shape (12 query heads per rank,
one latent head, D 576 / 512, 100K context; vLLM PR #50371 "Purpose" and
"Test Plan").  No dataset is involved: every value is N(0, 1) from a seeded
torch generator.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional

import numpy as np
import torch

BF16, FP8 = "bf16", "fp8"
NHD, HND = "nhd", "hnd"
SCALE_NONE, SCALE_TENSOR, SCALE_HEAD = "none", "tensor", "head"
FP8_E4M3_MAX = 448.0


@dataclasses.dataclass
class Workload:
    name: str
    num_q_heads: int
    num_kv_heads: int
    head_size: int          # dk
    head_size_v: int        # dv
    row_elems: int          # R
    k_off: int
    v_off: int
    block_size: int
    kv_dtype: str           # "bf16" | "fp8"
    scale_mode: str         # "none" | "tensor" | "head"
    layout: str             # "nhd" | "hnd"
    softmax_scale: float
    seq_lens: np.ndarray    # int32 [B]   keys per sequence, new tokens included
    q_lens: np.ndarray      # int32 [B]
    query_start_loc: np.ndarray  # int32 [B+1]
    block_table: np.ndarray      # int32 [B, max_blocks] (-1 = no page)
    num_blocks: int
    # context: every key/value of every sequence, in sequence order
    ctx_start: np.ndarray   # int64 [B+1] offsets into k_ctx / v_ctx
    k_ctx: torch.Tensor     # bf16 [sum L, Hkv, dk]
    v_ctx: Optional[torch.Tensor]  # bf16 [sum L, Hkv, dv] (None: V aliases K)
    q: torch.Tensor         # bf16 [T, Hq, dk]
    k_scale: Optional[np.ndarray]  # float32 [1] or [Hkv]
    v_scale: Optional[np.ndarray]
    max_splits: int = 16

    # ------------------------------------------------------------ helpers --
    @property
    def num_seqs(self) -> int:
        return int(self.seq_lens.shape[0])

    @property
    def num_tokens(self) -> int:
        return int(self.query_start_loc[-1])

    @property
    def max_query_len(self) -> int:
        return int(self.q_lens.max()) if self.q_lens.size else 0

    def slot_mapping_all(self) -> np.ndarray:
        """Slots of every context token (in k_ctx order)."""
        return slot_mapping_for(self, np.arange(self.num_seqs), new_only=False)

    def slot_mapping_new(self) -> np.ndarray:
        """Slots of the query tokens (the last q_len keys of each sequence),
        in query-token order: the write a decode / verify / prefill step
        performs before it attends."""
        return slot_mapping_for(self, np.arange(self.num_seqs), new_only=True)

    def new_kv_index(self) -> np.ndarray:
        """Row indices into k_ctx / v_ctx of the query tokens."""
        idx = []
        for b in range(self.num_seqs):
            L, ql = int(self.seq_lens[b]), int(self.q_lens[b])
            lo = int(self.ctx_start[b])
            n_new = min(ql, L)
            idx.extend(range(lo + L - n_new, lo + L))
            idx.extend([-1] * (ql - n_new))  # query rows without a key slot
        return np.asarray(idx, dtype=np.int64)

    def cache_bytes(self) -> int:
        e = 2 if self.kv_dtype == BF16 else 1
        return self.num_blocks * self.block_size * self.num_kv_heads * \
            self.row_elems * e


def slot_mapping_for(w: Workload, seqs, new_only: bool) -> np.ndarray:
    out = []
    for b in seqs:
        b = int(b)
        L = int(w.seq_lens[b])
        ql = int(w.q_lens[b])
        if new_only:
            n_new = min(ql, L)
            pos = list(range(L - n_new, L))
            pad = ql - n_new
        else:
            pos, pad = list(range(L)), 0
        for j in pos:
            out.append(int(w.block_table[b, j // w.block_size]) * w.block_size
                       + j % w.block_size)
        out.extend([-1] * pad)
    return np.asarray(out, dtype=np.int64)


def _randn(gen, shape, device):
    return torch.randn(*shape, generator=gen, dtype=torch.float32,
                       device=device).to(torch.bfloat16)


def make_workload(name: str, *, seq_lens, q_lens, num_q_heads=16,
                  num_kv_heads=4, head_size=192, head_size_v=128,
                  row_elems=None, k_off=0, v_off=None, block_size=16,
                  kv_dtype=BF16, scale_mode=SCALE_NONE, layout=NHD,
                  softmax_scale=None, seed=0, extra_blocks=0,
                  v_aliases_k=False, pad_q_heads=0, max_splits=16,
                  device="cpu") -> Workload:
    """Draw one workload.  Page placement is a random permutation of the
    pool of pages; unused block-table entries are -1 (never read)."""
    seq_lens = np.asarray(seq_lens, dtype=np.int32)
    q_lens = np.asarray(q_lens, dtype=np.int32)
    B = int(seq_lens.shape[0])
    if v_off is None:
        v_off = 0 if v_aliases_k else head_size
    if row_elems is None:
        row_elems = head_size if v_aliases_k else head_size + head_size_v
    if softmax_scale is None:
        softmax_scale = 1.0 / math.sqrt(head_size)
    gen = torch.Generator(device="cpu").manual_seed(seed)
    pages = [(int(L) + block_size - 1) // block_size for L in seq_lens]
    total_pages = sum(pages) + extra_blocks
    perm = torch.randperm(max(total_pages, 1), generator=gen).numpy()
    max_blocks = max(max(pages) if pages else 1, 1)
    bt = np.full((B, max_blocks), -1, dtype=np.int32)
    k = 0
    for b in range(B):
        for p in range(pages[b]):
            bt[b, p] = perm[k]
            k += 1
    qsl = np.zeros(B + 1, dtype=np.int32)
    qsl[1:] = np.cumsum(q_lens)
    cst = np.zeros(B + 1, dtype=np.int64)
    cst[1:] = np.cumsum(seq_lens.astype(np.int64))
    T = int(qsl[-1])
    nctx = int(cst[-1])
    dgen = gen
    if device != "cpu":
        dgen = torch.Generator(device=device).manual_seed(seed + 1)
    k_ctx = _randn(dgen, (nctx, num_kv_heads, head_size), device)
    v_ctx = None if v_aliases_k else _randn(
        dgen, (nctx, num_kv_heads, head_size_v), device)
    q = _randn(dgen, (T, num_q_heads, head_size), device)
    if pad_q_heads:
        # zero-valued extra query heads appended after the real ones
        q = torch.cat([q, torch.zeros(T, pad_q_heads, head_size,
                                      dtype=q.dtype, device=q.device)], 1)
        num_q_heads += pad_q_heads
    k_scale = v_scale = None
    if kv_dtype == FP8:
        k_scale = _choose_scales(k_ctx, scale_mode)
        v_scale = _choose_scales(v_ctx if v_ctx is not None else k_ctx,
                                 scale_mode)
    return Workload(
        name=name, num_q_heads=num_q_heads, num_kv_heads=num_kv_heads,
        head_size=head_size, head_size_v=head_size_v, row_elems=row_elems,
        k_off=k_off, v_off=v_off, block_size=block_size, kv_dtype=kv_dtype,
        scale_mode=scale_mode, layout=layout,
        softmax_scale=float(softmax_scale), seq_lens=seq_lens, q_lens=q_lens,
        query_start_loc=qsl, block_table=bt, num_blocks=max(total_pages, 1),
        ctx_start=cst, k_ctx=k_ctx, v_ctx=v_ctx, q=q, k_scale=k_scale,
        v_scale=v_scale, max_splits=max_splits)


def _choose_scales(x: torch.Tensor, mode: str) -> np.ndarray:
    """FP8 scales as the verify workload specifies them: absmax / 448 over
    the whole tensor or over each KV head (binary32)."""
    xf = x.float().abs()
    if mode == SCALE_TENSOR:
        a = xf.max().reshape(1)
    else:
        a = xf.amax(dim=(0, 2))
    s = (a / FP8_E4M3_MAX).cpu().numpy().astype(np.float32)
    s[s == 0] = 1.0
    return s


# ------------------------------------------------------- the named workloads --

def tiny(phase: str = "decode", layout=NHD, kv_dtype=BF16,
         scale_mode=SCALE_NONE, device="cpu") -> Workload:
    """2 sequences of 37 and 64 keys, Hq 16 / Hkv 4, K192/V128, block 16,
    random page placement, seed 0; q_len 1 (decode) or q_len = L (prefill)."""
    L = [37, 64]
    ql = [1, 1] if phase == "decode" else L
    return make_workload(f"tiny-{phase}", seq_lens=L, q_lens=ql,
                         layout=layout, kv_dtype=kv_dtype,
                         scale_mode=scale_mode, extra_blocks=3, seed=0,
                         max_splits=4, device=device)


def batched_decode(device="cpu", seed=0) -> Workload:
    """32 sequences, context U[2048, 8192], q_len 1, Hq 16 / Hkv 4,
    K192/V128, block 16, bf16, scale 1/sqrt(192)."""
    g = np.random.default_rng(seed)
    L = g.integers(2048, 8192, size=32, endpoint=True)
    return make_workload("batched-decode", seq_lens=L, q_lens=[1] * 32,
                         seed=seed, max_splits=16, device=device)


def long_prefill(n_tokens: int = 32768, device="cpu", seed=0) -> Workload:
    """One sequence of n_tokens, causal prefill over the paged cache."""
    return make_workload(f"prefill-{n_tokens}", seq_lens=[n_tokens],
                         q_lens=[n_tokens], seed=seed, device=device)


def verify_fp8(device="cpu", seed=0, n_real=16, n_pad=8,
               ctx=46_000) -> Workload:
    """16 sequences at ~46K keys (+-10% uniform), q_len 4 (1 + 3 draft
    tokens), FP8 E4M3 cache with per-head scales (absmax / 448), block 64,
    16 split-KV segments, plus 8 padded rows with seq_len 0."""
    g = np.random.default_rng(seed)
    lo, hi = int(ctx * 0.9), int(ctx * 1.1)
    L = list(g.integers(lo, hi, size=n_real, endpoint=True)) + [0] * n_pad
    return make_workload("verify-fp8", seq_lens=L, q_lens=[4] * len(L),
                         block_size=64, kv_dtype=FP8, scale_mode=SCALE_HEAD,
                         seed=seed, max_splits=16, device=device)


def mla_decode(batch: int = 1, heads: int = 12, ctx: int = 100_000,
               device="cpu", seed=0) -> Workload:
    """MLA-shaped decode: 1 latent KV head of 576, V = its first 512 dims,
    `heads` query heads (12, or 16 with heads 12..15 zero), block 64."""
    return make_workload(f"mla-b{batch}-h{heads}", seq_lens=[ctx] * batch,
                         q_lens=[1] * batch, num_q_heads=min(heads, 12),
                         pad_q_heads=max(heads - 12, 0),
                         num_kv_heads=1, head_size=576, head_size_v=512,
                         block_size=64, v_aliases_k=True,
                         softmax_scale=1.0 / math.sqrt(576), seed=seed,
                         max_splits=64, device=device)


# ------------------------------------------------------ device marshalling --

@dataclasses.dataclass
class DeviceWorkload:
    """The tensors of a workload on a CUDA device, ready for the library."""
    w: Workload
    cache: object            # paged_kv_asymmetric_gb300.Cache
    cache_buf: torch.Tensor  # uint8 storage: slack | cache | slack
    slack: int
    q: torch.Tensor
    k_ctx: torch.Tensor
    v_ctx: Optional[torch.Tensor]
    slots_all: torch.Tensor
    slots_new: torch.Tensor
    new_idx: torch.Tensor
    block_table: torch.Tensor
    seq_lens: torch.Tensor
    query_start_loc: torch.Tensor
    k_scale: Optional[torch.Tensor]
    v_scale: Optional[torch.Tensor]


def desc_of(w: Workload):
    from paged_kv_asymmetric_gb300 import (BF16 as _B, FP8_E4M3 as _F,
                                           NHD as _N, HND as _H, make_desc)
    return make_desc(
        dtype=_B if w.kv_dtype == BF16 else _F,
        layout=_N if w.layout == NHD else _H, num_blocks=w.num_blocks,
        block_size=w.block_size, num_kv_heads=w.num_kv_heads,
        row_elems=w.row_elems, k_off=w.k_off, head_size=w.head_size,
        v_off=w.v_off, head_size_v=w.head_size_v,
        scale_mode={SCALE_NONE: 0, SCALE_TENSOR: 1, SCALE_HEAD: 2}[w.scale_mode])


def to_device(w: Workload, device="cuda", fill_byte: int = 0xFF,
              slack: int = 4096) -> DeviceWorkload:
    """Copies a workload to the device.  The cache is allocated with `slack`
    guard bytes on both sides and every byte (guards included) set to
    fill_byte (0xFF reads as NaN in both bf16 and E4M3, so an unwritten slot
    that leaked into a result would show)."""
    from paged_kv_asymmetric_gb300 import Cache
    d = desc_of(w)
    nbytes = w.cache_bytes()
    buf = torch.full((nbytes + 2 * slack,), fill_byte, dtype=torch.uint8,
                     device=device)
    cache = Cache(buf[slack:slack + nbytes], d)
    f32 = lambda a: None if a is None else torch.from_numpy(
        np.asarray(a, dtype=np.float32)).to(device)
    return DeviceWorkload(
        w=w, cache=cache, cache_buf=buf, slack=slack,
        q=w.q.to(device).contiguous(), k_ctx=w.k_ctx.to(device),
        v_ctx=None if w.v_ctx is None else w.v_ctx.to(device),
        slots_all=torch.from_numpy(w.slot_mapping_all()).to(device),
        slots_new=torch.from_numpy(w.slot_mapping_new()).to(device),
        new_idx=torch.from_numpy(w.new_kv_index()).to(device),
        block_table=torch.from_numpy(w.block_table).to(device),
        seq_lens=torch.from_numpy(w.seq_lens).to(device),
        query_start_loc=torch.from_numpy(w.query_start_loc).to(device),
        k_scale=f32(w.k_scale), v_scale=f32(w.v_scale))
