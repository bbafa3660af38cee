"""Benchmark: paged decode HBM GB/s and prefill TFLOP/s (K192/V128) on GB300.

Headline step (``value``): one batched decode step of the library's hot path
on the batched-decode workload (32 sequences, context U[2048, 8192], q_len 1,
16 query / 4 KV heads, K 192 / V 128, block 16, bf16): write the step's new
K/V into the paged cache, split-KV decode with balanced ranges (at most 16
segments per sequence, cut on the device from seq_lens), merge.  ``value`` is the step's
algorithmic HBM bytes (every visible K|V row once per KV head, Q, O, block
table, and the write's reads and writes) per second of device time.  The
KV cache (419 MB) is larger than L2, so no flush is needed between steps.

``roofline`` is the decode kernel alone: its launches back to back on the
stream (no event between them), timed in a loop of their own after the
headline loop, which runs with no event inside it.

Also reported (``sub``): causal prefill TFLOP/s at 32,768 and 131,072 tokens
and their cache writes, the 32,768-token prefill over an FP8 cache,
speculative verify with an FP8 cache (16 x ~46K, q_len 4, 16 splits, 8
padded rows) and the MLA-shaped decode (100K context, 12 and 16 heads, batch
1 and 16).  Those are timed per launch with L2 flushed between launches;
the decode sub-benchmarks also time the decode and its merge launched back
to back as a step launches them (``step_ms``, one flush before the pair),
and, where the KV cache is larger than L2 (verify, MLA batch 16), a loop of
such steps with no flush and no event inside it (``loop_step_ms``), the
steps alternating between two copies of the cache so that no step can find
the previous step's pages in L2.
The prefill loads K/V tiles with TMA multicast between the two CTAs of a
cluster, which is for single-GPU jobs only: a run with more than one rank
takes no prefill measurement (and ``--only prefill`` refuses to run).

``--impl reference`` times the CPU oracle (the reference arm of this build:
no third-party implementation of this path runs on GB300) on a bounded sample
of the same workload.  With several GPUs (torchrun, ``--gpus N`` equal to
its WORLD_SIZE), every rank runs an independent replica of the decode step
(the path has no exchange step): ``scaling`` is weak.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "paged decode HBM GB/s & prefill TFLOP/s (K192/V128), % of GB300 roofline"
FALLBACK = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0,
            "bf16_tflops_sustained": 1700.0}
L2_FLUSH_BYTES = 512 << 20


# ------------------------------------------------------------- plumbing --

def dist_info():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def init_dist(ws, backend):
    if ws > 1 and not torch.distributed.is_initialized():
        torch.distributed.init_process_group(backend=backend)


def barrier(ws):
    if ws > 1:
        torch.distributed.barrier()


def max_over_ranks(x: float, ws: int, device=None) -> float:
    """The largest value of x over all ranks (x itself with one rank)."""
    if ws <= 1:
        return float(x)
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def sum_over_ranks(x: float, ws: int, device=None) -> float:
    if ws <= 1:
        return float(x)
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.SUM)
    return float(t.item())


PREFILL_KINDS = ("prefill", "prefill_fp8")


def require_single_gpu(ws: int, what: str) -> None:
    """The prefill's K/V tiles are multicast by TMA between the two CTAs of a
    cluster; that load is for jobs on one GPU only."""
    if ws != 1:
        raise RuntimeError(f"{what}: the cluster-multicast prefill runs in "
                           f"single-GPU jobs only (world size {ws})")


def sub_plan(args, ws: int):
    """The sub-measurements of a run, in order, as (kind, name, size).
    Prefill kinds appear only when the job has one rank."""
    plan = []
    if args.no_sub:
        return plan
    if ws == 1 and not args.skip_prefill:
        plan += [("prefill", "prefill_32k", 32768),
                 ("prefill_fp8", "prefill_fp8_32k", 32768),
                 ("prefill", "prefill_128k", 131072),
                 ("prefill_fp8", "prefill_fp8_128k", 131072)]
    plan.append(("verify", "verify_fp8", 16))
    plan += [("mla", f"mla_b{b}_h{h}", (b, h)) for b in (1, 16) for h in (12, 16)]
    return plan


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return d, "measured"
    return dict(FALLBACK), "fallback"


class ClockSampler:
    """nvidia-smi clock / throttle samples while the timed regions run."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.Q}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no nvidia-smi"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) >= 9:
                    rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None
        sm = [num(r[1]) for r in rows if num(r[1]) is not None]
        mx = [num(r[2]) for r in rows if num(r[2]) is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown",
                 "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4)
                          if r[5 + i].lower().startswith("active")})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(rows)}


def traffic_record(kernel: str):
    """DRAM bytes per launch from a committed ncu summary, if the kernel
    sources are unchanged since the capture (else None)."""
    import hashlib
    path = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        rec = json.load(f).get(kernel)
    if not rec:
        return None
    h = hashlib.sha256()
    for src in rec.get("sources", []):
        with open(os.path.join(ROOT, src), "rb") as f:
            h.update(f.read())
    if h.hexdigest() != rec.get("sha256"):
        return None
    return rec.get("bytes_per_launch")


# --------------------------------------------------- algorithmic counts --

def decode_bytes(w) -> int:
    """Visible K|V rows once per KV head (V inside K counted once), Q, O
    (bf16) and the block-table entries read."""
    e = 2 if w.kv_dtype == "bf16" else 1
    lo = min(w.k_off, w.v_off)
    hi = max(w.k_off + w.head_size, w.v_off + w.head_size_v)
    kv = int(np.sum(w.seq_lens.astype(np.int64))) * w.num_kv_heads * (hi - lo) * e
    q = w.num_tokens * w.num_q_heads * w.head_size * 2
    o = w.num_tokens * w.num_q_heads * w.head_size_v * 2
    bt = int(sum((int(L) + w.block_size - 1) // w.block_size for L in w.seq_lens)) * 4
    return kv + q + o + bt


def write_bytes(w, n_tokens: int) -> int:
    e = 2 if w.kv_dtype == "bf16" else 1
    per = w.num_kv_heads * (w.head_size + (w.head_size_v if w.v_ctx is not None else 0))
    return n_tokens * (per * 2 + per * e + 8)


def prefill_flops(w) -> float:
    """2 * (dk + dv) multiply-adds per visible (query row, key) pair and
    query head; masked pairs excluded."""
    tot = 0
    for b in range(w.num_seqs):
        L, ql = int(w.seq_lens[b]), int(w.q_lens[b])
        for_rows = 0
        # keys seen by query i: clamp(L - ql + i + 1, 0, L)
        first = L - ql + 1
        lo_i = max(0, -first + 1)
        n = ql - lo_i
        a = first + lo_i
        for_rows = n * a + n * (n - 1) // 2
        tot += for_rows
    return float(tot) * w.num_q_heads * 2 * (w.head_size + w.head_size_v)


# ----------------------------------------------------------- GPU arm ----

class Flusher:
    """Evicts L2 between timed launches: writes a buffer larger than L2 and
    then reads it back, so that L2 holds clean lines of the flush buffer (no
    write-back of flush data lands inside the next timed launch)."""
    def __init__(self, device):
        self.buf = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32,
                               device=device)
        self.sink = torch.empty((), dtype=torch.float32, device=device)

    def __call__(self):
        self.buf.fill_(1.0)
        torch.sum(self.buf, dim=0, out=self.sink)


def time_launches(fn, reps, warmup, flush=None):
    """Median device time (ms) of fn() over reps launches (and the minimum),
    events on the current stream, L2 flushed between launches when a flusher
    is given."""
    for _ in range(warmup):
        fn()
    ts = []
    for _ in range(reps):
        if flush is not None:
            flush()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record()
        fn()
        e1.record()
        e1.synchronize()
        ts.append(e0.elapsed_time(e1))
    return statistics.median(ts), min(ts)


def gpu_arm(args, ws, rank, local):
    import paged_kv_asymmetric_gb300 as pkv
    from paged_kv_asymmetric_gb300 import workloads as wl

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    pkv.load()  # raises if the library is not built
    pk, pk_kind = peaks()
    hbm = float(pk["hbm_gbs"])
    tf_burst = float(pk["bf16_tflops"])
    launches = 0

    # ---------------- sub-measurements --------------------------------
    flush = Flusher(dev)
    sub = {}
    reps = max(3, args.sub_reps)

    def attn_decode_sub(name, wk, splits, time_write=False, balanced=False):
        dwk = wl.to_device(wk, device=dev)

        def wr():
            pkv.kv_cache_write(dwk.k_ctx, dwk.v_ctx, dwk.slots_all, dwk.cache,
                               dwk.k_scale, dwk.v_scale)
        wr()
        wsub = {}
        if time_write:  # the whole context's cache write (e.g. the fp8 encode)
            mw, _ = time_launches(wr, reps, 2, flush)
            nw = int(dwk.k_ctx.shape[0])
            wb = write_bytes(wk, nw)
            wsub = {"write_ms": mw, "write_bytes": wb, "write_GBps": wb / (mw * 1e-3) / 1e9,
                    "write_frac_hbm": wb / (mw * 1e-3) / 1e9 / hbm}
        Tk, Hk, dvk = wk.num_tokens, wk.num_q_heads, wk.head_size_v
        pok = torch.empty(splits, Tk, Hk, dvk, dtype=torch.float32, device=dev)
        plk = torch.empty(splits, Tk, Hk, dtype=torch.float32, device=dev)
        outk = torch.empty(Tk, Hk, dvk, dtype=torch.bfloat16, device=dev)

        def dec(cache=None):
            cache = dwk.cache if cache is None else cache
            if balanced:
                pkv.paged_attn_decode_balanced(
                    dwk.q, cache, dwk.block_table, dwk.seq_lens, dwk.query_start_loc,
                    wk.softmax_scale, wk.max_query_len, splits, 0, partial_o=pok,
                    partial_lse=plk, k_scale=dwk.k_scale, v_scale=dwk.v_scale)
            else:
                pkv.paged_attn_decode(dwk.q, cache, dwk.block_table,
                                      dwk.seq_lens, dwk.query_start_loc,
                                      wk.softmax_scale, wk.max_query_len, splits,
                                      partial_o=pok, partial_lse=plk,
                                      k_scale=dwk.k_scale, v_scale=dwk.v_scale)

        def red():
            pkv.splitkv_reduce(pok, plk, out=outk)
        sinks = torch.linspace(-2.0, 2.0, Hk, dtype=torch.float32, device=dev)

        def red_sink():  # the same merge with an attention sink per head
            pkv.splitkv_reduce(pok, plk, out=outk, sinks=sinks)
        def step():  # the decode and its merge as a step launches them
            dec()
            red()
        md, _ = time_launches(dec, reps, 2, flush)
        mr, _ = time_launches(red, reps, 2, flush)
        ms, _ = time_launches(step, reps, 2, flush)
        mrs, _ = time_launches(red_sink, reps, 2, flush)
        b = decode_bytes(wk)
        loop = {}
        cache_bytes = dwk.cache.data.numel() * dwk.cache.data.element_size()
        if cache_bytes >= L2_FLUSH_BYTES:
            # steps back to back (inputs larger than L2): decode + merge, the
            # decode reading two copies of the cache in turn
            caches = (dwk.cache, pkv.Cache(dwk.cache.data.clone(), dwk.cache.desc))
            n_loop = 4 * max(10, reps)
            for i in range(4):
                dec(caches[i & 1])
                red()
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            torch.cuda.synchronize()
            e0.record()
            for i in range(n_loop):
                dec(caches[i & 1])
                red()
            e1.record()
            e1.synchronize()
            ml = e0.elapsed_time(e1) / n_loop
            loop = {"loop_step_ms": ml, "loop_step_frac_hbm": b / (ml * 1e-3) / 1e9 / hbm,
                    "loop_steps": n_loop}
            del caches

        sub[name] = {"decode_ms": md, "reduce_ms": mr, "splits": splits,
                     "segments": "balanced ranges (at most splits)" if balanced
                     else "equal segments",
                     "bytes": b, "GBps": b / ((md + mr) * 1e-3) / 1e9,
                     "decode_kernel_GBps": b / (md * 1e-3) / 1e9,
                     # each launch timed alone after an L2 flush
                     "frac_hbm": b / ((md + mr) * 1e-3) / 1e9 / hbm,
                     # decode then merge back to back (programmatic launch,
                     # partials still in L2), one L2 flush before the pair
                     "step_ms": ms, "step_frac_hbm": b / (ms * 1e-3) / 1e9 / hbm,
                     **loop, "reduce_sink_ms": mrs, **wsub}
        del dwk, pok, plk, outk
        torch.cuda.empty_cache()

    def prefill_sub(name, n_tokens):
        require_single_gpu(ws, name)
        wk = wl.long_prefill(n_tokens, device=dev)
        dwk = wl.to_device(wk, device=dev)
        nw = wk.k_ctx.shape[0]

        def wr():
            pkv.kv_cache_write(dwk.k_ctx, dwk.v_ctx, dwk.slots_all, dwk.cache)
        mw, _ = time_launches(wr, reps, 2, flush)
        wb = write_bytes(wk, nw)
        outk = torch.empty(wk.num_tokens, wk.num_q_heads, wk.head_size_v,
                           dtype=torch.bfloat16, device=dev)

        def pf():
            pkv.paged_attn_prefill(dwk.q, dwk.cache, dwk.block_table,
                                   dwk.seq_lens, dwk.query_start_loc,
                                   wk.softmax_scale, out=outk)
        mp, _ = time_launches(pf, reps, 2, flush)
        sinks = torch.linspace(-2.0, 2.0, wk.num_q_heads, dtype=torch.float32, device=dev)

        def pf_sink():  # the same prefill with an attention sink per head
            pkv.paged_attn_prefill(dwk.q, dwk.cache, dwk.block_table,
                                   dwk.seq_lens, dwk.query_start_loc,
                                   wk.softmax_scale, out=outk, sinks=sinks)
        mps, _ = time_launches(pf_sink, reps, 2, flush)
        fl = prefill_flops(wk)
        sub[name] = {"prefill_ms": mp, "tflop": fl / 1e12,
                     "TFLOPs": fl / (mp * 1e-3) / 1e12,
                     "frac_bf16": fl / (mp * 1e-3) / 1e12 / tf_burst,
                     "sink_ms": mps, "sink_TFLOPs": fl / (mps * 1e-3) / 1e12,
                     "write_ms": mw, "write_bytes": wb,
                     "write_GBps": wb / (mw * 1e-3) / 1e9,
                     "write_frac_hbm": wb / (mw * 1e-3) / 1e9 / hbm}
        del dwk, outk
        torch.cuda.empty_cache()

    def prefill_fp8_sub(name, n_tokens):
        # the same causal prefill over an FP8 E4M3 cache (per-head scales):
        # the codes are widened in the kernel, no workspace
        require_single_gpu(ws, name)
        wk = wl.make_workload(f"prefill-{n_tokens}-fp8", seq_lens=[n_tokens],
                              q_lens=[n_tokens], kv_dtype=wl.FP8,
                              scale_mode=wl.SCALE_HEAD, seed=0, device=dev)
        dwk = wl.to_device(wk, device=dev)
        pkv.kv_cache_write(dwk.k_ctx, dwk.v_ctx, dwk.slots_all, dwk.cache,
                           dwk.k_scale, dwk.v_scale)
        outk = torch.empty(wk.num_tokens, wk.num_q_heads, wk.head_size_v,
                           dtype=torch.bfloat16, device=dev)

        def pf8(ws=None):
            pkv.paged_attn_prefill(dwk.q, dwk.cache, dwk.block_table,
                                   dwk.seq_lens, dwk.query_start_loc,
                                   wk.softmax_scale, out=outk, k_scale=dwk.k_scale,
                                   v_scale=dwk.v_scale, workspace=ws)
        mp, _ = time_launches(pf8, reps, 2, flush)
        # the two-pass form: pages widened into a workspace, then the prefill
        nws = pkv.prefill_fp8_workspace_bytes(wk.num_seqs, dwk.block_table.shape[1],
                                              dwk.cache)
        wsp = torch.empty(nws, dtype=torch.uint8, device=dev)
        m2, _ = time_launches(lambda: pf8(wsp), reps, 2, flush)
        fl = prefill_flops(wk)
        sub[name] = {"prefill_ms": mp, "tflop": fl / 1e12,
                     "TFLOPs": fl / (mp * 1e-3) / 1e12,
                     "frac_bf16": fl / (mp * 1e-3) / 1e12 / tf_burst,
                     "form": "E4M3 widened in the kernel, no workspace",
                     "two_pass_ms": m2, "two_pass_TFLOPs": fl / (m2 * 1e-3) / 1e12,
                     "two_pass_frac_bf16": fl / (m2 * 1e-3) / 1e12 / tf_burst,
                     "two_pass_workspace_bytes": nws}
        del dwk, outk, wsp
        torch.cuda.empty_cache()

    if args.only:
        if args.only in PREFILL_KINDS:
            require_single_gpu(ws, f"--only {args.only}")
        sampler = ClockSampler(local)
        sampler.start()
        if args.only == "prefill":
            prefill_sub(f"prefill_{args.prefill_tokens}", args.prefill_tokens)
        elif args.only == "prefill_fp8":
            prefill_fp8_sub(f"prefill_fp8_{args.prefill_tokens}", args.prefill_tokens)
        elif args.only == "verify":
            attn_decode_sub("verify_fp8", wl.verify_fp8(device=dev), args.splits or 16,
                            time_write=True, balanced=True)
        elif args.only == "mla":
            s = pkv.decode_suggest_splits(1, 16, 1, 1, 100000, 64)
            attn_decode_sub("mla_b1_h16", wl.mla_decode(batch=1, heads=16,
                                                        device=dev), args.splits or s)
        elif args.only == "decode":
            wd = wl.batched_decode(device=dev)
            attn_decode_sub("batched_decode", wd, args.splits or wd.max_splits,
                            balanced=True)
        return {"only": args.only, "sub": sub, "clocks": sampler.stop()}

    # ---------------- headline: batched decode step -------------------
    w = wl.batched_decode(seed=rank)
    dw = wl.to_device(w, device=dev)
    pkv.kv_cache_write(dw.k_ctx, dw.v_ctx, dw.slots_all, dw.cache)
    S = w.max_splits
    T, Hq, dv = w.num_tokens, w.num_q_heads, w.head_size_v
    po = torch.empty(S, T, Hq, dv, dtype=torch.float32, device=dev)
    pl = torch.empty(S, T, Hq, dtype=torch.float32, device=dev)
    out = torch.empty(T, Hq, dv, dtype=torch.bfloat16, device=dev)
    new_idx = dw.new_idx
    k_new = dw.k_ctx[new_idx].contiguous()
    v_new = dw.v_ctx[new_idx].contiguous()
    stream = torch.cuda.current_stream()

    def decode_only():
        pkv.paged_attn_decode_balanced(dw.q, dw.cache, dw.block_table, dw.seq_lens,
                                       dw.query_start_loc, w.softmax_scale, 1, S, 0,
                                       partial_o=po, partial_lse=pl)

    def step():
        pkv.kv_cache_write(k_new, v_new, dw.slots_new, dw.cache)
        decode_only()
        pkv.splitkv_reduce(po, pl, out=out)

    step_bytes = decode_bytes(w) + write_bytes(w, T)
    for _ in range(max(3, args.warmup)):
        step()
    sampler = ClockSampler(local)
    sampler.start()
    torch.cuda.synchronize()
    barrier(ws)
    torch.cuda.synchronize()
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    t0.record(stream)
    for _ in range(args.steps):
        step()
    t1.record(stream)
    torch.cuda.synchronize()
    barrier(ws)
    torch.cuda.synchronize()
    ms_total = t0.elapsed_time(t1)
    launches += 3 * args.steps
    ms_total_max = max_over_ranks(ms_total, ws, dev)
    ms_step = ms_total_max / args.steps
    total_bytes = sum_over_ranks(step_bytes * args.steps, ws, dev)
    value = total_bytes / (ms_total_max * 1e-3) / 1e9

    # roofline: the decode kernel alone, its launches back to back with no
    # event between them (the 419 MB cache is larger than L2, so every
    # launch reads from HBM); average duration = loop time / launches
    n_roof = max(50, args.steps)
    for _ in range(3):
        decode_only()
    torch.cuda.synchronize()
    t0.record(stream)
    for _ in range(n_roof):
        decode_only()
    t1.record(stream)
    torch.cuda.synchronize()
    dec_ms = t0.elapsed_time(t1) / n_roof
    dec_alg = decode_bytes(w)
    dec_gbs = dec_alg / (dec_ms * 1e-3) / 1e9

    # ---------------- e2e: host buffers through the public API ---------
    # Every step's inputs (Q, new K/V, slots, block table, seq_lens,
    # query_start_loc) travel host -> device as one copy from a pinned
    # staging buffer on an upload stream, and its output device -> host on a
    # download stream; two device buffer sets let step k+1's upload and step
    # k's download overlap step k's kernels (one stream for both directions
    # would queue each upload behind the previous step's download, which
    # waits for that step's merge).  The timed region ends when the last
    # download lands.
    srcs = (dw.q, k_new, v_new, dw.slots_new, dw.block_table, dw.seq_lens,
            dw.query_start_loc)
    offs, off = [], 0
    for t in srcs:
        offs.append(off)
        off += (t.numel() * t.element_size() + 255) // 256 * 256
    h_in = torch.empty(off, dtype=torch.uint8).pin_memory()
    d_in = [torch.empty(off, dtype=torch.uint8, device=dev) for _ in range(2)]

    def views(buf):
        return [buf[o:o + t.numel() * t.element_size()].view(t.dtype).view(t.shape)
                for o, t in zip(offs, srcs)]
    for hv, t in zip(views(h_in), srcs):
        hv.copy_(t.cpu())
    d_views = [views(b) for b in d_in]
    outs = [torch.empty_like(out) for _ in range(2)]
    h_outs = [torch.empty(out.shape, dtype=out.dtype).pin_memory() for _ in range(2)]
    h2d = sum(t.numel() * t.element_size() for t in srcs)
    d2h = h_outs[0].numel() * h_outs[0].element_size()
    up = torch.cuda.Stream(device=dev)
    down = torch.cuda.Stream(device=dev)
    in_ready = [torch.cuda.Event() for _ in range(2)]
    in_free = [torch.cuda.Event() for _ in range(2)]
    out_ready = [torch.cuda.Event() for _ in range(2)]
    out_read = [torch.cuda.Event() for _ in range(2)]
    for e in in_free + out_read:
        e.record(stream)

    def e2e_step(k):
        b = k & 1
        d_q, d_k, d_v, d_slots, d_bt, d_sl, d_qsl = d_views[b]
        with torch.cuda.stream(up):
            up.wait_event(in_free[b])
            d_in[b].copy_(h_in, non_blocking=True)
            in_ready[b].record(up)
        stream.wait_event(in_ready[b])
        stream.wait_event(out_read[b])
        pkv.kv_cache_write(d_k, d_v, d_slots, dw.cache)
        pkv.paged_attn_decode_balanced(d_q, dw.cache, d_bt, d_sl, d_qsl,
                                       w.softmax_scale, 1, S, 0, partial_o=po,
                                       partial_lse=pl)
        in_free[b].record(stream)
        pkv.splitkv_reduce(po, pl, out=outs[b])
        out_ready[b].record(stream)
        with torch.cuda.stream(down):
            down.wait_event(out_ready[b])
            h_outs[b].copy_(outs[b], non_blocking=True)
            out_read[b].record(down)

    for k in range(3):
        e2e_step(k)
    torch.cuda.synchronize()
    barrier(ws)
    t0.record(stream)
    up.wait_stream(stream)  # no upload starts before the timed region
    for k in range(args.steps):
        e2e_step(k)
    stream.wait_stream(down)
    t1.record(stream)
    torch.cuda.synchronize()
    barrier(ws)
    e2e_ms = max_over_ranks(t0.elapsed_time(t1), ws, dev)
    launches += 3 * args.steps
    e2e_value = total_bytes / (e2e_ms * 1e-3) / 1e9
    # the downloaded output is the device result
    if not torch.equal(h_outs[(args.steps - 1) & 1], outs[(args.steps - 1) & 1].cpu()):
        raise RuntimeError("e2e output mismatch")

    for kind, name, size in sub_plan(args, ws):
        if kind == "prefill":
            prefill_sub(name, size)
        elif kind == "prefill_fp8":
            prefill_fp8_sub(name, size)
        elif kind == "verify":
            wv = wl.verify_fp8(device=dev)
            attn_decode_sub(name, wv, size, time_write=True, balanced=True)
            del wv
        elif kind == "mla":
            b, h = size
            wm = wl.mla_decode(batch=b, heads=h, device=dev)
            s = pkv.decode_suggest_splits(b, h, 1, 1, 100000, 64)
            attn_decode_sub(name, wm, s)
            del wm
    if ws > 1 and not args.no_sub:
        sub["prefill"] = ("not measured: the cluster-multicast prefill runs in "
                          "single-GPU jobs only")
    clocks = sampler.stop()

    traffic = traffic_record("decode_bf16_192")
    roof = {"kernel": "decode_kernel<192,128,bf16> (balanced ranges)", "bound": "hbm",
            "achieved": dec_gbs, "peak": hbm, "unit": "GB/s",
            "frac": dec_gbs / hbm, "peak_kind": pk_kind,
            "traffic": traffic,
            "algorithmic_bytes_per_launch": dec_alg,
            "avg_launch_ms": dec_ms, "launches_timed": n_roof,
            "timing": "back-to-back launches of the decode kernel alone, "
                      "CUDA events around the loop"}
    res = {
        "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": ws,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_step,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16", "data": "synthetic (seeded N(0,1), random page placement)",
        "config": {"workload": "batched-decode: 32 seqs, ctx U[2048,8192], q_len 1, "
                   "Hq16/Hkv4, K192/V128, block 16, bf16, 16 splits",
                   "segments": "balanced ranges cut on the device (at most 16 per sequence)",
                   "step": "kv_cache_write(new tokens) + paged_attn_decode_balanced + "
                           "splitkv_reduce",
                   "l2": "inputs larger than L2 (419 MB KV cache)",
                   "parallelism": f"replicas x{ws}"},
        "roofline": roof,
        "e2e": {"value": e2e_value, "unit": "GB/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h},
        "gpu_launches": launches,
        "clocks": clocks,
        "sub": sub,
    }
    if "prefill_32k" in sub:
        p = sub["prefill_32k"]
        res["prefill_tflops"] = p["TFLOPs"]
        res["roofline_prefill"] = {
            "kernel": "prefill_kernel (tcgen05)", "bound": "tensor",
            "achieved": p["TFLOPs"], "peak": tf_burst, "unit": "TFLOP/s",
            "frac": p["frac_bf16"], "peak_kind": pk_kind,
            "traffic": traffic_record("prefill"), "avg_launch_ms": p["prefill_ms"]}
    return res


# ------------------------------------------------------ oracle (CPU) ----

def oracle_decode_sample(target_s: float, seed: int = 0, nseq: int = 0):
    """The oracle on the first `nseq` sequences of the batched-decode workload:
    build its cache once, then repeat (write the step's new tokens, attend for
    the step's query rows) until about target_s seconds have passed."""
    import oracle
    from paged_kv_asymmetric_gb300 import workloads as wl
    from tests import refs

    w = wl.batched_decode(seed=seed)
    if nseq <= 0:  # one query row per host core, at most the whole batch
        nseq = max(1, min(w.num_seqs, os.cpu_count() or 1))
    seqs = list(range(nseq))
    cache = refs.oracle_cache(w, seqs=seqs)
    threads = os.cpu_count() or 1
    d = refs.oracle_desc(w)
    toks = np.arange(nseq, dtype=np.int32)
    kb, vb = refs.bf16_bits(w.k_ctx), refs.bf16_bits(w.v_ctx)
    idx = w.new_kv_index()[:nseq]
    slots = w.slot_mapping_new()[:nseq]
    sub_bytes = 0
    e = 2
    for b in seqs:
        sub_bytes += int(w.seq_lens[b]) * w.num_kv_heads * w.row_elems * e
    sub_bytes += nseq * w.num_q_heads * (w.head_size + w.head_size_v) * 2
    sub_bytes += write_bytes(w, nseq)
    n = 0
    t0 = time.perf_counter()
    while True:
        oracle.kv_cache_write(kb[idx], vb[idx], slots, cache, d)
        refs.oracle_attn(w, cache, tokens=toks, threads=threads)
        n += 1
        el = time.perf_counter() - t0
        if el >= target_s or n >= 1000:
            break
    return {"value": sub_bytes * n / el / 1e9, "unit": "GB/s",
            "cores": min(threads, nseq),
            "kind": "oracle",
            "sample": f"first {nseq} of 32 sequences of the batched-decode step "
                      f"(write + attention, threads over query rows), {n} "
                      f"repetitions in {el:.1f} s",
            "seconds_per_step": el / n}


def reference_arm(args, ws, rank):
    if rank != 0:
        return None
    base = oracle_decode_sample(target_s=max(2.0, args.ref_seconds / max(1, args.steps)))
    vals = []
    for _ in range(args.steps):
        vals.append(oracle_decode_sample(
            target_s=max(1.0, args.ref_seconds / max(1, args.steps)))["value"])
    v = statistics.mean(vals)
    return {
        "metric": METRIC, "value": v, "unit": "GB/s", "n_gpus": ws,
        "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": base["seconds_per_step"] * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f64", "data": "synthetic (seeded N(0,1), random page placement)",
        "config": {"workload": "batched-decode: 32 seqs, ctx U[2048,8192], q_len 1, "
                   "Hq16/Hkv4, K192/V128, block 16, bf16, 16 splits",
                   "step": "oracle: kv_cache_write(new tokens) + paged attention",
                   "parallelism": "host cores"},
        "impl": "reference",
        "cpu_baseline": {"value": v, "unit": "GB/s", "cores": base["cores"],
                         "kind": "oracle", "sample": base["sample"]},
        "e2e": {"value": v, "unit": "GB/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-sub", action="store_true")
    ap.add_argument("--skip-prefill", action="store_true")
    ap.add_argument("--only", choices=["prefill", "prefill_fp8", "verify", "mla", "decode"],
                    help="run one sub-measurement alone (for profiling)")
    ap.add_argument("--prefill-tokens", type=int, default=8192)
    ap.add_argument("--splits", type=int, default=0,
                    help="split-KV segments for --only decode / verify / mla "
                         "(default: the workload's own count)")
    ap.add_argument("--sub-reps", type=int, default=20)
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--ref-seconds", type=float, default=30.0)
    args = ap.parse_args(argv)
    ws, rank, local = dist_info()
    if args.gpus < 1 or args.gpus != ws:
        ap.error(f"--gpus {args.gpus} does not match the job's world size {ws}: "
                 "run N ranks with torch.distributed.run --nproc-per-node N")
    if args.impl == "reference":
        init_dist(ws, "gloo")
        res = reference_arm(args, ws, rank)
        if res is not None:
            print(json.dumps(res), flush=True)
        if ws > 1:
            torch.distributed.destroy_process_group()
        return 0
    init_dist(ws, "nccl")
    res = gpu_arm(args, ws, rank, local)
    if rank == 0:
        if ws == 1 and not args.only:
            res["cpu_baseline"] = oracle_decode_sample(args.cpu_seconds)
        print(json.dumps(res), flush=True)
    if ws > 1:
        torch.distributed.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
