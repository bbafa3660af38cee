"""Launch chaining invariant, checked on the sources (no GPU): every kernel
launched with programmatic dependent launch must trigger its dependents and
then wait for the kernel ahead of it (griddepcontrol.wait) before any
other statement of its body (only declarations and static_asserts may come
first).  A memory access above the wait would race with the kernel ahead."""
from __future__ import annotations

import os
import re

CSRC = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))),
                    "paged_kv_asymmetric_gb300", "csrc")


def _sources():
    out = {}
    for f in sorted(os.listdir(CSRC)):
        if f.endswith((".cu", ".cuh", ".h")):
            with open(os.path.join(CSRC, f)) as fh:
                out[f] = fh.read()
    return out


def _strip_comments(text):
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return re.sub(r"//[^\n]*", "", text)


def _pdl_kernels(srcs):
    names = set()
    for text in srcs.values():
        t = _strip_comments(text)
        for m in re.finditer(r"launch_pdl\(\s*([A-Za-z_]\w*)", t):
            names.add(m.group(1))
        # kernels chosen through a local function pointer, e.g.
        #   auto kernel = cond ? k<8> : k<16>;  launch_pdl(kernel, ...)
        for m in re.finditer(r"auto\s+(\w+)\s*=\s*([^;]*);", t):
            if re.search(r"launch_pdl\(\s*" + m.group(1) + r"\b", t):
                names.update(re.findall(r"([A-Za-z_]\w*_kernel)\s*<", m.group(2)))
    names.discard("kernel")
    names.discard("void")  # the helper's own signature
    return names


def _kernel_body(text, name):
    t = _strip_comments(text)
    m = re.search(r"__global__[^;{]*?\b" + name + r"\s*\(", t, flags=re.S)
    if m is None:
        return None
    i = t.index("{", m.end())  # the body's opening brace (after the parameters)
    depth, j = 0, i
    while True:
        if t[j] == "{":
            depth += 1
        elif t[j] == "}":
            depth -= 1
            if depth == 0:
                return t[i + 1:j]
        j += 1


def test_every_chained_kernel_waits_first():
    srcs = _sources()
    kernels = _pdl_kernels(srcs)
    # the write, decode and merge kernels of a decode step
    for must in ("cache_write_tok_kernel", "decode_kernel", "splitkv_reduce_warp4_kernel",
                 "splitkv_reduce_rows_kernel", "splitkv_reduce_kernel"):
        assert must in kernels, must
    for k in sorted(kernels):
        bodies = [b for b in (_kernel_body(t, k) for t in srcs.values()) if b is not None]
        assert bodies, f"no definition of {k}"
        for body in bodies:
            stmts = [s.strip() for s in body.split(";")]
            stmts = [s for s in stmts if s]
            lead = []
            for s in stmts:
                if s.startswith(("static_assert", "__shared__", "extern __shared__",
                                 "constexpr")):
                    continue
                lead.append(s)
                if len(lead) == 2:
                    break
            assert lead == ["pdl_trigger()", "pdl_wait()"], (k, lead)


def test_not_chained_kernels_do_not_wait():
    """The prefill and the FP8 widening pass launch plainly; a wait in them
    would be harmless but would mean a launch path forgot the attribute."""
    srcs = _sources()
    kernels = _pdl_kernels(srcs)
    assert "prefill_kernel" not in kernels
    assert "fp8_pages_to_bf16_kernel" not in kernels
