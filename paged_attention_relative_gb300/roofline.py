"""Algorithmic work of one forward call, for roofline reporting.

Counts the bytes a forward must move at least once and the flops of the two
contractions over the allowed (row, key) pairs.  Used by the benchmark only.
"""
from __future__ import annotations

import numpy as np

from .workloads import Case


def algorithmic_bytes(case: Case) -> int:
    """Bytes the forward must move at least once: every K/V row a request can
    attend to (per kv head), q, out, the used rel_logits band, table and lengths."""
    d = case.dims
    sq = case.seqlens_q
    sk = case.cache_seqlens.tolist()
    kv_rows = 0
    rel_elems = 0
    wl, wr = case.window_left, case.window_right
    for b in range(d["B"]):
        if sq[b] == 0:
            continue
        off = sk[b] - sq[b]
        hi = sk[b] - 1
        if case.causal:
            hi = min(hi, sq[b] - 1 + off)
        if wr >= 0:
            hi = min(hi, sq[b] - 1 + off + wr)
        lo = 0 if wl < 0 else max(0, off - wl)
        kv_rows += max(0, hi - lo + 1)
        rel_elems += _rel_band_elems(sq[b], sk[b], case.causal, wl, wr, case.rel_extent)
    kv = kv_rows * d["Hk"] * d["D"] * 2 * 2
    qo = 2 * d["T"] * d["H"] * d["D"] * 2
    rel_bytes = case.rel_logits.element_size() if case.rel_extent > 0 else 2  # bf16 or fp32
    rel = rel_elems * d["H"] * rel_bytes
    meta = case.block_table.numel() * 4 + case.cache_seqlens.numel() * 4 + case.cu_seqlens_q.numel() * 4
    return int(kv + qo + rel + meta)


def _rel_band_elems(sq, sk, causal, wl, wr, R):
    """Per-head count of (row, d) pairs with 0 <= d < R that some allowed key
    reaches; counted per row in closed form (no attention arithmetic)."""
    off = sk - sq
    tot = 0
    for i in range(sq):
        # keys j in [0, sk) with d = i + off - j in [0, R) and in the window
        dmax = min(R - 1, i + off)            # j >= 0
        dmin = max(0, i + off - (sk - 1))     # j <= sk-1
        if wl >= 0:
            dmax = min(dmax, wl)
        if wr >= 0:
            dmin = max(dmin, -wr)
        tot += max(0, dmax - dmin + 1)
    return tot


def algorithmic_flops(case: Case) -> int:
    """4*D flops per allowed (row, key) pair (QK^T and PV, one FMA = 2 flops)."""
    d = case.dims
    sq = case.seqlens_q
    sk = case.cache_seqlens.tolist()
    wl, wr = case.window_left, case.window_right
    pairs = 0
    for b in range(d["B"]):
        off = sk[b] - sq[b]
        i = np.arange(sq[b], dtype=np.int64)
        hi = np.full(sq[b], sk[b] - 1, dtype=np.int64)
        if case.causal:
            hi = np.minimum(hi, i + off)
        if wr >= 0:
            hi = np.minimum(hi, i + off + wr)
        lo = np.zeros(sq[b], dtype=np.int64)
        if wl >= 0:
            lo = np.maximum(lo, i + off - wl)
        pairs += int(np.maximum(0, hi - lo + 1).sum())
    return int(4 * d["D"] * pairs * d["H"])
