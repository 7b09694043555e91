"""The allocation-free decode entry point (rel_attn_paged_varlen_noalloc).

It serves callers that must not allocate device memory (a framework that owns
the device through its own pool, or a program that forbids allocation after
start-up): its split workspace is a fixed array inside the library.  These
tests call it through the C ABI, twice in a row on the same inputs (the
array keeps the previous call's contents, which must not leak into the
next), and compare with rel_attn_paged_varlen on the same inputs.  The file
name makes pytest collect it last.
"""
import ctypes

import pytest
import torch

from paged_attention_relative_gb300.workloads import batched_decode, long_decode, tiny_mixed
from tests.gpu_util import TOL_MAX, TOL_MEAN, TOL_SPLIT, to_dev

pytestmark = pytest.mark.gpu


def _call(fn, c, g, splits, out):
    from paged_attention_relative_gb300 import _lib as L
    descs = [L.describe(g[k]) for k in ("q", "key_cache", "value_cache", "block_table", "cache_seqlens",
                                        "cu_seqlens_q")]
    rel = L.describe(g["rel_logits"])
    od = L.describe(out)
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    st = fn(*[ctypes.byref(d) for d in descs], c.max_seqlen_q, ctypes.c_float(c.softmax_scale), int(c.causal),
            c.window_left, c.window_right, c.rel_extent, ctypes.byref(rel), splits, ctypes.byref(od), stream)
    torch.cuda.synchronize()
    return st


@pytest.mark.parametrize("make,splits", [(tiny_mixed, 3), (long_decode, 16), (batched_decode, 4),
                                         (batched_decode, 1)])
def test_noalloc_matches_allocating_entry_point_twice(make, splits):
    from paged_attention_relative_gb300 import _lib as L
    c = make(0)
    g = to_dev(c)
    ref_out = torch.empty_like(g["q"])
    assert _call(L.lib.rel_attn_paged_varlen, c, g, splits, ref_out) == 0
    for _ in range(2):
        out = torch.full_like(g["q"], float("nan"))
        st = _call(L.lib.rel_attn_paged_varlen_noalloc, c, g, splits, out)
        assert st == 0, L.lib.rel_attn_last_error().decode()
        diff = (out.float() - ref_out.float()).abs()
        assert torch.isfinite(out.float()).all()
        assert diff.max().item() <= min(TOL_SPLIT, TOL_MAX) and diff.mean().item() <= TOL_MEAN
    assert L.device_error() == 0


def test_noalloc_rejects_workspace_beyond_the_scratch():
    from paged_attention_relative_gb300 import _lib as L
    c = batched_decode(0)                      # 64 tokens x 64 heads x 129 floats per split
    g = to_dev(c)
    out = torch.empty_like(g["q"])
    st = _call(L.lib.rel_attn_paged_varlen_noalloc, c, g, 16, out)   # 16 splits -> 33.8 MB > 16 MiB
    assert st == 1
    msg = L.lib.rel_attn_last_error().decode()
    assert "static scratch" in msg and str(16 << 20) in msg
