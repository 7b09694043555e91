"""The allocation-free entry point (rel_attn_paged_varlen_noalloc).

It serves callers that must not allocate device memory (a framework that owns
the device through its own pool, or a program that forbids allocation after
start-up): its split workspace is a fixed array inside the library.  These
tests call it through the C ABI, twice in a row on the same inputs (the
array keeps the previous call's contents, which must not leak into the
next), and compare with rel_attn_paged_varlen and with the oracle on the same
inputs; they check that the calls leave the device's free memory unchanged
and that a workspace just under the array's size is accepted and one just
over it rejected.  The file name makes pytest collect it last.
"""
import ctypes

import pytest
import torch

from oracle import reference as ref
from paged_attention_relative_gb300.workloads import batched_decode, long_decode, make_case, tiny_mixed
from tests.gpu_util import TOL_MAX, TOL_MEAN, TOL_SPLIT, assert_close, to_dev

pytestmark = pytest.mark.gpu

SCRATCH = 16 << 20  # REL_ATTN_NOALLOC_SCRATCH_BYTES


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


def _prefill_case():
    return make_case(seed=31, seqlens_q=[70, 20], seqlens_k=[300, 90], num_heads=8, num_kv_heads=2,
                     head_dim=128, rel_extent=32)


@pytest.mark.parametrize("make,splits", [(tiny_mixed, 3), (long_decode, 16), (batched_decode, 4),
                                         (batched_decode, 1), (_prefill_case, 3)],
                         ids=["tiny_mixed-3", "long_decode-16", "batched_decode-4", "batched_decode-1",
                              "prefill-3"])
def test_noalloc_matches_allocating_entry_point_twice(make, splits):
    from paged_attention_relative_gb300 import _lib as L
    c = make(0) if make is not _prefill_case else make()
    g = to_dev(c)
    ref_out = torch.empty_like(g["q"])
    assert _call(L.lib.rel_attn_paged_varlen, c, g, splits, ref_out) == 0
    want = ref.forward(c)
    for _ in range(2):
        out = torch.full_like(g["q"], float("nan"))
        st = _call(L.lib.rel_attn_paged_varlen_noalloc, c, g, splits, out)
        assert st == 0, L.lib.rel_attn_last_error().decode()
        assert L.last_launch()["workspace_bytes"] == (
            splits * c.q.shape[0] * c.q.shape[1] * (c.q.shape[2] + 1) * 4 if splits > 1 else 0)
        diff = (out.float() - ref_out.float()).abs()
        assert torch.isfinite(out.float()).all()
        assert diff.max().item() <= min(TOL_SPLIT, TOL_MAX) and diff.mean().item() <= TOL_MEAN
        assert_close(out, want, what=f"noalloc {make.__name__} splits={splits}")
    assert L.device_error() == 0


def test_noalloc_leaves_free_device_memory_unchanged():
    from paged_attention_relative_gb300 import _lib as L
    c = batched_decode(0)
    g = to_dev(c)
    out = torch.empty_like(g["q"])
    # The first call loads the module (and its scratch array) if nothing has yet.
    assert _call(L.lib.rel_attn_paged_varlen_noalloc, c, g, 4, out) == 0
    torch.cuda.synchronize()
    free0, _ = torch.cuda.mem_get_info()
    for _ in range(3):
        assert _call(L.lib.rel_attn_paged_varlen_noalloc, c, g, 4, out) == 0
    torch.cuda.synchronize()
    free1, _ = torch.cuda.mem_get_info()
    assert free1 == free0, (free0, free1)


def test_noalloc_workspace_just_under_the_scratch_matches_oracle():
    """64 tokens x 64 heads x 129 floats x 4 bytes = 2,113,536 bytes per split:
    7 splits (14.8 MB) fit the 16 MiB array, 8 (16.9 MB) do not."""
    from paged_attention_relative_gb300 import _lib as L
    c = batched_decode(0)
    per_split = c.q.shape[0] * c.q.shape[1] * (c.q.shape[2] + 1) * 4
    assert 7 * per_split <= SCRATCH < 8 * per_split
    g = to_dev(c)
    out = torch.empty_like(g["q"])
    assert _call(L.lib.rel_attn_paged_varlen_noalloc, c, g, 7, out) == 0, L.lib.rel_attn_last_error().decode()
    assert L.last_launch()["num_splits"] == 7
    assert_close(out, ref.forward(c), what="noalloc 7 splits")
    st = _call(L.lib.rel_attn_paged_varlen_noalloc, c, g, 8, out)
    assert st == 1
    msg = L.lib.rel_attn_last_error().decode()
    assert "static scratch" in msg and str(SCRATCH) in msg and str(8 * per_split) in msg
    assert L.last_launch()["kernel"] == "none"
    assert L.device_error() == 0


def test_noalloc_rejects_workspace_beyond_the_scratch():
    from paged_attention_relative_gb300 import _lib as L
    c = batched_decode(0)                      # 64 tokens x 64 heads x 129 floats per split
    g = to_dev(c)
    out = torch.empty_like(g["q"])
    st = _call(L.lib.rel_attn_paged_varlen_noalloc, c, g, 16, out)   # 16 splits -> 33.8 MB > 16 MiB
    assert st == 1
    msg = L.lib.rel_attn_last_error().decode()
    assert "static scratch" in msg and str(SCRATCH) in msg
