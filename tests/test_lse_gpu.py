"""The log-sum-exp output (rel_attn_paged_varlen_lse, the return_lse=True form
of inkling_fa4_rel_attention in the vLLM API docs) against the fp64 oracle on
the decode kernel, the prefill kernel and the split combine.

Tolerance: each score s_j is an fp32 sum of D exact bf16 products (plus an
exact bf16 bias), so |ds_j| <= D * 2^-24 * scale * sum_k |q_k k_k| + 2^-24 |s_j|,
below 1e-4 for these inputs; the sum of the exps carries the relative error of
the hardware exp2 (about 2^-22 per term) and one log.  lse therefore lies
within max_j |ds_j| + a few 1e-6 of the exact value: 1e-3 + 1e-5 |lse| is a
bound with a wide margin.  Rows with no visible key are -inf on both sides.
"""
import numpy as np
import pytest
import torch

from oracle import reference as ref
from paged_attention_relative_gb300.workloads import make_case
from tests.gpu_util import assert_close, assert_no_device_error, to_dev, expected_prefill_kernel

pytestmark = pytest.mark.gpu

CASES = [
    # decode kernel (<= 64 packed rows)
    dict(name="decode_gqa4", seqlens_q=[1, 1, 1], seqlens_k=[700, 1, 0], num_heads=8, num_kv_heads=2,
         head_dim=128, rel_extent=64, kernel="decode"),
    dict(name="decode_multi_token_short_cache", seqlens_q=[4, 3], seqlens_k=[2, 300], num_heads=16,
         num_kv_heads=4, head_dim=64, rel_extent=16, kernel="decode"),
    dict(name="decode_window", seqlens_q=[2], seqlens_k=[900], num_heads=4, num_kv_heads=1, head_dim=128,
         window=(100, 0), rel_extent=40, kernel="decode"),
    # prefill kernel (> 64 packed rows)
    dict(name="prefill_gqa4", seqlens_q=[40, 17], seqlens_k=[300, 17], num_heads=8, num_kv_heads=2,
         head_dim=128, rel_extent=64, kernel="prefill"),
    dict(name="prefill_short_cache", seqlens_q=[100, 80], seqlens_k=[30, 0], num_heads=4, num_kv_heads=4,
         head_dim=128, rel_extent=16, kernel="prefill"),
    dict(name="prefill_window_noncausal", seqlens_q=[80], seqlens_k=[300], num_heads=4, num_kv_heads=4,
         head_dim=64, causal=False, window=(40, 25), rel_extent=24, kernel="prefill"),
]


def _call(c, g, splits, out, lse):
    import paged_attention_relative_gb300 as pa
    pa.rel_attn_paged_varlen_lse(g["q"], g["key_cache"], g["value_cache"], g["block_table"], g["cache_seqlens"],
                                 g["cu_seqlens_q"], c.max_seqlen_q, c.softmax_scale, c.causal, c.window_left,
                                 c.window_right, c.rel_extent, g["rel_logits"] if c.rel_extent > 0 else None,
                                 splits, out=out, softmax_lse=lse)
    torch.cuda.synchronize()


def assert_lse_close(got, want, what):
    got = got.double().cpu().numpy()
    inf_got, inf_want = np.isneginf(got), np.isneginf(want)
    assert np.array_equal(inf_got, inf_want), f"{what}: -inf rows differ"
    fin = ~inf_want
    assert np.isfinite(got[fin]).all(), f"{what}: non-finite lse"
    err = np.abs(got[fin] - want[fin])
    bound = 1e-3 + 1e-5 * np.abs(want[fin])
    assert (err <= bound).all(), f"{what}: lse max-abs {err.max():.3e}"


@pytest.mark.parametrize("cfg", CASES, ids=[c["name"] for c in CASES])
@pytest.mark.parametrize("splits", [1, 4])
def test_lse_matches_oracle(cfg, splits):
    import paged_attention_relative_gb300 as pa
    kw = dict(cfg)
    name, kernel = kw.pop("name"), kw.pop("kernel")
    c = make_case(seed=sum(map(ord, name)) % 991, **kw)
    g = to_dev(c)
    out = torch.empty_like(g["q"])
    lse = torch.full(c.q.shape[:2], float("nan"), dtype=torch.float32, device="cuda")
    _call(c, g, splits, out, lse)
    info = pa.last_launch()
    assert info["kernel"] == (expected_prefill_kernel(c) if kernel == "prefill" else kernel)
    want_out, want_lse = ref.forward(c, with_lse=True)
    assert_close(out, want_out, what=f"{name} out")
    assert_lse_close(lse, want_lse, f"{name} splits={splits} ({info['num_splits']} used)")
    assert_no_device_error()


def test_lse_into_transposed_buffer_and_same_out_as_plain_call():
    """An (H, T) buffer passed as its (T, H) transpose; out equals the plain call's bit for bit."""
    import paged_attention_relative_gb300 as pa
    c = make_case(seed=7, seqlens_q=[70, 33], seqlens_k=[500, 40], num_heads=8, num_kv_heads=2, head_dim=128,
                  rel_extent=32)
    g = to_dev(c)
    lse_ht = torch.full((c.q.shape[1], c.q.shape[0]), float("nan"), dtype=torch.float32, device="cuda")
    out = torch.empty_like(g["q"])
    _call(c, g, 3, out, lse_ht.t())
    plain = pa.rel_attn_paged_varlen(g["q"], g["key_cache"], g["value_cache"], g["block_table"],
                                     g["cache_seqlens"], g["cu_seqlens_q"], c.max_seqlen_q, c.softmax_scale,
                                     c.causal, c.window_left, c.window_right, c.rel_extent, g["rel_logits"], 3)
    torch.cuda.synchronize()
    assert torch.equal(out, plain)
    _, want_lse = ref.forward(c, with_lse=True)
    assert_lse_close(lse_ht.t(), want_lse, "transposed lse")
    assert_no_device_error()
