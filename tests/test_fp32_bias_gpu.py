"""fp32 rel_logits (values bf16 cannot hold) through the decode and prefill
kernels, with and without splits, a window, and the allocation-free decode
entry point, against the fp64 oracle on the same fp32 values."""
import pytest
import torch

from oracle import reference as ref
from paged_attention_relative_gb300.workloads import make_case
from tests.gpu_util import assert_close, assert_no_device_error, run, to_dev

pytestmark = pytest.mark.gpu

CASES = [
    dict(name="decode", seqlens_q=[1, 1, 2], seqlens_k=[300, 1000, 50], num_heads=8, num_kv_heads=2,
         head_dim=128, rel_extent=64, kernel="decode"),
    dict(name="decode_window", seqlens_q=[3], seqlens_k=[700], num_heads=16, num_kv_heads=4, head_dim=64,
         rel_extent=100, window=(200, 0), kernel="decode"),
    dict(name="prefill", seqlens_q=[40, 70], seqlens_k=[300, 200], num_heads=8, num_kv_heads=2, head_dim=128,
         rel_extent=48, kernel="prefill"),
    dict(name="prefill_odd_extent", seqlens_q=[90], seqlens_k=[400], num_heads=4, num_kv_heads=2, head_dim=64,
         rel_extent=37, window=(150, 0), kernel="prefill"),
]


def _fp32_case(cfg):
    kw = dict(cfg)
    name, kernel = kw.pop("name"), kw.pop("kernel")
    c = make_case(seed=sum(map(ord, name)) % 577, **kw)
    g = torch.Generator().manual_seed(1)
    rel = 2.0 * torch.randn(c.rel_logits.shape, generator=g)  # fp32 values, not bf16-representable
    return name, kernel, c.with_(rel_logits=rel)


@pytest.mark.parametrize("cfg", CASES, ids=[c["name"] for c in CASES])
@pytest.mark.parametrize("splits", [1, 3])
def test_fp32_rel_logits_match_oracle(cfg, splits):
    import paged_attention_relative_gb300 as pa
    name, kernel, c = _fp32_case(cfg)
    got = run(c, num_splits=splits)
    assert pa.last_launch()["kernel"] == kernel
    assert_close(got, ref.forward(c), what=f"{name} fp32 bias splits={splits}")
    assert_no_device_error()


def test_fp32_rel_logits_noalloc_decode():
    import paged_attention_relative_gb300 as pa
    _, _, c = _fp32_case(CASES[0])
    g = to_dev(c)
    out = torch.empty_like(g["q"])
    pa.rel_attn_paged_varlen_noalloc(g["q"], g["key_cache"], g["value_cache"], g["block_table"],
                                     g["cache_seqlens"], g["cu_seqlens_q"], c.max_seqlen_q, c.softmax_scale,
                                     c.causal, c.window_left, c.window_right, c.rel_extent, g["rel_logits"], 4,
                                     out=out)
    torch.cuda.synchronize()
    assert_close(out, ref.forward(c), what="noalloc fp32 bias")
    assert_no_device_error()
