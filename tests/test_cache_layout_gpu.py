"""Caches whose pages are not contiguous: key_cache and value_cache as the two
halves of one (num_blocks, 2, block_size, num_kv_heads, head_dim) buffer, so
the block stride is twice block_size times the slot stride.  The prefill
kernels then read each 16-key page as two 8-key TMA boxes instead of one;
decode is indifferent.  Every output is checked against the oracle, and the
same case through contiguous caches must give the identical result."""
import pytest
import torch

from oracle import reference as ref
from paged_attention_relative_gb300.workloads import make_case
from tests.gpu_util import assert_close, assert_no_device_error, expected_prefill_kernel, run, to_dev

pytestmark = pytest.mark.gpu

CASES = [
    dict(name="decode", seqlens_q=[1, 3, 2], seqlens_k=[300, 77, 16], num_heads=8, num_kv_heads=2, head_dim=128,
         rel_extent=16),
    dict(name="prefill_d128", seqlens_q=[150, 40], seqlens_k=[700, 40], num_heads=8, num_kv_heads=2, head_dim=128,
         rel_extent=64),
    dict(name="prefill_d64_window", seqlens_q=[200], seqlens_k=[900], num_heads=4, num_kv_heads=1, head_dim=64,
         rel_extent=32, window=(300, 0)),
    dict(name="prefill_d128_block32", seqlens_q=[130], seqlens_k=[333], num_heads=8, num_kv_heads=8, head_dim=128,
         rel_extent=0, block_size=32),
    dict(name="prefill_d256", seqlens_q=[70], seqlens_k=[260], num_heads=4, num_kv_heads=2, head_dim=256,
         rel_extent=16),
]


def _interleaved(kc, vc):
    """K and V as views of one buffer with the K/V index after the block index."""
    NB, BS, Hk, D = kc.shape
    kv = torch.empty((NB, 2, BS, Hk, D), dtype=kc.dtype, device=kc.device)
    kv[:, 0].copy_(kc)
    kv[:, 1].copy_(vc)
    return kv[:, 0], kv[:, 1]


@pytest.mark.parametrize("cfg", CASES, ids=[c["name"] for c in CASES])
@pytest.mark.parametrize("splits", [1, 3])
def test_interleaved_kv_buffer_matches_oracle(cfg, splits):
    import paged_attention_relative_gb300 as pa
    kw = dict(cfg)
    name = kw.pop("name")
    c = make_case(seed=40 + len(name), **kw)
    g = to_dev(c)
    base = run(c, g, num_splits=splits).clone()
    g["key_cache"], g["value_cache"] = _interleaved(g["key_cache"], g["value_cache"])
    assert not g["key_cache"].is_contiguous()
    got = run(c, g, num_splits=splits)
    kernel = pa.last_launch()["kernel"]
    if name == "decode":
        assert kernel == "decode"
    elif c.q.shape[2] == 256:
        assert kernel == "prefill_pair"
    else:
        assert kernel == expected_prefill_kernel(c)
    assert_close(got, ref.forward(c), what=f"{name} interleaved K/V splits={splits}")
    assert torch.equal(got, base), f"{name}: interleaved and contiguous caches disagree"
    assert_no_device_error()
