"""Paged KV-cache append (rel_attn_cache_append) against the oracle: bit-exact
whole caches after the write, on small ragged cases (empty requests, caches
shorter than the query, block size 32, head_dim 64), strided key/value views
of a packed projection, the full chunked-prefill write, and the attention run
on the caches the kernel wrote."""
import pytest
import torch

from oracle import reference as ref
from paged_attention_relative_gb300.workloads import chunked_prefill, make_case
from tests.gpu_util import assert_close, assert_no_device_error, run, to_dev

pytestmark = pytest.mark.gpu

CASES = [
    dict(name="ragged", seqlens_q=[3, 17, 40], seqlens_k=[100, 17, 333], num_heads=8, num_kv_heads=2,
         head_dim=128),
    dict(name="empty_and_short", seqlens_q=[0, 9, 5, 0], seqlens_k=[40, 4, 5, 0], num_heads=4, num_kv_heads=4,
         head_dim=64),
    dict(name="block32", seqlens_q=[33, 1], seqlens_k=[70, 32], num_heads=8, num_kv_heads=8, head_dim=128,
         block_size=32),
    # a request with new tokens but an empty cache writes nothing
    dict(name="empty_cache", seqlens_q=[3, 4], seqlens_k=[0, 10], num_heads=4, num_kv_heads=2, head_dim=128),
]


def _rows(c, seed):
    g = torch.Generator().manual_seed(seed)
    T, Hk, D = c.q.shape[0], c.key_cache.shape[2], c.key_cache.shape[3]
    return (torch.randn(T, Hk, D, generator=g).to(torch.bfloat16),
            torch.randn(T, Hk, D, generator=g).to(torch.bfloat16))


def _append(g, key, value):
    import paged_attention_relative_gb300 as pa
    pa.rel_attn_cache_append(key, value, g["key_cache"], g["value_cache"], g["block_table"], g["cache_seqlens"],
                             g["cu_seqlens_q"])
    torch.cuda.synchronize()
    assert pa.last_launch()["kernel"] == ("append" if key.shape[0] > 0 else "none")


@pytest.mark.parametrize("cfg", CASES, ids=[c["name"] for c in CASES])
def test_append_matches_oracle_bit_for_bit(cfg):
    kw = dict(cfg)
    name = kw.pop("name")
    c = make_case(seed=sum(map(ord, name)) % 313, rel_extent=8, **kw)
    key, value = _rows(c, 5)
    want_k, want_v = ref.cache_append(c, key, value)
    g = to_dev(c)
    _append(g, key.cuda(), value.cuda())
    assert torch.equal(g["key_cache"].cpu(), want_k)
    assert torch.equal(g["value_cache"].cpu(), want_v)
    assert_no_device_error()


def test_append_from_strided_views_of_a_packed_projection():
    """key and value as views into one (T, H + 2 Hk, D) projection output."""
    c = make_case(seed=6, seqlens_q=[7, 30], seqlens_k=[50, 30], num_heads=8, num_kv_heads=2, head_dim=128,
                  rel_extent=8)
    key, value = _rows(c, 6)
    qkv = torch.cat([c.q, key, value], dim=1).cuda()  # (T, 8 + 2 + 2, D)
    g = to_dev(c)
    _append(g, qkv[:, 8:10], qkv[:, 10:12])
    want_k, want_v = ref.cache_append(c, key, value)
    assert torch.equal(g["key_cache"].cpu(), want_k)
    assert torch.equal(g["value_cache"].cpu(), want_v)


def test_append_full_chunked_prefill_write_then_attend():
    """The chunked-prefill workload's 4 x 4096 new tokens written into its
    caches (whole caches compared), then the attention over what was written,
    checked on sampled rows."""
    import numpy as np
    c = chunked_prefill(0)
    key, value = _rows(c, 7)
    want_k, want_v = ref.cache_append(c, key, value)
    g = to_dev(c)
    _append(g, key.cuda(), value.cuda())
    assert torch.equal(g["key_cache"].cpu(), want_k)
    assert torch.equal(g["value_cache"].cpu(), want_v)
    c2 = c.with_(key_cache=want_k, value_cache=want_v)
    got = run(c2, g).float().cpu().numpy().astype(np.float64)
    rng = np.random.default_rng(3)
    T, H = c.q.shape[:2]
    idx = rng.choice(T * H, size=128, replace=False)
    t, h = idx // H, idx % H
    err = np.abs(got[t, h] - ref.forward_rows(c2, t, h))
    assert err.max() <= 2e-2 and err.mean() <= 2e-3, (err.max(), err.mean())
    assert_no_device_error()


def test_append_of_zero_tokens_is_a_no_op():
    c = make_case(seed=8, seqlens_q=[0, 0], seqlens_k=[20, 3], num_heads=4, num_kv_heads=2, head_dim=64)
    key = torch.empty(0, 2, 64, dtype=torch.bfloat16, device="cuda")
    g = to_dev(c)
    _append(g, key, key.clone())
    assert torch.equal(g["key_cache"].cpu(), c.key_cache)
