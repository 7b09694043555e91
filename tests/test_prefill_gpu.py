"""Parity of the tcgen05 prefill path (more than 64 GQA-packed rows per
request and kv head) against the fp64 oracle, through the C ABI: small cases
that span several 128-row and 128-key tiles with ragged tails, edge cases
(short caches, empty requests, windows, no bias, odd bias extents, splits,
block size 32, fp32 output, stale page tails), split-KV against one split
within 1e-3, and every output of the full-size chunked-prefill and mixed
windowed workloads against the oracle."""
import numpy as np
import pytest
import torch

from oracle import reference as ref
from paged_attention_relative_gb300.workloads import chunked_prefill, make_case, mixed_window
from tests.gpu_util import (assert_close, assert_no_device_error, assert_split_matches_single,
                            expected_prefill_kernel, run, to_dev)


@pytest.fixture(params=["1cta", "pair"])
def prefill_kernel(request, monkeypatch):
    """Run a test on the one-CTA kernel (the default) and on the CTA-pair
    kernel (REL_ATTN_PREFILL_PAIR=1)."""
    if request.param == "pair":
        monkeypatch.setenv("REL_ATTN_PREFILL_PAIR", "1")
    else:
        monkeypatch.delenv("REL_ATTN_PREFILL_PAIR", raising=False)
    return request.param

pytestmark = pytest.mark.gpu

SMALL = [
    dict(name="gqa4_two_tiles", seqlens_q=[40, 17], seqlens_k=[300, 17], num_heads=8, num_kv_heads=2,
         head_dim=128, rel_extent=64),
    dict(name="mha_130_tokens", seqlens_q=[130], seqlens_k=[200], num_heads=2, num_kv_heads=2, head_dim=128,
         rel_extent=33),
    dict(name="gqa8_d64", seqlens_q=[20, 9], seqlens_k=[150, 400], num_heads=16, num_kv_heads=2, head_dim=64,
         rel_extent=16),
    dict(name="gqa16_one_token_per_8", seqlens_q=[9, 30], seqlens_k=[1000, 31], num_heads=32, num_kv_heads=2,
         head_dim=128, rel_extent=100),
    dict(name="gqa3_ragged_rows", seqlens_q=[50], seqlens_k=[260], num_heads=6, num_kv_heads=2, head_dim=128,
         rel_extent=20),
    dict(name="noncausal", seqlens_q=[70, 33], seqlens_k=[90, 256], num_heads=4, num_kv_heads=2, head_dim=128,
         causal=False),
    dict(name="window_left", seqlens_q=[100], seqlens_k=[700], num_heads=4, num_kv_heads=1, head_dim=128,
         window=(130, 0), rel_extent=50),
    dict(name="window_both", seqlens_q=[80], seqlens_k=[300], num_heads=4, num_kv_heads=4, head_dim=64,
         causal=False, window=(40, 25)),
    dict(name="no_bias", seqlens_q=[66, 70], seqlens_k=[500, 70], num_heads=8, num_kv_heads=8, head_dim=128,
         rel_extent=0),
    dict(name="bias_r7", seqlens_q=[65], seqlens_k=[129], num_heads=2, num_kv_heads=1, head_dim=128,
         rel_extent=7),
    dict(name="bias_wide", seqlens_q=[70], seqlens_k=[90], num_heads=2, num_kv_heads=2, head_dim=64,
         rel_extent=300),
    dict(name="short_cache", seqlens_q=[100, 80], seqlens_k=[30, 0], num_heads=4, num_kv_heads=4, head_dim=128),
    dict(name="empty_requests", seqlens_q=[0, 90, 0, 20], seqlens_k=[40, 400, 0, 500], num_heads=8,
         num_kv_heads=2, head_dim=128),
    dict(name="block32", seqlens_q=[33], seqlens_k=[333], num_heads=8, num_kv_heads=2, head_dim=128,
         block_size=32),
    # four tokens per tile: one bias box holds all 32 heads of a 4-token sub-box
    dict(name="gqa32_four_tokens_per_tile", seqlens_q=[11, 6], seqlens_k=[400, 6], num_heads=64,
         num_kv_heads=2, head_dim=128, rel_extent=96),
    # each row sees only its own position (rows past a short cache see nothing)
    dict(name="window_diagonal_only", seqlens_q=[70, 40], seqlens_k=[70, 20], num_heads=4, num_kv_heads=2,
         head_dim=128, window=(0, 0), rel_extent=8),
    dict(name="window_left_noncausal", seqlens_q=[66], seqlens_k=[400], num_heads=4, num_kv_heads=2,
         head_dim=64, causal=False, window=(100, -1), rel_extent=24),
    # one token per tile (every row of a tile is a head of the same token)
    dict(name="gqa128_one_token_per_tile", seqlens_q=[3, 2], seqlens_k=[260, 70], num_heads=128,
         num_kv_heads=1, head_dim=64, rel_extent=40),
]


@pytest.mark.parametrize("cfg", SMALL, ids=[c["name"] for c in SMALL])
@pytest.mark.parametrize("splits", [1, 3])
def test_prefill_small_cases_match_oracle(cfg, splits, prefill_kernel):
    import paged_attention_relative_gb300 as pa
    kw = dict(cfg)
    name = kw.pop("name")
    kw.setdefault("rel_extent", 16)
    c = make_case(seed=(sum(map(ord, name)) % 997), **kw)
    got = run(c, num_splits=splits)
    assert pa.last_launch()["kernel"] == expected_prefill_kernel(c)
    assert_close(got, ref.forward(c), what=f"{name} splits={splits}")
    assert_no_device_error()


def test_prefill_split_matches_single_fp32(prefill_kernel):
    c = make_case(seed=3, seqlens_q=[64, 40], seqlens_k=[900, 600], num_heads=8, num_kv_heads=2, head_dim=128,
                  rel_extent=200)
    g = to_dev(c)
    for splits in (2, 4, 7):
        d32 = assert_split_matches_single(c, g, splits)
        print(f"prefill split {splits} vs single, fp32 out: max |diff| {d32:.3e}")
    a = torch.empty(c.q.shape, dtype=torch.float32, device="cuda")
    run(c, g, num_splits=4, out=a)
    assert_close(a, ref.forward(c), what="fp32 out")


def test_prefill_split_matches_single_concentrated_rows(prefill_kernel):
    """Rows whose weight sits on a few keys (a large bias at a few distances):
    a bf16 rounding of P that depended on the split would show here first."""
    c = make_case(seed=4, seqlens_q=[70, 130], seqlens_k=[700, 1000], num_heads=8, num_kv_heads=2,
                  head_dim=128, rel_extent=64)
    rel = c.rel_logits.float()
    rel[:, :, 5] += 12.0
    rel[:, :, 40] += 9.0
    c = c.with_(rel_logits=rel.to(torch.bfloat16))
    g = to_dev(c)
    for splits in (2, 3, 8):
        d32 = assert_split_matches_single(c, g, splits)
        print(f"prefill concentrated rows, split {splits} vs single, fp32 out: max |diff| {d32:.3e}")
    assert_close(run(c, g, num_splits=3), ref.forward(c), what="concentrated rows")


def test_prefill_stale_page_tail_does_not_leak(prefill_kernel):
    c = make_case(seed=5, seqlens_q=[70], seqlens_k=[101], num_heads=4, num_kv_heads=2, head_dim=128,
                  rel_extent=16)
    k = c.key_cache.clone()
    v = c.value_cache.clone()
    last = int(c.block_table[0, 100 // 16])
    k[last, 101 % 16:] = float("nan")
    v[last, 101 % 16:] = float("nan")
    c = c.with_(key_cache=k, value_cache=v)
    got = run(c)
    assert torch.isfinite(got.float()).all()
    assert_close(got, ref.forward(c), what="stale tail")


@pytest.fixture(scope="module")
def chunked_full():
    """The chunked-prefill workload (4 x 4096 new tokens on 4096 cached, 32/8
    heads, R 2048) on the device, with the oracle's output for every row."""
    c = chunked_prefill(0)
    return c, to_dev(c), ref.forward(c)


def _assert_full(got, want, what):
    err = np.abs(got.float().cpu().numpy().astype(np.float64) - want)
    assert np.isfinite(err).all(), what
    print(f"{what}: max-abs {err.max():.3e}, mean-abs {err.mean():.3e} over {err.size} outputs")
    assert err.max() <= 2e-2 and err.mean() <= 2e-3, (what, err.max(), err.mean())


@pytest.mark.parametrize("splits", [1, 3])
def test_chunked_prefill_every_output_matches_oracle(chunked_full, splits):
    import paged_attention_relative_gb300 as pa
    c, g, want = chunked_full
    got = run(c, g, num_splits=splits)
    assert pa.last_launch()["kernel"] == expected_prefill_kernel(c)
    assert pa.last_launch()["num_splits"] == splits
    _assert_full(got, want, f"chunked prefill splits={splits}")
    assert_no_device_error()


def test_chunked_prefill_split_matches_single_full_size(chunked_full):
    c, g, _ = chunked_full
    for splits in (2, 4):
        d32 = assert_split_matches_single(c, g, splits)
        print(f"chunked prefill split {splits} vs single, fp32 out: max |diff| {d32:.3e}")
    assert_no_device_error()


def test_mixed_window_every_output_matches_oracle():
    import paged_attention_relative_gb300 as pa
    c = mixed_window(0)
    got = run(c)
    assert pa.last_launch()["kernel"] == expected_prefill_kernel(c)
    _assert_full(got, ref.forward(c), "mixed window")
    assert_no_device_error()


def test_prefill_batch_above_compact_limit(prefill_kernel):
    """More than 256 requests: every request gets max_seqlen_q's query tiles
    (empty clusters leave at once) instead of the compact cluster list."""
    import paged_attention_relative_gb300 as pa
    rng = np.random.default_rng(11)
    sq = rng.integers(1, 41, size=300)
    sq[0] = 40
    sk = sq + rng.integers(0, 100, size=300)
    c = make_case(seed=12, seqlens_q=sq.tolist(), seqlens_k=sk.tolist(), num_heads=8, num_kv_heads=2,
                  head_dim=64, rel_extent=16)
    got = run(c)
    assert pa.last_launch()["kernel"] == expected_prefill_kernel(c)
    assert pa.last_launch()["grid"][2] == 300
    assert_close(got, ref.forward(c), what="300 requests")
    assert_no_device_error()


def test_prefill_compact_grid_with_inflated_max_seqlen_q(prefill_kernel):
    """max_seqlen_q far above the longest query: the compact launch is bounded
    by the rows (T / 64 pairs of 32-token tiles plus one per request) and
    still covers every pair."""
    import paged_attention_relative_gb300 as pa
    c = make_case(seed=13, seqlens_q=[1, 130, 0, 65, 7], seqlens_k=[300, 400, 10, 65, 900], num_heads=8,
                  num_kv_heads=2, head_dim=128, rel_extent=40)
    got = run(c, max_seqlen_q=8 * c.max_seqlen_q, num_splits=2)
    info = pa.last_launch()
    assert info["kernel"] == expected_prefill_kernel(c)
    T = c.q.shape[0]
    assert info["grid"][0] == 2 * ((T + 63) // 64 + 5)
    assert_close(got, ref.forward(c), what="inflated max_seqlen_q")
    assert_no_device_error()


@pytest.mark.parametrize("splits", [1, 3])
def test_prefill_strided_q_and_out_with_guard(splits, prefill_kernel):
    """q as a view into a packed (T, H + 2 Hk, D) projection, out as a view of a
    wider buffer: results match and nothing outside the out view is written."""
    c = make_case(seed=61, seqlens_q=[70, 33], seqlens_k=[300, 120], num_heads=8, num_kv_heads=2, head_dim=128,
                  rel_extent=24)
    g = to_dev(c)
    T, H, D = c.q.shape
    qkv = torch.zeros(T, H + 4, D, dtype=torch.bfloat16, device="cuda")
    qkv[:, :H] = g["q"]
    g["q"] = qkv[:, :H]
    big_o = torch.full((T, H, 2 * D), 7.0, dtype=torch.bfloat16, device="cuda")
    out = big_o[:, :, D:]
    run(c, g, out=out, num_splits=splits)
    assert_close(out, ref.forward(c), what=f"strided prefill splits={splits}")
    assert torch.all(big_o[:, :, :D] == 7.0)
    assert_no_device_error()
