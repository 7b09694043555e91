"""Parity of the tcgen05 prefill path (more than 64 GQA-packed rows per
request and kv head) against the fp64 oracle, through the C ABI: small cases
that span several 128-row and 128-key tiles with ragged tails, edge cases
(short caches, empty requests, windows, no bias, odd bias extents, splits,
block size 32, fp32 output, stale page tails), and the full-size chunked
prefill and mixed windowed workloads checked on sampled output rows."""
import numpy as np
import pytest
import torch

from oracle import reference as ref
from paged_attention_relative_gb300.workloads import chunked_prefill, make_case, mixed_window
from tests.gpu_util import assert_close, assert_no_device_error, run, to_dev

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
def test_prefill_small_cases_match_oracle(cfg, splits):
    import paged_attention_relative_gb300 as pa
    kw = dict(cfg)
    name = kw.pop("name")
    kw.setdefault("rel_extent", 16)
    c = make_case(seed=(sum(map(ord, name)) % 997), **kw)
    got = run(c, num_splits=splits)
    assert pa.last_launch()["kernel"] == "prefill"
    assert_close(got, ref.forward(c), what=f"{name} splits={splits}")
    assert_no_device_error()


def test_prefill_split_matches_single_fp32():
    c = make_case(seed=3, seqlens_q=[64, 40], seqlens_k=[900, 600], num_heads=8, num_kv_heads=2, head_dim=128,
                  rel_extent=200)
    g = to_dev(c)
    a = torch.empty(c.q.shape, dtype=torch.float32, device="cuda")
    b = torch.empty_like(a)
    run(c, g, num_splits=4, out=a)
    run(c, g, num_splits=1, out=b)
    # Both paths round every softmax weight p to bf16 (relative error <= 2^-9)
    # against their own reference maximum and keep everything else in fp32, so
    # each lies within 2^-9 * sum_j (p_j / l) |v_j| of the exact output and
    # the two within twice that: the attention of |V|, from the oracle.
    bound = torch.from_numpy(ref.forward(c.with_(value_cache=c.value_cache.abs()))).float().cuda()
    diff = (a - b).abs()
    assert (diff <= 2.0 ** -8 * bound + 1e-5).all(), f"split vs single {diff.max().item():.3e}"
    assert diff.mean().item() <= 1e-4
    assert_close(a, ref.forward(c), tol_max=5e-3, tol_mean=5e-4, what="fp32 out")


def test_prefill_stale_page_tail_does_not_leak():
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


def _sampled_rows(c, n, seed):
    rng = np.random.default_rng(seed)
    T, H = c.q.shape[:2]
    idx = rng.choice(T * H, size=min(n, T * H), replace=False)
    return idx // H, idx % H


@pytest.mark.parametrize("make", [chunked_prefill, mixed_window], ids=["chunked_prefill", "mixed_window"])
def test_full_size_workload_on_sampled_rows(make):
    import paged_attention_relative_gb300 as pa
    c = make(0)
    got = run(c).float().cpu().numpy().astype(np.float64)
    assert pa.last_launch()["kernel"] == "prefill"
    assert np.isfinite(got).all()
    t, h = _sampled_rows(c, 384, 1)
    want = ref.forward_rows(c, t, h)
    err = np.abs(got[t, h] - want)
    assert err.max() <= 2e-2 and err.mean() <= 2e-3, (err.max(), err.mean())
    # the last token of every request (the bias band and the causal diagonal)
    cu = c.cu_seqlens_q.tolist()
    last = [cu[b + 1] - 1 for b in range(len(cu) - 1) if cu[b + 1] > cu[b]]
    tt = np.repeat(last, 2)
    hh = np.tile([0, c.q.shape[1] - 1], len(last))
    err = np.abs(got[tt, hh] - ref.forward_rows(c, tt, hh))
    assert err.max() <= 2e-2, err.max()
    assert_no_device_error()


def test_prefill_batch_above_compact_limit():
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
    assert pa.last_launch()["kernel"] == "prefill"
    assert pa.last_launch()["grid"][2] == 300
    assert_close(got, ref.forward(c), what="300 requests")
    assert_no_device_error()


def test_prefill_compact_grid_with_inflated_max_seqlen_q():
    """max_seqlen_q far above the longest query: the compact launch is bounded
    by the rows (T / 64 pairs plus one per request) and still covers every pair."""
    import paged_attention_relative_gb300 as pa
    c = make_case(seed=13, seqlens_q=[1, 130, 0, 65, 7], seqlens_k=[300, 400, 10, 65, 900], num_heads=8,
                  num_kv_heads=2, head_dim=128, rel_extent=40)
    got = run(c, max_seqlen_q=8 * c.max_seqlen_q, num_splits=2)
    info = pa.last_launch()
    assert info["kernel"] == "prefill"
    T = c.q.shape[0]
    assert info["grid"][0] == 2 * ((T + 63) // 64 + 5)
    assert_close(got, ref.forward(c), what="inflated max_seqlen_q")
    assert_no_device_error()


@pytest.mark.parametrize("splits", [1, 3])
def test_prefill_strided_q_and_out_with_guard(splits):
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
