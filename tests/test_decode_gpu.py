"""Parity of the decode (<= 64 packed rows) path against the fp64 oracle,
through the C ABI, on the tiny, long-decode and batched-decode workloads and a
matrix of small edge cases (GQA ratios, head dims, windows, bias extents,
empty and ragged requests, short caches, splits, strided tensors, stale page
contents)."""
import numpy as np
import pytest
import torch

from oracle import reference as ref
from paged_attention_relative_gb300.workloads import (batched_decode, long_decode, make_case, tiny_mixed)
from tests.gpu_util import (assert_close, assert_no_device_error, assert_split_matches_single, run,
                            to_dev)

pytestmark = pytest.mark.gpu


def test_tiny_mixed_matches_oracle():
    import paged_attention_relative_gb300 as pa
    c = tiny_mixed(0)
    got = run(c)
    assert pa.last_launch()["kernel"] == "decode"
    assert_close(got, ref.forward(c), what="tiny_mixed")
    assert_no_device_error()


@pytest.fixture(scope="module")
def long_case():
    c = long_decode(0)
    return c, to_dev(c), ref.forward(c)


@pytest.mark.parametrize("splits", [16, 1, 5])
def test_long_decode_matches_oracle(long_case, splits):
    import paged_attention_relative_gb300 as pa
    c, g, want = long_case
    got = run(c, g, num_splits=splits)
    info = pa.last_launch()
    assert info["num_splits"] == splits and info["launches"] == (2 if splits > 1 else 1)
    assert_close(got, want, what=f"long_decode splits={splits}")
    assert_no_device_error()


def test_long_decode_split_equals_single(long_case):
    c, g, _ = long_case
    d32 = assert_split_matches_single(c, g, 16)
    print(f"long decode split 16 vs single, fp32 out: max |diff| {d32:.3e}")


def test_decode_split_matches_single_concentrated_rows():
    """Rows whose weight sits on a few keys (a large bias at a few distances):
    the case where a P rounding that depended on the split partition would
    move the output by most."""
    c = make_case(seed=8, seqlens_q=[1, 4, 2], seqlens_k=[3000, 900, 2000], num_heads=16, num_kv_heads=2,
                  head_dim=128, rel_extent=256)
    rel = c.rel_logits.float()
    rel[:, :, 3] += 12.0
    rel[:, :, 200] += 9.0
    c = c.with_(rel_logits=rel.to(torch.bfloat16))
    g = to_dev(c)
    for splits in (2, 5, 16):
        d32 = assert_split_matches_single(c, g, splits)
        print(f"decode concentrated rows, split {splits} vs single, fp32 out: max |diff| {d32:.3e}")
    assert_close(run(c, g, num_splits=5), ref.forward(c), what="concentrated rows")


def test_batched_decode_matches_oracle():
    c = batched_decode(0)
    g = to_dev(c)
    want = ref.forward(c)
    split = ref.num_splits(is_local=False, batch_size=64, max_query_len=1, num_heads=64, num_kv_heads=4,
                           max_kv_len=int(c.cache_seqlens.max()))
    assert split == 1
    assert_close(run(c, g, num_splits=split), want, what="batched_decode")
    a = run(c, g, num_splits=4)
    assert_close(a, want, what="batched_decode splits=4")
    assert_split_matches_single(c, g, 4)
    assert_no_device_error()


def test_fp32_out_matches_oracle():
    c = tiny_mixed(0)
    g = to_dev(c)
    for splits in (1, 3):
        out = torch.empty(c.q.shape, dtype=torch.float32, device="cuda")
        run(c, g, out=out, num_splits=splits)
        assert_close(out, ref.forward(c), tol_max=5e-3, tol_mean=5e-4, what=f"fp32 out splits={splits}")


SMALL = [
    dict(name="mha_d128", seqlens_q=[1, 3, 2], seqlens_k=[300, 77, 16], num_heads=4, num_kv_heads=4, head_dim=128),
    dict(name="gqa2_d64", seqlens_q=[7, 1], seqlens_k=[129, 1], num_heads=8, num_kv_heads=4, head_dim=64),
    dict(name="gqa8", seqlens_q=[8, 2], seqlens_k=[500, 1000], num_heads=16, num_kv_heads=2, head_dim=128),
    dict(name="gqa16_4tok", seqlens_q=[4, 1, 3], seqlens_k=[64, 640, 65], num_heads=32, num_kv_heads=2,
         head_dim=128, rel_extent=40),
    dict(name="rows64_mha", seqlens_q=[64, 10], seqlens_k=[200, 10], num_heads=2, num_kv_heads=2, head_dim=64),
    dict(name="noncausal", seqlens_q=[3, 5], seqlens_k=[50, 90], num_heads=4, num_kv_heads=1, head_dim=128,
         causal=False),
    dict(name="window_left", seqlens_q=[4, 2], seqlens_k=[400, 260], num_heads=8, num_kv_heads=2, head_dim=128,
         window=(100, 0)),
    dict(name="window_both_noncausal", seqlens_q=[6], seqlens_k=[300], num_heads=4, num_kv_heads=2,
         head_dim=64, causal=False, window=(37, 11)),
    dict(name="window_right_only", seqlens_q=[6], seqlens_k=[300], num_heads=4, num_kv_heads=2, head_dim=64,
         causal=False, window=(-1, 5)),
    dict(name="no_bias", seqlens_q=[2, 2], seqlens_k=[100, 33], num_heads=8, num_kv_heads=8, head_dim=128,
         rel_extent=0),
    dict(name="bias_r1", seqlens_q=[2, 2], seqlens_k=[100, 33], num_heads=8, num_kv_heads=4, head_dim=128,
         rel_extent=1),
    dict(name="bias_r7_odd", seqlens_q=[3], seqlens_k=[70], num_heads=4, num_kv_heads=2, head_dim=64,
         rel_extent=7),
    dict(name="bias_wider_than_cache", seqlens_q=[2], seqlens_k=[20], num_heads=4, num_kv_heads=2, head_dim=64,
         rel_extent=100),
    dict(name="short_cache_sk_lt_sq", seqlens_q=[6, 3], seqlens_k=[2, 0], num_heads=4, num_kv_heads=2,
         head_dim=64),
    dict(name="empty_requests", seqlens_q=[0, 3, 0, 1], seqlens_k=[50, 40, 0, 17], num_heads=4, num_kv_heads=2,
         head_dim=128),
    dict(name="block32", seqlens_q=[2, 1], seqlens_k=[95, 200], num_heads=8, num_kv_heads=2, head_dim=128,
         block_size=32),
    # each row sees only its own position (rows past a short cache see nothing)
    dict(name="window_diagonal_only", seqlens_q=[3, 5], seqlens_k=[40, 3], num_heads=4, num_kv_heads=2,
         head_dim=128, window=(0, 0)),
    dict(name="window_left_noncausal", seqlens_q=[4], seqlens_k=[200], num_heads=8, num_kv_heads=2, head_dim=64,
         causal=False, window=(20, -1)),
    dict(name="big_pool", seqlens_q=[1], seqlens_k=[1000], num_heads=8, num_kv_heads=8, head_dim=128,
         pool_blocks=400, extra_table_cols=5),
]


@pytest.mark.parametrize("cfg", SMALL, ids=[c["name"] for c in SMALL])
@pytest.mark.parametrize("splits", [1, 2, 3, 16])
def test_small_cases_match_oracle(cfg, splits):
    kw = dict(cfg)
    name = kw.pop("name")
    kw.setdefault("rel_extent", 16)
    c = make_case(seed=hash(name) % 1000, **kw)
    got = run(c, num_splits=splits)
    assert_close(got, ref.forward(c), what=f"{name} splits={splits}")
    assert_no_device_error()


def test_stale_page_tail_does_not_leak():
    """Slots past cache_seqlens in a request's last page hold NaN: masked keys
    must contribute nothing."""
    c = make_case(seed=5, seqlens_q=[1, 2], seqlens_k=[37, 90], num_heads=8, num_kv_heads=2, head_dim=128,
                  rel_extent=16)
    k = c.key_cache.clone()
    v = c.value_cache.clone()
    BS = k.shape[1]
    for b, sk in enumerate(c.cache_seqlens.tolist()):
        last = int(c.block_table[b, (sk - 1) // BS])
        k[last, sk % BS:] = float("nan")
        v[last, sk % BS:] = float("nan")
    c = c.with_(key_cache=k, value_cache=v)
    for splits in (1, 4):
        got = run(c, num_splits=splits)
        assert torch.isfinite(got.float()).all()
        assert_close(got, ref.forward(c), what=f"stale tail splits={splits}")


def test_strided_q_and_out():
    c = make_case(seed=6, seqlens_q=[3, 2], seqlens_k=[60, 30], num_heads=8, num_kv_heads=2, head_dim=128,
                  rel_extent=16)
    g = to_dev(c)
    T, H, D = c.q.shape
    big_q = torch.zeros(T, H + 3, D, dtype=torch.bfloat16, device="cuda")
    big_q[:, :H] = g["q"]
    g["q"] = big_q[:, :H]
    big_o = torch.full((T, H, 2 * D), 7.0, dtype=torch.bfloat16, device="cuda")
    out = big_o[:, :, :D]
    run(c, g, out=out)
    assert_close(out, ref.forward(c), what="strided")
    assert torch.all(big_o[:, :, D:] == 7.0)  # nothing written outside the view


def test_out_guard_band_untouched():
    c = tiny_mixed(0)
    g = to_dev(c)
    n = c.q.numel()
    buf = torch.full((n + 2048,), 3.0, dtype=torch.bfloat16, device="cuda")
    out = buf[1024:1024 + n].view_as(c.q)
    for splits in (1, 3):
        run(c, g, out=out, num_splits=splits)
        assert torch.all(buf[:1024] == 3.0) and torch.all(buf[1024 + n:] == 3.0)


def test_num_splits_above_kv_tiles_is_clamped():
    c = make_case(seed=7, seqlens_q=[1], seqlens_k=[40], num_heads=4, num_kv_heads=4, head_dim=64, rel_extent=8)
    got = run(c, num_splits=1000)
    assert_close(got, ref.forward(c), what="clamped splits")


def test_single_key_returns_v():
    c = make_case(seed=8, seqlens_q=[1, 1], seqlens_k=[1, 1], num_heads=4, num_kv_heads=2, head_dim=128,
                  rel_extent=4)
    got = run(c).float().cpu()
    for b in range(2):
        v0 = c.value_cache[int(c.block_table[b, 0]), 0]
        for h in range(4):
            assert torch.equal(got[b, h], v0[h // 2].float())


@pytest.mark.parametrize("splits", [1, 2])
def test_decode_more_requests_than_the_ranked_limit(splits):
    """700 requests (above the 256 the kernel ranks by length): CTAs take
    requests in index order; lengths include empty caches."""
    import numpy as np
    import paged_attention_relative_gb300 as pa
    rng = np.random.default_rng(17)
    sk = rng.integers(0, 400, size=700)
    c = make_case(seed=18, seqlens_q=[1] * 700, seqlens_k=sk.tolist(), num_heads=16, num_kv_heads=2,
                  head_dim=64, rel_extent=24)
    got = run(c, num_splits=splits)
    assert pa.last_launch()["kernel"] == "decode"
    assert_close(got, ref.forward(c), what=f"700 requests splits={splits}")
    assert_no_device_error()


@pytest.mark.parametrize("sq,kernel", [(16, "decode"), (17, "prefill")])
def test_kernel_boundary_at_64_packed_rows(sq, kernel):
    """64 GQA-packed rows (16 tokens x 4 heads) is the decode kernel's
    largest case; 65 and above go to the tensor-core prefill kernel."""
    import paged_attention_relative_gb300 as pa
    c = make_case(seed=19, seqlens_q=[sq, 3], seqlens_k=[500, 90], num_heads=8, num_kv_heads=2, head_dim=128,
                  rel_extent=40)
    got = run(c)
    assert pa.last_launch()["kernel"] == kernel
    assert_close(got, ref.forward(c), what=f"sq={sq}")


@pytest.mark.parametrize("sq", [[1, 2], [70, 20]], ids=["decode", "prefill"])
def test_block_size_64(sq):
    c = make_case(seed=20, seqlens_q=sq, seqlens_k=[333, 129], num_heads=8, num_kv_heads=2, head_dim=128,
                  rel_extent=32, block_size=64)
    assert_close(run(c, num_splits=2), ref.forward(c), what=f"block 64 {sq}")
    assert_no_device_error()
