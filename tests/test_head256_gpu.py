"""head_dim 256 against the fp64 oracle, through the C ABI: the decode kernel
(each 16-key slice on a pair of warps, one per dim half) and the CTA-pair
prefill kernel (2-SM MMAs, O in TMEM columns [256, 512)), with splits, the
split-vs-single bound, windows, bias extents that are and are not staged by
TMA, fp32 rel_logits, the log-sum-exp output, and one chunked-prefill case
checked on every output."""
import numpy as np
import pytest
import torch

from oracle import reference as ref
from paged_attention_relative_gb300.workloads import make_case
from tests.gpu_util import assert_close, assert_no_device_error, assert_split_matches_single, run, to_dev

pytestmark = pytest.mark.gpu

DECODE = [
    dict(name="mha", seqlens_q=[1, 3, 2], seqlens_k=[300, 77, 16], num_heads=4, num_kv_heads=4),
    dict(name="gqa8", seqlens_q=[2, 1], seqlens_k=[700, 1000], num_heads=16, num_kv_heads=2, rel_extent=64),
    dict(name="rows32", seqlens_q=[8, 3], seqlens_k=[200, 40], num_heads=8, num_kv_heads=2, rel_extent=24),
    dict(name="rows64", seqlens_q=[16, 5], seqlens_k=[333, 16], num_heads=8, num_kv_heads=2, rel_extent=7),
    dict(name="window", seqlens_q=[4, 2], seqlens_k=[400, 260], num_heads=8, num_kv_heads=2, window=(100, 0)),
    dict(name="noncausal_window", seqlens_q=[6], seqlens_k=[300], num_heads=4, num_kv_heads=2, causal=False,
         window=(37, 11)),
    dict(name="short_and_empty", seqlens_q=[0, 3, 6], seqlens_k=[50, 40, 2], num_heads=4, num_kv_heads=2),
    dict(name="block32", seqlens_q=[2, 1], seqlens_k=[95, 200], num_heads=8, num_kv_heads=2, block_size=32),
]

PREFILL = [
    dict(name="gqa4_two_tiles", seqlens_q=[40, 17], seqlens_k=[300, 17], num_heads=8, num_kv_heads=2,
         rel_extent=64),
    dict(name="mha_130", seqlens_q=[130], seqlens_k=[260], num_heads=2, num_kv_heads=2, rel_extent=32),
    dict(name="gqa8_ragged", seqlens_q=[20, 9, 33], seqlens_k=[150, 400, 33], num_heads=16, num_kv_heads=2,
         rel_extent=16),
    dict(name="gqa3_rows_126", seqlens_q=[50], seqlens_k=[260], num_heads=6, num_kv_heads=2, rel_extent=24),
    dict(name="window_left", seqlens_q=[100], seqlens_k=[700], num_heads=4, num_kv_heads=1, window=(130, 0),
         rel_extent=48),
    dict(name="noncausal_window", seqlens_q=[80], seqlens_k=[300], num_heads=4, num_kv_heads=4, causal=False,
         window=(40, 25)),
    dict(name="no_bias", seqlens_q=[66, 70], seqlens_k=[500, 70], num_heads=8, num_kv_heads=8, rel_extent=0),
    dict(name="bias_r7_per_element", seqlens_q=[65], seqlens_k=[129], num_heads=2, num_kv_heads=1,
         rel_extent=7),
    dict(name="short_cache", seqlens_q=[100, 80], seqlens_k=[30, 0], num_heads=4, num_kv_heads=4),
    dict(name="block32", seqlens_q=[33], seqlens_k=[333], num_heads=8, num_kv_heads=2, block_size=32),
]


def _case(cfg, seed_base):
    kw = dict(cfg)
    name = kw.pop("name")
    kw.setdefault("rel_extent", 16)
    return name, make_case(seed=seed_base + sum(map(ord, name)) % 997, head_dim=256, **kw)


@pytest.mark.parametrize("cfg", DECODE, ids=[c["name"] for c in DECODE])
@pytest.mark.parametrize("splits", [1, 3])
def test_decode_head256_matches_oracle(cfg, splits):
    import paged_attention_relative_gb300 as pa
    name, c = _case(cfg, 0)
    got = run(c, num_splits=splits)
    assert pa.last_launch()["kernel"] == "decode"
    assert_close(got, ref.forward(c), what=f"decode d256 {name} splits={splits}")
    assert_no_device_error()


@pytest.mark.parametrize("cfg", PREFILL, ids=[c["name"] for c in PREFILL])
@pytest.mark.parametrize("splits", [1, 3])
def test_prefill_head256_matches_oracle(cfg, splits):
    import paged_attention_relative_gb300 as pa
    name, c = _case(cfg, 1000)
    got = run(c, num_splits=splits)
    assert pa.last_launch()["kernel"] == "prefill_pair"
    assert_close(got, ref.forward(c), what=f"prefill d256 {name} splits={splits}")
    assert_no_device_error()


@pytest.mark.parametrize("kind", ["decode", "prefill"])
def test_head256_split_matches_single(kind):
    if kind == "decode":
        c = make_case(seed=7, seqlens_q=[1, 4], seqlens_k=[3000, 900], num_heads=16, num_kv_heads=2,
                      head_dim=256, rel_extent=256)
    else:
        c = make_case(seed=8, seqlens_q=[70, 130], seqlens_k=[700, 1000], num_heads=8, num_kv_heads=2,
                      head_dim=256, rel_extent=64)
    g = to_dev(c)
    for splits in (2, 5):
        d32 = assert_split_matches_single(c, g, splits)
        print(f"{kind} head_dim 256 split {splits} vs single, fp32 out: max |diff| {d32:.3e}")
    assert_no_device_error()


@pytest.mark.parametrize("kind", ["decode", "prefill"])
def test_head256_fp32_rel_logits_and_lse(kind):
    import paged_attention_relative_gb300 as pa
    sq = [2, 3] if kind == "decode" else [70, 40]
    c = make_case(seed=9, seqlens_q=sq, seqlens_k=[400, 260], num_heads=8, num_kv_heads=2, head_dim=256,
                  rel_extent=40)
    c = c.with_(rel_logits=torch.randn(c.rel_logits.shape, generator=torch.Generator().manual_seed(3)))
    g = to_dev(c)
    want, want_lse = ref.forward(c, with_lse=True)
    for splits in (1, 3):
        out, lse = pa.rel_attn_paged_varlen_lse(g["q"], g["key_cache"], g["value_cache"], g["block_table"],
                                                g["cache_seqlens"], g["cu_seqlens_q"], c.max_seqlen_q,
                                                c.softmax_scale, c.causal, c.window_left, c.window_right,
                                                c.rel_extent, g["rel_logits"], splits)
        torch.cuda.synchronize()
        assert_close(out, want, what=f"{kind} d256 fp32 bias splits={splits}")
        got = lse.cpu().double().numpy()
        fin = np.isfinite(want_lse)
        assert np.array_equal(np.isfinite(got), fin)
        assert np.all(np.abs(got[fin] - want_lse[fin]) <= 1e-3 + 1e-5 * np.abs(want_lse[fin]))
    assert_no_device_error()


def test_chunked_prefill_head256_every_output():
    """A chunked-prefill shape at head_dim 256 (1024 new tokens on a 1024-token
    prefix, 32/8 heads, rel_extent 512), every output against the oracle."""
    import paged_attention_relative_gb300 as pa
    c = make_case(seed=10, seqlens_q=[1024], seqlens_k=[2048], num_heads=32, num_kv_heads=8, head_dim=256,
                  rel_extent=512, rel_std=0.5)
    got = run(c)
    assert pa.last_launch()["kernel"] == "prefill_pair"
    err = np.abs(got.float().cpu().numpy().astype(np.float64) - ref.forward(c))
    print(f"chunked prefill d256: max-abs {err.max():.3e}, mean-abs {err.mean():.3e} over {err.size} outputs")
    assert err.max() <= 2e-2 and err.mean() <= 2e-3
    assert_no_device_error()
