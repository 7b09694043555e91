"""Calls captured in a CUDA graph: the query-length bucket (bucket_max_seqlen_q
in the vLLM API docs for fa4_rel_attention) as max_seqlen_q, then replays after
the cache lengths change on the device, each replay checked against the oracle."""
import pytest
import torch

from oracle import reference as ref
from paged_attention_relative_gb300.workloads import make_case
from tests.gpu_util import assert_close, assert_no_device_error, to_dev

pytestmark = pytest.mark.gpu


def _call(pa, c, g, out, max_seqlen_q, splits):
    pa.rel_attn_paged_varlen(g["q"], g["key_cache"], g["value_cache"], g["block_table"], g["cache_seqlens"],
                             g["cu_seqlens_q"], max_seqlen_q, c.softmax_scale, c.causal, c.window_left,
                             c.window_right, c.rel_extent, g["rel_logits"], splits, out=out)


@pytest.mark.parametrize("kind", ["decode", "prefill", "prefill_pair"])
def test_captured_call_replays_with_new_cache_lengths(kind, monkeypatch):
    import paged_attention_relative_gb300 as pa
    if kind == "prefill_pair":
        monkeypatch.setenv("REL_ATTN_PREFILL_PAIR", "1")
    if kind == "decode":
        c = make_case(seed=21, seqlens_q=[1, 1, 1], seqlens_k=[700, 1300, 260], num_heads=8, num_kv_heads=2,
                      head_dim=128, rel_extent=64)
        splits, shorter = 4, [333, 1000, 17]
    else:
        c = make_case(seed=22, seqlens_q=[70, 40], seqlens_k=[500, 300], num_heads=8, num_kv_heads=2,
                      head_dim=128, rel_extent=48)
        splits, shorter = 1, [200, 41]
    g = to_dev(c)
    out = torch.empty_like(g["q"])
    bucket = pa.rel_attn_bucket_max_seqlen_q(c.max_seqlen_q)
    assert bucket >= c.max_seqlen_q
    _call(pa, c, g, out, bucket, splits)  # first call outside the capture (library set-up)
    torch.cuda.synchronize()

    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        _call(pa, c, g, out, bucket, splits)
    out.zero_()
    graph.replay()
    torch.cuda.synchronize()
    assert_close(out, ref.forward(c), what=f"{kind} replay")

    # Same shapes, shorter caches: the captured launch reads the new lengths.
    new = torch.tensor(shorter, dtype=torch.int32)
    g["cache_seqlens"].copy_(new)
    c2 = c.with_(cache_seqlens=new)
    graph.replay()
    torch.cuda.synchronize()
    assert_close(out, ref.forward(c2), what=f"{kind} replay, new lengths")
    assert_no_device_error()
