"""Tensors that are not device memory of the current device (host memory,
pageable or pinned) are rejected with REL_ATTN_ERR_UNSUPPORTED before any
tensor map is encoded or kernel launched, on the decode and the prefill path
and in the cache append.  Nothing here reaches a kernel: the check runs on
the host."""
import pytest
import torch

from paged_attention_relative_gb300.workloads import make_case
from tests.gpu_util import assert_no_device_error, to_dev

pytestmark = pytest.mark.gpu

DECODE = dict(seqlens_q=[1, 2], seqlens_k=[100, 40], num_heads=8, num_kv_heads=4, head_dim=128, rel_extent=16)
PREFILL = dict(seqlens_q=[70], seqlens_k=[200], num_heads=8, num_kv_heads=2, head_dim=128, rel_extent=16)


def _call(c, g, out):
    import paged_attention_relative_gb300 as pa
    pa.rel_attn_paged_varlen(g["q"], g["key_cache"], g["value_cache"], g["block_table"], g["cache_seqlens"],
                             g["cu_seqlens_q"], c.max_seqlen_q, c.softmax_scale, c.causal, c.window_left,
                             c.window_right, c.rel_extent, g["rel_logits"], 1, out=out,
                             stream=torch.cuda.current_stream())


@pytest.mark.parametrize("shape", [DECODE, PREFILL], ids=["decode", "prefill"])
@pytest.mark.parametrize("which", ["key_cache", "value_cache", "rel_logits", "q", "block_table", "cu_seqlens_q",
                                   "out"])
@pytest.mark.parametrize("pinned", [False, True], ids=["pageable", "pinned"])
def test_host_tensor_is_rejected(shape, which, pinned):
    from paged_attention_relative_gb300 import _lib as L
    c = make_case(seed=21, **shape)
    g = to_dev(c)
    out = torch.empty_like(g["q"])
    host = (torch.empty_like(c.q) if which == "out" else getattr(c, which)).contiguous()
    if pinned:
        host = host.pin_memory()
    if which == "out":
        out = host
    else:
        g[which] = host
    with pytest.raises(L.RelAttnError) as ei:
        _call(c, g, out)
    assert ei.value.status == 2, str(ei.value)
    assert "not device memory of the current device" in str(ei.value)
    assert L.last_launch()["kernel"] == "none"
    assert_no_device_error()


def test_cache_append_rejects_host_cache():
    import paged_attention_relative_gb300 as pa
    from paged_attention_relative_gb300 import _lib as L
    c = make_case(seed=22, **PREFILL)
    g = to_dev(c)
    T, Hk, D = c.q.shape[0], c.key_cache.shape[2], c.key_cache.shape[3]
    key = torch.zeros(T, Hk, D, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(L.RelAttnError) as ei:
        pa.rel_attn_cache_append(key, key.clone(), c.key_cache, g["value_cache"], g["block_table"],
                                 g["cache_seqlens"], g["cu_seqlens_q"], stream=torch.cuda.current_stream())
    assert ei.value.status == 2 and "key_cache" in str(ei.value)
    assert_no_device_error()
