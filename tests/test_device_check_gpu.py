"""REL_ATTN_CHECK=1: a device-side check of the preconditions the kernels do
not test (block ids inside the cache, cache lengths inside the block table,
query lengths within max_seqlen_q) runs before the attention or the cache
append and turns a violation into REL_ATTN_ERR_DEVICE_CHECK without launching
them.  The check kernel reads only in-bounds entries (a cache length beyond
the table stops it before the table is read), so these cases are safe to run."""
import os

import pytest
import torch

from oracle import reference as ref
from paged_attention_relative_gb300.workloads import make_case
from tests.gpu_util import assert_close, run, to_dev

pytestmark = pytest.mark.gpu

DEVICE_CHECK = 5


@pytest.fixture
def checked(monkeypatch):
    monkeypatch.setenv("REL_ATTN_CHECK", "1")
    yield


def _case():
    return make_case(seed=41, seqlens_q=[3, 70], seqlens_k=[200, 300], num_heads=8, num_kv_heads=2,
                     head_dim=128, rel_extent=16)


def _call(c, g, **over):
    args = dict(max_seqlen_q=c.max_seqlen_q)
    args.update(over)
    return run(c, g, **args)


@pytest.mark.parametrize("bad", ["block_id", "cache_len", "max_seqlen_q"])
def test_violations_are_reported_before_the_attention_runs(checked, bad):
    import paged_attention_relative_gb300 as pa
    c = _case()
    g = to_dev(c)
    over = {}
    if bad == "block_id":
        g["block_table"][1, 3] = c.key_cache.shape[0] + 7
    elif bad == "cache_len":
        g["cache_seqlens"][0] = c.block_table.shape[1] * c.key_cache.shape[1] + 1
    else:
        over["max_seqlen_q"] = 69
    out_before = None
    with pytest.raises(pa.RelAttnError) as ei:
        out_before = _call(c, g, **over)
    assert ei.value.status == DEVICE_CHECK
    assert out_before is None
    assert pa.device_error() == 0


def test_valid_input_passes_the_check_and_matches_the_oracle(checked):
    c = _case()
    assert_close(_call(c, to_dev(c)), ref.forward(c), what="checked call")


def test_cache_append_checks_block_ids(checked):
    import paged_attention_relative_gb300 as pa
    c = _case()
    g = to_dev(c)
    g["block_table"][0, 0] = -1
    key = torch.zeros(c.q.shape[0], 2, 128, dtype=torch.bfloat16, device="cuda")
    before = g["key_cache"].clone()
    with pytest.raises(pa.RelAttnError) as ei:
        pa.rel_attn_cache_append(key, key.clone(), g["key_cache"], g["value_cache"], g["block_table"],
                                 g["cache_seqlens"], g["cu_seqlens_q"])
    assert ei.value.status == DEVICE_CHECK
    torch.cuda.synchronize()
    assert torch.equal(g["key_cache"], before)


def test_check_is_off_by_default():
    assert os.environ.get("REL_ATTN_CHECK") in (None, "", "0")
