"""Host-side checks of the C ABI that need no GPU: the library loads and
exports every function the headers declare, the split heuristic equals the
oracle's restatement, and argument validation rejects bad calls before any
device work."""
import os
import re

import numpy as np
import pytest
import torch

from oracle import reference as ref

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _lib():
    from paged_attention_relative_gb300 import _lib
    return _lib


def _declared_functions():
    names = set()
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if not fn.endswith(".h"):
            continue
        src = open(os.path.join(ROOT, "include", fn)).read()
        src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
        for m in re.finditer(r"^[A-Za-z_][\w \*]*?\b(rel_attn_\w+)\s*\(", src, flags=re.M):
            names.add(m.group(1))
    return names


def test_library_exports_every_declared_function():
    names = _declared_functions()
    assert {"rel_attn_paged_varlen", "rel_attn_num_splits", "rel_attn_last_error"} <= names
    L = _lib()
    for n in sorted(names):
        assert hasattr(L.lib, n), n
    assert names == set(L.EXPORTS)


def _golden(name):
    rows = []
    for line in open(os.path.join(ROOT, "tests", "golden", name)):
        line = line.split("#")[0].strip()
        if line:
            rows.append([int(x) for x in line.split()])
    return rows


def test_bucket_max_seqlen_q_matches_worked_values():
    L = _lib()
    for n, want in _golden("bucket_max_seqlen_q.txt"):
        assert L.rel_attn_bucket_max_seqlen_q(n) == want
    assert L.rel_attn_bucket_max_seqlen_q(1 << 30) == 1 << 30
    for bad in (-1, (1 << 30) + 1):
        assert L.lib.rel_attn_bucket_max_seqlen_q(bad) == -1


def test_num_splits_equals_oracle_on_worked_values():
    L = _lib()
    for is_local, B, mq, H, Hk, kv, cap, want in _golden("num_splits_cases.txt"):
        if cap == 9:
            continue  # the library runs on sm_103 only; the Hopper branch is not part of it
        assert L.rel_attn_num_splits(is_local, B, mq, H, Hk, kv) == want


def test_num_splits_equals_oracle_on_a_sweep():
    L = _lib()
    rng = np.random.default_rng(0)
    for _ in range(3000):
        Hk = int(rng.choice([1, 2, 4, 8, 16]))
        H = Hk * int(rng.choice([1, 2, 4, 8, 16]))
        B = int(rng.integers(1, 70))
        mq = int(rng.choice([1, 2, 4, 64, 255, 256, 257, 1024, 4096]))
        kv = int(rng.choice([0, 1, 127, 128, 129, 8192, 8193, 65536, 65537, 131072, 1 << 20]))
        loc = int(rng.integers(0, 2))
        want = ref.num_splits(is_local=bool(loc), batch_size=B, max_query_len=mq, num_heads=H,
                              num_kv_heads=Hk, max_kv_len=kv)
        assert L.rel_attn_num_splits(loc, B, mq, H, Hk, kv) == want


@pytest.mark.parametrize("args", [(0, 0, 1, 8, 8, 10), (0, 1, 0, 8, 8, 10), (0, 1, 1, 6, 4, 10),
                                  (0, 1, 1, 8, 0, 10), (0, 1, 1, 8, 8, -1)])
def test_num_splits_rejects_invalid_sizes(args):
    L = _lib()
    assert L.lib.rel_attn_num_splits(*args) == -1
    assert L.lib.rel_attn_last_error().decode()


def _cpu_case(**kw):
    from paged_attention_relative_gb300.workloads import make_case
    base = dict(seed=0, seqlens_q=[2, 1], seqlens_k=[20, 5], num_heads=4, num_kv_heads=2, head_dim=64,
                block_size=16, rel_extent=8)
    base.update(kw)
    return make_case(**base)


def _call(c, **over):
    L = _lib()
    args = dict(q=c.q, key_cache=c.key_cache, value_cache=c.value_cache, block_table=c.block_table,
                cache_seqlens=c.cache_seqlens, cu_seqlens_q=c.cu_seqlens_q, max_seqlen_q=c.max_seqlen_q,
                softmax_scale=c.softmax_scale, causal=c.causal, window_left=-1, window_right=-1,
                rel_extent=c.rel_extent, rel_logits=c.rel_logits, num_splits=1, out=torch.empty_like(c.q),
                stream=0)
    args.update(over)
    return L.rel_attn_paged_varlen(**args)


@pytest.mark.parametrize("over,status", [
    (dict(num_splits=0), 1),
    (dict(rel_extent=-1), 1),
    (dict(rel_extent=9), 1),                                   # rel_logits last dim is 8
    (dict(block_table=torch.zeros(3, 2, dtype=torch.int32)), 1),
    (dict(cache_seqlens=torch.zeros(2, dtype=torch.int64)), 1),
    (dict(cu_seqlens_q=torch.tensor([0, 3], dtype=torch.int32)), 1),
    (dict(out=torch.empty(3, 4, 32, dtype=torch.bfloat16)), 1),
])
def test_invalid_arguments_are_rejected_before_device_work(over, status):
    L = _lib()
    c = _cpu_case()
    with pytest.raises(L.RelAttnError) as ei:
        _call(c, **over)
    assert ei.value.status == status


def test_head_count_must_divide():
    L = _lib()
    c = _cpu_case(num_heads=6, num_kv_heads=4)
    with pytest.raises(L.RelAttnError) as ei:
        _call(c)
    assert ei.value.status == 1


def test_unsupported_head_dim_and_block_size():
    L = _lib()
    for kw in (dict(head_dim=96), dict(block_size=8)):
        c = _cpu_case(**kw)
        with pytest.raises(L.RelAttnError) as ei:
            _call(c)
        assert ei.value.status == 2, kw


def test_out_aliasing_q_is_rejected():
    L = _lib()
    c = _cpu_case()
    with pytest.raises(L.RelAttnError) as ei:
        _call(c, out=c.q)
    assert ei.value.status == 1


def test_non_contiguous_rel_logits_is_rejected():
    L = _lib()
    c = _cpu_case()
    rel = torch.empty(c.rel_logits.shape[0], c.rel_logits.shape[1], 16, dtype=torch.bfloat16)[:, :, :8]
    with pytest.raises(L.RelAttnError) as ei:
        _call(c, rel_logits=rel)
    assert ei.value.status == 1


def test_empty_batch_is_a_no_op():
    L = _lib()
    c = _cpu_case()
    q0 = c.q[:0]
    out = _call(c, q=q0, out=torch.empty_like(q0), rel_logits=c.rel_logits[:0],
                cu_seqlens_q=torch.zeros(3, dtype=torch.int32), max_seqlen_q=0)
    assert out.shape[0] == 0
    assert L.last_launch()["kernel"] == "none"


@pytest.mark.parametrize("make_lse", [
    lambda c, out: torch.empty(c.q.shape[0], c.q.shape[1] + 1, dtype=torch.float32),   # wrong shape
    lambda c, out: torch.empty(c.q.shape[0], c.q.shape[1], dtype=torch.bfloat16),      # wrong dtype
    lambda c, out: torch.empty(c.q.shape[0], dtype=torch.float32),                     # wrong rank
    lambda c, out: out.view(torch.float32)[:, :, 0],                                   # aliases out
], ids=["shape", "dtype", "rank", "aliases_out"])
def test_lse_argument_is_validated_before_device_work(make_lse):
    L = _lib()
    c = _cpu_case()
    out = torch.empty_like(c.q)
    with pytest.raises(L.RelAttnError) as ei:
        L.rel_attn_paged_varlen_lse(c.q, c.key_cache, c.value_cache, c.block_table, c.cache_seqlens,
                                    c.cu_seqlens_q, c.max_seqlen_q, c.softmax_scale, c.causal, -1, -1,
                                    c.rel_extent, c.rel_logits, 1, out=out, softmax_lse=make_lse(c, out), stream=0)
    assert ei.value.status == 1


@pytest.mark.parametrize("what", ["shape", "alias"])
def test_cache_append_validates_before_device_work(what):
    L = _lib()
    c = _cpu_case()
    T, Hk, D = c.q.shape[0], c.key_cache.shape[2], c.key_cache.shape[3]
    key = torch.zeros(T, Hk + 1, D, dtype=torch.bfloat16) if what == "shape" else c.key_cache[0, :T]
    value = torch.zeros(T, Hk, D, dtype=torch.bfloat16)
    if what == "alias":
        key = c.value_cache.view(-1, Hk, D)[:T]
    with pytest.raises(L.RelAttnError) as ei:
        L.rel_attn_cache_append(key, value, c.key_cache, c.value_cache, c.block_table, c.cache_seqlens,
                                c.cu_seqlens_q, stream=0)
    assert ei.value.status == 1


@pytest.mark.parametrize("ms", [0, -5, 10001])
def test_wait_timeout_self_test_rejects_out_of_range_limits(ms):
    L = _lib()
    assert L.lib.rel_attn_check_wait_timeout(ms, None) == 1


@pytest.mark.parametrize("over", [
    dict(num_splits=0), dict(rel_extent=-1), dict(rel_extent=9), dict(out="alias_q"),
    dict(block_table=torch.zeros(3, 2, dtype=torch.int32)), dict(max_seqlen_q=-1),
    dict(value_cache="strided"), dict(case=dict(head_dim=96)), dict(case=dict(block_size=8)),
    dict(case=dict(num_heads=6, num_kv_heads=4)),
], ids=["splits0", "rel_neg", "rel_shape", "alias", "table", "maxq", "v_strides", "d96", "bs8", "heads"])
def test_noalloc_validates_like_the_allocating_entry_point(over):
    """The allocation-free entry point shares the allocating one's validation:
    the same status for every bad call, before any device work."""
    L = _lib()
    over = dict(over)
    c = _cpu_case(**over.pop("case", {}))
    if over.get("out") == "alias_q":
        over["out"] = c.q
    if over.get("value_cache") == "strided":
        vc = torch.zeros(c.value_cache.shape[0], c.value_cache.shape[1], c.value_cache.shape[2],
                         2 * c.value_cache.shape[3], dtype=torch.bfloat16)
        over["value_cache"] = vc[..., :c.value_cache.shape[3]]
    statuses = []
    for fn in (L.rel_attn_paged_varlen, L.rel_attn_paged_varlen_noalloc):
        args = dict(q=c.q, key_cache=c.key_cache, value_cache=c.value_cache, block_table=c.block_table,
                    cache_seqlens=c.cache_seqlens, cu_seqlens_q=c.cu_seqlens_q, max_seqlen_q=c.max_seqlen_q,
                    softmax_scale=c.softmax_scale, causal=c.causal, window_left=-1, window_right=-1,
                    rel_extent=c.rel_extent, rel_logits=c.rel_logits, num_splits=1, out=torch.empty_like(c.q),
                    stream=0)
        args.update(over)
        with pytest.raises(L.RelAttnError) as ei:
            fn(**args)
        statuses.append(ei.value.status)
    assert statuses[0] == statuses[1] and statuses[0] in (1, 2), statuses
