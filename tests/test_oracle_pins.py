"""Pins for the fp64 oracle: checks against things other than the oracle itself.

Each test is chosen so that a plausible mistake in the oracle fails it: a
library routine (torch SDPA with torch's own lower-right causal mask and GQA
expansion), closed forms (single key, zero query, zero scale, empty rows),
invariants (page relabelling, unused rel_logits columns, bias shift), a
one-hot bias that must select one key per (token, head) — which fails on a
wrong distance sign, a kv-head instead of query-head index or a local instead
of global token index — and an independently written brute force.
"""
import math

import numpy as np
import pytest
import torch
import torch.nn.functional as F
from torch.nn.attention.bias import causal_lower_right

from oracle import reference as ref
from paged_attention_relative_gb300.workloads import make_case, tiny_mixed


def _kv_contig(c, b, which):
    """Gather request b's cache rows into (sk, Hk, D) float64 (no attention math)."""
    cache = c.key_cache if which == "k" else c.value_cache
    BS = cache.shape[1]
    sk = int(c.cache_seqlens[b])
    rows = [cache[int(c.block_table[b, j // BS]), j % BS] for j in range(sk)]
    return torch.stack(rows).double() if rows else torch.zeros(0, *cache.shape[2:], dtype=torch.float64)


def _small(seed, **kw):
    base = dict(seed=seed, seqlens_q=[3, 4], seqlens_k=[9, 13], num_heads=4, num_kv_heads=2,
                head_dim=8, block_size=4, rel_extent=6, causal=True)
    base.update(kw)
    return make_case(**base)


# --------------------------------------------------------------------- brute force

BRUTE_CASES = [
    dict(),
    dict(causal=False),
    dict(window=(2, 0)),
    dict(window=(3, 1), causal=False),
    dict(window=(-1, 2), causal=False),
    dict(rel_extent=0),
    dict(rel_extent=1),
    dict(seqlens_q=[5, 0, 2], seqlens_k=[2, 4, 7]),          # sk < sq and an empty request
    dict(num_heads=6, num_kv_heads=2, seqlens_q=[6], seqlens_k=[40], rel_extent=17),
    dict(num_heads=3, num_kv_heads=3, seqlens_q=[1, 1, 2], seqlens_k=[1, 16, 33], head_dim=16),
]


@pytest.mark.parametrize("i", range(len(BRUTE_CASES)))
def test_c_oracle_equals_python_brute_force(i):
    c = _small(100 + i, **BRUTE_CASES[i])
    np.testing.assert_allclose(ref.forward(c), ref.brute_force(c), rtol=0, atol=1e-12)


@pytest.mark.parametrize("i", range(len(BRUTE_CASES)))
def test_c_oracle_lse_equals_python_brute_force(i):
    c = _small(100 + i, **BRUTE_CASES[i])
    _, lse = ref.forward(c, with_lse=True)
    _, want = ref.brute_force(c, with_lse=True)
    assert np.array_equal(np.isneginf(lse), np.isneginf(want))
    fin = np.isfinite(want)
    np.testing.assert_allclose(lse[fin], want[fin], rtol=0, atol=1e-12)


def test_tiny_mixed_c_oracle_equals_brute_force():
    c = tiny_mixed(0)
    np.testing.assert_allclose(ref.forward(c), ref.brute_force(c), rtol=0, atol=1e-12)


# --------------------------------------------------------------------- library routine

@pytest.mark.parametrize("causal,sq,sk,H,Hk", [(True, [4, 7], [10, 7], 4, 2), (False, [3, 5], [8, 5], 6, 3),
                                                (True, [1, 2], [33, 2], 8, 1)])
def test_zero_bias_is_plain_attention_sdpa(causal, sq, sk, H, Hk):
    c = _small(7, seqlens_q=sq, seqlens_k=sk, num_heads=H, num_kv_heads=Hk, causal=causal, rel_extent=5)
    c = c.with_(rel_logits=torch.zeros_like(c.rel_logits))
    got = ref.forward(c)
    cu = c.cu_seqlens_q.tolist()
    for b in range(len(sq)):
        qb = c.q[cu[b]:cu[b + 1]].double().transpose(0, 1).unsqueeze(0)      # (1,H,sq,D)
        kb = _kv_contig(c, b, "k").transpose(0, 1).unsqueeze(0)                # (1,Hk,sk,D)
        vb = _kv_contig(c, b, "v").transpose(0, 1).unsqueeze(0)
        mask = causal_lower_right(sq[b], sk[b]) if causal else None
        want = F.scaled_dot_product_attention(qb, kb, vb, attn_mask=mask, scale=c.softmax_scale,
                                              enable_gqa=True)[0].transpose(0, 1)
        np.testing.assert_allclose(got[cu[b]:cu[b + 1]], want.numpy(), rtol=0, atol=1e-12)


def test_bias_only_is_torch_softmax_weighting():
    """scale = 0: scores are the bias alone, so the output is torch.softmax of the
    bias row over the keys times V.  Fails if the bias were scaled too."""
    c = _small(8, seqlens_q=[1], seqlens_k=[6], rel_extent=6, softmax_scale=0.0, causal=True)
    got = ref.forward(c)
    v = _kv_contig(c, 0, "v")
    for h in range(4):
        # key j sits at distance 5 - j; all six keys are in [0, 6)
        bias = torch.stack([c.rel_logits[0, h, 5 - j].double() for j in range(6)])
        w = torch.softmax(bias, 0)
        want = (w[:, None] * v[:, h // 2, :]).sum(0)
        np.testing.assert_allclose(got[0, h], want.numpy(), rtol=0, atol=1e-12)


# --------------------------------------------------------------------- closed forms

def test_single_key_returns_v_exactly():
    c = _small(9, seqlens_q=[1, 1, 1], seqlens_k=[1, 1, 1], rel_extent=3)
    got = ref.forward(c)
    for b in range(3):
        v0 = _kv_contig(c, b, "v")[0]
        for h in range(4):
            assert np.array_equal(got[b, h], v0[h // 2].numpy())


@pytest.mark.parametrize("window", [(-1, -1), (3, 0), (0, 0)])
def test_zero_query_zero_bias_is_mean_of_allowed_values(window):
    c = _small(10, seqlens_q=[4], seqlens_k=[11], window=window, rel_extent=4)
    c = c.with_(q=torch.zeros_like(c.q), rel_logits=torch.zeros_like(c.rel_logits))
    got = ref.forward(c)
    v = _kv_contig(c, 0, "v")
    for i in range(4):
        pos = i + 7
        lo = 0 if window[0] < 0 else max(0, pos - window[0])
        want = v[lo:pos + 1].mean(0)
        for h in range(4):
            np.testing.assert_allclose(got[i, h], want[h // 2].numpy(), rtol=0, atol=1e-12)


@pytest.mark.parametrize("window", [(-1, -1), (3, 0), (0, 0)])
def test_zero_scores_give_lse_log_of_visible_key_count(window):
    """Every visible score is 0, so lse = ln(number of visible keys)."""
    c = _small(10, seqlens_q=[4], seqlens_k=[11], window=window, rel_extent=4)
    c = c.with_(q=torch.zeros_like(c.q), rel_logits=torch.zeros_like(c.rel_logits))
    _, lse = ref.forward(c, with_lse=True)
    for i in range(4):
        pos = i + 7
        lo = 0 if window[0] < 0 else max(0, pos - window[0])
        np.testing.assert_allclose(lse[i], math.log(pos + 1 - lo), rtol=0, atol=1e-12)


def test_rows_without_keys_are_zero():
    """sk < sq, bottom-right causal: rows 0..2 of a 5-row request over 2 keys
    see no key; rows 3 and 4 see keys {0} and {0,1}."""
    c = _small(11, seqlens_q=[5], seqlens_k=[2])
    c = c.with_(q=torch.zeros_like(c.q))
    got, lse = ref.forward(c, with_lse=True)
    v = _kv_contig(c, 0, "v")
    assert np.all(got[:3] == 0.0)
    assert np.all(np.isneginf(lse[:3]))
    for h in range(4):
        # q = 0: row 3 sees key 0 at distance 0, row 4 keys 0 and 1 at distances 1 and 0
        assert lse[3, h] == float(c.rel_logits[3, h, 0])
        b1, b0 = float(c.rel_logits[4, h, 1]), float(c.rel_logits[4, h, 0])
        assert abs(lse[4, h] - math.log(math.exp(b1) + math.exp(b0))) < 1e-12
    for h in range(4):
        assert np.array_equal(got[3, h], v[0, h // 2].numpy())
        # two keys with scores b(d=1), b(d=0) from the bias alone
        b1 = c.rel_logits[4, h, 1].double()
        b0 = c.rel_logits[4, h, 0].double()
        w = torch.softmax(torch.stack([b1, b0]), 0)
        want = w[0] * v[0, h // 2] + w[1] * v[1, h // 2]
        np.testing.assert_allclose(got[4, h], want.numpy(), rtol=0, atol=1e-12)


def test_out_of_band_bias_is_zero_not_clamped():
    """q = 0 and rel = c on [0, R): in-band keys weigh e^c, out-of-band keys 1.
    A clamping reading would give every allowed key e^c (a plain mean)."""
    cval = 2.0
    c = _small(12, seqlens_q=[2], seqlens_k=[9], rel_extent=3, causal=True)
    c = c.with_(q=torch.zeros_like(c.q), rel_logits=torch.full_like(c.rel_logits, cval))
    got = ref.forward(c)
    v = _kv_contig(c, 0, "v")
    for i in range(2):
        pos = i + 7
        w = torch.tensor([math.exp(cval) if 0 <= pos - j < 3 else 1.0 for j in range(pos + 1)],
                         dtype=torch.float64)
        for h in range(4):
            want = (w[:, None] * v[:pos + 1, h // 2]).sum(0) / w.sum()
            np.testing.assert_allclose(got[i, h], want.numpy(), rtol=0, atol=1e-12)


def test_one_hot_bias_selects_one_key_per_token_and_head():
    """+30 at a distinct distance d*(t,h) per row: output ~ V at key pos - d*.
    Two requests so the global token index of the bias row is exercised."""
    c = _small(13, seqlens_q=[3, 4], seqlens_k=[10, 12], rel_extent=8, num_heads=4, num_kv_heads=2)
    rel = torch.zeros_like(c.rel_logits)
    rng = np.random.default_rng(5)
    target = {}
    cu = c.cu_seqlens_q.tolist()
    sk = c.cache_seqlens.tolist()
    for b in range(2):
        for i in range(cu[b + 1] - cu[b]):
            t = cu[b] + i
            for h in range(4):
                dstar = int(rng.integers(0, 8))
                rel[t, h, dstar] = 30.0
                target[(t, h)] = (b, i + sk[b] - (cu[b + 1] - cu[b]) - dstar)
    c = c.with_(rel_logits=rel)
    got = ref.forward(c)
    for (t, h), (b, j) in target.items():
        v = _kv_contig(c, b, "v")
        np.testing.assert_allclose(got[t, h], v[j, h // 2].numpy(), rtol=0, atol=1e-6)


# --------------------------------------------------------------------- invariants

def test_page_relabelling_is_bit_invariant():
    c = _small(14, seqlens_q=[3, 2, 5], seqlens_k=[17, 8, 30], block_size=4, pool_blocks=20)
    NB = c.key_cache.shape[0]
    perm = torch.from_numpy(np.random.default_rng(3).permutation(NB))
    inv = torch.argsort(perm)
    # physical block p moves to slot inv[p]
    k2 = torch.empty_like(c.key_cache)
    v2 = torch.empty_like(c.value_cache)
    k2[inv] = c.key_cache
    v2[inv] = c.value_cache
    table2 = inv[c.block_table.long()].to(torch.int32)
    c2 = c.with_(key_cache=k2, value_cache=v2, block_table=table2)
    assert np.array_equal(ref.forward(c), ref.forward(c2))


def test_appended_zero_columns_change_nothing():
    c = _small(15, rel_extent=4)
    wide = torch.cat([c.rel_logits, torch.zeros(*c.rel_logits.shape[:2], 5, dtype=torch.bfloat16)], 2)
    c2 = c.with_(rel_logits=wide, rel_extent=9)
    assert np.array_equal(ref.forward(c), ref.forward(c2))


def test_unreachable_columns_change_nothing():
    # window left 2: distances above 2 never occur; causal sk == sq: distances >= sk never occur
    c = _small(16, window=(2, 0), rel_extent=6)
    rel = c.rel_logits.clone()
    rel[:, :, 3:] = 99.0
    assert np.array_equal(ref.forward(c), ref.forward(c.with_(rel_logits=rel)))
    c = _small(17, seqlens_q=[5], seqlens_k=[5], rel_extent=9)
    rel = c.rel_logits.clone()
    rel[:, :, 5:] = -77.0
    assert np.array_equal(ref.forward(c), ref.forward(c.with_(rel_logits=rel)))


def test_bias_shift_invariance_when_every_key_is_in_band():
    c = _small(18, seqlens_q=[3, 4], seqlens_k=[6, 9], rel_extent=9, causal=True)
    # quarter steps in [-8, 8] stay exact in bf16 after adding 3
    base = torch.round(c.rel_logits.float().clamp(-8, 8) * 4) / 4
    c = c.with_(rel_logits=base.to(torch.bfloat16))
    c2 = c.with_(rel_logits=(base + 3.0).to(torch.bfloat16))
    o1, l1 = ref.forward(c, with_lse=True)
    o2, l2 = ref.forward(c2, with_lse=True)
    np.testing.assert_allclose(o1, o2, rtol=0, atol=1e-12)
    # the shift moves every visible score, so the log-sum-exp moves by exactly 3
    np.testing.assert_allclose(l2, l1 + 3.0, rtol=0, atol=1e-12)


def test_rows_entry_equals_full_forward():
    c = _small(19, seqlens_q=[3, 0, 6], seqlens_k=[7, 3, 20], window=(5, 0))
    full = ref.forward(c)
    rng = np.random.default_rng(0)
    t = rng.integers(0, c.q.shape[0], 12)
    h = rng.integers(0, c.q.shape[1], 12)
    rows = ref.forward_rows(c, t, h)
    assert np.array_equal(rows, full[t, h])


def test_lse_matches_log_of_softmax_denominator():
    """lse = log sum_j exp(s_j) over allowed keys: a single key gives lse = s_0."""
    c = _small(20, seqlens_q=[1], seqlens_k=[1], rel_extent=2)
    _, lse = ref.forward(c, with_lse=True)
    k0 = _kv_contig(c, 0, "k")[0]
    for h in range(4):
        s0 = c.softmax_scale * float(c.q[0, h].double() @ k0[h // 2]) + float(c.rel_logits[0, h, 0])
        assert abs(lse[0, h] - s0) < 1e-12


def test_oracle_rejects_bad_block_ids():
    c = _small(21)
    bad = c.block_table.clone()
    bad[0, 0] = 10_000
    with pytest.raises(ValueError):
        ref.forward(c.with_(block_table=bad))


# --------------------------------------------------------------------- heuristic

def _golden(name):
    import os
    path = os.path.join(os.path.dirname(__file__), "golden", name)
    rows = []
    for line in open(path):
        line = line.split("#")[0].strip()
        if line:
            rows.append([int(x) for x in line.split()])
    return rows


def test_num_splits_matches_worked_values():
    for is_local, B, mq, H, Hk, kv, cap, want in _golden("num_splits_cases.txt"):
        got = ref.num_splits(is_local=bool(is_local), batch_size=B, max_query_len=mq, num_heads=H,
                             num_kv_heads=Hk, max_kv_len=kv, capability_major=cap)
        assert got == want, (is_local, B, mq, H, Hk, kv, cap)


def test_bucket_max_seqlen_q_matches_worked_values():
    for n, want in _golden("bucket_max_seqlen_q.txt"):
        assert ref.bucket_max_seqlen_q(n) == want


# --------------------------------------------------------------------- cache append

def _new_rows(c, seed):
    g = torch.Generator().manual_seed(seed)
    T, Hk, D = c.q.shape[0], c.key_cache.shape[2], c.key_cache.shape[3]
    k = torch.randn(T, Hk, D, generator=g).to(torch.bfloat16)
    v = torch.randn(T, Hk, D, generator=g).to(torch.bfloat16)
    return k, v


def test_cache_append_round_trip_through_block_table():
    """Reading the request's last sq keys back through the (permuted) block
    table returns the appended rows bit for bit; every other slot is unchanged."""
    c = _small(40, seqlens_q=[3, 0, 5], seqlens_k=[9, 4, 13])
    key, value = _new_rows(c, 1)
    kc, vc = ref.cache_append(c, key, value)
    c2 = c.with_(key_cache=kc, value_cache=vc)
    cu = c.cu_seqlens_q.tolist()
    written = torch.zeros(kc.shape[:2], dtype=torch.bool)
    for b in range(3):
        sq, sk = cu[b + 1] - cu[b], int(c.cache_seqlens[b])
        got_k = _kv_contig(c2, b, "k")[sk - sq:]
        got_v = _kv_contig(c2, b, "v")[sk - sq:]
        assert torch.equal(got_k, key[cu[b]:cu[b + 1]].double())
        assert torch.equal(got_v, value[cu[b]:cu[b + 1]].double())
        assert torch.equal(_kv_contig(c2, b, "k")[:sk - sq], _kv_contig(c, b, "k")[:sk - sq])
        for pos in range(sk - sq, sk):
            written[int(c.block_table[b, pos // 4]), pos % 4] = True
    assert torch.equal(kc[~written], c.key_cache[~written])
    assert torch.equal(vc[~written], c.value_cache[~written])


def test_cache_append_skips_tokens_without_a_slot():
    """sk < sq: the first sq - sk tokens have negative positions and write
    nothing; a request with an empty cache writes nothing at all (which tells
    skipping apart from clamping the position to 0)."""
    c = _small(41, seqlens_q=[5, 3], seqlens_k=[2, 0])
    key, value = _new_rows(c, 2)
    kc, vc = ref.cache_append(c, key, value)
    got = _kv_contig(c.with_(key_cache=kc), 0, "k")
    assert torch.equal(got, key[3:5].double())
    untouched = torch.ones(kc.shape[:2], dtype=torch.bool)
    untouched[int(c.block_table[0, 0]), 0:2] = False
    assert torch.equal(kc[untouched], c.key_cache[untouched])
    assert torch.equal(vc[untouched], c.value_cache[untouched])


def test_append_then_attend_equals_sdpa_over_prefix_and_new_rows():
    """Appended rows are the keys the attention aligns with the new tokens:
    with zero bias, attending over the cache equals SDPA over [prefix, new]
    with torch's lower-right causal mask."""
    c = _small(42, seqlens_q=[4, 6], seqlens_k=[11, 6], rel_extent=0, head_dim=16)
    key, value = _new_rows(c, 3)
    kc, vc = ref.cache_append(c, key, value)
    c2 = c.with_(key_cache=kc, value_cache=vc)
    out = ref.forward(c2)
    cu = c.cu_seqlens_q.tolist()
    G = c.q.shape[1] // c.key_cache.shape[2]
    for b in range(2):
        sq, sk = cu[b + 1] - cu[b], int(c.cache_seqlens[b])
        k_all = torch.cat([_kv_contig(c, b, "k")[:sk - sq], key[cu[b]:cu[b + 1]].double()])
        v_all = torch.cat([_kv_contig(c, b, "v")[:sk - sq], value[cu[b]:cu[b + 1]].double()])
        q = c.q[cu[b]:cu[b + 1]].double().transpose(0, 1)                 # (H, sq, D)
        k = k_all.transpose(0, 1).repeat_interleave(G, 0)                  # (H, sk, D)
        v = v_all.transpose(0, 1).repeat_interleave(G, 0)
        want = F.scaled_dot_product_attention(q, k, v, attn_mask=causal_lower_right(sq, sk),
                                              scale=float(np.float32(c.softmax_scale)))
        np.testing.assert_allclose(out[cu[b]:cu[b + 1]], want.transpose(0, 1).numpy(), rtol=0, atol=1e-12)


@pytest.mark.parametrize("i", [0, 2, 8])
def test_fp32_rel_logits_c_oracle_equals_brute_force(i):
    """fp32 rel_logits (values bf16 cannot hold) take the same definition."""
    c = _small(100 + i, **BRUTE_CASES[i])
    g = torch.Generator().manual_seed(i)
    rel = c.rel_logits.float() + 1e-3 * torch.randn(c.rel_logits.shape, generator=g)
    c = c.with_(rel_logits=rel)
    out, lse = ref.forward(c, with_lse=True)
    want, want_lse = ref.brute_force(c, with_lse=True)
    np.testing.assert_allclose(out, want, rtol=0, atol=1e-12)
    fin = np.isfinite(want_lse)
    np.testing.assert_allclose(lse[fin], want_lse[fin], rtol=0, atol=1e-12)
    # and the fp32 values are used as they are, not rounded to bf16
    c16 = c.with_(rel_logits=rel.to(torch.bfloat16))
    assert np.abs(ref.forward(c16) - out).max() > 1e-6
