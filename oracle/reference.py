"""Python face of the oracle: the C definition through ctypes, a pure-Python
brute force for tiny inputs, and the split-count heuristic restated.

TEST INFRASTRUCTURE ONLY (tests, smoke check, CPU-baseline leg of the
benchmark).  The product library never imports this module.

Arguments are duck-typed: any object with the attributes of a workload case
(q, key_cache, value_cache, block_table, cache_seqlens, cu_seqlens_q,
softmax_scale, causal, window_left, window_right, rel_extent, rel_logits) as
CPU torch tensors / Python scalars.
"""
from __future__ import annotations

import ctypes
import math
import os

import numpy as np
import torch

from . import build as _build

_lib = None


def _load():
    global _lib
    if _lib is None:
        path = _build.build()
        lib = ctypes.CDLL(path)
        P = ctypes.c_void_p
        I64 = ctypes.c_int64
        I = ctypes.c_int
        D = ctypes.c_double
        common = [P, P, P, P, I64, P, P, I64, I64, I64, I64, I64, I64, I64, D, I, I, I, I64, P, I]
        lib.rel_attn_oracle_forward.argtypes = common + [P, P, I]
        lib.rel_attn_oracle_forward.restype = I
        lib.rel_attn_oracle_rows.argtypes = common + [I64, P, P, P, I]
        lib.rel_attn_oracle_rows.restype = I
        _lib = lib
    return _lib


def _bits(t: torch.Tensor) -> np.ndarray:
    assert t.dtype == torch.bfloat16
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def _i32(t: torch.Tensor) -> np.ndarray:
    return np.ascontiguousarray(t.detach().cpu().numpy().astype(np.int32))


def _common_args(c):
    q = _bits(c.q)
    kc = _bits(c.key_cache)
    vc = _bits(c.value_cache)
    bt = _i32(c.block_table)
    sk = _i32(c.cache_seqlens)
    cu = _i32(c.cu_seqlens_q)
    T, H, D = c.q.shape
    NB, BS, Hk, _ = c.key_cache.shape
    B = bt.shape[0]
    R = int(c.rel_extent)
    rel_f32 = R > 0 and c.rel_logits.dtype == torch.float32
    if R > 0:
        rel = (np.ascontiguousarray(c.rel_logits.detach().cpu().numpy()) if rel_f32 else _bits(c.rel_logits))
        assert rel.size == T * H * R
    else:
        rel = np.zeros(1, dtype=np.uint16)
    keep = (q, kc, vc, bt, sk, cu, rel)
    # the library takes softmax_scale as a float32; evaluate with that value
    scale = float(np.float32(c.softmax_scale))
    args = [q.ctypes.data, kc.ctypes.data, vc.ctypes.data, bt.ctypes.data, bt.shape[1],
            sk.ctypes.data, cu.ctypes.data, B, T, H, Hk, D, NB, BS, scale,
            int(bool(c.causal)), int(c.window_left), int(c.window_right), R, rel.ctypes.data, int(rel_f32)]
    return args, keep


def default_threads() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:  # pragma: no cover
        return os.cpu_count() or 1


def forward(c, num_threads: int | None = None, with_lse: bool = False):
    """out (T,H,D) fp64 [and lse (T,H) natural log] by the plain definition."""
    lib = _load()
    args, keep = _common_args(c)
    T, H, D = c.q.shape
    out = np.zeros((T, H, D), dtype=np.float64)
    lse = np.zeros((T, H), dtype=np.float64) if with_lse else None
    rc = lib.rel_attn_oracle_forward(*args, out.ctypes.data,
                                     lse.ctypes.data if with_lse else None,
                                     int(num_threads or default_threads()))
    if rc != 0:
        raise ValueError(f"oracle rejected the inputs (code {rc})")
    return (out, lse) if with_lse else out


def forward_rows(c, rows_t, rows_h, num_threads: int | None = None) -> np.ndarray:
    """out[t_k, h_k, :] for each listed row, fp64, shape (n, D)."""
    lib = _load()
    args, keep = _common_args(c)
    rt = np.ascontiguousarray(np.asarray(rows_t, dtype=np.int64))
    rh = np.ascontiguousarray(np.asarray(rows_h, dtype=np.int64))
    D = c.q.shape[2]
    out = np.zeros((rt.size, D), dtype=np.float64)
    rc = lib.rel_attn_oracle_rows(*args, rt.size, rt.ctypes.data, rh.ctypes.data,
                                  out.ctypes.data, int(num_threads or default_threads()))
    if rc != 0:
        raise ValueError(f"oracle rejected the inputs (code {rc})")
    return out


def brute_force(c, with_lse: bool = False):
    """Pure-Python loops over every (token, head, key, dim); tiny inputs only.

    Written independently of the C file: per output row it walks the request's
    keys, builds the score list with the bias rule of score_mod_rel_bias
    (distance, zero outside [0, R)), and takes the softmax-weighted mean of V.
    With ``with_lse`` it also returns log(sum exp(score)) per (token, head),
    -inf where no key is visible.
    """
    q = c.q.double().tolist()
    kc = c.key_cache.double().tolist()
    vc = c.value_cache.double().tolist()
    rel = c.rel_logits.double().tolist() if c.rel_extent > 0 else None
    table = c.block_table.tolist()
    seqk = c.cache_seqlens.tolist()
    cu = c.cu_seqlens_q.tolist()
    T, H, D = c.q.shape
    Hk = c.key_cache.shape[2]
    BS = c.key_cache.shape[1]
    group = H // Hk
    scale = float(np.float32(c.softmax_scale))
    wl, wr = c.window_left, c.window_right
    out = [[[0.0] * D for _ in range(H)] for _ in range(T)]
    lse = [[-math.inf] * H for _ in range(T)]
    for b in range(len(seqk)):
        n_q = cu[b + 1] - cu[b]
        n_k = seqk[b]
        for i in range(n_q):
            t = cu[b] + i
            pos = i + n_k - n_q          # key position of this query row
            for h in range(H):
                kvh = h // group
                scores, values = [], []
                for j in range(n_k):
                    if c.causal and j > pos:
                        continue
                    if wl >= 0 and j < pos - wl:
                        continue
                    if wr >= 0 and j > pos + wr:
                        continue
                    page, slot = table[b][j // BS], j % BS
                    kvec = kc[page][slot][kvh]
                    dot = sum(q[t][h][e] * kvec[e] for e in range(D))
                    dist = pos - j
                    bias = rel[t][h][dist] if (rel is not None and 0 <= dist < c.rel_extent) else 0.0
                    scores.append(scale * dot + bias)
                    values.append(vc[page][slot][kvh])
                if not scores:
                    continue
                top = max(scores)
                w = [math.exp(s - top) for s in scores]
                tot = sum(w)
                out[t][h] = [sum(w[n] * values[n][e] for n in range(len(w))) / tot for e in range(D)]
                lse[t][h] = top + math.log(tot)
    o = np.array(out, dtype=np.float64).reshape(T, H, D)
    return (o, np.array(lse, dtype=np.float64).reshape(T, H)) if with_lse else o


def cache_append(c, key: torch.Tensor, value: torch.Tensor):
    """New (key_cache, value_cache) after writing the new tokens' rows.

    Token i of request b (row t = cu_seqlens_q[b] + i) is the key at logical
    position pos = cache_seqlens[b] - sq_b + i: the bottom-right position the
    attention of inkling_fa4_rel_attention (vLLM API docs) gives query row i,
    so the new tokens are the last sq_b keys of the request.  Its row goes to
    slot pos % BS of physical block block_table[b, pos // BS] for every kv
    head; tokens with pos < 0 have no slot and are skipped.  Plain loops over
    requests and tokens; the inputs are not modified.
    """
    kc = c.key_cache.detach().cpu().clone()
    vc = c.value_cache.detach().cpu().clone()
    key = key.detach().cpu()
    value = value.detach().cpu()
    table = c.block_table.tolist()
    seqk = c.cache_seqlens.tolist()
    cu = c.cu_seqlens_q.tolist()
    BS = kc.shape[1]
    for b in range(len(seqk)):
        n_new = cu[b + 1] - cu[b]
        for i in range(n_new):
            pos = seqk[b] - n_new + i
            if pos < 0:
                continue
            blk, slot = table[b][pos // BS], pos % BS
            kc[blk, slot] = key[cu[b] + i]
            vc[blk, slot] = value[cu[b] + i]
    return kc, vc


# ---------------------------------------------------------------------------
# Split-count heuristic and scheduling-bound bucketing, restated from the vLLM
# API docs for vllm.models.inkling.nvidia.ops.fa4_rel_attention
# (inkling_fa4_num_splits and bucket_max_seqlen_q).
# ---------------------------------------------------------------------------

def num_splits(*, is_local: bool, batch_size: int, max_query_len: int, num_heads: int,
               num_kv_heads: int, max_kv_len: int, capability_major: int | None = 10) -> int:
    """Split-KV cap for relative-bias attention.

    Hopper (capability major 9) and local (windowed) attention get 1.  Otherwise
    the GQA-packed query rows are cut into 256-row tiles; the base CTA count is
    batch x kv heads x q tiles; the target CTA count is 256 for a single tile at
    batch 1, 128 for a single tile, else 64; batch-1 single-tile calls get a cap
    that depends on the kv-head count and the KV length; the result is the
    target/base ratio bounded by that cap and by the number of 128-key blocks,
    and never below 1.
    """
    if capability_major == 9:
        return 1
    if is_local:
        return 1
    rows = max_query_len * (num_heads // num_kv_heads)
    tiles = -(-rows // 256)
    base = batch_size * num_kv_heads * tiles
    single_b1 = tiles == 1 and batch_size == 1
    if single_b1:
        target = 256
    elif tiles == 1:
        target = 128
    else:
        target = 64
    cap = 128
    if single_b1:
        if num_kv_heads == 8:
            cap = 16
        elif num_kv_heads == 4 or max_kv_len <= 8192:
            cap = 32
        elif max_kv_len <= 65536:
            cap = 64
        else:
            cap = 128
    kv_blocks = -(-max_kv_len // 128)
    return max(1, min(target // base, cap, kv_blocks))


def bucket_max_seqlen_q(max_seqlen_q: int) -> int:
    """Smallest power of two >= max_seqlen_q (1 for 0 and 1)."""
    p = 1
    while p < max_seqlen_q:
        p *= 2
    return p
