"""Seeded synthetic inputs for paged varlen relative-bias attention.

This module only draws numbers and lays them out (lengths, a shuffled page pool,
a block table, bf16 tensors).  It holds none of the attention arithmetic, so the
CUDA path and the fp64 oracle can both be fed from it without sharing any of the
method's code.

Random streams come from numpy's PCG64 seeded through ``SeedSequence`` so that
the same seed gives the same inputs on x86_64 and aarch64 hosts.  Values are
drawn in float32 and rounded to bf16 (round-to-nearest-even) by torch.

Shapes follow the vLLM API docs for ``inkling_fa4_rel_attention`` (its
docstring): ``q`` is ``(num_tokens, num_heads, head_dim)``, the caches are
``(num_blocks, block_size, num_kv_heads, head_dim)``, ``rel_logits`` is
``(num_tokens, num_heads, rel_extent)``; ``block_table`` is the per-request
page table and ``cache_seqlens`` the per-request KV length (``seqused_k``).
"""
from __future__ import annotations

import math
from concurrent.futures import ThreadPoolExecutor
from dataclasses import dataclass, field, replace

import numpy as np
import torch

_CHUNK = 1 << 24

# Stream ids: one independent random stream per drawn quantity, so that the
# draws for one tensor never depend on the size of another.
_S_LENGTHS, _S_PERM, _S_Q, _S_K, _S_V, _S_REL = range(6)


def _rng(seed: int, stream: int, chunk: int = 0) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence([seed, stream, chunk])))


def _normal_bf16(seed: int, stream: int, shape, std: float = 1.0) -> torch.Tensor:
    """bf16 tensor of N(0, std^2) draws; chunked so large tensors fill in parallel."""
    n = int(np.prod(shape)) if len(shape) else 1
    out = torch.empty(n, dtype=torch.bfloat16)
    nchunks = max(1, (n + _CHUNK - 1) // _CHUNK)

    def fill(c):
        lo, hi = c * _CHUNK, min(n, (c + 1) * _CHUNK)
        x = _rng(seed, stream, c).standard_normal(hi - lo, dtype=np.float32)
        if std != 1.0:
            x *= np.float32(std)
        out[lo:hi] = torch.from_numpy(x).to(torch.bfloat16)

    if nchunks == 1:
        fill(0)
    else:
        with ThreadPoolExecutor(max_workers=min(8, nchunks)) as ex:
            list(ex.map(fill, range(nchunks)))
    return out.view(*shape)


@dataclass
class Case:
    """One call's worth of inputs (CPU tensors) plus its scalar arguments."""
    q: torch.Tensor              # (T, H, D) bf16
    key_cache: torch.Tensor      # (NB, BS, Hk, D) bf16
    value_cache: torch.Tensor    # (NB, BS, Hk, D) bf16
    block_table: torch.Tensor    # (B, MB) int32
    cache_seqlens: torch.Tensor  # (B,) int32
    cu_seqlens_q: torch.Tensor   # (B+1,) int32
    max_seqlen_q: int
    softmax_scale: float
    causal: bool
    window_left: int
    window_right: int
    rel_extent: int
    rel_logits: torch.Tensor     # (T, H, R) bf16
    num_splits: int
    name: str = ""
    meta: dict = field(default_factory=dict)

    @property
    def seqlens_q(self):
        cu = self.cu_seqlens_q.tolist()
        return [cu[i + 1] - cu[i] for i in range(len(cu) - 1)]

    @property
    def dims(self):
        T, H, D = self.q.shape
        NB, BS, Hk, _ = self.key_cache.shape
        return dict(B=self.block_table.shape[0], T=T, H=H, Hk=Hk, D=D, NB=NB, BS=BS,
                    MB=self.block_table.shape[1], R=self.rel_extent)

    def with_(self, **kw) -> "Case":
        return replace(self, **kw)


def make_case(*, seed: int, seqlens_q, seqlens_k, num_heads: int, num_kv_heads: int,
              head_dim: int, block_size: int = 16, rel_extent: int = 16,
              causal: bool = True, window=(-1, -1), softmax_scale: float | None = None,
              num_splits: int = 1, rel_std: float = 1.0, pool_blocks: int | None = None,
              extra_table_cols: int = 0, name: str = "") -> Case:
    """Build a case from explicit per-request lengths.

    The page pool holds ``sum_b ceil(sk_b / block_size)`` blocks (or
    ``pool_blocks`` if larger); a random permutation of the pool is dealt out to
    the requests in order, and the unused tail of each block-table row is 0.
    Draw order: block permutation, q, K, V, rel_logits.
    """
    sq = [int(x) for x in seqlens_q]
    sk = [int(x) for x in seqlens_k]
    assert len(sq) == len(sk)
    B = len(sq)
    T = sum(sq)
    H, Hk, D, BS, R = num_heads, num_kv_heads, head_dim, block_size, rel_extent
    nblk = [(k + BS - 1) // BS for k in sk]
    need = sum(nblk)
    NB = max(need, pool_blocks or 0, 1)
    MB = max(max(nblk) if nblk else 0, 1) + extra_table_cols
    perm = _rng(seed, _S_PERM).permutation(NB).astype(np.int32)
    table = np.zeros((B, MB), dtype=np.int32)
    pos = 0
    for b in range(B):
        table[b, :nblk[b]] = perm[pos:pos + nblk[b]]
        pos += nblk[b]
    cu = np.zeros(B + 1, dtype=np.int32)
    cu[1:] = np.cumsum(sq)
    q = _normal_bf16(seed, _S_Q, (T, H, D))
    k = _normal_bf16(seed, _S_K, (NB, BS, Hk, D))
    v = _normal_bf16(seed, _S_V, (NB, BS, Hk, D))
    rel = _normal_bf16(seed, _S_REL, (T, H, R), std=rel_std)
    if softmax_scale is None:
        softmax_scale = 1.0 / math.sqrt(D)
    return Case(q=q, key_cache=k, value_cache=v, block_table=torch.from_numpy(table),
                cache_seqlens=torch.tensor(sk, dtype=torch.int32),
                cu_seqlens_q=torch.from_numpy(cu), max_seqlen_q=max(sq) if sq else 0,
                softmax_scale=float(np.float32(softmax_scale)), causal=bool(causal),
                window_left=int(window[0]), window_right=int(window[1]), rel_extent=R,
                rel_logits=rel, num_splits=int(num_splits), name=name,
                meta=dict(seed=seed, pool_blocks=NB))


# ---------------------------------------------------------------------------
# The five named workloads.  Each is described by what it is and its sizes.
# ---------------------------------------------------------------------------

def tiny_mixed(seed: int = 0) -> Case:
    """2 requests, q lens [5,3], KV lens [37,20], 4/2 heads, head_dim 64,
    block_size 16, rel_extent 16, a permuted pool of 8 blocks, causal."""
    return make_case(seed=seed, seqlens_q=[5, 3], seqlens_k=[37, 20], num_heads=4,
                     num_kv_heads=2, head_dim=64, block_size=16, rel_extent=16,
                     causal=True, pool_blocks=8, num_splits=1, name="tiny_mixed")


def long_decode(seed: int = 0, num_splits: int = 16, kv_len: int = 131072) -> Case:
    """Batch-1 decode over 131072 cached tokens, 32/8 heads, head_dim 128,
    rel_extent 1024, shuffled blocks, causal."""
    return make_case(seed=seed, seqlens_q=[1], seqlens_k=[kv_len], num_heads=32,
                     num_kv_heads=8, head_dim=128, block_size=16, rel_extent=1024,
                     causal=True, num_splits=num_splits, name="long_decode")


def batched_decode(seed: int = 0, num_splits: int | None = None, batch: int = 64) -> Case:
    """64 decode requests with KV lens uniform in [1024, 8192], 64/4 heads,
    head_dim 128, rel_extent 512, non-contiguous pages, causal.  The split
    count defaults to the caller-provided heuristic value (1 here)."""
    sk = _rng(seed, _S_LENGTHS).integers(1024, 8192, size=batch, endpoint=True)
    return make_case(seed=seed, seqlens_q=[1] * batch, seqlens_k=sk.tolist(), num_heads=64,
                     num_kv_heads=4, head_dim=128, block_size=16, rel_extent=512,
                     causal=True, num_splits=1 if num_splits is None else num_splits,
                     name="batched_decode")


def chunked_prefill(seed: int = 0, batch: int = 4, q_len: int = 4096, prefix: int = 4096) -> Case:
    """4 requests each appending 4096 query tokens to a 4096-token prefix
    (seqlen_k 8192), 32/8 heads, head_dim 128, rel_extent 2048,
    rel_logits ~ N(0, 0.5^2), causal, one split."""
    return make_case(seed=seed, seqlens_q=[q_len] * batch, seqlens_k=[prefix + q_len] * batch,
                     num_heads=32, num_kv_heads=8, head_dim=128, block_size=16,
                     rel_extent=2048, causal=True, rel_std=0.5, num_splits=1,
                     name="chunked_prefill")


def chunked_prefill_d256(seed: int = 0, batch: int = 4, q_len: int = 4096, prefix: int = 4096) -> Case:
    """The chunked-prefill shape at head_dim 256 (the CTA-pair prefill
    kernel's size): 4 requests of 4096 query tokens on a 4096-token prefix,
    32/8 heads, rel_extent 2048, rel_logits ~ N(0, 0.5^2), causal, one split."""
    return make_case(seed=seed, seqlens_q=[q_len] * batch, seqlens_k=[prefix + q_len] * batch,
                     num_heads=32, num_kv_heads=8, head_dim=256, block_size=16,
                     rel_extent=2048, causal=True, rel_std=0.5, num_splits=1,
                     name="chunked_prefill_d256")


def mixed_window(seed: int = 0, batch: int = 32) -> Case:
    """32 requests, q lens log-uniform in [1, 2048], KV = prefix U[0, 32768] +
    q len, 32/8 heads, head_dim 128, window (4096, 0), rel_extent 512, causal."""
    r = _rng(seed, _S_LENGTHS)
    sq = np.clip(np.floor(np.exp(r.uniform(0.0, math.log(2049.0), size=batch))), 1, 2048).astype(int)
    prefix = r.integers(0, 32768, size=batch, endpoint=True)
    sk = prefix + sq
    return make_case(seed=seed, seqlens_q=sq.tolist(), seqlens_k=sk.tolist(), num_heads=32,
                     num_kv_heads=8, head_dim=128, block_size=16, rel_extent=512,
                     causal=True, window=(4096, 0), num_splits=1, name="mixed_window")


WORKLOADS = {
    "tiny_mixed": tiny_mixed,
    "long_decode": long_decode,
    "batched_decode": batched_decode,
    "chunked_prefill": chunked_prefill,
    "chunked_prefill_d256": chunked_prefill_d256,
    "mixed_window": mixed_window,
}
