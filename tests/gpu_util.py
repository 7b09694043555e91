"""Shared helpers of the GPU parity tests: move a case to the device, call
the library through the C ABI, compare with the fp64 oracle."""
import numpy as np
import torch

TOL_MAX = 2e-2    # max-abs error bound vs the fp64 oracle (bf16 output)
TOL_MEAN = 2e-3   # mean-abs error bound
TOL_SPLIT = 1e-3  # split vs one-split bound on the bf16 outputs

FIELDS = ("q", "key_cache", "value_cache", "block_table", "cache_seqlens", "cu_seqlens_q", "rel_logits")


def expected_prefill_kernel(c):
    """The prefill kernel the library picks for a case above 64 packed rows:
    the one-CTA kernel, or the CTA-pair kernel when REL_ATTN_PREFILL_PAIR=1
    asks for it on head_dim 128 with TMA-staged bf16 rel_logits (R a multiple
    of 8) or no bias."""
    import os
    D, R = c.q.shape[2], c.rel_extent
    staged = R == 0 or (c.rel_logits.dtype == torch.bfloat16 and R % 8 == 0)
    if D == 128 and staged and os.environ.get("REL_ATTN_PREFILL_PAIR", "") == "1":
        return "prefill_pair"
    return "prefill"


def to_dev(c, dev="cuda"):
    return {k: getattr(c, k).to(dev) for k in FIELDS}


def run(c, g=None, num_splits=None, out=None, **over):
    import paged_attention_relative_gb300 as pa
    g = g or to_dev(c)
    args = dict(max_seqlen_q=c.max_seqlen_q, softmax_scale=c.softmax_scale, causal=c.causal,
                window_left=c.window_left, window_right=c.window_right, rel_extent=c.rel_extent,
                num_splits=c.num_splits if num_splits is None else num_splits)
    args.update(over)
    out = pa.rel_attn_paged_varlen(g["q"], g["key_cache"], g["value_cache"], g["block_table"],
                                   g["cache_seqlens"], g["cu_seqlens_q"], args["max_seqlen_q"],
                                   args["softmax_scale"], args["causal"], args["window_left"],
                                   args["window_right"], args["rel_extent"],
                                   g["rel_logits"] if args["rel_extent"] > 0 else None, args["num_splits"],
                                   out=out)
    torch.cuda.synchronize()
    return out


def errors(got, want):
    got = got.float().cpu().numpy().astype(np.float64) if isinstance(got, torch.Tensor) else got
    e = np.abs(got - want)
    return float(e.max()) if e.size else 0.0, float(e.mean()) if e.size else 0.0


def assert_close(got, want, tol_max=TOL_MAX, tol_mean=TOL_MEAN, what=""):
    mx, mn = errors(got, want)
    assert np.isfinite(mx), f"{what}: non-finite output"
    assert mx <= tol_max and mn <= tol_mean, f"{what}: max-abs {mx:.3e} (<= {tol_max}), mean-abs {mn:.3e} (<= {tol_mean})"
    return mx, mn


def assert_no_device_error():
    import paged_attention_relative_gb300 as pa
    assert pa.device_error() == 0


def assert_split_matches_single(c, g, splits):
    """Split-KV + combine vs one split: within TOL_SPLIT on fp32 outputs (before
    the final bf16 rounding); on bf16 outputs within TOL_SPLIT or one bf16 ulp
    of the larger magnitude, since a correctly rounded pair of fp32 values that
    differ by less than TOL_SPLIT can still round one ulp apart."""
    a32 = torch.empty(c.q.shape, dtype=torch.float32, device="cuda")
    b32 = torch.empty_like(a32)
    run(c, g, num_splits=splits, out=a32)
    run(c, g, num_splits=1, out=b32)
    d32 = (a32 - b32).abs().max().item()
    assert d32 <= TOL_SPLIT, f"fp32 split vs single {d32:.3e}"
    a = run(c, g, num_splits=splits).float()
    b = run(c, g, num_splits=1).float()
    mag = torch.maximum(a.abs(), b.abs())
    ulp = torch.pow(2.0, torch.floor(torch.log2(mag.clamp_min(1e-30))) - 7)
    bad = ((a - b).abs() > torch.maximum(torch.full_like(ulp, TOL_SPLIT), ulp)).sum().item()
    assert bad == 0, f"{bad} bf16 outputs differ by more than max(TOL_SPLIT, 1 ulp)"
    return d32
