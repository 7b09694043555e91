"""Paged varlen attention with an additive relative-position bias, for GB300.

The compute path is the C-ABI library ``librel_attn.so`` (CUDA, sm_103a) built
in-tree from ``csrc/`` by ``build.py``; ``_lib`` is a thin ctypes binding with
the same entry-point names.  Importing the public functions loads the library
and raises if it has not been built: there is no CPU fallback.
"""
from __future__ import annotations


def __getattr__(name):
    if name in ("rel_attn_paged_varlen", "rel_attn_paged_varlen_lse", "rel_attn_paged_varlen_noalloc", "rel_attn_cache_append", "rel_attn_num_splits",
                "rel_attn_bucket_max_seqlen_q", "last_launch", "set_kernel_events", "device_error", "RelAttnError",
                "describe", "check_wait_timeout", "SITE_SELF_TEST"):
        from . import _lib
        return getattr(_lib, name)
    raise AttributeError(name)


__all__ = ["rel_attn_paged_varlen", "rel_attn_paged_varlen_lse", "rel_attn_paged_varlen_noalloc", "rel_attn_cache_append", "rel_attn_num_splits",
           "rel_attn_bucket_max_seqlen_q", "last_launch", "set_kernel_events", "device_error", "RelAttnError"]
