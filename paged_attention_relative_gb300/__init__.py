"""Paged varlen attention with an additive relative-position bias, for GB300.

The compute path is the C-ABI library ``librel_attn.so`` (CUDA, sm_103a) built
from ``csrc/``; this package is a thin ctypes binding over it.
"""
