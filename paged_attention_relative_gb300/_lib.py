"""ctypes binding of ``librel_attn.so`` (include/rel_attn.h, include/rel_attn_profile.h).

Argument marshalling only: torch tensors become borrowed ``rel_attn_tensor``
descriptors (data pointer, dtype, shape, strides), the current torch stream
becomes the ``cudaStream_t``.  Every step of the computation runs in the
library's CUDA kernels; there is no fallback path.  If the library has not
been built, importing this module raises.
"""
from __future__ import annotations

import ctypes
import os

import torch

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "librel_attn.so")

REL_ATTN_BF16, REL_ATTN_F32, REL_ATTN_I32 = 0, 1, 2
STATUS = {0: "OK", 1: "INVALID_ARGUMENT", 2: "UNSUPPORTED", 3: "CUDA", 4: "OUT_OF_MEMORY", 5: "DEVICE_CHECK"}
KERNELS = {0: "none", 1: "decode", 2: "prefill", 3: "append", 4: "prefill_pair"}

# Every function the headers declare, with its ctypes signature.
EXPORTS = ("rel_attn_paged_varlen", "rel_attn_paged_varlen_lse", "rel_attn_paged_varlen_noalloc", "rel_attn_num_splits",
           "rel_attn_cache_append",
           "rel_attn_bucket_max_seqlen_q",
           "rel_attn_last_error", "rel_attn_last_launch", "rel_attn_set_kernel_events", "rel_attn_device_error",
           "rel_attn_check_wait_timeout")


class RelAttnTensor(ctypes.Structure):
    _fields_ = [("data", ctypes.c_void_p), ("dtype", ctypes.c_int32), ("ndim", ctypes.c_int32),
                ("shape", ctypes.c_int64 * 4), ("stride", ctypes.c_int64 * 4)]


class LaunchInfo(ctypes.Structure):
    _fields_ = [("kernel", ctypes.c_int32), ("num_splits", ctypes.c_int32), ("grid", ctypes.c_int32 * 3),
                ("block", ctypes.c_int32), ("smem_bytes", ctypes.c_int32), ("launches", ctypes.c_int32),
                ("workspace_bytes", ctypes.c_int64)]


class RelAttnError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"{STATUS.get(status, status)}: {message}")
        self.status = status


def _load() -> ctypes.CDLL:
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"{LIB_PATH} is missing: build it with "
                          "`python -c 'import __graft_entry__ as g; g.build()'`")
    lib = ctypes.CDLL(LIB_PATH)
    P = ctypes.POINTER(RelAttnTensor)
    i32, f32 = ctypes.c_int32, ctypes.c_float
    lib.rel_attn_paged_varlen.argtypes = [P, P, P, P, P, P, i32, f32, i32, i32, i32, i32, P, i32, P, ctypes.c_void_p]
    lib.rel_attn_paged_varlen.restype = ctypes.c_int
    lib.rel_attn_paged_varlen_lse.argtypes = [P, P, P, P, P, P, i32, f32, i32, i32, i32, i32, P, i32, P, P,
                                              ctypes.c_void_p]
    lib.rel_attn_paged_varlen_lse.restype = ctypes.c_int
    lib.rel_attn_paged_varlen_noalloc.argtypes = lib.rel_attn_paged_varlen.argtypes
    lib.rel_attn_paged_varlen_noalloc.restype = ctypes.c_int
    lib.rel_attn_cache_append.argtypes = [P, P, P, P, P, P, P, ctypes.c_void_p]
    lib.rel_attn_cache_append.restype = ctypes.c_int
    lib.rel_attn_num_splits.argtypes = [i32] * 6
    lib.rel_attn_num_splits.restype = i32
    lib.rel_attn_bucket_max_seqlen_q.argtypes = [i32]
    lib.rel_attn_bucket_max_seqlen_q.restype = i32
    lib.rel_attn_last_error.argtypes = []
    lib.rel_attn_last_error.restype = ctypes.c_char_p
    lib.rel_attn_last_launch.argtypes = [ctypes.POINTER(LaunchInfo)]
    lib.rel_attn_last_launch.restype = ctypes.c_int
    lib.rel_attn_set_kernel_events.argtypes = [ctypes.c_void_p, ctypes.c_void_p]
    lib.rel_attn_set_kernel_events.restype = ctypes.c_int
    lib.rel_attn_device_error.argtypes = [ctypes.POINTER(ctypes.c_int32)]
    lib.rel_attn_device_error.restype = ctypes.c_int
    lib.rel_attn_check_wait_timeout.argtypes = [i32, ctypes.c_void_p]
    lib.rel_attn_check_wait_timeout.restype = ctypes.c_int
    return lib


lib = _load()

_DT = {torch.bfloat16: REL_ATTN_BF16, torch.float32: REL_ATTN_F32, torch.int32: REL_ATTN_I32}


def describe(t: torch.Tensor | None) -> RelAttnTensor | None:
    """Borrowed descriptor of a tensor (None stays None)."""
    if t is None:
        return None
    if t.dim() > 4:
        raise ValueError("rank > 4")
    d = RelAttnTensor()
    d.data = t.data_ptr() if t.numel() > 0 else None
    d.dtype = _DT.get(t.dtype, -1)
    d.ndim = t.dim()
    for i in range(t.dim()):
        d.shape[i] = t.shape[i]
        d.stride[i] = t.stride(i)
    return d


def _ref(d):
    return ctypes.byref(d) if d is not None else None


def _check(status: int):
    if status != 0:
        raise RelAttnError(status, lib.rel_attn_last_error().decode())


def _stream_handle(stream, device):
    """A cudaStream_t as an int: torch's current stream when None."""
    if stream is None:
        return torch.cuda.current_stream(device).cuda_stream
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return stream


def _attn_args(q, key_cache, value_cache, block_table, cache_seqlens, cu_seqlens_q, max_seqlen_q, softmax_scale,
               causal, window_left, window_right, rel_extent, rel_logits, num_splits):
    """The leading arguments shared by the three attention entry points (the
    byref objects keep their descriptors alive for the call)."""
    descs = [describe(t) for t in (q, key_cache, value_cache, block_table, cache_seqlens, cu_seqlens_q)]
    rel = describe(rel_logits) if rel_extent > 0 else None
    return [*[_ref(d) for d in descs], int(max_seqlen_q), float(softmax_scale), int(bool(causal)),
            int(window_left), int(window_right), int(rel_extent), _ref(rel), int(num_splits)]


def rel_attn_paged_varlen(q, key_cache, value_cache, block_table, cache_seqlens, cu_seqlens_q, max_seqlen_q,
                          softmax_scale, causal, window_left, window_right, rel_extent, rel_logits, num_splits,
                          out=None, stream=None):
    """Paged varlen attention with relative bias; see include/rel_attn.h.

    Same names and order as the C entry point.  ``out`` is allocated like
    ``q`` when None; ``stream`` defaults to torch's current stream.
    """
    if out is None:
        out = torch.empty_like(q)
    args = _attn_args(q, key_cache, value_cache, block_table, cache_seqlens, cu_seqlens_q, max_seqlen_q,
                      softmax_scale, causal, window_left, window_right, rel_extent, rel_logits, num_splits)
    od = describe(out)
    _check(lib.rel_attn_paged_varlen(*args, _ref(od), ctypes.c_void_p(_stream_handle(stream, q.device))))
    return out


def rel_attn_paged_varlen_lse(q, key_cache, value_cache, block_table, cache_seqlens, cu_seqlens_q, max_seqlen_q,
                              softmax_scale, causal, window_left, window_right, rel_extent, rel_logits, num_splits,
                              out=None, softmax_lse=None, stream=None):
    """The forward that also writes each row's natural-log sum-exp; see include/rel_attn.h.

    Returns ``(out, softmax_lse)``.  ``softmax_lse`` is allocated as a
    contiguous ``(T, H)`` fp32 tensor when None; any ``(T, H)`` fp32 view
    works (``lse_ht.t()`` for an ``(H, T)`` buffer).
    """
    if out is None:
        out = torch.empty_like(q)
    if softmax_lse is None:
        softmax_lse = torch.empty(q.shape[0], q.shape[1], dtype=torch.float32, device=q.device)
    args = _attn_args(q, key_cache, value_cache, block_table, cache_seqlens, cu_seqlens_q, max_seqlen_q,
                      softmax_scale, causal, window_left, window_right, rel_extent, rel_logits, num_splits)
    od, ld = describe(out), describe(softmax_lse)
    _check(lib.rel_attn_paged_varlen_lse(*args, _ref(od), _ref(ld),
                                         ctypes.c_void_p(_stream_handle(stream, q.device))))
    return out, softmax_lse


def rel_attn_paged_varlen_noalloc(q, key_cache, value_cache, block_table, cache_seqlens, cu_seqlens_q,
                                  max_seqlen_q, softmax_scale, causal, window_left, window_right, rel_extent,
                                  rel_logits, num_splits, out, stream=None):
    """The allocation-free decode entry point; ``out`` must be provided."""
    args = _attn_args(q, key_cache, value_cache, block_table, cache_seqlens, cu_seqlens_q, max_seqlen_q,
                      softmax_scale, causal, window_left, window_right, rel_extent, rel_logits, num_splits)
    od = describe(out)
    _check(lib.rel_attn_paged_varlen_noalloc(*args, _ref(od), ctypes.c_void_p(_stream_handle(stream, q.device))))
    return out


def rel_attn_cache_append(key, value, key_cache, value_cache, block_table, cache_seqlens, cu_seqlens_q,
                          stream=None):
    """Write the new tokens' key/value rows into the paged caches; see include/rel_attn.h."""
    d = [describe(t) for t in (key, value, key_cache, value_cache, block_table, cache_seqlens, cu_seqlens_q)]
    _check(lib.rel_attn_cache_append(*[_ref(x) for x in d], ctypes.c_void_p(_stream_handle(stream, key.device))))
    return key_cache, value_cache


def rel_attn_num_splits(is_local, batch_size, max_query_len, num_heads, num_kv_heads, max_kv_len) -> int:
    """Split-KV cap (include/rel_attn.h); raises on invalid sizes."""
    r = lib.rel_attn_num_splits(int(bool(is_local)), int(batch_size), int(max_query_len), int(num_heads),
                                int(num_kv_heads), int(max_kv_len))
    if r < 0:
        _check(-r)
    return r


def rel_attn_bucket_max_seqlen_q(max_seqlen_q) -> int:
    """Query-length bucket for graph-captured calls (include/rel_attn.h); raises on invalid input."""
    r = lib.rel_attn_bucket_max_seqlen_q(int(max_seqlen_q))
    if r < 0:
        _check(-r)
    return r


def last_launch() -> dict:
    info = LaunchInfo()
    _check(lib.rel_attn_last_launch(ctypes.byref(info)))
    return dict(kernel=KERNELS.get(info.kernel, info.kernel), num_splits=info.num_splits, grid=tuple(info.grid),
                block=info.block, smem_bytes=info.smem_bytes, launches=info.launches,
                workspace_bytes=info.workspace_bytes)


def set_kernel_events(begin: torch.cuda.Event | None, end: torch.cuda.Event | None):
    """Record ``begin``/``end`` around the main kernel of following calls.

    torch creates an event's CUDA handle lazily: record each event once before
    passing it here."""
    b = ctypes.c_void_p(begin.cuda_event) if begin is not None else None
    e = ctypes.c_void_p(end.cuda_event) if end is not None else None
    _check(lib.rel_attn_set_kernel_events(b, e))


def device_error() -> int:
    code = ctypes.c_int32(0)
    _check(lib.rel_attn_device_error(ctypes.byref(code)))
    return code.value


SITE_SELF_TEST = 99  # REL_ATTN_SITE_SELF_TEST


def check_wait_timeout(timeout_ms: int, stream=None):
    """Launch the bounded-wait self-test (include/rel_attn_profile.h)."""
    _check(lib.rel_attn_check_wait_timeout(int(timeout_ms), ctypes.c_void_p(_stream_handle(stream, None))))
