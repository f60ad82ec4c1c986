"""GB300 (sm_103a) exact attention forward — thin Python binding over libfa.so.

Every function here only marshals arguments into the C ABI declared in
``include/fa.h``; all of the computation runs in the library's CUDA kernel.
PyTorch is used for device memory and streams only.  There is no fallback:
if ``libfa.so`` has not been built, every call raises :class:`LibraryMissing`.

Functions with the C names (``fa_fwd``, ``fa_get_device_error``, ...) take
tensors or raw integer addresses.  :func:`attention_forward` is a convenience
wrapper that allocates O and LSE with PyTorch and checks the status.
"""
from __future__ import annotations

import ctypes
import math
import os
import threading

__all__ = [
    "FA_OK", "FA_ERR_INVALID_ARG", "FA_ERR_UNSUPPORTED", "FA_ERR_CUDA", "FA_ERR_TIMEOUT",
    "FA_ERR_BAD_SEQLENS", "FA_ERR_SCRATCH_LIMIT", "FA_DTYPE_FP16", "FA_DTYPE_BF16",
    "LibraryMissing", "FaError",
    "library_path", "load_library", "fa_fwd", "fa_fwd_ex", "fa_fwd_split", "fa_split_plan",
    "fa_fwd_split_noalloc", "fa_noalloc_scratch_bytes", "fa_fwd_kvcache", "attention_kvcache", "fa_kvcache_plan",
    "fa_get_device_error", "fa_debug_wait_timeout",
    "fa_debug_trace_read", "fa_shutdown", "fa_bwd", "fa_bwd_workspace_bytes",
    "fa_status_string", "fa_version", "attention_forward", "attention_backward",
    "EXPORTED_SYMBOLS",
]

FA_OK = 0
FA_ERR_INVALID_ARG = 1
FA_ERR_UNSUPPORTED = 2
FA_ERR_CUDA = 3
FA_ERR_TIMEOUT = 4
FA_ERR_BAD_SEQLENS = 5
FA_ERR_SCRATCH_LIMIT = 6
FA_DTYPE_FP16 = 0
FA_DTYPE_BF16 = 1

EXPORTED_SYMBOLS = ("fa_fwd", "fa_fwd_ex", "fa_fwd_split", "fa_split_plan",
                    "fa_fwd_split_noalloc", "fa_noalloc_scratch_bytes", "fa_fwd_kvcache",
                    "fa_kvcache_plan",
                    "fa_get_device_error", "fa_debug_wait_timeout",
                    "fa_debug_trace_read", "fa_shutdown", "fa_bwd", "fa_bwd_workspace_bytes",
                    "fa_status_string", "fa_version")

_HERE = os.path.dirname(os.path.abspath(__file__))
_lib = None
_lock = threading.Lock()


class LibraryMissing(RuntimeError):
    """libfa.so is not built (run ``__graft_entry__.build()``)."""


class FaError(RuntimeError):
    def __init__(self, status, where="fa_fwd"):
        self.status = status
        super().__init__(f"{where} failed: {status} ({fa_status_string(status)})")


def library_path() -> str:
    """In-tree libfa.so, or an ablation / debug build named by FA_LIB_VARIANT
    ("unfused", "threshold0", "trace")."""
    variant = os.environ.get("FA_LIB_VARIANT")
    return os.path.join(_HERE, f"libfa_{variant}.so" if variant else "libfa.so")


def load_library():
    """Load libfa.so (once) and declare the C signatures."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        path = library_path()
        if not os.path.exists(path):
            raise LibraryMissing(
                f"{path} is missing: build it with __graft_entry__.build() "
                "(nvcc, sm_103a); there is no fallback implementation")
        lib = ctypes.CDLL(path)
        vp, i32, f32 = ctypes.c_void_p, ctypes.c_int, ctypes.c_float
        lib.fa_fwd.argtypes = [vp, vp, vp, vp, vp, i32, i32, i32, i32, i32, i32, f32, i32,
                               vp, vp, vp, i32]
        lib.fa_fwd.restype = i32
        lib.fa_fwd_ex.argtypes = lib.fa_fwd.argtypes + [i32, i32, f32, vp]
        lib.fa_fwd_ex.restype = i32
        lib.fa_fwd_split.argtypes = lib.fa_fwd_ex.argtypes + [i32]
        lib.fa_fwd_split.restype = i32
        lib.fa_split_plan.argtypes = [i32] * 8 + [ctypes.POINTER(ctypes.c_longlong)]
        lib.fa_split_plan.restype = i32
        lib.fa_fwd_split_noalloc.argtypes = lib.fa_fwd_split.argtypes
        lib.fa_fwd_split_noalloc.restype = i32
        lib.fa_fwd_kvcache.argtypes = [vp, vp, vp, vp, vp, i32, i32, i32, i32, i32, f32, i32,
                                       vp, vp, i32, i32, i32, vp, i32, i32, i32, f32, vp, i32]
        lib.fa_fwd_kvcache.restype = i32
        lib.fa_kvcache_plan.argtypes = [i32] * 5 + [ctypes.c_longlong, i32,
                                                    ctypes.POINTER(ctypes.c_longlong)]
        lib.fa_kvcache_plan.restype = i32
        lib.fa_noalloc_scratch_bytes.argtypes = []
        lib.fa_noalloc_scratch_bytes.restype = ctypes.c_longlong
        lib.fa_get_device_error.argtypes = [vp]
        lib.fa_get_device_error.restype = i32
        lib.fa_debug_wait_timeout.argtypes = [ctypes.c_longlong, vp]
        lib.fa_debug_wait_timeout.restype = i32
        lib.fa_debug_trace_read.argtypes = [ctypes.POINTER(ctypes.c_ulonglong), i32]
        lib.fa_debug_trace_read.restype = i32
        lib.fa_bwd.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, i32, i32, i32, i32, i32, i32,
                               f32, i32, vp, vp, vp, ctypes.c_longlong, vp, i32]
        lib.fa_bwd.restype = i32
        lib.fa_bwd_workspace_bytes.argtypes = [i32, i32, i32]
        lib.fa_bwd_workspace_bytes.restype = ctypes.c_longlong
        lib.fa_shutdown.argtypes = []
        lib.fa_shutdown.restype = i32
        lib.fa_status_string.argtypes = [i32]
        lib.fa_status_string.restype = ctypes.c_char_p
        lib.fa_version.argtypes = []
        lib.fa_version.restype = i32
        _lib = lib
        return lib


def _addr(x):
    """Device / host address of a tensor, an int address, or None (NULL)."""
    if x is None:
        return None
    if isinstance(x, int):
        return x
    return x.data_ptr()


def _stream(s):
    if s is None:
        return None
    if isinstance(s, int):
        return s
    return s.cuda_stream  # torch.cuda.Stream


def fa_fwd(q, k, v, o, lse, B, Hq, Hkv, Sq, Sk, D, scale, causal,
           cu_seqlens_q, cu_seqlens_k, stream, dtype) -> int:
    """Call the C ``fa_fwd``; returns its status code (see include/fa.h)."""
    lib = load_library()
    return lib.fa_fwd(_addr(q), _addr(k), _addr(v), _addr(o), _addr(lse), int(B), int(Hq),
                      int(Hkv), int(Sq), int(Sk), int(D), float(scale), int(causal),
                      _addr(cu_seqlens_q), _addr(cu_seqlens_k), _stream(stream), int(dtype))


def fa_fwd_ex(q, k, v, o, lse, B, Hq, Hkv, Sq, Sk, D, scale, causal,
              cu_seqlens_q, cu_seqlens_k, stream, dtype, window_left=-1, window_right=-1,
              softcap=0.0, alibi_slopes=None) -> int:
    """Call the C ``fa_fwd_ex`` (local window, soft cap, ALiBi slopes)."""
    lib = load_library()
    return lib.fa_fwd_ex(_addr(q), _addr(k), _addr(v), _addr(o), _addr(lse), int(B), int(Hq),
                         int(Hkv), int(Sq), int(Sk), int(D), float(scale), int(causal),
                         _addr(cu_seqlens_q), _addr(cu_seqlens_k), _stream(stream), int(dtype),
                         int(window_left), int(window_right), float(softcap),
                         _addr(alibi_slopes))


def fa_fwd_split(q, k, v, o, lse, B, Hq, Hkv, Sq, Sk, D, scale, causal,
                 cu_seqlens_q, cu_seqlens_k, stream, dtype, window_left=-1, window_right=-1,
                 softcap=0.0, alibi_slopes=None, num_splits=0) -> int:
    """Call the C ``fa_fwd_split`` (split-KV forward + LSE merge)."""
    lib = load_library()
    return lib.fa_fwd_split(_addr(q), _addr(k), _addr(v), _addr(o), _addr(lse), int(B),
                            int(Hq), int(Hkv), int(Sq), int(Sk), int(D), float(scale),
                            int(causal), _addr(cu_seqlens_q), _addr(cu_seqlens_k),
                            _stream(stream), int(dtype), int(window_left), int(window_right),
                            float(softcap), _addr(alibi_slopes), int(num_splits))


def fa_fwd_split_noalloc(q, k, v, o, lse, B, Hq, Hkv, Sq, Sk, D, scale, causal,
                         cu_seqlens_q, cu_seqlens_k, stream, dtype, window_left=-1,
                         window_right=-1, softcap=0.0, alibi_slopes=None, num_splits=0) -> int:
    """Call the C ``fa_fwd_split_noalloc`` (split scratch in a fixed device array)."""
    lib = load_library()
    return lib.fa_fwd_split_noalloc(_addr(q), _addr(k), _addr(v), _addr(o), _addr(lse),
                                    int(B), int(Hq), int(Hkv), int(Sq), int(Sk), int(D),
                                    float(scale), int(causal), _addr(cu_seqlens_q),
                                    _addr(cu_seqlens_k), _stream(stream), int(dtype),
                                    int(window_left), int(window_right), float(softcap),
                                    _addr(alibi_slopes), int(num_splits))


def fa_fwd_kvcache(q, k_cache, v_cache, o, lse, B, Hq, Hkv, Sq, D, scale, causal,
                   cache_seqlens, block_table, max_blocks, page_rows, num_pages, stream, dtype,
                   window_left=-1, window_right=-1, softcap=0.0, alibi_slopes=None,
                   num_splits=0) -> int:
    """Call the C ``fa_fwd_kvcache`` (attention over a contiguous or paged KV cache)."""
    lib = load_library()
    return lib.fa_fwd_kvcache(_addr(q), _addr(k_cache), _addr(v_cache), _addr(o), _addr(lse),
                              int(B), int(Hq), int(Hkv), int(Sq), int(D), float(scale),
                              int(causal), _addr(cache_seqlens), _addr(block_table),
                              int(max_blocks), int(page_rows), int(num_pages), _stream(stream),
                              int(dtype), int(window_left), int(window_right), float(softcap),
                              _addr(alibi_slopes), int(num_splits))


def fa_kvcache_plan(B, Hq, Hkv, Sq, D, capacity, num_splits=0):
    """(split count or minus a status code, scratch bytes) of ``fa_fwd_kvcache``."""
    nbytes = ctypes.c_longlong(0)
    n = load_library().fa_kvcache_plan(int(B), int(Hq), int(Hkv), int(Sq), int(D),
                                       int(capacity), int(num_splits), ctypes.byref(nbytes))
    return n, nbytes.value


def fa_noalloc_scratch_bytes() -> int:
    return int(load_library().fa_noalloc_scratch_bytes())


def fa_split_plan(B, Hq, Hkv, Sq, Sk, D, varlen, num_splits=0):
    """(split count or minus a status code, scratch bytes) of ``fa_fwd_split``."""
    nbytes = ctypes.c_longlong(0)
    n = load_library().fa_split_plan(int(B), int(Hq), int(Hkv), int(Sq), int(Sk), int(D),
                                     int(bool(varlen)), int(num_splits), ctypes.byref(nbytes))
    return n, nbytes.value


def fa_get_device_error(stream=None) -> int:
    return load_library().fa_get_device_error(_stream(stream))


def fa_debug_wait_timeout(limit_cycles, stream=None) -> int:
    return load_library().fa_debug_wait_timeout(int(limit_cycles), _stream(stream))


def fa_debug_trace_read(n=2048):
    """(status, list of n clock stamps) from a trace build's buffer."""
    buf = (ctypes.c_ulonglong * n)()
    st = load_library().fa_debug_trace_read(buf, n)
    return st, list(buf)


def fa_shutdown() -> int:
    """Drop the library's cached per-device state (status-word and scratch
    addresses, SM counts, shared-memory opt-ins); later calls set it up again."""
    return load_library().fa_shutdown()


def fa_bwd(q, k, v, o, lse, dout, dq, dk, dv, B, Hq, Hkv, Sq, Sk, D, scale, causal,
           cu_seqlens_q, cu_seqlens_k, workspace, workspace_bytes, stream, dtype) -> int:
    """Call the C ``fa_bwd`` (gradients dq, dk, dv); returns its status code."""
    lib = load_library()
    return lib.fa_bwd(_addr(q), _addr(k), _addr(v), _addr(o), _addr(lse), _addr(dout), _addr(dq),
                      _addr(dk), _addr(dv), int(B), int(Hq), int(Hkv), int(Sq), int(Sk), int(D),
                      float(scale), int(causal), _addr(cu_seqlens_q), _addr(cu_seqlens_k),
                      _addr(workspace), int(workspace_bytes), _stream(stream), int(dtype))


def fa_bwd_workspace_bytes(B, Hq, Sq) -> int:
    """Device workspace bytes ``fa_bwd`` needs (or minus a status code)."""
    return int(load_library().fa_bwd_workspace_bytes(int(B), int(Hq), int(Sq)))


def attention_backward(q, k, v, out, lse, dout, causal=False, scale=None, stream=None,
                       cu_seqlens_q=None, cu_seqlens_k=None):
    """Gradients of exact attention on CUDA tensors; returns ``(dq, dk, dv)``.

    Dense: q / out / dout [B, Sq, Hq, D], k / v [B, Sk, Hkv, D], lse
    [B, Hq, Sq]; packed: q / out / dout [total_q, Hq, D], k / v [total_k, Hkv,
    D], lse [Hq, total_q] with int32 cu_seqlens, as :func:`attention_forward`
    returned them.  The workspace is a PyTorch allocation; everything else
    runs in ``fa_bwd``'s kernels.
    """
    import torch

    dtype = {torch.float16: FA_DTYPE_FP16, torch.bfloat16: FA_DTYPE_BF16}.get(q.dtype)
    if dtype is None:
        raise FaError(FA_ERR_UNSUPPORTED, "attention_backward (dtype)")
    for t in (q, k, v, out, lse, dout):
        if not t.is_contiguous():
            raise FaError(FA_ERR_INVALID_ARG, "attention_backward (contiguity)")
    if cu_seqlens_q is None:
        B, Sq, Hq, D = q.shape
        Sk, Hkv = k.shape[1], k.shape[2]
        rows_b = B
    else:
        Sq, Hq, D = q.shape
        Sk, Hkv = k.shape[0], k.shape[1]
        B, rows_b = cu_seqlens_q.numel() - 1, 1
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    if stream is None:
        stream = torch.cuda.current_stream(q.device)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    nbytes = fa_bwd_workspace_bytes(rows_b, Hq, Sq)
    if nbytes < 0:
        raise FaError(-nbytes, "fa_bwd_workspace_bytes")
    ws = torch.empty(max(nbytes, 16), dtype=torch.uint8, device=q.device)
    st = fa_bwd(q, k, v, out, lse, dout, dq, dk, dv, B, Hq, Hkv, Sq, Sk, D, scale,
                int(bool(causal)), cu_seqlens_q, cu_seqlens_k, ws, nbytes, stream, dtype)
    if st != FA_OK:
        raise FaError(st, "fa_bwd")
    return dq, dk, dv


def fa_status_string(status) -> str:
    return load_library().fa_status_string(int(status)).decode()


def fa_version() -> int:
    return load_library().fa_version()


def attention_forward(q, k, v, causal=False, scale=None, cu_seqlens_q=None,
                      cu_seqlens_k=None, out=None, lse=None, stream=None,
                      window_size=(-1, -1), softcap=0.0, alibi_slopes=None, num_splits=1):
    """Exact attention forward on CUDA tensors; returns ``(out, lse)``.

    Dense: q [B, Sq, Hq, D], k/v [B, Sk, Hkv, D] -> out like q, lse [B, Hq, Sq].
    Packed: q [total_q, Hq, D], k/v [total_k, Hkv, D] with int32 cu_seqlens of
    B + 1 offsets -> out like q, lse [Hq, total_q].
    ``window_size`` (left, right; -1 = unbounded), ``softcap`` and
    ``alibi_slopes`` (fp32 CUDA tensor [Hq]) select the score variants of
    ``fa_fwd_ex``; ``num_splits`` != 1 runs the split-KV path of
    ``fa_fwd_split`` (0 = chosen by the library).
    """
    import torch

    dtype = {torch.float16: FA_DTYPE_FP16, torch.bfloat16: FA_DTYPE_BF16}.get(q.dtype)
    if dtype is None:
        raise FaError(FA_ERR_UNSUPPORTED, "attention_forward (dtype)")
    for t in (q, k, v):
        if not t.is_contiguous():
            raise FaError(FA_ERR_INVALID_ARG, "attention_forward (contiguity)")
    if cu_seqlens_q is None:
        B, Sq, Hq, D = q.shape
        Sk, Hkv = k.shape[1], k.shape[2]
        lse_shape = (B, Hq, Sq)
    else:
        Sq, Hq, D = q.shape
        Sk, Hkv = k.shape[0], k.shape[1]
        B = cu_seqlens_q.numel() - 1
        lse_shape = (Hq, Sq)
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    if out is None:
        out = torch.empty_like(q)
    if lse is None:
        lse = torch.empty(lse_shape, dtype=torch.float32, device=q.device)
    if stream is None:
        stream = torch.cuda.current_stream(q.device)
    if alibi_slopes is not None and (alibi_slopes.dtype != torch.float32
                                     or alibi_slopes.shape != (Hq,)
                                     or not alibi_slopes.is_contiguous()):
        raise FaError(FA_ERR_INVALID_ARG, "attention_forward (alibi_slopes)")
    st = fa_fwd_split(q, k, v, out, lse, B, Hq, Hkv, Sq, Sk, D, scale, int(bool(causal)),
                      cu_seqlens_q, cu_seqlens_k, stream, dtype, window_size[0],
                      window_size[1], softcap, alibi_slopes, num_splits)
    if st != FA_OK:
        raise FaError(st)
    return out, lse


def attention_kvcache(q, k_cache, v_cache, cache_seqlens, block_table=None, causal=False,
                      scale=None, out=None, lse=None, stream=None, window_size=(-1, -1),
                      softcap=0.0, alibi_slopes=None, num_splits=0):
    """Attention of q [B, Sq, Hq, D] over a KV cache; returns ``(out, lse)``.

    Contiguous cache: k_cache / v_cache [B, capacity, Hkv, D].  Paged cache:
    k_cache / v_cache [num_pages, page_rows, Hkv, D] with an int32
    ``block_table`` [B, max_blocks].  ``cache_seqlens``: int32 [B] keys per
    sequence.  All tensors on the same CUDA device.
    """
    import torch

    dtype = {torch.float16: FA_DTYPE_FP16, torch.bfloat16: FA_DTYPE_BF16}.get(q.dtype)
    if dtype is None:
        raise FaError(FA_ERR_UNSUPPORTED, "attention_kvcache (dtype)")
    B, Sq, Hq, D = q.shape
    pages, page_rows, Hkv = k_cache.shape[0], k_cache.shape[1], k_cache.shape[2]
    max_blocks = block_table.shape[1] if block_table is not None else 1
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    if out is None:
        out = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((B, Hq, Sq), dtype=torch.float32, device=q.device)
    if stream is None:
        stream = torch.cuda.current_stream(q.device)
    st = fa_fwd_kvcache(q, k_cache, v_cache, out, lse, B, Hq, Hkv, Sq, D, scale,
                        int(bool(causal)), cache_seqlens, block_table, max_blocks, page_rows,
                        pages, stream, dtype, window_size[0], window_size[1], softcap,
                        alibi_slopes, num_splits)
    if st != FA_OK:
        raise FaError(st, "fa_fwd_kvcache")
    return out, lse
