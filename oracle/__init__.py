"""fp64 CPU oracle for the exact attention forward pass.

TEST INFRASTRUCTURE ONLY: the test suite, the package smoke check and the
benchmark's CPU-baseline / reference leg are the only callers.  The product
path (the CUDA library and its Python binding) never imports this package, and
this package imports nothing from the product.

The arithmetic lives in ``attention_oracle.c`` (plain C, fp64, OpenMP over
independent rows); this module only builds it with gcc and marshals arrays.

* :func:`attention` — the plain definition (full score row, softmax, O, LSE),
  optionally with a local window, a tanh soft cap and ALiBi slopes.
* :func:`attention_kvcache` — the same definition over a contiguous or paged
  KV cache (keys addressed through the block table, :func:`gather_kv_cache`).
* :func:`attention_online` — the streaming restatement with the lazy-rescale
  threshold and max lagging of the fork's v1.7 release notes (section 1.2),
  plus its skip / rescale counters and the largest P.
* :func:`attention_bwd` — the gradients dq, dk, dv of the plain definition
  for an upstream gradient dO (the backward pass of the v1.7 notes, section
  4.4), the derivative of softmax written out.

Both take the 16-bit inputs as exact float32 copies and address rows by their
LSE index (dense: ``(b * Hq + h) * Sq + i``; packed: ``h * total_q + t``).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "attention_oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile ``liboracle.so`` with gcc + OpenMP (no GPU needed)."""
    if (not force and os.path.exists(_LIB)
            and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC)):
        return _LIB
    tmp = _LIB + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fopenmp", "-fPIC", "-shared",
           "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        lib = ctypes.CDLL(build())
        f32p = ctypes.POINTER(ctypes.c_float)
        f64p = ctypes.POINTER(ctypes.c_double)
        i32p = ctypes.POINTER(ctypes.c_int32)
        i64p = ctypes.POINTER(ctypes.c_int64)
        c_int = ctypes.c_int
        common = [f32p, f32p, f32p, f64p, f64p,
                  c_int, c_int, c_int, c_int, c_int, c_int,
                  ctypes.c_double, c_int, i32p, i32p, i64p, ctypes.c_int64]
        lib.oracle_attention.argtypes = common + [c_int]
        lib.oracle_attention.restype = c_int
        lib.oracle_attention_ex.argtypes = (
            common[:13] + [c_int, c_int, ctypes.c_double, f64p] + common[13:] + [c_int])
        lib.oracle_attention_ex.restype = c_int
        lib.oracle_attention_online.argtypes = common + [
            c_int, ctypes.c_double, c_int, i64p, i64p, f64p, c_int]
        lib.oracle_attention_online.restype = c_int
        lib.oracle_attention_bwd.argtypes = [
            f32p, f32p, f32p, f32p, f64p, f64p, f64p,
            c_int, c_int, c_int, c_int, c_int, c_int, ctypes.c_double, c_int,
            i32p, i32p, c_int]
        lib.oracle_attention_bwd.restype = c_int
        lib.oracle_max_threads.argtypes = []
        lib.oracle_max_threads.restype = c_int
        _lib = lib
        return lib


def max_threads() -> int:
    return int(_load().oracle_max_threads())


def _as_f32(x):
    if hasattr(x, "detach"):  # torch tensor: upcast exactly on the CPU
        x = x.detach().to("cpu").float().numpy()
    return np.ascontiguousarray(x, dtype=np.float32)


def _ptr(a, ctype):
    return a.ctypes.data_as(ctypes.POINTER(ctype))


def _prep(q, k, v, B, Hq, Hkv, Sq, Sk, D, cu_seqlens_q, cu_seqlens_k, rows):
    q, k, v = _as_f32(q), _as_f32(k), _as_f32(v)
    varlen = cu_seqlens_q is not None
    if varlen:
        cu_q = np.ascontiguousarray(np.asarray(
            cu_seqlens_q.cpu() if hasattr(cu_seqlens_q, "cpu") else cu_seqlens_q),
            dtype=np.int32)
        cu_k = np.ascontiguousarray(np.asarray(
            cu_seqlens_k.cpu() if hasattr(cu_seqlens_k, "cpu") else cu_seqlens_k),
            dtype=np.int32)
        total_rows = Hq * int(cu_q[B])
    else:
        cu_q = cu_k = None
        total_rows = B * Hq * Sq
    if rows is None:
        rows = np.arange(total_rows, dtype=np.int64)
    rows = np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
    return q, k, v, cu_q, cu_k, rows


def attention(q, k, v, B, Hq, Hkv, Sq, Sk, D, scale, causal,
              cu_seqlens_q=None, cu_seqlens_k=None, rows=None, nthreads=0,
              window_left=-1, window_right=-1, softcap=0.0, alibi_slopes=None):
    """Plain-definition attention in fp64 for the requested rows.

    Optional variants: a local window (``window_left``, ``window_right``; a
    negative bound is unbounded), a tanh soft cap (``softcap`` > 0) and ALiBi
    (``alibi_slopes``: one slope per query head, natural-log units).

    Returns ``(o_rows [nrows, D] float64, lse_rows [nrows] float64)``; with
    ``rows=None`` every row, in LSE-index order.
    """
    lib = _load()
    q, k, v, cu_q, cu_k, rows = _prep(q, k, v, B, Hq, Hkv, Sq, Sk, D,
                                      cu_seqlens_q, cu_seqlens_k, rows)
    n = rows.shape[0]
    o = np.zeros((n, D), dtype=np.float64)
    lse = np.zeros((n,), dtype=np.float64)
    i32n = ctypes.POINTER(ctypes.c_int32)()
    slopes = None
    if alibi_slopes is not None:
        a = alibi_slopes.detach().cpu().double().numpy() if hasattr(alibi_slopes, "detach") \
            else alibi_slopes
        slopes = np.ascontiguousarray(np.asarray(a, dtype=np.float64))
        if slopes.shape != (Hq,):
            raise ValueError("alibi_slopes must hold one slope per query head")
    rc = lib.oracle_attention_ex(
        _ptr(q, ctypes.c_float), _ptr(k, ctypes.c_float), _ptr(v, ctypes.c_float),
        _ptr(o, ctypes.c_double), _ptr(lse, ctypes.c_double),
        B, Hq, Hkv, Sq, Sk, D, float(scale), int(bool(causal)),
        int(window_left), int(window_right), float(softcap),
        _ptr(slopes, ctypes.c_double) if slopes is not None else ctypes.POINTER(ctypes.c_double)(),
        _ptr(cu_q, ctypes.c_int32) if cu_q is not None else i32n,
        _ptr(cu_k, ctypes.c_int32) if cu_k is not None else i32n,
        _ptr(rows, ctypes.c_int64), n, int(nthreads))
    if rc != 0:
        raise ValueError(f"oracle_attention failed with status {rc}")
    return o, lse


def attention_online(q, k, v, B, Hq, Hkv, Sq, Sk, D, scale, causal,
                     cu_seqlens_q=None, cu_seqlens_k=None, rows=None,
                     block_n=128, threshold=8.0, lagging=True, nthreads=0):
    """Online-softmax restatement (fp64) with the lazy-rescale rule.

    Returns ``(o_rows, lse_rows, stats)`` where ``stats`` holds the number of
    skipped and performed rescales and the largest P seen.
    """
    lib = _load()
    q, k, v, cu_q, cu_k, rows = _prep(q, k, v, B, Hq, Hkv, Sq, Sk, D,
                                      cu_seqlens_q, cu_seqlens_k, rows)
    n = rows.shape[0]
    o = np.zeros((n, D), dtype=np.float64)
    lse = np.zeros((n,), dtype=np.float64)
    n_skip = ctypes.c_int64(0)
    n_rescale = ctypes.c_int64(0)
    max_p = ctypes.c_double(0.0)
    i32n = ctypes.POINTER(ctypes.c_int32)()
    rc = lib.oracle_attention_online(
        _ptr(q, ctypes.c_float), _ptr(k, ctypes.c_float), _ptr(v, ctypes.c_float),
        _ptr(o, ctypes.c_double), _ptr(lse, ctypes.c_double),
        B, Hq, Hkv, Sq, Sk, D, float(scale), int(bool(causal)),
        _ptr(cu_q, ctypes.c_int32) if cu_q is not None else i32n,
        _ptr(cu_k, ctypes.c_int32) if cu_k is not None else i32n,
        _ptr(rows, ctypes.c_int64), n, int(block_n), float(threshold),
        int(bool(lagging)), ctypes.byref(n_skip), ctypes.byref(n_rescale),
        ctypes.byref(max_p), int(nthreads))
    if rc != 0:
        raise ValueError(f"oracle_attention_online failed with status {rc}")
    return o, lse, {"skips": n_skip.value, "rescales": n_rescale.value,
                    "max_p": max_p.value}


def attention_bwd(q, k, v, dout, B, Hq, Hkv, Sq, Sk, D, scale, causal,
                  cu_seqlens_q=None, cu_seqlens_k=None, nthreads=0):
    """Gradients of plain-definition attention (fp64) for upstream gradient ``dout``.

    ``q`` / ``dout`` and ``k`` / ``v`` in the layouts of the C ABI (dense or
    packed).  Returns ``(dq, dk, dv)`` as float64 arrays shaped like ``q``,
    ``k`` and ``v``.
    """
    lib = _load()
    q, k, v, cu_q, cu_k, _ = _prep(q, k, v, B, Hq, Hkv, Sq, Sk, D,
                                   cu_seqlens_q, cu_seqlens_k, np.zeros(0, np.int64))
    do = _as_f32(dout)
    if do.shape != q.shape:
        raise ValueError("dout must have the shape of q")
    dq = np.zeros(q.shape, dtype=np.float64)
    dk = np.zeros(k.shape, dtype=np.float64)
    dv = np.zeros(v.shape, dtype=np.float64)
    i32n = ctypes.POINTER(ctypes.c_int32)()
    rc = lib.oracle_attention_bwd(
        _ptr(q, ctypes.c_float), _ptr(k, ctypes.c_float), _ptr(v, ctypes.c_float),
        _ptr(do, ctypes.c_float), _ptr(dq, ctypes.c_double), _ptr(dk, ctypes.c_double),
        _ptr(dv, ctypes.c_double), B, Hq, Hkv, Sq, Sk, D, float(scale), int(bool(causal)),
        _ptr(cu_q, ctypes.c_int32) if cu_q is not None else i32n,
        _ptr(cu_k, ctypes.c_int32) if cu_k is not None else i32n, int(nthreads))
    if rc != 0:
        raise ValueError(f"oracle_attention_bwd failed with status {rc}")
    return dq, dk, dv


def row_index_dense(b, h, i, Hq, Sq):
    """LSE index of dense row (b, h, i)."""
    return (np.asarray(b, dtype=np.int64) * Hq + h) * Sq + i


def row_index_packed(h, t, total_q):
    """LSE index of packed row (h, global token t)."""
    return np.asarray(h, dtype=np.int64) * total_q + t


def gather_kv_cache(cache, cache_seqlens, block_table=None):
    """Keys (or values) of each sequence read out of a KV cache, packed.

    Contiguous cache [B, capacity, Hkv, D]: sequence b's key j is cache[b, j].
    Paged cache [num_pages, page_rows, Hkv, D] with block_table [B, max_blocks]:
    key j of sequence b is row j % page_rows of page block_table[b, j // page_rows].
    Returns (packed [sum_b lk_b, Hkv, D] float32, cu_seqlens [B + 1] int32).
    """
    c = _as_f32(cache)
    lens = np.asarray(cache_seqlens.cpu() if hasattr(cache_seqlens, "cpu") else cache_seqlens,
                      dtype=np.int64)
    parts = []
    for b, lk in enumerate(lens):
        j = np.arange(int(lk))
        if block_table is None:
            parts.append(c[b, j])
        else:
            bt = np.asarray(block_table.cpu() if hasattr(block_table, "cpu") else block_table)
            page_rows = c.shape[1]
            parts.append(c[bt[b, j // page_rows], j % page_rows])
    packed = np.concatenate(parts, axis=0) if parts else np.zeros((0,) + c.shape[2:], np.float32)
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    return np.ascontiguousarray(packed), cu


def attention_kvcache(q, k_cache, v_cache, cache_seqlens, scale, causal, block_table=None,
                      rows=None, nthreads=0, window_left=-1, window_right=-1, softcap=0.0,
                      alibi_slopes=None):
    """Attention of q [B, Sq, Hq, D] over a KV cache (fp64, plain definition).

    Query token i of sequence b sits at position i + lk_b - Sq of its sequence
    (the bottom-right alignment of the plain path).  The cache is read by
    :func:`gather_kv_cache`; the attention itself is :func:`attention` on the
    resulting packed problem.  ``rows`` and the results use the LSE index of
    the [B, Hq, Sq] layout: (b * Hq + h) * Sq + i.
    """
    qf = _as_f32(q)
    B, Sq, Hq, D = qf.shape
    k, cu_k = gather_kv_cache(k_cache, cache_seqlens, block_table)
    v, _ = gather_kv_cache(v_cache, cache_seqlens, block_table)
    Hkv = k.shape[1] if k.ndim == 3 else _as_f32(k_cache).shape[2]
    cu_q = (np.arange(B + 1) * Sq).astype(np.int32)
    total_q = B * Sq
    if rows is None:
        rows = np.arange(B * Hq * Sq, dtype=np.int64)
    rows = np.asarray(rows, dtype=np.int64)
    b, rem = rows // (Hq * Sq), rows % (Hq * Sq)
    h, i = rem // Sq, rem % Sq
    packed_rows = h * total_q + b * Sq + i
    return attention(qf.reshape(total_q, Hq, D), k, v, B, Hq, Hkv, total_q, int(cu_k[-1]), D,
                     scale, causal, cu_q, cu_k, rows=packed_rows, nthreads=nthreads,
                     window_left=window_left, window_right=window_right, softcap=softcap,
                     alibi_slopes=alibi_slopes)
