"""Host-side checks of the C ABI (no GPU needed, no kernel launched).

libfa.so must load on a machine without a GPU, export every function that
include/fa.h declares, and reject invalid arguments before touching CUDA.
"""
import ctypes
import os
import re

import pytest

import exact_attention_forward_sm_gb300 as fa
from exact_attention_forward_sm_gb300 import _build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    _build.build()
    return fa.load_library()


def _declared_functions():
    text = open(os.path.join(ROOT, "include", "fa.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(fa_[a-z_0-9]+)\s*\(", text)))


def test_header_declares_the_exports():
    assert _declared_functions() == sorted(fa.EXPORTED_SYMBOLS)


def test_library_exports_every_declared_symbol(lib):
    for name in _declared_functions():
        assert hasattr(lib, name), name


def test_status_strings_and_version(lib):
    assert fa.fa_version() >= 100
    for code in range(7):
        assert fa.fa_status_string(code) not in ("", "unknown status")
    assert fa.fa_status_string(99) == "unknown status"


def _call(**kw):
    args = dict(q=16, k=16, v=16, o=16, lse=None, B=1, Hq=2, Hkv=2, Sq=8, Sk=8, D=64,
                scale=0.125, causal=0, cu_seqlens_q=None, cu_seqlens_k=None, stream=None,
                dtype=fa.FA_DTYPE_BF16)
    args.update(kw)
    return fa.fa_fwd(**args)


@pytest.mark.parametrize("bad", [
    dict(B=-1), dict(Hq=0), dict(Hkv=0), dict(Hq=3, Hkv=2), dict(Sq=-1), dict(Sk=-5),
    dict(D=0), dict(causal=2), dict(dtype=7), dict(scale=0.0), dict(scale=float("nan")),
    dict(scale=float("inf")), dict(cu_seqlens_q=64), dict(q=0), dict(o=0),
    dict(q=8), dict(v=24), dict(lse=2),
])
def test_invalid_arguments_rejected_without_launch(lib, bad):
    assert _call(**bad) == fa.FA_ERR_INVALID_ARG


def _call_ex(window_left=-1, window_right=-1, softcap=0.0, alibi_slopes=None, **kw):
    args = dict(q=16, k=16, v=16, o=16, lse=None, B=1, Hq=2, Hkv=2, Sq=8, Sk=8, D=64,
                scale=0.125, causal=0, cu_seqlens_q=None, cu_seqlens_k=None, stream=None,
                dtype=fa.FA_DTYPE_BF16)
    args.update(kw)
    return fa.fa_fwd_ex(**args, window_left=window_left, window_right=window_right,
                        softcap=softcap, alibi_slopes=alibi_slopes)


@pytest.mark.parametrize("bad", [
    dict(softcap=-1.0), dict(softcap=float("nan")), dict(softcap=float("inf")),
    dict(softcap=1e-40), dict(alibi_slopes=18), dict(B=-1), dict(causal=3),
])
def test_variant_arguments_rejected_without_launch(lib, bad):
    assert _call_ex(**bad) == fa.FA_ERR_INVALID_ARG


@pytest.mark.parametrize("splits", [-1, 129, 1 << 20])
def test_split_count_out_of_range_rejected(lib, splits):
    args = dict(q=16, k=16, v=16, o=16, lse=None, B=1, Hq=2, Hkv=2, Sq=8, Sk=8, D=64,
                scale=0.125, causal=0, cu_seqlens_q=None, cu_seqlens_k=None, stream=None,
                dtype=fa.FA_DTYPE_BF16)
    assert fa.fa_fwd_split(**args, num_splits=splits) == fa.FA_ERR_INVALID_ARG


def test_split_plan_forced_counts_and_scratch(lib):
    assert fa.fa_split_plan(2, 8, 2, 100, 5000, 128, 0, 4) == (4, 4 * 2 * 8 * 100 * 129 * 4)
    assert fa.fa_split_plan(3, 4, 4, 70, 90, 64, 1, 1) == (1, 0)
    assert fa.fa_split_plan(0, 4, 4, 70, 90, 64, 0, 0) == (1, 0)   # no rows: nothing to split
    assert fa.fa_split_plan(1, 3, 2, 8, 8, 64, 0, 2)[0] == -fa.FA_ERR_INVALID_ARG
    assert fa.fa_split_plan(1, 2, 2, 8, 8, 96, 0, 2)[0] == -fa.FA_ERR_UNSUPPORTED
    assert fa.fa_split_plan(1, 2, 2, 8, 8, 64, 0, 200)[0] == -fa.FA_ERR_INVALID_ARG


def _kvc(**kw):
    args = dict(q=16, k_cache=16, v_cache=16, o=16, lse=None, B=1, Hq=4, Hkv=2, Sq=1, D=64,
                scale=0.125, causal=0, cache_seqlens=16, block_table=None, max_blocks=1,
                page_rows=256, num_pages=1, stream=None, dtype=fa.FA_DTYPE_BF16)
    args.update(kw)
    return fa.fa_fwd_kvcache(**args)


@pytest.mark.parametrize("bad", [
    dict(page_rows=0), dict(block_table=16, page_rows=100), dict(block_table=16, max_blocks=0),
    dict(block_table=16, num_pages=0), dict(block_table=18), dict(cache_seqlens=0),
    dict(cache_seqlens=18), dict(num_splits=-1), dict(softcap=-2.0), dict(Hq=3),
    dict(q=8), dict(k_cache=0),
])
def test_kvcache_arguments_rejected_without_launch(lib, bad):
    assert _kvc(**bad) == fa.FA_ERR_INVALID_ARG


def test_kvcache_plan_forced_counts_and_scratch(lib):
    assert fa.fa_kvcache_plan(8, 32, 8, 1, 128, 4096, 5) == (5, 5 * 8 * 32 * 1 * 129 * 4)
    assert fa.fa_kvcache_plan(8, 32, 8, 1, 128, 4096, 1) == (1, 0)
    assert fa.fa_kvcache_plan(8, 12, 4, 1, 128, 4096, 1)[0] == -fa.FA_ERR_UNSUPPORTED
    assert fa.fa_kvcache_plan(8, 32, 8, 1, 128, 0, 1)[0] == -fa.FA_ERR_INVALID_ARG


@pytest.mark.parametrize("Hq,Hkv,D", [(6, 2, 64), (4, 2, 96), (256, 1, 64)])
def test_kvcache_unsupported(lib, Hq, Hkv, D):
    assert _kvc(Hq=Hq, Hkv=Hkv, D=D) == fa.FA_ERR_UNSUPPORTED


def test_variant_empty_problems_are_noops(lib):
    assert _call_ex(B=0, window_left=3, softcap=30.0) == fa.FA_OK
    assert _call_ex(Sq=0, alibi_slopes=16) == fa.FA_OK


@pytest.mark.parametrize("D", [32, 96, 192, 512])
def test_unbuilt_head_dims_unsupported(lib, D):
    assert _call(D=D) == fa.FA_ERR_UNSUPPORTED


def test_k_v_may_be_null_only_without_keys(lib):
    assert _call(k=0, v=0, Sk=4) == fa.FA_ERR_INVALID_ARG


def test_empty_problems_are_noops(lib):
    assert _call(B=0) == fa.FA_OK
    assert _call(Sq=0) == fa.FA_OK


def test_binding_raises_when_library_missing(tmp_path, monkeypatch):
    monkeypatch.setattr(fa, "_lib", None)
    monkeypatch.setattr(fa, "library_path", lambda: str(tmp_path / "libfa.so"))
    with pytest.raises(fa.LibraryMissing):
        fa.load_library()


def test_product_package_does_not_import_the_oracle():
    pkg = os.path.join(ROOT, "exact_attention_forward_sm_gb300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h")):
                src = open(os.path.join(dirpath, f)).read()
                assert "import oracle" not in src and "oracle." not in src.replace(
                    "the oracle", ""), f


def test_shutdown_without_a_gpu_is_ok(lib):
    # fa_shutdown only drops cached host-side values: no CUDA call is made
    assert fa.fa_shutdown() == fa.FA_OK
    assert fa.fa_shutdown() == fa.FA_OK


def _call_noalloc(num_splits=4, **kw):
    args = dict(q=16, k=16, v=16, o=16, lse=None, B=1, Hq=2, Hkv=2, Sq=8, Sk=8, D=64,
                scale=0.125, causal=0, cu_seqlens_q=None, cu_seqlens_k=None, stream=None,
                dtype=fa.FA_DTYPE_BF16)
    args.update(kw)
    return fa.fa_fwd_split_noalloc(**args, window_left=-1, window_right=-1, softcap=0.0,
                                   alibi_slopes=None, num_splits=num_splits)


@pytest.mark.parametrize("bad", [dict(B=-1), dict(Hq=3, Hkv=2), dict(D=0), dict(q=8),
                                 dict(num_splits=-1), dict(num_splits=129)])
def test_no_alloc_checks_arguments_before_any_cuda_call(lib, bad):
    # argument errors come back as such, before the fixed array is looked up
    assert _call_noalloc(**bad) == fa.FA_ERR_INVALID_ARG


def test_no_alloc_empty_problem_is_a_no_op(lib):
    assert _call_noalloc(B=0) == fa.FA_OK
    assert _call_noalloc(Sq=0) == fa.FA_OK


def _call_bwd(**kw):
    args = dict(q=16, k=16, v=16, o=16, lse=16, dout=16, dq=16, dk=16, dv=16, B=1, Hq=2, Hkv=2,
                Sq=8, Sk=8, D=64, scale=0.125, causal=0, cu_seqlens_q=None, cu_seqlens_k=None,
                workspace=16, workspace_bytes=1 << 20, stream=None, dtype=fa.FA_DTYPE_BF16)
    args.update(kw)
    return fa.fa_bwd(**args)


@pytest.mark.parametrize("bad", [dict(B=-1), dict(Hq=3, Hkv=2), dict(Sq=-1), dict(causal=2),
                                 dict(dtype=7), dict(scale=0.0), dict(scale=float("nan")),
                                 dict(q=8), dict(dq=None), dict(workspace=None),
                                 dict(workspace_bytes=8), dict(lse=18)])
def test_backward_invalid_arguments_rejected_without_launch(lib, bad):
    assert _call_bwd(**bad) == fa.FA_ERR_INVALID_ARG


@pytest.mark.parametrize("bad", [dict(D=256), dict(D=96)])
def test_backward_unsupported(lib, bad):
    assert _call_bwd(**bad) == fa.FA_ERR_UNSUPPORTED


@pytest.mark.parametrize("bad", [dict(cu_seqlens_q=64), dict(cu_seqlens_k=64),
                                 dict(cu_seqlens_q=66, cu_seqlens_k=64)])
def test_backward_packed_offsets_checked(lib, bad):
    # both offset arrays or neither, each 4-byte aligned
    assert _call_bwd(**bad) == fa.FA_ERR_INVALID_ARG


def test_backward_workspace_bytes(lib):
    # lse in log2 units (rows rounded up to 4 floats), then delta
    assert fa.fa_bwd_workspace_bytes(2, 4, 10) == 4 * 80 + 4 * 80
    assert fa.fa_bwd_workspace_bytes(1, 1, 3) == 4 * 4 + 4 * 3
    assert fa.fa_bwd_workspace_bytes(0, 4, 10) == 0
    assert fa.fa_bwd_workspace_bytes(-1, 4, 10) == -fa.FA_ERR_INVALID_ARG
    assert _call_bwd(B=0) == fa.FA_OK
