"""fa_fwd_split_noalloc: the split-KV path with its partial results in a fixed
device array inside the library instead of a per-call allocation.  The file
name sorts last, so in a full run these tests also execute after every other
GPU test of the same process (and they pass when run alone)."""
import pytest
import torch

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():  # pragma: no cover - collected on CPU machines too
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

import exact_attention_forward_sm_gb300 as fa  # noqa: E402
from exact_attention_forward_sm_gb300 import workloads as wl  # noqa: E402
from tests.gpu_util import check, to_device  # noqa: E402


@pytest.fixture(scope="module", autouse=True)
def _built():
    from exact_attention_forward_sm_gb300 import _build
    _build.build()
    fa.load_library()


def _call(fn, case, num_splits, stream):
    q, k, v, cu_q, cu_k = to_device(case)
    o = torch.full_like(q, float("nan"))
    shape = (case.Hq, case.Sq) if case.varlen else (case.B, case.Hq, case.Sq)
    lse = torch.full(shape, float("nan"), dtype=torch.float32, device=q.device)
    st = fn(q, k, v, o, lse, case.B, case.Hq, case.Hkv, case.Sq, case.Sk, case.D, case.scale,
            int(case.causal), cu_q, cu_k, stream, wl.DTYPE_CODE[case.dtype],
            num_splits=num_splits)
    return st, o, lse


@pytest.mark.parametrize("num_splits", [0, 4])
def test_two_calls_in_a_row_match_the_allocating_entry_point(num_splits):
    stream = torch.cuda.current_stream()
    cases = [wl.make_case(1, 8, 8, 256, 8192, 128, "bf16", True, seed=41),
             wl.make_case(2, 4, 2, 130, 3000, 64, "fp16", False, seed=42)]
    for case in cases:
        n, nbytes = fa.fa_split_plan(case.B, case.Hq, case.Hkv, case.Sq, case.Sk, case.D, 0,
                                     num_splits)
        assert n > 1 and 0 < nbytes <= fa.fa_noalloc_scratch_bytes()
    ref = [_call(fa.fa_fwd_split, c, num_splits, stream) for c in cases]
    # two no-alloc calls back to back on one stream, the second reusing the
    # array the first one wrote
    got = [_call(fa.fa_fwd_split_noalloc, c, num_splits, stream) for c in cases]
    assert fa.fa_get_device_error(stream) == fa.FA_OK
    for case, (st0, o0, l0), (st1, o1, l1) in zip(cases, ref, got):
        assert st0 == fa.FA_OK and st1 == fa.FA_OK
        assert torch.equal(o0, o1) and torch.equal(l0, l1)
        check(case, o1, l1, tag="noalloc")


def test_oversize_is_rejected_with_nothing_launched():
    stream = torch.cuda.current_stream()
    case = wl.make_case(1, 8, 8, 256, 8192, 128, "bf16", False, seed=43)
    splits = 64
    _, nbytes = fa.fa_split_plan(case.B, case.Hq, case.Hkv, case.Sq, case.Sk, case.D, 0, splits)
    assert nbytes > fa.fa_noalloc_scratch_bytes()
    st, o, lse = _call(fa.fa_fwd_split_noalloc, case, splits, stream)
    assert st == fa.FA_ERR_SCRATCH_LIMIT
    torch.cuda.synchronize()
    assert torch.isnan(o).all() and torch.isnan(lse).all()


def test_unsplit_call_needs_no_scratch():
    stream = torch.cuda.current_stream()
    case = wl.make_case(4, 16, 16, 2048, 2048, 128, "bf16", True, seed=44)
    st0, o0, l0 = _call(fa.fa_fwd_split, case, 1, stream)
    st1, o1, l1 = _call(fa.fa_fwd_split_noalloc, case, 1, stream)
    assert st0 == st1 == fa.FA_OK
    assert torch.equal(o0, o1) and torch.equal(l0, l1)


def test_splits_without_keys_overwrite_stale_partials():
    """A split that sees no key must still write its slot (weight zero) even
    though an earlier call left finite partials in the shared array: first a
    call that fills the array, then one with more splits than key tiles, and a
    packed problem whose sequences have very different key counts."""
    stream = torch.cuda.current_stream()
    filler = wl.make_case(1, 8, 8, 256, 8192, 128, "bf16", False, seed=45)
    st, _, _ = _call(fa.fa_fwd_split_noalloc, filler, 8, stream)
    assert st == fa.FA_OK
    cases = [
        (wl.make_case(1, 2, 2, 200, 300, 128, "bf16", False, seed=46), 16),  # 3 K/V tiles
        (wl.make_case(0, 4, 2, 0, 0, 64, "fp16", True, seed=47,
                      seqlens_q=[1, 130, 64, 0, 300], seqlens_k=[900, 130, 2000, 5, 301]), 6),
    ]
    for case, splits in cases:
        st0, o0, l0 = _call(fa.fa_fwd_split, case, splits, stream)
        st1, o1, l1 = _call(fa.fa_fwd_split_noalloc, case, splits, stream)
        assert st0 == fa.FA_OK and st1 == fa.FA_OK
        assert fa.fa_get_device_error(stream) == fa.FA_OK
        assert torch.equal(o0, o1) and torch.equal(l0, l1)
        check(case, o1, l1, tag=f"noalloc split{splits} after a filled array")


def test_shutdown_then_no_alloc_call_sets_up_again():
    """fa_shutdown() drops the cached array address; the next call looks it up
    again and still matches the allocating path."""
    stream = torch.cuda.current_stream()
    case = wl.make_case(1, 8, 8, 256, 4096, 64, "bf16", True, seed=48)
    _, o0, l0 = _call(fa.fa_fwd_split, case, 4, stream)
    assert fa.fa_shutdown() == fa.FA_OK
    st, o1, l1 = _call(fa.fa_fwd_split_noalloc, case, 4, stream)
    assert st == fa.FA_OK and fa.fa_get_device_error(stream) == fa.FA_OK
    assert torch.equal(o0, o1) and torch.equal(l0, l1)
