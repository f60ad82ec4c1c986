"""GPU parity of the split-KV path (``fa_fwd_split``): each query tile's keys
are cut into chunks processed by separate work units, whose normalised
partial O and LSE are merged by an LSE-weighted combine.  This is the
split-KV forward that the fork's v1.2 notes, section 3, list among the
dispatch sites (compute_attn_1rowblock_splitkv); the result must match the
oracle under the same gates as the unsplit path."""
import zlib

import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():  # pragma: no cover - collected on CPU machines too
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

import exact_attention_forward_sm_gb300 as fa  # noqa: E402
from exact_attention_forward_sm_gb300 import workloads as wl  # noqa: E402
from tests.gpu_util import check, run_gpu, to_device  # noqa: E402


@pytest.fixture(scope="module", autouse=True)
def _built():
    from exact_attention_forward_sm_gb300 import _build
    _build.build()
    fa.load_library()


def _seed(*key):
    return zlib.crc32(repr(key).encode()) % 100000


SHAPES = [
    # B, Hq, Hkv, Sq, Sk, D, dtype, causal
    (1, 2, 2, 128, 1024, 64, "fp16", False),
    (1, 4, 2, 300, 900, 128, "bf16", True),
    (2, 3, 1, 257, 640, 64, "bf16", True),      # odd group: two row blocks per unit
    (1, 8, 2, 64, 2000, 128, "fp16", True),     # GQA 4:1, few query rows
    (2, 2, 2, 700, 300, 128, "bf16", True),     # Sq > Sk: rows with no visible key
]


@pytest.mark.parametrize("splits", [2, 3, 7])
@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "b{}_hq{}_hkv{}_sq{}_sk{}_d{}_{}_{}".format(
    *s[:7], "causal" if s[7] else "full"))
def test_split_all_rows(shape, splits):
    B, Hq, Hkv, Sq, Sk, D, dtype, causal = shape
    case = wl.make_case(B, Hq, Hkv, Sq, Sk, D, dtype, causal, seed=_seed(shape, splits))
    o, lse = run_gpu(case, num_splits=splits)
    check(case, o, lse, tag=f"split{splits} {shape}")


def test_more_splits_than_key_tiles():
    # 3 K/V tiles, 16 splits: 13 chunks are empty and contribute weight 0
    case = wl.make_case(1, 2, 2, 200, 300, 128, "bf16", False, seed=31)
    o, lse = run_gpu(case, num_splits=16)
    check(case, o, lse, tag="split16 of 3 tiles")


@pytest.mark.parametrize("D,dtype", [(64, "fp16"), (128, "bf16")])
def test_split_packed_sequences(D, dtype):
    case = wl.make_case(0, 4, 2, 0, 0, D, dtype, True, seed=_seed("packed", D),
                        seqlens_q=[1, 130, 64, 0, 300], seqlens_k=[900, 130, 2000, 5, 301])
    o, lse = run_gpu(case, num_splits=4)
    check(case, o, lse, tag=f"split4 packed D{D}")


def test_split_with_variants():
    Hq = 4
    case = wl.make_case(1, Hq, 2, 256, 1500, 128, "bf16", True, seed=32, sigma=2.0,
                        window=(700, 0), softcap=20.0,
                        alibi_slopes=wl.alibi_slopes_geometric(Hq))
    o, lse = run_gpu(case, num_splits=5)
    check(case, o, lse, tag="split5 window softcap alibi")


def test_split_plan_splits_small_problems_only():
    n, nbytes = fa.fa_split_plan(1, 8, 8, 256, 8192, 128, 0, 0)
    assert n > 1 and nbytes == n * 8 * 256 * 129 * 4
    assert fa.fa_split_plan(4, 16, 16, 2048, 2048, 128, 0, 0) == (1, 0)


def test_split_auto_choice_matches_oracle():
    # 2 row tiles x 8 heads = 16 units on a GPU with far more multiprocessors:
    # the library splits the 64 K/V tiles of each unit
    case = wl.make_case(1, 8, 8, 256, 8192, 128, "bf16", False, seed=33)
    o, lse = run_gpu(case, num_splits=0)
    check(case, o, lse, tag="split auto")


def test_split_one_equals_unsplit_bitwise():
    case = wl.make_case(1, 4, 4, 300, 700, 64, "fp16", True, seed=34)
    o0, l0 = run_gpu(case)
    o1, l1 = run_gpu(case, num_splits=1)
    assert torch.equal(o0, o1) and torch.equal(l0, l1)


def test_split_deterministic_and_null_lse():
    case = wl.make_case(1, 4, 4, 128, 3000, 128, "bf16", False, seed=35)
    o0, l0 = run_gpu(case, num_splits=6)
    o1, l1 = run_gpu(case, num_splits=6)
    assert torch.equal(o0, o1) and torch.equal(l0, l1)
    o2, _ = run_gpu(case, with_lse=False, num_splits=6)
    assert torch.equal(o0, o2)


def test_split_no_keys():
    case = wl.make_case(1, 2, 2, 100, 0, 64, "fp16", False, seed=36)
    o, lse = run_gpu(case, num_splits=4)
    assert torch.all(o == 0) and torch.all(torch.isneginf(lse))


def test_split_leaves_rows_of_no_sequence_untouched():
    """Packed tokens outside [cu_seqlens_q[0], cu_seqlens_q[B]) belong to no
    sequence: neither the partial pass nor the merge may write their O."""
    dev = "cuda:0"
    lens = [40, 200]
    case = wl.make_case(0, 2, 2, 0, 0, 64, "bf16", False, seed=37, seqlens_q=lens,
                        seqlens_k=[500, 600])
    pad = 16
    q, k, v, _, _ = to_device(case)
    total = case.Sq + 2 * pad
    qq = torch.zeros((total, 2, 64), dtype=q.dtype, device=dev)
    qq[pad:pad + case.Sq] = q
    cu_q = (case.cu_seqlens_q + pad).to(dev)
    cu_k = case.cu_seqlens_k.to(dev)
    o = torch.full_like(qq, float("nan"))
    lse = torch.full((2, total), float("nan"), dtype=torch.float32, device=dev)
    st = fa.fa_fwd_split(qq, k, v, o, lse, 2, 2, 2, total, case.Sk, 64, case.scale, 0, cu_q,
                         cu_k, torch.cuda.current_stream(), fa.FA_DTYPE_BF16, num_splits=3)
    assert st == fa.FA_OK
    assert fa.fa_get_device_error(torch.cuda.current_stream()) == fa.FA_OK
    assert torch.isnan(o[:pad]).all() and torch.isnan(o[pad + case.Sq:]).all()
    assert torch.isnan(lse[:, :pad]).all() and torch.isnan(lse[:, pad + case.Sq:]).all()
    o_in, lse_in = o[pad:pad + case.Sq], lse[:, pad:pad + case.Sq]
    check(case, o_in.contiguous(), lse_in.contiguous(), tag="split padded packed")
