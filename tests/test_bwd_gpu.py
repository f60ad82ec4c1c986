"""GPU parity of the backward pass (``fa_bwd``) against the fp64 backward oracle.

The fork's v1.7 release notes validate a backward pass next to the forward
(section 4.4): finite dQ / dK / dV at S = 2048 causal in fp16 and bf16, and
gradient errors against an fp32 reference.  Here the library's gradients,
computed from its own forward output and LSE, are compared element by element
with ``oracle.attention_bwd`` (fp64, plain definition) on the same 16-bit
inputs and upstream gradient.

Gates per gradient tensor: cosine >= 0.9995 and max |g - ref| <= TOL *
max(max |ref|, 1e-3) with TOL = 2e-2 (bf16) / 1e-2 (fp16).  The kernels
round P and dS to the input type for the tensor-core products and the outputs
to it (bf16 keeps 8 significant bits: 2^-9 relative per rounding, 2^-8 per
output element at worst); the row term rowsum(dO * O) reads the 16-bit O, and
dS = P (dP - rowsum) cancels, so the gates sit a few output roundings above
that.

With FA_PARITY_REPORT=<path> set, every comparison appends its metrics to
that file as one JSON line.
"""
import json
import os

import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():  # pragma: no cover - collected on CPU machines too
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

import exact_attention_forward_sm_gb300 as fa  # noqa: E402
import oracle  # noqa: E402

TOL = {"bf16": 2e-2, "fp16": 1e-2}
COS_MIN = 0.9995
ABS_FLOOR = 1e-3
TORCH_DT = {"bf16": torch.bfloat16, "fp16": torch.float16}


@pytest.fixture(scope="module", autouse=True)
def _built():
    from exact_attention_forward_sm_gb300 import _build
    _build.build()
    fa.load_library()


def _draw(B, Hq, Hkv, Sq, Sk, D, dtype, seed, sigma=1.0):
    g = torch.Generator().manual_seed(seed)
    dt = TORCH_DT[dtype]
    q = (torch.randn(B, Sq, Hq, D, generator=g) * sigma).to(dt)
    k = (torch.randn(B, Sk, Hkv, D, generator=g) * sigma).to(dt)
    v = torch.randn(B, Sk, Hkv, D, generator=g).to(dt)
    do = torch.randn(B, Sq, Hq, D, generator=g).to(dt)
    return q, k, v, do


def _run(q, k, v, do, causal, scale=None):
    dev = "cuda:0"
    qd, kd, vd, dod = (t.to(dev).contiguous() for t in (q, k, v, do))
    out, lse = fa.attention_forward(qd, kd, vd, causal=causal, scale=scale)
    dq, dk, dv = fa.attention_backward(qd, kd, vd, out, lse, dod, causal=causal, scale=scale)
    st = fa.fa_get_device_error(torch.cuda.current_stream())
    assert st == fa.FA_OK, fa.fa_status_string(st)
    return dq, dk, dv


def _compare(name, got, ref, dtype):
    g = got.float().cpu().numpy().astype(np.float64)
    assert np.isfinite(g).all(), f"{name}: non-finite gradient"
    # a reference that vanishes (one key: dS = 0 exactly) is held to an
    # absolute floor: the rounding noise of dP - rowsum(dO * O) stays far below
    scale = max(np.max(np.abs(ref)), ABS_FLOOR)
    err = np.max(np.abs(g - ref)) / scale
    cos = float(np.sum(g * ref) / max(np.linalg.norm(g) * np.linalg.norm(ref), 1e-300))
    report = os.environ.get("FA_PARITY_REPORT")
    if report:
        with open(report, "a") as f:
            f.write(json.dumps({"case": os.environ.get("PYTEST_CURRENT_TEST", "").split(" ")[0],
                                "grad": name, "dtype": dtype, "err_of_max": err,
                                "cosine": cos}) + "\n")
    assert err <= TOL[dtype], f"{name}: max error {err:.3e} of max |ref|"
    if np.max(np.abs(ref)) > 0:
        assert cos >= COS_MIN, f"{name}: cosine {cos:.6f}"
    return err, cos


def _check(B, Hq, Hkv, Sq, Sk, D, dtype, causal, seed, sigma=1.0):
    q, k, v, do = _draw(B, Hq, Hkv, Sq, Sk, D, dtype, seed, sigma)
    dq, dk, dv = _run(q, k, v, do, causal)
    rq, rk, rv = oracle.attention_bwd(q, k, v, do, B, Hq, Hkv, Sq, Sk, D, D ** -0.5, causal)
    return {n: _compare(n, g, r, dtype) for n, g, r in
            (("dq", dq, rq), ("dk", dk, rk), ("dv", dv, rv))}


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("D,dtype", [(128, "bf16"), (64, "fp16"), (128, "fp16"), (64, "bf16")])
def test_gradients_several_tiles_ragged(causal, D, dtype):
    """Three query and key tiles with a ragged tail, GQA 2:1."""
    _check(2, 4, 2, 300, 300, D, dtype, causal, seed=D + 7 * causal + (dtype == "bf16"))


@pytest.mark.parametrize("Sq,Sk", [(200, 333), (333, 200), (1, 129), (129, 1)])
def test_gradients_unequal_lengths(Sq, Sk):
    """Bottom-right aligned causal masking with Sq != Sk; Sq > Sk leaves the
    first Sq - Sk rows without keys (dq = 0) and Sk = 1 / Sq = 1 edge tiles."""
    _check(1, 2, 2, Sq, Sk, 64, "fp16", True, seed=Sq * 1000 + Sk)
    _check(1, 2, 1, Sq, Sk, 128, "bf16", False, seed=Sq * 1000 + Sk + 1)


def test_gradients_gqa_4_to_1_wide_scores():
    _check(1, 8, 2, 257, 384, 128, "bf16", True, seed=41, sigma=1.6)


def test_repeatable_bit_for_bit():
    q, k, v, do = _draw(2, 4, 2, 256, 384, 128, "bf16", 5)
    a = _run(q, k, v, do, True)
    b = _run(q, k, v, do, True)
    for x, y in zip(a, b):
        assert torch.equal(x, y)


def test_no_queries_or_no_keys_give_zero_gradients():
    dev = "cuda:0"
    q = torch.randn(2, 0, 4, 64, device=dev, dtype=torch.bfloat16)
    k = torch.randn(2, 50, 2, 64, device=dev, dtype=torch.bfloat16)
    v = torch.randn_like(k)
    o = torch.empty_like(q)
    lse = torch.empty(2, 4, 0, device=dev)
    dk = torch.full_like(k, float("nan"))
    dv = torch.full_like(v, float("nan"))
    st = fa.fa_bwd(q, k, v, o, lse, o, o, dk, dv, 2, 4, 2, 0, 50, 64, 0.125, 1, None, None,
                   None, 0, torch.cuda.current_stream(), fa.FA_DTYPE_BF16)
    assert st == fa.FA_OK
    torch.cuda.synchronize()
    assert torch.count_nonzero(dk) == 0 and torch.count_nonzero(dv) == 0
    q = torch.randn(2, 30, 4, 64, device=dev, dtype=torch.bfloat16)
    k = torch.empty(2, 0, 2, 64, device=dev, dtype=torch.bfloat16)
    dq = torch.full_like(q, float("nan"))
    ws = torch.empty(fa.fa_bwd_workspace_bytes(2, 4, 30), dtype=torch.uint8, device=dev)
    lse = torch.full((2, 4, 30), float("-inf"), device=dev)
    st = fa.fa_bwd(q, k, k, q, lse, q, dq, k, k, 2, 4, 2, 30, 0, 64, 0.125, 0, None, None,
                   ws, ws.numel(), torch.cuda.current_stream(), fa.FA_DTYPE_BF16)
    assert st == fa.FA_OK
    torch.cuda.synchronize()
    assert torch.count_nonzero(dq) == 0


def test_full_size_causal_benchmark_shape():
    """B4 H16 S2048 D128 bf16 causal (the forward benchmark's shape; the
    release notes' backward finiteness check runs S = 2048 causal): every
    element of dq, dk, dv against the oracle."""
    _check(4, 16, 16, 2048, 2048, 128, "bf16", True, seed=2048)


def test_short_benchmark_shape():
    """B1 H2 S128 D64 fp16 non-causal, the short shape of the benchmark's
    backward workloads: one tile each way."""
    _check(1, 2, 2, 128, 128, 64, "fp16", False, seed=128)


def test_full_size_gqa_rising_bias_workload():
    """The GQA 4:1 workload with the rising per-key bias (B2 Hq32 Hkv8 S4096
    D128 bf16 causal), its own seeded inputs, every gradient element against
    the oracle.

    The workload carries its bias in channel D-1: q[..., D-1] = 1 and
    k[j, D-1] = b(j) ln2 / scale, up to |k| = 1256.  The row term
    Delta = rowsum(dO * O) is read from the 16-bit O (as the standard
    formulation does), so its rounding delta_i enters dq_i as
    scale * delta_i * sum_j P_ij k_j, and in channel D-1 that product is as
    large as dq itself (an fp64 emulation of the rounding alone moves that
    channel by up to its own size).  dk, dv and dq's other channels are held
    to the gates; channel D-1 of dq only to finiteness and to half of
    max |dq|."""
    from exact_attention_forward_sm_gb300 import workloads as wl
    case = wl.make_workload(wl.BY_NAME["b2_hq32_hkv8_s4096_d128_bf16_causal_risingbias"])
    g = torch.Generator().manual_seed(4096)
    do = torch.randn(tuple(case.q.shape), generator=g).to(case.q.dtype)
    dq, dk, dv = _run(case.q, case.k, case.v, do, True, scale=case.scale)
    rq, rk, rv = oracle.attention_bwd(case.q, case.k, case.v, do, case.B, case.Hq, case.Hkv,
                                      case.Sq, case.Sk, case.D, case.scale, True)
    _compare("dk", dk, rk, "bf16")
    _compare("dv", dv, rv, "bf16")
    _compare("dq[..., :D-1]", dq[..., :-1].contiguous(), rq[..., :-1], "bf16")
    carrier = dq[..., -1].float().cpu().numpy()
    assert np.isfinite(carrier).all()
    assert np.max(np.abs(carrier - rq[..., -1])) <= 0.5 * np.max(np.abs(rq))


def _packed(lens_q, lens_k, Hq, Hkv, D, dtype, seed):
    g = torch.Generator().manual_seed(seed)
    dt = TORCH_DT[dtype]
    tq, tk = sum(lens_q), sum(lens_k)
    q = torch.randn(tq, Hq, D, generator=g).to(dt)
    k = torch.randn(tk, Hkv, D, generator=g).to(dt)
    v = torch.randn(tk, Hkv, D, generator=g).to(dt)
    do = torch.randn(tq, Hq, D, generator=g).to(dt)
    cu_q = torch.tensor([0] + list(np.cumsum(lens_q)), dtype=torch.int32)
    cu_k = torch.tensor([0] + list(np.cumsum(lens_k)), dtype=torch.int32)
    return q, k, v, do, cu_q, cu_k


def _run_packed(q, k, v, do, cu_q, cu_k, causal):
    dev = "cuda:0"
    qd, kd, vd, dod = (t.to(dev).contiguous() for t in (q, k, v, do))
    cqd, ckd = cu_q.to(dev), cu_k.to(dev)
    out, lse = fa.attention_forward(qd, kd, vd, causal=causal, cu_seqlens_q=cqd,
                                    cu_seqlens_k=ckd)
    dq, dk, dv = fa.attention_backward(qd, kd, vd, out, lse, dod, causal=causal,
                                       cu_seqlens_q=cqd, cu_seqlens_k=ckd)
    st = fa.fa_get_device_error(torch.cuda.current_stream())
    assert st == fa.FA_OK, fa.fa_status_string(st)
    return dq, dk, dv


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("D,dtype", [(128, "bf16"), (64, "fp16")])
def test_packed_sequences(causal, D, dtype):
    """Packed sequences of mixed lengths (ragged tails, an empty sequence,
    Sq != Sk per sequence), GQA 2:1: every gradient element against the
    oracle on the same packed layout."""
    lens_q = [300, 1, 0, 129, 513, 64]
    lens_k = [300, 130, 17, 129, 400, 64]
    q, k, v, do, cu_q, cu_k = _packed(lens_q, lens_k, 4, 2, D, dtype, seed=D + causal)
    dq, dk, dv = _run_packed(q, k, v, do, cu_q, cu_k, causal)
    refs = oracle.attention_bwd(q, k, v, do, len(lens_q), 4, 2, sum(lens_q), sum(lens_k), D,
                                D ** -0.5, causal, cu_q, cu_k)
    for n, t, r in zip(("dq", "dk", "dv"), (dq, dk, dv), refs):
        _compare(n, t, r, dtype)


def test_packed_neighbours_hold_inf_and_nan():
    """Sequences 1 and 3 hold Inf / NaN in q, k, v and dO; the other
    sequences' tiles reach into those rows (the forward notes' varlen hazard).
    Their gradients must still match the oracle and stay finite."""
    lens = [300, 129, 1000, 64, 257]
    q, k, v, do, cu_q, cu_k = _packed(lens, lens, 4, 2, 128, "bf16", seed=77)
    for t, vals in ((q, (float("nan"), float("inf"))), (k, (float("inf"), float("nan"))),
                    (v, (float("nan"), float("-inf"))), (do, (float("inf"), float("nan")))):
        for n, b in enumerate((1, 3)):
            t[int(cu_q[b]):int(cu_q[b + 1])] = vals[n]
    dq, dk, dv = _run_packed(q, k, v, do, cu_q, cu_k, True)
    refs = oracle.attention_bwd(q, k, v, do, len(lens), 4, 2, sum(lens), sum(lens), 128,
                                128 ** -0.5, True, cu_q, cu_k)
    clean = np.concatenate([np.arange(int(cu_q[b]), int(cu_q[b + 1])) for b in (0, 2, 4)])
    for n, t, r in zip(("dq", "dk", "dv"), (dq, dk, dv), refs):
        _compare(n, t[torch.as_tensor(clean, device=t.device)].contiguous(), r[clean], "bf16")


def test_full_size_packed_workload():
    """The packed benchmark workload at full size (16 sequences of 64 to 8192
    tokens from its seeded recipe, H16, D64 fp16 causal) with a seeded
    upstream gradient: every element of dq, dk, dv against the oracle (about
    a minute and a half of fp64 work on 16 host cores)."""
    from exact_attention_forward_sm_gb300 import workloads as wl
    case = wl.make_workload(wl.BY_NAME["varlen16_l64to8192_h16_d64_fp16_causal"])
    g = torch.Generator().manual_seed(8192)
    do = torch.randn(tuple(case.q.shape), generator=g).to(case.q.dtype)
    assert case.scale == case.D ** -0.5  # the binding's default scale
    dq, dk, dv = _run_packed(case.q, case.k, case.v, do, case.cu_seqlens_q,
                             case.cu_seqlens_k, True)
    refs = oracle.attention_bwd(case.q, case.k, case.v, do, case.B, case.Hq, case.Hkv, case.Sq,
                                case.Sk, case.D, case.scale, True, case.cu_seqlens_q,
                                case.cu_seqlens_k)
    for n, t, r in zip(("dq", "dk", "dv"), (dq, dk, dv), refs):
        _compare(n, t, r, "fp16")
