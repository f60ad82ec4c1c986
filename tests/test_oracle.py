"""Pins for the fp64 CPU oracle, independent of the oracle's own code.

Each test checks the oracle against something the pages or the mathematics fix:
closed forms, an arbitrary-precision evaluation of the unshifted definition,
numpy brute force, invariances, the worked lazy-rescale example built from the
v1.7 release notes (section 1.2), and the LSE range printed in section 4.6.
A plausible mistake in the oracle (dropped max shift, log2 LSE, missing scale,
wrong causal diagonal, wrong GQA head, wrong packed offset, keep-new-max on a
skip) fails at least one of them.
"""
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
from exact_attention_forward_sm_gb300 import workloads as wl
from tests.helpers import REL_LINF_TOL, cosine, lse_max_abs, rel_linf

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _f64(x):
    return x.float().numpy().astype(np.float64)


def _run(case, **kw):
    return oracle.attention(case.q, case.k, case.v, case.B, case.Hq, case.Hkv,
                            case.Sq, case.Sk, case.D, case.scale, case.causal,
                            case.cu_seqlens_q, case.cu_seqlens_k, **kw)


def _run_online(case, **kw):
    return oracle.attention_online(case.q, case.k, case.v, case.B, case.Hq,
                                   case.Hkv, case.Sq, case.Sk, case.D, case.scale,
                                   case.causal, case.cu_seqlens_q,
                                   case.cu_seqlens_k, **kw)


def _dense_rows(o_rows, case):
    """Reshape LSE-ordered rows back to [B, Hq, Sq, D]."""
    return o_rows.reshape(case.B, case.Hq, case.Sq, case.D)


def _numpy_dense(case):
    """Brute force with numpy: softmax(scale * Q K^T + mask) V per (b, h)."""
    q, k, v = _f64(case.q), _f64(case.k), _f64(case.v)
    g = case.Hq // case.Hkv
    o = np.zeros((case.B, case.Hq, case.Sq, case.D))
    lse = np.zeros((case.B, case.Hq, case.Sq))
    i = np.arange(case.Sq)[:, None]
    j = np.arange(case.Sk)[None, :]
    vis = (j <= i + case.Sk - case.Sq) if case.causal else np.ones((case.Sq, case.Sk), bool)
    for b in range(case.B):
        for h in range(case.Hq):
            s = case.scale * q[b, :, h, :] @ k[b, :, h // g, :].T
            s = np.where(vis, s, -np.inf)
            mx = s.max(axis=1, keepdims=True)
            finite = np.isfinite(mx)
            e = np.where(finite, np.exp(s - np.where(finite, mx, 0.0)), 0.0)
            den = e.sum(axis=1, keepdims=True)
            with np.errstate(invalid="ignore", divide="ignore"):
                o[b, h] = np.where(den > 0, (e @ v[b, :, h // g, :]) / den, 0.0)
                lse[b, h] = np.where(den[:, 0] > 0,
                                     mx[:, 0] + np.log(np.where(den[:, 0] > 0, den[:, 0], 1.0)),
                                     -np.inf)
    return o, lse


# ---------------------------------------------------------------- closed forms

def test_single_key_gives_v_and_lse_is_the_score():
    """One visible key: softmax weight 1, so O = V[key] and LSE = s_00."""
    case = wl.make_case(1, 3, 3, 5, 1, 16, "fp16", causal=False, seed=1)
    o, lse = _run(case)
    o = _dense_rows(o, case)
    q, k, v = _f64(case.q), _f64(case.k), _f64(case.v)
    for h in range(3):
        for i in range(5):
            np.testing.assert_allclose(o[0, h, i], v[0, 0, h], rtol=0, atol=1e-15)
            s = case.scale * math.fsum(q[0, i, h, d] * k[0, 0, h, d] for d in range(16))
            assert abs(lse[h * 5 + i] - s) < 1e-12


def test_causal_row_zero_sees_only_key_zero():
    case = wl.make_case(2, 2, 2, 64, 64, 32, "bf16", causal=True, seed=2)
    o, _ = _run(case)
    o = _dense_rows(o, case)
    v = _f64(case.v)
    for b in range(2):
        for h in range(2):
            np.testing.assert_allclose(o[b, h, 0], v[b, 0, h], rtol=0, atol=1e-15)


@pytest.mark.parametrize("causal", [False, True])
def test_constant_scores_give_mean_of_visible_v(causal):
    """q = 0: all visible scores equal, O = mean of visible V rows, LSE = ln n."""
    S = 200
    case = wl.make_case(1, 2, 1, S, S, 16, "bf16", causal=causal, seed=3, zero_q=True)
    o, lse = _run(case)
    o = _dense_rows(o, case)
    v = _f64(case.v)[0, :, 0, :]
    for h in range(2):
        for i in (0, 1, 77, S - 1):
            n = i + 1 if causal else S
            np.testing.assert_allclose(o[0, h, i], v[:n].mean(axis=0), rtol=1e-12, atol=1e-14)
            assert abs(lse[h * S + i] - math.log(n)) < 1e-12


def test_unshifted_definition_in_arbitrary_precision():
    """O and LSE against exp(s_j) evaluated without any max shift at 50 digits."""
    mp = pytest.importorskip("mpmath")
    mp.mp.dps = 50
    case = wl.make_case(1, 2, 2, 7, 9, 8, "fp16", causal=True, seed=4, sigma=3.0)
    o, lse = _run(case)
    o = _dense_rows(o, case)
    q, k, v = _f64(case.q), _f64(case.k), _f64(case.v)
    for h in range(2):
        for i in range(7):
            n = min(9, i + 9 - 7 + 1)
            w = [mp.e ** (mp.mpf(case.scale) * mp.fsum(mp.mpf(q[0, i, h, d]) * mp.mpf(k[0, j, h, d])
                                                      for d in range(8))) for j in range(n)]
            z = mp.fsum(w)
            assert abs(float(mp.log(z)) - lse[h * 7 + i]) < 1e-12
            for d in range(8):
                ref = mp.fsum(w[j] * mp.mpf(v[0, j, h, d]) for j in range(n)) / z
                assert abs(float(ref) - o[0, h, i, d]) < 1e-12


def test_lse_range_matches_printed_probe_natural_log():
    """The printed LSE range for [2, 8, 512] (v1.7 notes, section 4.6)."""
    g = json.load(open(os.path.join(GOLDEN, "lse_natural_log_s512.json")))
    B, H, S = g["printed"]["shape"]
    case = wl.make_case(B, H, H, S, S, g["D"], "fp16", causal=g["causal"], seed=5,
                        zero_q=True)
    _, lse = _run(case)
    # constant scores: LSE_i = ln(i + 1) exactly, spanning [0, ln 512]
    assert abs(lse.max() - g["ln_512"]) < 1e-12
    assert abs(lse.min()) < 1e-12
    # the printed range brackets the natural-log reading and excludes base 2
    assert abs(lse.max() - g["printed"]["lse_max"]) < 0.01
    assert abs(lse.min() - g["printed"]["lse_min"]) < 0.05
    assert abs(math.log2(S) - g["printed"]["lse_max"]) > 2.0


# ------------------------------------------------------------------ invariance

def test_row_constant_shift_leaves_o_and_moves_lse():
    """Adding c_i to every score of row i keeps O and adds c_i to LSE."""
    D = 16
    base = wl.make_case(1, 1, 1, 33, 47, D, "bf16", causal=True, seed=6)
    base.q[..., D - 1] = 0
    base.k[..., D - 1] = 0
    shifted = wl.make_case(1, 1, 1, 33, 47, D, "bf16", causal=True, seed=6)
    shifted.q = base.q.clone().float()
    shifted.k = base.k.clone().float()
    shifted.v = base.v.clone().float()
    c = torch.linspace(-20.0, 30.0, 33, dtype=torch.float64)
    shifted.q[0, :, 0, D - 1] = (c / base.scale).float()
    shifted.k[..., D - 1] = 1.0
    c = shifted.q[0, :, 0, D - 1].double().numpy() * base.scale  # exact float32 c_i
    o0, lse0 = _run(base)
    o1, lse1 = _run(shifted)
    np.testing.assert_allclose(o1, o0, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(lse1 - lse0, c, rtol=0, atol=1e-12)


# ----------------------------------------------------------------- brute force

@pytest.mark.parametrize("shape", [
    # B, Hq, Hkv, Sq, Sk, D, causal
    (1, 1, 1, 17, 17, 8, False),
    (2, 3, 3, 40, 40, 16, True),
    (1, 4, 2, 31, 50, 8, True),     # Sq < Sk: bottom-right diagonal
    (1, 2, 1, 50, 31, 8, True),     # Sq > Sk: first 19 rows see no key
    (2, 8, 2, 20, 20, 16, False),   # GQA 4:1
])
def test_matches_numpy_brute_force(shape):
    B, Hq, Hkv, Sq, Sk, D, causal = shape
    case = wl.make_case(B, Hq, Hkv, Sq, Sk, D, "fp16", causal=causal, seed=7, sigma=2.0)
    o, lse = _run(case)
    o_ref, lse_ref = _numpy_dense(case)
    np.testing.assert_allclose(_dense_rows(o, case), o_ref, rtol=1e-10, atol=1e-12)
    lse = lse.reshape(B, Hq, Sq)
    assert np.array_equal(np.isneginf(lse), np.isneginf(lse_ref))
    fin = np.isfinite(lse_ref)
    np.testing.assert_allclose(lse[fin], lse_ref[fin], rtol=0, atol=1e-10)


def test_fully_masked_rows_are_zero_with_neg_inf_lse():
    case = wl.make_case(1, 1, 1, 10, 4, 8, "bf16", causal=True, seed=8)
    o, lse = _run(case)
    # row i sees keys j <= i - 6, so rows 0..5 see nothing
    assert np.all(o[:6] == 0.0) and np.all(np.isneginf(lse[:6]))
    assert np.all(np.isfinite(lse[6:]))


def test_gqa_equals_repeated_kv_heads():
    case = wl.make_case(2, 6, 2, 24, 24, 16, "bf16", causal=True, seed=9)
    o, lse = _run(case)
    rep = wl.make_case(2, 6, 6, 24, 24, 16, "bf16", causal=True, seed=9)
    rep.q, rep.k, rep.v = case.q, case.k.repeat_interleave(3, dim=2), case.v.repeat_interleave(3, dim=2)
    o2, lse2 = _run(rep)
    np.testing.assert_array_equal(o, o2)
    np.testing.assert_array_equal(lse, lse2)


def test_packed_sequences_equal_separate_dense_problems():
    lens_q, lens_k = [5, 1, 130, 64], [9, 1, 130, 70]
    case = wl.make_case(0, 4, 2, 0, 0, 16, "fp16", causal=True, seed=10,
                        seqlens_q=lens_q, seqlens_k=lens_k)
    o, lse = _run(case)
    cq, ck = case.cu_seqlens_q.tolist(), case.cu_seqlens_k.tolist()
    total_q = case.Sq
    for b in range(4):
        sub = wl.make_case(1, 4, 2, lens_q[b], lens_k[b], 16, "fp16", causal=True, seed=0)
        sub.q = case.q[cq[b]:cq[b + 1]].unsqueeze(0)
        sub.k = case.k[ck[b]:ck[b + 1]].unsqueeze(0)
        sub.v = case.v[ck[b]:ck[b + 1]].unsqueeze(0)
        o_ref, lse_ref = _numpy_dense(sub)
        for h in range(4):
            rows = h * total_q + np.arange(cq[b], cq[b + 1])
            np.testing.assert_allclose(o[rows], o_ref[0, h], rtol=1e-10, atol=1e-12)
            np.testing.assert_allclose(lse[rows], lse_ref[0, h], rtol=0, atol=1e-10)


def test_row_subset_matches_full_run():
    case = wl.make_case(2, 4, 4, 70, 70, 16, "bf16", causal=True, seed=11)
    o, lse = _run(case)
    rows = np.array([0, 69, 70, 139, 300, 559], dtype=np.int64)
    o_s, lse_s = _run(case, rows=rows)
    np.testing.assert_array_equal(o_s, o[rows])
    np.testing.assert_array_equal(lse_s, lse[rows])


# ------------------------------------------------ online restatement (lazy rescale)

def _worked_example():
    g = json.load(open(os.path.join(GOLDEN, "lazy_rescale_worked_example.json")))
    bn = g["block_n"]
    scale = g["scale"]
    b = np.repeat(np.array(g["block_log2_score"]), bn)
    n = b.size
    case = wl.make_case(1, 1, 1, 1, n, 2, "bf16", causal=False, seed=12, scale=scale)
    case.q = torch.tensor([[[[1.0, 0.0]]]], dtype=torch.float32)
    k = torch.zeros(1, n, 1, 2, dtype=torch.float64)
    k[0, :, 0, 0] = torch.from_numpy(b * math.log(2.0) / scale)
    case.k = k.float()
    case.v = torch.randn(1, n, 1, 2, generator=torch.Generator().manual_seed(3))
    return g, case


@pytest.mark.parametrize("variant,threshold,lagging", [
    ("threshold_8_lagging", 8.0, True),
    ("threshold_8_keep_new_max", 8.0, False),
    ("threshold_0_lagging", 0.0, True),
])
def test_worked_lazy_rescale_example(variant, threshold, lagging):
    g, case = _worked_example()
    o_ref, lse_ref = _run(case)
    o, lse, st = _run_online(case, block_n=g["block_n"], threshold=threshold, lagging=lagging)
    exp = g["expected"][variant]
    assert st["skips"] == exp["skips"] and st["rescales"] == exp["rescales"]
    assert abs(st["max_p"] - exp["max_p"]) <= 1e-5 * exp["max_p"]
    if lagging:
        np.testing.assert_allclose(o, o_ref, rtol=1e-12, atol=1e-13)
        assert abs(lse[0] - lse_ref[0]) < 1e-12
    else:
        # keep-new-max leaves block 0 on a stale base: a 2^7.99-fold overweight
        assert rel_linf(o, o_ref) > 1e-2


def _bias_case(seed, S=1024, D=32, causal=True):
    return wl.make_case(1, 2, 1, S, S, D, "bf16", causal=causal, seed=seed, rising_bias=True)


@pytest.mark.parametrize("seed", [20, 21, 22])
@pytest.mark.parametrize("kind", ["random", "rising_bias", "sigma2_noncausal"])
def test_naive_equals_online_threshold_0_and_8(seed, kind):
    if kind == "random":
        case = wl.make_case(1, 2, 2, 300, 300, 16, "fp16", causal=True, seed=seed)
    elif kind == "rising_bias":
        case = _bias_case(seed, S=300, D=16)
    else:
        case = wl.make_case(1, 2, 1, 280, 290, 16, "bf16", causal=False, seed=seed,
                            sigma=math.sqrt(2.0))
    o_n, lse_n = _run(case)
    for threshold in (0.0, 8.0):
        o, lse, st = _run_online(case, block_n=16, threshold=threshold, lagging=True)
        np.testing.assert_allclose(o, o_n, rtol=1e-12, atol=1e-12)
        np.testing.assert_allclose(lse, lse_n, rtol=1e-12, atol=1e-12)
        assert st["max_p"] <= 256.0
        if threshold == 8.0:
            assert st["skips"] > 0


def test_rising_bias_workload_exercises_skip_and_rescale():
    """The rising-bias recipe gives both skipped and performed rescales with the
    128-key blocks walked in ascending order; P stays <= 256 (v1.7 notes 1.2)."""
    case = _bias_case(23, S=4096, D=32)
    rows = oracle.row_index_dense(0, 0, np.arange(0, 4096, 97), case.Hq, case.Sq)
    o_n, lse_n = _run(case, rows=rows)
    o, lse, st = _run_online(case, rows=rows, block_n=128, threshold=8.0, lagging=True)
    assert st["skips"] > 0 and st["rescales"] > 0
    assert 1.0 < st["max_p"] <= 256.0
    np.testing.assert_allclose(o, o_n, rtol=1e-11, atol=1e-12)
    np.testing.assert_allclose(lse, lse_n, rtol=1e-12, atol=1e-9)


def test_rising_bias_named_workload_exercises_skip_and_rescale():
    """The named rising-bias workload itself (B2 Hq32 Hkv8 S4096 D128 bf16
    causal, its bias carried in bf16 channel D-1) gives both outcomes of the
    threshold-8 decision, walked in ascending 128-key blocks: a row sample over
    every (batch, head) pair records skipped and performed rescales, P stays
    <= 256 (v1.7 notes 1.2: threshold 8 with lagging bounds P by 2^8), and the
    online path equals the plain definition on those rows."""
    w = wl.BY_NAME["b2_hq32_hkv8_s4096_d128_bf16_causal_risingbias"]
    case = wl.make_workload(w)
    assert (case.B, case.Hq, case.Hkv, case.Sq, case.D, case.dtype) == (2, 32, 8, 4096, 128,
                                                                      "bf16")
    rng = np.random.default_rng(3)
    rows = []
    for b in range(case.B):
        for h in range(case.Hq):
            i = np.unique(np.concatenate([[0, 127, 128, 4095],
                                          rng.integers(0, case.Sq, size=12)]))
            rows.append(oracle.row_index_dense(b, h, i, case.Hq, case.Sq))
    all_rows = np.concatenate(rows)
    o_n, lse_n = _run(case, rows=all_rows)
    o, lse, st = _run_online(case, rows=all_rows, block_n=128, threshold=8.0, lagging=True)
    assert st["skips"] > 0 and st["rescales"] > 0, st
    assert 1.0 < st["max_p"] <= 256.0, st
    np.testing.assert_allclose(o, o_n, rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(lse, lse_n, rtol=1e-12, atol=1e-9)
    # each (batch, head) pair on its own sees both outcomes as well
    for r in rows:
        _, _, st_p = _run_online(case, rows=r, block_n=128, threshold=8.0, lagging=True)
        assert st_p["skips"] > 0 and st_p["rescales"] > 0, (r[:2], st_p)


def test_negative_control_keep_new_max_fails_the_gate():
    """The superseded skip rule (keep the new max) must fail the bf16 gate on
    the rising-bias inputs, so the suite can see the bug max lagging fixes."""
    case = _bias_case(24, S=2048, D=32)
    rows = oracle.row_index_dense(0, 1, np.arange(0, 2048, 13), case.Hq, case.Sq)
    o_n, _ = _run(case, rows=rows)
    o_bad, _, st = _run_online(case, rows=rows, block_n=128, threshold=8.0, lagging=False)
    assert st["skips"] > 0
    assert rel_linf(o_bad, o_n) > REL_LINF_TOL["bf16"]


def test_metrics_detect_a_transposed_or_dropped_term():
    """The gate metrics themselves: a wrong answer must fail them."""
    case = wl.make_case(1, 2, 2, 64, 64, 16, "bf16", causal=True, seed=25)
    o, lse = _run(case)
    assert rel_linf(o, o) == 0.0 and cosine(o, o) == pytest.approx(1.0)
    assert rel_linf(o[::-1], o) > 0.1
    assert lse_max_abs(lse + 2e-3, lse) > 1e-3
