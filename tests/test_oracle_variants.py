"""Pins for the oracle's score variants: local window, tanh soft cap, ALiBi.

The fork's v1.7 release notes list these next to the plain forward (section 2,
"Public APIs") and validate them in section 4.1 (tests 5-7) and section 4.6
(window (0, 0) gives O = V exactly; softcap with causal stays finite).  Each
test below checks the oracle against a closed form, an invariance that maps a
variant onto the already-pinned plain definition, or numpy brute force on tiny
inputs, so that a wrong sign, a wrong distance origin (top-left instead of
bottom-right), the soft cap applied before the scale, an off-by-one window
edge or a slope taken per K/V head fails at least one of them.
"""
import json
import math
import os

import numpy as np
import pytest
import torch
from scipy.special import logsumexp

import oracle
from exact_attention_forward_sm_gb300 import workloads as wl

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _f64(x):
    return x.float().numpy().astype(np.float64)


def _run(case, **kw):
    return oracle.attention(case.q, case.k, case.v, case.B, case.Hq, case.Hkv,
                            case.Sq, case.Sk, case.D, case.scale, case.causal,
                            case.cu_seqlens_q, case.cu_seqlens_k, **kw)


def _numpy_variant(case, wl_=-1, wr_=-1, softcap=0.0, slopes=None):
    """Brute force per (b, h): mask built from numpy's triangle helpers, scores
    from a dense matrix product, softmax via scipy's logsumexp."""
    q, k, v = _f64(case.q), _f64(case.k), _f64(case.v)
    g = case.Hq // case.Hkv
    out_o, out_l = [], []
    seqs = case.seq_lengths()
    cq = [0] + list(np.cumsum([a for a, _ in seqs]))
    ck = [0] + list(np.cumsum([b for _, b in seqs]))
    per = []
    for b, (lq, lk) in enumerate(seqs):
        off = lk - lq
        ones = np.ones((lq, lk), bool)
        vis = ones.copy()
        if case.causal:
            vis &= np.tril(ones, off)
        if wl_ >= 0:
            vis &= np.triu(ones, off - wl_)
        if wr_ >= 0:
            vis &= np.tril(ones, off + wr_)
        # |diag - j| with diag = i + off
        dist = np.abs(np.subtract.outer(np.arange(lq) + off, np.arange(lk)))
        for h in range(case.Hq):
            if case.varlen:
                qh = q[cq[b]:cq[b + 1], h, :]
                kh = k[ck[b]:ck[b + 1], h // g, :]
                vh = v[ck[b]:ck[b + 1], h // g, :]
            else:
                qh, kh, vh = q[b, :, h, :], k[b, :, h // g, :], v[b, :, h // g, :]
            s = case.scale * qh @ kh.T
            if softcap > 0:
                s = softcap * np.tanh(s / softcap)
            if slopes is not None:
                s = s - slopes[h] * dist
            s = np.where(vis, s, -np.inf)
            lse = logsumexp(s, axis=1) if lk > 0 else np.full(lq, -np.inf)
            w = np.where(np.isfinite(lse)[:, None], np.exp(s - lse[:, None]), 0.0)
            per.append((b, h, w @ vh, lse))
    # LSE-index order: dense (b, h, i); packed (h, token)
    if case.varlen:
        for h in range(case.Hq):
            for b in range(case.B):
                _, _, o, l = per[b * case.Hq + h]
                out_o.append(o)
                out_l.append(l)
    else:
        for _, _, o, l in per:
            out_o.append(o)
            out_l.append(l)
    return np.concatenate(out_o), np.concatenate(out_l)


def _close(a, b, tol=1e-12):
    a, b = np.asarray(a), np.asarray(b)
    fin = np.isfinite(b)
    assert np.array_equal(np.isfinite(a), fin)
    assert np.array_equal(a[~fin], b[~fin])
    if fin.any():
        assert np.max(np.abs(a[fin] - b[fin])) <= tol * max(1.0, np.max(np.abs(b[fin])))


# ------------------------------------------------------------------- window

def test_window_00_output_equals_v_golden():
    gold = json.load(open(os.path.join(GOLDEN, "window_00_output_equals_v.json")))
    wlft, wrgt = gold["window"]
    for causal in (False, True):
        for softcap in (0.0, gold["softcap_checked"]):
            c = wl.make_case(2, 4, 2, 37, 37, 16, "bf16", causal, seed=11)
            o, lse = _run(c, window_left=wlft, window_right=wrgt, softcap=softcap)
            v = _f64(c.v)                                    # [B, S, Hkv, D]
            want = np.stack([v[b, :, h // 2, :] for b in range(2) for h in range(4)])
            assert np.max(np.abs(o - want.reshape(-1, 16))) == gold["expected_max_abs_diff"]
            q, k = _f64(c.q), _f64(c.k)
            s = np.stack([np.einsum("id,id->i", q[b, :, h, :], k[b, :, h // 2, :])
                          for b in range(2) for h in range(4)]).reshape(-1) * c.scale
            if softcap:
                s = softcap * np.tanh(s / softcap)
            _close(lse, s, 1e-13)


def test_window_unbounded_and_causal_equivalences():
    c = wl.make_case(1, 2, 2, 50, 70, 16, "fp16", False, seed=12)
    base_o, base_l = _run(c)
    for wlft, wrgt in ((-1, -1), (70, 70), (1000, -5)):
        o, l = _run(c, window_left=wlft, window_right=wrgt)
        _close(o, base_o, 1e-15)
        _close(l, base_l, 1e-15)
    # right edge 0 on a non-causal problem is the bottom-right causal mask
    cc = wl.make_case(1, 2, 2, 50, 70, 16, "fp16", True, seed=12)
    co, cl = _run(cc)
    o, l = _run(c, window_right=0)
    _close(o, co, 1e-15)
    _close(l, cl, 1e-15)


@pytest.mark.parametrize("sq,sk", [(33, 33), (20, 45), (45, 20)])
@pytest.mark.parametrize("win", [(3, 5), (0, 7), (10, 0), (2, -1), (-1, 4), (0, 0)])
@pytest.mark.parametrize("causal", [False, True])
def test_window_brute_force(sq, sk, win, causal):
    c = wl.make_case(1, 2, 1, sq, sk, 8, "bf16", causal, seed=13 + sq + sk)
    o, l = _run(c, window_left=win[0], window_right=win[1])
    ro, rl = _numpy_variant(c, *win)
    _close(o, ro)
    _close(l, rl)


def test_window_packed_sequences_brute_force():
    c = wl.make_case(0, 3, 3, 0, 0, 8, "fp16", True, seed=14,
                     seqlens_q=[5, 40, 1, 17], seqlens_k=[9, 33, 20, 17])
    o, l = _run(c, window_left=6, window_right=2)
    ro, rl = _numpy_variant(c, 6, 2)
    _close(o, ro)
    _close(l, rl)


def test_window_row_without_keys_is_zero():
    # Sq > Sk non-causal with window (0, 0): rows whose diagonal i + Sk - Sq is
    # negative see no key at all
    c = wl.make_case(1, 1, 1, 12, 4, 8, "bf16", False, seed=15)
    o, l = _run(c, window_left=0, window_right=0)
    assert np.all(o[:8] == 0) and np.all(np.isneginf(l[:8]))
    assert np.all(np.isfinite(l[8:]))


# ------------------------------------------------------------------ softcap

def test_softcap_large_cap_is_plain():
    c = wl.make_case(1, 2, 2, 40, 40, 16, "bf16", True, seed=16, sigma=2.0)
    o0, l0 = _run(c)
    o, l = _run(c, softcap=1e9)
    _close(o, o0, 1e-13)
    _close(l, l0, 1e-13)


def test_softcap_identical_keys_closed_form():
    """All keys equal: every visible score of row i is the same s_i, so the
    weights are uniform: O = mean of the visible V rows and
    LSE = c tanh(s_i / c) + ln n_i."""
    c = wl.make_case(1, 1, 1, 30, 30, 8, "fp16", True, seed=17, sigma=3.0)
    c.k[:] = c.k[0, 0].clone()
    cap = 5.0
    o, l = _run(c, softcap=cap)
    q, k, v = _f64(c.q)[0, :, 0], _f64(c.k)[0, 0, 0], _f64(c.v)[0, :, 0]
    s = c.scale * q @ k
    n = np.arange(1, 31)
    _close(l, cap * np.tanh(s / cap) + np.log(n), 1e-13)
    _close(o, np.cumsum(v, axis=0) / n[:, None], 1e-13)


def test_softcap_saturates_and_bounds_lse():
    # scores far above the cap: every capped score is c, so LSE -> c + ln n
    c = wl.make_case(1, 1, 1, 16, 16, 8, "bf16", True, seed=18)
    c.k[:] = 1.0
    c.q[:] = 64.0
    cap = 2.0
    _, l = _run(c, softcap=cap)
    _close(l, cap + np.log(np.arange(1, 17)), 1e-12)
    # any input: |capped score| <= c, so ln n - c <= LSE <= ln n + c
    c = wl.make_case(1, 2, 2, 40, 40, 16, "bf16", False, seed=19, sigma=4.0)
    _, l = _run(c, softcap=cap)
    assert np.all(l <= math.log(40) + cap + 1e-12)
    assert np.all(l >= math.log(40) - cap - 1e-12)


@pytest.mark.parametrize("causal", [False, True])
def test_softcap_brute_force(causal):
    c = wl.make_case(2, 4, 2, 27, 35, 8, "bf16", causal, seed=20, sigma=3.0)
    o, l = _run(c, softcap=3.0)
    ro, rl = _numpy_variant(c, softcap=3.0)
    _close(o, ro)
    _close(l, rl)


# -------------------------------------------------------------------- ALiBi

def _geometric(a, n):
    """sum_{d=0}^{n-1} exp(-a d) in closed form."""
    return (1.0 - np.exp(-a * n)) / (1.0 - np.exp(-a))


@pytest.mark.parametrize("causal", [False, True])
def test_alibi_equal_scores_geometric_closed_form(causal):
    """q = 0: every score is 0, the weights are exp(-slope |i - j|), and
    LSE_i is a geometric series: causal sum_{d=0}^{i}; non-causal the two
    one-sided series around the diagonal."""
    S = 33
    c = wl.make_case(1, 2, 2, S, S, 8, "bf16", causal, seed=21, zero_q=True)
    slopes = np.array([0.5, 0.0625])
    _, l = _run(c, alibi_slopes=slopes)
    i = np.arange(S)
    want = []
    for a in slopes:
        if causal:
            want.append(np.log(_geometric(a, i + 1)))
        else:
            want.append(np.log(_geometric(a, i + 1) + _geometric(a, S - i) - 1.0))
    _close(l, np.concatenate(want), 1e-13)


def test_alibi_zero_slope_is_plain():
    c = wl.make_case(1, 2, 1, 30, 40, 16, "fp16", True, seed=22)
    o0, l0 = _run(c)
    o, l = _run(c, alibi_slopes=np.zeros(2))
    _close(o, o0, 0)
    _close(l, l0, 0)


@pytest.mark.parametrize("sq,sk", [(24, 24), (10, 31)])
def test_alibi_causal_equals_plain_with_linear_key_bias(sq, sk):
    """Under the causal mask -slope (diag - j) = slope j - slope diag: the same
    attention as a plain problem whose channel D-1 adds slope * j to every
    score, with LSE lower by slope * diag.  scale = 1 and slope = 1/4 keep every
    input exact in float32."""
    D, slope = 8, 0.25
    c = wl.make_case(1, 1, 1, sq, sk, D, "fp16", True, seed=23, scale=1.0)
    c.q[..., D - 1] = 0
    c.k[..., D - 1] = 0
    o_a, l_a = _run(c, alibi_slopes=np.array([slope]))
    c2 = wl.make_case(1, 1, 1, sq, sk, D, "fp16", True, seed=23, scale=1.0)
    c2.q[..., D - 1] = 1.0
    c2.k[0, :, 0, D - 1] = slope * torch.arange(sk, dtype=torch.float32)
    c2.v.copy_(c.v)
    c2.q[..., :D - 1] = c.q[..., :D - 1]
    c2.k[..., :D - 1] = c.k[..., :D - 1]
    o_p, l_p = _run(c2)
    diag = np.arange(sq) + sk - sq
    _close(o_a, o_p, 1e-13)
    _close(l_a, l_p - slope * diag, 1e-13)


@pytest.mark.parametrize("causal", [False, True])
def test_alibi_per_query_head_brute_force(causal):
    c = wl.make_case(2, 4, 2, 21, 29, 8, "bf16", causal, seed=24)
    slopes = np.array([0.7, 0.3, 0.11, 0.02])
    o, l = _run(c, alibi_slopes=slopes)
    ro, rl = _numpy_variant(c, slopes=slopes)
    _close(o, ro)
    _close(l, rl)


def test_all_variants_together_brute_force():
    c = wl.make_case(0, 4, 2, 0, 0, 8, "bf16", True, seed=25, sigma=2.5,
                     seqlens_q=[30, 3, 47], seqlens_k=[41, 3, 47])
    slopes = np.array([0.2, 0.05, 0.4, 0.01])
    o, l = _run(c, window_left=9, window_right=3, softcap=4.0, alibi_slopes=slopes)
    ro, rl = _numpy_variant(c, 9, 3, 4.0, slopes)
    _close(o, ro)
    _close(l, rl)
