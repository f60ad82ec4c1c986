"""Pins of the backward oracle (``oracle.attention_bwd``) to things other than
itself.

The fork's v1.7 release notes validate a backward pass (section 4.4: finite
gradients at S = 2048 causal, gradients against an fp32 reference, varlen
gradients finite); the oracle computes the gradients of the plain definition
of attention.  Here they are checked against:

* finite differences of the FORWARD oracle (an independent code path that is
  pinned by its own tests): L = sum dO * O, central differences at two step
  sizes combined by Richardson extrapolation, on inputs that are exact
  multiples of 2^-9 so every perturbed input is exact in fp32;
* closed forms: a single key (P = 1: dV = sum of dO over the rows that see
  it, dQ = dK = 0); zero queries (uniform P: dV_j = sum_i dO_i / n, dK = 0);
* invariants: sum_j dS_ij = 0 for every row, hence sum_j dK_j = 0, and
  sum_j dV_j = sum of dO over rows with at least one visible key;
* GQA: the gradients of a 2:1 grouped problem equal those of the same
  problem with K/V replicated per query head, summed over each group.
"""
import numpy as np
import pytest

import oracle


def _grid(rng, shape, step=2.0 ** -9, lim=2.0):
    """Random values that are exact multiples of ``step`` (exact in fp32)."""
    x = rng.uniform(-lim, lim, size=shape)
    return (np.round(x / step) * step).astype(np.float32)


def _loss(q, k, v, do, B, Hq, Hkv, Sq, Sk, D, scale, causal, cu_q=None, cu_k=None):
    o, _ = oracle.attention(q, k, v, B, Hq, Hkv, Sq, Sk, D, scale, causal, cu_q, cu_k)
    # o rows are in LSE-index order; reorder dO the same way
    return float(np.sum(o * _rows_of(do, B, Hq, Sq, D, cu_q)))


def _rows_of(x, B, Hq, Sq, D, cu_q):
    """[tokens, Hq, D] (or [B, Sq, Hq, D]) -> rows in LSE-index order."""
    if cu_q is None:
        return x.reshape(B, Sq, Hq, D).transpose(0, 2, 1, 3).reshape(-1, D).astype(np.float64)
    return x.transpose(1, 0, 2).reshape(-1, D).astype(np.float64)


def _finite_diff(which, args, kw):
    q, k, v, do = args
    arrs = {"q": q, "k": k, "v": v}
    base = arrs[which]
    grad = np.zeros(base.shape, dtype=np.float64)
    flat = base.reshape(-1)
    for idx in range(flat.size):
        est = []
        for e in (2.0 ** -7, 2.0 ** -8):
            vals = []
            for sgn in (1.0, -1.0):
                pert = flat.copy()
                pert[idx] = np.float32(flat[idx] + sgn * e)
                a = dict(arrs)
                a[which] = pert.reshape(base.shape)
                vals.append(_loss(a["q"], a["k"], a["v"], do, **kw))
            est.append((vals[0] - vals[1]) / (2 * e))
        # Richardson: (4 f(e/2) - f(e)) / 3 cancels the e^2 term
        grad.reshape(-1)[idx] = (4 * est[1] - est[0]) / 3
    return grad


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("Hq,Hkv,Sq,Sk", [(2, 1, 5, 7), (2, 2, 6, 4), (4, 2, 3, 3)])
def test_gradients_match_finite_differences_of_the_forward(causal, Hq, Hkv, Sq, Sk):
    rng = np.random.default_rng(Hq * 100 + Sq * 10 + Sk + int(causal))
    B, D, scale = 1, 4, 0.7
    q, k, v = _grid(rng, (B, Sq, Hq, D)), _grid(rng, (B, Sk, Hkv, D)), _grid(rng, (B, Sk, Hkv, D))
    do = _grid(rng, (B, Sq, Hq, D))
    kw = dict(B=B, Hq=Hq, Hkv=Hkv, Sq=Sq, Sk=Sk, D=D, scale=scale, causal=causal)
    dq, dk, dv = oracle.attention_bwd(q, k, v, do, B, Hq, Hkv, Sq, Sk, D, scale, causal)
    for name, g in (("q", dq), ("k", dk), ("v", dv)):
        fd = _finite_diff(name, (q, k, v, do), kw)
        err = np.max(np.abs(fd - g))
        assert err <= 1e-6 * max(1.0, np.max(np.abs(g))), (name, err)


def test_gradients_match_finite_differences_packed():
    """Two packed sequences of different lengths, causal, GQA 2:1."""
    rng = np.random.default_rng(11)
    Hq, Hkv, D, scale = 2, 1, 4, 0.5
    cu_q = np.array([0, 3, 7], np.int32)
    cu_k = np.array([0, 4, 9], np.int32)
    tq, tk = int(cu_q[-1]), int(cu_k[-1])
    q, k, v = _grid(rng, (tq, Hq, D)), _grid(rng, (tk, Hkv, D)), _grid(rng, (tk, Hkv, D))
    do = _grid(rng, (tq, Hq, D))
    kw = dict(B=2, Hq=Hq, Hkv=Hkv, Sq=tq, Sk=tk, D=D, scale=scale, causal=True,
              cu_q=cu_q, cu_k=cu_k)
    dq, dk, dv = oracle.attention_bwd(q, k, v, do, 2, Hq, Hkv, tq, tk, D, scale, True,
                                      cu_q, cu_k)
    for name, g in (("q", dq), ("k", dk), ("v", dv)):
        fd = _finite_diff(name, (q, k, v, do), kw)
        assert np.max(np.abs(fd - g)) <= 1e-6 * max(1.0, np.max(np.abs(g))), name


@pytest.mark.parametrize("causal", [False, True])
def test_single_key_closed_form(causal):
    """One key: P = 1 for every row that sees it, so dV = sum of those rows'
    dO (over the group's heads too), and dS = 0 gives dQ = dK = 0."""
    rng = np.random.default_rng(3)
    B, Hq, Hkv, Sq, Sk, D = 2, 4, 2, 5, 1, 8
    q, k, v = (rng.standard_normal(s).astype(np.float32)
               for s in ((B, Sq, Hq, D), (B, Sk, Hkv, D), (B, Sk, Hkv, D)))
    do = rng.standard_normal((B, Sq, Hq, D)).astype(np.float32)
    dq, dk, dv = oracle.attention_bwd(q, k, v, do, B, Hq, Hkv, Sq, Sk, D, 0.3, causal)
    assert np.max(np.abs(dq)) < 1e-12 and np.max(np.abs(dk)) < 1e-12
    # causal, bottom-right aligned: only the last query row sees key 0
    rows = slice(Sq - 1, Sq) if causal else slice(0, Sq)
    for b in range(B):
        for g in range(Hkv):
            want = do[b, rows, 2 * g:2 * g + 2].astype(np.float64).sum(axis=(0, 1))
            assert np.allclose(dv[b, 0, g], want, atol=1e-12)


def test_zero_queries_uniform_weights():
    """q = 0: every visible key gets P = 1/n, dK = scale * sum_i dS_ij q_i = 0
    and dV_j = sum_i dO_i / n (non-causal: n = Sk)."""
    rng = np.random.default_rng(4)
    B, Hq, Hkv, Sq, Sk, D = 1, 2, 2, 6, 9, 8
    q = np.zeros((B, Sq, Hq, D), np.float32)
    k, v = (rng.standard_normal((B, Sk, Hkv, D)).astype(np.float32) for _ in range(2))
    do = rng.standard_normal((B, Sq, Hq, D)).astype(np.float32)
    dq, dk, dv = oracle.attention_bwd(q, k, v, do, B, Hq, Hkv, Sq, Sk, D, 0.5, False)
    assert np.max(np.abs(dk)) < 1e-12
    for h in range(Hq):
        want = do[0, :, h].astype(np.float64).sum(axis=0) / Sk
        assert np.allclose(dv[0, :, h], np.broadcast_to(want, (Sk, D)), atol=1e-12)


@pytest.mark.parametrize("causal", [False, True])
def test_row_sums_of_ds_vanish(causal):
    """sum_j dS_ij = sum_j P_ij (dP_ij - sum_k P_ik dP_ik) = 0 for every row, so
    the key gradients sum to zero over the keys; the value gradients sum to
    the upstream gradient of every row with a visible key."""
    rng = np.random.default_rng(5)
    B, Hq, Hkv, Sq, Sk, D = 2, 4, 2, 40, 33, 16
    q, do = (rng.standard_normal((B, Sq, Hq, D)).astype(np.float32) for _ in range(2))
    k, v = (rng.standard_normal((B, Sk, Hkv, D)).astype(np.float32) for _ in range(2))
    dq, dk, dv = oracle.attention_bwd(q, k, v, do, B, Hq, Hkv, Sq, Sk, D, 0.25, causal)
    assert np.max(np.abs(dk.sum(axis=1))) < 1e-10
    seen = np.arange(Sq) + Sk - Sq >= 0 if causal else np.ones(Sq, bool)
    for g in range(Hkv):
        want = do[:, seen][:, :, 2 * g:2 * g + 2].astype(np.float64).sum(axis=(1, 2))
        assert np.allclose(dv[:, :, g].sum(axis=1), want, atol=1e-10)
    if causal:  # rows without a visible key (Sq > Sk) get no gradient
        assert np.all(dq[:, ~seen] == 0.0)


def test_gqa_equals_replicated_heads_summed():
    rng = np.random.default_rng(6)
    B, Hq, Hkv, Sq, Sk, D = 1, 4, 2, 12, 10, 8
    q, do = (rng.standard_normal((B, Sq, Hq, D)).astype(np.float32) for _ in range(2))
    k, v = (rng.standard_normal((B, Sk, Hkv, D)).astype(np.float32) for _ in range(2))
    dq, dk, dv = oracle.attention_bwd(q, k, v, do, B, Hq, Hkv, Sq, Sk, D, 0.35, True)
    kr, vr = np.repeat(k, 2, axis=2), np.repeat(v, 2, axis=2)
    dq1, dk1, dv1 = oracle.attention_bwd(q, kr, vr, do, B, Hq, Hq, Sq, Sk, D, 0.35, True)
    assert np.allclose(dq, dq1, atol=1e-12)
    assert np.allclose(dk, dk1.reshape(B, Sk, Hkv, 2, D).sum(axis=3), atol=1e-12)
    assert np.allclose(dv, dv1.reshape(B, Sk, Hkv, 2, D).sum(axis=3), atol=1e-12)
