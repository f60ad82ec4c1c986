"""Pins for the oracle's KV-cache path (attention of new tokens over a
contiguous or paged cache, the flash_attn_with_kvcache path run as test 4 of
the fork's v1.7 notes, section 4.1).

The oracle reads the cache through its block table and then applies the
pinned plain definition; these tests fix the addressing and the position
alignment independently: numpy brute force that reads cache rows by (page,
row) in a loop, paged == contiguous, rows past cache_seqlens never read (NaN
there changes nothing), and closed forms (window (0, 0) picks the newest key;
equal scores give ln(number of keys))."""
import math

import numpy as np
import pytest
import torch

import oracle


def _draw(shape, seed, dtype=torch.bfloat16):
    g = torch.Generator().manual_seed(seed)
    return torch.randn(shape, generator=g).to(dtype)


def _f64(x):
    return x.float().numpy().astype(np.float64)


def _brute(q, kc, vc, lens, scale, causal, table=None):
    """Loop over sequences / heads, reading key j from (page, row) explicitly."""
    q, kc, vc = _f64(q), _f64(kc), _f64(vc)
    B, Sq, Hq, D = q.shape
    Hkv = kc.shape[2]
    g = Hq // Hkv
    o = np.zeros((B, Hq, Sq, D))
    lse = np.zeros((B, Hq, Sq))
    for b in range(B):
        lk = int(lens[b])
        for h in range(Hq):
            keys, vals = [], []
            for j in range(lk):
                if table is None:
                    page, r = b, j
                else:
                    page, r = int(table[b, j // kc.shape[1]]), j % kc.shape[1]
                keys.append(kc[page, r, h // g])
                vals.append(vc[page, r, h // g])
            keys = np.array(keys).reshape(lk, D)
            vals = np.array(vals).reshape(lk, D)
            for i in range(Sq):
                pos = i + lk - Sq
                vis = [j for j in range(lk) if (not causal or j <= pos)]
                if not vis:
                    lse[b, h, i] = -np.inf
                    continue
                s = scale * keys[vis] @ q[b, i, h]
                m = s.max()
                w = np.exp(s - m)
                o[b, h, i] = w @ vals[vis] / w.sum()
                lse[b, h, i] = m + math.log(w.sum())
    return o.reshape(-1, D), lse.reshape(-1)


def _close(a, b, tol=1e-12):
    fin = np.isfinite(b)
    assert np.array_equal(np.isfinite(a), fin)
    assert np.max(np.abs(a[fin] - b[fin]), initial=0.0) <= tol * max(1.0, np.max(np.abs(b[fin]), initial=0.0))


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("Sq", [1, 3])
def test_contiguous_cache_brute_force(causal, Sq):
    B, Hq, Hkv, D, cap = 3, 4, 2, 8, 40
    q = _draw((B, Sq, Hq, D), 1)
    kc, vc = _draw((B, cap, Hkv, D), 2), _draw((B, cap, Hkv, D), 3)
    lens = torch.tensor([40, 7, 2], dtype=torch.int32)
    scale = 1 / math.sqrt(D)
    o, l = oracle.attention_kvcache(q, kc, vc, lens, scale, causal)
    ro, rl = _brute(q, kc, vc, lens.numpy(), scale, causal)
    _close(o, ro)
    _close(l, rl)


def test_paged_equals_contiguous_and_brute_force():
    B, Hq, Hkv, D, page_rows, Sq = 2, 4, 1, 8, 16, 2
    lens = np.array([37, 20])
    max_blocks = 3
    contig_k = _draw((B, max_blocks * page_rows, Hkv, D), 4)
    contig_v = _draw((B, max_blocks * page_rows, Hkv, D), 5)
    rng = np.random.default_rng(0)
    num_pages = 9
    perm = rng.permutation(num_pages)[:B * max_blocks].reshape(B, max_blocks)
    pk = torch.full((num_pages, page_rows, Hkv, D), float("nan"), dtype=torch.bfloat16)
    pv = pk.clone()
    for b in range(B):
        for blk in range(max_blocks):
            pk[perm[b, blk]] = contig_k[b, blk * page_rows:(blk + 1) * page_rows]
            pv[perm[b, blk]] = contig_v[b, blk * page_rows:(blk + 1) * page_rows]
    q = _draw((B, Sq, Hq, D), 6)
    scale = 0.3
    oc, lc = oracle.attention_kvcache(q, contig_k, contig_v, lens, scale, True)
    op, lp = oracle.attention_kvcache(q, pk, pv, lens, scale, True, block_table=perm)
    assert np.array_equal(oc, op) and np.array_equal(lc, lp)
    ro, rl = _brute(q, pk, pv, lens, scale, True, table=perm)
    _close(op, ro)
    _close(lp, rl)


def test_rows_past_cache_seqlens_are_never_read():
    B, Hq, Hkv, D, cap = 2, 2, 2, 8, 30
    q = _draw((B, 1, Hq, D), 7)
    kc, vc = _draw((B, cap, Hkv, D), 8), _draw((B, cap, Hkv, D), 9)
    lens = torch.tensor([11, 30], dtype=torch.int32)
    o0, l0 = oracle.attention_kvcache(q, kc, vc, lens, 0.35, False)
    kc[0, 11:] = float("nan")
    vc[0, 11:] = float("inf")
    o1, l1 = oracle.attention_kvcache(q, kc, vc, lens, 0.35, False)
    assert np.array_equal(o0, o1) and np.array_equal(l0, l1)


def test_window_00_decode_picks_the_newest_key():
    B, Hq, Hkv, D, cap = 3, 4, 4, 8, 25
    q = _draw((B, 1, Hq, D), 10)
    kc, vc = _draw((B, cap, Hkv, D), 11), _draw((B, cap, Hkv, D), 12)
    lens = np.array([25, 1, 13])
    o, l = oracle.attention_kvcache(q, kc, vc, lens, 0.5, True, window_left=0, window_right=0)
    want_o = np.stack([_f64(vc)[b, lens[b] - 1, h] for b in range(B) for h in range(Hq)])
    want_l = np.array([0.5 * _f64(q)[b, 0, h] @ _f64(kc)[b, lens[b] - 1, h]
                       for b in range(B) for h in range(Hq)])
    assert np.array_equal(o, want_o)
    _close(l, want_l, 1e-13)


def test_equal_scores_give_log_of_key_count():
    B, Hq, Hkv, D, cap, Sq = 2, 2, 1, 8, 50, 4
    q = torch.zeros((B, Sq, Hq, D), dtype=torch.bfloat16)
    kc, vc = _draw((B, cap, Hkv, D), 13), _draw((B, cap, Hkv, D), 14)
    lens = np.array([50, 9])
    o, l = oracle.attention_kvcache(q, kc, vc, lens, 0.5, True)
    want = []
    for b in range(B):
        for h in range(Hq):
            for i in range(Sq):
                want.append(math.log(i + lens[b] - Sq + 1))
    _close(l, np.array(want), 1e-13)
    # O = mean of the visible V rows
    o = o.reshape(B, Hq, Sq, D)
    for b in range(B):
        for i in range(Sq):
            n = i + lens[b] - Sq + 1
            assert np.allclose(o[b, 0, i], _f64(vc)[b, :n, 0].mean(axis=0), atol=1e-13)
