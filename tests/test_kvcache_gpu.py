"""GPU parity of attention over a KV cache (``fa_fwd_kvcache``): contiguous
and paged caches, packed GQA heads, several new tokens per sequence, split-KV
and the score variants, against the oracle's KV-cache path.  This is the
flash_attn_with_kvcache path run as test 4 of the fork's v1.7 notes, section
4.1; gates as for the plain path (O rel_Linf <= 2e-2 fp16 / 1e-2 bf16,
cosine >= 0.9995, LSE abs <= 1e-3)."""
import math
import zlib

import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():  # pragma: no cover - collected on CPU machines too
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

import exact_attention_forward_sm_gb300 as fa  # noqa: E402
import oracle  # noqa: E402
from exact_attention_forward_sm_gb300 import workloads as wl  # noqa: E402
from tests.helpers import COSINE_MIN, LSE_ABS_TOL, REL_LINF_TOL, cosine, lse_max_abs, rel_linf  # noqa: E402

DEV = "cuda:0"


@pytest.fixture(scope="module", autouse=True)
def _built():
    from exact_attention_forward_sm_gb300 import _build
    _build.build()
    fa.load_library()


def _seed(*key):
    return zlib.crc32(repr(key).encode()) % 100000


def _draw(shape, dtype, g, sigma=1.0):
    return (torch.randn(shape, generator=g) * sigma).to(wl.DTYPES[dtype])


def make_cache_case(B, Hq, Hkv, Sq, D, dtype, lens, page_rows=None, num_pages=None,
                    capacity=None, seed=0, sigma=1.0):
    """Draw q and a cache; paged when page_rows is given (random page order)."""
    g = torch.Generator().manual_seed(seed)
    q = _draw((B, Sq, Hq, D), dtype, g, sigma)
    lens = torch.tensor(lens, dtype=torch.int32)
    if page_rows is None:
        cap = capacity or max(1, int(lens.max()))
        kc = _draw((B, cap, Hkv, D), dtype, g, sigma)
        vc = _draw((B, cap, Hkv, D), dtype, g)
        return dict(q=q, kc=kc, vc=vc, lens=lens, table=None, page_rows=cap, num_pages=B,
                    max_blocks=1)
    max_blocks = max(1, math.ceil(int(lens.max()) / page_rows))
    num_pages = num_pages or B * max_blocks + 3
    kc = _draw((num_pages, page_rows, Hkv, D), dtype, g, sigma)
    vc = _draw((num_pages, page_rows, Hkv, D), dtype, g)
    perm = torch.randperm(num_pages, generator=g)[:B * max_blocks].reshape(B, max_blocks)
    return dict(q=q, kc=kc, vc=vc, lens=lens, table=perm.to(torch.int32), page_rows=page_rows,
                num_pages=num_pages, max_blocks=max_blocks)


def run_kvcache(c, causal, scale, num_splits=0, window=(-1, -1), softcap=0.0, slopes=None):
    q = c["q"].to(DEV)
    B, Sq, Hq, D = q.shape
    Hkv = c["kc"].shape[2]
    o = torch.full_like(q, float("nan"))
    lse = torch.full((B, Hq, Sq), float("nan"), dtype=torch.float32, device=DEV)
    table = c["table"].to(DEV).contiguous() if c["table"] is not None else None
    st = fa.fa_fwd_kvcache(q, c["kc"].to(DEV), c["vc"].to(DEV), o, lse, B, Hq, Hkv, Sq, D, scale,
                           int(causal), c["lens"].to(DEV), table, c["max_blocks"],
                           c["page_rows"], c["num_pages"], torch.cuda.current_stream(),
                           fa.FA_DTYPE_BF16 if q.dtype == torch.bfloat16 else fa.FA_DTYPE_FP16,
                           window[0], window[1], softcap,
                           slopes.to(DEV) if slopes is not None else None, num_splits)
    assert st == fa.FA_OK, fa.fa_status_string(st)
    dst = fa.fa_get_device_error(torch.cuda.current_stream())
    assert dst == fa.FA_OK, fa.fa_status_string(dst)
    return o, lse


def check_kvcache(c, o, lse, causal, scale, tag, **variants):
    ref_o, ref_l = oracle.attention_kvcache(c["q"], c["kc"], c["vc"], c["lens"], scale, causal,
                                            block_table=c["table"], **variants)
    B, Sq, Hq, D = c["q"].shape
    got_o = o.float().permute(0, 2, 1, 3).reshape(-1, D).cpu().numpy().astype(np.float64)
    got_l = lse.reshape(-1).cpu().numpy()
    assert np.all(np.isfinite(got_o)), f"{tag}: non-finite O"
    dtype = "bf16" if c["q"].dtype == torch.bfloat16 else "fp16"
    m = {"rel_linf": rel_linf(got_o, ref_o), "cosine": cosine(got_o, ref_o),
         "lse_err": lse_max_abs(got_l, ref_l)}
    assert m["rel_linf"] <= REL_LINF_TOL[dtype], f"{tag}: {m}"
    assert m["cosine"] >= COSINE_MIN, f"{tag}: {m}"
    assert m["lse_err"] <= LSE_ABS_TOL, f"{tag}: {m}"
    return m


@pytest.mark.parametrize("Hq,Hkv", [(32, 8), (8, 8), (16, 1), (4, 2)])
@pytest.mark.parametrize("Sq", [1, 5])
@pytest.mark.parametrize("causal", [False, True])
def test_contiguous_cache(Hq, Hkv, Sq, causal):
    D, dtype = 128, "bf16"
    c = make_cache_case(3, Hq, Hkv, Sq, D, dtype, [1500, 333, 129], capacity=1700,
                        seed=_seed(Hq, Hkv, Sq, causal))
    scale = 1 / math.sqrt(D)
    o, lse = run_kvcache(c, causal, scale)
    check_kvcache(c, o, lse, causal, scale, f"contig Hq{Hq} Hkv{Hkv} Sq{Sq}")


@pytest.mark.parametrize("page_rows", [128, 256])
@pytest.mark.parametrize("D,dtype", [(64, "fp16"), (128, "bf16")])
def test_paged_cache(page_rows, D, dtype):
    c = make_cache_case(4, 16, 4, 2, D, dtype, [2000, 1, 700, 256], page_rows=page_rows,
                        seed=_seed(page_rows, D))
    scale = 1 / math.sqrt(D)
    o, lse = run_kvcache(c, True, scale)
    check_kvcache(c, o, lse, True, scale, f"paged {page_rows} D{D}")


def test_tokens_spanning_two_tiles():
    # group 4: 32 tokens per tile, 70 new tokens -> three token blocks
    c = make_cache_case(2, 8, 2, 70, 64, "fp16", [900, 70], capacity=1024, seed=51)
    o, lse = run_kvcache(c, True, 0.125)
    check_kvcache(c, o, lse, True, 0.125, "70 new tokens")


@pytest.mark.parametrize("num_splits", [1, 3, 16])
def test_splits(num_splits):
    c = make_cache_case(2, 8, 8, 1, 128, "bf16", [4000, 1234], page_rows=256, seed=52)
    scale = 1 / math.sqrt(128)
    o, lse = run_kvcache(c, False, scale, num_splits=num_splits)
    check_kvcache(c, o, lse, False, scale, f"splits {num_splits}")


def test_auto_split_plan_fills_the_gpu():
    n, nbytes = fa.fa_kvcache_plan(8, 64, 8, 1, 128, 16384, 0)
    assert n > 1 and nbytes == n * 8 * 64 * 129 * 4
    c = make_cache_case(2, 16, 2, 1, 128, "bf16", [7000, 3000], capacity=8192, seed=58)
    o, lse = run_kvcache(c, True, 0.1, num_splits=0)
    check_kvcache(c, o, lse, True, 0.1, "auto splits")


def test_empty_and_tiny_caches():
    c = make_cache_case(4, 4, 2, 1, 64, "bf16", [0, 1, 2, 127], capacity=200, seed=53)
    o, lse = run_kvcache(c, True, 0.125)
    assert torch.all(o[0] == 0) and torch.all(torch.isneginf(lse[0]))
    check_kvcache(c, o, lse, True, 0.125, "tiny caches")


def _poison_cache_tail(c):
    """Cache rows past each sequence's length (and pages no sequence uses) hold
    NaN keys and Inf values; they must never reach the output."""
    kc, vc, lens = c["kc"].clone(), c["vc"].clone(), c["lens"].tolist()
    if c["table"] is None:
        for b, n in enumerate(lens):
            kc[b, n:] = float("nan")
            vc[b, n:] = float("inf")
    else:
        used = set()
        pr = c["page_rows"]
        for b, n in enumerate(lens):
            for blk in range(c["max_blocks"]):
                pg = int(c["table"][b, blk])
                used.add(pg)
                first = max(0, n - blk * pr)
                if first < pr:
                    kc[pg, first:] = float("nan")
                    vc[pg, first:] = float("inf")
        for pg in range(kc.shape[0]):
            if pg not in used:
                kc[pg] = float("nan")
                vc[pg] = float("-inf")
    c = dict(c)
    c["kc"], c["vc"] = kc, vc
    return c


@pytest.mark.parametrize("paged", [False, True])
@pytest.mark.parametrize("D,dtype", [(64, "fp16"), (128, "bf16")])
def test_cache_rows_past_the_length_hold_nan_and_inf(paged, D, dtype):
    lens = [1500, 333, 129, 1]
    if paged:
        c = make_cache_case(4, 16, 4, 3, D, dtype, lens, page_rows=256, seed=_seed("poison", D))
    else:
        c = make_cache_case(4, 16, 4, 3, D, dtype, lens, capacity=1700, seed=_seed("poison", D))
    c = _poison_cache_tail(c)
    scale = 1 / math.sqrt(D)
    for splits in (1, 3):
        o, lse = run_kvcache(c, True, scale, num_splits=splits)
        check_kvcache(c, o, lse, True, scale, f"poisoned cache tail paged={paged} D{D} s{splits}")


def test_variants_over_paged_cache():
    Hq = 8
    c = make_cache_case(2, Hq, 2, 3, 128, "bf16", [1800, 600], page_rows=128, seed=54,
                        sigma=2.0)
    slopes = wl.alibi_slopes_geometric(Hq)
    scale = 1 / math.sqrt(128)
    o, lse = run_kvcache(c, True, scale, num_splits=2, window=(500, 0), softcap=20.0,
                         slopes=slopes)
    check_kvcache(c, o, lse, True, scale, "paged variants", window_left=500, window_right=0,
                  softcap=20.0, alibi_slopes=slopes)


def test_window_00_decode_returns_newest_value():
    c = make_cache_case(3, 8, 4, 1, 64, "fp16", [300, 1, 129], page_rows=128, seed=55)
    o, _ = run_kvcache(c, True, 0.125, window=(0, 0))
    lens = c["lens"].tolist()
    for b in range(3):
        page = int(c["table"][b, (lens[b] - 1) // 128])
        want = c["vc"][page, (lens[b] - 1) % 128]          # [Hkv, D]
        assert torch.equal(o[b, 0].cpu(), want.repeat_interleave(2, dim=0))


def test_bad_cache_seqlens_and_table_reported():
    c = make_cache_case(2, 4, 4, 1, 64, "bf16", [100, 100], page_rows=128, seed=56)
    q = c["q"].to(DEV)
    o = torch.empty_like(q)
    for lens, table in (([100, 5000], c["table"]), ([100, 100], torch.tensor([[0], [999]]))):
        st = fa.fa_fwd_kvcache(q, c["kc"].to(DEV), c["vc"].to(DEV), o, None, 2, 4, 4, 1, 64,
                               0.125, 0, torch.tensor(lens, dtype=torch.int32, device=DEV),
                               table.to(torch.int32).to(DEV), 1, 128, c["num_pages"],
                               torch.cuda.current_stream(), fa.FA_DTYPE_BF16, num_splits=1)
        assert st == fa.FA_OK
        assert fa.fa_get_device_error(torch.cuda.current_stream()) == fa.FA_ERR_BAD_SEQLENS
    # the context is still usable
    o2, lse2 = run_kvcache(c, False, 0.125)
    check_kvcache(c, o2, lse2, False, 0.125, "after bad inputs")


@pytest.mark.parametrize("num_splits", [1, 2])
def test_many_units_per_cta(num_splits):
    """512+ units over the persistent grid: each CTA walks several long units
    whose two tiles share ring slots and run their MMA issue independently."""
    B, Hq, Hkv, D = 64, 32, 8, 128
    g = torch.Generator().manual_seed(59)
    lens = torch.randint(600, 1400, (B,), generator=g).tolist()
    c = make_cache_case(B, Hq, Hkv, 1, D, "bf16", lens, page_rows=256, seed=60)
    scale = 1 / math.sqrt(D)
    o, lse = run_kvcache(c, True, scale, num_splits=num_splits)
    o2, lse2 = run_kvcache(c, True, scale, num_splits=num_splits)
    assert torch.equal(o, o2) and torch.equal(lse, lse2)
    # compare a spread of sequences against the oracle
    pick = [0, 1, 17, 33, 62, 63]
    sub = dict(c)
    sub["q"] = c["q"][pick]
    sub["lens"] = c["lens"][pick]
    sub["table"] = c["table"][pick]
    check_kvcache(sub, o[pick], lse[pick], True, scale, f"many units splits {num_splits}")


def test_deterministic():
    c = make_cache_case(2, 16, 2, 2, 128, "bf16", [3000, 2500], page_rows=256, seed=57)
    a = run_kvcache(c, True, 0.1, num_splits=4)
    b = run_kvcache(c, True, 0.1, num_splits=4)
    assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])
