"""Helpers for the GPU parity tests: run a drawn case through the C ABI and
compare it with the fp64 oracle on the same 16-bit inputs.

With FA_PARITY_REPORT=<path> set, every comparison appends one JSON line with
its metrics to that file."""
import json
import os

import numpy as np
import torch

import exact_attention_forward_sm_gb300 as fa
from exact_attention_forward_sm_gb300 import workloads as wl
import oracle
from tests.helpers import COSINE_MIN, LSE_ABS_TOL, REL_LINF_TOL, cosine, lse_max_abs, rel_linf


def to_device(case, dev="cuda:0"):
    q, k, v = (t.to(dev).contiguous() for t in (case.q, case.k, case.v))
    cu_q = case.cu_seqlens_q.to(dev) if case.varlen else None
    cu_k = case.cu_seqlens_k.to(dev) if case.varlen else None
    return q, k, v, cu_q, cu_k


def run_gpu(case, dev="cuda:0", with_lse=True, stream=None, num_splits=None):
    """Run fa_fwd on the case (fa_fwd_ex with score variants, fa_fwd_split when
    ``num_splits`` is given); returns (o, lse) device tensors (library layout)."""
    q, k, v, cu_q, cu_k = to_device(case, dev)
    o = torch.full_like(q, float("nan"))
    shape = (case.Hq, case.Sq) if case.varlen else (case.B, case.Hq, case.Sq)
    lse = torch.full(shape, float("nan"), dtype=torch.float32, device=dev) if with_lse else None
    args = (q, k, v, o, lse, case.B, case.Hq, case.Hkv, case.Sq, case.Sk, case.D, case.scale,
            int(case.causal), cu_q, cu_k, stream or torch.cuda.current_stream(),
            wl.DTYPE_CODE[case.dtype])
    slopes = case.alibi_slopes.to(dev) if case.alibi_slopes is not None else None
    if num_splits is not None:
        st = fa.fa_fwd_split(*args, case.window_left, case.window_right, case.softcap, slopes,
                             num_splits)
    elif case.has_variants:
        st = fa.fa_fwd_ex(*args, case.window_left, case.window_right, case.softcap, slopes)
    else:
        st = fa.fa_fwd(*args)
    assert st == fa.FA_OK, fa.fa_status_string(st)
    dst = fa.fa_get_device_error(stream or torch.cuda.current_stream())
    assert dst == fa.FA_OK, fa.fa_status_string(dst)
    return o, lse


def rows_in_oracle_order(case, o, lse):
    """Library layout -> [rows, D] / [rows] in LSE-index order (float64)."""
    if case.varlen:
        o_rows = o.float().permute(1, 0, 2).reshape(-1, case.D)
    else:
        o_rows = o.float().permute(0, 2, 1, 3).reshape(-1, case.D)
    lse_rows = lse.reshape(-1) if lse is not None else None
    return o_rows, lse_rows


def oracle_rows(case, rows=None):
    return oracle.attention(case.q, case.k, case.v, case.B, case.Hq, case.Hkv, case.Sq,
                            case.Sk, case.D, case.scale, case.causal, case.cu_seqlens_q,
                            case.cu_seqlens_k, rows=rows, window_left=case.window_left,
                            window_right=case.window_right, softcap=case.softcap,
                            alibi_slopes=case.alibi_slopes)


def check(case, o, lse, rows=None, tag="", whole_tensor=True):
    """Compare GPU output rows (all, or the selected LSE indices) with the oracle
    under the acceptance gates; returns the metrics.  ``whole_tensor=False``
    skips the finiteness check of the rows outside ``rows`` (for inputs whose
    other rows are poisoned on purpose)."""
    # the whole output, compared rows or not: O finite (a row with no visible
    # key is 0), LSE finite or -inf (no visible key), never NaN or +inf
    if whole_tensor:
        assert bool(torch.isfinite(o).all()), f"{tag}: non-finite O in the output tensor"
        if lse is not None:
            assert not bool(torch.isnan(lse).any()), f"{tag}: NaN LSE in the output tensor"
            assert not bool(torch.isposinf(lse).any()), f"{tag}: +inf LSE in the output tensor"
    o_ref, lse_ref = oracle_rows(case, rows)
    o_rows, lse_rows = rows_in_oracle_order(case, o, lse)
    if rows is not None:
        idx = torch.as_tensor(np.asarray(rows), device=o_rows.device)
        o_rows = o_rows[idx]
        lse_rows = lse_rows[idx] if lse_rows is not None else None
    o_np = o_rows.cpu().numpy().astype(np.float64)
    assert np.all(np.isfinite(o_np)), f"{tag}: non-finite O"
    m = {"rel_linf": rel_linf(o_np, o_ref), "cosine": cosine(o_np, o_ref)}
    if lse_rows is not None:
        m["lse_err"] = lse_max_abs(lse_rows.cpu().numpy(), lse_ref)
    report = os.environ.get("FA_PARITY_REPORT")
    if report:
        with open(report, "a") as f:
            f.write(json.dumps({"case": tag, "dtype": case.dtype, "rows": int(o_np.shape[0]),
                                **m}) + "\n")
    tol = REL_LINF_TOL[case.dtype]
    assert m["rel_linf"] <= tol, f"{tag}: rel_Linf {m['rel_linf']:.3e} > {tol} {m}"
    assert m["cosine"] >= COSINE_MIN, f"{tag}: cosine {m['cosine']:.8f} {m}"
    if lse_rows is not None:
        assert m["lse_err"] <= LSE_ABS_TOL, f"{tag}: LSE err {m['lse_err']:.3e} {m}"
    return m


def sample_rows(case, per_head=64, heads=None, seed=0):
    """LSE indices of a spread of rows: sequence edges, tile edges and random."""
    rng = np.random.default_rng(seed)
    hs = range(case.Hq) if heads is None else heads
    out = []
    starts = [0]
    lens = [lq for lq, _ in case.seq_lengths()]
    if case.varlen:
        starts = case.cu_seqlens_q.tolist()[:-1]
    for h in hs:
        for b, lq in enumerate(lens):
            if lq == 0:
                continue
            cand = {0, 1, lq - 1, lq - 2}
            for e in (127, 128, 129, 255, 256, 257):
                if e < lq:
                    cand.add(e)
            cand.update(rng.integers(0, lq, size=max(0, per_head // len(lens))).tolist())
            cand = [c for c in sorted(cand) if 0 <= c < lq]
            for i in cand:
                if case.varlen:
                    out.append(h * case.Sq + starts[b] + i)
                else:
                    out.append((b * case.Hq + h) * case.Sq + i)
    return np.array(sorted(set(out)), dtype=np.int64)
