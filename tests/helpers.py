"""Comparison metrics shared by the tests (acceptance gates of the method).

O is judged by rel_Linf = max|O - O_ref| / max|O_ref| over all valid rows and by
the cosine of the flattened outputs; LSE by its max absolute error.  The gates
are fp16 rel_Linf <= 2e-2, bf16 rel_Linf <= 1e-2, cosine >= 0.9995 (release
notes v1.7, section 4) and LSE max abs error <= 1e-3.
"""
import numpy as np

REL_LINF_TOL = {"fp16": 2e-2, "bf16": 1e-2}
COSINE_MIN = 0.9995
LSE_ABS_TOL = 1e-3


def rel_linf(o, ref):
    o = np.asarray(o, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    den = np.max(np.abs(ref))
    num = np.max(np.abs(o - ref)) if o.size else 0.0
    return float(num / den) if den > 0 else float(num)


def cosine(o, ref):
    a = np.asarray(o, dtype=np.float64).ravel()
    b = np.asarray(ref, dtype=np.float64).ravel()
    na, nb = np.linalg.norm(a), np.linalg.norm(b)
    if na == 0 and nb == 0:
        return 1.0
    return float(np.dot(a, b) / (na * nb))


def lse_max_abs(lse, ref):
    lse = np.asarray(lse, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    both_inf = np.isneginf(lse) & np.isneginf(ref)
    with np.errstate(invalid="ignore"):
        d = np.where(both_inf, 0.0, np.abs(lse - ref))
    return float(np.max(d)) if d.size else 0.0
