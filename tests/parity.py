"""Parity comparisons between the CUDA library and the CPU oracle (tolerances written here).

Selection: identical except rows whose oracle deviation lies within 1e-3 (relative) of the
oracle's k-th largest deviation.  K/V: max-abs 2e-2 for bf16 storage, 1e-4 for fp32, against the oracle's unrounded value; a bf16
element also passes when it is one of the two bf16 neighbours of that value (the storage rounding).
Logits: max-abs 3e-2 for bf16, 1e-3 for fp32.
"""
from __future__ import annotations

import numpy as np

SEL_BAND = 1e-3
KV_TOL = {"bf16": 2e-2, "f32": 1e-4}
LOGIT_TOL = {"bf16": 3e-2, "f32": 1e-3}


def bf16_to_f64(t) -> np.ndarray:
    """torch tensor (any float dtype, any device) -> float64 numpy."""
    import torch
    return t.detach().to(torch.float32).cpu().numpy().astype(np.float64)


def threshold(dev: np.ndarray, k: int) -> float:
    if k <= 0:
        return float("inf")
    return float(np.sort(dev)[::-1][k - 1])


def selection_mismatch(gpu_sel, ref_sel, ref_dev, k):
    """Rows in exactly one of the two sets, and those among them outside the exemption band."""
    g, r = set(int(x) for x in gpu_sel), set(int(x) for x in ref_sel)
    diff = sorted(g ^ r)
    thr = threshold(ref_dev, k)
    bad = [j for j in diff if abs(ref_dev[j] - thr) > SEL_BAND * thr]
    return diff, bad


def assert_selection(gpu_sel, ref_sel, ref_dev, k):
    assert len(gpu_sel) == k and len(ref_sel) == k
    assert list(gpu_sel) == sorted(gpu_sel), "GPU selection not ascending"
    diff, bad = selection_mismatch(gpu_sel, ref_sel, ref_dev, k)
    assert not bad, f"selected rows differ outside the {SEL_BAND} band: {bad[:10]} (of {len(diff)} differing)"
    return diff


def bf16_neighbours(x: np.ndarray):
    """The bfloat16 values just below and just above x (equal when x is a bfloat16 number)."""
    m, e = np.frexp(np.asarray(x, np.float64))
    return np.ldexp(np.floor(np.ldexp(m, 8)), e - 8), np.ldexp(np.ceil(np.ldexp(m, 8)), e - 8)


def kv_error(gpu_kv: np.ndarray, ref_exact: np.ndarray, store: str):
    """Against the oracle's unrounded values: max-abs error, the count of elements beyond the
    tolerance, and how many of those are still one of the two bf16 neighbours of the exact value
    (the rounding of the stored value itself)."""
    err = np.abs(gpu_kv - ref_exact)
    tol = KV_TOL[store]
    over = err > tol
    n_nb = 0
    if store == "bf16" and over.any():
        lo, hi = bf16_neighbours(ref_exact[over])
        g = gpu_kv[over]
        n_nb = int(np.sum((g == lo) | (g == hi)))
    return float(err.max()) if err.size else 0.0, int(over.sum()), n_nb


def assert_kv(gpu_kv, ref_exact, store, what="K/V"):
    mx, n_over, n_nb = kv_error(gpu_kv, ref_exact, store)
    assert n_over == n_nb, (f"{what}: max abs error {mx:.3e}; {n_over - n_nb} elements beyond {KV_TOL[store]} "
                            f"that are not a bf16 neighbour of the exact value")
    return mx


def assert_logits(gpu_logits, ref_logits, store):
    mx = float(np.max(np.abs(gpu_logits - ref_logits)))
    assert mx <= LOGIT_TOL[store], f"logits max abs error {mx:.3e} > {LOGIT_TOL[store]}"
    return mx
