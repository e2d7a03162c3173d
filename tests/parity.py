"""Parity comparisons between the CUDA library and the CPU oracle (tolerances written here).

Selection: identical except rows whose oracle deviation lies within 1e-3 (relative) of the
oracle's k-th largest deviation.  K/V: max-abs 2e-2 for bf16 storage, 1e-4 for fp32.
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


def kv_error(gpu_kv: np.ndarray, ref_kv: np.ndarray, store: str):
    """max-abs error, plus the count of elements that exceed the tolerance but are within one
    storage ulp of the oracle value (the rounding of the stored value itself)."""
    err = np.abs(gpu_kv - ref_kv)
    tol = KV_TOL[store]
    over = err > tol
    n_ulp = 0
    if store == "bf16" and over.any():
        ulp = np.ldexp(1.0, np.frexp(np.abs(ref_kv[over]))[1] - 8)
        n_ulp = int(np.sum(err[over] <= ulp))
    return float(err.max()) if err.size else 0.0, int(over.sum()), n_ulp


def assert_kv(gpu_kv, ref_kv, store, what="K/V"):
    mx, n_over, n_ulp = kv_error(gpu_kv, ref_kv, store)
    assert n_over == n_ulp, f"{what}: max abs error {mx:.3e}; {n_over - n_ulp} elements beyond {KV_TOL[store]} and 1 ulp"
    return mx


def assert_logits(gpu_logits, ref_logits, store):
    mx = float(np.max(np.abs(gpu_logits - ref_logits)))
    assert mx <= LOGIT_TOL[store], f"logits max abs error {mx:.3e} > {LOGIT_TOL[store]}"
    return mx
