"""Parity comparisons between the CUDA library and the CPU oracle (tolerances written here).

Selection: identical except rows whose oracle deviation lies within 1e-3 (relative) of the
oracle's k-th largest deviation.  K/V: max-abs 2e-2 for bf16 storage, 1e-4 for fp32, against the oracle's
unrounded value.  Where |value| >= 8 the bf16 storage step itself is larger than 2e-2 (half an ulp is 1/32
there), so a bf16 element of such a value passes when it is one of the value's two bf16 neighbours (a
rounding that went either way); below 8 the 2e-2 bound holds as stated.  Such elements are counted.
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


def dev_error(gpu_dev, ref_dev, k):
    """Per-row deviation error relative to the larger of the row's own deviation and 1e-3 of the selection
    threshold (rows whose cached K/V equal their fresh K/V up to rounding, such as a chunk prefilled where
    it sits, have deviations near zero, where a relative error says nothing about the selection)."""
    thr = threshold(ref_dev, k) if k > 0 else float(np.max(ref_dev, initial=0.0))
    return np.abs(gpu_dev - ref_dev) / np.maximum(ref_dev, max(1e-3 * thr, 1e-30))


def bf16_neighbours(x: np.ndarray):
    """The bfloat16 values just below and just above x (equal when x is a bfloat16 number)."""
    m, e = np.frexp(np.asarray(x, np.float64))
    return np.ldexp(np.floor(np.ldexp(m, 8)), e - 8), np.ldexp(np.ceil(np.ldexp(m, 8)), e - 8)


BF16_STEP_ABOVE = 8.0    # |x| from which half a bf16 ulp (1/32) exceeds the 2e-2 bound


def kv_error(gpu_kv: np.ndarray, ref_exact: np.ndarray, store: str, tol: float = None):
    """Against the oracle's unrounded values: max-abs error, the count of elements beyond the
    tolerance, and how many of those are exempt (|x| >= 8 and a bf16 neighbour of the exact value)."""
    err = np.abs(gpu_kv - ref_exact)
    tol = KV_TOL[store] if tol is None else tol
    over = err > tol
    n_ex = 0
    if store == "bf16" and over.any():
        x, g = ref_exact[over], gpu_kv[over]
        lo, hi = bf16_neighbours(x)
        n_ex = int(np.sum((np.abs(x) >= BF16_STEP_ABOVE) & ((g == lo) | (g == hi))))
    return float(err.max()) if err.size else 0.0, int(over.sum()), n_ex


def assert_kv(gpu_kv, ref_exact, store, what="K/V", tol: float = None):
    """Asserts the K/V tolerance (KV_TOL, or `tol`) and returns the max abs error; the count of exempt
    elements (|x| >= 8, a bf16 neighbour of the exact value) is printed."""
    tol = KV_TOL[store] if tol is None else tol
    mx, n_over, n_ex = kv_error(gpu_kv, ref_exact, store, tol)
    assert n_over == n_ex, (f"{what}: max abs error {mx:.3e}; {n_over - n_ex} elements beyond {tol:.4g} "
                            f"that are not a bf16 neighbour of an exact value of magnitude >= {BF16_STEP_ABOVE}")
    if n_ex:
        print(f"{what}: {n_ex} of {gpu_kv.size} elements beyond {tol:.4g} are bf16 neighbours of exact values "
              f"of magnitude >= {BF16_STEP_ABOVE} (max abs error {mx:.4f})")
    return mx


def cascade_bounds(name: str):
    """Per-layer K/V bounds (max-abs, mean-abs) and the logits bound for a configuration whose recomputed rows
    are so many that the oracle's own spread under a rounding-sized perturbation of its stored values
    (tests/golden/cascade_spread.json, written by tests/golden/make_cascade_spread.py from the oracle alone)
    exceeds the tolerances (2e-2 K/V, 3e-2 logits): max-abs max(2e-2, 1.5 x spread), mean-abs 1.5 x spread, logits
    max(3e-2, 1.5 x spread)."""
    import json
    import os
    d = json.load(open(os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden", "cascade_spread.json")))[name]
    return ([max(KV_TOL["bf16"], 1.5 * v) for v in d["max"]], [1.5 * v for v in d["mean"]],
            max(LOGIT_TOL["bf16"], 1.5 * d["logits_max"]))


def rotation_tol(base_k, ref_k):
    """Bound on |GPU - oracle| for a K rotated in fp32 with fp32 (cos, sin) and rounded once to bf16:
    one bf16 ulp of the result, plus the fp32 rounding of the products, a few 2^-24 of the rotated
    pair's magnitude |x0| + |x1| (it dominates where the result cancels to near zero)."""
    ulp = np.ldexp(1.0, np.frexp(np.abs(ref_k))[1] - 8)
    pair = np.abs(base_k.reshape(base_k.shape[:-1] + (-1, 2))).sum(-1)
    return ulp + np.ldexp(np.repeat(pair, 2, axis=-1), -20)


def assert_logits(gpu_logits, ref_logits, store):
    mx = float(np.max(np.abs(gpu_logits - ref_logits)))
    assert mx <= LOGIT_TOL[store], f"logits max abs error {mx:.3e} > {LOGIT_TOL[store]}"
    return mx
