"""Write the stored oracle results of a full-size 8B-shape blend (test infrastructure).

The fp64 oracle needs minutes to tens of minutes of CPU for one blend at 8K and 32K context, more than
a GPU test run can spend; this script runs it once, offline, and stores what the GPU test compares
against.  It calls only ``oracle/`` (the blend) and ``workload/`` (the seeded inputs), never the CUDA
library.

Stored per (workload, seed, ratio), in ``fullsize_<workload>_s<seed>_r<ratio>.npz``:
  fingerprint   integer sums over strided samples of the token ids and of the weights' and chunk caches'
                bit patterns, so the test can tell that the generator made the same inputs on its machine
  k, selected   the oracle's top-k set (bit mask over the context rows)
  dev           every context row's check-layer deviation (float32)
  logits        the last row's logits (float32, all of the vocabulary)
  rows          a seeded sample of recomputed rows: the last query row, 7 more query rows and 24
                selected rows
  kv_layers     the layers stored for them: 1, 2, L/2 and L-1
  kv            their unrounded K and V at those layers, [layer][K|V][row][Hkv][hd] (float32)

Usage: python tests/golden/make_fullsize_golden.py llama8b-32k 6 0.15
"""
from __future__ import annotations

import os
import sys
import time

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(os.path.dirname(HERE))
sys.path.insert(0, ROOT)

import oracle  # noqa: E402
import workload  # noqa: E402


def golden_path(name: str, seed: int, ratio: float) -> str:
    return os.path.join(HERE, f"fullsize_{name}_s{seed}_r{ratio:.2f}.npz")


def fingerprint(spec, weights, req, caches) -> np.ndarray:
    """Integer sums over fixed strided samples of every input (the bfloat16 bit patterns and token ids):
    exact, so equal inputs give equal fingerprints on any machine."""
    def s(a, step=9973):
        return int(np.sum(np.asarray(a).reshape(-1)[::step].astype(np.int64)))
    parts = [s(req.tokens, 1), s(weights["embed"]), s(weights["lm_head"])]
    for lw in weights["layers"]:
        parts += [s(lw[name]) for name in ("wq", "wk", "wv", "wo", "w_gate", "w_up", "w_down")]
    parts += [s(caches[layer]) for layer in range(caches.shape[0])]
    return np.array(parts, np.int64)


def make_inputs(name: str, seed: int, ratio: float):
    spec = workload.WORKLOADS[name]
    w = workload.make_weights(spec.shape, seed)
    req = workload.make_request(spec, seed, ratio)
    caches = workload.synthetic_cache(spec.shape, seed, spec.n_ctx, workload.kv_std(spec.shape))
    return spec, w, req, caches


def main(name: str, seed: int, ratio: float) -> None:
    spec, w, req, caches = make_inputs(name, seed, ratio)
    L = spec.shape.n_layers
    layers = sorted({1, 2, L // 2, L - 1})
    t0 = time.time()
    ref = oracle.blend(spec.shape.as_dict(), w, req.tokens, caches, req.chunks, ratio, "bf16", exact_layers=layers)
    dt = time.time() - t0
    k = ref["k"]
    rows_all = ref["rows"]                                  # selected ascending, then the query rows
    rng = np.random.default_rng(1000 + seed)
    q_rows = rows_all[k:]
    pick_q = np.concatenate([[len(q_rows) - 1], rng.choice(len(q_rows) - 1, 7, replace=False)])
    pick_s = rng.choice(k, min(24, k), replace=False)
    pick = np.sort(np.concatenate([pick_s, k + pick_q]))   # indices into rows_all
    kv = np.zeros((len(layers), 2, len(pick)) + caches.shape[3:], np.float32)
    for li, layer in enumerate(layers):
        rows_l, k_ex, v_ex = ref["exact_rows"][layer]
        assert np.array_equal(rows_l, rows_all)
        kv[li, 0], kv[li, 1] = k_ex[pick], v_ex[pick]
    mask = np.zeros(spec.n_ctx, bool)
    mask[ref["selected"]] = True
    np.savez_compressed(golden_path(name, seed, ratio), fingerprint=fingerprint(spec, w, req, caches), k=k,
                        selected_mask=np.packbits(mask), dev=ref["dev"].astype(np.float32),
                        logits=ref["logits"].astype(np.float32), rows=rows_all[pick].astype(np.int32),
                        kv_layers=np.array(layers, np.int32), kv=kv, oracle_seconds=dt)
    print(f"{name} seed {seed} r={ratio}: k={k}, oracle {dt:.0f} s -> {golden_path(name, seed, ratio)}")


if __name__ == "__main__":
    main(sys.argv[1], int(sys.argv[2]), float(sys.argv[3]))
