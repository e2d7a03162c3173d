"""How closely the oracle agrees with itself when its stored values move by a rounding's worth (test
infrastructure; calls only ``oracle/`` and ``workload/``).

Every K/V value the blend stores is rounded to bfloat16 and read back by later rows and layers.  Two
implementations whose sums differ in the last float32 bits round a small share of those values to the
other bf16 neighbour, and the random-init model amplifies each such difference layer by layer.  This
script measures that amplification on the oracle alone: it runs a configuration twice, the second time
with every value multiplied by (1 + 1e-5 z), z ~ N(0, 1) from a fixed seed, just before its storage
rounding (the size of a float32 implementation's relative error; the re-RoPE'd cache rows included), with
the recomputed set of the plain run, and records per layer the max-abs and
the mean-abs distance of the perturbed run's stored values from the plain run's unrounded values, over
the rows the configuration recomputes, and the logits' max-abs distance.  The GPU parity tests hold a
configuration to the K/V tolerance of 2e-2 where this spread stays below it, and to 1.5 times the spread
where even the oracle's own spread exceeds it.

Written to ``cascade_spread.json`` (one entry per configuration).
Usage: python tests/golden/make_cascade_spread.py [prefill-8b | blend-8k-r0.30] ...
"""
from __future__ import annotations

import json
import os
import sys
import time

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(os.path.dirname(HERE))
sys.path.insert(0, ROOT)

import oracle  # noqa: E402
import oracle.cpu_blend as ob  # noqa: E402
import workload  # noqa: E402

PATH = os.path.join(HERE, "cascade_spread.json")
EPS = 1e-5


def config_inputs(name: str):
    """(cfg, weights, tokens, caches, chunks, ratio) of a named configuration."""
    if name == "prefill-8b":
        spec = workload.WORKLOADS["llama8b-3k"]
        w = workload.make_weights(spec.shape, spec.seeds[0])
        req = workload.make_request(spec, spec.seeds[0], spec.ratios[0])
        return spec.shape.as_dict(), w, req.chunk_tokens[0], None, [], 0.0
    if name == "blend-8k-r0.30":
        spec = workload.WORKLOADS["llama8b-8k"]
        w = workload.make_weights(spec.shape, 5)
        req = workload.make_request(spec, 5, 0.30)
        caches = workload.synthetic_cache(spec.shape, 5, spec.n_ctx, workload.kv_std(spec.shape))
        return spec.shape.as_dict(), w, req.tokens, caches, req.chunks, 0.30
    raise ValueError(name)


def spread(name: str) -> dict:
    cfg, w, tokens, caches, chunks, ratio = config_inputs(name)
    t0 = time.time()
    a = oracle.blend(cfg, w, tokens, caches, chunks, ratio, "bf16", keep_exact=True)
    rng = np.random.default_rng(12345)
    plain = ob.round_store

    def perturbed(x, store):
        if store == "bf16":
            x = np.asarray(x, np.float64)
            x = x * (1.0 + EPS * rng.standard_normal(x.shape))
        return plain(x, store)

    ob.round_store = perturbed
    try:   # the same recomputed set (the perturbation may swap rows whose deviations tie within it)
        b = oracle.blend(cfg, w, tokens, caches, chunks, ratio, "bf16", selected=a["selected"])
    finally:
        ob.round_store = plain
    rows = a["rows"]
    out = {"eps": EPS, "rows": "recomputed rows (the query rows and the selected rows)", "max": [], "mean": [],
           "oracle_seconds": round(time.time() - t0, 1)}
    for layer in range(cfg["n_layers"]):
        d = np.abs(b["out_kv"][layer][:, rows] - a["out_kv_exact"][layer][:, rows])
        out["max"].append(float(d.max()))
        out["mean"].append(float(d.mean()))
    out["logits_max"] = float(np.max(np.abs(b["logits"] - a["logits"])))
    return out


def main(names) -> None:
    data = json.load(open(PATH)) if os.path.exists(PATH) else {}
    for name in names:
        data[name] = spread(name)
        print(name, "max by layer", ["%.4f" % v for v in data[name]["max"]], "logits", data[name]["logits_max"])
        with open(PATH, "w") as f:
            json.dump(data, f, indent=1)


if __name__ == "__main__":
    main(sys.argv[1:] or ["prefill-8b", "blend-8k-r0.30"])
