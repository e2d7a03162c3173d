"""GPU parity at the full 8B-shape sizes, in the launch configuration bench.py times.

The chunk caches here are drawn by the workload generator (i.i.d. normal at the K/V scale of the
random-init model): a genuine per-chunk prefill at this shape costs the fp64 oracle ~8 TFLOP per
chunk.  The smaller configurations use genuine per-chunk prefills."""
import numpy as np
import pytest

import oracle
import parity
import workload

pytestmark = [pytest.mark.gpu, pytest.mark.slow]
torch = pytest.importorskip("torch")


@pytest.fixture(scope="module")
def cb():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__
    __graft_entry__.build()
    import cacheblend_selective_kv_gb300 as cbm
    return cbm


def test_llama8b_3k_full_blend(cb):
    spec = workload.WORKLOADS["llama8b-3k"]
    shape, seed, ratio = spec.shape, spec.seeds[0], spec.ratios[0]
    w = workload.make_weights(shape, seed)
    req = workload.make_request(spec, seed, ratio)
    caches = workload.synthetic_cache(shape, seed, spec.n_ctx, workload.kv_std(shape))
    model = cb.BlendModel(shape.as_dict(), w, max_tokens=spec.n_tokens, max_chunks=spec.n_chunks)
    cached = torch.from_numpy(caches.view(np.int16)).cuda().view(torch.bfloat16)
    out = model.blend(torch.from_numpy(req.tokens).cuda(), cached, req.chunks, ratio, want_dev=True)
    torch.cuda.synchronize()
    assert model.status() == 0
    g_sel = out["selected"].cpu().numpy()
    g_kv = parity.bf16_to_f64(out["out_kv"])
    g_lg = parity.bf16_to_f64(out["logits"])
    g_dev = out["dev"].cpu().numpy().astype(np.float64)
    model.close()
    del cached
    ref = oracle.blend(shape.as_dict(), w, req.tokens, caches, req.chunks, ratio, "bf16", keep_exact=True)
    diff = parity.assert_selection(g_sel, ref["selected"], ref["dev"], ref["k"])
    if diff:
        ref = oracle.blend(shape.as_dict(), w, req.tokens, caches, req.chunks, ratio, "bf16", selected=g_sel,
                           keep_exact=True)
    rows = ref["rows"]
    for l in (0, 1, 2, shape.n_layers // 2, shape.n_layers - 1):
        mx, n_over, n_nb = parity.kv_error(g_kv[l][:, rows], ref["out_kv_exact"][l][:, rows], "bf16")
        print(f"layer {l}: max abs {mx:.4f}, beyond tol {n_over}, of which bf16 neighbours {n_nb}")
    dev_rel = np.abs(g_dev - ref["dev"]) / ref["dev"]
    print(f"selection differs in {len(diff)} rows; deviation rel err max {dev_rel.max():.2e}")
    print(f"logits max abs {np.abs(g_lg - ref['logits']).max():.4f}")
    parity.assert_kv(g_kv, ref["out_kv_exact"], "bf16")
    parity.assert_logits(g_lg, ref["logits"], "bf16")
