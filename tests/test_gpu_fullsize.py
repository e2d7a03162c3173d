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


_MODELS = {}


def _model_for(cb, spec, seed):
    """Weights and a model handle per (workload, seed), kept for the next test of the same seed (one at a
    time: the 8B weights are 16 GB on each side)."""
    key = (spec.name, seed)
    if key not in _MODELS:
        for k in list(_MODELS):
            _MODELS.pop(k)[1].close()
        w = workload.make_weights(spec.shape, seed)
        _MODELS[key] = (w, cb.BlendModel(spec.shape.as_dict(), w, max_tokens=spec.n_tokens, max_chunks=spec.n_chunks))
    return _MODELS[key]


def _gpu_blend(cb, spec, seed, ratio, caches, want_dev=True, keep=False):
    shape = spec.shape
    req = workload.make_request(spec, seed, ratio)
    if keep:
        w, model = _model_for(cb, spec, seed)
    else:
        w = workload.make_weights(shape, seed)
        model = cb.BlendModel(shape.as_dict(), w, max_tokens=spec.n_tokens, max_chunks=spec.n_chunks)
    cached = torch.from_numpy(caches.view(np.int16)).cuda().view(torch.bfloat16)
    out = model.blend(torch.from_numpy(req.tokens).cuda(), cached, req.chunks, ratio, want_dev=want_dev)
    torch.cuda.synchronize()
    assert model.status() == 0
    res = dict(selected=out["selected"].cpu().numpy(), logits=parity.bf16_to_f64(out["logits"]), k=out["k"])
    if want_dev:
        res["dev"] = out["dev"].cpu().numpy().astype(np.float64)
    res["kv"] = out["out_kv"]          # stays on the device; sampled below
    del cached
    return w, req, res, model


def _kv_rows(res, layer, kv, rows):
    t = res["kv"][layer, kv, torch.as_tensor(rows, device=res["kv"].device)]
    return parity.bf16_to_f64(t)


def _sampled_checks(spec, w, req, res, caches, ratio, rng, n_sample=48):
    """Checks that need no full oracle blend: the selection is exactly the top-k of the GPU's own
    deviations; the deviations of sampled context rows match the oracle's row-restricted deviation;
    unselected context rows hold the re-RoPE'd cache at every layer."""
    shape = spec.shape
    k = res["k"]
    assert list(res["selected"]) == list(oracle.select_hkvd(res["dev"], k))
    rows = np.sort(rng.choice(spec.n_ctx, n_sample, replace=False))
    ref_dev = oracle.deviation_rows(shape.as_dict(), w, req.tokens, caches, req.chunks, rows, "bf16")
    rel = np.abs(res["dev"][rows] - ref_dev) / ref_dev
    assert rel.max() < 2e-3, rel.max()
    sel = set(res["selected"].tolist())
    unsel = np.array([r for r in rows if r not in sel])
    layers = [0, 1, shape.n_layers // 2, shape.n_layers - 1]
    placed = oracle.rerope(caches[layers], req.chunks, shape.rope_theta, "bf16")
    for li, layer in enumerate(layers):
        for kv in (0, 1):
            got = _kv_rows(res, layer, kv, unsel)
            ref = placed[li, kv, unsel]
            ulp = np.ldexp(1.0, np.frexp(np.abs(ref))[1] - 8)
            assert np.all(np.abs(got - ref) <= ulp), (layer, kv)
    return rel.max()


def test_llama8b_8k_r005_full_blend_seed3(cb):
    """8K context, 16 shuffled chunks, r = 0.05: the whole blend against the oracle."""
    spec = workload.WORKLOADS["llama8b-8k"]
    seed, ratio = 3, 0.05
    caches = workload.synthetic_cache(spec.shape, seed, spec.n_ctx, workload.kv_std(spec.shape))
    w, req, res, model = _gpu_blend(cb, spec, seed, ratio, caches)
    assert [c[1] for c in req.chunks] == [512 * i for i in range(16)]
    g_kv = parity.bf16_to_f64(res["kv"])
    model.close()
    ref = oracle.blend(spec.shape.as_dict(), w, req.tokens, caches, req.chunks, ratio, "bf16", keep_exact=True)
    diff = parity.assert_selection(res["selected"], ref["selected"], ref["dev"], ref["k"])
    if diff:
        ref = oracle.blend(spec.shape.as_dict(), w, req.tokens, caches, req.chunks, ratio, "bf16",
                           selected=res["selected"], keep_exact=True)
    print(f"8K r=0.05: {len(diff)} rows in the tie band; kv max {parity.kv_error(g_kv, ref['out_kv_exact'], 'bf16')[0]:.4f}")
    parity.assert_kv(g_kv, ref["out_kv_exact"], "bf16")
    parity.assert_logits(res["logits"], ref["logits"], "bf16")


C4_RUNS = [(s, r) for s in (3, 4, 5) for r in (0.05, 0.15, 0.30) if (s, r) != (3, 0.05)]


@pytest.mark.parametrize("seed,ratio", C4_RUNS)
def test_llama8b_8k_sampled(cb, seed, ratio):
    """The 8K configuration's sweep (seeds 3-5, each with its own shuffled chunk order, r in {0.05, 0.15,
    0.30}; seed 3 at r = 0.05 runs against the full oracle above): sampled checks on every other run."""
    spec = workload.WORKLOADS["llama8b-8k"]
    caches = workload.synthetic_cache(spec.shape, seed, spec.n_ctx, workload.kv_std(spec.shape))
    w, req, res, model = _gpu_blend(cb, spec, seed, ratio, caches, keep=True)
    rel = _sampled_checks(spec, w, req, res, caches, ratio, np.random.default_rng(seed))
    print(f"8K seed {seed} r={ratio}: sampled deviation rel err {rel:.2e}")
    if (seed, ratio) == C4_RUNS[-1]:
        for k in list(_MODELS):
            _MODELS.pop(k)[1].close()


def test_llama8b_32k_sampled(cb):
    """32K context (64 chunks + 128 query tokens), r = 0.15: sampled checks at full size."""
    spec = workload.WORKLOADS["llama8b-32k"]
    seed, ratio = spec.seeds[0], spec.ratios[0]
    caches = workload.synthetic_cache(spec.shape, seed, spec.n_ctx, workload.kv_std(spec.shape))
    w, req, res, model = _gpu_blend(cb, spec, seed, ratio, caches)
    rel = _sampled_checks(spec, w, req, res, caches, ratio, np.random.default_rng(seed), n_sample=32)
    print(f"32K r=0.15: sampled deviation rel err {rel:.2e}")
    model.close()


def test_llama8b_32k_full_reuse(cb):
    """32K context at r = 0 (full KV reuse): the query rows' K/V at every layer and the logits
    against the oracle; every context row is the re-RoPE'd cache."""
    spec = workload.WORKLOADS["llama8b-32k"]
    seed = spec.seeds[0]
    caches = workload.synthetic_cache(spec.shape, seed, spec.n_ctx, workload.kv_std(spec.shape))
    w, req, res, model = _gpu_blend(cb, spec, seed, 0.0, caches, want_dev=False)
    q_rows = np.arange(spec.n_ctx, spec.n_tokens)
    g_q = np.stack([np.stack([_kv_rows(res, l, kv, q_rows) for kv in (0, 1)]) for l in range(spec.shape.n_layers)])
    model.close()
    ref = oracle.blend(spec.shape.as_dict(), w, req.tokens, caches, req.chunks, 0.0, "bf16", keep_exact=True)
    parity.assert_kv(g_q, ref["out_kv_exact"][:, :, spec.n_ctx:], "bf16", "query-row K/V")
    parity.assert_logits(res["logits"], ref["logits"], "bf16")


def test_llama8b_3k_gradual(cb):
    """Gradual filtering at the 8B shape, 3K context: 0.30 at the check layer shrinking to 0.15 by
    layer 5 (the funnel schedule bench.py --gradual times).  Every shrinking layer's set, all K/V and
    the logits against the full oracle."""
    import test_gpu_gradual as tg
    spec = workload.WORKLOADS["llama8b-3k"]
    shape, seed = spec.shape, spec.seeds[0]
    ratios = workload.funnel_ratios(shape.n_layers, spec.ratios[0])
    w = workload.make_weights(shape, seed)
    req = workload.make_request(spec, seed, spec.ratios[0])
    caches = workload.synthetic_cache(shape, seed, spec.n_ctx, workload.kv_std(shape))
    r = tg.compare_gradual(cb, shape, w, req.tokens, caches, req.chunks, ratios, "bf16")
    print(f"8B 3K gradual: {r}")


def test_llama8b_3k_streamed_matches_device_resident(cb):
    """The 8B-shape 3K blend with its chunk caches streamed from pinned host memory layer by layer: K/V
    and logits within the parity tolerances of the device-resident blend (the residual GEMMs add split-K
    partial sums in a run-dependent order), and the copied-back K/V equal to the device K/V."""
    spec = workload.WORKLOADS["llama8b-3k"]
    shape, seed, ratio = spec.shape, spec.seeds[0], spec.ratios[0]
    w = workload.make_weights(shape, seed)
    req = workload.make_request(spec, seed, ratio)
    caches = workload.synthetic_cache(shape, seed, spec.n_ctx, workload.kv_std(shape))
    model = cb.BlendModel(shape.as_dict(), w, max_tokens=spec.n_tokens, max_chunks=spec.n_chunks)
    host = torch.from_numpy(caches.view(np.int16)).view(torch.bfloat16).pin_memory()
    tokens = torch.from_numpy(req.tokens).cuda()
    a = model.blend(tokens, host.cuda(), req.chunks, ratio)
    kv_host = torch.empty(a["out_kv"].shape, dtype=torch.bfloat16).pin_memory()
    b = model.blend_streamed(tokens, host, req.chunks, (ratio,) * (shape.n_layers - 1), out_kv_host=kv_host)
    torch.cuda.synchronize()
    assert model.status() == 0
    assert torch.equal(kv_host, b["out_kv"].cpu())
    ka, kb = parity.bf16_to_f64(a["out_kv"]), parity.bf16_to_f64(b["out_kv"])
    # 2e-2, or one bf16 step at the value (two roundings of sums taken in different orders)
    ulp = np.ldexp(1.0, np.frexp(np.maximum(np.abs(ka), 1e-30))[1] - 8)
    assert np.all(np.abs(ka - kb) <= np.maximum(2e-2, ulp))
    assert np.max(np.abs(parity.bf16_to_f64(a["logits"]) - parity.bf16_to_f64(b["logits"]))) <= 3e-2
    model.close()
