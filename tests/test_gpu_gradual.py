"""GPU parity of gradual filtering (the layer-by-layer funnel of Figure 9): cb_blend_gradual, called
through the C ABI, against the CPU oracle's blend_gradual on the same seeded inputs.  Tolerances are
in tests/parity.py; every layer's kept set is compared (identical except rows inside the tie band)."""
import numpy as np
import pytest

import oracle
import parity
import workload

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")

# a 5-layer fp32 model (the tiny configuration's widths) so that the set can shrink more than once
TINY5 = workload.ModelShape(n_layers=5, d_model=256, n_heads=4, n_kv_heads=2, head_dim=64, ffn_hidden=512,
                            vocab=1024, rope_theta=1e4, dtype="f32")


@pytest.fixture(scope="module")
def cb():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__
    __graft_entry__.build()
    import cacheblend_selective_kv_gb300 as cbm
    return cbm


_cache = {}


def tiny5_case():
    """3 chunks of 64 tokens, each prefilled alone by the oracle, plus a 16-token query (seed 0)."""
    if "tiny5" not in _cache:
        w = workload.make_weights(TINY5, 0)
        chunk_tokens = [workload.tokens(0, 10 + c, 64, TINY5.vocab) for c in range(3)]
        chunks = [(0, 64 * c, 64) for c in range(3)]
        toks = np.concatenate(chunk_tokens + [workload.tokens(0, 99, 16, TINY5.vocab)])
        caches = oracle.chunk_caches(TINY5.as_dict(), w, chunk_tokens, chunks, "f32").astype(np.float32)
        _cache["tiny5"] = (w, toks, chunks, caches)
    return _cache["tiny5"]


def device_cache(caches, store):
    if caches.dtype == np.uint16:
        return torch.from_numpy(caches.view(np.int16)).cuda().view(torch.bfloat16)
    t = torch.from_numpy(np.ascontiguousarray(caches, dtype=np.float32)).cuda()
    return t.to(torch.bfloat16) if store == "bf16" else t


def compare_gradual(cb, shape, w, toks, caches, chunks, ratios, store, model=None):
    """Run both sides; compare each shrinking layer's set, then K/V and logits."""
    own = model is None
    n_ctx = sum(c[2] for c in chunks)
    if own:
        model = cb.BlendModel(shape.as_dict(), w, max_tokens=len(toks), max_chunks=len(chunks))
    out = model.blend_gradual(torch.from_numpy(toks).cuda(), device_cache(caches, store), chunks, ratios,
                              want_dev=True)
    torch.cuda.synchronize()
    assert model.status() == 0, "device status bits set"
    g_sets = {l: s.cpu().numpy() for l, s in out["sets"].items()}
    g_devs = {l: d.cpu().numpy().astype(np.float64) for l, d in out["devs"].items()}
    follow = {}
    ref = oracle.blend_gradual(shape.as_dict(), w, toks, caches, chunks, ratios, store, keep_exact=True)
    assert sorted(g_sets) == sorted(ref["devs"]), "the shrinking layers differ"
    n_diff = 0
    for l in sorted(g_sets):
        k_l = ref["counts"][l - 1]
        cand = np.arange(n_ctx) if l == 1 else ref["sets"][l - 1]
        loc_g = np.searchsorted(cand, g_sets[l])
        assert np.array_equal(cand[np.minimum(loc_g, len(cand) - 1)], g_sets[l]), f"layer {l}: kept a non-candidate"
        loc_r = np.searchsorted(cand, ref["sets"][l])
        diff = parity.assert_selection(loc_g, loc_r, ref["devs"][l], k_l)
        rel = np.abs(g_devs[l] - ref["devs"][l]) / (np.abs(ref["devs"][l]) + 1e-6 * max(ref["devs"][l].max(), 1e-30))
        assert rel.max() < (1e-3 if store == "bf16" else 1e-4), f"layer {l}: deviation rel err {rel.max():.2e}"
        follow[l] = g_sets[l]
        if diff:   # follow the GPU through a tie inside the band before comparing later layers
            n_diff += len(diff)
            ref = oracle.blend_gradual(shape.as_dict(), w, toks, caches, chunks, ratios, store, selected=dict(follow),
                                       keep_exact=True)
    kv_err = parity.assert_kv(parity.bf16_to_f64(out["out_kv"]), ref["out_kv_exact"], store)
    lg_err = parity.assert_logits(parity.bf16_to_f64(out["logits"]), ref["logits"], store)
    if own:
        model.close()
    return dict(kv_err=kv_err, logits_err=lg_err, n_diff=n_diff, counts=ref["counts"])


@pytest.mark.parametrize("ratios", [(0.5, 0.35, 0.35, 0.2), (0.3, 0.3, 0.3, 0.3), (0.2, 0.1, 0.0, 0.0),
                                    (1.0, 0.6, 0.3, 0.05)],
                         ids=["funnel", "constant", "to-zero", "from-full"])
def test_tiny5_fp32_gradual(cb, ratios):
    w, toks, chunks, caches = tiny5_case()
    r = compare_gradual(cb, TINY5, w, toks, caches, chunks, ratios, "f32")
    print(r)


def test_constant_schedule_equals_blend(cb):
    """cb_blend_gradual with a constant schedule gives cb_blend's blend (same kernels, same order)."""
    w, toks, chunks, caches = tiny5_case()
    model = cb.BlendModel(TINY5.as_dict(), w, max_tokens=len(toks), max_chunks=len(chunks))
    t = torch.from_numpy(toks).cuda()
    a = model.blend(t, device_cache(caches, "f32"), chunks, 0.3)
    b = model.blend_gradual(t, device_cache(caches, "f32"), chunks, (0.3,) * 4)
    torch.cuda.synchronize()
    assert torch.equal(a["selected"], b["sets"][1])
    assert torch.equal(a["out_kv"], b["out_kv"])
    assert torch.equal(a["logits"], b["logits"])
    model.close()


def test_small_bf16_gradual(cb):
    spec = workload.WORKLOADS["small-bf16"]
    shape, seed = spec.shape, spec.seeds[0]
    w = workload.make_weights(shape, seed)
    req = workload.make_request(spec, seed, 0.3)
    caches = oracle.chunk_caches(shape.as_dict(), w, req.chunk_tokens, req.chunks, "bf16").astype(np.float32)
    ratios = (0.3, 0.25, 0.2, 0.2, 0.15, 0.15, 0.1)
    r = compare_gradual(cb, shape, w, req.tokens, caches, req.chunks, ratios, "bf16")
    print(r)


def test_gradual_validation(cb):
    w, toks, chunks, caches = tiny5_case()
    model = cb.BlendModel(TINY5.as_dict(), w, max_tokens=len(toks), max_chunks=len(chunks))
    t, c = torch.from_numpy(toks).cuda(), device_cache(caches, "f32")
    for bad in ((0.2, 0.3, 0.3, 0.3), (0.2, 0.2, 0.2), (0.2, 0.2, 0.2, 1.5)):
        with pytest.raises(cb.CacheBlendError) as ei:
            model.blend_gradual(t, c, chunks, bad)
        assert ei.value.code == cb.CB_ERR_INVALID_ARG
    model.close()
