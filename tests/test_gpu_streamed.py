"""GPU tests of the layer-wise load pipeline (cb_blend_streamed): chunk caches in pinned host memory,
copied layer by layer on a copy stream while earlier layers compute, finished layers copied back.
The streamed blend runs the same kernels as the device-resident one, so its results must match it
(and through it the oracle); the copied-back K/V must equal the device K/V."""
import numpy as np
import pytest

import oracle
import parity
import workload

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")


@pytest.fixture(scope="module")
def cb():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__
    __graft_entry__.build()
    import cacheblend_selective_kv_gb300 as cbm
    return cbm


def host_cache(caches, store):
    if caches.dtype == np.uint16:
        t = torch.from_numpy(caches.view(np.int16)).view(torch.bfloat16)
    else:
        t = torch.from_numpy(np.ascontiguousarray(caches, dtype=np.float32))
        if store == "bf16":
            t = t.to(torch.bfloat16)
    return t.pin_memory()


@pytest.mark.parametrize("ratios", [(0.3, 0.3, 0.3, 0.3), (0.5, 0.35, 0.35, 0.2)], ids=["constant", "funnel"])
def test_tiny5_streamed_equals_device_resident(cb, ratios):
    import test_gpu_gradual as tg
    w, toks, chunks, caches = tg.tiny5_case()
    model = cb.BlendModel(tg.TINY5.as_dict(), w, max_tokens=len(toks), max_chunks=len(chunks))
    t = torch.from_numpy(toks).cuda()
    ref = model.blend_gradual(t, tg.device_cache(caches, "f32"), chunks, ratios)
    hc = host_cache(caches, "f32")
    kv_host = torch.empty(ref["out_kv"].shape, dtype=ref["out_kv"].dtype).pin_memory()
    out = model.blend_streamed(t, hc, chunks, ratios, out_kv_host=kv_host)
    torch.cuda.synchronize()
    assert model.status() == 0
    assert torch.equal(out["out_kv"], ref["out_kv"])
    assert torch.equal(out["logits"], ref["logits"])
    assert torch.equal(kv_host, out["out_kv"].cpu())
    model.close()


def test_small_bf16_streamed_parity(cb):
    """Small bf16 configuration through the pipeline: the oracle's blend within the parity tolerances,
    and the host copy of every layer equal to the device K/V."""
    spec = workload.WORKLOADS["small-bf16"]
    shape, seed, ratio = spec.shape, spec.seeds[0], spec.ratios[0]
    w = workload.make_weights(shape, seed)
    req = workload.make_request(spec, seed, ratio)
    caches = oracle.chunk_caches(shape.as_dict(), w, req.chunk_tokens, req.chunks, "bf16").astype(np.float32)
    model = cb.BlendModel(shape.as_dict(), w, max_tokens=spec.n_tokens, max_chunks=spec.n_chunks)
    hc = host_cache(caches, "bf16")
    out_shape = (shape.n_layers, 2, spec.n_tokens, shape.n_kv_heads, shape.head_dim)
    kv_host = torch.empty(out_shape, dtype=torch.bfloat16).pin_memory()
    out = model.blend_streamed(torch.from_numpy(req.tokens).cuda(), hc, req.chunks, (ratio,) * (shape.n_layers - 1),
                               out_kv_host=kv_host)
    torch.cuda.synchronize()
    assert model.status() == 0
    assert torch.equal(kv_host, out["out_kv"].cpu())
    ref = oracle.blend(shape.as_dict(), w, req.tokens, caches, req.chunks, ratio, "bf16", keep_exact=True)
    parity.assert_kv(parity.bf16_to_f64(out["out_kv"]), ref["out_kv_exact"], "bf16")
    parity.assert_logits(parity.bf16_to_f64(out["logits"]), ref["logits"], "bf16")
    model.close()


def test_streamed_validation(cb):
    import test_gpu_gradual as tg
    w, toks, chunks, caches = tg.tiny5_case()
    model = cb.BlendModel(tg.TINY5.as_dict(), w, max_tokens=len(toks), max_chunks=len(chunks))
    t = torch.from_numpy(toks).cuda()
    hc = host_cache(caches, "f32")
    s = torch.cuda.Stream()
    out_kv = model.kv_buffer(len(toks))
    logits = torch.empty(1024, device="cuda")
    with pytest.raises(cb.CacheBlendError):      # the copy stream must not be the compute stream
        cb.cb_blend_streamed(model.handle, t, len(toks), hc, chunks, (0.3,) * 4, out_kv, logits, stream=s,
                             copy_stream=s)
    with pytest.raises(cb.CacheBlendError):      # chunks without a host cache
        cb.cb_blend_streamed(model.handle, t, len(toks), None, chunks, (0.3,) * 4, out_kv, logits, stream=s,
                             copy_stream=torch.cuda.Stream())
    # no chunks: a plain prefill through the pipeline (nothing to load) equals the device prefill
    a = model.blend_streamed(t, None, [], (0.0,) * 4)
    b = model.blend(t, None, [], 0.0)
    torch.cuda.synchronize()
    assert torch.equal(a["out_kv"], b["out_kv"]) and torch.equal(a["logits"], b["logits"])
    model.close()
