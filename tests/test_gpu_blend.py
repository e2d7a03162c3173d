"""GPU parity: the CUDA library, called through its C ABI, against the CPU oracle on the same seeded
inputs.  Tolerances are in tests/parity.py."""
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


_cache = {}


def setup_case(name, seed=None, ratio=None, synthetic=False):
    """Weights, request and chunk caches for a named workload (cached per module)."""
    spec = workload.WORKLOADS[name]
    seed = spec.seeds[0] if seed is None else seed
    ratio = spec.ratios[0] if ratio is None else ratio
    key = (name, seed, synthetic)
    if key not in _cache:
        shape = spec.shape
        w = workload.make_weights(shape, seed)
        req = workload.make_request(spec, seed, ratio)
        if synthetic:
            caches = workload.synthetic_cache(shape, seed, spec.n_ctx, workload.kv_std(shape))
        else:
            caches = oracle.chunk_caches(shape.as_dict(), w, req.chunk_tokens, req.chunks, shape.dtype)
            if shape.dtype == "bf16":
                caches = caches.astype(np.float32)
        _cache.clear()
        _cache[key] = (spec, w, req, caches)
    spec, w, req, caches = _cache[key]
    return spec, w, req, caches, ratio


def cached_tensor(caches, dtype):
    if caches.dtype == np.uint16:
        return torch.from_numpy(caches.view(np.int16)).cuda().view(torch.bfloat16)
    t = torch.from_numpy(np.ascontiguousarray(caches, dtype=np.float32)).cuda()
    return t.to(torch.bfloat16) if dtype == "bf16" else t


def run_and_compare(cb, name, ratio=None, synthetic=False, seed=None, model=None):
    spec, w, req, caches, ratio = setup_case(name, seed, ratio, synthetic)
    shape = spec.shape.as_dict()
    store = spec.shape.dtype
    own = model is None
    if own:
        model = cb.BlendModel(shape, w, max_tokens=spec.n_tokens, max_chunks=spec.n_chunks)
    tokens = torch.from_numpy(req.tokens).cuda()
    out = model.blend(tokens, cached_tensor(caches, store), req.chunks, ratio, want_dev=True)
    torch.cuda.synchronize()
    ref = oracle.blend(shape, w, req.tokens, caches, req.chunks, ratio, store, keep_exact=True)
    g_sel = out["selected"].cpu().numpy()
    g_dev = out["dev"].cpu().numpy().astype(np.float64)
    diff = parity.assert_selection(g_sel, ref["selected"], ref["dev"], ref["k"])
    if diff:   # follow the GPU through a tie inside the band
        ref = oracle.blend(shape, w, req.tokens, caches, req.chunks, ratio, store, selected=g_sel, keep_exact=True)
    rel_dev = np.max(np.abs(g_dev - ref["dev"]) / (np.abs(ref["dev"]) + 1e-6 * ref["dev"].max()))
    kv_err = parity.assert_kv(parity.bf16_to_f64(out["out_kv"]), ref["out_kv_exact"], store)
    lg_err = parity.assert_logits(parity.bf16_to_f64(out["logits"]), ref["logits"], store)
    assert model.status() == 0, "device status bits set"
    if own:
        model.close()
    return dict(kv_err=kv_err, logits_err=lg_err, dev_rel=float(rel_dev), n_diff=len(diff), k=ref["k"])


def test_tiny_fp32_blend(cb):
    r = run_and_compare(cb, "tiny-fp32")
    print(r)
    assert r["dev_rel"] < 1e-4


@pytest.mark.parametrize("ratio", [0.0, 0.01, 0.5, 1.0])
def test_tiny_fp32_ratio_extremes(cb, ratio):
    run_and_compare(cb, "tiny-fp32", ratio=ratio)


def test_small_bf16_blend(cb):
    r = run_and_compare(cb, "small-bf16")
    print(r)


def test_tensor_core_path_matches_cuda_core_path(cb, monkeypatch):
    """The tcgen05 GEMMs and the CUDA-core GEMMs give the same blend up to summation order."""
    spec, w, req, caches, ratio = setup_case("small-bf16")
    shape = spec.shape.as_dict()
    tokens = torch.from_numpy(req.tokens).cuda()
    outs = []
    for disable in ("0", "1"):
        monkeypatch.setenv("CB_DISABLE_TC", disable)
        model = cb.BlendModel(shape, w, max_tokens=spec.n_tokens, max_chunks=spec.n_chunks)
        outs.append(model.blend(tokens, cached_tensor(caches, "bf16"), req.chunks, ratio, want_dev=True))
        torch.cuda.synchronize()
        assert model.status() == 0
        model.close()
    a, b = outs
    dev_a, dev_b = a["dev"].cpu().numpy(), b["dev"].cpu().numpy()
    assert np.max(np.abs(dev_a - dev_b) / (np.abs(dev_b) + 1e-3 * dev_b.max())) < 1e-2
    kv_a, kv_b = parity.bf16_to_f64(a["out_kv"]), parity.bf16_to_f64(b["out_kv"])
    assert np.max(np.abs(kv_a[0] - kv_b[0])) < 2e-2        # layer 0: one GEMM each way


def test_tiny_prefill_matches_oracle(cb):
    spec, w, req, _, _ = setup_case("tiny-fp32")
    shape = spec.shape.as_dict()
    model = cb.BlendModel(shape, w, max_tokens=spec.n_tokens, max_chunks=spec.n_chunks)
    toks = req.chunk_tokens[1]
    kv = model.prefill_chunk(torch.from_numpy(toks).cuda())
    torch.cuda.synchronize()
    ref = oracle.blend(shape, w, toks, None, [], 0.0, "f32", keep_exact=True)
    parity.assert_kv(parity.bf16_to_f64(kv), ref["out_kv_exact"], "f32", "prefill K/V")
    model.close()


def test_small_bf16_prefill_matches_oracle(cb):
    """cb_blend with no cached chunks is a plain causal prefill (the chunk precompute, and the caller's
    fallback): on the small bf16 configuration, the whole request's 2080 tokens through the tensor-core
    path, every layer's K/V and the last row's logits against the oracle's prefill."""
    spec, w, req, _, _ = setup_case("small-bf16")
    shape = spec.shape.as_dict()
    model = cb.BlendModel(shape, w, max_tokens=spec.n_tokens, max_chunks=spec.n_chunks)
    out = model.blend(torch.from_numpy(req.tokens).cuda(), None, [], 0.0)
    torch.cuda.synchronize()
    assert model.status() == 0
    ref = oracle.blend(shape, w, req.tokens, None, [], 0.0, "bf16", keep_exact=True)
    kv_err = parity.assert_kv(parity.bf16_to_f64(out["out_kv"]), ref["out_kv_exact"], "bf16", "prefill K/V")
    lg_err = parity.assert_logits(parity.bf16_to_f64(out["logits"]), ref["logits"], "bf16")
    print(f"small bf16 prefill of {len(req.tokens)} tokens: K/V max abs {kv_err:.4f}, logits {lg_err:.4f}")
    model.close()


def test_inplace_blend_equals_out_of_place(cb):
    spec, w, req, caches, ratio = setup_case("small-bf16")
    shape = spec.shape.as_dict()
    model = cb.BlendModel(shape, w, max_tokens=spec.n_tokens, max_chunks=spec.n_chunks)
    tokens = torch.from_numpy(req.tokens).cuda()
    cached = cached_tensor(caches, "bf16")
    a = model.blend(tokens, cached, req.chunks, ratio)
    buf = model.kv_buffer(spec.n_tokens)
    buf[:, :, :spec.n_ctx] = cached
    b = model.blend(tokens, buf, req.chunks, ratio, out_kv=buf)
    torch.cuda.synchronize()
    # every reduction of the blend runs in a fixed order, so the two placements give the same bits
    assert torch.equal(a["selected"], b["selected"])
    assert torch.equal(a["out_kv"], b["out_kv"])
    assert torch.equal(a["logits"], b["logits"])
    model.close()


@pytest.mark.parametrize("name", ["tiny-fp32", "small-bf16"])
def test_blend_with_given_set_equals_blend(cb, name):
    """cb_blend_hkvd with the set cb_blend chose gives cb_blend's K/V and logits bit for bit; with another
    set (the oracle's top-k of a perturbed ratio) it matches the oracle following that set."""
    spec, w, req, caches, ratio = setup_case(name)
    shape = spec.shape.as_dict()
    store = spec.shape.dtype
    model = cb.BlendModel(shape, w, max_tokens=spec.n_tokens, max_chunks=spec.n_chunks)
    tokens = torch.from_numpy(req.tokens).cuda()
    cached = cached_tensor(caches, store)
    a = model.blend(tokens, cached, req.chunks, ratio)
    b = model.blend_hkvd(tokens, cached, req.chunks, a["selected"].clone())
    torch.cuda.synchronize()
    assert torch.equal(a["out_kv"], b["out_kv"]) and torch.equal(a["logits"], b["logits"])
    # a set that is not the top-k: every other context row
    sel = np.arange(0, spec.n_ctx, 2, dtype=np.int32)
    c = model.blend_hkvd(tokens, cached, req.chunks, torch.from_numpy(sel).cuda())
    torch.cuda.synchronize()
    assert model.status() == 0
    ref = oracle.blend(shape, w, req.tokens, caches, req.chunks, len(sel) / spec.n_ctx, store, selected=sel,
                       keep_exact=True)
    parity.assert_kv(parity.bf16_to_f64(c["out_kv"]), ref["out_kv_exact"], store)
    parity.assert_logits(parity.bf16_to_f64(c["logits"]), ref["logits"], store)
    # a set out of order is recorded, not faulted
    bad = torch.from_numpy(np.array([5, 3, spec.n_ctx + 7], np.int32)).cuda()
    model.blend_hkvd(tokens, cached, req.chunks, bad)
    torch.cuda.synchronize()
    assert model.status(clear=True) & cb.CB_STATUS_BAD_ROW
    model.close()


@pytest.mark.parametrize("name", ["tiny-fp32", "small-bf16"])
def test_blend_is_deterministic(cb, name):
    """Three blends of the same inputs give the same bits: the split-K partial sums of the residual GEMMs
    are added by the next RMSNorm in slot order, the deviation partials by the top-k kernel in a fixed
    order, and attention merges its key-range parts in part order, so no result depends on which CTA
    finished first."""
    spec, w, req, caches, ratio = setup_case(name)
    shape = spec.shape.as_dict()
    model = cb.BlendModel(shape, w, max_tokens=spec.n_tokens, max_chunks=spec.n_chunks)
    tokens = torch.from_numpy(req.tokens).cuda()
    cached = cached_tensor(caches, spec.shape.dtype)
    outs = [model.blend(tokens, cached, req.chunks, ratio, want_dev=True) for _ in range(3)]
    torch.cuda.synchronize()
    assert model.status() == 0
    for o in outs[1:]:
        for key in ("out_kv", "logits", "selected", "dev"):
            assert torch.equal(o[key], outs[0][key]), key
    model.close()


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_rerope_in_place(cb, dtype):
    """cb_rerope rotates K of every layer by each chunk's delta and leaves V alone."""
    shape = dict(workload.TINY.as_dict(), dtype=dtype)
    ms = workload.ModelShape(**{k: v for k, v in shape.items()})
    w = workload.make_weights(ms, 0)
    model = cb.BlendModel(shape, w, max_tokens=64, max_chunks=8)
    chunks = [(0, 0, 5), (100, 5, 17), (3, 22, 9), (40000, 31, 1), (7, 32, 30)]   # ragged, src past dst
    n_rows = 70
    raw = workload.normal(5, 77, (2, 2, n_rows, 2, 64), 1.0, dtype)
    ref = oracle.rerope(raw, chunks, shape["rope_theta"], dtype)
    kv = cb.to_device(raw)
    cb.cb_rerope(model.handle, kv, n_rows, chunks)
    torch.cuda.synchronize()
    got = parity.bf16_to_f64(kv)
    n_ctx = sum(c[2] for c in chunks)
    base = oracle.to_f64(raw)
    assert np.array_equal(got[:, 1], base[:, 1]), "V changed"
    assert np.array_equal(got[:, :, n_ctx:], base[:, :, n_ctx:]), "rows past the chunks changed"
    tol = 1e-5 if dtype == "f32" else 0.0
    err = np.abs(got[:, 0, :n_ctx] - ref[:, 0, :n_ctx])
    if dtype == "bf16":
        assert np.all(err <= parity.rotation_tol(base[:, 0, :n_ctx], ref[:, 0, :n_ctx])), float(err.max())
    else:
        assert err.max() <= tol, float(err.max())
    model.close()


def test_rerope_in_place_many_slabs(cb):
    """cb_rerope over 2 KB rows (8 KV heads x 128, bf16): many 16-row slabs per layer, a ragged last slab,
    chunk boundaries inside slabs, a one-row chunk, rows past the chunks left alone."""
    ms = workload.ModelShape(2, 1024, 8, 8, 128, 256, 64, 5e5, "bf16")
    w = workload.make_weights(ms, 0)
    model = cb.BlendModel(ms.as_dict(), w, max_tokens=1100, max_chunks=16)
    rng = np.random.default_rng(11)
    chunks, dst = [], 0
    for ln in (37, 200, 1, 333, 64, 299):
        chunks.append((int(rng.integers(0, 30000)), dst, ln))
        dst += ln
    n_ctx, n_rows = dst, 1000
    raw = workload.normal(6, 91, (2, 2, n_rows, 8, 128), 1.0, "bf16")
    ref = oracle.rerope(raw, chunks, ms.rope_theta, "bf16")
    kv = cb.to_device(raw)
    cb.cb_rerope(model.handle, kv, n_rows, chunks)
    torch.cuda.synchronize()
    got = parity.bf16_to_f64(kv)
    base = oracle.to_f64(raw)
    assert np.array_equal(got[:, 1], base[:, 1]), "V changed"
    assert np.array_equal(got[:, :, n_ctx:], base[:, :, n_ctx:]), "rows past the chunks changed"
    err = np.abs(got[:, 0, :n_ctx] - ref[:, 0, :n_ctx])
    assert np.all(err <= parity.rotation_tol(base[:, 0, :n_ctx], ref[:, 0, :n_ctx])), float(err.max())
    model.close()


def test_diag_words_after_a_clean_blend(cb):
    """cb_model_diag: 16 words; after a blend that met no error, the status bits and the record of a
    bounded wait that gave up are both zero."""
    spec, w, req, caches, ratio = setup_case("tiny-fp32")
    model = cb.BlendModel(spec.shape.as_dict(), w, max_tokens=spec.n_tokens, max_chunks=spec.n_chunks)
    tokens = torch.from_numpy(req.tokens).cuda()
    model.blend(tokens, cached_tensor(caches, "f32"), req.chunks, ratio)
    words = cb.cb_model_diag(model.handle)
    assert len(words) == 16
    assert words[0] == 0 and words[1] == 0, words[:8]
    assert model.status() == 0
    model.close()


@pytest.mark.parametrize("n", [1, 5, 8, 9, 100, 3072, 8192, 32768, 100003])
def test_select_hkvd_equals_stable_sort(cb, n):
    """The cluster radix select (cb_select_hkvd, the select step of every blend) against the oracle's
    top-k (a stable sort by decreasing deviation): bit for bit, with many exact ties (values drawn from a
    small set, so ties straddle every CTA's row range and the threshold), zeros, and k from 0 to n."""
    rng = np.random.default_rng(n)
    for trial, pool in enumerate((4, 97, None)):
        if pool is None:
            dev = rng.exponential(1.0, n).astype(np.float32)
        else:
            dev = rng.choice(np.linspace(0.0, 3.0, pool, dtype=np.float32), n)
        d = torch.from_numpy(dev).cuda()
        for k in sorted({0, 1, n // 3, n // 2, n - 1, n} - {-1}):
            if k < 0:
                continue
            out = torch.full((max(k, 1),), -1, dtype=torch.int32, device="cuda")
            cb.cb_select_hkvd(d, n, k, out)
            torch.cuda.synchronize()
            ref = oracle.select_hkvd(dev.astype(np.float64), k)
            assert np.array_equal(out[:k].cpu().numpy(), ref), (n, trial, k)


def test_topk_is_exact_on_gpu_deviations(cb):
    """The GPU's set is exactly the top-k (ties to the lower row) of the GPU's own deviations."""
    spec, w, req, caches, _ = setup_case("small-bf16")
    shape = spec.shape.as_dict()
    model = cb.BlendModel(shape, w, max_tokens=spec.n_tokens, max_chunks=spec.n_chunks)
    tokens = torch.from_numpy(req.tokens).cuda()
    for ratio in (0.0, 0.001, 0.15, 0.5, 0.999, 1.0):
        out = model.blend(tokens, cached_tensor(caches, "bf16"), req.chunks, ratio, want_dev=True)
        torch.cuda.synchronize()
        dev = out["dev"].cpu().numpy()
        assert list(out["selected"].cpu().numpy()) == list(oracle.select_hkvd(dev.astype(np.float64), out["k"]))
    model.close()


def test_validation_errors_enqueue_nothing(cb):
    spec, w, req, caches, _ = setup_case("tiny-fp32")
    shape = spec.shape.as_dict()
    model = cb.BlendModel(shape, w, max_tokens=spec.n_tokens, max_chunks=spec.n_chunks)
    tokens = torch.from_numpy(req.tokens).cuda()
    cached = cached_tensor(caches, "f32")
    bad = [
        dict(ratio=1.5), dict(ratio=-0.1), dict(ratio=float("nan")),
        dict(chunks=[(0, 0, 64), (0, 65, 64), (0, 129, 63)]),           # gap
        dict(chunks=[(0, 0, 64), (-1, 64, 64), (0, 128, 64)]),          # unknown source position
        dict(chunks=[(0, 0, 64), (0, 32, 64), (0, 96, 96)]),            # overlap
        dict(chunks=[(0, 0, 208)]),                                      # no query token
    ]
    for b in bad:
        with pytest.raises(cb.CacheBlendError) as ei:
            model.blend(tokens, cached, b.get("chunks", req.chunks), b.get("ratio", 0.25))
        assert ei.value.code == cb.CB_ERR_INVALID_ARG
    with pytest.raises(cb.CacheBlendError):
        big = torch.zeros(spec.n_tokens + 1, dtype=torch.int32, device="cuda")
        model.blend(big, cached, req.chunks, 0.25)
    torch.cuda.synchronize()
    model.close()


def test_tensor_core_attention_matches_cuda_core_attention(cb, monkeypatch):
    """The tcgen05 attention and the CUDA-core attention give the same blend (same GEMM path)."""
    spec, w, req, caches, ratio = setup_case("small-bf16")
    shape = spec.shape.as_dict()
    tokens = torch.from_numpy(req.tokens).cuda()
    outs = []
    for disable in ("0", "1"):
        monkeypatch.setenv("CB_DISABLE_TC_ATTN", disable)
        model = cb.BlendModel(shape, w, max_tokens=spec.n_tokens, max_chunks=spec.n_chunks)
        outs.append(model.blend(tokens, cached_tensor(caches, "bf16"), req.chunks, ratio, want_dev=True))
        torch.cuda.synchronize()
        assert model.status() == 0
        model.close()
    a, b = outs
    kv_a, kv_b = parity.bf16_to_f64(a["out_kv"]), parity.bf16_to_f64(b["out_kv"])
    assert np.max(np.abs(kv_a[1] - kv_b[1])) < 2e-2        # the check layer: one attention apart
    assert np.max(np.abs(kv_a - kv_b)) < 5e-2


def test_attention_rescale_path_head_dim_128(cb):
    """Large-magnitude keys make the running softmax max jump between key blocks, which exercises the
    tensor-core attention's in-TMEM rescale (warp-collective); head_dim 128 with 8 KV heads."""
    shape = workload.ModelShape(n_layers=2, d_model=256, n_heads=32, n_kv_heads=8, head_dim=128, ffn_hidden=512,
                                vocab=1024, rope_theta=5e5, dtype="bf16")
    w = workload.make_weights(shape, 3)
    chunks = [(0, i * 500, 500) for i in range(4)]
    toks = workload.tokens(3, 7, 2064, 1024)
    caches = workload.synthetic_cache(shape, 3, 2000, 4.0)
    model = cb.BlendModel(shape.as_dict(), w, max_tokens=2064, max_chunks=4)
    out = model.blend(torch.from_numpy(toks).cuda(), cb.to_device(caches), chunks, 0.5, want_dev=True)
    torch.cuda.synchronize()
    assert model.status() == 0
    ref = oracle.blend(shape.as_dict(), w, toks, caches, chunks, 0.5, "bf16", keep_exact=True)
    diff = parity.assert_selection(out["selected"].cpu().numpy(), ref["selected"], ref["dev"], ref["k"])
    assert not diff
    parity.assert_kv(parity.bf16_to_f64(out["out_kv"]), ref["out_kv_exact"], "bf16")
    parity.assert_logits(parity.bf16_to_f64(out["logits"]), ref["logits"], "bf16")
    model.close()


def test_cta_pair_gemms_match_single_cta_gemms(cb, monkeypatch):
    """The CTA-pair tcgen05 GEMMs (M = 256 over two SMs) and the single-CTA ones give the same blend up
    to summation order (split-K partial sums may differ in order)."""
    spec, w, req, caches, ratio = setup_case("small-bf16")
    shape = spec.shape.as_dict()
    tokens = torch.from_numpy(req.tokens).cuda()
    outs = []
    for pair in ("1", "0"):
        monkeypatch.setenv("CB_GEMM_PAIR", pair)
        model = cb.BlendModel(shape, w, max_tokens=spec.n_tokens, max_chunks=spec.n_chunks)
        outs.append(model.blend(tokens, cached_tensor(caches, "bf16"), req.chunks, ratio, want_dev=True))
        torch.cuda.synchronize()
        assert model.status() == 0
        model.close()
    a, b = outs
    dev_a, dev_b = a["dev"].cpu().numpy(), b["dev"].cpu().numpy()
    assert np.max(np.abs(dev_a - dev_b) / (np.abs(dev_b) + 1e-3 * dev_b.max())) < 1e-3
    kv_a, kv_b = parity.bf16_to_f64(a["out_kv"]), parity.bf16_to_f64(b["out_kv"])
    assert np.max(np.abs(kv_a[0] - kv_b[0])) < 1e-2
    assert np.max(np.abs(kv_a - kv_b)) < 3e-2


def test_ragged_projection_shapes(cb):
    """Output widths that are not multiples of a CTA pair's 256 weight rows (d_model 384, KV width 128,
    SwiGLU hidden 704 = 5.5 x 128) and a token count that is not a multiple of 16: the tiles past the
    end read zeros and store nothing."""
    shape = workload.ModelShape(n_layers=3, d_model=384, n_heads=6, n_kv_heads=2, head_dim=64, ffn_hidden=704,
                                vocab=1024, rope_theta=1e4, dtype="bf16")
    w = workload.make_weights(shape, 5)
    chunks = [(0, 0, 100), (0, 100, 77), (0, 177, 64)]
    n_ctx, n_tok = 241, 241 + 19
    toks = workload.tokens(5, 9, n_tok, 1024)
    caches = workload.synthetic_cache(shape, 5, n_ctx, workload.kv_std(shape))
    model = cb.BlendModel(shape.as_dict(), w, max_tokens=n_tok, max_chunks=3)
    out = model.blend(torch.from_numpy(toks).cuda(), cb.to_device(caches), chunks, 0.3, want_dev=True)
    torch.cuda.synchronize()
    assert model.status() == 0
    ref = oracle.blend(shape.as_dict(), w, toks, caches, chunks, 0.3, "bf16", keep_exact=True)
    diff = parity.assert_selection(out["selected"].cpu().numpy(), ref["selected"], ref["dev"], ref["k"])
    if diff:
        ref = oracle.blend(shape.as_dict(), w, toks, caches, chunks, 0.3, "bf16",
                           selected=out["selected"].cpu().numpy(), keep_exact=True)
    parity.assert_kv(parity.bf16_to_f64(out["out_kv"]), ref["out_kv_exact"], "bf16")
    parity.assert_logits(parity.bf16_to_f64(out["logits"]), ref["logits"], "bf16")
    model.close()
