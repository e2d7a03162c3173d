"""GPU tests of the paged blended K/V: gather/scatter through block tables, the blend over a paged pool
(chunk caches read through one table, blended K/V written through another, copy-on-write for shared
pages), and bad page ids recorded, not faulted."""
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


def pool_rows(pool, table, P, n_rows):
    """Logical rows 0..n_rows-1 read from a pool [L][2][n_pages*P][...] through a block table (reference)."""
    j = np.arange(n_rows)
    rows = np.asarray(table)[j // P] * P + j % P
    return pool[:, :, torch.from_numpy(rows).to(pool.device)]


@pytest.mark.parametrize("P", [16, 64, 256])
def test_gather_scatter_round_trip(cb, P):
    import test_gpu_gradual as tg
    w, toks, chunks, caches = tg.tiny5_case()
    model = cb.BlendModel(tg.TINY5.as_dict(), w, max_tokens=len(toks), max_chunks=len(chunks))
    n_rows = 197                                       # ragged: not a multiple of the page size
    n_pages = (n_rows + P - 1) // P + 5
    g = torch.Generator().manual_seed(P)
    pool = torch.randn((5, 2, n_pages * P, 2, 64), generator=g).cuda()
    table = torch.randperm(n_pages, generator=g)[: (n_rows + P - 1) // P].to(torch.int32)
    out = torch.empty((5, 2, n_rows, 2, 64), device="cuda")
    cb.cb_kv_gather_pages(model.handle, pool, n_pages, P, table.cuda(), n_rows, out)
    torch.cuda.synchronize()
    assert torch.equal(out, pool_rows(pool, table.numpy(), P, n_rows))
    pool2 = torch.zeros_like(pool)
    cb.cb_kv_scatter_pages(model.handle, out, n_rows, pool2, n_pages, P, table.cuda())
    torch.cuda.synchronize()
    assert torch.equal(pool_rows(pool2, table.numpy(), P, n_rows), out)
    assert model.status() == 0
    model.close()


@pytest.mark.parametrize("P,ratios", [(16, (0.3, 0.3, 0.3, 0.3)), (64, (0.5, 0.35, 0.35, 0.2)), (128, (0.25,) * 4)])
def test_paged_blend_equals_contiguous(cb, P, ratios):
    """Chunk caches scattered over shuffled pages; the first chunk's pages shared with another request
    (copy-on-write through the host page manager).  The blend over the pool equals the contiguous blend
    bit for bit, lands in the destination pages, and leaves the shared pages untouched."""
    import test_gpu_gradual as tg
    w, toks, chunks, caches = tg.tiny5_case()
    n_ctx, N = sum(c[2] for c in chunks), len(toks)
    model = cb.BlendModel(tg.TINY5.as_dict(), w, max_tokens=N, max_chunks=len(chunks))
    t = torch.from_numpy(toks).cuda()
    ref = model.blend_gradual(t, tg.device_cache(caches, "f32"), chunks, ratios)
    nb = (N + P - 1) // P
    n_pages = 3 * nb + 4
    pages = cb.Pages(n_pages)
    scramble = pages.alloc(n_pages)                     # take them all, then give back a shuffled subset
    rng = np.random.default_rng(P)
    keep = list(rng.permutation(scramble)[:nb])
    pages.release([p for p in scramble if p not in keep])
    src = keep                                          # the request's block table
    shared = src[: max(1, (chunks[0][2] // P))]         # another request holds the first chunk's pages
    pages.retain(shared)
    dst, n_cow = pages.plan_write(src)
    assert n_cow == len(shared) and all(d != s for d, s in zip(dst[:len(shared)], shared))
    pool = torch.zeros((5, 2, n_pages * P, 2, 64), device="cuda")
    ctx = tg.device_cache(caches, "f32")
    cb.cb_kv_scatter_pages(model.handle, ctx, n_ctx, pool, n_pages, P, torch.tensor(src, dtype=torch.int32).cuda())
    before = pool.clone()
    work = model.kv_buffer(N)
    logits = torch.empty(1024, device="cuda")
    cb.cb_blend_paged(model.handle, t, N, pool, n_pages, P, torch.tensor(src, dtype=torch.int32).cuda(),
                      torch.tensor(dst, dtype=torch.int32).cuda(), chunks, ratios, work, logits)
    torch.cuda.synchronize()
    assert model.status() == 0
    assert torch.equal(work, ref["out_kv"])
    assert torch.equal(logits, ref["logits"])
    assert torch.equal(pool_rows(pool, dst, P, N), ref["out_kv"])
    for sp in shared:                                   # shared pages are only read
        assert torch.equal(pool[:, :, sp * P:(sp + 1) * P], before[:, :, sp * P:(sp + 1) * P])
    pages.close()
    model.close()


def test_paged_blend_small_bf16_parity(cb):
    spec = workload.WORKLOADS["small-bf16"]
    shape, seed, ratio = spec.shape, spec.seeds[0], spec.ratios[0]
    w = workload.make_weights(shape, seed)
    req = workload.make_request(spec, seed, ratio)
    caches = oracle.chunk_caches(shape.as_dict(), w, req.chunk_tokens, req.chunks, "bf16").astype(np.float32)
    P, N, n_ctx = 32, spec.n_tokens, spec.n_ctx
    nb = (N + P - 1) // P
    n_pages = nb + 7
    table = torch.from_numpy(np.random.default_rng(3).permutation(n_pages)[:nb].astype(np.int32)).cuda()
    model = cb.BlendModel(shape.as_dict(), w, max_tokens=N, max_chunks=spec.n_chunks)
    pool = torch.zeros((shape.n_layers, 2, n_pages * P, shape.n_kv_heads, shape.head_dim), dtype=torch.bfloat16,
                       device="cuda")
    ctx = torch.from_numpy(caches).cuda().to(torch.bfloat16)
    cb.cb_kv_scatter_pages(model.handle, ctx, n_ctx, pool, n_pages, P, table)
    work = model.kv_buffer(N)
    logits = torch.empty(shape.vocab, device="cuda")
    cb.cb_blend_paged(model.handle, torch.from_numpy(req.tokens).cuda(), N, pool, n_pages, P, table, table,
                      req.chunks, (ratio,) * (shape.n_layers - 1), work, logits)
    torch.cuda.synchronize()
    assert model.status() == 0
    got = pool_rows(pool, table.cpu().numpy(), P, N)
    assert torch.equal(got, work)
    ref = oracle.blend(shape.as_dict(), w, req.tokens, caches, req.chunks, ratio, "bf16", keep_exact=True)
    parity.assert_kv(parity.bf16_to_f64(got), ref["out_kv_exact"], "bf16")
    parity.assert_logits(parity.bf16_to_f64(logits), ref["logits"], "bf16")
    model.close()


def test_bad_page_id_is_recorded_not_faulted(cb):
    """A page id past the pool is skipped by the kernels and reported in the status word."""
    import test_gpu_gradual as tg
    w, toks, chunks, caches = tg.tiny5_case()
    model = cb.BlendModel(tg.TINY5.as_dict(), w, max_tokens=len(toks), max_chunks=len(chunks))
    P, n_pages = 16, 8
    pool = torch.zeros((5, 2, n_pages * P, 2, 64), device="cuda")
    table = torch.tensor([0, 1, 99, 2], dtype=torch.int32, device="cuda")
    out = torch.full((5, 2, 64, 2, 64), 7.0, device="cuda")
    cb.cb_kv_gather_pages(model.handle, pool, n_pages, P, table, 64, out)
    torch.cuda.synchronize()
    assert model.status(clear=True) & cb.CB_STATUS_BAD_ROW
    assert torch.all(out[:, :, 32:48] == 7.0) and torch.all(out[:, :, :32] == 0.0)
    model.close()
