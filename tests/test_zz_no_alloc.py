"""cb_rerope_static -- re-RoPE without any device allocation -- checked against cb_rerope.

Some callers of this library cannot call cudaMalloc: a KV-cache manager that has reserved nearly
all device memory for its own block pool is the usual case.  Creating a model would allocate a
workspace sized for whole blends (and needs the weights), yet moving cached chunks to new positions
needs neither, so cb_rerope_static does it without a model handle, keeping its small per-call table
in a fixed device array inside the library.  These tests call both entry points through the C ABI on
the same inputs, twice in a row with different chunk layouts (the array keeps the previous call's
contents): the two must give the same bits (both rotate through one helper with fixed roundings, from
the same float64 angle table), and both must match the CPU oracle's re-RoPE within the rotation
tolerance of the re-RoPE parity tests.  The file is named to be collected last.
"""
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


LAYOUTS = [
    [(0, 0, 5), (100, 5, 17), (3, 22, 9), (40000, 31, 1), (7, 32, 30)],   # ragged, sources past their targets
    [(9, 0, 40), (0, 40, 20), (512, 60, 8)],
]


def _values(t):
    return t.detach().to(torch.float32).cpu().numpy().astype(np.float64)


@pytest.mark.parametrize("dtype,head_dim", [("f32", 64), ("bf16", 64), ("bf16", 128)])
def test_static_rerope_matches_model_rerope_on_two_calls(cb, dtype, head_dim):
    shape = workload.ModelShape(n_layers=2, d_model=256, n_heads=256 // head_dim * 2, n_kv_heads=2,
                                head_dim=head_dim, ffn_hidden=512, vocab=1024, rope_theta=5e5, dtype=dtype)
    model = cb.BlendModel(shape.as_dict(), workload.make_weights(shape, 0), max_tokens=80, max_chunks=8)
    n_rows = 70
    for call, chunks in enumerate(LAYOUTS):
        raw = workload.normal(5, 80 + call, (2, 2, n_rows, 2, head_dim), 1.0, dtype)
        a, b = cb.to_device(raw), cb.to_device(raw)
        cb.cb_rerope(model.handle, a, n_rows, chunks)
        cb.cb_rerope_static(b, n_rows, 2, 2, head_dim, shape.rope_theta, dtype, chunks)
        torch.cuda.synchronize()
        ga, gb = _values(a), _values(b)
        assert np.array_equal(ga, gb), f"call {call}: cb_rerope_static differs from cb_rerope"
        base = oracle.to_f64(raw)
        ref = oracle.rerope(raw, chunks, shape.rope_theta, dtype)
        n_ctx = sum(c[2] for c in chunks)
        err = np.abs(gb[:, 0, :n_ctx] - ref[:, 0, :n_ctx])
        if dtype == "f32":
            assert err.max() <= 1e-5, float(err.max())
        else:
            assert np.all(err <= parity.rotation_tol(base[:, 0, :n_ctx], ref[:, 0, :n_ctx])), float(err.max())
        assert np.array_equal(gb[:, 1], base[:, 1]), "V must stay untouched"
        assert np.array_equal(gb[:, :, n_ctx:], base[:, :, n_ctx:]), "rows past the chunks must stay untouched"
    assert model.status() == 0
    model.close()


def test_static_rerope_rejects_too_many_chunks(cb):
    n = cb.CB_STATIC_MAX_CHUNKS + 1
    kv = torch.zeros((1, 2, n, 1, 64), dtype=torch.float32, device="cuda")
    with pytest.raises(cb.CacheBlendError) as ei:
        cb.cb_rerope_static(kv, n, 1, 1, 64, 1e4, "f32", [(0, i, 1) for i in range(n)])
    assert ei.value.code == cb.CB_ERR_INVALID_ARG
    assert "limit" in cb.cb_last_error()
    torch.cuda.synchronize()
    assert torch.count_nonzero(kv).item() == 0
