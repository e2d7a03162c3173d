"""The C-ABI library builds, loads and exports every symbol the header declares; host-side
validation that needs no GPU."""
import ctypes
import glob
import os
import re

import pytest

import cacheblend_selective_kv_gb300 as cb
from oracle import selected_count

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    import __graft_entry__
    __graft_entry__.build()
    return cb.lib()


def declared_symbols():
    names = set()
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        text = open(h).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        for m in re.finditer(r"\b(cb_[a-z_0-9]+)\s*\(", text):
            names.add(m.group(1))
    return sorted(names)


def test_header_declares_the_boundary():
    names = declared_symbols()
    for n in cb.EXPORTED:
        assert n in names


def test_every_declared_symbol_is_exported(lib):
    for n in declared_symbols():
        assert hasattr(lib, n), f"{n} declared in include/ but not exported"


def test_selected_count_matches_oracle(lib):
    for n in (0, 1, 7, 192, 2048, 3072, 8192, 32768):
        for r in (0.0, 0.05, 0.1, 0.15, 0.25, 0.3, 0.5, 0.999, 1.0):
            assert cb.cb_selected_count(n, r) == selected_count(n, r), (n, r)
    assert cb.cb_selected_count(10, -0.1) == -1
    assert cb.cb_selected_count(10, 1.5) == -1
    assert cb.cb_selected_count(10, float("nan")) == -1


def _cfg(**kw):
    c = dict(n_layers=2, d_model=256, n_heads=4, n_kv_heads=2, head_dim=64, ffn_hidden=512, vocab=1024,
             rope_theta=1e4, rms_eps=1e-5, dtype="f32", max_tokens=256, max_chunks=8)
    c.update(kw)
    return c


def _fake_weights(L, ptr=4096):
    layer = {k: ptr for k in ("attn_norm", "wq", "wk", "wv", "wo", "mlp_norm", "w_gate", "w_up", "w_down")}
    return dict(embed=ptr, final_norm=ptr, lm_head=ptr, layers=[dict(layer) for _ in range(L)])


@pytest.mark.parametrize("bad,code", [
    (dict(head_dim=96), cb.CB_ERR_UNSUPPORTED),
    (dict(n_heads=6, n_kv_heads=4), cb.CB_ERR_INVALID_ARG),
    (dict(n_layers=1), cb.CB_ERR_INVALID_ARG),
    (dict(d_model=200), cb.CB_ERR_UNSUPPORTED),
    (dict(max_tokens=0), cb.CB_ERR_INVALID_ARG),
    (dict(max_chunks=cb.CB_MAX_CHUNKS + 1), cb.CB_ERR_INVALID_ARG),
    (dict(rope_theta=0.0), cb.CB_ERR_INVALID_ARG),
])
def test_create_rejects_bad_config_before_touching_the_gpu(lib, bad, code):
    with pytest.raises(cb.CacheBlendError) as ei:
        cb.cb_model_create(_cfg(**bad), _fake_weights(_cfg(**bad)["n_layers"]))
    assert ei.value.code == code
    assert cb.cb_last_error()


def test_create_rejects_null_and_misaligned_weights(lib):
    w = _fake_weights(2)
    w["layers"][1]["wo"] = 0
    with pytest.raises(cb.CacheBlendError) as ei:
        cb.cb_model_create(_cfg(), w)
    assert ei.value.code == cb.CB_ERR_INVALID_ARG
    w = _fake_weights(2)
    w["layers"][0]["w_up"] = 4096 + 8
    with pytest.raises(cb.CacheBlendError) as ei:
        cb.cb_model_create(_cfg(), w)
    assert "aligned" in cb.cb_last_error()


def test_calls_reject_null_model(lib):
    with pytest.raises(cb.CacheBlendError):
        cb.cb_blend(0, 4096, 10, 0, [], 0.1, 4096, 4096, stream=0)
    with pytest.raises(cb.CacheBlendError):
        cb.cb_rerope(0, 4096, 10, [(0, 0, 10)], stream=0)
    assert lib.cb_model_destroy(None) == cb.CB_OK


def test_select_hkvd_validation_enqueues_nothing(lib):
    """cb_select_hkvd rejects k outside [0, n] and null buffers on the host; k = 0 is a no-op."""
    for n, k in ((10, 11), (10, -1), (-1, 0)):
        with pytest.raises(cb.CacheBlendError) as ei:
            cb.cb_select_hkvd(4096, n, k, 4096, stream=0)
        assert ei.value.code == cb.CB_ERR_INVALID_ARG
    with pytest.raises(cb.CacheBlendError):
        cb.cb_select_hkvd(0, 10, 3, 4096, stream=0)
    cb.cb_select_hkvd(0, 10, 0, 0, stream=0)


def test_loading_controller_matches_oracle(lib):
    """The library's loading-controller arithmetic against the oracle's (host code, no GPU)."""
    from oracle import accounting
    for ptk in (131072.0, 524288.0, 163840.0):
        for n in (0, 512, 3072, 4096, 32768):
            for bw in (4.8e9, 5153960755.2, 2.5e10, 4.5e11):
                assert cb.cb_load_time(ptk, n, bw) == accounting.load_time(ptk, n, bw)
    for tp in (0.0, 0.02, 0.4667, 1.0, 3.0):
        for tl in (0.0, 0.004, 0.016, 0.05, 0.4, 2.0, 5.0):
            for rmin in (0.0, 0.15, 0.3):
                assert cb.cb_controller_ratio(tp, tl, rmin) == accounting.controller_ratio(tp, tl, rmin), (tp, tl, rmin)
    assert cb.cb_load_time(1.0, 1, 0.0) == -1.0
    assert cb.cb_controller_ratio(1.0, 0.1, 1.5) == -1.0
    tiers = [(2.0e11, 3.0), (4.8e9, 0.1), (2.5e10, 0.5), (2.5e10, 0.5)]
    for n in (512, 4096, 32768):
        for tp in (0.05, 0.5, 5.0, 50.0):
            for rmin in (0.05, 0.15, 1.0):
                assert cb.cb_pick_storage(tiers, 524288.0, n, tp, rmin) == \
                    accounting.pick_storage(tiers, 524288.0, n, tp, rmin), (n, tp, rmin)
    with pytest.raises(cb.CacheBlendError):
        cb.cb_pick_storage([], 1.0, 1, 1.0)


class _PagesModel:
    """Reference of the page bookkeeping rules (host logic): counts, lowest-free-first allocation,
    copy-on-write for shared pages."""

    def __init__(self, n):
        self.count = [0] * n

    def alloc(self, k):
        free = [i for i, c in enumerate(self.count) if c == 0]
        if k > len(free):
            return None
        for i in free[:k]:
            self.count[i] = 1
        return free[:k]

    def retain(self, ids):
        for i in ids:
            self.count[i] += 1

    def release(self, ids):
        for i in ids:
            self.count[i] -= 1

    def plan_write(self, table):
        need = sum(1 for t in table if self.count[t] > 1)
        if need > self.count.count(0):
            return None
        dst = []
        for t in table:
            if self.count[t] > 1:
                new = self.alloc(1)[0]
                self.count[t] -= 1
                dst.append(new)
            else:
                dst.append(t)
        return dst, need


def test_page_bookkeeping_matches_reference(lib):
    import random
    rng = random.Random(5)
    n = 64
    P, M = cb.Pages(n), _PagesModel(n)
    held = []                                    # tables of live "requests"
    for step in range(400):
        op = rng.random()
        if op < 0.35:
            k = rng.randint(1, 6)
            want = M.alloc(k)
            if want is None:
                with pytest.raises(cb.CacheBlendError):
                    P.alloc(k)
            else:
                assert P.alloc(k) == want
                held.append(list(want))
        elif op < 0.55 and held:
            t = rng.choice(held)
            share = t[: rng.randint(1, len(t))]
            P.retain(share)
            M.retain(share)
            held.append(list(share))
        elif op < 0.75 and held:
            t = rng.choice(held)
            want = M.plan_write(t)
            if want is None:
                with pytest.raises(cb.CacheBlendError):
                    P.plan_write(t)
            else:
                got = P.plan_write(t)
                assert got == (want[0], want[1])
                t[:] = want[0]
        elif held:
            t = held.pop(rng.randrange(len(held)))
            P.release(t)
            M.release(t)
        for i in range(n):
            assert P.count(i) == M.count[i]
        assert P.free() == M.count.count(0)
    with pytest.raises(cb.CacheBlendError):
        P.release([n + 3])
    assert P.count(-1) == -1
    P.close()


def test_gradual_layout_matches_oracle_sets(lib):
    """cb_gradual_layout (the order of cb_blend_gradual's out_selected and out_dev) against the layers the
    oracle's blend_gradual compares on a 5-layer fp32 model: its `devs` keys (the layers that rank rows) in
    layer order, the size of each such layer's set and the length of its deviation vector.  Invalid
    schedules are rejected."""
    import numpy as np
    import oracle
    import workload
    shape = workload.ModelShape(n_layers=5, d_model=256, n_heads=4, n_kv_heads=2, head_dim=64, ffn_hidden=512,
                                vocab=1024, rope_theta=1e4, dtype="f32")
    w = workload.make_weights(shape, 0)
    chunk_tokens = [workload.tokens(0, 10 + c, 64, shape.vocab) for c in range(3)]
    chunks = [(0, 64 * c, 64) for c in range(3)]
    toks = np.concatenate(chunk_tokens + [workload.tokens(0, 99, 16, shape.vocab)])
    caches = oracle.chunk_caches(shape.as_dict(), w, chunk_tokens, chunks, "f32")
    n_ctx = 192
    for ratios in ([0.5, 0.4, 0.4, 0.2], [0.3, 0.3, 0.3, 0.3], [0.5, 0.25, 0.0, 0.0], [1.0, 0.5, 0.5, 0.1]):
        ref = oracle.blend_gradual(shape.as_dict(), w, toks, caches, chunks, ratios, "f32")
        got = cb.cb_gradual_layout(n_ctx, ratios)
        layers = sorted(ref["devs"])
        assert [l for l, _, _ in got] == layers, ratios
        assert [kept for _, kept, _ in got] == [len(ref["sets"][l]) for l in layers], ratios
        assert [c for _, _, c in got] == [len(ref["devs"][l]) for l in layers], ratios
    with pytest.raises(ValueError):
        cb.cb_gradual_layout(n_ctx, [0.2, 0.3, 0.3, 0.3])          # growing
    with pytest.raises(ValueError):
        cb.cb_gradual_layout(n_ctx, [0.2, 1.5, 0.1, 0.1])          # ratio outside [0, 1]
    r = (ctypes.c_double * 4)(0.5, 0.4, 0.3, 0.2)
    assert lib.cb_gradual_layout(n_ctx, r, 4, None, None, None, 2) < 0   # more comparing layers than entries
    assert lib.cb_gradual_layout(n_ctx, r, 4, None, None, None, 4) == 4
