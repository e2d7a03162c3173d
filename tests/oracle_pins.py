"""Checks that pin the CPU oracle to things other than itself.

Each ``check_*`` takes the oracle module (``oracle.cpu_blend``) so that the mutation
tests can plant a mistake in it and confirm that some check fails.
"""
from __future__ import annotations

import numpy as np
import torch

import brute_force as bf
import workload

MICRO = workload.ModelShape(n_layers=3, d_model=64, n_heads=4, n_kv_heads=2, head_dim=16, ffn_hidden=96,
                            vocab=101, rope_theta=1e4, dtype="f32")
MICRO_CFG = MICRO.as_dict()
# ragged chunks (8, 6, 7 tokens) and a 5-token query
MICRO_CHUNK_LENS = (8, 6, 7)
MICRO_QUERY = 5

_cache = {}


def micro_weights():
    if "w" not in _cache:
        _cache["w"] = workload.make_weights(MICRO, seed=11, std=0.1)
    return _cache["w"]


def micro_request():
    """Chunk tokens, chunk layout (src 0, back to back), query, all tokens."""
    if "req" not in _cache:
        chunk_tokens = [workload.tokens(12, 100 + c, n, MICRO.vocab) for c, n in enumerate(MICRO_CHUNK_LENS)]
        chunks, at = [], 0
        for n in MICRO_CHUNK_LENS:
            chunks.append((0, at, n))
            at += n
        q = workload.tokens(12, 999, MICRO_QUERY, MICRO.vocab)
        toks = np.concatenate(chunk_tokens + [q])
        _cache["req"] = (chunk_tokens, chunks, q, toks)
    return _cache["req"]


def brute_caches():
    """Each chunk decoded alone from position 0 by the brute-force decoder (float64, unrounded)."""
    if "caches" not in _cache:
        chunk_tokens, chunks, _, _ = micro_request()
        parts = [bf.full_prefill(MICRO_CFG, micro_weights(), t)[0] for t in chunk_tokens]
        _cache["caches"] = np.concatenate(parts, axis=2)
    return _cache["caches"]


def brute_joint():
    if "joint" not in _cache:
        _, _, _, toks = micro_request()
        _cache["joint"] = bf.full_prefill(MICRO_CFG, micro_weights(), toks)
    return _cache["joint"]


def _close(a, b, tol, what):
    err = float(np.max(np.abs(np.asarray(a, np.float64) - np.asarray(b, np.float64)))) if np.size(a) else 0.0
    assert err <= tol, f"{what}: max abs error {err:.3e} > {tol:.1e}"
    return err


# ------------------------------------------------------------------------------------------------
def check_rope_matrix(ob):
    """rope(x, m) equals the explicit block-diagonal R_m x; R_m is orthogonal; R_0 = I."""
    rng = np.random.default_rng(0)
    for hd, theta in ((16, 1e4), (64, 1e4), (128, 5e5)):
        x = rng.standard_normal((7, 3, hd))
        pos = np.array([0, 1, 5, 63, 511, 4097, 32895])
        got = ob.rope(x, pos, theta)
        for r, m in enumerate(pos):
            R = bf.rotation_matrix(float(m), hd, theta)
            _close(got[r], x[r] @ R.T, 1e-9 * (1 + abs(m)), f"rope vs R_m (hd={hd}, m={m})")
            _close(R @ R.T, np.eye(hd), 1e-12, "R_m orthogonal")
        _close(ob.rope(x, np.zeros(7), theta), x, 0.0, "R_0 = I")


def check_rope_composition(ob):
    """R_{n-p} R_p = R_n (re-RoPE identity, section "位置恢复、KV 存储与加载流水线")."""
    rng = np.random.default_rng(1)
    x = rng.standard_normal((5, 2, 64))
    p = np.array([0, 3, 100, 700, 2000])
    n = np.array([9, 3, 40, 4096, 32000])
    _close(ob.rope(ob.rope(x, p, 1e4), n - p, 1e4), ob.rope(x, n, 1e4), 1e-9, "R_{n-p} R_p vs R_n")


def check_rmsnorm_silu(ob):
    """Closed forms: RMSNorm of a constant vector c*1 is g*c/sqrt(c^2+eps); silu(0)=0,
    silu(x) -> x for large x, silu(-x) = silu(x) - x."""
    g = np.linspace(0.5, 2.0, 32)
    for c in (1e-3, 0.5, -3.0):
        _close(ob.rmsnorm(np.full(32, c), g, 1e-5), g * c / np.sqrt(c * c + 1e-5), 1e-14, "rmsnorm constant")
    x = np.linspace(-8, 8, 101)
    _close(ob.silu(np.zeros(3)), np.zeros(3), 0.0, "silu(0)")
    _close(ob.silu(-x), ob.silu(x) - x, 1e-13, "silu odd part")
    _close(ob.silu(np.array([40.0])), np.array([40.0]), 1e-12, "silu large")


def check_attention_vs_sdpa(ob):
    """Causal GQA attention at arbitrary query positions against torch SDPA (float64)."""
    rng = np.random.default_rng(2)
    for Hq, Hkv in ((4, 4), (4, 2), (8, 2)):
        Nk, hd = 37, 16
        q_pos = np.array([0, 3, 4, 10, 20, 30, 36])
        k_pos = np.arange(Nk)
        q = rng.standard_normal((len(q_pos), Hq, hd))
        k = rng.standard_normal((Nk, Hkv, hd))
        v = rng.standard_normal((Nk, Hkv, hd))
        got = ob.attention(q, k, v, q_pos, k_pos, Hkv)
        mask = torch.from_numpy(k_pos[None, :] <= q_pos[:, None])
        ref = torch.nn.functional.scaled_dot_product_attention(
            torch.from_numpy(q).transpose(0, 1), torch.from_numpy(k).transpose(0, 1),
            torch.from_numpy(v).transpose(0, 1), attn_mask=mask, enable_gqa=True).transpose(0, 1).numpy()
        _close(got, ref, 1e-12, f"attention Hq={Hq} Hkv={Hkv}")
    # a query that sees one key returns that key's value exactly
    one = ob.attention(rng.standard_normal((1, 2, 8)), rng.standard_normal((4, 1, 8)),
                       np.arange(32.0).reshape(4, 1, 8), np.array([0]), np.arange(4), 1)
    _close(one[0, 0], np.arange(8.0), 0.0, "single visible key")


def check_prefill_vs_sequential(ob):
    """Batched prefill equals token-by-token decoding (K/V of every layer and logits)."""
    _, _, _, toks = micro_request()
    got = ob.prefill(MICRO_CFG, micro_weights(), toks, "f64")
    kv, logits = brute_joint()
    _close(got["out_kv"], kv, 1e-10, "prefill K/V")
    _close(got["logits"], logits, 1e-10, "prefill logits")


def check_relative_position(ob):
    """A chunk decoded alone at offset o has, at every layer, K = R_o K(at 0) and the same V;
    so re-RoPE of a cache made at src gives the cache made at dst."""
    chunk_tokens, _, _, _ = micro_request()
    w = micro_weights()
    t = chunk_tokens[1]
    at0, _ = bf.full_prefill(MICRO_CFG, w, t, first_pos=0)
    at9, _ = bf.full_prefill(MICRO_CFG, w, t, first_pos=9)
    moved = ob.rerope(at9, [(9, 0, len(t))], MICRO.rope_theta, "f64")
    _close(moved, at0, 1e-10, "rerope(cache@9 -> 0)")
    dummy = np.zeros(at0.shape[:2] + (9,) + at0.shape[3:])
    pad = np.concatenate([dummy, at0], axis=2)            # rows 0..8 are a dummy chunk
    moved2 = ob.rerope(pad, [(0, 0, 9), (0, 9, len(t))], MICRO.rope_theta, "f64")
    _close(moved2[:, :, 9:], at9, 1e-10, "rerope(cache@0 -> 9)")


def check_r1_full_prefill(ob):
    """ratio 1 (full recompute) reproduces the joint prefill exactly (float64 storage)."""
    _, chunks, _, toks = micro_request()
    got = ob.blend(MICRO_CFG, micro_weights(), toks, brute_caches(), chunks, 1.0, "f64")
    kv, logits = brute_joint()
    _close(got["out_kv"], kv, 1e-10, "r=1 K/V")
    _close(got["logits"], logits, 1e-10, "r=1 logits")


def check_r0_full_reuse(ob):
    """ratio 0 (full KV reuse): context rows are the placed caches at every layer, and the
    query rows are the query decoded after that fixed prefix."""
    _, chunks, q, toks = micro_request()
    got = ob.blend(MICRO_CFG, micro_weights(), toks, brute_caches(), chunks, 0.0, "f64")
    placed = bf.place_chunk_caches(MICRO_CFG, brute_caches(), chunks)
    n_ctx = placed.shape[2]
    _close(got["out_kv"][:, :, :n_ctx], placed, 1e-12, "r=0 context rows")
    qkv, logits = bf.extend_after_prefix(MICRO_CFG, micro_weights(), placed, q)
    _close(got["out_kv"][:, :, n_ctx:], qkv, 1e-10, "r=0 query rows")
    _close(got["logits"], logits, 1e-10, "r=0 logits")
    assert len(got["selected"]) == 0


def check_causal_prefix(ob):
    """The first chunk (placed at 0, prefilled at 0) equals the joint prefill's prefix for every ratio."""
    _, chunks, _, toks = micro_request()
    kv, _ = brute_joint()
    n0 = chunks[0][2]
    for r in (0.0, 0.34, 0.7, 1.0):
        got = ob.blend(MICRO_CFG, micro_weights(), toks, brute_caches(), chunks, r, "f64")
        _close(got["out_kv"][:, :, :n0], kv[:, :, :n0], 1e-10, f"prefix chunk at r={r}")


def check_deviation_definition(ob):
    """The check-layer deviation equals Δkv[j] = ||KV_full[1][j] - KV_pre[1][j]||^2 with KV_full
    the joint prefill (section "核心思想"), and the selection is its top-k."""
    _, chunks, _, toks = micro_request()
    kv_full, _ = brute_joint()
    placed = bf.place_chunk_caches(MICRO_CFG, brute_caches(), chunks)
    n_ctx = placed.shape[2]
    d = kv_full[1, :, :n_ctx] - placed[1]
    page = np.sum(d.reshape(2, n_ctx, -1) ** 2, axis=(0, 2))
    for r in (0.2, 0.5):
        got = ob.blend(MICRO_CFG, micro_weights(), toks, brute_caches(), chunks, r, "f64")
        _close(got["dev"], page, 1e-10 * max(1.0, page.max()), "deviation vs page definition")
        k = int(np.ceil(r * n_ctx - 1e-9))
        assert list(got["selected"]) == bf.top_k_by_sorting(page, k), "selection vs top-k of page Δkv"
    # rows of the first chunk (a true prefix) have zero deviation
    assert np.max(page[:chunks[0][2]]) < 1e-20


def check_topk_vs_sort(ob):
    rng = np.random.default_rng(3)
    for n in (1, 7, 64, 300):
        dev = np.round(rng.random(n) * 10) / 10          # many ties
        dev[rng.random(n) < 0.1] = 0.0
        for k in sorted({0, 1, n // 3, n // 2, n - 1, n}):
            assert list(ob.select_hkvd(dev, k)) == bf.top_k_by_sorting(dev, k), (n, k)


def check_selected_count(ob):
    assert ob.selected_count(192, 0.25) == 48
    assert ob.selected_count(2048, 0.15) == 308
    assert ob.selected_count(3072, 0.15) == 461
    assert ob.selected_count(8192, 0.05) == 410
    assert ob.selected_count(8192, 0.15) == 1229
    assert ob.selected_count(8192, 0.30) == 2458
    assert ob.selected_count(32768, 0.15) == 4916
    assert ob.selected_count(10, 0.1) == 1
    assert ob.selected_count(100, 0.0) == 0 and ob.selected_count(100, 1.0) == 100


def check_round_bf16(ob):
    """Round-to-nearest-even to bfloat16 against torch's float32 -> bfloat16 cast."""
    rng = np.random.default_rng(4)
    x = (rng.standard_normal(20000) * np.exp(rng.uniform(-20, 20, 20000))).astype(np.float32)
    # exact ties: 1 + 2^-8 (even below), 1 + 3 * 2^-8 (even above)
    x = np.concatenate([x, np.array([1 + 2 ** -8, 1 + 3 * 2 ** -8, -(1 + 2 ** -8), 0.0], np.float32)])
    ref = torch.from_numpy(x).to(torch.bfloat16).to(torch.float64).numpy()
    got = ob.round_bf16(x.astype(np.float64))
    assert np.array_equal(got, ref), "round_bf16 vs torch cast"


ALL_CHECKS = [check_rope_matrix, check_rope_composition, check_rmsnorm_silu, check_attention_vs_sdpa,
              check_prefill_vs_sequential, check_relative_position, check_r1_full_prefill,
              check_r0_full_reuse, check_causal_prefix, check_deviation_definition, check_topk_vs_sort,
              check_selected_count, check_round_bf16]


def check_deviation_rows(ob):
    """The row-restricted deviation equals the full blend's deviation on those rows."""
    _, chunks, _, toks = micro_request()
    full = ob.blend(MICRO_CFG, micro_weights(), toks, brute_caches(), chunks, 0.3, "f64")
    rows = [0, 3, 8, 13, 20]
    got = ob.deviation_rows(MICRO_CFG, micro_weights(), toks, brute_caches(), chunks, rows, "f64")
    _close(got, full["dev"][rows], 1e-10 * max(1.0, full["dev"].max()), "deviation_rows vs blend")


ALL_CHECKS.append(check_deviation_rows)


# ------------------------------------------------------------------------------------------------
# gradual filtering (Figure 9): a 5-layer micro model so that the set can shrink more than once
# ------------------------------------------------------------------------------------------------
MICRO5 = workload.ModelShape(n_layers=5, d_model=64, n_heads=4, n_kv_heads=2, head_dim=16, ffn_hidden=96,
                             vocab=101, rope_theta=1e4, dtype="f32")
MICRO5_CFG = MICRO5.as_dict()
# ratios of layers 1..4 over 21 context rows: k = 13, 10, 10, 5 (layer 3 keeps its set); the first
# chunk's 8 rows are a true prefix (zero deviation), so k_1 = 13 takes exactly the other rows
GRADUAL_RATIOS = (0.6, 0.45, 0.45, 0.2)


def micro5_weights():
    if "w5" not in _cache:
        _cache["w5"] = workload.make_weights(MICRO5, seed=13, std=0.1)
    return _cache["w5"]


def micro5_caches():
    if "caches5" not in _cache:
        chunk_tokens, _, _, _ = micro_request()
        parts = [bf.full_prefill(MICRO5_CFG, micro5_weights(), t)[0] for t in chunk_tokens]
        _cache["caches5"] = np.concatenate(parts, axis=2)
    return _cache["caches5"]


def check_gradual_vs_brute_force(ob):
    """The gradual-filtering blend against a row-by-row selective decoder written from the page's
    description of the funnel: K/V of every layer, logits, and each layer's kept rows."""
    _, chunks, _, toks = micro_request()
    got = ob.blend_gradual(MICRO5_CFG, micro5_weights(), toks, micro5_caches(), chunks, GRADUAL_RATIOS, "f64")
    placed = bf.place_chunk_caches(MICRO5_CFG, micro5_caches(), chunks)
    n_ctx = placed.shape[2]
    counts = [int(np.ceil(r * n_ctx - 1e-9)) for r in GRADUAL_RATIOS]
    assert counts == [13, 10, 10, 5] and list(got["counts"]) == counts
    kv, logits, kept = bf.selective_blend(MICRO5_CFG, micro5_weights(), toks, placed, n_ctx, counts)
    for layer in range(1, MICRO5.n_layers):
        assert list(got["sets"][layer]) == kept[layer], f"kept rows of layer {layer}"
    _close(got["out_kv"], kv, 1e-10, "gradual K/V")
    _close(got["logits"], logits, 1e-10, "gradual logits")


def check_gradual_sets_nested(ob):
    """S_{l+1} is a subset of S_l with k_l = ceil(r_l n_ctx) rows; only shrinking layers compare."""
    _, chunks, _, toks = micro_request()
    got = ob.blend_gradual(MICRO5_CFG, micro5_weights(), toks, micro5_caches(), chunks, GRADUAL_RATIOS, "f64")
    sets = got["sets"]
    for layer in range(1, MICRO5.n_layers):
        assert len(sets[layer]) == got["counts"][layer - 1]
        assert np.all(np.diff(sets[layer]) > 0)
        if layer > 1:
            assert set(sets[layer]) <= set(sets[layer - 1]), f"S_{layer} not within S_{layer - 1}"
    assert sorted(got["devs"]) == [1, 2, 4], "deviation compared at the check layer and shrinking layers only"
    # a shrinking layer ranks its candidates by their own deviation at that layer
    for layer in (2, 4):
        cand = sets[layer - 1]
        order = bf.top_k_by_sorting(got["devs"][layer], len(sets[layer]))
        assert list(cand[order]) == list(sets[layer])
    # a schedule whose counts grow is rejected
    try:
        ob.blend_gradual(MICRO5_CFG, micro5_weights(), toks, micro5_caches(), chunks, (0.3, 0.5, 0.5, 0.5), "f64")
    except ValueError:
        pass
    else:
        raise AssertionError("growing schedule accepted")


def check_gradual_constant_is_blend(ob):
    """A constant schedule never shrinks the set: the blend with one selection at the check layer."""
    _, chunks, _, toks = micro_request()
    for r in (0.0, 0.4, 1.0):
        one = ob.blend(MICRO_CFG, micro_weights(), toks, brute_caches(), chunks, r, "f64")
        grad = ob.blend_gradual(MICRO_CFG, micro_weights(), toks, brute_caches(), chunks, (r, r), "f64")
        _close(grad["out_kv"], one["out_kv"], 1e-12, f"constant schedule K/V (r={r})")
        _close(grad["logits"], one["logits"], 1e-12, f"constant schedule logits (r={r})")
        assert list(grad["sets"][1]) == list(one["selected"]) == list(grad["sets"][2])


ALL_CHECKS += [check_gradual_vs_brute_force, check_gradual_sets_nested, check_gradual_constant_is_blend]
