"""Plant plausible mistakes in the CPU oracle and confirm that a pin catches each one: in its building
blocks (RoPE, attention, RMSNorm, deviation, selection, rounding, gradual counts) and in the blend's own
control flow (which rows compete for selection, scatter before attention, which keys later layers see,
which row gives the logits).

Every mistake is planted in the oracle module on the CPU (monkeypatch), never in the
CUDA path."""
import inspect
import textwrap

import numpy as np
import pytest

import oracle.cpu_blend as ob
import oracle_pins as pins

_orig_rope, _orig_attention, _orig_rmsnorm = ob.rope, ob.attention, ob.rmsnorm
_orig_dev, _orig_sel, _orig_freqs, _orig_silu = ob.deviation, ob.select_hkvd, ob.rope_freqs, ob.silu
_orig_rerope, _orig_round = ob.rerope, ob.round_bf16
_orig_counts = ob.gradual_counts
_orig_blend = ob.blend


def rope_sign_flipped(x, pos, theta):
    return _orig_rope(x, -np.asarray(pos), theta)


def rope_freq_halved(hd, theta):
    return np.power(float(theta), -np.arange(hd // 2, dtype=np.float64) / hd)


def rope_half_split(x, pos, theta):
    """(i, i + hd/2) pairing instead of adjacent pairs."""
    hd = x.shape[-1]
    perm = np.arange(hd).reshape(2, hd // 2).T.reshape(-1)
    inv = np.argsort(perm)
    return _orig_rope(np.asarray(x)[..., perm], pos, theta)[..., inv]


def attention_gqa_modulo(q, k, v, q_pos, k_pos, n_kv_heads):
    Hq = q.shape[1]
    out = np.empty(q.shape, np.float64)
    for h in range(Hq):
        g = h % n_kv_heads
        out[:, h:h + 1] = _orig_attention(q[:, h:h + 1], k[:, g:g + 1], v[:, g:g + 1], q_pos, k_pos, 1)
    return out


def attention_no_scale(q, k, v, q_pos, k_pos, n_kv_heads):
    return _orig_attention(q * np.sqrt(q.shape[-1]), k, v, q_pos, k_pos, n_kv_heads)


def attention_strict_causal(q, k, v, q_pos, k_pos, n_kv_heads):
    """Masks the diagonal too (key at the query's own position hidden) -- but keeps row 0 alive."""
    return _orig_attention(q, k, v, np.asarray(q_pos) - 0.5 + (np.asarray(q_pos) == 0), k_pos, n_kv_heads)


def rmsnorm_no_eps(x, g, eps):
    return _orig_rmsnorm(x, g, 0.0)


def rmsnorm_mean_abs(x, g, eps):
    return x * g / (np.mean(np.abs(x), axis=-1, keepdims=True) + eps)


def silu_is_sigmoid(x):
    return 1.0 / (1.0 + np.exp(-x))


def deviation_k_only(k_new, v_new, k_pre, v_pre):
    return _orig_dev(k_new, v_new * 0, k_pre, v_pre * 0)


def deviation_unsquared(k_new, v_new, k_pre, v_pre):
    return np.sqrt(_orig_dev(k_new, v_new, k_pre, v_pre)) + np.abs(k_new - k_pre).reshape(len(k_new), -1).sum(1)


def select_ties_high(dev, k):
    n = len(dev)
    order = np.lexsort((-np.arange(n), -np.asarray(dev)))
    return np.sort(order[:k])


def select_smallest(dev, k):
    return np.sort(np.argsort(np.asarray(dev), kind="stable")[:k])


def rerope_wrong_direction(cached_kv, chunks, theta, store, out=None):
    return _orig_rerope(cached_kv, [(dst, src, ln) for src, dst, ln in chunks], theta, store, out=out)


def round_truncates(x):
    m, e = np.frexp(np.asarray(x, np.float64))
    return np.ldexp(np.trunc(np.ldexp(m, 8)), e - 8)


def gradual_counts_floor(n_ctx, ratios):
    return [int(np.floor(float(r) * n_ctx)) for r in ratios]


def gradual_counts_first_only(n_ctx, ratios):
    """The set chosen at the check layer kept to the end (no shrinking)."""
    ks = _orig_counts(n_ctx, ratios)
    return [ks[0]] * len(ks)


def rerope_rotates_v(cached_kv, chunks, theta, store, out=None):
    """V rotated by the position delta as well as K."""
    res = _orig_rerope(cached_kv, chunks, theta, store)
    swapped = np.ascontiguousarray(np.asarray(cached_kv)[:, ::-1])
    res[:, 1] = _orig_rerope(swapped, chunks, theta, store)[:, 0]
    if out is not None:
        out[...] = res
    return res


def _mutated(fn, *edits):
    """`fn` recompiled from its own source with snippets replaced, given as (old, new) pairs.  Each old
    snippet must occur once, so a change to the oracle that removes it fails loudly here instead of
    planting nothing."""
    src = textwrap.dedent(inspect.getsource(fn))
    for old, new in edits:
        assert src.count(old) == 1, f"mutation anchor not found once in {fn.__name__}: {old!r}"
        src = src.replace(old, new)
    ns = dict(vars(ob))
    exec(compile(src, f"<mutated {fn.__name__}>", "exec"), ns)
    return ns[fn.__name__]


# the blend's own control flow
blend_query_rows_in_pool = _mutated(          # query rows (no cache: compared with zeros) compete for the k slots
    _orig_blend,
    ("sel = select_hkvd(dev, kk) if selected is None",
     "sel = select_hkvd(np.concatenate([dev, deviation(k_new[n_ctx:], v_new[n_ctx:], 0 * k_new[n_ctx:], "
     "0 * v_new[n_ctx:])]), kk) if selected is None"))
blend_query_rows_in_pool.__name__ = "blend_query_rows_in_pool"
blend_attends_before_scatter = _mutated(
    _orig_blend,
    ("    out_kv[1, 0, A] = round_store(k_new[A], store)\n",
     "    stale = out_kv[1].astype(np.float64).copy()\n    out_kv[1, 0, A] = round_store(k_new[A], store)\n"),
    ("o = attention(q[A], out_kv[1, 0].astype(np.float64), out_kv[1, 1].astype(np.float64), A, pos, Hkv)",
     "o = attention(q[A], stale[0], stale[1], A, pos, Hkv)"))
blend_attends_before_scatter.__name__ = "blend_attends_before_scatter"
blend_attends_recomputed_rows_only = _mutated(
    _orig_blend,
    ("o = attention(q, out_kv[layer, 0].astype(np.float64), out_kv[layer, 1].astype(np.float64), A, pos, Hkv)",
     "o = attention(q, out_kv[layer, 0, A].astype(np.float64), out_kv[layer, 1, A].astype(np.float64), A, A, Hkv)"))
blend_attends_recomputed_rows_only.__name__ = "blend_attends_recomputed_rows_only"
blend_logits_of_first_row = _mutated(_orig_blend, ("logits = m.logits(hA[-1])", "logits = m.logits(hA[0])"))
blend_logits_of_first_row.__name__ = "blend_logits_of_first_row"


MUTATIONS = [
    ("rope", rope_sign_flipped), ("rope_freqs", rope_freq_halved), ("rope", rope_half_split),
    ("attention", attention_gqa_modulo), ("attention", attention_no_scale), ("attention", attention_strict_causal),
    ("rmsnorm", rmsnorm_no_eps), ("rmsnorm", rmsnorm_mean_abs), ("silu", silu_is_sigmoid),
    ("deviation", deviation_k_only), ("deviation", deviation_unsquared),
    ("select_hkvd", select_ties_high), ("select_hkvd", select_smallest),
    ("rerope", rerope_wrong_direction), ("round_bf16", round_truncates),
    ("gradual_counts", gradual_counts_floor), ("gradual_counts", gradual_counts_first_only),
    ("rerope", rerope_rotates_v),
    ("blend", blend_query_rows_in_pool), ("blend", blend_attends_before_scatter),
    ("blend", blend_attends_recomputed_rows_only), ("blend", blend_logits_of_first_row),
]


@pytest.mark.parametrize("name,bad", MUTATIONS, ids=[m[1].__name__ for m in MUTATIONS])
def test_pins_catch_mutation(monkeypatch, name, bad):
    monkeypatch.setattr(ob, name, bad)
    caught = []
    for check in pins.ALL_CHECKS:
        try:
            check(ob)
        except Exception:          # an assertion or a crash: either way the pin fails
            caught.append(check.__name__)
    assert caught, f"no pin caught the planted mistake {bad.__name__}"
