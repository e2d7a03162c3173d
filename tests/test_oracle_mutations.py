"""Plant plausible mistakes in the CPU oracle and confirm that a pin catches each one.

Every mistake is planted in the oracle module on the CPU (monkeypatch), never in the
CUDA path."""
import numpy as np
import pytest

import oracle.cpu_blend as ob
import oracle_pins as pins

_orig_rope, _orig_attention, _orig_rmsnorm = ob.rope, ob.attention, ob.rmsnorm
_orig_dev, _orig_sel, _orig_freqs, _orig_silu = ob.deviation, ob.select_hkvd, ob.rope_freqs, ob.silu
_orig_rerope, _orig_round = ob.rerope, ob.round_bf16
_orig_counts = ob.gradual_counts


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


def rerope_wrong_direction(cached_kv, chunks, theta, store):
    return _orig_rerope(cached_kv, [(dst, src, ln) for src, dst, ln in chunks], theta, store)


def round_truncates(x):
    m, e = np.frexp(np.asarray(x, np.float64))
    return np.ldexp(np.trunc(np.ldexp(m, 8)), e - 8)


def gradual_counts_floor(n_ctx, ratios):
    return [int(np.floor(float(r) * n_ctx)) for r in ratios]


def gradual_counts_first_only(n_ctx, ratios):
    """The set chosen at the check layer kept to the end (no shrinking)."""
    ks = _orig_counts(n_ctx, ratios)
    return [ks[0]] * len(ks)


MUTATIONS = [
    ("rope", rope_sign_flipped), ("rope_freqs", rope_freq_halved), ("rope", rope_half_split),
    ("attention", attention_gqa_modulo), ("attention", attention_no_scale), ("attention", attention_strict_causal),
    ("rmsnorm", rmsnorm_no_eps), ("rmsnorm", rmsnorm_mean_abs), ("silu", silu_is_sigmoid),
    ("deviation", deviation_k_only), ("deviation", deviation_unsquared),
    ("select_hkvd", select_ties_high), ("select_hkvd", select_smallest),
    ("rerope", rerope_wrong_direction), ("round_bf16", round_truncates),
    ("gradual_counts", gradual_counts_floor), ("gradual_counts", gradual_counts_first_only),
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
