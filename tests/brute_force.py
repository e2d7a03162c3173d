"""Brute-force reference used only to pin the CPU oracle (tiny inputs only).

Written independently of ``oracle/``: it decodes one token at a time with a
growing KV cache, builds each RoPE rotation as an explicit block-diagonal
matrix R_m from its definition (CacheBlend deep-dive page, section
"位置恢复、KV 存储与加载流水线"), and loops over heads and cached keys.
"""
from __future__ import annotations

import math

import numpy as np


def f64(a):
    a = np.asarray(a)
    if a.dtype == np.uint16:
        return (a.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    return a.astype(np.float64)


def rotation_matrix(m: float, hd: int, theta: float) -> np.ndarray:
    """R_m: block diagonal, block i = [[cos a, -sin a], [sin a, cos a]], a = m * theta^(-2i/hd)."""
    R = np.zeros((hd, hd))
    for i in range(hd // 2):
        a = m * theta ** (-(2.0 * i) / hd)
        R[2 * i, 2 * i] = math.cos(a)
        R[2 * i, 2 * i + 1] = -math.sin(a)
        R[2 * i + 1, 2 * i] = math.sin(a)
        R[2 * i + 1, 2 * i + 1] = math.cos(a)
    return R


def _norm(x, g, eps):
    return x * g / math.sqrt(float(np.dot(x, x)) / x.size + eps)


def _sigmoid_gate(x):
    return np.array([xi / (1.0 + math.exp(-xi)) for xi in x])


class SequentialDecoder:
    """Llama-style decoder run token by token over a KV cache."""

    def __init__(self, cfg: dict, weights: dict):
        self.c = cfg
        self.L = cfg["n_layers"]
        self.Hq, self.Hkv, self.hd = cfg["n_heads"], cfg["n_kv_heads"], cfg["head_dim"]
        self.theta, self.eps = cfg["rope_theta"], cfg.get("rms_eps", 1e-5)
        self.E = f64(weights["embed"])
        self.head = f64(weights["lm_head"])
        self.gf = f64(weights["final_norm"])
        self.layers = [{k: f64(v) for k, v in lw.items()} for lw in weights["layers"]]
        # cache[layer] = list of (position, K [Hkv][hd], V [Hkv][hd])
        self.cache = [[] for _ in range(self.L)]
        self._R = {}

    def R(self, m):
        if m not in self._R:
            self._R[m] = rotation_matrix(m, self.hd, self.theta)
        return self._R[m]

    def add_prefix(self, layer: int, pos: int, k: np.ndarray, v: np.ndarray):
        self.cache[layer].append((pos, np.array(k, np.float64), np.array(v, np.float64)))

    def step(self, token: int, pos: int):
        """Run one token through every layer; append its K/V; return its final hidden state."""
        hd, group = self.hd, self.Hq // self.Hkv
        h = self.E[token].copy()
        for li, W in enumerate(self.layers):
            x = _norm(h, W["attn_norm"], self.eps)
            Rm = self.R(pos)
            q = [Rm @ (W["wq"][i * hd:(i + 1) * hd] @ x) for i in range(self.Hq)]
            k = np.stack([Rm @ (W["wk"][i * hd:(i + 1) * hd] @ x) for i in range(self.Hkv)])
            v = np.stack([W["wv"][i * hd:(i + 1) * hd] @ x for i in range(self.Hkv)])
            self.cache[li].append((pos, k, v))
            o = []
            for i in range(self.Hq):
                g = i // group
                vis = [(kk[g], vv[g]) for (p, kk, vv) in self.cache[li] if p <= pos]
                s = [float(np.dot(q[i], kj)) / math.sqrt(hd) for kj, _ in vis]
                mx = max(s)
                e = [math.exp(sj - mx) for sj in s]
                z = sum(e)
                o.append(sum((ej / z) * vj for ej, (_, vj) in zip(e, vis)))
            h = h + W["wo"] @ np.concatenate(o)
            x = _norm(h, W["mlp_norm"], self.eps)
            h = h + W["w_down"] @ (_sigmoid_gate(W["w_gate"] @ x) * (W["w_up"] @ x))
        return h

    def logits(self, h):
        return self.head @ _norm(h, self.gf, self.eps)

    def kv(self, rows=None) -> np.ndarray:
        """Cache as [L][2][n][Hkv][hd], in insertion order."""
        n = len(self.cache[0])
        out = np.zeros((self.L, 2, n, self.Hkv, self.hd))
        for li in range(self.L):
            for j, (_, k, v) in enumerate(self.cache[li]):
                out[li, 0, j], out[li, 1, j] = k, v
        return out


def full_prefill(cfg, weights, tokens, first_pos: int = 0):
    """Decode every token from an empty cache at positions first_pos, first_pos+1, ...
    Returns (kv [L][2][n][Hkv][hd], logits of the last token)."""
    dec = SequentialDecoder(cfg, weights)
    h = None
    for j, t in enumerate(tokens):
        h = dec.step(int(t), first_pos + j)
    return dec.kv(), dec.logits(h)


def place_chunk_caches(cfg, cached_kv, chunks):
    """Full KV reuse: rotate each cached K by R_{dst-src} with an explicit matrix."""
    kv = f64(cached_kv).copy()
    hd, theta = cfg["head_dim"], cfg["rope_theta"]
    for src, dst, ln in chunks:
        R = rotation_matrix(dst - src, hd, theta)
        for li in range(kv.shape[0]):
            for j in range(dst, dst + ln):
                for g in range(kv.shape[3]):
                    kv[li, 0, j, g] = R @ kv[li, 0, j, g]
    return kv


def extend_after_prefix(cfg, weights, prefix_kv, query_tokens):
    """Query tokens decoded after a fixed prefix cache (positions 0..n_prefix-1):
    the full-KV-reuse baseline.  Returns (kv of the query rows, logits)."""
    dec = SequentialDecoder(cfg, weights)
    n_pre = prefix_kv.shape[2]
    for li in range(dec.L):
        for j in range(n_pre):
            dec.add_prefix(li, j, prefix_kv[li, 0, j], prefix_kv[li, 1, j])
    h = None
    for j, t in enumerate(query_tokens):
        h = dec.step(int(t), n_pre + j)
    return dec.kv()[:, :, n_pre:], dec.logits(h)


def top_k_by_sorting(dev, k):
    """Largest k by a full sort on (-dev, index); returned ascending."""
    order = sorted(range(len(dev)), key=lambda j: (-float(dev[j]), j))
    return sorted(order[:k])


def _layer_row(W, h, pos, R, Hq, Hkv, hd, eps):
    """One row's q (list of Hq vectors), k, v ([Hkv][hd]) at position pos, explicit per head."""
    x = _norm(h, W["attn_norm"], eps)
    Rm = R(pos)
    q = [Rm @ (W["wq"][i * hd:(i + 1) * hd] @ x) for i in range(Hq)]
    k = np.stack([Rm @ (W["wk"][i * hd:(i + 1) * hd] @ x) for i in range(Hkv)])
    v = np.stack([W["wv"][i * hd:(i + 1) * hd] @ x for i in range(Hkv)])
    return q, k, v


def _attend_row(q, kv_layer, pos, Hq, Hkv, hd):
    """Softmax attention of one row's heads over every key row at position <= pos."""
    group = Hq // Hkv
    o = []
    for i in range(Hq):
        g = i // group
        s = [float(np.dot(q[i], kv_layer[0][j][g])) / math.sqrt(hd) for j in range(pos + 1)]
        mx = max(s)
        e = [math.exp(sj - mx) for sj in s]
        z = sum(e)
        o.append(sum((e[j] / z) * kv_layer[1][j][g] for j in range(pos + 1)))
    return np.concatenate(o)


def selective_blend(cfg, weights, tokens, placed_kv, n_ctx, counts):
    """Blend with a per-layer shrinking recomputed set, one row at a time (micro inputs only).

    placed_kv: the chunk caches after placement, [L][2][n_ctx][Hkv][hd].  counts: k_l for layers
    1..L-1, non-increasing.  Layer 0 updates every row's hidden state and stores fresh K/V for the
    query rows only; at layer l >= 1 the rows holding an updated hidden state get fresh K/V, and when
    k_l is below the number of such context rows, each one's ||K_new - K_pre||^2 + ||V_new - V_pre||^2
    against the placed cache ranks them (ties to the lower row); the k_l largest and the query rows
    have their fresh K/V stored, attend, and carry their hidden state on.
    Returns (kv [L][2][N][Hkv][hd], logits of the last row, {layer: kept context rows})."""
    dec = SequentialDecoder(cfg, weights)
    L, Hq, Hkv, hd, eps = dec.L, dec.Hq, dec.Hkv, dec.hd, dec.eps
    N = len(tokens)
    kv = np.zeros((L, 2, N, Hkv, hd))
    kv[:, :, :n_ctx] = placed_kv
    h = {j: dec.E[int(tokens[j])].copy() for j in range(N)}
    live = list(range(N))
    kept = {}
    for li, W in enumerate(dec.layers):
        fresh = {j: _layer_row(W, h[j], j, dec.R, Hq, Hkv, hd, eps) for j in live}
        ctx_live = [j for j in live if j < n_ctx]
        if li == 0:
            keep = ctx_live
            store = [j for j in live if j >= n_ctx]
        else:
            k_l = counts[li - 1]
            if k_l < len(ctx_live):
                dev = {}
                for j in ctx_live:
                    dk = fresh[j][1] - kv[li, 0, j]
                    dv = fresh[j][2] - kv[li, 1, j]
                    dev[j] = float(np.sum(dk * dk) + np.sum(dv * dv))
                keep = sorted(sorted(ctx_live, key=lambda j: (-dev[j], j))[:k_l])
            else:
                keep = ctx_live
            kept[li] = list(keep)
            store = keep + [j for j in live if j >= n_ctx]
        for j in store:
            kv[li, 0, j], kv[li, 1, j] = fresh[j][1], fresh[j][2]
        live = keep + [j for j in live if j >= n_ctx]
        for j in live:
            hj = h[j] + W["wo"] @ _attend_row(fresh[j][0], kv[li], j, Hq, Hkv, hd)
            x = _norm(hj, W["mlp_norm"], eps)
            h[j] = hj + W["w_down"] @ (_sigmoid_gate(W["w_gate"] @ x) * (W["w_up"] @ x))
    return kv, dec.logits(h[N - 1]), kept
