"""CPU oracle of the CacheBlend blend step (plain numpy, float64 arithmetic).

TEST INFRASTRUCTURE ONLY.  Nothing on the product path imports this module;
only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline /
reference legs may call it.  It shares no code with the CUDA library.

Source of every step: the CacheBlend deep-dive page ("CacheBlend 完全拆解:RAG 多段
KV 缓存拼接,为什么还要重算一小部分 token").  Section names are quoted in the
docstrings below.

Readings taken where the page leaves a step open:
  R1  the check layer (full computation + deviation + selection) is layer index 1,
      the first layer whose input has seen other chunks; layer 0 recomputes hidden
      states for every row but reuses the (context-free) cached layer-0 K/V.
  R2  deviation = squared L2 over all KV heads and dims, K and V with equal weight,
      fresh (unrounded) K/V against the re-RoPE'd stored cache.
  R3  k = ceil(ratio * n_ctx) (minus 1e-9 to absorb representation error), clamped
      to [0, n_ctx]; query rows are always recomputed and never compete.
  R4  the set is chosen once at the check layer and kept for every later layer.
  R5  ties in deviation go to the lower position; the set is reported ascending.
  R6  within a layer the selected rows' fresh K/V are stored before attention, so
      selected queries see each other's fresh K/V ("assemble a complete K/V, then
      attend", Figure 5 of the page).
  R7  storage: out_kv is rounded once to the storage type (bf16 or f32, round to
      nearest even); activations stay unrounded float64.  Mode 'f64' keeps
      float64 storage for the exactness pins.
  R8  RoPE pairs are adjacent dims (2i, 2i+1), angle m * theta^(-2i/hd) in float64
      (the block-diagonal rotation of section "位置恢复、KV 存储与加载流水线").
  R9  Llama-style pre-norm decoder without biases; RMSNorm eps 1e-5; SwiGLU MLP;
      untied embedding / LM head.

Parity pins (tests/test_oracle_*.py): RoPE composition and orthogonality,
sequential-decode brute force, r = 1 equals a full joint prefill, r = 0 equals
full KV reuse, causal-prefix exactness, the page's Δkv definition, top-k against a
full sort, GQA against a library attention, bf16 rounding against a library cast.
The selected set at 0 < r < 1 is pinned only through the Δkv identity (the pages
print no worked example of a blend).
"""
from __future__ import annotations

import math
from concurrent.futures import ThreadPoolExecutor

import numpy as np

_POOL = None
_Q_BLOCK = 512       # query rows per attention block (memory bound only; rows are independent)
_ROW_BLOCK = 4096    # rows per MLP block (memory bound only)


def _pool():
    global _POOL
    if _POOL is None:
        _POOL = ThreadPoolExecutor(max_workers=16)
    return _POOL


# ----------------------------------------------------------------------------------------------
# number formats
# ----------------------------------------------------------------------------------------------
def to_f64(a: np.ndarray) -> np.ndarray:
    """bfloat16 bit patterns (uint16) or float arrays -> float64 values (exact)."""
    if a.dtype == np.uint16:
        flat = a.reshape(-1)
        out = np.empty(flat.shape, np.float64)
        step = max(1 << 20, -(-flat.size // 16))

        def conv(lo):
            hi = min(lo + step, flat.size)
            out[lo:hi] = (flat[lo:hi].astype(np.uint32) << 16).view(np.float32)

        list(_pool().map(conv, range(0, flat.size, step)))
        return out.reshape(a.shape)
    return np.asarray(a, dtype=np.float64)


def round_bf16(x: np.ndarray) -> np.ndarray:
    """Round float64 values to the nearest bfloat16 (8 significant bits), ties to even.

    bfloat16 keeps float32's exponent range and 8 significand bits; x = m * 2^e with
    m in [0.5, 1), so m * 2^8 rounded to an integer (np.rint: ties to even) is the
    bfloat16 significand.  (Subnormals and overflow do not occur here.)"""
    m, e = np.frexp(np.asarray(x, dtype=np.float64))
    return np.ldexp(np.rint(np.ldexp(m, 8)), e - 8)


def round_store(x: np.ndarray, store: str) -> np.ndarray:
    if store == "bf16":
        return round_bf16(x)
    if store == "f32":
        return np.asarray(x, np.float32).astype(np.float64)
    if store == "f64":
        return np.asarray(x, np.float64)
    raise ValueError(store)


# ----------------------------------------------------------------------------------------------
# model pieces (section "问题:拼接的 KV 缓存到底少了什么": Q_i = h_i W_Q, K_i = h_i W_K,
# V_i = h_i W_V, K rotated by position)
# ----------------------------------------------------------------------------------------------
def rope_freqs(head_dim: int, theta: float) -> np.ndarray:
    """theta_i = theta^(-2i/hd), i < hd/2 (float64)."""
    i = np.arange(head_dim // 2, dtype=np.float64)
    return np.power(float(theta), -2.0 * i / head_dim)


def rope(x: np.ndarray, pos, theta: float) -> np.ndarray:
    """Apply R_m to every head vector of x [n][H][hd] at positions pos [n].

    R_m is block diagonal; block i rotates dims (2i, 2i+1) by angle m * theta_i
    (section "位置恢复、KV 存储与加载流水线": q_m = R_m q, k_n = R_n k)."""
    x = np.asarray(x, np.float64)
    hd = x.shape[-1]
    ang = np.asarray(pos, np.float64)[:, None] * rope_freqs(hd, theta)[None, :]
    c = np.cos(ang)[:, None, :]
    s = np.sin(ang)[:, None, :]
    x0, x1 = x[..., 0::2], x[..., 1::2]
    out = np.empty_like(x)
    out[..., 0::2] = x0 * c - x1 * s
    out[..., 1::2] = x0 * s + x1 * c
    return out


def rmsnorm(x: np.ndarray, g: np.ndarray, eps: float) -> np.ndarray:
    ms = np.mean(x * x, axis=-1, keepdims=True)
    return x * g / np.sqrt(ms + eps)


def silu(x: np.ndarray) -> np.ndarray:
    return x / (1.0 + np.exp(-x))


def attention(q, k, v, q_pos, k_pos, n_kv_heads: int) -> np.ndarray:
    """Causal softmax attention with grouped KV heads.

    q [M][Hq][hd]; k, v [Nk][Hkv][hd]; query a sees key j iff k_pos[j] <= q_pos[a].
    q-head h reads KV head h // (Hq / Hkv); scores scaled by 1/sqrt(hd)."""
    M, Hq, hd = q.shape
    group = Hq // n_kv_heads
    q_pos = np.asarray(q_pos)
    k_pos = np.asarray(k_pos)
    out = np.empty((M, Hq, hd), np.float64)
    scale = 1.0 / math.sqrt(hd)
    sorted_keys = bool(np.all(k_pos[1:] >= k_pos[:-1]))
    for b0 in range(0, M, _Q_BLOCK):
        qp = q_pos[b0:b0 + _Q_BLOCK]
        # keys past the block's last position are invisible to all of its queries: with positions
        # sorted they are simply not scored (their softmax weight would be exactly zero)
        nk = int(np.searchsorted(k_pos, qp.max(), side="right")) if sorted_keys else k_pos.size
        visible = k_pos[None, :nk] <= qp[:, None]                   # [b][nk]

        def head(h):
            g = h // group
            s = (q[b0:b0 + _Q_BLOCK, h, :] @ k[:nk, g, :].T) * scale  # [b][nk]
            s = np.where(visible, s, -np.inf)
            s = s - s.max(axis=1, keepdims=True)
            p = np.exp(s)
            p /= p.sum(axis=1, keepdims=True)
            out[b0:b0 + _Q_BLOCK, h, :] = p @ v[:nk, g, :]

        list(_pool().map(head, range(Hq)))           # heads are independent
    return out


class Model:
    """Config dict + weights (as produced by the workload generator), widened to float64 per layer."""

    def __init__(self, cfg: dict, weights: dict):
        self.cfg = cfg
        self.w = weights
        self.L = cfg["n_layers"]
        self.d = cfg["d_model"]
        self.Hq = cfg["n_heads"]
        self.Hkv = cfg["n_kv_heads"]
        self.hd = cfg["head_dim"]
        self.theta = cfg["rope_theta"]
        self.eps = cfg.get("rms_eps", 1e-5)

    def layer(self, i: int) -> dict:
        return {k: to_f64(v) for k, v in self.w["layers"][i].items()}

    def embed_rows(self, tokens) -> np.ndarray:
        return to_f64(self.w["embed"][np.asarray(tokens)])

    # -- one decoder layer, split where the blend needs to intervene --------------------------
    def qkv(self, W: dict, h: np.ndarray, pos):
        """x = RMSNorm(h); q, k rotated at their positions; v plain.  Shapes [n][H][hd]."""
        n = h.shape[0]
        x = rmsnorm(h, W["attn_norm"], self.eps)
        q = rope((x @ W["wq"].T).reshape(n, self.Hq, self.hd), pos, self.theta)
        k = rope((x @ W["wk"].T).reshape(n, self.Hkv, self.hd), pos, self.theta)
        v = (x @ W["wv"].T).reshape(n, self.Hkv, self.hd)
        return q, k, v

    def q_only(self, W: dict, h: np.ndarray, pos):
        n = h.shape[0]
        x = rmsnorm(h, W["attn_norm"], self.eps)
        return rope((x @ W["wq"].T).reshape(n, self.Hq, self.hd), pos, self.theta)

    def finish(self, W: dict, h: np.ndarray, o: np.ndarray) -> np.ndarray:
        """h + o W_O, then h + W_down(silu(W_gate x) * W_up x) with x = RMSNorm(h)."""
        out = np.empty_like(h)
        for b0 in range(0, h.shape[0], _ROW_BLOCK):
            hb = h[b0:b0 + _ROW_BLOCK] + o[b0:b0 + _ROW_BLOCK].reshape(-1, self.Hq * self.hd) @ W["wo"].T
            x = rmsnorm(hb, W["mlp_norm"], self.eps)
            out[b0:b0 + _ROW_BLOCK] = hb + (silu(x @ W["w_gate"].T) * (x @ W["w_up"].T)) @ W["w_down"].T
        return out

    def logits(self, h_last: np.ndarray) -> np.ndarray:
        x = rmsnorm(h_last, to_f64(self.w["final_norm"]), self.eps)
        return to_f64(self.w["lm_head"]) @ x


# ----------------------------------------------------------------------------------------------
# the blend step
# ----------------------------------------------------------------------------------------------
def selected_count(n_ctx: int, ratio: float) -> int:
    """k = ceil(ratio * n_ctx), clamped to [0, n_ctx] (reading R3)."""
    k = math.ceil(float(ratio) * n_ctx - 1e-9)
    return int(min(max(k, 0), n_ctx))


def select_hkvd(dev: np.ndarray, k: int) -> np.ndarray:
    """The k rows of largest deviation (HKVD tokens), ties to the lower row, ascending.

    Section "选 token:HKVD、逐层过滤与 15% 这个经验值": rank tokens by KV deviation
    and keep the top fraction."""
    order = np.argsort(-np.asarray(dev, np.float64), kind="stable")
    return np.sort(order[:k]).astype(np.int64)


def rerope(cached_kv: np.ndarray, chunks, theta: float, store: str, out=None) -> np.ndarray:
    """Place chunk caches at their new offsets: K <- R_{dst-src} K, V unchanged.

    Section "位置恢复、KV 存储与加载流水线": a key cached at position p as k_p = R_p k
    becomes R_{n-p} k_p = R_n k at its new position n; V carries no position.
    cached_kv [L][2][n_ctx][Hkv][hd] holds the context rows in placed (dst) order.
    Returns float64 values rounded to the storage type (``out``, if given, receives them instead:
    any float array of the same shape that holds the storage type exactly)."""
    cached_kv = np.asarray(cached_kv)
    kv = np.empty(cached_kv.shape, np.float64) if out is None else out
    for layer in range(cached_kv.shape[0]):          # one layer at a time (memory only)
        kl = np.array(to_f64(cached_kv[layer, 0]), np.float64, copy=True)   # never a view of the input
        for src, dst, ln in chunks:
            rows = slice(dst, dst + ln)
            kl[rows] = round_store(rope(kl[rows], np.full(ln, dst - src), theta), store)
        kv[layer, 0] = kl
        kv[layer, 1] = to_f64(cached_kv[layer, 1])
    return kv


def deviation(k_new, v_new, k_pre, v_pre) -> np.ndarray:
    """Δkv[j] = ||K_new[j] - K_pre[j]||^2 + ||V_new[j] - V_pre[j]||^2 over all KV heads/dims.

    Section "核心思想:只重算偏差最大的那一小撮 token", KV-deviation formula (reading R2)."""
    n, width = k_new.shape[0], int(np.prod(k_new.shape[1:]))
    dk = (k_new - k_pre).reshape(n, width)
    dv = (v_new - v_pre).reshape(n, width)
    return np.sum(dk * dk, axis=1) + np.sum(dv * dv, axis=1)


def validate_chunks(chunks, n_tokens: int) -> int:
    """Chunks must tile [0, n_ctx) in dst order; src >= 0; at least one query row."""
    at = 0
    for src, dst, ln in chunks:
        if src < 0 or ln <= 0 or dst != at:
            raise ValueError("chunks must tile [0, n_ctx) in order with src >= 0")
        at += ln
    if at >= n_tokens:
        raise ValueError("need at least one query token after the context")
    return at


def blend(cfg: dict, weights: dict, tokens, cached_kv, chunks, ratio: float, store: str, selected=None,
          keep_exact: bool = False, exact_layers=None) -> dict:
    """One CacheBlend blend (sections "核心思想" and "选 token", Figures 5 and 9).

    1. re-RoPE the cached chunk K/V to their placed positions (V copied);
    2. embed all rows;
    3. layer 0: every row's hidden state is recomputed; context rows reuse their
       cached (context-free) K/V, query rows get fresh K/V (stored);
    4. check layer 1: fresh Q/K/V for every row; Δkv of each context row against
       its re-RoPE'd cache; the top-k rows plus the query rows form the set A;
       A's fresh K/V are stored; A attends over the blended K/V; O and MLP on A;
    5. layers 2..L-1: only A's rows: QKV, store, attend, O, MLP;
    6. logits of the last row.

    ``keep_exact`` also returns ``out_kv_exact``: the values before their rounding to the
    storage type (used to compare another implementation's rounded output against them).
    ``exact_layers`` (optional, a set of layer indices) returns ``exact_rows``: for each of those
    layers, (rows, K, V) of the rows computed fresh there, before rounding -- the same values as
    ``out_kv_exact`` at those rows, without a float64 copy of the whole cache.
    ``selected`` (optional) replaces the top-k choice by a given set of k rows -- used only
    to follow another implementation through a tie inside the comparison band.

    Returns dict(out_kv [L][2][N][Hkv][hd] float64, logits [V], selected [k],
    dev [n_ctx], k)."""
    m = Model(cfg, weights)
    tokens = np.asarray(tokens, np.int64)
    N = tokens.shape[0]
    n_ctx = validate_chunks(chunks, N)
    L, Hkv, hd = m.L, m.Hkv, m.hd
    pos = np.arange(N)

    kv_dtype = np.float64 if store == "f64" else np.float32   # bf16/f32 values are exact in f32
    out_kv = np.zeros((L, 2, N, Hkv, hd), kv_dtype)
    if n_ctx:
        rerope(cached_kv, chunks, m.theta, store, out=out_kv[:, :, :n_ctx])
    # unrounded values of everything stored (re-RoPE'd rows: the rotation before rounding)
    exact = np.zeros((L, 2, N, Hkv, hd), np.float64) if keep_exact else None
    if keep_exact and n_ctx:
        rerope(cached_kv, chunks, m.theta, "f64", out=exact[:, :, :n_ctx])
    exact_layers = set(exact_layers or ())
    exact_rows = {}

    def keep_rows(layer, rows, k_new, v_new):
        if layer in exact_layers:
            exact_rows[layer] = (np.asarray(rows).copy(), np.array(k_new, np.float64), np.array(v_new, np.float64))

    h = m.embed_rows(tokens)

    # layer 0: all rows; context K/V reused, query K/V fresh
    W = m.layer(0)
    q = m.q_only(W, h, pos)
    _, kq, vq = m.qkv(W, h[n_ctx:], pos[n_ctx:])
    out_kv[0, 0, n_ctx:] = round_store(kq, store)
    out_kv[0, 1, n_ctx:] = round_store(vq, store)
    if keep_exact:
        exact[0, 0, n_ctx:], exact[0, 1, n_ctx:] = kq, vq
    keep_rows(0, pos[n_ctx:], kq, vq)
    o = attention(q, out_kv[0, 0].astype(np.float64), out_kv[0, 1].astype(np.float64), pos, pos, Hkv)
    h = m.finish(W, h, o)
    del W

    # check layer 1: all rows' fresh q/k/v; deviation; selection
    W = m.layer(1)
    q, k_new, v_new = m.qkv(W, h, pos)
    dev = deviation(k_new[:n_ctx], v_new[:n_ctx], out_kv[1, 0, :n_ctx].astype(np.float64),
                    out_kv[1, 1, :n_ctx].astype(np.float64))
    kk = selected_count(n_ctx, ratio)
    sel = select_hkvd(dev, kk) if selected is None else np.sort(np.asarray(selected, np.int64))
    assert len(sel) == kk
    A = np.concatenate([sel, np.arange(n_ctx, N)])
    out_kv[1, 0, A] = round_store(k_new[A], store)
    out_kv[1, 1, A] = round_store(v_new[A], store)
    if keep_exact:
        exact[1, 0, A], exact[1, 1, A] = k_new[A], v_new[A]
    keep_rows(1, A, k_new[A], v_new[A])
    o = attention(q[A], out_kv[1, 0].astype(np.float64), out_kv[1, 1].astype(np.float64), A, pos, Hkv)
    hA = m.finish(W, h[A], o)
    del W, h, q, k_new, v_new

    # layers 2..L-1: only the selected rows and the query
    for layer in range(2, L):
        W = m.layer(layer)
        q, k_a, v_a = m.qkv(W, hA, A)
        out_kv[layer, 0, A] = round_store(k_a, store)
        out_kv[layer, 1, A] = round_store(v_a, store)
        if keep_exact:
            exact[layer, 0, A], exact[layer, 1, A] = k_a, v_a
        keep_rows(layer, A, k_a, v_a)
        o = attention(q, out_kv[layer, 0].astype(np.float64), out_kv[layer, 1].astype(np.float64), A, pos, Hkv)
        hA = m.finish(W, hA, o)
        del W

    logits = m.logits(hA[-1])
    return dict(out_kv=out_kv, out_kv_exact=exact, exact_rows=exact_rows, logits=logits, selected=sel, dev=dev, k=kk,
                rows=A)


def deviation_rows(cfg: dict, weights: dict, tokens, cached_kv, chunks, rows, store: str) -> np.ndarray:
    """The check-layer deviation Δkv of the given context rows only.

    Layer 0 of a context row depends only on its own token and the reused (re-RoPE'd) layer-0 K/V of
    the context rows at or before it, so the blend's steps 1-4 can be followed for a subset of rows:
    re-RoPE the caches of layers 0 and 1, layer 0 for those rows, their fresh layer-1 K/V, and the
    deviation against the stored layer-1 cache.  Equal to blend()['dev'][rows]."""
    m = Model(cfg, weights)
    tokens = np.asarray(tokens, np.int64)
    n_ctx = validate_chunks(chunks, tokens.shape[0])
    rows = np.asarray(rows, np.int64)
    assert rows.size and rows.max() < n_ctx
    kv01 = rerope(np.asarray(cached_kv)[:2], chunks, m.theta, store)        # layers 0 and 1
    h = m.embed_rows(tokens[rows])
    W = m.layer(0)
    q = m.q_only(W, h, rows)
    o = attention(q, kv01[0, 0], kv01[0, 1], rows, np.arange(n_ctx), m.Hkv)
    h = m.finish(W, h, o)
    _, k_new, v_new = m.qkv(m.layer(1), h, rows)
    return deviation(k_new, v_new, kv01[1, 0, rows], kv01[1, 1, rows])


def prefill(cfg: dict, weights: dict, tokens, store: str) -> dict:
    """Plain causal prefill at positions 0..N-1: the blend with no cached chunks."""
    return blend(cfg, weights, tokens, None, [], 0.0, store)


def chunk_caches(cfg: dict, weights: dict, chunk_tokens, chunks, store: str) -> np.ndarray:
    """Each chunk prefilled alone at positions src..src+len-1, stored at the storage
    type and concatenated in placed order: the cached_kv input of a blend."""
    parts = []
    for toks, (src, dst, ln) in zip(chunk_tokens, chunks):
        assert len(toks) == ln
        if src != 0:
            raise NotImplementedError("chunk caches are prefilled from position 0")
        parts.append(prefill(cfg, weights, toks, store)["out_kv"])
    return np.concatenate(parts, axis=2)


# ----------------------------------------------------------------------------------------------
# gradual filtering (Figure 9 of the page)
# ----------------------------------------------------------------------------------------------
def gradual_counts(n_ctx: int, ratios) -> list:
    """Per-layer selected counts k_l = ceil(r_l * n_ctx) for layers 1..L-1 (reading R3 per layer).

    Section "核心思想" (gradual filtering): r_1 > r_2 > ... so that S_{l+1} is a subset of S_l;
    a schedule that grows is rejected."""
    ks = [selected_count(n_ctx, r) for r in ratios]
    if any(not (0.0 <= float(r) <= 1.0) for r in ratios):
        raise ValueError("ratios must lie in [0, 1]")
    if any(b > a for a, b in zip(ks, ks[1:])):
        raise ValueError("the selected counts must not grow from layer to layer")
    return ks


def blend_gradual(cfg: dict, weights: dict, tokens, cached_kv, chunks, ratios, store: str, selected=None,
                  keep_exact: bool = False) -> dict:
    """CacheBlend blend with gradual filtering: the recomputed set shrinks layer by layer.

    Sections "核心思想" and "选 token" of the page (the funnel of Figure 9):
      * layer 0 and the check layer 1 are as in blend(); layer 1 keeps k_1 = ceil(r_1 n_ctx) rows S_1;
      * at a later layer l only the rows that carried an updated hidden state out of layer l-1
        (S_{l-1}, plus the query) get fresh Q/K/V; where k_l < k_{l-1}, each candidate's deviation ||KV_new - KV_pre||^2 against the re-RoPE'd
        cache of layer l (taken before the store) ranks the candidates again and S_l is the top k_l
        of them (ties to the lower position), so S_l is a subset of S_{l-1};
      * the fresh K/V of S_l and the query are stored (reading R10), then attention, O and MLP run
        for S_l plus the query only: theirs are the hidden states passed on.
    ``ratios`` has one entry per layer 1..L-1 and must give non-increasing counts.
    Readings added to R1-R9:
      R10 a layer that compares treats its candidates as the check layer treats every row: the
          fresh K/V of the rows it keeps are stored, and a candidate that drops out keeps its cached
          K/V from that layer on (its fresh K/V served only the comparison);
      R11 a layer whose count equals the previous one keeps the set without comparing (the page's
          check_flag off); the comparison would select every candidate anyway.
    ``selected`` (optional) maps a layer to the k_l rows to use there instead of the top-k choice
    (only to follow another implementation through a tie inside the comparison band).

    Returns dict(out_kv, out_kv_exact, logits, sets {layer: S_l ascending}, devs {layer: dev of
    that layer's candidates, in the candidates' order}, counts [k_1..k_{L-1}], rows: final A)."""
    m = Model(cfg, weights)
    tokens = np.asarray(tokens, np.int64)
    N = tokens.shape[0]
    n_ctx = validate_chunks(chunks, N)
    L, Hkv, hd = m.L, m.Hkv, m.hd
    if len(ratios) != L - 1:
        raise ValueError("one ratio per layer 1..L-1")
    counts = gradual_counts(n_ctx, ratios)
    selected = selected or {}
    pos = np.arange(N)
    query = np.arange(n_ctx, N)

    kv_dtype = np.float64 if store == "f64" else np.float32
    out_kv = np.zeros((L, 2, N, Hkv, hd), kv_dtype)
    if n_ctx:
        rerope(cached_kv, chunks, m.theta, store, out=out_kv[:, :, :n_ctx])
    exact = np.zeros((L, 2, N, Hkv, hd), np.float64) if keep_exact else None
    if keep_exact and n_ctx:
        rerope(cached_kv, chunks, m.theta, "f64", out=exact[:, :, :n_ctx])

    def store_rows(layer, rows, k_new, v_new):
        out_kv[layer, 0, rows] = round_store(k_new, store)
        out_kv[layer, 1, rows] = round_store(v_new, store)
        if keep_exact:
            exact[layer, 0, rows], exact[layer, 1, rows] = k_new, v_new

    h = m.embed_rows(tokens)
    # layer 0: every row, context K/V reused
    W = m.layer(0)
    q = m.q_only(W, h, pos)
    _, kq, vq = m.qkv(W, h[n_ctx:], pos[n_ctx:])
    store_rows(0, query, kq, vq)
    o = attention(q, out_kv[0, 0].astype(np.float64), out_kv[0, 1].astype(np.float64), pos, pos, Hkv)
    h = m.finish(W, h, o)
    del W

    sets, devs = {}, {}
    # check layer 1: every row compared, S_1 chosen among all context rows
    W = m.layer(1)
    q, k_new, v_new = m.qkv(W, h, pos)
    devs[1] = deviation(k_new[:n_ctx], v_new[:n_ctx], out_kv[1, 0, :n_ctx].astype(np.float64),
                        out_kv[1, 1, :n_ctx].astype(np.float64))
    sets[1] = np.sort(np.asarray(selected[1], np.int64)) if 1 in selected else select_hkvd(devs[1], counts[0])
    assert len(sets[1]) == counts[0]
    A = np.concatenate([sets[1], query])
    store_rows(1, A, k_new[A], v_new[A])
    o = attention(q[A], out_kv[1, 0].astype(np.float64), out_kv[1, 1].astype(np.float64), A, pos, Hkv)
    hA = m.finish(W, h[A], o)
    del W, h, q, k_new, v_new

    for layer in range(2, L):
        W = m.layer(layer)
        cand = sets[layer - 1]
        q, k_a, v_a = m.qkv(W, hA, A)          # fresh Q/K/V of S_{l-1} and the query
        k_prev, k_cur = counts[layer - 2], counts[layer - 1]
        if k_cur < k_prev:
            devs[layer] = deviation(k_a[:k_prev], v_a[:k_prev], out_kv[layer, 0, cand].astype(np.float64),
                                    out_kv[layer, 1, cand].astype(np.float64))
            if layer in selected:               # positions given: their indices among the candidates
                keep = np.searchsorted(cand, np.sort(np.asarray(selected[layer], np.int64)))
                assert len(keep) == k_cur and np.array_equal(cand[keep], np.sort(selected[layer]))
            else:
                keep = select_hkvd(devs[layer], k_cur)
            sets[layer] = cand[keep]
        else:
            keep = np.arange(k_prev)
            sets[layer] = cand
        local = np.concatenate([keep, np.arange(k_prev, k_prev + (N - n_ctx))])
        A = A[local]
        store_rows(layer, A, k_a[local], v_a[local])     # R10: the kept rows' fresh K/V, before attention
        o = attention(q[local], out_kv[layer, 0].astype(np.float64), out_kv[layer, 1].astype(np.float64), A,
                      pos, Hkv)
        hA = m.finish(W, hA[local], o)
        del W

    logits = m.logits(hA[-1])
    return dict(out_kv=out_kv, out_kv_exact=exact, logits=logits, sets=sets, devs=devs, counts=counts, rows=A)
