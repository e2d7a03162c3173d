"""Sizing arithmetic of the blend (CPU oracle; TEST INFRASTRUCTURE ONLY).

CacheBlend deep-dive page, section "把账算细:一份 KV 有多大,15% 重算值多少钱":
KV bytes per token = 2 * L * H_kv * d_head * bytes-per-element, and the recompute
share counted in token-layers (r of every layer, plus one full check layer).
Pinned by the page's own worked numbers in tests/golden/page_sizing_examples.txt.
"""
from __future__ import annotations


def kv_bytes_per_token(n_layers: int, n_kv_heads: int, head_dim: int, bytes_per_elem: float) -> float:
    """K and V of every layer for one token."""
    return 2 * n_layers * n_kv_heads * head_dim * bytes_per_elem


def kv_bytes(n_tokens: int, n_layers: int, n_kv_heads: int, head_dim: int, bytes_per_elem: float) -> float:
    return n_tokens * kv_bytes_per_token(n_layers, n_kv_heads, head_dim, bytes_per_elem)


def recompute_token_layers(n_tokens: int, n_layers: int, ratio: float) -> dict:
    """Token-layers recomputed when every layer redoes a fraction ``ratio`` of the
    tokens, plus the one check layer done for every token."""
    full = n_tokens * n_layers
    selective = n_tokens * n_layers * ratio
    with_check = selective + n_tokens
    return dict(full=full, selective=selective, selective_fraction=selective / full,
                with_check=with_check, with_check_fraction=with_check / full)


def load_time(per_token_kv_bytes: float, n_tokens: int, throughput_bytes_per_s: float) -> float:
    """T_load = PerTokenKVSize * L / Throughput(device) (section "位置恢复、KV 存储与加载流水线",
    loading controller; L here is the context length in tokens)."""
    return per_token_kv_bytes * n_tokens / throughput_bytes_per_s


def controller_ratio(t_prefill_s: float, t_load_s: float, r_min: float = 0.15) -> float:
    """Loading controller: the ratio whose recompute time r * T_prefill matches T_load,
    but never below the quality floor r* (15% on the page)."""
    r_match = t_load_s / t_prefill_s if t_prefill_s > 0 else 1.0
    return min(1.0, max(r_min, r_match))


def pick_storage(devices, per_token_kv_bytes: float, n_tokens: int, t_prefill_s: float, r_min: float = 0.15) -> int:
    """Storage tier choice of the loading controller: among the tiers whose load time stays within the
    recompute time at the quality floor (r_min * T_prefill), the cheapest per GB; when none does, fall
    back to the fastest ("SSD is cheaper than memory: use it when its bandwidth suffices, else memory").
    ``devices`` is a list of (throughput bytes/s, cost per GB); returns an index (ties: the first)."""
    budget = r_min * t_prefill_s
    ok = [i for i, (bw, _) in enumerate(devices) if load_time(per_token_kv_bytes, n_tokens, bw) <= budget]
    if ok:
        return min(ok, key=lambda i: (devices[i][1], i))
    return max(range(len(devices)), key=lambda i: (devices[i][0], -i))
