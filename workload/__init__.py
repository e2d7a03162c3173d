"""Seeded synthetic workloads for the CacheBlend blend step.

This package is the ONLY thing the CPU oracle and the GPU path share: it turns
a seed into weights, token ids and a chunk layout.  It contains no arithmetic of
the method itself (no projection, rotation, attention or selection).

The random numbers come from ``cbgen.c`` (counter-based SplitMix64 +
Box-Muller; the exact definition is in that file's header), so every element
of every tensor is a pure function of (seed, stream, index).

Workloads follow the pages' RAG setting (CacheBlend deep-dive page, section
"实测:质量、延迟与吞吐" / evaluation: 512-token chunks, top-6 retrieval):
uniform random token chunks stand in for retrieved passages; no dataset item is
reproduced.  Weights are random-init Llama-style, N(0, 0.02), norm gains 1.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from dataclasses import dataclass, field

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "cbgen.c")
_LIB = os.path.join(_HERE, "libcbgen.so")
_lib = None

# stream-id spaces (disjoint)
_S_EMBED, _S_HEAD = 1, 2
_S_LAYER = 256
_S_TOKENS = 1 << 32
_S_QUERY = 2 << 32
_S_PERM = 3 << 32
_S_CACHE = 4 << 32
_LAYER_TENSORS = ("wq", "wk", "wv", "wo", "w_gate", "w_up", "w_down")


def build(force: bool = False) -> str:
    """Compile libcbgen.so next to its source (portable C, OpenMP)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.run(["gcc", "-O2", "-std=c99", "-fopenmp", "-fPIC", "-shared", _SRC, "-o", tmp, "-lm"],
                       check=True)
        os.replace(tmp, _LIB)
    return _LIB


def _l():
    global _lib
    if _lib is None:
        build()
        lib = ctypes.CDLL(_LIB)
        u64, i64 = ctypes.c_uint64, ctypes.c_int64
        lib.cbgen_key.restype = u64
        lib.cbgen_key.argtypes = [u64, u64]
        lib.cbgen_draw.restype = u64
        lib.cbgen_draw.argtypes = [u64, u64]
        lib.cbgen_normal_f32.argtypes = [u64, u64, i64, i64, ctypes.c_double, ctypes.c_void_p]
        lib.cbgen_normal_bf16.argtypes = [u64, u64, i64, i64, ctypes.c_double, ctypes.c_void_p]
        lib.cbgen_fill_bf16.argtypes = [i64, ctypes.c_float, ctypes.c_void_p]
        lib.cbgen_tokens.argtypes = [u64, u64, i64, i64, ctypes.c_void_p]
        lib.cbgen_permutation.argtypes = [u64, u64, i64, ctypes.c_void_p]
        _lib = lib
    return _lib


# ----------------------------------------------------------------------------------------------
# primitive draws
# ----------------------------------------------------------------------------------------------
def key(seed: int, stream: int) -> int:
    return int(_l().cbgen_key(seed, stream))


def draw(k: int, i: int) -> int:
    return int(_l().cbgen_draw(k, i))


def normal(seed: int, stream: int, shape, std: float, dtype: str, first: int = 0, out=None) -> np.ndarray:
    """std * N(0,1) elements [first, first+prod(shape)) of a stream.

    dtype 'f32' -> float32 array; 'bf16' -> uint16 array of bfloat16 bit patterns.
    """
    n = int(np.prod(shape))
    if dtype == "bf16":
        a = np.empty(shape, np.uint16) if out is None else out
        _l().cbgen_normal_bf16(seed, stream, first, n, std, a.ctypes.data)
    elif dtype == "f32":
        a = np.empty(shape, np.float32) if out is None else out
        _l().cbgen_normal_f32(seed, stream, first, n, std, a.ctypes.data)
    else:
        raise ValueError(dtype)
    return a


def ones(shape, dtype: str) -> np.ndarray:
    if dtype == "bf16":
        a = np.empty(shape, np.uint16)
        _l().cbgen_fill_bf16(int(np.prod(shape)), 1.0, a.ctypes.data)
        return a
    return np.ones(shape, np.float32)


def tokens(seed: int, stream: int, n: int, vocab: int) -> np.ndarray:
    a = np.empty(n, np.int32)
    _l().cbgen_tokens(seed, stream, n, vocab, a.ctypes.data)
    return a


def permutation(seed: int, stream: int, n: int) -> np.ndarray:
    a = np.empty(n, np.int32)
    _l().cbgen_permutation(seed, stream, n, a.ctypes.data)
    return a


def bf16_bits_to_f32(a: np.ndarray) -> np.ndarray:
    """Reinterpret bfloat16 bit patterns (uint16) as float32 values (exact)."""
    return (a.astype(np.uint32) << 16).view(np.float32)


# ----------------------------------------------------------------------------------------------
# model configurations (Llama-style decoder shapes)
# ----------------------------------------------------------------------------------------------
@dataclass(frozen=True)
class ModelShape:
    n_layers: int
    d_model: int
    n_heads: int
    n_kv_heads: int
    head_dim: int
    ffn_hidden: int
    vocab: int
    rope_theta: float
    dtype: str            # storage / operand type of weights and KV: 'f32' or 'bf16'
    rms_eps: float = 1e-5

    @property
    def kv_row(self) -> int:          # elements of one token's K (or V) in one layer
        return self.n_kv_heads * self.head_dim

    def as_dict(self) -> dict:
        return dict(n_layers=self.n_layers, d_model=self.d_model, n_heads=self.n_heads,
                    n_kv_heads=self.n_kv_heads, head_dim=self.head_dim, ffn_hidden=self.ffn_hidden,
                    vocab=self.vocab, rope_theta=self.rope_theta, rms_eps=self.rms_eps, dtype=self.dtype)


@dataclass(frozen=True)
class WorkloadSpec:
    name: str
    shape: ModelShape
    n_chunks: int
    chunk_len: int
    n_query: int
    ratios: tuple
    seeds: tuple
    shuffle: bool = False

    @property
    def n_ctx(self) -> int:
        return self.n_chunks * self.chunk_len

    @property
    def n_tokens(self) -> int:
        return self.n_ctx + self.n_query


TINY = ModelShape(2, 256, 4, 2, 64, 512, 1024, 1e4, "f32")
SMALL = ModelShape(8, 1024, 16, 4, 64, 2816, 32000, 1e4, "bf16")
LLAMA8B = ModelShape(32, 4096, 32, 8, 128, 14336, 128256, 5e5, "bf16")

WORKLOADS = {
    "tiny-fp32": WorkloadSpec("tiny-fp32", TINY, 3, 64, 16, (0.25,), (0,)),
    "small-bf16": WorkloadSpec("small-bf16", SMALL, 4, 512, 32, (0.15,), (1,)),
    "llama8b-3k": WorkloadSpec("llama8b-3k", LLAMA8B, 6, 512, 64, (0.15,), (2,)),
    "llama8b-8k": WorkloadSpec("llama8b-8k", LLAMA8B, 16, 512, 64, (0.05, 0.15, 0.30), (3, 4, 5), shuffle=True),
    "llama8b-32k": WorkloadSpec("llama8b-32k", LLAMA8B, 64, 512, 128, (0.15,), (6,)),
}


def weight_shapes(s: ModelShape) -> dict:
    """Weight matrices in [out_features][in_features] row-major order."""
    d, hd = s.d_model, s.head_dim
    return dict(wq=(s.n_heads * hd, d), wk=(s.n_kv_heads * hd, d), wv=(s.n_kv_heads * hd, d),
                wo=(d, s.n_heads * hd), w_gate=(s.ffn_hidden, d), w_up=(s.ffn_hidden, d),
                w_down=(d, s.ffn_hidden))


def make_weights(s: ModelShape, seed: int, std: float = 0.02, layers=None) -> dict:
    """Random-init weights: every matrix N(0, std), RMSNorm gains 1.

    Returns {'embed': [V][d], 'lm_head': [V][d], 'final_norm': [d],
             'layers': [ {attn_norm, wq, wk, wv, wo, mlp_norm, w_gate, w_up, w_down}, ... ]}
    as uint16 (bf16 bits) or float32 arrays.
    """
    dt = s.dtype
    w = dict(embed=normal(seed, _S_EMBED, (s.vocab, s.d_model), std, dt),
             lm_head=normal(seed, _S_HEAD, (s.vocab, s.d_model), std, dt),
             final_norm=ones((s.d_model,), dt), layers=[])
    shapes = weight_shapes(s)
    for layer in range(s.n_layers) if layers is None else layers:
        lw = dict(attn_norm=ones((s.d_model,), dt), mlp_norm=ones((s.d_model,), dt))
        for t, name in enumerate(_LAYER_TENSORS):
            lw[name] = normal(seed, _S_LAYER * (layer + 1) + t + 1, shapes[name], std, dt)
        w["layers"].append(lw)
    return w


@dataclass
class Request:
    """One blend request: chunk tokens, their placement and the query."""
    spec: WorkloadSpec
    seed: int
    ratio: float
    chunk_tokens: list                     # per placed chunk (in dst order), int32 arrays
    chunks: list                           # per placed chunk: (src_pos, dst_pos, len)
    query: np.ndarray                      # int32 [n_query]
    tokens: np.ndarray = field(init=False)  # int32 [n_ctx + n_query], context then query

    def __post_init__(self):
        self.tokens = np.concatenate(list(self.chunk_tokens) + [self.query]).astype(np.int32)


def make_request(spec: WorkloadSpec, seed: int, ratio: float) -> Request:
    """Chunks of uniform random tokens, each to be prefilled alone at positions
    0..len-1 (src_pos 0) and placed back to back (dst_pos = slot * len), in a
    seeded random order when the workload shuffles; then a random query."""
    V = spec.shape.vocab
    order = permutation(seed, _S_PERM, spec.n_chunks) if spec.shuffle else np.arange(spec.n_chunks)
    chunk_tokens, chunks = [], []
    for slot, c in enumerate(order):
        chunk_tokens.append(tokens(seed, _S_TOKENS + int(c), spec.chunk_len, V))
        chunks.append((0, slot * spec.chunk_len, spec.chunk_len))
    q = tokens(seed, _S_QUERY, spec.n_query, V)
    return Request(spec, seed, ratio, chunk_tokens, chunks, q)


def synthetic_cache(s: ModelShape, seed: int, n_rows: int, std: float) -> np.ndarray:
    """A stand-in chunk cache [L][2][n_rows][Hkv][hd] of i.i.d. N(0, std) values.

    Used only where a genuine per-chunk prefill would cost the fp64 oracle too much
    (the 8B-shape configurations); ``std`` is chosen to match the K/V scale of the
    random-init model (0.02 * sqrt(d_model))."""
    out = np.empty((s.n_layers, 2, n_rows, s.n_kv_heads, s.head_dim),
                   np.uint16 if s.dtype == "bf16" else np.float32)
    for layer in range(s.n_layers):
        for kv in range(2):
            normal(seed, _S_CACHE + 2 * layer + kv, out.shape[2:], std, s.dtype, out=out[layer, kv])
    return out


def kv_std(s: ModelShape, std: float = 0.02) -> float:
    """Scale of K/V entries in a random-init model (unit-RMS input times N(0,std) weights)."""
    return std * float(np.sqrt(s.d_model))


def funnel_ratios(n_layers: int, r: float, r_first: float = None, steps: int = 4) -> tuple:
    """A gradual-filtering schedule for layers 1..n_layers-1: the check layer keeps r_first (2r by
    default, capped at 1), and the ratio shrinks in equal steps to r over the next `steps` layers,
    then stays at r (the funnel of Figure 9, settling near the target r).  Holds no method arithmetic:
    it only chooses inputs."""
    r1 = min(1.0, 2.0 * r) if r_first is None else r_first
    out = []
    for layer in range(1, n_layers):
        t = min(layer - 1, steps) / steps
        out.append(r1 + (r - r1) * t)
    return tuple(out)
