"""Python binding of libcacheblend (the GB300 CacheBlend blend-step library).

Argument marshalling only: every step of the blend runs in the CUDA library behind the C ABI
declared in ``include/cacheblend.h``.  PyTorch is used for device memory and streams.  There is
no fallback: if ``libcacheblend.so`` is missing or cannot be loaded, every call raises.

Entry points (same names as the C ABI): ``cb_model_create``, ``cb_model_destroy``,
``cb_rerope``, ``cb_blend``, ``cb_blend_gradual``, ``cb_selected_count``, ``cb_last_error``;
``BlendModel`` bundles a handle with the device tensors it borrows.
"""
from __future__ import annotations

import ctypes
import os

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libcacheblend.so")

CB_OK, CB_ERR_INVALID_ARG, CB_ERR_UNSUPPORTED, CB_ERR_OOM, CB_ERR_CUDA, CB_ERR_INTERNAL = 0, -1, -2, -3, -4, -5
CB_F32, CB_BF16 = 0, 1
CB_PREC_SPLIT, CB_PREC_BF16 = 0, 1
CB_MAX_CHUNKS = 1024
EXPORTED = ("cb_model_create", "cb_model_destroy", "cb_rerope", "cb_blend", "cb_blend_gradual", "cb_blend_streamed",
            "cb_selected_count", "cb_last_error", "cb_profile_enable", "cb_profile_read", "cb_model_status",
            "cb_rerope_static", "cb_model_diag", "cb_load_time", "cb_controller_ratio", "cb_pick_storage",
            "cb_blend_paged", "cb_kv_gather_pages", "cb_kv_scatter_pages", "cb_pages_create", "cb_pages_destroy",
            "cb_pages_alloc", "cb_pages_retain", "cb_pages_release", "cb_pages_plan_write", "cb_pages_count",
            "cb_pages_free", "cb_index_create", "cb_index_destroy", "cb_index_size", "cb_index_match",
            "cb_select_hkvd", "cb_blend_hkvd", "cb_gradual_layout")
CB_STATIC_MAX_CHUNKS = 256
CB_STATUS_BAD_TOKEN, CB_STATUS_WAIT_TIMEOUT, CB_STATUS_BAD_ROW = 1, 2, 4


class CbConfig(ctypes.Structure):
    _fields_ = [("n_layers", ctypes.c_int32), ("d_model", ctypes.c_int32), ("n_heads", ctypes.c_int32),
                ("n_kv_heads", ctypes.c_int32), ("head_dim", ctypes.c_int32), ("ffn_hidden", ctypes.c_int32),
                ("vocab", ctypes.c_int32), ("rope_theta", ctypes.c_double), ("rms_eps", ctypes.c_float),
                ("dtype", ctypes.c_int32), ("max_tokens", ctypes.c_int32), ("max_chunks", ctypes.c_int32),
                ("precision", ctypes.c_int32)]


_PP = ctypes.POINTER(ctypes.c_void_p)


class CbWeights(ctypes.Structure):
    _fields_ = [("embed", ctypes.c_void_p), ("final_norm", ctypes.c_void_p), ("lm_head", ctypes.c_void_p),
                ("attn_norm", _PP), ("wq", _PP), ("wk", _PP), ("wv", _PP), ("wo", _PP), ("mlp_norm", _PP),
                ("w_gate", _PP), ("w_up", _PP), ("w_down", _PP)]


class CbChunk(ctypes.Structure):
    _fields_ = [("src_pos", ctypes.c_int32), ("dst_pos", ctypes.c_int32), ("len", ctypes.c_int32)]


class CbStats(ctypes.Structure):
    _fields_ = [("n_tokens", ctypes.c_int32), ("n_ctx", ctypes.c_int32), ("n_selected", ctypes.c_int32),
                ("n_recompute", ctypes.c_int32), ("kernel_launches", ctypes.c_int32), ("reserved", ctypes.c_int32),
                ("gemm_flops", ctypes.c_double), ("attn_flops", ctypes.c_double),
                ("kv_bytes_moved", ctypes.c_double)]


class CbLayerIO(ctypes.Structure):
    _fields_ = [("cached_kv_host", ctypes.c_void_p), ("out_kv_host", ctypes.c_void_p), ("copy_stream", ctypes.c_void_p),
                ("copy_back_stream", ctypes.c_void_p)]


class CbPagedKV(ctypes.Structure):
    _fields_ = [("pool", ctypes.c_void_p), ("n_pages", ctypes.c_int64), ("page_size", ctypes.c_int32),
                ("src_table", ctypes.c_void_p), ("dst_table", ctypes.c_void_p)]


class CbKernelProfile(ctypes.Structure):
    _fields_ = [("name", ctypes.c_char * 24), ("launches", ctypes.c_int32), ("ms", ctypes.c_double),
                ("flops", ctypes.c_double), ("bytes", ctypes.c_double)]


class CacheBlendError(RuntimeError):
    def __init__(self, code: int, msg: str):
        super().__init__(f"[{code}] {msg}")
        self.code = code


_lib = None


def build(force: bool = False) -> str:
    from . import buildlib
    return buildlib.build(force=force)


def lib() -> ctypes.CDLL:
    """Load libcacheblend.so (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"libcacheblend.so is not built ({LIB_PATH}); run __graft_entry__.build()")
        L = ctypes.CDLL(LIB_PATH)
        vp, i32, i64 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64
        L.cb_model_create.restype = ctypes.c_int
        L.cb_model_create.argtypes = [ctypes.POINTER(CbConfig), ctypes.POINTER(CbWeights), ctypes.POINTER(vp)]
        L.cb_model_destroy.restype = ctypes.c_int
        L.cb_model_destroy.argtypes = [vp]
        L.cb_rerope.restype = ctypes.c_int
        L.cb_rerope.argtypes = [vp, vp, i64, ctypes.POINTER(CbChunk), i32, vp]
        L.cb_blend.restype = ctypes.c_int
        L.cb_blend.argtypes = [vp, vp, i32, vp, ctypes.POINTER(CbChunk), i32, ctypes.c_double, vp, vp, vp, vp,
                               ctypes.POINTER(CbStats), vp]
        L.cb_blend_gradual.restype = ctypes.c_int
        L.cb_blend_gradual.argtypes = [vp, vp, i32, vp, ctypes.POINTER(CbChunk), i32, ctypes.POINTER(ctypes.c_double),
                                       i32, vp, vp, vp, vp, ctypes.POINTER(CbStats), vp]
        L.cb_blend_streamed.restype = ctypes.c_int
        L.cb_blend_streamed.argtypes = [vp, vp, i32, ctypes.POINTER(CbLayerIO), ctypes.POINTER(CbChunk), i32,
                                        ctypes.POINTER(ctypes.c_double), i32, vp, vp, vp, vp, ctypes.POINTER(CbStats), vp]
        L.cb_load_time.restype = ctypes.c_double
        L.cb_load_time.argtypes = [ctypes.c_double, i64, ctypes.c_double]
        L.cb_controller_ratio.restype = ctypes.c_double
        L.cb_controller_ratio.argtypes = [ctypes.c_double, ctypes.c_double, ctypes.c_double]
        L.cb_pick_storage.restype = i32
        L.cb_pick_storage.argtypes = [ctypes.POINTER(ctypes.c_double), ctypes.POINTER(ctypes.c_double), i32,
                                      ctypes.c_double, i64, ctypes.c_double, ctypes.c_double]
        L.cb_blend_paged.restype = ctypes.c_int
        L.cb_blend_paged.argtypes = [vp, vp, i32, ctypes.POINTER(CbPagedKV), ctypes.POINTER(CbChunk), i32,
                                     ctypes.POINTER(ctypes.c_double), i32, vp, vp, vp, vp, ctypes.POINTER(CbStats), vp]
        L.cb_kv_gather_pages.restype = ctypes.c_int
        L.cb_kv_gather_pages.argtypes = [vp, ctypes.POINTER(CbPagedKV), i32, vp, vp]
        L.cb_kv_scatter_pages.restype = ctypes.c_int
        L.cb_kv_scatter_pages.argtypes = [vp, vp, i32, ctypes.POINTER(CbPagedKV), vp]
        ip = ctypes.POINTER(ctypes.c_int32)
        L.cb_pages_create.restype = ctypes.c_int
        L.cb_pages_create.argtypes = [i64, ctypes.POINTER(vp)]
        L.cb_pages_destroy.restype = ctypes.c_int
        L.cb_pages_destroy.argtypes = [vp]
        L.cb_pages_alloc.restype = ctypes.c_int
        L.cb_pages_alloc.argtypes = [vp, i32, ip]
        L.cb_pages_retain.restype = ctypes.c_int
        L.cb_pages_retain.argtypes = [vp, ip, i32]
        L.cb_pages_release.restype = ctypes.c_int
        L.cb_pages_release.argtypes = [vp, ip, i32]
        L.cb_pages_plan_write.restype = i32
        L.cb_pages_plan_write.argtypes = [vp, ip, i32, ip]
        L.cb_pages_count.restype = i32
        L.cb_pages_count.argtypes = [vp, i32]
        L.cb_pages_free.restype = i64
        L.cb_pages_free.argtypes = [vp]
        L.cb_index_create.restype = ctypes.c_int
        L.cb_index_create.argtypes = [i32, vp, vp, vp, vp, i32, i32, ctypes.POINTER(vp)]
        L.cb_index_destroy.restype = ctypes.c_int
        L.cb_index_destroy.argtypes = [vp]
        L.cb_index_size.restype = i32
        L.cb_index_size.argtypes = [vp, i32]
        L.cb_index_match.restype = ctypes.c_int
        L.cb_index_match.argtypes = [vp, vp, i32, i32, i32, i32, vp, i32, vp, vp]
        L.cb_selected_count.restype = i32
        L.cb_selected_count.argtypes = [i32, ctypes.c_double]
        L.cb_gradual_layout.restype = i32
        L.cb_gradual_layout.argtypes = [i32, ctypes.POINTER(ctypes.c_double), i32, vp, vp, vp, i32]
        L.cb_select_hkvd.restype = ctypes.c_int
        L.cb_select_hkvd.argtypes = [vp, i32, i32, vp, vp]
        L.cb_blend_hkvd.restype = ctypes.c_int
        L.cb_blend_hkvd.argtypes = [vp, vp, i32, vp, ctypes.POINTER(CbChunk), i32, vp, i32, vp, vp,
                                    ctypes.POINTER(CbStats), vp]
        L.cb_profile_enable.restype = ctypes.c_int
        L.cb_profile_enable.argtypes = [vp, i32, i32]
        L.cb_profile_read.restype = i32
        L.cb_profile_read.argtypes = [vp, ctypes.POINTER(CbKernelProfile), i32]
        L.cb_rerope_static.restype = ctypes.c_int
        L.cb_rerope_static.argtypes = [vp, i64, i32, i32, i32, ctypes.c_double, i32, ctypes.POINTER(CbChunk), i32, vp]
        L.cb_model_diag.restype = ctypes.c_int
        L.cb_model_diag.argtypes = [vp, ctypes.POINTER(ctypes.c_uint32)]
        L.cb_model_status.restype = ctypes.c_int
        L.cb_model_status.argtypes = [vp, ctypes.POINTER(ctypes.c_uint32), i32]
        L.cb_last_error.restype = ctypes.c_char_p
        L.cb_last_error.argtypes = []
        _lib = L
    return _lib


def cb_last_error() -> str:
    return lib().cb_last_error().decode()


def _check(code: int):
    if code != CB_OK:
        raise CacheBlendError(code, cb_last_error())


def cb_selected_count(n_ctx: int, ratio: float) -> int:
    return int(lib().cb_selected_count(n_ctx, ratio))


def cb_gradual_layout(n_ctx: int, ratios):
    """The comparing layers of a gradual schedule as a list of (layer, kept rows, compared rows), in the order
    cb_blend_gradual writes out_selected and out_dev.  Raises on an invalid schedule."""
    r = (ctypes.c_double * len(ratios))(*[float(x) for x in ratios])
    cap = len(ratios)
    lay, kept, cmp_ = (ctypes.c_int32 * cap)(), (ctypes.c_int32 * cap)(), (ctypes.c_int32 * cap)()
    n = int(lib().cb_gradual_layout(int(n_ctx), r, len(ratios), ctypes.addressof(lay), ctypes.addressof(kept),
                                    ctypes.addressof(cmp_), cap))
    if n < 0:
        raise ValueError(f"cb_gradual_layout: invalid schedule (status {n})")
    return [(int(lay[i]), int(kept[i]), int(cmp_[i])) for i in range(n)]


def cb_select_hkvd(dev, n: int, k: int, out_rows, stream=None) -> None:
    """The k rows of largest dev[0..n) (ties to the lower row), ascending, into out_rows (device tensors)."""
    _check(lib().cb_select_hkvd(_ptr(dev), n, k, _ptr(out_rows), _stream(stream)))


def _chunks(chunks):
    arr = (CbChunk * max(1, len(chunks)))()
    for i, (s, d, n) in enumerate(chunks):
        arr[i] = CbChunk(int(s), int(d), int(n))
    return arr


def _ptr(t) -> int:
    if t is None:
        return 0
    return t if isinstance(t, int) else int(t.data_ptr())


def _stream(stream) -> int:
    if stream is None:
        import torch
        stream = torch.cuda.current_stream()
    return stream if isinstance(stream, int) else int(stream.cuda_stream)


def cb_model_create(config: dict, weights: dict) -> int:
    """config: shape dict (n_layers, d_model, n_heads, n_kv_heads, head_dim, ffn_hidden, vocab, rope_theta,
    rms_eps, dtype 'bf16'|'f32', max_tokens, max_chunks, precision 'split'|'bf16'); weights: device pointers / tensors with keys
    embed, final_norm, lm_head and 'layers' (list of dicts of per-layer tensors)."""
    cfg = CbConfig(config["n_layers"], config["d_model"], config["n_heads"], config["n_kv_heads"],
                   config["head_dim"], config["ffn_hidden"], config["vocab"], float(config["rope_theta"]),
                   float(config.get("rms_eps", 1e-5)), CB_BF16 if config["dtype"] == "bf16" else CB_F32,
                   int(config["max_tokens"]), int(config.get("max_chunks", 256)),
                   CB_PREC_BF16 if config.get("precision", "split") == "bf16" else CB_PREC_SPLIT)
    L = config["n_layers"]
    tabs = {}
    for name in ("attn_norm", "wq", "wk", "wv", "wo", "mlp_norm", "w_gate", "w_up", "w_down"):
        tabs[name] = (ctypes.c_void_p * L)(*[_ptr(weights["layers"][i][name]) for i in range(L)])
    w = CbWeights(_ptr(weights["embed"]), _ptr(weights["final_norm"]), _ptr(weights["lm_head"]),
                  *[ctypes.cast(tabs[n], _PP) for n in ("attn_norm", "wq", "wk", "wv", "wo", "mlp_norm",
                                                         "w_gate", "w_up", "w_down")])
    h = ctypes.c_void_p()
    _check(lib().cb_model_create(ctypes.byref(cfg), ctypes.byref(w), ctypes.byref(h)))
    return h.value


def cb_model_destroy(handle: int) -> None:
    _check(lib().cb_model_destroy(handle))


def cb_rerope(handle: int, kv, n_rows: int, chunks, stream=None) -> None:
    _check(lib().cb_rerope(handle, _ptr(kv), int(n_rows), _chunks(chunks), len(chunks), _stream(stream)))


def cb_rerope_static(kv, n_rows: int, n_layers: int, n_kv_heads: int, head_dim: int, rope_theta: float, dtype: str,
                     chunks, stream=None) -> None:
    """In-place re-RoPE without a model handle and without any device allocation (see the header)."""
    _check(lib().cb_rerope_static(_ptr(kv), int(n_rows), int(n_layers), int(n_kv_heads), int(head_dim),
                                  float(rope_theta), CB_BF16 if dtype == "bf16" else CB_F32, _chunks(chunks),
                                  len(chunks), _stream(stream)))


def cb_blend(handle: int, tokens, n_tokens: int, cached_kv, chunks, ratio: float, out_kv, out_logits,
             out_selected=None, out_dev=None, stream=None, stats: bool = False):
    st = CbStats()
    _check(lib().cb_blend(handle, _ptr(tokens), int(n_tokens), _ptr(cached_kv), _chunks(chunks), len(chunks),
                          float(ratio), _ptr(out_kv), _ptr(out_logits), _ptr(out_selected), _ptr(out_dev),
                          ctypes.byref(st) if stats else None, _stream(stream)))
    if stats:
        return {f: getattr(st, f) for f, _ in CbStats._fields_}
    return None


def cb_blend_hkvd(handle: int, tokens, n_tokens: int, cached_kv, chunks, hkvd, k: int, out_kv, out_logits,
                  stream=None, stats: bool = False):
    """A blend whose recomputed context rows are the caller's (device int32 [k], ascending)."""
    st = CbStats()
    _check(lib().cb_blend_hkvd(handle, _ptr(tokens), int(n_tokens), _ptr(cached_kv), _chunks(chunks), len(chunks),
                               _ptr(hkvd), int(k), _ptr(out_kv), _ptr(out_logits), ctypes.byref(st) if stats else None,
                               _stream(stream)))
    if stats:
        return {f: getattr(st, f) for f, _ in CbStats._fields_}
    return None


def cb_blend_gradual(handle: int, tokens, n_tokens: int, cached_kv, chunks, ratios, out_kv, out_logits,
                     out_selected=None, out_dev=None, stream=None, stats: bool = False):
    """Gradual filtering: ratios[l - 1] is the ratio of layer l (n_layers - 1 entries, non-increasing counts)."""
    st = CbStats()
    r = (ctypes.c_double * max(1, len(ratios)))(*[float(x) for x in ratios])
    _check(lib().cb_blend_gradual(handle, _ptr(tokens), int(n_tokens), _ptr(cached_kv), _chunks(chunks), len(chunks),
                                  r, len(ratios), _ptr(out_kv), _ptr(out_logits), _ptr(out_selected), _ptr(out_dev),
                                  ctypes.byref(st) if stats else None, _stream(stream)))
    if stats:
        return {f: getattr(st, f) for f, _ in CbStats._fields_}
    return None


def cb_blend_streamed(handle: int, tokens, n_tokens: int, cached_kv_host, chunks, ratios, out_kv, out_logits,
                      out_kv_host=None, out_selected=None, out_dev=None, stream=None, copy_stream=None,
                      copy_back_stream=None, stats: bool = False):
    """Layer-wise load pipeline: the chunk caches come from pinned host memory (cached_kv_host), one layer
    per copy on copy_stream; out_kv_host (optional, pinned) receives each finished layer."""
    st = CbStats()
    r = (ctypes.c_double * max(1, len(ratios)))(*[float(x) for x in ratios])
    io = CbLayerIO(_ptr(cached_kv_host) or None, _ptr(out_kv_host) or None, _stream(copy_stream),
                   _stream(copy_back_stream) if copy_back_stream is not None else None)
    _check(lib().cb_blend_streamed(handle, _ptr(tokens), int(n_tokens), ctypes.byref(io), _chunks(chunks), len(chunks),
                                   r, len(ratios), _ptr(out_kv), _ptr(out_logits), _ptr(out_selected), _ptr(out_dev),
                                   ctypes.byref(st) if stats else None, _stream(stream)))
    if stats:
        return {f: getattr(st, f) for f, _ in CbStats._fields_}
    return None


def _paged(pool, n_pages, page_size, src_table=None, dst_table=None):
    return CbPagedKV(_ptr(pool) or None, int(n_pages), int(page_size), _ptr(src_table) or None, _ptr(dst_table) or None)


def cb_blend_paged(handle: int, tokens, n_tokens: int, pool, n_pages: int, page_size: int, src_table, dst_table, chunks,
                   ratios, work_kv, out_logits, out_selected=None, out_dev=None, stream=None, stats: bool = False):
    """Blend over a paged pool: chunk caches read through src_table, blended K/V written through dst_table
    (device int32 tables); work_kv is the caller's contiguous working copy."""
    st = CbStats()
    r = (ctypes.c_double * max(1, len(ratios)))(*[float(x) for x in ratios])
    pg = _paged(pool, n_pages, page_size, src_table, dst_table)
    _check(lib().cb_blend_paged(handle, _ptr(tokens), int(n_tokens), ctypes.byref(pg), _chunks(chunks), len(chunks),
                                r, len(ratios), _ptr(work_kv), _ptr(out_logits), _ptr(out_selected), _ptr(out_dev),
                                ctypes.byref(st) if stats else None, _stream(stream)))
    if stats:
        return {f: getattr(st, f) for f, _ in CbStats._fields_}
    return None


def cb_kv_gather_pages(handle: int, pool, n_pages: int, page_size: int, table, n_rows: int, out_kv, stream=None):
    pg = _paged(pool, n_pages, page_size, table, None)
    _check(lib().cb_kv_gather_pages(handle, ctypes.byref(pg), int(n_rows), _ptr(out_kv), _stream(stream)))


def cb_kv_scatter_pages(handle: int, kv, n_rows: int, pool, n_pages: int, page_size: int, table, stream=None):
    pg = _paged(pool, n_pages, page_size, None, table)
    _check(lib().cb_kv_scatter_pages(handle, _ptr(kv), int(n_rows), ctypes.byref(pg), _stream(stream)))


class Pages:
    """Host-side page bookkeeping of a pool (cb_pages_*): reference counts, allocation, copy-on-write plans."""

    def __init__(self, n_pages: int):
        h = ctypes.c_void_p()
        _check(lib().cb_pages_create(int(n_pages), ctypes.byref(h)))
        self.h = h.value

    @staticmethod
    def _arr(ids):
        return (ctypes.c_int32 * max(1, len(ids)))(*[int(i) for i in ids])

    def alloc(self, n: int) -> list:
        a = (ctypes.c_int32 * max(1, n))()
        _check(lib().cb_pages_alloc(self.h, int(n), a))
        return [a[i] for i in range(n)]

    def retain(self, ids):
        _check(lib().cb_pages_retain(self.h, self._arr(ids), len(ids)))

    def release(self, ids):
        _check(lib().cb_pages_release(self.h, self._arr(ids), len(ids)))

    def plan_write(self, table) -> tuple:
        """(dst table, number of copy-on-write pages)."""
        d = (ctypes.c_int32 * max(1, len(table)))()
        n = int(lib().cb_pages_plan_write(self.h, self._arr(table), len(table), d))
        if n < 0:
            raise CacheBlendError(n, cb_last_error())
        return [d[i] for i in range(len(table))], n

    def count(self, i: int) -> int:
        return int(lib().cb_pages_count(self.h, int(i)))

    def free(self) -> int:
        return int(lib().cb_pages_free(self.h))

    def close(self):
        if self.h:
            lib().cb_pages_destroy(self.h)
            self.h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


class FragmentIndex:
    """cb_index_*: an immutable fragment index on the device (built from host arrays) and its matcher."""

    def __init__(self, chunk_size: int, tokens, occ_ids, old_st, ns, max_tokens: int):
        t = np.ascontiguousarray(tokens, dtype=np.uint32).reshape(-1)
        o, s_, n_ = (np.ascontiguousarray(a, dtype=np.int32) for a in (occ_ids, old_st, ns))
        h = ctypes.c_void_p()
        _check(lib().cb_index_create(int(chunk_size), t.ctypes.data, o.ctypes.data, s_.ctypes.data, n_.ctypes.data,
                                     len(o), int(max_tokens), ctypes.byref(h)))
        self.h, self.chunk_size = h.value, chunk_size

    def size(self, what: int) -> int:
        return int(lib().cb_index_size(self.h, int(what)))

    def match_async(self, tokens, ns: int, out, out_count, stride: int = 1, greedy: bool = True, stream=None):
        """Enqueue a match: out (device int32 [max][3]) and out_count (device int32 [1])."""
        _check(lib().cb_index_match(self.h, _ptr(tokens), int(tokens.shape[0]), int(ns), int(stride),
                                    1 if greedy else 0, _ptr(out), int(out.shape[0]), _ptr(out_count),
                                    _stream(stream)))

    def match(self, tokens, ns: int, stride: int = 1, greedy: bool = True, max_out: int = 4096) -> list:
        """Matches as (occupant id, old_st, cur_st) triples (synchronises)."""
        import torch
        out = torch.empty((max_out, 3), dtype=torch.int32, device=tokens.device)
        cnt = torch.zeros(1, dtype=torch.int32, device=tokens.device)
        self.match_async(tokens, ns, out, cnt, stride, greedy)
        n = int(cnt.item())
        return [tuple(int(v) for v in r) for r in out[:min(n, max_out)].cpu().tolist()]

    def close(self):
        if self.h:
            lib().cb_index_destroy(self.h)
            self.h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def cb_load_time(per_token_kv_bytes: float, n_tokens: int, throughput_bytes_per_s: float) -> float:
    return float(lib().cb_load_time(float(per_token_kv_bytes), int(n_tokens), float(throughput_bytes_per_s)))


def cb_controller_ratio(t_prefill_s: float, t_load_s: float, r_min: float = 0.15) -> float:
    return float(lib().cb_controller_ratio(float(t_prefill_s), float(t_load_s), float(r_min)))


def cb_pick_storage(devices, per_token_kv_bytes: float, n_tokens: int, t_prefill_s: float, r_min: float = 0.15) -> int:
    """devices: list of (throughput bytes/s, cost per GB); returns the chosen index."""
    n = len(devices)
    bw = (ctypes.c_double * max(1, n))(*[float(d[0]) for d in devices])
    cost = (ctypes.c_double * max(1, n))(*[float(d[1]) for d in devices])
    i = int(lib().cb_pick_storage(bw, cost, n, float(per_token_kv_bytes), int(n_tokens), float(t_prefill_s),
                                  float(r_min)))
    if i < 0:
        raise CacheBlendError(i, cb_last_error())
    return i


def cb_model_status(handle: int, clear: bool = False) -> int:
    """Device status bits (CB_STATUS_*) recorded by the kernels; synchronises."""
    v = ctypes.c_uint32()
    _check(lib().cb_model_status(handle, ctypes.byref(v), 1 if clear else 0))
    return v.value


def cb_model_diag(handle: int) -> list:
    """16 diagnostic words (status bits, then the first bounded wait that gave up); synchronises."""
    w = (ctypes.c_uint32 * 16)()
    _check(lib().cb_model_diag(handle, w))
    return list(w)


def cb_profile_enable(handle: int, enable: bool = True, max_launches: int = 65536) -> None:
    _check(lib().cb_profile_enable(handle, 1 if enable else 0, int(max_launches)))


def cb_profile_read(handle: int) -> list:
    """Per kernel class: name, launches, ms, flops, bytes since the last read (synchronises)."""
    arr = (CbKernelProfile * 32)()
    n = lib().cb_profile_read(handle, arr, 32)
    if n < 0:
        raise CacheBlendError(n, cb_last_error())
    return [dict(name=arr[i].name.decode(), launches=arr[i].launches, ms=arr[i].ms, flops=arr[i].flops,
                 bytes=arr[i].bytes) for i in range(n)]


# ------------------------------------------------------------------------------------------------
# convenience: a model handle that owns the device copies of its weights
# ------------------------------------------------------------------------------------------------
def to_device(a: np.ndarray, device="cuda"):
    """numpy float32 or bfloat16-bit-pattern (uint16) array -> torch tensor on the device."""
    import torch
    if a.dtype == np.uint16:
        return torch.from_numpy(a.view(np.int16)).to(device).view(torch.bfloat16)
    return torch.from_numpy(np.ascontiguousarray(a)).to(device)


class BlendModel:
    """A cb_model handle plus the device weights it borrows."""

    def __init__(self, shape: dict, weights: dict, max_tokens: int, max_chunks: int = 256, device="cuda",
                 precision: str = "split"):
        import torch
        self.shape = dict(shape)
        self.device = torch.device(device)
        self.weights = {k: to_device(weights[k], device) for k in ("embed", "final_norm", "lm_head")}
        self.weights["layers"] = [{k: to_device(v, device) for k, v in lw.items()} for lw in weights["layers"]]
        cfg = dict(shape, max_tokens=max_tokens, max_chunks=max_chunks, precision=precision)
        self.handle = cb_model_create(cfg, self.weights)
        self.max_tokens = max_tokens
        self.kv_dtype = torch.bfloat16 if shape["dtype"] == "bf16" else torch.float32

    def status(self, clear: bool = False) -> int:
        return cb_model_status(self.handle, clear)

    def close(self):
        if self.handle:
            cb_model_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def kv_buffer(self, n_rows: int):
        import torch
        s = self.shape
        return torch.empty((s["n_layers"], 2, n_rows, s["n_kv_heads"], s["head_dim"]), dtype=self.kv_dtype,
                           device=self.device)

    def blend(self, tokens, cached_kv, chunks, ratio, out_kv=None, stream=None, want_dev=False, stats=False):
        """Run cb_blend; returns dict(out_kv, logits, selected, dev?, stats?).  Asynchronous on `stream`."""
        import torch
        n = int(tokens.shape[0])
        n_ctx = sum(c[2] for c in chunks)
        k = cb_selected_count(n_ctx, ratio)
        if out_kv is None:
            out_kv = self.kv_buffer(n)
        logits = torch.empty(self.shape["vocab"], dtype=torch.float32, device=self.device)
        sel = torch.empty(max(k, 1), dtype=torch.int32, device=self.device)
        dev = torch.empty(max(n_ctx, 1), dtype=torch.float32, device=self.device) if want_dev else None
        st = cb_blend(self.handle, tokens, n, cached_kv, chunks, ratio, out_kv, logits,
                      sel if k > 0 else None, dev, stream, stats)
        out = dict(out_kv=out_kv, logits=logits, selected=sel[:k], k=k)
        if want_dev:
            out["dev"] = dev[:n_ctx]
        if stats:
            out["stats"] = st
        return out

    def blend_hkvd(self, tokens, cached_kv, chunks, hkvd, out_kv=None, stream=None):
        """Run cb_blend_hkvd with the given recomputed context rows (device int32, ascending); returns
        dict(out_kv, logits).  Asynchronous on `stream`."""
        import torch
        n = int(tokens.shape[0])
        if out_kv is None:
            out_kv = self.kv_buffer(n)
        logits = torch.empty(self.shape["vocab"], dtype=torch.float32, device=self.device)
        cb_blend_hkvd(self.handle, tokens, n, cached_kv, chunks, hkvd, int(hkvd.numel()), out_kv, logits, stream)
        return dict(out_kv=out_kv, logits=logits)

    def blend_gradual(self, tokens, cached_kv, chunks, ratios, out_kv=None, stream=None, want_dev=False,
                      stats=False):
        """Run cb_blend_gradual; returns dict(out_kv, logits, counts [k_1..k_{L-1}], sets {layer: positions} for
        the check layer and every shrinking layer, devs {layer: deviations}?, stats?).  The sets and
        deviations are device tensors (asynchronous on `stream`)."""
        import torch
        n = int(tokens.shape[0])
        n_ctx = sum(c[2] for c in chunks)
        counts = [cb_selected_count(n_ctx, r) for r in ratios]
        try:
            layout = cb_gradual_layout(n_ctx, ratios)      # the library's own order of the outputs
        except ValueError:
            layout = []                                    # cb_blend_gradual below rejects it with its own error
        n_sel = sum(kept for _, kept, _ in layout)
        n_dev = sum(cmp_ for _, _, cmp_ in layout)
        if out_kv is None:
            out_kv = self.kv_buffer(n)
        logits = torch.empty(self.shape["vocab"], dtype=torch.float32, device=self.device)
        sel = torch.empty(max(n_sel, 1), dtype=torch.int32, device=self.device)
        dev = torch.empty(max(n_dev, 1), dtype=torch.float32, device=self.device) if want_dev else None
        st = cb_blend_gradual(self.handle, tokens, n, cached_kv, chunks, ratios, out_kv, logits,
                              sel if n_sel > 0 else None, dev, stream, stats)
        sets, devs, at, dat = {}, {}, 0, 0
        for l, kept, nd in layout:
            sets[l] = sel[at:at + kept]
            at += kept
            if want_dev:
                devs[l] = dev[dat:dat + nd]
                dat += nd
        out = dict(out_kv=out_kv, logits=logits, counts=counts, sets=sets)
        if want_dev:
            out["devs"] = devs
        if stats:
            out["stats"] = st
        return out

    def blend_streamed(self, tokens, cached_kv_host, chunks, ratios, out_kv=None, out_kv_host=None, stream=None,
                       copy_stream=None, copy_back_stream=None, stats=False):
        """Run cb_blend_streamed (chunk caches in pinned host memory, loaded layer by layer); returns
        dict(out_kv, out_kv_host, logits, stats?).  Asynchronous on `stream`."""
        import torch
        n = int(tokens.shape[0])
        if out_kv is None:
            out_kv = self.kv_buffer(n)
        logits = torch.empty(self.shape["vocab"], dtype=torch.float32, device=self.device)
        if copy_stream is None:
            copy_stream = torch.cuda.Stream(self.device)
        st = cb_blend_streamed(self.handle, tokens, n, cached_kv_host, chunks, ratios, out_kv, logits,
                               out_kv_host=out_kv_host, stream=stream, copy_stream=copy_stream,
                               copy_back_stream=copy_back_stream, stats=stats)
        out = dict(out_kv=out_kv, out_kv_host=out_kv_host, logits=logits)
        if stats:
            out["stats"] = st
        return out

    def prefill_chunk(self, tokens, stream=None):
        """A chunk prefilled alone at positions 0..len-1 (cb_blend with no cached chunks): its K/V cache."""
        return self.blend(tokens, None, [], 0.0, stream=stream)["out_kv"]
