"""Python binding of libtokenselect (token-level KV selection, sm_103a).

Argument marshalling only: every function below passes device pointers and
sizes to the C ABI declared in include/tokenselect.h, under the same names,
and raises TokenSelectError on a non-OK status. All arithmetic of the decode
step runs in the CUDA kernels of the library. There is no CPU fallback: if
libtokenselect.so is missing the import of the library fails loudly.

Tensors are torch tensors on the context's device; ``None`` passes NULL.
Streams default to torch's current stream.
"""
from __future__ import annotations

import ctypes
import os
from ctypes import POINTER, c_char_p, c_double, c_float, c_int, c_int64, c_void_p

__all__ = [
    "TokenSelectError", "Config", "SelectParams", "library", "library_path",
    "TS_KV_F32", "TS_KV_BF16", "TS_SELECT_TOPK", "TS_SELECT_TOPP", "STATUS",
    "TS_SCORE_HEAD_SOFT_VOTE", "TS_SCORE_LOGIT_SUM", "TS_SCORE_HEAD_HARD_VOTE", "ts_score_fn",
    "ts_prefill_chunk", "ts_select_blocks", "ts_append_kv",
    "ts_create", "ts_destroy", "ts_cache_create", "ts_cache_destroy", "ts_cache_reset",
    "ts_cache_check", "ts_score", "ts_select", "ts_sparse_attend", "ts_decode_step",
    "ts_get_status", "ts_status_str", "ts_version", "ts_profile_enable", "ts_profile_read",
    "ts_kernel_count", "ts_debug_phase_ns", "ts_sparse_attend_noalloc", "ts_set_wait_limit",
    "ts_inject_barrier_skip", "Context", "Cache", "Profile", "PROF_FAMILIES",
]

TS_KV_F32, TS_KV_BF16 = 0, 1
TS_SELECT_TOPK, TS_SELECT_TOPP = 0, 1
TS_SCORE_HEAD_SOFT_VOTE, TS_SCORE_LOGIT_SUM, TS_SCORE_HEAD_HARD_VOTE = 0, 1, 2
STATUS = {
    0: "TS_OK", 1: "TS_ERR_INVALID_ARG", 2: "TS_ERR_SHAPE", 3: "TS_ERR_UNSUPPORTED",
    4: "TS_ERR_CUDA", 5: "TS_ERR_PAGE_OOB", 6: "TS_ERR_CAPACITY", 7: "TS_ERR_TIMEOUT",
    8: "TS_ERR_COOP_UNAVAILABLE", 9: "TS_ERR_SEQ_LEN", 10: "TS_ERR_SCRATCH_LIMIT",
}
STATUS_CODE = {v: k for k, v in STATUS.items()}

library_path = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libtokenselect.so")


class TokenSelectError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {STATUS.get(status, status)}")


class Config(ctypes.Structure):
    _fields_ = [("n_q_heads", c_int), ("n_kv_heads", c_int), ("head_dim", c_int),
                ("page_size", c_int), ("kv_dtype", c_int), ("max_batch", c_int),
                ("max_pages_per_seq", c_int), ("num_pages", c_int64)]


class Profile(ctypes.Structure):
    _fields_ = [("ms", c_double * 6), ("launches", c_int64 * 6)]


PROF_FAMILIES = ("check", "score", "vote", "select", "attend", "step")


class SelectParams(ctypes.Structure):
    _fields_ = [("mode", c_int), ("k", c_int), ("n_sink", c_int), ("n_local", c_int),
                ("top_p", c_float), ("theta", c_float), ("softmax_scale", c_float), ("score_fn", c_int)]


_lib = None
_SIGS = {
    "ts_version": (c_int, []),
    "ts_status_str": (c_char_p, [c_int]),
    "ts_create": (c_int, [POINTER(c_void_p), POINTER(Config)]),
    "ts_destroy": (c_int, [c_void_p]),
    "ts_cache_create": (c_int, [c_void_p, POINTER(c_void_p), c_int, c_int]),
    "ts_cache_destroy": (c_int, [c_void_p]),
    "ts_cache_reset": (c_int, [c_void_p, c_void_p]),
    "ts_cache_check": (c_int, [c_void_p, c_void_p, c_int, c_void_p, c_int, c_float, c_void_p,
                               c_void_p, c_void_p]),
    "ts_score": (c_int, [c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_int, c_void_p,
                         c_float, c_void_p, c_int64, c_void_p]),
    "ts_score_fn": (c_int, [c_void_p, POINTER(SelectParams), c_void_p, c_void_p, c_void_p, c_void_p, c_int,
                            c_void_p, c_void_p, c_int64, c_void_p]),
    "ts_select": (c_int, [c_void_p, c_void_p, c_int, c_void_p, c_void_p, c_int64, c_void_p, c_int,
                          c_void_p, POINTER(SelectParams), c_void_p, c_int64, c_void_p, c_void_p]),
    "ts_sparse_attend": (c_int, [c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_void_p,
                                 c_int64, c_void_p, c_int, c_float, c_void_p, c_void_p, c_void_p]),
    "ts_decode_step": (c_int, [c_void_p, c_void_p, c_int, c_void_p, c_void_p, c_void_p, c_void_p,
                               c_void_p, c_int, POINTER(SelectParams), c_void_p, c_int64, c_void_p,
                               c_int64, c_void_p, c_void_p, c_void_p, c_void_p, c_void_p]),
    "ts_get_status": (c_int, [c_void_p, POINTER(c_int), c_void_p]),
    "ts_append_kv": (c_int, [c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_int, c_void_p, c_void_p, c_void_p]),
    "ts_select_blocks": (c_int, [c_void_p, c_void_p, c_int64, c_void_p, c_int, c_int, c_int, c_void_p, c_int64,
                                 c_void_p, c_void_p]),
    "ts_prefill_chunk": (c_int, [c_void_p, c_void_p, c_int, c_void_p, c_void_p, c_void_p, c_void_p, c_int,
                                 POINTER(SelectParams), c_void_p, c_int64, c_void_p, c_int64, c_void_p, c_void_p,
                                 c_void_p, c_void_p]),
    "ts_set_wait_limit": (c_int, [c_void_p, ctypes.c_uint64]),
    "ts_inject_barrier_skip": (c_int, [c_void_p, c_int, c_int]),
    "ts_profile_enable": (c_int, [c_void_p, c_int]),
    "ts_profile_read": (c_int, [c_void_p, c_void_p, c_int]),
    "ts_kernel_count": (c_int, [c_void_p, POINTER(c_int64)]),
    "ts_debug_phase_ns": (c_int, [c_void_p, c_void_p, c_void_p]),
    "ts_sparse_attend_noalloc": (c_int, [c_int, c_int, c_int, c_int, c_void_p, c_void_p, c_void_p, c_int64,
                                         c_void_p, c_int, c_void_p, c_int64, c_void_p, c_int, c_float,
                                         c_void_p, c_void_p, c_void_p, c_void_p]),
}


def library() -> ctypes.CDLL:
    """The loaded libtokenselect.so (built in-tree by token_level_sparse_gb300.build)."""
    global _lib
    if _lib is None:
        if not os.path.exists(library_path):
            raise ImportError(f"{library_path} is missing: build it with "
                              "`python -m token_level_sparse_gb300.build` (nvcc, sm_103a)")
        lib = ctypes.CDLL(library_path)
        for name, (res, args) in _SIGS.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _lib = lib
    return _lib


def _check(st: int, where: str):
    if st != 0:
        raise TokenSelectError(st, where)


def _p(t):
    """Device pointer of a tensor (None -> NULL; ints pass through)."""
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _s(stream):
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _params(mode=TS_SELECT_TOPK, k=2048, n_sink=4, n_local=512, top_p=0.9, theta=0.9, softmax_scale=0.0,
            score_fn=TS_SCORE_HEAD_SOFT_VOTE):
    if isinstance(mode, SelectParams):
        return mode
    return SelectParams(mode, k, n_sink, n_local, top_p, theta, softmax_scale, score_fn)


# ---------------------------------------------------------------- raw calls

def ts_version() -> int:
    return library().ts_version()


def ts_status_str(status: int) -> str:
    return library().ts_status_str(status).decode()


def ts_create(cfg: Config) -> int:
    h = c_void_p()
    _check(library().ts_create(ctypes.byref(h), ctypes.byref(cfg)), "ts_create")
    return h.value


def ts_destroy(ctx: int) -> None:
    _check(library().ts_destroy(ctx), "ts_destroy")


def ts_cache_create(ctx: int, n_layers: int, capacity: int) -> int:
    h = c_void_p()
    _check(library().ts_cache_create(ctx, ctypes.byref(h), n_layers, capacity), "ts_cache_create")
    return h.value


def ts_cache_destroy(cache: int) -> None:
    _check(library().ts_cache_destroy(cache), "ts_cache_destroy")


def ts_cache_reset(cache: int, stream=None) -> None:
    _check(library().ts_cache_reset(cache, _s(stream)), "ts_cache_reset")


def ts_cache_check(ctx, cache, layer, q, B, theta, hit, cos_out=None, stream=None) -> None:
    _check(library().ts_cache_check(ctx, cache, layer, _p(q), B, theta, _p(hit), _p(cos_out), _s(stream)),
           "ts_cache_check")


def ts_score(ctx, q, k_pool, page_table, seq_lens, B, skip, scale, vote, vote_stride, stream=None) -> None:
    _check(library().ts_score(ctx, _p(q), _p(k_pool), _p(page_table), _p(seq_lens), B, _p(skip), scale,
                              _p(vote), vote_stride, _s(stream)), "ts_score")


def ts_score_fn(ctx, params, q, k_pool, page_table, seq_lens, B, skip, vote, vote_stride, stream=None) -> None:
    _check(library().ts_score_fn(ctx, ctypes.byref(params), _p(q), _p(k_pool), _p(page_table), _p(seq_lens), B,
                                 _p(skip), _p(vote), vote_stride, _s(stream)), "ts_score_fn")


def ts_select(ctx, cache, layer, q, vote, vote_stride, seq_lens, B, hit, params, idx, idx_stride, count,
              stream=None) -> None:
    _check(library().ts_select(ctx, cache, layer, _p(q), _p(vote), vote_stride, _p(seq_lens), B, _p(hit),
                               ctypes.byref(params), _p(idx), idx_stride, _p(count), _s(stream)), "ts_select")


def ts_sparse_attend(ctx, q, k_pool, v_pool, page_table, idx, idx_stride, count, B, scale, out, lse=None,
                     stream=None) -> None:
    _check(library().ts_sparse_attend(ctx, _p(q), _p(k_pool), _p(v_pool), _p(page_table), _p(idx),
                                      idx_stride, _p(count), B, scale, _p(out), _p(lse), _s(stream)),
           "ts_sparse_attend")


def ts_decode_step(ctx, cache, layer, q, k_pool, v_pool, page_table, seq_lens, B, params, vote, vote_stride,
                   idx, idx_stride, count, out, lse=None, hit=None, stream=None) -> None:
    _check(library().ts_decode_step(ctx, cache, layer, _p(q), _p(k_pool), _p(v_pool), _p(page_table),
                                    _p(seq_lens), B, ctypes.byref(params), _p(vote), vote_stride, _p(idx),
                                    idx_stride, _p(count), _p(out), _p(lse), _p(hit), _s(stream)),
           "ts_decode_step")


def ts_sparse_attend_noalloc(n_q_heads, n_kv_heads, head_dim, kv_dtype, q, k_pool, v_pool, num_pages,
                             page_table, max_pages_per_seq, idx, idx_stride, count, B, scale, out, lse=None,
                             status=None, stream=None) -> None:
    """Sparse attention with no context and no allocation (fixed static scratch)."""
    _check(library().ts_sparse_attend_noalloc(n_q_heads, n_kv_heads, head_dim, kv_dtype, _p(q), _p(k_pool),
                                              _p(v_pool), num_pages, _p(page_table), max_pages_per_seq, _p(idx),
                                              idx_stride, _p(count), B, scale, _p(out), _p(lse), _p(status),
                                              _s(stream)), "ts_sparse_attend_noalloc")


def ts_get_status(ctx, stream=None) -> int:
    v = c_int(0)
    _check(library().ts_get_status(ctx, ctypes.byref(v), _s(stream)), "ts_get_status")
    return v.value


def ts_prefill_chunk(ctx, q, c, k_pool, v_pool, page_table, seq_lens, B, params, vote, vote_stride, idx,
                     idx_stride, count, out, lse=None, stream=None) -> None:
    _check(library().ts_prefill_chunk(ctx, _p(q), c, _p(k_pool), _p(v_pool), _p(page_table), _p(seq_lens), B,
                                      ctypes.byref(params), _p(vote), vote_stride, _p(idx), idx_stride, _p(count),
                                      _p(out), _p(lse), _s(stream)), "ts_prefill_chunk")


def ts_select_blocks(ctx, vote, vote_stride, seq_lens, B, block, budget, idx, idx_stride, count, stream=None):
    _check(library().ts_select_blocks(ctx, _p(vote), vote_stride, _p(seq_lens), B, block, budget, _p(idx),
                                      idx_stride, _p(count), _s(stream)), "ts_select_blocks")


def ts_append_kv(ctx, k_new, v_new, page_table, seq_lens, B, k_pool, v_pool, stream=None) -> None:
    _check(library().ts_append_kv(ctx, _p(k_new), _p(v_new), _p(page_table), _p(seq_lens), B, _p(k_pool),
                                  _p(v_pool), _s(stream)), "ts_append_kv")


def ts_set_wait_limit(ctx, ns: int) -> None:
    _check(library().ts_set_wait_limit(ctx, int(ns)), "ts_set_wait_limit")


def ts_inject_barrier_skip(ctx, cta: int, barrier: int) -> None:
    _check(library().ts_inject_barrier_skip(ctx, cta, barrier), "ts_inject_barrier_skip")


def ts_profile_enable(ctx, on: bool) -> None:
    _check(library().ts_profile_enable(ctx, 1 if on else 0), "ts_profile_enable")


def ts_profile_read(ctx, keep: bool = False) -> dict:
    """{family: (ms, launches)} added up over the recorded brackets."""
    p = Profile()
    _check(library().ts_profile_read(ctx, ctypes.byref(p), 1 if keep else 0), "ts_profile_read")
    return {f: (p.ms[i], p.launches[i]) for i, f in enumerate(PROF_FAMILIES)}


def ts_debug_phase_ns(ctx, stream=None) -> list:
    """Phase-boundary times (ns) of CTA 0 in the last persistent step kernel."""
    buf = (ctypes.c_uint64 * 64)()
    _check(library().ts_debug_phase_ns(ctx, buf, _s(stream)), "ts_debug_phase_ns")
    return list(buf)


def ts_kernel_count(ctx) -> int:
    v = c_int64(0)
    _check(library().ts_kernel_count(ctx, ctypes.byref(v)), "ts_kernel_count")
    return v.value


# ------------------------------------------------------- handle wrappers

class Context:
    """Owns a ts_ctx for one head geometry and pool; tensors in, nothing computed here."""

    def __init__(self, n_q_heads, n_kv_heads, head_dim, kv_dtype, max_batch, max_pages_per_seq,
                 num_pages, page_size=16):
        self.cfg = Config(n_q_heads, n_kv_heads, head_dim, page_size, kv_dtype, max_batch,
                          max_pages_per_seq, num_pages)
        self.handle = ts_create(self.cfg)
        self.max_tokens = max_pages_per_seq * page_size

    def close(self):
        if self.handle:
            ts_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def cache(self, n_layers, capacity):
        return Cache(self, n_layers, capacity)

    def score(self, q, k_pool, page_table, seq_lens, vote, skip=None, scale=0.0, stream=None):
        ts_score(self.handle, q, k_pool, page_table, seq_lens, q.shape[0], skip, scale, vote,
                 vote.stride(0), stream)

    def score_fn(self, params, q, k_pool, page_table, seq_lens, vote, skip=None, stream=None):
        ts_score_fn(self.handle, params, q, k_pool, page_table, seq_lens, q.shape[0], skip, vote, vote.stride(0),
                    stream)

    def select(self, vote, seq_lens, params, idx, count, cache=None, layer=0, q=None, hit=None, stream=None):
        ts_select(self.handle, cache.handle if cache else None, layer, q, vote, vote.stride(0), seq_lens,
                  seq_lens.shape[0], hit, params, idx, idx.stride(0), count, stream)

    def sparse_attend(self, q, k_pool, v_pool, page_table, idx, count, out, lse=None, scale=0.0, stream=None):
        ts_sparse_attend(self.handle, q, k_pool, v_pool, page_table, idx, idx.stride(0), count, q.shape[0],
                         scale, out, lse, stream)

    def decode_step(self, q, k_pool, v_pool, page_table, seq_lens, params, idx, count, out, lse=None,
                    hit=None, vote=None, cache=None, layer=0, stream=None):
        ts_decode_step(self.handle, cache.handle if cache else None, layer, q, k_pool, v_pool, page_table,
                       seq_lens, q.shape[0], params, vote, vote.stride(0) if vote is not None else 0, idx,
                       idx.stride(0), count, out, lse, hit, stream)

    def prefill_chunk(self, q, k_pool, v_pool, page_table, seq_lens, params, idx, count, out, lse=None, vote=None,
                      stream=None):
        """q [B][c][H][d]: one selection from the chunk's mean query, causal attention of every query."""
        ts_prefill_chunk(self.handle, q, q.shape[1], k_pool, v_pool, page_table, seq_lens, q.shape[0], params,
                         vote, vote.stride(0) if vote is not None else 0, idx, idx.stride(0), count, out, lse, stream)

    def append_kv(self, k_new, v_new, page_table, seq_lens, k_pool, v_pool, stream=None):
        """k_new / v_new [B][H_kv][d]: the current token's rows into position seq_lens[b] - 1."""
        ts_append_kv(self.handle, k_new, v_new, page_table, seq_lens, seq_lens.shape[0], k_pool, v_pool, stream)

    def select_blocks(self, vote, seq_lens, block, budget, idx, count, stream=None):
        ts_select_blocks(self.handle, vote, vote.stride(0), seq_lens, seq_lens.shape[0], block, budget, idx,
                         idx.stride(0), count, stream)

    def status(self, stream=None) -> int:
        return ts_get_status(self.handle, stream)


class Cache:
    """Owns a ts_cache (Selection Cache state: C_Q, C_T per sequence and layer)."""

    def __init__(self, ctx: Context, n_layers: int, capacity: int):
        self.ctx = ctx
        self.handle = ts_cache_create(ctx.handle, n_layers, capacity)

    def reset(self, stream=None):
        ts_cache_reset(self.handle, stream)

    def check(self, layer, q, theta, hit, cos_out=None, stream=None):
        ts_cache_check(self.ctx.handle, self.handle, layer, q, q.shape[0], theta, hit, cos_out, stream)

    def close(self):
        if self.handle:
            ts_cache_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def params(**kw) -> SelectParams:
    """SelectParams with the paper's defaults (k 2048, 4 sinks, 512 local, theta 0.9)."""
    return _params(**kw)
