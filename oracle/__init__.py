"""CPU oracle of the lightning-indexer path — TEST INFRASTRUCTURE ONLY.

Only the tests, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline leg may
import this package. The product path (``deepseek_v4_sparse_gb300``) never does.

The arithmetic lives in ``ds4x_oracle.c`` (plain C, IEEE double, OpenMP over tokens);
this module compiles it with gcc when needed and wraps it for numpy arrays (host
memory). fp16/bf16 tensors are numpy uint16 arrays of raw bits. See the C file's
header for the passages each function follows and for how it is pinned.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "ds4x_oracle.c")
_LIB = os.path.join(_HERE, "libds4x_oracle.so")
_lock = threading.Lock()
_lib = None

DTYPES = {"f16": 0, "bf16": 1}


def build(force: bool = False, src: str = _SRC, out: str = _LIB) -> str:
    """Compile an oracle shared library (gcc, OpenMP). Returns its path."""
    if force or not os.path.exists(out) or os.path.getmtime(out) < os.path.getmtime(src):
        tmp = out + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-std=c11",
                               "-Wall", "-o", tmp, src, "-lm"])
        os.replace(tmp, out)
    return out


def _bind(lib):
    P = ctypes.c_void_p
    i32, i64, f32 = ctypes.c_int32, ctypes.c_int64, ctypes.c_float
    lib.ds4x_ref_indexer_score.argtypes = [P, P, P, P, i32, i32, i32, i32, i32, P, i64]
    lib.ds4x_ref_topk_ex.argtypes = [P, i64, P, i32, i32, i32, i32, P, P, ctypes.c_int]
    lib.ds4x_ref_sparse_attn.argtypes = [P, P, ctypes.c_int, P, i32, i32, i32, i32, i32, f32, P, P]
    lib.ds4x_ref_index_and_attend.argtypes = [P, P, P, P, P, P, ctypes.c_int, i32, i32, i32, i32,
                                              i32, i32, i32, i32, f32, P, P, P]
    lib.ds4x_ref_local_pooled_attn.argtypes = [P, P, P, ctypes.c_int, P, P, i32, i32, i32, i32, i32, i32,
                                               i32, i32, f32, P, P]
    lib.ds4x_ref_index_and_attend_local.argtypes = [P, P, P, P, P, P, P, ctypes.c_int, i32, i32, i32, i32,
                                                    i32, i32, i32, i32, i32, i32, i32, f32, P, P, P]
    lib.ds4x_ref_compress.argtypes = [P, P, P, ctypes.c_int, i32, i32, i32, P, P, i32, P, P, P]
    lib.ds4x_ref_decode.argtypes = [P, P, P, P, P, ctypes.c_int, i32, i32, P, P, i32, i32, i32, i32, i32, i32,
                                    i32, i32, i32, f32, P, P, P, P, P]
    lib.ds4x_ref_decode_local.argtypes = [P, P, P, P, P, ctypes.c_int, i32, i32, P, P, i32, i32, i32, i32, i32,
                                          i32, i32, i32, i32, f32, P, i32, P, i32, P, P, P, P, P]
    lib.ds4x_ref_n_visible.argtypes = [i64, i64, i64]
    lib.ds4x_ref_n_visible.restype = i64
    lib.ds4x_ref_decode16.argtypes = [ctypes.c_uint16, ctypes.c_int]
    lib.ds4x_ref_decode16.restype = ctypes.c_double
    lib.ds4x_ref_encode16.argtypes = [ctypes.c_double, ctypes.c_int]
    lib.ds4x_ref_encode16.restype = ctypes.c_uint16
    for f in ("ds4x_ref_indexer_score", "ds4x_ref_topk_ex", "ds4x_ref_sparse_attn",
              "ds4x_ref_index_and_attend", "ds4x_ref_decode", "ds4x_ref_local_pooled_attn",
              "ds4x_ref_index_and_attend_local", "ds4x_ref_compress", "ds4x_ref_decode_local"):
        getattr(lib, f).restype = ctypes.c_int
    return lib


def _ptr(a: np.ndarray | None):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


class Oracle:
    """numpy-facing wrapper of one compiled oracle library (host memory only)."""

    def __init__(self, lib_path: str):
        self.path = lib_path
        self.lib = _bind(ctypes.CDLL(lib_path))

    def n_visible(self, p: int, ratio: int, S: int) -> int:
        return int(self.lib.ds4x_ref_n_visible(p, ratio, S))

    def decode16(self, x: int, dtype: str) -> float:
        return float(self.lib.ds4x_ref_decode16(x, DTYPES[dtype]))

    def encode16(self, x: float, dtype: str) -> int:
        return int(self.lib.ds4x_ref_encode16(x, DTYPES[dtype]))

    def indexer_score(self, q, w, k, positions, ratio, S=None, ld=None):
        """q [T,H,D], w [T,H], k [>=S, D] fp16 bits; returns scores [T, ld] float32
        (columns >= S are left NaN so that writes beyond S are detectable)."""
        q, w, k = _c(q, np.uint16), _c(w, np.uint16), _c(k, np.uint16)
        positions = _c(positions, np.int32)
        T, H, D = q.shape
        S = k.shape[0] if S is None else S
        ld = S if ld is None else ld
        out = np.full((T, ld), np.nan, dtype=np.float32)
        rc = self.lib.ds4x_ref_indexer_score(_ptr(q), _ptr(w), _ptr(k), _ptr(positions), T, H, D,
                                             S, ratio, _ptr(out), ld)
        assert rc == 0, rc
        return out

    def topk(self, scores, positions, S, ratio, k_top, shortcut=True):
        """scores [T, ld] float32; returns (indices [T,k_top] int32, counts [T] int32)."""
        scores = _c(scores, np.float32)
        positions = _c(positions, np.int32)
        T, ld = scores.shape
        idx = np.empty((T, k_top), dtype=np.int32)
        cnt = np.empty((T,), dtype=np.int32)
        rc = self.lib.ds4x_ref_topk_ex(_ptr(scores), ld, _ptr(positions), T, S, ratio, k_top,
                                       _ptr(idx), _ptr(cnt), 1 if shortcut else 0)
        assert rc == 0, rc
        return idx, cnt

    def sparse_attn(self, q_attn, kv, dtype, indices, S, scale):
        """q_attn [T,Hq,Dkv], kv [>=S,Dkv] raw bits of `dtype`; indices [T,k_top] int32.
        Returns (out [T,Hq,Dkv] uint16 bits, lse [T,Hq] float32)."""
        q_attn, kv = _c(q_attn, np.uint16), _c(kv, np.uint16)
        indices = _c(indices, np.int32)
        T, Hq, Dkv = q_attn.shape
        k_top = indices.shape[1]
        out = np.empty((T, Hq, Dkv), dtype=np.uint16)
        lse = np.empty((T, Hq), dtype=np.float32)
        rc = self.lib.ds4x_ref_sparse_attn(_ptr(q_attn), _ptr(kv), DTYPES[dtype], _ptr(indices), T,
                                           Hq, Dkv, S, k_top, scale, _ptr(out), _ptr(lse))
        assert rc == 0, rc
        return out, lse

    def index_and_attend(self, q, w, k, positions, q_attn, kv, kv_dtype, S, ratio, k_top, scale):
        """The whole path. Returns (indices, out bits, lse)."""
        q, w, k = _c(q, np.uint16), _c(w, np.uint16), _c(k, np.uint16)
        q_attn, kv = _c(q_attn, np.uint16), _c(kv, np.uint16)
        positions = _c(positions, np.int32)
        T, H, D = q.shape
        _, Hq, Dkv = q_attn.shape
        idx = np.empty((T, k_top), dtype=np.int32)
        out = np.empty((T, Hq, Dkv), dtype=np.uint16)
        lse = np.empty((T, Hq), dtype=np.float32)
        rc = self.lib.ds4x_ref_index_and_attend(_ptr(q), _ptr(w), _ptr(k), _ptr(positions),
                                                _ptr(q_attn), _ptr(kv), DTYPES[kv_dtype], T, H, D,
                                                S, ratio, k_top, Hq, Dkv, scale, _ptr(idx),
                                                _ptr(out), _ptr(lse))
        assert rc == 0, rc
        return idx, out, lse

    def local_pooled_attn(self, q_attn, kv, kv_local, dtype, indices, positions, S, local_pos0, window,
                          scale):
        """One softmax over the selected pooled rows of kv [>=S, Dkv] and the raw window rows
        of kv_local [L, Dkv] (row r = position local_pos0 + r). Returns (out bits, lse)."""
        q_attn, kv, kv_local = _c(q_attn, np.uint16), _c(kv, np.uint16), _c(kv_local, np.uint16)
        indices, positions = _c(indices, np.int32), _c(positions, np.int32)
        T, Hq, Dkv = q_attn.shape
        k_top = indices.shape[1]
        out = np.empty((T, Hq, Dkv), dtype=np.uint16)
        lse = np.empty((T, Hq), dtype=np.float32)
        rc = self.lib.ds4x_ref_local_pooled_attn(_ptr(q_attn), _ptr(kv), _ptr(kv_local), DTYPES[dtype],
                                                 _ptr(indices), _ptr(positions), T, Hq, Dkv, S, k_top,
                                                 local_pos0, kv_local.shape[0], window, scale, _ptr(out),
                                                 _ptr(lse))
        assert rc == 0, rc
        return out, lse

    def index_and_attend_local(self, q, w, k, positions, q_attn, kv, kv_local, kv_dtype, S, ratio, k_top,
                               local_pos0, window, scale):
        """The whole path with local-plus-pooled attention. Returns (indices, out bits, lse)."""
        q, w, k = _c(q, np.uint16), _c(w, np.uint16), _c(k, np.uint16)
        q_attn, kv, kv_local = _c(q_attn, np.uint16), _c(kv, np.uint16), _c(kv_local, np.uint16)
        positions = _c(positions, np.int32)
        T, H, D = q.shape
        _, Hq, Dkv = q_attn.shape
        idx = np.empty((T, k_top), dtype=np.int32)
        out = np.empty((T, Hq, Dkv), dtype=np.uint16)
        lse = np.empty((T, Hq), dtype=np.float32)
        rc = self.lib.ds4x_ref_index_and_attend_local(
            _ptr(q), _ptr(w), _ptr(k), _ptr(positions), _ptr(q_attn), _ptr(kv), _ptr(kv_local),
            DTYPES[kv_dtype], T, H, D, S, ratio, k_top, Hq, Dkv, local_pos0, kv_local.shape[0], window, scale,
            _ptr(idx), _ptr(out), _ptr(lse))
        assert rc == 0, rc
        return idx, out, lse

    def compress(self, x, g, bias, dtype, ratio, fx=None, fg=None):
        """x, g [T, D] raw bits of `dtype`, bias [ratio, D] float32, frontier fx, fg [f, D] (f < ratio,
        None = empty). Returns (rows [(f+T)//ratio, D], new frontier x, new frontier g)."""
        x, g = _c(x, np.uint16), _c(g, np.uint16)
        bias = _c(bias, np.float32)
        T, D = x.shape
        f = 0 if fx is None else fx.shape[0]
        fx = np.zeros((1, D), np.uint16) if fx is None else _c(fx, np.uint16)
        fg = np.zeros((1, D), np.uint16) if fg is None else _c(fg, np.uint16)
        n_out, rem = (f + T) // ratio, (f + T) % ratio
        rows = np.empty((n_out, D), dtype=np.uint16)
        fx_out = np.empty((rem, D), dtype=np.uint16)
        fg_out = np.empty((rem, D), dtype=np.uint16)
        rc = self.lib.ds4x_ref_compress(_ptr(x), _ptr(g), _ptr(bias), DTYPES[dtype], T, D, ratio, _ptr(fx), _ptr(fg),
                                        f, _ptr(rows), _ptr(fx_out), _ptr(fg_out))
        assert rc == 0, rc
        return rows, fx_out, fg_out

    def decode(self, q, w, q_attn, k, kv, kv_dtype, S0, pos0, ratio, k_new, kv_new, k_top, scale):
        """The decode loop on copies of k / kv (capacity = their row count).
        Returns (indices, out bits, lse, positions, S per step, k after, kv after)."""
        q, w, q_attn = _c(q, np.uint16), _c(w, np.uint16), _c(q_attn, np.uint16)
        k, kv = np.array(k, dtype=np.uint16, copy=True), np.array(kv, dtype=np.uint16, copy=True)
        n_new = 0 if k_new is None else k_new.shape[0]
        k_new = None if k_new is None else _c(k_new, np.uint16)
        kv_new = None if kv_new is None else _c(kv_new, np.uint16)
        n_steps, H, D = q.shape
        _, Hq, Dkv = q_attn.shape
        idx = np.empty((n_steps, k_top), dtype=np.int32)
        out = np.empty((n_steps, Hq, Dkv), dtype=np.uint16)
        lse = np.empty((n_steps, Hq), dtype=np.float32)
        pos = np.empty((n_steps,), dtype=np.int32)
        s_steps = np.empty((n_steps,), dtype=np.int32)
        rc = self.lib.ds4x_ref_decode(_ptr(q), _ptr(w), _ptr(q_attn), _ptr(k), _ptr(kv), DTYPES[kv_dtype],
                                      k.shape[0], S0, _ptr(k_new), _ptr(kv_new), n_new, pos0, n_steps, H, D,
                                      ratio, k_top, Hq, Dkv, scale, _ptr(pos), _ptr(idx), _ptr(out), _ptr(lse),
                                      _ptr(s_steps))
        assert rc == 0, rc
        return idx, out, lse, pos, s_steps, k, kv

    def decode_local(self, q, w, q_attn, k, kv, kv_dtype, S0, pos0, ratio, k_new, kv_new, k_top, scale, kv_raw,
                     kv_raw_new, window):
        """decode() with the raw window, on copies of k / kv / kv_raw. Returns (indices, out bits, lse,
        positions, S per step, k after, kv after, kv_raw after)."""
        q, w, q_attn = _c(q, np.uint16), _c(w, np.uint16), _c(q_attn, np.uint16)
        k, kv = np.array(k, dtype=np.uint16, copy=True), np.array(kv, dtype=np.uint16, copy=True)
        kv_raw = np.array(kv_raw, dtype=np.uint16, copy=True)
        kv_raw_new = _c(kv_raw_new, np.uint16)
        n_new = 0 if k_new is None else k_new.shape[0]
        k_new = None if k_new is None else _c(k_new, np.uint16)
        kv_new = None if kv_new is None else _c(kv_new, np.uint16)
        n_steps, H, D = q.shape
        _, Hq, Dkv = q_attn.shape
        idx = np.empty((n_steps, k_top), dtype=np.int32)
        out = np.empty((n_steps, Hq, Dkv), dtype=np.uint16)
        lse = np.empty((n_steps, Hq), dtype=np.float32)
        pos = np.empty((n_steps,), dtype=np.int32)
        s_steps = np.empty((n_steps,), dtype=np.int32)
        rc = self.lib.ds4x_ref_decode_local(_ptr(q), _ptr(w), _ptr(q_attn), _ptr(k), _ptr(kv), DTYPES[kv_dtype],
                                            k.shape[0], S0, _ptr(k_new), _ptr(kv_new), n_new, pos0, n_steps, H, D,
                                            ratio, k_top, Hq, Dkv, scale, _ptr(kv_raw), kv_raw.shape[0],
                                            _ptr(kv_raw_new), window, _ptr(pos), _ptr(idx), _ptr(out), _ptr(lse),
                                            _ptr(s_steps))
        assert rc == 0, rc
        return idx, out, lse, pos, s_steps, k, kv, kv_raw


def default() -> Oracle:
    """The oracle built from ds4x_oracle.c (compiled on first use)."""
    global _lib
    with _lock:
        if _lib is None:
            _lib = Oracle(build())
    return _lib


def n_visible(p, ratio, S):
    return default().n_visible(p, ratio, S)


def decode16(x, dtype):
    return default().decode16(x, dtype)


def encode16(x, dtype):
    return default().encode16(x, dtype)


def indexer_score(*a, **kw):
    return default().indexer_score(*a, **kw)


def topk(*a, **kw):
    return default().topk(*a, **kw)


def sparse_attn(*a, **kw):
    return default().sparse_attn(*a, **kw)


def index_and_attend(*a, **kw):
    return default().index_and_attend(*a, **kw)


def decode(*a, **kw):
    return default().decode(*a, **kw)


def local_pooled_attn(*a, **kw):
    return default().local_pooled_attn(*a, **kw)


def index_and_attend_local(*a, **kw):
    return default().index_and_attend_local(*a, **kw)


def compress(*a, **kw):
    return default().compress(*a, **kw)


def decode_local(*a, **kw):
    return default().decode_local(*a, **kw)
