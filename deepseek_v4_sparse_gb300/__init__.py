"""Python binding of libds4x.so — the GB300 lightning-indexer path.

Thin argument marshalling over the C ABI declared in include/ds4x.h: torch tensors
(device memory) are passed as raw pointers together with the current CUDA stream; every
step of the computation runs in the library's CUDA kernels. There is no fallback: if
libds4x.so has not been built (``python -c "import __graft_entry__ as g; g.build()"``)
every call raises.

Entry points (same names as the C ABI, without the ``ds4x_`` prefix):
  indexer_score, topk, sparse_attn, index_and_attend, workspace_bytes, decode,
  decode_workspace_bytes, topk_workspace_bytes, topk_static_scratch, device_status,
  selftest_bounded_wait, last_launch_count
"""
from __future__ import annotations

import ctypes
import math
import os
import threading

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libds4x.so")

OK, ERR_INVALID, ERR_UNSUPPORTED, ERR_CUDA, ERR_WORKSPACE, ERR_TIMEOUT = 0, -1, -2, -3, -4, -5
F16, BF16 = 0, 1
MAX_KTOP = 1024
MAX_WINDOW = 1024
MAX_RATIO = 65536
EXPORTS = (
    "ds4x_indexer_score", "ds4x_topk", "ds4x_topk_workspace_bytes", "ds4x_sparse_attn",
    "ds4x_index_and_attend", "ds4x_workspace_bytes", "ds4x_status_string",
    "ds4x_last_launch_count", "ds4x_device_status", "ds4x_selftest_bounded_wait",
    "ds4x_topk_static_scratch", "ds4x_decode", "ds4x_decode_workspace_bytes",
    "ds4x_index_and_attend_host", "ds4x_index_and_attend_host_bytes",
    "ds4x_local_pooled_attn", "ds4x_index_and_attend_local", "ds4x_workspace_bytes_local",
    "ds4x_index_and_attend_local_host", "ds4x_index_and_attend_local_host_bytes", "ds4x_compress",
    "ds4x_decode_local", "ds4x_decode_local_workspace_bytes",
)

_lock = threading.Lock()
_lib = None


class Ds4xError(RuntimeError):
    def __init__(self, fn: str, status: int):
        super().__init__(f"{fn} failed: {status_string(status)} ({status})")
        self.status = status


def load(path: str = LIB_PATH) -> ctypes.CDLL:
    """Load libds4x.so (once) and declare the C signatures."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(path):
            raise RuntimeError(f"libds4x.so is not built ({path}); run deepseek_v4_sparse_gb300.build.build()")
        lib = ctypes.CDLL(path)
        P, i32, i64, f32, sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_float, ctypes.c_size_t
        lib.ds4x_indexer_score.argtypes = [P, P, P, P, i32, i32, i32, i32, i32, P, i64, P]
        lib.ds4x_topk.argtypes = [P, i64, P, i32, i32, i32, i32, P, P, P, sz, P]
        lib.ds4x_topk_workspace_bytes.argtypes = [i32, i32, i32]
        lib.ds4x_topk_workspace_bytes.restype = sz
        lib.ds4x_sparse_attn.argtypes = [P, P, ctypes.c_int, P, i32, i32, i32, i32, i32, f32, P, P, P]
        lib.ds4x_index_and_attend.argtypes = [P, P, P, P, P, P, ctypes.c_int, i32, i32, i32, i32, i32,
                                              i32, i32, i32, f32, P, P, P, P, sz, P]
        lib.ds4x_workspace_bytes.argtypes = [i32, i32, i32]
        lib.ds4x_workspace_bytes.restype = sz
        lib.ds4x_index_and_attend_host.argtypes = [P, P, P, P, P, P, ctypes.c_int, i32, i32, i32, i32, i32,
                                                   i32, i32, i32, f32, P, P, P, i32, P, sz, P]
        lib.ds4x_index_and_attend_host_bytes.argtypes = [i32, i32, i32, i32, i32, i32, i32, i32]
        lib.ds4x_index_and_attend_host_bytes.restype = sz
        lib.ds4x_local_pooled_attn.argtypes = [P, P, P, ctypes.c_int, P, P, i32, i32, i32, i32, i32, i32, i32,
                                               i32, f32, P, P, P]
        lib.ds4x_index_and_attend_local.argtypes = [P, P, P, P, P, P, P, ctypes.c_int, i32, i32, i32, i32, i32,
                                                    i32, i32, i32, i32, i32, i32, f32, P, P, P, P, sz, P]
        lib.ds4x_workspace_bytes_local.argtypes = [i32, i32, i32, i32]
        lib.ds4x_workspace_bytes_local.restype = sz
        lib.ds4x_index_and_attend_local_host.argtypes = [P, P, P, P, P, P, P, ctypes.c_int, i32, i32, i32, i32,
                                                         i32, i32, i32, i32, i32, i32, i32, f32, P, P, P, i32, P,
                                                         sz, P]
        lib.ds4x_index_and_attend_local_host_bytes.argtypes = [i32, i32, i32, i32, i32, i32, i32, i32, i32, i32]
        lib.ds4x_index_and_attend_local_host_bytes.restype = sz
        lib.ds4x_compress.argtypes = [P, P, P, ctypes.c_int, i32, i32, i32, P, P, i32, P, P, P, P]
        lib.ds4x_decode.argtypes = [P, P, P, P, P, ctypes.c_int, i32, i32, P, P, i32, i32, i32, i32, i32, i32, i32,
                                    i32, i32, f32, P, P, P, P, P, sz, ctypes.POINTER(i32), P]
        lib.ds4x_decode_local.argtypes = [P, P, P, P, P, ctypes.c_int, i32, i32, P, P, i32, i32, i32, i32, i32, i32,
                                          i32, i32, i32, f32, P, i32, P, i32, P, P, P, P, P, sz, ctypes.POINTER(i32), P]
        lib.ds4x_decode_local_workspace_bytes.argtypes = [i32, i32, i32]
        lib.ds4x_decode_local_workspace_bytes.restype = sz
        lib.ds4x_decode_workspace_bytes.argtypes = [i32, i32]
        lib.ds4x_decode_workspace_bytes.restype = sz
        lib.ds4x_status_string.argtypes = [ctypes.c_int]
        lib.ds4x_status_string.restype = ctypes.c_char_p
        lib.ds4x_last_launch_count.argtypes = []
        lib.ds4x_device_status.argtypes = [P, ctypes.c_int]
        lib.ds4x_selftest_bounded_wait.argtypes = [i64, P]
        for f in ("ds4x_indexer_score", "ds4x_topk", "ds4x_sparse_attn", "ds4x_index_and_attend", "ds4x_decode",
                  "ds4x_index_and_attend_host", "ds4x_local_pooled_attn", "ds4x_index_and_attend_local",
                  "ds4x_index_and_attend_local_host", "ds4x_compress", "ds4x_decode_local",
                  "ds4x_last_launch_count", "ds4x_device_status", "ds4x_selftest_bounded_wait"):
            getattr(lib, f).restype = ctypes.c_int
        _lib = lib
        return lib


def status_string(status: int) -> str:
    return load().ds4x_status_string(status).decode()


def _check(fn: str, rc: int):
    if rc != OK:
        raise Ds4xError(fn, rc)


# ---------------------------------------------------------------------------- torch helpers
def _torch():
    import torch
    return torch


def _ptr(t):
    if t is None:
        return None
    torch = _torch()
    if isinstance(t, torch.Tensor):
        if not t.is_cuda:
            raise ValueError("tensors passed to libds4x must live on a CUDA device")
        if not t.is_contiguous():
            raise ValueError("tensors passed to libds4x must be contiguous")
        return ctypes.c_void_p(t.data_ptr())
    return ctypes.c_void_p(int(t))


def _stream(stream):
    if stream is None:
        torch = _torch()
        return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    if hasattr(stream, "cuda_stream"):
        return ctypes.c_void_p(stream.cuda_stream)
    return ctypes.c_void_p(int(stream))


# Buffers of host-entry calls whose work may still be running: the copies read and write host memory
# asynchronously, and PyTorch recycles a freed page-locked block (or a device block of another
# stream) without knowing about copies it did not issue, so each call's tensors stay referenced
# until an event recorded after it on its stream has completed.
_inflight = []


def _keep_until_done(stream, tensors):
    torch = _torch()
    if stream is None:
        s = torch.cuda.current_stream()
    elif isinstance(stream, torch.cuda.Stream):
        s = stream
    else:
        s = torch.cuda.ExternalStream(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))
    ev = torch.cuda.Event()
    ev.record(s)
    _inflight[:] = [(e, t) for (e, t) in _inflight if not e.query()]
    _inflight.append((ev, tuple(x for x in tensors if x is not None)))


def _kv_dtype(t) -> int:
    torch = _torch()
    if t.dtype == torch.float16:
        return F16
    if t.dtype == torch.bfloat16:
        return BF16
    raise ValueError(f"kv / q_attn must be float16 or bfloat16, got {t.dtype}")


def _need(t, dtype, name):
    if t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")


def _need_positions(positions, T: int):
    """positions must be int32 with at least one entry per token (the kernels read T of them)."""
    _need(positions, _torch().int32, "positions")
    if positions.numel() < T:
        raise ValueError(f"positions holds {positions.numel()} entries for {T} tokens")


# ------------------------------------------------------------------------------ entry points
def workspace_bytes(T: int, S: int, k_top: int) -> int:
    return int(load().ds4x_workspace_bytes(T, S, k_top))


def topk_workspace_bytes(T: int, S: int, k_top: int) -> int:
    return int(load().ds4x_topk_workspace_bytes(T, S, k_top))


def last_launch_count() -> int:
    return int(load().ds4x_last_launch_count())


def indexer_score(q, w, k, positions, ratio: int, scores=None, S: int | None = None, stream=None):
    """scores[t, s] = sum_h w[t,h] relu(q[t,h,:] . k[s,:]) for visible s, -inf for masked.
    q [T,H,D] fp16, w [T,H] fp16, k [>=S, D] fp16, positions [T] int32 (CUDA tensors)."""
    torch = _torch()
    _need(q, torch.float16, "q"); _need(w, torch.float16, "w"); _need(k, torch.float16, "k")
    T, H, D = q.shape
    _need_positions(positions, T)
    S = k.shape[0] if S is None else S
    if scores is None:
        scores = torch.empty((T, S), dtype=torch.float32, device=q.device)
    _need(scores, torch.float32, "scores")
    rc = load().ds4x_indexer_score(_ptr(q), _ptr(w), _ptr(k), _ptr(positions), T, H, D, S, ratio,
                                   _ptr(scores), scores.shape[1] if scores.dim() == 2 else S,
                                   _stream(stream))
    _check("ds4x_indexer_score", rc)
    return scores


def topk(scores, positions, S: int, ratio: int, k_top: int = 512, indices=None, counts=None,
         workspace=None, stream=None):
    """Exact per-token top-k of the visible scores, ascending row order, -1 padded."""
    torch = _torch()
    _need(scores, torch.float32, "scores")
    T, ld = scores.shape
    _need_positions(positions, T)
    dev = scores.device
    if indices is None:
        indices = torch.empty((T, k_top), dtype=torch.int32, device=dev)
    if counts is None:
        counts = torch.empty((T,), dtype=torch.int32, device=dev)
    need = topk_workspace_bytes(T, S, k_top)
    if workspace is None and need > 0:
        workspace = torch.empty((need,), dtype=torch.uint8, device=dev)
    wbytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    rc = load().ds4x_topk(_ptr(scores), ld, _ptr(positions), T, S, ratio, k_top, _ptr(indices),
                          _ptr(counts), _ptr(workspace), wbytes, _stream(stream))
    _check("ds4x_topk", rc)
    return indices, counts


def sparse_attn(q_attn, kv, indices, S: int | None = None, scale: float | None = None, out=None,
                lse=None, want_lse: bool = True, stream=None):
    """64-head MQA over the selected rows. q_attn [T,64,512], kv [>=S,512] (fp16 or bf16)."""
    torch = _torch()
    dt = _kv_dtype(q_attn)
    if kv.dtype != q_attn.dtype:
        raise ValueError("kv and q_attn must have the same dtype")
    T, Hq, Dkv = q_attn.shape
    S = kv.shape[0] if S is None else S
    k_top = indices.shape[1]
    scale = 1.0 / math.sqrt(Dkv) if scale is None else scale
    if out is None:
        out = torch.empty_like(q_attn)
    if lse is None and want_lse:
        lse = torch.empty((T, Hq), dtype=torch.float32, device=q_attn.device)
    rc = load().ds4x_sparse_attn(_ptr(q_attn), _ptr(kv), dt, _ptr(indices), T, Hq, Dkv, S, k_top,
                                 scale, _ptr(out), _ptr(lse), _stream(stream))
    _check("ds4x_sparse_attn", rc)
    return out, lse


def index_and_attend(q, w, k, positions, q_attn, kv, ratio: int, k_top: int = 512, S: int | None = None,
                     scale: float | None = None, indices=None, out=None, lse=None, workspace=None,
                     want_lse: bool = True, stream=None):
    """The whole path: score -> top-k -> sparse MQA. Returns (indices, out, lse)."""
    torch = _torch()
    dt = _kv_dtype(q_attn)
    T, H, D = q.shape
    _, Hq, Dkv = q_attn.shape
    S = k.shape[0] if S is None else S
    scale = 1.0 / math.sqrt(Dkv) if scale is None else scale
    dev = q.device
    if indices is None:
        indices = torch.empty((T, k_top), dtype=torch.int32, device=dev)
    if out is None:
        out = torch.empty_like(q_attn)
    if lse is None and want_lse:
        lse = torch.empty((T, Hq), dtype=torch.float32, device=dev)
    need = workspace_bytes(T, S, k_top)
    if workspace is None and need > 0:
        workspace = torch.empty((need,), dtype=torch.uint8, device=dev)
    wbytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    rc = load().ds4x_index_and_attend(_ptr(q), _ptr(w), _ptr(k), _ptr(positions), _ptr(q_attn), _ptr(kv),
                                      dt, T, H, D, S, ratio, k_top, Hq, Dkv, scale, _ptr(indices),
                                      _ptr(out), _ptr(lse), _ptr(workspace), wbytes, _stream(stream))
    _check("ds4x_index_and_attend", rc)
    return indices, out, lse


def _host_ptr(t):
    """A contiguous CPU tensor's host address (page-locked memory lets the copies overlap)."""
    if t is None:
        return None
    if t.is_cuda or not t.is_contiguous():
        raise ValueError("host tensors passed to ds4x_index_and_attend_host must be contiguous CPU tensors")
    return ctypes.c_void_p(t.data_ptr())


def index_and_attend_host_bytes(T: int, H: int, D: int, S: int, k_top: int, Hq: int, Dkv: int,
                                n_chunks: int = 0) -> int:
    return int(load().ds4x_index_and_attend_host_bytes(T, H, D, S, k_top, Hq, Dkv, n_chunks))


def index_and_attend_host(q, w, k, positions, q_attn, kv, ratio: int, k_top: int = 512, S: int | None = None,
                          scale: float | None = None, n_chunks: int = 0, indices=None, out=None, lse=None,
                          device_buffer=None, want_lse: bool = True, device=None, stream=None):
    """The whole path on host (CPU) tensors: copies in, computes, copies out, overlapped by sub-chunks
    of tokens.  Outputs are page-locked CPU tensors, valid once `stream` is synchronised.  The copies
    run after the call returns: every tensor passed or created here stays referenced until the
    call's work on `stream` is done.  Returns (indices, out, lse)."""
    torch = _torch()
    dt = _kv_dtype(q_attn)
    T, H, D = q.shape
    _, Hq, Dkv = q_attn.shape
    S = k.shape[0] if S is None else S
    scale = 1.0 / math.sqrt(Dkv) if scale is None else scale
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
    if indices is None:
        indices = torch.empty((T, k_top), dtype=torch.int32).pin_memory()
    if out is None:
        out = torch.empty(q_attn.shape, dtype=q_attn.dtype).pin_memory()
    if lse is None and want_lse:
        lse = torch.empty((T, Hq), dtype=torch.float32).pin_memory()
    need = index_and_attend_host_bytes(T, H, D, S, k_top, Hq, Dkv, n_chunks)
    if device_buffer is None:
        device_buffer = torch.empty((max(need, 16),), dtype=torch.uint8, device=dev)
    dbytes = device_buffer.numel() * device_buffer.element_size()
    rc = load().ds4x_index_and_attend_host(
        _host_ptr(q), _host_ptr(w), _host_ptr(k), _host_ptr(positions), _host_ptr(q_attn), _host_ptr(kv), dt, T,
        H, D, S, ratio, k_top, Hq, Dkv, scale, _host_ptr(indices), _host_ptr(out), _host_ptr(lse), n_chunks,
        _ptr(device_buffer), dbytes, _stream(stream))
    _check("ds4x_index_and_attend_host", rc)
    _keep_until_done(stream, (q, w, k, positions, q_attn, kv, indices, out, lse, device_buffer))
    return indices, out, lse


# ------------------------------------------------------------------ local-plus-pooled attention
def _rows(t):
    return 0 if t is None else int(t.shape[0])


def workspace_bytes_local(T: int, S: int, k_top: int, window: int) -> int:
    return int(load().ds4x_workspace_bytes_local(T, S, k_top, window))


def local_pooled_attn(q_attn, kv, kv_local, indices, positions, local_pos0: int, window: int,
                      S: int | None = None, scale: float | None = None, out=None, lse=None,
                      want_lse: bool = True, stream=None):
    """One softmax over the selected pooled rows of kv and the raw window rows of kv_local
    [L, 512] (row r = position local_pos0 + r). Returns (out, lse)."""
    torch = _torch()
    dt = _kv_dtype(q_attn)
    if kv.dtype != q_attn.dtype or (kv_local is not None and kv_local.dtype != q_attn.dtype):
        raise ValueError("kv, kv_local and q_attn must have the same dtype")
    T, Hq, Dkv = q_attn.shape
    S = kv.shape[0] if S is None else S
    k_top = indices.shape[1]
    scale = 1.0 / math.sqrt(Dkv) if scale is None else scale
    if out is None:
        out = torch.empty_like(q_attn)
    if lse is None and want_lse:
        lse = torch.empty((T, Hq), dtype=torch.float32, device=q_attn.device)
    rc = load().ds4x_local_pooled_attn(_ptr(q_attn), _ptr(kv), _ptr(kv_local), dt, _ptr(indices), _ptr(positions),
                                       T, Hq, Dkv, S, k_top, local_pos0, _rows(kv_local), window, scale, _ptr(out),
                                       _ptr(lse), _stream(stream))
    _check("ds4x_local_pooled_attn", rc)
    return out, lse


def index_and_attend_local(q, w, k, positions, q_attn, kv, kv_local, ratio: int, local_pos0: int, window: int,
                           k_top: int = 512, S: int | None = None, scale: float | None = None, indices=None,
                           out=None, lse=None, workspace=None, want_lse: bool = True, stream=None):
    """The whole path with local-plus-pooled attention. Returns (indices, out, lse)."""
    torch = _torch()
    dt = _kv_dtype(q_attn)
    T, H, D = q.shape
    _, Hq, Dkv = q_attn.shape
    S = k.shape[0] if S is None else S
    scale = 1.0 / math.sqrt(Dkv) if scale is None else scale
    dev = q.device
    if indices is None:
        indices = torch.empty((T, k_top), dtype=torch.int32, device=dev)
    if out is None:
        out = torch.empty_like(q_attn)
    if lse is None and want_lse:
        lse = torch.empty((T, Hq), dtype=torch.float32, device=dev)
    need = workspace_bytes_local(T, S, k_top, window)
    if workspace is None and need > 0:
        workspace = torch.empty((need,), dtype=torch.uint8, device=dev)
    wbytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    rc = load().ds4x_index_and_attend_local(_ptr(q), _ptr(w), _ptr(k), _ptr(positions), _ptr(q_attn), _ptr(kv),
                                            _ptr(kv_local), dt, T, H, D, S, ratio, k_top, Hq, Dkv, local_pos0,
                                            _rows(kv_local), window, scale, _ptr(indices), _ptr(out), _ptr(lse),
                                            _ptr(workspace), wbytes, _stream(stream))
    _check("ds4x_index_and_attend_local", rc)
    return indices, out, lse


def index_and_attend_local_host_bytes(T: int, H: int, D: int, S: int, k_top: int, Hq: int, Dkv: int, L: int,
                                      window: int, n_chunks: int = 0) -> int:
    return int(load().ds4x_index_and_attend_local_host_bytes(T, H, D, S, k_top, Hq, Dkv, L, window, n_chunks))


def index_and_attend_local_host(q, w, k, positions, q_attn, kv, kv_local, ratio: int, local_pos0: int,
                                window: int, k_top: int = 512, S: int | None = None, scale: float | None = None,
                                n_chunks: int = 0, indices=None, out=None, lse=None, device_buffer=None,
                                want_lse: bool = True, device=None, stream=None):
    """index_and_attend_host with the raw window (kv_local a CPU tensor too)."""
    torch = _torch()
    dt = _kv_dtype(q_attn)
    T, H, D = q.shape
    _, Hq, Dkv = q_attn.shape
    S = k.shape[0] if S is None else S
    L = _rows(kv_local)
    scale = 1.0 / math.sqrt(Dkv) if scale is None else scale
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
    if indices is None:
        indices = torch.empty((T, k_top), dtype=torch.int32).pin_memory()
    if out is None:
        out = torch.empty(q_attn.shape, dtype=q_attn.dtype).pin_memory()
    if lse is None and want_lse:
        lse = torch.empty((T, Hq), dtype=torch.float32).pin_memory()
    need = index_and_attend_local_host_bytes(T, H, D, S, k_top, Hq, Dkv, L, window, n_chunks)
    if device_buffer is None:
        device_buffer = torch.empty((max(need, 16),), dtype=torch.uint8, device=dev)
    dbytes = device_buffer.numel() * device_buffer.element_size()
    rc = load().ds4x_index_and_attend_local_host(
        _host_ptr(q), _host_ptr(w), _host_ptr(k), _host_ptr(positions), _host_ptr(q_attn), _host_ptr(kv),
        _host_ptr(kv_local), dt, T, H, D, S, ratio, k_top, Hq, Dkv, local_pos0, L, window, scale,
        _host_ptr(indices), _host_ptr(out), _host_ptr(lse), n_chunks, _ptr(device_buffer), dbytes, _stream(stream))
    _check("ds4x_index_and_attend_local_host", rc)
    _keep_until_done(stream, (q, w, k, positions, q_attn, kv, kv_local, indices, out, lse, device_buffer))
    return indices, out, lse


# ------------------------------------------------------------------------------- compressor
def compress(x, g, bias, ratio: int, frontier_x=None, frontier_g=None, rows=None, frontier_x_out=None,
             frontier_g_out=None, stream=None):
    """One gated-pooled row per `ratio` positions of the sequence frontier + (x, g).
    x, g [T, D] and the frontier [f, D] (f < ratio) fp16 or bf16; bias [ratio, D] fp32.
    Returns (rows [(f+T)//ratio, D], new frontier x, new frontier g [(f+T)%ratio, D])."""
    torch = _torch()
    dt = _kv_dtype(x)
    T, D = x.shape
    f = 0 if frontier_x is None else int(frontier_x.shape[0])
    n_out, rem = (f + T) // ratio, (f + T) % ratio
    if rows is None:
        rows = torch.empty((n_out, D), dtype=x.dtype, device=x.device)
    if frontier_x_out is None:
        frontier_x_out = torch.empty((rem, D), dtype=x.dtype, device=x.device)
    if frontier_g_out is None:
        frontier_g_out = torch.empty((rem, D), dtype=x.dtype, device=x.device)
    rc = load().ds4x_compress(_ptr(x), _ptr(g), _ptr(bias), dt, T, D, ratio, _ptr(frontier_x), _ptr(frontier_g), f,
                              _ptr(rows) if n_out else None, _ptr(frontier_x_out) if rem else None,
                              _ptr(frontier_g_out) if rem else None, _stream(stream))
    _check("ds4x_compress", rc)
    return rows, frontier_x_out, frontier_g_out


def decode_workspace_bytes(capacity: int, k_top: int = 512) -> int:
    return int(load().ds4x_decode_workspace_bytes(capacity, k_top))


def decode(q, w, q_attn, k, kv, S0: int, pos0: int, ratio: int, k_new=None, kv_new=None, k_top: int = 512,
           scale: float | None = None, positions=None, indices=None, out=None, lse=None, workspace=None,
           want_lse: bool = True, stream=None):
    """n_steps = q.shape[0] decode steps at positions pos0, pos0+1, ...; rows of k_new / kv_new are
    appended to k / kv (capacity = k.shape[0]) as the positions complete them.
    Returns (indices, out, lse, positions, S_final)."""
    torch = _torch()
    dt = _kv_dtype(kv)
    n_steps, H, D = q.shape
    _, Hq, Dkv = q_attn.shape
    capacity = k.shape[0]
    if kv.shape[0] != capacity:
        raise ValueError("k and kv must have the same capacity")
    n_new = 0 if k_new is None else k_new.shape[0]
    scale = 1.0 / math.sqrt(Dkv) if scale is None else scale
    dev = q.device
    if positions is None:
        positions = torch.empty((n_steps,), dtype=torch.int32, device=dev)
    if indices is None:
        indices = torch.empty((n_steps, k_top), dtype=torch.int32, device=dev)
    if out is None:
        out = torch.empty_like(q_attn)
    if lse is None and want_lse:
        lse = torch.empty((n_steps, Hq), dtype=torch.float32, device=dev)
    if workspace is None:
        workspace = torch.empty((max(decode_workspace_bytes(capacity, k_top), 16),), dtype=torch.uint8, device=dev)
    s_final = ctypes.c_int32(0)
    rc = load().ds4x_decode(_ptr(q), _ptr(w), _ptr(q_attn), _ptr(k), _ptr(kv), dt, capacity, S0, _ptr(k_new),
                            _ptr(kv_new), n_new, pos0, n_steps, H, D, ratio, k_top, Hq, Dkv, scale, _ptr(positions),
                            _ptr(indices), _ptr(out), _ptr(lse), _ptr(workspace),
                            workspace.numel() * workspace.element_size(), ctypes.byref(s_final), _stream(stream))
    _check("ds4x_decode", rc)
    return indices, out, lse, positions, int(s_final.value)


def decode_local_workspace_bytes(capacity: int, k_top: int = 512, window: int = 128) -> int:
    return int(load().ds4x_decode_local_workspace_bytes(capacity, k_top, window))


def decode_local(q, w, q_attn, k, kv, S0: int, pos0: int, ratio: int, kv_raw, kv_raw_new, window: int,
                 k_new=None, kv_new=None, k_top: int = 512, scale: float | None = None, positions=None,
                 indices=None, out=None, lse=None, workspace=None, want_lse: bool = True, stream=None):
    """decode() with local-plus-pooled attention: kv_raw [raw_capacity, 512] holds the raw row of
    each position (rows below pos0 are the window's history), kv_raw_new [n_steps, 512] the steps'
    own raw rows, written at rows pos0.. by the call. Returns (indices, out, lse, positions, S_final)."""
    torch = _torch()
    dt = _kv_dtype(kv)
    n_steps, H, D = q.shape
    _, Hq, Dkv = q_attn.shape
    capacity = k.shape[0]
    if kv.shape[0] != capacity:
        raise ValueError("k and kv must have the same capacity")
    if kv_raw.dtype != kv.dtype or kv_raw_new.dtype != kv.dtype:
        raise ValueError("kv_raw and kv_raw_new must have kv's dtype")
    n_new = 0 if k_new is None else k_new.shape[0]
    scale = 1.0 / math.sqrt(Dkv) if scale is None else scale
    dev = q.device
    if positions is None:
        positions = torch.empty((n_steps,), dtype=torch.int32, device=dev)
    if indices is None:
        indices = torch.empty((n_steps, k_top), dtype=torch.int32, device=dev)
    if out is None:
        out = torch.empty_like(q_attn)
    if lse is None and want_lse:
        lse = torch.empty((n_steps, Hq), dtype=torch.float32, device=dev)
    if workspace is None:
        workspace = torch.empty((max(decode_local_workspace_bytes(capacity, k_top, window), 16),), dtype=torch.uint8,
                                device=dev)
    s_final = ctypes.c_int32(0)
    rc = load().ds4x_decode_local(_ptr(q), _ptr(w), _ptr(q_attn), _ptr(k), _ptr(kv), dt, capacity, S0, _ptr(k_new),
                                  _ptr(kv_new), n_new, pos0, n_steps, H, D, ratio, k_top, Hq, Dkv, scale, _ptr(kv_raw),
                                  kv_raw.shape[0], _ptr(kv_raw_new), window, _ptr(positions), _ptr(indices),
                                  _ptr(out), _ptr(lse), _ptr(workspace), workspace.numel() * workspace.element_size(),
                                  ctypes.byref(s_final), _stream(stream))
    _check("ds4x_decode_local", rc)
    return indices, out, lse, positions, int(s_final.value)


def device_status(stream=None, clear: bool = True) -> int:
    return int(load().ds4x_device_status(_stream(stream), 1 if clear else 0))


def selftest_bounded_wait(timeout_ns: int, stream=None):
    _check("ds4x_selftest_bounded_wait", load().ds4x_selftest_bounded_wait(timeout_ns, _stream(stream)))


TOPK_STATIC_SCRATCH_BYTES = 4 << 20


def topk_static_scratch(scores, positions, S: int, ratio: int, k_top: int = 512, indices=None, counts=None,
                        stream=None):
    """ds4x_topk without a workspace, for callers that may not allocate device memory while they
    run (the split mode's candidate lists use a fixed array inside the library instead). The
    output tensors must be passed in by such callers; calls overlapping on the GPU must not be
    issued (they share that array)."""
    torch = _torch()
    _need(scores, torch.float32, "scores")
    T, ld = scores.shape
    _need_positions(positions, T)
    if indices is None:
        indices = torch.empty((T, k_top), dtype=torch.int32, device=scores.device)
    if counts is None:
        counts = torch.empty((T,), dtype=torch.int32, device=scores.device)
    lib = load()
    fn = lib.ds4x_topk_static_scratch
    P = ctypes.c_void_p
    fn.argtypes = [P, ctypes.c_int64, P, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32, P, P, P]
    fn.restype = ctypes.c_int
    _check("ds4x_topk_static_scratch", fn(_ptr(scores), ld, _ptr(positions), T, S, ratio, k_top, _ptr(indices),
                                          _ptr(counts), _stream(stream)))
    return indices, counts
