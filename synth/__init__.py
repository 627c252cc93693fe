"""Seeded synthetic inputs for the lightning-indexer path.

This module only draws numbers; it holds none of the indexer's arithmetic. Both the
CPU oracle tests and the CUDA path (tests, bench) take their inputs from here, so
the two sides always see the same bytes.

Generator: a counter-based splitmix64. Element i of stream `name` is
``mix(base(name) + i * GAMMA)`` where ``mix`` is the splitmix64 finaliser and
``base(name) = mix(seed ^ fnv1a64(name))``. From the 64-bit words:
  * uniform integers in [lo, hi]:  lo + (u mod (hi - lo + 1))
  * U[0,1):                        (u >> 11) * 2^-53
  * N(0,1):                        Box-Muller on the word pair (2i, 2i+1):
                                   r = sqrt(-2 ln u1), u1 = ((u >> 11) + 1) * 2^-53,
                                   element 2i = r cos(2 pi u2), element 2i+1 = r sin(2 pi u2)
Floating values are formed in float64, rounded to float32 (round-to-nearest-even) and
then to fp16 / bf16 (round-to-nearest-even). fp16/bf16 tensors are returned as numpy
uint16 arrays holding the raw bits.

Workloads follow the shapes of the pages' prefill chunks (2048 query tokens at 8k/32k/
64k context, ratio-4 compressed rows) and of 1M-context decode; see WORKLOADS.
"""
from __future__ import annotations

import math
import os
from dataclasses import dataclass, field

import numpy as np

MASK64 = (1 << 64) - 1
GAMMA = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)
_CHUNK = 1 << 22


def _mix_int(z: int) -> int:
    z &= MASK64
    z = ((z ^ (z >> 30)) * 0xBF58476D1CE4E5B9) & MASK64
    z = ((z ^ (z >> 27)) * 0x94D049BB133111EB) & MASK64
    return z ^ (z >> 31)


def _fnv1a64(s: str) -> int:
    h = 0xCBF29CE484222325
    for b in s.encode():
        h = ((h ^ b) * 0x100000001B3) & MASK64
    return h


def stream_base(seed: int, name: str) -> int:
    return _mix_int((seed ^ _fnv1a64(name)) & MASK64)


def words(seed: int, name: str, n: int, offset: int = 0) -> np.ndarray:
    """n consecutive 64-bit words (elements offset..offset+n-1) of stream `name`."""
    base = np.uint64(stream_base(seed, name))
    out = np.empty(n, dtype=np.uint64)
    with np.errstate(over="ignore"):
        for a in range(0, n, _CHUNK):
            b = min(n, a + _CHUNK)
            z = base + (np.arange(a + offset, b + offset, dtype=np.uint64) * GAMMA)
            z = (z ^ (z >> np.uint64(30))) * _M1
            z = (z ^ (z >> np.uint64(27))) * _M2
            out[a:b] = z ^ (z >> np.uint64(31))
    return out


def uniform_int(seed: int, name: str, n: int, lo: int, hi: int) -> np.ndarray:
    u = words(seed, name, n)
    return (np.int64(lo) + (u % np.uint64(hi - lo + 1)).astype(np.int64))


def uniform01(seed: int, name: str, n: int) -> np.ndarray:
    u = words(seed, name, n)
    return (u >> np.uint64(11)).astype(np.float64) * (2.0 ** -53)


def normal(seed: int, name: str, n: int, offset: int = 0) -> np.ndarray:
    """N(0,1) float64 values, elements offset..offset+n-1 of the stream."""
    p0 = offset // 2
    p1 = (offset + n + 1) // 2
    out = np.empty(2 * (p1 - p0), dtype=np.float64)
    for a in range(p0, p1, _CHUNK):
        b = min(p1, a + _CHUNK)
        u = words(seed, name, 2 * (b - a), offset=2 * a)
        u1 = ((u[0::2] >> np.uint64(11)).astype(np.float64) + 1.0) * (2.0 ** -53)
        u2 = (u[1::2] >> np.uint64(11)).astype(np.float64) * (2.0 ** -53)
        r = np.sqrt(-2.0 * np.log(u1))
        t = 2.0 * math.pi * u2
        seg = out[2 * (a - p0): 2 * (b - p0)]
        seg[0::2] = r * np.cos(t)
        seg[1::2] = r * np.sin(t)
    s = offset - 2 * p0
    return out[s:s + n]


def to_f16_bits(x: np.ndarray) -> np.ndarray:
    return np.asarray(x, dtype=np.float64).astype(np.float32).astype(np.float16).view(np.uint16)


def to_bf16_bits(x: np.ndarray) -> np.ndarray:
    u = np.asarray(x, dtype=np.float64).astype(np.float32).view(np.uint32).astype(np.uint64)
    r = (u + np.uint64(0x7FFF) + ((u >> np.uint64(16)) & np.uint64(1))) >> np.uint64(16)
    return r.astype(np.uint16)


def f16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    return np.asarray(b, dtype=np.uint16).view(np.float16).astype(np.float32)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def to_bits(x: np.ndarray, dtype: str) -> np.ndarray:
    return to_f16_bits(x) if dtype == "f16" else to_bf16_bits(x)


def bits_to_f32(b: np.ndarray, dtype: str) -> np.ndarray:
    return f16_bits_to_f32(b) if dtype == "f16" else bf16_bits_to_f32(b)


@dataclass(frozen=True)
class Workload:
    """Shapes and value recipe of one synthetic workload."""
    name: str
    T: int            # query tokens in the chunk
    H: int            # indexer heads
    D: int            # indexer dim
    S: int            # compressed rows present
    ratio: int        # tokens per compressed row
    pos0: int         # position of the first query token (tokens are consecutive)
    kind: str         # "int" (exact small integers) or "normal"
    kv_dtype: str     # "f16" or "bf16"
    Hq: int = 64
    Dkv: int = 512
    k_top: int = 512
    decode_steps: int = 0   # >0: a decode loop of this many single-token steps
    extra_rows: int = 0     # rows appended during the decode loop
    window: int = 0         # >0: raw sliding-window rows joined to the pooled ones (local-plus-pooled)
    tags: tuple = field(default_factory=tuple)

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.Dkv)

    @property
    def rows_capacity(self) -> int:
        return self.S + self.extra_rows


WORKLOADS = {
    # exact check: every product and sum is an exact fp32 value
    "tiny_exact": Workload("tiny_exact", T=512, H=16, D=64, S=1024, ratio=4, pos0=3584,
                           kind="int", kv_dtype="f16"),
    "prefill_8k": Workload("prefill_8k", T=2048, H=64, D=128, S=2048, ratio=4, pos0=6144,
                           kind="normal", kv_dtype="bf16"),
    "prefill_32k": Workload("prefill_32k", T=2048, H=64, D=128, S=8192, ratio=4, pos0=30720,
                            kind="normal", kv_dtype="bf16"),
    "prefill_64k": Workload("prefill_64k", T=2048, H=64, D=128, S=16384, ratio=4, pos0=63488,
                            kind="normal", kv_dtype="bf16"),
    # ratio-128 layer kind: every pooled row is attended (n_vis <= 512: sequential indices, no scoring)
    "pooled_64k_r128": Workload("pooled_64k_r128", T=2048, H=64, D=128, S=512, ratio=128, pos0=63488,
                                kind="normal", kv_dtype="bf16"),
    # local-plus-pooled attention: the 8k chunk with a 128-position raw window per token
    "prefill_8k_local128": Workload("prefill_8k_local128", T=2048, H=64, D=128, S=2048, ratio=4, pos0=6144,
                                    kind="normal", kv_dtype="bf16", window=128),
    "decode_1m": Workload("decode_1m", T=1, H=64, D=128, S=262144, ratio=4, pos0=1048575,
                          kind="normal", kv_dtype="bf16", decode_steps=256, extra_rows=64),
}


@dataclass
class Inputs:
    """Host copies of one workload's tensors (raw 16-bit storage for fp16/bf16)."""
    wl: Workload
    q: np.ndarray          # [T, H, D] uint16 (fp16 bits)
    w: np.ndarray          # [T, H] uint16 (fp16 bits)
    k: np.ndarray          # [rows, D] uint16 (fp16 bits)
    positions: np.ndarray  # [T] int32
    q_attn: np.ndarray     # [T, Hq, Dkv] uint16 (kv dtype bits)
    kv: np.ndarray         # [rows, Dkv] uint16 (kv dtype bits)
    kv_local: np.ndarray | None = None  # [L, Dkv] raw window rows (kv dtype bits), row r = position local_pos0 + r
    local_pos0: int = 0


_PARALLEL_MIN = 1 << 24


def _normal_bits_piece(job):
    seed, name, n, offset, dtype = job
    return to_bits(normal(seed, name, n, offset), dtype)


def normal_bits(seed: int, name: str, n: int, dtype: str) -> np.ndarray:
    """to_bits(normal(seed, name, n), dtype), drawn in pieces on a thread pool when n is large
    (numpy's array operations release the GIL); the counter-based stream makes the pieces
    independent, so the bits equal those of the single-piece draw."""
    workers = min(16, os.cpu_count() or 1)
    if n < _PARALLEL_MIN or workers < 2:
        return to_bits(normal(seed, name, n), dtype)
    import concurrent.futures as cf
    piece = ((n + 4 * workers - 1) // (4 * workers) + 1) & ~1     # even: whole Box-Muller pairs
    jobs = [(seed, name, min(piece, n - a), a, dtype) for a in range(0, n, piece)]
    with cf.ThreadPoolExecutor(workers) as ex:
        return np.concatenate(list(ex.map(_normal_bits_piece, jobs)))


def _bits(seed, wl: Workload, name: str, n: int, int_range, dtype: str) -> np.ndarray:
    if wl.kind == "int":
        return to_bits(uniform_int(seed, f"{wl.name}/{name}", n, *int_range).astype(np.float64), dtype)
    return normal_bits(seed, f"{wl.name}/{name}", n, dtype)


def make_inputs(wl: Workload, seed: int = 0, T: int | None = None, S: int | None = None,
                pos0: int | None = None, rows: int | None = None) -> Inputs:
    """Generate a workload's tensors. T/S/pos0/rows override the workload's sizes
    (used for down-scaled parity cases); the value recipe stays the same."""
    T = wl.T if T is None else T
    S = wl.S if S is None else S
    pos0 = wl.pos0 if pos0 is None else pos0
    rows = (S + wl.extra_rows) if rows is None else rows
    H, D, Hq, Dkv = wl.H, wl.D, wl.Hq, wl.Dkv
    q = _bits(seed, wl, "q", T * H * D, (-3, 3), "f16").reshape(T, H, D)
    k = _bits(seed, wl, "k", rows * D, (-3, 3), "f16").reshape(rows, D)
    if wl.kind == "int":
        sel = uniform_int(seed, f"{wl.name}/w", T * H, 0, 2)
        w = to_f16_bits(np.array([0.25, 0.5, 1.0])[sel]).reshape(T, H)
    else:
        w = to_f16_bits(uniform01(seed, f"{wl.name}/w", T * H) / 8.0).reshape(T, H)
    kvd = wl.kv_dtype
    q_attn = _bits(seed, wl, "q_attn", T * Hq * Dkv, (-2, 2), kvd).reshape(T, Hq, Dkv)
    kv = _bits(seed, wl, "kv", rows * Dkv, (-2, 2), kvd).reshape(rows, Dkv)
    positions = (pos0 + np.arange(T, dtype=np.int64)).astype(np.int32)
    kv_local, local_pos0 = None, 0
    if wl.window > 0:
        # the raw rows a prefill chunk needs: the window - 1 positions before it and its own
        local_pos0 = max(0, pos0 - wl.window + 1)
        L = pos0 + T - local_pos0
        kv_local = _bits(seed, wl, "kv_local", L * Dkv, (-2, 2), kvd).reshape(L, Dkv)
    return Inputs(wl, q, w, k, positions, q_attn, kv, kv_local, local_pos0)


def local_rows(seed: int, tag: str, L: int, Dkv: int, kind: str, kv_dtype: str) -> np.ndarray:
    """A raw-window row buffer [L, Dkv] for edge-case tests (kv dtype bits)."""
    wl = Workload(tag, T=0, H=1, D=1, S=0, ratio=1, pos0=0, kind=kind, kv_dtype=kv_dtype, Dkv=Dkv)
    return _bits(seed, wl, "kv_local", L * Dkv, (-2, 2), kv_dtype).reshape(L, Dkv)


def custom_inputs(seed: int, tag: str, T: int, H: int, D: int, rows: int, Hq: int, Dkv: int,
                  kind: str, kv_dtype: str, positions: np.ndarray, w_kind: str = "pos"):
    """Free-form inputs for edge-case tests. w_kind: "pos" = U(0,1)/8, "signed" = N(0,1),
    "pow2" = {1/4,1/2,1}."""
    wl = Workload(tag, T=T, H=H, D=D, S=rows, ratio=1, pos0=0, kind=kind, kv_dtype=kv_dtype,
                  Hq=Hq, Dkv=Dkv)
    q = _bits(seed, wl, "q", T * H * D, (-3, 3), "f16").reshape(T, H, D)
    k = _bits(seed, wl, "k", rows * D, (-3, 3), "f16").reshape(rows, D)
    if w_kind == "pow2":
        sel = uniform_int(seed, f"{tag}/w", T * H, 0, 2)
        w = to_f16_bits(np.array([0.25, 0.5, 1.0])[sel]).reshape(T, H)
    elif w_kind == "signed":
        w = to_f16_bits(normal(seed, f"{tag}/w", T * H)).reshape(T, H)
    else:
        w = to_f16_bits(uniform01(seed, f"{tag}/w", T * H) / 8.0).reshape(T, H)
    q_attn = _bits(seed, wl, "q_attn", T * Hq * Dkv, (-2, 2), kv_dtype).reshape(T, Hq, Dkv)
    kv = _bits(seed, wl, "kv", rows * Dkv, (-2, 2), kv_dtype).reshape(rows, Dkv)
    return Inputs(wl, q, w, k, np.asarray(positions, dtype=np.int32), q_attn, kv)


def compress_inputs(seed: int, tag: str, T: int, D: int, ratio: int, dtype: str, n_frontier: int = 0):
    """Compressor inputs: raw rows x and gate logits g [T, D] (N(0,1), dtype bits), a held-over
    frontier fx, fg [n_frontier, D] drawn the same way, and the per-position bias [ratio, D]
    (N(0,1), float32)."""
    x = normal_bits(seed, f"{tag}/x", T * D, dtype).reshape(T, D)
    g = normal_bits(seed, f"{tag}/g", T * D, dtype).reshape(T, D)
    fx = normal_bits(seed, f"{tag}/fx", n_frontier * D, dtype).reshape(n_frontier, D)
    fg = normal_bits(seed, f"{tag}/fg", n_frontier * D, dtype).reshape(n_frontier, D)
    bias = normal(seed, f"{tag}/bias", ratio * D).astype(np.float32).reshape(ratio, D)
    return x, g, fx, fg, bias
