"""The C-ABI library without a GPU: it builds, loads, exports every declared symbol, and
rejects bad arguments on the host before any launch."""
import ctypes
import os
import re
import subprocess

import pytest

import deepseek_v4_sparse_gb300 as ds4x
from deepseek_v4_sparse_gb300 import build as ds4x_build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "ds4x.h")


@pytest.fixture(scope="module")
def lib():
    ds4x_build.build()
    return ds4x.load()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(ds4x_\w+)\s*\(", text)))


def test_header_declares_the_abi():
    names = declared_functions()
    for n in ("ds4x_indexer_score", "ds4x_topk", "ds4x_sparse_attn", "ds4x_index_and_attend"):
        assert n in names
    assert set(names) == set(ds4x.EXPORTS)


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name
    out = subprocess.run(["nm", "-D", "--defined-only", ds4x.LIB_PATH], capture_output=True, text=True).stdout
    exported = set(re.findall(r"\bT (ds4x_\w+)", out))
    assert set(declared_functions()) <= exported


def test_status_strings(lib):
    for code in (0, -1, -2, -3, -4, -5):
        assert ds4x.status_string(code).startswith("DS4X_")
    assert "UNKNOWN" in ds4x.status_string(-99)


def _p(v):
    return ctypes.c_void_p(v)


def test_invalid_arguments_rejected_without_launch(lib):
    A = 0x10000  # an aligned, never dereferenced address: validation fails before any use
    # negative sizes
    assert lib.ds4x_indexer_score(_p(A), _p(A), _p(A), _p(A), -1, 64, 128, 10, 4, _p(A), 10, None) == ds4x.ERR_INVALID
    # ld < S
    assert lib.ds4x_indexer_score(_p(A), _p(A), _p(A), _p(A), 4, 64, 128, 10, 4, _p(A), 9, None) == ds4x.ERR_INVALID
    # ratio < 1
    assert lib.ds4x_indexer_score(_p(A), _p(A), _p(A), _p(A), 4, 64, 128, 10, 0, _p(A), 10, None) == ds4x.ERR_INVALID
    # null and misaligned pointers
    assert lib.ds4x_indexer_score(None, _p(A), _p(A), _p(A), 4, 64, 128, 10, 4, _p(A), 10, None) == ds4x.ERR_INVALID
    assert lib.ds4x_indexer_score(_p(A + 2), _p(A), _p(A), _p(A), 4, 64, 128, 10, 4, _p(A), 10, None) == ds4x.ERR_INVALID
    # unsupported head / dim
    assert lib.ds4x_indexer_score(_p(A), _p(A), _p(A), _p(A), 4, 48, 128, 10, 4, _p(A), 10, None) == ds4x.ERR_UNSUPPORTED
    assert lib.ds4x_indexer_score(_p(A), _p(A), _p(A), _p(A), 4, 64, 96, 10, 4, _p(A), 10, None) == ds4x.ERR_UNSUPPORTED
    # top-k: k_top out of range, null output
    assert lib.ds4x_topk(_p(A), 10, _p(A), 4, 10, 4, 0, _p(A), None, None, 0, None) == ds4x.ERR_INVALID
    assert lib.ds4x_topk(_p(A), 10, _p(A), 4, 10, 4, 4096, _p(A), None, None, 0, None) == ds4x.ERR_UNSUPPORTED
    assert lib.ds4x_topk(_p(A), 10, _p(A), 4, 10, 4, 512, None, None, None, 0, None) == ds4x.ERR_INVALID
    # attention: shapes the library has no kernel for, bad dtype
    assert lib.ds4x_sparse_attn(_p(A), _p(A), 1, _p(A), 4, 32, 512, 10, 512, 0.1, _p(A), None, None) == ds4x.ERR_UNSUPPORTED
    assert lib.ds4x_sparse_attn(_p(A), _p(A), 1, _p(A), 4, 64, 256, 10, 512, 0.1, _p(A), None, None) == ds4x.ERR_UNSUPPORTED
    assert lib.ds4x_sparse_attn(_p(A), _p(A), 7, _p(A), 4, 64, 512, 10, 512, 0.1, _p(A), None, None) == ds4x.ERR_INVALID
    # fused entry: workspace missing / too small
    assert lib.ds4x_index_and_attend(_p(A), _p(A), _p(A), _p(A), _p(A), _p(A), 1, 4, 64, 128, 10, 4, 512, 64, 512,
                                     0.1, _p(A), _p(A), None, None, 0, None) == ds4x.ERR_WORKSPACE
    assert lib.ds4x_index_and_attend(_p(A), _p(A), _p(A), _p(A), _p(A), _p(A), 1, 4, 64, 128, 10, 4, 512, 64, 512,
                                     0.1, _p(A), _p(A), None, _p(A), 16, None) == ds4x.ERR_WORKSPACE
    # self-test argument range
    assert lib.ds4x_selftest_bounded_wait(10, None) == ds4x.ERR_INVALID


def test_empty_calls_are_noops(lib):
    A = 0x10000
    assert lib.ds4x_indexer_score(_p(A), _p(A), _p(A), _p(A), 0, 64, 128, 10, 4, _p(A), 10, None) == ds4x.OK
    assert lib.ds4x_topk(_p(A), 10, _p(A), 0, 10, 4, 512, _p(A), None, None, 0, None) == ds4x.OK
    assert lib.ds4x_sparse_attn(_p(A), _p(A), 1, _p(A), 0, 64, 512, 10, 512, 0.1, _p(A), None, None) == ds4x.OK


def _decode(lib, capacity=100, S0=90, n_new=4, pos0=359, n_steps=8, H=64, D=128, ratio=4, k_top=512, dtype=1,
            ws=0, q=0x10000, S_final=None):
    A = 0x10000
    return lib.ds4x_decode(_p(q), _p(A), _p(A), _p(A), _p(A), dtype, capacity, S0, _p(A), _p(A), n_new, pos0,
                           n_steps, H, D, ratio, k_top, 64, 512, 0.1, _p(A), _p(A), _p(A), None, _p(A), ws,
                           S_final, None)


def test_decode_arguments_rejected_without_launch(lib):
    assert _decode(lib, capacity=80) == ds4x.ERR_INVALID          # S0 > capacity
    assert _decode(lib, n_steps=-1) == ds4x.ERR_INVALID
    assert _decode(lib, ratio=0) == ds4x.ERR_INVALID
    assert _decode(lib, pos0=-1) == ds4x.ERR_INVALID
    assert _decode(lib, pos0=2**31 - 4) == ds4x.ERR_INVALID       # positions would overflow int32
    assert _decode(lib, dtype=5) == ds4x.ERR_INVALID
    assert _decode(lib, H=48) == ds4x.ERR_UNSUPPORTED
    assert _decode(lib, k_top=2048) == ds4x.ERR_UNSUPPORTED
    assert _decode(lib, k_top=510) == ds4x.ERR_UNSUPPORTED        # index rows would lose 16-byte alignment
    assert _decode(lib, q=0x10002) == ds4x.ERR_INVALID            # misaligned
    assert _decode(lib, ws=16) == ds4x.ERR_WORKSPACE
    s = ctypes.c_int32(-7)
    assert _decode(lib, n_steps=0, S_final=ctypes.byref(s)) == ds4x.OK   # nothing to do, nothing launched
    assert s.value == 90


def test_workspace_sizes(lib):
    # the fused entry keeps T x S fp32 scores (rounded up to 256 bytes)
    assert ds4x.workspace_bytes(2048, 2048, 512) >= 2048 * 2048 * 4
    assert ds4x.workspace_bytes(0, 2048, 512) == 0
    # one decode token over a long row is split and needs candidate scratch
    assert ds4x.topk_workspace_bytes(1, 262208, 512) > 0
    assert ds4x.topk_workspace_bytes(2048, 16384, 512) == 0
    # the decode loop sizes its workspace for one token at full capacity
    assert ds4x.decode_workspace_bytes(262208, 512) >= ds4x.workspace_bytes(1, 262208, 512) >= 262208 * 4
    assert ds4x.decode_workspace_bytes(0, 512) == 0


def _host(lib, T=64, S=100, H=64, k_top=512, n_chunks=0, dtype=1, buf=0x10000, nbytes=1 << 40, q=0x10000):
    A = 0x10000
    return lib.ds4x_index_and_attend_host(_p(q), _p(A), _p(A), _p(A), _p(A), _p(A), dtype, T, H, 128, S, 4, k_top, 64,
                                          512, 0.1, _p(A), _p(A), None, n_chunks, _p(buf) if buf else None, nbytes,
                                          None)


def test_host_path_arguments_rejected_without_launch(lib):
    assert _host(lib, n_chunks=-1) == ds4x.ERR_INVALID
    assert _host(lib, dtype=5) == ds4x.ERR_INVALID
    assert _host(lib, buf=0) == ds4x.ERR_INVALID                  # no device buffer
    assert _host(lib, buf=0x10004) == ds4x.ERR_INVALID            # device buffer not 16-byte aligned
    assert _host(lib, q=0) == ds4x.ERR_INVALID
    assert _host(lib, H=48) == ds4x.ERR_UNSUPPORTED
    assert _host(lib, k_top=2048) == ds4x.ERR_UNSUPPORTED
    assert _host(lib, nbytes=16) == ds4x.ERR_WORKSPACE
    assert _host(lib, T=0) == ds4x.OK                            # nothing to do, nothing enqueued


def test_host_path_staging_sizes(lib):
    T, H, D, S, k_top, Hq, Dkv = 2048, 64, 128, 2048, 512, 64, 512
    per_token_slot = H * D * 2 + Hq * Dkv * 2 + k_top * 4 + Hq * Dkv * 2       # q, q_attn, indices, out
    shared = S * D * 2 + S * Dkv * 2 + T * (H * 2 + 4 + Hq * 4)                # k, kv; w, positions, lse of all
    for n in (1, 3, 4, 8, 16):
        tc = -(-T // n)
        slots = min(n, 3)
        b = ds4x.index_and_attend_host_bytes(T, H, D, S, k_top, Hq, Dkv, n)
        # the shared parts, the fused workspace of one sub-chunk, up to three slots of one sub-chunk
        low = shared + ds4x.workspace_bytes(tc, S, k_top) + slots * tc * per_token_slot
        assert low <= b <= low + 20 * 256, (n, b - low)
    assert ds4x.index_and_attend_host_bytes(T, H, D, S, k_top, Hq, Dkv, 0) == \
        ds4x.index_and_attend_host_bytes(T, H, D, S, k_top, Hq, Dkv, 4)      # default: sub-chunks of ~512 tokens
    assert ds4x.index_and_attend_host_bytes(0, H, D, S, k_top, Hq, Dkv, 0) == 0
    assert ds4x.index_and_attend_host_bytes(T, H, D, S, k_top, Hq, Dkv, -1) == 0


def _local_attn(lib, T=4, S=10, L=100, lp0=0, window=128, kv_local=0x10000, dtype=1, positions=0x10000, k_top=512):
    A = 0x10000
    return lib.ds4x_local_pooled_attn(_p(A), _p(A), _p(kv_local) if kv_local else None, dtype, _p(A),
                                      _p(positions) if positions else None, T, 64, 512, S, k_top, lp0, L, window, 0.1,
                                      _p(A), None, None)


def _local_fused(lib, T=4, S=10, L=100, lp0=0, window=128, ws=0, nbytes=0):
    A = 0x10000
    return lib.ds4x_index_and_attend_local(_p(A), _p(A), _p(A), _p(A), _p(A), _p(A), _p(A), 1, T, 64, 128, S, 4, 512,
                                           64, 512, lp0, L, window, 0.1, _p(A), _p(A), None,
                                           _p(ws) if ws else None, nbytes, None)


def test_local_arguments_rejected_without_launch(lib):
    assert _local_attn(lib, lp0=-1) == ds4x.ERR_INVALID                 # buffer before position 0
    assert _local_attn(lib, L=-1) == ds4x.ERR_INVALID
    assert _local_attn(lib, window=-1) == ds4x.ERR_INVALID
    assert _local_attn(lib, window=ds4x.MAX_WINDOW + 1) == ds4x.ERR_UNSUPPORTED
    assert _local_attn(lib, kv_local=0) == ds4x.ERR_INVALID             # rows in reach but no buffer
    assert _local_attn(lib, kv_local=0x10008) == ds4x.ERR_INVALID       # misaligned buffer
    assert _local_attn(lib, positions=0) == ds4x.ERR_INVALID            # positions are required
    assert _local_attn(lib, dtype=3) == ds4x.ERR_INVALID
    assert _local_attn(lib, k_top=2048) == ds4x.ERR_UNSUPPORTED
    assert _local_attn(lib, T=0) == ds4x.OK                             # nothing to do
    assert _local_fused(lib, lp0=-5) == ds4x.ERR_INVALID
    assert _local_fused(lib) == ds4x.ERR_WORKSPACE                      # S > 0 needs the score workspace
    assert _local_fused(lib, ws=0x10000, nbytes=16) == ds4x.ERR_WORKSPACE
    A = 0x10000
    assert lib.ds4x_index_and_attend_local_host(
        _p(A), _p(A), _p(A), _p(A), _p(A), _p(A), None, 1, 4, 64, 128, 10, 4, 512, 64, 512, 0, 100, 128, 0.1,
        _p(A), _p(A), None, 0, _p(A), 1 << 40, None) == ds4x.ERR_INVALID    # window rows but no host buffer


def test_local_workspace_and_staging_sizes(lib):
    T, H, D, S, k_top, Hq, Dkv = 2048, 64, 128, 2048, 512, 64, 512
    # a full chunk never splits: the window adds nothing to the workspace
    assert ds4x.workspace_bytes_local(T, S, k_top, 128) == ds4x.workspace_bytes(T, S, k_top)
    assert ds4x.workspace_bytes_local(T, S, k_top, 0) == ds4x.workspace_bytes(T, S, k_top)
    # one token splits its chunks; the window's chunks take part, so the split scratch can grow
    assert ds4x.workspace_bytes_local(1, S, k_top, 128) >= ds4x.workspace_bytes(1, S, k_top)
    assert ds4x.workspace_bytes_local(1, S, k_top, ds4x.MAX_WINDOW + 1) == 0
    L = T + 127
    for n in (1, 4):
        plain = ds4x.index_and_attend_host_bytes(T, H, D, S, k_top, Hq, Dkv, n)
        local = ds4x.index_and_attend_local_host_bytes(T, H, D, S, k_top, Hq, Dkv, L, 128, n)
        # the window's rows are staged once, beside k and kv
        assert L * Dkv * 2 <= local - plain <= L * Dkv * 2 + 256
        assert ds4x.index_and_attend_local_host_bytes(T, H, D, S, k_top, Hq, Dkv, L, 0, n) == plain


def _compress(lib, T=16, D=128, ratio=4, nf=0, x=0x10000, fx=0x10000, rows=0x10000, fxo=0x10000, bias=0x10000,
              dtype=0):
    A = 0x10000
    return lib.ds4x_compress(_p(x) if x else None, _p(A), _p(bias) if bias else None, dtype, T, D, ratio,
                             _p(fx) if fx else None, _p(A), nf, _p(rows) if rows else None, _p(fxo) if fxo else None,
                             _p(A), None)


def test_compress_arguments_rejected_without_launch(lib):
    assert _compress(lib, D=100) == ds4x.ERR_INVALID             # rows of whole 16-byte units
    assert _compress(lib, D=0) == ds4x.ERR_INVALID
    assert _compress(lib, ratio=0) == ds4x.ERR_INVALID
    assert _compress(lib, ratio=ds4x.MAX_RATIO + 1) == ds4x.ERR_INVALID
    assert _compress(lib, nf=4) == ds4x.ERR_INVALID              # a frontier is shorter than a block
    assert _compress(lib, nf=-1) == ds4x.ERR_INVALID
    assert _compress(lib, T=-1) == ds4x.ERR_INVALID
    assert _compress(lib, dtype=9) == ds4x.ERR_INVALID
    assert _compress(lib, x=0) == ds4x.ERR_INVALID               # new positions but no rows
    assert _compress(lib, x=0x10002) == ds4x.ERR_INVALID         # misaligned
    assert _compress(lib, nf=2, fx=0) == ds4x.ERR_INVALID        # a frontier but no buffer
    assert _compress(lib, rows=0) == ds4x.ERR_INVALID            # 4 blocks complete but nowhere to write
    assert _compress(lib, bias=0) == ds4x.ERR_INVALID
    assert _compress(lib, T=6, fxo=0) == ds4x.ERR_INVALID        # 2 positions left over, no frontier out
    assert _compress(lib, T=0) == ds4x.OK                        # nothing to do, nothing launched


def test_plain_c_caller(lib, tmp_path):
    # the header compiles as C11 and a C program links the library and gets the host-side answers
    exe = tmp_path / "c_abi_check"
    pkg = os.path.dirname(ds4x.LIB_PATH)
    subprocess.check_call(["gcc", "-std=c11", "-Wall", "-Wextra", "-Werror", "-I", os.path.join(ROOT, "include"),
                           os.path.join(ROOT, "tests", "c_abi_check.c"), "-o", str(exe), ds4x.LIB_PATH,
                           "-Wl,-rpath," + pkg])
    r = subprocess.run([str(exe)], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, r.stderr
    assert "c abi ok" in r.stdout
