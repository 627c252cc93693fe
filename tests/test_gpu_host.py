"""The fused path on host buffers (copies in, work, copies out, overlapped by sub-chunks of
tokens) against the CPU oracle."""
import numpy as np
import pytest
import torch

import deepseek_v4_sparse_gb300 as ds4x
import oracle
import synth
from parity import check_attn, check_index_sets

pytestmark = pytest.mark.gpu


def _host16(bits: np.ndarray, dtype: str, pin: bool):
    t = torch.from_numpy(np.ascontiguousarray(bits).view(np.int16))
    t = t.view(torch.float16 if dtype == "f16" else torch.bfloat16)
    return t.pin_memory() if pin else t


@pytest.mark.parametrize("n_chunks,pin", [(1, True), (3, True), (4, False), (0, True)])
def test_host_path_matches_oracle(n_chunks, pin):
    # 150 tokens of the 8k recipe: one, three (ragged: 50 tokens each), four (38, 38, 38, 36)
    # sub-chunks, and the default; page-locked and pageable host memory
    wl = synth.WORKLOADS["prefill_8k"]
    T = 150
    inp = synth.make_inputs(wl, seed=9, T=T, pos0=wl.pos0 + 700)
    pos = torch.from_numpy(inp.positions.copy())
    if pin:
        pos = pos.pin_memory()
    idx, out, lse = ds4x.index_and_attend_host(
        _host16(inp.q, "f16", pin), _host16(inp.w, "f16", pin), _host16(inp.k, "f16", pin), pos,
        _host16(inp.q_attn, wl.kv_dtype, pin), _host16(inp.kv, wl.kv_dtype, pin), wl.ratio, wl.k_top,
        S=wl.S, scale=wl.scale, n_chunks=n_chunks)
    torch.cuda.synchronize()
    assert ds4x.device_status() == ds4x.OK
    gidx = idx.numpy()
    ref_scores = oracle.indexer_score(inp.q, inp.w, inp.k, inp.positions, wl.ratio, S=wl.S)
    ref_idx, _ = oracle.topk(ref_scores, inp.positions, wl.S, wl.ratio, wl.k_top)
    check_index_sets(gidx, ref_idx, ref_scores, inp.positions, wl.ratio, wl.S, wl.k_top)
    ref_out, ref_lse = oracle.sparse_attn(inp.q_attn, inp.kv, wl.kv_dtype, gidx, wl.S, wl.scale)
    check_attn(out.view(torch.int16).numpy().view(np.uint16), ref_out, wl.kv_dtype, lse.numpy(), ref_lse)


def test_host_path_back_to_back_calls_share_nothing_stale():
    # two calls on the same stream and device buffer with different inputs: the second call's
    # copies wait for the first call's work, and each returns its own results
    wl = synth.WORKLOADS["prefill_8k"]
    T = 64
    a = synth.make_inputs(wl, seed=21, T=T, pos0=wl.pos0 + 100)
    b = synth.make_inputs(wl, seed=22, T=T, pos0=wl.pos0 + 1900)
    need = ds4x.index_and_attend_host_bytes(T, wl.H, wl.D, wl.S, wl.k_top, wl.Hq, wl.Dkv, 2)
    buf = torch.empty((need,), dtype=torch.uint8, device="cuda")
    res = []
    for inp in (a, b):
        res.append(ds4x.index_and_attend_host(
            _host16(inp.q, "f16", True), _host16(inp.w, "f16", True), _host16(inp.k, "f16", True),
            torch.from_numpy(inp.positions.copy()).pin_memory(), _host16(inp.q_attn, wl.kv_dtype, True),
            _host16(inp.kv, wl.kv_dtype, True), wl.ratio, wl.k_top, S=wl.S, scale=wl.scale, n_chunks=2,
            device_buffer=buf))
    torch.cuda.synchronize()
    for inp, (idx, out, lse) in zip((a, b), res):
        ref_scores = oracle.indexer_score(inp.q, inp.w, inp.k, inp.positions, wl.ratio, S=wl.S)
        ref_idx, _ = oracle.topk(ref_scores, inp.positions, wl.S, wl.ratio, wl.k_top)
        check_index_sets(idx.numpy(), ref_idx, ref_scores, inp.positions, wl.ratio, wl.S, wl.k_top)
        ref_out, ref_lse = oracle.sparse_attn(inp.q_attn, inp.kv, wl.kv_dtype, idx.numpy(), wl.S, wl.scale)
        check_attn(out.view(torch.int16).numpy().view(np.uint16), ref_out, wl.kv_dtype, lse.numpy(), ref_lse)


def test_host_path_one_token_sub_chunks_long_row():
    # two decode-recipe tokens over 32768 rows, one per sub-chunk: each sub-chunk is one token
    # over a long row (the top-k's one-token mode with the scorer's bounds), the second reusing the
    # device buffer the first one used
    wl = synth.WORKLOADS["decode_1m"]
    S = 32768
    inp = synth.make_inputs(wl, seed=4, T=2, S=S, pos0=wl.ratio * S + 5, rows=S)
    idx, out, lse = ds4x.index_and_attend_host(
        _host16(inp.q, "f16", True), _host16(inp.w, "f16", True), _host16(inp.k, "f16", True),
        torch.from_numpy(inp.positions.copy()).pin_memory(), _host16(inp.q_attn, wl.kv_dtype, True),
        _host16(inp.kv, wl.kv_dtype, True), wl.ratio, wl.k_top, S=S, scale=wl.scale, n_chunks=2)
    torch.cuda.synchronize()
    assert ds4x.device_status() == ds4x.OK
    gidx = idx.numpy()
    ref_scores = oracle.indexer_score(inp.q, inp.w, inp.k, inp.positions, wl.ratio, S=S)
    ref_idx, _ = oracle.topk(ref_scores, inp.positions, S, wl.ratio, wl.k_top)
    check_index_sets(gidx, ref_idx, ref_scores, inp.positions, wl.ratio, S, wl.k_top)
    ref_out, ref_lse = oracle.sparse_attn(inp.q_attn, inp.kv, wl.kv_dtype, gidx, S, wl.scale)
    check_attn(out.view(torch.int16).numpy().view(np.uint16), ref_out, wl.kv_dtype, lse.numpy(), ref_lse)
