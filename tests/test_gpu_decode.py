"""The decode loop (one token per step, rows appended as positions complete them) and the split
attention it runs on (a token's chunks spread over CTAs and merged by their softmax statistics),
against the CPU oracle."""
import dataclasses

import numpy as np
import pytest
import torch

import deepseek_v4_sparse_gb300 as ds4x
import oracle
import synth
from parity import check_attn, check_index_sets, dev16, host16, to_device

pytestmark = pytest.mark.gpu


def _decode_case(S0, extra, n_steps, seed=0):
    wl = synth.WORKLOADS["decode_1m"]
    pos0 = wl.ratio * S0 - 1                      # step 0 sees exactly the S0 resident rows
    inp = synth.make_inputs(wl, seed=seed, T=n_steps, S=S0, pos0=pos0, rows=S0 + extra)
    k0, kv0 = inp.k.copy(), inp.kv.copy()
    k0[S0:] = 0
    kv0[S0:] = 0
    return wl, inp, pos0, k0, kv0, inp.k[S0:].copy(), inp.kv[S0:].copy()


def _run_and_check(S0, extra, n_steps, steps_to_check=None):
    wl, inp, pos0, k0, kv0, k_new, kv_new = _decode_case(S0, extra, n_steps)
    d_k, d_kv = dev16(k0, "f16"), dev16(kv0, wl.kv_dtype)
    idx, out, lse, pos, S_final = ds4x.decode(
        dev16(inp.q, "f16"), dev16(inp.w, "f16"), dev16(inp.q_attn, wl.kv_dtype), d_k, d_kv, S0, pos0, wl.ratio,
        k_new=dev16(k_new, "f16"), kv_new=dev16(kv_new, wl.kv_dtype), k_top=wl.k_top, scale=wl.scale)
    torch.cuda.synchronize()
    assert ds4x.device_status() == ds4x.OK
    ridx, rout, rlse, rpos, rS, rk, rkv = oracle.decode(inp.q, inp.w, inp.q_attn, k0, kv0, wl.kv_dtype, S0, pos0,
                                                        wl.ratio, k_new, kv_new, wl.k_top, wl.scale)
    assert np.array_equal(pos.cpu().numpy(), rpos)
    assert S_final == int(rS[-1])
    # the appended rows: bit-exact copies of the staged rows, at rows S0.. in order
    assert np.array_equal(host16(d_k), rk) and np.array_equal(host16(d_kv), rkv)
    gidx, gout, glse = idx.cpu().numpy(), host16(out), lse.cpu().numpy()
    for i in (range(n_steps) if steps_to_check is None else steps_to_check):
        S = int(rS[i])
        ref_scores = oracle.indexer_score(inp.q[i:i + 1], inp.w[i:i + 1], rk, rpos[i:i + 1], wl.ratio, S=S)
        check_index_sets(gidx[i:i + 1], ridx[i:i + 1], ref_scores, rpos[i:i + 1], wl.ratio, S, wl.k_top)
        # attention of the step on the GPU's own selection (selection and attention errors apart)
        ref_out, ref_lse = oracle.sparse_attn(inp.q_attn[i:i + 1], rkv, wl.kv_dtype, gidx[i:i + 1], S, wl.scale)
        check_attn(gout[i:i + 1], ref_out, wl.kv_dtype, glse[i:i + 1], ref_lse)
    return rS


def test_decode_downscaled_vs_oracle():
    # the 1M-context decode recipe on 4096 resident rows: 24 steps, a row appended every 4th
    rS = _run_and_check(S0=4096, extra=16, n_steps=24)
    assert list(rS[:4]) == [4096] * 4 and rS[4] == 4097 and rS[-1] == 4101


def test_decode_staged_rows_run_out():
    # 2 staged rows for 5 needed: later steps see the rows that exist (n_vis = min(S, ...))
    rS = _run_and_check(S0=2048, extra=2, n_steps=20)
    assert rS[-1] == 2050


def test_decode_full_size_first_steps():
    # the 1M-context decode itself (262144 resident rows, capacity 262208): the first 6 steps,
    # including the first append, compared with the oracle in full
    rS = _run_and_check(S0=262144, extra=64, n_steps=6)
    assert list(rS) == [262144] * 4 + [262145] * 2


def test_decode_full_size_whole_call_sampled():
    # the 1M-context decode as the benchmark runs it: 256 steps over 262144 resident rows with 64
    # staged rows.  Rows per step follow the append rule (the oracle's decode loop is pinned to
    # the same closed form); steps on both sides of three appends and the call's last step are
    # compared with the oracle on the rows present at that step.
    S0, extra, n_steps = 262144, 64, 256
    wl, inp, pos0, k0, kv0, k_new, kv_new = _decode_case(S0, extra, n_steps, seed=5)
    d_k, d_kv = dev16(k0, "f16"), dev16(kv0, wl.kv_dtype)
    idx, out, lse, pos, S_final = ds4x.decode(
        dev16(inp.q, "f16"), dev16(inp.w, "f16"), dev16(inp.q_attn, wl.kv_dtype), d_k, d_kv, S0, pos0, wl.ratio,
        k_new=dev16(k_new, "f16"), kv_new=dev16(kv_new, wl.kv_dtype), k_top=wl.k_top, scale=wl.scale)
    torch.cuda.synchronize()
    assert ds4x.device_status() == ds4x.OK
    cap = k0.shape[0]
    rpos = pos0 + np.arange(n_steps, dtype=np.int64)
    rS = np.minimum(np.minimum(S0 + extra, cap), np.maximum(S0, (rpos + 1) // wl.ratio))
    assert np.array_equal(pos.cpu().numpy(), rpos.astype(np.int32)) and S_final == int(rS[-1]) == S0 + 63
    # the rows after the call: the staged rows appended in order, the rest untouched
    n_app = int(rS[-1]) - S0
    rk, rkv = k0.copy(), kv0.copy()
    rk[S0:S0 + n_app], rkv[S0:S0 + n_app] = k_new[:n_app], kv_new[:n_app]
    assert np.array_equal(host16(d_k), rk) and np.array_equal(host16(d_kv), rkv)
    gidx, gout, glse = idx.cpu().numpy(), host16(out), lse.cpu().numpy()
    steps = [0, 3, 4, 127, 128, 255]
    assert [int(rS[i]) for i in steps] == [262144, 262144, 262145, 262175, 262176, 262207]
    for i in steps:
        S = int(rS[i])
        p_i = rpos[i:i + 1].astype(np.int32)
        ref_scores = oracle.indexer_score(inp.q[i:i + 1], inp.w[i:i + 1], rk, p_i, wl.ratio, S=S)
        ref_idx, _ = oracle.topk(ref_scores, p_i, S, wl.ratio, wl.k_top)
        check_index_sets(gidx[i:i + 1], ref_idx, ref_scores, p_i, wl.ratio, S, wl.k_top)
        ref_out, ref_lse = oracle.sparse_attn(inp.q_attn[i:i + 1], rkv, wl.kv_dtype, gidx[i:i + 1], S, wl.scale)
        check_attn(gout[i:i + 1], ref_out, wl.kv_dtype, glse[i:i + 1], ref_lse)


@pytest.mark.parametrize("T,k_top,kv_dtype", [(1, 512, "bf16"), (16, 512, "bf16"), (50, 512, "bf16"), (76, 512, "bf16"),
                                               (1, 300, "bf16"), (1, 512, "f16"), (16, 512, "f16")])
def test_split_attention_matches_oracle(T, k_top, kv_dtype):
    # few tokens: the fused path splits each token's attention over CTAs (uneven splits at
    # T = 50, a partial last chunk at k_top = 300) and merges the parts, which are stored in the
    # kv dtype (both dtypes)
    wl = dataclasses.replace(synth.WORKLOADS["prefill_8k"], kv_dtype=kv_dtype)
    inp = synth.make_inputs(wl, seed=3, T=T, pos0=wl.pos0 + wl.T - T)
    d = to_device(inp)
    assert ds4x.workspace_bytes(T, wl.S, k_top) >= T * wl.S * 4
    fidx, fout, flse = ds4x.index_and_attend(d["q"], d["w"], d["k"], d["positions"], d["q_attn"], d["kv"],
                                             wl.ratio, k_top, S=wl.S, scale=wl.scale)
    # the standalone attention (one CTA per token) on the same selection
    sout, slse = ds4x.sparse_attn(d["q_attn"], d["kv"], fidx, S=wl.S, scale=wl.scale)
    torch.cuda.synchronize()
    assert ds4x.device_status() == ds4x.OK
    gidx = fidx.cpu().numpy()
    ref_out, ref_lse = oracle.sparse_attn(inp.q_attn, inp.kv, wl.kv_dtype, gidx, wl.S, wl.scale)
    check_attn(host16(fout), ref_out, wl.kv_dtype, flse.cpu().numpy(), ref_lse)
    check_attn(host16(sout), ref_out, wl.kv_dtype, slse.cpu().numpy(), ref_lse)
    ref_scores = oracle.indexer_score(inp.q, inp.w, inp.k, inp.positions, wl.ratio, S=wl.S)
    ref_idx, _ = oracle.topk(ref_scores, inp.positions, wl.S, wl.ratio, k_top)
    check_index_sets(gidx, ref_idx, ref_scores, inp.positions, wl.ratio, wl.S, k_top)


# --------------------------------------------------- the decode loop with the raw window
@pytest.mark.parametrize("S0,extra,n_steps,window", [(4096, 16, 24, 128), (2048, 4, 12, 100), (262144, 64, 6, 128)])
def test_decode_local_vs_oracle(S0, extra, n_steps, window):
    # each step attends to its selected pooled rows and the raw rows of its last `window` positions;
    # the raw history below pos0 is the caller's, the steps' own raw rows are written by the call
    wl, inp, pos0, k0, kv0, k_new, kv_new = _decode_case(S0, extra, n_steps, seed=3)
    raw_cap = pos0 + n_steps + 5
    hist = synth.local_rows(3, f"decode_raw_{S0}", window, wl.Dkv, "normal", wl.kv_dtype)
    kv_raw = np.zeros((raw_cap, wl.Dkv), dtype=np.uint16)
    kv_raw[pos0 - window:pos0] = hist                 # the window's history
    kv_raw_new = synth.local_rows(4, f"decode_raw_new_{S0}", n_steps, wl.Dkv, "normal", wl.kv_dtype)
    d_k, d_kv, d_raw = dev16(k0, "f16"), dev16(kv0, wl.kv_dtype), dev16(kv_raw, wl.kv_dtype)
    idx, out, lse, pos, S_final = ds4x.decode_local(
        dev16(inp.q, "f16"), dev16(inp.w, "f16"), dev16(inp.q_attn, wl.kv_dtype), d_k, d_kv, S0, pos0, wl.ratio,
        d_raw, dev16(kv_raw_new, wl.kv_dtype), window, k_new=dev16(k_new, "f16"), kv_new=dev16(kv_new, wl.kv_dtype),
        k_top=wl.k_top, scale=wl.scale)
    torch.cuda.synchronize()
    assert ds4x.device_status() == ds4x.OK
    ridx, rout, rlse, rpos, rS, rk, rkv, rraw = oracle.decode_local(
        inp.q, inp.w, inp.q_attn, k0, kv0, wl.kv_dtype, S0, pos0, wl.ratio, k_new, kv_new, wl.k_top, wl.scale,
        kv_raw, kv_raw_new, window)
    assert np.array_equal(pos.cpu().numpy(), rpos) and S_final == int(rS[-1])
    assert np.array_equal(host16(d_raw), rraw)                   # the steps' raw rows, in place
    gidx, gout, glse = idx.cpu().numpy(), host16(out), lse.cpu().numpy()
    for i in range(n_steps):
        S = int(rS[i])
        ref_scores = oracle.indexer_score(inp.q[i:i + 1], inp.w[i:i + 1], rk, rpos[i:i + 1], wl.ratio, S=S)
        check_index_sets(gidx[i:i + 1], ridx[i:i + 1], ref_scores, rpos[i:i + 1], wl.ratio, S, wl.k_top)
        ref_out, ref_lse = oracle.local_pooled_attn(inp.q_attn[i:i + 1], rkv, rraw, wl.kv_dtype, gidx[i:i + 1],
                                                    rpos[i:i + 1], S, 0, window, wl.scale)
        check_attn(gout[i:i + 1], ref_out, wl.kv_dtype, glse[i:i + 1], ref_lse)
