"""Local-plus-pooled attention (the raw sliding window joined to the selected pooled rows in one
softmax) through the C ABI, against the CPU oracle on the same seeded inputs."""
import numpy as np
import pytest
import torch

import deepseek_v4_sparse_gb300 as ds4x
import oracle
import synth
from parity import check_attn, check_index_sets, dev16, host16, to_device, union_rows_bound, window_positions

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from deepseek_v4_sparse_gb300 import build
    build.build()
    ds4x.load()
    yield
    torch.cuda.synchronize()
    assert ds4x.device_status() == ds4x.OK, "a bounded device wait timed out during the tests"


def _attn_case(tag, positions, S, L, local_pos0, seed=3, dtype="bf16", kind="normal"):
    inp = synth.custom_inputs(seed, tag, len(positions), 64, 128, S, 64, 512, kind, dtype, positions)
    kvl = synth.local_rows(seed, tag, L, 512, kind, dtype)
    return inp, kvl


def _gpu_local(inp, kvl, idx, local_pos0, window, S, dtype="bf16"):
    d = to_device(inp)
    out, lse = ds4x.local_pooled_attn(d["q_attn"], d["kv"], dev16(kvl, dtype) if kvl.shape[0] else None,
                                      torch.from_numpy(idx).cuda(), d["positions"], local_pos0, window, S=S)
    torch.cuda.synchronize()
    assert ds4x.device_status() == ds4x.OK
    return host16(out), lse.cpu().numpy()


def test_window_off_is_the_pooled_kernel_bit_for_bit():
    rng = np.random.default_rng(1)
    S, T, L = 700, 12, 300
    pos = np.arange(T) * 50 + 2000
    inp, kvl = _attn_case("local_off", pos, S, L, 1900)
    idx = np.sort(np.stack([rng.choice(S, 512, replace=False) for _ in range(T)]), axis=1).astype(np.int32)
    idx[3, 100:] = -1
    d = to_device(inp)
    ref_out, ref_lse = ds4x.sparse_attn(d["q_attn"], d["kv"], torch.from_numpy(idx).cuda(), S=S)
    ref_out, ref_lse = host16(ref_out), ref_lse.cpu().numpy()
    for window, rows, lp0 in ((0, L, 1900), (128, 0, 1900), (128, L, 10**6)):
        out, lse = _gpu_local(inp, kvl[:rows], idx, lp0, window, S)
        assert np.array_equal(out, ref_out) and np.array_equal(lse, ref_lse), (window, rows, lp0)


@pytest.mark.parametrize("window", [1, 64, 100, 128, 1024])
def test_window_rows_only(window):
    # no pooled row: tokens at the sequence start (fewer than `window` positions exist), inside the
    # buffer, with the window reaching before the buffer, and past the buffer's end
    L, lp0 = 900, 40
    pos = np.array([0, 5, 39, 40, 41, 63, 64, 130, 500, 938, 939, 1000, 1500, 2000, -3], dtype=np.int64)
    inp, kvl = _attn_case(f"local_only_{window}", pos, 16, L, lp0)
    idx = np.full((len(pos), 512), -1, dtype=np.int32)
    out, lse = _gpu_local(inp, kvl, idx, lp0, window, 16)
    ref_out, ref_lse = oracle.local_pooled_attn(inp.q_attn, inp.kv, kvl, "bf16", idx, inp.positions, 16, lp0,
                                                window, 1 / np.sqrt(512))
    check_attn(out, ref_out, "bf16", lse, ref_lse,
               extra=union_rows_bound(inp.kv, idx, 16, kvl, inp.positions, lp0, window, ref_out, "bf16"))
    for t, p in enumerate(pos):
        rows = window_positions(int(p), window, lp0, L)
        if not rows:
            assert np.all(out[t] == 0) and np.all(np.isneginf(lse[t])), t
        elif len(rows) == 1:
            assert all(np.array_equal(out[t, h], kvl[rows[0] - lp0]) for h in range(64)), t


@pytest.mark.parametrize("dtype", ["bf16", "f16"])
def test_pooled_and_window_rows(dtype):
    # random selections (some padded, some out of range) plus a 128-position window
    rng = np.random.default_rng(2)
    S, L, lp0, W = 1500, 700, 5873, 128
    pos = np.concatenate([[5873, 5880, 6000], 6000 + rng.integers(0, 572, 37)]).astype(np.int64)
    inp, kvl = _attn_case(f"local_union_{dtype}", pos, S, L, lp0, dtype=dtype)
    idx = np.sort(np.stack([rng.choice(S, 512, replace=False) for _ in range(len(pos))]), axis=1).astype(np.int32)
    idx[1, 7:] = -1
    idx[2, ::5] = S + 9
    out, lse = _gpu_local(inp, kvl, idx, lp0, W, S, dtype)
    ref_out, ref_lse = oracle.local_pooled_attn(inp.q_attn, inp.kv, kvl, dtype, idx, inp.positions, S, lp0, W,
                                                1 / np.sqrt(512))
    check_attn(out, ref_out, dtype, lse, ref_lse,
               extra=union_rows_bound(inp.kv, idx, S, kvl, inp.positions, lp0, W, ref_out, dtype))


def _local_inputs(name, T, seed=0, at_end=True):
    wl = synth.WORKLOADS[name]
    pos0 = wl.pos0 + wl.T - T if at_end else wl.pos0
    return wl, synth.make_inputs(wl, seed=seed, T=T, pos0=pos0)


def test_fused_local_exact_integer_indices():
    # the integer workload with a window: indices bit-exact, attention within tolerance
    base = synth.WORKLOADS["tiny_exact"]
    T, W = 200, 128
    inp = synth.make_inputs(base, seed=0, T=T)
    lp0 = int(inp.positions[0]) - W + 1
    kvl = synth.local_rows(0, "tiny_exact_local", T + W - 1, 512, "int", "f16")
    d = to_device(inp)
    fidx, fout, flse = ds4x.index_and_attend_local(d["q"], d["w"], d["k"], d["positions"], d["q_attn"], d["kv"],
                                                   dev16(kvl, "f16"), base.ratio, lp0, W, base.k_top, S=base.S)
    torch.cuda.synchronize()
    assert ds4x.device_status() == ds4x.OK
    ref_idx, ref_out, ref_lse = oracle.index_and_attend_local(inp.q, inp.w, inp.k, inp.positions, inp.q_attn, inp.kv,
                                                              kvl, "f16", base.S, base.ratio, base.k_top, lp0, W,
                                                              base.scale)
    assert np.array_equal(fidx.cpu().numpy(), ref_idx)
    check_attn(host16(fout), ref_out, "f16", flse.cpu().numpy(), ref_lse)


@pytest.mark.parametrize("T", [1, 3, 160])
def test_fused_local_normal(T):
    # T = 1 and 3 take the split mode (a token's pooled and window chunks over several CTAs, merged)
    wl, inp = _local_inputs("prefill_8k_local128", T, seed=1)
    d = to_device(inp)
    kvl = dev16(inp.kv_local, wl.kv_dtype)
    fidx, fout, flse = ds4x.index_and_attend_local(d["q"], d["w"], d["k"], d["positions"], d["q_attn"], d["kv"], kvl,
                                                   wl.ratio, inp.local_pos0, wl.window, wl.k_top, S=wl.S)
    torch.cuda.synchronize()
    assert ds4x.device_status() == ds4x.OK
    gidx = fidx.cpu().numpy()
    ref_scores = oracle.indexer_score(inp.q, inp.w, inp.k, inp.positions, wl.ratio, S=wl.S)
    ref_idx, _ = oracle.topk(ref_scores, inp.positions, wl.S, wl.ratio, wl.k_top)
    check_index_sets(gidx, ref_idx, ref_scores, inp.positions, wl.ratio, wl.S, wl.k_top)
    ref_out, ref_lse = oracle.local_pooled_attn(inp.q_attn, inp.kv, inp.kv_local, wl.kv_dtype, gidx, inp.positions,
                                                wl.S, inp.local_pos0, wl.window, wl.scale)
    check_attn(host16(fout), ref_out, wl.kv_dtype, flse.cpu().numpy(), ref_lse)


def test_fused_local_full_size_sampled():
    # the benchmark's workload and launch shape; sampled tokens against the oracle
    wl = synth.WORKLOADS["prefill_8k_local128"]
    inp = synth.make_inputs(wl, seed=0)
    d = to_device(inp)
    fidx, fout, flse = ds4x.index_and_attend_local(d["q"], d["w"], d["k"], d["positions"], d["q_attn"], d["kv"],
                                                   dev16(inp.kv_local, wl.kv_dtype), wl.ratio, inp.local_pos0,
                                                   wl.window, wl.k_top, S=wl.S)
    torch.cuda.synchronize()
    assert ds4x.device_status() == ds4x.OK
    sample = np.array([0, 1, 127, 128, 777, 1500, wl.T - 1])
    gidx = fidx.cpu().numpy()[sample]
    q, w, pos = inp.q[sample], inp.w[sample], inp.positions[sample]
    ref_scores = oracle.indexer_score(q, w, inp.k, pos, wl.ratio, S=wl.S)
    ref_idx, _ = oracle.topk(ref_scores, pos, wl.S, wl.ratio, wl.k_top)
    check_index_sets(gidx, ref_idx, ref_scores, pos, wl.ratio, wl.S, wl.k_top)
    ref_out, ref_lse = oracle.local_pooled_attn(inp.q_attn[sample], inp.kv, inp.kv_local, wl.kv_dtype, gidx, pos,
                                                wl.S, inp.local_pos0, wl.window, wl.scale)
    check_attn(host16(fout)[sample], ref_out, wl.kv_dtype, flse.cpu().numpy()[sample], ref_lse)


@pytest.mark.parametrize("n_chunks", [1, 3])
def test_local_host_entry(n_chunks):
    wl, inp = _local_inputs("prefill_8k_local128", 96, seed=2)
    kvt = torch.bfloat16

    def h16(a, dt):
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16).copy()).view(dt).pin_memory()

    h = dict(q=h16(inp.q, torch.float16), w=h16(inp.w, torch.float16), k=h16(inp.k, torch.float16),
             qa=h16(inp.q_attn, kvt), kv=h16(inp.kv, kvt), kvl=h16(inp.kv_local, kvt),
             pos=torch.from_numpy(inp.positions.copy()).pin_memory())
    idx, out, lse = ds4x.index_and_attend_local_host(h["q"], h["w"], h["k"], h["pos"], h["qa"], h["kv"], h["kvl"],
                                                     wl.ratio, inp.local_pos0, wl.window, wl.k_top, S=wl.S,
                                                     n_chunks=n_chunks)
    torch.cuda.synchronize()
    assert ds4x.device_status() == ds4x.OK
    gidx = idx.numpy()
    ref_scores = oracle.indexer_score(inp.q, inp.w, inp.k, inp.positions, wl.ratio, S=wl.S)
    ref_idx, _ = oracle.topk(ref_scores, inp.positions, wl.S, wl.ratio, wl.k_top)
    check_index_sets(gidx, ref_idx, ref_scores, inp.positions, wl.ratio, wl.S, wl.k_top)
    ref_out, ref_lse = oracle.local_pooled_attn(inp.q_attn, inp.kv, inp.kv_local, wl.kv_dtype, gidx, inp.positions,
                                                wl.S, inp.local_pos0, wl.window, wl.scale)
    check_attn(out.view(torch.int16).numpy().view(np.uint16), ref_out, wl.kv_dtype, lse.numpy(), ref_lse)
