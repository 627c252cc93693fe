"""CUDA path (through the C ABI) against the CPU oracle on the same seeded inputs."""
import numpy as np
import pytest
import torch

import deepseek_v4_sparse_gb300 as ds4x
import oracle
import synth
from parity import (check_attn, check_index_sets, check_scores, dev16, few_rows_bound, host16, n_vis,
                    to_device)

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


def run_all(inp, S=None):
    d = to_device(inp)
    wl = inp.wl
    S = wl.S if S is None else S
    scores = ds4x.indexer_score(d["q"], d["w"], d["k"], d["positions"], wl.ratio, S=S)
    idx, cnt = ds4x.topk(scores, d["positions"], S, wl.ratio, wl.k_top)
    out, lse = ds4x.sparse_attn(d["q_attn"], d["kv"], idx, S=S, scale=wl.scale)
    fidx, fout, flse = ds4x.index_and_attend(d["q"], d["w"], d["k"], d["positions"], d["q_attn"], d["kv"],
                                             wl.ratio, wl.k_top, S=S, scale=wl.scale)
    torch.cuda.synchronize()
    assert ds4x.device_status() == ds4x.OK
    return dict(scores=scores.cpu().numpy(), idx=idx.cpu().numpy(), cnt=cnt.cpu().numpy(),
                out=host16(out), lse=lse.cpu().numpy(), fidx=fidx.cpu().numpy(), fout=host16(fout),
                flse=flse.cpu().numpy())


# ------------------------------------------------------------------------ bounded waits
def test_bounded_wait_reports_timeout():
    ds4x.device_status(clear=True)
    ds4x.selftest_bounded_wait(2_000_000)  # 2 ms, nothing ever completes the barrier
    assert ds4x.device_status(clear=True) == ds4x.ERR_TIMEOUT
    assert ds4x.device_status(clear=True) == ds4x.OK


# ---------------------------------------------------------------- exact-integer config
def test_tiny_exact_bit_exact():
    wl = synth.WORKLOADS["tiny_exact"]
    inp = synth.make_inputs(wl, seed=0)
    g = run_all(inp)
    ref_scores = oracle.indexer_score(inp.q, inp.w, inp.k, inp.positions, wl.ratio, S=wl.S)
    check_scores(g["scores"], ref_scores, inp.positions, wl.ratio, wl.S, exact=True)
    ref_idx, ref_cnt = oracle.topk(ref_scores, inp.positions, wl.S, wl.ratio, wl.k_top)
    assert np.array_equal(g["idx"], ref_idx), "indices differ from the oracle"
    assert np.array_equal(g["cnt"], ref_cnt)
    assert np.array_equal(g["fidx"], ref_idx), "fused-path indices differ from the oracle"
    ref_out, ref_lse = oracle.sparse_attn(inp.q_attn, inp.kv, "f16", ref_idx, wl.S, wl.scale)
    check_attn(g["out"], ref_out, "f16", g["lse"], ref_lse)
    check_attn(g["fout"], ref_out, "f16", g["flse"], ref_lse)


# ---------------------------------------------------------- N(0,1) configs, down-scaled
@pytest.mark.parametrize("name,T", [("prefill_8k", 160), ("prefill_32k", 40)])
def test_normal_downscaled(name, T):
    wl = synth.WORKLOADS[name]
    # the last T tokens of the chunk (they see the most rows)
    inp = synth.make_inputs(wl, seed=0, T=T, pos0=wl.pos0 + wl.T - T)
    g = run_all(inp)
    ref_scores = oracle.indexer_score(inp.q, inp.w, inp.k, inp.positions, wl.ratio, S=wl.S)
    check_scores(g["scores"], ref_scores, inp.positions, wl.ratio, wl.S, exact=False)
    # same fp32 scores in, same decision out: top-k of the GPU's scores is bit-exact
    idx_on_gpu_scores, cnt = oracle.topk(g["scores"], inp.positions, wl.S, wl.ratio, wl.k_top)
    assert np.array_equal(g["idx"], idx_on_gpu_scores)
    assert np.array_equal(g["cnt"], cnt)
    ref_idx, _ = oracle.topk(ref_scores, inp.positions, wl.S, wl.ratio, wl.k_top)
    check_index_sets(g["fidx"], ref_idx, ref_scores, inp.positions, wl.ratio, wl.S, wl.k_top)
    ref_out, ref_lse = oracle.sparse_attn(inp.q_attn, inp.kv, wl.kv_dtype, g["idx"], wl.S, wl.scale)
    check_attn(g["out"], ref_out, wl.kv_dtype, g["lse"], ref_lse)
    ref_fout, ref_flse = oracle.sparse_attn(inp.q_attn, inp.kv, wl.kv_dtype, g["fidx"], wl.S, wl.scale)
    check_attn(g["fout"], ref_fout, wl.kv_dtype, g["flse"], ref_flse)


# ----------------------------------------------------------------------------- edge cases
def _edge_inputs(tag, positions, S, kind="normal", kv_dtype="bf16", H=64, D=128, w_kind="pos", seed=1):
    T = len(positions)
    return synth.custom_inputs(seed, tag, T, H, D, S, 64, 512, kind, kv_dtype, np.array(positions), w_kind)


@pytest.mark.parametrize("ratio", [1, 4, 128])
def test_visibility_edges(ratio):
    # n_vis in {0, 1, 2, 511, 512, 513, ...}; S not a multiple of 128; T not a multiple of
    # the scorer's token group; a negative position sees no row
    S = 1000
    nv = [0, 1, 2, 511, 512, 513, 700, 999, 1000, 1000, 37, 128, 129]
    positions = [n * ratio - 1 for n in nv]
    assert [n_vis(p, ratio, S) for p in positions] == nv
    raw = _edge_inputs(f"edge_r{ratio}", positions, S)
    wl = synth.Workload(raw.wl.name, T=len(nv), H=64, D=128, S=S, ratio=ratio, pos0=0, kind="normal",
                        kv_dtype="bf16")
    inp = synth.Inputs(wl, raw.q, raw.w, raw.k, raw.positions, raw.q_attn, raw.kv)
    g = run_all(inp)
    ref_scores = oracle.indexer_score(inp.q, inp.w, inp.k, inp.positions, ratio, S=S)
    check_scores(g["scores"], ref_scores, inp.positions, ratio, S, exact=False)
    idx_ref_on_gpu, cnt_ref = oracle.topk(g["scores"], inp.positions, S, ratio, wl.k_top)
    assert np.array_equal(g["idx"], idx_ref_on_gpu) and np.array_equal(g["cnt"], cnt_ref)
    ref_idx, _ = oracle.topk(ref_scores, inp.positions, S, ratio, wl.k_top)
    check_index_sets(g["fidx"], ref_idx, ref_scores, inp.positions, ratio, S, wl.k_top)
    # tokens here see as few as 1 row: the few-row rounding bound applies on top of the spec's
    ref_out, ref_lse = oracle.sparse_attn(inp.q_attn, inp.kv, "bf16", g["idx"], S, wl.scale)
    check_attn(g["out"], ref_out, "bf16", g["lse"], ref_lse,
               extra=few_rows_bound(inp.kv, g["idx"], ref_out, "bf16", S))
    ref_fout, ref_flse = oracle.sparse_attn(inp.q_attn, inp.kv, "bf16", g["fidx"], S, wl.scale)
    check_attn(g["fout"], ref_fout, "bf16", g["flse"], ref_flse,
               extra=few_rows_bound(inp.kv, g["fidx"], ref_fout, "bf16", S))


@pytest.mark.parametrize("H,D", [(16, 64), (16, 128), (32, 64), (32, 128), (64, 64), (64, 128), (128, 64),
                                 (128, 128)])
def test_score_shapes_both_tile_widths(H, D):
    # every supported indexer shape, bit-exact on integer inputs, at token counts that take the
    # narrow tile (all tokens in max(64, H) columns: one token for H >= 64, up to 4 for H = 16)
    # and the wide one (four 64-head tokens per tile), with a ragged row count
    S, ratio = 1000, 1
    narrow_tokens = max(64, H) // H
    for T in sorted({1, narrow_tokens, narrow_tokens + 1, 9}):
        positions = [S - 1 - 37 * t for t in range(T)]          # n_vis from 1000 down
        raw = _edge_inputs(f"shape_{H}_{D}_{T}", positions, S, kind="int", kv_dtype="f16", H=H, D=D,
                           w_kind="pow2")
        d = to_device(raw)
        scores = ds4x.indexer_score(d["q"], d["w"], d["k"], d["positions"], ratio, S=S)
        torch.cuda.synchronize()
        assert ds4x.device_status() == ds4x.OK
        ref = oracle.indexer_score(raw.q, raw.w, raw.k, raw.positions, ratio, S=S)
        check_scores(scores.cpu().numpy(), ref, raw.positions, ratio, S, exact=True)


def test_score_work_split_sparse_tiles():
    # far fewer scored tiles than CTAs, after leading token groups that see nothing (their rows
    # are written -inf by whichever CTA holds them), with groups of differing widths in between
    S, ratio = 3000, 4
    nv = [0] * 21 + [5, 130, 0, 700, 1, 2999, 3000, 64, 0, 256, 257]
    positions = [n * ratio - 1 if n > 0 else -1 for n in nv]
    raw = _edge_inputs("score_split", positions, S, kind="int", kv_dtype="f16", w_kind="pow2")
    d = to_device(raw)
    scores = ds4x.indexer_score(d["q"], d["w"], d["k"], d["positions"], ratio, S=S)
    torch.cuda.synchronize()
    assert ds4x.device_status() == ds4x.OK
    ref = oracle.indexer_score(raw.q, raw.w, raw.k, raw.positions, ratio, S=S)
    check_scores(scores.cpu().numpy(), ref, raw.positions, ratio, S, exact=True)


def test_all_equal_scores_tie_break():
    # q = 0 -> every visible score is exactly 0 -> the k lowest rows win
    S, T = 900, 5
    positions = np.array([899, 600, 513, 512, 100], dtype=np.int32)
    inp = _edge_inputs("ties", positions, S, kind="int", kv_dtype="f16", H=16, D=64, w_kind="pow2")
    inp.q[:] = 0
    wl = synth.Workload("ties", T=T, H=16, D=64, S=S, ratio=1, pos0=0, kind="int", kv_dtype="f16")
    inp = synth.Inputs(wl, inp.q, inp.w, inp.k, inp.positions, inp.q_attn, inp.kv)
    g = run_all(inp)
    for t in range(T):
        n = min(S, int(positions[t]) + 1)
        want = list(range(min(n, 512))) + [-1] * (512 - min(n, 512))
        assert list(g["idx"][t]) == want
        assert list(g["fidx"][t]) == want


def test_integer_config_many_ties_random_k():
    # small integer scores (many exact ties) with a k_top that is not a multiple of 128
    wl0 = synth.WORKLOADS["tiny_exact"]
    inp = synth.make_inputs(wl0, seed=3, T=37, pos0=4000)
    S, k_top = wl0.S, 300
    d = to_device(inp)
    scores = ds4x.indexer_score(d["q"], d["w"], d["k"], d["positions"], wl0.ratio, S=S)
    idx, cnt = ds4x.topk(scores, d["positions"], S, wl0.ratio, k_top)
    out, lse = ds4x.sparse_attn(d["q_attn"], d["kv"], idx, S=S, scale=wl0.scale)
    torch.cuda.synchronize()
    ref_scores = oracle.indexer_score(inp.q, inp.w, inp.k, inp.positions, wl0.ratio, S=S)
    check_scores(scores.cpu().numpy(), ref_scores, inp.positions, wl0.ratio, S, exact=True)
    ref_idx, ref_cnt = oracle.topk(ref_scores, inp.positions, S, wl0.ratio, k_top)
    assert np.array_equal(idx.cpu().numpy(), ref_idx)
    ref_out, ref_lse = oracle.sparse_attn(inp.q_attn, inp.kv, "f16", ref_idx, S, wl0.scale)
    check_attn(host16(out), ref_out, "f16", lse.cpu().numpy(), ref_lse)


def test_attention_invalid_and_out_of_range_indices():
    rng = np.random.default_rng(0)
    S, T = 300, 6
    inp = _edge_inputs("attn_idx", np.full(T, 10**6), S)
    idx = np.stack([rng.choice(S, 512, replace=True) for _ in range(T)]).astype(np.int32)
    idx[0, :] = -1                       # no valid row
    idx[1, 5:] = -1                      # five rows
    idx[2, ::3] = S + 7                  # out of range entries are skipped
    idx[3, :] = 17                       # the same row 512 times
    d = to_device(inp)
    out, lse = ds4x.sparse_attn(d["q_attn"], d["kv"], torch.from_numpy(idx).cuda(), S=S)
    torch.cuda.synchronize()
    ref_out, ref_lse = oracle.sparse_attn(inp.q_attn, inp.kv, "bf16", idx, S, 1 / np.sqrt(512))
    check_attn(host16(out), ref_out, "bf16", lse.cpu().numpy(), ref_lse,
               extra=few_rows_bound(inp.kv, idx, ref_out, "bf16", S))
    assert np.all(np.isneginf(lse[0].cpu().numpy()))


def test_split_topk_decode_row():
    # one token over a long row: the row is split across CTAs and merged
    S = 262144 + 37
    rng = np.random.default_rng(11)
    scores = rng.standard_normal((1, S)).astype(np.float32)
    scores[0, 1000:1300] = scores[0, 1000]          # a run of exact ties
    pos = np.array([4 * S + 3], dtype=np.int32)
    assert ds4x.topk_workspace_bytes(1, S, 512) > 0
    idx, cnt = ds4x.topk(torch.from_numpy(scores).cuda(), torch.from_numpy(pos).cuda(), S, 4, 512)
    torch.cuda.synchronize()
    ref_idx, ref_cnt = oracle.topk(scores, pos, S, 4, 512)
    assert np.array_equal(idx.cpu().numpy(), ref_idx)
    assert np.array_equal(cnt.cpu().numpy(), ref_cnt)


@pytest.mark.parametrize("S", [2048, 4096, 8192, 16384])
@pytest.mark.parametrize("pad", [0, 1])
def test_topk_one_cta_rounds_exact(S, pad):
    # one CTA per token with the keys in registers, at every row-length class: a dense cluster of
    # repeated adjacent floats behind two far outliers (a boundary bin of more rows than are
    # ranked directly: a second round, then a direct rank among ties), equal scores under 100
    # larger ones (a pure tie at the boundary), N(0,1), a ragged visible count, a row of equal
    # scores; pad = 1 makes the row pitch odd so that most rows start unaligned
    rng = np.random.default_rng(S + pad)
    ld = S + pad
    sc = rng.standard_normal((5, ld)).astype(np.float32)
    sc[0, :S] = (np.float32(3.0).view(np.int32) + rng.integers(0, 400, S)).astype(np.int32).view(np.float32)
    sc[0, 5], sc[0, S - 7] = -1e30, 1e30
    sc[1, :S] = 0.5
    sc[1, rng.choice(S, 100, replace=False)] = 1.0 + rng.random(100).astype(np.float32)
    sc[4, :] = -2.0
    pos = np.array([4 * S - 1, 4 * S - 1, 4 * S - 1, 4 * (S - 37) - 1, 4 * S + 100], dtype=np.int32)
    idx, cnt = ds4x.topk(torch.from_numpy(sc).cuda(), torch.from_numpy(pos).cuda(), S, 4, 512)
    torch.cuda.synchronize()
    assert ds4x.device_status() == ds4x.OK
    ref_idx, ref_cnt = oracle.topk(sc, pos, S, 4, 512)
    assert np.array_equal(idx.cpu().numpy(), ref_idx)
    assert np.array_equal(cnt.cpu().numpy(), ref_cnt)


@pytest.mark.parametrize("S", [2048, 8192, 12000, 16384, 40000, 65536])
@pytest.mark.parametrize("k_top", [300, 512, 1024])
def test_topk_many_tokens_exact(S, k_top):
    # at least one token per SM, so every row takes the one-CTA-per-token kernels: keys in registers
    # up to 4096 rows, the row staged in shared memory up to 32768, the streaming one-pass select
    # (running threshold, ballot compaction) beyond.  N(0,1) rows, small integers (long runs of
    # ties), a row whose best scores all sit in one eighth of it, a row of equal scores, and visible
    # counts from just above k_top to the whole row
    T = 160
    rng = np.random.default_rng(S * 7 + k_top)
    sc = rng.standard_normal((T, S)).astype(np.float32)
    sc[1::4] = rng.integers(-3, 4, size=sc[1::4].shape).astype(np.float32)
    seg = S // 8
    sc[2::4, 3 * seg:4 * seg] += 50.0
    sc[3] = 1.5
    nv = rng.integers(k_top + 1, S + 1, size=T)
    nv[:8] = [S, S, S, S, k_top + 1, k_top + 2, min(S, 2048), S - 1]
    pos = (4 * nv - 1).astype(np.int32)
    assert ds4x.topk_workspace_bytes(T, S, k_top) == 0
    idx, cnt = ds4x.topk(torch.from_numpy(sc).cuda(), torch.from_numpy(pos).cuda(), S, 4, k_top)
    torch.cuda.synchronize()
    assert ds4x.device_status() == ds4x.OK
    ref_idx, ref_cnt = oracle.topk(sc, pos, S, 4, k_top)
    assert np.array_equal(cnt.cpu().numpy(), ref_cnt)
    bad = np.nonzero(np.any(idx.cpu().numpy() != ref_idx, axis=1))[0]
    assert bad.size == 0, f"tokens {bad[:8]} differ from the oracle"


@pytest.mark.parametrize("case", ["boundary_overflow", "all_equal", "few_tokens"])
def test_long_row_topk_exact(case):
    # long rows over many CTAs: a boundary bin with more rows than the candidate buffer (the last
    # CTA ranks the whole row), a row of equal scores (lowest rows win), several tokens at once
    rng = np.random.default_rng(12)
    S, T = 262144, 1
    if case == "boundary_overflow":
        scores = np.floor(rng.standard_normal((1, S)) / 1.5).astype(np.float32)   # ~17k rows tie at 1.0
    elif case == "all_equal":
        scores = np.full((1, S), 3.25, dtype=np.float32)
    else:
        T = 7
        scores = rng.standard_normal((T, S)).astype(np.float32)
        scores[3, 5000:9000] = scores[3].max()                                    # a tied block on top
    pos = (4 * S - 1 - np.arange(T) * 40000).astype(np.int32)                      # different n per token
    idx, cnt = ds4x.topk(torch.from_numpy(scores).cuda(), torch.from_numpy(pos).cuda(), S, 4, 512)
    torch.cuda.synchronize()
    assert ds4x.device_status() == ds4x.OK
    ref_idx, ref_cnt = oracle.topk(scores, pos, S, 4, 512)
    assert np.array_equal(idx.cpu().numpy(), ref_idx)
    assert np.array_equal(cnt.cpu().numpy(), ref_cnt)
    if case == "all_equal":
        assert np.array_equal(ref_idx[0], np.arange(512))


# ------------------------------------------------------- one token over a long row, fused
def _fused_one_token(inp):
    d = to_device(inp)
    wl = inp.wl
    scores = ds4x.indexer_score(d["q"], d["w"], d["k"], d["positions"], wl.ratio, S=wl.S)
    fidx, _, _ = ds4x.index_and_attend(d["q"], d["w"], d["k"], d["positions"], d["q_attn"], d["kv"],
                                       wl.ratio, wl.k_top, S=wl.S, scale=wl.scale)
    torch.cuda.synchronize()
    assert ds4x.device_status() == ds4x.OK
    return scores.cpu().numpy(), fidx.cpu().numpy()


@pytest.mark.parametrize("case,S,n", [("random", 65536 + 37, None), ("random", 16384, None),
                                      ("random", 12000, None), ("partly_visible", 50000, 30001),
                                      ("all_ties", 20000, None), ("top_ties", 40000, None),
                                      ("int_ties", 40000, None), ("int_ties", 65536, None)])
def test_one_token_fused_topk_exact(case, S, n):
    # One token over a long row in the fused path (a decode step). The scorer hands the top-k a
    # lower bound on the k_top-th key; the top-k ranks only the rows at or above it when their
    # count lies in [k_top, its list's capacity] and its boundary bin is small (random and integer
    # scores), else goes on with its histogram phases (every score equal; 600 rows sharing the
    # top score; a row of which only part is visible, so the bound falls to the lowest key).
    # Rows under 16384 have too few scorer CTAs for the bound. The indices must equal the oracle's
    # top-k of the scores the GPU computed.
    n = S if n is None else n
    kind = "int" if case == "int_ties" else "normal"
    raw = _edge_inputs(f"one_{case}_{S}", [n - 1], S, kind=kind, w_kind="pow2" if kind == "int" else "pos", seed=2)
    wl = synth.Workload(raw.wl.name, T=1, H=64, D=128, S=S, ratio=1, pos0=0, kind=kind, kv_dtype="bf16")
    inp = synth.Inputs(wl, raw.q, raw.w, raw.k, raw.positions, raw.q_attn, raw.kv)
    if case == "all_ties":
        inp.q[:] = 0
    if case == "top_ties":  # 600 spread rows become twice the best row: twice its score, exactly
        scores, _ = _fused_one_token(inp)
        best = int(np.argmax(scores[0, :n]))
        k16 = inp.k.view(np.float16)
        k16[np.arange(17, n, n // 600)[:600]] = k16[best] * np.float16(2)
    scores, fidx = _fused_one_token(inp)
    vis = scores[0, :n]
    if case == "all_ties":
        assert np.all(vis == 0)
    if case == "top_ties":
        assert np.count_nonzero(vis == vis.max()) == 600
    ref_idx, _ = oracle.topk(scores, inp.positions, S, 1, wl.k_top)
    assert np.array_equal(fidx, ref_idx)


# --------------------------------------- full-size workloads in the benchmark's launch shape
@pytest.mark.parametrize("name", ["prefill_8k", "prefill_32k", "prefill_64k"])
def test_full_size_sampled(name):
    wl = synth.WORKLOADS[name]
    inp = synth.make_inputs(wl, seed=0)
    d = to_device(inp)
    fidx, fout, flse = ds4x.index_and_attend(d["q"], d["w"], d["k"], d["positions"], d["q_attn"], d["kv"],
                                             wl.ratio, wl.k_top, S=wl.S, scale=wl.scale)
    torch.cuda.synchronize()
    assert ds4x.device_status() == ds4x.OK
    sample = np.array([0, 1, 517, 1024, 1500, wl.T - 2, wl.T - 1])
    gidx = fidx.cpu().numpy()[sample]
    gout = host16(fout)[sample]
    glse = flse.cpu().numpy()[sample]
    q, w, pos = inp.q[sample], inp.w[sample], inp.positions[sample]
    ref_scores = oracle.indexer_score(q, w, inp.k, pos, wl.ratio, S=wl.S)
    ref_idx, _ = oracle.topk(ref_scores, pos, wl.S, wl.ratio, wl.k_top)
    check_index_sets(gidx, ref_idx, ref_scores, pos, wl.ratio, wl.S, wl.k_top)
    ref_out, ref_lse = oracle.sparse_attn(inp.q_attn[sample], inp.kv, wl.kv_dtype, gidx, wl.S, wl.scale)
    check_attn(gout, ref_out, wl.kv_dtype, glse, ref_lse)
    # every token: a valid, ascending selection of k_top visible rows
    allidx = fidx.cpu().numpy()
    nv = np.minimum(wl.S, (inp.positions.astype(np.int64) + 1) // wl.ratio)
    assert np.all(np.diff(allidx, axis=1) > 0)
    assert np.all(allidx[:, 0] >= 0) and np.all(allidx[:, -1] < nv)


def test_scores_full_64k_rows_elementwise():
    # the 64k chunk's scorer in its wide-tile launch (4 tokens x 64 heads a tile) over all 16384
    # rows, element by element against the oracle: the last 20 tokens of the chunk (five token
    # groups, each seeing 15868..16384 rows, so the masked tails differ)
    wl = synth.WORKLOADS["prefill_64k"]
    T = 20
    inp = synth.make_inputs(wl, seed=0, T=T, pos0=wl.pos0 + wl.T - T)
    d = to_device(inp)
    scores = ds4x.indexer_score(d["q"], d["w"], d["k"], d["positions"], wl.ratio, S=wl.S)
    torch.cuda.synchronize()
    assert ds4x.device_status() == ds4x.OK
    ref = oracle.indexer_score(inp.q, inp.w, inp.k, inp.positions, wl.ratio, S=wl.S)
    check_scores(scores.cpu().numpy(), ref, inp.positions, wl.ratio, wl.S, exact=False)


def test_scores_decode_rows_elementwise():
    # the decode step's scorer (one token: the narrow tile) over a 1M-context row of 262181
    # compressed rows, element by element against the oracle: a token that sees every row, the
    # decode loop's first position (the last 37 rows masked) and one far back (a long masked tail)
    wl = synth.WORKLOADS["decode_1m"]
    S = 262144 + 37
    pos = np.array([4 * S + 10, wl.pos0, 4 * 200000 - 1], dtype=np.int32)
    inp = synth.make_inputs(wl, seed=2, T=3, S=S, rows=S)
    d = to_device(inp)
    got = []
    for t in range(3):     # one call per token: each takes the narrow, single-token tile
        pt = torch.from_numpy(pos[t:t + 1].copy()).cuda()
        got.append(ds4x.indexer_score(d["q"][t:t + 1], d["w"][t:t + 1], d["k"], pt, wl.ratio, S=S))
    torch.cuda.synchronize()
    assert ds4x.device_status() == ds4x.OK
    ref = oracle.indexer_score(inp.q, inp.w, inp.k, pos, wl.ratio, S=S)
    check_scores(torch.cat(got).cpu().numpy(), ref, pos, wl.ratio, S, exact=False)
    assert [n_vis(p, wl.ratio, S) for p in pos] == [S, 262144, 200000]


def test_pooled_ratio128_all_rows():
    # the ratio-128 layer kind: a token at the end of a 64k chunk sees at most 512 pooled rows, so
    # the fused path skips scoring and attends every visible row (sequential indices)
    wl = synth.WORKLOADS["pooled_64k_r128"]
    T = 96
    inp = synth.make_inputs(wl, seed=5, T=T, pos0=wl.pos0 + wl.T - T)
    d = to_device(inp)
    fidx, fout, flse = ds4x.index_and_attend(d["q"], d["w"], d["k"], d["positions"], d["q_attn"], d["kv"],
                                             wl.ratio, wl.k_top, S=wl.S, scale=wl.scale)
    torch.cuda.synchronize()
    assert ds4x.device_status() == ds4x.OK
    gidx = fidx.cpu().numpy()
    ref_scores = oracle.indexer_score(inp.q, inp.w, inp.k, inp.positions, wl.ratio, S=wl.S)
    ref_idx, _ = oracle.topk(ref_scores, inp.positions, wl.S, wl.ratio, wl.k_top)
    assert np.array_equal(gidx, ref_idx)
    nv = [n_vis(p, wl.ratio, wl.S) for p in inp.positions]
    assert all(np.array_equal(gidx[t, :nv[t]], np.arange(nv[t])) for t in range(T))
    ref_out, ref_lse = oracle.sparse_attn(inp.q_attn, inp.kv, wl.kv_dtype, gidx, wl.S, wl.scale)
    check_attn(host16(fout), ref_out, wl.kv_dtype, flse.cpu().numpy(), ref_lse)


def test_pooled_ratio128_full_chunk_sampled():
    # the benchmark's ratio-128 workload at its full size: every token takes the shortcut; sampled
    # tokens' attention against the oracle, every token's indices against the closed form
    wl = synth.WORKLOADS["pooled_64k_r128"]
    inp = synth.make_inputs(wl, seed=0)
    d = to_device(inp)
    fidx, fout, flse = ds4x.index_and_attend(d["q"], d["w"], d["k"], d["positions"], d["q_attn"], d["kv"],
                                             wl.ratio, wl.k_top, S=wl.S, scale=wl.scale)
    torch.cuda.synchronize()
    assert ds4x.device_status() == ds4x.OK
    gidx = fidx.cpu().numpy()
    nv = np.minimum(wl.S, (inp.positions.astype(np.int64) + 1) // wl.ratio)
    want = np.where(np.arange(wl.k_top)[None, :] < nv[:, None], np.arange(wl.k_top)[None, :], -1)
    assert np.array_equal(gidx, want)
    sample = np.array([0, 1, 700, 1400, wl.T - 1])
    ref_out, ref_lse = oracle.sparse_attn(inp.q_attn[sample], inp.kv, wl.kv_dtype, gidx[sample], wl.S, wl.scale)
    check_attn(host16(fout)[sample], ref_out, wl.kv_dtype, flse.cpu().numpy()[sample], ref_lse)

