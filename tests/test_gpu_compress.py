"""The compressor through the C ABI against the CPU oracle on the same seeded inputs."""
import numpy as np
import pytest
import torch

import deepseek_v4_sparse_gb300 as ds4x
import oracle
import synth
from parity import dev16, host16

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
    assert ds4x.device_status() == ds4x.OK


def _gpu(x, g, fx, fg, bias, ratio, dtype):
    rows, fxo, fgo = ds4x.compress(dev16(x, dtype), dev16(g, dtype), torch.from_numpy(bias).cuda(), ratio,
                                   dev16(fx, dtype) if fx.shape[0] else None,
                                   dev16(fg, dtype) if fg.shape[0] else None)
    torch.cuda.synchronize()
    return host16(rows), host16(fxo), host16(fgo)


def block_absmax(x, fx, ratio, dtype):
    """max_i |x_i[d]| over each block's positions (frontier rows first), [n_out, D] float64."""
    seq = np.concatenate([fx, x]) if fx is not None and fx.shape[0] else x
    n_out = seq.shape[0] // ratio
    v = np.abs(synth.bits_to_f32(seq[:n_out * ratio], dtype).astype(np.float64))
    return v.reshape(n_out, ratio, -1).max(axis=1)


def check_rows(got, ref, dtype, xmax, ratio):
    """fp32 pooling on the GPU, fp64 in the oracle, each rounded once to the 16-bit type.  The
    GPU's fp32 value of a row differs from the exact one by the rounding of its weighted sum
    (up to ratio * 2^-24 of the largest term) and of its weights (gate sum and product, the
    ex2.approx result: about 10 * 2^-24 relative each), i.e. by at most (ratio + 32) * 2^-24 *
    max_i |x_i| when the block's terms cancel.  The two roundings to 16 bits add one unit in the
    last place (2^-7 / 2^-10 of |result| at most, 2^-24 below the normal range)."""
    g = synth.bits_to_f32(got, dtype).astype(np.float64)
    r = synth.bits_to_f32(ref, dtype).astype(np.float64)
    ulp = 2.0 ** (-7 if dtype == "bf16" else -10)
    err = np.abs(g - r) - (ulp * np.abs(r) + 2.0 ** -24 + (ratio + 32) * 2.0 ** -24 * xmax)
    assert err.max(initial=-1) <= 0, f"compressor error {np.abs(g - r).max()}"
    # almost every row matches bit for bit; a flip needs the fp32 result within ~1e-7 of a midpoint
    assert np.mean(got == ref) > 0.99


@pytest.mark.parametrize("dtype,D,ratio,T,f", [
    ("bf16", 512, 4, 2048, 0),      # the kv rows of a 2048-token chunk at ratio 4
    ("f16", 128, 4, 2048, 3),       # the indexer's k rows, with a held-over partial block
    ("bf16", 512, 128, 2048, 0),    # a ratio-128 layer
    ("bf16", 512, 128, 300, 100),   # a frontier deep into its block, a partial block left over
    ("f16", 8, 3, 50, 2),           # odd ratio, one 8-channel group
    ("bf16", 136, 7, 33, 6),        # 17 channel groups: no power-of-two slab
    ("bf16", 512, 4, 1, 2),         # no block completes: the frontier grows from both sources
    ("bf16", 512, 4, 1, 3),         # decode: the one new position completes a block
    ("f16", 128, 4, 0, 3),          # nothing new: the frontier is copied through
])
def test_compress_vs_oracle(dtype, D, ratio, T, f):
    x, g, fx, fg, bias = synth.compress_inputs(1, f"cmp_{dtype}_{D}_{ratio}_{T}_{f}", T, D, ratio, dtype, f)
    rows, fxo, fgo = _gpu(x, g, fx, fg, bias, ratio, dtype)
    rrows, rfx, rfg = oracle.compress(x, g, bias, dtype, ratio, fx if f else None, fg if f else None)
    assert rows.shape == rrows.shape and fxo.shape == rfx.shape
    if rows.size:
        check_rows(rows, rrows, dtype, block_absmax(x, fx, ratio, dtype), ratio)
    assert np.array_equal(fxo, rfx) and np.array_equal(fgo, rfg)


def test_compress_ratio_one_is_identity():
    x, g, _, _, bias = synth.compress_inputs(2, "cmp_r1", 64, 256, 1, "bf16")
    rows, _, _ = _gpu(x, g, x[:0], g[:0], bias, 1, "bf16")
    assert np.array_equal(rows, x)


def test_compress_dominant_gate_selects_row():
    ratio, D, T = 16, 64, 160
    x, _, _, _, _ = synth.compress_inputs(3, "cmp_dom", T, D, ratio, "f16")
    rng = np.random.default_rng(3)
    pick = rng.integers(0, ratio, size=(T // ratio, D))
    gv = np.zeros((T, D))
    for j in range(T // ratio):
        gv[j * ratio + pick[j], np.arange(D)] = 100.0
    rows, _, _ = _gpu(x, synth.to_f16_bits(gv), x[:0], x[:0], np.zeros((ratio, D), np.float32), ratio, "f16")
    for j in range(T // ratio):
        assert np.array_equal(rows[j], x[j * ratio + pick[j], np.arange(D)]), j


@pytest.mark.parametrize("ratio", [4, 128])
def test_compress_split_calls_equal_one_bit_for_bit(ratio):
    # a block's arithmetic does not depend on which call supplied its positions
    D, N = 512, 1100
    x, g, _, _, bias = synth.compress_inputs(4, f"cmp_split_{ratio}", N, D, ratio, "bf16")
    whole, wfx, wfg = _gpu(x, g, x[:0], g[:0], bias, ratio, "bf16")
    parts, fx, fg = [], x[:0], g[:0]
    for a, b in ((0, 5), (5, 517), (517, 518), (518, N)):
        r, fx, fg = _gpu(x[a:b], g[a:b], fx, fg, bias, ratio, "bf16")
        parts.append(r)
    assert np.array_equal(np.concatenate(parts), whole)
    assert np.array_equal(fx, wfx) and np.array_equal(fg, wfg)


def test_compress_streaming_batch_full_size():
    # the benchmark's bandwidth case: a 64k-token batch of kv rows at ratio 4 with a 3-position frontier
    D, ratio, T, f = 512, 4, 65536, 3
    x, g, fx, fg, bias = synth.compress_inputs(0, "bench_kv_64k_r4", T, D, ratio, "bf16", f)
    rows, fxo, fgo = _gpu(x, g, fx, fg, bias, ratio, "bf16")
    rrows, rfx, rfg = oracle.compress(x, g, bias, "bf16", ratio, fx, fg)
    assert rows.shape == rrows.shape == ((T + f) // ratio, D)
    check_rows(rows, rrows, "bf16", block_absmax(x, fx, ratio, "bf16"), ratio)
    assert np.array_equal(fxo, rfx) and np.array_equal(fgo, rfg)



def _streamed(n_out, f, D, ratio):
    """Whether a call takes the streamed path: ratio <= 4, D a power of two <= 512, and at least
    two stages (32 KB of x rows each) of whole blocks for every SM after the frontier's block."""
    if ratio not in (1, 2, 4) or D > 512 or D & (D - 1):
        return False
    bps = (16384 // D) // ratio
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    return n_out - (1 if f else 0) >= 2 * sms * bps


@pytest.mark.parametrize("dtype,D,ratio,T,f", [
    ("bf16", 512, 4, 20003, 3),   # a held-over block 0, a ragged last stage, a partial block left over
    ("f16", 128, 4, 40001, 1),    # the indexer's k rows: 128-position stages
    ("bf16", 512, 2, 12001, 1),
    ("bf16", 256, 1, 20000, 0),   # ratio 1: every position is a row
    ("f16", 8, 4, 640002, 2),     # one 8-channel group a row: 2048-position stages
])
def test_compress_streamed_batches_vs_oracle(dtype, D, ratio, T, f):
    assert _streamed((T + f) // ratio, f, D, ratio)
    x, g, fx, fg, bias = synth.compress_inputs(5, f"cmp_stream_{dtype}_{D}_{ratio}_{T}_{f}", T, D, ratio, dtype, f)
    rows, fxo, fgo = _gpu(x, g, fx, fg, bias, ratio, dtype)
    rrows, rfx, rfg = oracle.compress(x, g, bias, dtype, ratio, fx if f else None, fg if f else None)
    assert rows.shape == rrows.shape and fxo.shape == rfx.shape
    check_rows(rows, rrows, dtype, block_absmax(x, fx, ratio, dtype), ratio)
    assert np.array_equal(fxo, rfx) and np.array_equal(fgo, rfg)


def test_compress_streamed_and_one_pass_paths_agree_bit_for_bit():
    # a long batch split so that the middle call streams and the short ones take the one-pass
    # kernel: every block comes out the same bits as from the one streamed call
    D, ratio, N = 512, 4, 20000
    assert _streamed(N // ratio, 0, D, ratio) and not _streamed(249, 1, D, ratio)
    x, g, _, _, bias = synth.compress_inputs(6, "cmp_paths", N, D, ratio, "bf16")
    whole, wfx, wfg = _gpu(x, g, x[:0], g[:0], bias, ratio, "bf16")
    parts, fx, fg = [], x[:0], g[:0]
    for a, b in ((0, 5), (5, 19005), (19005, N)):
        r, fx, fg = _gpu(x[a:b], g[a:b], fx, fg, bias, ratio, "bf16")
        parts.append(r)
    assert _streamed((19005 - 5 + 1) // ratio, 1, D, ratio)
    assert np.array_equal(np.concatenate(parts), whole)
    assert np.array_equal(fx, wfx) and np.array_equal(fg, wfg)
