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


def check_rows(got, ref, dtype):
    """fp32 pooling on the GPU, fp64 in the oracle, each rounded once: at most one unit in the
    last place of the 16-bit result apart."""
    g = synth.bits_to_f32(got, dtype).astype(np.float64)
    r = synth.bits_to_f32(ref, dtype).astype(np.float64)
    ulp = 2.0 ** (-7 if dtype == "bf16" else -10)
    err = np.abs(g - r) - (ulp * np.abs(r) + 2.0 ** -24)
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
        check_rows(rows, rrows, dtype)
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
    check_rows(rows, rrows, "bf16")
    assert np.array_equal(fxo, rfx) and np.array_equal(fgo, rfg)

