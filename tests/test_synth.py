"""The input generator: large draws are split into pieces on threads; the pieces must give the
same bits as one sequential draw (the stream is counter-based)."""
import numpy as np

import synth


def test_parallel_normal_draw_equals_sequential():
    n = synth._PARALLEL_MIN + 12345            # odd length: the last Box-Muller pair is split
    for dtype in ("f16", "bf16"):
        a = synth.normal_bits(3, "check/normal", n, dtype)
        b = synth.to_bits(synth.normal(3, "check/normal", n), dtype)
        assert a.dtype == np.uint16 and np.array_equal(a, b)


def test_normal_offsets_are_stream_positions():
    full = synth.normal(5, "check/offsets", 1001)
    for off in (0, 1, 2, 333, 998):
        assert np.array_equal(synth.normal(5, "check/offsets", 1001 - off, offset=off), full[off:])
