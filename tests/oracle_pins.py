"""Pins of the CPU oracle against facts that do not come from the oracle itself.

Each check takes an ``oracle.Oracle`` and raises AssertionError when the oracle
disagrees with the independent fact. tests/test_oracle.py runs them on the real oracle;
tests/test_oracle_mutants.py runs them on copies of the oracle with one planted
mistake each and requires that some check fails.

Independent facts used:
  * the IEEE binary16 / bfloat16 encodings (numpy's float16, the float32 bit layout,
    exact rational rounding with fractions.Fraction);
  * a hand-worked example (tests/golden/indexer_worked_example.txt);
  * an int64 recomputation of 4*score on integer inputs (exact closed form);
  * a float64 numpy evaluation of the definition (different summation order);
  * brute-force ranking with Python's sorted() on tiny inputs;
  * the selection invariants (dominance, mask, count, ascending order, shortcut);
  * closed-form attention cases (zero query, single row, two rows) and a textbook
    float64 numpy softmax-attention;
  * for the decode loop: the closed-form row count of every step, the appended bytes, and a
    numpy brute-force (definition score, sorted() ranking, textbook attention) of each step;
  * for local-plus-pooled attention: a textbook float64 causal sliding-window attention, a
    float64 softmax over the union of both row sources, the log-sum-exp merge identity of two
    one-source results, the exact rational mean for a zero query, a one-row window giving that
    row, and the pooled result whenever no raw row is in reach;
  * for the compressor: the exact rational mean of each block under equal gates, a dominant gate
    selecting its position's row, a float64 numpy gated pooling, and the equality of one call with
    any two calls that carry the frontier.
"""
from __future__ import annotations

import math
import os
from fractions import Fraction

import numpy as np

import synth

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden",
                      "indexer_worked_example.txt")


# ----------------------------------------------------------------------------- helpers
def _f16(x):
    return synth.to_f16_bits(np.asarray(x, dtype=np.float64))


def _f16_val(bits):
    return synth.f16_bits_to_f32(bits).astype(np.float64)


def _bits_val(bits, dtype):
    return synth.bits_to_f32(bits, dtype).astype(np.float64)


def parse_golden(path=GOLDEN):
    vals = {}
    for line in open(path):
        line = line.split("#", 1)[0].strip()
        if not line:
            continue
        key, rest = line.split(":", 1)
        vals[key.strip()] = [float(v) for v in rest.split()]
    return vals


def _rand_int_case(seed, T, H, D, S, lo=-3, hi=3, w_pow2=True):
    q = synth.uniform_int(seed, "pin/q", T * H * D, lo, hi).reshape(T, H, D)
    k = synth.uniform_int(seed, "pin/k", S * D, lo, hi).reshape(S, D)
    sel = synth.uniform_int(seed, "pin/w", T * H, 0, 2)
    w4 = np.array([1, 2, 4])[sel].reshape(T, H)  # 4*w with w in {1/4, 1/2, 1}
    return q, k, w4


def _brute_topk(row, n, k_top):
    order = sorted(range(n), key=lambda s: (-row[s], s))
    sel = sorted(order[:k_top])
    return sel + [-1] * (k_top - len(sel))


# ------------------------------------------------------------------- number formats
def check_f16_decode_exhaustive(o):
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ref = bits.view(np.float16).astype(np.float64)
    got = np.array([o.decode16(int(b), "f16") for b in bits])
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])


def check_bf16_decode_exhaustive(o):
    bits = np.arange(65536, dtype=np.uint32)
    with np.errstate(invalid="ignore"):
        ref = (bits << 16).astype(np.uint32).view(np.float32).astype(np.float64)
    got = np.array([o.decode16(int(b), "bf16") for b in bits])
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])


def _rne_fraction(x: Fraction, mant: int, ebits: int):
    """Exact round-to-nearest-even of a rational into a binary format, as a Fraction
    (or +-inf)."""
    bias = (1 << (ebits - 1)) - 1
    emin, emax = 1 - bias, bias
    a = abs(x)
    if a == 0:
        return Fraction(0)
    E = math.floor(math.log2(a))
    while Fraction(2) ** E > a:
        E -= 1
    while Fraction(2) ** (E + 1) <= a:
        E += 1
    E = max(E, emin)
    q = Fraction(2) ** (E - mant)
    m = a / q
    r = math.floor(m)
    rem = m - r
    if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and r % 2 == 1):
        r += 1
    val = r * q
    if val >= Fraction(2) ** (emax + 1):
        return math.inf if x > 0 else -math.inf
    return val if x > 0 else -val


def check_encode_rne(o):
    rng = np.random.default_rng(7)
    # random magnitudes across the normal and subnormal ranges, plus exact ties
    xs = list(rng.standard_normal(400) * np.exp2(rng.integers(-30, 18, 400)))
    xs += [1 + 2 ** -11, 1 + 3 * 2 ** -11, 2 ** -25, 3 * 2 ** -25, 65519.0, 65520.0, 1e-9, -0.0,
           0.880797077977882, 1 + 2 ** -8, 1 + 3 * 2 ** -8, 2 ** -134, 3 * 2 ** -134]
    for x in xs:
        for dtype, mant, ebits in (("f16", 10, 5), ("bf16", 7, 8)):
            got = o.decode16(o.encode16(float(x), dtype), dtype)
            want = _rne_fraction(Fraction(float(x)), mant, ebits)
            if isinstance(want, float):
                assert got == want, (x, dtype, got, want)
            else:
                assert Fraction(got) == want, (x, dtype, got, float(want))
    # numpy's double -> half conversion (round to nearest even) as a second witness
    ys = rng.standard_normal(2000) * np.exp2(rng.integers(-26, 16, 2000))
    with np.errstate(over="ignore"):
        ref = ys.astype(np.float16).view(np.uint16)
    got = np.array([o.encode16(float(y), "f16") for y in ys], dtype=np.uint16)
    assert np.array_equal(got, ref)


# ------------------------------------------------------------------------ visibility
def check_visibility(o):
    # row s visible iff (s+1)*ratio <= p+1, counted by brute force
    for ratio in (1, 2, 4, 128):
        for S in (0, 1, 7, 300):
            for p in list(range(0, 40)) + [511, 512, 4095, 65535]:
                brute = sum(1 for s in range(S) if (s + 1) * ratio <= p + 1)
                assert o.n_visible(p, ratio, S) == brute, (p, ratio, S)


# ------------------------------------------------------------------ worked example
def check_golden_example(o):
    g = parse_golden()
    T, H, D, S = (int(g[k][0]) for k in ("T", "H", "D", "S"))
    ratio, k_top = int(g["ratio"][0]), int(g["k_top"][0])
    pos = np.array(g["positions"], dtype=np.int32)
    q = _f16(np.array(g["q"]).reshape(T, H, D))
    w = _f16(np.array(g["w"]).reshape(T, H))
    k = _f16(np.array(g["k"]).reshape(S, D))
    sc = o.indexer_score(q, w, k, pos, ratio)
    want = np.array(g["scores"], dtype=np.float32).reshape(T, S)
    assert np.array_equal(sc, want), (sc, want)
    idx, cnt = o.topk(sc, pos, S, ratio, k_top)
    assert np.array_equal(idx, np.array(g["indices"], dtype=np.int32).reshape(T, k_top)), idx
    assert np.array_equal(cnt, np.array(g["counts"], dtype=np.int32)), cnt
    Hq, Dkv = int(g["attn_Hq"][0]), int(g["attn_Dkv"][0])
    kv = _f16(np.array(g["attn_kv"]).reshape(-1, Dkv))
    qa = _f16(np.array(g["attn_q"]).reshape(T, Hq, Dkv))
    ai = np.array(g["attn_indices"], dtype=np.int32).reshape(T, -1)
    out, lse = o.sparse_attn(qa, kv, "f16", ai, kv.shape[0], float(g["attn_scale"][0]))
    want_out = np.array(g["attn_out"]).reshape(T, Hq, Dkv)
    assert np.array_equal(_f16_val(out), want_out), (_f16_val(out), want_out)
    want_lse = np.array(g["attn_lse"], dtype=np.float64).reshape(T, Hq)
    fin = np.isfinite(want_lse)
    assert np.array_equal(np.isinf(lse), ~fin)
    assert np.allclose(lse[fin], want_lse[fin], rtol=1e-6, atol=0)
    idx2, out2, lse2 = o.index_and_attend(q, w, k, pos, _f16(np.zeros((T, 64, 8))),
                                          _f16(np.zeros((S, 8))), "f16", S, ratio, k_top, 1.0)
    assert np.array_equal(idx2, idx)


# ------------------------------------------------------------------------- scoring
def check_scores_int64_closed_form(o):
    T, H, D, S, ratio = 9, 16, 64, 70, 4
    q, k, w4 = _rand_int_case(11, T, H, D, S)
    pos = np.array([0, 3, 4, 100, 150, 255, 279, 280, 400], dtype=np.int32)
    sc = o.indexer_score(_f16(q), _f16(w4 / 4.0), _f16(k), pos, ratio, ld=S + 3)
    dots = np.einsum("thd,sd->ths", q.astype(np.int64), k.astype(np.int64))
    four = (w4[:, :, None].astype(np.int64) * np.maximum(dots, 0)).sum(axis=1)  # 4*score
    for t in range(T):
        n = min(S, (int(pos[t]) + 1) // ratio)
        assert np.array_equal(sc[t, :n].astype(np.float64) * 4.0, four[t, :n].astype(np.float64))
        assert np.all(np.isneginf(sc[t, n:S]))
        assert np.all(np.isnan(sc[t, S:]))  # columns past S are never written


def check_scores_float_vs_numpy(o):
    T, H, D, S, ratio = 5, 8, 32, 40, 2
    rng = np.random.default_rng(3)
    q = _f16(rng.standard_normal((T, H, D)))
    k = _f16(rng.standard_normal((S, D)))
    w = _f16(rng.standard_normal((T, H)))         # signed weights
    pos = np.array([10, 30, 50, 79, 200], dtype=np.int32)
    sc = o.indexer_score(q, w, k, pos, ratio)
    qf, kf, wf = _f16_val(q), _f16_val(k), _f16_val(w)
    ref = np.einsum("th,ths->ts", wf, np.maximum(np.einsum("thd,sd->ths", qf, kf), 0.0))
    for t in range(T):
        n = min(S, (int(pos[t]) + 1) // ratio)
        assert np.allclose(sc[t, :n], ref[t, :n], rtol=2e-7, atol=1e-12)
        assert np.all(np.isneginf(sc[t, n:]))


# --------------------------------------------------------------------------- top-k
def check_topk_brute_force(o):
    rng = np.random.default_rng(5)
    for trial in range(12):
        T = 6
        S = int(rng.integers(1, 60))
        ratio = int(rng.choice([1, 2, 4]))
        k_top = int(rng.choice([1, 2, 5, 8, 16]))
        # few distinct values -> many ties
        sc = rng.integers(-4, 5, size=(T, S)).astype(np.float32) * 0.5
        pos = rng.integers(0, S * ratio + 5, size=T).astype(np.int32)
        idx, cnt = o.topk(sc, pos, S, ratio, k_top)
        for t in range(T):
            n = min(S, (int(pos[t]) + 1) // ratio)
            want = _brute_topk(list(sc[t]), n, k_top)
            assert list(idx[t]) == want, (trial, t, list(idx[t]), want)
            assert cnt[t] == min(n, k_top)


def check_topk_invariants(o):
    wl = synth.WORKLOADS["tiny_exact"]
    inp = synth.make_inputs(wl, seed=0, T=24)
    sc = o.indexer_score(inp.q, inp.w, inp.k, inp.positions, wl.ratio, S=wl.S)
    idx, cnt = o.topk(sc, inp.positions, wl.S, wl.ratio, wl.k_top)
    for t in range(idx.shape[0]):
        n = min(wl.S, (int(inp.positions[t]) + 1) // wl.ratio)
        sel = idx[t][idx[t] >= 0]
        assert len(sel) == min(n, wl.k_top) == cnt[t]
        assert np.all(np.diff(sel) > 0)                      # ascending, distinct
        assert np.all(sel < n)                               # masked rows never chosen
        if n > wl.k_top:
            chosen = np.zeros(n, dtype=bool)
            chosen[sel] = True
            lo = sc[t, :n][chosen].min()
            hi = sc[t, :n][~chosen].max()
            assert lo >= hi                                  # dominance
            if lo == hi:                                     # ties go to the lower row
                assert np.nonzero(chosen & (sc[t, :n] == lo))[0].max() < \
                    np.nonzero(~chosen & (sc[t, :n] == hi))[0].min()


def check_shortcut(o):
    S, ratio, k_top = 600, 1, 512
    rng = np.random.default_rng(9)
    sc = rng.standard_normal((8, S)).astype(np.float32)
    pos = np.array([0, 1, 2, 100, 510, 511, 512, 599], dtype=np.int32)  # n = 1,2,3,101,511,512,513,600
    a, ca = o.topk(sc, pos, S, ratio, k_top, shortcut=True)
    b, cb = o.topk(sc, pos, S, ratio, k_top, shortcut=False)
    for t in range(8):
        n = min(S, int(pos[t]) + 1)
        if n <= k_top:
            assert list(a[t]) == list(range(n)) + [-1] * (k_top - n)
    assert np.array_equal(a, b) and np.array_equal(ca, cb)
    # a token that sees nothing
    z, cz = o.topk(sc[:1], np.array([-1], dtype=np.int32), S, ratio, k_top)
    assert np.all(z == -1) and cz[0] == 0


# ----------------------------------------------------------------------- attention
def check_attn_zero_query_is_mean(o):
    rng = np.random.default_rng(1)
    S, Dkv, Hq = 40, 16, 3
    kv = synth.to_bf16_bits(rng.standard_normal((S, Dkv)))
    qa = np.zeros((2, Hq, Dkv), dtype=np.uint16)           # +0.0 bits
    ind = np.array([[3, 7, 11, 20, 39, -1], [0, 1, 2, 5, 8, 13]], dtype=np.int32)
    out, lse = o.sparse_attn(qa, kv, "bf16", ind, S, 0.3)
    kvf = _bits_val(kv, "bf16")
    for t in range(2):
        rows = [i for i in ind[t] if i >= 0]
        # equal logits -> equal weights: the exact rational mean, rounded to nearest even
        mean = [_rne_fraction(sum(Fraction(float(v)) for v in kvf[rows, d]) / len(rows), 7, 8)
                for d in range(Dkv)]
        for h in range(Hq):
            got = _bits_val(out[t, h], "bf16")
            assert all(Fraction(float(g)) == m for g, m in zip(got, mean)), (got, mean)
            assert abs(lse[t, h] - math.log(len(rows))) < 1e-6


def check_attn_single_row(o):
    rng = np.random.default_rng(2)
    S, Dkv, Hq = 10, 32, 4
    kv = synth.to_f16_bits(rng.standard_normal((S, Dkv)))
    qa = synth.to_f16_bits(rng.standard_normal((3, Hq, Dkv)))
    ind = np.array([[4, -1, -1], [-1, 9, -1], [-1, -1, 0]], dtype=np.int32)
    out, lse = o.sparse_attn(qa, kv, "f16", ind, S, 0.125)
    for t, r in enumerate([4, 9, 0]):
        for h in range(Hq):
            assert np.array_equal(out[t, h], kv[r])          # softmax of one logit is 1
            logit = 0.125 * float(np.dot(_f16_val(qa[t, h]), _f16_val(kv[r])))
            assert abs(lse[t, h] - logit) <= 1e-6 * max(1.0, abs(logit))


def check_attn_two_rows_logistic(o):
    # rows e0 and e1, q = [a, b]: p1 = 1/(1 + exp(-(b-a)*scale)), out = [1-p1, p1]
    S, Dkv = 2, 8
    kv = np.zeros((S, Dkv)); kv[0, 0] = 1; kv[1, 1] = 1
    cases = [(0.0, 1.0), (2.0, -1.0), (0.5, 0.5), (-3.0, 4.0)]
    qa = np.zeros((len(cases), 1, Dkv))
    for i, (a, b) in enumerate(cases):
        qa[i, 0, 0], qa[i, 0, 1] = a, b
    ind = np.array([[0, 1]] * len(cases), dtype=np.int32)
    out, lse = o.sparse_attn(_f16(qa), _f16(kv), "f16", ind, S, 0.75)
    for i, (a, b) in enumerate(cases):
        p1 = 1.0 / (1.0 + math.exp(-(b - a) * 0.75))
        want = np.zeros(Dkv); want[0], want[1] = 1 - p1, p1
        assert np.array_equal(out[i, 0], _f16(want)), (out[i, 0], want)
        assert abs(lse[i, 0] - math.log(math.exp(0.75 * a) + math.exp(0.75 * b))) < 1e-6


def check_attn_vs_textbook(o):
    rng = np.random.default_rng(4)
    S, Dkv, Hq, T, k_top = 50, 64, 8, 3, 12
    kv = synth.to_bf16_bits(rng.standard_normal((S, Dkv)))
    qa = synth.to_bf16_bits(rng.standard_normal((T, Hq, Dkv)))
    ind = np.stack([rng.choice(S, k_top, replace=False) for _ in range(T)]).astype(np.int32)
    ind[1, -3:] = -1
    ind[2, 0] = S + 5                                        # out of range -> skipped
    scale = 1.0 / math.sqrt(Dkv)
    out, lse = o.sparse_attn(qa, kv, "bf16", ind, S, scale)
    kvf, qf = _bits_val(kv, "bf16"), _bits_val(qa, "bf16")
    for t in range(T):
        rows = [int(i) for i in ind[t] if 0 <= i < S]
        V = kvf[rows]
        logits = scale * qf[t] @ V.T                         # [Hq, n]
        m = logits.max(axis=1, keepdims=True)
        p = np.exp(logits - m)
        ref = (p / p.sum(axis=1, keepdims=True)) @ V
        assert np.allclose(_bits_val(out[t], "bf16"), ref, rtol=2 ** -8, atol=1e-6)
        assert np.allclose(lse[t], (m[:, 0] + np.log(p.sum(axis=1))), rtol=1e-6, atol=1e-6)


def check_index_and_attend_composes(o):
    wl = synth.WORKLOADS["tiny_exact"]
    inp = synth.make_inputs(wl, seed=0, T=6, S=1024)
    # include tokens that take the shortcut (positions below k_top*ratio)
    pos = np.array([5, 2047, 2048, 2051, 4000, 4095], dtype=np.int32)
    idx, out, lse = o.index_and_attend(inp.q, inp.w, inp.k, pos, inp.q_attn, inp.kv, "f16",
                                       wl.S, wl.ratio, wl.k_top, wl.scale)
    sc = o.indexer_score(inp.q, inp.w, inp.k, pos, wl.ratio, S=wl.S)
    idx2, _ = o.topk(sc, pos, wl.S, wl.ratio, wl.k_top)
    out2, lse2 = o.sparse_attn(inp.q_attn, inp.kv, "f16", idx2, wl.S, wl.scale)
    assert np.array_equal(idx, idx2)
    assert np.array_equal(out, out2) and np.array_equal(lse, lse2)


def decode_rows_closed_form(S0, capacity, n_new, pos0, ratio, n_steps):
    """Rows present at each decode step: the visible count floor((p+1)/ratio), never below S0,
    capped by the staged rows and the capacity."""
    return [min(S0 + n_new, capacity, max(S0, (pos0 + i + 1) // ratio)) for i in range(n_steps)]


def _tiny_decode_case(seed=7):
    rng = np.random.default_rng(seed)
    capacity, S0, n_new, H, D, Hq, Dkv = 40, 30, 3, 4, 16, 4, 32
    k = _f16(rng.standard_normal((capacity, D)))
    kv = synth.to_bf16_bits(rng.standard_normal((capacity, Dkv)))
    k[S0:] = 0
    kv[S0:] = 0
    k_new = _f16(rng.standard_normal((n_new, D)))
    kv_new = synth.to_bf16_bits(rng.standard_normal((n_new, Dkv)))
    n_steps = 10
    q = _f16(rng.standard_normal((n_steps, H, D)))
    w = _f16(rng.uniform(0.0, 1.0, (n_steps, H)) / 8)
    qa = synth.to_bf16_bits(rng.standard_normal((n_steps, Hq, Dkv)))
    return dict(k=k, kv=kv, k_new=k_new, kv_new=kv_new, q=q, w=w, qa=qa, S0=S0, pos0=59, ratio=2,
                k_top=8, n_steps=n_steps, capacity=capacity, n_new=n_new)


def check_decode_schedule(o):
    c = _tiny_decode_case()
    idx, out, lse, pos, s_steps, k_after, kv_after = o.decode(
        c["q"], c["w"], c["qa"], c["k"], c["kv"], "bf16", c["S0"], c["pos0"], c["ratio"], c["k_new"],
        c["kv_new"], c["k_top"], 0.25)
    assert list(pos) == [c["pos0"] + i for i in range(c["n_steps"])]
    want = decode_rows_closed_form(c["S0"], c["capacity"], c["n_new"], c["pos0"], c["ratio"], c["n_steps"])
    assert list(s_steps) == want, (list(s_steps), want)
    # appended rows carry the staged bytes, in order; rows before S0 and after are untouched
    S = int(s_steps[-1])
    assert np.array_equal(k_after[c["S0"]:S], c["k_new"][:S - c["S0"]])
    assert np.array_equal(kv_after[c["S0"]:S], c["kv_new"][:S - c["S0"]])
    assert np.array_equal(k_after[:c["S0"]], c["k"][:c["S0"]]) and not k_after[S:].any()
    # the 1M-context decode: 63 rows appended over 256 steps from position 1048575
    assert decode_rows_closed_form(262144, 262208, 64, 1048575, 4, 256)[-1] - 262144 == 63


def check_decode_steps_brute_force(o):
    c = _tiny_decode_case()
    scale = 0.25
    idx, out, lse, pos, s_steps, k_after, _ = o.decode(
        c["q"], c["w"], c["qa"], c["k"], c["kv"], "bf16", c["S0"], c["pos0"], c["ratio"], c["k_new"],
        c["kv_new"], c["k_top"], scale)
    rows_k = np.concatenate([c["k"][:c["S0"]], c["k_new"]])
    rows_kv = np.concatenate([c["kv"][:c["S0"]], c["kv_new"]])
    kf, kvf = _f16_val(rows_k), _bits_val(rows_kv, "bf16")
    for i in range(c["n_steps"]):
        p = c["pos0"] + i
        S = min(c["S0"] + c["n_new"], max(c["S0"], (p + 1) // c["ratio"]))
        n = min(S, (p + 1) // c["ratio"])
        qf, wf = _f16_val(c["q"][i]), _f16_val(c["w"][i])
        dots = qf @ kf[:n].T                                  # [H, n]
        score = (wf[:, None] * np.maximum(dots, 0.0)).sum(axis=0).astype(np.float32)
        ranked = sorted(range(n), key=lambda s_: (-float(score[s_]), s_))[:c["k_top"]]
        sel = sorted(ranked) + [-1] * (c["k_top"] - min(n, c["k_top"]))
        assert list(idx[i]) == sel, (i, list(idx[i]), sel)
        V = kvf[sorted(ranked)]
        logits = scale * _bits_val(c["qa"][i], "bf16") @ V.T
        m = logits.max(axis=1, keepdims=True)
        pr = np.exp(logits - m)
        ref = (pr / pr.sum(axis=1, keepdims=True)) @ V
        assert np.allclose(_bits_val(out[i], "bf16"), ref, rtol=2 ** -8, atol=1e-6)
        assert np.allclose(lse[i], m[:, 0] + np.log(pr.sum(axis=1)), rtol=1e-6, atol=1e-6)


# ------------------------------------------------------------ local-plus-pooled attention
def _softmax_rows(qf, V, scale):
    """Textbook float64 softmax attention of the heads qf [Hq, Dkv] over the rows V [n, Dkv]."""
    logits = scale * qf @ V.T
    m = logits.max(axis=1, keepdims=True)
    p = np.exp(logits - m)
    return (p / p.sum(axis=1, keepdims=True)) @ V, m[:, 0] + np.log(p.sum(axis=1))


def _raw_window(p, W, local_pos0, L):
    """Positions of the raw rows a token at p attends: p-W < a <= p, a >= 0, held by the buffer."""
    return [a for a in range(p - W + 1, p + 1) if a >= 0 and local_pos0 <= a < local_pos0 + L]


def check_local_only_vs_textbook(o):
    # no pooled row at all: causal sliding-window attention over a raw sequence X, of which the
    # buffer holds positions 6..19; tokens before, inside and after the buffer, and p < 0
    rng = np.random.default_rng(11)
    N, Dkv, Hq, W, lp0, L = 24, 32, 4, 5, 6, 14
    X = synth.to_bf16_bits(rng.standard_normal((N, Dkv)))
    pos = np.array([0, 3, 6, 8, 10, 13, 19, 21, 30, -2], dtype=np.int32)
    T = len(pos)
    qa = synth.to_bf16_bits(rng.standard_normal((T, Hq, Dkv)))
    ind = np.full((T, 4), -1, dtype=np.int32)
    scale = 0.3
    out, lse = o.local_pooled_attn(qa, X, X[lp0:lp0 + L], "bf16", ind, pos, 2, lp0, W, scale)
    Xf = _bits_val(X, "bf16")
    for t, p in enumerate(pos):
        rows = [a for a in range(max(0, p - W + 1, lp0), min(p, lp0 + L - 1) + 1)]
        assert rows == _raw_window(int(p), W, lp0, L)
        if not rows:
            assert np.all(out[t] == 0) and np.all(np.isneginf(lse[t])), (t, p)
            continue
        if len(rows) == 1:                                   # one row: softmax weight exactly 1
            assert all(np.array_equal(out[t, h], X[rows[0]]) for h in range(Hq))
        ref, rlse = _softmax_rows(_bits_val(qa[t], "bf16"), Xf[rows], scale)
        assert np.allclose(_bits_val(out[t], "bf16"), ref, rtol=2 ** -8, atol=1e-6), (t, p)
        assert np.allclose(lse[t], rlse, rtol=1e-6, atol=1e-6)


def _union_case(seed, dtype):
    rng = np.random.default_rng(seed)
    S, N, Dkv, Hq, W, lp0, k_top = 30, 40, 32, 4, 7, 9, 6
    L = 25                                                   # raw positions 9..33
    kv = synth.to_bits(rng.standard_normal((S, Dkv)), dtype)
    X = synth.to_bits(rng.standard_normal((N, Dkv)), dtype)
    pos = np.array([9, 12, 20, 33, 36, 5], dtype=np.int32)
    T = len(pos)
    qa = synth.to_bits(rng.standard_normal((T, Hq, Dkv)), dtype)
    ind = np.stack([rng.choice(S, k_top, replace=False) for _ in range(T)]).astype(np.int32)
    ind[1, -2:] = -1
    ind[2, 0] = S + 3                                        # out of range -> skipped
    ind[4, :] = -1                                           # window rows only
    return dict(S=S, W=W, lp0=lp0, L=L, kv=kv, X=X, kv_local=X[lp0:lp0 + L], pos=pos, qa=qa, ind=ind)


def check_local_pooled_union_vs_textbook(o):
    c = _union_case(12, "bf16")
    scale = 1.0 / math.sqrt(32)
    out, lse = o.local_pooled_attn(c["qa"], c["kv"], c["kv_local"], "bf16", c["ind"], c["pos"], c["S"],
                                   c["lp0"], c["W"], scale)
    kvf, Xf = _bits_val(c["kv"], "bf16"), _bits_val(c["X"], "bf16")
    for t, p in enumerate(c["pos"]):
        pooled = [int(i) for i in c["ind"][t] if 0 <= i < c["S"]]
        raw = _raw_window(int(p), c["W"], c["lp0"], c["L"])
        V = np.concatenate([kvf[pooled], Xf[raw]])
        ref, rlse = _softmax_rows(_bits_val(c["qa"][t], "bf16"), V, scale)
        assert np.allclose(_bits_val(out[t], "bf16"), ref, rtol=2 ** -8, atol=1e-6), t
        assert np.allclose(lse[t], rlse, rtol=1e-6, atol=1e-6), t


def check_local_pooled_lse_merge(o):
    # softmax over a union = the two one-source results weighted by exp(lse_i - lse):
    #   lse = log(e^lse_p + e^lse_l),  out = e^(lse_p - lse) out_p + e^(lse_l - lse) out_l
    c = _union_case(13, "f16")
    scale = 0.2
    T = len(c["pos"])
    out, lse = o.local_pooled_attn(c["qa"], c["kv"], c["kv_local"], "f16", c["ind"], c["pos"], c["S"],
                                   c["lp0"], c["W"], scale)
    out_p, lse_p = o.sparse_attn(c["qa"], c["kv"], "f16", c["ind"], c["S"], scale)
    none = np.full_like(c["ind"], -1)
    out_l, lse_l = o.local_pooled_attn(c["qa"], c["kv"], c["kv_local"], "f16", none, c["pos"], c["S"],
                                       c["lp0"], c["W"], scale)
    lp, ll = lse_p.astype(np.float64), lse_l.astype(np.float64)
    merged_lse = np.logaddexp(lp, ll)
    assert np.allclose(lse, merged_lse, rtol=1e-6, atol=1e-6)
    wp = np.exp(lp - merged_lse)[..., None]
    wl = np.exp(ll - merged_lse)[..., None]
    op, ol = _bits_val(out_p, "f16"), _bits_val(out_l, "f16")
    merged = wp * op + wl * ol
    got = _bits_val(out, "f16")
    # every output carries one f16 rounding (2^-11 relative, 2^-25 absolute below the normal
    # range) and the lse values are fp32 (the weights then err by ~1e-6 relative)
    bound = (2 ** -11 * (wp * np.abs(op) + wl * np.abs(ol) + np.abs(got)) + 1e-5 * (np.abs(op) + np.abs(ol))
             + 2 ** -24)
    assert np.all(np.abs(got - merged) <= bound), np.abs(got - merged).max()
    assert T == out.shape[0]


def check_local_zero_query_is_mean(o):
    # equal logits: the output is the exact rational mean of every pooled and raw row, rounded once
    c = _union_case(14, "bf16")
    qa = np.zeros_like(c["qa"])
    out, lse = o.local_pooled_attn(qa, c["kv"], c["kv_local"], "bf16", c["ind"], c["pos"], c["S"],
                                   c["lp0"], c["W"], 0.5)
    kvf, Xf = _bits_val(c["kv"], "bf16"), _bits_val(c["X"], "bf16")
    for t, p in enumerate(c["pos"]):
        rows = [kvf[int(i)] for i in c["ind"][t] if 0 <= i < c["S"]]
        rows += [Xf[a] for a in _raw_window(int(p), c["W"], c["lp0"], c["L"])]
        n = len(rows)
        mean = [_rne_fraction(sum(Fraction(float(r[d])) for r in rows) / n, 7, 8) for d in range(len(rows[0]))]
        for h in range(qa.shape[1]):
            got = _bits_val(out[t, h], "bf16")
            assert all(Fraction(float(g)) == m for g, m in zip(got, mean)), (t, h)
            assert abs(lse[t, h] - math.log(n)) < 1e-6


def check_local_window_off_is_sparse_attn(o):
    # no raw row in reach (window 0, an empty buffer, a buffer past every token): the pooled
    # result, bit for bit
    c = _union_case(15, "bf16")
    ref = o.sparse_attn(c["qa"], c["kv"], "bf16", c["ind"], c["S"], 0.25)
    for kv_local, lp0, W in ((c["kv_local"], c["lp0"], 0), (c["kv_local"][:0], c["lp0"], 7),
                             (c["kv_local"], 1000, 7)):
        got = o.local_pooled_attn(c["qa"], c["kv"], kv_local, "bf16", c["ind"], c["pos"], c["S"], lp0, W, 0.25)
        assert np.array_equal(got[0], ref[0]) and np.array_equal(got[1], ref[1])


def check_index_and_attend_local_composes(o):
    wl = synth.WORKLOADS["tiny_exact"]
    inp = synth.make_inputs(wl, seed=0, T=6, S=1024)
    pos = np.array([5, 2047, 2048, 2051, 4000, 4095], dtype=np.int32)
    rng = np.random.default_rng(16)
    lp0, L, W = 1990, 2106, 64
    kv_local = synth.to_f16_bits(rng.integers(-2, 3, size=(L, wl.Dkv)).astype(np.float64))
    idx, out, lse = o.index_and_attend_local(inp.q, inp.w, inp.k, pos, inp.q_attn, inp.kv, kv_local, "f16",
                                             wl.S, wl.ratio, wl.k_top, lp0, W, wl.scale)
    idx2, _, _ = o.index_and_attend(inp.q, inp.w, inp.k, pos, inp.q_attn, inp.kv, "f16", wl.S, wl.ratio,
                                    wl.k_top, wl.scale)
    out2, lse2 = o.local_pooled_attn(inp.q_attn, inp.kv, kv_local, "f16", idx2, pos, wl.S, lp0, W, wl.scale)
    assert np.array_equal(idx, idx2)
    assert np.array_equal(out, out2) and np.array_equal(lse, lse2)


# ----------------------------------------------------------------------------- compressor
def _softmax_pool_numpy(seq_x, seq_g, bias, ratio, dtype):
    """Textbook float64 gated pooling of whole blocks of the sequence rows."""
    xf, gf = _bits_val(seq_x, dtype), _bits_val(seq_g, dtype)
    n_out = xf.shape[0] // ratio
    out = np.empty((n_out, xf.shape[1]))
    for j in range(n_out):
        z = gf[j * ratio:(j + 1) * ratio] + bias.astype(np.float64)      # [ratio, D]
        a = np.exp(z - z.max(axis=0))
        out[j] = (a * xf[j * ratio:(j + 1) * ratio]).sum(axis=0) / a.sum(axis=0)
    return out


def check_compress_equal_gates_is_mean(o):
    # equal gates: every block row is the exact rational mean of its positions, rounded once;
    # a 3-position frontier at ratio 4 puts the first block across the call boundary
    rng = np.random.default_rng(21)
    ratio, D, T, f = 4, 24, 13, 3
    xs = synth.to_bf16_bits(rng.standard_normal((f + T, D)))
    g = np.full((f + T, D), synth.to_bf16_bits(np.array([0.75]))[0], dtype=np.uint16)
    bias = np.zeros((ratio, D), np.float32)
    rows, fx, fg = o.compress(xs[f:], g[f:], bias, "bf16", ratio, xs[:f], g[:f])
    assert rows.shape == (4, D) and fx.shape == (0, D)
    xv = _bits_val(xs, "bf16")
    for j in range(4):
        for d in range(D):
            mean = sum(Fraction(float(v)) for v in xv[j * ratio:(j + 1) * ratio, d]) / ratio
            assert Fraction(float(_bits_val(rows[j:j + 1, d], "bf16")[0])) == _rne_fraction(mean, 7, 8), (j, d)


def check_compress_dominant_gate_selects_row(o):
    # one position's gate 100 above the others: its weight is 1 to far below rounding
    rng = np.random.default_rng(22)
    ratio, D, T = 8, 16, 40
    x = synth.to_f16_bits(rng.standard_normal((T, D)))
    gv = np.zeros((T, D))
    pick = rng.integers(0, ratio, size=(T // ratio, D))
    for j in range(T // ratio):
        gv[j * ratio + pick[j], np.arange(D)] = 100.0
    rows, _, _ = o.compress(x, synth.to_f16_bits(gv), np.zeros((ratio, D), np.float32), "f16", ratio)
    for j in range(T // ratio):
        assert np.array_equal(rows[j], x[j * ratio + pick[j], np.arange(D)]), j


def check_compress_vs_numpy(o):
    rng = np.random.default_rng(23)
    for dtype, ratio, D, T, f in (("bf16", 4, 32, 29, 2), ("f16", 16, 8, 50, 15), ("bf16", 128, 4, 300, 0)):
        xs = synth.to_bits(rng.standard_normal((f + T, D)), dtype)
        gs = synth.to_bits(2 * rng.standard_normal((f + T, D)), dtype)
        bias = rng.standard_normal((ratio, D)).astype(np.float32)
        rows, fx, fg = o.compress(xs[f:], gs[f:], bias, dtype, ratio, xs[:f] if f else None, gs[:f] if f else None)
        ref = _softmax_pool_numpy(xs, gs, bias, ratio, dtype)
        got = _bits_val(rows, dtype)
        ulp = 2.0 ** (-8 if dtype == "bf16" else -11)
        assert np.all(np.abs(got - ref) <= ulp * np.abs(ref) + 1e-7), (dtype, ratio, np.abs(got - ref).max())
        rem = (f + T) % ratio
        assert np.array_equal(fx, xs[f + T - rem:]) and np.array_equal(fg, gs[f + T - rem:])


def check_compress_split_calls_equal_one(o):
    # compressing a sequence in one call equals any split into two calls with the frontier carried
    rng = np.random.default_rng(24)
    ratio, D, N = 4, 12, 37
    xs = synth.to_bf16_bits(rng.standard_normal((N, D)))
    gs = synth.to_bf16_bits(rng.standard_normal((N, D)))
    bias = rng.standard_normal((ratio, D)).astype(np.float32)
    whole, wfx, wfg = o.compress(xs, gs, bias, "bf16", ratio)
    for cut in (0, 1, 3, 4, 5, 18, 36, 37):
        r1, fx, fg = o.compress(xs[:cut], gs[:cut], bias, "bf16", ratio)
        r2, fx2, fg2 = o.compress(xs[cut:], gs[cut:], bias, "bf16", ratio, fx, fg)
        assert np.array_equal(np.concatenate([r1, r2]), whole), cut
        assert np.array_equal(fx2, wfx) and np.array_equal(fg2, wfg), cut


def _tiny_decode_local_case(seed=8):
    c = _tiny_decode_case(seed)
    rng = np.random.default_rng(seed + 100)
    raw_cap = c["pos0"] + c["n_steps"] + 3
    kv_raw = synth.to_bf16_bits(rng.standard_normal((raw_cap, c["kv"].shape[1])))   # history below pos0
    kv_raw_new = synth.to_bf16_bits(rng.standard_normal((c["n_steps"], c["kv"].shape[1])))
    c.update(kv_raw=kv_raw, kv_raw_new=kv_raw_new, window=5)
    return c


def check_decode_local_window_off(o):
    # window 0: the plain decode loop, bit for bit
    c = _tiny_decode_local_case()
    a = o.decode(c["q"], c["w"], c["qa"], c["k"], c["kv"], "bf16", c["S0"], c["pos0"], c["ratio"], c["k_new"],
                 c["kv_new"], c["k_top"], 0.25)
    b = o.decode_local(c["q"], c["w"], c["qa"], c["k"], c["kv"], "bf16", c["S0"], c["pos0"], c["ratio"], c["k_new"],
                       c["kv_new"], c["k_top"], 0.25, c["kv_raw"], c["kv_raw_new"], 0)
    for x, y in zip(a[:5], b[:5]):
        assert np.array_equal(x, y)


def check_decode_local_steps_brute_force(o):
    # each step against numpy: the definition score, sorted() ranking, and a textbook softmax over
    # the selected pooled rows together with the raw rows of the step's last `window` positions
    c = _tiny_decode_local_case()
    scale, W = 0.25, c["window"]
    idx, out, lse, pos, s_steps, _, _, raw_after = o.decode_local(
        c["q"], c["w"], c["qa"], c["k"], c["kv"], "bf16", c["S0"], c["pos0"], c["ratio"], c["k_new"], c["kv_new"],
        c["k_top"], scale, c["kv_raw"], c["kv_raw_new"], W)
    p0, n = c["pos0"], c["n_steps"]
    assert np.array_equal(raw_after[p0:p0 + n], c["kv_raw_new"])          # the steps' raw rows in place
    assert np.array_equal(raw_after[:p0], c["kv_raw"][:p0])               # the history untouched
    rows_k = np.concatenate([c["k"][:c["S0"]], c["k_new"]])
    rows_kv = np.concatenate([c["kv"][:c["S0"]], c["kv_new"]])
    kf, kvf, rawf = _f16_val(rows_k), _bits_val(rows_kv, "bf16"), _bits_val(raw_after, "bf16")
    for i in range(n):
        p = p0 + i
        S = min(c["S0"] + c["n_new"], max(c["S0"], (p + 1) // c["ratio"]))
        nv = min(S, (p + 1) // c["ratio"])
        qf, wf = _f16_val(c["q"][i]), _f16_val(c["w"][i])
        score = (wf[:, None] * np.maximum(qf @ kf[:nv].T, 0.0)).sum(axis=0).astype(np.float32)
        ranked = sorted(sorted(range(nv), key=lambda s_: (-float(score[s_]), s_))[:c["k_top"]])
        assert list(idx[i]) == ranked + [-1] * (c["k_top"] - len(ranked)), i
        V = np.concatenate([kvf[ranked], rawf[max(0, p - W + 1):p + 1]])
        ref, rlse = _softmax_rows(_bits_val(c["qa"][i], "bf16"), V, scale)
        assert np.allclose(_bits_val(out[i], "bf16"), ref, rtol=2 ** -8, atol=1e-6), i
        assert np.allclose(lse[i], rlse, rtol=1e-6, atol=1e-6), i


ALL_CHECKS = [
    check_f16_decode_exhaustive, check_bf16_decode_exhaustive, check_encode_rne,
    check_visibility, check_golden_example, check_scores_int64_closed_form,
    check_scores_float_vs_numpy, check_topk_brute_force, check_topk_invariants,
    check_shortcut, check_attn_zero_query_is_mean, check_attn_single_row,
    check_attn_two_rows_logistic, check_attn_vs_textbook, check_index_and_attend_composes,
    check_decode_schedule, check_decode_steps_brute_force, check_local_only_vs_textbook,
    check_local_pooled_union_vs_textbook, check_local_pooled_lse_merge, check_local_zero_query_is_mean,
    check_local_window_off_is_sparse_attn, check_index_and_attend_local_composes,
    check_compress_equal_gates_is_mean, check_compress_dominant_gate_selects_row, check_compress_vs_numpy,
    check_compress_split_calls_equal_one, check_decode_local_window_off, check_decode_local_steps_brute_force,
]
