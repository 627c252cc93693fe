"""Helpers shared by the GPU parity tests: host<->device marshalling of the synthetic
inputs and the tolerance rules.

Tolerances (from the path's definition of acceptable error):
  * exact-integer inputs: scores and indices bit-exact;
  * N(0,1) inputs: |s_gpu - s_ref| <= 1e-3*|s_ref| + 1e-6 on visible scores, masked entries
    exactly -inf; index sets may differ only in rows whose oracle score lies within
    1e-3*|s_k| of the oracle's k-th score s_k;
  * attention: |o_gpu - o_ref| <= 2e-3 + 1e-2*|o_ref|, with the GPU's own indices fed to
    the oracle so that selection and attention errors stay separate.
"""
import numpy as np
import torch

import synth

SCORE_RTOL, SCORE_ATOL = 1e-3, 1e-6
ATTN_ATOL, ATTN_RTOL = 2e-3, 1e-2


def dev16(a: np.ndarray, dtype: str, device="cuda"):
    t = torch.from_numpy(np.ascontiguousarray(a).view(np.int16).copy())
    return t.view(torch.float16 if dtype == "f16" else torch.bfloat16).to(device)


def host16(t) -> np.ndarray:
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def to_device(inp):
    kvd = inp.wl.kv_dtype
    return dict(q=dev16(inp.q, "f16"), w=dev16(inp.w, "f16"), k=dev16(inp.k, "f16"),
                q_attn=dev16(inp.q_attn, kvd), kv=dev16(inp.kv, kvd),
                positions=torch.from_numpy(inp.positions.copy()).cuda())


def n_vis(p, ratio, S):
    return 0 if p < 0 else min(S, (int(p) + 1) // ratio)


def check_scores(gpu: np.ndarray, ref: np.ndarray, positions, ratio, S, exact: bool):
    for t in range(gpu.shape[0]):
        n = n_vis(positions[t], ratio, S)
        assert np.all(np.isneginf(gpu[t, n:S])), f"token {t}: masked entries not -inf"
        g, r = gpu[t, :n].astype(np.float64), ref[t, :n].astype(np.float64)
        if exact:
            bad = np.nonzero(g != r)[0]
            assert bad.size == 0, f"token {t}: {bad.size} scores differ, first row {bad[0]}: {g[bad[0]]} vs {r[bad[0]]}"
        else:
            err = np.abs(g - r) - (SCORE_RTOL * np.abs(r) + SCORE_ATOL)
            assert err.max(initial=-1) <= 0, f"token {t}: score error {np.abs(g - r).max()} above tolerance"


def check_index_sets(gpu_idx: np.ndarray, ref_idx: np.ndarray, ref_scores: np.ndarray, positions, ratio, S,
                     k_top):
    """Selections must agree except for rows whose oracle score ties (within tolerance) the
    oracle's k-th score; each GPU row list must be valid (ascending, distinct, visible)."""
    for t in range(gpu_idx.shape[0]):
        n = n_vis(positions[t], ratio, S)
        g = gpu_idx[t]
        gs = g[g >= 0]
        assert len(gs) == min(n, k_top), f"token {t}: {len(gs)} rows selected"
        assert np.all(g[len(gs):] == -1)
        assert np.all(np.diff(gs) > 0) and (len(gs) == 0 or (gs[0] >= 0 and gs[-1] < n))
        rs = ref_idx[t][ref_idx[t] >= 0]
        diff = np.setxor1d(gs, rs)
        if diff.size == 0:
            continue
        row = ref_scores[t, :n].astype(np.float64)
        kth = np.sort(row)[::-1][k_top - 1]
        tol = 1e-3 * abs(kth) + 1e-6
        assert np.all(np.abs(row[diff] - kth) <= tol), \
            f"token {t}: rows {diff[:8]} differ beyond the tie tolerance of the k-th score {kth}"


def few_rows_bound(kv_bits: np.ndarray, indices: np.ndarray, ref_bits: np.ndarray, dtype: str, S: int):
    """Extra error allowed when a token has few valid rows (the configs' tokens all have 512).

    The probabilities enter the second product rounded to the kv dtype: p~ = p (1 + d),
    |d| <= u (u = 2^-9 for bf16, 2^-11 for fp16), and the sums use the same rounded values, so
    each normalised weight is off by at most 2u relative and
        |o_gpu - o_ref| <= 2u * sum_j w_j |v_j - o_ref| <= 2u * max_j |v_j - o_ref|.
    With hundreds of rows the rounding errors average out far below the spec tolerance; with
    a handful of rows and cancelling values they need not."""
    u = 2.0 ** -9 if dtype == "bf16" else 2.0 ** -11
    kv = synth.bits_to_f32(kv_bits, dtype).astype(np.float64)
    ref = synth.bits_to_f32(ref_bits, dtype).astype(np.float64)
    bound = np.zeros_like(ref)
    for t in range(ref.shape[0]):
        rows = [int(i) for i in indices[t] if 0 <= i < S]
        if rows:
            V = kv[rows]                                         # [n, Dkv]
            bound[t] = 2 * u * np.abs(V[None, :, :] - ref[t][:, None, :]).max(axis=1)
    return bound


def window_positions(p: int, window: int, local_pos0: int, L: int):
    """Raw positions a token at p attends in local-plus-pooled attention."""
    return [a for a in range(max(0, p - window + 1, local_pos0), min(p, local_pos0 + L - 1) + 1)]


def union_rows_bound(kv_bits, indices, S, kv_local_bits, positions, local_pos0, window, ref_bits, dtype):
    """few_rows_bound over the union of a token's pooled rows and its raw window rows."""
    u = 2.0 ** -9 if dtype == "bf16" else 2.0 ** -11
    kv = synth.bits_to_f32(kv_bits, dtype).astype(np.float64)
    kvl = synth.bits_to_f32(kv_local_bits, dtype).astype(np.float64)
    ref = synth.bits_to_f32(ref_bits, dtype).astype(np.float64)
    L = kvl.shape[0]
    bound = np.zeros_like(ref)
    for t in range(ref.shape[0]):
        rows = [kv[int(i)] for i in indices[t] if 0 <= i < S]
        rows += [kvl[a - local_pos0] for a in window_positions(int(positions[t]), window, local_pos0, L)]
        if rows:
            V = np.stack(rows)
            bound[t] = 2 * u * np.abs(V[None, :, :] - ref[t][:, None, :]).max(axis=1)
    return bound


def check_attn(gpu_bits: np.ndarray, ref_bits: np.ndarray, dtype: str, gpu_lse=None, ref_lse=None,
               extra=None):
    g = synth.bits_to_f32(gpu_bits, dtype).astype(np.float64)
    r = synth.bits_to_f32(ref_bits, dtype).astype(np.float64)
    assert np.all(np.isfinite(g)), "non-finite attention output"
    err = np.abs(g - r) - (ATTN_ATOL + ATTN_RTOL * np.abs(r) + (0.0 if extra is None else extra))
    worst = np.unravel_index(np.argmax(err), err.shape)
    assert err.max() <= 0, f"attention error {np.abs(g - r)[worst]} at {worst}: {g[worst]} vs {r[worst]}"
    if gpu_lse is not None:
        fin = np.isfinite(ref_lse)
        assert np.array_equal(np.isfinite(gpu_lse), fin)
        # lse = m + log(sum of the rounded probabilities), consistent with the normalisation of
        # out; with few rows the rounding (<= u relative per term) can move it by up to ~2u
        lse_atol = 1e-4 + (0.0 if extra is None else 2.0 ** -8)
        lerr = np.abs(gpu_lse[fin] - ref_lse[fin])
        assert np.all(lerr <= lse_atol + 1e-4 * np.abs(ref_lse[fin])), f"lse error {lerr.max()}"
