"""ds4x_topk_static_scratch: top-k for callers that cannot allocate device memory.

Some callers of this library may not allocate device memory while they run — a serving
process that handed all of HBM to its KV cache at start-up, or a plugin inside a host framework
that owns the allocator — so they cannot give ds4x_topk the workspace its split mode needs.
The allocation-free variant keeps that scratch in a fixed array inside the library. These tests
call it through the C ABI and require the same indices and counts as ds4x_topk and as the CPU
oracle's top-k on the same fp32 scores (top-k results are compared bit for bit everywhere in this
suite), on two calls in a row, since every call reuses the same array.
"""
import ctypes

import numpy as np
import pytest
import torch

import deepseek_v4_sparse_gb300 as ds4x
import oracle

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from deepseek_v4_sparse_gb300 import build
    build.build()
    lib = ds4x.load()
    P = ctypes.c_void_p
    i32 = ctypes.c_int32
    lib.ds4x_topk_static_scratch.argtypes = [P, ctypes.c_int64, P, i32, i32, i32, i32, P, P, P]
    lib.ds4x_topk_static_scratch.restype = ctypes.c_int
    return lib


def _p(t):
    return ctypes.c_void_p(t.data_ptr()) if t is not None else None


def static_topk(lib, scores, positions, S, ratio, k_top):
    T = scores.shape[0]
    idx = torch.full((T, k_top), -7, dtype=torch.int32, device="cuda")
    cnt = torch.full((T,), -7, dtype=torch.int32, device="cuda")
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    rc = lib.ds4x_topk_static_scratch(_p(scores), scores.shape[1], _p(positions), T, S, ratio, k_top,
                                      _p(idx), _p(cnt), stream)
    assert rc == ds4x.OK, ds4x.status_string(rc)
    return idx, cnt


def workspace_topk(scores, positions, S, ratio, k_top):
    return ds4x.topk(scores, positions, S, ratio, k_top)


@pytest.mark.parametrize("T,S,ratio", [(1, 262144 + 37, 4), (3, 70000, 1), (200, 4096, 4)])
def test_matches_workspace_entry_on_two_calls(lib, T, S, ratio):
    rng = np.random.default_rng(T * 1000 + S)
    # the first two cases split each row over many CTAs (the mode whose scratch is the fixed
    # array): one cooperative launch, or three launches where it cannot be resident at once
    split = ds4x.topk_workspace_bytes(T, S, 512) > 0
    assert split == (T < 100), "the cases are chosen to cover both modes"
    for call in range(2):
        scores = rng.standard_normal((T, S)).astype(np.float32)
        if call == 1:
            scores[:, 100:400] = scores[0, 100]               # exact ties on the second call
        pos = (S * ratio - 1 - rng.integers(0, 5 * ratio, size=T)).astype(np.int32)
        pos[0] = S * ratio + 11                               # one token sees every row
        d_scores = torch.from_numpy(scores).cuda()
        d_pos = torch.from_numpy(pos).cuda()
        a_idx, a_cnt = static_topk(lib, d_scores, d_pos, S, ratio, 512)
        launches = ds4x.last_launch_count()
        assert launches in ((1, 3) if split else (1,)), f"call {call}: {launches} launches"
        b_idx, b_cnt = workspace_topk(d_scores, d_pos, S, ratio, 512)
        torch.cuda.synchronize()
        assert torch.equal(a_idx, b_idx), f"call {call}: indices differ from ds4x_topk"
        assert torch.equal(a_cnt, b_cnt), f"call {call}: counts differ from ds4x_topk"
        r_idx, r_cnt = oracle.topk(scores, pos, S, ratio, 512)
        assert np.array_equal(a_idx.cpu().numpy(), r_idx), f"call {call}: indices differ from the oracle"
        assert np.array_equal(a_cnt.cpu().numpy(), r_cnt), f"call {call}: counts differ from the oracle"
    assert ds4x.device_status() == ds4x.OK


def test_rejects_requests_beyond_the_fixed_array(lib):
    T, S, k_top = 100, 262144, 512
    need = ds4x.topk_workspace_bytes(T, S, k_top)
    assert need > ds4x.TOPK_STATIC_SCRATCH_BYTES
    scores = torch.zeros((T, S), dtype=torch.float32, device="cuda")
    pos = torch.full((T,), 4 * S, dtype=torch.int32, device="cuda")
    idx = torch.full((T, k_top), -7, dtype=torch.int32, device="cuda")
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    rc = lib.ds4x_topk_static_scratch(_p(scores), S, _p(pos), T, S, 4, k_top, _p(idx), None, stream)
    assert rc == ds4x.ERR_WORKSPACE
    torch.cuda.synchronize()
    assert bool((idx == -7).all()), "a rejected call must not touch its outputs"
