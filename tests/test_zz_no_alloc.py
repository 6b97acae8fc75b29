"""The no-allocation entry point lmhead_two_stage_local_noalloc, through the
C ABI, against lmhead_two_stage on the same inputs.

Some callers cannot allocate device memory at call time (a serving engine
that has given all free HBM to its KV-cache pool, or C code without a device
allocator), so this variant keeps its scratch in a fixed static device array
instead of a caller workspace. Two calls in a row, on different hidden
states, must each match the workspace entry point within the parity
tolerances; sizes beyond the array are refused. This file is collected last.
"""
import ctypes

import numpy as np
import pytest

from gpu_util import dev_bf16, dev_i32, host, lib, make_case
import parity as P

pytestmark = pytest.mark.gpu


def _noalloc(L, W, A, B, h, tok, n, d, r, M, T, k, temp, out):
    import torch
    ids, lg, q = out
    return L.load().lmhead_two_stage_local_noalloc(
        W.data_ptr(), A.data_ptr(), B.data_ptr(), h.data_ptr(), tok.data_ptr(), n, d, r, M, T, k,
        ctypes.c_float(temp), ids.data_ptr(), lg.data_ptr(), q.data_ptr(),
        torch.cuda.current_stream().cuda_stream)


def test_noalloc_matches_two_stage_on_two_calls():
    import torch
    L = lib()
    n, d, r, T, k = 3000, 128, 32, 256, 2          # 12 tiles, ragged last tile
    case = make_case(n, d, r, 24, seed=31, plain_h=True)
    W, A, B, tok = dev_bf16(case["W"]), dev_bf16(case["A"]), dev_bf16(case["B"]), dev_i32(case["tok"])
    K = L.candidate_count(L.LOCAL, n, T, k)
    for call, (rows, temp) in enumerate(((slice(0, 11), 1.0), (slice(11, 24), 0.7))):
        h = dev_bf16(np.ascontiguousarray(case["h"][rows]))
        M = h.shape[0]
        ref_ids, ref_lg, ref_q = (host(t) for t in L.two_stage(L.LOCAL, W, A, B, h, tok, T, k,
                                                                temperature=temp))
        out = (torch.full((M, K), -1, dtype=torch.int32, device="cuda"),
               torch.full((M, K), float("nan"), device="cuda"),
               torch.full((M, K), float("nan"), device="cuda"))
        assert _noalloc(L, W, A, B, h, tok, n, d, r, M, T, k, temp, out) == 0, f"call {call}"
        ids, lg, q = (host(t) for t in out)
        assert L.last_device_error() == 0
        for m in range(M):                         # same candidate set per tile
            for t0 in range(0, K, k):
                assert set(ids[m, t0:t0 + k]) == set(ref_ids[m, t0:t0 + k])
        order = [np.argsort(ids[m]) for m in range(M)]
        ref_order = [np.argsort(ref_ids[m]) for m in range(M)]
        lg_s = np.stack([lg[m, o] for m, o in enumerate(order)])
        ref_lg_s = np.stack([ref_lg[m, o] for m, o in enumerate(ref_order)])
        assert np.all(np.abs(lg_s - ref_lg_s) <= P.LOGIT_REL * np.maximum(np.abs(ref_lg_s), 1.0))
        q_s = np.stack([q[m, o] for m, o in enumerate(order)])
        ref_q_s = np.stack([ref_q[m, o] for m, o in enumerate(ref_order)])
        assert np.abs(q_s - ref_q_s).max() <= P.Q_ABS


def test_noalloc_refuses_sizes_beyond_its_scratch():
    import torch
    L = lib()
    n, d, r = 512, 64, 16
    case = make_case(n, d, r, 257, seed=32)
    W, A, B, tok = dev_bf16(case["W"]), dev_bf16(case["A"]), dev_bf16(case["B"]), dev_i32(case["tok"])
    h = dev_bf16(case["h"])
    K = L.candidate_count(L.LOCAL, n, 128, 2)
    out = (torch.full((257, K), -1, dtype=torch.int32, device="cuda"),
           torch.zeros((257, K), device="cuda"), torch.zeros((257, K), device="cuda"))
    assert _noalloc(L, W, A, B, h, tok, n, d, r, 257, 128, 2, 1.0, out) == -5   # M > 256
    assert _noalloc(L, W, A, B, h, tok, n, d, r, 4, 128, 33, 1.0, out) == -5    # k_tile > 32
    torch.cuda.synchronize()
    assert (host(out[0]) == -1).all()              # nothing was enqueued
