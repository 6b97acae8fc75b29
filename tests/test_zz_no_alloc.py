"""The no-allocation entry point lmhead_two_stage_local_noalloc, through the
C ABI, against the oracle on the same inputs.

Some callers cannot allocate device memory at call time (a serving engine
that has given all free HBM to its KV-cache pool, or C code without a device
allocator), so this variant keeps its scratch in a fixed static device array
instead of a caller workspace. Two calls in a row, on different hidden
states, must each match the oracle within the parity tolerances that the
workspace entry point meets; sizes beyond the array are refused.
This file is collected last.
"""
import ctypes

import numpy as np
import pytest

from gpu_util import dev_bf16, dev_i32, host, lib, make_case, oracle_scores
import parity as P

pytestmark = pytest.mark.gpu


def _noalloc(L, W, A, B, h, tok, n, d, r, M, T, k, temp, out):
    import torch
    ids, lg, q = out
    return L.load().lmhead_two_stage_local_noalloc(
        W.data_ptr(), A.data_ptr(), B.data_ptr(), h.data_ptr(), tok.data_ptr(), n, d, r, M, T, k,
        ctypes.c_float(temp), ids.data_ptr(), lg.data_ptr(), q.data_ptr(),
        torch.cuda.current_stream().cuda_stream)


def _against_oracle(case, rows, T, k, temp, ids, lg, q):
    """The new entry point's output against the oracle: ids by the boundary
    rule with the u-rounding slack, logits and q against fp64 W[id].h."""
    sub = dict(case)
    sub["h"] = case["h"][rows]
    _, S, h64, SL = oracle_scores(sub, with_slack=True)
    P.check_ids("local", ids, S, case["tok"], T, k, slack_pos=SL)
    ex = P.exact_logits(case["W"], h64, ids)
    P.check_logits(lg, ex)
    P.check_q(q, ex, temp)


@pytest.mark.parametrize("n,d,r,T,k,calls", [
    # 12 tiles, ragged last tile; 11 and 13 hidden vectors (tensor-core
    # scoring, its tile counters in the fixed scratch)
    (3000, 128, 32, 256, 2, ((slice(0, 11), 1.0), (slice(11, 24), 0.7))),
    # 96-row tiles (not a multiple of 128: the CUDA-core tile kernel)
    (3000, 128, 32, 96, 2, ((slice(0, 5), 1.0), (slice(5, 12), 0.7))),
    # the decode-loop shape: one and two hidden vectors, r = 256, 256-row
    # tiles (the warp-per-row scoring kernel), ragged last tile of 64 rows
    (4160, 256, 256, 256, 2, ((slice(0, 1), 1.0), (slice(1, 3), 0.8))),
])
def test_noalloc_matches_oracle_on_two_calls(n, d, r, T, k, calls):
    import torch
    L = lib()
    case = make_case(n, d, r, 24, seed=31, plain_h=True)
    W, A, B, tok = dev_bf16(case["W"]), dev_bf16(case["A"]), dev_bf16(case["B"]), dev_i32(case["tok"])
    K = L.candidate_count(L.LOCAL, n, T, k)
    for call, (rows, temp) in enumerate(calls):
        h = dev_bf16(np.ascontiguousarray(case["h"][rows]))
        M = h.shape[0]
        out = (torch.full((M, K), -1, dtype=torch.int32, device="cuda"),
               torch.full((M, K), float("nan"), device="cuda"),
               torch.full((M, K), float("nan"), device="cuda"))
        assert _noalloc(L, W, A, B, h, tok, n, d, r, M, T, k, temp, out) == 0, f"call {call}"
        ids, lg, q = (host(t) for t in out)
        assert L.last_device_error() == 0
        _against_oracle(case, np.arange(24)[rows], T, k, temp, ids, lg, q)


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
