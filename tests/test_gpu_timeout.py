"""The bounded-wait timeout path of the tensor-core kernels, exercised
without faulting or hanging the GPU: with a role-wait budget of zero every
wait between the warp roles tests its barrier once, so a call gives up at its
first wait that is not already complete. The kernel then records
LMHEAD_ERR_TIMEOUT, drains its own copies and MMAs, frees its tensor memory
and returns. The status must reach the host, and the next call on the same
stream, with the default budget, must be correct again."""
import numpy as np
import pytest

import oracle as O

from gpu_util import dev_bf16, dev_i32, host, lib, make_case, oracle_scores
import parity as P

pytestmark = pytest.mark.gpu

ERR_TIMEOUT = -8


@pytest.fixture(scope="module")
def L():
    return lib()


def _timed_out(L, fn):
    L.debug_set_wait_cycles(0)
    try:
        fn()
        status = L.last_device_error()
    finally:
        L.debug_set_wait_cycles(-1)
    return status


@pytest.mark.parametrize("mode,C,k,M", [("local", 256, 2, 24),    # fused score + top-k, 256-row MMAs
                                        ("local", 128, 4, 80),    # 128-row MMAs
                                        ("local", 200, 2, 9),     # tiles cut between CTAs
                                        ("global", 300, 0, 5)])   # score writeback
def test_timeout_is_reported_and_the_next_call_recovers(L, mode, C, k, M):
    case = make_case(6000, 256, 32, M, seed=41, plain_h=True)
    W, A, B, h = (dev_bf16(case[x]) for x in ("W", "A", "B", "h"))
    tok = dev_i32(case["tok"])
    md = L.LOCAL if mode == "local" else L.GLOBAL
    L.two_stage(md, W, A, B, h, tok, C, k)      # launch set-up done once
    assert L.last_device_error() == 0
    assert _timed_out(L, lambda: L.two_stage(md, W, A, B, h, tok, C, k)) == ERR_TIMEOUT
    assert L.last_device_error() == 0           # read and cleared
    ids, lg, q = L.two_stage(md, W, A, B, h, tok, C, k)
    assert L.last_device_error() == 0
    _, S, h64, SL = oracle_scores(case, with_slack=True)
    ids = host(ids)
    P.check_ids(mode, ids, S, case["tok"], C, k, slack_pos=SL)
    ex = P.exact_logits(case["W"], h64, ids)
    P.check_logits(host(lg), ex)
    P.check_q(host(q), ex)


def test_dense_head_timeout_recovers(L):
    case = make_case(5000, 128, 16, 3, seed=42, plain_h=True)
    W, h = dev_bf16(case["W"]), dev_bf16(case["h"])
    L.dense_head(W, h)
    assert L.last_device_error() == 0
    assert _timed_out(L, lambda: L.dense_head(W, h)) == ERR_TIMEOUT
    lg, q = L.dense_head(W, h)
    assert L.last_device_error() == 0
    Z = O.bf16_bits_to_f64(case["h"]) @ O.bf16_bits_to_f64(case["W"]).T
    P.check_logits(host(lg), Z)


def test_budget_setter_round_trips(L):
    default = L.debug_set_wait_cycles(12345)
    assert default > 10 ** 9                     # about a second of SM cycles
    assert L.debug_set_wait_cycles(-1) == 12345
    assert L.debug_set_wait_cycles(-1) == default
