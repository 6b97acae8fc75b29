"""The vocabulary-sharded local head on one GPU: the shards run one after
another (each on its own slice of A and W), their (max, sum) stats are
stacked as an all-gather would, and every shard finishes its q. The shards'
outputs side by side must match the oracle of the unsharded head: with
tile-aligned shards the candidates are the same, and q is the softmax over
all of them."""
import numpy as np
import pytest
import torch

import oracle as O
import synth

from gpu_util import dev_bf16, dev_i32, host, lib, make_case, oracle_scores, workload_case
import parity as P

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def L():
    return lib()


def _run_shards(L, case, T, k, G, temperature, rows=None):
    from draft_lm_head_gb300 import shard as S
    B = dev_bf16(case["B"])
    h = dev_bf16(case["h"])
    outs = []
    for p0, p1 in S.shard_ranges(case["n"], T, G):
        Ws, As, toks, roi = S.shard_inputs(case["W"], case["A"], case["tok"], p0, p1)
        outs.append(L.shard_two_stage(dev_bf16(Ws), dev_bf16(As), B, h, dev_i32(toks),
                                      dev_i32(roi), T, k, temperature))
    all_stats = torch.stack([o[2] for o in outs])
    qs = [L.shard_softmax(all_stats, o[1], temperature) for o in outs]
    assert L.last_device_error() == 0
    ids = np.concatenate([host(o[0]) for o in outs], axis=1)
    lg = np.concatenate([host(o[1]) for o in outs], axis=1)
    q = np.concatenate([host(x) for x in qs], axis=1)
    return ids, lg, q


def _check(case, T, k, ids, lg, q, temperature, rows=None):
    rows = np.arange(case["M"]) if rows is None else np.asarray(rows)
    sub = dict(case)
    sub["h"] = case["h"][rows]
    _, S, h64, SL = oracle_scores(sub, with_slack=True, M_call=case["M"])
    assert ids.shape[1] == O.local_candidate_count(case["n"], T, k)
    counts = P.check_ids("local", ids[rows], S, case["tok"], T, k, slack_pos=SL)
    ex = P.exact_logits(case["W"], h64, ids[rows])
    P.check_logits(lg[rows], ex)
    P.check_q(q[rows], ex, temperature)
    return counts


@pytest.mark.parametrize("n,d,r,T,k,M,G", [
    (3000, 128, 32, 256, 2, 5, 2),      # ragged last tile in the last shard
    (4096, 256, 32, 128, 4, 3, 3),      # three shards, GEMV-free small M
    (20000, 64, 16, 256, 8, 17, 2),     # tensor-core scoring, ready counters
    (4160, 256, 256, 256, 2, 1, 2),     # one hidden vector: the GEMV scoring kernel
])
def test_shards_match_the_unsharded_oracle(L, n, d, r, T, k, M, G):
    case = make_case(n, d, r, M, seed=51, plain_h=True)
    temp = 0.8
    ids, lg, q = _run_shards(L, case, T, k, G, temp)
    _check(case, T, k, ids, lg, q, temp)
    # the same candidate sets, tile by tile, as the unsharded call
    W, A, B, h, tok = (dev_bf16(case["W"]), dev_bf16(case["A"]), dev_bf16(case["B"]),
                       dev_bf16(case["h"]), dev_i32(case["tok"]))
    ref_ids, _, ref_q = (host(t) for t in L.two_stage(L.LOCAL, W, A, B, h, tok, T, k,
                                                        temperature=temp))
    same = all(set(ids[m, j:j + k]) == set(ref_ids[m, j:j + k])
               for m in range(M) for j in range(0, ids.shape[1], k))
    if same:
        np.testing.assert_allclose(q, ref_q, atol=P.Q_ABS)


def test_shards_on_the_headline_head(L):
    """n=128256, d=4096, r=256, shuffled rows, tile 256, k_tile 2, M=64,
    two shards of 250 and 251 tiles; parity on sampled rows."""
    wl = synth.workload(2)
    case = workload_case(wl, 64)
    case["h"] = synth.make_plain_hidden(wl.d, 64, wl.index)
    ids, lg, q = _run_shards(L, case, wl.T, wl.k_tile, 2, 20.0)
    counts = _check(case, wl.T, wl.k_tile, ids, lg, q, 20.0, rows=[0, 17, 40, 63])
    P.record("wl2 local 2 vocabulary shards, plain h, T=20 M=64 (4 rows)", **counts)


def test_shard_argument_checks(L):
    case = make_case(512, 64, 16, 2, seed=52)
    B, h = dev_bf16(case["B"]), dev_bf16(case["h"])
    from draft_lm_head_gb300 import shard as S
    Ws, As, toks, roi = S.shard_inputs(case["W"], case["A"], case["tok"], 0, 256)
    with pytest.raises(L.LmheadError):           # temperature must be positive
        L.shard_two_stage(dev_bf16(Ws), dev_bf16(As), B, h, dev_i32(toks), dev_i32(roi), 128, 2, 0.0)
    with pytest.raises(ValueError):              # row_of_id of the wrong length for W's ids
        L.shard_two_stage(dev_bf16(Ws), dev_bf16(As), B, h, dev_i32(toks[:-1]), dev_i32(roi), 128, 2)
