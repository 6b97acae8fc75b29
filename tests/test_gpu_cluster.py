"""Cluster-level two-stage head (groups of consecutive rows, the G best
groups by their best low-rank score, exact logits of every row inside them)
vs the fp64 oracle, through the C ABI: several group sizes (tensor-core and
CUDA-core selection paths), G from one group to all of them, temperatures,
and the full-size head of the Llama-3-8B-shaped workload."""
import numpy as np
import pytest

import oracle as O
import synth

from gpu_util import dev_bf16, host, lib, make_case, oracle_scores, workload_case
import parity as P

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def L():
    return lib()


def _run(L, case, group, G, temperature=1.0):
    W, A, B, h = (dev_bf16(case[k]) for k in ("W", "A", "B", "h"))
    out = L.cluster_two_stage(W, A, B, h, group, G, temperature, with_group_scores=True)
    assert L.last_device_error() == 0
    return [host(t) for t in out]


def _check(case, group, G, groups, ids, lg, q, gs, temperature=1.0, rows=None):
    rows = np.arange(case["M"]) if rows is None else np.asarray(rows)
    sub = dict(case)
    sub["h"] = case["h"][rows]
    u, S, h64, SL = oracle_scores(sub, with_slack=True, M_call=case["M"])
    groups, ids, lg, q, gs = groups[rows], ids[rows], lg[rows], q[rows], gs[rows]
    excused = P.check_groups(groups, S, group, G, slack_pos=SL)
    M = len(rows)
    # reported group scores: best first, each the group's best fp32 score
    assert np.all(np.diff(gs, axis=1) <= 0)
    A64 = O.bf16_bits_to_f64(case["A"])
    ng = case["n"] // group
    for m in range(M):
        mag = (np.abs(A64) @ np.abs(u[m])).reshape(ng, group).max(axis=1)
        want = S[m].reshape(ng, group).max(axis=1)
        slack = SL[m].reshape(ng, group).max(axis=1)
        g = groups[m]
        assert np.all(np.abs(gs[m] - want[g]) <= 1e-5 * mag[g] + 1e-6 + slack[g])
    # candidates: the GPU's own groups expanded, bit-exact
    want_ids = (groups[:, :, None].astype(np.int64) * group + np.arange(group)).reshape(M, G * group)
    assert np.array_equal(ids, want_ids)
    ex = P.exact_logits(case["W"], h64, ids)
    P.check_logits(lg, ex)
    P.check_q(q, ex, temperature)
    return excused


@pytest.fixture(scope="module")
def tiny():
    # the tiny workload's shapes (n=4096, d=256, r=32), head rows unshuffled, 5 hidden vectors
    return make_case(4096, 256, 32, 5, seed=21, shuffle=False)


@pytest.mark.parametrize("group,G", [(128, 1), (128, 4), (128, 32), (32, 17), (64, 3), (256, 2),
                                     (512, 8), (4096, 1), (8, 100), (1, 64), (16, 256)])
def test_cluster_tiny(L, tiny, group, G):
    out = _run(L, tiny, group, G)
    assert out[1].shape == (5, G * group)
    _check(tiny, group, G, *out)


def test_cluster_all_groups_is_dense_softmax(L, tiny):
    groups, ids, lg, q, gs = _run(L, tiny, 128, 32, 0.6)
    _check(tiny, 128, 32, groups, ids, lg, q, gs, 0.6)
    h64 = O.bf16_bits_to_f64(tiny["h"])
    Z = h64 @ O.bf16_bits_to_f64(tiny["W"]).T / 0.6
    for m in range(5):
        full = np.zeros(4096)
        full[ids[m]] = q[m]
        ref = np.exp(Z[m] - Z[m].max())
        np.testing.assert_allclose(full, ref / ref.sum(), atol=P.Q_ABS)


@pytest.mark.parametrize("M", [1, 17, 64])
def test_cluster_longer_rows(L, M):
    case = make_case(20000, 64, 16, M, seed=22, shuffle=False)
    for group, G in ((160, 3), (100, 7), (40, 50)):
        out = _run(L, case, group, G)
        _check(case, group, G, *out, rows=None if M <= 17 else [0, 5, 31, 63])


def test_cluster_full_size_head(L):
    """n=128256, d=4096, r=256, unshuffled, M=64, 128-row groups, G=8 (1024
    candidates, the global route's C): parity on sampled rows, and recall of
    the exact full-head Top-{1,8,64} next to the token-level routes."""
    wl = synth.workload(2)
    case = workload_case(wl, 64, shuffle=False)
    groups, ids, lg, q, gs = _run(L, case, 128, 8)
    assert ids.shape == (64, 1024)
    rows = [0, 1, 13, 32, 63]
    _check(case, 128, 8, groups, ids, lg, q, gs, rows=rows)
    h64 = O.bf16_bits_to_f64(case["h"][rows])
    Z = h64 @ O.bf16_bits_to_f64(case["W"]).T
    rec = {k: float(np.mean([O.recall_at(ids[m], Z[i], k) for i, m in enumerate(rows)]))
           for k in (1, 8, 64)}
    print("cluster 128x8 recall", rec)
    assert rec[1] > 0.5
