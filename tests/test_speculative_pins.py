"""Pins of the speculative-step oracle (oracle/speculative_oracle.py) against
what the pages and the mathematics fix, independent of the oracle itself:
brute force on tiny inputs, hand-computed cases, the Gumbel-max theorem, and
the page's own exactness exercise (output distribution = target, TV < 0.01),
with the page's listing form of the residual shown to fail it (reading R17)."""
import itertools

import numpy as np
import pytest

import oracle as O


def test_draft_topk_brute_force_and_ties():
    rng = np.random.default_rng(1)
    for _ in range(50):
        K = 9
        q = rng.choice(np.array([0.05, 0.1, 0.2, 0.3], dtype=np.float32), size=K)  # many ties
        ids = rng.permutation(40)[:K].astype(np.int32)
        for k in (1, 3, K):
            got_ids, got_q, _ = O.draft_topk(q, ids, k)
            # brute force: the first k of all (q desc, id asc) orderings is unique
            ref = sorted(zip((-q.astype(np.float64)).tolist(), ids.tolist()))[:k]
            assert got_ids.tolist() == [i for _, i in ref]
            assert np.array_equal(got_q, q[[list(ids).index(i) for _, i in ref]])


def test_draft_value_is_fp32_product():
    q = np.array([0.7, 0.2, 0.1], dtype=np.float32)
    ids = np.array([5, 3, 9], dtype=np.int32)
    _, top_q, val = O.draft_topk(q, ids, 2, parent_value=0.3)
    assert val.dtype == np.float32
    assert val[0] == np.float32(np.float32(0.3) * np.float32(0.7))
    # a chain of expansions multiplies confidences along the path ([E1])
    _, _, v2 = O.draft_topk(q, ids, 1, parent_value=val[0])
    assert v2[0] == np.float32(val[0] * np.float32(0.7))


def test_gumbel_max_matches_q():
    # Gumbel-max theorem: argmax(log q + G) is distributed as q
    q = np.array([0.5, 0.25, 0.125, 0.0625, 0.0625, 0.0], dtype=np.float32)
    ids = np.arange(6, dtype=np.int32)
    rng = np.random.default_rng(2)
    N = 60000
    U = rng.random((N, 6))
    U = np.clip(U, 1e-12, 1 - 1e-12)
    counts = np.zeros(6)
    for row in U:
        counts[O.gumbel_sample(q, ids, row)[1]] += 1
    tv = 0.5 * np.abs(counts / N - q).sum()
    assert tv < 0.01
    assert counts[5] == 0  # q = 0 is never drawn


def test_gumbel_degenerate_cases():
    ids = np.array([7, 3, 11], dtype=np.int32)
    u = np.array([0.9, 0.001, 0.5])
    assert O.gumbel_sample(np.array([0, 1, 0], dtype=np.float32), ids, u)[0] == 3
    # hand value: u = exp(-1) gives g = 0, so the score is log q
    s = O.gumbel_scores(np.array([0.25]), np.array([np.exp(-1.0)]))
    assert s[0] == pytest.approx(np.log(0.25), abs=1e-12)


def test_inverse_cdf_hand_values():
    w = np.array([0.1, 0.2, 0.7])
    assert O.inverse_cdf_sample(w, 0.05) == 0
    assert O.inverse_cdf_sample(w, 0.10) == 1     # sum(w[:1]) = 0.1 is not > 0.1
    assert O.inverse_cdf_sample(w, 0.29) == 1
    assert O.inverse_cdf_sample(w, 0.31) == 2
    assert O.inverse_cdf_sample(2 * w, 0.31) == 2  # scale-free
    assert O.inverse_cdf_sample(np.array([0.0, 0.0, 1.0]), 0.0) == 2  # zero weights never chosen


def test_residual_hand_values():
    p = np.array([0.1, 0.4, 0.2, 0.3])
    w = O.residual(p, np.array([1, 2]), np.array([0.5, 0.1]))
    assert np.allclose(w, [0.1, 0.0, 0.1, 0.3])


def test_verify_chain_hand_case():
    # n = 4, Kd = 2. Position 0: q(x0=1) = 0.5, p(1) = 0.4 -> ratio 0.8, r0 = 0.7 accepts.
    # Position 1: q(x1=2) = 0.6, p(2) = 0.3 -> ratio 0.5, r1 = 0.9 rejects; with
    # p1 = [0.2, 0.1, 0.3, 0.4] and q1 = {2: 0.6, 1: 0.4} the residual (p - q)+ is
    # [0.2, 0, 0, 0.4].
    p = np.array([[0.1, 0.4, 0.2, 0.3], [0.2, 0.1, 0.3, 0.4], [0.25, 0.25, 0.25, 0.25]])
    x = np.array([1, 2])
    cand_ids = [np.array([1, 3]), np.array([2, 1])]
    cand_q = [np.array([0.5, 0.5], dtype=np.float32), np.array([0.6, 0.4], dtype=np.float32)]
    n_acc, out = O.verify_chain(p, x, cand_ids, cand_q, r=np.array([0.7, 0.9]), u=np.array([0.0, 0.5, 0.0]))
    assert n_acc == 1
    assert out == [1, 3]          # u * 0.6 = 0.3 > cumsum 0.2 -> index 3
    n_acc, out = O.verify_chain(p, x, cand_ids, cand_q, r=np.array([0.7, 0.4]), u=np.array([0.0, 0.0, 0.6]))
    assert n_acc == 2 and out == [1, 2, 2]   # both accepted; bonus from p[2] at u = 0.6


def _tv_of_first_token(residual_fn, trials=40000, seed=3):
    rng = np.random.default_rng(seed)
    n = 12
    p = rng.random(n) ** 2
    p /= p.sum()
    cand = np.array([0, 2, 3, 5, 8, 11])
    qc = rng.random(cand.size).astype(np.float64) + 0.1
    qc = (qc / qc.sum()).astype(np.float32)
    counts = np.zeros(n)
    U = rng.random((trials, cand.size))
    R = rng.random(trials)
    V = rng.random(trials)
    for i in range(trials):
        x = O.gumbel_sample(qc, cand, U[i])[0]
        qx = np.float32(qc[np.nonzero(cand == x)[0][0]])
        if np.float32(R[i]) < np.float32(np.float32(p[x]) / qx):
            tok = x
        else:
            w = residual_fn(p, cand, qc, x, qx)
            tok = O.inverse_cdf_sample(w, V[i])
        counts[tok] += 1
    return 0.5 * np.abs(counts / trials - p).sum()


def test_exactness_tv_below_001():
    # the page's exercise: the output of draft + accept/reject is distributed as p
    tv = _tv_of_first_token(lambda p, cand, qc, x, qx: O.residual(p, cand, qc))
    assert tv < 0.01


def test_listing_residual_form_fails_exactness():
    # R17: subtracting the scalar q(x) (the page's listing) does not preserve p
    tv = _tv_of_first_token(lambda p, cand, qc, x, qx: np.maximum(p - float(qx), 0.0))
    assert tv > 0.02


def test_verify_chain_equal_distributions_accept_everything():
    rng = np.random.default_rng(4)
    n, Kd = 10, 3
    cand = [np.array([1, 4, 6]) for _ in range(Kd)]
    qs = []
    p = np.zeros((Kd + 1, n))
    for t in range(Kd):
        qv = rng.random(3) + 0.2
        qv = (qv / qv.sum()).astype(np.float32)
        qs.append(qv)
        p[t, cand[t]] = qv  # target equals the draft distribution
    p[Kd] = 1.0 / n
    for trial in range(50):
        x = np.array([cand[t][trial % 3] for t in range(Kd)])
        n_acc, out = O.verify_chain(p, x, cand, qs, rng.random(Kd) * 0.999, rng.random(Kd + 1))
        assert n_acc == Kd and out[:Kd] == x.tolist()


def test_verify_chain_rejects_non_candidate_draft():
    with pytest.raises(ValueError):
        O.verify_chain(np.ones((2, 3)) / 3, np.array([2]), [np.array([0, 1])],
                       [np.array([0.5, 0.5], dtype=np.float32)], np.array([0.5]), np.array([0.5, 0.5]))
