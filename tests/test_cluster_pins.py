"""Pins of the cluster-level oracle (oracle/cluster_oracle.py) against values
fixed by hand, brute force over tokens on tiny inputs, and two special cases
that reduce to textbook definitions: one group per token is the plain global
Top-G of the low-rank scores, and all groups selected is the full-vocabulary
softmax of W.h."""
import math

import numpy as np
import pytest
from scipy.special import softmax

import oracle as O


def test_hand_case():
    s = np.array([0.1, 0.9, 0.5, 0.2, -1.0, 0.95, 0.3, 0.3])
    g = O.group_scores(s, 2)
    assert g.tolist() == [0.9, 0.5, 0.95, 0.3]
    sel = O.select_groups(g, 2)
    assert sel.tolist() == [2, 0]
    assert O.group_candidates(sel, 2).tolist() == [4, 5, 0, 1]
    assert O.select_groups(g, 4).tolist() == [2, 0, 1, 3]


def test_ties_by_smaller_group():
    s = np.array([1.0, 0.0, 0.0, 1.0, 0.5, 1.0, 0.0, 0.0, 1.0])
    g = O.group_scores(s, 3)
    assert g.tolist() == [1.0, 1.0, 1.0]
    assert O.select_groups(g, 2).tolist() == [0, 1]


def test_ragged_group_refused():
    with pytest.raises(ValueError):
        O.group_scores(np.zeros(10), 4)
    with pytest.raises(ValueError):
        O.select_groups(np.zeros(3), 4)


def test_group_of_one_is_global_topk():
    rng = np.random.default_rng(3)
    for _ in range(20):
        s = rng.choice(np.array([-1.0, 0.0, 0.25, 0.5, 2.0]), size=17)  # ties
        sel = O.select_groups(O.group_scores(s, 1), 6)
        ref = [i for _, i in sorted(zip((-s).tolist(), range(17)))[:6]]
        assert sel.tolist() == ref


def test_brute_force_selection_tiny():
    """Over every row of random tiny heads: each selected group holds a token
    scoring at least as high as every token of every unselected group, with
    the tie rule, and the candidates are whole aligned blocks."""
    rng = np.random.default_rng(4)
    n, d, r, group, G, M = 24, 16, 4, 4, 3, 3
    W = O.round_to_bf16(rng.standard_normal((n, d)))
    A = O.round_to_bf16(rng.standard_normal((n, r)))
    B = O.round_to_bf16(rng.standard_normal((r, d)))
    h = O.round_to_bf16(rng.standard_normal((M, d)))
    out = O.cluster_two_stage(W, A, B, h, group, G)
    for m in range(M):
        u = out["u"][m]
        # scores by exact sums over the row, independent of the oracle's matmul
        sc = [math.fsum(float(A[i, k]) * float(u[k]) for k in range(r)) for i in range(n)]
        best = [max(sc[g * group:(g + 1) * group]) for g in range(n // group)]
        np.testing.assert_allclose(out["gscores"][m], best, rtol=1e-12, atol=1e-12)
        ranked = sorted(range(n // group), key=lambda g: (-best[g], g))
        assert out["groups"][m].tolist() == ranked[:G]
        ids = out["ids"][m]
        assert len(ids) == G * group and len(set(ids.tolist())) == G * group
        for j, g in enumerate(out["groups"][m]):
            assert ids[j * group:(j + 1) * group].tolist() == list(range(g * group, (g + 1) * group))
        logit = [math.fsum(float(W[i, k]) * float(h[m, k]) for k in range(d)) for i in ids]
        np.testing.assert_allclose(out["logits"][m], logit, rtol=1e-12, atol=1e-12)


def test_all_groups_is_dense_softmax():
    rng = np.random.default_rng(5)
    n, d, r, group, M = 32, 24, 6, 8, 2
    W = O.round_to_bf16(rng.standard_normal((n, d)))
    A = O.round_to_bf16(rng.standard_normal((n, r)))
    B = O.round_to_bf16(rng.standard_normal((r, d)))
    h = O.round_to_bf16(rng.standard_normal((M, d)))
    for T in (1.0, 0.7):
        out = O.cluster_two_stage(W, A, B, h, group, n // group, temperature=T)
        for m in range(M):
            full = np.zeros(n)
            full[out["ids"][m]] = out["q"][m]
            ref = softmax((W @ h[m]) / T)
            np.testing.assert_allclose(full, ref, rtol=1e-12, atol=1e-15)
            assert sorted(out["ids"][m].tolist()) == list(range(n))


def test_group_scores_are_tile_maxima_of_local_topk():
    """Consistency with the token-level oracle: a tile of T rows keeping
    k_tile = 1 keeps exactly the group's best row."""
    rng = np.random.default_rng(6)
    s = rng.standard_normal(64)
    ids, vals = O.local_topk(s, np.arange(64), 16, 1)
    np.testing.assert_array_equal(vals, O.group_scores(s, 16))
    assert all(ids[g] // 16 == g for g in range(4))
