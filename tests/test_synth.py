"""Sanity of the seeded synthetic inputs (shapes, determinism, recipe)."""
import numpy as np

import synth


def test_head_is_deterministic_and_bf16():
    W1 = synth.make_head(300, 64, 0)
    W2 = synth.make_head(300, 64, 0, block=37)
    assert W1.dtype == np.uint16 and W1.shape == (300, 64)
    assert np.array_equal(W1, W2)
    Wf = synth.bf16_bits_to_f64(W1)
    # rank-64 structure X.Y/8 has unit-variance entries; noise adds 0.05^2
    assert 0.8 < Wf.std() < 1.2


def test_zipf_counts_follow_ranks():
    c = synth.zipf_counts(1000, 1.1, 0)
    s = np.sort(c)[::-1]
    assert s[0] > 10 * s[9] > 0
    assert len(set(np.argsort(-c, kind="stable")[:5].tolist())) == 5
    assert c.sum() <= 10 ** 9


def test_hidden_recipe_points_at_target():
    W = synth.make_head(500, 256, 0)
    h, t = synth.make_hidden(W, 4, 0)
    Wf, hf = synth.bf16_bits_to_f64(W), synth.bf16_bits_to_f64(h)
    for m in range(4):
        cos = Wf @ hf[m] / np.linalg.norm(Wf, axis=1) / np.linalg.norm(hf[m])
        assert np.argmax(cos) == t[m]


def test_tree_rows_mix_parent():
    W = synth.make_head(200, 64, 3)
    h, _ = synth.make_tree_hidden(W, 2, 3)
    assert h.shape == (20, 64)
    hf = synth.bf16_bits_to_f64(h)
    # a child correlates with its parent more than with an unrelated root
    c = np.corrcoef(hf)
    assert c[4, 1] > abs(c[4, 10])


def test_perm_is_permutation():
    p = synth.shuffle_perm(1000, 2)
    assert p.dtype == np.int32 and np.array_equal(np.sort(p), np.arange(1000))
