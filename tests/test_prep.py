"""The offline Freq-aware SVD of the product (Gram + eigh in fp64, then bf16)
against the oracle's literal SVD of F^1/2 W."""
import numpy as np

import oracle as O
import synth
from draft_lm_head_gb300 import prep


def test_prep_matches_oracle_svd():
    n, d, r = 600, 48, 12
    W = synth.make_head(n, d, 21)
    counts = synth.zipf_counts(n, 1.1, 21)
    perm = synth.shuffle_perm(n, 21)
    fac = prep.freq_aware_factors(W, counts, r, perm, block=97)
    W64 = O.bf16_bits_to_f64(W)
    f = O.smooth_freq(counts)
    A, B, S = O.freq_aware_svd(W64, f, r)
    assert np.allclose(fac["eigenvalues"], S ** 2, rtol=1e-9, atol=1e-6 * S[0] ** 2)
    assert np.array_equal(fac["token_ids"], perm)
    AB_prep = O.bf16_bits_to_f64(fac["A"]) @ O.bf16_bits_to_f64(fac["B"])
    AB_ora = (A @ B)[perm]
    rel = np.linalg.norm(AB_prep - AB_ora) / np.linalg.norm(AB_ora)
    assert rel < 1e-2          # bf16 rounding of both factors
    # the rounding-free identity A = W B^T holds for the prep's factors too
    A_ref = W64[perm] @ O.bf16_bits_to_f64(fac["B"]).T
    assert np.abs(O.bf16_bits_to_f64(fac["A"]) - A_ref).max() <= 2 ** -7 * np.abs(A_ref).max()


def test_prep_identity_order_and_full_rank():
    n, d = 200, 16
    W = synth.make_head(n, d, 22)
    fac = prep.freq_aware_factors(W, np.zeros(n, dtype=np.int64), d)
    assert np.array_equal(fac["token_ids"], np.arange(n))
    AB = O.bf16_bits_to_f64(fac["A"]) @ O.bf16_bits_to_f64(fac["B"])
    W64 = O.bf16_bits_to_f64(W)
    assert np.linalg.norm(AB - W64) / np.linalg.norm(W64) < 1e-2


def test_pruned_rows_match_the_oracle():
    import synth
    rng = np.random.default_rng(3)
    counts = rng.integers(0, 50, 400)          # many ties
    W = synth.make_head(400, 16, 0)
    Wp, kept = prep.pruned_rows(W, counts, 123)
    want = O.pruned_ids(O.smooth_freq(counts), 123)
    assert np.array_equal(kept, want)
    assert np.array_equal(Wp, W[want])
