"""The parity rules themselves (tests/parity.py), on hand-built cases: the
projection's rounding depth per kernel, the u check at an exact bf16
midpoint, and the split of excused ids into the 1e-3 band and the u-slack."""
import numpy as np

import parity as P


def test_projection_depth_per_kernel():
    # GEMV: 7 (FMA chain) + VPT - 1 + 5 (butterfly) + 3 (warp partials)
    assert P.projection_depth(256, 1) == 15        # VPT 1
    assert P.projection_depth(4096, 8) == 18       # VPT 4
    assert P.projection_depth(2880, 2) == 18       # vpt 3 runs as VPT 4
    assert P.projection_depth(5120, 4) == 22       # vpt 5 runs as VPT 8 (M <= 4)
    # tensor cores: 2 per 16-wide MMA step of the CTA's slice + KS - 1
    assert P.projection_depth(4096, 64) == 2 * 32 + 7   # KS 8, slices of 512
    assert P.projection_depth(5120, 8) == 2 * 40 + 7    # vpt 5 at M > 4: tensor cores
    assert P.projection_depth(2880, 80) == 2 * 32 + 5   # KS 6, 480 -> 512 columns
    assert P.projection_depth(96, 300) == 2 * 8 + 0     # KS 1, 96 -> 128 columns
    g = P.u_gamma(4096, 64)
    assert 71 * 2.0 ** -24 < g < 71.01 * 2.0 ** -24


def _bits(*vals):
    # bf16 bit patterns of exactly representable values
    return np.array([np.float32(v).view(np.uint32) >> 16 for v in vals], dtype=np.uint16)


def test_check_u_accepts_only_ambiguous_neighbours():
    h = np.array([[1.0, 1.0, 1.0]])
    # exact u = 1 + 2^-8 + 2^-30: just above the midpoint of 1 and 1 + 2^-7;
    # the oracle rounds to fp32 first (the 2^-30 is lost), then ties to even: 1
    B = np.array([[1.0, 2.0 ** -8, 2.0 ** -30]])
    assert P.check_u(_bits(1.0)[None], B, h) == (0, 1)
    assert P.check_u(_bits(1.0 + 2.0 ** -7)[None], B, h) == (1, 1)
    for wrong in (1.0 + 2.0 ** -6, 1.0 - 2.0 ** -8):
        try:
            P.check_u(_bits(wrong)[None], B, h)
        except AssertionError:
            pass
        else:
            raise AssertionError("a value that is not a bf16 neighbour passed")
    # exact u = 1 + 2^-9 is a quarter ulp from 1: only 1 is correct
    B2 = np.array([[1.0, 2.0 ** -9, 0.0]])
    assert P.check_u(_bits(1.0)[None], B2, h) == (0, 0)
    try:
        P.check_u(_bits(1.0 + 2.0 ** -7)[None], B2, h)
    except AssertionError:
        pass
    else:
        raise AssertionError("a flip of an unambiguous element passed")


def test_check_u_under_cancellation():
    # exact u = 2^-20, but the fp32 error bound (15 roundings of |terms| ~ 2)
    # is ~1.8e-6: any bf16 value the interval [x - e, x + e] rounds to is right
    h = np.array([[1.0, 1.0, 1.0]])
    B = np.array([[1.0, -1.0, 2.0 ** -20]])
    e = P.u_gamma(3, 1) * (2.0 + 2.0 ** -20)
    assert e > 2.0 ** -20
    assert P.check_u(_bits(2.0 ** -19)[None], B, h) == (1, 1)
    assert P.check_u(_bits(0.0)[None], B, h) == (1, 1)
    for wrong in (2.0 ** -17, -(2.0 ** -19)):
        try:
            P.check_u(_bits(wrong)[None], B, h)
        except AssertionError:
            pass
        else:
            raise AssertionError("a value outside the error interval passed")
    sl = P.u_slack(np.array([[1.0]]), B, h)
    assert e - 2.0 ** -26 <= sl[0, 0] <= e + 2.0 ** -26   # both ends rounded to bf16


def test_u_slack_counts_only_ambiguous_elements():
    h = np.array([[1.0, 1.0, 1.0]])
    B = np.array([[1.0, 2.0 ** -8, 2.0 ** -30],     # ambiguous (ulp 2^-7)
                  [1.0, 2.0 ** -9, 0.0]])           # not
    A = np.array([[3.0, 5.0], [-2.0, 7.0]])
    sl = P.u_slack(A, B, h)
    np.testing.assert_allclose(sl, [[3.0 * 2.0 ** -7, 2.0 * 2.0 ** -7]])


def test_excused_ids_split_band_and_slack():
    # oracle top-2 of a 4-entry tile (token ids 0..3): scores 10, 9, 8.995, 5
    scores = np.array([[10.0, 9.0, 8.995, 5.0]])
    tok = np.arange(4)
    # id 2 for id 1: gap 0.005 < 1e-3 * 9 = 0.009 -> band
    r = P.check_ids("local", np.array([[0, 2]]), scores, tok, 4, 2)
    assert (r["band"], r["slack"]) == (2, 0)
    # scores 10, 9, 8.98: gap 0.02 is outside the band, inside a slack of 0.02
    s2 = np.array([[10.0, 9.0, 8.98, 5.0]])
    sl = np.array([[0.0, 0.01, 0.011, 0.0]])
    r = P.check_ids("local", np.array([[0, 2]]), s2, tok, 4, 2, slack_pos=sl)
    assert (r["band"], r["slack"]) == (1, 1)      # id 1 itself is at gap 0
    try:
        P.check_ids("local", np.array([[0, 2]]), s2, tok, 4, 2)
    except AssertionError:
        pass
    else:
        raise AssertionError("an id outside the band passed without slack")
    try:
        P.check_ids("local", np.array([[0, 3]]), scores, tok, 4, 2)
    except AssertionError:
        pass
    else:
        raise AssertionError("a wrong id passed")
