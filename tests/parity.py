"""Parity rules between the CUDA path and the fp64 oracle.

* Ids: per row (and per tile in local mode) the GPU's candidate set equals the
  oracle's, except at boundary ranks: an element in either difference is
  excused only if its oracle score is within 1e-3*|s_C| of s_C, the oracle's
  C-th best score (global) or k_tile-th best within its tile (local), widened
  by the u-rounding slack below. Excused elements are counted and returned.
* u-rounding slack (reading R3: u is rounded to bf16 after an fp32 sum): the
  GPU's fp32 sum s of B[k].h[m] lies within e = gamma_D * sum_i |B[k,i] h[m,i]|
  of the exact value x, gamma_D = D u / (1 - D u), u = 2^-24, where D is the
  largest number of fp32 roundings a product passes through in the
  projection kernel the library runs at (d, M); see projection_depth(). Its
  bf16 rounding is therefore one of the bf16 values from bf16(x - e) to
  bf16(x + e) (rounding is monotone), and any of them is correct. Usually
  that is the oracle's value or its neighbour; where the sum cancels (|x|
  far below e) it can be several bf16 steps away. A position j's score then
  moves by at most slack_j = sum_k |A[j,k]| * dev_k, dev_k the larger
  distance from the oracle's u_k to those two ends (0 where they agree).
  check_u() verifies the GPU's own u against that interval: the model is
  checked, not assumed.
* Logits: |L_gpu - L_exact| <= 2e-3 * max(|L_exact|, 1), L_exact = W[id].h in
  fp64 for the GPU's own ids.
* q: within 1e-4 absolute of the softmax of the exact logits over the GPU's
  own candidate set (equal to the oracle's q whenever the sets are equal).
"""
from __future__ import annotations

import numpy as np

import oracle as O

ID_REL = 1e-3
LOGIT_REL = 2e-3
Q_ABS = 1e-4


U_UNIT = 2.0 ** -24   # unit roundoff of fp32

# Every checked case appends a summary here; tests/conftest.py prints them at
# the end of the session (band / slack counts, u flips, how much q spreads).
REPORT = []


def record(case, **fields):
    REPORT.append({"case": case, **fields})


def projection_depth(d, M):
    """Largest number of fp32 roundings one product B[k,i]*h[m,i] passes
    through before u[m,k] is rounded to bf16, for the projection kernel the
    library runs at (d, M) (the dispatch of launch_project_u):

    * M <= 8, d <= 8192 (GEMV; vpt = ceil(d/1024) 16-byte pieces per thread,
      run as a template of VPT = 1, 2, 4 or, at M <= 4, 8): an 8-term FMA chain
      from zero (7 roundings: the first product is exact), the thread's sum of
      VPT such chains (VPT - 1), a 5-level warp butterfly and the sum of the
      4 warps' partials from zero (3): D = 14 + VPT.
    * d <= 5120 otherwise (tensor cores): the cluster of KS = min(8,
      ceil(d/512)) CTAs splits d into slices of kslice = 64*ceil(d/KS/64);
      each CTA accumulates kslice/16 MMA steps (K = 16) in fp32 TMEM. The
      tensor core's internal alignment may truncate rather than round, so a
      step counts as 2 roundings (an error of one fp32 ulp, 2u, of the
      magnitudes summed); then the KS partials are added from zero in rank
      order (KS - 1): D = 2*kslice/16 + KS - 1.
    * otherwise (CUDA cores, 8-element pieces strided over a warp): a chain
      of 8*ceil(d/256) FMAs per lane, then the 5-level butterfly."""
    if M <= 8 and d <= 8192:
        vpt = (d + 1023) // 1024
        VPT = 1 if vpt <= 1 else 2 if vpt <= 2 else 4 if vpt <= 4 else (8 if M <= 4 else 0)
        if VPT:
            return 14 + VPT
    if d <= 5120:
        KS = min(8, (d + 511) // 512)
        per_cta = -(-d // KS)                            # ceil(d / KS)
        kslice = -(-per_cta // 64) * 64                 # rounded up to 64 columns
        return 2 * (kslice // 16) + KS - 1
    return 8 * ((d + 255) // 256) - 1 + 5


def u_gamma(d, M):
    D = projection_depth(d, M)
    return D * U_UNIT / (1.0 - D * U_UNIT)


def _u_exact(B64, h64):
    exact = h64 @ B64.T                                  # M x r
    mag = np.abs(h64) @ np.abs(B64).T                   # sum_i |B[k,i] h[m,i]|
    return exact, mag


def u_interval(B64, h64, M_call):
    """Per element of u: the exact value x and the lowest and highest bf16
    values the projection may return, bf16(x - e) and bf16(x + e), e the
    fp32 error bound of the kernel the library runs at (d, M_call)."""
    exact, mag = _u_exact(B64, h64)
    e = u_gamma(B64.shape[1], M_call) * mag
    return exact, O.round_to_bf16(exact - e), O.round_to_bf16(exact + e)


def u_slack(A64, B64, h64, M_call=None):
    """Per row m and position p: the most the score of p can move when u
    takes another value of its interval (see the module docstring). M_call
    is the number of hidden vectors of the library call (it picks the
    projection kernel); default h64's rows."""
    M_call = h64.shape[0] if M_call is None else M_call
    _, lo, hi = u_interval(B64, h64, M_call)
    want = O.project_u(B64, h64)
    dev = np.maximum(np.abs(hi - want), np.abs(lo - want))
    return dev @ np.abs(A64).T                          # M x n by position


def check_u(gpu_u_bits, B64, h64, M_call=None):
    """The GPU's u against the oracle's: every element equals the oracle's
    bf16 rounding or lies in its interval [bf16(x - e), bf16(x + e)].
    Returns (elements that differ from the oracle, elements whose interval
    holds more than one value)."""
    M_call = h64.shape[0] if M_call is None else M_call
    want = O.project_u(B64, h64)
    got = O.bf16_bits_to_f64(gpu_u_bits)
    exact, lo, hi = u_interval(B64, h64, M_call)
    bad = (got != want) & ~((got >= lo) & (got <= hi))
    if bad.any():
        m, k = np.argwhere(bad)[0]
        raise AssertionError(f"u[{m},{k}]: gpu {got[m, k]!r} oracle {want[m, k]!r} exact "
                             f"{exact[m, k]!r}, allowed [{lo[m, k]!r}, {hi[m, k]!r}]")
    return int((got != want).sum()), int((lo != hi).sum())


def _check_set(gpu, ora, score_of, slack_of, s_C, id_C, where):
    """Excused elements of the symmetric difference, as (band, slack): band
    = within 1e-3*|s_C| of s_C, slack = excused only by the u-rounding slack."""
    g, o = set(gpu.tolist()), set(ora.tolist())
    if len(g) != len(gpu):
        raise AssertionError(f"{where}: duplicate ids in GPU output")
    band = slack = 0
    bad = []
    for x in g ^ o:
        gap = abs(score_of[x] - s_C)
        if gap < ID_REL * abs(s_C):
            band += 1
        elif gap < ID_REL * abs(s_C) + slack_of[x] + slack_of[id_C]:
            slack += 1
        else:
            bad.append(x)
    if bad:
        raise AssertionError(f"{where}: {len(bad)} ids differ beyond the boundary band "
                             f"(e.g. id {bad[0]} score {score_of[bad[0]]:.6g} vs s_C {s_C:.6g}, "
                             f"slack {slack_of[bad[0]] + slack_of[id_C]:.3g})")
    return band, slack


def check_ids(mode, gpu_ids, scores_pos, token_ids, C_or_tile, k_tile=0, slack_pos=None):
    """gpu_ids: M x K int array. scores_pos: oracle scores M x n by position;
    slack_pos: u-rounding slack M x n by position (or None). Returns the
    excused boundary elements as {"band": b, "slack": s, "compared": c}: b
    within the 1e-3 band, s needing the u-rounding slack, c ids compared."""
    M = gpu_ids.shape[0]
    n = scores_pos.shape[1]
    token_ids = np.asarray(token_ids)
    band = slack = 0
    for m in range(M):
        score_of = np.empty(n)
        score_of[token_ids] = scores_pos[m]
        slack_of = np.zeros(n)
        if slack_pos is not None:
            slack_of[token_ids] = slack_pos[m]
        if mode == "global":
            ora, vals = O.global_topk(scores_pos[m], token_ids, C_or_tile)
            b, s = _check_set(gpu_ids[m], ora, score_of, slack_of, vals[-1], ora[-1], f"row {m}")
            band, slack = band + b, slack + s
        else:
            T = C_or_tile
            off = 0
            for t0 in range(0, n, T):
                seg = slice(t0, min(n, t0 + T))
                ora, vals = O.global_topk(scores_pos[m][seg], token_ids[seg], k_tile)
                cnt = len(ora)
                b, s = _check_set(gpu_ids[m, off:off + cnt], ora, score_of, slack_of,
                                  vals[-1], ora[-1], f"row {m} tile {t0 // T}")
                band, slack = band + b, slack + s
                off += cnt
            assert off == gpu_ids.shape[1]
    return {"band": band, "slack": slack, "compared": int(gpu_ids.size)}


def check_order(mode, gpu_ids, gpu_scores, C_or_tile, k_tile, n):
    """GPU-reported approximate scores are non-increasing within each
    global row / local tile."""
    M, K = gpu_ids.shape
    if mode == "global":
        assert np.all(np.diff(gpu_scores, axis=1) <= 0)
        return
    off = 0
    for t0 in range(0, n, C_or_tile):
        cnt = min(k_tile, min(n, t0 + C_or_tile) - t0)
        assert np.all(np.diff(gpu_scores[:, off:off + cnt], axis=1) <= 0)
        off += cnt


def exact_logits(W_bits, h64, ids):
    """fp64 W[ids[m,j]] . h[m] for every GPU id (decoding only those rows)."""
    M, K = ids.shape
    out = np.empty((M, K))
    for m in range(M):
        rows = O.bf16_bits_to_f64(W_bits[ids[m]])
        out[m] = O.candidate_logits(rows, h64[m], np.arange(K))
    return out


def check_logits(gpu_L, exact):
    err = np.abs(gpu_L - exact)
    bound = LOGIT_REL * np.maximum(np.abs(exact), 1.0)
    bad = err > bound
    if bad.any():
        i = np.argwhere(bad)[0]
        raise AssertionError(f"logit mismatch at {tuple(i)}: gpu {gpu_L[tuple(i)]:.7g} "
                             f"exact {exact[tuple(i)]:.7g}")
    return int((np.abs(exact) < 1.0).sum())  # entries where the floor applied


def check_q(gpu_q, exact_L, temperature=1.0):
    """q within Q_ABS of the softmax of the exact logits over the GPU's set.
    Returns how much the check bites: the median over rows of the largest q
    and of the number of candidates with q > Q_ABS (a one-hot row has 1)."""
    qmax, live = [], []
    for m in range(gpu_q.shape[0]):
        want = O.candidate_softmax(exact_L[m], temperature)
        err = np.abs(gpu_q[m] - want).max()
        if err > Q_ABS:
            raise AssertionError(f"q row {m}: max abs error {err:.3g}")
        assert abs(gpu_q[m].sum() - 1.0) < 1e-3
        qmax.append(float(want.max()))
        live.append(int((want > Q_ABS).sum()))
    return {"q_max_median": float(np.median(qmax)), "q_live_median": float(np.median(live))}


def check_groups(gpu_groups, scores_pos, group, G, slack_pos=None):
    """Cluster-level selection: per row, the GPU's G groups equal the
    oracle's G best groups by their best low-rank score, except at boundary
    ranks (same band as check_ids, the slack of a group being its rows'
    largest). Scores are by row of the head as stored (no shuffle).
    Returns the number of excused groups."""
    M, n = scores_pos.shape
    ng = n // group
    excused = 0
    for m in range(M):
        gsc = O.group_scores(scores_pos[m], group)
        gsl = (np.zeros(ng) if slack_pos is None
               else np.asarray(slack_pos[m]).reshape(ng, group).max(axis=1))
        ora = O.select_groups(gsc, G)
        b, s = _check_set(np.asarray(gpu_groups[m]), ora, gsc, gsl, gsc[ora[-1]], ora[-1],
                          f"row {m} groups")
        excused += b + s
    return excused
