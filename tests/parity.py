"""Parity rules between the CUDA path and the fp64 oracle.

* Ids: per row (and per tile in local mode) the GPU's candidate set equals the
  oracle's, except at boundary ranks: an element in either difference is
  excused only if its oracle score is within 1e-3*|s_C| of s_C, the oracle's
  C-th best score (global) or k_tile-th best within its tile (local), widened
  by the u-rounding slack below. Excused elements are counted and returned.
* u-rounding slack (reading R3: u is rounded to bf16 after an fp32 sum): an
  element of u whose exact value B[k].h[m] lies within the fp32 summation
  error of a bf16 rounding midpoint may legitimately round either way. The
  bound is gamma * sum_i |B[k,i] h[m,i]| with gamma = 128 * 2^-24, the
  depth of the kernel's blocked fp32 summation (16-term MMA steps, at most
  d/16/KS steps per CTA, KS <= 8 cluster partials; < 64 roundings at
  d <= 5120) with a factor 2 margin. A flip moves the score of row j by at
  most |A[j,k]| * ulp(u_k), so slack_j = sum over ambiguous k of that.
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


U_GAMMA = 128 * 2.0 ** -24


def u_slack(A64, B64, h64):
    """Per row m and position p: the most the score of p can move when the
    ambiguous elements of u round the other way (see the module docstring)."""
    exact = h64 @ B64.T                                  # M x r
    mag = np.abs(h64) @ np.abs(B64).T                   # sum_i |B[k,i] h[m,i]|
    ax = np.abs(exact)
    _, e = np.frexp(np.where(ax > 0, ax, 1.0))          # ax = f * 2^e, 0.5 <= f < 1
    ulp = np.ldexp(1.0, e - 8)                          # bf16: 8 significant bits
    mid = (np.floor(ax / ulp) + 0.5) * ulp
    amb = np.abs(ax - mid) <= U_GAMMA * mag
    return (amb * ulp) @ np.abs(A64).T                  # M x n by position


def _check_set(gpu, ora, score_of, slack_of, s_C, id_C, where):
    g, o = set(gpu.tolist()), set(ora.tolist())
    if len(g) != len(gpu):
        raise AssertionError(f"{where}: duplicate ids in GPU output")
    diff = g ^ o
    bad = [x for x in diff
           if not abs(score_of[x] - s_C) < ID_REL * abs(s_C) + slack_of[x] + slack_of[id_C]]
    if bad:
        raise AssertionError(f"{where}: {len(bad)} ids differ beyond the boundary band "
                             f"(e.g. id {bad[0]} score {score_of[bad[0]]:.6g} vs s_C {s_C:.6g}, "
                             f"slack {slack_of[bad[0]] + slack_of[id_C]:.3g})")
    return len(diff)


def check_ids(mode, gpu_ids, scores_pos, token_ids, C_or_tile, k_tile=0, slack_pos=None):
    """gpu_ids: M x K int array. scores_pos: oracle scores M x n by position;
    slack_pos: u-rounding slack M x n by position (or None). Returns the
    number of excused boundary elements."""
    M = gpu_ids.shape[0]
    n = scores_pos.shape[1]
    token_ids = np.asarray(token_ids)
    excused = 0
    for m in range(M):
        score_of = np.empty(n)
        score_of[token_ids] = scores_pos[m]
        slack_of = np.zeros(n)
        if slack_pos is not None:
            slack_of[token_ids] = slack_pos[m]
        if mode == "global":
            ora, vals = O.global_topk(scores_pos[m], token_ids, C_or_tile)
            excused += _check_set(gpu_ids[m], ora, score_of, slack_of, vals[-1], ora[-1],
                                  f"row {m}")
        else:
            T = C_or_tile
            off = 0
            for t0 in range(0, n, T):
                seg = slice(t0, min(n, t0 + T))
                ora, vals = O.global_topk(scores_pos[m][seg], token_ids[seg], k_tile)
                cnt = len(ora)
                excused += _check_set(gpu_ids[m, off:off + cnt], ora, score_of, slack_of,
                                      vals[-1], ora[-1], f"row {m} tile {t0 // T}")
                off += cnt
            assert off == gpu_ids.shape[1]
    return excused


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
    for m in range(gpu_q.shape[0]):
        want = O.candidate_softmax(exact_L[m], temperature)
        err = np.abs(gpu_q[m] - want).max()
        if err > Q_ABS:
            raise AssertionError(f"q row {m}: max abs error {err:.3g}")
        assert abs(gpu_q[m].sum() - 1.0) < 1e-3


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
        excused += _check_set(np.asarray(gpu_groups[m]), ora, gsc, gsl, gsc[ora[-1]], ora[-1],
                              f"row {m} groups")
    return excused
