"""Parity rules between the CUDA path and the fp64 oracle.

* Ids: per row (and per tile in local mode) the GPU's candidate set equals the
  oracle's, except at boundary ranks: an element in either difference is
  excused only if its oracle score is within 1e-3*|s_C| of s_C, the oracle's
  C-th best score (global) or k_tile-th best within its tile (local).
  Excused elements are counted and returned.
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


def _check_set(gpu, ora, score_of, s_C, where):
    g, o = set(gpu.tolist()), set(ora.tolist())
    if len(g) != len(gpu):
        raise AssertionError(f"{where}: duplicate ids in GPU output")
    diff = g ^ o
    bad = [x for x in diff if not abs(score_of[x] - s_C) < ID_REL * abs(s_C)]
    if bad:
        raise AssertionError(f"{where}: {len(bad)} ids differ beyond the boundary band "
                             f"(e.g. id {bad[0]} score {score_of[bad[0]]:.6g} vs s_C {s_C:.6g})")
    return len(diff)


def check_ids(mode, gpu_ids, scores_pos, token_ids, C_or_tile, k_tile=0):
    """gpu_ids: M x K int array. scores_pos: oracle scores M x n by position.
    Returns the number of excused boundary elements."""
    M = gpu_ids.shape[0]
    n = scores_pos.shape[1]
    token_ids = np.asarray(token_ids)
    excused = 0
    for m in range(M):
        score_of = np.empty(n)
        score_of[token_ids] = scores_pos[m]
        if mode == "global":
            ora, vals = O.global_topk(scores_pos[m], token_ids, C_or_tile)
            excused += _check_set(gpu_ids[m], ora, score_of, vals[-1], f"row {m}")
        else:
            T = C_or_tile
            off = 0
            for t0 in range(0, n, T):
                seg = slice(t0, min(n, t0 + T))
                ora, vals = O.global_topk(scores_pos[m][seg], token_ids[seg], k_tile)
                cnt = len(ora)
                excused += _check_set(gpu_ids[m, off:off + cnt], ora, score_of, vals[-1],
                                      f"row {m} tile {t0 // T}")
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
