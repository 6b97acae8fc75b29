"""CPU oracle of the cluster-level two-stage head (the third route).

TEST INFRASTRUCTURE ONLY, like lmhead_oracle: nothing in the product path
imports it, and it shares no code with the CUDA library.

Source: [E4] "EAGLE-4" design notes, qingkeai.online/blog/EAGLE, section
"EAGLE Efficient LM Head", the third of the three routes tried: the tokens are
split into groups (128 tokens per group in the example), a few groups are
selected first, then the logits of every token inside the selected groups are
computed and the draft token is sampled from them. The same section says the
route lost acceptance length against the full head, which is why the notes
chose the token-level route; it is built here as a second candidate scheme on
the same library.

Readings where the section is silent (numbered R21-R23):
  R21 A group is `group` consecutive rows of the head as stored (rows
      [g*group, (g+1)*group)), so a selected group is one contiguous block of
      W. The group size must divide n (every vocabulary size in the workloads
      is a multiple of 128); a ragged last group is refused.
  R22 The group selector is the token-level route's own first stage: a
      group's score is the largest low-rank score A(Bh) among its rows (u in
      bf16 as in R3, scores never below fp32). The G groups with the largest
      scores are kept, ties by the smaller group index; they are listed best
      first.
  R23 A row's candidates are its selected groups' rows, group by group in
      that order, ascending inside a group (G*group ids); logits are the exact
      W[ids].h and q their softmax as in R7.
"""
from __future__ import annotations

import numpy as np

from .lmhead_oracle import candidate_logits, candidate_softmax, lowrank_scores, project_u

__all__ = ["group_scores", "select_groups", "group_candidates", "cluster_two_stage"]


def group_scores(scores_row: np.ndarray, group: int) -> np.ndarray:
    """R22: the maximum low-rank score of each group of `group` consecutive
    rows. scores_row has n entries, n a multiple of `group` (R21)."""
    s = np.asarray(scores_row, dtype=np.float64)
    n = s.shape[0]
    if group < 1 or n % group:
        raise ValueError("the group size must divide n (R21)")
    best = np.empty(n // group)
    for g in range(n // group):
        best[g] = s[g * group:(g + 1) * group].max()
    return best


def select_groups(gscores: np.ndarray, G: int) -> np.ndarray:
    """R22: indices of the G best groups, score descending, ties by the
    smaller index."""
    gs = np.asarray(gscores, dtype=np.float64)
    if not 1 <= G <= gs.shape[0]:
        raise ValueError("G must be in [1, number of groups]")
    return np.lexsort((np.arange(gs.shape[0]), -gs))[:G].astype(np.int64)


def group_candidates(groups: np.ndarray, group: int) -> np.ndarray:
    """R23: every row of the selected groups, group by group in selection
    order, ascending inside a group."""
    out = []
    for g in np.asarray(groups):
        out.extend(range(int(g) * group, (int(g) + 1) * group))
    return np.asarray(out, dtype=np.int64)


def cluster_two_stage(W, A, B, h, group: int, G: int, temperature: float = 1.0):
    """The third route of [E4] row by row: u = bf16(B h), low-rank scores,
    group scores, the G best groups, exact logits of all their rows, softmax.
    W, A, B, h are float64 arrays of bf16 values (A in the head's row order).
    Returns dict(u, scores, gscores, groups, ids, logits, q); the last five
    are lists of per-row arrays."""
    u = project_u(B, h)
    S = lowrank_scores(A, u)
    out = {"u": u, "scores": S, "gscores": [], "groups": [], "ids": [], "logits": [], "q": []}
    for m in range(S.shape[0]):
        gsc = group_scores(S[m], group)
        sel = select_groups(gsc, G)
        ids = group_candidates(sel, group)
        L = candidate_logits(W, h[m], ids)
        out["gscores"].append(gsc)
        out["groups"].append(sel)
        out["ids"].append(ids)
        out["logits"].append(L)
        out["q"].append(candidate_softmax(L, temperature))
    return out
