"""CPU oracle of the steps that consume the draft distribution q.

TEST INFRASTRUCTURE ONLY, like lmhead_oracle: nothing in the product path
imports it, and it shares no code with the CUDA library.

Sources:
* [E1] "EAGLE -> EAGLE-2 -> EAGLE-3 -> DFlash" (course.zhidx.com), the
  EAGLE-2 dynamic draft tree, "Expansion Phase": a node's value is the
  product of the draft confidences along its path; only the top nodes by
  value of the current layer are expanded, each into its most likely draft
  tokens.
* [P2] "Speculative decoding and EAGLE" (ai-engineering.com.cn), the
  exactness rule: for each drafted token x, draw r ~ U(0, 1); accept if
  r < p(x) / q(x); otherwise draw the replacement from (p - q)+ normalised
  and stop; when every drafted token is accepted, draw one more token from
  the target. The page's exercise checks the output distribution against
  plain sampling from the target (total variation < 0.01 over 10K samples).

Readings (numbered R17-R20):
  R17 The page's printed listing subtracts the scalar q(x_t) from the target
      row; the exactness the page states (the output is distributed as p)
      holds for the pointwise residual (p - q)+ with the whole draft
      distribution q, so that is what is computed here. A test shows the
      listing's form failing the page's own TV check.
  R18 q is the head's candidate-supported distribution: zero outside the
      row's candidates. A drafted token is one of its row's candidates.
  R19 Random draws are inputs. Sampling from q (the drafter's own draw) uses
      the Gumbel-max construction on per-candidate uniforms; the residual and
      bonus draws use the inverse CDF in vocabulary order with one uniform.
  R20 Draft selection order: q descending, ties by the smaller vocabulary id;
      a child's value is the parent's value times q, rounded to fp32 (the
      precision the kernel multiplies in).
"""
from __future__ import annotations

import numpy as np

__all__ = ["draft_topk", "gumbel_scores", "gumbel_sample", "inverse_cdf_sample",
           "residual", "verify_chain"]


def draft_topk(q: np.ndarray, ids: np.ndarray, k_sel: int, parent_value: float = 1.0):
    """EAGLE-2 expansion of one node ([E1], Expansion Phase): its k_sel most
    likely draft tokens (q descending, ties by smaller id, R20) and their path
    values parent_value * q (fp32 product)."""
    q = np.asarray(q, dtype=np.float32)
    ids = np.asarray(ids)
    order = np.lexsort((ids, -q.astype(np.float64)))[:k_sel]
    top_q = q[order]
    value = np.float32(parent_value) * top_q  # fp32 x fp32 -> fp32
    return ids[order], top_q, value.astype(np.float32)


def gumbel_scores(q: np.ndarray, u: np.ndarray) -> np.ndarray:
    """log q_j + g_j with g_j = -log(-log u_j) (fp64); -inf where q_j = 0."""
    q64 = np.asarray(q, dtype=np.float64)
    u64 = np.asarray(u, dtype=np.float64)
    with np.errstate(divide="ignore"):
        s = np.log(q64) - np.log(-np.log(u64))
    s[q64 <= 0] = -np.inf
    return s


def gumbel_sample(q: np.ndarray, ids: np.ndarray, u: np.ndarray):
    """One draw from q by Gumbel-max (R19): the candidate with the largest
    perturbed log-probability (ties by smaller id). Returns (id, index, scores)."""
    s = gumbel_scores(q, u)
    j = int(np.lexsort((np.asarray(ids), -s))[0])
    return int(ids[j]), j, s


def inverse_cdf_sample(w: np.ndarray, u: float) -> int:
    """Smallest index v with sum(w[:v+1]) > u * sum(w) (fp64, vocabulary
    order; w >= 0, sum > 0)."""
    w64 = np.asarray(w, dtype=np.float64)
    c = np.cumsum(w64)
    return int(min(np.searchsorted(c, u * c[-1], side="right"), w64.size - 1))


def residual(p_row: np.ndarray, cand_ids: np.ndarray, cand_q: np.ndarray) -> np.ndarray:
    """(p - q)+ over the whole vocabulary, q zero outside the candidates (R17, R18)."""
    w = np.asarray(p_row, dtype=np.float64).copy()
    w[np.asarray(cand_ids)] -= np.asarray(cand_q, dtype=np.float64)
    return np.maximum(w, 0.0)


def verify_chain(p: np.ndarray, x: np.ndarray, cand_ids: np.ndarray, cand_q: np.ndarray,
                 r: np.ndarray, u: np.ndarray):
    """The exactness rule over one chain of Kd drafted tokens ([P2]).

    p: (Kd + 1) x n target probabilities; x: Kd drafted vocabulary ids;
    cand_ids, cand_q: Kd x K candidate lists of the drafter (q per R18);
    r: Kd accept uniforms; u: Kd + 1 sampling uniforms.
    The accept test is taken in fp32, the precision the kernel decides it in:
    fp32(r) < fp32(p(x)) / fp32(q(x)).
    Returns (accepted count, output tokens: the accepted drafts followed by the
    replacement or bonus token)."""
    Kd = len(x)
    out = []
    for t in range(Kd):
        ids_t = np.asarray(cand_ids[t])
        hit = np.nonzero(ids_t == x[t])[0]
        if hit.size == 0:
            raise ValueError("drafted token is not a candidate of its row (R18)")
        qx = np.float32(cand_q[t][hit[0]])
        px = np.float32(p[t][x[t]])
        if np.float32(r[t]) < np.float32(px / qx):
            out.append(int(x[t]))
            continue
        w = residual(p[t], ids_t, cand_q[t])
        if not w.sum() > 0:  # p <= q everywhere: then p = q and rejection cannot happen
            w = np.asarray(p[t], dtype=np.float64)
        out.append(inverse_cdf_sample(w, float(u[t])))
        return t, out
    out.append(inverse_cdf_sample(p[Kd], float(u[Kd])))
    return Kd, out
