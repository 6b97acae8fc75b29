"""fp64 CPU oracle of the two-stage draft LM head.

TEST INFRASTRUCTURE ONLY. Nothing in the product path imports this module:
only tests/, the smoke check in __graft_entry__ and bench.py's CPU-baseline
leg may use it. It shares no code with the CUDA library (draft_lm_head_gb300)
and imports nothing from it.

Every function is a plain, slow restatement of what the pages define, in
NumPy float64, on the same bf16 input bits that the GPU consumes. Sources:

* [E4] "EAGLE-4" design notes, qingkeai.online/blog/EAGLE:
  - section "EAGLE Efficient LM Head" (two-stage, token level: a cheap
    full-vocabulary score, Top-k candidates, exact logits of the candidates
    from the original hidden state);
  - section "A training-free version: Freq-aware SVD" and its equation
    (A = F^-1/2 U_r S_r, B = V_r^T where F^1/2 W = U S V^T; smoothed f_i > 0;
    candidates from Top-k of A(Bh));
  - section "A Local Top-k based variant" (the original flow u = B h,
    scores = A u, ids = topk(scores, C), logits = W[ids] h; the fused flow
    with a per-vocab-tile top-k_tile written through tile.token_ids and
    concatenated; vocabulary rows shuffled before tiling).
* [E1] "EAGLE -> EAGLE-2 -> EAGLE-3 -> DFlash" (course.zhidx.com), section
  1.3: the drafter maps its feature through the LM head to a distribution and
  samples from it. [P2] "Speculative decoding and EAGLE"
  (ai-engineering.com.cn): the draft distribution q is what the accept/reject
  rule consumes. Together these are why stage 2 ends in a softmax.

Readings where the pages are silent (numbered R3-R15):
  R3  u is rounded to bf16 after the projection (the pseudocode's u = B @ h on
      bf16 tensors); the rounding is decided in fp32, as the kernel decides it.
  R4  scores are never rounded below fp32 (fp64 here).
  R5  Top-k ties: the smaller vocabulary id wins.
  R6  a partial last tile keeps min(k_tile, rows) candidates.
  R7  q is the softmax restricted to a row's own candidates, divided by a
      temperature (1 by default); non-candidates have q = 0.
  R8  local mode keeps all tiles x k_tile candidates (no re-selection).
  R9  the shuffle permutes the rows of A only; ids are reported in
      vocabulary space through token_ids (position -> vocabulary id).
  R10 every hidden vector (row of h) gets its own candidates and its own q.
  R15 the pruned head keeps the n_keep most frequent tokens (ties: smaller id).
"""
from __future__ import annotations

import math

import numpy as np

__all__ = [
    "bf16_bits_to_f64", "round_f64_to_f32", "round_to_bf16", "smooth_freq",
    "freq_aware_svd", "freq_svd_gram", "project_u", "lowrank_scores",
    "topk_order", "global_topk", "local_topk", "candidate_logits",
    "candidate_softmax", "dense_logits", "pruned_ids", "exact_topk",
    "recall_at", "two_stage", "local_candidate_count",
]


# ------------------------------------------------------------------ numbers
def bf16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    """Exact value of bf16 bit patterns (uint16) as float64.

    A bf16 number is the upper 16 bits of an IEEE binary32: sign, 8-bit
    exponent, 7-bit fraction. Decoded here field by field.
    """
    b = np.asarray(bits, dtype=np.int64)
    sign = np.where(b >> 15, -1.0, 1.0)
    exp = (b >> 7) & 0xFF
    frac = (b & 0x7F).astype(np.float64)
    normal = sign * np.ldexp(1.0 + frac / 128.0, (exp - 127).astype(np.int64))
    sub = sign * np.ldexp(frac / 128.0, -126)
    out = np.where(exp == 0, sub, normal)
    out = np.where(exp == 0xFF, np.where(frac == 0, sign * np.inf, np.nan), out)
    return out.astype(np.float64)


def _round_to_precision(x: np.ndarray, mant_bits: int, emin: int) -> np.ndarray:
    """Round float64 values to a binary format with `mant_bits` significant
    bits (implicit bit included) and minimum normal exponent `emin`, nearest
    with ties to even. Overflow is not handled (inputs here are small)."""
    x = np.asarray(x, dtype=np.float64)
    out = np.zeros_like(x)
    nz = x != 0
    _, e = np.frexp(x[nz])            # x = m * 2^e, 0.5 <= |m| < 1
    e = np.maximum(e - 1, emin)       # exponent of the leading bit
    quantum = np.ldexp(1.0, e - (mant_bits - 1))
    out[nz] = np.rint(x[nz] / quantum) * quantum   # rint: ties to even
    return out


def round_f64_to_f32(x: np.ndarray) -> np.ndarray:
    """IEEE binary32 rounding (24 significant bits), as float64 values."""
    return _round_to_precision(x, 24, -126)


def round_to_bf16(x: np.ndarray) -> np.ndarray:
    """bf16 rounding (8 significant bits, binary32 exponent range)."""
    return _round_to_precision(x, 8, -126)


# ----------------------------------------------------------- Freq-aware SVD
def smooth_freq(counts: np.ndarray) -> np.ndarray:
    """[E4] Freq-aware SVD: the frequency weights must be smoothed so every
    f_i > 0. Reading: add-one smoothing of the raw counts."""
    return np.asarray(counts, dtype=np.float64) + 1.0


def freq_aware_svd(W: np.ndarray, f: np.ndarray, r: int):
    """[E4] Freq-aware SVD equation, taken literally.

    F = diag(f). Take the SVD of F^1/2 W = U S V^T, keep the r largest
    singular values, and undo the row scaling on the left factor:
    A = F^-1/2 U_r S_r (n x r), B = V_r^T (r x d). Returns (A, B, S) where S
    holds all singular values of F^1/2 W.
    """
    W = np.asarray(W, dtype=np.float64)
    sq = np.sqrt(np.asarray(f, dtype=np.float64))
    U, S, Vt = np.linalg.svd(sq[:, None] * W, full_matrices=False)
    A = (U[:, :r] * S[:r]) / sq[:, None]
    B = Vt[:r].copy()
    return A, B, S


def freq_svd_gram(W: np.ndarray, f: np.ndarray, r: int):
    """Same factors through the Gram matrix, for heads too tall for a direct
    SVD. With F^1/2 W = U S V^T, (F^1/2 W)^T (F^1/2 W) = W^T F W = V S^2 V^T,
    so V_r are its top-r eigenvectors, and U_r S_r = F^1/2 W V_r gives
    A = F^-1/2 U_r S_r = W V_r and B = V_r^T. Returns (A, B, S) with S the
    singular values sqrt(max(eig, 0)) in descending order."""
    W = np.asarray(W, dtype=np.float64)
    G = W.T @ (np.asarray(f, dtype=np.float64)[:, None] * W)
    evals, evecs = np.linalg.eigh(G)
    order = np.argsort(evals)[::-1]
    V = evecs[:, order[:r]]
    return W @ V, V.T.copy(), np.sqrt(np.maximum(evals[order], 0.0))


# ------------------------------------------------------------- stage 1
def project_u(B: np.ndarray, h: np.ndarray) -> np.ndarray:
    """[E4] u = B @ h per hidden vector. Reading R3: u is stored in bf16 and
    the rounding is decided in fp32: the exact fp64 product is rounded to
    binary32, then to bf16. Returns float64 values on the bf16 grid, M x r."""
    u = np.asarray(h, dtype=np.float64) @ np.asarray(B, dtype=np.float64).T
    return round_to_bf16(round_f64_to_f32(u))


def lowrank_scores(A: np.ndarray, u: np.ndarray) -> np.ndarray:
    """[E4] scores = A @ u for every vocabulary row (fp64, reading R4).
    A is indexed by position (row order as stored); returns M x n."""
    return np.asarray(u, dtype=np.float64) @ np.asarray(A, dtype=np.float64).T


def topk_order(scores: np.ndarray, ids: np.ndarray) -> np.ndarray:
    """Indices of `scores` sorted by (score descending, id ascending) (R5)."""
    return np.lexsort((np.asarray(ids), -np.asarray(scores, dtype=np.float64)))


def global_topk(scores_row: np.ndarray, token_ids: np.ndarray, C: int):
    """[E4] original flow: ids = topk(scores, C) over the whole vocabulary.
    scores_row is indexed by position; token_ids maps position -> vocabulary
    id. Returns (vocab ids, scores), best first."""
    order = topk_order(scores_row, token_ids)[:C]
    return np.asarray(token_ids)[order].astype(np.int64), np.asarray(scores_row)[order]


def local_candidate_count(n: int, T: int, k_tile: int) -> int:
    """Candidates per row of local mode: every tile keeps min(k_tile, rows)."""
    full, tail = divmod(n, T)
    return full * min(k_tile, T) + (min(k_tile, tail) if tail else 0)


def local_topk(scores_row: np.ndarray, token_ids: np.ndarray, T: int, k_tile: int):
    """[E4] Local Top-k variant: for each vocabulary tile of T consecutive
    positions, keep the top k_tile by score (R5 ties, R6 short last tile) and
    store tile.token_ids[local_ids]; ids = concat over tiles in tile order.
    Returns (vocab ids, scores), tile order, best first within a tile."""
    scores_row = np.asarray(scores_row, dtype=np.float64)
    token_ids = np.asarray(token_ids)
    n = scores_row.shape[0]
    ids, vals = [], []
    for t0 in range(0, n, T):
        seg = slice(t0, min(n, t0 + T))
        order = topk_order(scores_row[seg], token_ids[seg])[:k_tile]
        ids.append(token_ids[seg][order])
        vals.append(scores_row[seg][order])
    return np.concatenate(ids).astype(np.int64), np.concatenate(vals)


# ------------------------------------------------------------- stage 2
def candidate_logits(W: np.ndarray, h_row: np.ndarray, ids: np.ndarray) -> np.ndarray:
    """[E4] logits = W[ids] @ h with the original hidden state, fp64."""
    return np.asarray(W, dtype=np.float64)[np.asarray(ids)] @ np.asarray(h_row, dtype=np.float64)


def candidate_softmax(logits: np.ndarray, temperature: float = 1.0) -> np.ndarray:
    """Draft distribution over one row's candidates (reading R7):
    q_j = exp((L_j - max L)/T) / sum_k exp((L_k - max L)/T)."""
    z = (np.asarray(logits, dtype=np.float64) - np.max(logits)) / temperature
    e = np.exp(z)
    return e / e.sum()


def dense_logits(W: np.ndarray, h: np.ndarray) -> np.ndarray:
    """[E4] the full LM head whose cost motivates the method: W h for all n."""
    return np.asarray(h, dtype=np.float64) @ np.asarray(W, dtype=np.float64).T


def pruned_ids(f: np.ndarray, n_keep: int) -> np.ndarray:
    """[E4] the vocabulary-pruning baseline (keep the n_keep most frequent
    tokens, 32000 in the pages). Ties: smaller id. Returned ascending."""
    f = np.asarray(f, dtype=np.float64)
    order = np.lexsort((np.arange(f.shape[0]), -f))[:n_keep]
    return np.sort(order).astype(np.int64)


# ------------------------------------------------------------- metrics
def exact_topk(Z_row: np.ndarray, K: int) -> np.ndarray:
    """Top-K vocabulary ids of the exact full-head logits (Z desc, id asc)."""
    return topk_order(Z_row, np.arange(Z_row.shape[0]))[:K].astype(np.int64)


def recall_at(cand_ids: np.ndarray, Z_row: np.ndarray, K: int) -> float:
    """|candidates ∩ exact Top-K| / K."""
    top = exact_topk(Z_row, K)
    return float(np.isin(top, np.asarray(cand_ids)).sum()) / K


# ------------------------------------------------------------- composition
def two_stage(W, A, B, h, token_ids, mode: str, C_or_tile: int, k_tile: int = 0,
              temperature: float = 1.0):
    """Both flows of [E4], row by row (R10). W, A, B, h are float64 arrays of
    bf16 values; A is in position order, token_ids maps position -> vocab id.
    mode 'global': ids = topk(A u, C); mode 'local': per-tile top-k_tile.
    Returns dict(u, scores, ids, approx, logits, q), ids/approx/logits/q as
    lists of per-row arrays."""
    u = project_u(B, h)
    S = lowrank_scores(A, u)
    out = {"u": u, "scores": S, "ids": [], "approx": [], "logits": [], "q": []}
    for m in range(S.shape[0]):
        if mode == "global":
            ids, s = global_topk(S[m], token_ids, C_or_tile)
        elif mode == "local":
            ids, s = local_topk(S[m], token_ids, C_or_tile, k_tile)
        else:
            raise ValueError(mode)
        L = candidate_logits(W, h[m], ids)
        out["ids"].append(ids)
        out["approx"].append(s)
        out["logits"].append(L)
        out["q"].append(candidate_softmax(L, temperature))
    return out


def fsum_dot(a, b) -> float:
    """Correctly rounded dot product (math.fsum) for small brute-force pins."""
    return math.fsum(float(x) * float(y) for x, y in zip(a, b))
