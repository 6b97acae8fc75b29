"""Offline preparation of the low-rank selection head (host, fp64).

EAGLE-4 notes (qingkeai.online/blog/EAGLE), section "A training-free version:
Freq-aware SVD": weight each row of the full head W (n x d) by its smoothed
token frequency, take a truncated SVD, and undo the row weighting:

    F = diag(f),  F^1/2 W = U S V^T,  A = F^-1/2 U_r S_r (n x r),  B = V_r^T (r x d).

The pages place this step offline ("count token frequencies and do one
decomposition"; no training); it never runs per call. For heads with
n >> d the decomposition goes through the d x d Gram matrix:
W^T F W = V S^2 V^T, so V_r are its top-r eigenvectors and
F^-1/2 U_r S_r = F^-1/2 (F^1/2 W V_r) = W V_r. Hence A = W V_r, B = V_r^T,
computed in fp64 in row blocks and rounded to bf16 (through fp32, nearest-even).

The section "A Local Top-k based variant" recommends shuffling vocabulary
rows before tiling; `perm` (position -> vocabulary id) reorders the rows of
A, and is what the kernels take as `token_ids`.

Smoothing: the pages only require f_i > 0; this uses add-one smoothing of raw
counts (the frequency scale cancels in A B).
"""
from __future__ import annotations

from typing import Optional

import numpy as np

__all__ = ["smoothed_frequency", "freq_aware_factors", "bf16_bits", "pruned_rows"]


def smoothed_frequency(counts: np.ndarray) -> np.ndarray:
    return np.asarray(counts, dtype=np.float64) + 1.0


def bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round to bf16 via fp32 (both nearest-even); uint16 bit patterns."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    return ((u + np.uint32(0x7FFF) + ((u >> np.uint32(16)) & np.uint32(1))) >> np.uint32(16)).astype(np.uint16)


def _bits_to_f64(b: np.ndarray) -> np.ndarray:
    return (np.ascontiguousarray(b, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)


def freq_aware_factors(W_bits: np.ndarray, counts: np.ndarray, r: int,
                       perm: Optional[np.ndarray] = None, block: int = 8192) -> dict:
    """Freq-aware SVD factors of a bf16 head.

    Returns dict(A=uint16 n x r in position order, B=uint16 r x d,
    token_ids=int32 n, eigenvalues=float64 d (descending) of W^T F W).
    """
    n, d = W_bits.shape
    if not 1 <= r <= d:
        raise ValueError(f"rank r={r} must be in [1, d={d}]")
    f = smoothed_frequency(counts)
    G = np.zeros((d, d), dtype=np.float64)
    for r0 in range(0, n, block):
        Wb = _bits_to_f64(W_bits[r0:r0 + block])
        G += Wb.T @ (f[r0:r0 + block, None] * Wb)
    evals, evecs = np.linalg.eigh(G)
    order = np.argsort(evals)[::-1]
    V = np.ascontiguousarray(evecs[:, order[:r]])
    token_ids = (np.arange(n, dtype=np.int32) if perm is None
                 else np.ascontiguousarray(perm, dtype=np.int32))
    A = np.empty((n, r), dtype=np.uint16)
    for r0 in range(0, n, block):
        rows = token_ids[r0:r0 + block]
        A[r0:r0 + rows.size] = bf16_bits(_bits_to_f64(W_bits[rows]) @ V)
    B = bf16_bits(V.T)
    return {"A": A, "B": B, "token_ids": token_ids, "eigenvalues": evals[order]}


def pruned_rows(W_bits: np.ndarray, counts: np.ndarray, n_keep: int = 32000):
    """The comparison head of the EAGLE-4 notes' "EAGLE Efficient LM Head"
    section that keeps only the n_keep most frequent tokens (32000 there),
    built offline: returns (W_pruned, kept), kept the vocabulary ids in
    ascending order (ties in frequency go to the smaller id) and W_pruned
    their rows of W copied contiguously (the layout lmhead_pruned_head
    takes; output column j belongs to kept[j])."""
    n = W_bits.shape[0]
    if not 1 <= n_keep <= n:
        raise ValueError(f"n_keep={n_keep} must be in [1, n={n}]")
    f = smoothed_frequency(counts)
    kept = np.sort(np.argsort(-f, kind="stable")[:n_keep]).astype(np.int64)
    return np.ascontiguousarray(W_bits[kept]), kept
