"""Seeded synthetic inputs for the two-stage draft LM head.

This module is shared by the CUDA path's tests/bench and by the fp64 oracle's
tests. It holds only input generation: random heads W, token counts, hidden
states h, the vocabulary-row shuffle and the draft-tree layout. None of the
head's own arithmetic (frequency smoothing, the Freq-aware SVD, scoring,
Top-k, logits, softmax) lives here.

The recipes stand in for the heads of the models the pages talk about
(Llama-3-8B, GPT-OSS-120B, a wider model) and for their missing benchmark
text, since neither weights nor data are available:

* W = X.Y/sqrt(64) + 0.05.N(0,1) with X (n x 64), Y (64 x d) i.i.d. N(0,1):
  a rank-64 structure plus noise. X.Y/8 is formed in fp64, cast to fp32,
  the fp32 noise added in fp32, and the sum rounded to bf16 (nearest-even).
  The bf16 bits are the head from then on.
* Token counts: rank k (1-based) of a Zipf(s) law gets
  floor(1e9 * k^-s / H_{n,s}) counts, assigned to token pi_f[k-1] for a
  seeded permutation pi_f. (Smoothing is the method's step, not done here.)
* h[m] = 0.5*sqrt(d)*W[t_m]/||W[t_m]|| + N(0,1), computed in fp64 from the
  bf16 W, rounded to bf16; t_m uniform over the vocabulary.
* Draft tree (8 sequences x 10 nodes): parent = [-1,0,0,0,1,1,1,2,2,3];
  a node's h is 0.5*(parent's unrounded h) + 0.5*(a fresh recipe draw).
* Vocabulary shuffle: a seeded permutation pi; position i of the shuffled
  low-rank factor holds vocabulary row pi[i].

Seeds: stream s of workload c uses numpy PCG64 seeded with 1000*c + s
(0: X, 1: Y, 2: W noise, 3: pi_f, 4: pi, 5: t, 6: h noise).
"""
from __future__ import annotations

import dataclasses
import hashlib
import os
from typing import Optional

import numpy as np

__all__ = [
    "Workload", "WORKLOADS", "workload", "rng", "bf16_bits_from_f32",
    "bf16_bits_to_f64", "bf16_bits_to_f32", "make_head", "zipf_counts",
    "shuffle_perm", "make_hidden", "make_tree_hidden", "TREE_PARENT",
    "make_plain_hidden", "head_cache",
]

TREE_PARENT = (-1, 0, 0, 0, 1, 1, 1, 2, 2, 3)


@dataclasses.dataclass(frozen=True)
class Workload:
    """One synthetic workload: head shape, batch sizes and selection knobs."""
    index: int          # workload number (seed base = 1000 * head_seed_index)
    name: str
    n: int              # vocabulary
    d: int              # hidden size
    r: int              # rank of the low-rank factor
    zipf_s: float
    Ms: tuple           # hidden vectors per call
    C: int              # global Top-k budget
    T: int              # local tile rows (0 = local mode not used)
    k_tile: int
    head_seed_index: int  # workloads that share a head share its seeds
    shuffle: bool = True
    tree: bool = False

    @property
    def tiles(self) -> int:
        return -(-self.n // self.T) if self.T else 0


WORKLOADS = (
    Workload(0, "tiny n4096 d256 r32", 4096, 256, 32, 1.1, (1,), 128, 128, 4, 0),
    Workload(1, "llama3-8b head n128256 d4096 r256 global", 128256, 4096, 256,
             1.1, (1, 4, 8), 1024, 256, 2, 1, shuffle=False),
    Workload(2, "llama3-8b head n128256 d4096 r256 local", 128256, 4096, 256,
             1.1, (1, 8, 16, 32, 64), 1002, 256, 2, 1),
    Workload(3, "gpt-oss-120b head n201088 d2880 r256 tree", 201088, 2880, 256,
             1.1, (80,), 1024, 256, 2, 3, tree=True),
    Workload(4, "wide head n151936 d5120 r512", 151936, 5120, 512, 1.0,
             (1, 8, 32, 128, 512), 1024, 256, 4, 4),
)


def workload(i: int) -> Workload:
    return WORKLOADS[i]


def rng(seed_index: int, stream: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(1000 * seed_index + stream))


# ---------------------------------------------------------------- bf16 bits
def bf16_bits_from_f32(x: np.ndarray) -> np.ndarray:
    """Round fp32 values to bf16 (nearest, ties to even); return uint16 bits."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    lsb = (u >> np.uint32(16)) & np.uint32(1)
    return ((u + np.uint32(0x7FFF) + lsb) >> np.uint32(16)).astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (np.ascontiguousarray(b, dtype=np.uint16).astype(np.uint32)
            << np.uint32(16)).view(np.float32)


def bf16_bits_to_f64(b: np.ndarray) -> np.ndarray:
    return bf16_bits_to_f32(b).astype(np.float64)


# ---------------------------------------------------------------- generators
def make_head(n: int, d: int, seed_index: int, block: int = 8192) -> np.ndarray:
    """Synthetic LM head W (n x d) as bf16 bits (uint16), row-major."""
    X = rng(seed_index, 0).standard_normal((n, 64))
    Y = rng(seed_index, 1).standard_normal((64, d))
    noise_rng = rng(seed_index, 2)
    out = np.empty((n, d), dtype=np.uint16)
    for r0 in range(0, n, block):
        r1 = min(n, r0 + block)
        base = (X[r0:r1] @ Y / 8.0).astype(np.float32)
        base += np.float32(0.05) * noise_rng.standard_normal((r1 - r0, d), dtype=np.float32)
        out[r0:r1] = bf16_bits_from_f32(base)
    return out


def zipf_counts(n: int, s: float, seed_index: int) -> np.ndarray:
    """Raw (unsmoothed) token counts, int64, indexed by vocabulary id."""
    ranks = np.arange(1, n + 1, dtype=np.float64)
    w = ranks ** (-s)
    cnt = np.floor(1e9 * w / w.sum()).astype(np.int64)
    pi_f = rng(seed_index, 3).permutation(n)
    counts = np.empty(n, dtype=np.int64)
    counts[pi_f] = cnt
    return counts


def shuffle_perm(n: int, seed_index: int) -> np.ndarray:
    """Position -> vocabulary id for the shuffled low-rank rows (int32)."""
    return rng(seed_index, 4).permutation(n).astype(np.int32)


def _recipe_f64(W_bits: np.ndarray, t: np.ndarray, noise: np.ndarray) -> np.ndarray:
    d = W_bits.shape[1]
    rows = bf16_bits_to_f64(W_bits[t])
    norms = np.sqrt((rows * rows).sum(axis=1, keepdims=True))
    return 0.5 * np.sqrt(d) * rows / norms + noise


def make_hidden(W_bits: np.ndarray, M: int, seed_index: int,
                stream_offset: int = 0) -> tuple:
    """h (M x d) bf16 bits and the target ids t (M,) of the recipe."""
    n, d = W_bits.shape
    t = rng(seed_index, 5 + 10 * stream_offset).integers(0, n, size=M)
    noise = rng(seed_index, 6 + 10 * stream_offset).standard_normal((M, d))
    h = _recipe_f64(W_bits, t, noise)
    return bf16_bits_from_f32(h.astype(np.float32)), t


def make_plain_hidden(d: int, M: int, seed_index: int, stream_offset: int = 0) -> np.ndarray:
    """h ~ N(0,1) without the W[t] spike (keeps softmax non-degenerate)."""
    z = rng(seed_index, 7 + 10 * stream_offset).standard_normal((M, d))
    return bf16_bits_from_f32(z.astype(np.float32))


def make_tree_hidden(W_bits: np.ndarray, n_seq: int, seed_index: int) -> tuple:
    """Draft-tree hidden states, rows ordered (sequence, node)."""
    n, d = W_bits.shape
    nodes = len(TREE_PARENT)
    M = n_seq * nodes
    t = rng(seed_index, 5).integers(0, n, size=M)
    noise = rng(seed_index, 6).standard_normal((M, d))
    fresh = _recipe_f64(W_bits, t, noise)
    h = np.empty((M, d), dtype=np.float64)
    for s in range(n_seq):
        for k, p in enumerate(TREE_PARENT):
            i = s * nodes + k
            h[i] = fresh[i] if p < 0 else 0.5 * h[s * nodes + p] + 0.5 * fresh[i]
    return bf16_bits_from_f32(h.astype(np.float32)), t


# ---------------------------------------------------------------- disk cache
def head_cache(key: str, builder, root: Optional[str] = None):
    """Memoise a dict of arrays in an .npz under <repo>/_cache (git-ignored)."""
    root = root or os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "_cache")
    os.makedirs(root, exist_ok=True)
    path = os.path.join(root, hashlib.sha1(key.encode()).hexdigest()[:16] + ".npz")
    if os.path.exists(path):
        with np.load(path) as z:
            return {k: z[k] for k in z.files}
    arrays = builder()
    tmp = path + f".{os.getpid()}.tmp.npz"
    np.savez(tmp, **arrays)
    os.replace(tmp, path)
    return arrays
