"""Helpers shared by the GPU tests: building the library, moving seeded
inputs to the device, and running the oracle on the same bits."""
from __future__ import annotations

import functools

import numpy as np

import oracle as O
import synth


@functools.lru_cache(maxsize=None)
def lib():
    import torch
    if not torch.cuda.is_available():
        raise RuntimeError("GPU tests need CUDA")
    from draft_lm_head_gb300 import build
    build.build()
    import draft_lm_head_gb300 as L
    L.load() if hasattr(L, "load") else None
    return L


def dev_bf16(bits: np.ndarray):
    import torch
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).cuda().view(torch.bfloat16)


def dev_i32(x: np.ndarray):
    import torch
    return torch.from_numpy(np.ascontiguousarray(x, dtype=np.int32)).cuda()


def host(t) -> np.ndarray:
    return t.detach().cpu().numpy()


def make_case(n, d, r, M, seed, shuffle=True, zipf_s=1.1, plain_h=False):
    """A seeded synthetic head and its Freq-aware SVD factors (host, bits)."""
    from draft_lm_head_gb300 import prep
    W = synth.make_head(n, d, seed)
    counts = synth.zipf_counts(n, zipf_s, seed)
    perm = synth.shuffle_perm(n, seed) if shuffle else None
    fac = prep.freq_aware_factors(W, counts, r, perm)
    if plain_h:
        h = synth.make_plain_hidden(d, M, seed)
    else:
        h, _ = synth.make_hidden(W, M, seed)
    return {"W": W, "A": fac["A"], "B": fac["B"], "tok": fac["token_ids"], "h": h,
            "counts": counts, "n": n, "d": d, "r": r, "M": M}


def workload_head(wl):
    """The seeded head of a workload with its Freq-aware SVD factors in
    vocabulary order (cached under _cache/); rows are shuffled per use."""
    from draft_lm_head_gb300 import prep

    def builder():
        W = synth.make_head(wl.n, wl.d, wl.head_seed_index)
        counts = synth.zipf_counts(wl.n, wl.zipf_s, wl.head_seed_index)
        fac = prep.freq_aware_factors(W, counts, wl.r)
        return {"W": W, "counts": counts, "A": fac["A"], "B": fac["B"]}

    key = f"head:{wl.head_seed_index}:{wl.n}:{wl.d}:{wl.r}:{wl.zipf_s}"
    return synth.head_cache(key, builder)


def workload_case(wl, M, shuffle=None, tree=None, stream_offset=0):
    head = workload_head(wl)
    shuffle = wl.shuffle if shuffle is None else shuffle
    tok = synth.shuffle_perm(wl.n, wl.index) if shuffle else np.arange(wl.n, dtype=np.int32)
    tree = wl.tree if tree is None else tree
    if tree:
        h, t = synth.make_tree_hidden(head["W"], M // len(synth.TREE_PARENT), wl.index)
    else:
        h, t = synth.make_hidden(head["W"], M, wl.index, stream_offset)
    return {"W": head["W"], "A": np.ascontiguousarray(head["A"][tok]), "B": head["B"], "tok": tok,
            "h": h, "t": t, "counts": head["counts"], "n": wl.n, "d": wl.d, "r": wl.r, "M": M}


def oracle_scores(case, with_slack=False, M_call=None):
    """Oracle u (bf16 grid, fp64) and position-ordered scores M x n (and the
    u-rounding slack of tests/parity.py when asked). M_call: hidden vectors
    of the library call that produced the GPU side (it picks the projection
    kernel, hence the slack); default the rows of case["h"]."""
    import parity
    A64 = O.bf16_bits_to_f64(case["A"])
    B64 = O.bf16_bits_to_f64(case["B"])
    h64 = O.bf16_bits_to_f64(case["h"])
    u = O.project_u(B64, h64)
    S = O.lowrank_scores(A64, u)
    if with_slack:
        return u, S, h64, parity.u_slack(A64, B64, h64, M_call)
    return u, S, h64
