"""GB300-native two-stage draft LM head: Python binding of liblmhead.so.

Argument marshalling only: every step of the head runs in the library's CUDA
kernels; PyTorch supplies device memory and streams. Tensors are CUDA,
contiguous, row-major; bf16 tensors may be torch.bfloat16 or 16-bit integer
views of bf16 bits. Names follow the C ABI (include/lmhead.h) without the
`lmhead_` prefix.

    ids, logits, q = two_stage(LOCAL, W, A, B, h, token_ids, T, k_tile)

Offline preparation of A and B (the Freq-aware SVD) is in
draft_lm_head_gb300.prep.
"""
from __future__ import annotations

import functools
from typing import Optional

import torch

from ._lib import LIB_PATH, LmheadError, check, load, status_string  # noqa: F401

GLOBAL = 0
LOCAL = 1

__all__ = [
    "GLOBAL", "LOCAL", "LmheadError", "candidate_count", "workspace_size", "project_u",
    "lowrank_score_topk", "gather_logits", "candidate_softmax", "two_stage", "dense_head",
    "pruned_head", "cluster_candidate_count", "cluster_workspace_size", "cluster_two_stage",
    "draft_select", "verify_chain", "last_device_error", "debug_set_wait_cycles", "version",
    "Workspace", "shard_workspace_size", "shard_two_stage", "shard_softmax",
]

_BF16_OK = (torch.bfloat16, torch.int16, torch.uint16) if hasattr(torch, "uint16") else (
    torch.bfloat16, torch.int16)


def _stream_ptr(stream: Optional[torch.cuda.Stream]) -> int:
    s = stream if stream is not None else torch.cuda.current_stream()
    return s.cuda_stream


def _bf16(t: torch.Tensor, name: str) -> int:
    if not t.is_cuda or t.dtype not in _BF16_OK or not t.is_contiguous():
        raise TypeError(f"{name}: expected a contiguous CUDA bf16 tensor, got {t.dtype} "
                        f"on {t.device} (contiguous={t.is_contiguous()})")
    return t.data_ptr()


def _typed(t: Optional[torch.Tensor], dtype, name: str) -> int:
    if t is None:
        return 0
    if not t.is_cuda or t.dtype != dtype or not t.is_contiguous():
        raise TypeError(f"{name}: expected a contiguous CUDA {dtype} tensor")
    return t.data_ptr()


def _check_shapes(device, **named) -> None:
    """Host-side size checks before any pointer reaches the library: the C ABI
    takes sizes from the caller, so a tensor of the wrong shape would make a
    kernel read or write outside it. named: name -> (tensor or None, shape)."""
    for name, (t, want) in named.items():
        if t is None:
            continue
        if tuple(t.shape) != tuple(want):
            raise ValueError(f"{name}: expected shape {tuple(want)}, got {tuple(t.shape)}")
        if device is not None and t.device != device:
            raise ValueError(f"{name}: on {t.device}, expected {device}")


def version() -> int:
    return load().lmhead_version()


@functools.lru_cache(maxsize=4096)
def candidate_count(mode: int, n: int, C_or_tile: int, k_tile: int = 0) -> int:
    K = load().lmhead_candidate_count(mode, n, C_or_tile, k_tile)
    if K < 0:
        raise LmheadError(int(K), "candidate_count")
    return int(K)


@functools.lru_cache(maxsize=4096)
def workspace_size(mode: int, n: int, d: int, r: int, M: int, C_or_tile: int,
                   k_tile: int = 0) -> int:
    return int(load().lmhead_workspace_size(mode, n, d, r, M, C_or_tile, k_tile))


class Workspace:
    """A reusable device workspace (grows on demand; 256-byte aligned)."""

    def __init__(self, device=None):
        self.device = device
        self.buf = None

    def get(self, nbytes: int, device) -> torch.Tensor:
        if self.buf is None or self.buf.numel() < nbytes or self.buf.device != device:
            self.buf = torch.empty(max(nbytes, 256), dtype=torch.uint8, device=device)
        return self.buf


def _ws(workspace, nbytes, device):
    if workspace is None:
        return torch.empty(max(nbytes, 256), dtype=torch.uint8, device=device)
    if isinstance(workspace, Workspace):
        return workspace.get(nbytes, device)
    return workspace


def project_u(B: torch.Tensor, h: torch.Tensor, out: Optional[torch.Tensor] = None,
              stream=None) -> torch.Tensor:
    r, d = B.shape
    M = h.shape[0]
    _check_shapes(B.device, h=(h, (M, d)), out=(out, (M, r)))
    u = out if out is not None else torch.empty((M, r), dtype=torch.bfloat16, device=h.device)
    check(load().lmhead_project_u(_bf16(B, "B"), _bf16(h, "h"), d, r, M, _bf16(u, "u"),
                                  _stream_ptr(stream)), "project_u")
    return u


def lowrank_score_topk(mode: int, A: torch.Tensor, B: torch.Tensor, h: torch.Tensor,
                       token_ids: Optional[torch.Tensor], C_or_tile: int, k_tile: int = 0,
                       with_scores: bool = False, workspace=None, stream=None):
    n, r = A.shape
    d = B.shape[1]
    M = h.shape[0]
    _check_shapes(A.device, B=(B, (r, d)), h=(h, (M, d)), token_ids=(token_ids, (n,)))
    K = candidate_count(mode, n, C_or_tile, k_tile)
    ids = torch.empty((M, K), dtype=torch.int32, device=h.device)
    scores = torch.empty((M, K), dtype=torch.float32, device=h.device) if with_scores else None
    nbytes = workspace_size(mode, n, d, r, M, C_or_tile, k_tile)
    ws = _ws(workspace, nbytes, h.device)
    check(load().lmhead_lowrank_score_topk(
        mode, _bf16(A, "A"), _bf16(B, "B"), _bf16(h, "h"), _typed(token_ids, torch.int32, "token_ids"),
        n, d, r, M, C_or_tile, k_tile, ids.data_ptr(), _typed(scores, torch.float32, "scores"),
        ws.data_ptr(), ws.numel(), _stream_ptr(stream)), "lowrank_score_topk")
    return (ids, scores) if with_scores else ids


def gather_logits(W: torch.Tensor, h: torch.Tensor, ids: torch.Tensor,
                  out: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    n, d = W.shape
    M, K = ids.shape
    _check_shapes(W.device, h=(h, (M, d)), ids=(ids, (M, K)), out=(out, (M, K)))
    L = out if out is not None else torch.empty((M, K), dtype=torch.float32, device=h.device)
    check(load().lmhead_gather_logits(_bf16(W, "W"), _bf16(h, "h"), _typed(ids, torch.int32, "ids"),
                                      n, d, M, K, _typed(L, torch.float32, "out"),
                                      _stream_ptr(stream)), "gather_logits")
    return L


def candidate_softmax(logits: torch.Tensor, temperature: float = 1.0,
                      out: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    M, K = logits.shape
    _check_shapes(logits.device, out=(out, (M, K)))
    q = out if out is not None else torch.empty_like(logits)
    check(load().lmhead_candidate_softmax(_typed(logits, torch.float32, "logits"), M, K,
                                          float(temperature), _typed(q, torch.float32, "out"),
                                          _stream_ptr(stream)), "candidate_softmax")
    return q


def two_stage(mode: int, W: torch.Tensor, A: torch.Tensor, B: torch.Tensor, h: torch.Tensor,
              token_ids: Optional[torch.Tensor], C_or_tile: int, k_tile: int = 0,
              temperature: float = 1.0, workspace=None, out=None, stream=None):
    """The whole head: returns (ids, logits, q), each M x K."""
    n, d = W.shape
    r = A.shape[1]
    M = h.shape[0]
    K = candidate_count(mode, n, C_or_tile, k_tile)
    if out is None:
        ids = torch.empty((M, K), dtype=torch.int32, device=h.device)
        L = torch.empty((M, K), dtype=torch.float32, device=h.device)
        q = torch.empty((M, K), dtype=torch.float32, device=h.device)
    else:
        ids, L, q = out
    _check_shapes(W.device, A=(A, (n, r)), B=(B, (r, d)), h=(h, (M, d)),
                  token_ids=(token_ids, (n,)), ids=(ids, (M, K)), logits=(L, (M, K)),
                  q=(q, (M, K)))
    nbytes = workspace_size(mode, n, d, r, M, C_or_tile, k_tile)
    ws = _ws(workspace, nbytes, h.device)
    check(load().lmhead_two_stage(
        mode, _bf16(W, "W"), _bf16(A, "A"), _bf16(B, "B"), _bf16(h, "h"),
        _typed(token_ids, torch.int32, "token_ids"), n, d, r, M, C_or_tile, k_tile,
        float(temperature), _typed(ids, torch.int32, "ids"), _typed(L, torch.float32, "logits"),
        _typed(q, torch.float32, "q"), ws.data_ptr(), ws.numel(), _stream_ptr(stream)),
        "two_stage")
    return ids, L, q


def dense_head(W: torch.Tensor, h: torch.Tensor, temperature: float = 1.0, with_q: bool = True,
               out=None, stream=None):
    n, d = W.shape
    M = h.shape[0]
    if out is None:
        L = torch.empty((M, n), dtype=torch.float32, device=h.device)
        q = torch.empty((M, n), dtype=torch.float32, device=h.device) if with_q else None
    else:
        L, q = out
    _check_shapes(W.device, h=(h, (M, d)), logits=(L, (M, n)), q=(q, (M, n)))
    check(load().lmhead_dense_head(_bf16(W, "W"), _bf16(h, "h"), n, d, M, float(temperature),
                                   _typed(L, torch.float32, "logits"), _typed(q, torch.float32, "q"),
                                   _stream_ptr(stream)), "dense_head")
    return L, q


def pruned_head(W_pruned: torch.Tensor, h: torch.Tensor, temperature: float = 1.0,
                with_q: bool = True, out=None, stream=None):
    n_keep, d = W_pruned.shape
    M = h.shape[0]
    if out is None:
        L = torch.empty((M, n_keep), dtype=torch.float32, device=h.device)
        q = torch.empty((M, n_keep), dtype=torch.float32, device=h.device) if with_q else None
    else:
        L, q = out
    _check_shapes(W_pruned.device, h=(h, (M, d)), logits=(L, (M, n_keep)), q=(q, (M, n_keep)))
    check(load().lmhead_pruned_head(_bf16(W_pruned, "W_pruned"), _bf16(h, "h"), n_keep, d, M,
                                    float(temperature), _typed(L, torch.float32, "logits"),
                                    _typed(q, torch.float32, "q"), _stream_ptr(stream)),
          "pruned_head")
    return L, q


def shard_workspace_size(n_shard: int, d: int, r: int, M: int, T: int, k_tile: int) -> int:
    return int(load().lmhead_shard_workspace_size(n_shard, d, r, M, T, k_tile))


def shard_two_stage(W_shard: torch.Tensor, A_shard: torch.Tensor, B: torch.Tensor,
                    h: torch.Tensor, token_ids_shard: torch.Tensor, row_of_id: torch.Tensor,
                    T: int, k_tile: int, temperature: float = 1.0, workspace=None, out=None,
                    stream=None):
    """One vocabulary shard of the local head (see lmhead_shard_two_stage):
    returns (ids, logits, stats), stats M x 2 (max, sum of exponentials)."""
    n_shard, r = A_shard.shape
    d = B.shape[1]
    M = h.shape[0]
    n_vocab = row_of_id.shape[0]
    K = candidate_count(LOCAL, n_shard, T, k_tile)
    dev = h.device
    if out is None:
        ids = torch.empty((M, K), dtype=torch.int32, device=dev)
        L = torch.empty((M, K), dtype=torch.float32, device=dev)
        stats = torch.empty((M, 2), dtype=torch.float32, device=dev)
    else:
        ids, L, stats = out
    _check_shapes(A_shard.device, W_shard=(W_shard, (n_shard, d)), B=(B, (r, d)), h=(h, (M, d)),
                  token_ids_shard=(token_ids_shard, (n_shard,)), ids=(ids, (M, K)),
                  logits=(L, (M, K)), stats=(stats, (M, 2)))
    nbytes = shard_workspace_size(n_shard, d, r, M, T, k_tile)
    ws = _ws(workspace, nbytes, dev)
    check(load().lmhead_shard_two_stage(
        _bf16(W_shard, "W_shard"), _bf16(A_shard, "A_shard"), _bf16(B, "B"), _bf16(h, "h"),
        _typed(token_ids_shard, torch.int32, "token_ids_shard"),
        _typed(row_of_id, torch.int32, "row_of_id"), n_vocab, n_shard, d, r, M, T, k_tile,
        float(temperature), _typed(ids, torch.int32, "ids"), _typed(L, torch.float32, "logits"),
        _typed(stats, torch.float32, "stats"), ws.data_ptr(), ws.numel(), _stream_ptr(stream)),
        "shard_two_stage")
    return ids, L, stats


def shard_softmax(all_stats: torch.Tensor, logits: torch.Tensor, temperature: float = 1.0,
                  out: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """q of one shard's candidates from every shard's stats (G x M x 2)."""
    M, K = logits.shape
    G = all_stats.shape[0]
    _check_shapes(logits.device, all_stats=(all_stats, (G, M, 2)), out=(out, (M, K)))
    q = out if out is not None else torch.empty_like(logits)
    check(load().lmhead_shard_softmax(
        _typed(all_stats, torch.float32, "all_stats"), G, _typed(logits, torch.float32, "logits"),
        M, K, float(temperature), _typed(q, torch.float32, "out"), _stream_ptr(stream)),
        "shard_softmax")
    return q


def last_device_error(stream=None) -> int:
    """Synchronise the stream and return (and clear) the device error status."""
    return int(load().lmhead_last_device_error(_stream_ptr(stream)))


def debug_set_wait_cycles(cycles: int) -> int:
    """Test hook: the role-wait budget of the tensor-core kernels in SM cycles
    (0 = test each wait once, < 0 = the default). Returns the previous one."""
    return int(load().lmhead_debug_set_wait_cycles(int(cycles)))


@functools.lru_cache(maxsize=4096)
def cluster_candidate_count(n: int, group: int, G: int) -> int:
    K = load().lmhead_cluster_candidate_count(n, group, G)
    if K < 0:
        raise LmheadError(int(K), "cluster_candidate_count")
    return int(K)


@functools.lru_cache(maxsize=4096)
def cluster_workspace_size(n: int, d: int, r: int, M: int, group: int, G: int) -> int:
    return int(load().lmhead_cluster_workspace_size(n, d, r, M, group, G))


def cluster_two_stage(W: torch.Tensor, A: torch.Tensor, B: torch.Tensor, h: torch.Tensor,
                      group: int, G: int, temperature: float = 1.0, with_group_scores=False,
                      workspace=None, out=None, stream=None):
    """The cluster-level head: returns (groups M x G, ids, logits, q each
    M x G*group), plus the groups' scores when with_group_scores."""
    n, d = W.shape
    r = A.shape[1]
    M = h.shape[0]
    K = cluster_candidate_count(n, group, G)
    dev = h.device
    if out is None:
        groups = torch.empty((M, G), dtype=torch.int32, device=dev)
        ids = torch.empty((M, K), dtype=torch.int32, device=dev)
        L = torch.empty((M, K), dtype=torch.float32, device=dev)
        q = torch.empty((M, K), dtype=torch.float32, device=dev)
    else:
        groups, ids, L, q = out
    _check_shapes(W.device, A=(A, (n, r)), B=(B, (r, d)), h=(h, (M, d)), groups=(groups, (M, G)),
                  ids=(ids, (M, K)), logits=(L, (M, K)), q=(q, (M, K)))
    gs = torch.empty((M, G), dtype=torch.float32, device=dev) if with_group_scores else None
    nbytes = cluster_workspace_size(n, d, r, M, group, G)
    ws = _ws(workspace, nbytes, dev)
    check(load().lmhead_cluster_two_stage(
        _bf16(W, "W"), _bf16(A, "A"), _bf16(B, "B"), _bf16(h, "h"), n, d, r, M, group, G,
        float(temperature), _typed(groups, torch.int32, "groups"),
        _typed(gs, torch.float32, "group_scores"), _typed(ids, torch.int32, "ids"),
        _typed(L, torch.float32, "logits"), _typed(q, torch.float32, "q"), ws.data_ptr(),
        ws.numel(), _stream_ptr(stream)), "cluster_two_stage")
    return (groups, ids, L, q, gs) if with_group_scores else (groups, ids, L, q)


def draft_select(q: torch.Tensor, ids: torch.Tensor, k_sel: int,
                 parent_value: Optional[torch.Tensor] = None,
                 uniforms: Optional[torch.Tensor] = None, stream=None):
    """EAGLE-2 expansion of each row of q: its k_sel most likely candidates with
    their path values, and (given uniforms) one Gumbel-max draw. Returns
    (top_ids, top_q, top_value, sample_id, sample_q); the last two are None
    without uniforms."""
    M, K = q.shape
    dev = q.device
    _check_shapes(dev, ids=(ids, (M, K)), parent_value=(parent_value, (M,)),
                  uniforms=(uniforms, (M, K)))
    top_ids = torch.empty((M, k_sel), dtype=torch.int32, device=dev)
    top_q = torch.empty((M, k_sel), dtype=torch.float32, device=dev)
    top_value = torch.empty((M, k_sel), dtype=torch.float32, device=dev)
    sid = torch.empty(M, dtype=torch.int32, device=dev) if uniforms is not None else None
    sq = torch.empty(M, dtype=torch.float32, device=dev) if uniforms is not None else None
    check(load().lmhead_draft_select(
        _typed(q, torch.float32, "q"), _typed(ids, torch.int32, "ids"), M, K, k_sel,
        _typed(parent_value, torch.float32, "parent_value"),
        _typed(uniforms, torch.float32, "uniforms"), top_ids.data_ptr(), top_q.data_ptr(),
        top_value.data_ptr(), _typed(sid, torch.int32, "sample_id"),
        _typed(sq, torch.float32, "sample_q"), _stream_ptr(stream)), "draft_select")
    return top_ids, top_q, top_value, sid, sq


def verify_chain(p: torch.Tensor, x: torch.Tensor, cand_ids: torch.Tensor, cand_q: torch.Tensor,
                 r: torch.Tensor, u: torch.Tensor, stream=None):
    """The exactness rule over B chains: p B x (Kd+1) x n, x B x Kd, cand_ids /
    cand_q B x Kd x K, r B x Kd, u B x (Kd+1). Returns (tokens B x (Kd+1),
    accepted counts B)."""
    B, Kd1, n = p.shape
    Kd = Kd1 - 1
    K = cand_ids.shape[-1]
    dev = p.device
    _check_shapes(dev, x=(x, (B, Kd)), cand_ids=(cand_ids, (B, Kd, K)),
                  cand_q=(cand_q, (B, Kd, K)), r=(r, (B, Kd)), u=(u, (B, Kd + 1)))
    tokens = torch.empty((B, Kd + 1), dtype=torch.int32, device=dev)
    count = torch.empty(B, dtype=torch.int32, device=dev)
    check(load().lmhead_verify_chain(
        _typed(p, torch.float32, "p"), n, B, Kd, _typed(x, torch.int32, "x"),
        _typed(cand_ids, torch.int32, "cand_ids"), _typed(cand_q, torch.float32, "cand_q"), K,
        _typed(r, torch.float32, "r"), _typed(u, torch.float32, "u"), tokens.data_ptr(),
        count.data_ptr(), _stream_ptr(stream)), "verify_chain")
    return tokens, count
