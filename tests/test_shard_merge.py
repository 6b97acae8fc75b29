"""Host side of the vocabulary-sharded head, no GPU: the tile-aligned shard
ranges and per-shard inputs, the all-gather of the shards' (max, sum) stats
over two gloo ranks, and the fact the sharding rests on: with tile-aligned
shards the shards' local Top-k candidates are the unsharded head's, and the
softmax over their union is rebuilt exactly from per-shard (max, sum) pairs."""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import oracle as O
import synth
from draft_lm_head_gb300 import shard as S


def test_shard_ranges_are_tile_aligned_and_cover_the_head():
    for n, T, G in ((128256, 256, 2), (128256, 256, 8), (1000, 128, 3), (201088, 256, 4)):
        rs = S.shard_ranges(n, T, G)
        assert rs[0][0] == 0 and rs[-1][1] == n and len(rs) == G
        for (a0, a1), (b0, b1) in zip(rs, rs[1:]):
            assert a1 == b0 and a0 % T == 0
        assert all(p0 % T == 0 for p0, _ in rs)


def test_shard_inputs_map_ids_to_local_rows():
    W = synth.make_head(300, 8, 0)
    A = np.arange(300 * 4, dtype=np.uint16).reshape(300, 4)
    tok = synth.shuffle_perm(300, 0)
    Ws, As, toks, roi = S.shard_inputs(W, A, tok, 128, 256)
    assert np.array_equal(As, A[128:256]) and np.array_equal(toks, tok[128:256])
    assert np.array_equal(Ws, W[tok[128:256]])
    held = roi >= 0
    assert held.sum() == 128 and np.array_equal(np.sort(np.nonzero(held)[0]), np.sort(toks))
    assert np.array_equal(Ws[roi[toks]], W[toks])


def test_tile_aligned_shards_keep_the_candidates():
    rng = np.random.default_rng(61)
    n, T, k = 1000, 64, 3
    scores = rng.standard_normal(n)
    tok = rng.permutation(n).astype(np.int32)
    whole, _ = O.local_topk(scores, tok, T, k)
    parts = [O.local_topk(scores[p0:p1], tok[p0:p1], T, k)[0] for p0, p1 in S.shard_ranges(n, T, 3)]
    assert np.array_equal(np.concatenate(parts), whole)


def _stats(L, temp):
    z = L / temp
    mx = z.max()
    return np.array([mx, np.exp(z - mx).sum()])


def _merge(all_stats, L, temp):
    # the combination lmhead_shard_softmax computes, restated
    gm = all_stats[:, 0].max()
    Z = (all_stats[:, 1] * np.exp(all_stats[:, 0] - gm)).sum()
    return np.exp(L / temp - gm) / Z


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, out_dir):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        rng = np.random.default_rng(62)
        Lall = rng.standard_normal((3, 50)) * 30.0     # 3 rows, 50 candidates in all
        cut = [0, 20, 50]
        mine = Lall[:, cut[rank]:cut[rank + 1]]
        st = torch.tensor(np.stack([_stats(row, 2.0) for row in mine]), dtype=torch.float64)
        gathered = S.gather_stats(st).numpy()           # G x M x 2, rank order
        q = np.stack([_merge(gathered[:, m], mine[m], 2.0) for m in range(3)])
        np.save(os.path.join(out_dir, f"r{rank}.npy"), np.concatenate([gathered.ravel(), q.ravel()]))
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_two_ranks_exchange_stats_and_rebuild_the_softmax(tmp_path):
    mp.start_processes(_rank, args=(2, _free_port(), str(tmp_path)), nprocs=2,
                       start_method="spawn", join=True)
    rng = np.random.default_rng(62)
    Lall = rng.standard_normal((3, 50)) * 30.0
    r0, r1 = np.load(tmp_path / "r0.npy"), np.load(tmp_path / "r1.npy")
    g0, g1 = r0[:12].reshape(2, 3, 2), r1[:12].reshape(2, 3, 2)
    assert np.array_equal(g0, g1)                       # both ranks hold the same table
    for m in range(3):                                  # in rank order
        np.testing.assert_allclose(g0[0, m], _stats(Lall[m, :20], 2.0))
        np.testing.assert_allclose(g0[1, m], _stats(Lall[m, 20:], 2.0))
    q = np.concatenate([r0[12:].reshape(3, 20), r1[12:].reshape(3, 30)], axis=1)
    for m in range(3):
        np.testing.assert_allclose(q[m], O.candidate_softmax(Lall[m], 2.0), rtol=1e-12, atol=1e-15)


def test_gather_stats_without_a_process_group():
    st = torch.zeros((4, 2))
    assert tuple(S.gather_stats(st).shape) == (1, 4, 2)
