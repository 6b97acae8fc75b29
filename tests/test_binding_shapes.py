"""The Python binding checks every tensor's shape against the sizes it passes
to the C ABI, before any pointer is taken (the library trusts the sizes it is
given). CPU tensors suffice: the shape check comes first."""
import pytest
import torch

import draft_lm_head_gb300 as L


def bf(*shape):
    return torch.zeros(shape, dtype=torch.bfloat16)


def f32(*shape):
    return torch.zeros(shape, dtype=torch.float32)


def i32(*shape):
    return torch.zeros(shape, dtype=torch.int32)


def test_project_u_shapes():
    with pytest.raises(ValueError, match="h: expected shape"):
        L.project_u(bf(32, 256), bf(2, 128))
    with pytest.raises(ValueError, match="out: expected shape"):
        L.project_u(bf(32, 256), bf(2, 256), out=bf(2, 16))


def test_two_stage_shapes():
    W, A, B, h = bf(1000, 64), bf(1000, 16), bf(16, 64), bf(3, 64)
    with pytest.raises(ValueError, match="A: expected shape"):
        L.two_stage(L.LOCAL, W, bf(999, 16), B, h, None, 128, 2)
    with pytest.raises(ValueError, match="B: expected shape"):
        L.two_stage(L.LOCAL, W, A, bf(16, 32), h, None, 128, 2)
    with pytest.raises(ValueError, match="token_ids: expected shape"):
        L.two_stage(L.LOCAL, W, A, B, h, i32(500), 128, 2)
    K = L.candidate_count(L.LOCAL, 1000, 128, 2)
    with pytest.raises(ValueError, match="q: expected shape"):
        L.two_stage(L.LOCAL, W, A, B, h, None, 128, 2, out=(i32(3, K), f32(3, K), f32(3, K - 1)))
    with pytest.raises(ValueError, match="h: expected shape"):
        L.lowrank_score_topk(L.LOCAL, A, B, bf(3, 32), None, 128, 2)


def test_gather_softmax_and_dense_shapes():
    with pytest.raises(ValueError, match="h: expected shape"):
        L.gather_logits(bf(100, 64), bf(2, 64), i32(3, 10))
    with pytest.raises(ValueError, match="out: expected shape"):
        L.gather_logits(bf(100, 64), bf(3, 64), i32(3, 10), out=f32(3, 11))
    with pytest.raises(ValueError, match="out: expected shape"):
        L.candidate_softmax(f32(3, 10), out=f32(10, 3))
    with pytest.raises(ValueError, match="logits: expected shape"):
        L.dense_head(bf(100, 64), bf(3, 64), out=(f32(3, 99), None))
    with pytest.raises(ValueError, match="h: expected shape"):
        L.pruned_head(bf(100, 64), bf(3, 32))


def test_cluster_shapes():
    W, A, B, h = bf(1024, 64), bf(1024, 16), bf(16, 64), bf(2, 64)
    with pytest.raises(ValueError, match="A: expected shape"):
        L.cluster_two_stage(W, bf(1000, 16), B, h, 128, 2)
    K = L.cluster_candidate_count(1024, 128, 2)
    with pytest.raises(ValueError, match="groups: expected shape"):
        L.cluster_two_stage(W, A, B, h, 128, 2, out=(i32(2, 3), i32(2, K), f32(2, K), f32(2, K)))


def test_after_q_shapes():
    q = f32(4, 50)
    with pytest.raises(ValueError, match="ids: expected shape"):
        L.draft_select(q, i32(4, 49), 3)
    with pytest.raises(ValueError, match="uniforms: expected shape"):
        L.draft_select(q, i32(4, 50), 3, uniforms=f32(4, 5))
    with pytest.raises(ValueError, match="parent_value: expected shape"):
        L.draft_select(q, i32(4, 50), 3, parent_value=f32(3))
    p = f32(2, 4, 100)  # B = 2 chains, Kd = 3 drafts
    good = dict(x=i32(2, 3), cand_ids=i32(2, 3, 8), cand_q=f32(2, 3, 8), r=f32(2, 3), u=f32(2, 4))
    for name, bad in (("x", i32(2, 2)), ("cand_q", f32(2, 3, 7)), ("r", f32(3, 3)),
                      ("u", f32(2, 3))):
        args = dict(good, **{name: bad})
        with pytest.raises(ValueError, match=f"{name}: expected shape"):
            L.verify_chain(p, **args)
