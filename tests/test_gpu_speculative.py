"""CUDA steps after q vs the oracle (oracle/speculative_oracle.py): EAGLE-2
draft selection with path values and a Gumbel-max draw, and chain
verification (the exactness rule with the pointwise residual)."""
import numpy as np
import pytest

import oracle as O

from gpu_util import host, lib

pytestmark = pytest.mark.gpu

GUMBEL_TOL = 1e-5   # fp32 log(q) - log(-log u) against fp64: a few ulps of values ~ 10
CDF_TOL = 1e-4      # fp32 sums over ~125-element slices then 1024 partials, relative to W


@pytest.fixture(scope="module")
def L():
    return lib()


def _softmax_rows(x):
    x = x - x.max(axis=-1, keepdims=True)
    e = np.exp(x)
    return (e / e.sum(axis=-1, keepdims=True)).astype(np.float32)


def _t(a):
    import torch
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


@pytest.mark.parametrize("K", [1, 5, 300, 1002, 4096])
@pytest.mark.parametrize("k_sel", [1, 4, 8, 16])
def test_draft_select(L, K, k_sel):
    if k_sel > K:
        pytest.skip("k_sel > K")
    rng = np.random.default_rng(31 * K + k_sel)
    M = 7
    q = _softmax_rows(rng.standard_normal((M, K)) * 3)
    q[1] = np.float32(1.0 / K)                                   # every value tied
    q[2] = np.round(q[2] * 64) / 64                              # coarse values, many ties
    ids = np.stack([rng.permutation(200000)[:K] for _ in range(M)]).astype(np.int32)
    parent = rng.random(M).astype(np.float32)
    U = np.clip(rng.random((M, K)), 1e-7, 1 - 1e-7).astype(np.float32)
    ti, tq, tv, si, sq = L.draft_select(_t(q), _t(ids), k_sel, _t(parent), _t(U))
    ti, tq, tv, si, sq = map(host, (ti, tq, tv, si, sq))
    excused = 0
    for m in range(M):
        oi, oq, ov = O.draft_topk(q[m], ids[m], k_sel, parent[m])
        assert np.array_equal(ti[m], oi) and np.array_equal(tq[m], oq) and np.array_equal(tv[m], ov)
        gid, gj, s = O.gumbel_sample(q[m], ids[m], U[m].astype(np.float64))
        if si[m] != gid:
            j = int(np.nonzero(ids[m] == si[m])[0][0])
            assert s[gj] - s[j] <= GUMBEL_TOL * (1 + abs(s[gj])), (m, si[m], gid)
            excused += 1
        j = int(np.nonzero(ids[m] == si[m])[0][0])
        assert sq[m] == q[m][j]
    assert excused <= 1


def test_draft_select_without_draw(L):
    rng = np.random.default_rng(9)
    q = _softmax_rows(rng.standard_normal((3, 50)))
    ids = np.stack([rng.permutation(1000)[:50] for _ in range(3)]).astype(np.int32)
    ti, tq, tv, si, sq = L.draft_select(_t(q), _t(ids), 4)
    assert si is None and sq is None
    for m in range(3):
        oi, oq, ov = O.draft_topk(q[m], ids[m], 4)
        assert np.array_equal(host(ti)[m], oi) and np.array_equal(host(tv)[m], ov)


def _chain_case(rng, B, Kd, K, n, equal_rows):
    p = np.empty((B, Kd + 1, n), dtype=np.float32)
    cid = np.empty((B, Kd, K), dtype=np.int32)
    cq = np.empty((B, Kd, K), dtype=np.float32)
    x = np.empty((B, Kd), dtype=np.int32)
    for b in range(B):
        for t in range(Kd + 1):
            p[b, t] = _softmax_rows(rng.standard_normal(n) * 2.5)
        for t in range(Kd):
            cid[b, t] = rng.permutation(n)[:K]
            cq[b, t] = _softmax_rows(rng.standard_normal(K) * 2)
            if b in equal_rows:   # target = draft: every draft is accepted
                p[b, t] = 0.0
                p[b, t, cid[b, t]] = cq[b, t]
            x[b, t] = O.gumbel_sample(cq[b, t], cid[b, t], rng.random(K))[0]
    r = rng.random((B, Kd)).astype(np.float32) * np.float32(0.999)
    u = rng.random((B, Kd + 1)).astype(np.float32)
    return p, x, cid, cq, r, u


def _check_chain(p, x, cid, cq, r, u, tokens, count):
    excused = 0
    for b in range(p.shape[0]):
        n_acc, out = O.verify_chain(p[b], x[b], cid[b], cq[b], r[b], u[b])
        assert count[b] == n_acc, b
        assert list(tokens[b, :n_acc]) == out[:n_acc]
        assert np.all(tokens[b, n_acc + 1:] == -1)
        vg, vo = int(tokens[b, n_acc]), out[n_acc]
        if vg != vo:
            t = n_acc
            w = p[b, t].astype(np.float64) if t == len(x[b]) else O.residual(p[b, t], cid[b, t], cq[b, t])
            c = np.cumsum(w)
            target = float(u[b, t]) * c[-1]
            lo = c[vg - 1] if vg > 0 else 0.0
            assert w[vg] > 0 and lo - CDF_TOL * c[-1] <= target <= c[vg] + CDF_TOL * c[-1], (b, vg, vo)
            excused += 1
    return excused


@pytest.mark.parametrize("n", [1000, 128256])
def test_verify_chain(L, n):
    rng = np.random.default_rng(n)
    B, Kd, K = 8, 3, 64
    p, x, cid, cq, r, u = _chain_case(rng, B, Kd, K, n, equal_rows={0, 3})
    tokens, count = L.verify_chain(_t(p), _t(x), _t(cid), _t(cq), _t(r), _t(u))
    tokens, count = host(tokens), host(count)
    assert count[0] == Kd and count[3] == Kd
    assert _check_chain(p, x, cid, cq, r, u, tokens, count) <= 1
    assert L.last_device_error() == 0


def test_verify_chain_bonus_only_and_bad_draft(L):
    rng = np.random.default_rng(5)
    n = 777
    p = _softmax_rows(rng.standard_normal((3, 1, n)))
    u = rng.random((3, 1)).astype(np.float32)
    import torch
    empty_i = torch.empty((3, 0, 1), dtype=torch.int32, device="cuda")
    empty_f = torch.empty((3, 0, 1), dtype=torch.float32, device="cuda")
    tokens, count = L.verify_chain(_t(p), torch.empty((3, 0), dtype=torch.int32, device="cuda"),
                                   empty_i, empty_f, torch.empty((3, 0), dtype=torch.float32,
                                                                 device="cuda"), _t(u))
    assert np.all(host(count) == 0)
    tk = host(tokens)
    for b in range(3):
        vg = int(tk[b, 0])
        c = np.cumsum(p[b, 0].astype(np.float64))
        target = float(u[b, 0]) * c[-1]
        lo = c[vg - 1] if vg > 0 else 0.0
        assert lo - CDF_TOL * c[-1] <= target <= c[vg] + CDF_TOL * c[-1]
    # a drafted token outside its row's candidates: count -1, device check error, no fault
    p2, x, cid, cq, r, u2 = _chain_case(rng, 2, 2, 16, 500, equal_rows=set())
    x[1, 0] = next(v for v in range(500) if v not in set(cid[1, 0].tolist()))
    tokens, count = L.verify_chain(_t(p2), _t(x), _t(cid), _t(cq), _t(r), _t(u2))
    assert host(count)[1] == -1
    assert L.last_device_error() == -7
    assert L.last_device_error() == 0


@pytest.mark.parametrize("n", [40, 70, 300, 2049])
def test_verify_chain_small_vocabularies(L, n):
    """Vocabularies of a few 32-entry chunks: most CTAs of a chain's cluster
    own an empty slice (n = 40 has two chunks for eight CTAs)."""
    rng = np.random.default_rng(1000 + n)
    B, Kd, K = 6, 2, 8
    p, x, cid, cq, r, u = _chain_case(rng, B, Kd, K, n, equal_rows={1})
    tokens, count = L.verify_chain(_t(p), _t(x), _t(cid), _t(cq), _t(r), _t(u))
    tokens, count = host(tokens), host(count)
    assert count[1] == Kd
    assert _check_chain(p, x, cid, cq, r, u, tokens, count) <= 1
    assert L.last_device_error() == 0
