"""CUDA path vs the fp64 oracle on the five seeded workloads at full size,
through the C ABI, in the launch configuration the bench times.

Workloads (seeded, synthetic; see synth/):
  0  n=4096   d=256  r=32,  M=1: global C=128; local tile 128, k_tile 4 (shuffled and identity)
  1  n=128256 d=4096 r=256, M in {1,4,8}: global C=1024 (identity order)
  2  same head, shuffled, M in {1,8,16,32,64}: local tile 256, k_tile 2 (1002 candidates);
     global C=1002 and 1024 for the recall comparison
  3  n=201088 d=2880 r=256, M=80 (8 sequences x 10-node tree): local 256/2; global C=1024
  4  n=151936 d=5120 r=512, M in {1,8,32,128,512}: local 256/4; dense; pruned 32000
Recall of the exact full-head Top-{1,8,64} is printed, and written to
$LMHEAD_REPORT_DIR/recall_*.json when that variable names a folder (a report,
not a pass/fail criterion).
"""
import json
import os

import numpy as np
import pytest

import oracle as O
import synth

from gpu_util import dev_bf16, dev_i32, host, lib, oracle_scores, workload_case
import parity as P

pytestmark = pytest.mark.gpu

OUT = os.environ.get("LMHEAD_REPORT_DIR", "")


@pytest.fixture(scope="module")
def L():
    return lib()


def _run(L, case, mode, C, k, temperature=1.0):
    W, A, B = dev_bf16(case["W"]), dev_bf16(case["A"]), dev_bf16(case["B"])
    h, tok = dev_bf16(case["h"]), dev_i32(case["tok"])
    md = L.LOCAL if mode == "local" else L.GLOBAL
    ids, lg, q = L.two_stage(md, W, A, B, h, tok, C, k, temperature=temperature)
    assert L.last_device_error() == 0
    return host(ids), host(lg), host(q)


def _gpu_u(L, case):
    """u as the library's projection computes it for this call's (d, M)
    (the kernel is chosen by d and M only, and sums in a fixed order)."""
    import torch
    u = L.project_u(dev_bf16(case["B"]), dev_bf16(case["h"]))
    return host(u.view(torch.int16)).view(np.uint16)


def _check(L, case, mode, C, k, ids, lg, q, rows=None, temperature=1.0, name=None):
    """Parity of one call on the rows `rows` (default all), recorded in the
    session's parity report: excused ids split into the 1e-3 band and the
    u-rounding slack, u elements that rounded the other way, and the spread
    of q (so a one-hot q, where the 1e-4 check is vacuous, shows)."""
    rows = np.arange(case["M"]) if rows is None else np.asarray(rows)
    sub = dict(case)
    sub["h"] = case["h"][rows]
    _, S, h64, SL = oracle_scores(sub, with_slack=True, M_call=case["M"])
    counts = P.check_ids(mode, ids[rows], S, case["tok"], C, k, slack_pos=SL)
    ex = P.exact_logits(case["W"], h64, ids[rows])
    floor = P.check_logits(lg[rows], ex)
    bite = P.check_q(q[rows], ex, temperature)
    flips, amb = P.check_u(_gpu_u(L, case)[rows], O.bf16_bits_to_f64(case["B"]), h64,
                           M_call=case["M"])
    label = name or f"{mode} n={case['n']} M={case['M']}"
    P.record(label, mode=mode, M=int(case["M"]), rows=int(len(rows)), **counts,
             logit_floor=floor, **bite, u_flips=flips, u_ambiguous=amb,
             temperature=float(temperature))
    return counts


def _candidate_temperature(case, mode, C, k):
    """The temperature at which q bites: the standard deviation of the exact
    logits over the oracle's own candidates of row 0 (oracle only)."""
    A64 = O.bf16_bits_to_f64(case["A"])
    h0 = O.bf16_bits_to_f64(case["h"][:1])
    u = O.project_u(O.bf16_bits_to_f64(case["B"]), h0)
    S = O.lowrank_scores(A64, u)[0]
    if mode == "local":
        ids, _ = O.local_topk(S, case["tok"], C, k)
    else:
        ids, _ = O.global_topk(S, case["tok"], C)
    Lx = O.candidate_logits(O.bf16_bits_to_f64(case["W"][ids]), h0[0], np.arange(len(ids)))
    return float(np.std(Lx))


def _dense_exact(W_bits, h64, block=16384):
    Z = np.empty((h64.shape[0], W_bits.shape[0]))
    for r0 in range(0, W_bits.shape[0], block):
        Z[:, r0:r0 + block] = h64 @ O.bf16_bits_to_f64(W_bits[r0:r0 + block]).T
    return Z


def _report(name, payload):
    if os.path.isdir(OUT):
        with open(os.path.join(OUT, f"recall_{name}.json"), "w") as fh:
            json.dump(payload, fh, indent=1)
    print(name, json.dumps(payload))


def test_workload0_tiny(L):
    wl = synth.workload(0)
    for shuffle in (True, False):
        case = workload_case(wl, 1, shuffle=shuffle)
        ids, lg, q = _run(L, case, "local", wl.T, wl.k_tile)
        assert ids.shape == (1, 128)
        _check(L, case, "local", wl.T, wl.k_tile, ids, lg, q,
               name=f"wl0 local 128/4 {'shuffled' if shuffle else 'identity'} M=1")
    case = workload_case(wl, 1)
    ids, lg, q = _run(L, case, "global", wl.C, 0)
    _check(L, case, "global", wl.C, 0, ids, lg, q, name="wl0 global C=128 M=1")


@pytest.mark.parametrize("M", [1, 4, 8])
def test_workload1_global(L, M):
    wl = synth.workload(1)
    case = workload_case(wl, M)
    ids, lg, q = _run(L, case, "global", wl.C, 0)
    assert ids.shape == (M, 1024)
    _check(L, case, "global", wl.C, 0, ids, lg, q, name=f"wl1 global C=1024 M={M}")


@pytest.mark.parametrize("M", [1, 8, 16, 32, 64])
def test_workload2_local(L, M):
    wl = synth.workload(2)
    case = workload_case(wl, M)
    ids, lg, q = _run(L, case, "local", wl.T, wl.k_tile)
    assert ids.shape == (M, 1002)
    _check(L, case, "local", wl.T, wl.k_tile, ids, lg, q, name=f"wl2 local 256/2 M={M}")
    if M == 64:
        h64 = O.bf16_bits_to_f64(case["h"])
        Z = _dense_exact(case["W"], h64)
        g1002, gl2, gq2 = _run(L, case, "global", 1002, 0)
        _check(L, case, "global", 1002, 0, g1002, gl2, gq2, rows=[0, 31, 63],
               name="wl2 global C=1002 M=64 (3 rows)")
        g1024, gl4, gq4 = _run(L, case, "global", 1024, 0)
        _check(L, case, "global", 1024, 0, g1024, gl4, gq4, rows=[0, 31, 63],
               name="wl2 global C=1024 M=64 (3 rows)")
        rep = {}
        for name, cand in (("local_1002", ids), ("global_1002", g1002), ("global_1024", g1024)):
            rep[name] = {f"recall@{k}": float(np.mean([O.recall_at(cand[m], Z[m], k) for m in range(M)]))
                         for k in (1, 8, 64)}
        _report("workload2", rep)
        assert rep["local_1002"]["recall@1"] > 0.9


def test_workload3_tree(L):
    wl = synth.workload(3)
    case = workload_case(wl, 80)
    ids, lg, q = _run(L, case, "local", wl.T, wl.k_tile)
    assert ids.shape == (80, 1572)
    _check(L, case, "local", wl.T, wl.k_tile, ids, lg, q, name="wl3 tree local 256/2 M=80")
    gi, gl, gq = _run(L, case, "global", wl.C, 0)
    _check(L, case, "global", wl.C, 0, gi, gl, gq, rows=[0, 1, 9, 37, 79],
           name="wl3 tree global C=1024 M=80 (5 rows)")
    h64 = O.bf16_bits_to_f64(case["h"][:16])
    Z = _dense_exact(case["W"], h64)
    rep = {name: {f"recall@{k}": float(np.mean([O.recall_at(c[m], Z[m], k) for m in range(16)]))
                  for k in (1, 8, 64)} for name, c in (("local_1572", ids), ("global_1024", gi))}
    _report("workload3", rep)


@pytest.mark.parametrize("M", [1, 8, 32, 128, 512])
def test_workload4_wide(L, M):
    wl = synth.workload(4)
    case = workload_case(wl, M)
    ids, lg, q = _run(L, case, "local", wl.T, wl.k_tile)
    assert ids.shape == (M, 2376)
    rows = None if M <= 32 else sorted({0, 1, M // 2, M - 1, *range(7, M, M // 6)})
    _check(L, case, "local", wl.T, wl.k_tile, ids, lg, q, rows=rows,
           name=f"wl4 local 256/4 M={M}" + ("" if rows is None else f" ({len(rows)} rows)"))


@pytest.mark.parametrize("index,M", [(2, 16), (3, 80), (4, 8)])
def test_q_bites_plain_hidden(L, index, M):
    """q parity where it is not one-hot: hidden states N(0,1) without the
    W[t] spike, temperature = std of the exact logits over the candidates."""
    wl = synth.workload(index)
    case = workload_case(wl, M)
    case["h"] = synth.make_plain_hidden(wl.d, M, wl.index)
    T = _candidate_temperature(case, "local", wl.T, wl.k_tile)
    ids, lg, q = _run(L, case, "local", wl.T, wl.k_tile, temperature=T)
    _check(L, case, "local", wl.T, wl.k_tile, ids, lg, q, temperature=T,
           name=f"wl{index} local plain h, T=std(L) M={M}")
    live = [int((q[m] > P.Q_ABS).sum()) for m in range(M)]
    assert np.median(live) >= 20, "q is nearly one-hot: the check would not bite"


def test_q_bites_recipe_hidden(L):
    """The spike recipe at T = std(L over candidates) (workload 2, M = 8),
    local and global."""
    wl = synth.workload(2)
    case = workload_case(wl, 8)
    for mode, C, k in (("local", wl.T, wl.k_tile), ("global", 1024, 0)):
        T = _candidate_temperature(case, mode, C, k)
        ids, lg, q = _run(L, case, mode, C, k, temperature=T)
        _check(L, case, mode, C, k, ids, lg, q, temperature=T,
               name=f"wl2 {mode} recipe h, T=std(L) M=8")


@pytest.mark.parametrize("M", [1, 32])
def test_workload4_dense_and_pruned(L, M):
    wl = synth.workload(4)
    case = workload_case(wl, M)
    W, h = dev_bf16(case["W"]), dev_bf16(case["h"])
    lg, q = L.dense_head(W, h)
    rows = [0, M - 1]
    h64 = O.bf16_bits_to_f64(case["h"][rows])
    Z = _dense_exact(case["W"], h64)
    P.check_logits(host(lg)[rows], Z)
    for i, m in enumerate(rows):
        assert np.abs(host(q)[m] - O.candidate_softmax(Z[i])).max() < P.Q_ABS
    keep = O.pruned_ids(O.smooth_freq(case["counts"]), 32000)
    lp, qp = L.pruned_head(dev_bf16(case["W"][keep]), h)
    P.check_logits(host(lp)[rows], Z[:, keep])
    for i, m in enumerate(rows):
        assert np.abs(host(qp)[m] - O.candidate_softmax(Z[i, keep])).max() < P.Q_ABS


def test_workload2_draft_select_and_verify(L):
    # the steps after q on the headline head: q and ids from the two-stage call,
    # targets p = the dense head's full-vocabulary softmax of the same hidden vectors
    import torch
    wl = synth.workload(2)
    Bc, Kd = 4, 3
    M = Bc * (Kd + 1)
    case = workload_case(wl, M)
    W, A, B = dev_bf16(case["W"]), dev_bf16(case["A"]), dev_bf16(case["B"])
    h, tok = dev_bf16(case["h"]), dev_i32(case["tok"])
    ids, lg, q = L.two_stage(L.LOCAL, W, A, B, h, tok, wl.T, wl.k_tile, temperature=0.8)
    _, p = L.dense_head(W, h, 0.8)
    rng = np.random.default_rng(7)
    K = ids.shape[1]
    U = np.clip(rng.random((M, K)), 1e-7, 1 - 1e-7).astype(np.float32)
    parent = rng.random(M).astype(np.float32)
    ti, tq, tv, si, sq = L.draft_select(q, ids, 8, torch.from_numpy(parent).cuda(),
                                        torch.from_numpy(U).cuda())
    qh, ih = host(q), host(ids)
    for m in range(M):
        oi, oq, ov = O.draft_topk(qh[m], ih[m], 8, parent[m])
        assert np.array_equal(host(ti)[m], oi) and np.array_equal(host(tv)[m], ov)
        gid, gj, s = O.gumbel_sample(qh[m], ih[m], U[m].astype(np.float64))
        j = int(np.nonzero(ih[m] == host(si)[m])[0][0])
        assert s[gj] - s[j] <= 1e-5 * (1 + abs(s[gj]))
    # chains: row (b, t) of the batch is position t of chain b; drafts are the draws above
    rows = np.arange(M).reshape(Bc, Kd + 1)
    ph = host(p).reshape(Bc, Kd + 1, -1)
    cid = ih[rows[:, :Kd]]
    cq = qh[rows[:, :Kd]]
    x = host(si)[rows[:, :Kd]].astype(np.int32)
    r = rng.random((Bc, Kd)).astype(np.float32)
    u = rng.random((Bc, Kd + 1)).astype(np.float32)
    tokens, count = L.verify_chain(p.reshape(Bc, Kd + 1, -1).contiguous(),
                                   torch.from_numpy(x).cuda(), torch.from_numpy(cid).cuda(),
                                   torch.from_numpy(cq).cuda(), torch.from_numpy(r).cuda(),
                                   torch.from_numpy(u).cuda())
    tokens, count = host(tokens), host(count)
    for b in range(Bc):
        n_acc, out = O.verify_chain(ph[b], x[b], cid[b], cq[b], r[b], u[b])
        assert count[b] == n_acc and list(tokens[b, :n_acc]) == out[:n_acc]
        vg, vo = int(tokens[b, n_acc]), out[n_acc]
        if vg != vo:
            w = ph[b, n_acc].astype(np.float64) if n_acc == Kd else \
                O.residual(ph[b, n_acc], cid[b, n_acc], cq[b, n_acc])
            c = np.cumsum(w)
            target = float(u[b, n_acc]) * c[-1]
            lo = c[vg - 1] if vg > 0 else 0.0
            assert w[vg] > 0 and lo - 1e-4 * c[-1] <= target <= c[vg] + 1e-4 * c[-1]
    assert L.last_device_error() == 0
