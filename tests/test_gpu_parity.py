"""CUDA path vs the fp64 oracle on small seeded heads (several tiles, ragged
tails, edge cases), through the C ABI. Full-size workloads are in
test_gpu_workloads.py."""
import numpy as np
import pytest

import oracle as O
import synth

from gpu_util import dev_bf16, dev_i32, host, lib, make_case, oracle_scores
import parity as P

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def L():
    return lib()


@pytest.fixture(scope="module")
def small():
    return make_case(1000, 64, 16, 17, seed=11)


def _dev(case):
    return (dev_bf16(case["W"]), dev_bf16(case["A"]), dev_bf16(case["B"]),
            dev_bf16(case["h"]), dev_i32(case["tok"]))


def test_project_u(L, small):
    # every M the projection dispatches on: GEMV (M <= 8) and tensor cores
    for M in (1, 2, 8, 9, 17):
        W, A, B, h, tok = _dev(small)
        h = h[:M].contiguous()
        u = L.project_u(B, h)
        flips, amb = P.check_u(host(u.view(__import__("torch").int16)).view(np.uint16),
                               O.bf16_bits_to_f64(small["B"]), O.bf16_bits_to_f64(small["h"][:M]))
        P.record(f"project_u d=64 r=16 M={M}", u_flips=flips, u_ambiguous=amb)


@pytest.mark.parametrize("M", [1, 3, 17])
@pytest.mark.parametrize("T,k", [(128, 1), (128, 2), (128, 4), (100, 32), (7, 3), (1000, 16),
                                 (4096, 8), (128, 40), (300, 300)])
def test_local_select(L, small, M, T, k):
    case = dict(small)
    case["h"] = small["h"][:M]
    W, A, B, h, tok = _dev(case)
    ids, sc = L.lowrank_score_topk(L.LOCAL, A, B, h, tok, T, k, with_scores=True)
    _, S, _, SL = oracle_scores(case, with_slack=True)
    P.check_ids("local", host(ids), S, case["tok"], T, k, slack_pos=SL)
    P.check_order("local", host(ids), host(sc), T, k, case["n"])
    assert ids.shape[1] == O.local_candidate_count(case["n"], T, k)
    assert L.last_device_error() == 0


@pytest.mark.parametrize("M", [1, 5])
@pytest.mark.parametrize("C", [1, 64, 777, 1000])
def test_global_select(L, small, M, C):
    case = dict(small)
    case["h"] = small["h"][:M]
    W, A, B, h, tok = _dev(case)
    ids, sc = L.lowrank_score_topk(L.GLOBAL, A, B, h, tok, C, with_scores=True)
    _, S, _, SL = oracle_scores(case, with_slack=True)
    P.check_ids("global", host(ids), S, case["tok"], C, slack_pos=SL)
    P.check_order("global", host(ids), host(sc), C, 0, case["n"])


def test_global_select_long_rows(L):
    # rows long enough for the multi-pass radix path (> 8192 keys)
    case = make_case(20000, 64, 16, 3, seed=12)
    W, A, B, h, tok = _dev(case)
    _, S, _, SL = oracle_scores(case, with_slack=True)
    for C in (1, 100, 1024, 4096):
        ids = L.lowrank_score_topk(L.GLOBAL, A, B, h, tok, C)
        P.check_ids("global", host(ids), S, case["tok"], C, slack_pos=SL)


@pytest.mark.parametrize("M", [1, 2, 16])
def test_global_select_several_ctas_order(L, M):
    # the several-CTA selection on random scores (n = 30001: odd rows, off a
    # 16-byte boundary after the first): ids against the oracle, every row
    # score-descending with equal scores by ascending id and no id twice.
    # r = 256: M <= 2 counts the first histogram in the GEMV score writeback;
    # M = 16 places the keys two to a lane.
    n, d, r = 30001, 256, 256
    case = make_case(n, d, r, M, seed=41, plain_h=True)
    W, A, B, h, tok = _dev(case)
    _, S, _, SL = oracle_scores(case, with_slack=True)
    for C in (1, 64, 1000, 4096):
        ids, sc = L.lowrank_score_topk(L.GLOBAL, A, B, h, tok, C, with_scores=True)
        ids, sc = host(ids), host(sc)
        P.check_ids("global", ids, S, case["tok"], C, slack_pos=SL)
        P.check_order("global", ids, sc, C, 0, n)
        for m in range(M):
            assert np.unique(ids[m]).size == C, (C, m)
            tie = sc[m, 1:] == sc[m, :-1]
            assert np.all(ids[m, 1:][tie] > ids[m, :-1][tie]), (C, m)
    assert L.last_device_error() == 0


@pytest.mark.parametrize("M", [1, 3])
def test_global_select_all_scores_tied(L, M):
    # every row of A equal: all scores tie, so the Top-C is exactly the C
    # smallest vocabulary ids, in ascending order (rows long enough for the
    # several-CTAs-per-row selection)
    import torch
    n, r, d = 12000, 16, 64
    case = make_case(n, d, r, M, seed=15)
    A = np.repeat(case["A"][:1], n, axis=0)
    tok = dev_i32(case["tok"])
    for C in (1, 777, 4096):
        ids, sc = L.lowrank_score_topk(L.GLOBAL, dev_bf16(A), dev_bf16(case["B"]),
                                       dev_bf16(case["h"]), tok, C, with_scores=True)
        ids, sc = host(ids), host(sc)
        for m in range(M):
            assert np.array_equal(ids[m], np.arange(C)), (C, m)
            assert np.all(sc[m] == sc[m, 0])
    assert L.last_device_error() == 0


@pytest.mark.parametrize("n_tie", [2000, 5000])
@pytest.mark.parametrize("M", [1, 2, 3])
def test_global_select_three_score_levels(L, M, n_tie):
    # every row of A is 2a, a or a/2 for one row a with a.u > 0, and the
    # hidden rows are h, h/2, 2h: each row's scores are exactly 2s, s and s/2
    # (power-of-two scaling is exact in bf16 and in the fp32 sums). With 700
    # rows at 2s and n_tie rows at s, the Top-1024 is the 2s rows by id, then
    # the 324 smallest ids of the s rows. 2000 tied rows leave the several-CTA
    # selection's final range with 2000 keys (the ranking takes its chunks in
    # turns); 5000 are more than its lists hold (one CTA finishes the row). M
    # <= 2 counts the first histogram in the GEMV score writeback (r = 256),
    # M = 3 in a pass kernel. n % 4 = 3: rows after the first start off a
    # 16-byte boundary (the score scans' scalar head and tail).
    n, d, r, C, n_hi = 20003, 64, 256, 1024, 700
    g = np.random.default_rng(71)
    B = synth.bf16_bits_from_f32((g.standard_normal((r, d)) / 8).astype(np.float32))
    h0 = g.standard_normal(d).astype(np.float32)
    h = synth.bf16_bits_from_f32(np.stack([h0 * c for c in (1.0, 0.5, 2.0)[:M]]).astype(np.float32))
    u = O.project_u(O.bf16_bits_to_f64(B), O.bf16_bits_to_f64(h[:1]))[0]
    a = (np.where(u >= 0, 1.0, -1.0) * (0.5 + g.random(r))).astype(np.float32)
    a = synth.bf16_bits_to_f32(synth.bf16_bits_from_f32(a))
    perm = g.permutation(n)
    A = np.empty((n, r), dtype=np.float32)
    A[:] = 0.5 * a
    A[perm[:n_hi]] = 2.0 * a
    A[perm[n_hi:n_hi + n_tie]] = a
    tok = g.permutation(n).astype(np.int32)
    ids, sc = L.lowrank_score_topk(L.GLOBAL, dev_bf16(synth.bf16_bits_from_f32(A)), dev_bf16(B),
                                   dev_bf16(h), dev_i32(tok), C, with_scores=True)
    ids, sc = host(ids), host(sc)
    want = np.concatenate([np.sort(tok[perm[:n_hi]]),
                           np.sort(tok[perm[n_hi:n_hi + n_tie]])[:C - n_hi]])
    for m in range(M):
        assert np.array_equal(ids[m], want), m
        assert np.all(sc[m, :n_hi] == sc[m, 0]) and np.all(sc[m, n_hi:] == sc[m, n_hi])
        assert sc[m, n_hi] > 0 and sc[m, 0] == 2 * sc[m, n_hi]
    assert L.last_device_error() == 0


def test_scores_match_oracle(L, small):
    W, A, B, h, tok = _dev(small)
    ids, sc = L.lowrank_score_topk(L.LOCAL, A, B, h, tok, 128, 4, with_scores=True)
    _, S, _ = oracle_scores(small)
    ids, sc = host(ids), host(sc)
    A64 = O.bf16_bits_to_f64(small["A"])
    inv = np.empty(small["n"], dtype=np.int64)
    inv[small["tok"]] = np.arange(small["n"])
    u = O.project_u(O.bf16_bits_to_f64(small["B"]), O.bf16_bits_to_f64(small["h"]))
    for m in range(ids.shape[0]):
        pos = inv[ids[m]]
        bound = 1e-5 * (np.abs(A64[pos]) @ np.abs(u[m])) + 1e-6
        assert np.all(np.abs(sc[m] - S[m, pos]) <= bound)


@pytest.mark.parametrize("mode,C,k", [("local", 128, 2), ("local", 64, 40), ("global", 300, 0)])
@pytest.mark.parametrize("temp", [1.0, 0.37])
def test_two_stage(L, mode, C, k, temp):
    case = make_case(1500, 128, 24, 6, seed=13, plain_h=True)
    W, A, B, h, tok = _dev(case)
    md = L.LOCAL if mode == "local" else L.GLOBAL
    ids, lg, q = L.two_stage(md, W, A, B, h, tok, C, k, temperature=temp)
    _, S, h64, SL = oracle_scores(case, with_slack=True)
    ids = host(ids)
    P.check_ids(mode, ids, S, case["tok"], C, k, slack_pos=SL)
    ex = P.exact_logits(case["W"], h64, ids)
    P.check_logits(host(lg), ex)
    P.check_q(host(q), ex, temp)


@pytest.mark.parametrize("T,k", [(256, 2), (64, 8), (32, 1)])
@pytest.mark.parametrize("M", [1, 2, 3, 4])
def test_two_stage_gemv_scoring(L, M, T, k):
    # up to four hidden vectors at r = 256 take the CUDA-core scoring kernel
    # (tiles of 32-256 rows in one 256-row CTA; one, two or four vectors per
    # CTA). d = 264: W rows and h end off
    # a 256-element step; n = 5003: the last tile is partial and the last CTA
    # holds tile slots past n.
    case = make_case(5003, 264, 256, M, seed=23, plain_h=True)
    W, A, B, h, tok = _dev(case)
    ids, lg, q = L.two_stage(L.LOCAL, W, A, B, h, tok, T, k, temperature=0.7)
    _, S, h64, SL = oracle_scores(case, with_slack=True)
    ids = host(ids)
    P.check_ids("local", ids, S, case["tok"], T, k, slack_pos=SL)
    ex = P.exact_logits(case["W"], h64, ids)
    P.check_logits(host(lg), ex)
    P.check_q(host(q), ex, 0.7)
    assert L.last_device_error() == 0


@pytest.mark.parametrize("M", [1, 2, 4])
def test_gemv_scoring_rank_512(L, M):
    # r = 512 on the CUDA-core GEMV kernel (two 16-byte pieces of a row per
    # lane, four rows a batch): local two-stage calls over a few tile sizes,
    # and the global route on rows long enough for the several-CTA selection
    # (the GEMV writeback counts its first histogram)
    case = make_case(9001, 520, 512, M, seed=29, plain_h=True)
    W, A, B, h, tok = _dev(case)
    _, S, h64, SL = oracle_scores(case, with_slack=True)
    for T, k in ((256, 2), (64, 4)):
        ids, lg, q = L.two_stage(L.LOCAL, W, A, B, h, tok, T, k, temperature=0.7)
        ids = host(ids)
        P.check_ids("local", ids, S, case["tok"], T, k, slack_pos=SL)
        ex = P.exact_logits(case["W"], h64, ids)
        P.check_logits(host(lg), ex)
        P.check_q(host(q), ex, 0.7)
    for C in (1, 1000):
        ids, sc = L.lowrank_score_topk(L.GLOBAL, A, B, h, tok, C, with_scores=True)
        P.check_ids("global", host(ids), S, case["tok"], C, slack_pos=SL)
        P.check_order("global", host(ids), host(sc), C, 0, case["n"])
    assert L.last_device_error() == 0


def test_two_stage_identity_token_ids(L):
    case = make_case(1024, 64, 16, 2, seed=14, shuffle=False)
    W, A, B, h, _ = _dev(case)
    ids, lg, q = L.two_stage(L.LOCAL, W, A, B, h, None, 128, 4)
    _, S, h64, SL = oracle_scores(case, with_slack=True)
    P.check_ids("local", host(ids), S, np.arange(1024), 128, 4, slack_pos=SL)
    ex = P.exact_logits(case["W"], h64, host(ids))
    P.check_logits(host(lg), ex)
    P.check_q(host(q), ex)


def test_unit_tiles_cover_vocabulary(L):
    case = make_case(300, 32, 8, 2, seed=15, plain_h=True)
    W, A, B, h, tok = _dev(case)
    ids, lg, q = L.two_stage(L.LOCAL, W, A, B, h, tok, 1, 1)
    ids = host(ids)
    assert np.array_equal(ids[0], case["tok"]) and np.array_equal(ids[1], case["tok"])
    h64 = O.bf16_bits_to_f64(case["h"])
    Z = O.dense_logits(O.bf16_bits_to_f64(case["W"]), h64)
    for m in range(2):
        want = O.candidate_softmax(Z[m])[case["tok"]]
        assert np.abs(host(q)[m] - want).max() < P.Q_ABS


def test_one_tile_equals_global(L, small):
    W, A, B, h, tok = _dev(small)
    g = host(L.lowrank_score_topk(L.GLOBAL, A, B, h, tok, 16))
    l = host(L.lowrank_score_topk(L.LOCAL, A, B, h, tok, small["n"], 16))
    assert np.array_equal(g, l)


def test_gather_logits_and_bad_id(L, small):
    import torch
    W, A, B, h, tok = _dev(small)
    rng = np.random.default_rng(5)
    ids = rng.integers(0, small["n"], size=(small["M"], 37)).astype(np.int32)
    ids[0, :3] = [0, small["n"] - 1, 0]
    got = host(L.gather_logits(W, h, dev_i32(ids)))
    h64 = O.bf16_bits_to_f64(small["h"])
    P.check_logits(got, P.exact_logits(small["W"], h64, ids))
    assert L.last_device_error() == 0
    bad = ids.copy()
    bad[1, 5] = small["n"]
    bad[2, 0] = -1
    got = host(L.gather_logits(W, h, dev_i32(bad)))
    assert np.isnan(got[1, 5]) and np.isnan(got[2, 0])
    assert np.isfinite(np.delete(got.ravel(), [1 * 37 + 5, 2 * 37])).all()
    assert L.last_device_error() == -7   # LMHEAD_ERR_DEVICE_CHECK, then cleared
    assert L.last_device_error() == 0
    torch.cuda.synchronize()


@pytest.mark.parametrize("K", [1, 5, 1002, 70000, 200000, 300000])
@pytest.mark.parametrize("temp", [1.0, 3.0])
def test_candidate_softmax(L, K, temp):
    import torch
    x = np.random.default_rng(K).standard_normal((3, K)).astype(np.float32) * 6
    q = host(L.candidate_softmax(torch.from_numpy(x).cuda(), temp))
    for m in range(3):
        assert np.abs(q[m] - O.candidate_softmax(x[m].astype(np.float64), temp)).max() < P.Q_ABS
    # aliasing the output onto the input is allowed
    t = torch.from_numpy(x).cuda()
    L.candidate_softmax(t, temp, out=t)
    assert np.abs(host(t) - q).max() < 1e-6


@pytest.mark.parametrize("M", [1, 9])
def test_dense_and_pruned_head(L, M):
    case = make_case(700, 64, 16, M, seed=16, plain_h=True)
    W, A, B, h, tok = _dev(case)
    lg, q = L.dense_head(W, h, 0.8)
    h64 = O.bf16_bits_to_f64(case["h"])
    Z = O.dense_logits(O.bf16_bits_to_f64(case["W"]), h64)
    P.check_logits(host(lg), Z)
    for m in range(M):
        assert np.abs(host(q)[m] - O.candidate_softmax(Z[m], 0.8)).max() < P.Q_ABS
    keep = O.pruned_ids(O.smooth_freq(case["counts"]), 200)
    Wp = dev_bf16(case["W"][keep])
    lp, qp = L.pruned_head(Wp, h)
    P.check_logits(host(lp), Z[:, keep])
    for m in range(M):
        assert np.abs(host(qp)[m] - O.candidate_softmax(Z[m, keep])).max() < P.Q_ABS


def test_deterministic_repeats(L, small):
    W, A, B, h, tok = _dev(small)
    outs = [tuple(host(t) for t in L.two_stage(L.LOCAL, W, A, B, h, tok, 128, 4)) for _ in range(3)]
    for o in outs[1:]:
        for a, b in zip(outs[0], o):
            assert np.array_equal(a, b)


def test_host_validation_errors(L, small):
    import torch
    W, A, B, h, tok = _dev(small)
    with pytest.raises(L.LmheadError) as e:
        L.two_stage(L.LOCAL, W, A, B, h, tok, 4, 8)       # k_tile > T
    assert e.value.status == -2
    with pytest.raises(L.LmheadError) as e:
        L.two_stage(L.GLOBAL, W, A, B, h, tok, small["n"] + 1)
    assert e.value.status == -2
    tiny = torch.empty(16, dtype=torch.uint8, device="cuda")
    with pytest.raises(L.LmheadError) as e:
        L.two_stage(L.GLOBAL, W, A, B, h, tok, 64, workspace=tiny)
    assert e.value.status == -4


# Local mode at larger M: the gather takes the candidates in blocks of 16
# tiles (ragged last block when the tile count is not a multiple of 16);
# tiles of a multiple of 128 rows and not, d not a multiple of 64, M above
# one 128-row TMEM block of the scoring kernel, k_tile up to 8.
@pytest.mark.parametrize("M", [16, 33, 150])
@pytest.mark.parametrize("T,k", [(128, 2), (256, 4), (64, 8), (100, 3), (7, 3)])
def test_two_stage_larger_m(L, M, T, k):
    case = make_case(1500, 200, 24, M, seed=17, plain_h=True)
    W, A, B, h, tok = _dev(case)
    ids, lg, q = L.two_stage(L.LOCAL, W, A, B, h, tok, T, k, temperature=0.7)
    _, S, h64, SL = oracle_scores(case, with_slack=True)
    ids = host(ids)
    P.check_ids("local", ids, S, case["tok"], T, k, slack_pos=SL)
    ex = P.exact_logits(case["W"], h64, ids)
    P.check_logits(host(lg), ex)
    P.check_q(host(q), ex, 0.7)
    assert L.last_device_error() == 0


# Tiles of many 128-row chunks with a long per-tile list: the scoring kernel's
# epilogue then trails its MMAs by several chunks when the end of the work is
# signalled (the end marker must wait for its accumulator slot like a chunk).
@pytest.mark.parametrize("M", [1, 17, 33, 64, 150])
@pytest.mark.parametrize("n,T,k", [(1500, 4096, 8), (5000, 1024, 8), (5000, 2048, 4)])
def test_local_long_tiles(L, M, n, T, k):
    case = make_case(n, 64, 16, M, seed=19, plain_h=True)
    W, A, B, h, tok = _dev(case)
    ids, sc = L.lowrank_score_topk(L.LOCAL, A, B, h, tok, T, k, with_scores=True)
    assert L.last_device_error() == 0
    _, S, _, SL = oracle_scores(case, with_slack=True)
    P.check_ids("local", host(ids), S, case["tok"], T, k, slack_pos=SL)
    P.check_order("local", host(ids), host(sc), T, k, n)


# More 256-row tiles than SMs (n = 50000 is 196 tiles, the last one ragged):
# tiles claimed dynamically past the first round, 256-row MMAs, one and two
# 128-lane blocks of hidden vectors.
@pytest.mark.parametrize("M", [3, 64, 150])
@pytest.mark.parametrize("k", [1, 2, 8])
def test_local_more_tiles_than_sms(L, M, k):
    case = make_case(50000, 64, 16, M, seed=23, plain_h=True)
    W, A, B, h, tok = _dev(case)
    ids, sc = L.lowrank_score_topk(L.LOCAL, A, B, h, tok, 256, k, with_scores=True)
    assert L.last_device_error() == 0
    _, S, _, SL = oracle_scores(case, with_slack=True)
    P.check_ids("local", host(ids), S, case["tok"], 256, k, slack_pos=SL)
    P.check_order("local", host(ids), host(sc), 256, k, 50000)


# One or two hidden vectors at r = 256 take the warp-per-row GEMV scoring
# kernel: every tile size it serves (32-256 rows), k_tile 1 to 8 (3 is not a
# power of two), a ragged last CTA block and a ragged last tile.
@pytest.mark.parametrize("M", [1, 2])
@pytest.mark.parametrize("T,k", [(32, 1), (64, 3), (128, 4), (256, 2), (256, 8)])
def test_local_gemv_small_batches(L, M, T, k):
    case = make_case(5037, 512, 256, M, seed=29, plain_h=True)
    W, A, B, h, tok = _dev(case)
    ids, sc = L.lowrank_score_topk(L.LOCAL, A, B, h, tok, T, k, with_scores=True)
    assert L.last_device_error() == 0
    _, S, _, SL = oracle_scores(case, with_slack=True)
    P.check_ids("local", host(ids), S, case["tok"], T, k, slack_pos=SL)
    P.check_order("local", host(ids), host(sc), T, k, 5037)
    assert ids.shape[1] == O.local_candidate_count(5037, T, k)
    lg_ids, lg, q = L.two_stage(L.LOCAL, W, A, B, h, tok, T, k)
    h64 = O.bf16_bits_to_f64(case["h"])
    ex = P.exact_logits(case["W"], h64, host(lg_ids))
    P.check_logits(host(lg), ex)
    P.check_q(host(q), ex)


@pytest.mark.parametrize("M", [1, 9])
def test_local_wide_rank_cuda_cores(L, M):
    # r = 1280 is beyond the tensor-core scoring (r <= 512): the CUDA-core
    # kernel holds u (8 x r fp32 = 40 KB) next to ~13 KB of static shared
    # memory, over the 48 KB default
    case = make_case(3000, 1536, 1280, M, seed=19, plain_h=True)
    W, A, B, h, tok = _dev(case)
    ids, lg, q = L.two_stage(L.LOCAL, W, A, B, h, tok, 256, 4)
    assert L.last_device_error() == 0
    _, S, h64, SL = oracle_scores(case, with_slack=True)
    ids = host(ids)
    P.check_ids("local", ids, S, case["tok"], 256, 4, slack_pos=SL)
    ex = P.exact_logits(case["W"], h64, ids)
    P.check_logits(host(lg), ex)
    P.check_q(host(q), ex)


@pytest.mark.parametrize("M", [1, 17, 300])
def test_dense_head_blocks(L, M):
    # tensor cores at every M (N = M hidden vectors per MMA, M > 256 in blocks
    # of 256); n not a multiple of 128
    case = make_case(1000, 96, 16, M, seed=18, plain_h=True)
    W, A, B, h, tok = _dev(case)
    lg, q = L.dense_head(W, h)
    h64 = O.bf16_bits_to_f64(case["h"])
    Z = O.dense_logits(O.bf16_bits_to_f64(case["W"]), h64)
    P.check_logits(host(lg), Z)
    qq = host(q)
    for m in (0, M // 2, M - 1):
        assert np.abs(qq[m] - O.candidate_softmax(Z[m])).max() < P.Q_ABS
    assert L.last_device_error() == 0
