"""Pins of the oracle's next-row functions against what the pages and the
mathematics fix, not against the oracle itself:
  * the exact best-path walk (reading R17): exhaustive search over all 16^L
    slot paths with the same fp32 left-to-right sums, a special case that
    reduces to the greedy walk, a hand case where greedy is myopic, and the
    invariant best >= greedy;
  * the selector evaluation (reading R18): Table 1's printed acceptance
    lengths through the closed form, hand cases, and planted data whose mean
    acceptance lengths and conditional recalls match the closed form."""
import itertools
import math

import numpy as np
import pytest

import oracle
from conftest import read_golden_rows

K = 16


# ---------------------------------------------------------------------------
# exact best path
# ---------------------------------------------------------------------------
def brute_best(S):
    """All K^L paths of one sequence (S: [L, K, K] f32), sums in fp32 left to
    right: (max score, list of every path attaining it)."""
    L = S.shape[0]
    acc = S[0, 0, :].astype(np.float32)                       # [K]: paths of length 1
    for t in range(1, L):
        acc = (acc[..., None] + S[t][(None,) * (t - 1) + (slice(None), slice(None))]).astype(np.float32)
    best = acc.max()
    return best, [tuple(int(x) for x in p) for p in np.argwhere(acc == best)]


@pytest.mark.parametrize("L", [1, 2, 3])
def test_viterbi_matches_exhaustive_search(L):
    rng = np.random.default_rng(100 + L)
    B = 24
    S = rng.standard_normal((B, L, K, K)).astype(np.float32)
    ci = rng.integers(0, 5000, (B, L, K)).astype(np.int32)
    tok, slot, score = oracle.walk_viterbi(S, ci)
    unique = 0
    for b in range(B):
        best, paths = brute_best(S[b])
        assert score[b] == best
        if len(paths) == 1:
            unique += 1
            assert tuple(slot[b]) == paths[0]
        assert tuple(slot[b]) in paths
        assert list(tok[b]) == [ci[b, t, slot[b, t]] for t in range(L)]
    assert unique >= B - 2


def test_viterbi_without_predecessor_dependence_is_the_greedy_walk():
    # S[t][i][j] = u_t[j] for every i: the best path is the per-position arg-max
    rng = np.random.default_rng(7)
    B, L = 16, 12
    u = rng.standard_normal((B, L, 1, K)).astype(np.float32)
    S = np.broadcast_to(u, (B, L, K, K)).copy()
    ci = rng.integers(0, 1000, (B, L, K)).astype(np.int32)
    _, vslot, _ = oracle.walk_viterbi(S, ci)
    _, gslot, _, _ = oracle.walk(S, ci, temperature=0.0)
    assert np.array_equal(vslot, gslot)
    assert np.array_equal(vslot, u[:, :, 0, :].argmax(-1))


def test_viterbi_hand_case_where_greedy_is_myopic():
    S = np.full((1, 2, K, K), -1.0, np.float32)
    S[0, 0, 0, 0] = 1.0          # greedy takes slot 0 first ...
    S[0, 0, 0, 1] = 0.9
    S[0, 1, 0, :] = -10.0        # ... and then has nowhere good to go
    S[0, 1, 1, 5] = 5.0          # the best path goes through slot 1 to slot 5
    ci = np.arange(2 * K, dtype=np.int32).reshape(1, 2, K)
    tok, slot, score = oracle.walk_viterbi(S, ci)
    _, gslot, _, _ = oracle.walk(S, ci, temperature=0.0)
    assert list(gslot[0]) == [0, 0]
    assert list(slot[0]) == [1, 5] and list(tok[0]) == [1, K + 5]
    assert score[0] == np.float32(np.float32(0.9) + np.float32(5.0))


def test_viterbi_ties_take_the_lowest_slots():
    S = np.zeros((1, 3, K, K), np.float32)     # every path scores 0
    ci = np.zeros((1, 3, K), np.int32)
    _, slot, score = oracle.walk_viterbi(S, ci)
    assert list(slot[0]) == [0, 0, 0] and score[0] == 0.0


def test_viterbi_score_is_at_least_the_greedy_path():
    rng = np.random.default_rng(11)
    B, L = 64, 16
    S = (rng.standard_normal((B, L, K, K)) * 2).astype(np.float32)
    ci = rng.integers(0, 1000, (B, L, K)).astype(np.int32)
    _, _, vscore = oracle.walk_viterbi(S, ci)
    _, gslot, _, _ = oracle.walk(S, ci, temperature=0.0)
    for b in range(B):
        g = np.float32(S[b, 0, 0, gslot[b, 0]])
        for t in range(1, L):
            g = np.float32(g + S[b, t, gslot[b, t - 1], gslot[b, t]])
        assert vscore[b] >= g
    assert (vscore > -np.inf).all()


# ---------------------------------------------------------------------------
# selector evaluation
# ---------------------------------------------------------------------------
def test_closed_form_accept_reproduces_table1():
    for row in read_golden_rows("table1_recall.txt"):
        r = [float(x) for x in row[1:8]]
        printed = float(row[8])
        al = oracle.closed_form_accept(r)
        assert math.floor(al * 100) / 100 == printed   # printed truncated to 2 decimals


def test_selector_eval_hand_cases():
    L = 4
    gt = np.array([[10, 11, 12, 13],      # top-1 everywhere
                   [10, 11, 12, 13],      # in the 16 but never top-1
                   [10, 11, 12, 13],      # top-1, top-1, absent, top-1
                   [10, 11, 12, 13]], np.int32)
    ci = np.full((4, L, K), 99, np.int32)
    ci[:, :, 1:] = np.arange(200, 200 + K - 1)
    ci[0, :, 0] = gt[0]
    ci[1, :, 7] = gt[1]
    ci[2, [0, 1, 3], 0] = gt[2, [0, 1, 3]]
    a1, a16, counts = oracle.selector_eval(gt, ci)
    assert list(a1) == [5, 1, 3, 1]
    assert list(a16) == [5, 5, 3, 1]
    # sequence 3 has no hits at all
    assert list(counts[0]) == [4, 2, 4, 3]            # t=0: all alive; hits: seq 0 and 2 / 0, 1, 2
    assert list(counts[1]) == [2, 2, 3, 3]
    assert list(counts[2]) == [2, 1, 3, 2]
    assert list(counts[3]) == [1, 1, 2, 2]


def test_selector_eval_planted_matches_the_closed_form():
    # Table 1's recalls planted independently per position: E[accept] = closed form,
    # and each position's conditional hit ratio estimates its recall
    rows = {row[0]: [float(x) for x in row[1:8]] for row in read_golden_rows("table1_recall.txt")}
    r1, r16 = np.array(rows["recall@1"]), np.array(rows["recall@16"])
    B, L = 20000, 7
    rng = np.random.default_rng(3)
    gt = rng.integers(0, 1 << 20, (B, L)).astype(np.int32)
    ci = rng.integers(1 << 21, 1 << 22, (B, L, K)).astype(np.int32)   # never a true token
    u = rng.random((B, L))
    top = u < r1
    inside = (~top) & (u < r16)
    slot = rng.integers(1, K, (B, L))
    bb, tt = np.nonzero(top)
    ci[bb, tt, 0] = gt[bb, tt]
    bb, tt = np.nonzero(inside)
    ci[bb, tt, slot[bb, tt]] = gt[bb, tt]
    a1, a16, counts = oracle.selector_eval(gt, ci)
    for acc, r in ((a1, r1), (a16, r16)):
        expect = oracle.closed_form_accept(r)
        assert abs(acc.mean() - expect) < 4 * acc.std() / math.sqrt(B)
    for t in range(L):
        for n_col, h_col, r in ((0, 1, r1[t]), (2, 3, r16[t])):
            n, h = counts[t, n_col], counts[t, h_col]
            sd = math.sqrt(r * (1 - r) / n)
            assert abs(h / n - r) < 4 * sd + 1e-9


# ---------------------------------------------------------------------------
# best path vs greedy on planted data (acceptance length through the T=0 verify)
# ---------------------------------------------------------------------------
def planted_acceptance(seed, B, L, V, mu, sigma=1.0):
    from draft_selection_dflash2_gb300 import synth
    S, ci, _, true_tok = synth.planted_path(seed, B, L, V, mu=mu, sigma=sigma)
    target = synth.target_planted(seed + 1, true_tok, V, agree=1.0)
    gtok, gslot, gq, _ = oracle.walk(S, ci, temperature=0.0)
    vtok, vslot, _ = oracle.walk_viterbi(S, ci)
    ag, _, _ = oracle.verify(target, gtok, gslot, gq, ci, temperature=0.0)
    av, _, _ = oracle.verify(target, vtok, vslot, gq, ci, temperature=0.0)
    lead = lambda tok: 1 + np.cumprod(tok == true_tok, axis=1).sum(axis=1)   # noqa: E731
    return ag, av, lead(gtok), lead(vtok)


def test_planted_path_without_noise_is_found_by_both_walks():
    ag, av, lg, lv = planted_acceptance(1, 32, 12, 600, mu=5.0, sigma=0.0)
    assert (ag == 13).all() and (av == 13).all()


def test_best_path_accepts_more_than_greedy_on_planted_data():
    # the verifier's acceptance equals 1 + the leading run of true tokens (the
    # planted target's arg-max is the true token), for both walks; the best path
    # uses later positions' evidence, so its mean acceptance is higher
    ag, av, lg, lv = planted_acceptance(2, 256, 16, 800, mu=3.0)
    assert np.array_equal(ag, lg) and np.array_equal(av, lv)
    assert av.mean() > ag.mean() + 0.5


# ---------------------------------------------------------------------------
# projection-form selector (reading R19), pinned to the table form (already
# pinned) through embeddings whose projections are exact
# ---------------------------------------------------------------------------
def _proj_case(seed, B, L, V, d, r=256):
    from draft_selection_dflash2_gb300 import synth
    rng = np.random.default_rng(seed)
    ci = rng.integers(0, V, (B, L, K)).astype(np.int32)
    cv = rng.standard_normal((B, L, K)).astype(np.float32)
    lv = rng.integers(0, V, B).astype(np.int32)
    H = rng.random((B, L, r))
    return synth, rng, ci, cv, lv, H


def test_projection_with_one_hot_embeddings_is_the_table_form():
    # E(v) = e_v: A(v) = column v of W_A exactly, so the table A[v, q] = W_A[q, v]
    B, L, V, d = 3, 5, 48, 64
    synth, rng, ci, cv, lv, H = _proj_case(1, B, L, V, d)
    E = np.zeros((V, d), np.uint16)
    E[np.arange(V), np.arange(V)] = synth.bf16_bits(np.float32(1.0))
    WA = synth.bf16_bits(rng.standard_normal((256, d)).astype(np.float32))
    WB = synth.bf16_bits(rng.standard_normal((256, d)).astype(np.float32))
    lv[1] = V + 7                                   # out of range: clamped and reported by both
    S, bad = oracle.pair_scores_proj(ci, cv, lv, H, E, WA, WB)
    St, bad_t = oracle.pair_scores(ci, cv, lv, H, np.ascontiguousarray(WA[:, :V].T),
                                   np.ascontiguousarray(WB[:, :V].T))
    assert bad and bad_t
    assert np.allclose(S, St, rtol=1e-13, atol=1e-13)


def test_projection_with_integer_embeddings_matches_exact_tables():
    # entries in {-1, 0, 1}: E W^T is an exact integer table (numpy integer matmul)
    B, L, V, d = 2, 4, 300, 64
    synth, rng, ci, cv, lv, H = _proj_case(2, B, L, V, d)
    Ei = rng.integers(-1, 2, (V, d))
    WAi = rng.integers(-1, 2, (256, d))
    WBi = rng.integers(-1, 2, (256, d))
    bits = lambda a: synth.bf16_bits(a.astype(np.float32))          # noqa: E731
    S, bad = oracle.pair_scores_proj(ci, cv, lv, H, bits(Ei), bits(WAi), bits(WBi))
    St, _ = oracle.pair_scores(ci, cv, lv, H, bits(Ei @ WAi.T), bits(Ei @ WBi.T))
    assert not bad
    assert np.allclose(S, St, rtol=1e-13, atol=1e-12)
    # a zero W_B removes the pair term: the scores are the candidate logits
    S0, _ = oracle.pair_scores_proj(ci, cv, lv, H, bits(Ei), bits(WAi), bits(0 * WBi))
    assert np.array_equal(S0, np.broadcast_to(cv[:, :, None, :], S0.shape).astype(np.float64))


# ---------------------------------------------------------------------------
# conv fused into the producing GEMM (reading R20), pinned to the conv
# (already pinned) through GEMMs whose output is exact in bf16
# ---------------------------------------------------------------------------
def _conv_parts(seed, B, L, d, bias):
    from draft_selection_dflash2_gb300 import synth
    c = synth.conv_inputs(seed, B, L, d, with_bias=bias)
    h = synth.normal_bits(seed + 50, (B, L, d))
    return synth, c, h


def test_fused_conv_with_identity_projection_is_the_conv():
    # W = I (K = d) and A = x: the GEMM returns x exactly
    B, L, d = 2, 5, 64
    synth, c, h = _conv_parts(1, B, L, d, True)
    I = np.zeros((d, d), np.uint16)
    I[np.arange(d), np.arange(d)] = synth.bf16_bits(np.float32(1.0))
    y = oracle.gemm_conv2tap(c.x, I, c.x_prev, h, c.k0, c.k1, c.W_c, b_c=c.b_c)
    ref = oracle.conv2tap(c.x, c.x_prev, c.k0, c.k1, c.W_c, b_c=c.b_c, h_bits=h)
    assert np.allclose(y, ref, rtol=1e-14, atol=1e-14)


def test_fused_conv_with_integer_projection_matches_conv_of_exact_x():
    # A, W in {-1, 0, 1} with K = 96: A W^T is an exact integer (numpy integer matmul),
    # exact in bf16, so the conv of its bf16 image is the fused result
    B, L, d, K = 3, 4, 128, 96
    synth, c, h = _conv_parts(2, B, L, d, False)
    rng = np.random.default_rng(9)
    Ai, Wi = rng.integers(-1, 2, (B, L, K)), rng.integers(-1, 2, (d, K))
    bits = lambda a: synth.bf16_bits(a.astype(np.float32))          # noqa: E731
    y = oracle.gemm_conv2tap(bits(Ai), bits(Wi), c.x_prev, h, c.k0, c.k1, c.W_c)
    ref = oracle.conv2tap(bits(Ai @ Wi.T), c.x_prev, c.k0, c.k1, c.W_c, h_bits=h)
    assert np.allclose(y, ref, rtol=1e-14, atol=1e-13)
    # k0 = 0, k1 = 1, no correction: y is x shifted by one position, the first
    # position of each block reading x_prev
    zero = np.zeros_like(c.k0)
    one = np.full_like(c.k1, synth.bf16_bits(np.float32(1.0)))
    y1 = oracle.gemm_conv2tap(bits(Ai), bits(Wi), c.x_prev, h, zero, one, 0 * c.W_c)
    x = (Ai @ Wi.T).astype(np.float64)
    assert np.array_equal(y1[:, 1:], x[:, :-1])
    assert np.array_equal(y1[:, 0], synth.bf16_to_f32(c.x_prev).astype(np.float64))
