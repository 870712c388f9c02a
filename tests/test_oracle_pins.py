"""Pins the CPU oracle to what the pages and the mathematics fix.

Each test checks the oracle against something other than itself: a published
known-answer vector, a closed form, a special case that reduces to a textbook
or library routine, an invariant, or brute force on a tiny input.  They are
chosen so that a dropped term, a wrong sign or index, or a transposed operand
in the oracle fails at least one of them.
"""
import math

import numpy as np
import pytest
from scipy import signal, stats

import oracle
from conftest import read_golden_rows
from draft_selection_dflash2_gb300 import synth

K = 16


def f32_bits(vals):
    return synth.bf16_bits(np.asarray(vals, np.float32))


# ---------------------------------------------------------------------------
# Philox4x32-10
# ---------------------------------------------------------------------------


def test_philox_known_answers():
    rows = read_golden_rows("philox4x32_10_kat.txt")
    assert len(rows) == 3
    for row in rows:
        v = [int(x, 16) for x in row]
        out = oracle.philox4x32_10(v[0:4], v[4:6])
        assert [int(x) for x in out] == v[6:10]


def test_uniform24_counter_layout():
    # u = (x0 >> 8) * 2^-24 of Philox(ctr = (b, t | stream << 24, off_lo, off_hi), key = seed).
    seed, b, t, stream, off = 0x1234_5678_9ABC_DEF0, 7, 5, 2, (3 << 32) | 11
    out = oracle.philox4x32_10([b, t | (stream << 24), 11, 3], [0x9ABCDEF0, 0x12345678])
    assert oracle.uniform24(seed, b, t, stream, off) == (int(out[0]) >> 8) / 2.0**24


def test_uniform24_is_uniform():
    u = np.array([oracle.uniform24(1, b, 0, 0, 0) for b in range(20000)])
    assert u.min() >= 0.0 and u.max() < 1.0
    assert stats.kstest(u, "uniform").pvalue > 1e-4


# ---------------------------------------------------------------------------
# top-16
# ---------------------------------------------------------------------------


def brute_topk(row_f32, k):
    order = sorted(range(len(row_f32)), key=lambda v: (-row_f32[v], v))
    return order[:k]


def test_topk_brute_force_with_ties():
    rng = np.random.default_rng(3)
    for V in (16, 17, 40, 129):
        # values from a tiny set so that exact ties are everywhere
        vals = rng.choice(np.array([-2.0, -0.5, 0.0, 0.25, 1.0, 3.0], np.float32), size=(9, V))
        bits = f32_bits(vals)
        got_v, got_i = oracle.topk(bits, k=K)
        for r in range(9):
            ref = brute_topk(list(synth.bf16_to_f32(bits[r])), K)
            assert list(got_i[r]) == ref
            assert np.array_equal(got_v[r], synth.bf16_to_f32(bits[r])[ref])


def test_topk_planted_token_is_slot0():
    rng = np.random.default_rng(5)
    U = synth.logits_planted(rng, 12, 4096, plant=12.0)
    # the planted id is where the +12 went: the largest value by far
    planted = np.argmax(synth.bf16_to_f32(U), axis=1)
    _, idx = oracle.topk(U, k=K)
    assert np.array_equal(idx[:, 0], planted)


def test_topk_signed_zero_and_nan():
    row = np.full(32, -np.inf, np.float32)
    row[[3, 9, 20]] = [-0.0, 0.0, -0.0]   # three equal zeros: ids 3, 9, 20 in id order
    row[5] = np.nan                         # NaN ranks below -inf
    row[7] = 1.0
    vals, idx = oracle.topk(f32_bits(row)[None, :], k=K)
    assert list(idx[0, :4]) == [7, 3, 9, 20]
    assert 5 not in idx[0]
    # the 12 remaining slots are -inf entries in id order
    rest = [v for v in range(32) if v not in (3, 5, 7, 9, 20)][:12]
    assert list(idx[0, 4:]) == rest


def test_topk_respects_ld_and_V():
    rng = np.random.default_rng(8)
    V, ld = 100, 112
    bits = np.zeros((3, ld), np.uint16)
    bits[:, :V] = f32_bits(rng.standard_normal((3, V)))
    bits[:, V:] = f32_bits(np.full(ld - V, 50.0))  # padding must never be read
    _, idx = oracle.topk(bits, k=K, V=V)
    assert idx.max() < V
    for r in range(3):
        assert list(idx[r]) == brute_topk(list(synth.bf16_to_f32(bits[r, :V])), K)


# ---------------------------------------------------------------------------
# gate
# ---------------------------------------------------------------------------


def test_gate_zero_weights_is_one_half():
    h = f32_bits(np.random.default_rng(0).standard_normal((5, 64)))
    H = oracle.gate(h, np.zeros((256, 64), np.uint16))
    assert np.all(H == 0.5)


def test_gate_bias_only_is_logistic():
    b = np.linspace(-6, 6, 256).astype(np.float32)
    H = oracle.gate(np.zeros((2, 32), np.uint16), np.zeros((256, 32), np.uint16), b)
    ref = np.array([1.0 / (1.0 + math.exp(-float(x))) for x in b])
    assert np.allclose(H, ref[None, :], rtol=0, atol=1e-15)


def test_gate_single_entry_orientation():
    # h[m] = 2 e_5 and W_H[q, 5] = a_q: pre-activation = 2 a_q; W_H[q, k != 5] is
    # set to junk that a transposed product would pick up.
    d, r = 16, 256
    a = np.linspace(-1, 1, r).astype(np.float32)
    W = np.full((r, d), 3.0, np.float32)
    W[:, 5] = a
    h = np.zeros((1, d), np.float32)
    h[0, 5] = 2.0
    H = oracle.gate(f32_bits(h), f32_bits(W))
    Wb = synth.bf16_to_f32(f32_bits(W))
    ref = [1.0 / (1.0 + math.exp(-2.0 * float(Wb[q, 5]))) for q in range(r)]
    assert np.allclose(H[0], ref, rtol=0, atol=1e-15)


def test_gate_symmetry():
    rng = np.random.default_rng(1)
    h = f32_bits(rng.standard_normal((3, 48)))
    W = f32_bits(rng.standard_normal((256, 48)) * 0.1)
    b = rng.standard_normal(256).astype(np.float32)
    negW = W ^ np.uint16(0x8000)
    H = oracle.gate(h, W, b)
    Hn = oracle.gate(h, negW, -b)
    assert np.allclose(H + Hn, 1.0, rtol=0, atol=1e-14)


# ---------------------------------------------------------------------------
# pair scores
# ---------------------------------------------------------------------------


def _cands(rng, B, L, V):
    idx = np.stack([np.stack([rng.choice(V, K, replace=False) for _ in range(L)]) for _ in range(B)])
    val = np.sort(rng.standard_normal((B, L, K)).astype(np.float32), axis=-1)[..., ::-1]
    return idx.astype(np.int32), np.ascontiguousarray(synth.bf16_to_f32(f32_bits(val)))


def test_pairs_zero_embeddings_reduce_to_logits():
    rng = np.random.default_rng(2)
    B, L, V, r = 2, 5, 300, 256
    ci, cv = _cands(rng, B, L, V)
    H = rng.random((B, L, r))
    z = np.zeros((V, r), np.uint16)
    S, bad = oracle.pair_scores(ci, cv, np.array([1, 2], np.int32), H, z, z)
    assert not bad
    assert np.array_equal(S, np.broadcast_to(cv[:, :, None, :].astype(np.float64), S.shape))


def test_pairs_roles_of_predecessor_and_candidate():
    # A carries the predecessor, B the current candidate, H the position's gate.
    rng = np.random.default_rng(4)
    B, L, V, r = 1, 3, 200, 256
    ci, cv = _cands(rng, B, L, V)
    last = np.array([150], np.int32)
    ci[0, 0, 6] = 151  # candidate j=6 at t=0
    H = np.full((B, L, r), 0.5)
    H[0, 2, 9] = 0.25
    A = np.zeros((V, r), np.float32)
    Bm = np.zeros((V, r), np.float32)
    A[150, 9] = 2.0                   # predecessor of t = 0
    Bm[151, 9] = 3.0                  # candidate 6 at t = 0
    p2 = ci[0, 1, 3]                  # predecessor slot 3 at t = 2
    c2 = ci[0, 2, 11]                 # candidate slot 11 at t = 2
    A[p2, 9] = -1.5
    Bm[c2, 9] = 4.0
    S, _ = oracle.pair_scores(ci, cv, last, H, f32_bits(A), f32_bits(Bm))
    expect = np.broadcast_to(cv[:, :, None, :].astype(np.float64), S.shape).copy()
    expect[0, 0, :, 6] += 2.0 * 0.5 * 3.0          # every row at t = 0 (one predecessor)
    if c2 != 151:
        expect[0, 2, 3, 11] += -1.5 * 0.25 * 4.0
    assert np.array_equal(S, expect)
    # swapping the two tables must not give the same scores
    S_swapped, _ = oracle.pair_scores(ci, cv, last, H, f32_bits(Bm), f32_bits(A))
    assert not np.array_equal(S, S_swapped)


def test_pairs_bilinear_scaling():
    rng = np.random.default_rng(6)
    B, L, V, r = 2, 4, 128, 256
    ci, cv = _cands(rng, B, L, V)
    H = rng.random((B, L, r))
    A = f32_bits(rng.standard_normal((V, r)) * 0.25)
    Bm = f32_bits(rng.standard_normal((V, r)) * 0.25)
    last = np.array([3, 4], np.int32)
    S1, _ = oracle.pair_scores(ci, cv, last, H, A, Bm)
    A2 = f32_bits(synth.bf16_to_f32(A) * 2.0)  # exact in bf16
    S2, _ = oracle.pair_scores(ci, cv, last, H, A2, Bm)
    base = cv[:, :, None, :].astype(np.float64)
    assert np.allclose(S2 - base, 2.0 * (S1 - base), rtol=1e-12, atol=1e-12)
    # t = 0: the 16 rows are the same predecessor
    assert np.array_equal(S1[:, 0], np.broadcast_to(S1[:, 0, :1, :], S1[:, 0].shape))


def test_pairs_out_of_range_id_is_clamped_and_flagged():
    rng = np.random.default_rng(7)
    ci, cv = _cands(rng, 1, 2, 64)
    H = rng.random((1, 2, 256))
    A = f32_bits(rng.standard_normal((64, 256)))
    Bm = f32_bits(rng.standard_normal((64, 256)))
    S_hi, bad = oracle.pair_scores(ci, cv, np.array([1000], np.int32), H, A, Bm)
    S_ok, bad_ok = oracle.pair_scores(ci, cv, np.array([63], np.int32), H, A, Bm)
    assert bad and not bad_ok
    assert np.array_equal(S_hi, S_ok)


# ---------------------------------------------------------------------------
# walk
# ---------------------------------------------------------------------------


def test_walk_zero_embeddings_is_per_position_top1():
    rng = np.random.default_rng(9)
    B, L, V = 3, 6, 500
    ci, cv = _cands(rng, B, L, V)
    z = np.zeros((V, 256), np.uint16)
    S, _ = oracle.pair_scores(ci, cv, np.array([0, 1, 2], np.int32), rng.random((B, L, 256)), z, z)
    tok, slot, q, _ = oracle.walk(S.astype(np.float32), ci)
    assert np.all(slot == 0)
    assert np.array_equal(tok, ci[:, :, 0])
    assert np.array_equal(q, np.eye(K, dtype=np.float32)[np.zeros((B, L), int)])


def test_walk_greedy_brute_force():
    rng = np.random.default_rng(10)
    B, L = 4, 7
    S = rng.standard_normal((B, L, K, K)).astype(np.float32)
    S[:, :, :, 3] = S[:, :, :, 8]  # plant exact ties between slots 3 and 8
    ci = rng.integers(0, 1000, (B, L, K)).astype(np.int32)
    tok, slot, _, _ = oracle.walk(S, ci)
    for b in range(B):
        prev = None
        for t in range(L):
            best, best_pair = None, None
            for i in range(K):
                for j in range(K):
                    if (t == 0 and i != 0) or (t > 0 and i != prev):
                        continue
                    if best is None or S[b, t, i, j] > best:
                        best, best_pair = S[b, t, i, j], (i, j)
            assert slot[b, t] == best_pair[1]
            assert tok[b, t] == ci[b, t, best_pair[1]]
            prev = best_pair[1]


def test_walk_t0_reads_only_row0():
    rng = np.random.default_rng(11)
    S = rng.standard_normal((2, 3, K, K)).astype(np.float32)
    ci = rng.integers(0, 99, (2, 3, K)).astype(np.int32)
    S2 = S.copy()
    S2[:, 0, 1:, :] = rng.standard_normal((2, K - 1, K))
    a = oracle.walk(S, ci, temperature=0.7, seed=3)
    b = oracle.walk(S2, ci, temperature=0.7, seed=3)
    assert np.array_equal(a[1], b[1])


def test_walk_sampling_distribution_and_q():
    # one position, many sequences: slot frequencies ~ softmax(S/T); q closed form
    T = 0.8
    row = np.linspace(-1.0, 1.2, K).astype(np.float32)[::-1].copy()
    n = 40000
    S = np.broadcast_to(row, (n, 1, K, K)).astype(np.float32)
    ci = np.broadcast_to(np.arange(K, dtype=np.int32), (n, 1, K)).copy()
    _, slot, q, _ = oracle.walk(S, ci, temperature=T, seed=12)
    for j in range(K):
        for i in range(K):
            assert q[0, 0, i] / q[0, 0, j] == pytest.approx(math.exp((row[i] - row[j]) / T), rel=1e-6)
    assert q[0, 0].sum() == pytest.approx(1.0, abs=1e-6)
    counts = np.bincount(slot[:, 0], minlength=K)
    q64 = q[0, 0].astype(np.float64)
    assert stats.chisquare(counts, q64 / q64.sum() * n).pvalue > 1e-4


def test_walk_low_temperature_matches_greedy():
    rng = np.random.default_rng(13)
    S = (rng.standard_normal((6, 8, K, K)) * 3).astype(np.float32)
    ci = rng.integers(0, 99, (6, 8, K)).astype(np.int32)
    g = oracle.walk(S, ci)
    s = oracle.walk(S, ci, temperature=1e-4, seed=1)
    assert np.array_equal(g[1], s[1])


def test_walk_seed_and_offset_change_draws():
    S = np.zeros((64, 4, K, K), np.float32)
    ci = np.zeros((64, 4, K), np.int32)
    a = oracle.walk(S, ci, temperature=1.0, seed=1, offset=0)[1]
    b = oracle.walk(S, ci, temperature=1.0, seed=1, offset=1)[1]
    c = oracle.walk(S, ci, temperature=1.0, seed=2, offset=0)[1]
    assert not np.array_equal(a, b) and not np.array_equal(a, c)
    # with all scores equal, slot = floor(16 u) for the Philox uniform of (b, t, stream 0)
    for bb in range(8):
        for t in range(4):
            assert a[bb, t] == int(16 * oracle.uniform24(1, bb, t, 0, 0))


# ---------------------------------------------------------------------------
# conv
# ---------------------------------------------------------------------------


def _conv_case(seed, B=2, L=5, d=64):
    return synth.conv_inputs(seed, B, L, d)


def test_conv_identity():
    c = _conv_case(0)
    d = c.x.shape[-1]
    y = oracle.conv2tap(c.x, c.x_prev, f32_bits(np.ones(d)), np.zeros(d, np.uint16),
                        np.zeros_like(c.W_c))
    assert np.array_equal(y, synth.bf16_to_f32(c.x).astype(np.float64))


def test_conv_shift_reads_last_verified_at_t0():
    c = _conv_case(1)
    d = c.x.shape[-1]
    y = oracle.conv2tap(c.x, c.x_prev, np.zeros(d, np.uint16), f32_bits(np.ones(d)),
                        np.zeros_like(c.W_c))
    x = synth.bf16_to_f32(c.x)
    assert np.array_equal(y[:, 0], synth.bf16_to_f32(c.x_prev))
    assert np.array_equal(y[:, 1:], x[:, :-1])


def test_conv_static_kernel_is_textbook_fir():
    c = _conv_case(2)
    x = synth.bf16_to_f32(c.x).astype(np.float64)
    xp = synth.bf16_to_f32(c.x_prev).astype(np.float64)
    k0 = synth.bf16_to_f32(c.k0).astype(np.float64)
    k1 = synth.bf16_to_f32(c.k1).astype(np.float64)
    y = oracle.conv2tap(c.x, c.x_prev, c.k0, c.k1, np.zeros_like(c.W_c))
    B, L, d = x.shape
    for b in range(B):
        seq = np.concatenate([xp[b][None, :], x[b]], axis=0)
        for ch in range(d):
            ref = signal.lfilter([k0[ch], k1[ch]], [1.0], seq[:, ch])[1:]
            assert np.allclose(y[b, :, ch], ref, rtol=1e-13, atol=1e-13)


def test_conv_group_mapping_via_bias():
    # W_c = 0, b_c = beta: channel ch uses beta[ch // 16] on x_t and beta[G + ch // 16] on x_{t-1}
    c = _conv_case(3, d=64)
    G = 4
    beta = np.array([0.5, -1.0, 2.0, 0.25, 1.5, -0.75, 0.125, 3.0], np.float32)
    x = synth.bf16_to_f32(c.x).astype(np.float64)
    xp = synth.bf16_to_f32(c.x_prev).astype(np.float64)
    k0 = synth.bf16_to_f32(c.k0).astype(np.float64)
    k1 = synth.bf16_to_f32(c.k1).astype(np.float64)
    y = oracle.conv2tap(c.x, c.x_prev, c.k0, c.k1, np.zeros_like(c.W_c), b_c=beta)
    for b in range(x.shape[0]):
        seq = np.concatenate([xp[b][None, :], x[b]], axis=0)
        for ch in range(64):
            g = ch // 16
            ref = signal.lfilter([k0[ch] + beta[g], k1[ch] + beta[G + g]], [1.0], seq[:, ch])[1:]
            assert np.allclose(y[b, :, ch], ref, rtol=1e-13, atol=1e-13)


def test_conv_correction_orientation_one_hot_hidden():
    # h[m] = s_m e_7 (h given separately from x): c[m, n] = s_m W_c[n, 7]
    rng = np.random.default_rng(4)
    B, L, d = 1, 4, 32
    G = d // 16
    c = synth.conv_inputs(5, B, L, d)
    W = np.full((2 * G, d), 9.0, np.float32)     # junk outside column 7
    W[:, 7] = [0.5, -0.25, 1.0, 2.0]
    s = np.array([1.0, -2.0, 0.5, 4.0], np.float32)
    h = np.zeros((B, L, d), np.float32)
    h[0, :, 7] = s
    y = oracle.conv2tap(c.x, c.x_prev, c.k0, c.k1, f32_bits(W), h_bits=f32_bits(h))
    x = synth.bf16_to_f32(c.x)[0].astype(np.float64)
    xp = synth.bf16_to_f32(c.x_prev)[0].astype(np.float64)
    k0 = synth.bf16_to_f32(c.k0).astype(np.float64)
    k1 = synth.bf16_to_f32(c.k1).astype(np.float64)
    for t in range(L):
        prev = xp if t == 0 else x[t - 1]
        for ch in range(d):
            g = ch // 16
            ref = (k0[ch] + s[t] * W[g, 7]) * x[t, ch] + (k1[ch] + s[t] * W[G + g, 7]) * prev[ch]
            assert y[0, t, ch] == pytest.approx(ref, rel=1e-13, abs=1e-13)
    del rng


# ---------------------------------------------------------------------------
# verify
# ---------------------------------------------------------------------------


def _greedy_target(rng, B, L, V, argmax_tok, plant=10.0):
    tg = rng.standard_normal((B, L + 1, V)).astype(np.float32)
    for b in range(B):
        tg[b, np.arange(L + 1), argmax_tok[b]] += plant
    return f32_bits(tg)


def test_verify_greedy_reproduces_target_tokens():
    rng = np.random.default_rng(14)
    B, L, V = 5, 6, 50
    g = rng.integers(0, V, (B, L + 1))
    tg = _greedy_target(rng, B, L, V, g)
    draft = g[:, :L].copy().astype(np.int32)
    mism = [0, 2, 5, 6, 3]  # position of the first mismatch (6 = none)
    for b, n in enumerate(mism):
        if n < L:
            draft[b, n] = (g[b, n] + 1) % V
            if n + 1 < L:
                draft[b, n + 1] = (g[b, n + 1] + 2) % V  # later positions are ignored
    slot = np.zeros((B, L), np.int32)
    dq = np.ones((B, L, K), np.float32)
    ci = np.zeros((B, L, K), np.int32)
    acc, out, _ = oracle.verify(tg, draft, slot, dq, ci)
    for b, n in enumerate(mism):
        assert acc[b] == n + 1
        assert list(out[b, :n + 1]) == list(g[b, :n + 1])   # the target's own greedy tokens
        assert np.all(out[b, n + 1:] == -1)


def test_verify_greedy_tie_is_lowest_id():
    B, L, V = 1, 1, 20
    tg = np.zeros((B, L + 1, V), np.float32)
    tg[0, 0, [4, 11]] = 5.0
    tg[0, 1, [2, 17]] = 7.0
    bits = f32_bits(tg)
    acc, out, _ = oracle.verify(bits, np.array([[11]], np.int32), np.zeros((1, 1), np.int32),
                                np.ones((1, 1, K), np.float32), np.zeros((1, 1, K), np.int32))
    assert acc[0] == 1 and out[0, 0] == 4
    acc, out, _ = oracle.verify(bits, np.array([[4]], np.int32), np.zeros((1, 1), np.int32),
                                np.ones((1, 1, K), np.float32), np.zeros((1, 1, K), np.int32))
    assert acc[0] == 2 and list(out[0]) == [4, 2]


def test_acceptance_closed_form_reproduces_table1():
    # AL = 1 + sum_k prod_{i<k} r_i (the +1 is the verifier's token): Table 1's printed values.
    for row in read_golden_rows("table1_recall.txt"):
        r = [float(x) for x in row[1:8]]
        printed = float(row[8])
        al = 1.0 + sum(np.prod(r[:k]) for k in range(1, 8))
        assert math.floor(al * 100) / 100 == printed  # printed truncated to 2 decimals
        assert abs(al - printed) < 0.01


def test_verify_greedy_mean_acceptance_closed_form():
    # planted argmax agreement r per position => E[accept_len] = 1 + sum_{k=1}^{L} r^k
    B, L, V, r = 3000, 16, 64, 0.85
    rng = np.random.default_rng(15)
    draft = rng.integers(0, V, (B, L)).astype(np.int32)
    tg = synth.target_planted(16, draft, V, agree=r, plant=12.0)
    acc, _, _ = oracle.verify(tg, draft, np.zeros((B, L), np.int32), np.ones((B, L, K), np.float32),
                              np.zeros((B, L, K), np.int32))
    expect = 1.0 + sum(r**k for k in range(1, L + 1))
    assert expect == pytest.approx(6.2459, abs=1e-4)
    sd = acc.std() / math.sqrt(B)
    assert abs(acc.mean() - expect) < 4 * sd


def _softmax(z):
    z = z - z.max()
    e = np.exp(z)
    return e / e.sum()


@pytest.mark.parametrize("T", [1.0, 0.6])
def test_verify_rejection_sampling_is_lossless(T):
    # the first emitted token is distributed as softmax(target_0 / T), whatever q is
    V, L, n = 64, 2, 30000
    rng = np.random.default_rng(17)
    t0 = (rng.standard_normal(V) * 1.5).astype(np.float32)
    tg = np.zeros((n, L + 1, V), np.uint16)
    tg[:] = f32_bits(np.stack([t0, rng.standard_normal(V), rng.standard_normal(V)]).astype(np.float32))
    cand = rng.choice(V, K, replace=False).astype(np.int32)
    S = np.zeros((n, L, K, K), np.float32)
    S[:] = rng.standard_normal(K).astype(np.float32)[None, None, None, :] * 2
    ci = np.broadcast_to(cand, (n, L, K)).copy()
    tok, slot, q, _ = oracle.walk(S, ci, temperature=T, seed=5)
    acc, out, _ = oracle.verify(tg, tok, slot, q, ci, temperature=T, seed=6)
    p = _softmax(synth.bf16_to_f32(tg[0, 0]).astype(np.float64) / T)
    counts = np.bincount(out[:, 0], minlength=V)
    keep = p * n >= 5
    obs, exp = counts[keep], p[keep] * n
    if (~keep).any():
        obs, exp = np.append(obs, counts[~keep].sum()), np.append(exp, p[~keep].sum() * n)
    assert stats.chisquare(obs, exp).pvalue > 1e-4
    assert np.all((acc >= 1) & (acc <= L + 1))


def test_verify_all_accepted_draws_bonus_from_last_row():
    # q = p exactly on a 16-token support => every draft accepted (u q < p); the bonus is from p_L
    V, L, n, T = 16, 1, 20000, 1.0
    rng = np.random.default_rng(18)
    rows = np.zeros((L + 1, V), np.float32)
    rows[0] = -1e4  # not used
    rows[1] = rng.standard_normal(V)
    tg = np.broadcast_to(f32_bits(rows), (n, L + 1, V)).copy()
    z0 = np.array([0.0] * V, np.float32)
    tg[:, 0] = f32_bits(z0)  # p_0 uniform over 16 tokens
    ci = np.broadcast_to(np.arange(K, dtype=np.int32), (n, L, K)).copy()
    S = np.zeros((n, L, K, K), np.float32)  # q uniform
    tok, slot, q, _ = oracle.walk(S, ci, temperature=T, seed=9)
    acc, out, _ = oracle.verify(tg, tok, slot, q, ci, temperature=T, seed=10)
    assert np.all(acc == 2)
    p = _softmax(synth.bf16_to_f32(tg[0, 1]).astype(np.float64))
    counts = np.bincount(out[:, 1], minlength=V)
    assert stats.chisquare(counts, p * n).pvalue > 1e-4


# ---------------------------------------------------------------------------
# fused LM head (restated unfused)
# ---------------------------------------------------------------------------


def test_lmhead_topk_matches_library_matmul_and_sort():
    rng = np.random.default_rng(19)
    M, d, V = 6, 96, 700
    hid = f32_bits(rng.standard_normal((M, d)))
    W = f32_bits(rng.standard_normal((V, d)) * 0.1)
    rows = np.array([0, 3, 5], np.int64)
    vals, idx = oracle.lmhead_topk(hid, W, rows)
    logits = synth.bf16_to_f32(hid).astype(np.float64) @ synth.bf16_to_f32(W).astype(np.float64).T
    for i, m in enumerate(rows):
        order = np.lexsort((np.arange(V), -logits[m]))[:K]
        assert list(idx[i]) == list(order)
        assert np.allclose(vals[i], logits[m, order], rtol=1e-12, atol=1e-12)


def test_verify_philox_streams_are_pinned():
    # p_0 uniform over V = 16 (all-zero logits: exp(0) = 1, Z = 16, exact) and q one-hot
    # at the drafted token x: accept iff u1 < 1/16 with u1 = uniform24(seed, b, 0, stream 1);
    # a rejection draws the floor(15 u2)-th token != x with u2 = uniform24(seed, b, 0, stream 2);
    # an acceptance (L = 1) draws the bonus floor(16 u3) from the uniform row 1, u3 = stream 2 at t = 1.
    V, L, n, seed, off = 16, 1, 400, 21, 5
    tg = np.zeros((n, L + 1, V), np.uint16)
    rng = np.random.default_rng(22)
    x = rng.integers(0, V, (n, 1)).astype(np.int32)
    ci = np.broadcast_to(np.arange(K, dtype=np.int32), (n, L, K)).copy()
    slot = x.copy()
    q = np.zeros((n, L, K), np.float32)
    q[np.arange(n), 0, x[:, 0]] = 1.0
    acc, out, _ = oracle.verify(tg, x, slot, q, ci, temperature=1.0, seed=seed, offset=off)
    n_acc = 0
    for b in range(n):
        u1 = oracle.uniform24(seed, b, 0, 1, off)
        if u1 < 1.0 / 16:
            n_acc += 1
            assert acc[b] == 2 and out[b, 0] == x[b, 0]
            assert out[b, 1] == int(16 * oracle.uniform24(seed, b, 1, 2, off))
        else:
            others = [v for v in range(V) if v != x[b, 0]]
            assert acc[b] == 1
            assert out[b, 0] == others[int(15 * oracle.uniform24(seed, b, 0, 2, off))]
    assert 5 < n_acc < 60


# ---------------------------------------------------------------------------
# the walk's fp32 2^x
# ---------------------------------------------------------------------------


def test_exp2_neg_exact_points():
    assert oracle.exp2_neg(0.0) == 1.0
    assert oracle.exp2_neg(-1.0) == 0.5
    assert oracle.exp2_neg(-126.0) == 2.0**-126
    assert oracle.exp2_neg(-127.0) == 0.0
    assert oracle.exp2_neg(float("-inf")) == 0.0
    assert oracle.exp2_neg(float("nan")) == 0.0
    for n in range(0, 126):
        assert oracle.exp2_neg(-float(n)) == 2.0 ** -n


def test_exp2_neg_within_one_ulp_of_exact():
    # against the exact value (math.exp2 in double), over [-126, 0] including
    # the rint half-way points; one fp32 ulp relative = 2^-23
    xs = np.concatenate([np.linspace(-126.0, 0.0, 200001, dtype=np.float32),
                         np.arange(-125.5, 0.0, 1.0, dtype=np.float32),
                         -np.logspace(-8, 0, 2001).astype(np.float32)])
    for x in xs:
        got = oracle.exp2_neg(float(x))
        ref = math.exp2(float(x))
        assert abs(got - ref) <= 2.0**-23 * ref, (float(x), got, ref)


# ---------------------------------------------------------------------------
# reading R21: the sampled verification's fixed-point weights, and the fp32
# walk, against plain fp64 restatements of the definitions
# ---------------------------------------------------------------------------


def test_verify_weights_are_floor_of_scaled_exp2():
    rng = np.random.default_rng(40)
    for T in (1.0, 0.6, 2.5):
        row = f32_bits(rng.standard_normal(3000) * 3)
        W, Z = oracle.verify_weights(row, T)
        lf = synth.bf16_to_f32(row).astype(np.float64)
        c = float(np.float32(1.44269504) / np.float32(T))
        x = (lf - lf.max()) * c
        exact = np.exp2(x) * 2.0**40
        # the row's largest logit weighs exactly 2^40; every weight is floor(w 2^40)
        # for an fp32 w within one fp32 ulp of 2^x, x = (l - M) c carrying one
        # fp32 rounding (relative 2^-24, so 2^x moves by ln 2 |x| 2^-24 relative)
        assert int(W[np.argmax(lf)]) == 2**40
        err = np.abs(W.astype(np.float64) - exact)
        assert np.all(err <= exact * (np.abs(x) * 2.0**-24 + 2.0**-23) + 1.0)
        assert Z == int(np.sum(W.astype(object)))   # exact integer sum, any order


def test_verify_weights_nan_and_degenerate_rows():
    row = f32_bits(np.array([1.0, np.nan, 3.0, -np.inf, 3.0], np.float32))
    W, Z = oracle.verify_weights(row, 1.0)
    assert W[1] == 0 and W[3] == 0 and W[2] == 2**40 and W[4] == 2**40 and Z == int(W.sum())
    for bad in (np.full(8, np.nan, np.float32), np.full(8, -np.inf, np.float32)):
        W, Z = oracle.verify_weights(f32_bits(bad), 1.0)
        assert Z == 0


def test_verify_no_finite_logit_emits_the_argmax():
    # Z = 0: the accept test fails (0 < 0 is false) and the token is the row's
    # arg-max in top-k order (all NaN or all -inf: id 0; one +inf: that id)
    V, L = 32, 1
    rows = np.zeros((3, L + 1, V), np.float32)
    rows[0, 0] = np.nan
    rows[1, 0] = -np.inf
    rows[2, 0] = -np.inf
    rows[2, 0, 7] = np.inf
    tg = f32_bits(rows)
    ci = np.broadcast_to(np.arange(K, dtype=np.int32), (3, L, K)).copy()
    q = np.full((3, L, K), 1.0 / K, np.float32)
    acc, out, _ = oracle.verify(tg, np.ones((3, L), np.int32), np.ones((3, L), np.int32), q, ci,
                                temperature=1.0, seed=2)
    assert list(acc) == [1, 1, 1] and list(out[:, 0]) == [0, 0, 7]


def _fp64_verify(tg_bits, tok, slot, q, ci, T, seed, offset):
    """The plain definition in fp64 (softmax by np.exp, residual max(0, p - q),
    inverse CDF in id order) with each decision's margin."""
    B, L1, V = tg_bits.shape
    L = L1 - 1
    acc = np.zeros(B, np.int32)
    out = np.full((B, L1), -1, np.int32)
    margin = np.full(B, np.inf)

    def p_of(b, t):
        z = synth.bf16_to_f32(tg_bits[b, t]).astype(np.float64) / T
        e = np.exp(z - z.max())
        return e / e.sum()

    def draw(w, u, b):
        cdf = np.cumsum(w)
        tgt = u * cdf[-1]
        v = int(np.searchsorted(cdf, tgt, side="right"))
        lo = cdf[v - 1] if v > 0 else 0.0
        margin[b] = min(margin[b], min(cdf[v] - tgt, tgt - lo) / cdf[-1])
        return v

    for b in range(B):
        n = L
        for t in range(L):
            p = p_of(b, t)
            qx = float(q[b, t, slot[b, t]])
            u1 = oracle.uniform24(seed, b, t, 1, offset)
            margin[b] = min(margin[b], abs(u1 * qx - p[tok[b, t]]) / p[tok[b, t]])
            if u1 * qx < p[tok[b, t]]:
                continue
            r = p.copy()
            for j in range(K):
                r[ci[b, t, j]] = max(0.0, p[ci[b, t, j]] - float(q[b, t, j]))
            n = t
            out[b, t] = draw(r, oracle.uniform24(seed, b, t, 2, offset), b)
            break
        if n == L:
            out[b, L] = draw(p_of(b, L), oracle.uniform24(seed, b, L, 2, offset), b)
        out[b, :n] = tok[b, :n]
        acc[b] = n + 1
    return acc, out, margin


@pytest.mark.parametrize("T", [1.0, 0.6])
def test_verify_fixed_point_agrees_with_fp64_definition(T):
    # R21's integer decisions equal the fp64 definition's wherever the latter is
    # not within 1e-9 (relative) of a boundary: the fixed point changes no
    # decision that floating point can resolve
    rng = np.random.default_rng(41)
    B, L, V = 300, 4, 600
    S = (rng.standard_normal((B, L, K, K)) * 2).astype(np.float32)
    ci = np.stack([np.stack([rng.choice(V, K, replace=False) for _ in range(L)]) for _ in range(B)]).astype(np.int32)
    tok, slot, q, _ = oracle.walk(S, ci, temperature=T, seed=3)
    tg = synth.target_planted(42, tok, V, agree=0.7, plant=3.0)
    acc, out, _ = oracle.verify(tg, tok, slot, q, ci, temperature=T, seed=4, offset=1)
    facc, fout, fmargin = _fp64_verify(tg, tok, slot, q, ci, T, 4, 1)
    ok = fmargin > 1e-9
    assert ok.sum() >= B - 2
    assert np.array_equal(acc[ok], facc[ok]) and np.array_equal(out[ok], fout[ok])
    assert 1.0 < acc.mean() < L + 1


def test_walk_fp32_agrees_with_fp64_definition():
    # R5's fp32 draw against w = exp((S - max) / T) in fp64: equal except where
    # u Z lies within 1e-6 Z of a CDF boundary
    rng = np.random.default_rng(43)
    B, L = 400, 8
    for T in (1.0, 0.5, 2.0):
        S = (rng.standard_normal((B, L, K, K)) * 2).astype(np.float32)
        ci = rng.integers(0, 1000, (B, L, K)).astype(np.int32)
        _, slot, _, _ = oracle.walk(S, ci, temperature=T, seed=7, offset=2)
        checked = 0
        for b in range(B):
            prev = 0
            for t in range(L):
                s = S[b, t, prev].astype(np.float64)
                w = np.exp((s - s.max()) / T)
                cdf = np.cumsum(w)
                tgt = oracle.uniform24(7, b, t, 0, 2) * cdf[-1]
                if np.min(np.abs(cdf - tgt)) < 1e-6 * cdf[-1]:
                    break   # later steps follow a predecessor that may legitimately differ
                assert slot[b, t] == int(np.searchsorted(cdf, tgt, side="right")), (T, b, t)
                checked += 1
                prev = slot[b, t]
        assert checked >= 0.99 * B * L


def test_walk_nan_scores_never_win():
    # greedy: the lowest slot of the largest non-NaN score (numpy's nanargmax);
    # all NaN: slot 0.  Sampled: a NaN slot has q = 0; a row without a positive
    # weight (all NaN or -inf) takes the greedy slot with q one-hot.
    rng = np.random.default_rng(44)
    B, L = 64, 6
    S = rng.standard_normal((B, L, K, K)).astype(np.float32)
    S[rng.random(S.shape) < 0.3] = np.nan
    S[0, 0, 0, :] = np.nan
    S[1, 0, 0, :] = -np.inf
    S[2, 0, 0, 0] = np.nan
    ci = rng.integers(0, 1000, (B, L, K)).astype(np.int32)
    _, slot, q, _ = oracle.walk(S, ci)
    for b in range(B):
        prev = 0
        for t in range(L):
            row = S[b, t, prev]
            expect = 0 if np.all(np.isnan(row)) else int(np.nanargmax(row))
            assert slot[b, t] == expect
            prev = expect
    _, slot1, q1, _ = oracle.walk(S, ci, temperature=1.0, seed=3)
    assert slot1[0, 0] == 0 and q1[0, 0, 0] == 1.0 and q1[0, 0].sum() == 1.0
    assert slot1[1, 0] == 0 and q1[1, 0, 0] == 1.0
    for b in range(B):
        prev = 0
        for t in range(L):
            row = S[b, t, prev]
            if not np.all(np.isnan(row) | np.isneginf(row)):
                assert np.all(q1[b, t][np.isnan(row)] == 0.0)
                assert not np.isnan(row[slot1[b, t]])
            prev = slot1[b, t]
