"""The exact best-path walk and the Table 1 selector evaluation on the GPU vs
the oracle: slots, tokens, scores and counts bit-exact (the path is an integer
decided by fp32 sums formed in the same order on both sides)."""
import numpy as np
import pytest
import torch

import oracle
from draft_selection_dflash2_gb300 import api, synth
from gpu_common import f32, handle, host, i32  # noqa: F401

pytestmark = pytest.mark.gpu
K = 16


@pytest.mark.parametrize("B,L", [(1, 1), (3, 2), (5, 3), (128, 16), (257, 7), (9, 64), (64, 16)])
def test_viterbi_matches_oracle(handle, B, L):
    rng = np.random.default_rng(B * 131 + L)
    S = (rng.standard_normal((B, L, K, K)) * 2).astype(np.float32)
    ci = rng.integers(0, 151936, (B, L, K)).astype(np.int32)
    tok, slot, score = api.walk_viterbi(handle, f32(S), i32(ci))
    otok, oslot, oscore = oracle.walk_viterbi(S, ci)
    assert np.array_equal(host(slot), oslot)
    assert np.array_equal(host(tok), otok)
    assert np.array_equal(host(score).view(np.uint32), oscore.view(np.uint32))


def test_viterbi_ties_and_nan(handle):
    B, L = 4, 6
    S = np.zeros((B, L, K, K), np.float32)        # sequence 0: every path ties
    rng = np.random.default_rng(5)
    S[1:] = rng.integers(-2, 3, (B - 1, L, K, K)).astype(np.float32)   # many integer ties
    S[3, 2, 4, :] = np.nan                       # NaN never wins a comparison
    S[3, 0, 0, 7] = np.nan
    ci = rng.integers(0, 1000, (B, L, K)).astype(np.int32)
    tok, slot, score = api.walk_viterbi(handle, f32(S), i32(ci))
    otok, oslot, oscore = oracle.walk_viterbi(S, ci)
    assert np.array_equal(host(slot), oslot) and np.array_equal(host(tok), otok)
    assert list(host(slot)[0]) == [0] * L
    g, o = host(score), oscore
    assert np.array_equal(np.isnan(g), np.isnan(o)) and np.array_equal(g[~np.isnan(g)], o[~np.isnan(o)])


def test_viterbi_on_the_pipeline_scores_beats_greedy(handle):
    # on pair scores of the full-cycle shapes, the best path scores at least the greedy one
    B, L = 32, 16
    rng = np.random.default_rng(2)
    S = (rng.standard_normal((B, L, K, K)) * 3).astype(np.float32)
    ci = rng.integers(0, 151936, (B, L, K)).astype(np.int32)
    _, vslot, vscore = api.walk_viterbi(handle, f32(S), i32(ci))
    _, gslot, _ = api.walk(handle, f32(S), i32(ci), temperature=0.0)
    gs, vs = host(gslot), host(vscore)
    for b in range(B):
        g = np.float32(S[b, 0, 0, gs[b, 0]])
        for t in range(1, L):
            g = np.float32(g + S[b, t, gs[b, t - 1], gs[b, t]])
        assert vs[b] >= g


def planted_eval_inputs(seed, B, L, r1, r16):
    rng = np.random.default_rng(seed)
    gt = rng.integers(0, 1 << 20, (B, L)).astype(np.int32)
    ci = rng.integers(1 << 21, 1 << 22, (B, L, K)).astype(np.int32)
    u = rng.random((B, L))
    top = u < r1
    inside = (~top) & (u < r16)
    slot = rng.integers(1, K, (B, L))
    bb, tt = np.nonzero(top)
    ci[bb, tt, 0] = gt[bb, tt]
    bb, tt = np.nonzero(inside)
    ci[bb, tt, slot[bb, tt]] = gt[bb, tt]
    return gt, ci


@pytest.mark.parametrize("B,L", [(1, 1), (7, 3), (5000, 7), (1000, 16), (300, 64)])
def test_selector_eval_matches_oracle(handle, B, L):
    r1 = np.linspace(0.85, 0.7, L)
    r16 = np.linspace(0.995, 0.85, L)
    gt, ci = planted_eval_inputs(B + L, B, L, r1, r16)
    a1, a16, counts = api.selector_eval(handle, i32(gt), i32(ci))
    o1, o16, ocounts = oracle.selector_eval(gt, ci)
    assert np.array_equal(host(a1), o1) and np.array_equal(host(a16), o16)
    assert np.array_equal(host(counts), ocounts)


def test_selector_eval_empty_batch_zeroes_counts(handle):
    L = 5
    counts = torch.full((L, 4), 77, dtype=torch.int64, device="cuda")
    gt = torch.empty((0, L), dtype=torch.int32, device="cuda")
    ci = torch.empty((0, L, K), dtype=torch.int32, device="cuda")
    api.selector_eval(handle, gt, ci, counts=counts)
    assert (host(counts) == 0).all()


def test_selector_eval_on_gpu_top16_candidates(handle):
    # the candidates of the GPU top-16 and of the oracle top-16 (computed separately)
    # give the same evaluation; the true token is planted at a varying rank
    B, L, V = 64, 8, 4096
    rng = np.random.default_rng(9)
    U = synth.logits_planted(rng, B * L, V)
    vals, idx = api.topk(handle, torch.from_numpy(U.view(np.int16)).cuda().view(torch.bfloat16))
    _, oidx = oracle.topk(U)
    gt = oidx.reshape(B, L, K)[:, :, 0].copy()
    swap = rng.random((B, L)) < 0.3           # some true tokens sit at rank 2..20 instead
    alt = np.argsort(-synth.bf16_to_f32(U), axis=1, kind="stable")[:, 2:21]
    pick = alt[np.arange(B * L), rng.integers(0, 19, B * L)].reshape(B, L)
    gt = np.where(swap, pick, gt).astype(np.int32)
    a1, a16, counts = api.selector_eval(handle, i32(gt), idx.view(B, L, K))
    o1, o16, ocounts = oracle.selector_eval(gt, oidx.reshape(B, L, K))
    assert np.array_equal(host(a1), o1) and np.array_equal(host(a16), o16)
    assert np.array_equal(host(counts), ocounts)


def test_selector_eval_unaligned_candidates(handle):
    # candidate ids starting 4 bytes past a 16-byte boundary take the scalar-load path
    B, L = 777, 9
    r1 = np.full(L, 0.8)
    r16 = np.full(L, 0.95)
    gt, ci = planted_eval_inputs(4, B, L, r1, r16)
    flat = torch.empty(B * L * K + 1, dtype=torch.int32, device="cuda")
    flat[1:].copy_(torch.from_numpy(ci.reshape(-1)))
    cand = flat[1:].view(B, L, K)
    assert cand.data_ptr() % 16 == 4
    a1, a16, counts = api.selector_eval(handle, i32(gt), cand)
    o1, o16, ocounts = oracle.selector_eval(gt, ci)
    assert np.array_equal(host(a1), o1) and np.array_equal(host(a16), o16)
    assert np.array_equal(host(counts), ocounts)


def test_best_path_vs_greedy_acceptance_on_planted_data(handle):
    # both walks and the T=0 verify on the GPU give the oracle's acceptance lengths,
    # and the best path accepts more than greedy on planted pair scores
    B, L, V = 256, 16, 800
    S, ci, _, true_tok = synth.planted_path(2, B, L, V, mu=3.0)
    target = synth.target_planted(3, true_tok, V, agree=1.0)
    dS, dci = f32(S), i32(ci)
    dtg = torch.from_numpy(target.view(np.int16)).cuda().view(torch.bfloat16)
    gtok, gslot, gq = api.walk(handle, dS, dci, temperature=0.0)
    vtok, vslot, _ = api.walk_viterbi(handle, dS, dci)
    ag, _ = api.verify(handle, dtg, gtok, gslot, gq, dci, temperature=0.0)
    av, _ = api.verify(handle, dtg, vtok, vslot, gq, dci, temperature=0.0)
    otok, oslot, oq, _ = oracle.walk(S, ci, temperature=0.0)
    vt, vs, _ = oracle.walk_viterbi(S, ci)
    oag, _, _ = oracle.verify(target, otok, oslot, oq, ci, temperature=0.0)
    oav, _, _ = oracle.verify(target, vt, vs, oq, ci, temperature=0.0)
    assert np.array_equal(host(ag), oag) and np.array_equal(host(av), oav)
    assert host(av).mean() > host(ag).mean() + 0.5
