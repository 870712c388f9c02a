"""Verification kernels vs the oracle.

T = 0: acceptance lengths and emitted tokens bit-exact.
T > 0: bit-exact as well.  Both sides take the target distribution in exact
fixed point (each weight floor(exp2_neg((l - M) c) 2^40), summed as integers,
which no parallel order changes), so every accept test and every draw is the
same integer decision on both sides, for every sequence.  Losslessness is
checked statistically on V = 64."""
import numpy as np
import pytest
import torch
from scipy import stats

import oracle
from draft_selection_dflash2_gb300 import api, synth
from gpu_common import bf, f32, handle, host, i32  # noqa: F401

pytestmark = pytest.mark.gpu
K = 16


def draft(seed, B, L, V, T):
    rng = np.random.default_rng(seed)
    ci = np.stack([np.stack([rng.choice(V, K, replace=V < K) for _ in range(L)]) for _ in range(B)])
    ci = ci.astype(np.int32)
    S = (rng.standard_normal((B, L, K, K)) * 2).astype(np.float32)
    tok, slot, q, _ = oracle.walk(S, ci, temperature=float(np.float32(T)), seed=seed)
    return tok, slot, q, ci


def padded(target, V):
    """Target logits with the leading dimension rounded up to a multiple of 8;
    the padding holds large values that must never be read."""
    ld = (V + 7) // 8 * 8
    if ld == V:
        return target
    out = np.full(target.shape[:2] + (ld,), synth.bf16_bits(np.float32(1e4)), np.uint16)
    out[..., :V] = target
    return out


@pytest.mark.parametrize("B,L,V", [(1, 8, 4096), (16, 16, 151936), (128, 16, 8200), (5, 1, 4099),
                                   (9, 64, 1000), (3, 5, 17), (2, 3, 9)])
def test_greedy_verify_exact(handle, B, L, V):
    tok, slot, q, ci = draft(B + L, B, L, V, 0.0)
    target = padded(synth.target_planted(B * 3 + L, tok, V, agree=0.85), V)
    acc, out = api.verify(handle, bf(target), i32(tok), V=V)
    oacc, oout, _ = oracle.verify(target, tok, slot, q, ci, V=V)
    assert np.array_equal(host(acc), oacc) and np.array_equal(host(out), oout)


@pytest.mark.parametrize("T", [1.0, 0.7])
@pytest.mark.parametrize("B,L,V,plant", [(64, 16, 8200, 12.0), (16, 16, 151936, 16.0), (40, 4, 4099, 6.0),
                                         (6, 5, 17, 2.0), (3, 2, 1 << 20, 8.0)])
def test_sampled_verify_matches_oracle(handle, B, L, V, plant, T):
    tok, slot, q, ci = draft(B * 7 + L, B, L, V, T)
    target = padded(synth.target_planted(B + 1, tok, V, agree=0.85, plant=plant), V)
    Tf = float(np.float32(T))
    acc, out = api.verify(handle, bf(target), i32(tok), i32(slot), f32(q), i32(ci), temperature=T,
                          seed=11, offset=2, V=V)
    oacc, oout, _ = oracle.verify(target, tok, slot, q, ci, temperature=Tf, seed=11, offset=2, V=V)
    assert np.array_equal(host(acc), oacc) and np.array_equal(host(out), oout)
    assert handle.device_error() == 0


@pytest.mark.parametrize("T", [0.05, 3.0])
def test_sampled_verify_extreme_temperatures(handle, T):
    # T = 0.05: nearly every weight floors to 0 and the draws sit on a few ids;
    # T = 3: weights are flat and the sums long
    B, L, V = 24, 8, 30011
    tok, slot, q, ci = draft(5, B, L, V, T)
    target = padded(synth.target_planted(6, tok, V, agree=0.8, plant=1.0), V)
    Tf = float(np.float32(T))
    for seed in (1, 2):
        acc, out = api.verify(handle, bf(target), i32(tok), i32(slot), f32(q), i32(ci), temperature=T, seed=seed, V=V)
        oacc, oout, _ = oracle.verify(target, tok, slot, q, ci, temperature=Tf, seed=seed, V=V)
        assert np.array_equal(host(acc), oacc) and np.array_equal(host(out), oout)


def test_sampled_verify_degenerate_rows(handle):
    """Rows with no finite logit (all NaN, all -inf: the token is the arg-max,
    id 0; one +inf among -inf: that id), NaN scattered through a row, a
    candidate id repeated within a position, a NaN proposal weight: each side
    follows the same rules, so the outputs agree exactly."""
    B, L, V = 8, 4, 5000
    tok, slot, q, ci = draft(21, B, L, V, 1.0)
    target = synth.target_planted(22, tok, V, agree=0.85, plant=10.0)
    f = lambda x: int(synth.bf16_bits(np.float32([x]))[0])   # noqa: E731
    target[0, 0, :] = 0x7FC0                              # all NaN
    target[1, 0, :] = f(-np.inf)                          # all -inf
    target[2, 0, :] = f(-np.inf)
    target[2, 0, 123] = f(np.inf)                         # one +inf
    rng = np.random.default_rng(23)
    target[3][rng.random(target[3].shape) < 0.2] = 0x7FC0  # NaN scattered
    ci[4, 0, 5] = ci[4, 0, 2]                             # a repeated candidate id
    ci[4, 1, :] = ci[4, 1, 0]                             # one id in every slot
    q[5, 0, 3] = np.nan                                   # a NaN proposal weight
    tok[6, 0] = ci[6, 0, 0]
    target[6, 0, ci[6, 0, 0]] = f(-3.0)                   # forced rejection of the top candidate
    acc, out = api.verify(handle, bf(target), i32(tok), i32(slot), f32(q), i32(ci), temperature=1.0, seed=4, V=V)
    oacc, oout, _ = oracle.verify(target, tok, slot, q, ci, temperature=1.0, seed=4, V=V)
    assert list(oout[:3, 0]) == [0, 0, 123]
    assert np.array_equal(host(acc), oacc) and np.array_equal(host(out), oout)
    assert handle.device_error() == 0


def test_sampled_verify_out_of_range_draft_is_rejected_and_flagged(handle):
    B, L, V = 4, 3, 3000
    tok, slot, q, ci = draft(25, B, L, V, 1.0)
    target = synth.target_planted(26, tok, V, agree=1.0, plant=20.0)
    tok[1, 0] = V + 5          # weighs 0: always rejected
    slot[2, 1] = 40            # clamped to slot 15
    acc, out = api.verify(handle, bf(target), i32(tok), i32(slot), f32(q), i32(ci), temperature=1.0, seed=2, V=V)
    oacc, oout, _ = oracle.verify(target, tok, slot, q, ci, temperature=1.0, seed=2, V=V)
    assert oacc[1] == 1
    assert np.array_equal(host(acc), oacc) and np.array_equal(host(out), oout)
    bits = handle.device_error()
    assert bits & api.DEVERR_BAD_TOKEN and bits & api.DEVERR_BAD_SLOT


def test_verify_full_size_both_temperatures(handle):
    # the benchmark's shape and launch configuration: B=128, L=16, V=151936
    # (661 MB of target logits), where the grid's warps equal sequences x chunks;
    # every sequence is compared at both temperatures
    B, L, V = 128, 16, 151936
    tok, slot, q, ci = draft(12, B, L, V, 1.0)
    target = synth.target_planted(13, tok, V, agree=0.85, plant=8.0)
    tg = bf(target)
    acc, out = api.verify(handle, tg, i32(tok), V=V)
    oacc, oout, _ = oracle.verify(target, tok, slot, q, ci, V=V)
    assert np.array_equal(host(acc), oacc) and np.array_equal(host(out), oout)
    assert oacc.mean() > 4.0   # most sequences reach deep positions: the tail of the pass is covered
    # sampled: a plant of 8 on N(0,1) logits is ~1% of the mass at T=1 (rejections,
    # residual draws); a plant of 14 is ~80% (long accepted prefixes, bonus draws)
    for plant in (8.0, 14.0):
        if plant != 8.0:
            target = synth.target_planted(14, tok, V, agree=0.85, plant=plant)
            tg = bf(target)
        for seed, offset, T in ((5, 1, 1.0), (6, 0, 0.7)):
            acc, out = api.verify(handle, tg, i32(tok), i32(slot), f32(q), i32(ci), temperature=T, seed=seed,
                                  offset=offset, V=V)
            oacc, oout, _ = oracle.verify(target, tok, slot, q, ci, temperature=float(np.float32(T)), seed=seed,
                                          offset=offset, V=V)
            assert np.array_equal(host(acc), oacc) and np.array_equal(host(out), oout)
        if plant == 14.0:
            assert oacc.mean() > 2.0
    assert handle.device_error() == 0


def test_sampled_verify_is_lossless_on_gpu(handle):
    V, L, n, T = 64, 2, 20000, 1.0
    rng = np.random.default_rng(31)
    t0 = (rng.standard_normal(V) * 1.5).astype(np.float32)
    rows = np.stack([t0, rng.standard_normal(V), rng.standard_normal(V)]).astype(np.float32)
    target = np.broadcast_to(synth.bf16_bits(rows), (n, L + 1, V)).copy()
    cand = rng.choice(V, K, replace=False).astype(np.int32)
    ci = np.broadcast_to(cand, (n, L, K)).copy()
    S = np.zeros((n, L, K, K), np.float32)
    S[:] = (rng.standard_normal(K) * 2).astype(np.float32)
    tok, slot, q = api.walk(handle, f32(S), i32(ci), temperature=T, seed=5)
    acc, out = api.verify(handle, bf(target), tok, slot, q, i32(ci), temperature=T, seed=6)
    first = host(out)[:, 0]
    p = np.exp(synth.bf16_to_f32(target[0, 0]).astype(np.float64) / T)
    p /= p.sum()
    counts = np.bincount(first, minlength=V)
    keep = p * n >= 5
    obs, exp = counts[keep], p[keep] * n
    if (~keep).any():
        obs, exp = np.append(obs, counts[~keep].sum()), np.append(exp, p[~keep].sum() * n)
    assert stats.chisquare(obs, exp).pvalue > 1e-4


def test_greedy_verify_nan_and_ties(handle):
    """Arg-max order of the pages' greedy rule as the oracle reads it: NaN ranks
    below -inf (an all-NaN row's arg-max is id 0), -0 equals +0, and equal
    values go to the lowest id, wherever in the row (and in which chunk) they lie."""
    B, L, V = 6, 4, 9000
    tok, slot, q, ci = draft(7, B, L, V, 0.0)
    target = synth.target_planted(8, tok, V, agree=0.85)
    rng = np.random.default_rng(9)
    f = lambda x: int(synth.bf16_bits(np.float32([x]))[0])   # noqa: E731
    target[rng.random(target.shape) < 0.05] = 0x7FC0  # NaN scattered everywhere
    target[0, 1, :] = 0x7FC0                          # all NaN: arg-max 0
    target[1, 0, :] = f(-1.0)
    target[1, 0, 8000] = 0x8000                       # -0 at a later id ...
    target[1, 0, 50] = f(0.0)                         # ... equals +0 at id 50
    target[2, 0, :] = f(-2.0)
    target[2, 0, [100, 8000]] = f(3.0)                # a tie in two chunks: id 100
    tok[2, 0] = 8000
    target[3, :, tok[3]] = 0x7FC0                     # the draft's own logit is NaN
    acc, out = api.verify(handle, bf(target), i32(tok), V=V)
    oacc, oout, _ = oracle.verify(target, tok, slot, q, ci, V=V)
    assert oout[0, 1] == 0 and oout[1, 0] == 50 and oout[2, 0] == 100
    assert np.array_equal(host(acc), oacc) and np.array_equal(host(out), oout)


@pytest.mark.parametrize("T", [0.0, 1.0])
def test_verify_empty_block(handle, T):
    # L = 0: no draft, only the bonus row; the draft tensors are empty (null pointers)
    B, L, V, K = 5, 0, 4099, 16
    rng = np.random.default_rng(17)
    target = padded(synth.bf16_bits(rng.standard_normal((B, L + 1, V)).astype(np.float32)), V)
    tok, slot = np.zeros((B, L), np.int32), np.zeros((B, L), np.int32)
    q, ci = np.zeros((B, L, K), np.float32), np.zeros((B, L, K), np.int32)
    acc, out = api.verify(handle, bf(target), i32(tok), i32(slot), f32(q), i32(ci), temperature=T, seed=3, V=V)
    oacc, oout, _ = oracle.verify(target, tok, slot, q, ci, temperature=T, seed=3, V=V)
    assert np.array_equal(host(acc), oacc) and np.array_equal(host(out), oout)
    assert handle.device_error() == 0


def test_greedy_mean_acceptance_closed_form_on_gpu(handle):
    B, L, V, r = 4096, 16, 512, 0.85
    rng = np.random.default_rng(8)
    tok = rng.integers(0, V, (B, L)).astype(np.int32)
    target = synth.target_planted(9, tok, V, agree=r, plant=12.0)
    acc, _ = api.verify(handle, bf(target), i32(tok))
    a = host(acc)
    expect = 1.0 + sum(r**k for k in range(1, L + 1))
    assert abs(a.mean() - expect) < 4 * a.std() / np.sqrt(B)


def test_verify_workspace_is_the_callers(handle):
    """The call's scratch is the caller's workspace: a short or missing one is
    refused (DFLASH2_ERR_WORKSPACE) before anything launches, a misaligned one
    too (DFLASH2_ERR_MISALIGNED), and one workspace serves calls of any size up
    to the one it was sized for, inside a CUDA graph capture as well."""
    B, L, V = 6, 5, 3001
    tok, slot, q, ci = draft(3, B, L, V, 1.0)
    target = padded(synth.target_planted(4, tok, V, agree=0.85), V)
    need = api.verify_workspace(handle, B, L, V)
    assert need > 0
    tg, tk, sl, qq, cc = bf(target), i32(tok), i32(slot), f32(q), i32(ci)
    short = torch.empty(need - 8, dtype=torch.uint8, device="cuda")
    with pytest.raises(api.Dflash2Error) as e:
        api.verify(handle, tg, tk, sl, qq, cc, temperature=1.0, V=V, workspace=short)
    assert e.value.status == -7
    big = torch.empty(need + 512, dtype=torch.uint8, device="cuda")
    with pytest.raises(api.Dflash2Error) as e:
        api.verify(handle, tg, tk, sl, qq, cc, temperature=1.0, V=V, workspace=big[8:])
    assert e.value.status == -3
    ws = big[:need]
    stream = torch.cuda.Stream()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.stream(stream):
        api.verify(handle, tg, tk, sl, qq, cc, temperature=1.0, seed=9, V=V, workspace=ws)
        torch.cuda.synchronize()
        with torch.cuda.graph(graph, stream=stream):
            acc0, out0 = api.verify(handle, tg, tk, V=V, workspace=ws)
            acc1, out1 = api.verify(handle, tg, tk, sl, qq, cc, temperature=1.0, seed=9, V=V, workspace=ws)
        graph.replay()
    torch.cuda.synchronize()
    oacc0, oout0, _ = oracle.verify(target, tok, slot, q, ci, V=V)
    oacc1, oout1, _ = oracle.verify(target, tok, slot, q, ci, temperature=1.0, seed=9, V=V)
    assert np.array_equal(host(acc0), oacc0) and np.array_equal(host(out0), oout0)
    assert np.array_equal(host(acc1), oacc1) and np.array_equal(host(out1), oout1)
    # a smaller problem in the same workspace
    acc, out = api.verify(handle, tg[:2, :3].contiguous(), tk[:2, :2].contiguous(), V=V, workspace=ws)
    oacc, oout, _ = oracle.verify(target[:2, :3], tok[:2, :2], slot[:2, :2], q[:2, :2], ci[:2, :2], V=V)
    assert np.array_equal(host(acc), oacc) and np.array_equal(host(out), oout)
