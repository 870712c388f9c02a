"""Verification kernels vs the oracle.

T = 0: acceptance lengths and emitted tokens bit-exact.
T > 0: exact except sequences whose oracle decision margin is below 1e-4
(relative), where fp32 exponentials may legitimately flip a draw; those are
counted and must be rare.  Losslessness is checked statistically on V = 64."""
import numpy as np
import pytest
import torch
from scipy import stats

import oracle
from draft_selection_dflash2_gb300 import api, synth
from gpu_common import bf, f32, handle, host, i32  # noqa: F401

pytestmark = pytest.mark.gpu
K = 16


# The GPU forms p(x) and the residual CDF from fp32 exponentials summed in
# fp64 (relative error ~1e-6); decisions closer than that to their boundary may
# legitimately flip and are excused (counted).
ACCEPT_MARGIN = 1e-5     # |u q - p(x)| / p(x)
DRAW_MARGIN = 2e-6       # distance to the drawn token's CDF interval / total mass


def excused(margin):
    return (margin[:, 0] < ACCEPT_MARGIN) | (margin[:, 1] < DRAW_MARGIN)


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
                                         (6, 5, 17, 2.0)])
def test_sampled_verify_matches_oracle(handle, B, L, V, plant, T):
    tok, slot, q, ci = draft(B * 7 + L, B, L, V, T)
    target = padded(synth.target_planted(B + 1, tok, V, agree=0.85, plant=plant), V)
    Tf = float(np.float32(T))
    acc, out = api.verify(handle, bf(target), i32(tok), i32(slot), f32(q), i32(ci), temperature=T,
                          seed=11, offset=2, V=V)
    oacc, oout, margin = oracle.verify(target, tok, slot, q, ci, temperature=Tf, seed=11, offset=2, V=V)
    gacc, gout = host(acc), host(out)
    near = excused(margin)
    assert near.sum() <= max(2, B // 10)
    ok = ~near
    assert np.array_equal(gacc[ok], oacc[ok]) and np.array_equal(gout[ok], oout[ok])
    assert handle.device_error() == 0


def test_verify_full_size_both_temperatures(handle):
    # the benchmark's shape and launch configuration: B=128, L=16, V=151936
    # (661 MB of target logits), where the grid's warps equal sequences x chunks
    B, L, V = 128, 16, 151936
    tok, slot, q, ci = draft(12, B, L, V, 1.0)
    target = synth.target_planted(13, tok, V, agree=0.85, plant=8.0)
    tg = bf(target)
    acc, out = api.verify(handle, tg, i32(tok), V=V)
    oacc, oout, _ = oracle.verify(target, tok, slot, q, ci, V=V)
    assert np.array_equal(host(acc), oacc) and np.array_equal(host(out), oout)
    assert oacc.mean() > 4.0   # most sequences reach deep positions: the tail of the pass is covered
    acc, out = api.verify(handle, tg, i32(tok), i32(slot), f32(q), i32(ci), temperature=1.0, seed=5, offset=1,
                          V=V)
    oacc, oout, margin = oracle.verify(target, tok, slot, q, ci, temperature=1.0, seed=5, offset=1, V=V)
    # with 151936 ids a drawn token's own mass is ~7e-6 of the total, so many draws
    # land within the draw margin of a neighbour; the accept tests rarely do
    accept_ok = margin[:, 0] >= ACCEPT_MARGIN
    assert accept_ok.sum() >= B - 2
    assert np.array_equal(host(acc)[accept_ok], oacc[accept_ok])
    ok = ~excused(margin)
    assert ok.sum() >= B // 4
    assert np.array_equal(host(out)[ok], oout[ok])
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
    oacc, oout, margin = oracle.verify(target, tok, slot, q, ci, temperature=T, seed=3, V=V)
    ok = ~excused(margin)
    assert ok.sum() >= B - 1
    assert np.array_equal(host(acc), oacc) and np.array_equal(host(out)[ok], oout[ok])
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


def test_verify_scratch_grows_outside_capture_only(handle):
    """The per-row scratch lives in the handle: a call that fits runs inside a
    CUDA graph capture, a call that would need a larger buffer is refused there
    (DFLASH2_ERR_WORKSPACE) without breaking the capture, and the same call
    grows the buffer outside capture."""
    h = api.Handle(0)
    small = dict(B=4, L=4, V=1000)
    tok, slot, q, ci = draft(3, small["B"], small["L"], small["V"], 0.0)
    target = synth.target_planted(4, tok, small["V"], agree=0.85)
    big_B, big_L, big_V = 20000, 16, 8   # 340k rows: well past the initial 1 MiB
    big_tok = np.zeros((big_B, big_L), np.int32)
    big_target = np.zeros((big_B, big_L + 1, big_V), np.uint16)
    tg, tk, btg, btk = bf(target), i32(tok), bf(big_target), i32(big_tok)
    stream = torch.cuda.Stream()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.stream(stream):
        api.verify(h, tg, tk, V=small["V"])
        torch.cuda.synchronize()
        with torch.cuda.graph(graph, stream=stream):
            acc, out = api.verify(h, tg, tk, V=small["V"])
            with pytest.raises(api.Dflash2Error):
                api.verify(h, btg, btk, V=big_V)
        graph.replay()
    torch.cuda.synchronize()
    oacc, oout, _ = oracle.verify(target, tok, slot, q, ci, V=small["V"])
    assert np.array_equal(host(acc), oacc) and np.array_equal(host(out), oout)
    bacc, _ = api.verify(h, btg, btk, V=big_V)   # grows the scratch
    assert (host(bacc) >= 1).all()
    h.close()
