"""End-to-end draft-block head on the GPU vs the chained oracle.

Chain: [conv x n] -> top-16 -> gate + pair scores -> walk -> verify.
Each side runs its own chain from the same generated inputs (no oracle input
comes from the GPU).  Rules: each conv application within one bf16 ulp; top-16
bit-exact; S within 1e-3 rel / 1e-4 abs.  The walks read their own S, which
differ by at most dS = max |S_gpu - S_oracle| (measured, ~1e-6): a greedy step
whose oracle margin (best - runner-up) exceeds 2 dS cannot change its arg-max,
and a sampled step whose draw lies further than max(1e-5, 8 c dS) (relative to
Z) from its CDF bounds cannot change its slot, so every such step is compared,
up to each sequence's first step without that margin (after it the two walks
may legitimately follow different predecessors).  At most 5% of sequences may
have such a step.  Verification is exact (fixed-point weights on both sides):
at T = 0 every sequence whose two drafts agree gives the same acceptance length
and tokens; at T > 0 the proposals q still differ in their last bits (each walk
rounds its own S), so the comparison covers every sequence whose decisions
those differences cannot flip, and at most 10% may lack that margin."""
import numpy as np
import pytest

import oracle
from draft_selection_dflash2_gb300 import api, synth
from gpu_common import assert_close, bf, f32, handle, host, i32  # noqa: F401

pytestmark = pytest.mark.gpu
K = 16


def bf16_ulp(v):
    e = np.floor(np.log2(np.maximum(np.abs(v), 2.0**-126)))
    return 2.0 ** (e - 7)


def compared_prefix(tight):
    """Per sequence, the number of leading steps before the first tight decision."""
    B, L = tight.shape
    first = np.where(tight.any(axis=1), tight.argmax(axis=1), L)
    return first


def robust_to_q(target, otok, oslot, oq, gq, ci, oacc, oout, T, seed, offset=0):
    """Per sequence: whether none of the oracle's sampled decisions can flip when
    each proposal weight moves from the oracle's q to the GPU's (the two walks
    read slightly different S), recomputed from the oracle's own fixed-point
    weights: an accept test (u1 q) Z < W_x moves by at most u1 |dq| Z; a
    residual draw's target and its token's interval bounds move by at most
    sum_j (|dq_j| Z + 1) each (an exact 0 where the two q agree bit for bit).
    The bonus draw does not read q."""
    B, L = otok.shape
    V = target.shape[-1]
    dq = np.abs(gq.astype(np.float64) - oq.astype(np.float64))
    same = gq.view(np.uint32) == oq.view(np.uint32)
    ok = np.ones(B, bool)
    for b in range(B):
        n = int(oacc[b]) - 1
        for t in range(min(n + 1, L)):
            j = oslot[b, t]
            if same[b, t, j]:
                continue
            W, Z = oracle.verify_weights(target[b, t], T)
            u1 = oracle.uniform24(seed, b, t, 1, offset)
            lhs = u1 * float(oq[b, t, j]) * Z
            if abs(lhs - float(W[otok[b, t]])) <= 2.0 * u1 * dq[b, t, j] * Z + 2.0:
                ok[b] = False
                break
        if ok[b] and n < L and not same[b, n].all():
            W, Z = oracle.verify_weights(target[b, n], T)
            Q = np.zeros(V, np.float64)
            cand = np.zeros(V, bool)
            for j in range(K):
                Q[ci[b, n, j]] += np.floor(min(max(float(oq[b, n, j]), 0.0), 1.0) * Z)
                cand[ci[b, n, j]] = True
            R = np.where(cand, np.maximum(W.astype(np.float64) - Q, 0.0), W.astype(np.float64))
            total = R.sum()
            if total <= 0:
                continue
            cdf = np.cumsum(R)
            U2 = round(oracle.uniform24(seed, b, n, 2, offset) * 2**24)
            tgt = np.floor(U2 * total / 2**24)
            v = int(oout[b, n])
            lo = cdf[v - 1] if v > 0 else 0.0
            slack = 2.0 * float(np.sum(np.where(same[b, n], 0.0, dq[b, n] * Z + 1.0)))
            if min(tgt - lo, cdf[v] - tgt) <= slack:
                ok[b] = False
    return ok


def chain(h, seed, B, L, V, d, logits="planted", conv_apps=0, temperatures=(0.0,), emb=0.02):
    """Runs the GPU chain and the oracle chain side by side.  Each side feeds
    its own outputs forward; the only shared inputs come from the generator."""
    sel = synth.selector_inputs(seed, B, L, V, d, logits=logits, emb_std=emb)
    o_h, g_h = sel.h, bf(sel.h)
    if conv_apps:
        # each application reads its own activation (a new sublayer boundary);
        # the last output is the hidden state that feeds the gate
        for a in range(conv_apps):
            x = synth.normal_bits(seed + 100 + a, (B, L, d))
            x_prev = synth.normal_bits(seed + 200 + a, (B, d))
            k0, k1, W_c = synth.conv_layer_params(seed + 10 + a, d)
            g_cur = api.conv2tap(h, bf(x), bf(x_prev), bf(k0), bf(k1), bf(W_c))
            oy = oracle.conv2tap(x, x_prev, k0, k1, W_c)
            got = synth.bf16_to_f32(host(g_cur)).astype(np.float64)
            assert np.all(np.abs(got - oy) <= bf16_ulp(oy) + 1e-4), f"application {a}"
        o_h, g_h = synth.bf16_bits(oy.astype(np.float32)), g_cur
    U = sel.U.reshape(B * L, V)
    vals, idx = api.topk(h, bf(U))
    ov, oi = oracle.topk(U)
    assert np.array_equal(host(idx), oi) and np.array_equal(host(vals), ov)
    ci, cv = oi.reshape(B, L, K), ov.reshape(B, L, K)
    S, gate = api.pair_scores(h, idx.view(B, L, K), vals.view(B, L, K), i32(sel.last_verified), g_h,
                              bf(sel.W_H), None, bf(sel.A), bf(sel.Bt))
    H = oracle.gate(o_h.reshape(B * L, d), sel.W_H, sel.b_H).reshape(B, L, 256)
    oS, _ = oracle.pair_scores(ci, cv, sel.last_verified, H, sel.A, sel.Bt)
    assert_close(host(S), oS, what="S")
    o_S32 = oS.astype(np.float32)
    dS = float(np.max(np.abs(host(S).astype(np.float64) - o_S32.astype(np.float64))))
    assert dS < 1e-4
    results = {}
    greedy_otok = None
    for T in temperatures:
        Tf = float(np.float32(T))
        tok, slot, q = api.walk(h, S, idx.view(B, L, K), temperature=T, seed=1)
        otok, oslot, oq, margin = oracle.walk(o_S32, ci, temperature=Tf, seed=1)
        if T == 0:
            greedy_otok = otok
            tight = margin <= 2.0 * dS
        else:
            tight = margin <= max(1e-5, 8.0 * (1.4427 / Tf) * dS)
        n_cmp = compared_prefix(tight)
        gtok = host(tok)
        for b in range(B):
            assert np.array_equal(gtok[b, :n_cmp[b]], otok[b, :n_cmp[b]]), f"sequence {b}"
        assert (n_cmp < L).sum() <= max(1, 0.05 * B), f"{(n_cmp < L).sum()} of {B} sequences have a tight step"
        same_draft = np.all(gtok == otok, axis=1)
        assert (~same_draft).sum() <= max(1, 0.05 * B)
        # the target is planted on the oracle's greedy draft; both sides verify their own draft
        target = synth.target_planted(seed + 5, greedy_otok, V, agree=0.85,
                                      plant=8.0 if T == 0 else 14.0)
        acc, out = api.verify(h, bf(target), tok, slot, q, idx.view(B, L, K), temperature=T, seed=1)
        oacc, oout, _ = oracle.verify(target, otok, oslot, oq, ci, temperature=Tf, seed=1)
        ok = same_draft
        if T > 0:
            # the proposals differ by the walks' own rounding of slightly different
            # S: compare every sequence whose decisions that difference cannot flip
            gq = host(q)
            assert float(np.max(np.abs(gq.astype(np.float64) - oq)[same_draft], initial=0.0)) < 1e-4
            ok = ok & robust_to_q(target, otok, oslot, oq, gq, ci, oacc, oout, Tf, 1)
            assert (~ok).sum() <= max(1, 0.1 * B), f"{(~ok).sum()} of {B} sequences without margin"
        assert np.array_equal(host(acc)[ok], oacc[ok]) and np.array_equal(host(out)[ok], oout[ok])
        results[T] = host(acc)
    assert h.device_error() == 0
    return results


def test_tiny_selector(handle):
    chain(handle, 0, 1, 8, 4096, 512)


def test_tiny_selector_stress_embeddings(handle):
    chain(handle, 1, 4, 8, 4096, 512, emb=0.25)


def test_qwen3_4b_shaped_head(handle):
    chain(handle, 2, 1, 16, 151936, 2560, logits="zipf", conv_apps=1, temperatures=(0.0, 1.0))


def test_batch_sweep_b32(handle):
    chain(handle, 3, 32, 16, 151936, 5120)


def test_full_cycle_reduced_batch(handle):
    acc = chain(handle, 4, 8, 16, 151936, 5120, conv_apps=10, temperatures=(0.0, 1.0))
    assert np.all((acc[0.0] >= 1) & (acc[0.0] <= 17))


def test_full_cycle_benchmark_batch(handle):
    # the benchmark's workload: B=128, L=16, V=151936, d=5120, conv x10, both temperatures
    acc = chain(handle, 5, 128, 16, 151936, 5120, conv_apps=10, temperatures=(0.0, 1.0))
    assert acc[0.0].mean() > 4.0 and np.all((acc[1.0] >= 1) & (acc[1.0] <= 17))
