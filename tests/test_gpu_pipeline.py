"""End-to-end draft-block head on the GPU vs the chained oracle.

Chain: [conv x n] -> top-16 -> gate + pair scores -> walk -> verify.
Each side runs its own chain from the same generated inputs (no oracle input
comes from the GPU).  Rules: top-16 bit-exact; S within 1e-3 rel / 1e-4 abs;
each conv application within one bf16 ulp; walk choices exact for every sequence whose oracle
decision margin exceeds 1e-3 (greedy, absolute) or 1e-5 (sampled, relative to
Z) -- the rest are counted and must be rare; verification exact on sequences
whose drafts agree, except sampled decisions within 1e-4 (relative) of their
boundary."""
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
    results = {}
    greedy_otok = None
    for T in temperatures:
        Tf = float(np.float32(T))
        tok, slot, q = api.walk(h, S, idx.view(B, L, K), temperature=T, seed=1)
        otok, oslot, oq, margin = oracle.walk(o_S32, ci, temperature=Tf, seed=1)
        if T == 0:
            greedy_otok = otok
        # compare every step up to each sequence's first tight decision (after
        # it the two walks may legitimately follow different predecessors)
        tight = margin < (1e-3 if T == 0 else 1e-5)
        n_cmp = compared_prefix(tight)
        gtok = host(tok)
        for b in range(B):
            assert np.array_equal(gtok[b, :n_cmp[b]], otok[b, :n_cmp[b]]), f"sequence {b}"
        assert n_cmp.sum() >= 0.5 * B * L, f"only {n_cmp.sum()} of {B * L} steps comparable"
        same_draft = n_cmp == L
        # the target is planted on the oracle's greedy draft; both sides verify their own draft
        target = synth.target_planted(seed + 5, greedy_otok, V, agree=0.85,
                                      plant=8.0 if T == 0 else 14.0)
        acc, out = api.verify(h, bf(target), tok, slot, q, idx.view(B, L, K), temperature=T, seed=1)
        oacc, oout, vmargin = oracle.verify(target, otok, oslot, oq, ci, temperature=Tf, seed=1)
        ok = same_draft & (vmargin[:, 0] >= 1e-5) & (vmargin[:, 1] >= 2e-6)
        assert ok.sum() >= B // 2
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
