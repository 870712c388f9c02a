"""Gate + pair-score kernels vs the oracle (fp32 accumulation: 1e-3 rel / 1e-4 abs)."""
import numpy as np
import pytest

import oracle
from draft_selection_dflash2_gb300 import api, synth
from gpu_common import assert_close, bf, handle, host, i32  # noqa: F401

pytestmark = pytest.mark.gpu
K = 16


def run_case(h, sel, logits_bits=None):
    B, L, V, d = sel.B, sel.L, sel.V, sel.d
    U = sel.U.reshape(B * L, V) if logits_bits is None else logits_bits
    ov, oi = oracle.topk(U)
    ci, cv = oi.reshape(B, L, K), ov.reshape(B, L, K)
    S, gate = api.pair_scores(h, i32(ci), __import__("gpu_common").f32(cv), i32(sel.last_verified), bf(sel.h),
                              bf(sel.W_H), None, bf(sel.A), bf(sel.Bt))
    H = oracle.gate(sel.h.reshape(B * L, d), sel.W_H, sel.b_H)
    oS, bad = oracle.pair_scores(ci, cv, sel.last_verified, H.reshape(B, L, 256), sel.A, sel.Bt)
    return host(S), host(gate), oS, H, bad


@pytest.mark.parametrize("B,L,V,d,emb", [(1, 8, 4096, 512, 0.02), (1, 8, 4096, 512, 0.25),
                                         (3, 5, 4096, 512, 0.25), (1, 16, 151936, 2560, 0.02),
                                         (8, 16, 151936, 5120, 0.25), (16, 16, 4096, 2560, 0.25),
                                         (48, 16, 8192, 5120, 0.02), (2, 1, 4096, 512, 0.25),
                                         (96, 16, 8192, 512, 0.25)])
def test_pair_scores_match_oracle(handle, B, L, V, d, emb):
    sel = synth.selector_inputs(B * 100 + L, B, L, V, d, emb_std=emb)
    S, gate, oS, H, bad = run_case(handle, sel)
    assert not bad
    assert_close(gate.reshape(B * L, 256), H, what="gate")
    assert_close(S, oS, what="S")
    assert handle.device_error() == 0


def test_zero_embeddings_give_candidate_logits_exactly(handle):
    sel = synth.selector_inputs(7, 2, 6, 4096, 512)
    sel.A[:] = 0
    sel.Bt[:] = 0
    S, _, oS, _, _ = run_case(handle, sel)
    assert np.array_equal(S, oS.astype(np.float32))


def test_t0_rows_equal_and_bad_last_verified_flagged(handle):
    sel = synth.selector_inputs(8, 2, 4, 4096, 512, emb_std=0.25)
    sel.last_verified[:] = [5000, -3]      # out of range: clamped to V-1 and 0
    S, _, oS, _, bad = run_case(handle, sel)
    assert bad
    assert handle.device_error() & api.DEVERR_BAD_TOKEN
    assert_close(S, oS, what="S")
    assert np.array_equal(S[:, 0], np.broadcast_to(S[:, 0, :1], S[:, 0].shape))


def test_gate_bias(handle):
    import torch
    sel = synth.selector_inputs(9, 2, 4, 4096, 512)
    b = np.linspace(-2, 2, 256).astype(np.float32)
    ov, oi = oracle.topk(sel.U.reshape(8, 4096))
    from gpu_common import f32
    S, gate = api.pair_scores(handle, i32(oi.reshape(2, 4, K)), f32(ov.reshape(2, 4, K)),
                              i32(sel.last_verified), bf(sel.h), bf(sel.W_H), f32(b), bf(sel.A), bf(sel.Bt))
    H = oracle.gate(sel.h.reshape(8, 512), sel.W_H, b)
    assert_close(host(gate).reshape(8, 256), H, what="gate with bias")
    del torch
