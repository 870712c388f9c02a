"""The projection-form selector and the gate folded into the fused head, on the
GPU, against the oracle (fp32 tensor-core accumulation: 1e-3 rel / 1e-4 abs on
scores and gate values), and against the table form where both are exact."""
import numpy as np
import pytest
import torch

import oracle
from draft_selection_dflash2_gb300 import api, synth
from gpu_common import assert_close, bf, f32, handle, host, i32  # noqa: F401

pytestmark = pytest.mark.gpu
K = 16


# ---------------------------------------------------------------------------
# gate folded into the fused LM head
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("M,V,d,with_bias", [(200, 5000, 256, False), (1, 777, 128, True),
                                             (1024, 151936, 5120, True)])
def test_lmhead_gate_matches_plain_head_and_oracle_gate(handle, M, V, d, with_bias):
    hid = synth.normal_bits(M + d, (M, d))
    W = synth.normal_bits(M + d + 1, (V, d), std=0.02)
    W_H = synth.normal_bits(M + d + 2, (256, d), std=0.02)
    b = np.linspace(-1, 1, 256).astype(np.float32) if with_bias else None
    dh, dW = bf(hid), bf(W)
    vals, idx, gate = api.lmhead_topk_gate(handle, dh, dW, bf(W_H), f32(b) if b is not None else None)
    pv, pi = api.lmhead_topk(handle, dh, dW)
    assert handle.device_error() == 0
    # the extra tile changes nothing in the top-16: same tiles, same products
    assert np.array_equal(host(idx), host(pi))
    assert np.array_equal(host(vals).view(np.uint32), host(pv).view(np.uint32))
    rows = np.arange(M) if M <= 256 else np.sort(np.random.default_rng(1).choice(M, 64, replace=False))
    H = oracle.gate(hid[rows], W_H, b)
    assert_close(host(gate)[rows], H, what="gate")


# ---------------------------------------------------------------------------
# projection-form pair scores
# ---------------------------------------------------------------------------
def proj_inputs(seed, B, L, V, d):
    rng = np.random.default_rng(seed)
    ci = rng.integers(0, V, (B, L, K)).astype(np.int32)
    cv = rng.standard_normal((B, L, K)).astype(np.float32)
    lv = rng.integers(0, V, B).astype(np.int32)
    H = rng.random((B, L, 256)).astype(np.float32)
    E = synth.normal_bits(seed + 1, (V, d))
    WA = synth.normal_bits(seed + 2, (256, d), std=1.0 / np.sqrt(d))
    WB = synth.normal_bits(seed + 3, (256, d), std=1.0 / np.sqrt(d))
    return ci, cv, lv, H, E, WA, WB


def run_proj(h, ci, cv, lv, H, E, WA, WB):
    S, P = api.pair_scores_proj(h, i32(ci), f32(cv), i32(lv), f32(H), bf(E), bf(WA), bf(WB))
    return host(S), host(P)


@pytest.mark.parametrize("B,L,V,d", [(1, 3, 4096, 512), (3, 5, 4096, 512), (2, 16, 151936, 2560),
                                     (5, 7, 20000, 5120), (1, 1, 64, 64)])
def test_pair_scores_proj_matches_oracle(handle, B, L, V, d):
    ci, cv, lv, H, E, WA, WB = proj_inputs(B * 1000 + L, B, L, V, d)
    S, P = run_proj(handle, ci, cv, lv, H, E, WA, WB)
    assert handle.device_error() == 0
    oS, bad = oracle.pair_scores_proj(ci, cv, lv, H.astype(np.float64), E, WA, WB)
    assert not bad
    assert_close(S, oS, what="S")
    assert np.array_equal(S[:, 0], np.broadcast_to(S[:, 0, :1], S[:, 0].shape))
    # the projections themselves, for a few rows (numpy matmul of the widened operands)
    Ef, WAf, WBf = (synth.bf16_to_f32(a).astype(np.float64) for a in (E, WA, WB))
    n_cand = B * L * K
    for m in sorted({0, n_cand - 1, n_cand, n_cand + B - 1, (n_cand // 2)}):
        tok = ci.reshape(-1)[m] if m < n_cand else lv[m - n_cand]
        assert_close(P[m, :256], WAf @ Ef[tok], what=f"A row {m}")
        assert_close(P[m, 256:], WBf @ Ef[tok], what=f"B row {m}")


def test_pair_scores_proj_equals_table_form_on_exact_data(handle):
    # entries in {-1, 0, 1} and H = 1: every projection is an exact small integer,
    # the tables E W^T are exact in bf16, and both forms run the same products
    B, L, V, d = 4, 6, 700, 128
    rng = np.random.default_rng(5)
    ci = rng.integers(0, V, (B, L, K)).astype(np.int32)
    cv = rng.standard_normal((B, L, K)).astype(np.float32)
    lv = rng.integers(0, V, B).astype(np.int32)
    Ei, WAi, WBi = rng.integers(-1, 2, (V, d)), rng.integers(-1, 2, (256, d)), rng.integers(-1, 2, (256, d))
    bits = lambda a: synth.bf16_bits(a.astype(np.float32))          # noqa: E731
    ones = np.ones((B, L, 256), np.float32)
    S, _ = run_proj(handle, ci, cv, lv, ones, bits(Ei), bits(WAi), bits(WBi))
    # table form through the same pair products: the gate GEMM gives H = sigmoid(0) = 0.5
    # for h = 0, so feed the tables scaled by 2 on one side to get H * A = A exactly
    hs = np.zeros((B, L, d), np.uint16)
    W_H = np.zeros((256, d), np.uint16)
    St, gate = api.pair_scores(handle, i32(ci), f32(cv), i32(lv), bf(hs), bf(W_H), None,
                               bf(bits(2 * (Ei @ WAi.T))), bf(bits(Ei @ WBi.T)))
    assert np.all(host(gate) == 0.5)
    assert np.array_equal(S.view(np.uint32), host(St).view(np.uint32))


def test_pair_scores_proj_flags_bad_ids(handle):
    B, L, V, d = 2, 4, 4096, 256
    ci, cv, lv, H, E, WA, WB = proj_inputs(9, B, L, V, d)
    lv[:] = [V + 5, -2]
    ci[1, 2, 3] = V
    S, _ = run_proj(handle, ci, cv, lv, H, E, WA, WB)
    assert handle.device_error() & api.DEVERR_BAD_TOKEN        # reading clears it
    oS, bad = oracle.pair_scores_proj(ci, cv, lv, H.astype(np.float64), E, WA, WB)
    assert bad
    assert_close(S, oS, what="S")


def test_pair_scores_proj_full_size_sampled_sequences(handle):
    # the benchmark's shape: B=128, L=16, V=151936, d=5120; two sequences checked in fp64
    B, L, V, d = 128, 16, 151936, 5120
    ci, cv, lv, H, E, WA, WB = proj_inputs(11, B, L, V, d)
    S, _ = run_proj(handle, ci, cv, lv, H, E, WA, WB)
    assert handle.device_error() == 0
    sel = np.array([0, 77])
    oS, _ = oracle.pair_scores_proj(ci[sel], cv[sel], lv[sel], H[sel].astype(np.float64), E, WA, WB)
    assert_close(S[sel], oS, what="S (sampled sequences)")


def test_pair_scores_proj_workspace_too_small(handle):
    B, L, V, d = 1, 2, 256, 64
    ci, cv, lv, H, E, WA, WB = proj_inputs(3, B, L, V, d)
    small = torch.empty((B * L * K, 512), dtype=torch.float32, device="cuda")   # misses the B extra rows
    with pytest.raises(RuntimeError, match="WORKSPACE"):
        api.pair_scores_proj(handle, i32(ci), f32(cv), i32(lv), f32(H), bf(E), bf(WA), bf(WB), P=small)
    assert api.pair_scores_proj_workspace(handle, B, L) == (B * L * K + B) * 512 * 4
