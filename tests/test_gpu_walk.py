"""Walk kernel vs the oracle on identical generated scores.

Greedy choices are compared exactly.  Sampled draws are taken in fp32 by the
same sequence of correctly rounded IEEE operations on both sides (2^x by Cody-
Waite reduction and a degree-7 Taylor polynomial), so slots, tokens and the
proposal distributions q must agree bit for bit, with no tolerance."""
import numpy as np
import pytest

import oracle
from draft_selection_dflash2_gb300 import api
from gpu_common import f32, handle, host, i32  # noqa: F401

pytestmark = pytest.mark.gpu
K = 16


def scores(seed, B, L, scale=1.0, ties=False):
    rng = np.random.default_rng(seed)
    S = (rng.standard_normal((B, L, K, K)) * scale).astype(np.float32)
    if ties:
        S[..., 5] = S[..., 2]
        S[..., 11] = S[..., 2]
    ci = rng.integers(0, 151936, (B, L, K)).astype(np.int32)
    return S, ci


@pytest.mark.parametrize("B,L", [(1, 8), (1, 16), (5, 3), (128, 16), (256, 16), (7, 64)])
def test_greedy_walk_exact(handle, B, L):
    S, ci = scores(B * 31 + L, B, L, ties=True)
    tok, slot, q = api.walk(handle, f32(S), i32(ci))
    otok, oslot, oq, _ = oracle.walk(S, ci)
    assert np.array_equal(host(slot), oslot) and np.array_equal(host(tok), otok)
    assert np.array_equal(host(q), oq)


@pytest.mark.parametrize("T", [1.0, 0.5, 2.0, 0.07])
@pytest.mark.parametrize("B,L", [(1, 16), (128, 16), (33, 7)])
def test_sampled_walk_exact(handle, B, L, T):
    S, ci = scores(B + L + int(T * 10), B, L, scale=2.0)
    Tf = float(np.float32(T))
    for seed, offset in ((1, 0), (1, 7), (99, (5 << 32) + 3)):
        tok, slot, q = api.walk(handle, f32(S), i32(ci), temperature=T, seed=seed, offset=offset)
        otok, oslot, oq, _ = oracle.walk(S, ci, temperature=Tf, seed=seed, offset=offset)
        assert np.array_equal(host(slot), oslot) and np.array_equal(host(tok), otok)
        assert np.array_equal(host(q).view(np.uint32), oq.view(np.uint32))


def test_sampled_walk_large_score_spread(handle):
    # weights underflow to 0 (exp2 argument below -126) for most slots
    S, ci = scores(5, 64, 16, scale=400.0)
    tok, slot, q = api.walk(handle, f32(S), i32(ci), temperature=0.3, seed=4)
    otok, oslot, oq, _ = oracle.walk(S, ci, temperature=float(np.float32(0.3)), seed=4)
    assert np.array_equal(host(slot), oslot)
    assert np.array_equal(host(q).view(np.uint32), oq.view(np.uint32))


def test_walk_without_q(handle):
    S, ci = scores(3, 4, 8)
    tok, slot, q = api.walk(handle, f32(S), i32(ci), temperature=1.0, seed=3, want_q=False)
    assert q is None
    otok, oslot, _, _ = oracle.walk(S, ci, temperature=1.0, seed=3)
    assert np.array_equal(host(slot), oslot)


@pytest.mark.parametrize("T", [0.0, 1.0])
def test_walk_nan_scores(handle, T):
    """NaN never beats a number (the lowest slot of the largest non-NaN score
    wins; all NaN: slot 0), in any slot, at either temperature; a sampled row
    with no positive weight (all NaN or -inf) takes the greedy slot with q
    one-hot.  Every lane must reach the same slot, or later steps would mix
    predecessors: slots, tokens and q are compared bit for bit."""
    rng = np.random.default_rng(77)
    B, L = 96, 12
    S = rng.standard_normal((B, L, K, K)).astype(np.float32)
    S[rng.random(S.shape) < 0.25] = np.nan
    S[0, 0, 0, :] = np.nan
    S[1, 0, 0, :] = -np.inf
    S[2, 0, 0, 0] = np.nan
    S[3, :, :, 7] = np.nan
    S[4, 1] = np.nan
    S[5, 2] = -np.inf
    ci = rng.integers(0, 151936, (B, L, K)).astype(np.int32)
    tok, slot, q = api.walk(handle, f32(S), i32(ci), temperature=T, seed=8)
    otok, oslot, oq, _ = oracle.walk(S, ci, temperature=float(np.float32(T)), seed=8)
    assert np.array_equal(host(slot), oslot) and np.array_equal(host(tok), otok)
    assert np.array_equal(host(q).view(np.uint32), oq.view(np.uint32))
    assert (oslot >= 0).all()
    assert handle.device_error() == 0
