"""Race and bounds evidence without compute-sanitizer.

Every entry point runs twice on the same inputs and must give byte-identical
outputs (a race between CTAs, or a read of memory that another call left
behind, shows up as a difference), and writes its outputs into buffers padded
on both sides with a canary pattern that must survive (an out-of-bounds write
shows up as a changed canary)."""
import numpy as np
import pytest
import torch

from draft_selection_dflash2_gb300 import api, synth
from gpu_common import bf, handle, host  # noqa: F401

pytestmark = pytest.mark.gpu
K = 16
PAD = 4096          # canary bytes on each side (keeps every alignment)
CANARY = 0x5A


class Guarded:
    """Output tensors carved out of canary-filled byte buffers."""

    def __init__(self):
        self.bufs = []

    def __call__(self, shape, dtype):
        n = int(np.prod(shape)) * torch.tensor([], dtype=dtype).element_size()
        buf = torch.full((n + 2 * PAD,), CANARY, dtype=torch.uint8, device="cuda")
        self.bufs.append((buf, n))
        return buf[PAD:PAD + n].view(dtype).view(shape)

    def check(self):
        torch.cuda.synchronize()
        for buf, n in self.bufs:
            b = buf.cpu().numpy()
            assert (b[:PAD] == CANARY).all() and (b[PAD + n:] == CANARY).all(), "canary overwritten"


def twice(fn):
    outs = []
    for _ in range(2):
        g = Guarded()
        res = fn(g)
        g.check()
        outs.append([host(t).copy() for t in res])
    for a, b in zip(*outs):
        assert a.tobytes() == b.tobytes()
    return outs[0]


@pytest.fixture(scope="module")
def sel():
    return synth.selector_inputs(9, 32, 16, 151936, 5120)


def test_topk_and_selector_stages(handle, sel):
    B, L, V, d = 32, 16, 151936, 5120
    U = bf(sel.U.reshape(B * L, V))
    hs, W_H, A, Bt = bf(sel.h), bf(sel.W_H), bf(sel.A), bf(sel.Bt)
    lv = torch.from_numpy(sel.last_verified).cuda()

    def run(g):
        vals, idx = api.topk(handle, U, vals=g((B * L, K), torch.float32), idx=g((B * L, K), torch.int32))
        ci, cv = idx.view(B, L, K), vals.view(B, L, K)
        S, gate = api.pair_scores(handle, ci, cv, lv, hs, W_H, None, A, Bt, gate=g((B, L, 256), torch.float32),
                                  S=g((B, L, K, K), torch.float32))
        out = [vals, idx, S, gate]
        for T in (0.0, 1.0):
            tok, slot, q = api.walk(handle, S, ci, temperature=T, seed=3, draft_tok=g((B, L), torch.int32),
                                    draft_slot=g((B, L), torch.int32), draft_q=g((B, L, K), torch.float32))
            out += [tok, slot, q]
        vt, vs, sc = api.walk_viterbi(handle, S, ci, draft_tok=g((B, L), torch.int32),
                                      draft_slot=g((B, L), torch.int32), score=g((B,), torch.float32))
        a1, a16, cnt = api.selector_eval(handle, out[4], ci, accept1=g((B,), torch.int32),
                                         accept16=g((B,), torch.int32), counts=g((L, 4), torch.int64))
        return out + [vt, vs, sc, a1, a16, cnt]

    twice(run)
    assert handle.device_error() == 0


def test_conv_and_fused_conv(handle):
    B, L, d = 16, 16, 5120
    c = synth.conv_inputs(4, B, L, d)
    x, xp, k0, k1, W_c = bf(c.x), bf(c.x_prev), bf(c.k0), bf(c.k1), bf(c.W_c)
    A = bf(synth.normal_bits(5, (B, L, 1024)))
    W = bf(synth.normal_bits(6, (d, 1024), std=1024 ** -0.5))

    def run(g):
        y = api.conv2tap(handle, x, xp, k0, k1, W_c, y=g((B, L, d), torch.bfloat16))
        y32 = api.conv2tap(handle, x, xp, k0, k1, W_c, y=g((B, L, d), torch.float32))
        ws = g(((api.gemm_conv2tap_workspace(handle, B, L, d) + 3) // 4,), torch.float32)
        yf, cw = api.gemm_conv2tap(handle, A, W, xp, x, k0, k1, W_c, c_work=ws, y=g((B, L, d), torch.bfloat16))
        return [y, y32, yf, cw]

    twice(run)
    assert handle.device_error() == 0


@pytest.mark.parametrize("T", [0.0, 1.0])
def test_verify(handle, T):
    B, L, V = 128, 16, 151936
    rng = np.random.default_rng(7)
    tok = rng.integers(0, V, (B, L)).astype(np.int32)
    ci = np.concatenate([tok[..., None], rng.integers(0, V, (B, L, K - 1))], axis=-1).astype(np.int32)
    q = rng.dirichlet(np.ones(K), (B, L)).astype(np.float32)
    slot = np.zeros((B, L), np.int32)
    target = bf(synth.target_planted(8, tok, V, agree=0.85, plant=8.0 if T == 0 else 14.0))
    dev = lambda a: torch.from_numpy(a).cuda()  # noqa: E731
    tk, sl, qq, cc = dev(tok), dev(slot), dev(q), dev(ci)

    def run(g):
        ws = g((api.verify_workspace(handle, B, L, V),), torch.uint8)
        acc, out = api.verify(handle, target, tk, sl, qq, cc, temperature=T, seed=5, accept_len=g((B,), torch.int32),
                              out_tok=g((B, L + 1), torch.int32), workspace=ws)
        return [acc, out]

    twice(run)
    assert handle.device_error() == 0


def test_lmhead_forms(handle):
    M, V, d = 256, 30000, 1024
    hid = bf(synth.normal_bits(11, (M, d)))
    W = bf(synth.normal_bits(12, (V, d), std=0.02))
    W_H = bf(synth.normal_bits(13, (256, d), std=0.02))
    E = bf(synth.normal_bits(14, (V, d)))
    W_A = bf(synth.normal_bits(15, (256, d), std=d ** -0.5))
    W_B = bf(synth.normal_bits(16, (256, d), std=d ** -0.5))

    def run(g):
        ws = g((api.lmhead_topk_workspace(handle, M, V, d),), torch.uint8)
        v, i = api.lmhead_topk(handle, hid, W, vals=g((M, K), torch.float32), idx=g((M, K), torch.int32), workspace=ws)
        v2, i2, gate = api.lmhead_topk_gate(handle, hid, W, W_H, vals=g((M, K), torch.float32),
                                            idx=g((M, K), torch.int32), gate=g((M, 256), torch.float32), workspace=ws)
        B, L = 16, 16
        ci, cv = i.view(B, L, K), v.view(B, L, K)
        lv = ci[:, 0, 0].contiguous()
        P = g((B * L * K + B, 512), torch.float32)
        S, _ = api.pair_scores_proj(handle, ci, cv, lv, gate.view(B, L, 256), E, W_A, W_B, P=P,
                                    S=g((B, L, K, K), torch.float32))
        return [v, i, v2, i2, gate, S]

    twice(run)
    assert handle.device_error() == 0
