"""Runs one stage of the draft-block head on seeded synthetic inputs of the
full-cycle workload's shape (B sequences, L=16, V=151936, d=5120), a few
times, so that a profiler (ncu) can capture that stage's kernels alone.

  python -m draft_selection_dflash2_gb300.profile_stage --stage topk [--B 128] [--reps 3]

Stages: topk, pairs (gate + pair scores), walk0, walk1, conv (one application),
verify0, verify1, lmhead (M=1024 hidden rows against the full vocabulary),
lmhead_gate (the same with the context gate folded in), viterbi (the exact
best-path walk on N(0, 4) scores of B sequences), eval (the Table 1 selector
evaluation of B sequences of 7 positions with uniform candidate ids and the
true token in slot 0 of 80% of the rows), proj (projection-form pair scores
of B sequences: A, B projected from an N(0, 1) [V, d] embedding) and gemm_conv
(the conv fused into an output projection with K = d).
"""
import argparse
import os
import sys

import numpy as np

sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))

from draft_selection_dflash2_gb300 import api, synth  # noqa: E402

L, V, D, R, K = 16, 151936, 5120, 256, 16


def bf(torch, a):
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).cuda().view(torch.bfloat16)


def main():
    import torch

    ap = argparse.ArgumentParser()
    ap.add_argument("--stage", required=True,
                    choices=["topk", "pairs", "walk0", "walk1", "conv", "verify0", "verify1", "lmhead",
                             "lmhead_gate", "viterbi", "eval", "proj", "gemm_conv"])
    ap.add_argument("--B", type=int, default=128)
    ap.add_argument("--reps", type=int, default=3)
    args = ap.parse_args()
    torch.cuda.set_device(0)
    B = args.B
    h = api.Handle(0)
    rng = np.random.default_rng(0)
    if args.stage == "topk":
        U = bf(torch, synth.logits_planted(rng, B * L, V))
        run = lambda: api.topk(h, U)  # noqa: E731
    elif args.stage in ("pairs", "walk0", "walk1"):
        U = bf(torch, synth.logits_planted(rng, B * L, V))
        vals, idx = api.topk(h, U)
        del U
        hs = bf(torch, synth.normal_bits(1, (B, L, D)))
        W_H = bf(torch, synth.normal_bits(2, (R, D), std=0.02))
        A = bf(torch, synth.normal_bits(3, (V, R), std=0.02))
        Bt = bf(torch, synth.normal_bits(4, (V, R), std=0.02))
        lv = torch.from_numpy(rng.integers(0, V, B).astype(np.int32)).cuda()
        ci, cv = idx.view(B, L, K), vals.view(B, L, K)
        if args.stage == "pairs":
            run = lambda: api.pair_scores(h, ci, cv, lv, hs, W_H, None, A, Bt)  # noqa: E731
        else:
            S, _ = api.pair_scores(h, ci, cv, lv, hs, W_H, None, A, Bt)
            T = 0.0 if args.stage == "walk0" else 1.0
            run = lambda: api.walk(h, S, ci, temperature=T, seed=1)  # noqa: E731
    elif args.stage == "conv":
        x = bf(torch, synth.normal_bits(1, (B, L, D)))
        xp = bf(torch, synth.normal_bits(2, (B, D)))
        k0, k1, W_c = (bf(torch, a) for a in synth.conv_layer_params(3, D))
        y = torch.empty((B, L, D), dtype=torch.bfloat16, device="cuda")
        cws = torch.empty(api.conv2tap_workspace(h, B, L, D), dtype=torch.uint8, device="cuda")
        run = lambda: api.conv2tap(h, x, xp, k0, k1, W_c, y=y, workspace=cws)  # noqa: E731
    elif args.stage in ("verify0", "verify1"):
        T = 0.0 if args.stage == "verify0" else 1.0
        tok = rng.integers(0, V, (B, L)).astype(np.int32)
        ci = np.concatenate([tok[..., None], rng.integers(0, V, (B, L, K - 1))], axis=-1).astype(np.int32)
        slot = np.zeros((B, L), np.int32)
        q = np.full((B, L, K), 1.0 / K, np.float32)
        target = bf(torch, synth.target_planted(5, tok, V, agree=0.85, plant=8.0))
        dev = lambda a: torch.from_numpy(a).cuda()  # noqa: E731
        tok_d, slot_d, q_d, ci_d = dev(tok), dev(slot), dev(q), dev(ci)
        ws = torch.empty(api.verify_workspace(h, B, L, V), dtype=torch.uint8, device="cuda")
        run = lambda: api.verify(h, target, tok_d, slot_d, q_d, ci_d, temperature=T, seed=1, workspace=ws)  # noqa: E731
    elif args.stage == "viterbi":
        g = torch.Generator(device="cuda")
        g.manual_seed(5)
        S = torch.randn((B, L, K, K), generator=g, device="cuda") * 2
        ci = torch.randint(0, V, (B, L, K), generator=g, device="cuda", dtype=torch.int32)
        run = lambda: api.walk_viterbi(h, S, ci)  # noqa: E731
    elif args.stage == "eval":
        g = torch.Generator(device="cuda")
        g.manual_seed(6)
        Le = 7
        gt = torch.randint(0, V, (B, Le), generator=g, device="cuda", dtype=torch.int32)
        cand = torch.randint(0, V, (B, Le, K), generator=g, device="cuda", dtype=torch.int32)
        hit = torch.rand((B, Le), generator=g, device="cuda") < 0.8
        cand[:, :, 0] = torch.where(hit, gt, cand[:, :, 0])
        run = lambda: api.selector_eval(h, gt, cand)  # noqa: E731
    elif args.stage == "gemm_conv":
        A = bf(torch, synth.normal_bits(1, (B, L, D)))
        Wp = bf(torch, synth.normal_bits(2, (D, D), std=D ** -0.5))
        hs = bf(torch, synth.normal_bits(3, (B, L, D)))
        xp = bf(torch, synth.normal_bits(4, (B, D)))
        k0, k1, W_c = (bf(torch, a) for a in synth.conv_layer_params(5, D))
        run = lambda: api.gemm_conv2tap(h, A, Wp, xp, hs, k0, k1, W_c)  # noqa: E731
    elif args.stage == "proj":
        g = torch.Generator(device="cuda")
        g.manual_seed(7)
        ci = torch.randint(0, V, (B, L, K), generator=g, device="cuda", dtype=torch.int32)
        cv = torch.randn((B, L, K), generator=g, device="cuda")
        lv = torch.randint(0, V, (B,), generator=g, device="cuda", dtype=torch.int32)
        H = torch.rand((B, L, R), generator=g, device="cuda")
        E = torch.randn((V, D), generator=g, device="cuda").to(torch.bfloat16)
        WA = (torch.randn((R, D), generator=g, device="cuda") / D ** 0.5).to(torch.bfloat16)
        WB = (torch.randn((R, D), generator=g, device="cuda") / D ** 0.5).to(torch.bfloat16)
        run = lambda: api.pair_scores_proj(h, ci, cv, lv, H, E, WA, WB)  # noqa: E731
    else:
        M = 1024
        hidden = bf(torch, synth.normal_bits(1, (M, D)))
        W = bf(torch, synth.normal_bits(2, (V, D), std=0.02))
        ws = torch.empty(max(api.lmhead_topk_workspace(h, M, V, D), 256), dtype=torch.uint8, device="cuda")
        if args.stage == "lmhead_gate":
            W_H = bf(torch, synth.normal_bits(3, (R, D), std=0.02))
            run = lambda: api.lmhead_topk_gate(h, hidden, W, W_H, workspace=ws)  # noqa: E731
        else:
            run = lambda: api.lmhead_topk(h, hidden, W, workspace=ws)  # noqa: E731
    for _ in range(args.reps):
        run()
    torch.cuda.synchronize()
    assert h.device_error() == 0
    print(f"{args.stage}: {args.reps} runs ok")
    h.close()


if __name__ == "__main__":
    main()
