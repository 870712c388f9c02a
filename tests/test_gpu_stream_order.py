"""Stream order with programmatic dependent launch.

The step's kernels may start while the previous kernel in the stream is still
running and wait (griddepcontrol.wait) before their first global access.  These
tests put PyTorch kernels between the library's calls on one stream -- each
rewriting a call's input just before it, or reading its output just after --
and check every iteration's result against the oracle, so that a kernel that
read an input (or wrote an output) before its predecessor finished would
show up as a wrong result."""
import numpy as np
import pytest
import torch

import oracle
from draft_selection_dflash2_gb300 import api, synth
from gpu_common import bf, handle, host  # noqa: F401

pytestmark = pytest.mark.gpu


def test_topk_inputs_rewritten_between_calls(handle):
    rows, V, n = 64, 32768, 6
    rng = np.random.default_rng(21)
    srcs = [synth.logits_planted(rng, rows, V) for _ in range(n)]
    dev_src = [bf(s) for s in srcs]
    logits = torch.empty_like(dev_src[0])
    vals = torch.empty((rows, 16), dtype=torch.float32, device="cuda")
    idx = torch.empty((rows, 16), dtype=torch.int32, device="cuda")
    outs = []
    for i in range(n):
        logits.copy_(dev_src[i])                 # a PyTorch kernel writes the input ...
        api.topk(handle, logits, vals=vals, idx=idx)
        outs.append((vals.clone(), idx.clone()))  # ... and PyTorch kernels read the output
    torch.cuda.synchronize()
    for i in range(n):
        ov, oi = oracle.topk(srcs[i])
        assert np.array_equal(host(outs[i][1]), oi) and np.array_equal(host(outs[i][0]), ov)
    assert handle.device_error() == 0


def test_conv_inputs_rewritten_and_outputs_reused(handle):
    # a PyTorch copy rewrites x before every application; two output buffers
    # alternate, each cloned by PyTorch right after the call that wrote it
    B, L, d, n = 8, 16, 512, 5
    cs = [synth.conv_inputs(31 + i, B, L, d) for i in range(n)]
    xs = [bf(c.x) for c in cs]
    x = torch.empty_like(xs[0])
    ys = [torch.empty_like(x), torch.empty_like(x)]
    outs = []
    for i, c in enumerate(cs):
        x.copy_(xs[i])
        y = api.conv2tap(handle, x, bf(c.x_prev), bf(c.k0), bf(c.k1), bf(c.W_c), y=ys[i % 2])
        outs.append(y.clone())
    torch.cuda.synchronize()
    for i, c in enumerate(cs):
        oy = oracle.conv2tap(c.x, c.x_prev, c.k0, c.k1, c.W_c)
        got = synth.bf16_to_f32(host(outs[i]).view(np.uint16)).astype(np.float64)
        ulp = 2.0 ** (np.floor(np.log2(np.maximum(np.abs(oy), 2.0 ** -126))) - 7)
        assert np.all(np.abs(got - oy) <= ulp + 1e-6), f"application {i}"
    assert handle.device_error() == 0
