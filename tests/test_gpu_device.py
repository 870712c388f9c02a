"""The handle's device must be the current device.

Kernels launch on the calling thread's current device and write the handle's
error word on the handle's device, so a compute call made while another device
is current is refused before anything launches (DFLASH2_ERR_INVALID_ARG).  The
refusal needs a second device to provoke; the positive case runs anywhere."""
import numpy as np
import pytest
import torch

import oracle
from draft_selection_dflash2_gb300 import api, synth
from gpu_common import bf, handle, host  # noqa: F401

pytestmark = pytest.mark.gpu


def test_calls_on_the_handles_device_run(handle):
    rng = np.random.default_rng(1)
    U = synth.logits_planted(rng, 8, 4096)
    torch.cuda.set_device(handle.device)
    vals, idx = api.topk(handle, bf(U))
    ov, oi = oracle.topk(U)
    assert np.array_equal(host(idx), oi) and np.array_equal(host(vals), ov)


@pytest.mark.skipif(torch.cuda.device_count() < 2, reason="needs a second CUDA device")
def test_calls_from_another_device_are_refused(handle):
    rng = np.random.default_rng(2)
    U = bf(synth.logits_planted(rng, 8, 4096))
    vals = torch.full((8, 16), -7.0, device=U.device)
    idx = torch.full((8, 16), -7, dtype=torch.int32, device=U.device)
    other = 1 if handle.device == 0 else 0
    torch.cuda.set_device(other)
    try:
        with pytest.raises(api.Dflash2Error) as e:
            api.topk(handle, U, vals=vals, idx=idx)
        assert e.value.status == -1
        with pytest.raises(api.Dflash2Error) as e:
            api.lmhead_topk_noalloc(handle, bf(synth.normal_bits(3, (16, 64))), bf(synth.normal_bits(4, (64, 64))))
        assert e.value.status == -1
    finally:
        torch.cuda.set_device(handle.device)
    assert (vals == -7.0).all() and (idx == -7).all()   # nothing ran
