"""Failure detection without a GPU fault.

Every wait in the library's kernels is bounded.  The self-test entry point runs
one kernel whose two waits nothing can satisfy (an mbarrier no thread arrives
on, a global word no one writes) with a short limit: both give up, the error
word gets DFLASH2_DEVERR_TIMEOUT, the kernel returns normally and the context
stays usable for the next call.  Host-side argument errors answer before
anything launches."""
import time

import numpy as np
import pytest
import torch

import oracle
from draft_selection_dflash2_gb300 import api, synth
from gpu_common import bf, handle, host  # noqa: F401

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("limit_ms", [1, 20])
def test_unsatisfied_waits_give_up_and_the_context_survives(handle, limit_ms):
    assert handle.device_error() == 0
    words = torch.zeros(2, dtype=torch.int32, device="cuda")
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    api.selftest_wait_timeout(handle, limit_ms * 1_000_000, words)
    torch.cuda.synchronize()
    elapsed = time.perf_counter() - t0
    res = int(host(words)[1])
    assert res == 4, f"result word {res}: bit 2 = the kernel returned, bits 0/1 = a wait was satisfied"
    assert handle.device_error() == api.DEVERR_TIMEOUT
    assert 2 * limit_ms * 1e-3 <= elapsed < 1.0 + 2 * limit_ms * 1e-3
    # the context is intact: a regular call runs and agrees with the oracle
    rng = np.random.default_rng(limit_ms)
    U = synth.logits_planted(rng, 16, 8192)
    vals, idx = api.topk(handle, bf(U))
    ov, oi = oracle.topk(U)
    assert np.array_equal(host(idx), oi) and np.array_equal(host(vals), ov)
    assert handle.device_error() == 0


def test_selftest_rejects_limits_beyond_the_library_bound(handle):
    words = torch.zeros(2, dtype=torch.int32, device="cuda")
    for bad in (0, 3_000_000_000):
        with pytest.raises(api.Dflash2Error) as e:
            api.selftest_wait_timeout(handle, bad, words)
        assert e.value.status == -1


def test_argument_errors_launch_nothing(handle):
    # each refused call leaves its outputs untouched
    rng = np.random.default_rng(3)
    U = bf(synth.logits_planted(rng, 8, 4096))
    vals = torch.full((8, 16), -7.0, device="cuda")
    idx = torch.full((8, 16), -7, dtype=torch.int32, device="cuda")
    for kw, status in ((dict(k=8), -2), (dict(V=8), -2)):
        with pytest.raises(api.Dflash2Error) as e:
            api.topk(handle, U, vals=vals, idx=idx, **kw)
        assert e.value.status == status
    with pytest.raises(api.Dflash2Error) as e:
        api.topk(handle, U[:, 1:], vals=vals, idx=idx)     # logits 2 bytes off 16-byte alignment
    assert e.value.status == -3
    torch.cuda.synchronize()
    assert (vals == -7.0).all() and (idx == -7).all()
