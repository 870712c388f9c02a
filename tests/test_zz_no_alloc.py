"""The allocation-free LM-head entry point against the regular one.

dflash2_lmhead_topk_noalloc serves callers that cannot allocate device memory
(an engine whose memory pool owns the whole GPU, or a serving loop that must
not pay the device synchronisation a cudaMalloc/cudaFree can cause): its
scratch is a fixed array inside the library instead of a caller-provided
workspace.  Run through the C ABI twice in a row, it must give exactly what
dflash2_lmhead_topk gives on the same inputs, since the same kernels run;
this file is collected last so that a stop at the first failure has already
run every other test."""
import numpy as np
import pytest

from draft_selection_dflash2_gb300 import api, synth
from gpu_common import bf, handle, host  # noqa: F401

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("M,V,d", [(256, 20000, 512), (1024, 151936, 5120)])
def test_noalloc_matches_workspace_call_twice(handle, M, V, d):
    hid = bf(synth.normal_bits(40 + M, (M, d)))
    W = bf(synth.normal_bits(41 + M, (V, d), std=0.02))
    ref_v, ref_i = api.lmhead_topk(handle, hid, W)
    ref_v, ref_i = host(ref_v), host(ref_i)
    for _ in range(2):
        v, i = api.lmhead_topk_noalloc(handle, hid, W)
        assert np.array_equal(host(i), ref_i)
        assert np.array_equal(host(v).view(np.uint32), ref_v.view(np.uint32))
    assert handle.device_error() == 0


def test_noalloc_rejects_problems_beyond_the_fixed_scratch(handle):
    import torch
    # 40000 rows x 1 run x 16 keys x 8 bytes > 4 MiB of fixed scratch
    hid = torch.zeros((40000, 64), dtype=torch.bfloat16, device="cuda")
    W = torch.zeros((4096, 64), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(api.Dflash2Error) as e:
        api.lmhead_topk_noalloc(handle, hid, W)
    assert e.value.status == -7
