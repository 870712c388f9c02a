"""Shared helpers for the GPU parity tests (numpy bf16 bits <-> CUDA tensors)."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

K = 16


def dev():
    return torch.device("cuda:0")


def bf(a):
    """numpy uint16 bf16 bits -> CUDA bfloat16 tensor (same bytes)."""
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(dev()).view(torch.bfloat16)


def i32(a):
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32)).to(dev())


def f32(a):
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(dev())


def host(t):
    t = t.detach()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).cpu().numpy().view(np.uint16)
    return t.cpu().numpy()


def assert_close(got, ref, rtol=1e-3, atol=1e-4, what=""):
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    err = np.abs(got - ref)
    bad = err > atol + rtol * np.abs(ref)
    assert not bad.any(), (f"{what}: {bad.sum()} of {bad.size} outside rtol={rtol} atol={atol}; "
                           f"max abs err {err.max():.3e}")


@pytest.fixture(scope="session")
def handle():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from draft_selection_dflash2_gb300 import api, build
    build.build()
    torch.cuda.set_device(0)
    h = api.Handle(0)
    yield h
    h.close()
