"""The two-tap conv fused into its producing GEMM, on the GPU, against the
oracle (fp32 accumulation over K products: 1e-3 rel / 1e-4 abs on fp32 output,
one bf16 ulp + 1e-4 abs on bf16 output), and bit for bit against the unfused path (the
conv kernel on an exact x) where the GEMM output is exact."""
import numpy as np
import pytest
import torch

import oracle
from draft_selection_dflash2_gb300 import api, synth
from gpu_common import assert_close, bf, f32, handle, host  # noqa: F401

pytestmark = pytest.mark.gpu


def inputs(seed, B, L, K, d, bias=False):
    c = synth.conv_inputs(seed, B, L, d, with_bias=bias)
    A = synth.normal_bits(seed + 1, (B, L, K))
    W = synth.normal_bits(seed + 2, (d, K), std=1.0 / np.sqrt(K))
    h = synth.normal_bits(seed + 3, (B, L, d))
    return c, A, W, h


def run(hd, c, A, W, h, y_fp32=True):
    y, cw = api.gemm_conv2tap(hd, bf(A), bf(W), bf(c.x_prev), bf(h), bf(c.k0), bf(c.k1), bf(c.W_c),
                              b_c=None if c.b_c is None else f32(c.b_c), y_fp32=y_fp32)
    return host(y), host(cw)


@pytest.mark.parametrize("B,L,K,d,bias", [(2, 16, 256, 512, False), (3, 5, 192, 256, True), (1, 1, 64, 64, False),
                                          (4, 7, 512, 2560, True), (2, 64, 128, 320, False),
                                          (8, 16, 5120, 5120, False), (1280, 16, 64, 512, True)])
def test_fused_conv_matches_oracle(handle, B, L, K, d, bias):
    # (1280, 16, ...): 160 row tiles, more correction tiles than SMs
    c, A, W, h = inputs(B * 31 + L + K, B, L, K, d, bias)
    y, cw = run(handle, c, A, W, h)
    assert handle.device_error() == 0
    oy = oracle.gemm_conv2tap(A, W, c.x_prev, h, c.k0, c.k1, c.W_c, b_c=c.b_c)
    assert_close(y, oy, rtol=1e-3, atol=1e-4, what="y")


def bf16_ulp(v):
    e = np.floor(np.log2(np.maximum(np.abs(v), 2.0**-126)))
    return 2.0 ** (e - 7)


def test_fused_conv_bf16_within_one_ulp(handle):
    c, A, W, h = inputs(3, 4, 16, 1024, 2560)
    y, _ = run(handle, c, A, W, h, y_fp32=False)
    oy = oracle.gemm_conv2tap(A, W, c.x_prev, h, c.k0, c.k1, c.W_c)
    got = synth.bf16_to_f32(y).astype(np.float64)
    assert np.all(np.abs(got - oy) <= bf16_ulp(oy) + 1e-4)


def exact_case(seed, B, L, K, d):
    """A, W, hs in {-1, 0, 1} and W_c in {-1, 0, 1} / 64: x = A W^T and the correction
    are exact in any summation order, and x is exact in bf16 (|x| <= K <= 256)."""
    rng = np.random.default_rng(seed)
    c = synth.conv_inputs(seed, B, L, d)
    Ai, Wi = rng.integers(-1, 2, (B, L, K)), rng.integers(-1, 2, (d, K))
    bits = lambda a: synth.bf16_bits(np.asarray(a, np.float32))          # noqa: E731
    h = bits(rng.integers(-1, 2, (B, L, d)))
    c.W_c = bits(rng.integers(-1, 2, c.W_c.shape) / 64.0)
    return c, bits(Ai), bits(Wi), h, bits(Ai @ Wi.T)


@pytest.mark.parametrize("B,L,K,d", [(4, 16, 128, 256), (3, 7, 192, 512)])
def test_fused_conv_equals_unfused_on_exact_data(handle, B, L, K, d):
    c, A, W, h, x = exact_case(B + L, B, L, K, d)
    for y_fp32 in (True, False):
        y, _ = run(handle, c, A, W, h, y_fp32=y_fp32)
        yu = host(api.conv2tap(handle, bf(x), bf(c.x_prev), bf(c.k0), bf(c.k1), bf(c.W_c), hs=bf(h),
                               y_fp32=y_fp32))
        assert np.array_equal(y.view(np.uint8), yu.view(np.uint8))


def test_fused_conv_shift_crosses_warps(handle):
    # k0 = 0, k1 = 1, no correction: y is x one position later; with L = 7 a tile holds
    # 126 rows, and rows 32, 64 and 96 take x_{t-1} from the previous warp
    B, L, K, d = 18, 7, 128, 256
    c, A, W, h, x = exact_case(5, B, L, K, d)
    c.k0[:] = 0
    c.k1[:] = synth.bf16_bits(np.float32(1.0))
    c.W_c[:] = 0
    y, _ = run(handle, c, A, W, h, y_fp32=True)
    xf = synth.bf16_to_f32(x)
    assert np.array_equal(y[:, 1:], xf[:, :-1])
    assert np.array_equal(y[:, 0], synth.bf16_to_f32(c.x_prev))


def test_fused_conv_workspace_too_small(handle):
    c, A, W, h = inputs(4, 1, 4, 64, 64)
    small = torch.empty((3, 8), dtype=torch.float32, device="cuda")
    with pytest.raises(api.Dflash2Error, match="WORKSPACE"):
        api.gemm_conv2tap(handle, bf(A), bf(W), bf(c.x_prev), bf(h), bf(c.k0), bf(c.k1), bf(c.W_c), c_work=small)
    # the correction (4 rows x 8 columns of fp32), then a counter per row, rounded to 16 bytes
    assert api.gemm_conv2tap_workspace(handle, 1, 4, 64) == 4 * 8 * 4 + 16
