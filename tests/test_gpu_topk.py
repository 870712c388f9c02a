"""Top-16 kernel vs the oracle: indices and values bit-exact (ties -> lowest id)."""
import numpy as np
import pytest

import oracle
from draft_selection_dflash2_gb300 import api, synth
from gpu_common import bf, handle, host  # noqa: F401

pytestmark = pytest.mark.gpu


def run(h, bits, V=None):
    vals, idx = api.topk(h, bf(bits), V=V)
    return host(vals), host(idx)


def check(h, bits, V=None):
    gv, gi = run(h, bits, V)
    ov, oi = oracle.topk(bits, V=V)
    assert np.array_equal(gi, oi), f"idx mismatch in {np.where((gi != oi).any(1))[0][:8]}"
    assert np.array_equal(gv, ov, equal_nan=True)   # a row of NaN ranks NaN logits (lowest ids first)
    assert h.device_error() == 0


@pytest.mark.parametrize("rows,V", [(8, 4096), (1, 16), (3, 17), (5, 4099), (16, 151936), (40, 50000),
                                    (300, 8200)])
def test_topk_planted(handle, rows, V):
    # the leading dimension is padded to a multiple of 8 (16-byte rows); the
    # ragged tail V % 8 is read with scalar loads
    rng = np.random.default_rng(rows * 7 + V)
    ld = (V + 7) // 8 * 8
    bits = synth.logits_planted(rng, rows, V, ld=ld)
    if ld == V:
        check(handle, bits)
    else:
        gv, gi = run(handle, bits, V=V)
        ov, oi = oracle.topk(bits, V=V)
        assert np.array_equal(gi, oi) and np.array_equal(gv, ov)


def test_topk_zipf_qwen3_4b_head(handle):
    rng = np.random.default_rng(1)
    check(handle, synth.logits_zipf(rng, 16, 151936))


def test_topk_padded_leading_dimension(handle):
    rng = np.random.default_rng(2)
    V, ld = 4099, 4112
    bits = synth.logits_planted(rng, 6, V, ld=ld)
    bits[:, V:] = synth.bf16_bits(np.full(ld - V, 100.0, np.float32))  # must never be read
    gv, gi = run(handle, bits, V=V)
    ov, oi = oracle.topk(bits, V=V)
    assert np.array_equal(gi, oi) and np.array_equal(gv, ov)


def test_topk_ties_everywhere(handle):
    rng = np.random.default_rng(3)
    vals = rng.choice(np.array([-1.0, 0.0, 0.5, 2.0], np.float32), size=(12, 30000))
    check(handle, synth.bf16_bits(vals))


def test_topk_all_equal_and_signed_zero(handle):
    rows = np.zeros((4, 9000), np.float32)
    rows[1, ::2] = -0.0
    rows[2] = -np.inf
    rows[2, 8000] = -0.0
    rows[3, 100:200] = np.nan
    check(handle, synth.bf16_bits(rows))


def test_topk_adversarial_ascending_rows(handle):
    # every element beats the running threshold: exercises the candidate buffer folds
    base = np.linspace(-8, 8, 40000, dtype=np.float32)
    rows = np.stack([base, base[::-1], np.roll(base, 12345)])
    check(handle, synth.bf16_bits(rows))


def test_topk_edge_rows_on_the_whole_row_path(handle):
    # enough rows that each CTA takes whole rows (the persistent form with a
    # ranking warp): ties, signed zeros, NaN runs, all -inf but one, ascending
    # and descending ramps, planted rows, interleaved so that consecutive rows
    # of one CTA differ in kind
    V = 9000
    rng = np.random.default_rng(6)
    kinds = []
    kinds.append(rng.choice(np.array([-1.0, 0.0, 0.5, 2.0], np.float32), size=V))
    z = np.zeros(V, np.float32)
    z[::2] = -0.0
    kinds.append(z)
    n = rng.standard_normal(V).astype(np.float32)
    n[100:4000] = np.nan
    kinds.append(n)
    f = np.full(V, -np.inf, np.float32)
    f[8000] = -0.0
    kinds.append(f)
    kinds.append(np.linspace(-8, 8, V, dtype=np.float32))
    kinds.append(np.linspace(8, -8, V, dtype=np.float32))
    kinds.append(np.full(V, np.nan, np.float32))
    rows = np.stack([kinds[i % len(kinds)] if i % 3 else rng.standard_normal(V).astype(np.float32)
                     for i in range(1024)])
    check(handle, synth.bf16_bits(rows))


@pytest.mark.parametrize("rows,V", [(3, 1_000_000), (2, 6_500_000)])
def test_topk_long_rows(handle, rows, V):
    # V = 1M: each row is split over a cluster until a segment fits the group
    # history (196,608 logits); V = 6.5M exceeds it even over 16 CTAs and
    # takes the running-threshold stream
    rng = np.random.default_rng(V + rows)
    check(handle, synth.logits_planted(rng, rows, V))


def test_topk_many_rows_multiple_launches(handle):
    rng = np.random.default_rng(4)
    bits = synth.bf16_bits(rng.standard_normal((70000, 24)).astype(np.float32))
    check(handle, bits)


def test_topk_batch_sweep_full_size_sampled_rows(handle):
    # B = 256, L = 16, V = 151936 (1.25 GB of logits): the launch configuration
    # the benchmark times; the oracle checks 48 sampled rows.
    import torch
    B, L, V = 256, 16, 151936
    rows = B * L
    rng = np.random.default_rng(5)
    dev_logits = torch.empty((rows, V), dtype=torch.bfloat16, device="cuda:0")
    picked = np.sort(rng.choice(rows, 48, replace=False))
    host_rows = {}
    for r0 in range(0, rows, 512):
        chunk = synth.logits_planted(np.random.default_rng(1000 + r0), 512, V)
        dev_logits[r0:r0 + 512] = bf(chunk)
        for r in picked[(picked >= r0) & (picked < r0 + 512)]:
            host_rows[int(r)] = chunk[r - r0]
    vals, idx = api.topk(handle, dev_logits)
    gv, gi = host(vals), host(idx)
    sample = np.stack([host_rows[int(r)] for r in picked])
    ov, oi = oracle.topk(sample)
    assert np.array_equal(gi[picked], oi) and np.array_equal(gv[picked], ov)
    # every row: sorted descending, ids distinct and in range
    assert np.all(np.diff(gv, axis=1) <= 0)
    assert gi.min() >= 0 and gi.max() < V
    srt = np.sort(gi, axis=1)
    assert np.all(srt[:, 1:] != srt[:, :-1])
    del dev_logits


def test_topk_rejects_bad_arguments(handle):
    import torch
    x = torch.zeros((4, 64), dtype=torch.bfloat16, device="cuda:0")
    with pytest.raises(api.Dflash2Error) as e:
        api.topk(handle, x, k=8)
    assert e.value.status == -2
    with pytest.raises(api.Dflash2Error) as e:
        api.topk(handle, x[:, 1:])          # misaligned base pointer
    assert e.value.status == -3
    with pytest.raises(api.Dflash2Error) as e:
        api.topk(handle, x, V=8)            # V < 16
    assert e.value.status == -2
