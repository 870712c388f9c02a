"""Seeded synthetic inputs for the DFlash 2 draft-block head.

This module is the only thing the CUDA path and the CPU oracle share.  It
draws random tensors with the shapes and value distributions of the workloads
the pages describe (block of 16 drafted positions, top-16 candidates, 256-D
selector embeddings, a ~152k vocabulary) and holds none of the method's
arithmetic.  The pages measure on GSM8K / MATH-500 / HumanEval / MBPP /
MT-Bench with trained drafters; none of those are available, so these seeded
draws stand in for them.  Nothing here is derived from any benchmark item.

bf16 tensors are returned as numpy uint16 bit patterns (round-to-nearest-even
from float32), so that both sides read the same bytes.
"""
from dataclasses import dataclass, field

import numpy as np

# ---------------------------------------------------------------------------
# dtype helpers
# ---------------------------------------------------------------------------


def bf16_bits(x) -> np.ndarray:
    """float32 -> bf16 bit patterns, round to nearest even (NaN kept quiet)."""
    f = np.ascontiguousarray(x, dtype=np.float32)
    u = f.view(np.uint32)
    rounding = np.uint32(0x7FFF) + ((u >> np.uint32(16)) & np.uint32(1))
    out = ((u + rounding) >> np.uint32(16)).astype(np.uint16)
    nan = np.isnan(f)
    if nan.any():
        out[nan] = np.uint16(0x7FC0)
    return out


def bf16_to_f32(bits) -> np.ndarray:
    b = np.ascontiguousarray(bits, dtype=np.uint16)
    return (b.astype(np.uint32) << np.uint32(16)).view(np.float32)


def _normal_bits(rng, shape, mean=0.0, std=1.0, chunk=1 << 26) -> np.ndarray:
    """N(mean, std^2) drawn in float32 and rounded to bf16, in chunks to bound memory."""
    n = int(np.prod(shape))
    out = np.empty(n, np.uint16)
    for s in range(0, n, chunk):
        e = min(n, s + chunk)
        v = rng.standard_normal(e - s, dtype=np.float32)
        if std != 1.0:
            v *= np.float32(std)
        if mean != 0.0:
            v += np.float32(mean)
        out[s:e] = bf16_bits(v)
    return out.reshape(shape)


# ---------------------------------------------------------------------------
# drafter logits U
# ---------------------------------------------------------------------------


def logits_planted(rng, rows: int, V: int, plant: float = 4.0, ld: int = None) -> np.ndarray:
    """U ~ N(0, 1) rounded to bf16, plus +plant at one uniform id per row.

    Returns uint16 [rows, ld] (columns >= V, if any, hold -inf padding)."""
    ld = V if ld is None else ld
    out = np.empty((rows, ld), np.uint16)
    planted = rng.integers(0, V, size=rows)
    for s in range(0, rows, 256):
        e = min(rows, s + 256)
        v = rng.standard_normal((e - s, V), dtype=np.float32)
        v[np.arange(e - s), planted[s:e]] += np.float32(plant)
        out[s:e, :V] = bf16_bits(v)
    if ld > V:
        out[:, V:] = np.uint16(0xFF80)
    return out


def zipf_bias(rng, V: int, s: float = 1.1) -> np.ndarray:
    """Log-Zipf prior: bias(v) = -s * ln(1 + pi(v)) for a seeded permutation pi."""
    perm = rng.permutation(V)
    return (-s * np.log1p(perm.astype(np.float64))).astype(np.float32)


def logits_zipf(rng, rows: int, V: int, sigma: float = 2.0, s: float = 1.1) -> np.ndarray:
    """U ~ N(0, sigma^2) + Zipf(s)-ranked bias (shared by all rows), bf16 [rows, V]."""
    bias = zipf_bias(rng, V, s)
    out = np.empty((rows, V), np.uint16)
    for r0 in range(0, rows, 256):
        r1 = min(rows, r0 + 256)
        v = rng.standard_normal((r1 - r0, V), dtype=np.float32)
        v *= np.float32(sigma)
        v += bias[None, :]
        out[r0:r1] = bf16_bits(v)
    return out


# ---------------------------------------------------------------------------
# selector / conv / head parameters
# ---------------------------------------------------------------------------


@dataclass
class SelectorInputs:
    U: np.ndarray            # uint16 [B, L, V]
    h: np.ndarray            # uint16 [B, L, d]
    W_H: np.ndarray          # uint16 [r, d]
    b_H: np.ndarray          # float32 [r]
    A: np.ndarray            # uint16 [V, r]
    Bt: np.ndarray           # uint16 [V, r]
    last_verified: np.ndarray  # int32 [B]
    B: int = 0
    L: int = 0
    V: int = 0
    d: int = 0
    r: int = 256


def selector_inputs(seed: int, B: int, L: int, V: int, d: int, r: int = 256,
                    logits: str = "planted", emb_std: float = 0.02,
                    gate_std: float = 0.02) -> SelectorInputs:
    """Inputs of the top-16 + pair-score + walk stages.

    logits: "planted" (N(0,1) + one +4 per position) or "zipf" (N(0,2) +
    Zipf(1.1)-ranked bias).  emb_std = 0.25 gives the stress set in which the
    pair term is large enough to change choices."""
    rng = np.random.default_rng(seed)
    if logits == "planted":
        U = logits_planted(rng, B * L, V)
    elif logits == "zipf":
        U = logits_zipf(rng, B * L, V)
    else:
        raise ValueError(logits)
    U = U.reshape(B, L, V)
    h = _normal_bits(rng, (B, L, d))
    W_H = _normal_bits(rng, (r, d), std=gate_std)
    b_H = np.zeros(r, np.float32)
    A = _normal_bits(rng, (V, r), std=emb_std)
    Bt = _normal_bits(rng, (V, r), std=emb_std)
    last_verified = rng.integers(0, V, size=B).astype(np.int32)
    return SelectorInputs(U=U, h=h, W_H=W_H, b_H=b_H, A=A, Bt=Bt,
                          last_verified=last_verified, B=B, L=L, V=V, d=d, r=r)


@dataclass
class ConvInputs:
    x: np.ndarray        # uint16 [B, L, d]
    x_prev: np.ndarray   # uint16 [B, d]
    k0: np.ndarray       # uint16 [d]
    k1: np.ndarray       # uint16 [d]
    W_c: np.ndarray      # uint16 [2d/16, d]
    b_c: np.ndarray = None  # float32 [2d/16] or None


def conv_inputs(seed: int, B: int, L: int, d: int, w_std: float = 0.01,
                with_bias: bool = False) -> ConvInputs:
    """x, x_prev ~ N(0,1); k0, k1 ~ N(0.5, 0.1); W_c ~ N(0, w_std^2); all bf16."""
    rng = np.random.default_rng(seed)
    x = _normal_bits(rng, (B, L, d))
    x_prev = _normal_bits(rng, (B, d))
    k0 = _normal_bits(rng, (d,), mean=0.5, std=0.1)
    k1 = _normal_bits(rng, (d,), mean=0.5, std=0.1)
    W_c = _normal_bits(rng, (2 * (d // 16), d), std=w_std)
    b_c = rng.standard_normal(2 * (d // 16), dtype=np.float32) * np.float32(0.05) if with_bias else None
    return ConvInputs(x=x, x_prev=x_prev, k0=k0, k1=k1, W_c=W_c, b_c=b_c)


def conv_layer_params(seed: int, d: int, w_std: float = 0.01):
    """(k0, k1, W_c) for one conv application."""
    rng = np.random.default_rng(seed)
    k0 = _normal_bits(rng, (d,), mean=0.5, std=0.1)
    k1 = _normal_bits(rng, (d,), mean=0.5, std=0.1)
    W_c = _normal_bits(rng, (2 * (d // 16), d), std=w_std)
    return k0, k1, W_c


def normal_bits(seed: int, shape, mean=0.0, std=1.0) -> np.ndarray:
    """Seeded N(mean, std^2) tensor as bf16 bits."""
    return _normal_bits(np.random.default_rng(seed), shape, mean=mean, std=std)


# ---------------------------------------------------------------------------
# synthetic target logits with planted argmax agreement
# ---------------------------------------------------------------------------


def target_planted(seed: int, draft_tok: np.ndarray, V: int, agree: float = 0.85,
                   plant: float = 8.0) -> np.ndarray:
    """Target logits [B, L+1, V] bf16: N(0,1) noise; at each drafted position t
    a seeded Bernoulli(agree) decides whether +plant goes on draft_tok[b, t]
    (agreement) or on a uniform id != draft_tok[b, t]; the bonus row t = L gets
    +plant at a uniform id.  draft_tok is an input (whoever drafted it)."""
    rng = np.random.default_rng(seed)
    dt = np.asarray(draft_tok, np.int64)
    B, L = dt.shape
    agreeing = rng.random((B, L)) < agree
    other = rng.integers(0, V - 1, size=(B, L))
    other = other + (other >= dt)          # uniform over ids != draft
    where = np.where(agreeing, dt, other)
    bonus = rng.integers(0, V, size=(B, 1))
    where = np.concatenate([where, bonus], axis=1)
    out = np.empty((B, L + 1, V), np.uint16)
    for b in range(B):
        v = rng.standard_normal((L + 1, V), dtype=np.float32)
        v[np.arange(L + 1), where[b]] += np.float32(plant)
        out[b] = bf16_bits(v)
    return out


def planted_path(seed: int, B: int, L: int, V: int, mu: float = 3.0, sigma: float = 1.0, K: int = 16):
    """Pair scores with a planted true slot path, for comparing walks.

    Per sequence: 16 distinct candidate ids per position (uniform in [0, V)),
    a uniform true slot p_t per position, and S f32 [B, L, 16, 16] of
    N(0, sigma^2) noise plus mu on the true transition: at t = 0 on column p_0
    of every row (the rows of position 0 are equal), at t >= 1 on
    (p_{t-1}, p_t).  Returns (S, cand_idx, true_slot, true_tok)."""
    rng = np.random.default_rng(seed)
    cand = np.empty((B, L, K), np.int32)
    for b in range(B):
        for t in range(L):
            cand[b, t] = rng.choice(V, K, replace=V < K)
    p = rng.integers(0, K, (B, L))
    S = (rng.standard_normal((B, L, K, K), dtype=np.float32) * np.float32(sigma)).astype(np.float32)
    S[:, 0] = S[:, 0, :1, :]
    bb = np.arange(B)
    S[bb, 0, :, p[:, 0]] += np.float32(mu)
    for t in range(1, L):
        S[bb, t, p[:, t - 1], p[:, t]] += np.float32(mu)
    tok = np.take_along_axis(cand, p[:, :, None], axis=2)[:, :, 0]
    return S, cand, p.astype(np.int32), tok.astype(np.int32)


def target_noise(seed: int, B: int, L: int, V: int, std: float = 1.0) -> np.ndarray:
    """Unplanted target logits [B, L+1, V], N(0, std^2) bf16."""
    return _normal_bits(np.random.default_rng(seed), (B, L + 1, V), std=std)


# ---------------------------------------------------------------------------
# named workloads (shapes and distributions of the pages' setting)
# ---------------------------------------------------------------------------


@dataclass(frozen=True)
class Workload:
    name: str
    B: int
    L: int
    V: int
    d: int
    r: int = 256
    K: int = 16
    logits: str = "planted"
    temperatures: tuple = (0.0,)
    conv_apps: int = 0
    verify: bool = False
    notes: str = ""


TINY_SELECTOR = Workload("tiny selector B=1 L=8 V=4096 d=512", B=1, L=8, V=4096, d=512)
QWEN3_4B_HEAD = Workload("Qwen3-4B-shaped head B=1 L=16 V=151936 d=2560", B=1, L=16, V=151936,
                         d=2560, logits="zipf", temperatures=(0.0, 1.0), conv_apps=1)
BATCH_SWEEP = tuple(Workload(f"batch sweep B={b} L=16 V=151936 d=5120", B=b, L=16, V=151936,
                             d=5120) for b in (1, 8, 32, 128, 256))
FULL_CYCLE = Workload("full draft-verify cycle B=128 L=16 V=151936 d=5120", B=128, L=16,
                      V=151936, d=5120, temperatures=(0.0, 1.0), conv_apps=10, verify=True)
LMHEAD = dict(name="fused LM-head top-16 M=1024 d=5120 V=151936", M=1024, d=5120, V=151936)
