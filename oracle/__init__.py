"""CPU oracle for the DFlash 2 draft-block head -- TEST INFRASTRUCTURE ONLY.

A plain, slow, obviously-correct restatement of "DFlash 2: Keep Drafting
Parallel" in C++17 (fp64), wrapped here with ctypes over numpy arrays.  Only the
tests, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline leg may
import this package; the product path never does.  It shares no code with the
CUDA library.  bf16 tensors are passed as uint16 bit patterns.

Every function here is pinned by ``tests/test_oracle_pins.py`` against
properties the pages and the mathematics fix (closed forms, special cases that
reduce to textbook routines, brute force on tiny inputs, published Philox
known-answer vectors).
"""
import ctypes
import os

import numpy as np

from . import build as _build

_lib = None


def _load():
    global _lib
    if _lib is None:
        path = _build.build()
        lib = ctypes.CDLL(path)
        P = ctypes.c_void_p
        I64 = ctypes.c_int64
        I = ctypes.c_int
        D = ctypes.c_double
        U64 = ctypes.c_uint64
        lib.oracle_philox4x32_10.argtypes = [P, P, P]
        lib.oracle_philox4x32_10.restype = None
        lib.oracle_uniform24.argtypes = [U64, U64, U64, ctypes.c_uint32, U64]
        lib.oracle_uniform24.restype = D
        lib.oracle_exp2_neg.argtypes = [ctypes.c_float]
        lib.oracle_exp2_neg.restype = ctypes.c_float
        lib.oracle_verify_weights.argtypes = [P, I64, D, P]
        lib.oracle_verify_weights.restype = U64
        lib.oracle_topk.argtypes = [P, I64, I64, I64, I, P, P, I]
        lib.oracle_topk.restype = None
        lib.oracle_gate.argtypes = [P, P, P, I64, I64, I64, P, I]
        lib.oracle_gate.restype = None
        lib.oracle_pair_scores.argtypes = [P, P, P, P, P, P, I64, I64, I64, I64, I64, P, I]
        lib.oracle_pair_scores.restype = I
        lib.oracle_gemm_conv2tap.argtypes = [P, P, P, P, P, P, P, P, I64, I64, I64, I64, P, I]
        lib.oracle_gemm_conv2tap.restype = None
        lib.oracle_pair_scores_proj.argtypes = [P, P, P, P, P, P, P, I64, I64, I64, I64, I64, I64, P, I]
        lib.oracle_pair_scores_proj.restype = I
        lib.oracle_walk.argtypes = [P, P, I64, I64, I64, D, U64, U64, P, P, P, P, I]
        lib.oracle_walk.restype = None
        lib.oracle_conv2tap.argtypes = [P, P, P, P, P, P, P, I64, I64, I64, P, I]
        lib.oracle_conv2tap.restype = None
        lib.oracle_verify.argtypes = [P, I64, P, P, P, P, I64, I64, I64, I64, D, U64, U64, P, P, P, I]
        lib.oracle_verify.restype = None
        lib.oracle_lmhead_topk.argtypes = [P, P, I64, I64, P, I64, I, P, P, I]
        lib.oracle_lmhead_topk.restype = None
        lib.oracle_walk_viterbi.argtypes = [P, P, I64, I64, I64, P, P, P, I]
        lib.oracle_walk_viterbi.restype = None
        lib.oracle_selector_eval.argtypes = [P, P, I64, I64, I64, P, P, P]
        lib.oracle_selector_eval.restype = None
        lib.oracle_threads.argtypes = [I]
        lib.oracle_threads.restype = I
        _lib = lib
    return _lib


def _p(a):
    return None if a is None else ctypes.c_void_p(a.ctypes.data)


def _c(a, dtype):
    if a is None:
        return None
    return np.ascontiguousarray(a, dtype=dtype)


def default_threads() -> int:
    return int(os.environ.get("DFLASH2_ORACLE_THREADS", os.cpu_count() or 1))


def threads_used(nthreads: int) -> int:
    return int(_load().oracle_threads(nthreads))


def philox4x32_10(ctr, key):
    ctr = _c(ctr, np.uint32)
    key = _c(key, np.uint32)
    out = np.zeros(4, np.uint32)
    _load().oracle_philox4x32_10(_p(ctr), _p(key), _p(out))
    return out


def uniform24(seed, b, t, stream, offset=0):
    return float(_load().oracle_uniform24(seed, b, t, stream, offset))


def exp2_neg(x: float) -> float:
    """The walk's fp32 2^x (x <= 0): Cody-Waite reduction + degree-7 Taylor polynomial."""
    return float(_load().oracle_exp2_neg(float(x)))


def verify_weights(row_bits, temperature):
    """Reading R21: fixed-point weights of one target row -> (W uint64 [V], Z)."""
    row = _c(row_bits, np.uint16)
    W = np.zeros(row.shape[0], np.uint64)
    Z = _load().oracle_verify_weights(_p(row), row.shape[0], float(temperature), _p(W))
    return W, int(Z)


def topk(logits_bits, k=16, V=None, nthreads=None):
    """logits_bits: uint16 [rows, ld]; returns (vals f32 [rows,k], idx i32 [rows,k])."""
    x = _c(logits_bits, np.uint16)
    rows, ld = x.shape
    V = ld if V is None else V
    vals = np.zeros((rows, k), np.float32)
    idx = np.zeros((rows, k), np.int32)
    _load().oracle_topk(_p(x), rows, V, ld, k, _p(vals), _p(idx), nthreads or default_threads())
    return vals, idx


def gate(h_bits, W_H_bits, b_H=None, nthreads=None):
    """h: uint16 [M, d]; W_H: uint16 [r, d]; b_H: f32 [r] or None -> H f64 [M, r]."""
    h = _c(h_bits, np.uint16)
    W = _c(W_H_bits, np.uint16)
    b = _c(b_H, np.float32)
    M, d = h.shape
    r = W.shape[0]
    H = np.zeros((M, r), np.float64)
    _load().oracle_gate(_p(h), _p(W), _p(b), M, d, r, _p(H), nthreads or default_threads())
    return H


def pair_scores(cand_idx, cand_val, last_verified, H, A_bits, B_bits, nthreads=None):
    """cand_*: [B, L, K]; H: f64 [B, L, r]; A, B: uint16 [V, r] -> (S f64 [B,L,K,K], bad_id flag)."""
    ci = _c(cand_idx, np.int32)
    cv = _c(cand_val, np.float32)
    lv = _c(last_verified, np.int32)
    Hh = _c(H, np.float64)
    A = _c(A_bits, np.uint16)
    Bt = _c(B_bits, np.uint16)
    B, L, K = ci.shape
    V, r = A.shape
    S = np.zeros((B, L, K, K), np.float64)
    bad = _load().oracle_pair_scores(_p(ci), _p(cv), _p(lv), _p(Hh), _p(A), _p(Bt), B, L, K, r, V,
                                     _p(S), nthreads or default_threads())
    return S, bool(bad)


def pair_scores_proj(cand_idx, cand_val, last_verified, H, E_bits, WA_bits, WB_bits, nthreads=None):
    """Projection form (reading R19): cand_*: [B, L, K]; H: f64 [B, L, r]; E: uint16 [V, d];
    W_A, W_B: uint16 [r, d] -> (S f64 [B, L, K, K], bad_id flag)."""
    ci = _c(cand_idx, np.int32)
    cv = _c(cand_val, np.float32)
    lv = _c(last_verified, np.int32)
    Hh = _c(H, np.float64)
    E = _c(E_bits, np.uint16)
    WA = _c(WA_bits, np.uint16)
    WB = _c(WB_bits, np.uint16)
    B, L, K = ci.shape
    V, d = E.shape
    r = WA.shape[0]
    S = np.zeros((B, L, K, K), np.float64)
    bad = _load().oracle_pair_scores_proj(_p(ci), _p(cv), _p(lv), _p(Hh), _p(E), _p(WA), _p(WB), B, L, K, r, V, d,
                                          _p(S), nthreads or default_threads())
    return S, bool(bad)


def walk(S, cand_idx, temperature=0.0, seed=0, offset=0, nthreads=None):
    """S: f32 [B, L, K, K] -> (draft_tok, draft_slot, draft_q, margin [B, L] per step)."""
    Sf = _c(S, np.float32)
    ci = _c(cand_idx, np.int32)
    B, L, K, _ = Sf.shape
    tok = np.zeros((B, L), np.int32)
    slot = np.zeros((B, L), np.int32)
    q = np.zeros((B, L, K), np.float32)
    margin = np.zeros((B, L), np.float64)
    _load().oracle_walk(_p(Sf), _p(ci), B, L, K, float(temperature), seed, offset, _p(tok), _p(slot),
                        _p(q), _p(margin), nthreads or default_threads())
    return tok, slot, q, margin


def walk_viterbi(S, cand_idx, nthreads=None):
    """Exact best path over S f32 [B, L, K, K] (reading R17) -> (draft_tok, draft_slot, score [B])."""
    Sf = _c(S, np.float32)
    ci = _c(cand_idx, np.int32)
    B, L, K, _ = Sf.shape
    tok = np.zeros((B, L), np.int32)
    slot = np.zeros((B, L), np.int32)
    score = np.zeros((B,), np.float32)
    _load().oracle_walk_viterbi(_p(Sf), _p(ci), B, L, K, _p(tok), _p(slot), _p(score), nthreads or default_threads())
    return tok, slot, score


def selector_eval(gt, cand_idx):
    """Table 1 evaluation (reading R18): gt int32 [B, L], cand_idx int32 [B, L, K] ->
    (accept1 [B], accept16 [B], counts int64 [L, 4] = (n1, hit1, n16, hit16) per position)."""
    g = _c(gt, np.int32)
    ci = _c(cand_idx, np.int32)
    B, L, K = ci.shape
    a1 = np.zeros((B,), np.int32)
    a16 = np.zeros((B,), np.int32)
    counts = np.zeros((L, 4), np.int64)
    _load().oracle_selector_eval(_p(g), _p(ci), B, L, K, _p(a1), _p(a16), _p(counts))
    return a1, a16, counts


def closed_form_accept(recalls):
    """Expected acceptance length 1 + sum_k prod_{t<=k} r_t for conditional per-position
    acceptance rates r_t (Table 1's note: the verifier's next token is included)."""
    total, prod = 1.0, 1.0
    for r in recalls:
        prod *= float(r)
        total += prod
    return total


def conv2tap(x_bits, x_prev_bits, k0_bits, k1_bits, W_c_bits, b_c=None, h_bits=None, nthreads=None):
    """x: uint16 [B, L, d]; x_prev: [B, d]; k0, k1: [d]; W_c: [2d/16, d] -> y f64 [B, L, d]."""
    x = _c(x_bits, np.uint16)
    xp = _c(x_prev_bits, np.uint16)
    h = _c(h_bits, np.uint16)
    k0 = _c(k0_bits, np.uint16)
    k1 = _c(k1_bits, np.uint16)
    W = _c(W_c_bits, np.uint16)
    bc = _c(b_c, np.float32)
    B, L, d = x.shape
    y = np.zeros((B, L, d), np.float64)
    _load().oracle_conv2tap(_p(x), _p(xp), _p(h), _p(k0), _p(k1), _p(W), _p(bc), B, L, d, _p(y),
                            nthreads or default_threads())
    return y


def gemm_conv2tap(A_bits, W_bits, x_prev_bits, h_bits, k0_bits, k1_bits, W_c_bits, b_c=None, nthreads=None):
    """Conv fused into the producing GEMM (reading R20): A: uint16 [B, L, K]; W: uint16 [d, K];
    x_prev: uint16 [B, d]; h: uint16 [B, L, d] -> y f64 [B, L, d] with x = A W^T exact."""
    A = _c(A_bits, np.uint16)
    W = _c(W_bits, np.uint16)
    xp = _c(x_prev_bits, np.uint16)
    hh = _c(h_bits, np.uint16)
    k0, k1, Wc = _c(k0_bits, np.uint16), _c(k1_bits, np.uint16), _c(W_c_bits, np.uint16)
    bc = _c(b_c, np.float32)
    B, L, K = A.shape
    d = W.shape[0]
    y = np.zeros((B, L, d), np.float64)
    _load().oracle_gemm_conv2tap(_p(A), _p(W), _p(xp), _p(hh), _p(k0), _p(k1), _p(Wc), _p(bc), B, L, K, d, _p(y),
                                 nthreads or default_threads())
    return y


def verify(target_bits, draft_tok, draft_slot, draft_q, cand_idx, temperature=0.0, seed=0, offset=0,
           V=None, nthreads=None):
    """target: uint16 [B, L+1, ld] -> (accept_len [B], out_tok [B, L+1], margin [B, 2]).

    margin[:, 0]: smallest relative accept-test margin; margin[:, 1]: smallest
    draw margin relative to the total weight (both +inf at temperature 0).  At
    T > 0 the decisions are taken on reading R21's exact fixed-point weights."""
    tg = _c(target_bits, np.uint16)
    dt = _c(draft_tok, np.int32)
    ds = _c(draft_slot, np.int32)
    dq = _c(draft_q, np.float32)
    ci = _c(cand_idx, np.int32)
    B, L1, ld = tg.shape
    L = L1 - 1
    K = ci.shape[-1]
    V = ld if V is None else V
    acc = np.zeros(B, np.int32)
    out = np.zeros((B, L + 1), np.int32)
    margin = np.zeros((B, 2), np.float64)
    _load().oracle_verify(_p(tg), ld, _p(dt), _p(ds), _p(dq), _p(ci), B, L, K, V, float(temperature),
                          seed, offset, _p(acc), _p(out), _p(margin), nthreads or default_threads())
    return acc, out, margin


def lmhead_topk(hidden_bits, W_bits, rows, k=16, nthreads=None):
    """hidden: uint16 [M, d]; W: uint16 [V, d]; rows: row ids -> (vals f64 [n,k], idx i32 [n,k])."""
    hid = _c(hidden_bits, np.uint16)
    W = _c(W_bits, np.uint16)
    rw = _c(rows, np.int64)
    V, d = W.shape
    n = rw.shape[0]
    vals = np.zeros((n, k), np.float64)
    idx = np.zeros((n, k), np.int32)
    _load().oracle_lmhead_topk(_p(hid), _p(W), V, d, _p(rw), n, k, _p(vals), _p(idx),
                               nthreads or default_threads())
    return vals, idx
