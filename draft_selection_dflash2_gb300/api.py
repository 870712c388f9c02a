"""Python binding of the DFlash 2 draft-block head (argument marshalling only).

Every function has the name of the C entry point it calls (without the
``dflash2_`` prefix) and runs entirely in the CUDA library: torch tensors only
supply device memory and the current stream.  bf16 tensors may be given as
torch.bfloat16 or as int16/uint16 bit patterns.  Outputs that are not passed in
are allocated with torch before the call (the library itself never allocates).
"""
import ctypes

import torch

from . import _lib

K = 16
EMBED = 256

STATUS = {0: "OK", -1: "INVALID_ARG", -2: "UNSUPPORTED", -3: "MISALIGNED", -4: "CUDA",
          -5: "TIMEOUT", -6: "DEVICE", -7: "WORKSPACE"}
DEVERR_BAD_TOKEN = 0x1
DEVERR_TIMEOUT = 0x2
DEVERR_BAD_SLOT = 0x4


class Dflash2Error(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        msg = _lib.load().dflash2_status_string(status).decode()
        super().__init__(f"{where}: {STATUS.get(status, status)} ({msg})")


def _check(status: int, where: str):
    if status != 0:
        raise Dflash2Error(status, where)


def _ptr(t):
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("expected a CUDA tensor")
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _is16(t):
    return t.dtype in (torch.bfloat16, torch.int16, torch.uint16)


def _need(cond, what):
    if not cond:
        raise ValueError(what)


class Handle:
    """Owns a dflash2_handle (device error word) bound to one CUDA device."""

    def __init__(self, device: int = None):
        self._lib = _lib.load()
        if device is None:
            device = torch.cuda.current_device()
        self.device = device
        h = ctypes.c_void_p()
        _check(self._lib.dflash2_create(device, ctypes.byref(h)), "dflash2_create")
        self._h = h

    @property
    def ptr(self):
        return self._h

    @property
    def num_sms(self) -> int:
        return int(self._lib.dflash2_num_sms(self._h))

    def device_error(self, stream=None, clear: bool = True) -> int:
        bits = ctypes.c_uint32(0)
        _check(self._lib.dflash2_get_device_error(self._h, _stream(stream), ctypes.byref(bits),
                                                  1 if clear else 0), "dflash2_get_device_error")
        return int(bits.value)

    def close(self):
        if self._h is not None and self._h.value:
            _check(self._lib.dflash2_destroy(self._h), "dflash2_destroy")
        self._h = None

    def __enter__(self):
        return self

    def __exit__(self, *exc):
        self.close()

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def topk(h: Handle, logits, V: int = None, vals=None, idx=None, k: int = K, stream=None):
    """logits [rows, ld] bf16 -> (vals fp32 [rows, 16], idx int32 [rows, 16])."""
    _need(_is16(logits) and logits.dim() == 2 and logits.stride(1) == 1, "logits: 2-D bf16, unit stride")
    rows, ld = logits.shape[0], logits.stride(0)
    V = logits.shape[1] if V is None else V
    dev = logits.device
    vals = torch.empty((rows, k), dtype=torch.float32, device=dev) if vals is None else vals
    idx = torch.empty((rows, k), dtype=torch.int32, device=dev) if idx is None else idx
    _check(h._lib.dflash2_topk(h.ptr, _ptr(logits), rows, V, ld, k, _ptr(vals), _ptr(idx),
                               _stream(stream)), "dflash2_topk")
    return vals, idx


def pair_scores_workspace(h: Handle, B: int, L: int, d: int) -> int:
    return int(h._lib.dflash2_pair_scores_workspace(h.ptr, B, L, d))


def pair_scores(h: Handle, cand_idx, cand_val, last_verified, hs, W_H, b_H, A, Bt, V: int = None,
                gate=None, S=None, workspace=None, stream=None):
    """-> (S fp32 [B, L, 16, 16], gate fp32 [B, L, 256]).

    workspace: device bytes (uint8 tensor) of at least pair_scores_workspace(h, B, L, d);
    allocated here by torch when None."""
    B, L, k = cand_idx.shape
    _need(k == K, "cand_idx: [B, L, 16]")
    d = hs.shape[-1]
    V = A.shape[0] if V is None else V
    dev = cand_idx.device
    for name, t in (("hs", hs), ("W_H", W_H), ("A", A), ("Bt", Bt)):
        _need(_is16(t) and t.is_contiguous(), f"{name}: contiguous bf16")
    gate = torch.empty((B, L, EMBED), dtype=torch.float32, device=dev) if gate is None else gate
    S = torch.empty((B, L, K, K), dtype=torch.float32, device=dev) if S is None else S
    if workspace is None:
        workspace = torch.empty(max(pair_scores_workspace(h, B, L, d), 256), dtype=torch.uint8, device=dev)
    _check(h._lib.dflash2_pair_scores(h.ptr, _ptr(cand_idx), _ptr(cand_val), _ptr(last_verified),
                                      _ptr(hs), _ptr(W_H), _ptr(b_H), _ptr(A), _ptr(Bt), B, L, d, V,
                                      _ptr(gate), _ptr(S), _ptr(workspace),
                                      workspace.numel() * workspace.element_size(), _stream(stream)),
           "dflash2_pair_scores")
    return S, gate


def walk(h: Handle, S, cand_idx, temperature: float = 0.0, seed: int = 0, offset: int = 0,
         draft_tok=None, draft_slot=None, draft_q=None, want_q: bool = True, stream=None):
    """-> (draft_tok int32 [B, L], draft_slot int32 [B, L], draft_q fp32 [B, L, 16] or None)."""
    B, L = S.shape[0], S.shape[1]
    dev = S.device
    draft_tok = torch.empty((B, L), dtype=torch.int32, device=dev) if draft_tok is None else draft_tok
    draft_slot = torch.empty((B, L), dtype=torch.int32, device=dev) if draft_slot is None else draft_slot
    if draft_q is None and want_q:
        draft_q = torch.empty((B, L, K), dtype=torch.float32, device=dev)
    _check(h._lib.dflash2_walk(h.ptr, _ptr(S), _ptr(cand_idx), B, L, float(temperature), seed, offset,
                               _ptr(draft_tok), _ptr(draft_slot), _ptr(draft_q), _stream(stream)),
           "dflash2_walk")
    return draft_tok, draft_slot, draft_q


def walk_viterbi(h: Handle, S, cand_idx, draft_tok=None, draft_slot=None, score=None, want_score: bool = True,
                 stream=None):
    """Exact best path -> (draft_tok int32 [B, L], draft_slot int32 [B, L], score fp32 [B] or None)."""
    B, L = S.shape[0], S.shape[1]
    dev = S.device
    draft_tok = torch.empty((B, L), dtype=torch.int32, device=dev) if draft_tok is None else draft_tok
    draft_slot = torch.empty((B, L), dtype=torch.int32, device=dev) if draft_slot is None else draft_slot
    if score is None and want_score:
        score = torch.empty((B,), dtype=torch.float32, device=dev)
    _check(h._lib.dflash2_walk_viterbi(h.ptr, _ptr(S), _ptr(cand_idx), B, L, _ptr(draft_tok), _ptr(draft_slot),
                                       _ptr(score), _stream(stream)),
           "dflash2_walk_viterbi")
    return draft_tok, draft_slot, score


def selector_eval(h: Handle, gt, cand_idx, accept1=None, accept16=None, counts=None, stream=None):
    """Table 1 evaluation -> (accept1 int32 [B], accept16 int32 [B], counts int64 [L, 4])."""
    B, L = gt.shape
    dev = gt.device
    accept1 = torch.empty((B,), dtype=torch.int32, device=dev) if accept1 is None else accept1
    accept16 = torch.empty((B,), dtype=torch.int32, device=dev) if accept16 is None else accept16
    counts = torch.empty((L, 4), dtype=torch.int64, device=dev) if counts is None else counts
    _check(h._lib.dflash2_selector_eval(h.ptr, _ptr(gt), _ptr(cand_idx), B, L, _ptr(accept1), _ptr(accept16),
                                        _ptr(counts), _stream(stream)),
           "dflash2_selector_eval")
    return accept1, accept16, counts


def conv2tap_workspace(h: Handle, B: int, L: int, d: int) -> int:
    return int(h._lib.dflash2_conv2tap_workspace(h.ptr, B, L, d))


def conv2tap(h: Handle, x, x_prev, k0, k1, W_c, b_c=None, hs=None, y=None, y_fp32: bool = False,
             workspace=None, stream=None):
    """x [B, L, d] bf16 -> y [B, L, d] (bf16, or fp32 when y_fp32).

    workspace: device bytes (uint8 tensor) of at least conv2tap_workspace(h, B, L, d);
    allocated here by torch when None."""
    B, L, d = x.shape
    dev = x.device
    if y is None:
        y = torch.empty((B, L, d), dtype=torch.float32 if y_fp32 else torch.bfloat16, device=dev)
    y_is_fp32 = 1 if y.dtype == torch.float32 else 0
    if workspace is None:
        workspace = torch.empty(max(conv2tap_workspace(h, B, L, d), 256), dtype=torch.uint8, device=dev)
    _check(h._lib.dflash2_conv2tap(h.ptr, _ptr(x), _ptr(x_prev), _ptr(hs), _ptr(k0), _ptr(k1), _ptr(W_c),
                                   _ptr(b_c), B, L, d, _ptr(y), y_is_fp32, _ptr(workspace),
                                   workspace.numel() * workspace.element_size(), _stream(stream)),
           "dflash2_conv2tap")
    return y


def gemm_conv2tap_workspace(h: Handle, B: int, L: int, d: int) -> int:
    return h._lib.dflash2_gemm_conv2tap_workspace(h.ptr, B, L, d)


def gemm_conv2tap(h: Handle, A, W, x_prev, hs, k0, k1, W_c, b_c=None, c_work=None, y=None, y_fp32: bool = False,
                  stream=None):
    """Conv fused into its producing GEMM: A [B, L, K] bf16, W [d, K] bf16 -> (y [B, L, d], c fp32 [B*L, 2d/16]).

    c_work: workspace of at least gemm_conv2tap_workspace(h, B, L, d) bytes (the correction, then
    per-row-tile counters); allocated when None."""
    B, L, Kd = A.shape
    d = W.shape[0]
    dev = A.device
    for name, t in (("A", A), ("W", W), ("x_prev", x_prev), ("hs", hs), ("W_c", W_c)):
        _need(_is16(t) and t.is_contiguous(), f"{name}: contiguous bf16")
    if c_work is None:
        c_work = torch.empty(((gemm_conv2tap_workspace(h, B, L, d) + 3) // 4,), dtype=torch.float32, device=dev)
    if y is None:
        y = torch.empty((B, L, d), dtype=torch.float32 if y_fp32 else torch.bfloat16, device=dev)
    y_is_fp32 = 1 if y.dtype == torch.float32 else 0
    _check(h._lib.dflash2_gemm_conv2tap(h.ptr, _ptr(A), _ptr(W), _ptr(x_prev), _ptr(hs), _ptr(k0), _ptr(k1),
                                        _ptr(W_c), _ptr(b_c), B, L, Kd, d, _ptr(c_work),
                                        c_work.numel() * c_work.element_size(), _ptr(y), y_is_fp32, _stream(stream)),
           "dflash2_gemm_conv2tap")
    n = 2 * (d // 16)
    return y, c_work.view(-1)[: B * L * n].view(B * L, n)


def verify_workspace(h: Handle, B: int, L: int, V: int) -> int:
    return int(h._lib.dflash2_verify_workspace(h.ptr, B, L, V))


def verify(h: Handle, target, draft_tok, draft_slot=None, draft_q=None, cand_idx=None,
           temperature: float = 0.0, seed: int = 0, offset: int = 0, V: int = None,
           accept_len=None, out_tok=None, workspace=None, stream=None):
    """target [B, L+1, V(ld)] bf16 -> (accept_len int32 [B], out_tok int32 [B, L+1]).

    workspace: device bytes (uint8 tensor) of at least verify_workspace(h, B, L, V);
    allocated here by torch when None."""
    B, L1 = target.shape[0], target.shape[1]
    ld = target.stride(1)
    V = target.shape[2] if V is None else V
    dev = target.device
    accept_len = torch.empty((B,), dtype=torch.int32, device=dev) if accept_len is None else accept_len
    out_tok = torch.empty((B, L1), dtype=torch.int32, device=dev) if out_tok is None else out_tok
    if workspace is None:
        workspace = torch.empty(max(verify_workspace(h, B, L1 - 1, V), 256), dtype=torch.uint8, device=dev)
    _check(h._lib.dflash2_verify(h.ptr, _ptr(target), ld, _ptr(draft_tok), _ptr(draft_slot), _ptr(draft_q),
                                 _ptr(cand_idx), B, L1 - 1, V, float(temperature), seed, offset,
                                 _ptr(accept_len), _ptr(out_tok), _ptr(workspace),
                                 workspace.numel() * workspace.element_size(), _stream(stream)), "dflash2_verify")
    return accept_len, out_tok


def lmhead_topk_workspace(h: Handle, M: int, V: int, d: int) -> int:
    return int(h._lib.dflash2_lmhead_topk_workspace(h.ptr, M, V, d))


def lmhead_topk(h: Handle, hidden, W, vals=None, idx=None, workspace=None, stream=None):
    """hidden [M, d] bf16, W [V, d] bf16 -> (vals fp32 [M, 16], idx int32 [M, 16])."""
    M, d = hidden.shape
    V = W.shape[0]
    dev = hidden.device
    vals = torch.empty((M, K), dtype=torch.float32, device=dev) if vals is None else vals
    idx = torch.empty((M, K), dtype=torch.int32, device=dev) if idx is None else idx
    need = lmhead_topk_workspace(h, M, V, d)
    if workspace is None:
        workspace = torch.empty(max(need, 256), dtype=torch.uint8, device=dev)
    _check(h._lib.dflash2_lmhead_topk(h.ptr, _ptr(hidden), _ptr(W), M, V, d, _ptr(vals), _ptr(idx),
                                      _ptr(workspace), workspace.numel(), _stream(stream)),
           "dflash2_lmhead_topk")
    return vals, idx


def lmhead_topk_gate(h: Handle, hidden, W, W_H, b_H=None, vals=None, idx=None, gate=None, workspace=None,
                     stream=None):
    """Fused LM head + top-16 + context gate -> (vals fp32 [M, 16], idx int32 [M, 16], gate fp32 [M, 256])."""
    for name, t in (("hidden", hidden), ("W", W), ("W_H", W_H)):
        _need(_is16(t) and t.is_contiguous(), f"{name}: contiguous bf16")
    M, d = hidden.shape
    V = W.shape[0]
    dev = hidden.device
    vals = torch.empty((M, K), dtype=torch.float32, device=dev) if vals is None else vals
    idx = torch.empty((M, K), dtype=torch.int32, device=dev) if idx is None else idx
    gate = torch.empty((M, EMBED), dtype=torch.float32, device=dev) if gate is None else gate
    if workspace is None:
        workspace = torch.empty(max(lmhead_topk_workspace(h, M, V, d), 256), dtype=torch.uint8, device=dev)
    _check(h._lib.dflash2_lmhead_topk_gate(h.ptr, _ptr(hidden), _ptr(W), _ptr(W_H), _ptr(b_H), M, V, d, _ptr(vals),
                                           _ptr(idx), _ptr(gate), _ptr(workspace), workspace.numel(),
                                           _stream(stream)), "dflash2_lmhead_topk_gate")
    return vals, idx, gate


def pair_scores_proj_workspace(h: Handle, B: int, L: int) -> int:
    return h._lib.dflash2_pair_scores_proj_workspace(h.ptr, B, L)


def pair_scores_proj(h: Handle, cand_idx, cand_val, last_verified, gate, E, W_A, W_B, P=None, S=None, stream=None):
    """Projection-form pair scores -> (S fp32 [B, L, 16, 16], P fp32 [B*L*16 + B, 512])."""
    B, L, k = cand_idx.shape
    _need(k == K, "cand_idx: [B, L, 16]")
    for name, t in (("E", E), ("W_A", W_A), ("W_B", W_B)):
        _need(_is16(t) and t.is_contiguous(), f"{name}: contiguous bf16")
    V, d = E.shape
    dev = cand_idx.device
    if P is None:
        P = torch.empty((B * L * K + B, 2 * EMBED), dtype=torch.float32, device=dev)
    S = torch.empty((B, L, K, K), dtype=torch.float32, device=dev) if S is None else S
    _check(h._lib.dflash2_pair_scores_proj(h.ptr, _ptr(cand_idx), _ptr(cand_val), _ptr(last_verified), _ptr(gate),
                                           _ptr(E), _ptr(W_A), _ptr(W_B), B, L, d, V, _ptr(P),
                                           P.numel() * P.element_size(), _ptr(S), _stream(stream)),
           "dflash2_pair_scores_proj")
    return S, P


def lmhead_topk_noalloc(h: Handle, hidden, W, vals=None, idx=None, stream=None):
    """lmhead_topk for callers that cannot allocate: the library's fixed
    device scratch replaces the workspace (calls sharing a device must not
    overlap on the GPU).  Outputs not passed in are allocated here, by torch."""
    M, d = hidden.shape
    V = W.shape[0]
    dev = hidden.device
    vals = torch.empty((M, K), dtype=torch.float32, device=dev) if vals is None else vals
    idx = torch.empty((M, K), dtype=torch.int32, device=dev) if idx is None else idx
    _check(h._lib.dflash2_lmhead_topk_noalloc(h.ptr, _ptr(hidden), _ptr(W), M, V, d, _ptr(vals), _ptr(idx),
                                              _stream(stream)), "dflash2_lmhead_topk_noalloc")
    return vals, idx



def selftest_wait_timeout(h: Handle, limit_ns: int, words=None, stream=None):
    """Runs the library's bounded-wait self-test: one kernel whose two waits
    cannot be satisfied gives up after limit_ns each.  Returns the result word
    (bit 2 = the kernel reached its end; bits 0/1 = a wait was satisfied)."""
    if words is None:
        words = torch.zeros(2, dtype=torch.int32, device=torch.device("cuda", h.device))
    _check(h._lib.dflash2_selftest_wait_timeout(h.ptr, int(limit_ns), _ptr(words), _stream(stream)),
           "dflash2_selftest_wait_timeout")
    return words
