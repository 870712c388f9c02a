"""ctypes loader for libdflash2.so (the CUDA kernels behind the C ABI).

There is no fallback: if the library has not been built for this machine,
loading raises immediately.
"""
import ctypes
import os
import re

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libdflash2.so")
HEADER = os.path.join(os.path.dirname(HERE), "include", "dflash2.h")

P = ctypes.c_void_p
I64 = ctypes.c_int64
U64 = ctypes.c_uint64
I32 = ctypes.c_int
U32P = ctypes.POINTER(ctypes.c_uint32)
F32 = ctypes.c_float
SZ = ctypes.c_size_t

# name -> (restype, argtypes); mirrors include/dflash2.h
SIGNATURES = {
    "dflash2_version": (I32, []),
    "dflash2_status_string": (ctypes.c_char_p, [I32]),
    "dflash2_create": (I32, [I32, ctypes.POINTER(P)]),
    "dflash2_destroy": (I32, [P]),
    "dflash2_num_sms": (I32, [P]),
    "dflash2_get_device_error": (I32, [P, P, U32P, I32]),
    "dflash2_topk": (I32, [P, P, I64, I64, I64, I32, P, P, P]),
    "dflash2_pair_scores_workspace": (SZ, [P, I64, I64, I64]),
    "dflash2_pair_scores": (I32, [P, P, P, P, P, P, P, P, P, I64, I64, I64, I64, P, P, P, SZ, P]),
    "dflash2_walk": (I32, [P, P, P, I64, I64, F32, U64, U64, P, P, P, P]),
    "dflash2_walk_viterbi": (I32, [P, P, P, I64, I64, P, P, P, P]),
    "dflash2_selector_eval": (I32, [P, P, P, I64, I64, P, P, P, P]),
    "dflash2_conv2tap_workspace": (SZ, [P, I64, I64, I64]),
    "dflash2_conv2tap": (I32, [P, P, P, P, P, P, P, P, I64, I64, I64, P, I32, P, SZ, P]),
    "dflash2_verify_workspace": (SZ, [P, I64, I64, I64]),
    "dflash2_verify": (I32, [P, P, I64, P, P, P, P, I64, I64, I64, F32, U64, U64, P, P, P, SZ, P]),
    "dflash2_lmhead_topk_workspace": (SZ, [P, I64, I64, I64]),
    "dflash2_lmhead_topk": (I32, [P, P, P, I64, I64, I64, P, P, P, SZ, P]),
    "dflash2_lmhead_topk_gate": (I32, [P, P, P, P, P, I64, I64, I64, P, P, P, P, SZ, P]),
    "dflash2_pair_scores_proj_workspace": (SZ, [P, I64, I64]),
    "dflash2_gemm_conv2tap_workspace": (SZ, [P, I64, I64, I64]),
    "dflash2_gemm_conv2tap": (I32, [P, P, P, P, P, P, P, P, P, I64, I64, I64, I64, P, SZ, P, I32, P]),
    "dflash2_pair_scores_proj": (I32, [P, P, P, P, P, P, P, P, I64, I64, I64, I64, P, SZ, P, P]),
    "dflash2_lmhead_topk_noalloc": (I32, [P, P, P, I64, I64, I64, P, P, P]),
    "dflash2_selftest_wait_timeout": (I32, [P, U64, P, P]),
}

_lib = None


def declared_functions(header: str = HEADER):
    """Function names declared in the public header."""
    text = open(header).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(dflash2_[a-z_0-9]+)\s*\(", text)))


def load():
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(
                f"{LIB_PATH} is missing: build it first "
                "(python -c 'import __graft_entry__ as g; g.build()')")
        lib = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in SIGNATURES.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _lib = lib
    return _lib
