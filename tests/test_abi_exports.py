"""The C-ABI library loads on any host and exports every entry point the
public header declares; host-side argument checks answer without a GPU."""
import ctypes

import pytest

from draft_selection_dflash2_gb300 import _lib, build


@pytest.fixture(scope="module")
def lib():
    build.build()
    return _lib.load()


def test_header_declares_the_six_calls():
    names = _lib.declared_functions()
    for call in ("dflash2_topk", "dflash2_pair_scores", "dflash2_walk", "dflash2_conv2tap",
                 "dflash2_verify", "dflash2_lmhead_topk"):
        assert call in names


def test_every_declared_symbol_is_exported(lib):
    for name in _lib.declared_functions():
        assert hasattr(lib, name), name
        assert name in _lib.SIGNATURES, f"{name} has no ctypes signature"


def test_status_strings(lib):
    assert lib.dflash2_status_string(0) == b"ok"
    assert lib.dflash2_status_string(-7) == b"workspace too small"
    assert lib.dflash2_version() >= 100


def test_null_handle_is_rejected_without_a_device(lib):
    null = ctypes.c_void_p(None)
    one = ctypes.c_void_p(16)
    assert lib.dflash2_topk(null, one, 4, 64, 64, 16, one, one, null) == -1
    assert lib.dflash2_walk(null, one, one, 1, 4, 0.0, 0, 0, one, one, null, null) == -1
    assert lib.dflash2_verify(null, one, 64, one, null, null, null, 1, 4, 64, 0.0, 0, 0, one, one,
                              one, 1 << 20, null) == -1
    assert lib.dflash2_conv2tap(null, one, one, null, one, one, one, null, 1, 4, 64, one, 1, one, 1 << 20,
                                null) == -1
    assert lib.dflash2_pair_scores(null, one, one, one, one, one, null, one, one, 1, 4, 64, 64, one,
                                   one, one, 1 << 20, null) == -1
    assert lib.dflash2_lmhead_topk(null, one, one, 4, 64, 64, one, one, one, 256, null) == -1
    assert lib.dflash2_create(0, None) == -1


def test_workspace_queries_are_host_only(lib):
    null = ctypes.c_void_p(None)
    assert lib.dflash2_lmhead_topk_workspace(null, 1024, 151936, 5120) == 0
    assert lib.dflash2_verify_workspace(null, 128, 16, 151936) == 0
    assert lib.dflash2_gemm_conv2tap_workspace(null, 128, 16, 5120) == 0
    assert lib.dflash2_conv2tap_workspace(null, 128, 16, 5120) == 0
    assert lib.dflash2_pair_scores_workspace(null, 128, 16, 5120) == 0


def test_handle_allocates_only_its_error_word():
    # the library's only cudaMalloc is the handle's error word in dflash2_create
    import os
    import re
    csrc = os.path.join(os.path.dirname(_lib.HERE), "draft_selection_dflash2_gb300", "csrc")
    hits = []
    for name in sorted(os.listdir(csrc)):
        text = open(os.path.join(csrc, name)).read()
        for m in re.finditer(r"\bcudaMalloc\w*\s*\(", text):
            hits.append((name, text[:m.start()].count("\n") + 1))
    assert [h[0] for h in hits] == ["api.cu"], hits
    api_src = open(os.path.join(csrc, "api.cu")).read()
    assert api_src.count("cudaMalloc(") == 1 and "cudaMalloc(&h->err" in api_src
