"""Host-side checks of the C ABI: the library loads, exports every declared symbol, and rejects
bad arguments before launching anything (no GPU needed)."""
import ctypes
import os
import re

import pytest

import diffusion_decoding_gb300 as dd
from diffusion_decoding_gb300 import build as cuda_build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    cuda_build.build()
    return dd.lib()


def declared_functions():
    src = open(os.path.join(ROOT, "include", "dllm.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(dllm_\w+)\s*\(", src)))


def test_every_declared_symbol_is_exported(lib):
    names = declared_functions()
    assert len(names) >= 14
    raw = ctypes.CDLL(dd.LIB_PATH)
    for n in names:
        assert hasattr(raw, n), f"{n} declared in dllm.h but not exported"
    # and the binding covers the same set
    assert set(names) <= set(dd._SIGS), set(names) - set(dd._SIGS)


def _shape(**kw):
    d = dict(B=2, L=8, V=1024, dtype=dd.DLLM_BF16, row_stride=1024)
    d.update(kw)
    return dd.dllm_shape(d["B"], d["L"], d["V"], d["dtype"], d["row_stride"])


@pytest.mark.parametrize("kw,expect", [
    (dict(B=0), dd.DLLM_ERR_INVALID_ARG),
    (dict(V=0), dd.DLLM_ERR_INVALID_ARG),
    (dict(L=1025), dd.DLLM_ERR_UNSUPPORTED),
    (dict(dtype=7), dd.DLLM_ERR_UNSUPPORTED),
    (dict(row_stride=1000), dd.DLLM_ERR_INVALID_ARG),
    (dict(B=2048, L=1024), dd.DLLM_ERR_UNSUPPORTED),
])
def test_shape_validation(lib, kw, expect):
    sh = _shape(**kw)
    st = dd.dllm_stats(16, 16, 16, 16)
    rc = lib.dllm_decode_stats(256, ctypes.byref(sh), None, ctypes.byref(st), 256, None)
    assert rc == expect, lib.dllm_last_error()
    assert lib.dllm_last_error()


def test_pointer_validation(lib):
    sh = _shape()
    st = dd.dllm_stats(16, 16, 16, 16)
    bs = dd.dllm_block_state(16, 16, 16, 16, 16)
    assert lib.dllm_decode_stats(None, ctypes.byref(sh), None, ctypes.byref(st), 256, None) \
        == dd.DLLM_ERR_INVALID_ARG
    assert lib.dllm_decode_stats(9, ctypes.byref(sh), None, ctypes.byref(st), 256, None) \
        == dd.DLLM_ERR_INVALID_ARG  # logits not aligned to the bf16 element
    # rows that are not 16-byte aligned are read element by element by every call, but a
    # pointer not aligned to its element is rejected before anything is launched
    odd = _shape(V=1024, row_stride=1028)
    assert lib.dllm_commit_threshold_smooth(257, ctypes.byref(odd), ctypes.byref(st),
                                            ctypes.byref(bs), 0.9, -1, 256, 64, 256, 16, 16,
                                            256, 1 << 30, None) == dd.DLLM_ERR_INVALID_ARG
    assert lib.dllm_smooth_probs(259, ctypes.byref(sh), ctypes.byref(st), ctypes.byref(bs), 64,
                                 16, 16, 256, 1 << 30, None) == dd.DLLM_ERR_INVALID_ARG
    assert lib.dllm_decode_stats(256, ctypes.byref(sh), None, ctypes.byref(st), 128, None) \
        == dd.DLLM_ERR_INVALID_ARG  # misaligned workspace
    bad = dd.dllm_block_state(16, 0, 16, 16, 16)
    assert lib.dllm_commit_threshold(256, ctypes.byref(sh), ctypes.byref(st), ctypes.byref(bad),
                                     0.9, -1, 256, None) == dd.DLLM_ERR_INVALID_ARG
    assert lib.dllm_commit_hierarchical(256, ctypes.byref(sh), ctypes.byref(st),
                                        ctypes.byref(bs), 0.6, 0, -1, 256, None) \
        == dd.DLLM_ERR_INVALID_ARG
    assert lib.dllm_commit_credit(256, ctypes.byref(sh), ctypes.byref(st), ctypes.byref(bs),
                                  16, 16, 17, 0.7, 0.3, 0.9, -1, 256, None) \
        == dd.DLLM_ERR_UNSUPPORTED
    assert lib.dllm_commit_credit(256, ctypes.byref(sh), ctypes.byref(st), ctypes.byref(bs),
                                  None, 16, 8, 0.7, 0.3, 0.9, -1, 256, None) \
        == dd.DLLM_ERR_INVALID_ARG
    assert lib.dllm_kv_refresh_mask(ctypes.byref(bs), 2, 8, -1, 4, 16, 16, 16, None) \
        == dd.DLLM_ERR_INVALID_ARG
    assert lib.dllm_block_state_reset(ctypes.byref(bad), 2, 8, None, None, 0, None) \
        == dd.DLLM_ERR_INVALID_ARG  # a null state array
    assert lib.dllm_block_state_reset(ctypes.byref(bs), 0, 8, None, None, 0, None) \
        == dd.DLLM_ERR_INVALID_ARG
    assert lib.dllm_block_state_reset(ctypes.byref(bs), 2, 1025, None, None, 0, None) \
        == dd.DLLM_ERR_UNSUPPORTED
    assert lib.dllm_block_state_reset(ctypes.byref(bs), 2, 8, 16, 16, 17, None) \
        == dd.DLLM_ERR_INVALID_ARG  # K beyond the slot limit
    assert lib.dllm_kv_refresh_mask(ctypes.byref(bs), 2, 8, 65530, 4, 16, 16, 16, None) \
        == dd.DLLM_ERR_UNSUPPORTED
    assert lib.dllm_prepare_embedding(16, 100, 24, 16, None) == dd.DLLM_ERR_UNSUPPORTED
    assert lib.dllm_smooth_embed(256, ctypes.byref(_shape(V=1020, row_stride=1024)),
                                 ctypes.byref(st), ctypes.byref(bs), 256, 40, 256, 16, 16, 256,
                                 1 << 30, None) == dd.DLLM_ERR_UNSUPPORTED  # d % 16 != 0
    assert lib.dllm_smooth_embed(256, ctypes.byref(sh), ctypes.byref(st), ctypes.byref(bs), 256,
                                 64, 256, 16, 16, 256, 16, None) == dd.DLLM_ERR_INVALID_ARG
    assert lib.dllm_get_status(256, None, None) == dd.DLLM_ERR_INVALID_ARG
    # loop capture: checked before any CUDA call
    assert lib.dllm_capture_condition(None, 0, None) == dd.DLLM_ERR_INVALID_ARG
    assert lib.dllm_capture_if_begin(16, 16, 1) == dd.DLLM_ERR_INVALID_ARG  # one stream for both
    no_mask = dd.dllm_block_state(None, 16, 16, 16, 16)
    assert lib.dllm_loop_continue(ctypes.byref(no_mask), 2, 8, 1, None) == dd.DLLM_ERR_INVALID_ARG
    assert lib.dllm_loop_continue(ctypes.byref(bs), 0, 8, 1, None) == dd.DLLM_ERR_INVALID_ARG
    assert lib.dllm_loop_continue(ctypes.byref(bs), 2, 1025, 1, None) == dd.DLLM_ERR_UNSUPPORTED


def test_workspace_sizes(lib):
    sh = _shape(B=32, L=32, V=126464, row_stride=126464)
    n = dd.dllm_workspace_bytes(sh)
    assert n >= 32 * 32 * 16 * 12  # partials for every 32 KB slice of every row (fp32 worst case)
    assert dd.dllm_workspace_bytes(_shape(B=0)) == 0
    assert dd.dllm_embedding_t_elems(126463, 2048) == 2048 * 126464
    assert dd.dllm_embedding_t_elems(1001, 16) == 16 * 1024
