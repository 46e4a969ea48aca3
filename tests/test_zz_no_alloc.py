"""The allocation-free entry point, for callers that cannot allocate device memory.

dllm_commit_threshold_static takes no workspace: its scratch is a fixed static array inside the
library.  It must give the same results as dllm_commit_threshold with a caller-allocated
workspace, call after call (the static scratch keeps the previous call's contents), and both
must match the oracle.  This file is collected last so that a failure here never hides the
other tests.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
import synth
from gpu_runner import to_device
from harness import close, guarded_logits, oracle_step

import diffusion_decoding_gb300 as dd

pytestmark = pytest.mark.gpu

STATIC_BYTES = 4 << 20  # DLLM_STATIC_WORKSPACE_BYTES


def _host(state: dd.BlockState, stats: dd.StatsBuffers):
    return ({k: getattr(state, k).cpu().numpy() for k in
             ("masked", "tokens", "committed_now", "n_commit", "eos_hit")},
            {k: getattr(stats, k).cpu().numpy() for k in ("row_max", "lse", "conf", "argmax")})


def _static_call(logits, shape, stats, state, tau, eos_id):
    st, bs = stats.c(), state.c()
    return dd.lib().dllm_commit_threshold_static(
        logits.data_ptr(), ctypes.byref(shape), ctypes.byref(st), ctypes.byref(bs), tau, eos_id,
        torch.cuda.current_stream().cuda_stream)


def _matches_oracle(tag, s_host, t_host, ost, s_ref):
    for k in ("masked", "tokens", "committed_now", "n_commit", "eos_hit"):
        assert np.array_equal(s_host[k].reshape(getattr(ost, k).shape), getattr(ost, k)), \
            f"{tag}: {k} differs from the oracle"
    assert np.array_equal(t_host["argmax"], s_ref.argmax), f"{tag}: argmax"
    assert close(t_host["row_max"], s_ref.row_max, 0.0), f"{tag}: row_max"
    for k in ("lse", "conf"):
        assert close(t_host[k], getattr(s_ref, k)), f"{tag}: {k}"


def _two_calls(w, seed, calibrated):
    """Two decode steps in a row: the caller-workspace call and the static call on the same
    margin-guarded logits, each compared with the other and with the oracle trajectory."""
    dt = dd.DLLM_BF16 if w.dtype == "bf16" else dd.DLLM_F32
    shape = dd.make_shape(w.B, w.L, w.V, dt)
    assert dd.dllm_workspace_bytes(shape) <= STATIC_BYTES
    ref_state, ref_stats = dd.BlockState(w.B, w.L), dd.StatsBuffers(w.B * w.L)
    st_state, st_stats = dd.BlockState(w.B, w.L), dd.StatsBuffers(w.B * w.L)
    ws = dd.workspace(dd.dllm_workspace_bytes(shape))
    ost = oracle.BlockState(w.B, w.L)
    for it in range(2):  # two calls in a row through the same static scratch
        lg_h, _, s = guarded_logits(w, seed, it, ost, calibrated)
        s_ref, _ = oracle_step(w, ost, lg_h, s)
        lg = to_device(lg_h)
        dd.dllm_commit_threshold(lg, shape, ref_stats, ref_state, w.tau, w.eos_id, ws)
        rc = _static_call(lg, shape, st_stats, st_state, w.tau, w.eos_id)
        assert rc == dd.DLLM_OK, dd.lib().dllm_last_error()
        torch.cuda.synchronize()
        (a_s, a_t), (b_s, b_t) = _host(ref_state, ref_stats), _host(st_state, st_stats)
        for k in a_s:
            assert np.array_equal(a_s[k], b_s[k]), f"call {it}: {k}"
        assert np.array_equal(a_t["argmax"], b_t["argmax"])
        for k in ("row_max", "lse", "conf"):
            assert close(b_t[k], a_t[k]), f"call {it}: {k}"
        _matches_oracle(f"static call {it}", b_s, b_t, ost, s_ref)
        _matches_oracle(f"workspace call {it}", a_s, a_t, ost, s_ref)
        assert a_s["n_commit"].sum() >= w.B or it > 0


@pytest.mark.parametrize("w,calibrated", [
    (synth.WORKLOADS["threshold_loop"].scaled(B=4, L=32, V=20000, eos_id=2), True),
    (synth.WORKLOADS["smooth_step"], False),
])
def test_static_scratch_matches_caller_workspace_two_calls(w, calibrated):
    _two_calls(w, seed=123, calibrated=calibrated)


def test_static_scratch_at_its_size_limit():
    # 16 x 129 rows of V = 130048: 127 records of 16 bytes per row (counted at the fp32 slice
    # size) plus the 256-byte header fill the static array exactly
    w = synth.WORKLOADS["smooth_step"].scaled(B=16, L=129, V=130048)
    shape = dd.make_shape(w.B, w.L, w.V, dd.DLLM_BF16)
    assert dd.dllm_workspace_bytes(shape) == STATIC_BYTES
    _two_calls(w, seed=321, calibrated=False)


@pytest.mark.parametrize("B,L,V", [(16, 129, 130049), (16, 130, 130048), (1024, 1024, 126464)])
def test_static_scratch_rejects_shapes_beyond_its_size(B, L, V):
    # one vocabulary element, or one position per sequence, more than the limit case
    shape = dd.make_shape(B, L, V, dd.DLLM_BF16)
    assert dd.dllm_workspace_bytes(shape) > STATIC_BYTES
    stats, state = dd.StatsBuffers(1), dd.BlockState(1, 1)
    dummy = torch.empty(8, dtype=torch.bfloat16, device="cuda")
    rc = _static_call(dummy, shape, stats, state, 0.9, -1)
    assert rc == dd.DLLM_ERR_UNSUPPORTED
    assert "static" in dd.lib().dllm_last_error().decode()
