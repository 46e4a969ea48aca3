"""GPU: the conditional sections that stop a captured decode loop on the device.

The whole-loop parity (every workload's loop, plain and with early stop, against the oracle) is
in test_gpu_commit.py; these cases cover the capture calls themselves: a section's default
condition, nesting, the condition set from inside a section, and the errors outside a capture.
"""
import numpy as np
import pytest
import torch

import oracle
import synth
from gpu_runner import GpuDecoder, to_device
from harness import guarded_logits, oracle_step

import diffusion_decoding_gb300 as dd

pytestmark = pytest.mark.gpu


def _graph(body_fn):
    g = torch.cuda.CUDAGraph()
    cap = torch.cuda.Stream()
    cap.wait_stream(torch.cuda.current_stream())
    torch.cuda.synchronize()
    with torch.cuda.stream(cap):
        with torch.cuda.graph(g, stream=cap):
            body_fn(cap)
    torch.cuda.current_stream().wait_stream(cap)
    return g


@pytest.mark.parametrize("default", [0, 1])
def test_section_runs_on_its_default_condition(default):
    x = torch.zeros(4, device="cuda")
    s2 = torch.cuda.Stream()

    def body(cap):
        h = dd.dllm_capture_condition(default, cap)
        x.add_(1)                      # always
        dd.dllm_capture_if_begin(h, s2, cap)
        with torch.cuda.stream(s2):
            x.add_(10)                 # only when the condition is non-zero
        dd.dllm_capture_if_end(s2)
        x.mul_(2)                      # after the section

    g = _graph(body)
    for rep in range(3):               # the default is assigned again at every launch
        x.zero_()
        g.replay()
        torch.cuda.synchronize()
        assert torch.equal(x, torch.full_like(x, 2 * (1 + 10 * default))), rep


def _decode(w, seed, iters):
    """Oracle trajectory: per-iteration logits (device) and the state after each iteration."""
    ost = oracle.BlockState(w.B, w.L, w.K)
    lgs, states = [], []
    for it in range(iters):
        lg, _, s = guarded_logits(w, seed, it, ost, calibrated=True)
        oracle_step(w, ost, lg, s)
        lgs.append(to_device(lg))
        states.append(ost.copy())
    return lgs, states


def test_nested_sections_follow_the_device_condition():
    # iteration 0 plain; iteration 1 in a section enabled by iteration 0; iteration 2 in a
    # section nested inside it, enabled by iteration 1.  With the block still decoding after
    # iteration 1 all three run; on a block finished by iteration 0 (forced below), neither runs.
    w = synth.WORKLOADS["threshold_loop"].scaled(B=2, L=16, V=4096, max_iters=3, eos_id=-1)
    lgs, states = _decode(w, 31, 3)
    assert states[0].masked.any(axis=1).all() and states[1].masked.any(), \
        "the trajectory must still be decoding after iterations 0 and 1"
    gpu = GpuDecoder(w)
    s2, s3 = torch.cuda.Stream(), torch.cuda.Stream()
    ran = torch.zeros(3, dtype=torch.int32, device="cuda")
    finish = torch.zeros(1, dtype=torch.int32, device="cuda")  # 1: end the block after it 0

    def body(cap):
        gpu.state.reset()
        h1 = dd.dllm_capture_condition(0, cap)
        gpu.step(lgs[0])
        ran[0].add_(1)
        # a block that was made to finish: every position committed (masked = 0)
        gpu.state.masked.mul_((1 - finish).to(torch.uint8))
        dd.dllm_loop_continue(gpu.state, h1, cap)
        dd.dllm_capture_if_begin(h1, s2, cap)
        with torch.cuda.stream(s2):
            h2 = dd.dllm_capture_condition(0, s2)   # its node lives in this section's body
            gpu.step(lgs[1])
            ran[1].add_(1)
            dd.dllm_loop_continue(gpu.state, h2, s2)
            dd.dllm_capture_if_begin(h2, s3, s2)
            with torch.cuda.stream(s3):
                gpu.step(lgs[2])
                ran[2].add_(1)
            dd.dllm_capture_if_end(s3)
        dd.dllm_capture_if_end(s2)

    g = _graph(body)
    for force_end, expect in ((0, [1, 1, 1]), (1, [1, 0, 0]), (0, [1, 1, 1])):
        finish.fill_(force_end)
        ran.zero_()
        g.replay()
        torch.cuda.synchronize()
        assert ran.cpu().tolist() == expect, force_end
        if not force_end:
            hs = gpu.host_state()
            for k in ("masked", "tokens", "committed_now", "n_commit"):
                assert np.array_equal(hs[k], getattr(states[2], k)), k


@pytest.mark.parametrize("L", [40, 32])  # byte loads; 16 positions per load
def test_loop_continue_reads_stopped_sequences(L):
    # the block decodes while some sequence has a masked position and no EOS
    w = synth.WORKLOADS["threshold_loop"].scaled(B=3, L=L, V=1024, max_iters=2)
    gpu = GpuDecoder(w)
    s2 = torch.cuda.Stream()
    ran = torch.zeros(1, dtype=torch.int32, device="cuda")

    def body(cap):
        h = dd.dllm_capture_condition(1, cap)     # default 1: only dllm_loop_continue clears it
        dd.dllm_loop_continue(gpu.state, h, cap)
        dd.dllm_capture_if_begin(h, s2, cap)
        with torch.cuda.stream(s2):
            ran.add_(1)
        dd.dllm_capture_if_end(s2)

    g = _graph(body)
    st = gpu.state

    def one_masked(b, i):
        m = np.zeros((3, L), np.uint8)
        m[b, i] = 1
        return m

    cases = [
        (np.zeros((3, L), np.uint8), [0, 0, 0], 0),   # nothing masked
        (one_masked(1, 0), [0, 1, 0], 0),             # only in a sequence that hit EOS
        (one_masked(1, 0), [0, 0, 0], 1),
        (one_masked(2, L - 1), [1, 1, 0], 1),         # the very last position
        (one_masked(0, L - 1), [1, 0, 0], 0),
        (np.ones((3, L), np.uint8), [1, 1, 1], 0),    # everything masked, every sequence done
    ]
    for masked, eos, expect in cases:
        st.masked.copy_(torch.from_numpy(masked.reshape(-1)).cuda())
        st.eos_hit.copy_(torch.tensor(eos, dtype=torch.int32, device="cuda"))
        ran.zero_()
        g.replay()
        torch.cuda.synchronize()
        assert int(ran.item()) == expect, (int(masked.sum()), eos)


def test_loop_continue_on_the_largest_block():
    # B*L = 2^20 positions (1024 x 1024): one CTA tests 65,536 16-byte vectors of mask bytes
    B = L = 1024
    state = dd.BlockState(B, L)
    s2 = torch.cuda.Stream()
    ran = torch.zeros(1, dtype=torch.int32, device="cuda")

    def body(cap):
        h = dd.dllm_capture_condition(0, cap)
        dd.dllm_loop_continue(state, h, cap)
        dd.dllm_capture_if_begin(h, s2, cap)
        with torch.cuda.stream(s2):
            ran.add_(1)
        dd.dllm_capture_if_end(s2)

    g = _graph(body)
    for last_masked, eos_last, expect in ((None, 0, 0), (B * L - 1, 0, 1), (B * L - 1, 1, 0),
                                          (5 * L + 7, 0, 1)):
        state.masked.zero_()
        state.eos_hit.zero_()
        if last_masked is not None:
            state.masked[last_masked] = 1
        state.eos_hit[B - 1] = eos_last
        ran.zero_()
        g.replay()
        torch.cuda.synchronize()
        assert int(ran.item()) == expect, (last_masked, eos_last)


def test_capture_calls_outside_a_capture_are_rejected():
    w = synth.WORKLOADS["threshold_loop"].scaled(B=1, L=8, V=1024)
    gpu = GpuDecoder(w)
    s = torch.cuda.Stream()
    with pytest.raises(dd.DllmError) as e:
        dd.dllm_loop_continue(gpu.state, 1, s)
    assert e.value.status == dd.DLLM_ERR_INVALID_ARG
    with pytest.raises(dd.DllmError) as e:
        dd.dllm_capture_condition(0, s)
    assert e.value.status == dd.DLLM_ERR_INVALID_ARG
    with pytest.raises(dd.DllmError) as e:
        dd.dllm_capture_if_begin(1, torch.cuda.Stream(), s)
    assert e.value.status == dd.DLLM_ERR_INVALID_ARG
    torch.cuda.synchronize()
