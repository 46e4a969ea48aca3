"""Run the CUDA path through the Python binding of the C ABI (GPU tests only)."""
from __future__ import annotations

import numpy as np
import torch

import diffusion_decoding_gb300 as dd


def to_device(lg: np.ndarray) -> torch.Tensor:
    """float32 array, or uint16 bf16 bit patterns, -> CUDA tensor of the same values."""
    if lg.dtype == np.uint16:
        return torch.from_numpy(lg.view(np.int16)).view(torch.bfloat16).cuda()
    return torch.from_numpy(lg).cuda()


class GpuDecoder:
    """Device state + buffers for one workload; step() runs one fused commit call."""

    def __init__(self, w):
        self.w = w
        dt = dd.DLLM_BF16 if w.dtype == "bf16" else dd.DLLM_F32
        self.shape = dd.make_shape(w.B, w.L, w.V, dt)
        self.state = dd.BlockState(w.B, w.L, w.K)
        self.stats = dd.StatsBuffers(w.B * w.L)
        self.ws = dd.workspace(dd.dllm_workspace_bytes(self.shape))

    def step(self, logits_dev: torch.Tensor | None) -> None:
        w = self.w
        if w.strategy in ("threshold", "smooth"):
            dd.dllm_commit_threshold(logits_dev, self.shape, self.stats, self.state, w.tau,
                                     w.eos_id, self.ws)
        elif w.strategy == "hierarchical":
            dd.dllm_commit_hierarchical(logits_dev, self.shape, self.stats, self.state, w.tau_low,
                                        w.min_width, w.eos_id, self.ws)
        elif w.strategy == "hierarchical_levels":
            dd.dllm_commit_hierarchical_levels(logits_dev, self.shape, self.stats, self.state,
                                               w.tau_low, w.min_width, w.eos_id, self.ws)
        elif w.strategy == "credit_tracked":
            dd.dllm_commit_credit_tracked(logits_dev, self.shape, self.stats, self.state, w.K,
                                          w.decay, w.boost, w.tau, w.eos_id, self.ws)
        else:
            dd.dllm_commit_credit(logits_dev, self.shape, self.stats, self.state, w.K, w.decay,
                                  w.boost, w.tau, w.eos_id, self.ws)

    def host_state(self):
        s = self.state
        B, L = self.w.B, self.w.L
        return dict(masked=s.masked.cpu().numpy().reshape(B, L),
                    tokens=s.tokens.cpu().numpy().reshape(B, L),
                    committed_now=s.committed_now.cpu().numpy().reshape(B, L),
                    n_commit=s.n_commit.cpu().numpy(), eos_hit=s.eos_hit.cpu().numpy(),
                    cand_id=s.cand_id.cpu().numpy().reshape(B, L, -1),
                    cand_credit=s.cand_credit.cpu().numpy().reshape(B, L, -1))

    def host_stats(self):
        st = self.stats
        return dict(row_max=st.row_max.cpu().numpy(), lse=st.lse.cpu().numpy(),
                    conf=st.conf.cpu().numpy(), argmax=st.argmax.cpu().numpy())


def capture_loop(gpu: GpuDecoder, lgs, iters: int, every: int = 0, rec=None):
    """The whole decode loop as one CUDA graph: the block reset, then `iters` commit calls
    (iteration it on lgs[min(it, len(lgs) - 1)]), each followed by a device copy of that
    iteration's n_commit into rec[it] when rec is given.  With every = k > 0 the loop stops on
    the device: before iterations k, 2k, ... dllm_loop_continue tests the block and the rest of
    the loop is captured inside a conditional section on that test, each section nested in the
    one before, so once the block is finished the remaining iterations do not run at all (their
    rec rows keep whatever they held)."""
    g = torch.cuda.CUDAGraph()
    cap = torch.cuda.Stream()
    depth = (iters - 1) // every if every else 0
    bodies = [torch.cuda.Stream() for _ in range(depth)]  # one per nesting level
    cap.wait_stream(torch.cuda.current_stream())
    torch.cuda.synchronize()
    with torch.cuda.stream(cap):
        with torch.cuda.graph(g, stream=cap):
            gpu.state.reset()
            cur, level = cap, 0
            for it in range(iters):
                if every and it > 0 and it % every == 0:
                    h = dd.dllm_capture_condition(0, cur)
                    dd.dllm_loop_continue(gpu.state, h, cur)
                    dd.dllm_capture_if_begin(h, bodies[level], cur)
                    cur, level = bodies[level], level + 1
                with torch.cuda.stream(cur):
                    gpu.step(lgs[min(it, len(lgs) - 1)])
                    if rec is not None:
                        rec[it].copy_(gpu.state.n_commit)
            for body in reversed(bodies):
                dd.dllm_capture_if_end(body)
    torch.cuda.current_stream().wait_stream(cap)
    return g
