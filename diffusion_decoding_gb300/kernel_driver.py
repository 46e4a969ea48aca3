"""Run one kernel family of the decode step a fixed number of times, for external profilers.

    python -m diffusion_decoding_gb300.kernel_driver {stats|probs|gemm|step|fused} [n [B L]]

The inputs have the smoothing-step sizes (B=16, L=64, V=126464 bf16 logits, d=2048 embedding
table; about 0.8 GB on the device), so every launch reads more than the L2 holds; `stats`
takes another block shape as B and L (every position masked, as in a loop's first
iteration).  Nothing is timed here: a profiler (ncu) attaches to the launches.  `stats` runs
the fused statistics + threshold commit; `probs` the probability rows; `gemm` the smoothing
GEMM (after one probability pass); `step` the whole step (commit, probabilities, GEMM, KV
refresh) through the separate calls; `fused` the whole step through the single-read call.
"""
import sys

import torch

import diffusion_decoding_gb300 as dd

B_, L_, V, D = 16, 64, 126464, 2048
PREFIX, WINDOW, TAU = 1024, 4, 0.9


def main(argv) -> None:
    what = argv[0] if argv else "step"
    n = int(argv[1]) if len(argv) > 1 else 4
    if what not in ("stats", "probs", "gemm", "step", "fused"):
        raise SystemExit(f"unknown kernel family {what!r}")
    B, L = (int(argv[2]), int(argv[3])) if what == "stats" and len(argv) > 3 else (B_, L_)
    dev = torch.device("cuda")
    g = torch.Generator(device=dev)
    g.manual_seed(7)
    shape = dd.make_shape(B, L, V, dd.DLLM_BF16)
    lg = torch.randn(B, L, V, device=dev, generator=g).mul_(2).to(torch.bfloat16)
    state, stats = dd.BlockState(B, L), dd.StatsBuffers(B * L)
    ws = dd.workspace(dd.dllm_workspace_bytes(shape))
    if what == "stats":
        for _ in range(n):
            state.reset()
            dd.dllm_commit_threshold(lg, shape, stats, state, TAU, -1, ws)
        torch.cuda.synchronize()
        return
    Et = torch.randn(dd.dllm_embedding_t_elems(V, D), device=dev, generator=g)
    Et = Et.mul_(0.02).to(torch.bfloat16)
    ws_s = dd.workspace(dd.dllm_smooth_workspace_bytes(shape, D))
    out = torch.empty(B * L, D, device=dev)
    row_ids = torch.empty(B * L, dtype=torch.int32, device=dev)
    M = torch.zeros(1, dtype=torch.int32, device=dev)
    T = PREFIX + L
    refresh = torch.empty(B * T, dtype=torch.uint8, device=dev)
    idx = torch.empty(B * T, dtype=torch.int32, device=dev)
    count = torch.empty(B, dtype=torch.int32, device=dev)
    state.reset()
    dd.dllm_commit_threshold(lg, shape, stats, state, TAU, -1, ws)
    if what == "gemm":
        dd.dllm_smooth_probs(lg, shape, stats, state, D, row_ids, M, ws_s)
    for _ in range(n):
        if what == "probs":
            dd.dllm_smooth_probs(lg, shape, stats, state, D, row_ids, M, ws_s)
        elif what == "gemm":
            dd.dllm_smooth_gemm(shape, Et, D, out, M, ws_s)
        elif what == "fused":
            state.reset()
            dd.dllm_commit_threshold_smooth(lg, shape, stats, state, TAU, -1, Et, D, out,
                                            row_ids, M, ws_s)
            dd.dllm_kv_refresh_mask(state, PREFIX, WINDOW, refresh, idx, count)
        else:
            state.reset()
            dd.dllm_commit_threshold(lg, shape, stats, state, TAU, -1, ws)
            dd.dllm_smooth_probs(lg, shape, stats, state, D, row_ids, M, ws_s)
            dd.dllm_smooth_gemm(shape, Et, D, out, M, ws_s)
            dd.dllm_kv_refresh_mask(state, PREFIX, WINDOW, refresh, idx, count)
    torch.cuda.synchronize()
    if dd.dllm_get_status(ws_s) != dd.DLLM_OK:
        raise SystemExit("smoothing reported an error status")


if __name__ == "__main__":
    main(sys.argv[1:])
    print("ok")
