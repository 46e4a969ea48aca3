"""Decode state on the GPU: checkpoint/resume, determinism of the smoothing step, and capture of
the whole step in a CUDA graph."""
import numpy as np
import pytest
import torch

import synth
from gpu_runner import GpuDecoder, to_device

import diffusion_decoding_gb300 as dd

pytestmark = pytest.mark.gpu


def test_credit_state_checkpoint_resume_is_bit_identical():
    # the whole decode state is (mask, tokens, committed_now, n_commit, eos_hit, candidate ids,
    # credits): 12 steps, copy it to the host, reload it into fresh buffers, 12 more steps
    w = synth.WORKLOADS["credit_loop"].scaled(B=4, L=32, V=9000, max_iters=24)
    lgs = [to_device(synth.logits(w, seed=55, it=i, calibrated=True)) for i in range(24)]
    straight = GpuDecoder(w)
    for lg in lgs:
        straight.step(lg)
    first = GpuDecoder(w)
    for lg in lgs[:12]:
        first.step(lg)
    saved = {k: v.cpu().clone() for k, v in vars(first.state).items() if torch.is_tensor(v)}
    resumed = GpuDecoder(w)
    for k, v in saved.items():
        getattr(resumed.state, k).copy_(v)
    for lg in lgs[12:]:
        resumed.step(lg)
    a, b = straight.host_state(), resumed.host_state()
    for k in a:
        assert np.array_equal(a[k], b[k]), k


@pytest.mark.parametrize("B,L,K", [(1, 1, 1), (3, 100, 8), (64, 1024, 16)])
def test_block_state_reset_gives_a_fresh_block(B, L, K):
    # every array scribbled over, then one reset: the oracle's fresh state, exactly
    import oracle
    st = dd.BlockState(B, L, K)
    g = torch.Generator(device="cuda").manual_seed(B * L + K)
    for t in (st.masked, st.committed_now):
        t.copy_(torch.randint(0, 256, t.shape, generator=g, device="cuda").to(t.dtype))
    for t in (st.tokens, st.n_commit, st.eos_hit, st.cand_id):
        t.copy_(torch.randint(-9, 99999, t.shape, generator=g, device="cuda").to(t.dtype))
    st.cand_credit.uniform_(0.0, 3.0, generator=g)
    st.reset()
    ref = oracle.BlockState(B, L, K)
    for k in ("masked", "tokens", "committed_now", "n_commit", "eos_hit", "cand_id"):
        assert np.array_equal(getattr(st, k).cpu().numpy().reshape(getattr(ref, k).shape),
                              getattr(ref, k)), k
    assert np.array_equal(st.cand_credit.cpu().numpy().reshape(ref.cand_credit.shape),
                          ref.cand_credit.astype(np.float32))


def test_block_state_reset_without_credit_slots_leaves_them():
    st = dd.BlockState(2, 16, 8)
    st.cand_id.fill_(7)
    st.cand_credit.fill_(1.5)
    st.masked.zero_()
    dd.dllm_block_state_reset(st, credit=False)
    assert bool((st.masked == 1).all()) and bool((st.cand_id == 7).all())
    assert bool((st.cand_credit == 1.5).all())


def _smooth_setup(w, seed=9):
    gpu = GpuDecoder(w)
    E = synth.embedding_table(seed, w.V, w.d)
    Et = torch.empty(dd.dllm_embedding_t_elems(w.V, w.d), dtype=torch.int16, device="cuda")
    dd.dllm_prepare_embedding(torch.from_numpy(E.view(np.int16)).cuda(), Et)
    R, T = w.B * w.L, w.prefix_len + w.L
    bufs = dict(out=torch.zeros(R, w.d, device="cuda"),
                row_ids=torch.empty(R, dtype=torch.int32, device="cuda"),
                M=torch.zeros(1, dtype=torch.int32, device="cuda"),
                ws=dd.workspace(dd.dllm_smooth_workspace_bytes(gpu.shape, w.d)),
                refresh=torch.empty(w.B * T, dtype=torch.uint8, device="cuda"),
                idx=torch.empty(w.B * T, dtype=torch.int32, device="cuda"),
                count=torch.empty(w.B, dtype=torch.int32, device="cuda"))
    return gpu, Et, bufs


def _smooth_step(w, gpu, Et, b, lg):
    gpu.step(lg)
    dd.dllm_smooth_embed(lg, gpu.shape, gpu.stats, gpu.state, Et, w.d, b["out"], b["row_ids"],
                         b["M"], b["ws"])
    dd.dllm_kv_refresh_mask(gpu.state, w.prefix_len, w.window, b["refresh"], b["idx"], b["count"])


def test_smoothing_is_deterministic_with_split_k():
    # small M -> the planner splits K; partial sums are reduced in a fixed order
    w = synth.WORKLOADS["smooth_step"].scaled(B=2, L=16, V=8192, d=256, prefix_len=8)
    shape = dd.make_shape(w.B, w.L, w.V, dd.DLLM_BF16)
    assert dd.dllm_smooth_plan_info(shape, w.d)["split_k"] > 1
    lg = to_device(synth.logits(w, seed=4, calibrated=True))
    outs = []
    for _ in range(2):
        gpu, Et, b = _smooth_setup(w)
        _smooth_step(w, gpu, Et, b, lg)
        torch.cuda.synchronize()
        outs.append(b["out"].clone())
    assert torch.equal(outs[0], outs[1])


def test_whole_step_captured_in_a_cuda_graph_matches_eager():
    w = synth.WORKLOADS["smooth_step"].scaled(B=4, L=64, V=4096, d=512, prefix_len=32)
    lg = to_device(synth.logits(w, seed=6, calibrated=True))
    gpu_e, Et, be = _smooth_setup(w)
    _smooth_step(w, gpu_e, Et, be, lg)
    gpu_g, _, bg = _smooth_setup(w)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            _smooth_step(w, gpu_g, Et, bg, lg)
    g.replay()
    torch.cuda.synchronize()
    M = int(be["M"].item())
    assert int(bg["M"].item()) == M
    assert torch.equal(be["out"][:M], bg["out"][:M])
    for k in ("row_ids", "refresh", "idx", "count"):
        assert torch.equal(be[k], bg[k]), k
    a, b = gpu_e.host_state(), gpu_g.host_state()
    for k in ("masked", "tokens", "committed_now"):
        assert np.array_equal(a[k], b[k]), k
