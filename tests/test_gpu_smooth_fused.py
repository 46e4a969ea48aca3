"""GPU vs oracle: single-read smoothing (dllm_commit_threshold_smooth), the threshold commit and
the iteration smoothing of one step with every logit read from HBM once."""
import numpy as np
import pytest
import torch

import oracle
import synth
from gpu_runner import GpuDecoder, to_device
from harness import close, guarded_logits, oracle_step
from test_gpu_smooth import _table, lane_group_sample, smooth_close

import diffusion_decoding_gb300 as dd

pytestmark = pytest.mark.gpu


def _layout(lg: np.ndarray, stride: int, offset: int) -> torch.Tensor:
    """Rows of lg at `stride` elements, starting `offset` elements into a device buffer; the gaps
    hold huge values that must never be read."""
    B, L, V = lg.shape
    pad = np.uint16(0x7F7F) if lg.dtype == np.uint16 else np.float32(3e38)
    buf = np.full(offset + B * L * stride, pad, lg.dtype)
    buf[offset:].reshape(B * L, stride)[:, :V] = lg.reshape(B * L, V)
    return to_device(buf)[offset:]


def _fused_case(w, seed, calibrated, sample_rows=None, masked0=None, eos0=None,
                padded=False, stride=None, offset=0, ws=None):
    gpu = GpuDecoder(w)
    ost = oracle.BlockState(w.B, w.L)
    if masked0 is not None:
        ost.masked[:] = masked0
        gpu.state.masked.copy_(torch.from_numpy(masked0.reshape(-1)).cuda())
    if eos0 is not None:  # sequences already stopped: nothing of theirs is read or smoothed
        ost.eos_hit[:] = eos0
        gpu.state.eos_hit.copy_(torch.from_numpy(eos0.astype(np.int32)).cuda())
    lg, _, s = guarded_logits(w, seed, 0, ost, calibrated)
    rows_read = np.flatnonzero(oracle.active_rows(ost.masked, ost.eos_hit))
    s_ref, _ = oracle_step(w, ost, lg, s)
    E, Et = _table(w.V, w.d)
    R = w.B * w.L
    out = torch.full((R, w.d), float("nan"), dtype=torch.float32, device="cuda")
    row_ids = torch.empty(R, dtype=torch.int32, device="cuda")
    M = torch.zeros(1, dtype=torch.int32, device="cuda")
    if ws is None:
        ws = dd.workspace(dd.dllm_smooth_workspace_bytes(gpu.shape, w.d))
    dt = dd.DLLM_BF16 if w.dtype == "bf16" else dd.DLLM_F32
    shape, lgd = gpu.shape, to_device(lg)
    if padded:  # rows padded by 8 elements holding huge values that must never be read
        stride = w.V + 8
    if stride is not None or offset:
        stride = w.V if stride is None else stride
        lgd = _layout(lg, stride, offset)
        shape = dd.make_shape(w.B, w.L, w.V, dt, row_stride=stride)
    dd.dllm_commit_threshold_smooth(lgd, shape, gpu.stats, gpu.state, w.tau,
                                    w.eos_id, Et, w.d, out, row_ids, M, ws)
    torch.cuda.synchronize()
    assert dd.dllm_get_status(ws) == dd.DLLM_OK
    hs = gpu.host_state()
    for k in ("masked", "tokens", "committed_now", "n_commit"):
        assert np.array_equal(hs[k], getattr(ost, k)), k
    st = gpu.host_stats()
    assert np.array_equal(st["argmax"], s_ref.argmax)
    assert np.array_equal(st["row_max"], s_ref.row_max.astype(np.float32))
    for k in ("lse", "conf"):
        assert close(st[k], getattr(s_ref, k)), k
    ids_ref = oracle.smooth_rows(ost.masked, ost.eos_hit)
    Mg = int(M.item())
    assert Mg == len(ids_ref)
    rid = row_ids.cpu().numpy()
    assert np.array_equal(rid[:Mg], ids_ref) and (rid[Mg:] == -1).all()
    o = out.cpu().numpy()
    assert np.isnan(o[Mg:]).all(), "rows >= M must stay untouched"
    # the single-read call's GEMM rows are the rows read (before the commit), in order
    js = np.arange(Mg) if sample_rows is None else lane_group_sample(
        np.searchsorted(rows_read, ids_ref))
    ids = ids_ref[js].astype(np.int32)
    ref = oracle.smooth_embed(lg.reshape(R, w.V), s_ref.lse, ids, E)
    scale = oracle.smooth_embed(lg.reshape(R, w.V), s_ref.lse, ids, E & np.uint16(0x7FFF))
    smooth_close(o[js], ref, scale)
    return Mg


@pytest.mark.parametrize("B,L,V,d", [
    (1, 8, 1024, 32),        # one CTA per row (no cluster exchange)
    (3, 100, 2056, 160),     # ragged row tile, V not a multiple of 64
    (2, 64, 20000, 272),     # clusters of 2 CTAs per row
    (4, 64, 126464, 512),    # clusters of 8 CTAs per row (the full vocabulary)
])
def test_fused_small_all_rows(B, L, V, d):
    w = synth.WORKLOADS["smooth_step"].scaled(B=B, L=L, V=V, d=d, prefix_len=16)
    assert _fused_case(w, seed=B * 1000 + V, calibrated=True) > 0


@pytest.mark.parametrize("d", [16, 65536])
def test_fused_embedding_width_limits(d):
    # the narrowest table (one 16-wide column tile) and the widest the call takes (4096 column
    # tiles of 16 columns per 256-wide pair tile)
    w = synth.WORKLOADS["smooth_step"].scaled(B=1, L=16, V=1024, d=d, prefix_len=4)
    assert _fused_case(w, seed=d, calibrated=True) > 0


@pytest.mark.parametrize("V,dtype", [
    (1000, "bf16"),    # one CTA per row, a partial last 64-element slab
    (20008, "bf16"),   # clusters of 2, the second CTA's slice ends inside a slab
    (8200, "f32"),     # clusters of 2 over fp32 rows
    (8, "f32"),        # a row of two vectors (smoothing needs V a multiple of 8)
    (150000, "bf16"),  # rows longer than 8 x 16384 elements: the shared-memory (wide) form
    (140000, "f32"),
])
def test_fused_ragged_vocab_padded_stride(V, dtype):
    w = synth.WORKLOADS["smooth_step"].scaled(B=2, L=40, V=V, d=48, prefix_len=4, dtype=dtype)
    assert _fused_case(w, seed=V, calibrated=V > 16, padded=True) > 0


@pytest.mark.parametrize("V,dtype,extra,offset", [
    (1001, "bf16", 0, 0),     # V not a multiple of 8
    (20000, "bf16", 3, 0),    # an odd row stride
    (20000, "bf16", 0, 1),    # rows one element off 16-byte alignment
    (8191, "f32", 1, 1),      # all three, fp32
    (126464, "bf16", 1, 0),   # the full vocabulary at an odd stride
])
def test_fused_unaligned_rows_take_the_elementwise_path(V, dtype, extra, offset):
    # rows the single-read kernels cannot copy whole: same results through the element-wise
    # statistics and probability kernels
    w = synth.WORKLOADS["smooth_step"].scaled(B=2, L=24, V=V, d=64, prefix_len=4, dtype=dtype)
    assert _fused_case(w, seed=V + extra, calibrated=True, stride=V + extra, offset=offset) > 0


def test_fused_partial_mask_and_fp32():
    w = synth.WORKLOADS["smooth_step"].scaled(B=2, L=48, V=8192, d=64, dtype="f32",
                                              prefix_len=8)
    rng = np.random.default_rng(7)
    m0 = (rng.random((w.B, w.L)) < 0.6).astype(np.uint8)
    assert _fused_case(w, seed=5, calibrated=True, masked0=m0) > 0


def test_fused_full_size_sampled_rows():
    w = synth.WORKLOADS["smooth_step"]
    Mg = _fused_case(w, synth.workloads.SEEDS[w.key], calibrated=False, sample_rows="lanes")
    assert Mg == w.B * w.L - w.B


def test_fused_with_a_stopped_sequence():
    w = synth.WORKLOADS["smooth_step"].scaled(B=3, L=32, V=20000, d=128, prefix_len=8)
    eos0 = np.array([0, 1, 0], np.int32)
    Mg = _fused_case(w, seed=9, calibrated=True, eos0=eos0)
    assert 0 < Mg < 2 * w.L


def test_fused_step_on_a_finished_block_then_reset():
    # nothing is masked: no row is read, M = 0 and every GEMM CTA pair leaves at once.  A block
    # reset launched right behind the step must not overtake the step's kept-row map, which
    # still reads the (finished) block state: M stays 0 and every row id -1, call after call.
    w = synth.WORKLOADS["smooth_step"].scaled(B=4, L=64, V=20000, d=256, prefix_len=8)
    gpu = GpuDecoder(w)
    E, Et = _table(w.V, w.d)
    R = w.B * w.L
    lg = to_device(synth.logits(w, seed=3, calibrated=True))
    out = torch.full((R, w.d), float("nan"), dtype=torch.float32, device="cuda")
    row_ids = torch.zeros(R, dtype=torch.int32, device="cuda")
    M = torch.full((1,), 99, dtype=torch.int32, device="cuda")
    ws = dd.workspace(dd.dllm_smooth_workspace_bytes(gpu.shape, w.d))
    for _ in range(20):
        gpu.state.masked.zero_()
        dd.dllm_commit_threshold_smooth(lg, gpu.shape, gpu.stats, gpu.state, w.tau, w.eos_id, Et,
                                        w.d, out, row_ids, M, ws)
        gpu.state.reset()
        torch.cuda.synchronize()
        assert int(M.item()) == 0
        assert bool((row_ids == -1).all())
        assert bool((gpu.state.masked == 1).all())
    assert bool(torch.isnan(out).all()), "no output row may be written"
    assert dd.dllm_get_status(ws) == dd.DLLM_OK


def test_fused_calls_share_a_workspace_across_shapes():
    # One smoothing workspace, sized for the largest shape, serves calls of three shapes in turn,
    # twice (the first shape's plan splits K: partial sums in the workspace, added in a fixed
    # order); every call matches the oracle.
    shapes = [dict(B=4, L=64, V=126464, d=512), dict(B=2, L=64, V=20000, d=272),
              dict(B=3, L=100, V=2056, d=160)]
    ws_list = [synth.WORKLOADS["smooth_step"].scaled(prefix_len=16, **kw) for kw in shapes]
    need = max(dd.dllm_smooth_workspace_bytes(GpuDecoder(w).shape, w.d) for w in ws_list)
    ws = dd.workspace(need)
    assert dd.dllm_smooth_plan_info(GpuDecoder(ws_list[0]).shape, ws_list[0].d)["split_k"] > 1
    for rep in range(2):
        for i, w in enumerate(ws_list):
            assert _fused_case(w, seed=100 * rep + i, calibrated=True, ws=ws) > 0
    assert dd.dllm_get_status(ws) == dd.DLLM_OK
