"""GPU vs oracle: iteration smoothing (probability rows + tcgen05 GEMM) and the KV refresh."""
import numpy as np
import pytest
import torch

import oracle
import synth
from gpu_runner import GpuDecoder, to_device
from harness import guarded_logits, oracle_step

import diffusion_decoding_gb300 as dd

pytestmark = pytest.mark.gpu


def smooth_close(g: np.ndarray, o: np.ndarray, scale: np.ndarray, rtol=2e-3) -> None:
    """Per element |g-o| <= rtol * sum_v P_v |E_v,c| (the magnitude of the terms summed: an
    entry that is a near-cancelling sum has no meaningful relative error of its own); per row
    relative L2 <= rtol."""
    g = np.asarray(g, np.float64)
    bound = rtol * scale
    bad = np.abs(g - o) > bound
    assert not bad.any(), f"{bad.sum()} elements outside the bound; worst " \
                          f"{np.max(np.abs(g - o) / np.maximum(bound, 1e-30)):.3g}x"
    rel = np.linalg.norm(g - o, axis=1) / np.maximum(np.linalg.norm(o, axis=1), 1e-30)
    assert (rel <= rtol).all(), rel.max()


def lane_group_sample(gemm_rows: np.ndarray) -> np.ndarray:
    """Kept-row indices to check at full size: two per 32-row group of the GEMM's rows (the
    rows of one TMEM lane quarter, read back by one epilogue warp), so every epilogue warp of
    every CTA of every row pair is checked.  gemm_rows[j] is the GEMM row of kept row j."""
    groups = np.asarray(gemm_rows) // 32
    sel = []
    for g in np.unique(groups):
        js = np.flatnonzero(groups == g)
        sel += [int(js[0]), int(js[len(js) // 2])]
    return np.unique(np.array(sel, np.int64))


def _table(V, d, seed=77):
    E = synth.embedding_table(seed, V, d)
    Et = torch.empty(dd.dllm_embedding_t_elems(V, d), dtype=torch.int16, device="cuda")
    dd.dllm_prepare_embedding(torch.from_numpy(E.view(np.int16)).cuda(), Et)
    return E, Et


def _smooth_case(w, seed, calibrated, sample_rows=None):
    """One full step: threshold commit, smoothing, refresh; returns GPU and oracle results."""
    gpu = GpuDecoder(w)
    ost = oracle.BlockState(w.B, w.L)
    lg, _, s = guarded_logits(w, seed, 0, ost, calibrated)
    s_ref, _ = oracle_step(w, ost, lg, s)
    E, Et = _table(w.V, w.d)
    R = w.B * w.L
    out = torch.full((R, w.d), float("nan"), dtype=torch.float32, device="cuda")
    row_ids = torch.empty(R, dtype=torch.int32, device="cuda")
    M = torch.zeros(1, dtype=torch.int32, device="cuda")
    ws_s = dd.workspace(dd.dllm_smooth_workspace_bytes(gpu.shape, w.d))
    T = w.prefix_len + w.L
    refresh = torch.empty(w.B * T, dtype=torch.uint8, device="cuda")
    idx = torch.empty(w.B * T, dtype=torch.int32, device="cuda")
    count = torch.empty(w.B, dtype=torch.int32, device="cuda")
    lgd = to_device(lg)
    gpu.step(lgd)
    dd.dllm_smooth_embed(lgd, gpu.shape, gpu.stats, gpu.state, Et, w.d, out, row_ids, M, ws_s)
    dd.dllm_kv_refresh_mask(gpu.state, w.prefix_len, w.window, refresh, idx, count)
    torch.cuda.synchronize()
    assert dd.dllm_get_status(ws_s) == dd.DLLM_OK
    # commits, rows, refresh: exact
    hs = gpu.host_state()
    for k in ("masked", "tokens", "committed_now", "n_commit"):
        assert np.array_equal(hs[k], getattr(ost, k)), k
    ids_ref = oracle.smooth_rows(ost.masked, ost.eos_hit)
    Mg = int(M.item())
    assert Mg == len(ids_ref)
    rid = row_ids.cpu().numpy()
    assert np.array_equal(rid[:Mg], ids_ref) and (rid[Mg:] == -1).all()
    ref_r, ref_i, ref_c = oracle.kv_refresh(ost.committed_now, w.prefix_len, w.window)
    assert np.array_equal(refresh.cpu().numpy().reshape(w.B, T), ref_r)
    assert np.array_equal(idx.cpu().numpy().reshape(w.B, T), ref_i)
    assert np.array_equal(count.cpu().numpy(), ref_c)
    # soft embeddings: all rows or a sample, against the oracle's own lse
    o = out.cpu().numpy()
    assert np.isnan(o[Mg:]).all(), "rows >= M must stay untouched"
    # the separate smoothing call's GEMM rows are the kept rows themselves
    js = np.arange(Mg) if sample_rows is None else lane_group_sample(np.arange(Mg))
    ids = ids_ref[js].astype(np.int32)
    ref = oracle.smooth_embed(lg.reshape(R, w.V), s_ref.lse, ids, E)
    scale = oracle.smooth_embed(lg.reshape(R, w.V), s_ref.lse, ids, E & np.uint16(0x7FFF))
    smooth_close(o[js], ref, scale)
    return Mg


@pytest.mark.parametrize("B,L,V,d", [
    (1, 8, 1024, 32),        # one row tile, one column tile
    (3, 100, 2056, 160),     # 3 row tiles with a ragged last one, V not a multiple of 64
    (2, 64, 4096, 272),      # column tiles of unequal widths
    (4, 64, 6000, 2048),     # full embedding width
])
def test_smooth_small_all_rows(B, L, V, d):
    w = synth.WORKLOADS["smooth_step"].scaled(B=B, L=L, V=V, d=d, prefix_len=16)
    Mg = _smooth_case(w, seed=B * 1000 + V, calibrated=True)
    assert Mg > 0


def test_smooth_step_full_sampled_rows():
    w = synth.WORKLOADS["smooth_step"]
    Mg = _smooth_case(w, synth.workloads.SEEDS[w.key], calibrated=False, sample_rows="lanes")
    assert Mg == w.B * w.L - w.B  # literal workload: one fallback commit per sequence


@pytest.mark.parametrize("V,dtype,extra,offset", [
    (1001, "bf16", 0, 0),     # V not a multiple of 8
    (20000, "bf16", 3, 1),    # an odd row stride, rows one element off alignment
    (8191, "f32", 1, 1),
])
def test_smooth_unaligned_rows(V, dtype, extra, offset):
    # the separate calls (commit, then probabilities + GEMM) on rows that are not 16-byte
    # aligned: the probability rows are read element by element; same results as the oracle
    from test_gpu_smooth_fused import _layout
    w = synth.WORKLOADS["smooth_step"].scaled(B=2, L=24, V=V, d=64, prefix_len=4, dtype=dtype)
    ost = oracle.BlockState(w.B, w.L)
    lg, _, s = guarded_logits(w, V, 0, ost, True)
    s_ref, _ = oracle_step(w, ost, lg, s)
    E, Et = _table(w.V, w.d)
    R = w.B * w.L
    dt = dd.DLLM_BF16 if dtype == "bf16" else dd.DLLM_F32
    shape = dd.make_shape(w.B, w.L, V, dt, row_stride=V + extra)
    lgd = _layout(lg, V + extra, offset)
    state, stats = dd.BlockState(w.B, w.L), dd.StatsBuffers(R)
    ws = dd.workspace(dd.dllm_workspace_bytes(shape))
    ws_s = dd.workspace(dd.dllm_smooth_workspace_bytes(shape, w.d))
    out = torch.full((R, w.d), float("nan"), dtype=torch.float32, device="cuda")
    row_ids = torch.empty(R, dtype=torch.int32, device="cuda")
    M = torch.zeros(1, dtype=torch.int32, device="cuda")
    dd.dllm_commit_threshold(lgd, shape, stats, state, w.tau, w.eos_id, ws)
    dd.dllm_smooth_embed(lgd, shape, stats, state, Et, w.d, out, row_ids, M, ws_s)
    torch.cuda.synchronize()
    assert np.array_equal(state.masked.cpu().numpy().reshape(w.B, w.L), ost.masked)
    ids_ref = oracle.smooth_rows(ost.masked, ost.eos_hit)
    Mg = int(M.item())
    assert Mg == len(ids_ref) and np.array_equal(row_ids.cpu().numpy()[:Mg], ids_ref)
    o = out.cpu().numpy()
    assert np.isnan(o[Mg:]).all()
    ids = ids_ref.astype(np.int32)
    ref = oracle.smooth_embed(lg.reshape(R, V), s_ref.lse, ids, E)
    scale = oracle.smooth_embed(lg.reshape(R, V), s_ref.lse, ids, E & np.uint16(0x7FFF))
    smooth_close(o[:Mg], ref, scale)


def test_smooth_skips_when_nothing_is_masked():
    w = synth.WORKLOADS["smooth_step"].scaled(B=2, L=8, V=1024, d=32)
    gpu = GpuDecoder(w)
    gpu.state.masked.zero_()
    E, Et = _table(w.V, w.d)
    out = torch.full((16, 32), 7.0, device="cuda")
    row_ids = torch.empty(16, dtype=torch.int32, device="cuda")
    M = torch.full((1,), 99, dtype=torch.int32, device="cuda")
    ws = dd.workspace(dd.dllm_smooth_workspace_bytes(gpu.shape, w.d))
    lg = to_device(synth.logits(w, seed=1))
    dd.dllm_decode_stats(lg, gpu.shape, None, gpu.stats, gpu.ws)
    dd.dllm_smooth_embed(lg, gpu.shape, gpu.stats, gpu.state, Et, w.d, out, row_ids, M, ws)
    torch.cuda.synchronize()
    assert int(M.item()) == 0 and (row_ids.cpu() == -1).all() and (out.cpu() == 7.0).all()


def test_embedding_relayout_is_a_blocked_transpose():
    V, d = 1001, 48
    E, Et = _table(V, d)
    Vp = dd.dllm_embedding_t_elems(V, d) // d
    assert Vp == 1024
    # Et[(v // 64) * d + c][v % 64] = E[v][c]
    et = Et.cpu().numpy().view(np.uint16).reshape(Vp // 64, d, 64)
    full = et.transpose(1, 0, 2).reshape(d, Vp)
    assert np.array_equal(full[:, :V], E.T) and (full[:, V:] == 0).all()


@pytest.mark.parametrize("B,L,P,w", [(1, 1, 0, 0), (3, 64, 1024, 4), (2, 300, 5, 9),
                                     (4, 1024, 0, 1), (2, 16, 3, 40)])
def test_kv_refresh_random_patterns(B, L, P, w):
    rng = np.random.default_rng(B * L + P)
    com = (rng.random((B, L)) < 0.1).astype(np.uint8)
    com[0, :] = 0  # one sequence with no commit
    state = dd.BlockState(B, L)
    state.committed_now.copy_(torch.from_numpy(com.reshape(-1)))
    T = P + L
    refresh = torch.empty(B * T, dtype=torch.uint8, device="cuda")
    idx = torch.empty(B * T, dtype=torch.int32, device="cuda")
    count = torch.empty(B, dtype=torch.int32, device="cuda")
    dd.dllm_kv_refresh_mask(state, P, w, refresh, idx, count)
    r, i, c = oracle.kv_refresh(com, P, w)
    assert np.array_equal(refresh.cpu().numpy().reshape(B, T), r)
    assert np.array_equal(idx.cpu().numpy().reshape(B, T), i)
    assert np.array_equal(count.cpu().numpy(), c)


def test_bounded_wait_times_out_and_reports_status():
    # a wait that nothing satisfies gives up after its limit and records DLLM_ERR_TIMEOUT; the
    # context stays usable and the status word resets once read
    ws = dd.workspace(256)
    dd.dllm_selftest_wait_timeout(ws, 20000)  # 20 ms
    assert dd.dllm_get_status(ws) == dd.DLLM_ERR_TIMEOUT
    assert dd.dllm_get_status(ws) == dd.DLLM_OK
    x = torch.ones(4, device="cuda")
    assert float((x * 2).sum().item()) == 8.0
