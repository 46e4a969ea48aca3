"""GPU vs oracle: statistics and the three commit strategies, element by element.

Small cases span several vocabulary slices with ragged tails; the full cases are the five
workloads at their stated sizes, in the launch configuration the benchmark uses.
"""
import numpy as np
import pytest
import torch

import oracle
import synth
from gpu_runner import GpuDecoder, capture_loop, to_device
from harness import close, guarded_logits, oracle_step

import diffusion_decoding_gb300 as dd

pytestmark = pytest.mark.gpu


def _compare_step(gpu: GpuDecoder, ost: oracle.BlockState, os_, scores=None, tag=""):
    hs = gpu.host_state()
    for k in ("masked", "tokens", "committed_now", "n_commit", "eos_hit"):
        assert np.array_equal(hs[k], getattr(ost, k)), f"{tag}: {k} differs"
    st = gpu.host_stats()
    assert np.array_equal(st["argmax"], os_.argmax), f"{tag}: argmax differs"
    assert close(st["row_max"], os_.row_max, 0.0), f"{tag}: row_max differs"
    assert close(st["lse"], os_.lse), f"{tag}: lse differs"
    assert close(st["conf"], os_.conf), f"{tag}: conf differs"
    if gpu.w.strategy == "credit":
        assert np.array_equal(hs["cand_id"], ost.cand_id), f"{tag}: candidate ids differ"
        assert close(hs["cand_credit"], ost.cand_credit), f"{tag}: credits differ"


def _run_loop(w, seed, calibrated=False, max_iters=None, graph=False):
    """Eager loop checked against the oracle after every iteration.  With graph=True the same
    loop is then run once more as one CUDA graph (below) on the same device logits."""
    gpu = GpuDecoder(w)
    ost = oracle.BlockState(w.B, w.L, w.K)
    iters = w.max_iters if max_iters is None else max_iters
    n_done = 0
    kept, n_commits = [], []
    for it in range(iters):
        running = ((ost.masked.sum(1) > 0) & (ost.eos_hit == 0)).any()
        if not running:
            break
        lg, _, s = guarded_logits(w, seed, it, ost, calibrated)
        s_ref, scores = oracle_step(w, ost, lg, s)
        lgd = to_device(lg)
        gpu.step(lgd)
        torch.cuda.synchronize()
        _compare_step(gpu, ost, s_ref, scores, tag=f"{w.key} iter {it}")
        n_done += 1
        if graph:
            kept.append(lgd)
            n_commits.append(ost.n_commit.copy())
    if graph:
        _graph_loop_matches_oracle(w, kept, ost, np.array(n_commits), iters)
    return gpu, ost, n_done


def _graph_loop_matches_oracle(w, lgs, ost, n_commits, iters):
    """The whole decode loop as one CUDA graph (dInfer explainer, system optimisations: CUDA
    graphs and loop unrolling keep the host out of the iterations), plain and stopping on the
    device (a continue test every 4 iterations, and every iteration on short loops).  Each form
    is replayed twice over a scribbled state; iteration it records its n_commit in rec[it].
    Iterations after the oracle's loop has ended reuse its last logits: every sequence is
    stopped by then, so an iteration that runs must commit nothing, and with the device stop
    only the iterations up to the next test after the end may run (the rest keep the fill
    value).  The final state and every recorded n_commit must equal the oracle trajectory's."""
    n = len(n_commits)
    forms = [0, 4] + ([1] if iters <= 24 else [])
    for every in forms:
        gpu = GpuDecoder(w)
        rec = torch.empty((iters, w.B), dtype=torch.int32, device="cuda")
        g = capture_loop(gpu, lgs, iters, every, rec)
        tag = f"{w.key} graph (test every {every})"
        # with a test every k iterations, the iterations after the end that still run are
        # those before the first test that comes after the end
        ran_to = iters if every == 0 else min(iters, -(-n // every) * every)
        for rep in range(2):
            st = gpu.state
            st.masked.zero_()
            st.tokens.fill_(12345)
            st.eos_hit.fill_(1)
            st.cand_id.fill_(7)
            st.cand_credit.fill_(2.5)
            rec.fill_(-7)
            g.replay()
            torch.cuda.synchronize()
            hs = gpu.host_state()
            for k in ("masked", "tokens", "eos_hit"):
                assert np.array_equal(hs[k], getattr(ost, k)), f"{tag} {rep}: {k} differs"
            if w.strategy == "credit":
                assert np.array_equal(hs["cand_id"], ost.cand_id), f"{tag} {rep}: candidate ids"
                assert close(hs["cand_credit"], ost.cand_credit), f"{tag} {rep}: credits"
            got = rec.cpu().numpy()
            assert np.array_equal(got[:n], n_commits), f"{tag} {rep}: n_commit per iteration"
            assert (got[n:ran_to] == 0).all(), f"{tag} {rep}: iterations after the end committed"
            assert (got[ran_to:] == -7).all(), f"{tag} {rep}: iterations after a stop ran"


# ------------------------------------------------------------------ statistics

@pytest.mark.parametrize("V", [1, 7, 8, 9, 100, 2049, 5003, 33001, 126464])
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_stats_ragged_sizes(V, dtype):
    w = synth.WORKLOADS["threshold_loop"].scaled(B=3, L=5, V=V, dtype=dtype, eos_id=-1,
                                                  plant="fixed" if V > 16 else "none")
    lg = synth.logits(w, seed=V, it=1)
    rng = np.random.default_rng(V)
    masked = (rng.random(w.B * w.L) < 0.7).astype(np.uint8)
    ref = oracle.stats(lg, masked)
    stats = dd.StatsBuffers(w.B * w.L)
    # rows padded to a 16-byte stride (the ABI's row alignment); the padding is never read
    stride = -(-V // 8) * 8
    buf = np.full((w.B, w.L, stride), 0x7F7F if dtype == "bf16" else 3e38, lg.dtype)
    buf[:, :, :V] = lg
    shape = dd.make_shape(w.B, w.L, V, dd.DLLM_BF16 if dtype == "bf16" else dd.DLLM_F32,
                          row_stride=stride)
    ws = dd.workspace(dd.dllm_workspace_bytes(shape))
    dd.dllm_decode_stats(to_device(buf), shape, torch.from_numpy(masked).cuda(), stats, ws)
    torch.cuda.synchronize()
    assert np.array_equal(stats.argmax.cpu().numpy(), ref.argmax)
    assert close(stats.row_max.cpu().numpy(), ref.row_max, 0.0)
    assert close(stats.lse.cpu().numpy(), ref.lse)
    assert close(stats.conf.cpu().numpy(), ref.conf)
    # no mask: every row computed
    dd.dllm_decode_stats(to_device(buf), shape, None, stats, ws)
    full = oracle.stats(lg)
    assert np.array_equal(stats.argmax.cpu().numpy(), full.argmax)
    assert close(stats.conf.cpu().numpy(), full.conf)


@pytest.mark.parametrize("B,L,V,dtype,frac", [
    (16, 64, 126464, "bf16", 0.3),   # 1024 rows: the persistent grid over the rows read
    (8, 64, 126464, "bf16", 0.02),   # a nearly decided block
    (8, 64, 126464, "bf16", 0.0),    # nothing read: every row reports -inf
    (64, 64, 20001, "f32", 0.5),     # 4096 rows (the largest listed), fp32 rows read by scalar loads
    (65, 64, 20000, "bf16", 0.5),    # 4160 rows: one warp per item again
    (4, 256, 126464, "bf16", 1.0),   # every row read
])
def test_stats_over_partly_read_blocks(B, L, V, dtype, frac):
    # statistics of the rows read, and -inf for the others, when the grid is persistent and
    # its warps share out the rows read (blocks of up to 4096 rows that need more than one
    # wave of CTAs), at and beyond its size limit
    w = synth.WORKLOADS["threshold_loop"].scaled(B=B, L=L, V=V, dtype=dtype, eos_id=-1,
                                                  plant="fixed")
    lg = synth.logits(w, seed=B + L, it=1)
    rng = np.random.default_rng(B * L)
    masked = (rng.random(B * L) < frac).astype(np.uint8)
    ref = oracle.stats(lg, masked)
    stats = dd.StatsBuffers(B * L)
    stats.argmax.fill_(12345)
    shape = dd.make_shape(B, L, V, dd.DLLM_BF16 if dtype == "bf16" else dd.DLLM_F32)
    ws = dd.workspace(dd.dllm_workspace_bytes(shape))
    dd.dllm_decode_stats(to_device(lg), shape, torch.from_numpy(masked).cuda(), stats, ws)
    torch.cuda.synchronize()
    assert np.array_equal(stats.argmax.cpu().numpy(), ref.argmax)
    assert close(stats.row_max.cpu().numpy(), ref.row_max, 0.0)
    assert close(stats.lse.cpu().numpy(), ref.lse)
    assert close(stats.conf.cpu().numpy(), ref.conf)


def test_stats_padded_row_stride_and_ties():
    B, L, V, pad = 2, 3, 4000, 64
    rng = np.random.default_rng(1)
    base = rng.integers(-3, 4, size=(B * L, V)).astype(np.float32)  # many exact ties
    buf = np.zeros((B * L, V + pad), np.float32)
    buf[:, :V] = base
    buf[:, V:] = 1e4  # padding must never be read
    t = torch.from_numpy(buf).cuda()
    shape = dd.make_shape(B, L, V, dd.DLLM_F32, row_stride=V + pad)
    stats = dd.StatsBuffers(B * L)
    ws = dd.workspace(dd.dllm_workspace_bytes(shape))
    dd.dllm_decode_stats(t, shape, None, stats, ws)
    ref = oracle.stats(base)
    assert np.array_equal(stats.argmax.cpu().numpy(), ref.argmax)
    assert close(stats.lse.cpu().numpy(), ref.lse)


# ------------------------------------------------------------------ rows not 16-byte aligned

def _unaligned(lg: np.ndarray, stride: int, offset: int) -> torch.Tensor:
    """Rows of lg at `stride` elements, starting `offset` elements into a device buffer; the gaps
    hold huge values that must never be read."""
    B, L, V = lg.shape
    pad = np.uint16(0x7F7F) if lg.dtype == np.uint16 else np.float32(3e38)
    buf = np.full(offset + B * L * stride, pad, lg.dtype)
    buf[offset:].reshape(B * L, stride)[:, :V] = lg.reshape(B * L, V)
    return to_device(buf)[offset:]


@pytest.mark.parametrize("V", [1, 7, 9, 2049, 33001])
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("offset", [0, 1])
def test_stats_unaligned_rows(V, dtype, offset):
    # stride = V (odd or not a multiple of 16 bytes), logits possibly one element into a buffer
    w = synth.WORKLOADS["threshold_loop"].scaled(B=3, L=5, V=V, dtype=dtype, eos_id=-1,
                                                  plant="fixed" if V > 16 else "none")
    lg = synth.logits(w, seed=V + offset, it=1)
    rng = np.random.default_rng(V)
    masked = (rng.random(w.B * w.L) < 0.7).astype(np.uint8)
    ref = oracle.stats(lg, masked)
    stats = dd.StatsBuffers(w.B * w.L)
    shape = dd.make_shape(w.B, w.L, V, dd.DLLM_BF16 if dtype == "bf16" else dd.DLLM_F32,
                          row_stride=V)
    ws = dd.workspace(dd.dllm_workspace_bytes(shape))
    dd.dllm_decode_stats(_unaligned(lg, V, offset), shape, torch.from_numpy(masked).cuda(),
                         stats, ws)
    torch.cuda.synchronize()
    assert np.array_equal(stats.argmax.cpu().numpy(), ref.argmax)
    assert close(stats.row_max.cpu().numpy(), ref.row_max, 0.0)
    assert close(stats.lse.cpu().numpy(), ref.lse)
    assert close(stats.conf.cpu().numpy(), ref.conf)


@pytest.mark.parametrize("key,V,extra,offset,dtype", [
    ("threshold_loop", 20001, 0, 0, "bf16"),
    ("threshold_loop", 5003, 0, 1, "f32"),
    ("hierarchical_loop", 4097, 1, 0, "bf16"),
    ("credit_loop", 9001, 3, 1, "bf16"),
])
def test_loops_on_unaligned_rows(key, V, extra, offset, dtype):
    w = synth.WORKLOADS[key].scaled(B=2, L=16, V=V, dtype=dtype, max_iters=6)
    gpu = GpuDecoder(w)
    gpu.shape = dd.make_shape(w.B, w.L, V, dd.DLLM_BF16 if dtype == "bf16" else dd.DLLM_F32,
                              row_stride=V + extra)
    ost = oracle.BlockState(w.B, w.L, w.K)
    n_done = 0
    for it in range(w.max_iters):
        if not ((ost.masked.sum(1) > 0) & (ost.eos_hit == 0)).any():
            break
        lg, _, s = guarded_logits(w, 77, it, ost, True)
        s_ref, scores = oracle_step(w, ost, lg, s)
        gpu.step(_unaligned(lg, V + extra, offset))
        torch.cuda.synchronize()
        _compare_step(gpu, ost, s_ref, scores, tag=f"{key} unaligned iter {it}")
        n_done += 1
    assert n_done >= 2


def test_stats_deterministic():
    w = synth.WORKLOADS["credit_loop"].scaled(B=4, L=8)
    lg = to_device(synth.logits(w, seed=3))
    shape = dd.make_shape(w.B, w.L, w.V, dd.DLLM_BF16)
    ws = dd.workspace(dd.dllm_workspace_bytes(shape))
    a, b = dd.StatsBuffers(w.B * w.L), dd.StatsBuffers(w.B * w.L)
    dd.dllm_decode_stats(lg, shape, None, a, ws)
    dd.dllm_decode_stats(lg, shape, None, b, ws)
    for k in ("row_max", "lse", "conf", "argmax"):
        assert torch.equal(getattr(a, k), getattr(b, k))


# ------------------------------------------------------------------ the five workloads

def test_threshold_single_step_full():
    w = synth.WORKLOADS["threshold_single"]
    gpu, ost, n = _run_loop(w, synth.workloads.SEEDS[w.key])
    assert n == 1 and ost.n_commit[0] >= 1


def test_threshold_loop_full():
    w = synth.WORKLOADS["threshold_loop"]
    gpu, ost, n = _run_loop(w, synth.workloads.SEEDS[w.key], graph=True)
    assert n >= 1


@pytest.mark.parametrize("seed", [5, 6])
def test_threshold_loop_calibrated_small(seed):
    w = synth.WORKLOADS["threshold_loop"].scaled(B=4, L=32, V=20000)
    gpu, ost, n = _run_loop(w, seed, calibrated=True, graph=True)
    assert n >= 2


def test_hierarchical_loop_full():
    w = synth.WORKLOADS["hierarchical_loop"]
    gpu, ost, n = _run_loop(w, synth.workloads.SEEDS[w.key], graph=True)
    assert ost.masked.sum() == 0


@pytest.mark.parametrize("L,min_width", [(64, 2), (100, 3), (33, 1)])
def test_hierarchical_calibrated_small(L, min_width):
    w = synth.WORKLOADS["hierarchical_loop"].scaled(B=5, L=L, V=8200, min_width=min_width,
                                                     max_iters=L)
    gpu, ost, n = _run_loop(w, 40 + L, calibrated=True, graph=True)
    assert ost.masked.sum() == 0


def test_credit_loop_full():
    w = synth.WORKLOADS["credit_loop"]
    gpu, ost, n = _run_loop(w, synth.workloads.SEEDS[w.key], graph=True)
    assert n == w.max_iters


@pytest.mark.parametrize("K", [8, 3, 16])
def test_credit_calibrated_small(K):
    w = synth.WORKLOADS["credit_loop"].scaled(B=6, L=24, V=12000, K=K, max_iters=20)
    gpu, ost, n = _run_loop(w, 70 + K, calibrated=True, graph=True)
    assert n >= 5


def test_large_block_epilogue():
    # L = 1024 positions: the epilogue loops 4 positions per thread, scans cross 8 warps.
    # The planted-peak recipe (not the calibrated one) keeps 2048 confidences clear of tau_low.
    w = synth.WORKLOADS["hierarchical_loop"].scaled(B=2, L=1024, V=2048, max_iters=3)
    _run_loop(w, 90, calibrated=False)


# ------------------------------------------------------------------ edge cases

@pytest.mark.parametrize("B,L,V,dtype", [(1024, 1024, 8, "bf16"), (2, 3, 2, "f32")])
def test_extreme_shapes_statistics_and_commit(B, L, V, dtype):
    # the most rows a call takes (B*L = 2^20, L = 1024) and the smallest vocabulary: statistics
    # of every row against the oracle, then a threshold no confidence reaches from below
    # (tau = -1: every masked position commits its argmax), so no decision rests on rounding
    w = synth.WORKLOADS["threshold_loop"].scaled(B=B, L=L, V=V, dtype=dtype, eos_id=-1,
                                                  plant="none")
    lg = synth.logits(w, seed=B + V, it=0)
    rng = np.random.default_rng(B + V)
    masked = (rng.random(B * L) < 0.8).astype(np.uint8)
    ref = oracle.stats(lg, masked)
    shape = dd.make_shape(B, L, V, dd.DLLM_BF16 if dtype == "bf16" else dd.DLLM_F32)
    ws = dd.workspace(dd.dllm_workspace_bytes(shape))
    stats = dd.StatsBuffers(B * L)
    lgd = to_device(lg)
    dd.dllm_decode_stats(lgd, shape, torch.from_numpy(masked).cuda(), stats, ws)
    torch.cuda.synchronize()
    assert np.array_equal(stats.argmax.cpu().numpy(), ref.argmax)
    assert close(stats.row_max.cpu().numpy(), ref.row_max, 0.0)
    assert close(stats.lse.cpu().numpy(), ref.lse)
    assert close(stats.conf.cpu().numpy(), ref.conf)
    state = dd.BlockState(B, L)
    state.masked.copy_(torch.from_numpy(masked).cuda())
    dd.dllm_commit_threshold(lgd, shape, stats, state, -1.0, -1, ws)
    torch.cuda.synchronize()
    full = oracle.stats(lg)
    tokens = state.tokens.cpu().numpy()
    assert np.array_equal(state.committed_now.cpu().numpy(), masked)
    assert np.array_equal(tokens[masked == 1], full.argmax[masked == 1])
    assert (tokens[masked == 0] == -1).all() and not state.masked.cpu().numpy().any()
    assert np.array_equal(state.n_commit.cpu().numpy(), masked.reshape(B, L).sum(1))

def test_stopped_sequences_are_untouched():
    w = synth.WORKLOADS["threshold_loop"].scaled(B=3, L=8, V=512, eos_id=-1)
    gpu = GpuDecoder(w)
    gpu.state.masked.view(3, 8)[0].zero_()        # nothing masked
    gpu.state.eos_hit[1] = 1                      # EOS already hit
    before = gpu.host_state()
    lg = to_device(synth.logits(w, seed=2))
    gpu.step(lg)
    after = gpu.host_state()
    assert after["n_commit"].tolist()[:2] == [0, 0] and after["n_commit"][2] >= 1
    assert np.array_equal(after["masked"][:2], before["masked"][:2])
    st = gpu.host_stats()
    assert (st["argmax"].reshape(3, 8)[:2] == -1).all()
    assert np.isneginf(st["lse"].reshape(3, 8)[:2]).all()


def test_commit_only_matches_fused():
    w = synth.WORKLOADS["credit_loop"].scaled(B=4, L=16, V=3000, max_iters=6)
    fused, split = GpuDecoder(w), GpuDecoder(w)
    for it in range(w.max_iters):
        lg = to_device(synth.logits(w, seed=11, it=it, calibrated=True))
        fused.step(lg)
        dd.dllm_decode_stats(lg, split.shape, split.state.masked, split.stats, split.ws)
        # rows of stopped sequences are skipped by the fused call; none stop here
        split.step(None)
        a, b = fused.host_state(), split.host_state()
        for k in a:
            assert np.array_equal(a[k], b[k]), k


def test_graph_capture_replays_steps():
    w = synth.WORKLOADS["threshold_loop"].scaled(B=2, L=16, V=4096, max_iters=4)
    lgs = [to_device(synth.logits(w, seed=8, it=i, calibrated=True)) for i in range(4)]
    eager = GpuDecoder(w)
    for lg in lgs:
        eager.step(lg)
    graphed = GpuDecoder(w)
    s = torch.cuda.Stream()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            for lg in lgs:
                graphed.step(lg)
    graphed.state.reset()
    g.replay()
    torch.cuda.synchronize()
    a, b = eager.host_state(), graphed.host_state()
    for k in a:
        assert np.array_equal(a[k], b[k]), k


def test_status_word_stays_ok():
    w = synth.WORKLOADS["threshold_single"]
    gpu = GpuDecoder(w)
    gpu.step(to_device(synth.logits(w, seed=1)))
    assert dd.dllm_get_status(gpu.ws) == dd.DLLM_OK
