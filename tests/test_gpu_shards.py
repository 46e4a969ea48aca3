"""GPU vs oracle: vocabulary-sharded statistics (tensor-parallel output layer) simulated on one
GPU.  Each shard's columns are reduced by dllm_decode_stats, merged by dllm_merge_shard_stats,
and must match the whole-row statistics; committing from the merged statistics must equal the
commit over the whole rows, and per-shard smoothing with the merged lse must sum to the
whole-row smoothing."""
import numpy as np
import pytest
import torch

import oracle
import synth
from gpu_runner import GpuDecoder, to_device
from harness import close, guarded_logits, oracle_step

import diffusion_decoding_gb300 as dd
from diffusion_decoding_gb300.tp import vocab_range

pytestmark = pytest.mark.gpu


def _shard_stats_gpu(lg, masked, n, dtype):
    """Per-shard statistics on the GPU; shard rows padded to a 16-byte stride."""
    R, V = lg.shape
    out = []
    for k in range(n):
        first, cnt = vocab_range(V, n, k)
        stride = -(-cnt // 8) * 8
        buf = np.zeros((R, stride), lg.dtype)
        buf[:, :cnt] = lg[:, first:first + cnt]
        shape = dd.make_shape(1, R, cnt, dtype, row_stride=stride)
        st = dd.StatsBuffers(R)
        ws = dd.workspace(dd.dllm_workspace_bytes(shape))
        m = None if masked is None else torch.from_numpy(masked).cuda()
        dd.dllm_decode_stats(to_device(buf), shape, m, st, ws)
        out.append((st, first))
    return out


@pytest.mark.parametrize("n", [2, 3, 8])
@pytest.mark.parametrize("V,dtype", [(4096, "f32"), (126464, "bf16"), (5003, "bf16")])
def test_merged_shard_statistics_match_whole_rows(n, V, dtype):
    w = synth.WORKLOADS["threshold_loop"].scaled(B=2, L=16, V=V, dtype=dtype, eos_id=-1,
                                                  plant="fixed")
    lg = synth.logits(w, seed=V + n, it=0).reshape(w.B * w.L, V)
    rng = np.random.default_rng(n)
    masked = (rng.random(w.B * w.L) < 0.75).astype(np.uint8)
    dt = dd.DLLM_BF16 if dtype == "bf16" else dd.DLLM_F32
    shards = _shard_stats_gpu(lg, masked, n, dt)
    out = dd.StatsBuffers(w.B * w.L)
    dd.dllm_merge_shard_stats(shards, w.B * w.L, out)
    torch.cuda.synchronize()
    ref = oracle.stats(lg, masked)
    assert np.array_equal(out.argmax.cpu().numpy(), ref.argmax)
    assert np.array_equal(out.row_max.cpu().numpy(), ref.row_max.astype(np.float32))
    for k in ("lse", "conf"):
        assert close(getattr(out, k).cpu().numpy(), getattr(ref, k)), k


def test_commit_and_smoothing_from_shards_equal_whole_rows():
    w = synth.WORKLOADS["smooth_step"].scaled(B=2, L=32, V=12000, d=256, prefix_len=16)
    n = 3                                   # 4000 ids per shard (multiples of 8)
    ost = oracle.BlockState(w.B, w.L)
    lg, _, s = guarded_logits(w, 21, 0, ost, calibrated=True)
    s_ref, _ = oracle_step(w, ost, lg, s)
    R = w.B * w.L
    lg2 = lg.reshape(R, w.V)
    # whole-vocabulary statistics from the shards, then commit from statistics only
    shards = _shard_stats_gpu(lg2, None, n, dd.DLLM_BF16)
    merged = dd.StatsBuffers(R)
    dd.dllm_merge_shard_stats(shards, R, merged)
    gpu = GpuDecoder(w)
    ws = dd.workspace(dd.dllm_workspace_bytes(gpu.shape))
    dd.dllm_commit_threshold(None, gpu.shape, merged, gpu.state, w.tau, w.eos_id, ws)
    torch.cuda.synchronize()
    hs = gpu.host_state()
    for k in ("masked", "tokens", "committed_now", "n_commit"):
        assert np.array_equal(hs[k], getattr(ost, k)), k
    # smoothing: each shard's probabilities (merged lse) times its rows of E, summed
    E = synth.embedding_table(3, w.V, w.d)
    total = torch.zeros(R, w.d, device="cuda")
    Mh = None
    for k in range(n):
        first, cnt = vocab_range(w.V, n, k)
        shape_k = dd.make_shape(w.B, w.L, cnt, dd.DLLM_BF16)
        Ek = np.ascontiguousarray(E[first:first + cnt])
        Et = torch.empty(dd.dllm_embedding_t_elems(cnt, w.d), dtype=torch.int16, device="cuda")
        dd.dllm_prepare_embedding(torch.from_numpy(Ek.view(np.int16)).cuda(), Et)
        out = torch.zeros(R, w.d, device="cuda")
        row_ids = torch.empty(R, dtype=torch.int32, device="cuda")
        M = torch.zeros(1, dtype=torch.int32, device="cuda")
        ws_s = dd.workspace(dd.dllm_smooth_workspace_bytes(shape_k, w.d))
        lgk = to_device(np.ascontiguousarray(lg2[:, first:first + cnt]))
        dd.dllm_smooth_embed(lgk, shape_k, merged, gpu.state, Et, w.d, out, row_ids, M, ws_s)
        total += out
        torch.cuda.synchronize()
        Mh = int(M.item())
    ids = oracle.smooth_rows(ost.masked, ost.eos_hit)
    assert Mh == len(ids)
    ref = oracle.smooth_embed(lg2, s_ref.lse, ids.astype(np.int32), E)
    scale = oracle.smooth_embed(lg2, s_ref.lse, ids.astype(np.int32), E & np.uint16(0x7FFF))
    g = total[:Mh].cpu().numpy().astype(np.float64)
    assert (np.abs(g - ref) <= 2e-3 * scale).all()
