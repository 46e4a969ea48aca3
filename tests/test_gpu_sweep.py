"""GPU vs oracle over seeded random shapes: whole decode loops of every strategy, and the
single-read smoothing call.

The fixed cases elsewhere sit on chosen edges; these draw B, L, V, dtype, candidate slots,
loop length, row strides and offsets from a seeded generator, so that shapes nobody picked by
hand (a one-position block, a 10-element vocabulary, K = 1, odd strides with fp32 rows) run
through the same element-by-element comparison.  Every draw satisfies the margin guard (the
generator is deterministic; the guard is checked when the logits are drawn).
"""
import numpy as np
import pytest

import synth
from test_gpu_commit import _run_loop
from test_gpu_smooth_fused import _fused_case

pytestmark = pytest.mark.gpu

KEYS = ("threshold_loop", "hierarchical_loop", "hierarchical_levels_loop", "credit_loop",
        "credit_tracked_loop")


def _loop_case(seed):
    rng = np.random.default_rng(1000 + seed)
    key = KEYS[seed % len(KEYS)]
    B = int(rng.integers(1, 9))
    L = int(rng.integers(1, 97))
    V = int(rng.choice([int(rng.integers(2, 200)), int(rng.integers(200, 9000)),
                        int(rng.integers(9000, 70000))]))
    V = max(V, 4)  # the credit recipes plant token ids from 3 up
    dtype = "f32" if rng.random() < 0.3 else "bf16"
    K = int(rng.integers(1, 9))
    iters = int(rng.integers(2, 7))
    calibrated = bool(rng.random() < 0.5)
    return key, dict(B=B, L=L, V=V, dtype=dtype, K=K, max_iters=iters), calibrated


@pytest.mark.parametrize("seed", range(120))
def test_random_loop_matches_oracle(seed):
    # every iteration eagerly, then the whole loop as one graph, plain and stopping on the
    # device (a continue test every 4 iterations and every iteration)
    key, kw, calibrated = _loop_case(seed)
    w = synth.WORKLOADS[key].scaled(**kw)
    _run_loop(w, seed, calibrated=calibrated, graph=True)


def _smooth_case(seed):
    rng = np.random.default_rng(5000 + seed)
    B = int(rng.integers(1, 7))
    L = int(rng.integers(1, 81))
    V = int(rng.choice([int(rng.integers(8, 300)), int(rng.integers(300, 12000)),
                        int(rng.integers(12000, 60000))]))
    d = 16 * int(rng.integers(1, 49))
    dtype = "f32" if rng.random() < 0.3 else "bf16"
    extra = int(rng.choice([0, 0, 8, 3]))   # row padding: none, aligned, odd
    offset = int(rng.choice([0, 0, 0, 1]))  # rows one element off 16-byte alignment
    kw = dict(B=B, L=L, V=V, d=d, dtype=dtype, prefix_len=int(rng.integers(0, 64)))
    return kw, extra, offset


@pytest.mark.parametrize("seed", range(48))
def test_random_single_read_smoothing_matches_oracle(seed):
    kw, extra, offset = _smooth_case(seed)
    w = synth.WORKLOADS["smooth_step"].scaled(**kw)
    stride = w.V + extra if (extra or offset) else None
    _fused_case(w, seed=seed, calibrated=True, stride=stride, offset=offset)
