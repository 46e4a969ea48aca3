"""The five decode-step workloads: shapes, input distributions and method parameters.

Each workload names what it is; ``WORKLOADS`` maps a short key to it.  Numbers only: no
arithmetic of the decode step lives here.
"""
from __future__ import annotations

from dataclasses import dataclass, replace


@dataclass(frozen=True)
class Workload:
    key: str
    title: str
    strategy: str          # threshold | hierarchical | credit | smooth, or a variant:
                           # hierarchical_levels | credit_tracked
    B: int
    L: int
    V: int
    dtype: str             # "f32" or "bf16"
    std: float             # logits ~ N(0, std)
    plant: str             # none | sparse | fixed | stable
    peak_lo: float = 0.0   # planted peak height ~ U[peak_lo, peak_hi] (sparse: fixed peak_lo)
    peak_hi: float = 0.0
    n_planted: int = 0     # sparse plants over the whole batch
    p_stable: float = 0.0  # credit workload: chance the planted id is the position's stable id
    calib_lo: float = -2.0  # calibrated variant: peak = ln V + std^2/2 + U[calib_lo, calib_hi]
    calib_hi: float = 4.0
    tau: float = 0.9
    tau_low: float = 0.6
    min_width: int = 2
    K: int = 8
    decay: float = 0.7
    boost: float = 0.3
    eos_id: int = -1
    max_iters: int = 1
    d: int = 0             # embedding width (smoothing)
    prefix_len: int = 0    # cached prefix (KV refresh)
    window: int = 0        # refresh neighbourhood

    def scaled(self, **kw) -> "Workload":
        """Same recipe at other sizes (the parity tests' small cases)."""
        return replace(self, **kw)


WORKLOADS = {
    "threshold_single": Workload(
        key="threshold_single",
        title="threshold decoding, one step, B=1 L=32 V=4096 fp32, 8 planted +8.0 peaks",
        strategy="threshold", B=1, L=32, V=4096, dtype="f32", std=1.0, plant="sparse",
        peak_lo=8.0, n_planted=8, tau=0.9, max_iters=1),
    "threshold_loop": Workload(
        key="threshold_loop",
        title="threshold decoding to completion, B=1 L=32 V=126464 bf16, EOS id 2",
        strategy="threshold", B=1, L=32, V=126464, dtype="bf16", std=2.0, plant="fixed",
        peak_lo=2.0, peak_hi=12.0, tau=0.9, eos_id=2, max_iters=32),
    "hierarchical_loop": Workload(
        key="hierarchical_loop",
        title="hierarchical decoding to completion, B=8 L=64 V=126464 bf16",
        strategy="hierarchical", B=8, L=64, V=126464, dtype="bf16", std=2.0, plant="fixed",
        peak_lo=2.0, peak_hi=12.0, tau_low=0.6, min_width=2, max_iters=64),
    "credit_loop": Workload(
        key="credit_loop",
        title="credit decoding, 24 steps, B=32 L=32 V=126464 bf16, K=8 candidates",
        strategy="credit", B=32, L=32, V=126464, dtype="bf16", std=2.0, plant="stable",
        peak_lo=2.0, peak_hi=12.0, p_stable=0.7, K=8, decay=0.7, boost=0.3, tau=0.9,
        max_iters=24),
    "smooth_step": Workload(
        key="smooth_step",
        title="threshold commit + iteration smoothing + KV refresh, B=16 L=64 V=126464 d=2048",
        strategy="smooth", B=16, L=64, V=126464, dtype="bf16", std=2.0, plant="none",
        tau=0.9, d=2048, prefix_len=1024, window=4, max_iters=1),
    # the strategy variants (the readings the configured workloads do not take), at the
    # hierarchical and credit shapes
    "hierarchical_levels_loop": Workload(
        key="hierarchical_levels_loop",
        title="hierarchical decoding, a centre per level, to completion, B=8 L=64 V=126464 bf16",
        strategy="hierarchical_levels", B=8, L=64, V=126464, dtype="bf16", std=2.0,
        plant="fixed", peak_lo=2.0, peak_hi=12.0, tau_low=0.6, min_width=2, max_iters=64),
    "credit_tracked_loop": Workload(
        key="credit_tracked_loop",
        title="credit decoding, every tracked candidate credited, 24 steps, B=32 L=32 "
              "V=126464 bf16, K=8",
        strategy="credit_tracked", B=32, L=32, V=126464, dtype="bf16", std=2.0, plant="stable",
        peak_lo=2.0, peak_hi=12.0, p_stable=0.7, K=8, decay=0.7, boost=0.3, tau=0.9,
        max_iters=24),
}

# fixed seeds per workload (1000 + position in the list)
SEEDS = {k: 1000 + i for i, k in enumerate(WORKLOADS)}
