"""Seeded synthetic inputs for the parallel-decode step.

This package only makes inputs: Philox-4x32-10 normal draws (``philox.c``), bf16 rounding of
those draws, and the planted-peak recipes of the benchmark workloads.  It holds none of the
decode step's arithmetic.  The oracle side and the CUDA side of every test consume the same
buffers it returns; logits are returned as float32 arrays or as uint16 arrays of bf16 bits.
"""
from __future__ import annotations

import ctypes
import math
import os
import subprocess

import numpy as np

from .workloads import WORKLOADS, Workload  # noqa: F401

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "philox.c")
_LIB = os.path.join(_HERE, "libsynth.so")
_lib = None
_THREADS = max(1, min(32, os.cpu_count() or 1))

# stream ids separate the draws of one seed: (iteration, attempt, purpose)
_NOISE, _PEAK_POS, _PEAK_ID, _PEAK_H, _STABLE, _TABLE = range(6)


def build(force: bool = False) -> str:
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off", _SRC,
               "-o", _LIB + ".tmp", "-lm", "-lpthread"]
        subprocess.run(cmd, check=True)
        os.replace(_LIB + ".tmp", _LIB)
    return _LIB


def _load():
    global _lib
    if _lib is None:
        build()
        _lib = ctypes.CDLL(_LIB)
        _lib.synth_normal_f32.argtypes = [ctypes.c_uint64, ctypes.c_uint64, ctypes.c_uint64,
                                          ctypes.c_int64, ctypes.c_double, ctypes.c_double,
                                          ctypes.c_void_p, ctypes.c_int]
        _lib.synth_f32_to_bf16.argtypes = [ctypes.c_void_p, ctypes.c_int64, ctypes.c_void_p,
                                           ctypes.c_int]
    return _lib


def stream_id(it: int, attempt: int, purpose: int) -> int:
    return (int(it) << 32) | (int(attempt) << 8) | int(purpose)


def normal_f32(seed: int, stream: int, n: int, mean: float = 0.0, std: float = 1.0,
               offset: int = 0) -> np.ndarray:
    out = np.empty(n, np.float32)
    rc = _load().synth_normal_f32(seed, stream, offset, n, mean, std,
                                  out.ctypes.data_as(ctypes.c_void_p), _THREADS)
    if rc:
        raise RuntimeError("synth_normal_f32 failed")
    return out


def to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round finite float32 values to bf16 (nearest even); returns the uint16 bit patterns."""
    x = np.ascontiguousarray(x, np.float32)
    out = np.empty(x.shape, np.uint16)
    _load().synth_f32_to_bf16(x.ctypes.data_as(ctypes.c_void_p), x.size,
                              out.ctypes.data_as(ctypes.c_void_p), _THREADS)
    return out


def bf16_bits_to_f32(h: np.ndarray) -> np.ndarray:
    return (h.astype(np.uint32) << 16).view(np.float32)


def _rng(seed: int, it: int, attempt: int, purpose: int) -> np.random.Generator:
    return np.random.Generator(np.random.Philox(key=[seed, stream_id(it, attempt, purpose)]))


# ---------------------------------------------------------------- planted-peak recipes

def _planted_ids_fixed(seed: int, B: int, L: int, V: int) -> np.ndarray:
    """Per-seed planted token per position, uniform over [3, V) (ids 0..2 stay special)."""
    return _rng(seed, 0, 0, _PEAK_ID).integers(3, V, size=(B, L), dtype=np.int64)


def _peak_heights(w: Workload, seed: int, it: int, attempt: int, B: int, L: int,
                  calibrated: bool) -> np.ndarray:
    g = _rng(seed, it, attempt, _PEAK_H)
    if calibrated:
        # planted logit ~ ln(sum of the noise exponentials) + u, using the closed-form mean
        # ln(V) + std^2/2 of that sum, so that confidences spread over ~[0.1, 0.98]
        base = math.log(w.V) + 0.5 * w.std * w.std
        return base + g.uniform(w.calib_lo, w.calib_hi, size=(B, L))
    return g.uniform(w.peak_lo, w.peak_hi, size=(B, L))


def planted_ids(w: Workload, seed: int, it: int = 0, attempt: int = 0) -> np.ndarray:
    """Token id planted at each position in iteration ``it`` ([B, L], -1 = no plant)."""
    B, L, V = w.B, w.L, w.V
    if w.plant == "none":
        return np.full((B, L), -1, np.int64)
    if w.plant == "fixed":
        ids = _planted_ids_fixed(seed, B, L, V)
        if w.eos_id >= 0:
            # one seeded position per sequence in the second half of the block carries EOS
            pos = _rng(seed, 0, 0, _PEAK_POS).integers(L // 2, L, size=B)
            ids[np.arange(B), pos] = w.eos_id
        return ids
    if w.plant == "stable":
        stable = _rng(seed, 0, 0, _STABLE).integers(3, V, size=(B, L), dtype=np.int64)
        g = _rng(seed, it, attempt, _PEAK_ID)
        keep = g.random(size=(B, L)) < w.p_stable
        fresh = g.integers(3, V, size=(B, L), dtype=np.int64)
        return np.where(keep, stable, fresh)
    if w.plant == "sparse":
        # a fixed number of seeded positions (over the whole batch) get one seeded id each
        g = _rng(seed, it, attempt, _PEAK_POS)
        ids = np.full((B, L), -1, np.int64)
        flat = g.choice(B * L, size=min(w.n_planted, B * L), replace=False)
        ids.reshape(-1)[flat] = g.integers(0, V, size=len(flat))
        return ids
    raise ValueError(w.plant)


def logits_f32(w: Workload, seed: int, it: int = 0, attempt: int = 0,
               calibrated: bool = False) -> np.ndarray:
    """The fp32 draw std*N(0,1) + planted peaks, shape [B, L, V] (before any bf16 rounding)."""
    B, L, V = w.B, w.L, w.V
    x = normal_f32(seed, stream_id(it, attempt, _NOISE), B * L * V, 0.0, w.std).reshape(B, L, V)
    if calibrated and w.plant == "none":
        # the calibrated variant of an unplanted workload plants one fixed id per position
        w = w.scaled(plant="fixed", eos_id=-1)
    ids = planted_ids(w, seed, it, attempt)
    if w.plant == "sparse":
        heights = np.full((B, L), w.peak_lo, np.float64)
    else:
        heights = _peak_heights(w, seed, it, attempt, B, L, calibrated)
    b_idx, l_idx = np.nonzero(ids >= 0)
    x[b_idx, l_idx, ids[b_idx, l_idx]] += heights[b_idx, l_idx].astype(np.float32)
    return x


def logits(w: Workload, seed: int, it: int = 0, attempt: int = 0,
           calibrated: bool = False) -> np.ndarray:
    """Logits in the workload's dtype: float32 array, or uint16 bf16 bit patterns."""
    x = logits_f32(w, seed, it, attempt, calibrated)
    if w.dtype == "f32":
        return x
    return to_bf16_bits(x)


def embedding_table(seed: int, V: int, d: int, std: float = 0.02) -> np.ndarray:
    """bf16 bit patterns of E ~ N(0, std), shape [V, d] row-major."""
    return to_bf16_bits(normal_f32(seed, stream_id(0, 0, _TABLE), V * d, 0.0, std)).reshape(V, d)
