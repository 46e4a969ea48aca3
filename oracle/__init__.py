"""Oracle for the parallel-decode step: ctypes wrapper around ``dllm_oracle.cpp``.

TEST INFRASTRUCTURE ONLY.  The test suite, the smoke check and the benchmark's CPU-baseline leg
are the only callers.  The product path (the CUDA library and its Python binding) never imports
this package, and this package imports nothing from the product.

Every function takes and returns numpy arrays; all arithmetic happens in the C++ file, in double,
one row at a time, in the order its comments state.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "dllm_oracle.cpp")
_LIB = os.path.join(_HERE, "liboracle.so")
_lib = None

F32, BF16 = 0, 1


def build(force: bool = False) -> str:
    """Compile the oracle with plain g++ (no fast-math, no FMA contraction)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        cmd = ["g++", "-O2", "-std=c++17", "-fPIC", "-shared", "-ffp-contract=off",
               "-fno-fast-math", _SRC, "-o", _LIB + ".tmp"]
        subprocess.run(cmd, check=True)
        os.replace(_LIB + ".tmp", _LIB)
    return _LIB


def _load():
    global _lib
    if _lib is None:
        build()
        _lib = ctypes.CDLL(_LIB)
        vp, i32, i64, dbl = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_double
        _lib.orc_stats.argtypes = [vp, i32, i64, i64, i64, vp, vp, vp, vp, vp]
        _lib.orc_active_rows.argtypes = [i32, i32, vp, vp, vp]
        _lib.orc_commit_threshold.argtypes = [i32, i32, vp, vp, vp, vp, vp, vp, vp, dbl, i32]
        _lib.orc_commit_hierarchical.argtypes = [i32, i32, vp, vp, vp, vp, vp, vp, vp, dbl, i32,
                                                 i32]
        _lib.orc_commit_credit.argtypes = [i32, i32, vp, vp, vp, vp, vp, vp, vp, vp, vp, i32, dbl,
                                           dbl, dbl, i32, vp]
        _lib.orc_smooth_rows.argtypes = [i32, i32, vp, vp, vp, vp]
        _lib.orc_smooth_embed.argtypes = [vp, i32, i64, i64, vp, vp, i64, vp, i64, vp]
        _lib.orc_prob_row_bf16.argtypes = [vp, i32, i64, i64, i64, dbl, vp]
        _lib.orc_round_to_bf16.argtypes = [vp, i64, vp]
        _lib.orc_kv_refresh.argtypes = [i32, i32, vp, i32, i32, vp, vp, vp]
        _lib.orc_merge_shard_stats.argtypes = [i32, i64, vp, vp, vp, vp, vp, vp, vp, vp]
        _lib.orc_commit_hierarchical_levels.argtypes = [i32, i32, vp, vp, vp, vp, vp, vp, vp,
                                                        dbl, i32, i32]
        _lib.orc_commit_credit_tracked.argtypes = [i32, i32, vp, i32, i64, i64, vp, vp, vp, vp,
                                                   vp, vp, vp, vp, vp, vp, i32, dbl, dbl, dbl,
                                                   i32, vp, vp]
        for name in ("orc_stats", "orc_active_rows", "orc_commit_threshold",
                     "orc_commit_hierarchical", "orc_commit_credit", "orc_smooth_rows",
                     "orc_smooth_embed", "orc_prob_row_bf16", "orc_round_to_bf16",
                     "orc_kv_refresh", "orc_merge_shard_stats",
                     "orc_commit_hierarchical_levels", "orc_commit_credit_tracked"):
            getattr(_lib, name).restype = ctypes.c_int
    return _lib


def _p(a: np.ndarray | None):
    if a is None:
        return None
    assert a.flags["C_CONTIGUOUS"], "oracle arrays must be C-contiguous"
    return a.ctypes.data_as(ctypes.c_void_p)


def _check(rc: int, name: str) -> None:
    if rc != 0:
        raise ValueError(f"oracle {name} rejected its arguments (rc={rc})")


def _dtype_code(logits: np.ndarray) -> int:
    if logits.dtype == np.float32:
        return F32
    if logits.dtype == np.uint16:  # bf16 bit patterns
        return BF16
    raise TypeError("logits must be float32 or uint16 bf16 bit patterns")


class Stats:
    """Per-row softmax statistics in double: row_max, lse, conf, argmax."""

    def __init__(self, R: int):
        self.row_max = np.empty(R, np.float64)
        self.lse = np.empty(R, np.float64)
        self.conf = np.empty(R, np.float64)
        self.argmax = np.empty(R, np.int32)


def stats(logits: np.ndarray, active: np.ndarray | None = None) -> Stats:
    """logits: [R, V] (or [B, L, V]) float32 or bf16 bits; active: uint8 [R] or None (all)."""
    lg = np.ascontiguousarray(logits)
    V = lg.shape[-1]
    R = lg.size // V
    st = Stats(R)
    act = None if active is None else np.ascontiguousarray(active.reshape(R), np.uint8)
    rc = _load().orc_stats(_p(lg), _dtype_code(lg), R, V, V, _p(act), _p(st.row_max), _p(st.lse),
                           _p(st.conf), _p(st.argmax))
    _check(rc, "stats")
    return st


def active_rows(masked: np.ndarray, eos_hit: np.ndarray) -> np.ndarray:
    B, L = masked.shape
    out = np.empty((B, L), np.uint8)
    _load().orc_active_rows(B, L, _p(np.ascontiguousarray(masked, np.uint8)),
                            _p(np.ascontiguousarray(eos_hit, np.int32)), _p(out))
    return out


class BlockState:
    """Decode state of B blocks of L positions (the oracle's own copy, mutated in place)."""

    def __init__(self, B: int, L: int, K: int = 0):
        self.B, self.L, self.K = B, L, K
        self.masked = np.ones((B, L), np.uint8)
        self.tokens = np.full((B, L), -1, np.int32)
        self.committed_now = np.zeros((B, L), np.uint8)
        self.n_commit = np.zeros(B, np.int32)
        self.eos_hit = np.zeros(B, np.int32)
        self.cand_id = np.full((B, L, max(K, 1)), -1, np.int32)
        self.cand_credit = np.zeros((B, L, max(K, 1)), np.float64)

    def copy(self) -> "BlockState":
        c = BlockState(self.B, self.L, self.K)
        for k in ("masked", "tokens", "committed_now", "n_commit", "eos_hit", "cand_id",
                  "cand_credit"):
            setattr(c, k, getattr(self, k).copy())
        return c


def commit_threshold(st: BlockState, conf: np.ndarray, argmax: np.ndarray, tau: float,
                     eos_id: int = -1) -> None:
    conf = np.ascontiguousarray(conf, np.float64)
    argmax = np.ascontiguousarray(argmax, np.int32)
    rc = _load().orc_commit_threshold(st.B, st.L, _p(conf), _p(argmax), _p(st.masked),
                                      _p(st.tokens), _p(st.committed_now), _p(st.n_commit),
                                      _p(st.eos_hit), float(tau), int(eos_id))
    _check(rc, "commit_threshold")


def commit_hierarchical(st: BlockState, conf: np.ndarray, argmax: np.ndarray, tau_low: float,
                        min_width: int, eos_id: int = -1) -> None:
    conf = np.ascontiguousarray(conf, np.float64)
    argmax = np.ascontiguousarray(argmax, np.int32)
    rc = _load().orc_commit_hierarchical(st.B, st.L, _p(conf), _p(argmax), _p(st.masked),
                                         _p(st.tokens), _p(st.committed_now), _p(st.n_commit),
                                         _p(st.eos_hit), float(tau_low), int(min_width),
                                         int(eos_id))
    _check(rc, "commit_hierarchical")


def commit_credit(st: BlockState, conf: np.ndarray, argmax: np.ndarray, decay: float,
                  boost: float, tau: float, eos_id: int = -1) -> np.ndarray:
    """Returns the boosted scores (0 for rows not read)."""
    conf = np.ascontiguousarray(conf, np.float64)
    argmax = np.ascontiguousarray(argmax, np.int32)
    score = np.zeros((st.B, st.L), np.float64)
    rc = _load().orc_commit_credit(st.B, st.L, _p(conf), _p(argmax), _p(st.masked), _p(st.tokens),
                                   _p(st.committed_now), _p(st.n_commit), _p(st.eos_hit),
                                   _p(st.cand_id), _p(st.cand_credit), st.K, float(decay),
                                   float(boost), float(tau), int(eos_id), _p(score))
    _check(rc, "commit_credit")
    return score


def commit_hierarchical_levels(st: BlockState, conf: np.ndarray, argmax: np.ndarray,
                               tau_low: float, min_width: int, eos_id: int = -1) -> None:
    conf = np.ascontiguousarray(conf, np.float64)
    argmax = np.ascontiguousarray(argmax, np.int32)
    rc = _load().orc_commit_hierarchical_levels(st.B, st.L, _p(conf), _p(argmax), _p(st.masked),
                                                _p(st.tokens), _p(st.committed_now),
                                                _p(st.n_commit), _p(st.eos_hit), float(tau_low),
                                                int(min_width), int(eos_id))
    _check(rc, "commit_hierarchical_levels")


def commit_credit_tracked(st: BlockState, logits: np.ndarray, s: "Stats", decay: float,
                          boost: float, tau: float, eos_id: int = -1):
    """Returns (boosted score, candidate token) of every row (0 / -1 for rows not read)."""
    lg = np.ascontiguousarray(logits)
    V = lg.shape[-1]
    score = np.zeros((st.B, st.L), np.float64)
    token = np.full((st.B, st.L), -1, np.int32)
    rc = _load().orc_commit_credit_tracked(
        st.B, st.L, _p(lg), _dtype_code(lg), V, V, _p(np.ascontiguousarray(s.lse, np.float64)),
        _p(np.ascontiguousarray(s.conf, np.float64)), _p(np.ascontiguousarray(s.argmax, np.int32)),
        _p(st.masked), _p(st.tokens), _p(st.committed_now), _p(st.n_commit), _p(st.eos_hit),
        _p(st.cand_id), _p(st.cand_credit), st.K, float(decay), float(boost), float(tau),
        int(eos_id), _p(score), _p(token))
    _check(rc, "commit_credit_tracked")
    return score, token


def smooth_rows(masked: np.ndarray, eos_hit: np.ndarray) -> np.ndarray:
    B, L = masked.shape
    ids = np.empty(B * L, np.int32)
    M = np.zeros(1, np.int32)
    _load().orc_smooth_rows(B, L, _p(np.ascontiguousarray(masked, np.uint8)),
                            _p(np.ascontiguousarray(eos_hit, np.int32)), _p(ids), _p(M))
    return ids[: int(M[0])].copy()


def smooth_embed(logits: np.ndarray, lse: np.ndarray, row_ids: np.ndarray,
                 E_bf16: np.ndarray) -> np.ndarray:
    """logits [R, V]; lse [R] (double); row_ids [M]; E bf16 bits [V, d] -> S [M, d] double."""
    lg = np.ascontiguousarray(logits)
    V = lg.shape[-1]
    E = np.ascontiguousarray(E_bf16, np.uint16)
    assert E.shape[0] == V
    d = E.shape[1]
    ids = np.ascontiguousarray(row_ids, np.int32)
    out = np.empty((len(ids), d), np.float64)
    rc = _load().orc_smooth_embed(_p(lg), _dtype_code(lg), V, V,
                                  _p(np.ascontiguousarray(lse, np.float64)), _p(ids), len(ids),
                                  _p(E), d, _p(out))
    _check(rc, "smooth_embed")
    return out


def prob_row_bf16(logits: np.ndarray, r: int, lse_r: float) -> np.ndarray:
    lg = np.ascontiguousarray(logits)
    V = lg.shape[-1]
    p = np.empty(V, np.float64)
    _load().orc_prob_row_bf16(_p(lg), _dtype_code(lg), V, V, int(r), float(lse_r), _p(p))
    return p


def round_to_bf16(x: np.ndarray) -> np.ndarray:
    x = np.ascontiguousarray(x, np.float64)
    y = np.empty_like(x)
    _load().orc_round_to_bf16(_p(x), x.size, _p(y))
    return y


def kv_refresh(committed_now: np.ndarray, prefix_len: int, window: int):
    B, L = committed_now.shape
    T = prefix_len + L
    refresh = np.empty((B, T), np.uint8)
    idx = np.empty((B, T), np.int32)
    count = np.empty(B, np.int32)
    rc = _load().orc_kv_refresh(B, L, _p(np.ascontiguousarray(committed_now, np.uint8)),
                                int(prefix_len), int(window), _p(refresh), _p(idx), _p(count))
    _check(rc, "kv_refresh")
    return refresh, idx, count


def merge_shard_stats(shards: list, offsets) -> Stats:
    """Merge per-shard Stats (each over its own vocabulary columns, local argmax) of the same R
    rows; offsets[k] = first vocabulary id of shard k."""
    n = len(shards)
    R = shards[0].row_max.size
    rm = np.ascontiguousarray(np.stack([s.row_max for s in shards]), np.float64)
    ls = np.ascontiguousarray(np.stack([s.lse for s in shards]), np.float64)
    am = np.ascontiguousarray(np.stack([s.argmax for s in shards]), np.int32)
    off = np.ascontiguousarray(offsets, np.int64)
    out = Stats(R)
    rc = _load().orc_merge_shard_stats(n, R, _p(rm), _p(ls), _p(am), _p(off), _p(out.row_max),
                                       _p(out.lse), _p(out.conf), _p(out.argmax))
    _check(rc, "merge_shard_stats")
    return out
