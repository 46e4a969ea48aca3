"""Python binding of ``libdllm`` — the GB300 (sm_103a) parallel-decode step of a diffusion LM.

Each ``dllm_*`` function here marshals its arguments and calls the C entry point of the same
name (``include/dllm.h``); every step of the computation runs in the library's CUDA kernels.
Tensors must live on the current CUDA device; PyTorch provides device memory and streams only.

The library is built in-tree by ``diffusion_decoding_gb300.build.build()``.  Importing works
without it (so that host-side code and the CPU tests run), but every call raises if the shared
library is missing: there is no fallback path.
"""
from __future__ import annotations

import ctypes
import os

import torch

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libdllm.so")

DLLM_OK, DLLM_ERR_INVALID_ARG, DLLM_ERR_UNSUPPORTED, DLLM_ERR_CUDA, DLLM_ERR_TIMEOUT = range(5)
DLLM_F32, DLLM_BF16 = 0, 1

_c_i32, _c_i64, _c_f32, _c_vp, _c_sz = (ctypes.c_int32, ctypes.c_int64, ctypes.c_float,
                                        ctypes.c_void_p, ctypes.c_size_t)


class DllmError(RuntimeError):
    def __init__(self, status: int, name: str, msg: str):
        super().__init__(f"{name} -> status {status}: {msg}")
        self.status = status


class dllm_shape(ctypes.Structure):
    _fields_ = [("B", _c_i32), ("L", _c_i32), ("V", _c_i32), ("dtype", _c_i32),
                ("row_stride", _c_i64)]


class dllm_block_state(ctypes.Structure):
    _fields_ = [("masked", _c_vp), ("tokens", _c_vp), ("committed_now", _c_vp),
                ("n_commit", _c_vp), ("eos_hit", _c_vp)]


class dllm_stats(ctypes.Structure):
    _fields_ = [("row_max", _c_vp), ("lse", _c_vp), ("conf", _c_vp), ("argmax", _c_vp)]


class dllm_shard_stats(ctypes.Structure):
    _fields_ = [("stats", dllm_stats), ("vocab_offset", _c_i64)]


_SIGS = {
    "dllm_last_error": (ctypes.c_char_p, []),
    "dllm_workspace_bytes": (_c_sz, [ctypes.POINTER(dllm_shape)]),
    "dllm_decode_stats": (_c_i32, [_c_vp, ctypes.POINTER(dllm_shape), _c_vp,
                                   ctypes.POINTER(dllm_stats), _c_vp, _c_vp]),
    "dllm_commit_threshold": (_c_i32, [_c_vp, ctypes.POINTER(dllm_shape),
                                       ctypes.POINTER(dllm_stats),
                                       ctypes.POINTER(dllm_block_state), _c_f32, _c_i32, _c_vp,
                                       _c_vp]),
    "dllm_commit_hierarchical": (_c_i32, [_c_vp, ctypes.POINTER(dllm_shape),
                                          ctypes.POINTER(dllm_stats),
                                          ctypes.POINTER(dllm_block_state), _c_f32, _c_i32,
                                          _c_i32, _c_vp, _c_vp]),
    "dllm_commit_hierarchical_levels": (_c_i32, [_c_vp, ctypes.POINTER(dllm_shape),
                                                 ctypes.POINTER(dllm_stats),
                                                 ctypes.POINTER(dllm_block_state), _c_f32,
                                                 _c_i32, _c_i32, _c_vp, _c_vp]),
    "dllm_commit_credit_tracked": (_c_i32, [_c_vp, ctypes.POINTER(dllm_shape),
                                            ctypes.POINTER(dllm_stats),
                                            ctypes.POINTER(dllm_block_state), _c_vp, _c_vp,
                                            _c_i32, _c_f32, _c_f32, _c_f32, _c_i32, _c_vp,
                                            _c_vp]),
    "dllm_commit_credit": (_c_i32, [_c_vp, ctypes.POINTER(dllm_shape),
                                    ctypes.POINTER(dllm_stats), ctypes.POINTER(dllm_block_state),
                                    _c_vp, _c_vp, _c_i32, _c_f32, _c_f32, _c_f32, _c_i32, _c_vp,
                                    _c_vp]),
    "dllm_embedding_t_elems": (_c_sz, [_c_i32, _c_i32]),
    "dllm_prepare_embedding": (_c_i32, [_c_vp, _c_i32, _c_i32, _c_vp, _c_vp]),
    "dllm_smooth_workspace_bytes": (_c_sz, [ctypes.POINTER(dllm_shape), _c_i32]),
    "dllm_smooth_embed": (_c_i32, [_c_vp, ctypes.POINTER(dllm_shape), ctypes.POINTER(dllm_stats),
                                   ctypes.POINTER(dllm_block_state), _c_vp, _c_i32, _c_vp, _c_vp,
                                   _c_vp, _c_vp, _c_sz, _c_vp]),
    "dllm_smooth_plan_info": (_c_i32, [ctypes.POINTER(dllm_shape), _c_i32, _c_vp]),
    "dllm_commit_threshold_smooth": (_c_i32, [_c_vp, ctypes.POINTER(dllm_shape),
                                              ctypes.POINTER(dllm_stats),
                                              ctypes.POINTER(dllm_block_state), _c_f32, _c_i32,
                                              _c_vp, _c_i32, _c_vp, _c_vp, _c_vp, _c_vp, _c_sz,
                                              _c_vp]),
    "dllm_smooth_probs": (_c_i32, [_c_vp, ctypes.POINTER(dllm_shape), ctypes.POINTER(dllm_stats),
                                   ctypes.POINTER(dllm_block_state), _c_i32, _c_vp, _c_vp, _c_vp,
                                   _c_sz, _c_vp]),
    "dllm_smooth_gemm": (_c_i32, [ctypes.POINTER(dllm_shape), _c_vp, _c_i32, _c_vp, _c_vp, _c_vp,
                                  _c_sz, _c_vp]),
    "dllm_block_state_reset": (_c_i32, [ctypes.POINTER(dllm_block_state), _c_i32, _c_i32, _c_vp,
                                        _c_vp, _c_i32, _c_vp]),
    "dllm_kv_refresh_mask": (_c_i32, [ctypes.POINTER(dllm_block_state), _c_i32, _c_i32, _c_i32,
                                      _c_i32, _c_vp, _c_vp, _c_vp, _c_vp]),
    "dllm_get_status": (_c_i32, [_c_vp, _c_vp, ctypes.POINTER(_c_i32)]),
    "dllm_merge_shard_stats": (_c_i32, [ctypes.POINTER(dllm_shard_stats), _c_i32, _c_i64,
                                        ctypes.POINTER(dllm_stats), _c_vp]),
    "dllm_selftest_wait_timeout": (_c_i32, [_c_vp, ctypes.c_uint32, _c_vp]),
    "dllm_commit_threshold_static": (_c_i32, [_c_vp, ctypes.POINTER(dllm_shape),
                                              ctypes.POINTER(dllm_stats),
                                              ctypes.POINTER(dllm_block_state), _c_f32, _c_i32,
                                              _c_vp]),
    "dllm_capture_condition": (_c_i32, [_c_vp, ctypes.c_uint32, ctypes.POINTER(ctypes.c_uint64)]),
    "dllm_capture_if_begin": (_c_i32, [_c_vp, _c_vp, ctypes.c_uint64]),
    "dllm_capture_if_end": (_c_i32, [_c_vp]),
    "dllm_loop_continue": (_c_i32, [ctypes.POINTER(dllm_block_state), _c_i32, _c_i32,
                                    ctypes.c_uint64, _c_vp]),
}

_lib = None


def lib() -> ctypes.CDLL:
    """The loaded C library; raises if it has not been built."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: build it with "
                               "diffusion_decoding_gb300.build.build() (no CPU fallback exists)")
        handle = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in _SIGS.items():
            fn = getattr(handle, name)
            fn.restype = res
            fn.argtypes = args
        _lib = handle
    return _lib


def _ptr(t):
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(stream):
    s = torch.cuda.current_stream() if stream is None else stream
    return s.cuda_stream


def _check(status: int, name: str) -> None:
    if status != DLLM_OK:
        raise DllmError(status, name, lib().dllm_last_error().decode())


# ------------------------------------------------------------------ descriptors

def make_shape(B: int, L: int, V: int, dtype: int, row_stride: int | None = None) -> dllm_shape:
    return dllm_shape(B, L, V, dtype, V if row_stride is None else row_stride)


def shape_of(logits: torch.Tensor) -> dllm_shape:
    """Shape descriptor of a [B, L, V] (or [B, L, row_stride] sliced to V) logits tensor."""
    B, L, V = logits.shape
    if logits.dtype == torch.bfloat16:
        dt = DLLM_BF16
    elif logits.dtype == torch.float32:
        dt = DLLM_F32
    else:
        raise TypeError("logits must be bfloat16 or float32")
    if logits.stride(2) != 1 or logits.stride(0) != L * logits.stride(1):
        raise ValueError("logits rows must be contiguous and evenly strided")
    return dllm_shape(B, L, V, dt, logits.stride(1))


class StatsBuffers:
    """Device arrays for row_max, lse, conf and argmax ([B*L] each)."""

    def __init__(self, R: int, device=None):
        dev = device or torch.device("cuda")
        self.row_max = torch.empty(R, dtype=torch.float32, device=dev)
        self.lse = torch.empty(R, dtype=torch.float32, device=dev)
        self.conf = torch.empty(R, dtype=torch.float32, device=dev)
        self.argmax = torch.empty(R, dtype=torch.int32, device=dev)

    def c(self) -> dllm_stats:
        return dllm_stats(_ptr(self.row_max), _ptr(self.lse), _ptr(self.conf), _ptr(self.argmax))


class BlockState:
    """Device decode state of B blocks of L positions (fresh: everything masked)."""

    def __init__(self, B: int, L: int, K: int = 0, device=None):
        dev = device or torch.device("cuda")
        self.B, self.L, self.K = B, L, K
        self.masked = torch.ones(B * L, dtype=torch.uint8, device=dev)
        self.tokens = torch.full((B * L,), -1, dtype=torch.int32, device=dev)
        self.committed_now = torch.zeros(B * L, dtype=torch.uint8, device=dev)
        self.n_commit = torch.zeros(B, dtype=torch.int32, device=dev)
        self.eos_hit = torch.zeros(B, dtype=torch.int32, device=dev)
        self.cand_id = torch.full((B * L, max(K, 1)), -1, dtype=torch.int32, device=dev)
        self.cand_credit = torch.zeros((B * L, max(K, 1)), dtype=torch.float32, device=dev)

    def c(self) -> dllm_block_state:
        return dllm_block_state(_ptr(self.masked), _ptr(self.tokens), _ptr(self.committed_now),
                                _ptr(self.n_commit), _ptr(self.eos_hit))

    def reset(self, stream=None) -> None:
        """A new block, by one kernel (dllm_block_state_reset), credit slots included."""
        dllm_block_state_reset(self, stream=stream)


def workspace(nbytes: int, device=None) -> torch.Tensor:
    """Zero-filled device workspace (256-byte aligned: torch allocations are 512-aligned)."""
    return torch.zeros(max(int(nbytes), 256), dtype=torch.uint8, device=device or "cuda")


# ------------------------------------------------------------------ entry points

def dllm_workspace_bytes(shape: dllm_shape) -> int:
    return int(lib().dllm_workspace_bytes(ctypes.byref(shape)))


def dllm_decode_stats(logits, shape, masked, stats: StatsBuffers, ws, stream=None) -> None:
    st = stats.c()
    _check(lib().dllm_decode_stats(_ptr(logits), ctypes.byref(shape), _ptr(masked),
                                   ctypes.byref(st), _ptr(ws), _stream(stream)),
           "dllm_decode_stats")


def dllm_commit_threshold(logits, shape, stats: StatsBuffers, state: BlockState, tau: float,
                          eos_id: int, ws, stream=None) -> None:
    st, bs = stats.c(), state.c()
    _check(lib().dllm_commit_threshold(_ptr(logits), ctypes.byref(shape), ctypes.byref(st),
                                       ctypes.byref(bs), tau, eos_id, _ptr(ws), _stream(stream)),
           "dllm_commit_threshold")


def dllm_commit_hierarchical(logits, shape, stats: StatsBuffers, state: BlockState,
                             tau_low: float, min_width: int, eos_id: int, ws,
                             stream=None) -> None:
    st, bs = stats.c(), state.c()
    _check(lib().dllm_commit_hierarchical(_ptr(logits), ctypes.byref(shape), ctypes.byref(st),
                                          ctypes.byref(bs), tau_low, min_width, eos_id, _ptr(ws),
                                          _stream(stream)),
           "dllm_commit_hierarchical")


def dllm_commit_hierarchical_levels(logits, shape, stats: StatsBuffers, state: BlockState,
                                    tau_low: float, min_width: int, eos_id: int, ws,
                                    stream=None) -> None:
    st, bs = stats.c(), state.c()
    _check(lib().dllm_commit_hierarchical_levels(_ptr(logits), ctypes.byref(shape),
                                                 ctypes.byref(st), ctypes.byref(bs), tau_low,
                                                 min_width, eos_id, _ptr(ws), _stream(stream)),
           "dllm_commit_hierarchical_levels")


def dllm_commit_credit_tracked(logits, shape, stats: StatsBuffers, state: BlockState, K: int,
                               decay: float, boost: float, tau: float, eos_id: int, ws,
                               stream=None) -> None:
    st, bs = stats.c(), state.c()
    _check(lib().dllm_commit_credit_tracked(_ptr(logits), ctypes.byref(shape), ctypes.byref(st),
                                            ctypes.byref(bs), _ptr(state.cand_id),
                                            _ptr(state.cand_credit), K, decay, boost, tau, eos_id,
                                            _ptr(ws), _stream(stream)),
           "dllm_commit_credit_tracked")


def dllm_commit_credit(logits, shape, stats: StatsBuffers, state: BlockState, K: int,
                       decay: float, boost: float, tau: float, eos_id: int, ws,
                       stream=None) -> None:
    st, bs = stats.c(), state.c()
    _check(lib().dllm_commit_credit(_ptr(logits), ctypes.byref(shape), ctypes.byref(st),
                                    ctypes.byref(bs), _ptr(state.cand_id),
                                    _ptr(state.cand_credit), K, decay, boost, tau, eos_id,
                                    _ptr(ws), _stream(stream)),
           "dllm_commit_credit")


def dllm_embedding_t_elems(V: int, d: int) -> int:
    return int(lib().dllm_embedding_t_elems(V, d))


def dllm_prepare_embedding(E: torch.Tensor, Et: torch.Tensor, stream=None) -> None:
    """E: [V, d] bf16 (or int16 bit patterns); Et: dllm_embedding_t_elems(V, d) elements."""
    V, d = E.shape
    _check(lib().dllm_prepare_embedding(_ptr(E), V, d, _ptr(Et), _stream(stream)),
           "dllm_prepare_embedding")


def dllm_smooth_workspace_bytes(shape: dllm_shape, d: int) -> int:
    return int(lib().dllm_smooth_workspace_bytes(ctypes.byref(shape), d))


def dllm_smooth_embed(logits, shape, stats: StatsBuffers, state: BlockState, Et, d: int, out,
                      row_ids, M, ws, stream=None) -> None:
    st, bs = stats.c(), state.c()
    _check(lib().dllm_smooth_embed(_ptr(logits), ctypes.byref(shape), ctypes.byref(st),
                                   ctypes.byref(bs), _ptr(Et), d, _ptr(out), _ptr(row_ids),
                                   _ptr(M), _ptr(ws), ws.numel(), _stream(stream)),
           "dllm_smooth_embed")


def dllm_commit_threshold_smooth(logits, shape, stats: StatsBuffers, state: BlockState,
                                 tau: float, eos_id: int, Et, d: int, out, row_ids, M, ws,
                                 stream=None) -> None:
    st, bs = stats.c(), state.c()
    _check(lib().dllm_commit_threshold_smooth(_ptr(logits), ctypes.byref(shape), ctypes.byref(st),
                                              ctypes.byref(bs), tau, eos_id, _ptr(Et), d,
                                              _ptr(out), _ptr(row_ids), _ptr(M), _ptr(ws),
                                              ws.numel(), _stream(stream)),
           "dllm_commit_threshold_smooth")


def dllm_smooth_plan_info(shape, d: int) -> dict:
    info = (_c_i32 * 6)()
    _check(lib().dllm_smooth_plan_info(ctypes.byref(shape), d, info), "dllm_smooth_plan_info")
    keys = ("m_tiles", "n_tiles", "bn_max", "split_k", "stages", "launches")
    return dict(zip(keys, (int(x) for x in info)))


def dllm_smooth_probs(logits, shape, stats: StatsBuffers, state: BlockState, d: int, row_ids, M,
                      ws, stream=None) -> None:
    st, bs = stats.c(), state.c()
    _check(lib().dllm_smooth_probs(_ptr(logits), ctypes.byref(shape), ctypes.byref(st),
                                   ctypes.byref(bs), d, _ptr(row_ids), _ptr(M), _ptr(ws),
                                   ws.numel(), _stream(stream)),
           "dllm_smooth_probs")


def dllm_smooth_gemm(shape, Et, d: int, out, M, ws, stream=None) -> None:
    _check(lib().dllm_smooth_gemm(ctypes.byref(shape), _ptr(Et), d, _ptr(out), _ptr(M), _ptr(ws),
                                  ws.numel(), _stream(stream)),
           "dllm_smooth_gemm")


def dllm_block_state_reset(state: BlockState, credit: bool = True, stream=None) -> None:
    bs = state.c()
    K = state.cand_id.shape[1]
    _check(lib().dllm_block_state_reset(ctypes.byref(bs), state.B, state.L,
                                        _ptr(state.cand_id) if credit else None,
                                        _ptr(state.cand_credit) if credit else None,
                                        K if credit else 0, _stream(stream)),
           "dllm_block_state_reset")


def dllm_kv_refresh_mask(state: BlockState, prefix_len: int, window: int, refresh, idx, count,
                         stream=None) -> None:
    bs = state.c()
    _check(lib().dllm_kv_refresh_mask(ctypes.byref(bs), state.B, state.L, prefix_len, window,
                                      _ptr(refresh), _ptr(idx), _ptr(count), _stream(stream)),
           "dllm_kv_refresh_mask")


def dllm_commit_threshold_static(logits, shape, stats: StatsBuffers, state: BlockState, tau: float,
                                 eos_id: int, stream=None) -> None:
    """dllm_commit_threshold for callers that cannot allocate: no workspace argument, the
    scratch is a fixed static array inside the library (see include/dllm.h)."""
    st, bs = stats.c(), state.c()
    _check(lib().dllm_commit_threshold_static(_ptr(logits), ctypes.byref(shape),
                                              ctypes.byref(st), ctypes.byref(bs), tau, eos_id,
                                              _stream(stream)),
           "dllm_commit_threshold_static")


def dllm_capture_condition(default_value: int = 0, stream=None) -> int:
    """A condition handle in the graph `stream` is capturing (see include/dllm.h)."""
    h = ctypes.c_uint64(0)
    _check(lib().dllm_capture_condition(_stream(stream), int(default_value), ctypes.byref(h)),
           "dllm_capture_condition")
    return int(h.value)


def dllm_capture_if_begin(handle: int, body_stream, stream=None) -> None:
    """Conditional IF node on `handle` in the graph `stream` is capturing; its body is captured
    on body_stream until dllm_capture_if_end."""
    _check(lib().dllm_capture_if_begin(_stream(stream), body_stream.cuda_stream, int(handle)),
           "dllm_capture_if_begin")


def dllm_capture_if_end(body_stream) -> None:
    _check(lib().dllm_capture_if_end(body_stream.cuda_stream), "dllm_capture_if_end")


def dllm_loop_continue(state: BlockState, handle: int, stream=None) -> None:
    """Inside a capture: sets `handle` to whether some sequence of the block still decodes."""
    bs = state.c()
    _check(lib().dllm_loop_continue(ctypes.byref(bs), state.B, state.L, int(handle),
                                    _stream(stream)), "dllm_loop_continue")


def dllm_selftest_wait_timeout(ws, limit_us: int, stream=None) -> None:
    _check(lib().dllm_selftest_wait_timeout(_ptr(ws), limit_us, _stream(stream)),
           "dllm_selftest_wait_timeout")


def dllm_merge_shard_stats(shards, rows: int, out: StatsBuffers, stream=None) -> None:
    """shards: list of (statistics of one vocabulary shard, its first vocabulary id); each
    statistics object has row_max, lse, conf (float32) and argmax (int32) device tensors."""
    arr = (dllm_shard_stats * len(shards))(*[
        dllm_shard_stats(dllm_stats(_ptr(st.row_max), _ptr(st.lse), _ptr(st.conf),
                                    _ptr(st.argmax)), int(off))
        for st, off in shards])
    _check(lib().dllm_merge_shard_stats(arr, len(shards), int(rows), ctypes.byref(out.c()),
                                        _stream(stream)), "dllm_merge_shard_stats")


def dllm_get_status(ws, stream=None) -> int:
    out = _c_i32(0)
    _check(lib().dllm_get_status(_ptr(ws), _stream(stream), ctypes.byref(out)), "dllm_get_status")
    return int(out.value)
