"""GB300 GatedDeltaNet record / replay with innovation-tape capture.

A thin ctypes binding over ``libgdn.so`` (C ABI: ``include/gdn.h``).  The
functions below only check tensor metadata, allocate missing outputs with
PyTorch and forward raw device pointers plus the current CUDA stream; every
step of the computation runs in the library's sm_103a kernels.  There is no
CPU or PyTorch fallback: if the library has not been built (``build()``) or
cannot be loaded, every call raises ``GdnError``.

Entry points (same names as the C ABI):

* ``gdn_step_record`` -- T gated delta-rule steps; writes y, the final state
  and the delta tape (optionally k_log / g_log), "metaltile-std
  gated_delta_replay.rs", kernel gated_delta_step_record.
* ``gdn_step_record_mapped`` -- the same with the tiled GQA mapping
  ``hk = hv % Hk`` available (``mapping="tiled"``).
* ``gdn_chunk_prefill`` -- the record recurrence for long calls in chunks of
  16 steps on the tensor cores (float32-accurate; optional tape outputs;
  needs a workspace of ``gdn_chunk_prefill_workspace_size`` bytes, which
  the binding allocates when none is given).
* ``gdn_step_record_tstate`` / ``gdn_state_replay_tstate`` -- record and
  replay with the state stored in the input element type (chosen by the
  binding when ``state_in`` has the inputs' bf16/f16 dtype).
* ``gdn_chunk_replay`` -- the replay of a long accepted prefix as one
  tensor-core contraction (tcgen05; float32-accurate; workspace allocated by
  the binding when none is given).
* ``gdn_state_replay`` -- re-fold the accepted tape prefix onto a snapshot,
  same page, kernel state_replay.
* ``gdn_state_replay_per_seq`` -- the same with one accepted count per
  sequence (an int32 device tensor).
* ``gqa_repeat_tiled`` -- ``dst[t,h,k] = src[t,h%hg,k]``, "mlx-native
  repeat_tiled.rs".
"""
from __future__ import annotations

import ctypes
import os
import threading
from collections import namedtuple
from typing import Optional

import torch

from . import _build

__all__ = ["GdnError", "build", "load", "lib_path", "gdn_step_record", "gdn_step_record_mapped",
           "gdn_chunk_prefill", "gdn_chunk_prefill_workspace_size", "gdn_chunk_prefill_noalloc",
           "gdn_chunk_replay", "gdn_chunk_replay_workspace_size",
           "gdn_step_record_tstate", "gdn_state_replay_tstate",
           "gdn_state_replay", "gdn_state_replay_per_seq", "gqa_repeat_tiled", "RecordOutputs",
           "STATUS_NAMES", "DTYPE_CODES", "GQA_MAPPINGS"]

STATUS_NAMES = {0: "GDN_OK", 1: "GDN_ERR_INVALID_ARGUMENT", 2: "GDN_ERR_UNSUPPORTED",
                3: "GDN_ERR_MISALIGNED", 4: "GDN_ERR_CUDA"}
DTYPE_CODES = {torch.float32: 0, torch.bfloat16: 1, torch.float16: 2}
GQA_MAPPINGS = {"block": 0, "tiled": 1}
EXPORTED = ("gdn_step_record", "gdn_step_record_mapped", "gdn_chunk_prefill",
            "gdn_chunk_prefill_workspace_size", "gdn_chunk_prefill_noalloc", "gdn_chunk_replay",
            "gdn_chunk_replay_workspace_size", "gdn_step_record_tstate",
            "gdn_state_replay_tstate", "gdn_state_replay",
            "gdn_state_replay_per_seq", "gqa_repeat_tiled", "gdn_status_string",
            "gdn_last_error", "gdn_abi_version", "gdn_wait_status", "gdn_set_wait_bound",
            "gdn_inject_wait_expiry", "gdn_force_launch_failures")

RecordOutputs = namedtuple("RecordOutputs", "y state_out delta_log k_log g_log")

_lock = threading.Lock()
_lib: Optional[ctypes.CDLL] = None
_P = ctypes.c_void_p
_I = ctypes.c_int64


class GdnError(RuntimeError):
    """A non-OK status from libgdn.so, or the library is missing."""

    def __init__(self, msg: str, status: int = -1):
        super().__init__(msg)
        self.status = status


def lib_path() -> str:
    return _build.LIB_PATH


def build(force: bool = False) -> str:
    """Compile libgdn.so for sm_103a (in-tree) and return its path."""
    return _build.build(force=force)


def _declare(lib: ctypes.CDLL) -> None:
    lib.gdn_step_record.argtypes = [_P] * 12 + [_I] * 6 + [ctypes.c_int, _P]
    lib.gdn_step_record.restype = ctypes.c_int
    lib.gdn_step_record_mapped.argtypes = [_P] * 12 + [_I] * 6 + [ctypes.c_int] * 2 + [_P]
    lib.gdn_step_record_mapped.restype = ctypes.c_int
    lib.gdn_chunk_prefill.argtypes = [_P] * 12 + [_I] * 6 + [ctypes.c_int, _P, ctypes.c_size_t,
                                                           ctypes.c_int, _P]
    lib.gdn_chunk_prefill.restype = ctypes.c_int
    lib.gdn_chunk_prefill_noalloc.argtypes = [_P] * 12 + [_I] * 6 + [ctypes.c_int] * 2 + [_P]
    lib.gdn_chunk_prefill_noalloc.restype = ctypes.c_int
    lib.gdn_step_record_tstate.argtypes = [_P] * 12 + [_I] * 6 + [ctypes.c_int] * 2 + [_P]
    lib.gdn_step_record_tstate.restype = ctypes.c_int
    lib.gdn_state_replay_tstate.argtypes = [_P] * 6 + [_I] * 6 + [_P, ctypes.c_int, _P]
    lib.gdn_state_replay_tstate.restype = ctypes.c_int
    lib.gdn_chunk_replay.argtypes = [_P] * 6 + [_I] * 6 + [_P, _P, ctypes.c_size_t, ctypes.c_int, _P]
    lib.gdn_chunk_replay.restype = ctypes.c_int
    lib.gdn_chunk_replay_workspace_size.argtypes = [_I] * 5
    lib.gdn_chunk_replay_workspace_size.restype = ctypes.c_size_t
    lib.gdn_chunk_prefill_workspace_size.argtypes = [_I] * 3
    lib.gdn_chunk_prefill_workspace_size.restype = ctypes.c_size_t
    lib.gdn_state_replay.argtypes = [_P] * 6 + [_I] * 6 + [ctypes.c_int, _P]
    lib.gdn_state_replay.restype = ctypes.c_int
    lib.gdn_state_replay_per_seq.argtypes = [_P] * 6 + [_I] * 5 + [_P, ctypes.c_int, _P]
    lib.gdn_state_replay_per_seq.restype = ctypes.c_int
    lib.gqa_repeat_tiled.argtypes = [_P, _P] + [_I] * 4 + [ctypes.c_int, ctypes.c_size_t,
                                                            ctypes.c_size_t, _P]
    lib.gqa_repeat_tiled.restype = ctypes.c_int
    lib.gdn_status_string.argtypes = [ctypes.c_int]
    lib.gdn_status_string.restype = ctypes.c_char_p
    lib.gdn_last_error.argtypes = []
    lib.gdn_last_error.restype = ctypes.c_char_p
    lib.gdn_abi_version.argtypes = []
    lib.gdn_abi_version.restype = ctypes.c_int
    lib.gdn_wait_status.argtypes = [ctypes.POINTER(ctypes.c_int)]
    lib.gdn_wait_status.restype = ctypes.c_int
    lib.gdn_set_wait_bound.argtypes = [_I]
    lib.gdn_set_wait_bound.restype = ctypes.c_int
    lib.gdn_inject_wait_expiry.argtypes = [ctypes.c_int]
    lib.gdn_inject_wait_expiry.restype = ctypes.c_int
    lib.gdn_force_launch_failures.argtypes = [ctypes.c_int]
    lib.gdn_force_launch_failures.restype = ctypes.c_int


def load(path: Optional[str] = None) -> ctypes.CDLL:
    """Load libgdn.so (raises GdnError if it is missing: no fallback)."""
    global _lib
    with _lock:
        if _lib is not None and path is None:
            return _lib
        p = path or lib_path()
        if not os.path.exists(p):
            raise GdnError(f"libgdn.so not found at {p}; build it first "
                           "(linear_attention_recurrence_step_gb300.build())")
        lib = ctypes.CDLL(p)
        _declare(lib)
        if path is None:
            _lib = lib
        return lib


def _check(status: int, what: str) -> None:
    if status != 0:
        lib = load()
        msg = lib.gdn_last_error().decode(errors="replace")
        raise GdnError(f"{what}: {STATUS_NAMES.get(status, status)}: {msg}", status)


def _ptr(t: Optional[torch.Tensor]) -> Optional[int]:
    return None if t is None else t.data_ptr()


def _stream(device: torch.device, stream) -> int:
    if stream is None:
        stream = torch.cuda.current_stream(device)
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def _need(t: torch.Tensor, name: str, shape, dtype, device) -> None:
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.device != device:
        raise ValueError(f"{name} is on {t.device}, expected {device}")
    if t.dtype != dtype:
        raise ValueError(f"{name} has dtype {t.dtype}, expected {dtype}")
    if tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} has shape {tuple(t.shape)}, expected {tuple(shape)}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def gdn_step_record(q, k, v, g, beta, state_in, mask=None, *, y=None, state_out=None,
                    delta_log=None, k_log=None, g_log=None, capture_tape: bool = False,
                    gqa: str = "block", stream=None) -> RecordOutputs:
    """Run T record steps.  Missing outputs are allocated (uninitialised where
    the mask skips a step).  ``capture_tape=True`` also allocates k_log/g_log.
    ``state_out=state_in`` runs in place.  ``gqa="tiled"`` reads key head
    ``hv % Hk`` (C entry point gdn_step_record_mapped) instead of the block
    mapping ``hv // (Hv/Hk)``."""
    if gqa not in GQA_MAPPINGS:
        raise ValueError(f"gqa must be one of {sorted(GQA_MAPPINGS)}")
    B, T, Hk, Dk = q.shape
    Hv, Dv = v.shape[2], v.shape[3]
    dt, dev = q.dtype, q.device
    if dt not in DTYPE_CODES:
        raise ValueError(f"unsupported dtype {dt}")
    _need(q, "q", (B, T, Hk, Dk), dt, dev)
    _need(k, "k", (B, T, Hk, Dk), dt, dev)
    _need(v, "v", (B, T, Hv, Dv), dt, dev)
    _need(g, "g", (B, T, Hv), dt, dev)
    _need(beta, "beta", (B, T, Hv), dt, dev)
    # the state is float32, or (state in T) the input element type
    sdt = state_in.dtype if isinstance(state_in, torch.Tensor) else torch.float32
    tstate = sdt == dt and dt != torch.float32
    _need(state_in, "state_in", (B, Hv, Dv, Dk), dt if tstate else torch.float32, dev)
    if mask is not None:
        _need(mask, "mask", (B, T), torch.int32 if mask.dtype == torch.int32 else torch.uint32, dev)
    if y is None:
        y = torch.empty((B, T, Hv, Dv), dtype=dt, device=dev)
    if state_out is None:
        state_out = torch.empty_like(state_in)
    if delta_log is None:
        delta_log = torch.empty((B, T, Hv, Dv), dtype=dt, device=dev)
    if capture_tape:
        if k_log is None:
            k_log = torch.empty((B, T, Hv, Dk), dtype=dt, device=dev)
        if g_log is None:
            g_log = torch.empty((B, T, Hv), dtype=dt, device=dev)
    _need(y, "y", (B, T, Hv, Dv), dt, dev)
    _need(state_out, "state_out", (B, Hv, Dv, Dk), state_in.dtype, dev)
    _need(delta_log, "delta_log", (B, T, Hv, Dv), dt, dev)
    if k_log is not None:
        _need(k_log, "k_log", (B, T, Hv, Dk), dt, dev)
    if g_log is not None:
        _need(g_log, "g_log", (B, T, Hv), dt, dev)
    ptrs = (_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(state_in), _ptr(mask), _ptr(y),
            _ptr(state_out), _ptr(delta_log), _ptr(k_log), _ptr(g_log), B, T, Hk, Hv, Dk, Dv)
    if tstate:
        st = load().gdn_step_record_tstate(*ptrs, GQA_MAPPINGS[gqa], DTYPE_CODES[dt],
                                           _stream(dev, stream))
        _check(st, "gdn_step_record_tstate")
    elif gqa == "block":
        st = load().gdn_step_record(*ptrs, DTYPE_CODES[dt], _stream(dev, stream))
        _check(st, "gdn_step_record")
    else:
        st = load().gdn_step_record_mapped(*ptrs, GQA_MAPPINGS[gqa], DTYPE_CODES[dt],
                                           _stream(dev, stream))
        _check(st, "gdn_step_record_mapped")
    return RecordOutputs(y, state_out, delta_log, k_log, g_log)


def gdn_step_record_mapped(q, k, v, g, beta, state_in, mask=None, *, mapping: str,
                           **kw) -> RecordOutputs:
    """``gdn_step_record`` with an explicit GQA mapping ("block" or "tiled")."""
    return gdn_step_record(q, k, v, g, beta, state_in, mask, gqa=mapping, **kw)


def gdn_chunk_prefill_workspace_size(B: int, T: int, Hv: int) -> int:
    """Bytes of device workspace gdn_chunk_prefill needs (0 for invalid sizes)."""
    return int(load().gdn_chunk_prefill_workspace_size(B, T, Hv))


def gdn_chunk_prefill(q, k, v, g, beta, state_in, mask=None, *, y=None, state_out=None,
                      delta_log=None, k_log=None, g_log=None, write_delta: bool = True,
                      capture_tape: bool = False, gqa: str = "block", workspace=None,
                      stream=None) -> RecordOutputs:
    """The record recurrence in chunks of 16 steps on the tensor cores.

    Same inputs and outputs as ``gdn_step_record`` (float32-accurate, not
    bit-identical to the step form).  ``write_delta=False`` skips the delta
    tape; ``workspace`` (a device tensor of at least
    ``gdn_chunk_prefill_workspace_size(B, T, Hv)`` bytes) is allocated when
    not given; ``workspace="static"`` calls gdn_chunk_prefill_noalloc."""
    if gqa not in GQA_MAPPINGS:
        raise ValueError(f"gqa must be one of {sorted(GQA_MAPPINGS)}")
    B, T, Hk, Dk = q.shape
    Hv, Dv = v.shape[2], v.shape[3]
    dt, dev = q.dtype, q.device
    if dt not in DTYPE_CODES:
        raise ValueError(f"unsupported dtype {dt}")
    _need(q, "q", (B, T, Hk, Dk), dt, dev)
    _need(k, "k", (B, T, Hk, Dk), dt, dev)
    _need(v, "v", (B, T, Hv, Dv), dt, dev)
    _need(g, "g", (B, T, Hv), dt, dev)
    _need(beta, "beta", (B, T, Hv), dt, dev)
    _need(state_in, "state_in", (B, Hv, Dv, Dk), torch.float32, dev)
    if mask is not None:
        _need(mask, "mask", (B, T), torch.int32 if mask.dtype == torch.int32 else torch.uint32, dev)
    if y is None:
        y = torch.empty((B, T, Hv, Dv), dtype=dt, device=dev)
    if state_out is None:
        state_out = torch.empty_like(state_in)
    if delta_log is None and write_delta:
        delta_log = torch.empty((B, T, Hv, Dv), dtype=dt, device=dev)
    if capture_tape:
        if k_log is None:
            k_log = torch.empty((B, T, Hv, Dk), dtype=dt, device=dev)
        if g_log is None:
            g_log = torch.empty((B, T, Hv), dtype=dt, device=dev)
    _need(y, "y", (B, T, Hv, Dv), dt, dev)
    _need(state_out, "state_out", (B, Hv, Dv, Dk), torch.float32, dev)
    if delta_log is not None:
        _need(delta_log, "delta_log", (B, T, Hv, Dv), dt, dev)
    if k_log is not None:
        _need(k_log, "k_log", (B, T, Hv, Dk), dt, dev)
    if g_log is not None:
        _need(g_log, "g_log", (B, T, Hv), dt, dev)
    if isinstance(workspace, str):
        if workspace != "static":
            raise ValueError('workspace must be a device tensor, None or "static"')
        st = load().gdn_chunk_prefill_noalloc(
            _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(state_in), _ptr(mask), _ptr(y),
            _ptr(state_out), _ptr(delta_log), _ptr(k_log), _ptr(g_log), B, T, Hk, Hv, Dk, Dv,
            GQA_MAPPINGS[gqa], DTYPE_CODES[dt], _stream(dev, stream))
        _check(st, "gdn_chunk_prefill_noalloc")
        return RecordOutputs(y, state_out, delta_log, k_log, g_log)
    need = gdn_chunk_prefill_workspace_size(B, T, Hv)
    if workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=dev)
    if workspace.device != dev or not workspace.is_contiguous():
        raise ValueError("workspace must be a contiguous tensor on the inputs' device")
    st = load().gdn_chunk_prefill(
        _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(state_in), _ptr(mask), _ptr(y),
        _ptr(state_out), _ptr(delta_log), _ptr(k_log), _ptr(g_log), B, T, Hk, Hv, Dk, Dv,
        GQA_MAPPINGS[gqa], _ptr(workspace), workspace.numel() * workspace.element_size(),
        DTYPE_CODES[dt], _stream(dev, stream))
    _check(st, "gdn_chunk_prefill")
    return RecordOutputs(y, state_out, delta_log, k_log, g_log)


def gdn_chunk_prefill_noalloc(q, k, v, g, beta, state_in, mask=None, **kw) -> RecordOutputs:
    """``gdn_chunk_prefill`` on the library's static 32 MiB device scratch, for
    callers that may not allocate device memory when they call (no workspace
    argument; calls on one device share the scratch and must not overlap in
    time)."""
    return gdn_chunk_prefill(q, k, v, g, beta, state_in, mask, workspace="static", **kw)


def gdn_state_replay(delta_log, k_log, g_log, state_in, mask=None, *, accepted,
                     state_out=None, stream=None) -> torch.Tensor:
    """Fold the tape prefix [0, accepted) onto ``state_in``; returns state_out.

    ``accepted`` is an int (one count for the batch) or an int32 device
    tensor of shape [B] (one count per sequence; C entry point
    gdn_state_replay_per_seq)."""
    B, T, Hv, Dv = delta_log.shape
    Dk = k_log.shape[3]
    dt, dev = delta_log.dtype, delta_log.device
    if dt not in DTYPE_CODES:
        raise ValueError(f"unsupported dtype {dt}")
    _need(delta_log, "delta_log", (B, T, Hv, Dv), dt, dev)
    _need(k_log, "k_log", (B, T, Hv, Dk), dt, dev)
    _need(g_log, "g_log", (B, T, Hv), dt, dev)
    sdt = state_in.dtype if isinstance(state_in, torch.Tensor) else torch.float32
    tstate = sdt == dt and dt != torch.float32
    _need(state_in, "state_in", (B, Hv, Dv, Dk), dt if tstate else torch.float32, dev)
    if mask is not None:
        _need(mask, "mask", (B, T), torch.int32 if mask.dtype == torch.int32 else torch.uint32, dev)
    if state_out is None:
        state_out = torch.empty_like(state_in)
    _need(state_out, "state_out", (B, Hv, Dv, Dk), state_in.dtype, dev)
    ptrs = (_ptr(delta_log), _ptr(k_log), _ptr(g_log), _ptr(state_in), _ptr(mask),
            _ptr(state_out), B, T, Hv, Dk, Dv)
    if tstate:
        per_seq = accepted if isinstance(accepted, torch.Tensor) else None
        if per_seq is not None:
            _need(per_seq, "accepted", (B,), torch.int32, dev)
        st = load().gdn_state_replay_tstate(*ptrs, 0 if per_seq is not None else int(accepted),
                                            _ptr(per_seq), DTYPE_CODES[dt], _stream(dev, stream))
        _check(st, "gdn_state_replay_tstate")
    elif isinstance(accepted, torch.Tensor):
        _need(accepted, "accepted", (B,), torch.int32, dev)
        st = load().gdn_state_replay_per_seq(*ptrs, _ptr(accepted), DTYPE_CODES[dt],
                                             _stream(dev, stream))
        _check(st, "gdn_state_replay_per_seq")
    else:
        st = load().gdn_state_replay(*ptrs, int(accepted), DTYPE_CODES[dt], _stream(dev, stream))
        _check(st, "gdn_state_replay")
    return state_out


def gdn_chunk_replay_workspace_size(B: int, T: int, Hv: int, Dk: int, Dv: int) -> int:
    """Bytes of device workspace gdn_chunk_replay needs (0 for invalid sizes)."""
    return int(load().gdn_chunk_replay_workspace_size(B, T, Hv, Dk, Dv))


def gdn_chunk_replay(delta_log, k_log, g_log, state_in, mask=None, *, accepted,
                     state_out=None, workspace=None, stream=None) -> torch.Tensor:
    """Replay of the accepted tape prefix as one tensor-core contraction.

    ``accepted`` is an int or an int32 device tensor [B] (per sequence).
    Float32-accurate, not bit-identical to ``gdn_state_replay``."""
    B, T, Hv, Dv = delta_log.shape
    Dk = k_log.shape[3]
    dt, dev = delta_log.dtype, delta_log.device
    if dt not in DTYPE_CODES:
        raise ValueError(f"unsupported dtype {dt}")
    _need(delta_log, "delta_log", (B, T, Hv, Dv), dt, dev)
    _need(k_log, "k_log", (B, T, Hv, Dk), dt, dev)
    _need(g_log, "g_log", (B, T, Hv), dt, dev)
    _need(state_in, "state_in", (B, Hv, Dv, Dk), torch.float32, dev)
    if mask is not None:
        _need(mask, "mask", (B, T), torch.int32 if mask.dtype == torch.int32 else torch.uint32, dev)
    if state_out is None:
        state_out = torch.empty_like(state_in)
    _need(state_out, "state_out", (B, Hv, Dv, Dk), torch.float32, dev)
    per_seq = None
    if isinstance(accepted, torch.Tensor):
        _need(accepted, "accepted", (B,), torch.int32, dev)
        per_seq, accepted = accepted, 0
    need = gdn_chunk_replay_workspace_size(B, T, Hv, Dk, Dv)
    if workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=dev)
    if workspace.device != dev or not workspace.is_contiguous():
        raise ValueError("workspace must be a contiguous tensor on the inputs' device")
    st = load().gdn_chunk_replay(
        _ptr(delta_log), _ptr(k_log), _ptr(g_log), _ptr(state_in), _ptr(mask), _ptr(state_out),
        B, T, Hv, Dk, Dv, int(accepted), _ptr(per_seq), _ptr(workspace),
        workspace.numel() * workspace.element_size(), DTYPE_CODES[dt], _stream(dev, stream))
    _check(st, "gdn_chunk_replay")
    return state_out


def gdn_state_replay_per_seq(delta_log, k_log, g_log, state_in, mask=None, *,
                             accepted: torch.Tensor, **kw) -> torch.Tensor:
    """``gdn_state_replay`` with per-sequence accepted counts ([B] int32, device)."""
    if not isinstance(accepted, torch.Tensor):
        raise TypeError("accepted must be an int32 device tensor of shape [B]")
    return gdn_state_replay(delta_log, k_log, g_log, state_in, mask, accepted=accepted, **kw)


def gqa_repeat_tiled(src, h: int, *, dst=None, stream=None) -> torch.Tensor:
    """Tiled GQA broadcast ``[seq,hg,k] -> [seq,h,k]``, ``dst[t,hh,x] = src[t,hh%hg,x]``."""
    seq, hg, kd = src.shape
    dt, dev = src.dtype, src.device
    if dt not in DTYPE_CODES:
        raise ValueError(f"unsupported dtype {dt}")
    if not src.is_contiguous():
        raise ValueError("src must be contiguous")
    if dst is None:
        dst = torch.empty((seq, h, kd), dtype=dt, device=dev)
    _need(dst, "dst", (seq, h, kd), dt, dev)
    st = load().gqa_repeat_tiled(_ptr(src), _ptr(dst), seq, hg, h, kd, DTYPE_CODES[dt],
                                 src.numel() * src.element_size(),
                                 dst.numel() * dst.element_size(), _stream(dev, stream))
    _check(st, "gqa_repeat_tiled")
    return dst


def wait_status() -> bool:
    """Whether a bounded wait of a pipelined kernel ran out since the last
    call (C entry point gdn_wait_status; reads and clears the flag).  Call it
    after synchronising the streams that ran the kernels."""
    lib = load()
    flag = ctypes.c_int(0)
    _check(lib.gdn_wait_status(ctypes.byref(flag)), "gdn_wait_status")
    return bool(flag.value)


def set_wait_bound(cycles: int) -> None:
    """Testing hook: the bound (GPU clock cycles) on the pipelined kernels'
    pipeline waits; 0 restores the default (C entry point gdn_set_wait_bound)."""
    _check(load().gdn_set_wait_bound(int(cycles)), "gdn_set_wait_bound")


def inject_wait_expiry(on: bool) -> None:
    """Testing hook: while on, each pipelined kernel takes one wait that
    nothing completes (C entry point gdn_inject_wait_expiry)."""
    _check(load().gdn_inject_wait_expiry(1 if on else 0), "gdn_inject_wait_expiry")


def force_launch_failures(n: int) -> None:
    """Testing hook: the next ``n`` calls that pass their argument checks fail
    with GDN_ERR_CUDA before touching the device (C entry point
    gdn_force_launch_failures)."""
    _check(load().gdn_force_launch_failures(int(n)), "gdn_force_launch_failures")
