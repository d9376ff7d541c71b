"""Float64 CPU oracle for the GatedDeltaNet record / replay step (test infrastructure).

TEST INFRASTRUCTURE ONLY: the test-suite, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline leg are the only callers.  The CUDA library never
imports, links or runs anything here, and nothing here imports the CUDA
library.

The arithmetic lives in ``gdn_oracle.c`` (plain C, float64, the page kernels'
loop order); this module compiles it with gcc on first use and wraps it with
ctypes.  Functions take and return float64 numpy arrays holding the exact
values the GPU sees (see ``workloads.widen``).

Parity status of each function (what pins it; tests/test_oracle_pins.py):

* ``record`` -- pinned: hand-derived worked example (tests/golden), closed
  forms (outer-product write, reset g=0), the delta-rule projection identity
  at every step, an independent matrix-form restatement, permutation
  equivariance, masked-step identity; the tiled GQA mapping equals the
  pinned repeat followed by a record on the expanded heads.
* ``replay`` -- pinned: accepted=T reproduces record, accepted=a reproduces
  record on the first a tokens, accepted=0 / all-masked identity, NaN in
  unused tape slots never reaches the state, worked example; per-sequence
  accepted counts reproduce, sequence by sequence, a record over that
  sequence's own prefix.
* ``repeat_tiled`` -- pinned: numpy fancy indexing, bit-exact.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from typing import Optional

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
SOURCE = os.path.join(_HERE, "gdn_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "libgdn_oracle.so")
_lock = threading.Lock()
_default: Optional["OracleLib"] = None

_D = ctypes.POINTER(ctypes.c_double)
_U32 = ctypes.POINTER(ctypes.c_uint32)
_P64 = ctypes.POINTER(ctypes.c_int64)
_I64 = ctypes.c_int64


def compile_c(src: str, out: str) -> str:
    """Compile an oracle C source into a shared library at ``out``."""
    os.makedirs(os.path.dirname(out), exist_ok=True)
    tmp = out + f".{os.getpid()}.tmp"
    cmd = ["gcc", "-std=c11", "-O2", "-ffp-contract=off", "-fno-fast-math",
           "-fopenmp", "-shared", "-fPIC", src, "-o", tmp]
    subprocess.run(cmd, check=True)
    os.replace(tmp, out)
    return out


def build(force: bool = False) -> str:
    """Compile the oracle shared library with gcc (if stale); return its path."""
    stale = (not os.path.exists(_LIB_PATH)
             or os.path.getmtime(_LIB_PATH) < os.path.getmtime(SOURCE))
    if force or stale:
        compile_c(SOURCE, _LIB_PATH)
    return _LIB_PATH


class OracleLib:
    """ctypes view of one compiled oracle library."""

    def __init__(self, path: str):
        lib = ctypes.CDLL(path)
        lib.gdn_oracle_record.argtypes = [_I64] * 7 + [_D] * 6 + [_U32] + [_D] * 5
        lib.gdn_oracle_record.restype = None
        lib.gdn_oracle_replay.argtypes = [_I64] * 6 + [_P64] + [_D] * 4 + [_U32, _D]
        lib.gdn_oracle_replay.restype = None
        lib.gdn_oracle_repeat_tiled.argtypes = [_I64] * 5 + [ctypes.c_void_p] * 2
        lib.gdn_oracle_repeat_tiled.restype = None
        lib.gdn_oracle_max_threads.restype = ctypes.c_int
        lib.gdn_oracle_set_threads.argtypes = [ctypes.c_int]
        self.lib = lib
        self.path = path

    def record(self, *a, **kw):
        return _record(self.lib, *a, **kw)

    def replay(self, *a, **kw):
        return _replay(self.lib, *a, **kw)

    def repeat_tiled(self, *a, **kw):
        return _repeat_tiled(self.lib, *a, **kw)


def default() -> OracleLib:
    global _default
    with _lock:
        if _default is None:
            _default = OracleLib(build())
    return _default


def _f64(a, shape) -> np.ndarray:
    a = np.ascontiguousarray(a, dtype=np.float64)
    if a.shape != tuple(shape):
        raise ValueError(f"expected shape {tuple(shape)}, got {a.shape}")
    return a


def _dp(a: Optional[np.ndarray]):
    return None if a is None else a.ctypes.data_as(_D)


def _mask(mask, B, T):
    if mask is None:
        return None, None
    m = np.ascontiguousarray(mask, dtype=np.uint32)
    if m.shape != (B, T):
        raise ValueError(f"mask must be [B,T]=({B},{T}), got {m.shape}")
    return m, m.ctypes.data_as(_U32)


def max_threads() -> int:
    return int(default().lib.gdn_oracle_max_threads())


def set_threads(n: int) -> None:
    default().lib.gdn_oracle_set_threads(int(n))


def record(*a, **kw):
    """Float64 record step (see ``_record``)."""
    return default().record(*a, **kw)


def replay(*a, **kw):
    """Float64 replay (see ``_replay``)."""
    return default().replay(*a, **kw)


def repeat_tiled(*a, **kw):
    """Tiled GQA repeat (see ``_repeat_tiled``)."""
    return default().repeat_tiled(*a, **kw)


GQA_MAPPINGS = {"block": 0, "tiled": 1}


def _record(lib, q, k, v, g, beta, state, mask=None, *, capture_tape: bool = True,
            fill: float = float("nan"), gqa: str = "block"):
    """Float64 record step.  Returns dict y, state_out, delta_log[, k_log, g_log].

    y / delta_log / k_log / g_log start filled with ``fill`` so that positions
    the method leaves untouched (masked steps) stay recognisable.  ``gqa``
    picks the key head of value head hv: "block" hv // (Hv/Hk), "tiled"
    hv % Hk.
    """
    if gqa not in GQA_MAPPINGS:
        raise ValueError(f"gqa must be one of {sorted(GQA_MAPPINGS)}")
    q = np.asarray(q)
    B, T, Hk, Dk = q.shape
    Hv, Dv = np.asarray(v).shape[2], np.asarray(v).shape[3]
    if Hk <= 0 or Hv % Hk != 0:
        raise ValueError("Hv must be a positive multiple of Hk")
    q = _f64(q, (B, T, Hk, Dk))
    k = _f64(k, (B, T, Hk, Dk))
    v = _f64(v, (B, T, Hv, Dv))
    g = _f64(g, (B, T, Hv))
    beta = _f64(beta, (B, T, Hv))
    s_in = _f64(state, (B, Hv, Dv, Dk))
    m, mp = _mask(mask, B, T)
    y = np.full((B, T, Hv, Dv), fill)
    dl = np.full((B, T, Hv, Dv), fill)
    s_out = np.empty((B, Hv, Dv, Dk))
    kl = np.full((B, T, Hv, Dk), fill) if capture_tape else None
    gl = np.full((B, T, Hv), fill) if capture_tape else None
    lib.gdn_oracle_record(B, T, Hk, Hv, Dk, Dv, GQA_MAPPINGS[gqa], _dp(q), _dp(k), _dp(v), _dp(g),
                          _dp(beta), _dp(s_in), mp, _dp(y), _dp(s_out), _dp(dl),
                          _dp(kl), _dp(gl))
    out = dict(y=y, state_out=s_out, delta_log=dl)
    if capture_tape:
        out.update(k_log=kl, g_log=gl)
    return out


def _replay(lib, delta_log, k_log, g_log, state, mask=None, *, accepted):
    """Float64 replay of the accepted tape prefix onto ``state``; returns state_out.

    ``accepted`` is one int >= 0 for the whole batch, or a length-B sequence
    of per-sequence counts (a negative entry accepts nothing).
    """
    dl = np.asarray(delta_log)
    B, T, Hv, Dv = dl.shape
    Dk = np.asarray(k_log).shape[3]
    per_seq = None
    if np.ndim(accepted) == 0:
        if accepted < 0:
            raise ValueError("accepted must be >= 0")
        scalar = int(accepted)
    else:
        per_seq = np.ascontiguousarray(accepted, dtype=np.int64)
        if per_seq.shape != (B,):
            raise ValueError(f"per-sequence accepted must have shape ({B},)")
        scalar = 0
    dl = _f64(dl, (B, T, Hv, Dv))
    kl = _f64(k_log, (B, T, Hv, Dk))
    gl = _f64(g_log, (B, T, Hv))
    s_in = _f64(state, (B, Hv, Dv, Dk))
    m, mp = _mask(mask, B, T)
    s_out = np.empty((B, Hv, Dv, Dk))
    lib.gdn_oracle_replay(B, T, Hv, Dk, Dv, scalar,
                          None if per_seq is None else per_seq.ctypes.data_as(_P64), _dp(dl), _dp(kl), _dp(gl),
                          _dp(s_in), mp, _dp(s_out))
    return s_out


def _repeat_tiled(lib, src: np.ndarray, h: int) -> np.ndarray:
    """Tiled GQA repeat ``[seq,hg,k] -> [seq,h,k]`` of any fixed-size dtype, bit-exact."""
    src = np.ascontiguousarray(src)
    seq, hg, kd = src.shape
    if hg <= 0 or h % hg != 0:
        raise ValueError("h must be a positive multiple of hg")
    dst = np.empty((seq, h, kd), dtype=src.dtype)
    lib.gdn_oracle_repeat_tiled(seq, hg, h, kd, src.dtype.itemsize,
                                src.ctypes.data, dst.ctypes.data)
    return dst
