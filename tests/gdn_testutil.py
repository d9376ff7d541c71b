"""Helpers shared by the tests: device transfer and the comparison rule.

Comparison rule (per element, float64):
    |got - want| <= atol + rtol * |want|  (+ half a unit in the last place of
    the stored type when the output is stored in bf16 / f16)
with atol = rtol = 1e-4 for float32 problems and 1e-3 for bf16 / f16 inputs
(the page's registered tolerance is 1e-3 for every dtype; float32 runs are
held ten times tighter).  ``want`` is always the unrounded float64 oracle
value; the half-ulp term admits a correctly rounded store of it.
"""
from __future__ import annotations

import numpy as np

import workloads

TOL = {"f32": 1e-4, "bf16": 1e-3, "f16": 1e-3}
SIG_BITS = {"f32": 24, "bf16": 8, "f16": 11}
MIN_EXP = {"f32": -126, "bf16": -126, "f16": -14}


def half_ulp(x: np.ndarray, dtype: str) -> np.ndarray:
    """Half the spacing of ``dtype`` values at magnitude |x| (0 for f32 outputs
    compared against an f64 value is not used: f32 stores get the f32 ulp)."""
    ax = np.abs(np.asarray(x, dtype=np.float64))
    _, e = np.frexp(np.maximum(ax, np.finfo(np.float64).tiny))
    e = np.maximum(e, MIN_EXP[dtype] + 1)
    return np.ldexp(1.0, e - SIG_BITS[dtype] - 1)


def excess(got, want, in_dtype: str, stored: str | None = None, extra=None) -> np.ndarray:
    """Per-element amount by which |got - want| exceeds the bound (<= 0 passes).
    ``extra`` adds a derived per-element bound (e.g. tape_rounding_bound)."""
    got = np.asarray(got, dtype=np.float64)
    want = np.asarray(want, dtype=np.float64)
    t = TOL[in_dtype]
    bound = t + t * np.abs(want)
    if extra is not None:
        bound = bound + extra
    if stored is not None:
        bound = bound + half_ulp(np.maximum(np.abs(want), np.abs(got)), stored)
    return np.abs(got - want) - bound


def assert_close(got, want, in_dtype: str, stored: str | None = None, what: str = "",
                 extra=None):
    ex = excess(got, want, in_dtype, stored, extra)
    if ex.size and not (ex <= 0).all():
        bad = np.argwhere(~(ex <= 0))
        i = tuple(bad[0])
        raise AssertionError(
            f"{what}: {len(bad)} of {ex.size} elements out of tolerance; first at {i}: "
            f"got {np.asarray(got)[i]!r} want {np.asarray(want)[i]!r} (excess {ex[i]:.3e})")


def tape_rounding_bound(k_log, g_log, delta, mask, accepted: int, dtype: str) -> np.ndarray:
    """Per-element bound on how far two replays can drift apart when their
    delta tapes were rounded to ``dtype`` independently (the GPU rounds its
    f32 delta, the oracle path rounds its f64 delta): each tape entry may land
    on the neighbouring representable value, one ulp away, and replay carries
    that error as  s <- g s + k (delta + e).  So
        bound[b,hv,dv,i] = sum_t |k[b,t,hv,i]| ulp(delta[b,t,hv,dv]) prod_{t'>t} |g[b,t',hv]|
    over the replayed (accepted, unmasked) steps.  Arrays are float64 oracle
    values: k_log [B,T,Hv,Dk], g_log [B,T,Hv], delta [B,T,Hv,Dv]."""
    B, T, Hv, Dv = delta.shape
    Dk = k_log.shape[3]
    act = np.ones((B, T), bool) if mask is None else mask.astype(bool)
    bound = np.zeros((B, Hv, Dv, Dk))
    for t in range(min(accepted, T)):
        on = act[:, t][:, None, None, None]
        ulp = 2.0 * half_ulp(np.nan_to_num(delta[:, t]), dtype)          # [B,Hv,Dv]
        step = np.abs(np.nan_to_num(g_log[:, t]))[:, :, None, None] * bound + \
            ulp[..., None] * np.abs(np.nan_to_num(k_log[:, t]))[:, :, None, :]
        bound = np.where(on, step, bound)
    return bound


def torch_dtype(dtype: str):
    import torch
    return {"f32": torch.float32, "bf16": torch.bfloat16, "f16": torch.float16}[dtype]


def to_dev(arr: np.ndarray, dev):
    """Storage array (see workloads) -> torch tensor on ``dev``, same bits."""
    import torch
    if arr.dtype == np.uint16:
        return torch.from_numpy(np.ascontiguousarray(arr).view(np.int16)).view(torch.bfloat16).to(dev)
    if arr.dtype == np.uint32:
        return torch.from_numpy(np.ascontiguousarray(arr).astype(np.int32)).to(dev)
    return torch.from_numpy(np.ascontiguousarray(arr)).to(dev)


def to_host_f64(t) -> np.ndarray:
    import torch
    return t.detach().to(torch.float64).cpu().numpy()


def storage_of(t) -> np.ndarray:
    """Torch tensor -> numpy array in workloads' storage form (bf16 as uint16 bits)."""
    import torch
    t = t.detach().cpu()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view(np.uint16)
    return t.numpy()


def round_to(x: np.ndarray, dtype: str) -> np.ndarray:
    """Round float64 values through float32 to the storage type; storage array."""
    return workloads.to_storage(np.asarray(x, dtype=np.float64).astype(np.float32), dtype)


def device_inputs(case, dev):
    """q, k, v, g, beta, state, mask of a workloads.Case on ``dev``."""
    q, k, v, g, beta = (to_dev(getattr(case, n), dev) for n in ("q", "k", "v", "g", "beta"))
    state = to_dev(case.state, dev)
    mask = None if case.mask is None else to_dev(case.mask, dev)
    return q, k, v, g, beta, state, mask


# ------------------------------------------------------------ guard bands
# Canary bytes around output buffers stand in for a memory checker: an
# output allocated with guarded_full sits between two 256-byte bands of a
# fixed pattern, and after every GPU test (tests/conftest.py) each band
# registered during the test must still hold it, so a kernel that writes past
# either end of its output is caught.
GUARD_BYTES = 256          # keeps the output 256-byte aligned
GUARD_PATTERN = 0xA5
_GUARDS = []


def guarded_full(shape, fill, dtype, dev):
    """torch.full(shape, fill) with canary bands before and after it."""
    import torch
    shape = tuple(int(x) for x in shape)
    n = 1
    for x in shape:
        n *= x
    nbytes = n * torch.empty((), dtype=dtype).element_size()
    raw = torch.empty(2 * GUARD_BYTES + nbytes, dtype=torch.uint8, device=dev)
    raw.fill_(GUARD_PATTERN)
    out = raw[GUARD_BYTES:GUARD_BYTES + nbytes].view(dtype).view(shape)
    out.fill_(fill)
    _GUARDS.append((raw, nbytes))
    return out


def guarded_like(t, fill=float("nan")):
    return guarded_full(t.shape, fill, t.dtype, t.device)


def reset_guards():
    _GUARDS.clear()


def broken_guards():
    """Descriptions of the bands that no longer hold the pattern."""
    bad = []
    for i, (raw, nbytes) in enumerate(_GUARDS):
        head = raw[:GUARD_BYTES]
        tail = raw[GUARD_BYTES + nbytes:]
        if not bool((head == GUARD_PATTERN).all()) or not bool((tail == GUARD_PATTERN).all()):
            bad.append(f"guarded buffer {i} ({nbytes} bytes): a write landed outside it")
    return bad
