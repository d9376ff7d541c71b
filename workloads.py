"""Seeded synthetic inputs for the GatedDeltaNet record / replay step.

This module is the input recipe and nothing else: random draws, the
L2-normalisation of q/k head rows, the sigmoid that makes beta, the mask
patterns, and the casts to the storage dtype (round-to-nearest-even for
bf16/f16).  None of the recurrence's arithmetic lives here.  The float64
oracle and the CUDA path both consume these arrays unchanged, which is the
only thing the two sides share.

Arrays are returned in their *storage* form:

* ``f32``  -> ``numpy.float32``
* ``bf16`` -> ``numpy.uint16`` holding the bf16 bit patterns
* ``f16``  -> ``numpy.float16``

``widen(arr, dtype)`` gives the exact float64 value of every element, which
is what the oracle is fed.

Shapes follow the GatedDeltaNet record kernel's tensors on the
"metaltile-std gated_delta_replay.rs" page (kernel argument list of
``gated_delta_step_record``): q, k ``[B,T,Hk,Dk]``; v ``[B,T,Hv,Dv]``;
g, beta ``[B,T,Hv]``; state ``[B,Hv,Dv,Dk]`` (always float32 here);
mask ``[B,T]`` uint32.

Draw order for one case, from ``numpy.random.default_rng(seed)``:
q, k, v (standard normal, float32), g (uniform on ``g_range``), the
pre-sigmoid normal for beta, the state (normal, std ``state_std``, unless
zeros), then the mask draw, then ``accepted`` when it is random.
"""
from __future__ import annotations

from dataclasses import dataclass, field
from typing import Dict, Optional, Tuple

import numpy as np

DTYPES = ("f32", "bf16", "f16")

# Named workloads.  Sizes, distributions and structure are the five
# configurations this library is measured and checked on.
CONFIGS: Dict[str, dict] = {
    # tiny f32 parity case: record then replay with accepted=3
    "tiny_f32": dict(B=1, T=4, Hk=2, Hv=4, Dk=32, Dv=32, dtype="f32",
                     g_range=(0.9, 1.0), state="normal", mask="none",
                     accepted=3, seed=1000),
    # one decode token per sequence, bf16 inputs, f32 state
    "decode_b32_bf16": dict(B=32, T=1, Hk=16, Hv=32, Dk=128, Dv=128,
                            dtype="bf16", g_range=(0.9, 1.0), state="normal",
                            mask="none", accepted=1, seed=1001),
    # speculative verify: 8 drafts, per-sequence valid prefix L_b~U{1..8},
    # replay accepted~U{0..8} (one draw)
    "spec_verify_b16_t8_bf16": dict(B=16, T=8, Hk=16, Hv=32, Dk=128, Dv=128,
                                    dtype="bf16", g_range=(0.9, 1.0),
                                    state="normal", mask="prefix",
                                    accepted="uniform", seed=1002),
    # large-batch rollback: B=128, 16 drafts, Bernoulli(0.8) mask, replay 11
    "rollback_b128_t16_bf16": dict(B=128, T=16, Hk=16, Hv=32, Dk=128, Dv=128,
                                   dtype="bf16", g_range=(0.9, 1.0),
                                   state="normal", mask="bernoulli:0.8",
                                   accepted=11, seed=1003),
    # long prefill: tiled GQA repeat of q/k 16 -> 32 heads, then record over
    # 4096 steps from a zero state, f32
    "long_prefill_t4096_f32": dict(B=1, T=4096, Hk=16, Hv=32, Dk=128, Dv=128,
                                   dtype="f32", g_range=(0.95, 1.0),
                                   state="zeros", mask="none",
                                   accepted=4096, seed=1004, repeat=True),
}

CONFIG_ORDER = ("tiny_f32", "decode_b32_bf16", "spec_verify_b16_t8_bf16",
                "rollback_b128_t16_bf16", "long_prefill_t4096_f32")


# ---------------------------------------------------------------- dtype casts
def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 values to bf16 (nearest, ties to even); return the bits."""
    b = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    nan = np.isnan(x)
    rounded = (b + (((b >> 16) & np.uint32(1)) + np.uint32(0x7FFF))) >> 16
    out = rounded.astype(np.uint16)
    if nan.any():
        out[nan] = np.uint16(0x7FC0)
    return out


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    """Exact float32 value of bf16 bit patterns."""
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def to_storage(x32: np.ndarray, dtype: str) -> np.ndarray:
    """Cast float32 values to the storage form of ``dtype``."""
    if dtype == "f32":
        return np.ascontiguousarray(x32, dtype=np.float32)
    if dtype == "bf16":
        return f32_to_bf16_bits(x32)
    if dtype == "f16":
        return np.ascontiguousarray(x32.astype(np.float16))
    raise ValueError(f"unknown dtype {dtype!r}")


def widen(arr: np.ndarray, dtype: str) -> np.ndarray:
    """Exact float64 value of a storage array."""
    if dtype == "bf16":
        return bf16_bits_to_f32(arr).astype(np.float64)
    return np.asarray(arr).astype(np.float64)


def elem_size(dtype: str) -> int:
    return {"f32": 4, "bf16": 2, "f16": 2}[dtype]


# ------------------------------------------------------------------ the case
@dataclass
class Case:
    """One seeded problem in storage form (see module docstring)."""
    B: int
    T: int
    Hk: int
    Hv: int
    Dk: int
    Dv: int
    dtype: str
    q: np.ndarray
    k: np.ndarray
    v: np.ndarray
    g: np.ndarray
    beta: np.ndarray
    state: np.ndarray          # float32 [B,Hv,Dv,Dk]
    mask: Optional[np.ndarray]  # uint32 [B,T] or None (no mask)
    accepted: int
    name: str = "custom"
    meta: dict = field(default_factory=dict)

    def f64(self, name: str) -> np.ndarray:
        arr = getattr(self, name)
        if name == "state":
            return arr.astype(np.float64)
        return widen(arr, self.dtype)

    @property
    def shape_kwargs(self) -> dict:
        return dict(B=self.B, T=self.T, Hk=self.Hk, Hv=self.Hv, Dk=self.Dk, Dv=self.Dv)


def _l2_normalise_rows(x: np.ndarray) -> np.ndarray:
    """Divide every last-axis row by its L2 norm (float32, norm floored at 1e-12)."""
    x = x.astype(np.float32)
    n = np.sqrt(np.sum(x * x, axis=-1, keepdims=True, dtype=np.float32))
    return (x / np.maximum(n, np.float32(1e-12))).astype(np.float32)


def _sigmoid32(x: np.ndarray) -> np.ndarray:
    x = x.astype(np.float32)
    return (np.float32(1.0) / (np.float32(1.0) + np.exp(-x))).astype(np.float32)


def make_case(B: int, T: int, Hk: int, Hv: int, Dk: int, Dv: int, *,
              dtype: str = "f32", seed: int = 0,
              g_range: Tuple[float, float] = (0.9, 1.0),
              state: str = "normal", state_std: float = 0.1,
              mask: str = "none", accepted="T", name: str = "custom",
              normalise_qk: bool = True) -> Case:
    """Draw one case.

    mask: ``"none"`` (no mask pointer), ``"prefix"`` (mask[b,t]=1 for
    t<L_b, L_b~U{1..T}), ``"bernoulli:p"`` (independent per (b,t)),
    ``"all_off"`` or ``"all_on"`` (explicit mask array).
    accepted: an int, ``"T"``, or ``"uniform"`` (one draw from U{0..T}).
    """
    if dtype not in DTYPES:
        raise ValueError(f"unknown dtype {dtype!r}")
    rng = np.random.default_rng(seed)
    q = rng.standard_normal((B, T, Hk, Dk), dtype=np.float32)
    k = rng.standard_normal((B, T, Hk, Dk), dtype=np.float32)
    if normalise_qk:
        q = _l2_normalise_rows(q)
        k = _l2_normalise_rows(k)
    v = rng.standard_normal((B, T, Hv, Dv), dtype=np.float32)
    lo, hi = g_range
    g = rng.uniform(lo, hi, size=(B, T, Hv)).astype(np.float32)
    beta = _sigmoid32(rng.standard_normal((B, T, Hv), dtype=np.float32))
    if state == "zeros":
        s = np.zeros((B, Hv, Dv, Dk), dtype=np.float32)
    elif state == "normal":
        s = (rng.standard_normal((B, Hv, Dv, Dk), dtype=np.float32)
             * np.float32(state_std)).astype(np.float32)
    else:
        raise ValueError(f"unknown state recipe {state!r}")

    m: Optional[np.ndarray]
    meta: dict = {}
    if mask == "none":
        m = None
    elif mask == "all_on":
        m = np.ones((B, T), dtype=np.uint32)
    elif mask == "all_off":
        m = np.zeros((B, T), dtype=np.uint32)
    elif mask == "prefix":
        lengths = rng.integers(1, T + 1, size=B)
        m = (np.arange(T)[None, :] < lengths[:, None]).astype(np.uint32)
        meta["prefix_lengths"] = lengths
    elif mask.startswith("bernoulli:"):
        p = float(mask.split(":", 1)[1])
        m = (rng.random((B, T)) < p).astype(np.uint32)
    else:
        raise ValueError(f"unknown mask recipe {mask!r}")

    if accepted == "T":
        acc = T
    elif accepted == "uniform":
        acc = int(rng.integers(0, T + 1))
    else:
        acc = int(accepted)

    return Case(B=B, T=T, Hk=Hk, Hv=Hv, Dk=Dk, Dv=Dv, dtype=dtype,
                q=to_storage(q, dtype), k=to_storage(k, dtype),
                v=to_storage(v, dtype), g=to_storage(g, dtype),
                beta=to_storage(beta, dtype), state=s, mask=m,
                accepted=acc, name=name, meta=meta)


def make_config(name: str, *, batch: Optional[int] = None) -> Case:
    """Draw the named workload; ``batch`` overrides B (rank shards, samples)."""
    c = dict(CONFIGS[name])
    seed = c.pop("seed")
    c.pop("repeat", None)
    if batch is not None:
        c["B"] = int(batch)
    return make_case(seed=seed, name=name, **c)


def uses_repeat(name: str) -> bool:
    """Whether the workload expands q/k with the tiled GQA repeat first."""
    return bool(CONFIGS[name].get("repeat", False))
