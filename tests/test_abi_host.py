"""Host-side tests of the C ABI (no GPU needed).

* libgdn.so builds for sm_103a, loads, and exports every function that
  include/gdn.h declares;
* every argument check of include/gdn.h returns its status before anything
  is launched.  Each call below carries at least one invalid argument, so it
  can never reach a kernel (the fake pointers are never dereferenced).
"""
from __future__ import annotations

import ctypes
import os
import re

import pytest

import linear_attention_recurrence_step_gb300 as gdn

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "gdn.h")

OK, INVALID, UNSUPPORTED, MISALIGNED, CUDA = 0, 1, 2, 3, 4
F32, BF16, F16 = 0, 1, 2
A = 0x10000  # fake, 16-byte aligned device addresses (never dereferenced)


def P(i: int) -> int:
    return A * (i + 1)


@pytest.fixture(scope="module")
def lib():
    gdn.build()
    return gdn.load()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    text = re.sub(r"//[^\n]*", "", text)
    names = re.findall(r"^[A-Za-z_][\w \t\*]*?\b(\w+)\s*\(", text, flags=re.M)
    return sorted(set(n for n in names if n not in ("defined",)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for want in ("gdn_step_record", "gdn_step_record_mapped", "gdn_chunk_prefill",
                 "gdn_chunk_prefill_workspace_size", "gdn_chunk_prefill_noalloc",
                 "gdn_chunk_replay", "gdn_chunk_replay_workspace_size", "gdn_state_replay",
                 "gdn_state_replay_per_seq", "gqa_repeat_tiled",
                 "gdn_status_string", "gdn_last_error", "gdn_abi_version"):
        assert want in names
    assert set(names) == set(gdn.EXPORTED)


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), f"libgdn.so does not export {name}"
    assert lib.gdn_abi_version() == 7


def test_library_is_sm103a():
    # the build passes exactly one -gencode, for sm_103a
    from linear_attention_recurrence_step_gb300 import _build
    assert _build.ARCH_FLAGS == ["-gencode", "arch=compute_103a,code=sm_103a"]
    assert os.path.exists(_build.LIB_PATH)


def test_status_strings(lib):
    for code, name in gdn.STATUS_NAMES.items():
        assert lib.gdn_status_string(code).decode() == name


def rec(lib, **kw):
    args = dict(q=P(0), k=P(1), v=P(2), g=P(3), beta=P(4), state_in=P(5), mask=None,
                y=P(6), state_out=P(7), delta_log=P(8), k_log=None, g_log=None,
                B=2, T=3, Hk=2, Hv=4, Dk=64, Dv=32, dtype=BF16, stream=None)
    args.update(kw)
    return lib.gdn_step_record(*args.values())


def rep(lib, **kw):
    args = dict(delta_log=P(0), k_log=P(1), g_log=P(2), state_in=P(3), mask=None,
                state_out=P(4), B=2, T=3, Hv=4, Dk=64, Dv=32, accepted=2, dtype=BF16,
                stream=None)
    args.update(kw)
    return lib.gdn_state_replay(*args.values())


def rec_mapped(lib, mapping=1, **kw):
    args = dict(q=P(0), k=P(1), v=P(2), g=P(3), beta=P(4), state_in=P(5), mask=None,
                y=P(6), state_out=P(7), delta_log=P(8), k_log=None, g_log=None,
                B=2, T=3, Hk=2, Hv=4, Dk=64, Dv=32, mapping=mapping, dtype=BF16, stream=None)
    args.update(kw)
    return lib.gdn_step_record_mapped(*args.values())


def chunk(lib, **kw):
    ws = lib.gdn_chunk_prefill_workspace_size(2, 3, 4)
    args = dict(q=P(0), k=P(1), v=P(2), g=P(3), beta=P(4), state_in=P(5), mask=None,
                y=P(6), state_out=P(7), delta_log=None, k_log=None, g_log=None,
                B=2, T=3, Hk=2, Hv=4, Dk=64, Dv=32, mapping=0, workspace=P(9),
                workspace_bytes=ws, dtype=F32, stream=None)
    args.update(kw)
    return lib.gdn_chunk_prefill(*args.values())


def test_chunk_workspace_size(lib):
    # one block of 2 x 16 x 16 + 2 x 16 floats per (b, hv, 16-step chunk)
    assert lib.gdn_chunk_prefill_workspace_size(1, 4096, 32) == 32 * 256 * 544 * 4
    assert lib.gdn_chunk_prefill_workspace_size(2, 17, 3) == 2 * 3 * 2 * 544 * 4
    assert lib.gdn_chunk_prefill_workspace_size(0, 5, 5) == 0
    assert lib.gdn_chunk_prefill_workspace_size(1 << 40, 1 << 30, 64) == 0


CHUNK_CASES = {
    "null workspace": (dict(workspace=None), INVALID),
    "workspace too small": (dict(workspace_bytes=100), INVALID),
    "workspace misaligned": (dict(workspace=P(9) + 8), MISALIGNED),
    "mapping=3": (dict(mapping=3), INVALID),
    "null y": (dict(y=None), INVALID),
    "T=0": (dict(T=0), INVALID),
    "Hv%Hk": (dict(Hk=3), INVALID),
    "Dk=80": (dict(Dk=80), UNSUPPORTED),
    "dtype": (dict(dtype=7), UNSUPPORTED),
    "q misaligned": (dict(q=P(0) + 4), MISALIGNED),
    "state overlap": (dict(state_out=P(5) + 16), INVALID),
    # more CTAs than a grid holds (2^31 - 1) is refused, not launched short:
    # 2^30 chunks of 16 steps, or 2^30 blocks of 16 rows, for 4 value heads
    "grid chunks": (dict(T=16 << 30, state_out=P(5), workspace_bytes=1 << 50), INVALID),
    "grid rows": (dict(Dv=16 << 30, state_out=P(5), workspace_bytes=1 << 50), INVALID),
}


@pytest.mark.parametrize("name", sorted(CHUNK_CASES))
def test_chunk_prefill_rejects(lib, name):
    kw, want = CHUNK_CASES[name]
    assert chunk(lib, **kw) == want
    msg = lib.gdn_last_error().decode()
    assert msg.startswith("gdn_chunk_prefill")
    if name == "workspace too small":
        assert "need 17408 bytes, have 100" in msg  # 2 x 4 x 1 x 544 x 4
    if name.startswith("grid"):
        assert "grid too large" in msg


def creplay(lib, **kw):
    ws = lib.gdn_chunk_replay_workspace_size(2, 3, 4, 64, 32)
    args = dict(delta_log=P(0), k_log=P(1), g_log=P(2), state_in=P(3), mask=None,
                state_out=P(4), B=2, T=3, Hv=4, Dk=64, Dv=32, accepted=2, per_seq=None,
                workspace=P(9), workspace_bytes=ws, dtype=F32, stream=None)
    args.update(kw)
    return lib.gdn_chunk_replay(*args.values())


def test_chunk_replay_workspace_size(lib):
    # decay weights [B,Hv,T] + totals [B,Hv] (16-byte padded) + partial sums
    # when the steps are split (fewer than 304 CTAs from the tiles alone at
    # Dk <= 128, where two CTAs share each of the 152 SMs; 152 above): 32
    # tiles of 4096 steps take 9 splits of 464 steps at Dk = 128, 4 at 256
    B, T, Hv, Dk, Dv = 1, 4096, 32, 128, 128
    w, gam = 32 * 4096 * 4, 32 * 4
    assert lib.gdn_chunk_replay_workspace_size(B, T, Hv, Dk, Dv) == w + gam + 9 * 32 * 128 * 128 * 4
    assert lib.gdn_chunk_replay_workspace_size(B, T, Hv, 256, Dv) == w + gam + 4 * 32 * 128 * 256 * 4
    assert lib.gdn_chunk_replay_workspace_size(128, 16, 32, 128, 128) == 128 * 32 * 16 * 4 + 128 * 32 * 4
    assert lib.gdn_chunk_replay_workspace_size(0, 16, 32, 128, 128) == 0


@pytest.mark.parametrize("B,Hv,T,Dk,splits", [
    (1, 32, 4096, 128, 9),    # 32 tiles: 304 // 32 = 9 splits of 464 steps (288 CTAs)
    (1, 100, 4096, 128, 3),   # 100 tiles: 3 splits (300 CTAs)
    (2, 152, 4096, 128, 1),   # 304 tiles fill the GPU alone: no split, no partial sums
    (1, 32, 4096, 256, 4),    # Dk = 256, one CTA per SM: 152 // 32 = 4 splits
    (1, 1, 100, 128, 7),      # a short tape splits no finer than its 16-step stages
])
def test_chunk_replay_split_plan(lib, B, Hv, T, Dk, splits):
    """The tensor-core replay splits the steps of each tile over CTAs until
    the tiles fill 152 SMs (two CTAs each up to Dk = 128, one above), in
    whole 16-step stages; the partial sums of the splits are the workspace
    beyond the decay weights and totals."""
    Dv = 128
    w = -(-B * Hv * T * 4 // 16) * 16
    gam = -(-B * Hv * 4 // 16) * 16
    part = 0 if splits == 1 else splits * B * Hv * Dv * Dk * 4
    assert lib.gdn_chunk_replay_workspace_size(B, T, Hv, Dk, Dv) == w + gam + part


CREPLAY_CASES = {
    "null workspace": (dict(workspace=None), INVALID),
    "workspace too small": (dict(workspace_bytes=16), INVALID),
    "accepted<0": (dict(accepted=-1), INVALID),
    "null k_log": (dict(k_log=None), INVALID),
    "Dk=80": (dict(Dk=80), UNSUPPORTED),
    "dtype": (dict(dtype=4), UNSUPPORTED),
    "state misaligned": (dict(state_in=P(3) + 4), MISALIGNED),
    "per_seq misaligned": (dict(per_seq=P(10) + 2), MISALIGNED),
    "state overlap": (dict(state_out=P(3) + 16), INVALID),
    # 2^32 (b, hv) tiles: more CTAs than a grid holds
    "grid tiles": (dict(B=1 << 20, Hv=1 << 12, state_out=P(3), workspace_bytes=1 << 62), INVALID),
}


@pytest.mark.parametrize("name", sorted(CREPLAY_CASES))
def test_chunk_replay_rejects(lib, name):
    kw, want = CREPLAY_CASES[name]
    assert creplay(lib, **kw) == want
    msg = lib.gdn_last_error().decode()
    assert msg.startswith("gdn_chunk_replay")
    if name.startswith("grid"):
        assert "grid too large" in msg


def rec_ts(lib, **kw):
    args = dict(q=P(0), k=P(1), v=P(2), g=P(3), beta=P(4), state_in=P(5), mask=None,
                y=P(6), state_out=P(7), delta_log=P(8), k_log=None, g_log=None,
                B=2, T=3, Hk=2, Hv=4, Dk=64, Dv=32, mapping=0, dtype=BF16, stream=None)
    args.update(kw)
    return lib.gdn_step_record_tstate(*args.values())


def rep_ts(lib, **kw):
    args = dict(delta_log=P(0), k_log=P(1), g_log=P(2), state_in=P(3), mask=None,
                state_out=P(4), B=2, T=3, Hv=4, Dk=64, Dv=32, accepted=2, per_seq=None,
                dtype=BF16, stream=None)
    args.update(kw)
    return lib.gdn_state_replay_tstate(*args.values())


TSTATE_CASES = {
    "record mapping=5": (rec_ts, dict(mapping=5), INVALID),
    "record state misaligned": (rec_ts, dict(state_in=P(5) + 8), MISALIGNED),
    # bf16 state: 2 x 4 x 32 x 64 x 2 bytes = 32768; an 8-byte offset overlaps
    "record state overlap": (rec_ts, dict(state_out=P(5) + 16), INVALID),
    "record Dk=48": (rec_ts, dict(Dk=48), UNSUPPORTED),
    "replay accepted<0": (rep_ts, dict(accepted=-3), INVALID),
    "replay per_seq misaligned": (rep_ts, dict(per_seq=P(9) + 2), MISALIGNED),
    "replay null g_log": (rep_ts, dict(g_log=None), INVALID),
}


@pytest.mark.parametrize("name", sorted(TSTATE_CASES))
def test_tstate_rejects(lib, name):
    fn, kw, want = TSTATE_CASES[name]
    assert fn(lib, **kw) == want
    assert lib.gdn_last_error().decode().startswith(
        "gdn_step_record_tstate" if fn is rec_ts else "gdn_state_replay_tstate")


def rep_seq(lib, **kw):
    args = dict(delta_log=P(0), k_log=P(1), g_log=P(2), state_in=P(3), mask=None,
                state_out=P(4), B=2, T=3, Hv=4, Dk=64, Dv=32, accepted=P(5), dtype=BF16,
                stream=None)
    args.update(kw)
    return lib.gdn_state_replay_per_seq(*args.values())


def rpt(lib, **kw):
    args = dict(src=P(0), dst=P(8), seq=4, hg=2, h=6, k=8, dtype=F32,
                src_bytes=4 * 2 * 8 * 4, dst_bytes=4 * 6 * 8 * 4, stream=None)
    args.update(kw)
    return lib.gqa_repeat_tiled(*args.values())


RECORD_CASES = {
    "B=0": (dict(B=0), INVALID),
    "T=0": (dict(T=0), INVALID),
    "Hk=0": (dict(Hk=0), INVALID),
    "Dv=-1": (dict(Dv=-1), INVALID),
    "Hv%Hk": (dict(Hk=3), INVALID),
    "null q": (dict(q=None), INVALID),
    "null state_out": (dict(state_out=None), INVALID),
    "null delta_log": (dict(delta_log=None), INVALID),
    "Dk%32": (dict(Dk=48), UNSUPPORTED),
    "Dk=96 not compiled": (dict(Dk=96), UNSUPPORTED),
    "Dk=512 not compiled": (dict(Dk=512), UNSUPPORTED),
    "dtype": (dict(dtype=9), UNSUPPORTED),
    "overflow": (dict(B=1 << 40, T=1 << 20), INVALID),
    "q misaligned": (dict(q=P(0) + 4), MISALIGNED),
    "state_in misaligned": (dict(state_in=P(5) + 8), MISALIGNED),
    "v odd address bf16": (dict(v=P(2) + 1), MISALIGNED),
    "mask misaligned": (dict(mask=P(9) + 2), MISALIGNED),
    "k_log misaligned": (dict(k_log=P(10) + 8), MISALIGNED),
    "state overlap": (dict(state_out=P(5) + 16), INVALID),
}


@pytest.mark.parametrize("name", sorted(RECORD_CASES))
def test_record_rejects(lib, name):
    kw, want = RECORD_CASES[name]
    assert rec(lib, **kw) == want
    assert lib.gdn_last_error().decode().startswith("gdn_step_record")


MAPPED_CASES = {
    "mapping=2": (dict(mapping=2), INVALID),
    "mapping=-1": (dict(mapping=-1), INVALID),
    "tiled Hv%Hk": (dict(Hk=3), INVALID),
    "tiled B=0": (dict(B=0), INVALID),
    "tiled Dk=96": (dict(Dk=96), UNSUPPORTED),
    "tiled k misaligned": (dict(k=P(1) + 8), MISALIGNED),
    "block null v": (dict(mapping=0, v=None), INVALID),
}


@pytest.mark.parametrize("name", sorted(MAPPED_CASES))
def test_record_mapped_rejects(lib, name):
    kw, want = MAPPED_CASES[name]
    assert rec_mapped(lib, **kw) == want
    assert lib.gdn_last_error().decode().startswith("gdn_step_record_mapped")


PER_SEQ_CASES = {
    "null accepted": (dict(accepted=None), INVALID),
    "accepted misaligned": (dict(accepted=P(5) + 2), MISALIGNED),
    "T=0": (dict(T=0), INVALID),
    "null g_log": (dict(g_log=None), INVALID),
    "Dk=48": (dict(Dk=48), UNSUPPORTED),
    "state overlap": (dict(state_out=P(3) + 32), INVALID),
}


@pytest.mark.parametrize("name", sorted(PER_SEQ_CASES))
def test_replay_per_seq_rejects(lib, name):
    kw, want = PER_SEQ_CASES[name]
    assert rep_seq(lib, **kw) == want
    assert lib.gdn_last_error().decode().startswith("gdn_state_replay_per_seq")


REPLAY_CASES = {
    "B=0": (dict(B=0), INVALID),
    "Dv=0": (dict(Dv=0), INVALID),
    "accepted<0": (dict(accepted=-1), INVALID),
    "null k_log": (dict(k_log=None), INVALID),
    "null g_log": (dict(g_log=None), INVALID),
    "Dk=80": (dict(Dk=80), UNSUPPORTED),
    "dtype": (dict(dtype=-1), UNSUPPORTED),
    "k_log misaligned": (dict(k_log=P(1) + 2), MISALIGNED),
    "state overlap": (dict(state_out=P(3) + 32), INVALID),
    "overflow": (dict(B=1 << 50, Dv=1 << 20), INVALID),
}


@pytest.mark.parametrize("name", sorted(REPLAY_CASES))
def test_replay_rejects(lib, name):
    kw, want = REPLAY_CASES[name]
    assert rep(lib, **kw) == want
    assert lib.gdn_last_error().decode().startswith("gdn_state_replay")


REPEAT_CASES = {
    # the error rules of dispatch_repeat_tiled_f32 ("mlx-native repeat_tiled.rs")
    "seq=0": (dict(seq=0), INVALID),
    "hg=0": (dict(hg=0), INVALID),
    "h=0": (dict(h=0), INVALID),
    "k=0": (dict(k=0), INVALID),
    "h%hg": (dict(h=5), INVALID),
    "src too small": (dict(src_bytes=4 * 2 * 8 * 4 - 1), INVALID),
    "dst too small": (dict(dst_bytes=4 * 6 * 8 * 4 - 4), INVALID),
    "src overflow": (dict(seq=1 << 40, k=1 << 30), INVALID),
    "null src": (dict(src=None), INVALID),
    "overlap": (dict(dst=P(0) + 64), INVALID),
    "dtype": (dict(dtype=5), UNSUPPORTED),
    "misaligned f32": (dict(src=P(0) + 2), MISALIGNED),
}


@pytest.mark.parametrize("name", sorted(REPEAT_CASES))
def test_repeat_rejects(lib, name):
    kw, want = REPEAT_CASES[name]
    assert rpt(lib, **kw) == want
    msg = lib.gdn_last_error().decode()
    assert msg.startswith("gqa_repeat_tiled")
    if name == "src too small":
        assert "need 256 bytes, have 255" in msg


def test_python_binding_refuses_without_library(tmp_path):
    with pytest.raises(gdn.GdnError):
        gdn.load(str(tmp_path / "missing.so"))


# ------------------------------------------------- testing hooks (no device)
def test_forced_launch_failures_stop_before_the_device(lib):
    """gdn_force_launch_failures(n): the next n calls that pass validation
    return GDN_ERR_CUDA without touching the device; a call that fails
    validation does not consume one.  Exactly n valid calls are made here (a
    further valid call with these fake pointers would reach the device)."""
    try:
        assert lib.gdn_force_launch_failures(2) == OK
        assert rec(lib, B=0) == INVALID                      # validation first, nothing consumed
        assert rec(lib) == CUDA
        msg = lib.gdn_last_error().decode()
        assert msg.startswith("gdn_step_record") and "forced by gdn_force_launch_failures" in msg
        assert rpt(lib) == CUDA
        assert "forced" in lib.gdn_last_error().decode()
    finally:
        assert lib.gdn_force_launch_failures(0) == OK
    assert lib.gdn_force_launch_failures(-1) == INVALID


def test_wait_hooks_reject_bad_arguments(lib):
    assert lib.gdn_set_wait_bound(-1) == INVALID
    assert lib.gdn_set_wait_bound(0) == OK
    assert lib.gdn_inject_wait_expiry(0) == OK
    assert lib.gdn_wait_status(None) == INVALID
    assert lib.gdn_last_error().decode().startswith("gdn_wait_status")
