"""GPU parity of the persistent TMA-fed replay (replay_stream.cuh).

gdn_state_replay calls with Dk = 128, 2 to 16 steps and 16-byte aligned
delta_log rows run on the stream kernel (single-step calls stay on the FP32
replay kernel); the same call with delta_log moved off its 16-byte boundary
runs the FP32 replay kernel.  Both fold the same
steps with the same f32 operations in the same order, so their results must
be bit-identical for every tape type; each case is also held to the oracle.
The cases cover fewer blocks than SMs and several blocks per group, ragged
row blocks (Dv = 72, 200), every mask form, accepted = 0 / inside / T /
beyond T, per-sequence counts (negative, 0, inside, beyond T), in-place
state, NaN in tape slots that are never read, calls large enough that most
blocks are handed out by the launch's counter rather than the CTAs' fixed
shares, and launches on two streams at once.
"""
from __future__ import annotations

import numpy as np
import pytest

import oracle
import workloads
from gdn_testutil import (assert_close, device_inputs, guarded_like, round_to, to_dev,
                          to_host_f64)

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

import linear_attention_recurrence_step_gb300 as gdn  # noqa: E402


@pytest.fixture(scope="module")
def dev():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    gdn.load()
    return torch.device("cuda:0")


def _host_tape(case):
    """The oracle's record tape rounded to the tape dtype (no GPU value)."""
    ref = oracle.record(case.f64("q"), case.f64("k"), case.f64("v"), case.f64("g"), case.f64("beta"),
                        case.f64("state"), case.mask)
    dt = case.dtype
    return (round_to(np.nan_to_num(ref["delta_log"]), dt), round_to(np.nan_to_num(ref["k_log"]), dt),
            round_to(np.nan_to_num(ref["g_log"]), dt))


def _off16(t):
    """A copy of t whose data starts one element past a 16-byte boundary."""
    buf = torch.empty(t.numel() + 8, dtype=t.dtype, device=t.device)
    v = buf[1:1 + t.numel()].view(t.shape)
    v.copy_(t)
    assert v.data_ptr() % 16 != 0
    return v


def _both(dtape, dkl, dgl, s0, mask, **kw):
    stream = gdn.gdn_state_replay(dtape, dkl, dgl, s0, mask, state_out=guarded_like(s0), **kw)
    fp32 = gdn.gdn_state_replay(_off16(dtape), dkl, dgl, s0, mask, **kw)
    torch.cuda.synchronize()
    return stream, fp32


SPECS = [
    dict(B=1, T=2, Hk=1, Hv=2, Dv=128, dtype="bf16", mask="none", seed=1401),            # 4 blocks, fewer than SMs
    dict(B=4, T=8, Hk=2, Hv=8, Dv=128, dtype="bf16", mask="prefix", seed=1402),
    dict(B=8, T=16, Hk=4, Hv=16, Dv=128, dtype="bf16", mask="bernoulli:0.8", seed=1403),  # 256 blocks
    dict(B=3, T=13, Hk=2, Hv=4, Dv=72, dtype="f32", mask="bernoulli:0.6", seed=1404),     # ragged blocks
    dict(B=2, T=16, Hk=1, Hv=3, Dv=200, dtype="f16", mask="all_on", seed=1405),
    dict(B=20, T=16, Hk=8, Hv=32, Dv=128, dtype="bf16", mask="bernoulli:0.8", seed=1406),  # 1280 blocks
    # 2048 ragged blocks: past the CTAs' fixed shares, so handed out by the counter
    dict(B=16, T=16, Hk=8, Hv=32, Dv=200, dtype="f16", mask="prefix", seed=1407),
]


@pytest.mark.parametrize("spec", SPECS, ids=lambda s: f"{s['dtype']}-B{s['B']}T{s['T']}Hv{s['Hv']}"
                                                    f"Dv{s['Dv']}-{s['mask']}")
def test_stream_replay_matches_fp32_kernel_and_oracle(dev, spec):
    case = workloads.make_case(Dk=128, **spec)
    tape, kl, gl = _host_tape(case)
    dt = case.dtype
    dtape, dkl, dgl = to_dev(tape, dev), to_dev(kl, dev), to_dev(gl, dev)
    _, _, _, _, _, s0, mask = device_inputs(case, dev)
    for acc in sorted({0, 1, case.T // 2, case.T, case.T + 3}):
        stream, fp32 = _both(dtape, dkl, dgl, s0, mask, accepted=acc)
        assert torch.equal(stream, fp32), f"accepted={acc}"
        ref = oracle.replay(workloads.widen(tape, dt), workloads.widen(kl, dt), workloads.widen(gl, dt),
                            case.f64("state"), case.mask, accepted=acc)
        assert_close(to_host_f64(stream), ref, dt, None, f"replay accepted={acc}")


def test_stream_replay_per_sequence_in_place_and_unused_slots(dev):
    case = workloads.make_case(B=6, T=16, Hk=2, Hv=4, Dk=128, Dv=128, dtype="bf16", seed=1410,
                               mask="bernoulli:0.7")
    tape, kl, gl = _host_tape(case)
    acc = np.array([-3, 0, 5, 16, 40, 11], dtype=np.int32)
    dacc = torch.from_numpy(acc).to(dev)
    # tape slots at or past each sequence's count hold NaN: never read
    tape_n, kl_n, gl_n = tape.copy(), kl.copy(), gl.copy()
    nan16 = np.uint16(0x7fc0)
    for b, a in enumerate(np.clip(acc, 0, case.T)):
        tape_n[b, a:] = nan16
        kl_n[b, a:] = nan16
        gl_n[b, a:] = nan16
    dtape, dkl, dgl = to_dev(tape_n, dev), to_dev(kl_n, dev), to_dev(gl_n, dev)
    _, _, _, _, _, s0, mask = device_inputs(case, dev)
    stream = gdn.gdn_state_replay_per_seq(dtape, dkl, dgl, s0, mask, accepted=dacc,
                                          state_out=guarded_like(s0))
    fp32 = gdn.gdn_state_replay_per_seq(_off16(dtape), dkl, dgl, s0, mask, accepted=dacc)
    torch.cuda.synchronize()
    assert torch.equal(stream, fp32)
    assert not torch.isnan(stream).any()
    ref = oracle.replay(workloads.widen(tape, "bf16"), workloads.widen(kl, "bf16"),
                        workloads.widen(gl, "bf16"), case.f64("state"), case.mask,
                        accepted=acc.astype(np.int64))
    assert_close(to_host_f64(stream), ref, "bf16", None, "per-sequence stream replay")
    s1 = s0.clone()
    gdn.gdn_state_replay_per_seq(dtape, dkl, dgl, s1, mask, accepted=dacc, state_out=s1)
    torch.cuda.synchronize()
    assert torch.equal(s1, stream), "in-place equals out-of-place"


def test_stream_replay_f32_record_bit_exact(dev):
    """A float32 record's own tape, replayed over every prefix length, lands
    on the record of that prefix bit for bit (same operations as record)."""
    case = workloads.make_case(B=2, T=16, Hk=2, Hv=4, Dk=128, Dv=128, dtype="f32", seed=1420,
                               mask="bernoulli:0.8")
    q, k, v, g, beta, s0, mask = device_inputs(case, dev)
    full = gdn.gdn_step_record(q, k, v, g, beta, s0, mask, capture_tape=True)
    for a in (3, 9, 16):
        sub = gdn.gdn_step_record(q[:, :a].contiguous(), k[:, :a].contiguous(), v[:, :a].contiguous(),
                                  g[:, :a].contiguous(), beta[:, :a].contiguous(), s0,
                                  mask[:, :a].contiguous(), capture_tape=False)
        st = gdn.gdn_state_replay(full.delta_log, full.k_log, full.g_log, s0, mask, accepted=a)
        torch.cuda.synchronize()
        assert torch.equal(st, sub.state_out), f"accepted={a}"


def test_stream_replay_two_streams_and_counter_slot_reuse(dev):
    """The persistent replay hands its blocks out from a per-launch counter
    (one of 256 slots, reset by each launch's last CTA).  Launches alternating
    between two streams, so that two run at once, and more launches than
    there are slots, all give the result of a lone call.  Batch 32 has 2048
    blocks, more than the CTAs' fixed shares, so the counter is in use."""
    case = workloads.make_config("rollback_b128_t16_bf16", batch=32)
    q, k, v, g, beta, s0, mask = device_inputs(case, dev)
    rec = gdn.gdn_step_record(q, k, v, g, beta, s0, mask, capture_tape=True)
    ref = gdn.gdn_state_replay(rec.delta_log, rec.k_log, rec.g_log, s0, mask, accepted=11)
    torch.cuda.synchronize()
    streams = [torch.cuda.Stream(dev), torch.cuda.Stream(dev)]
    per = 8  # output buffers per stream, reused in stream order
    outs = [[torch.empty_like(s0) for _ in range(per)] for _ in streams]
    launches = 0
    while launches < 300:
        for o in outs:
            for t in o:
                t.fill_(float("nan"))
        torch.cuda.synchronize()
        for i in range(per):
            for si, st in enumerate(streams):
                with torch.cuda.stream(st):
                    gdn.gdn_state_replay(rec.delta_log, rec.k_log, rec.g_log, s0, mask, accepted=11,
                                         state_out=outs[si][i])
                launches += 1
        torch.cuda.synchronize()
        for si in range(len(streams)):
            for i in range(per):
                assert torch.equal(outs[si][i], ref), f"launch batch ending at {launches}: stream {si}, buffer {i}"


def test_stream_replay_counter_per_sequence_and_unused_slots(dev):
    """Per-sequence counts and NaN in unread tape slots on a call large enough
    (3072 blocks) that most blocks come from the launch's counter: bit-equal
    to the FP32 replay kernel and within the oracle's tolerance."""
    case = workloads.make_case(B=48, T=16, Hk=2, Hv=32, Dk=128, Dv=128, dtype="bf16", seed=1411,
                               mask="bernoulli:0.8")
    tape, kl, gl = _host_tape(case)
    rng = np.random.default_rng(1412)
    acc = rng.integers(-2, case.T + 5, size=case.B).astype(np.int32)
    dacc = torch.from_numpy(acc).to(dev)
    tape_n, kl_n, gl_n = tape.copy(), kl.copy(), gl.copy()
    nan16 = np.uint16(0x7fc0)
    for b, a in enumerate(np.clip(acc, 0, case.T)):
        tape_n[b, a:] = nan16
        kl_n[b, a:] = nan16
        gl_n[b, a:] = nan16
    dtape, dkl, dgl = to_dev(tape_n, dev), to_dev(kl_n, dev), to_dev(gl_n, dev)
    _, _, _, _, _, s0, mask = device_inputs(case, dev)
    stream = gdn.gdn_state_replay_per_seq(dtape, dkl, dgl, s0, mask, accepted=dacc,
                                          state_out=guarded_like(s0))
    fp32 = gdn.gdn_state_replay_per_seq(_off16(dtape), dkl, dgl, s0, mask, accepted=dacc)
    torch.cuda.synchronize()
    assert torch.equal(stream, fp32)
    assert not torch.isnan(stream).any()
    ref = oracle.replay(workloads.widen(tape, "bf16"), workloads.widen(kl, "bf16"),
                        workloads.widen(gl, "bf16"), case.f64("state"), case.mask,
                        accepted=acc.astype(np.int64))
    assert_close(to_host_f64(stream), ref, "bf16", None, "per-sequence stream replay, counter-fed")
