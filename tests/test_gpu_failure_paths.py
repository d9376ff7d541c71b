"""Failure paths on the GPU, made without any fault.

* Bounded waits: with the wait bound of the tensor-core kernels shortened to
  one clock cycle (gdn_set_wait_bound) and one wait that nothing completes
  injected (gdn_inject_wait_expiry), their pipeline waits run out.  The
  kernels must return (no hang), poison what they could not finish with NaN,
  raise the flag gdn_wait_status reports, and leave the context usable: the
  next calls with the default bound give the normal results and no flag.
* Forced launch failures: gdn_force_launch_failures makes the next call
  return GDN_ERR_CUDA before anything is enqueued (its outputs stay
  untouched); the call after it runs normally.
"""
from __future__ import annotations

import numpy as np
import pytest

import workloads
from gdn_testutil import device_inputs

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

import linear_attention_recurrence_step_gb300 as gdn  # noqa: E402


@pytest.fixture(scope="module")
def dev():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    gdn.load()
    return torch.device("cuda:0")


@pytest.fixture
def restore_hooks():
    yield
    gdn.inject_wait_expiry(False)
    gdn.set_wait_bound(0)
    gdn.force_launch_failures(0)


def _record(case, dev):
    q, k, v, g, beta, s0, mask = device_inputs(case, dev)
    out = gdn.gdn_step_record(q, k, v, g, beta, s0, mask, capture_tape=True)
    torch.cuda.synchronize()
    return out


def test_record_wait_expiry_is_reported(dev, restore_hooks):
    case = workloads.make_config("rollback_b128_t16_bf16", batch=8)  # the tcgen05 record path
    assert not gdn.wait_status()
    clean = _record(case, dev)
    assert not gdn.wait_status()
    gdn.set_wait_bound(1)
    gdn.inject_wait_expiry(True)
    bad = _record(case, dev)
    assert gdn.wait_status(), "an expired wait must raise the flag"
    assert torch.isnan(bad.state_out).any(), "the unfinished units are poisoned with NaN"
    assert not gdn.wait_status(), "reading the flag clears it"
    gdn.inject_wait_expiry(False)
    gdn.set_wait_bound(0)
    again = _record(case, dev)
    assert not gdn.wait_status()
    assert torch.equal(again.state_out, clean.state_out), "the context must stay usable"


def test_chunk_replay_wait_expiry_is_reported(dev, restore_hooks):
    case = workloads.make_case(B=8, T=64, Hk=8, Hv=32, Dk=128, Dv=128, dtype="f32", seed=1301,
                               mask="none")
    q, k, v, g, beta, s0, mask = device_inputs(case, dev)
    rec = gdn.gdn_step_record(q, k, v, g, beta, s0, mask, capture_tape=True)
    clean = gdn.gdn_chunk_replay(rec.delta_log, rec.k_log, rec.g_log, s0, mask, accepted=case.T)
    torch.cuda.synchronize()
    assert not gdn.wait_status()
    gdn.set_wait_bound(1)
    gdn.inject_wait_expiry(True)
    bad = gdn.gdn_chunk_replay(rec.delta_log, rec.k_log, rec.g_log, s0, mask, accepted=case.T)
    torch.cuda.synchronize()
    assert gdn.wait_status()
    assert torch.isnan(bad).any()
    gdn.inject_wait_expiry(False)
    gdn.set_wait_bound(0)
    again = gdn.gdn_chunk_replay(rec.delta_log, rec.k_log, rec.g_log, s0, mask, accepted=case.T)
    torch.cuda.synchronize()
    assert not gdn.wait_status()
    assert torch.equal(again, clean)


@pytest.mark.parametrize("batch", [4, 32])
def test_stream_replay_wait_expiry_is_reported(dev, restore_hooks, batch):
    """The persistent TMA-fed replay (bf16 tape, 16 steps, Dk = 128): its
    ring waits give up, every row it could not fold is NaN, the flag is
    raised, and the next call runs normally.  Batch 4 (256 blocks) runs on
    each CTA's fixed share alone; batch 32 (2048 blocks) also hands blocks
    out from the launch's counter, so a failing CTA takes every block left
    there and writes it as NaN."""
    case = workloads.make_config("rollback_b128_t16_bf16", batch=batch)
    q, k, v, g, beta, s0, mask = device_inputs(case, dev)
    rec = gdn.gdn_step_record(q, k, v, g, beta, s0, mask, capture_tape=True)
    clean = gdn.gdn_state_replay(rec.delta_log, rec.k_log, rec.g_log, s0, mask, accepted=11)
    torch.cuda.synchronize()
    assert not gdn.wait_status()
    gdn.set_wait_bound(1)
    gdn.inject_wait_expiry(True)
    bad = gdn.gdn_state_replay(rec.delta_log, rec.k_log, rec.g_log, s0, mask, accepted=11)
    torch.cuda.synchronize()
    assert gdn.wait_status()
    assert torch.isnan(bad).all(), "both compute groups stop at their first block"
    gdn.inject_wait_expiry(False)
    gdn.set_wait_bound(0)
    again = gdn.gdn_state_replay(rec.delta_log, rec.k_log, rec.g_log, s0, mask, accepted=11)
    torch.cuda.synchronize()
    assert not gdn.wait_status()
    assert torch.equal(again, clean)


def test_forced_launch_failure_enqueues_nothing(dev, restore_hooks):
    case = workloads.make_config("rollback_b128_t16_bf16", batch=2)
    q, k, v, g, beta, s0, mask = device_inputs(case, dev)
    sentinel = torch.full_like(s0, float("nan"))
    gdn.force_launch_failures(1)
    with pytest.raises(gdn.GdnError) as err:
        gdn.gdn_step_record(q, k, v, g, beta, s0, mask, state_out=sentinel)
    assert err.value.args[0].startswith("gdn_step_record") and "GDN_ERR_CUDA" in err.value.args[0]
    torch.cuda.synchronize()
    assert torch.isnan(sentinel).all(), "a failed call must not write its outputs"
    out = gdn.gdn_step_record(q, k, v, g, beta, s0, mask, state_out=sentinel)
    torch.cuda.synchronize()
    assert not torch.isnan(out.state_out).any()
    assert np.isfinite(out.state_out.cpu().numpy()).all()
