"""gdn_chunk_prefill_noalloc: the chunked prefill on the library's static
device scratch, for callers that cannot allocate device memory when they
call (a runtime whose pool allocator owns all of HBM, a plugin host without
access to the allocator, a serving loop that may not call cudaMalloc).  The
source pages have no counterpart to this entry point.

* two calls in a row on different inputs, each bit-equal to
  gdn_chunk_prefill on a caller workspace (same kernels, same arithmetic):
  the second call must not see what the first left in the shared scratch;
* parity with the float64 oracle;
* a problem whose workspace exceeds the 32 MiB static block is refused with
  GDN_ERR_UNSUPPORTED before anything is launched.

This file is collected last, so a run that stops at the first failure has
already run every other test; it also passes alone in a fresh process.
"""
from __future__ import annotations

import pytest

import oracle
import workloads
from gdn_testutil import assert_close, device_inputs, to_host_f64

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

import linear_attention_recurrence_step_gb300 as gdn  # noqa: E402

STATIC_SCRATCH = 32 << 20
UNSUPPORTED = 2


@pytest.fixture(scope="module")
def dev():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    gdn.load()
    return torch.device("cuda:0")


def _call_pair(case, dev):
    q, k, v, g, beta, s0, mask = device_inputs(case, dev)
    a = gdn.gdn_chunk_prefill_noalloc(q, k, v, g, beta, s0, mask, gqa="tiled", capture_tape=True)
    b = gdn.gdn_chunk_prefill(q, k, v, g, beta, s0, mask, gqa="tiled", capture_tape=True)
    torch.cuda.synchronize()
    on = torch.from_numpy(case.mask.astype(bool)).to(dev)
    assert torch.equal(a.state_out, b.state_out)
    assert torch.equal(a.y[on], b.y[on]) and torch.equal(a.delta_log[on], b.delta_log[on])
    return a


def test_noalloc_two_calls_match_workspace_call_and_oracle(dev):
    # two calls in a row on different problems (the second smaller, so every
    # scratch block it uses still holds the first call's data when it
    # starts): both must equal the workspace entry point bit for bit
    first = workloads.make_case(B=2, T=77, Hk=2, Hv=4, Dk=128, Dv=48, dtype="f32", seed=801,
                                mask="bernoulli:0.8")
    second = workloads.make_case(B=1, T=40, Hk=2, Hv=4, Dk=128, Dv=48, dtype="f32", seed=802,
                                 mask="bernoulli:0.8")
    for case in (first, second):
        a = _call_pair(case, dev)
        ref = oracle.record(case.f64("q"), case.f64("k"), case.f64("v"), case.f64("g"),
                            case.f64("beta"), case.f64("state"), case.mask, gqa="tiled")
        act = case.mask.astype(bool)
        assert_close(to_host_f64(a.state_out), ref["state_out"], "f32", None, "state_out")
        assert_close(to_host_f64(a.y)[act], ref["y"][act], "f32", None, "y")


def test_noalloc_long_prefill_fits(dev):
    # the long-prefill workload needs 17.8 MB of workspace: inside the block
    case = workloads.make_config("long_prefill_t4096_f32")
    assert gdn.gdn_chunk_prefill_workspace_size(case.B, case.T, case.Hv) <= STATIC_SCRATCH
    q, k, v, g, beta, s0, mask = device_inputs(case, dev)
    a = gdn.gdn_chunk_prefill_noalloc(q, k, v, g, beta, s0, mask, gqa="tiled")
    b = gdn.gdn_chunk_prefill(q, k, v, g, beta, s0, mask, gqa="tiled")
    torch.cuda.synchronize()
    assert torch.equal(a.state_out, b.state_out) and torch.equal(a.y, b.y)


def test_noalloc_refuses_oversized_problem(dev):
    # B * Hv * ceil(T/16) * 2176 bytes > 32 MiB: refused on the host
    B, T, Hk, Hv, Dk, Dv = 8, 4096, 16, 32, 128, 128
    need = gdn.gdn_chunk_prefill_workspace_size(B, T, Hv)
    assert need > STATIC_SCRATCH
    lib = gdn.load()
    fake = 0x10000  # never dereferenced: the size check comes first
    st = lib.gdn_chunk_prefill_noalloc(*([fake] * 7), fake, fake, None, None, None,
                                       B, T, Hk, Hv, Dk, Dv, 0, 0, None)
    assert st == UNSUPPORTED
    msg = lib.gdn_last_error().decode()
    assert msg.startswith("gdn_chunk_prefill_noalloc") and str(need) in msg
