"""GPU parity of the tcgen05 record path against the float64 oracle.

bf16 record calls of 7 to 16 steps with Dk = 128 and Dv a multiple of 128
run on the tensor-core kernel of record_tc.cuh (TMA-fed, accumulators in
tensor memory).  These cases are chosen to route there and cover what that
kernel adds: several 128-row units per tile (Dv = 256), more units than one
wave of the persistent grid, calls shorter than the 16-step chunk (down to
the 7-step threshold and the speculative-verify shape), every mask form, the
tiled GQA mapping, tape capture on and off, scale folds inside the chunk,
in-place state, NaN in masked input slots, a state_out that is 16- but not
32-byte aligned, and the eligibility edges
(T = 6 and T = 17, v not 16-byte aligned) that fall back to the other
kernels.
"""
from __future__ import annotations

import numpy as np
import pytest

import oracle
import workloads
from gdn_testutil import assert_close, device_inputs, guarded_full, to_host_f64

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

import linear_attention_recurrence_step_gb300 as gdn  # noqa: E402

SENTINEL = float("nan")


@pytest.fixture(scope="module")
def dev():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    gdn.load()
    return torch.device("cuda:0")


def _outputs(case, dev, capture=True):
    B, T, Hv, Dv, Dk = case.B, case.T, case.Hv, case.Dv, case.Dk
    # guarded: the conftest checks the canary bands around every output
    out = dict(y=guarded_full((B, T, Hv, Dv), SENTINEL, torch.bfloat16, dev),
               delta_log=guarded_full((B, T, Hv, Dv), SENTINEL, torch.bfloat16, dev),
               state_out=guarded_full((B, Hv, Dv, Dk), SENTINEL, torch.float32, dev))
    if capture:
        out["k_log"] = guarded_full((B, T, Hv, Dk), SENTINEL, torch.bfloat16, dev)
        out["g_log"] = guarded_full((B, T, Hv), SENTINEL, torch.bfloat16, dev)
    return out


def _record(case, dev, capture=True, gqa="block", inputs=None):
    q, k, v, g, beta, s0, mask = inputs if inputs is not None else device_inputs(case, dev)
    out = _outputs(case, dev, capture)
    gdn.gdn_step_record(q, k, v, g, beta, s0, mask, gqa=gqa, **out)
    torch.cuda.synchronize()
    return out, s0


def _check(case, got, gqa="block", capture=True, row_relative=False):
    ref = oracle.record(case.f64("q"), case.f64("k"), case.f64("v"), case.f64("g"),
                        case.f64("beta"), case.f64("state"), case.mask, gqa=gqa)
    act = np.ones((case.B, case.T), bool) if case.mask is None else case.mask.astype(bool)
    st = to_host_f64(got["state_out"])
    if row_relative:
        # states of ~1e10 under growth: f32 carries absolute error in
        # proportion to each row's magnitude
        scale = np.abs(ref["state_out"]).max(axis=-1, keepdims=True)
        assert (np.abs(st - ref["state_out"]) <= 1e-3 * scale).all(), "state_out (row-relative)"
    else:
        assert_close(st, ref["state_out"], "bf16", None, "state_out")
        y = to_host_f64(got["y"])
        dl = to_host_f64(got["delta_log"])
        assert_close(y[act], ref["y"][act], "bf16", "bf16", "y")
        assert_close(dl[act], ref["delta_log"][act], "bf16", "bf16", "delta_log")
    assert np.isnan(to_host_f64(got["y"])[~act]).all(), "masked y written"
    assert np.isnan(to_host_f64(got["delta_log"])[~act]).all(), "masked delta_log written"
    if capture:
        kl = to_host_f64(got["k_log"])
        gl = to_host_f64(got["g_log"])
        np.testing.assert_array_equal(kl[act], ref["k_log"][act])
        np.testing.assert_array_equal(gl[act], ref["g_log"][act])
        assert np.isnan(kl[~act]).all() and np.isnan(gl[~act]).all(), "masked tape slots written"
    return ref


TC_SPECS = [
    dict(B=2, T=16, Hk=2, Hv=4, Dv=128, mask="bernoulli:0.8", seed=1201),
    dict(B=1, T=12, Hk=1, Hv=2, Dv=128, mask="none", seed=1202),
    dict(B=3, T=13, Hk=2, Hv=4, Dv=128, mask="prefix", seed=1203),
    dict(B=2, T=16, Hk=1, Hv=3, Dv=256, mask="bernoulli:0.6", seed=1204),   # two units per tile
    dict(B=16, T=16, Hk=8, Hv=32, Dv=128, mask="bernoulli:0.8", seed=1205),  # 512 units: several per warpgroup
    dict(B=2, T=15, Hk=4, Hv=4, Dv=128, mask="all_on", seed=1206),
    dict(B=2, T=16, Hk=2, Hv=4, Dv=128, mask="all_off", seed=1207),
    dict(B=16, T=8, Hk=16, Hv=32, Dv=128, mask="prefix", seed=1208),         # the speculative-verify shape
    dict(B=3, T=7, Hk=2, Hv=6, Dv=256, mask="bernoulli:0.7", seed=1209),     # the shortest call routed here
]


@pytest.mark.parametrize("spec", TC_SPECS, ids=lambda s: f"B{s['B']}T{s['T']}Hk{s['Hk']}Hv{s['Hv']}"
                                                       f"Dv{s['Dv']}-{s['mask']}")
def test_tc_record_matches_oracle(dev, spec):
    case = workloads.make_case(Dk=128, dtype="bf16", **spec)
    got, s0 = _record(case, dev)
    _check(case, got)
    if spec["mask"] == "all_off":
        assert torch.equal(got["state_out"], s0), "all-masked call must leave the state unchanged"


def test_tc_record_tiled_mapping_and_no_capture(dev):
    case = workloads.make_case(B=3, T=16, Hk=2, Hv=8, Dk=128, Dv=128, dtype="bf16", seed=1210,
                               mask="bernoulli:0.7")
    got, _ = _record(case, dev, capture=False, gqa="tiled")
    _check(case, got, gqa="tiled", capture=False)


@pytest.mark.parametrize("g_range,row_relative", [((0.0, 0.0), False),   # resets
                                                  ((0.1, 0.25), False),  # folds below 2^-32 inside the chunk
                                                  ((4.0, 5.0), True)])   # folds above 2^32 (growth)
def test_tc_record_decay_edges(dev, g_range, row_relative):
    case = workloads.make_case(B=2, T=16, Hk=2, Hv=4, Dk=128, Dv=128, dtype="bf16", seed=1220,
                               g_range=g_range, mask="bernoulli:0.8")
    got, _ = _record(case, dev)
    _check(case, got, row_relative=row_relative)


def test_tc_record_in_place(dev):
    case = workloads.make_config("rollback_b128_t16_bf16", batch=4)
    q, k, v, g, beta, s0, mask = device_inputs(case, dev)
    ref = gdn.gdn_step_record(q, k, v, g, beta, s0, mask, capture_tape=True)
    s_in = s0.clone()
    out = gdn.gdn_step_record(q, k, v, g, beta, s_in, mask, state_out=s_in, capture_tape=True)
    torch.cuda.synchronize()
    assert out.state_out.data_ptr() == s_in.data_ptr()
    assert torch.equal(s_in, ref.state_out), "in-place record differs from out-of-place"
    on = torch.from_numpy(case.mask.astype(bool)).to(dev)
    assert torch.equal(out.y[on], ref.y[on]) and torch.equal(out.delta_log[on], ref.delta_log[on])


def test_tc_record_ignores_masked_inputs(dev):
    """NaN in the q / k / v / g / beta slots of masked steps never reaches an
    output: the masked rows of K enter the products as zeros."""
    case = workloads.make_case(B=2, T=16, Hk=2, Hv=4, Dk=128, Dv=128, dtype="bf16", seed=1230,
                               mask="bernoulli:0.6")
    clean, _ = _record(case, dev)
    off = ~case.mask.astype(bool)
    dirty_case = workloads.Case(**case.__dict__)
    nan_bf16 = np.uint16(0x7fc0)
    for name in ("q", "k", "v", "g", "beta"):
        arr = getattr(case, name).copy()
        arr[off] = nan_bf16
        setattr(dirty_case, name, arr)
    dirty, _ = _record(dirty_case, dev)
    on = torch.from_numpy(case.mask.astype(bool)).to(dev)
    assert torch.equal(dirty["state_out"], clean["state_out"])
    assert torch.equal(dirty["y"][on], clean["y"][on])
    assert torch.equal(dirty["delta_log"][on], clean["delta_log"][on])


def test_tc_record_eligibility_edges(dev):
    """T = 6 (below the threshold), T = 17 (two chunks) and a v tensor that is
    not 16-byte aligned take the other record kernels; all still match the
    oracle."""
    for T, seed in ((6, 1242), (17, 1240)):
        case = workloads.make_case(B=2, T=T, Hk=2, Hv=4, Dk=128, Dv=128, dtype="bf16", seed=seed,
                                   mask="bernoulli:0.8")
        got, _ = _record(case, dev)
        _check(case, got)
    case = workloads.make_case(B=2, T=16, Hk=2, Hv=4, Dk=128, Dv=128, dtype="bf16", seed=1241,
                               mask="bernoulli:0.8")
    q, k, v, g, beta, s0, mask = device_inputs(case, dev)
    buf = torch.empty(v.numel() + 1, dtype=torch.bfloat16, device=dev)
    v_off = buf[1:].view(v.shape)  # 2 bytes past a 16-byte boundary
    v_off.copy_(v)
    assert v_off.data_ptr() % 16 != 0
    got, _ = _record(case, dev, inputs=(q, k, v_off, g, beta, s0, mask))
    _check(case, got)


def test_tc_record_state_out_16_byte_offset(dev):
    """A state_out that is 16- but not 32-byte aligned (the ABI asks for 16)
    gives a result bit-identical to an aligned output, and nothing around it
    is written."""
    case = workloads.make_case(B=2, T=12, Hk=2, Hv=4, Dk=128, Dv=256, dtype="bf16", seed=1250,
                               mask="bernoulli:0.8")
    inputs = device_inputs(case, dev)
    ref, _ = _record(case, dev, inputs=inputs)
    assert ref["state_out"].data_ptr() % 32 == 0
    q, k, v, g, beta, s0, mask = inputs
    n = s0.numel()
    raw = guarded_full((n + 8,), SENTINEL, torch.float32, dev)
    off = (4 - (raw.data_ptr() // 4) % 8) % 8  # floats to 16 bytes past a 32-byte boundary
    so = raw[off:off + n].view(s0.shape)
    assert so.data_ptr() % 32 == 16
    out = _outputs(case, dev)
    out["state_out"] = so
    gdn.gdn_step_record(q, k, v, g, beta, s0, mask, **out)
    torch.cuda.synchronize()
    assert torch.equal(so, ref["state_out"])
    assert torch.isnan(raw[:off]).all() and torch.isnan(raw[off + n:]).all()
    for name in ("y", "delta_log", "k_log", "g_log"):
        assert torch.equal(out[name].view(torch.int16), ref[name].view(torch.int16)), name
