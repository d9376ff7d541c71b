"""Chains of dependent library calls launched without synchronisation.

Every kernel of the library is launched as a programmatic dependent launch:
it may be scheduled while the kernel before it in the stream is still
running, and it reads and writes global memory only after that kernel has
completed (griddepcontrol.wait).  These chains feed each call's outputs to
the next and write in place into buffers the previous call reads, through
every launcher (tcgen05 record, persistent stream replay, FP32 record and
replay, chunked prefill, tensor-core replay, tiled repeat).  A chain run with
no synchronisation must give results bit-identical to the same chain with a
device synchronisation after every call; a captured step replayed as a CUDA
graph many times must give the eager result every time.
"""
from __future__ import annotations

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


def _nan(shape, dtype, dev):
    return torch.full(shape, float("nan"), dtype=dtype, device=dev)


def _bits(t):
    return t.view(torch.int32) if t.dtype == torch.float32 else t.view(torch.int16)


def _decode_chain(dev, sync):
    """bf16: record (tcgen05, T = 16) -> replay in place onto the state the
    record read (stream kernel) -> record of 5 steps in place (FP32 kernel) ->
    single-step replay in place (FP32 replay kernel), four rounds."""
    c16 = workloads.make_case(B=4, T=16, Hk=2, Hv=4, Dk=128, Dv=256, dtype="bf16", seed=1301,
                              mask="bernoulli:0.8")
    c5 = workloads.make_case(B=4, T=5, Hk=2, Hv=4, Dk=128, Dv=256, dtype="bf16", seed=1302)
    q, k, v, g, beta, s0, mask = device_inputs(c16, dev)
    q5, k5, v5, g5, b5, _, _ = device_inputs(c5, dev)
    s = s0.clone()
    seen = []
    for i in range(4):
        shp = (c16.B, c16.T, c16.Hv, c16.Dv)
        rec = gdn.gdn_step_record(q, k, v, g, beta, s, mask, capture_tape=True,
                                  y=_nan(shp, torch.bfloat16, dev), delta_log=_nan(shp, torch.bfloat16, dev))
        if sync:
            torch.cuda.synchronize()
        gdn.gdn_state_replay(rec.delta_log, rec.k_log, rec.g_log, s, mask, accepted=11 - i, state_out=s)
        if sync:
            torch.cuda.synchronize()
        r5 = gdn.gdn_step_record(q5, k5, v5, g5, b5, s, None, state_out=s, capture_tape=True)
        if sync:
            torch.cuda.synchronize()
        gdn.gdn_state_replay(r5.delta_log, r5.k_log, r5.g_log, s, None, accepted=1, state_out=s)
        if sync:
            torch.cuda.synchronize()
        seen += [rec.y, rec.delta_log, rec.state_out, r5.y, s.clone()]
    torch.cuda.synchronize()
    return seen


def _prefill_chain(dev, sync):
    """f32: tiled repeat of q and k -> chunked prefill -> tensor-core replay
    in place onto the state the prefill read, three rounds."""
    case = workloads.make_case(B=1, T=80, Hk=2, Hv=4, Dk=128, Dv=128, dtype="f32", seed=1303,
                               g_range=(0.95, 1.0), mask="bernoulli:0.9")
    q, k, v, g, beta, s0, mask = device_inputs(case, dev)
    s = s0.clone()
    seen = []
    for i in range(3):
        qx = gdn.gqa_repeat_tiled(q.view(case.T, case.Hk, case.Dk), case.Hv)
        kx = gdn.gqa_repeat_tiled(k.view(case.T, case.Hk, case.Dk), case.Hv)
        if sync:
            torch.cuda.synchronize()
        shp = (1, case.T, case.Hv, case.Dv)
        out = gdn.gdn_chunk_prefill(qx.view(1, case.T, case.Hv, case.Dk), kx.view(1, case.T, case.Hv, case.Dk),
                                    v, g, beta, s, mask, capture_tape=True,
                                    y=_nan(shp, torch.float32, dev), delta_log=_nan(shp, torch.float32, dev))
        if sync:
            torch.cuda.synchronize()
        gdn.gdn_chunk_replay(out.delta_log, out.k_log, out.g_log, s, mask, accepted=case.T - 7 * i,
                             state_out=s)
        if sync:
            torch.cuda.synchronize()
        seen += [qx, kx, out.y, out.delta_log, out.state_out, s.clone()]
    torch.cuda.synchronize()
    return seen


@pytest.mark.parametrize("chain", [_decode_chain, _prefill_chain], ids=["record-replay", "prefill-replay"])
def test_unsynchronised_chain_is_bit_identical(dev, chain):
    free = chain(dev, sync=False)
    stepped = chain(dev, sync=True)
    assert len(free) == len(stepped)
    for i, (a, b) in enumerate(zip(free, stepped)):
        # masked slots of y / delta_log are left unwritten: NaN in both runs
        if a.shape != b.shape:
            raise AssertionError(f"output {i}: shapes differ")
        ba, bb = _bits(a), _bits(b)
        same = ba == bb
        both_nan = torch.isnan(a.float()) & torch.isnan(b.float())
        assert bool((same | both_nan).all()), f"output {i} differs between the two runs"


def test_graph_replays_reuse_the_counter_slot(dev):
    """A captured record + replay step (the replay's blocks past its fixed
    shares come from a per-launch counter slot, fixed in the graph) replayed
    300 times in one stream: every replay resets the slot it used, so every
    replay gives the eager result, and the dependent launches inside the
    graph keep their order."""
    case = workloads.make_config("rollback_b128_t16_bf16", batch=32)  # 2048 replay blocks: counter in use
    q, k, v, g, beta, s0, mask = device_inputs(case, dev)
    shp = (case.B, case.T, case.Hv, case.Dv)
    out = dict(y=torch.empty(shp, dtype=torch.bfloat16, device=dev),
               delta_log=torch.empty(shp, dtype=torch.bfloat16, device=dev),
               k_log=torch.empty((case.B, case.T, case.Hv, case.Dk), dtype=torch.bfloat16, device=dev),
               g_log=torch.empty((case.B, case.T, case.Hv), dtype=torch.bfloat16, device=dev),
               state_out=torch.empty_like(s0))
    s_rep = torch.empty_like(s0)

    def step():
        gdn.gdn_step_record(q, k, v, g, beta, s0, mask, **out)
        gdn.gdn_state_replay(out["delta_log"], out["k_log"], out["g_log"], s0, mask, accepted=11,
                             state_out=s_rep)

    step()
    torch.cuda.synchronize()
    ref_rec, ref_rep = out["state_out"].clone(), s_rep.clone()
    side = torch.cuda.Stream(dev)
    side.wait_stream(torch.cuda.current_stream(dev))
    with torch.cuda.stream(side):
        step()  # warm-up on the capture stream
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=side):
        step()
    for i in range(300):
        if i % 50 == 0:
            out["state_out"].fill_(float("nan"))
            s_rep.fill_(float("nan"))
        graph.replay()
        if i % 50 == 49:
            torch.cuda.synchronize()
            assert torch.equal(out["state_out"], ref_rec), f"record after replay {i}"
            assert torch.equal(s_rep, ref_rep), f"replay after replay {i}"
