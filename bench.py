#!/usr/bin/env python
"""Benchmark: GatedDeltaNet record + replay tokens/s and achieved HBM GB/s.

One step = the whole hot path over one batch of the workload: the record
kernel (T steps, delta tape plus k_log / g_log capture) followed by the
replay kernel (the accepted prefix folded onto the pre-record snapshot).
The default workload is the 128-sequence rollback case (B=128, T=16,
Hk=16, Hv=32, Dk=Dv=128, bf16 inputs and tape, f32 state, Bernoulli(0.8)
mask, accepted=11); ``--config`` picks another named workload.

Timing: W untimed warm-up steps, then K steps between CUDA events on the
launching stream, bracketed by a barrier and torch.cuda.synchronize(); with
N processes (torchrun) every rank runs its own full batch (weak scaling, no
data-path collective) and the maximum time over ranks is used.  Replay folds
onto its own copy of the snapshot (not the buffer record just read), and when
one buffer set fits in L2 the steps rotate over enough sets that a set is
read again only after twice the L2 capacity of other traffic; at the default
size one set (1 GiB) is already far larger than L2.  The timed K steps have
no event between their kernels (an event there delays the next kernel's
launch by a few microseconds and keeps it from starting while the one before
it finishes); per-kernel durations come from a second pass over the same K
steps with an event pair around each launch (``config.kernel_timing``).
Beside the
measured peak, ``roofline.same_size_copy`` gives the rate of a plain
device-to-device copy moving as many bytes as the dominant kernel (L2-cold),
the most one pass over that much data reaches on this GPU, and each
kernel's fraction of it.

``--impl reference`` times the float64 CPU oracle on the same workload (a
bounded batch sample per step) and prints the same JSON line.
"""
from __future__ import annotations

import argparse
import hashlib
import glob
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import workloads  # noqa: E402

METRIC = "GDN record+replay tokens/s and achieved HBM GB/s (% of GB300 peak), 1 GPU"
DEFAULT_CONFIG = "rollback_b128_t16_bf16"
FALLBACK_HBM_GBS = 6800.0
L2_BYTES = 129 * 1024 * 1024
KERNEL_SOURCES = os.path.join(ROOT, "linear_attention_recurrence_step_gb300", "csrc")


# ---------------------------------------------------------------- accounting
CHUNK_MIN_T = 256  # bench "auto": calls this long take the chunked prefill


def algorithmic_bytes(case, accepted: int, capture: bool = True):
    """Bytes the method must move (each touched once), per launch.

    Record: the state read and written once (f32), plus for every active
    (b, t): the q and k rows of its key head, the v row, g and beta, the y and
    delta_log rows written (and k_log / g_log when captured), plus the mask.
    Replay: the state read and written once, plus for every active (b, t) with
    t < accepted: the delta_log row, the k_log row and g_log, plus the mask
    entries it reads.  Masked-off and unaccepted steps move nothing."""
    eb = workloads.elem_size(case.dtype)
    B, T, Hk, Hv, Dk, Dv = case.B, case.T, case.Hk, case.Hv, case.Dk, case.Dv
    act = np.ones((B, T), bool) if case.mask is None else case.mask.astype(bool)
    n_act = int(act.sum())
    state = B * Hv * Dv * Dk * 4
    mask_b = 0 if case.mask is None else B * T * 4
    per_step_rec = (2 * Hk * Dk + Hv * Dv + 2 * Hv + 2 * Hv * Dv) * eb
    if capture:
        per_step_rec += (Hv * Dk + Hv) * eb
    rec = 2 * state + n_act * per_step_rec + mask_b
    steps = min(accepted, T)
    n_rep = int(act[:, :steps].sum())
    rep = 2 * state + n_rep * (Hv * Dv + Hv * Dk + Hv) * eb + \
        (0 if case.mask is None else B * steps * 4)
    return rec, rep


def algorithmic_bytes_all_positions(case, accepted: int, capture: bool = True):
    """The same, counting every position whether its mask is on or off:
    record moves every (b, t) row, replay every (b, t) row with t < accepted
    (an upper bound on the bytes a masked call has to move)."""
    eb = workloads.elem_size(case.dtype)
    B, T, Hk, Hv, Dk, Dv = case.B, case.T, case.Hk, case.Hv, case.Dk, case.Dv
    state = B * Hv * Dv * Dk * 4
    mask_b = 0 if case.mask is None else B * T * 4
    per_step_rec = (2 * Hk * Dk + Hv * Dv + 2 * Hv + 2 * Hv * Dv) * eb
    if capture:
        per_step_rec += (Hv * Dk + Hv) * eb
    steps = min(accepted, T)
    rec = 2 * state + B * T * per_step_rec + mask_b
    rep = 2 * state + B * steps * (Hv * Dv + Hv * Dk + Hv) * eb + (0 if case.mask is None else B * steps * 4)
    return rec, rep


def hbm_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def kernel_source_hash() -> str:
    h = hashlib.sha256()
    for p in sorted(glob.glob(os.path.join(KERNEL_SOURCES, "*"))):
        if p.endswith((".cu", ".cuh", ".h")):
            h.update(open(p, "rb").read())
    return h.hexdigest()[:16]


def measured_traffic(kernel: str, workload: str):
    """DRAM bytes per launch from the committed ncu summary, if it was taken
    on the current kernel sources (else None)."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            t = json.load(f)
    except Exception:
        return None
    if t.get("kernel_source_hash") != kernel_source_hash():
        return None
    entry = t.get("kernels", {}).get(f"{kernel}:{workload}")
    return None if entry is None else entry.get("dram_bytes_per_launch")


# ---------------------------------------------------------------- clocks
class ClockSampler:
    """nvidia-smi clock / throttle samples while the timed region runs."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id: str | None):
        self.gpu_id = gpu_id
        self.proc = None
        self.lines = []

    def __enter__(self):
        cmd = ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
               "-lms", "100"]
        if self.gpu_id:
            cmd += ["-i", self.gpu_id]
        try:
            self.proc = subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL,
                                         text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
            time.sleep(0.25)
        except Exception:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(0.15)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
            self.thread.join(timeout=2)

    def summary(self):
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 7:
                continue
            try:
                sm.append(float(parts[0]))
                mx.append(float(parts[1]))
            except ValueError:
                continue
            for name, val in zip(names, parts[3:7]):
                if val.lower() == "active":
                    reasons.add(name)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx),
                "reasons": sorted(reasons), "samples": len(sm)}


# ---------------------------------------------------------------- our arm
def _dist_init(world):
    import torch
    import torch.distributed as dist
    if world > 1 and not dist.is_initialized():
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    return dist if world > 1 else None


def max_over_ranks(x: float, dist, device=None) -> float:
    """Max of a scalar over ranks (timing only: not part of the data path)."""
    if dist is None:
        return x
    import torch
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def rank_seed(base_seed: int, rank: int) -> int:
    """Each rank draws its own batch (independent shard of the job)."""
    return base_seed + 7919 * rank


def _make_rank_case(config: str, rank: int, batch=None):
    spec = dict(workloads.CONFIGS[config])
    seed = rank_seed(spec.pop("seed"), rank)
    spec.pop("repeat", None)
    if batch is not None:
        spec["B"] = int(batch)
    return workloads.make_case(seed=seed, name=config, **spec)


def run_ours(args, rank, world, local_rank):
    import torch
    import linear_attention_recurrence_step_gb300 as gdn

    dist = _dist_init(world)
    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    lib = gdn.load()
    case = _make_rank_case(args.config, rank, args.batch)
    record_path = args.record
    if record_path == "auto":
        record_path = "chunk" if case.T >= CHUNK_MIN_T else "step"
    # the tiled GQA expansion is read in place by the record kernels unless
    # the materialised repeat is asked for
    replay_path = args.replay
    if replay_path == "auto":
        replay_path = "chunk" if min(case.accepted, case.T) >= CHUNK_MIN_T else "step"
    fused_gqa = workloads.uses_repeat(args.config) and args.gqa == "fused"
    uses_repeat = workloads.uses_repeat(args.config) and not fused_gqa
    dt = case.dtype
    tdt = {"f32": torch.float32, "bf16": torch.bfloat16, "f16": torch.float16}[dt]
    code = gdn.DTYPE_CODES[tdt]
    B, T, Hk, Hv, Dk, Dv = case.B, case.T, case.Hk, case.Hv, case.Dk, case.Dv
    acc = case.accepted

    def host(arr):
        if arr.dtype == np.uint16:
            return torch.from_numpy(arr.view(np.int16)).view(torch.bfloat16)
        if arr.dtype == np.uint32:
            return torch.from_numpy(arr.astype(np.int32))
        return torch.from_numpy(np.ascontiguousarray(arr))

    names = ["q", "k", "v", "g", "beta"]
    h_in = {n: host(getattr(case, n)).pin_memory() for n in names}
    h_in["state"] = host(case.state).pin_memory()
    if case.mask is not None:
        h_in["mask"] = host(case.mask).pin_memory()
    d_in = {n: t.to(dev) for n, t in h_in.items()}
    Hk_rec = Hv if uses_repeat else Hk
    eb = workloads.elem_size(dt)
    stream = torch.cuda.current_stream(dev)
    sp = stream.cuda_stream

    def alloc_set(inputs=None):
        """One full set of device buffers for a step: inputs (copied from
        ``inputs`` or allocated) and every output / workspace."""
        d = dict(inputs) if inputs is not None else {n: torch.empty_like(t, device=dev)
                                                     for n, t in h_in.items()}
        if uses_repeat:
            d["qx"] = torch.empty((B, T, Hv, Dk), dtype=tdt, device=dev)
            d["kx"] = torch.empty((B, T, Hv, Dk), dtype=tdt, device=dev)
        d["y"] = torch.empty((B, T, Hv, Dv), dtype=tdt, device=dev)
        d["dl"] = torch.empty_like(d["y"])
        d["kl"] = torch.empty((B, T, Hv, Dk), dtype=tdt, device=dev)
        d["gl"] = torch.empty((B, T, Hv), dtype=tdt, device=dev)
        d["s_rec"] = torch.empty_like(d["state"])
        d["s_rep"] = torch.empty_like(d["state"])
        # replay folds onto its own copy of the pre-record snapshot (a serving
        # loop keeps the snapshot apart from the state record reads)
        d["snap"] = d["state"].clone()
        if record_path == "chunk":
            d["ws"] = torch.empty(lib.gdn_chunk_prefill_workspace_size(B, T, Hv), dtype=torch.uint8,
                                  device=dev)
        if replay_path == "chunk":
            d["rws"] = torch.empty(lib.gdn_chunk_replay_workspace_size(B, T, Hv, Dk, Dv),
                                   dtype=torch.uint8, device=dev)
        return d

    def check(st, what):
        if st != 0:
            raise RuntimeError(f"{what}: {gdn.STATUS_NAMES.get(st)}: {lib.gdn_last_error().decode()}")

    def make_launcher(d, sp):
        """The step's launches on buffer set ``d`` and stream ``sp`` (C ABI calls only)."""
        P = lambda name: d[name].data_ptr()
        mask_p = P("mask") if "mask" in d else None
        rec_args = ((P("qx") if uses_repeat else P("q")), (P("kx") if uses_repeat else P("k")), P("v"),
                    P("g"), P("beta"), P("state"), mask_p, P("y"), P("s_rec"), P("dl"), P("kl"),
                    P("gl"), B, T, Hk_rec, Hv, Dk, Dv, code, sp)
        if record_path == "chunk":
            rec_call = (lib.gdn_chunk_prefill, rec_args[:18] + (1 if fused_gqa else 0, P("ws"),
                                                                d["ws"].numel(), code, sp), "chunk prefill")
        elif fused_gqa:
            rec_call = (lib.gdn_step_record_mapped, rec_args[:18] + (1, code, sp), "record (tiled mapping)")
        else:
            rec_call = (lib.gdn_step_record, rec_args, "record")
        if replay_path == "chunk":
            rep_call = (lib.gdn_chunk_replay, (P("dl"), P("kl"), P("gl"), P("snap"), mask_p, P("s_rep"),
                                               B, T, Hv, Dk, Dv, acc, None, P("rws"), d["rws"].numel(),
                                               code, sp), "replay (tensor-core contraction)")
        else:
            rep_call = (lib.gdn_state_replay, (P("dl"), P("kl"), P("gl"), P("snap"), mask_p, P("s_rep"),
                                               B, T, Hv, Dk, Dv, acc, code, sp), "replay")
        rpts = []
        if uses_repeat:
            for src, dst in (("q", "qx"), ("k", "kx")):
                rpts.append((P(src), P(dst), B * T, Hk, Hv, Dk, code, B * T * Hk * Dk * eb,
                             B * T * Hv * Dk * eb, sp))

        def launch(ev=None, ev_stream=None):
            for r in rpts:
                check(lib.gqa_repeat_tiled(*r), "repeat")
            if ev is not None:
                ev[0].record(ev_stream)
            check(rec_call[0](*rec_call[1]), rec_call[2])
            if ev is not None:
                ev[1].record(ev_stream)
            check(rep_call[0](*rep_call[1]), rep_call[2])
            if ev is not None:
                ev[2].record(ev_stream)
        return launch

    set0 = alloc_set(d_in)
    y, dl, s_rep = set0["y"], set0["dl"], set0["s_rep"]
    # When one buffer set fits in L2 the steps rotate over several, so that a
    # set is read again only after at least twice the L2 capacity of other
    # traffic (no step finds its inputs in L2 from the step before).
    set_bytes = sum(t.numel() * t.element_size() for t in set0.values())
    n_sets = 1 if set_bytes >= 2 * L2_BYTES else min(16, -(-2 * L2_BYTES // set_bytes) + 1)
    timed_sets = [set0] + [alloc_set({n: t.clone() for n, t in d_in.items()}) for _ in range(n_sets - 1)]
    launchers_t = [make_launcher(d, sp) for d in timed_sets]
    step_no = [0]

    def step(ev=None):
        launchers_t[step_no[0] % n_sets](ev, stream)
        step_no[0] += 1

    n_replay = 1
    if replay_path == "chunk":
        plan_split = set0["rws"].numel() > (B * Hv * T * 4 + 15) // 16 * 16 + (B * Hv * 4 + 15) // 16 * 16
        n_replay = 3 if plan_split else 2
    launches_per_step = (2 if record_path == "chunk" else 1) + n_replay + (2 if uses_repeat else 0)
    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()

    K = args.steps
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(K)]
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    gpu_id = None
    try:
        gpu_id = "GPU-" + str(torch.cuda.get_device_properties(dev).uuid)
    except Exception:
        pass
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize()
    with ClockSampler(gpu_id if rank == 0 else None) as clocks:
        # the measured pass: K steps, an event only before the first and after
        # the last (an event between two kernels delays the second one's launch
        # and keeps it from being scheduled while the first is finishing)
        t0.record(stream)
        for i in range(K):
            step()
        t1.record(stream)
        torch.cuda.synchronize()
        # the same K steps again with an event before and after each kernel:
        # each kernel's mean duration, for the roofline figures
        for i in range(K):
            step(evs[i])
        torch.cuda.synchronize()
    if gdn.wait_status():
        raise RuntimeError("a bounded wait of a pipelined kernel ran out during the timed steps: "
                           "the outputs and the timing are not valid")
    if dist is not None:
        dist.barrier()
    elapsed_ms = t0.elapsed_time(t1)
    rec_ms = statistics.fmean(e[0].elapsed_time(e[1]) for e in evs)
    rep_ms = statistics.fmean(e[1].elapsed_time(e[2]) for e in evs)
    elapsed_ms = max_over_ranks(elapsed_ms, dist, dev)

    tokens_per_step = B * T
    ms_per_step = elapsed_ms / K
    value = world * tokens_per_step * K / (elapsed_ms / 1e3)
    rec_b, rep_b = algorithmic_bytes(case, acc, capture=True)
    rec_all, rep_all = algorithmic_bytes_all_positions(case, acc, capture=True)
    peak, peak_src = hbm_peak()
    rec_gbs = rec_b / (rec_ms * 1e-3) / 1e9
    rep_gbs = rep_b / (rep_ms * 1e-3) / 1e9
    step_bytes = rec_b + rep_b
    if uses_repeat:
        step_bytes += 2 * (B * T * Hk * Dk + B * T * Hv * Dk) * eb
    step_gbs = step_bytes / (ms_per_step * 1e-3) / 1e9


    # ---- end to end through the C ABI with host buffers (pinned): every step
    # copies its inputs host -> device, runs both kernels and copies y, the
    # delta tape and the replayed state device -> host.  Steps are pipelined
    # the way a serving loop runs them: three device buffer sets, one stream
    # each for uploads, kernels and downloads, so the upload of step i+1 and
    # the download of step i-1 overlap the kernels of step i.  (With two sets
    # the upload of step i+1 would wait for the download of step i-1, which
    # shares its set, and the two copies would run one after the other.)
    NE = 3
    e2e_steps = max(1, min(args.e2e_steps, K))
    h_y = [torch.empty(y.shape, dtype=tdt).pin_memory() for _ in range(NE)]
    h_dl = [torch.empty(dl.shape, dtype=tdt).pin_memory() for _ in range(NE)]
    h_st = [torch.empty(s_rep.shape, dtype=torch.float32).pin_memory() for _ in range(NE)]
    d2h = sum(t.numel() * t.element_size() for t in (h_y[0], h_dl[0], h_st[0]))
    # the device buffer sets; the uploaded state is also the snapshot replay
    # folds onto (record writes s_rec, never state)
    sets = [alloc_set() for _ in range(NE)]
    for d in sets:
        d["snap"] = d["state"]
    # The step's own inputs (q, k, v, g, beta, mask) of each set live in one
    # device buffer at 256-byte aligned offsets, mirrored by one pinned host
    # buffer, so a step uploads them with one copy (the state separately).
    small = [n for n in h_in if n != "state"]
    offs, nb = {}, 0
    for n in small:
        offs[n] = nb
        nb += -(-h_in[n].numel() * h_in[n].element_size() // 256) * 256

    def packed_view(buf, n):
        t = h_in[n]
        return buf[offs[n]:offs[n] + t.numel() * t.element_size()].view(t.dtype).view(t.shape)

    h_pack = torch.empty(nb, dtype=torch.uint8).pin_memory()
    h2d = nb + h_in["state"].numel() * h_in["state"].element_size()
    for n in small:
        packed_view(h_pack, n).copy_(h_in[n])
    for d in sets:
        d["pack"] = torch.empty(nb, dtype=torch.uint8, device=dev)
        for n in small:
            d[n] = packed_view(d["pack"], n)
    s_up, s_run, s_down = (torch.cuda.Stream(dev) for _ in range(3))
    launchers = [make_launcher(d, s_run.cuda_stream) for d in sets]
    up_done = [torch.cuda.Event() for _ in range(NE)]
    run_done = [torch.cuda.Event() for _ in range(NE)]
    down_done = [torch.cuda.Event() for _ in range(NE)]
    for e in down_done:
        e.record(s_down)

    def e2e_step(i):
        k = i % NE
        d = sets[k]
        s_up.wait_event(down_done[k])   # this set's previous step is fully drained
        with torch.cuda.stream(s_up):
            d["pack"].copy_(h_pack, non_blocking=True)
            d["state"].copy_(h_in["state"], non_blocking=True)
        up_done[k].record(s_up)
        s_run.wait_event(up_done[k])
        launchers[k]()
        run_done[k].record(s_run)
        s_down.wait_event(run_done[k])
        with torch.cuda.stream(s_down):
            h_y[k].copy_(d["y"], non_blocking=True)
            h_dl[k].copy_(d["dl"], non_blocking=True)
            h_st[k].copy_(d["s_rep"], non_blocking=True)
        down_done[k].record(s_down)

    for i in range(min(3, args.warmup)):
        e2e_step(i)
    torch.cuda.synchronize()
    if dist is not None:
        dist.barrier()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(s_up)
    s_run.wait_event(e0)
    s_down.wait_event(e0)
    for i in range(e2e_steps):
        e2e_step(i)
    s_down.wait_event(run_done[(e2e_steps - 1) % NE])
    e1.record(s_down)
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks(e0.elapsed_time(e1), dist, dev)
    e2e_value = world * tokens_per_step * e2e_steps / (e2e_ms / 1e3)

    # ---- the same loop with the recurrent state resident in HBM, as a
    # serving loop keeps it: every step copies only the step's own inputs (q,
    # k, v, g, beta, mask) host -> device and its output y device -> host.
    h2d_res = nb
    d2h_res = h_y[0].numel() * h_y[0].element_size()
    for d in sets:
        d["state"].copy_(d_in["state"])  # the resident snapshot, uploaded once (untimed)
    torch.cuda.synchronize()

    def e2e_step_resident(i):
        k = i % NE
        d = sets[k]
        s_up.wait_event(down_done[k])
        with torch.cuda.stream(s_up):
            d["pack"].copy_(h_pack, non_blocking=True)
        up_done[k].record(s_up)
        s_run.wait_event(up_done[k])
        launchers[k]()
        run_done[k].record(s_run)
        s_down.wait_event(run_done[k])
        with torch.cuda.stream(s_down):
            h_y[k].copy_(d["y"], non_blocking=True)
        down_done[k].record(s_down)

    for i in range(min(3, args.warmup)):
        e2e_step_resident(i)
    torch.cuda.synchronize()
    if dist is not None:
        dist.barrier()
    e0.record(s_up)
    s_run.wait_event(e0)
    s_down.wait_event(e0)
    for i in range(e2e_steps):
        e2e_step_resident(i)
    s_down.wait_event(run_done[(e2e_steps - 1) % NE])
    e1.record(s_down)
    torch.cuda.synchronize()
    e2e_res_ms = max_over_ranks(e0.elapsed_time(e1), dist, dev)
    e2e_res_value = world * tokens_per_step * e2e_steps / (e2e_res_ms / 1e3)

    if rank != 0:
        if dist is not None:
            dist.destroy_process_group()
        return None

    dominant = "record" if rec_ms >= rep_ms else "replay"
    dom_ms = rec_ms if dominant == "record" else rep_ms
    dom_b = rec_b if dominant == "record" else rep_b
    achieved = dom_b / (dom_ms * 1e-3) / 1e9
    traffic = measured_traffic(dominant, args.config)
    # ---- context for the fractions: a plain device-to-device copy moving as
    # many bytes as the dominant kernel (half read, half written), L2-cold
    # through rotating buffer pairs -- what one pass over that much data
    # reaches here (the measured peak is taken at GB sizes; a short pass
    # cannot hide its ramp).
    copy_each = max(1, round(dom_b / 2 / 2**20)) * 2**20  # whole MiB of float32
    pairs = 1 if 2 * copy_each >= 2 * L2_BYTES else -(-2 * L2_BYTES // (2 * copy_each)) + 1
    c_src = [torch.ones(copy_each // 4, dtype=torch.float32, device=dev) for _ in range(pairs)]
    c_dst = [torch.empty(copy_each // 4, dtype=torch.float32, device=dev) for _ in range(pairs)]
    c_reps = int(min(2000, max(20, 5e-3 * peak * 1e9 / (2 * copy_each))))
    for i in range(2 * pairs):
        c_dst[i % pairs].copy_(c_src[i % pairs])
    c0, c1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    c0.record()
    for i in range(c_reps):
        c_dst[i % pairs].copy_(c_src[i % pairs])
    c1.record()
    torch.cuda.synchronize()
    copy_gbs = 2 * copy_each * c_reps / (c0.elapsed_time(c1) * 1e-3) / 1e9
    del c_src, c_dst
    out = {
        "metric": METRIC,
        "value": value,
        "unit": "tokens/s",
        "n_gpus": world,
        "steps": K,
        "warmup": args.warmup,
        "ms_per_step": ms_per_step,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f32",
        "data": "synthetic",
        "config": {
            "workload": args.config, "B": B, "T": T, "Hk": Hk, "Hv": Hv, "Dk": Dk, "Dv": Dv,
            "io_dtype": dt, "state_dtype": "f32", "accepted": acc,
            "mask": workloads.CONFIGS[args.config]["mask"],
            "tape_capture": "delta_log+k_log+g_log",
            "record_path": ("gdn_chunk_prefill (chunk-local + scan kernels)" if record_path == "chunk"
                            else "gdn_step_record"),
            "replay_path": ("gdn_chunk_replay (tcgen05 contraction)" if replay_path == "chunk"
                            else "gdn_state_replay"),
            "gqa": ("tiled, read in place" if fused_gqa else
                    "tiled repeat materialised" if uses_repeat else "block"),
            "l2": (f"one buffer set of {set_bytes >> 20} MiB (at least twice the {L2_BYTES >> 20} MiB L2)"
                   if n_sets == 1 else
                   f"{n_sets} rotating buffer sets of {set_bytes >> 20} MiB (a set is reused after "
                   f"{(n_sets - 1) * set_bytes >> 20} MiB of other traffic, at least twice the "
                   f"{L2_BYTES >> 20} MiB L2)") + "; replay reads its own copy of the snapshot",
            "parallelism": f"{world} independent batch shard(s), no collective",
            "kernel_timing": ("kernels.*.us: a second pass over the same K steps with CUDA events "
                              "before and after each kernel; value and ms_per_step come from the "
                              "first pass, with no event between kernels"),
        },
        "hbm_gbs_step": step_gbs,
        "hbm_frac_step": step_gbs / peak,
        "roofline": {"bound": "hbm", "kernel": dominant, "achieved": achieved, "peak": peak,
                     "unit": "GB/s", "frac": achieved / peak, "traffic": traffic,
                     "algorithmic_bytes": dom_b, "bytes_counted": "active (unmasked) rows",
                     "peak_source": peak_src,
                     "same_size_copy": {"bytes_each_way": copy_each, "gbs": copy_gbs,
                                        "frac_of_peak": copy_gbs / peak,
                                        "kernel_frac_of_copy": achieved / copy_gbs}},
        "kernels": {
            "record": {"us": rec_ms * 1e3, "algorithmic_bytes": rec_b, "gbs": rec_gbs,
                       "frac": rec_gbs / peak, "frac_of_same_size_copy": rec_gbs / copy_gbs,
                       "algorithmic_bytes_all_positions": rec_all,
                       "frac_all_positions": rec_all / (rec_ms * 1e-3) / 1e9 / peak},
            "replay": {"us": rep_ms * 1e3, "algorithmic_bytes": rep_b, "gbs": rep_gbs,
                       "frac": rep_gbs / peak, "frac_of_same_size_copy": rep_gbs / copy_gbs,
                       "algorithmic_bytes_all_positions": rep_all,
                       "frac_all_positions": rep_all / (rep_ms * 1e-3) / 1e9 / peak},
        },
        "e2e": {"value": e2e_value, "unit": "tokens/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "steps": e2e_steps,
                "mode": "pinned host buffers; every input including the f32 state uploaded (q, k, v, "
                        "g, beta and the mask as one packed buffer of 256-byte aligned tensors, the "
                        "state as a second copy) and y, delta_log and the replayed state downloaded "
                        "every step; uploads, kernels and downloads pipelined on three streams over "
                        "three device buffer sets"},
        "e2e_resident_state": {"value": e2e_res_value, "unit": "tokens/s",
                               "h2d_bytes_per_step": h2d_res, "d2h_bytes_per_step": d2h_res,
                               "steps": e2e_steps,
                               "mode": "recurrent state kept in HBM between steps; q, k, v, g, beta, "
                                       "mask uploaded as one packed buffer and y downloaded every "
                                       "step (pinned, pipelined as above)"},
        "gpu_launches": launches_per_step * K,
        "clocks": clocks.summary(),
    }
    if world == 1 and not args.no_cpu_baseline:
        out["cpu_baseline"] = cpu_baseline(case, args.cpu_seconds)
    if dist is not None:
        dist.destroy_process_group()
    return out


# ---------------------------------------------------------------- oracle legs
def _oracle_inputs(orc, case, bs: int):
    """Float64 inputs of the first ``bs`` sequences (q / k expanded when the
    workload uses the tiled repeat; that expansion is part of the timed work)."""
    sl = slice(0, bs)
    return dict(q=case.f64("q")[sl].copy(), k=case.f64("k")[sl].copy(),
                v=case.f64("v")[sl].copy(), g=case.f64("g")[sl].copy(),
                beta=case.f64("beta")[sl].copy(), state=case.f64("state")[sl].copy(),
                mask=None if case.mask is None else case.mask[sl].copy())


def _oracle_step(orc, case, inp):
    """One oracle record + replay on prepared float64 inputs."""
    q, k = inp["q"], inp["k"]
    if workloads.uses_repeat(case.name):
        Bs = q.shape[0]
        q = orc.repeat_tiled(q.reshape(Bs * case.T, case.Hk, case.Dk), case.Hv).reshape(
            Bs, case.T, case.Hv, case.Dk)
        k = orc.repeat_tiled(k.reshape(Bs * case.T, case.Hk, case.Dk), case.Hv).reshape(
            Bs, case.T, case.Hv, case.Dk)
    rec = orc.record(q, k, inp["v"], inp["g"], inp["beta"], inp["state"], inp["mask"])
    orc.replay(rec["delta_log"], rec["k_log"], rec["g_log"], inp["state"], inp["mask"],
               accepted=case.accepted)


def cpu_baseline(case, seconds: float):
    """The float64 oracle, as it stands, on the host cores: whole-batch record
    + replay repeated for about ``seconds``; tokens/s."""
    import oracle
    oracle.build()
    threads = oracle.max_threads()
    inp = _oracle_inputs(oracle, case, case.B)
    t_start = time.perf_counter()
    reps = 0
    while True:
        _oracle_step(oracle, case, inp)
        reps += 1
        el = time.perf_counter() - t_start
        if el >= seconds or reps >= 1000:
            break
    value = reps * case.B * case.T / el
    sample = (f"{reps} x full batch (B={case.B}, T={case.T}) record+replay, {el:.1f} s, float64, "
              f"OpenMP over (b, hv)")
    # the same on one core, for about a third of the time
    oracle.set_threads(1)
    try:
        t_start = time.perf_counter()
        reps1 = 0
        while True:
            _oracle_step(oracle, case, inp)
            reps1 += 1
            el1 = time.perf_counter() - t_start
            if el1 >= seconds / 3 or reps1 >= 1000:
                break
    finally:
        oracle.set_threads(threads)
    return {"value": value, "unit": "tokens/s", "cores": threads, "kind": "oracle", "sample": sample,
            "host_cpus": os.cpu_count(),
            "single_thread": {"value": reps1 * case.B * case.T / el1, "unit": "tokens/s", "cores": 1,
                              "sample": f"{reps1} x full batch, {el1:.1f} s"}}


def run_reference(args, rank, world):
    if rank != 0:
        return None
    import oracle
    oracle.build()
    case = workloads.make_config(args.config, batch=args.batch)
    threads = oracle.max_threads()
    # size the per-step batch sample so the whole run stays within ~2 minutes
    one = _oracle_inputs(oracle, case, 1)
    t = time.perf_counter()
    _oracle_step(oracle, case, one)
    t1 = time.perf_counter() - t
    budget = 120.0 / max(1, args.steps + args.warmup)
    bs = int(max(1, min(case.B, budget / max(t1, 1e-6))))
    inp = _oracle_inputs(oracle, case, bs)
    for i in range(args.warmup):
        _oracle_step(oracle, case, inp)
    t = time.perf_counter()
    for i in range(args.steps):
        _oracle_step(oracle, case, inp)
    el = time.perf_counter() - t
    value = args.steps * bs * case.T / el
    out = {
        "impl": "reference",
        "metric": METRIC,
        "value": value,
        "unit": "tokens/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": el / args.steps * 1e3,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f64",
        "data": "synthetic",
        "config": {"workload": args.config, "B": case.B, "T": case.T, "Hk": case.Hk,
                   "Hv": case.Hv, "Dk": case.Dk, "Dv": case.Dv, "io_dtype": case.dtype,
                   "accepted": case.accepted, "batch_sample_per_step": bs},
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": threads, "kind": "oracle",
                         "sample": f"{bs} of {case.B} sequences per step, record+replay, "
                                   "float64 oracle, OpenMP over (b, hv)"},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    return out


def parse_args(argv=None):
    p = argparse.ArgumentParser(description=__doc__.split("\n\n")[0])
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=2000)
    p.add_argument("--warmup", type=int, default=20)
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--config", choices=sorted(workloads.CONFIGS), default=DEFAULT_CONFIG)
    p.add_argument("--e2e-steps", type=int, default=50)
    p.add_argument("--cpu-seconds", type=float, default=10.0)
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--record", choices=("auto", "step", "chunk"), default="auto",
                   help="record entry point: step form, chunked prefill, or by T (auto)")
    p.add_argument("--replay", choices=("auto", "step", "chunk"), default="auto",
                   help="replay entry point: step form, tensor-core contraction, or by accepted (auto)")
    p.add_argument("--gqa", choices=("fused", "repeat"), default="fused",
                   help="workloads with the tiled GQA expansion: read in place, or materialise")
    p.add_argument("--batch", type=int, default=None,
                   help="override B (smaller cases for profiler captures; not a bench line)")
    args = p.parse_args(argv)
    if args.warmup < 3:
        p.error("--warmup must be >= 3")
    if args.steps < 1:
        p.error("--steps must be >= 1")
    return args


def main(argv=None):
    args = parse_args(argv)
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if world != args.gpus and "WORLD_SIZE" in os.environ:
        print(f"warning: --gpus {args.gpus} but WORLD_SIZE={world}; using WORLD_SIZE",
              file=sys.stderr)
    if args.impl == "reference":
        out = run_reference(args, rank, world)
    else:
        out = run_ours(args, rank, world, local_rank)
    if out is not None:
        print(json.dumps(out))


if __name__ == "__main__":
    main()
