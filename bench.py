"""Benchmark: GatedDeltaNet verify + commit, verified rows/s and HBM GB/s.

One step = one pass of the whole verify + commit path over a 36-layer stack
of Qwen3.5-shaped GDN layers (B = 16 requests, k = 3 drafts -> 4 rows each,
H_qk = 16, H_v = 32, d_k = d_v = 128, bf16 inputs, fp32 state), one layer
call after another on one stream.  Every step moves ~2.5 GB, far more than
the 126 MB L2, so no flush is needed between steps.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--mode fused|replay|snapshot]
    python bench.py --impl reference ...   # the fp64 CPU oracle on host cores

Prints one JSON line (rank 0).  Under torchrun every rank runs its own
replica of the stack (weak scaling, no collective on the data path); the
time is the max over ranks.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from speculative_decode_gateddeltanet_gb300.inputs import (CONFIGS, RAGGED, SINGLE, STACK, SWEEP,  # noqa: E402
                                                           deferred_bytes, make_layer, make_step, spec_bytes,
                                                           workload_layers)

METRIC = "GDN verify+commit verified rows/sec and achieved HBM GB/s (% of peak), 1 GB300"
UNIT = "rows/s"
KERNEL_SRC = os.path.join(ROOT, "speculative_decode_gateddeltanet_gb300", "csrc", "gdn_spec.cu")
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "traffic.txt")
PEAKS_FILE = os.path.join(ROOT, "MEASURED_PEAKS.json")
FALLBACK_HBM_GBS = 6800.0


def kernel_source_hash() -> str:
    with open(KERNEL_SRC, "rb") as f:
        return hashlib.sha256(f.read()).hexdigest()[:16]


def measured_traffic(workload: str, mode: str):
    """(dram bytes read, dram bytes written) in one launch of the dominant
    kernel, from the committed ncu summary, if it was taken on the current
    kernel source; else None."""
    if not os.path.exists(TRAFFIC_FILE):
        return None
    h = kernel_source_hash()
    for line in open(TRAFFIC_FILE):
        parts = line.split()
        if len(parts) == 5 and not line.startswith("#") and parts[:3] == [workload, mode, h]:
            return float(parts[3]), float(parts[4])
    return None


def hbm_peak():
    try:
        with open(PEAKS_FILE) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, "fallback"


# ------------------------------------------------------------ distributed
def dist_setup():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    if ws <= 1:
        return 0, 1, 0
    import torch.distributed as dist

    rank, local = int(os.environ["RANK"]), int(os.environ.get("LOCAL_RANK", "0"))
    backend = "nccl" if torch.cuda.is_available() else "gloo"
    if torch.cuda.is_available():
        torch.cuda.set_device(local)
    dist.init_process_group(backend=backend)
    return rank, ws, local


def barrier(ws):
    if ws > 1:
        import torch.distributed as dist

        dist.barrier()


def max_over_ranks(value: float, ws: int) -> float:
    if ws <= 1:
        return value
    import torch.distributed as dist

    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([value], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ----------------------------------------------------------------- clocks
class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons during the timed region."""

    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device: int):
        self.proc = None
        self.path = None
        try:
            uuid = str(torch.cuda.get_device_properties(device).uuid)
            sel = uuid if uuid.startswith("GPU-") else f"GPU-{uuid}"
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", sel, f"--query-gpu={self.Q}", "--format=csv,noheader,nounits",
                 "-lms", "200"], stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        rows = []
        for line in open(self.path):
            f = [x.strip() for x in line.split(",")]
            if len(f) >= 9:
                rows.append(f)
        os.unlink(self.path)
        if not rows:
            return None
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({n for r in rows for n, v in zip(names, r[5:9]) if v.lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(rows)}


# ------------------------------------------------------------ CUDA arm
def layer_footprint(spec) -> int:
    """Bytes of distinct device data one layer call touches: its requests'
    state slices and conv windows (read and written in place), x, g, beta, o,
    the taps and the work buffer."""
    e = spec.elem_bytes
    state = spec.B * spec.H_v * spec.d_v * spec.d_k * 4
    conv = spec.B * spec.C * (spec.W - 1) * e + spec.C * spec.W * e
    rows = spec.B * spec.R * (spec.C * e + spec.H_v * 8 + spec.H_v * spec.d_v * 4)
    work = 4 * spec.B * spec.R * (2 * spec.H_qk * spec.d_k + spec.H_v * spec.d_v + 4 * spec.H_v)
    return state + conv + rows + work


def l2_bytes(device) -> int:
    props = torch.cuda.get_device_properties(device)
    return int(getattr(props, "L2_cache_size", 0) or 129 * 2**20)


def workload_specs(layers: int, batch: int | None = None, workload: str = "stack"):
    """(LayerSpec, seed) of each layer call of one step of the workload."""
    from dataclasses import replace

    if workload == "ragged":  # B=256 requests of 2, 4 or 9 rows, 64 value heads, 10 % inactive
        base = CONFIGS[RAGGED]
        specs = [(replace(base, name=f"ragged-{layers}L-B256-k1_3_8"), 4000 + i) for i in range(layers)]
    elif workload == "single":  # the single-layer B=1, k=3 call, as distinct layers so L2 cannot hold them
        base = CONFIGS[SINGLE]
        specs = [(replace(base, name=f"qwen35-{layers}L-B1-k3"), 1000 + i) for i in range(layers)]
    elif workload == "sweep":  # the batch sweep's k=2 calls (2B-slot pools), at --batch B, as distinct layers
        b = 16 if batch is None else batch
        base = replace(CONFIGS[SWEEP], B=b)
        specs = [(replace(base, name=f"qwen35-{layers}L-B{b}-k2"), 2000 + 100 * b + i) for i in range(layers)]
        batch = None
    else:
        specs = workload_layers(STACK, layers=layers)
    out = []
    for spec, seed in specs:
        if batch is not None and batch != spec.B:
            spec = replace(spec, B=batch, name=f"qwen35-{layers}L-B{batch}-k{spec.k}")
        out.append((spec, seed))
    return out


def build_stack(layers: int, device: str, batch: int | None = None, workload: str = "stack"):
    from speculative_decode_gateddeltanet_gb300 import gdn

    host, devs = [], []
    for spec, seed in workload_specs(layers, batch, workload):
        layer = make_layer(spec, seed)
        host.append(layer)
        devs.append(gdn.DeviceLayer(layer, device, snapshot=False))
    return host, devs


def run_cuda(args, rank, ws, local):
    from speculative_decode_gateddeltanet_gb300 import build as pkg_build

    pkg_build.build()
    from speculative_decode_gateddeltanet_gb300 import gdn

    device = f"cuda:{local}"
    torch.cuda.set_device(local)
    if args.layers is None:
        # The workload's default layer count, raised until the distinct data one step touches is at
        # least twice the L2: the timed steps then cannot find earlier steps' data in L2.
        default = 4 if args.workload == "ragged" else 36
        probe = workload_specs(1, args.batch, args.workload)[0][0]
        need = -(-2 * l2_bytes(device) // layer_footprint(probe))
        args.layers = max(default, need)
    host, devs = build_stack(args.layers, device, args.batch, args.workload)
    spec = host[0]["spec"]
    if args.mode == "snapshot":
        for d in devs:
            d.scratch_S = torch.empty((spec.B, spec.R, spec.H_v, spec.d_v, spec.d_k), device=device)
            d.scratch_cs = torch.empty((spec.B, spec.R, spec.C, spec.W - 1), dtype=d.x.dtype, device=device)
    stream = torch.cuda.Stream(device)
    sp = stream.cuda_stream
    # deferred: each layer's pending rows are a previous decode step of the same shape, already on the
    # device; the call commits their accepted prefix and verifies the current rows
    pending, prevs = [], []
    if args.mode == "deferred":
        for h in host:
            ps = make_step(h, h["spec"], h["seed"] + 7919)
            pending.append({k: ps[k].to(device).contiguous() for k in ("x", "g", "beta", "n_rows", "accept_len")})
    # A step's per-call inputs (x, g, beta, slot ids, row and accept counts) live in one device arena
    # that one copy from a pinned host arena refills, and every layer's o in one buffer that one copy
    # reads back: the end-to-end leg moves each step's host data in two transfers.
    step_keys = ("x", "g", "beta", "slot_ids", "n_rows") + (("accept_len",) if args.mode != "deferred" else ())
    parts = []
    for i, (h, d) in enumerate(zip(host, devs)):
        for k in step_keys:
            parts.append((d, k, getattr(d, k)))
        if args.mode == "deferred":
            parts.append((pending[i], "accept_len", pending[i]["accept_len"]))
    offs, total = [], 0
    for _, _, t in parts:
        offs.append(total)
        total += (t.numel() * t.element_size() + 255) // 256 * 256
    dev_arena = torch.zeros(total, dtype=torch.uint8, device=device)
    host_arena = torch.zeros(total, dtype=torch.uint8).pin_memory()
    for (owner, k, t), off in zip(parts, offs):
        nb = t.numel() * t.element_size()
        view = dev_arena[off:off + nb].view(t.dtype).view(t.shape)
        view.copy_(t)
        host_arena[off:off + nb].view(t.dtype).view(t.shape).copy_(t.cpu())
        if isinstance(owner, dict):
            owner[k] = view
        else:
            setattr(owner, k, view)
    o_all = torch.full((len(devs),) + tuple(devs[0].o.shape), float("nan"), device=device)
    for i, d in enumerate(devs):
        d.o = o_all[i]
    host_o = torch.empty(o_all.shape, dtype=o_all.dtype).pin_memory()
    cargs = [d.args() for d in devs]
    if args.stable:
        # every layer has slots of its own and nothing else on the stream writes them, slot_ids or
        # n_rows, so each call may fetch its state while the call before it drains
        for a in cargs:
            a.flags |= gdn.FLAG_STATE_STABLE
    if args.mode == "deferred":
        # one untimed deferred call per layer with nothing pending writes the pending step's carry;
        # every timed call then commits that step's accepted rows from it and writes its own carry
        for d, a, t in zip(devs, cargs, pending):
            t["carry_in"] = torch.empty(gdn.carry_bytes(a) // 4, device=device)
            t["carry_out"] = torch.empty_like(t["carry_in"])
            first = gdn.make_args(x=t["x"], g=t["g"], beta=t["beta"], conv_w=d.conv_w, conv_state=d.conv_state,
                                  ssm_state=d.ssm_state, slot_ids=d.slot_ids, n_rows=t["n_rows"], o=d.o,
                                  work=d.work, status=d.status, H_qk=spec.H_qk, carry=t["carry_in"])
            gdn.gdn_verify_deferred(first, None, sp)
            a.carry = t["carry_out"].data_ptr()
            a.accept_len = None
            prevs.append(gdn.make_prev(x=t["x"], n_rows=t["n_rows"], accept_len=t["accept_len"],
                                       carry=t["carry_in"]))
        torch.cuda.synchronize()

    def call(a, i):
        if args.mode == "fused":
            gdn.gdn_verify_commit(a, sp)
        elif args.mode == "deferred":
            gdn.gdn_verify_deferred(a, prevs[i], sp)
        else:
            m = gdn.REPLAY if args.mode == "replay" else gdn.SNAPSHOT
            gdn.gdn_verify(a, m, sp)
            gdn.gdn_commit(a, m, sp)

    def step():
        if args.mode in ("fused", "deferred"):
            for i, a in enumerate(cargs):
                call(a, i)
        else:
            m = gdn.REPLAY if args.mode == "replay" else gdn.SNAPSHOT
            for a in cargs:
                gdn.gdn_verify(a, m, sp)
                gdn.gdn_commit(a, m, sp)

    calls_per_step = len(cargs) * (1 if args.mode in ("fused", "deferred") else 2)
    # kernels per layer: prologue + rows kernel per call; a snapshot commit is one kernel
    kernels_per_layer = {"fused": 2, "deferred": 2, "replay": 4, "snapshot": 3}[args.mode]
    # --graph: the step's launches captured once into a CUDA graph and replayed
    graph = None

    def run_step():
        if graph is not None:
            graph.replay()
        else:
            step()
    rows_per_step = sum(int(h["n_rows"].clamp(min=0).sum()) for h in host)
    if args.mode == "deferred":
        bytes_per_step = sum(deferred_bytes(h["spec"], h["n_rows"], t["n_rows"].cpu(), t["accept_len"].cpu())
                             for h, t in zip(host, pending))
    else:
        bytes_per_step = sum(spec_bytes(h["spec"], h["n_rows"]) for h in host)

    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            step()
    torch.cuda.synchronize()
    if args.graph:
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=stream):
            step()
        with torch.cuda.stream(stream):
            for _ in range(args.warmup):
                run_step()
        torch.cuda.synchronize()

    # ---- device-resident timed region ----
    sampler = ClockSampler(local) if rank == 0 else None
    if sampler:
        time.sleep(0.4)
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(ws)
    torch.cuda.synchronize()
    ev0.record(stream)
    with torch.cuda.stream(stream):
        for _ in range(args.steps):
            run_step()
    ev1.record(stream)
    torch.cuda.synchronize()
    barrier(ws)
    clocks = sampler.stop() if sampler else None
    ms = max_over_ranks(ev0.elapsed_time(ev1), ws)
    ms_step = ms / args.steps
    value = rows_per_step * ws / (ms_step / 1e3)
    for d in devs:
        assert int(d.status.item()) == 0, "device status bits set"

    # ---- end to end: pinned host inputs -> device -> call -> o back to host ----
    h2d = host_arena.numel()
    d2h = host_o.numel() * host_o.element_size()

    def e2e_step():
        dev_arena.copy_(host_arena, non_blocking=True)
        run_step()
        host_o.copy_(o_all, non_blocking=True)

    e2e_steps = max(3, min(args.steps, 200))
    with torch.cuda.stream(stream):
        for _ in range(3):
            e2e_step()
    torch.cuda.synchronize()
    barrier(ws)
    ev0.record(stream)
    with torch.cuda.stream(stream):
        for _ in range(e2e_steps):
            e2e_step()
    ev1.record(stream)
    torch.cuda.synchronize()
    barrier(ws)
    e2e_ms = max_over_ranks(ev0.elapsed_time(ev1), ws) / e2e_steps

    peak, peak_kind = hbm_peak()
    traffic = measured_traffic(spec.name, args.mode)
    per_launch_bytes = bytes_per_step / len(cargs)
    launch_s = ms_step / 1e3 / calls_per_step
    achieved = (per_launch_bytes / launch_s / 1e9 if args.mode in ("fused", "deferred")
                else bytes_per_step / (ms_step / 1e3) / 1e9)
    out = {
        "metric": METRIC, "value": round(value, 1), "unit": UNIT, "n_gpus": ws, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms_step, 5), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": {"workload": spec.name, "layers": len(cargs), "B": spec.B, "k": spec.k, "rows_per_layer":
                   rows_per_step // len(cargs), "H_qk": spec.H_qk, "H_v": spec.H_v, "d_k": spec.d_k,
                   "d_v": spec.d_v, "storage": "bf16 x/conv, fp32 g/beta/state/o", "mode": args.mode,
                   "launch": "cuda graph replay" if args.graph else "stream launches",
                   "state_stable": bool(args.stable),
                   "l2": "inputs larger than L2: each step touches %.0f MB of distinct data (%d layers; "
                         "L2 %.0f MB) and streams %.2f GB"
                         % (sum(layer_footprint(h["spec"]) for h in host) / 1e6, len(cargs),
                            l2_bytes(device) / 1e6, bytes_per_step / 1e9)},
        "hbm_gbs": round(bytes_per_step * ws / (ms_step / 1e3) / 1e9, 1),
        "bytes_per_row": round(bytes_per_step / rows_per_step),
        "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                     "frac": round(achieved / peak, 4), "peak_kind": peak_kind,
                     "kernel": "rows_kernel<128, %s>" % args.mode,
                     "traffic": None if traffic is None else traffic[0] + traffic[1],
                     "traffic_read": None if traffic is None else traffic[0],
                     "traffic_write": None if traffic is None else traffic[1],
                     "traffic_note": "ncu dram__bytes_read.sum + dram__bytes_write.sum of one rows-kernel launch, "
                                     "inside its own window: the committed state it writes (2 MiB per request) "
                                     "stays dirty in L2 and reaches DRAM while later kernels run, so the window "
                                     "shows its reads (state, staged rows) and almost none of its writes",
                     "algorithmic_bytes_per_launch": round(per_launch_bytes)},
        "e2e": {"value": round(rows_per_step * ws / (e2e_ms / 1e3), 1), "unit": UNIT,
                "ms_per_step": round(e2e_ms, 5), "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h},
        "gpu_launches": kernels_per_layer * len(cargs) * args.steps,
        "clocks": clocks,
    }
    if rank == 0 and ws == 1 and not args.no_cpu_baseline:
        out["cpu_baseline"] = cpu_baseline(host, budget_s=args.cpu_seconds)
    return out


# ------------------------------------------------------------ greedy acceptance
def run_accept(args, rank, ws, local):
    """Device-side greedy acceptance on the verify shape: B=16 requests of
    4 rows over the 151936-token vocabulary in bf16, L distinct calls per
    step (a step's logits at least twice the L2)."""
    from speculative_decode_gateddeltanet_gb300 import build as pkg_build
    from speculative_decode_gateddeltanet_gb300.inputs import make_accept_case

    pkg_build.build()
    from speculative_decode_gateddeltanet_gb300 import gdn

    device = f"cuda:{local}"
    torch.cuda.set_device(local)
    B, R, V = 16, 4, 151936
    # enough distinct calls (at least 12) that the logits a step reads (its valid rows') are at
    # least twice the L2
    need = 2 * l2_bytes(device)
    calls, read = [], 0
    i = 0
    while len(calls) < 12 or read < need:
        c = make_accept_case(B, R, V, seed=9000 + i)
        calls.append({k: c[k].to(device) for k in ("logits", "drafts", "n_rows")}
                     | {"target": torch.empty((B, R), dtype=torch.int32, device=device),
                        "acc": torch.empty(B, dtype=torch.int32, device=device)})
        read += int(c["n_rows"].sum()) * V * 2
        i += 1
    L = len(calls)
    rows = sum(int(c["n_rows"].sum()) for c in calls)
    nbytes = sum(int(c["n_rows"].sum()) * V * 2 for c in calls)  # the valid rows' logits, read once
    stream = torch.cuda.Stream(device)

    def step():
        for c in calls:
            gdn.greedy_accept(c["logits"], c["drafts"], c["n_rows"], c["target"], c["acc"], stream=stream)

    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            step()
    torch.cuda.synchronize()
    sampler = ClockSampler(local) if rank == 0 else None
    if sampler:
        time.sleep(0.4)
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(ws)
    ev0.record(stream)
    with torch.cuda.stream(stream):
        for _ in range(args.steps):
            step()
    ev1.record(stream)
    torch.cuda.synchronize()
    barrier(ws)
    clocks = sampler.stop() if sampler else None
    ms_step = max_over_ranks(ev0.elapsed_time(ev1), ws) / args.steps
    peak, peak_kind = hbm_peak()
    gbs = nbytes / (ms_step / 1e3) / 1e9
    return {"metric": "greedy acceptance: verify rows/s (argmax over the vocabulary + accepted prefix)",
            "value": round(rows * ws / (ms_step / 1e3), 1), "unit": "rows/s", "n_gpus": ws,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_step, 5),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic",
            "config": {"workload": f"accept-B{B}-R{R}-V{V}", "calls_per_step": L,
                       "l2": "inputs larger than L2: %.0f MB of logits per step" % (nbytes / 1e6)},
            "roofline": {"bound": "hbm", "achieved": round(gbs, 1), "peak": peak, "unit": "GB/s",
                         "frac": round(gbs / peak, 4), "peak_kind": peak_kind,
                         "kernel": "argmax_kernel<bf16> + accept_kernel", "traffic": None},
            "gpu_launches": 2 * L * args.steps, "clocks": clocks}


# ------------------------------------------------------------ oracle arm
def oracle_rows_per_second(layers: list, budget_s: float):
    """Time the oracle on one thread over whole layer calls of the workload
    (cycling over its layers) until the budget is used."""
    import oracle

    rows, secs, calls = 0, 0.0, 0
    while secs < budget_s:
        layer = layers[calls % len(layers)]
        r = oracle.verify_commit(layer)
        rows += int(layer["n_rows"].clamp(min=0).sum())
        secs += r["seconds"]
        calls += 1
    return rows, secs, calls


def oracle_rows_per_second_threads(layers: list, budget_s: float, threads: int):
    """The oracle over all host cores: each layer call's requests spread over
    ``threads`` threads (``oracle.verify_commit_threads``), cycling over the
    given layers until the wall-time budget is used."""
    import oracle

    rows, secs, calls, used = 0, 0.0, 0, 1
    while secs < budget_s:
        layer = layers[calls % len(layers)]
        r = oracle.verify_commit_threads(layer, threads)
        rows += int(layer["n_rows"].clamp(min=0).sum())
        secs += r["seconds"]
        used = r["threads"]
        calls += 1
    return rows, secs, calls, used


def host_threads() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except (AttributeError, OSError):
        return os.cpu_count() or 1


def cpu_baseline(layers: list, budget_s: float = 12.0):
    """The oracle on the host, on the bench's own host-side layers (the same
    seeded inputs the GPU ran): all cores (the reported value) and one core,
    half the budget each, cycling over at most four layers."""
    layers = layers[:4]
    spec = layers[0]["spec"]
    rows1, secs1, calls1 = oracle_rows_per_second(layers, budget_s / 2)
    rows, secs, calls, used = oracle_rows_per_second_threads(layers, budget_s / 2, host_threads())
    return {"value": round(rows / secs, 1), "unit": UNIT, "cores": used, "kind": "oracle",
            "sample": f"fp64 C oracle, fused verify+commit, each layer call's {spec.B} requests spread over {used} "
                      f"host threads: {calls} calls ({rows} rows) cycling over {len(layers)} layers of "
                      f"{spec.name}, {secs:.1f} s wall",
            "one_core": {"value": round(rows1 / secs1, 1), "unit": UNIT, "cores": 1,
                         "sample": f"single thread, {calls1} whole layer calls ({rows1} rows) of the same layers, "
                                   f"{secs1:.1f} s"}}


def run_reference(args, rank, ws):
    """The oracle as it stands, on the host cores, on the same workload: each
    step is one layer call of the stack (its 16 requests over the host's
    threads), capped so the whole run stays within a few minutes."""
    import oracle

    if rank != 0:
        return None
    spec, seed = workload_layers(STACK, layers=1)[0]
    layer = make_layer(spec, seed)
    threads = host_threads()
    r = oracle.verify_commit_threads(layer, threads)
    t_call = max(r["seconds"], 1e-4)
    budget = 150.0
    steps = args.steps
    if (args.steps + args.warmup) * t_call > budget:  # bounded sample: fewer requests per step
        per_step = max(1, min(spec.B, int(spec.B * budget / ((args.steps + args.warmup) * t_call))))
    else:
        per_step = spec.B
    sub = dict(layer)
    sub["n_rows"] = layer["n_rows"].clone()
    sub["n_rows"][per_step:] = 0
    rows_step = int(sub["n_rows"].clamp(min=0).sum())
    for _ in range(args.warmup):
        oracle.verify_commit_threads(sub, threads)
    t, used = 0.0, 1
    for _ in range(steps):
        r = oracle.verify_commit_threads(sub, threads)
        t += r["seconds"]
        used = r["threads"]
    ms_step = t / steps * 1e3
    value = rows_step / (ms_step / 1e3)
    sample = (f"fp64 C oracle, fused verify+commit: {per_step} of the {spec.B} requests of one layer of the "
              f"36-layer B=16 k=3 stack per step ({rows_step} rows), spread over {used} host threads")
    return {"metric": METRIC, "value": round(value, 1), "unit": UNIT, "n_gpus": ws, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": round(ms_step, 4), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "impl": "reference",
            "config": {"workload": spec.name, "layers": 36, "B": spec.B, "k": spec.k, "mode": "fused"},
            "cpu_baseline": {"value": round(value, 1), "unit": UNIT, "cores": used, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": round(value, 1), "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--mode", choices=["fused", "replay", "snapshot", "deferred"], default="fused",
                    help="deferred: each call commits the previous step's accepted rows from that step's "
                         "carry and verifies the current ones (gdn_verify_deferred)")
    ap.add_argument("--layers", type=int, default=None,
                    help="layer calls per step (default 36 for the stack, 4 for the ragged batch)")
    ap.add_argument("--workload", choices=["stack", "ragged", "single", "sweep"], default="stack",
                    help="stack: 36 Qwen3.5-shaped layers at B=16, k=3; ragged: B=256 requests with k in "
                         "{1,3,8} and 64 value heads (about 1 GB of state per layer); single: the B=1, k=3 "
                         "call as 36 distinct layers; sweep: the batch sweep's k=2 call at --batch B (2B-slot "
                         "pools), as 36 distinct layers")
    ap.add_argument("--batch", type=int, default=None, help="requests per layer (default: the workload's 16)")
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--accept", action="store_true",
                    help="time the device-side greedy acceptance instead of the verify + commit step")
    ap.add_argument("--stable", action="store_true",
                    help="set GDN_FLAG_STATE_STABLE on every call: each call fetches its state while the call "
                         "before it drains")
    ap.add_argument("--no-graph", dest="graph", action="store_false",
                    help="launch each step's kernels on the stream instead of replaying the step captured "
                         "as a CUDA graph")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    rank, ws, local = dist_setup()
    if args.impl == "reference":
        out = run_reference(args, rank, ws)
    elif args.accept:
        out = run_accept(args, rank, ws, local)
    else:
        out = run_cuda(args, rank, ws, local)
    if rank == 0 and out is not None:
        print(json.dumps(out), flush=True)
    if ws > 1:
        import torch.distributed as dist

        dist.destroy_process_group()


if __name__ == "__main__":
    main()
