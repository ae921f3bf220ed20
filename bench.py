"""Benchmark of the selective-scan hot path on B300: state updates/s and achieved HBM GB/s.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl reference]

One step = one pass of the whole hot path over one batch of synthetic input: for a prefill
workload one call of ssm_selective_scan_fwd (conv prologue + Delta + discretisation +
recurrence + readout + gate, plus the chunk-carry kernel when the scan is chunked); for the
decode workload its 64 consecutive ssm_selective_state_update calls. Inputs are resident in
HBM; L2 is flushed (a 256 MiB write) before every timed step, outside the step's events.
Each step is timed with CUDA events on the launching stream.

Prints ONE JSON line (rank 0). Under torchrun every rank runs its own copy of the workload
(weak scaling, no collective on the data path); the step time is the max over ranks.
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
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

DEFAULT_WORKLOAD = "longscan_bf16_b1_d1536_l131072_n16"
METRIC = "selective-scan state updates/s (B*L*D*N) and HBM GB/s vs B300 peak"
UNIT = "updates/s"
FALLBACK_HBM_GBS = 6400.0
SPEC_HBM_GBS = 8000.0  # the part's nominal HBM3e bandwidth, reported beside the measured copy peak


def _peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            p = json.load(f)
        return float(p.get("hbm_gbs", FALLBACK_HBM_GBS)), "measured"
    return FALLBACK_HBM_GBS, "fallback"


def _sm_max_mhz() -> float:
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            return float(json.load(f).get("sm_max_mhz", 2032.0))
    return 2032.0


# Pipe model of one state update on this part (measured by a throughput probe on the B300:
# ex2.approx.f32 issues at 4 cycles per warp instruction per SMSP, i.e. 32 results per clock per
# SM; packed fma.rn.f32x2 at 2 cycles per warp instruction, overlapping fully with ex2; lg2,
# tanh and rcp at half the ex2 rate). Every update of the main pass and of the carry pass needs
# one exp2, so the special-function pipe alone allows 32 updates per clock per SM: that is the
# floor the scan kernels are held against. The four FMA-pipe operations of a main-pass update
# (Delta*A, Delta*u*B, the recurrence, the readout) cost the same four cycles per 32 updates on
# the FMA pipe, so a perfect kernel would keep both pipes full; the per-token element-wise work
# (conv, SiLU, softplus, gate) comes on top.
UPDATES_PER_CLK_PER_SM = 32


def _as_graph(fn, dev):
    """Capture fn (library calls on the current stream) once into a CUDA graph; return a
    function that replays it on the current stream."""
    import torch

    side = torch.cuda.Stream(dev)
    side.wait_stream(torch.cuda.current_stream(dev))
    with torch.cuda.stream(side):
        fn()  # one eager call: kernel attributes are set outside the capture
    torch.cuda.synchronize(dev)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.stream(side):
        with torch.cuda.graph(graph, stream=side):
            fn()
    torch.cuda.synchronize(dev)
    return graph.replay


class _Packed:
    """Named tensors laid out back to back (256-byte aligned) in one flat byte buffer, so that a
    step's inputs (or results) cross PCIe in one copy; `views` holds the named tensors as views
    into the buffer (non-tensor entries pass through)."""

    def __init__(self, tensors, device=None, pin=False):
        import torch

        meta, off = [], 0
        for name, v in tensors.items():
            if isinstance(v, torch.Tensor):
                nb = v.numel() * v.element_size()
                meta.append((name, off, v.dtype, tuple(v.shape), nb))
                off += (nb + 255) // 256 * 256
        self.buf = torch.empty(max(off, 256), dtype=torch.uint8, device=device)
        if pin:
            self.buf = self.buf.pin_memory()
        self.views = {k: v for k, v in tensors.items() if not isinstance(v, torch.Tensor)}
        for name, o, dt, shape, nb in meta:
            self.views[name] = self.buf[o:o + nb].view(dt).view(shape)

    @property
    def nbytes(self) -> int:
        return self.buf.numel()


def alu_roofline(w, seconds: float, chunk_len: int, sms: int):
    """Scan step time against its special-function-pipe floor: main + carry updates, one exp2
    each, at 32 per clock per SM at the maximum SM clock. The per-token element-wise work (conv,
    SiLU, softplus, gate) is extra, so frac stays below 1 even for a perfect scan."""
    if w.kind != "scan":
        return None
    per_t = w.batch * w.dim * w.dstate
    nchunks = (w.seqlen + chunk_len - 1) // chunk_len if w.seqlen > 0 else 1
    u_main = per_t * w.seqlen
    u_carry = per_t * min(w.seqlen, (nchunks - 1) * chunk_len) if nchunks > 1 else 0
    rate = sms * UPDATES_PER_CLK_PER_SM * _sm_max_mhz() * 1e6
    floor_s = (u_main + u_carry) / rate
    return {"bound": "alu", "achieved": u_main / seconds / 1e9, "peak": u_main / floor_s / 1e9,
            "unit": "Gupdates/s", "frac": floor_s / seconds, "carry_updates": u_carry,
            "model": f"one ex2 per main or carry update at {UPDATES_PER_CLK_PER_SM} per clock per SM (measured); "
                     f"{sms} SMs at {_sm_max_mhz():.0f} MHz"}


def algorithmic_bytes(w) -> int:
    """Bytes every input read once / every output written once, per step (no per-step state)."""
    es = 2 if w.io == "bf16" else 4
    N, K = w.dstate, w.d_conv
    if w.kind == "decode":
        ch = w.batch * w.dim
        per = (ch * N * 4 * 2                      # state read + write
               + ch * (K - 1) * es * 2             # window read + write
               + ch * es * 4                       # x, delta, z in; y out
               + w.batch * N * es * 2              # B, C
               + w.dim * N * 4                     # A
               + w.dim * 4 * 3                     # D, delta_bias, conv bias
               + w.dim * K * 4)                    # conv weights
        return per * w.steps
    tokens = w.batch * w.dim * w.seqlen
    b = tokens * es * 4                            # x (or u), delta, z in; y out
    b += 2 * w.batch * N * w.seqlen * es           # B, C
    b += w.batch * w.dim * N * 4                   # h_last out
    b += w.dim * N * 4                             # A
    b += w.dim * 4 * 2                             # D, delta_bias
    if K:
        b += w.dim * 4 + w.dim * K * 4             # conv bias, conv weights
    return b


def bwd_algorithmic_bytes(w) -> int:
    """Bytes of one backward step, every input read once and every output written once: u,
    delta, z, dout in and du, ddelta, dz out (io dtype); B, C in (io) and dB, dC out (fp32);
    h0, dh_last in and dh0 out; A, D, bias in and dA, dD, dbias out (fp32)."""
    es = 2 if w.io == "bf16" else 4
    tok = w.batch * w.dim * w.seqlen
    bnl = w.batch * w.dstate * w.seqlen
    return (tok * es * 7 + bnl * (2 * es + 2 * 4) + w.batch * w.dim * w.dstate * 4 * 3
            + w.dim * w.dstate * 4 * 2 + w.dim * 4 * 4)


# The sources each kind of workload's kernels are built from: a traffic figure stays valid
# while their code is unchanged (comments and whitespace do not count, see source_code_only).
_KERNEL_SOURCES = {
    "scan": ("ssm_scan.cu", "ssm_api.cu", "ssm_device.cuh", "ssm_internal.h", "ssm_bounds.cuh"),
    "decode": ("ssm_decode.cu", "ssm_api.cu", "ssm_device.cuh", "ssm_internal.h", "ssm_bounds.cuh"),
    "backward": ("ssm_scan_bwd.cu", "ssm_api.cu", "ssm_device.cuh", "ssm_internal.h", "ssm_bounds.cuh"),
    "ssd": ("ssm_ssd.cu", "ssm_umma.cuh", "ssm_api.cu", "ssm_device.cuh", "ssm_internal.h"),
}


def source_code_only(text: str) -> str:
    """C / C++ / CUDA source without its comments, with every run of whitespace collapsed to one
    space: two sources that differ only in comments or layout compile to the same kernels and
    give the same string. String and character literals are kept as they are."""
    out, i, n = [], 0, len(text)
    while i < n:
        ch = text[i]
        if ch in "\"'":  # literal: copy through the closing quote, honouring escapes
            j = i + 1
            while j < n and text[j] != ch:
                j += 2 if text[j] == "\\" else 1
            out.append(text[i:j + 1])
            i = j + 1
        elif text.startswith("//", i):
            j = text.find("\n", i)
            i = n if j < 0 else j
            out.append(" ")
        elif text.startswith("/*", i):
            j = text.find("*/", i + 2)
            i = n if j < 0 else j + 2
            out.append(" ")
        else:
            out.append(ch)
            i += 1
    return " ".join("".join(out).split())


def kernel_source_hash(kind: str = "scan") -> str:
    h = hashlib.sha256()
    for name in _KERNEL_SOURCES[kind]:
        with open(os.path.join(ROOT, "selective_state_space_145_b300", "csrc", name), encoding="utf-8") as f:
            h.update(name.encode() + source_code_only(f.read()).encode())
    return h.hexdigest()[:16]


def traffic_from_profiles(workload: str, kind: str = "scan"):
    """DRAM bytes per step from a committed ncu summary, if its kernel-source hash is current."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        t = json.load(f)
    e = t.get(workload)
    if not e or e.get("kernel_source_hash") != kernel_source_hash(kind):
        return None
    return e.get("dram_bytes_per_step")


class ClockSampler:
    """nvidia-smi clock / throttle-reason sampling during the timed region."""

    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.Q}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, ValueError):
            self.proc = None
        return self

    def __exit__(self, *exc):
        self.lines = []
        if self.proc is not None:
            time.sleep(0.25)
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                out, _ = self.proc.communicate()
            self.lines = [ln for ln in out.splitlines() if ln.strip()]
        return False

    def summary(self):
        rows = []
        for ln in getattr(self, "lines", []):
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                rows.append((float(f[1]), float(f[2]), f[5], f[6], f[7], f[8]))
            except ValueError:
                continue
        if not rows:
            return None
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[2 + i].lower() == "active"})
        return {"sm_mhz": statistics.median(r[0] for r in rows), "sm_max_mhz": max(r[1] for r in rows),
                "reasons": reasons, "samples": len(rows)}


def _dist():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def reduce_max(value: float, world: int, device=None) -> float:
    if world <= 1:
        return value
    import torch
    import torch.distributed as dist

    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(world: int):
    if world > 1:
        import torch.distributed as dist

        dist.barrier()


# ---------------------------------------------------------------- CPU oracle (baseline / reference arm)

def oracle_sample_rate(w, target_s: float = 10.0, max_channels: int = 1024, reverse: bool = False,
                       zoh: bool = False):
    """Time the fp64 oracle, as it stands, on a bounded sample of the workload's channels.

    Returns (updates/s, cores, sample description)."""
    import numpy as np

    import oracle
    from selective_state_space_145_b300 import inputs

    cores = oracle.oracle.default_threads()
    if w.kind == "decode":
        q = inputs.decode_inputs(min(w.batch, 16), w.dim, w.dstate, w.d_conv, w.io, w.seed, steps=1)
        state, win = q["state"].double().numpy(), q["conv_state"].double().numpy()
        ups = 0
        t0 = time.perf_counter()
        reps = 0
        while time.perf_counter() - t0 < target_s:
            _, state, win = oracle.state_update(state, win, q["x"][0], q["delta"][0], q["A"], q["B"][0], q["C"][0],
                                                q["D"], q["z"][0], q["delta_bias"], True, q["conv_w"], q["conv_b"],
                                                nthreads=cores, zoh=zoh)
            ups += state.size
            reps += 1
        dt = time.perf_counter() - t0
        return ups / dt, cores, f"{reps} decode steps of {state.shape[0]} sequences x {w.dim} channels"
    # prefill: full-length rows of a subset of channels
    nch = max(1, min(max_channels, w.batch * w.dim))
    bsub = 1
    dsub = min(w.dim, nch)
    p = inputs.scan_inputs(bsub, dsub, w.seqlen, w.dstate, w.d_conv, w.io, w.seed, salient_frac=w.salient_frac)
    # size the sample so it takes about target_s
    L = w.seqlen
    probe_len = min(L, 256)
    t0 = time.perf_counter()
    oracle.selective_scan(p["x"][..., :probe_len], p["delta"][..., :probe_len], p["A"], p["B"][..., :probe_len],
                          p["C"][..., :probe_len], p["D"], p["z"][..., :probe_len], p["delta_bias"], True,
                          p["conv_w"], p["conv_b"], nthreads=cores, reverse=reverse, zoh=zoh)
    per_step = (time.perf_counter() - t0) / probe_len
    use_len = int(max(probe_len, min(L, target_s / max(per_step, 1e-9))))
    sub = {k: (v[..., :use_len] if k in ("x", "delta", "z", "B", "C") else v) for k, v in p.items()}
    reps = 0
    t0 = time.perf_counter()
    while True:
        oracle.selective_scan(sub["x"], sub["delta"], sub["A"], sub["B"], sub["C"], sub["D"], sub["z"],
                              sub["delta_bias"], True, sub["conv_w"], sub["conv_b"], nthreads=cores,
                              reverse=reverse, zoh=zoh)
        reps += 1
        if time.perf_counter() - t0 >= target_s or reps >= 10000:
            break
    dt = time.perf_counter() - t0
    ups = reps * dsub * use_len * w.dstate
    return ups / dt, cores, (f"{reps} pass(es) over {dsub} channels x {use_len} steps x N={w.dstate} "
                             f"of the workload's inputs (fp64, {cores} threads)")


def run_reference(args, w):
    world, rank, _ = _dist()
    if rank != 0:
        return 0
    rates = []
    desc, cores = "", 1
    budget = max(2.0, 120.0 / max(1, args.steps + args.warmup))
    for i in range(args.warmup + args.steps):
        r, cores, desc = oracle_sample_rate(w, target_s=budget, reverse=args.reverse, zoh=args.zoh)
        if i >= args.warmup:
            rates.append(r)
    value = statistics.mean(rates)
    line = {"metric": METRIC, "value": value, "unit": UNIT, "impl": "reference", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": w.updates / value * 1e3,
            "ms_per_step_basis": "one whole step of the workload at the oracle's sampled rate",
            "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": config_of(w, args.reverse, args.zoh, s4d_real=args.s4d_real),
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle", "sample": desc},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


def config_of(w, reverse: bool = False, zoh: bool = False, eager: bool = False, s4d_real: bool = False):
    c = {"workload": w.name, "kind": w.kind, "io": w.io, "batch": w.batch, "d_inner": w.dim, "seqlen": w.seqlen,
         "d_state": w.dstate, "d_conv": w.d_conv, "l2": "flushed before every timed step (256 MiB write)",
         "launch": "direct library calls" if eager else "the step's library calls replayed from one CUDA graph"}
    if reverse:
        c["direction"] = "backward (SSM_SCAN_REVERSE)"
    if zoh:
        c["discretisation"] = "zero-order hold (SSM_SCAN_ZOH)"
    if s4d_real:
        c["a_structure"] = ("opt-in S4D-real path (SSM_SCAN_S4D_REAL): Abar_n = Abar_0^(n+1), valid because the "
                            "workload's A is -(n+1); not the generic measurement")
    if w.d_model:
        c.update({"d_model": w.d_model, "expand": w.expand})
    if w.kind == "decode":
        c["decode_steps_per_step"] = w.steps
    if w.salient_frac:
        c["salient_frac"] = w.salient_frac
    return c


# ---------------------------------------------------------------- GPU arm

def run_gpu(args, w):
    import torch

    world, rank, local = _dist()
    if world > 1:
        import torch.distributed as dist

        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    dev = torch.device("cuda", local if world > 1 else 0)
    torch.cuda.set_device(dev)

    import selective_state_space_145_b300 as ssm
    from selective_state_space_145_b300 import inputs

    import dataclasses

    p = inputs.workload_inputs(w if world == 1 else dataclasses.replace(w, seed=w.seed + 1000 * rank))
    g = {k: (v.to(dev) if isinstance(v, torch.Tensor) else v) for k, v in p.items()}
    flush = torch.empty(256 * 1024 * 1024 // 4, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)

    if w.kind == "decode":
        state0, win0 = g["state"].clone(), g["conv_state"].clone()

        def step():
            for t in range(w.steps):
                ssm.ssm_selective_state_update(g["state"], g["conv_state"], g["x"][t], g["delta"][t], g["A"],
                                               g["B"][t], g["C"][t], g["D"], g["z"][t], g["delta_bias"], True,
                                               g["conv_w"], g["conv_b"], y=ybuf[t], zoh=args.zoh)

        ybuf = torch.empty(w.steps, w.batch, w.dim, dtype=g["x"].dtype, device=dev)
        cl = 0
        launches_per_step = w.steps
        kernels = ["decode_kernel"]
        # the 64 token steps are replayed from one CUDA graph, as a serving loop would run them
        if not args.eager:
            step = _as_graph(step, dev)
    else:
        cl = args.chunk_len or ssm.ssm_scan_default_chunk_len(w.batch, w.dim, w.seqlen, w.dstate, g["x"].dtype)
        cl = (cl + 63) // 64 * 64
        nchunks = (w.seqlen + cl - 1) // cl
        ws_bytes = ssm.ssm_scan_workspace_bytes(w.batch, w.dim, w.seqlen, w.dstate, args.chunk_len, g["x"].dtype)
        ws = torch.empty(max(ws_bytes, 1), dtype=torch.uint8, device=dev)
        out = torch.empty_like(g["x"])
        h_last = torch.empty(w.batch, w.dim, w.dstate, dtype=torch.float32, device=dev)

        def step():
            ssm.ssm_selective_scan_fwd(g["x"], g["delta"], g["A"], g["B"], g["C"], g["D"], g["z"], g["delta_bias"],
                                       True, g["conv_w"], g["conv_b"], None, None, workspace=ws, out=out,
                                       h_last=h_last, chunk_len=args.chunk_len, reverse=args.reverse,
                                       zoh=args.zoh, s4d_real=args.s4d_real)

        launches_per_step = 2 if nchunks > 1 else 1
        main = "scan_main1_kernel or scan_main_kernel (the plan's main pass)"
        kernels = ["scan_carry_kernel", main] if nchunks > 1 else [main]
        if not args.eager:
            step = _as_graph(step, dev)

    for _ in range(args.warmup):
        flush.zero_()
        step()
    torch.cuda.synchronize(dev)
    barrier(world)

    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    with ClockSampler(dev.index if dev.index is not None else 0) as clk:
        torch.cuda.synchronize(dev)
        barrier(world)
        for i in range(args.steps):
            flush.zero_()
            starts[i].record(stream)
            step()
            ends[i].record(stream)
        torch.cuda.synchronize(dev)
        barrier(world)
    step_ms = [s.elapsed_time(e) for s, e in zip(starts, ends)]
    ms_local = statistics.mean(step_ms)
    ms = reduce_max(ms_local, world, dev)

    updates = w.updates
    value = updates * world / (ms * 1e-3)
    bytes_step = algorithmic_bytes(w)
    peak, peak_kind = _peaks()
    achieved = bytes_step / (ms * 1e-3) / 1e9

    # end to end through the public API with host buffers: every step uploads its inputs from
    # pinned host memory, makes the call(s) and downloads its results into pinned host memory.
    # Steps are pipelined the way a streaming caller would run them: two buffer sets, uploads on
    # one stream, the calls on the compute stream, downloads on a third, so step i+1's upload
    # overlaps step i's call and download (PCIe moves both directions at once). Events order
    # every reuse of a buffer; the timed region runs from before the first upload to after the
    # last download.
    e2e = None
    if rank == 0 or world > 1:
        # every input of a step in one pinned buffer and one device buffer per set: one upload copy
        hpack = _Packed(p, pin=True)
        for k, v in p.items():
            if isinstance(v, torch.Tensor):
                hpack.views[k].copy_(v)
        host = hpack.views
        nbuf = 2
        dpacks = [_Packed(p, device=dev) for _ in range(nbuf)]
        bufs = [dp.views for dp in dpacks]
        s_up, s_down = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
        ev = {name: [torch.cuda.Event() for _ in range(nbuf)] for name in ("up", "used", "done", "down")}
        if w.kind == "decode":
            outs = [{"y": torch.empty(w.steps, w.batch, w.dim, dtype=host["x"].dtype, device=dev)}
                    for _ in range(nbuf)]
            host_out = [{"y": torch.empty(w.steps, w.batch, w.dim, dtype=host["x"].dtype).pin_memory(),
                         "state": torch.empty_like(host["state"]).pin_memory()} for _ in range(nbuf)]

            def eager(d, o):
                for t in range(w.steps):
                    ssm.ssm_selective_state_update(d["state"], d["conv_state"], d["x"][t], d["delta"][t], d["A"],
                                                   d["B"][t], d["C"][t], d["D"], d["z"][t], d["delta_bias"], True,
                                                   d["conv_w"], d["conv_b"], y=o["y"][t], zoh=args.zoh)

            replays = [_as_graph(lambda d=d, o=o: eager(d, o), dev) for d, o in zip(bufs, outs)]

            def call(d, o):
                replays[next(i for i, bb in enumerate(bufs) if bb is d)]()

            def download(k):
                host_out[k]["y"].copy_(outs[k]["y"], non_blocking=True)
                host_out[k]["state"].copy_(bufs[k]["state"], non_blocking=True)

            d2h = sum(v.numel() * v.element_size() for v in host_out[0].values())
        else:
            # the results of a step in one device buffer and one pinned buffer: one download copy
            res = {"out": out, "h_last": h_last}
            opacks = [_Packed(res, device=dev) for _ in range(nbuf)]
            outs = [op.views for op in opacks]
            hopacks = [_Packed(res, pin=True) for _ in range(nbuf)]

            def call(d, o):
                ssm.ssm_selective_scan_fwd(d["x"], d["delta"], d["A"], d["B"], d["C"], d["D"], d["z"],
                                           d["delta_bias"], True, d["conv_w"], d["conv_b"], None, None,
                                           workspace=ws, out=o["out"], h_last=o["h_last"],
                                           chunk_len=args.chunk_len, reverse=args.reverse, zoh=args.zoh,
                                           s4d_real=args.s4d_real)

            def download(k):
                hopacks[k].buf.copy_(opacks[k].buf, non_blocking=True)

            d2h = opacks[0].nbytes

        def e2e_step(i):
            k = i % nbuf
            with torch.cuda.stream(s_up):
                s_up.wait_event(ev["used"][k])          # the call two steps back is done with buffer k
                dpacks[k].buf.copy_(hpack.buf, non_blocking=True)
                ev["up"][k].record(s_up)
            stream.wait_event(ev["up"][k])
            stream.wait_event(ev["down"][k])            # the download two steps back has read buffer k
            with torch.cuda.stream(stream):
                call(bufs[k], outs[k])
                ev["used"][k].record(stream)
            with torch.cuda.stream(s_down):
                s_down.wait_event(ev["used"][k])
                download(k)
                ev["down"][k].record(s_down)

        h2d = hpack.nbytes
        for i in range(2 * nbuf):
            e2e_step(i)
        torch.cuda.synchronize(dev)
        n_e2e = max(3, min(args.steps, 20))
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(s_up)
        for i in range(n_e2e):
            e2e_step(i)
        e1.record(s_down)
        torch.cuda.synchronize(dev)
        e2e_ms = reduce_max(e0.elapsed_time(e1) / n_e2e, world, dev)
        e2e = {"value": updates * world / (e2e_ms * 1e-3), "unit": UNIT, "h2d_bytes_per_step": int(h2d),
               "d2h_bytes_per_step": int(d2h), "ms_per_step": e2e_ms,
               "pipeline": "2 buffer sets; one packed upload, the call(s) and one packed download per step on three streams, overlapped across steps"}

    if rank != 0:
        if world > 1:
            import torch.distributed as dist

            dist.destroy_process_group()
        return 0

    cpu = None
    if world == 1 and not args.no_cpu_baseline:
        r, cores, desc = oracle_sample_rate(w, target_s=args.cpu_seconds, reverse=args.reverse, zoh=args.zoh)
        cpu = {"value": r, "unit": UNIT, "cores": cores, "kind": "oracle", "sample": desc}

    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f32", "data": "synthetic (seeded; shapes and distributions of the workload)",
        "config": config_of(w, args.reverse, args.zoh, args.eager, args.s4d_real),
        "hbm_gbs": achieved,
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
                     "traffic": traffic_from_profiles(w.name, w.kind), "peak_source": peak_kind,
                     "spec_gbs": SPEC_HBM_GBS, "frac_of_spec": achieved / SPEC_HBM_GBS,
                     "algorithmic_bytes_per_step": bytes_step,
                     "timed": "whole step (" + " + ".join(kernels) + "), CUDA events on the launching stream"},
        "roofline_alu": alu_roofline(w, ms * 1e-3, cl, torch.cuda.get_device_properties(dev).multi_processor_count)
        if w.kind == "scan" else None,
        "cpu_baseline": cpu,
        "e2e": e2e,
        "gpu_launches": launches_per_step * args.steps,
        "clocks": clk.summary(),
        "step_ms_min": min(step_ms), "step_ms_max": max(step_ms),
    }
    print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist

        dist.destroy_process_group()
    return 0


def run_gpu_bwd(args, w):
    """The scan's backward pass on the workload's shapes (x taken as the scan input u): one
    ssm_selective_scan_bwd call per step, CUDA events on the launching stream, L2 flushed
    before every step outside the events."""
    import torch

    world, rank, local = _dist()
    if world > 1:
        import torch.distributed as dist

        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    dev = torch.device("cuda", local if world > 1 else 0)
    torch.cuda.set_device(dev)

    import dataclasses

    import selective_state_space_145_b300 as ssm
    from selective_state_space_145_b300 import inputs

    p = inputs.workload_inputs(w if world == 1 else dataclasses.replace(w, seed=w.seed + 1000 * rank))
    gen = torch.Generator().manual_seed(w.seed + 7)
    dout = torch.randn(w.batch, w.dim, w.seqlen, generator=gen).to(p["x"].dtype)
    dhl = torch.randn(w.batch, w.dim, w.dstate, generator=gen)
    g = {k: (v.to(dev) if isinstance(v, torch.Tensor) else v) for k, v in p.items()}
    dout_d, dhl_d = dout.to(dev), dhl.to(dev)
    flush = torch.empty(256 * 1024 * 1024 // 4, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)
    ws = torch.empty(max(1, ssm.ssm_scan_bwd_workspace_bytes(w.batch, w.dim, w.seqlen, w.dstate, g["x"].dtype)),
                     dtype=torch.uint8, device=dev)
    args_bwd = (g["x"], g["delta"], g["A"], g["B"], g["C"], dout_d, g["D"], g["z"], g["delta_bias"], True, g["h0"],
                dhl_d)
    grads = ssm.ssm_selective_scan_bwd(*args_bwd, workspace=ws)

    def step():
        ssm.ssm_selective_scan_bwd(*args_bwd, workspace=ws, grads=grads)

    if not args.eager:
        step = _as_graph(step, dev)

    for _ in range(args.warmup):
        flush.zero_()
        step()
    torch.cuda.synchronize(dev)
    barrier(world)
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    with ClockSampler(dev.index if dev.index is not None else 0) as clk:
        torch.cuda.synchronize(dev)
        barrier(world)
        for i in range(args.steps):
            flush.zero_()
            starts[i].record(stream)
            step()
            ends[i].record(stream)
        torch.cuda.synchronize(dev)
        barrier(world)
    ms = reduce_max(statistics.mean(s.elapsed_time(e) for s, e in zip(starts, ends)), world, dev)
    # the conv prologue's backward (block workloads): du -> dx, dconv_w, dconv_b, timed alone
    conv_ms = None
    if w.d_conv:
        cws = torch.empty(max(1, int(ssm.lib().ssm_conv_bwd_workspace_bytes(w.batch, w.dim, w.seqlen, w.d_conv,
                                                                            1 if w.io == "bf16" else 0))),
                          dtype=torch.uint8, device=dev)
        cargs = (g["x"], g["conv_w"], grads["du"], g["conv_b"])

        def conv_step():
            ssm.ssm_causal_conv1d_bwd(*cargs, workspace=cws)

        if not args.eager:
            conv_step = _as_graph(conv_step, dev)
        for _ in range(3):
            conv_step()
        cs = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
        ce = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
        for i in range(args.steps):
            flush.zero_()
            cs[i].record(stream)
            conv_step()
            ce[i].record(stream)
        torch.cuda.synchronize(dev)
        conv_ms = statistics.mean(s.elapsed_time(e) for s, e in zip(cs, ce))
    updates = w.updates
    bytes_step = bwd_algorithmic_bytes(w)
    peak, peak_kind = _peaks()
    achieved = bytes_step / (ms * 1e-3) / 1e9
    if rank != 0:
        if world > 1:
            import torch.distributed as dist

            dist.destroy_process_group()
        return 0
    cpu = None
    if world == 1 and not args.no_cpu_baseline:
        import oracle

        nch = min(w.dim, 64)
        sub = inputs.scan_inputs(1, nch, w.seqlen, w.dstate, 0, w.io, w.seed, with_h0=True)
        sd = torch.randn(1, nch, w.seqlen, generator=gen).to(sub["x"].dtype)
        cores = oracle.oracle.default_threads()
        reps, t0 = 0, time.perf_counter()
        while time.perf_counter() - t0 < args.cpu_seconds and reps < 1000:
            oracle.selective_scan_bwd(sub["x"], sub["delta"], sub["A"], sub["B"], sub["C"], sd, sub["D"], sub["z"],
                                      sub["delta_bias"], True, sub["h0"], None, nthreads=cores)
            reps += 1
        dt = time.perf_counter() - t0
        cpu = {"value": reps * nch * w.seqlen * w.dstate / dt, "unit": UNIT, "cores": cores, "kind": "oracle",
               "sample": f"{reps} backward pass(es) over {nch} channels x {w.seqlen} steps x N={w.dstate} (fp64)"}
    cfg = config_of(w)
    cfg["pass"] = "backward (ssm_selective_scan_bwd; x taken as the scan input u)"
    line = {
        "metric": METRIC, "value": updates * world / (ms * 1e-3), "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic (seeded)", "config": cfg,
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
                     "traffic": traffic_from_profiles(w.name + "#backward", "backward"), "peak_source": peak_kind,
                     "algorithmic_bytes_per_step": bytes_step,
                     "timed": "whole step (scan_bwd_ckpt_kernel + scan_bwd_kernel + scan_bwd_reduce_kernel)"},
        "cpu_baseline": cpu, "e2e": None, "gpu_launches": 3 * args.steps, "clocks": clk.summary(),
        "conv_backward_ms": conv_ms,
        "conv_backward_gbs": (None if conv_ms is None else
                              w.batch * w.dim * w.seqlen * (2 if w.io == "bf16" else 4) * 3 / (conv_ms * 1e-3) / 1e9),
    }
    print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist

        dist.destroy_process_group()
    return 0


# ---------------------------------------------------------------- state-space-duality layer

SSD_Q = 128  # the kernel's chunk length


def ssd_algorithmic_bytes(w) -> int:
    """x, dt, B, C read once, y and the final state written once, parameters read once."""
    tok = w.batch * w.seqlen
    return (tok * w.nheads * w.headdim * 2 * 2 + tok * w.nheads * 2 + 2 * tok * w.dstate * 2
            + w.batch * w.nheads * w.headdim * w.dstate * 4 + w.nheads * 4 * 3)


def ssd_flops(w):
    """Tensor-core FLOPs of one step of the chunked dual form, per chunk of Q steps and head:
    C B^T (2 Q^2 N), the masked product with X (2 Q^2 P), C H_in (2 Q N P) and the chunk's state
    increment B^T X (2 N Q P). Returns (algorithmic, executed): the kernel multiplies the three
    operands it computes (G', H_in and the decay-scaled B) as hi + lo bf16 pairs, which doubles
    three of the four."""
    Q, N, P = SSD_Q, w.dstate, w.headdim
    units = w.batch * w.nheads * ((w.seqlen + Q - 1) // Q)
    alg = 2 * Q * Q * N + 2 * Q * Q * P + 2 * Q * N * P + 2 * N * Q * P
    exe = 2 * Q * Q * N + 4 * Q * Q * P + 4 * Q * N * P + 4 * N * Q * P
    return units * alg, units * exe


def _bf16_peak_tflops():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            p = json.load(f)
        if "bf16_tflops" in p:
            return float(p["bf16_tflops"]), "measured (cuBLAS bf16 burst)"
    return 1800.0, "fallback"


def ssd_config_of(w, eager: bool = False):
    return {"workload": w.name, "kind": "ssd", "io": "bf16", "batch": w.batch, "seqlen": w.seqlen,
            "nheads": w.nheads, "headdim": w.headdim, "d_state": w.dstate, "chunk": SSD_Q,
            "d_model": w.d_model, "expand": w.expand, "l2": "flushed before every timed step (256 MiB write)",
            "launch": "direct library calls" if eager else "the step's library call replayed from one CUDA graph"}


def ssd_oracle_rate(w, target_s: float = 10.0):
    """The fp64 oracle on a bounded sample of (batch, head) pairs at the full sequence length."""
    import oracle
    from selective_state_space_145_b300 import inputs

    cores = oracle.oracle.default_threads()
    p = inputs.ssd_workload_inputs(w)
    pairs = 1
    t0 = time.perf_counter()
    oracle.ssd(p["x"][:1, :, :1], p["dt"][:1, :, :1], p["A"][:1], p["B"][:1], p["C"][:1], p["D"][:1],
               p["dt_bias"][:1], True, None, nthreads=cores)
    one = max(time.perf_counter() - t0, 1e-6)
    heads = int(max(1, min(w.nheads, target_s / one)))
    reps, t0 = 0, time.perf_counter()
    while True:
        oracle.ssd(p["x"][:1, :, :heads], p["dt"][:1, :, :heads], p["A"][:heads], p["B"][:1], p["C"][:1],
                   p["D"][:heads], p["dt_bias"][:heads], True, None, nthreads=cores)
        reps += 1
        if time.perf_counter() - t0 >= target_s or reps >= 1000:
            break
    dt = time.perf_counter() - t0
    pairs = reps * heads
    ups = pairs * w.seqlen * w.headdim * w.dstate
    return ups / dt, cores, (f"{reps} pass(es) over {heads} head(s) of one sequence x {w.seqlen} steps "
                             f"x {w.headdim} x {w.dstate} state (fp64, {cores} threads)")


def run_reference_ssd(args, w):
    world, rank, _ = _dist()
    if rank != 0:
        return 0
    rates, desc, cores = [], "", 1
    budget = max(2.0, 120.0 / max(1, args.steps + args.warmup))
    for i in range(args.warmup + args.steps):
        r, cores, desc = ssd_oracle_rate(w, target_s=budget)
        if i >= args.warmup:
            rates.append(r)
    value = statistics.mean(rates)
    print(json.dumps({"metric": METRIC, "value": value, "unit": UNIT, "impl": "reference", "n_gpus": args.gpus,
                      "steps": args.steps, "warmup": args.warmup, "ms_per_step": w.updates / value * 1e3,
                      "ms_per_step_basis": "one whole step of the workload at the oracle's sampled rate",
                      "higher_is_better": True,
                      "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
                      "config": ssd_config_of(w),
                      "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle", "sample": desc},
                      "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}),
          flush=True)
    return 0


def run_gpu_ssd(args, w):
    """One ssm_ssd_fwd call per step (one kernel after clearing the status word)."""
    import torch

    world, rank, local = _dist()
    if world > 1:
        import torch.distributed as dist

        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    dev = torch.device("cuda", local if world > 1 else 0)
    torch.cuda.set_device(dev)
    import dataclasses

    import selective_state_space_145_b300 as ssm
    from selective_state_space_145_b300 import inputs

    p = inputs.ssd_workload_inputs(w if world == 1 else dataclasses.replace(w, seed=w.seed + 1000 * rank))
    g = {k: (v.to(dev) if isinstance(v, torch.Tensor) else v) for k, v in p.items()}
    flush = torch.empty(256 * 1024 * 1024 // 4, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)
    wsb = ssm.ssm_ssd_workspace_bytes(w.batch, w.seqlen, w.nheads, w.headdim, w.dstate, torch.bfloat16)
    ws = torch.zeros(max(1, wsb), dtype=torch.uint8, device=dev)
    y = torch.empty_like(g["x"])
    h_last = torch.empty(w.batch, w.nheads, w.headdim, w.dstate, dtype=torch.float32, device=dev)

    def call(d, yo, ho):
        ssm.ssm_ssd_fwd(d["x"], d["dt"], d["A"], d["B"], d["C"], d["D"], d["dt_bias"], True, None, workspace=ws,
                        out=yo, h_last=ho)

    step = (lambda: call(g, y, h_last))
    if not args.eager:
        step = _as_graph(step, dev)
    for _ in range(args.warmup):
        flush.zero_()
        step()
    torch.cuda.synchronize(dev)
    if int(ws[:4].view(torch.int32).item()) != 0:
        raise RuntimeError("ssm_ssd_fwd: a tensor-core wait ran out")
    barrier(world)
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    with ClockSampler(dev.index if dev.index is not None else 0) as clk:
        torch.cuda.synchronize(dev)
        barrier(world)
        for i in range(args.steps):
            flush.zero_()
            starts[i].record(stream)
            step()
            ends[i].record(stream)
        torch.cuda.synchronize(dev)
        barrier(world)
    step_ms = [s_.elapsed_time(e_) for s_, e_ in zip(starts, ends)]
    ms = reduce_max(statistics.mean(step_ms), world, dev)

    # end to end with host buffers, pipelined as for the scans: two buffer sets, uploads, calls and
    # downloads on three streams
    # one upload and one download copy per step, as for the scans
    hpack = _Packed(p, pin=True)
    for k_, v in p.items():
        if isinstance(v, torch.Tensor):
            hpack.views[k_].copy_(v)
    nbuf = 2
    dpacks = [_Packed(p, device=dev) for _ in range(nbuf)]
    bufs = [dp.views for dp in dpacks]
    res = {"y": y, "h_last": h_last}
    opacks = [_Packed(res, device=dev) for _ in range(nbuf)]
    outs = [op.views for op in opacks]
    hopacks = [_Packed(res, pin=True) for _ in range(nbuf)]
    s_up, s_down = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    ev = {name: [torch.cuda.Event() for _ in range(nbuf)] for name in ("up", "used", "down")}

    def e2e_step(i):
        k = i % nbuf
        with torch.cuda.stream(s_up):
            s_up.wait_event(ev["used"][k])
            dpacks[k].buf.copy_(hpack.buf, non_blocking=True)
            ev["up"][k].record(s_up)
        stream.wait_event(ev["up"][k])
        stream.wait_event(ev["down"][k])
        with torch.cuda.stream(stream):
            call(bufs[k], outs[k]["y"], outs[k]["h_last"])
            ev["used"][k].record(stream)
        with torch.cuda.stream(s_down):
            s_down.wait_event(ev["used"][k])
            hopacks[k].buf.copy_(opacks[k].buf, non_blocking=True)
            ev["down"][k].record(s_down)

    for i in range(2 * nbuf):
        e2e_step(i)
    torch.cuda.synchronize(dev)
    n_e2e = max(3, min(args.steps, 20))
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(s_up)
    for i in range(n_e2e):
        e2e_step(i)
    e1.record(s_down)
    torch.cuda.synchronize(dev)
    e2e_ms = reduce_max(e0.elapsed_time(e1) / n_e2e, world, dev)
    h2d = hpack.nbytes
    d2h = opacks[0].nbytes

    if rank != 0:
        if world > 1:
            import torch.distributed as dist

            dist.destroy_process_group()
        return 0
    cpu = None
    if world == 1 and not args.no_cpu_baseline:
        r, cores, desc = ssd_oracle_rate(w, target_s=args.cpu_seconds)
        cpu = {"value": r, "unit": UNIT, "cores": cores, "kind": "oracle", "sample": desc}
    peak_gbs, peak_kind = _peaks()
    bytes_step = ssd_algorithmic_bytes(w)
    gbs = bytes_step / (ms * 1e-3) / 1e9
    alg, exe = ssd_flops(w)
    tf_peak, tf_kind = _bf16_peak_tflops()
    tf = alg / (ms * 1e-3) / 1e12
    line = {
        "metric": METRIC, "value": w.updates * world / (ms * 1e-3), "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic (seeded; shapes and distributions of the workload)",
        "config": ssd_config_of(w, args.eager),
        "roofline": {"bound": "tensor", "achieved": tf, "peak": tf_peak, "unit": "TFLOP/s", "frac": tf / tf_peak,
                     "traffic": traffic_from_profiles(w.name, "ssd"), "peak_source": tf_kind,
                     "algorithmic_flops_per_step": alg, "executed_flops_per_step": exe,
                     "executed_tflops": exe / (ms * 1e-3) / 1e12,
                     "timed": "whole step (ssd_fused_kernel), CUDA events on the launching stream"},
        "roofline_hbm": {"bound": "hbm", "achieved": gbs, "peak": peak_gbs, "unit": "GB/s", "frac": gbs / peak_gbs,
                         "peak_source": peak_kind, "algorithmic_bytes_per_step": bytes_step},
        "cpu_baseline": cpu,
        "e2e": {"value": w.updates * world / (e2e_ms * 1e-3), "unit": UNIT, "h2d_bytes_per_step": int(h2d),
                "d2h_bytes_per_step": int(d2h), "ms_per_step": e2e_ms,
                "pipeline": "2 buffer sets; one packed upload, the call(s) and one packed download per step on three streams, overlapped across steps"},
        "gpu_launches": args.steps, "clocks": clk.summary(),
        "step_ms_min": min(step_ms), "step_ms_max": max(step_ms),
    }
    print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist

        dist.destroy_process_group()
    return 0


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD)
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--seqlen", type=int, default=None,
                    help="override the workload's sequence length (smaller cases for profiling)")
    ap.add_argument("--batch", type=int, default=None, help="override the workload's batch size")
    ap.add_argument("--chunk-len", type=int, default=0,
                    help="scan chunk length (0 = the library's default policy)")
    ap.add_argument("--reverse", action="store_true", help="time the backward scan (SSM_SCAN_REVERSE)")
    ap.add_argument("--zoh", action="store_true", help="zero-order-hold discretisation (SSM_SCAN_ZOH)")
    ap.add_argument("--s4d-real", action="store_true",
                    help="the opt-in S4D-real path (SSM_SCAN_S4D_REAL); labelled in config, never the default")
    ap.add_argument("--backward", action="store_true", help="time the scan's backward pass")
    ap.add_argument("--eager", action="store_true",
                    help="time direct library calls instead of replaying the step from a CUDA graph")
    args = ap.parse_args(argv)
    import dataclasses

    from selective_state_space_145_b300 import inputs

    args.warmup = max(args.warmup, 3)  # at least 3 untimed warm-up steps
    if args.workload in inputs.SSD_WORKLOADS:
        w = inputs.SSD_WORKLOADS[args.workload]
        if args.reverse or args.zoh or args.backward or args.chunk_len or args.s4d_real:
            ap.error("the state-space-duality workload takes none of --reverse, --zoh, --backward, --chunk-len, "
                     "--s4d-real")
        if args.seqlen is not None or args.batch is not None:
            w = dataclasses.replace(w, seqlen=args.seqlen if args.seqlen is not None else w.seqlen,
                                    batch=args.batch if args.batch is not None else w.batch)
            w = dataclasses.replace(w, name=f"{w.name}[batch={w.batch},seqlen={w.seqlen}]")
        return run_reference_ssd(args, w) if args.impl == "reference" else run_gpu_ssd(args, w)
    w = inputs.WORKLOADS[args.workload]
    if args.reverse and w.kind != "scan":
        ap.error("--reverse applies to the scan workloads only")
    if args.s4d_real and (w.kind != "scan" or args.backward):
        ap.error("--s4d-real applies to the forward scan workloads only")
    if args.seqlen is not None or args.batch is not None:
        w = dataclasses.replace(w, seqlen=args.seqlen if args.seqlen is not None else w.seqlen,
                                batch=args.batch if args.batch is not None else w.batch)
        w = dataclasses.replace(w, name=f"{w.name}[batch={w.batch},seqlen={w.seqlen}]")
    if args.impl == "reference":
        return run_reference(args, w)
    if args.backward:
        if w.kind != "scan" or args.impl != "ours":
            ap.error("--backward times this library's backward pass on a scan workload")
        return run_gpu_bwd(args, w)
    return run_gpu(args, w)


if __name__ == "__main__":
    sys.exit(main())
