"""Benchmark of the GB300 hyper-connection read.

Metric: microseconds per hyper-connection read and achieved HBM GB/s with cold
weights at T = 1..8.  One step is the cold read sweep at n=4, d=2560, K=320:
for every T in (1, 2, 3, 4, 5, 6, 8) with the pending write off and on, 300
independent reads rotated over 16 weight sets (16 x 13.1 MB > the 129 MB L2),
each with its own output buffers, enqueued as one hc_read_batch (the library
runs reads that share no memory side by side on its internal streams), each
case captured once as a CUDA graph and replayed.  Before capture, every
weight set's W_down and W_up are also registered in tile order with the
handle (hc_read_register_down_tiles / _up_tiles, a one-time setup outside
the timed region): the kernels fetch their weight tiles from them, with
results bit for bit those of the weights as given, whose sweep is reported
too.  `value` is the algorithmic
bytes of every read of the step divided by the step time (GB/s, higher is
better); `us_per_read` gives the per-case times.

Also reported on the same line: the same sweep as 300 hc_read calls on one
stream, the 96-read chained window graph (T=4; hc_read_batch, the persistent
window kernel, and 96 hc_read calls), the scaled-up width (d=4096, K=512) and
the T=16/32/64 batches, the same sweep over Q8_0 weights, the roofline of the read, an end-to-end figure through
host buffers, and the FP64 oracle timed on one host core (a baseline only).

`--impl reference` times the FP64 oracle as the reference arm (host cores, a
bounded sample of the same workload per step).

Multi-GPU: one process per GPU (torchrun); every rank runs the same workload
on its own GPU (replicas, weak scaling, no collective on the data path).
"""

from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

import synth  # noqa: E402

METRIC = "µs per hyper-connection read and achieved HBM GB/s (cold weights) at T=1..8"
EPS = 1e-6
SWEEP_T = (1, 2, 3, 4, 5, 6, 8)
CALLS = 300
SETS = 16
NOMINAL_HBM_GBS = 7900.0  # GB300 HBM3e nominal, context beside the measured copy rate
WINDOW_READS = 96
WINDOW_T = 4


def read_bytes(g: synth.Geometry, T: int, pending: bool) -> int:
    """Algorithmic bytes of one read: each byte the read must move, once.

    weights 4*K*N (W_down + W_up, BF16) + w_norm and gate 8*N + per token:
    R in and out 8*N, mean 4*d, lo 4*K, pending 4*N when on.
    """
    per_token = 8 * g.N + 4 * g.d + 4 * g.K + (4 * g.N if pending else 0)
    return 4 * g.K * g.N + 8 * g.N + T * per_token


def read_bytes_q8(g: synth.Geometry, T: int, pending: bool) -> int:
    """Algorithmic bytes of one Q8_0 read: quants 2*K*N (one byte a weight,
    both projections) and scales 2*2*K*N/32 (binary16 per 32-weight block)
    in place of the BF16 weights; the rest as read_bytes."""
    return read_bytes(g, T, pending) - 4 * g.K * g.N + 2 * g.K * g.N + 4 * g.K * g.N // 32


def sweep_cases():
    return [(T, p) for T in SWEEP_T for p in (False, True)]


# --------------------------------------------------------------------- helpers

def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def max_over_ranks(dist, seconds: float, device=None) -> float:
    """The largest of the ranks' values (a time), by one all-reduce (MAX);
    `dist` is torch.distributed with a process group, or None on one rank."""
    if dist is None:
        return seconds
    import torch
    t = torch.tensor([seconds], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_gbs(world: int, bytes_per_step: int, steps: int, seconds: float) -> float:
    """Whole-job throughput: every rank moved bytes_per_step per step (weak
    scaling, replicas), over the slowest rank's time."""
    return world * bytes_per_step * steps / seconds / 1e9


def _code_only(text: str) -> str:
    """C++ source without its comments, whitespace runs collapsed (the
    sources hashed here hold no comment markers inside string literals)."""
    text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
    text = re.sub(r"//[^\n]*", " ", text)
    return " ".join(text.split())


def kernel_source_hash(names=None) -> str:
    """Hash of the CUDA sources' code (all of them, or the files in `names`);
    comments and layout do not change it."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "hyper_connection_residual_gb300", "csrc")
    for name in sorted(names if names is not None else os.listdir(csrc)):
        with open(os.path.join(csrc, name), encoding="utf-8") as f:
            h.update(name.encode())
            h.update(_code_only(f.read()).encode())
    return h.hexdigest()[:16]


# The device code of the T=1 read kernels, whose DRAM counters profiles/traffic.json records.
T1_KERNEL_SOURCES = ("hc_kernels.cuh", "hc_ptx.cuh")


def measured_peaks() -> dict:
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return {"hbm_gbs": float(d["hbm_gbs"]), "source": "measured"}
    return {"hbm_gbs": 6800.0, "source": "fallback"}


def profiled_traffic() -> dict | None:
    """DRAM bytes per read from a committed ncu summary, if it matches these kernels."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        d = json.load(f)
    if d.get("kernel_hash") != kernel_source_hash(T1_KERNEL_SOURCES):
        return None
    return d


class ClockSampler:
    """nvidia-smi sampling of SM clock and throttle reasons while it runs."""

    FIELDS = ("clocks.sm,clocks.max.sm,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id: str | None):
        self.gpu_id = gpu_id
        self.proc = None
        self.lines: list[str] = []
        self._t = None

    def __enter__(self):
        cmd = ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
               "-lms", "100"]
        if self.gpu_id:
            cmd[1:1] = ["-i", self.gpu_id]
        try:
            self.proc = subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL,
                                         text=True)
            self._t = threading.Thread(target=self._drain, daemon=True)
            self._t.start()
        except OSError:
            self.proc = None
        return self

    def _drain(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            if self._t is not None:
                self._t.join(timeout=2)

    def summary(self) -> dict:
        sm, mx, reasons = [], [], set()
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
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
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted(reasons), "samples": len(sm)}


def gpu_uuid(dev) -> str | None:
    import torch
    try:
        u = str(torch.cuda.get_device_properties(dev).uuid)
    except Exception:  # noqa: BLE001 - older torch
        return None
    return u if u.startswith("GPU-") else f"GPU-{u}"


# --------------------------------------------------------------------- oracle arms

class OracleWork:
    """The FP64 oracle, as it stands, on the sweep's inputs (prepared once,
    outside any timed region); one host thread."""

    def __init__(self):
        import oracle
        self.g = synth.G1
        self.orc = oracle.default()
        self.ws = [synth.weight_set(self.g, j) for j in range(2)]
        self.act = synth.activations(self.g, max(SWEEP_T), True)
        self.k = 0

    def read(self, case) -> int:
        """One oracle read of `case` = (T, pending); returns its algorithmic bytes."""
        T, p = case
        g, w, act = self.g, self.ws[self.k % len(self.ws)], self.act
        self.k += 1
        self.orc.read(g.n, g.d, g.K, R=act.R[:T], P=act.P[:T] if p else None, w_norm=w.w_norm,
                      W_down=w.W_down, W_up=w.W_up, gate=w.gate, eps=EPS)
        return read_bytes(g, T, p)

    def sample(self, seconds: float, cases):
        """Cycle the cases, one read each, until `seconds` have passed."""
        done, reads = 0, 0
        t0 = time.perf_counter()
        while True:
            done += self.read(cases[reads % len(cases)])
            reads += 1
            el = time.perf_counter() - t0
            if el >= seconds:
                return done, reads, el


def run_reference(args):
    world, rank, _ = dist_env()
    if rank != 0:
        return 0
    cases = sweep_cases()
    work = OracleWork()
    # one step = one oracle read of one case of the sweep, cycling through the cases
    for s in range(args.warmup):
        work.read(cases[s % len(cases)])
    total_bytes = 0
    t0 = time.perf_counter()
    for s in range(args.steps):
        total_bytes += work.read(cases[s % len(cases)])
    elapsed = time.perf_counter() - t0
    gbs = total_bytes / elapsed / 1e9
    line = {
        "impl": "reference", "metric": METRIC, "value": gbs, "unit": "GB/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1e3 * elapsed / max(1, args.steps), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": "cold read sweep, n=4 d=2560 K=320, T in (1,2,3,4,5,6,8), "
                               "pending off/on; one FP64 oracle read per step, cycling the cases"},
        "us_per_read": 1e6 * elapsed / max(1, args.steps),
        "cpu_baseline": {"value": gbs, "unit": "GB/s", "cores": 1, "kind": "oracle",
                         "sample": f"{args.steps} oracle reads, one per step over the sweep's 14 cases"},
        "e2e": {"value": gbs, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


# --------------------------------------------------------------------- GPU arm

class Sweep:
    """Device-resident inputs and one captured graph per case.

    Every read has its own R and P (distinct buffers: a read's activations are
    never another read's, as in a verify window) and, with batch=True, its own
    out, mean and lo; per T they are one contiguous block of `calls` reads
    ([calls][T][...]), which the end-to-end leg copies in and out whole.
    batch=True: the case's reads are one hc_read_batch.  batch=False: one
    hc_read call per read on the stream, all into one set of output buffers."""

    def __init__(self, hc, torch, dev, g: synth.Geometry, Ts, pendings, sets: int, calls: int,
                 stream, batch: bool = True, q8: bool = False, tiles: bool = False):
        self.g, self.calls, self.batch, self.q8 = g, calls, batch, q8
        self.torch, self.hc, self.dev, self.stream = torch, hc, dev, stream
        Tmax = max(Ts)
        self.ws = []
        for j in range(sets):
            if q8:
                w = synth.q8_weight_set(g, j)
                self.ws.append(dict(
                    w_norm=torch.from_numpy(w.w_norm).to(dev), gate=torch.from_numpy(w.gate).to(dev),
                    Wd_q=torch.from_numpy(w.Wd_q).to(dev), Wd_scale=torch.from_numpy(w.Wd_scale.view(np.int16)).to(dev),
                    Wu_q=torch.from_numpy(w.Wu_q).to(dev), Wu_scale=torch.from_numpy(w.Wu_scale.view(np.int16)).to(dev)))
                continue
            w = synth.weight_set(g, j)
            self.ws.append(dict(
                w_norm=torch.from_numpy(w.w_norm).to(dev), gate=torch.from_numpy(w.gate).to(dev),
                W_down=torch.from_numpy(w.W_down.view(np.int16)).to(dev),
                W_up=torch.from_numpy(w.W_up.view(np.int16)).to(dev)))
        # One activation draw per T, copied into every read's own buffers; each
        # case has its own buffers (the end-to-end leg refills one case's
        # inputs while another case runs).
        self.act = {}
        nout = calls if batch else 1
        for T in sorted(set(Ts)):
            a = synth.activations(g, T, True)
            R1 = torch.from_numpy(a.R).to(dev)
            for p in pendings:
                blk = dict(R=R1.unsqueeze(0).repeat(calls, 1, 1).contiguous(),
                           out=torch.empty(nout, T, g.N, device=dev), mean=torch.empty(nout, T, g.d, device=dev),
                           lo=torch.empty(nout, T, g.K, device=dev))
                if p:
                    blk["P"] = torch.from_numpy(a.P).to(dev).unsqueeze(0).repeat(calls, 1, 1).contiguous()
                self.act[(T, p)] = blk
        self.rd = hc.Read(g.n, g.d, g.K, T_max=max(8, Tmax), eps=EPS)
        # tiles: every weight set's W_down and W_up also in tile order,
        # registered with the handle before capture (hc_read_register_down_tiles,
        # hc_read_register_up_tiles; no up tiles where no kernel takes them).
        self.tiles = []
        if tiles:
            for w in self.ws:
                self.tiles.append(self.rd.down_tiles(w["W_down"]))
                self.tiles.append(self.rd.up_tiles(w["W_up"]))
        self.cases = [(T, p) for T in Ts for p in pendings]
        self.graphs = {}
        for case in self.cases:
            self.graphs[case] = self._capture(*case)

    def _desc(self, T, pending, j):
        a = self.act[(T, pending)]
        o = j if self.batch else 0
        return dict(R=a["R"][j], P=a["P"][j] if pending else None, out=a["out"][o], mean=a["mean"][o],
                    lo=a["lo"][o], **self.ws[j % len(self.ws)])

    def _capture(self, T, pending):
        hc = self.hc
        descs = [self._desc(T, pending, j) for j in range(self.calls)]
        with self.torch.cuda.stream(self.stream):
            hc.hc_graph_begin(self.stream)
            if self.batch:
                (self.rd.batch_q8 if self.q8 else self.rd.batch)(descs, T, stream=self.stream)
            elif self.q8:
                for d in descs:
                    self.rd.q8(d["R"], d["w_norm"], d["Wd_q"], d["Wd_scale"], d["Wu_q"], d["Wu_scale"],
                               d["gate"], d["P"], T, d["out"], d["mean"], d["lo"], stream=self.stream)
            else:
                for d in descs:
                    self.rd(d["R"], d["w_norm"], d["W_down"], d["W_up"], d["gate"], d["P"], T,
                            d["out"], d["mean"], d["lo"], stream=self.stream)
            return hc.hc_graph_end(self.stream)

    def plan(self, case):
        T, pending = case
        descs = [self._desc(T, pending, j) for j in range(self.calls)]
        return (self.rd.batch_q8_plan if self.q8 else self.rd.batch_plan)(descs, T)

    def block(self, case):
        """The case's device buffers: R, (P), out, mean, lo, each [calls][T][...]."""
        return self.act[case]

    def replay(self, case):
        self.hc.hc_graph_launch(self.graphs[case], self.stream)

    def bytes_per_replay(self, case):
        return self.calls * (read_bytes_q8 if self.q8 else read_bytes)(self.g, *case)

    def close(self):
        for gr in self.graphs.values():
            self.hc.hc_graph_destroy(gr)
        self.graphs = {}
        self.rd.close()


def time_cases(torch, sweep: Sweep, steps: int, warmup: int, stream):
    """Replay every case `steps` times; returns (total seconds, per-case seconds)."""
    for _ in range(warmup):
        for case in sweep.cases:
            sweep.replay(case)
    stream.synchronize()
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(len(sweep.cases) + 1)]
           for _ in range(steps)]
    per_case = {c: 0.0 for c in sweep.cases}
    start = torch.cuda.Event(enable_timing=True)
    stop = torch.cuda.Event(enable_timing=True)
    start.record(stream)
    for s in range(steps):
        evs[s][0].record(stream)
        for i, case in enumerate(sweep.cases):
            sweep.replay(case)
            evs[s][i + 1].record(stream)
    stop.record(stream)
    stop.synchronize()
    for s in range(steps):
        for i, case in enumerate(sweep.cases):
            per_case[case] += evs[s][i].elapsed_time(evs[s][i + 1]) / 1e3
    return start.elapsed_time(stop) / 1e3, per_case


def run_window(torch, hc, dev, stream, replays: int, batch: bool):
    """96 chained reads (out_i is R_{i+1}) with distinct weight sets, T=4,
    captured once and replayed: one hc_read_batch (batch=True: the persistent
    window kernel) or 96 hc_read calls."""
    g = synth.G1
    T = WINDOW_T
    ws = []
    for j in range(WINDOW_READS):
        w = synth.weight_set(g, 100 + j)
        ws.append(dict(w_norm=torch.from_numpy(w.w_norm).to(dev), gate=torch.from_numpy(w.gate).to(dev),
                       W_down=torch.from_numpy(w.W_down.view(np.int16)).to(dev),
                       W_up=torch.from_numpy(w.W_up.view(np.int16)).to(dev)))
    act = synth.activations(g, T, False)
    R0 = torch.from_numpy(act.R).to(dev)
    bufs = [torch.empty(T, g.N, device=dev) for _ in range(WINDOW_READS + 1)]
    mean = torch.empty(T, g.d, device=dev)
    lo = torch.empty(T, g.K, device=dev)
    rd = hc.Read(g.n, g.d, g.K, T_max=8, eps=EPS)
    descs = [dict(R=bufs[i], P=None, out=bufs[i + 1], mean=mean, lo=lo, **ws[i]) for i in range(WINDOW_READS)]
    plan = rd.batch_plan(descs, T)
    with torch.cuda.stream(stream):
        hc.hc_graph_begin(stream)
        if batch:
            rd.batch(descs, T, stream=stream)
        else:
            for d in descs:
                rd(d["R"], d["w_norm"], d["W_down"], d["W_up"], d["gate"], None, T,
                   d["out"], d["mean"], d["lo"], stream=stream)
        graph = hc.hc_graph_end(stream)
    bufs[0].copy_(R0)
    torch.cuda.synchronize()
    for _ in range(3):
        hc.hc_graph_launch(graph, stream)
    stream.synchronize()
    a = torch.cuda.Event(enable_timing=True)
    b = torch.cuda.Event(enable_timing=True)
    a.record(stream)
    for _ in range(replays):
        hc.hc_graph_launch(graph, stream)
    b.record(stream)
    b.synchronize()
    sec = a.elapsed_time(b) / 1e3 / replays
    hc.hc_graph_destroy(graph)
    ok = rd.check() == hc.HC_OK
    rd.close()
    nbytes = WINDOW_READS * read_bytes(g, T, False)
    return {"reads": WINDOW_READS, "T": T, "replays": replays,
            "path": ("persistent window kernel" if plan == 1 else f"batch plan {plan}") if batch
            else "one hc_read call per read",
            "us_per_replay": sec * 1e6, "us_per_read": sec * 1e6 / WINDOW_READS,
            "GBps": nbytes / sec / 1e9, "bytes_per_replay": nbytes, "status_ok": ok}


def run_profile_case():
    """Four cold reads at T=1 and four at T=8 (pending on), each after a 256 MB
    write that flushes L2, with the weight sets' W_down registered in tile
    order as in the headline sweep; used as the small case of ncu captures."""
    import torch
    import hyper_connection_residual_gb300 as hc
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    g = synth.G1
    ws = []
    for j in range(4):
        w = synth.weight_set(g, j)
        ws.append(dict(w_norm=torch.from_numpy(w.w_norm).to(dev), gate=torch.from_numpy(w.gate).to(dev),
                       W_down=torch.from_numpy(w.W_down.view(np.int16)).to(dev),
                       W_up=torch.from_numpy(w.W_up.view(np.int16)).to(dev)))
    act = synth.activations(g, 8, True)
    R = torch.from_numpy(act.R).to(dev)
    P = torch.from_numpy(act.P).to(dev)
    out = torch.empty(8, g.N, device=dev)
    mean = torch.empty(8, g.d, device=dev)
    lo = torch.empty(8, g.K, device=dev)
    flush = torch.empty(64 * 1024 * 1024, device=dev)
    with hc.Read(g.n, g.d, g.K, T_max=8, eps=EPS) as rd:
        tiles = [rd.down_tiles(w["W_down"]) for w in ws] + [rd.up_tiles(w["W_up"]) for w in ws]  # as the headline
        for T in (1, 8):
            for w in ws:
                flush.zero_()
                rd(R, w["w_norm"], w["W_down"], w["W_up"], w["gate"], P, T, out, mean, lo)
        torch.cuda.synchronize()
        assert rd.check() == hc.HC_OK
    print("profile case done")
    return 0


def run_profile_wide_case():
    """Cold reads on the wide tensor-memory pair, each after a 256 MB write that
    flushes L2: three at T=16 (one pass), three at T=64 (four passes), pending
    off; a small case for ncu captures."""
    import torch
    import hyper_connection_residual_gb300 as hc
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    g = synth.G1
    ws = []
    for j in range(3):
        w = synth.weight_set(g, j)
        ws.append(dict(w_norm=torch.from_numpy(w.w_norm).to(dev), gate=torch.from_numpy(w.gate).to(dev),
                       W_down=torch.from_numpy(w.W_down.view(np.int16)).to(dev),
                       W_up=torch.from_numpy(w.W_up.view(np.int16)).to(dev)))
    act = synth.activations(g, 64, False)
    R = torch.from_numpy(act.R).to(dev)
    out = torch.empty(64, g.N, device=dev)
    mean = torch.empty(64, g.d, device=dev)
    lo = torch.empty(64, g.K, device=dev)
    flush = torch.empty(64 * 1024 * 1024, device=dev)
    with hc.Read(g.n, g.d, g.K, T_max=64, eps=EPS) as rd:
        for T in (16, 64):
            for w in ws:
                flush.zero_()
                rd(R, w["w_norm"], w["W_down"], w["W_up"], w["gate"], None, T, out, mean, lo)
        torch.cuda.synchronize()
        assert rd.check() == hc.HC_OK
    print("profile case done")
    return 0


def run_profile_q8_case():
    """Cold reads after a 256 MB L2 flush each: two BF16 and two Q8_0 reads at
    T=4 (the same tensor-core kernels over the two weight formats), then two
    Q8_0 reads each at T=1, T=2 and T=8 (pending on); a small case for ncu."""
    import torch
    import hyper_connection_residual_gb300 as hc
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    g = synth.G1
    bf, q8 = [], []
    for j in range(2):
        w = synth.weight_set(g, j)
        bf.append(dict(w_norm=torch.from_numpy(w.w_norm).to(dev), gate=torch.from_numpy(w.gate).to(dev),
                       W_down=torch.from_numpy(w.W_down.view(np.int16)).to(dev),
                       W_up=torch.from_numpy(w.W_up.view(np.int16)).to(dev)))
        w = synth.q8_weight_set(g, j)
        q8.append(dict(w_norm=torch.from_numpy(w.w_norm).to(dev), gate=torch.from_numpy(w.gate).to(dev),
                       Wd_q=torch.from_numpy(w.Wd_q).to(dev), Wd_scale=torch.from_numpy(w.Wd_scale.view(np.int16)).to(dev),
                       Wu_q=torch.from_numpy(w.Wu_q).to(dev), Wu_scale=torch.from_numpy(w.Wu_scale.view(np.int16)).to(dev)))
    act = synth.activations(g, 8, True)
    R = torch.from_numpy(act.R).to(dev)
    P = torch.from_numpy(act.P).to(dev)
    out = torch.empty(8, g.N, device=dev)
    mean = torch.empty(8, g.d, device=dev)
    lo = torch.empty(8, g.K, device=dev)
    flush = torch.empty(64 * 1024 * 1024, device=dev)
    with hc.Read(g.n, g.d, g.K, T_max=8, eps=EPS) as rd:
        for w in bf:
            flush.zero_()
            rd(R, w["w_norm"], w["W_down"], w["W_up"], w["gate"], P, 4, out, mean, lo)
        for T in (4, 1, 2, 8):
            for w in q8:
                flush.zero_()
                rd.q8(R, w["w_norm"], w["Wd_q"], w["Wd_scale"], w["Wu_q"], w["Wu_scale"], w["gate"], P, T,
                      out, mean, lo)
        torch.cuda.synchronize()
        assert rd.check() == hc.HC_OK
    print("profile case done")
    return 0


Q2_ROWS, Q2_COLS, Q2_COPIES = 12288, 2560, 24


def q2_bytes(rows: int, cols: int, ncols: int) -> int:
    """Algorithmic bytes of one Q2_0 product: codes, scales, x and y once."""
    return rows * cols // 4 + rows * (cols // 64) * 2 + ncols * cols * 4 + ncols * rows * 4


def run_q2_sweep(torch, hc, dev, stream, steps: int = 5, warmup: int = 3, calls: int = CALLS):
    """The Q2_0 product of the decode windows' attn_q (2560 -> 12288) at 1..4
    columns, cold: 300 products per case rotated over 24 copies of the weights
    (212 MB, more than L2), one input, own outputs, captured once as a CUDA
    graph and replayed; as one hc_q2_0_matvec_batch (independent products
    share a persistent launch) and as 300 hc_q2_0_matvec calls (each waits for
    the one before).  Returns {mode: {ncols: (seconds per product, GB/s)}}."""
    m = synth.q2_0_matrix(Q2_ROWS, Q2_COLS, j=0)
    Wq0 = torch.from_numpy(m.Wq).to(dev)
    Ws0 = torch.from_numpy(m.Wscale.view(np.int16)).to(dev)
    copies = [(Wq0.clone(), Ws0.clone()) for _ in range(Q2_COPIES)]
    x = torch.from_numpy(synth.q2_0_columns(Q2_COLS, 4, j=0)).to(dev)
    ys = [torch.empty(4, Q2_ROWS, device=dev) for _ in range(Q2_COPIES)]
    out = {"batch": {}, "chained": {}}
    for mode in out:
        for ncols in (1, 2, 3, 4):
            xv = x[:ncols]
            prods = [(*copies[i % Q2_COPIES], xv, ys[i % Q2_COPIES][:ncols]) for i in range(calls)]
            torch.cuda.synchronize()
            with torch.cuda.stream(stream):
                hc.hc_graph_begin(stream)
                if mode == "batch":
                    hc.hc_q2_0_matvec_batch(prods, Q2_ROWS, Q2_COLS, ncols, stream=stream)
                else:
                    for p in prods:
                        hc.hc_q2_0_matvec(*p, stream=stream)
                graph = hc.hc_graph_end(stream)
            for _ in range(warmup):
                hc.hc_graph_launch(graph, stream)
            stream.synchronize()
            ea = torch.cuda.Event(enable_timing=True)
            eb = torch.cuda.Event(enable_timing=True)
            ea.record(stream)
            for _ in range(steps):
                hc.hc_graph_launch(graph, stream)
            eb.record(stream)
            eb.synchronize()
            hc.hc_graph_destroy(graph)
            sec = ea.elapsed_time(eb) / 1e3 / (steps * calls)
            out[mode][ncols] = (sec, q2_bytes(Q2_ROWS, Q2_COLS, ncols) / sec / 1e9)
    del copies, ys
    return out


def run_profile_q2_case():
    """Q2_0 products (2560 -> 12288): one at 1 column and one at 4 columns, then
    one batch of 24 at 4 columns over 24 copies of the weights (212 MB), each
    after a 256 MB write that flushes L2; a small case for ncu."""
    import torch
    import hyper_connection_residual_gb300 as hc
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    m = synth.q2_0_matrix(Q2_ROWS, Q2_COLS, j=0)
    Wq = torch.from_numpy(m.Wq).to(dev)
    Ws = torch.from_numpy(m.Wscale.view(np.int16)).to(dev)
    copies = [(Wq.clone(), Ws.clone()) for _ in range(Q2_COPIES)]
    x = torch.from_numpy(synth.q2_0_columns(Q2_COLS, 4, j=0)).to(dev)
    ys = [torch.empty(4, Q2_ROWS, device=dev) for _ in range(Q2_COPIES)]
    flush = torch.empty(64 * 1024 * 1024, device=dev)
    for ncols in (1, 4):
        flush.zero_()
        hc.hc_q2_0_matvec(Wq, Ws, x[:ncols], ys[0][:ncols])
    flush.zero_()
    hc.hc_q2_0_matvec_batch([(*copies[i], x, ys[i]) for i in range(Q2_COPIES)], Q2_ROWS, Q2_COLS, 4)
    torch.cuda.synchronize()
    print("profile case done")
    return 0


def run_gpu(args):
    import torch
    import hyper_connection_residual_gb300 as hc

    world, rank, local = dist_env()
    if not torch.cuda.is_available():
        raise SystemExit("bench.py: no CUDA device (the read has no CPU path)")
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    hc.load()
    pg = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
        pg = dist

    stream = torch.cuda.Stream(device=dev)
    g = synth.G1
    calls = args.calls
    sweep = Sweep(hc, torch, dev, g, SWEEP_T, (False, True), SETS, calls, stream, tiles=True)
    step_bytes = sum(sweep.bytes_per_replay(c) for c in sweep.cases)
    plans = {sweep.plan(c) for c in sweep.cases}

    # ---- timed region (device-resident inputs)
    if pg:
        pg.barrier()
    torch.cuda.synchronize()
    with ClockSampler(gpu_uuid(dev) if rank == 0 else None) as clocks:
        total, per_case = time_cases(torch, sweep, args.steps, args.warmup, stream)
    torch.cuda.synchronize()
    total = max_over_ranks(pg, total, dev)
    if pg:
        pg.barrier()
    value = whole_job_gbs(world, step_bytes, args.steps, total)
    us_per_read = {f"T{T}_{'pend' if p else 'nopend'}": 1e6 * per_case[(T, p)] / (args.steps * calls)
                   for (T, p) in sweep.cases}
    gbs_per_case = {f"T{T}_{'pend' if p else 'nopend'}":
                    read_bytes(g, T, p) * args.steps * calls / per_case[(T, p)] / 1e9
                    for (T, p) in sweep.cases}

    # ---- end to end: every read's R (and P) in from pinned host memory and
    # every read's out and mean back, every step.  As a serving loop would:
    # host-to-device copies on one stream, the reads on the compute stream,
    # device-to-host copies on a third, ordered per case by events, so that a
    # case's inputs arrive while the case before it runs.
    host = {}
    for case in sweep.cases:
        b = sweep.block(case)
        host[case] = {k: torch.empty(b[k].shape, dtype=b[k].dtype).pin_memory()
                      for k in ("R", "P", "out", "mean") if k in b}
        host[case]["R"].copy_(b["R"])
        if "P" in b:
            host[case]["P"].copy_(b["P"])
    h2d = sum(calls * T * g.N * 4 * (2 if p else 1) for (T, p) in sweep.cases)
    d2h = sum(calls * T * (g.N + g.d) * 4 for (T, p) in sweep.cases)
    e2e_steps = max(3, min(args.steps, 20))
    up_st = torch.cuda.Stream(device=dev)
    down_st = torch.cuda.Stream(device=dev)
    ev = {c: {k: torch.cuda.Event() for k in ("in", "run", "out")} for c in sweep.cases}
    if pg:
        pg.barrier()
    torch.cuda.synchronize()
    ea = torch.cuda.Event(enable_timing=True)
    eb = torch.cuda.Event(enable_timing=True)
    ea.record(stream)
    up_st.wait_event(ea)
    for _ in range(e2e_steps):
        for case in sweep.cases:
            b, hb, e = sweep.block(case), host[case], ev[case]
            up_st.wait_event(e["run"])      # the case's previous run has read its inputs
            with torch.cuda.stream(up_st):
                b["R"].copy_(hb["R"], non_blocking=True)
                if "P" in b:
                    b["P"].copy_(hb["P"], non_blocking=True)
            e["in"].record(up_st)
            stream.wait_event(e["in"])
            stream.wait_event(e["out"])     # the case's previous outputs are back on the host
            sweep.replay(case)
            e["run"].record(stream)
            down_st.wait_event(e["run"])
            with torch.cuda.stream(down_st):
                hb["out"].copy_(b["out"], non_blocking=True)
                hb["mean"].copy_(b["mean"], non_blocking=True)
            e["out"].record(down_st)
    stream.wait_stream(up_st)
    stream.wait_stream(down_st)
    eb.record(stream)
    eb.synchronize()
    e2e_sec = ea.elapsed_time(eb) / 1e3
    e2e_sec = max_over_ranks(pg, e2e_sec, dev)
    e2e_value = whole_job_gbs(world, step_bytes, e2e_steps, e2e_sec)
    sweep.close()
    del host

    extra = {}
    if not args.quick:
        single = Sweep(hc, torch, dev, g, SWEEP_T, (False, True), SETS, calls, stream, batch=False,
                       tiles=True)
        ts, pc = time_cases(torch, single, 5, 3, stream)
        extra["sweep_one_stream_per_call"] = {
            "note": "the same 300 reads per case as hc_read calls on one stream, one set of outputs",
            "us_per_read": {f"T{T}_{'pend' if p else 'nopend'}": 1e6 * pc[(T, p)] / (5 * calls)
                            for (T, p) in single.cases},
            "GBps": sum(single.bytes_per_replay(c) for c in single.cases) * 5 / ts / 1e9}
        single.close()
        extra["window_96_reads_T4"] = run_window(torch, hc, dev, stream, replays=100, batch=True)
        extra["window_96_reads_T4_per_call"] = run_window(torch, hc, dev, stream, replays=20, batch=False)
        for key, tl in (("batch_T16_32_64", True), ("batch_T16_32_64_weights_as_given", False)):
            big = Sweep(hc, torch, dev, g, (16, 32, 64), (False,), SETS, CALLS, stream, tiles=tl)
            tb, pc = time_cases(torch, big, 5, 3, stream)
            extra[key] = {f"T{T}": {"us_per_read": 1e6 * pc[(T, p)] / (5 * CALLS),
                                    "GBps": read_bytes(g, T, p) * 5 * CALLS / pc[(T, p)] / 1e9}
                          for (T, p) in big.cases}
            big.close()
        q8 = Sweep(hc, torch, dev, g, SWEEP_T, (False, True), SETS, CALLS, stream, q8=True)
        tq, pc = time_cases(torch, q8, 5, 3, stream)
        extra["q8_0_sweep"] = {
            "note": "the sweep's reads over Q8_0 weights (int8 quants, one binary16 scale per 32 weights: "
                    "6.96 MB a weight set), one hc_read_batch_q8 per case",
            "batch_plan": sorted({q8.plan(c) for c in q8.cases}),
            "us_per_read": {f"T{T}_{'pend' if p else 'nopend'}": 1e6 * pc[(T, p)] / (5 * CALLS)
                            for (T, p) in q8.cases},
            "GBps_per_case": {f"T{T}_{'pend' if p else 'nopend'}":
                              read_bytes_q8(g, T, p) * 5 * CALLS / pc[(T, p)] / 1e9 for (T, p) in q8.cases},
            "GBps": sum(q8.bytes_per_replay(c) for c in q8.cases) * 5 / tq / 1e9}
        q8.close()
        q8s = Sweep(hc, torch, dev, g, SWEEP_T, (False,), SETS, calls, stream, batch=False, q8=True)
        ts8, pc = time_cases(torch, q8s, 5, 3, stream)
        extra["q8_0_sweep_one_stream_per_call"] = {
            "note": "the Q8_0 sweep's reads (pending off) as hc_read_q8 calls on one stream, one set of outputs",
            "us_per_read": {f"T{T}_nopend": 1e6 * pc[(T, p)] / (5 * calls) for (T, p) in q8s.cases}}
        q8s.close()
        q2 = run_q2_sweep(torch, hc, dev, stream)
        hbm = measured_peaks()["hbm_gbs"]
        extra["q2_0_matvec_attn_q"] = {
            "note": "Q2_0 product 2560 -> 12288 (two-bit codes, one binary16 scale per 64 weights: "
                    "8,847,360 B of weights), 300 products per case rotated over 24 copies of the "
                    "weights (212 MB), one input, CUDA-graph replay; bytes = weights + x + y once",
            "us_per_call": {f"ncols{n}": 1e6 * v[0] for n, v in q2["batch"].items()},
            "GBps": {f"ncols{n}": v[1] for n, v in q2["batch"].items()},
            "frac_of_measured_hbm": {f"ncols{n}": v[1] / hbm for n, v in q2["batch"].items()},
            "us_per_call_chained": {f"ncols{n}": 1e6 * v[0] for n, v in q2["chained"].items()},
            "chained_note": "the same 300 products as single hc_q2_0_matvec calls: each waits for "
                            "the one before (the engine's case when x comes from the previous layer)",
            "pages_rtx2080ti_us": {"ncols1": 24.8, "ncols2": 31.4, "ncols3": 31.3, "ncols4": 36.6},
        }
        g2 = synth.G2
        wide = Sweep(hc, torch, dev, g2, SWEEP_T, (True,), 12, CALLS, stream)
        tw, pc = time_cases(torch, wide, 5, 3, stream)
        extra["wide_d4096_K512_pend"] = {f"T{T}": {"us_per_read": 1e6 * pc[(T, p)] / (5 * CALLS),
                                                   "GBps": read_bytes(g2, T, p) * 5 * CALLS / pc[(T, p)] / 1e9}
                                         for (T, p) in wide.cases}
        wide.close()
        # The headline sweep without the tile-ordered copies (W_down as given),
        # and the scaled-up width with them (every T there takes them).
        tl = Sweep(hc, torch, dev, g, SWEEP_T, (False, True), SETS, CALLS, stream)
        tt, pc = time_cases(torch, tl, 5, 3, stream)
        extra["sweep_weights_as_given"] = {
            "note": "the headline sweep with no tile-ordered weights registered: every kernel "
                    "fetches its tiles from W_down [K][N] and W_up [N][K] themselves",
            "us_per_read": {f"T{T}_{'pend' if p else 'nopend'}": 1e6 * pc[(T, p)] / (5 * CALLS)
                            for (T, p) in tl.cases},
            "frac_of_measured_hbm": {f"T{T}_{'pend' if p else 'nopend'}":
                                     read_bytes(g, T, p) * 5 * CALLS / pc[(T, p)] / 1e9 / hbm
                                     for (T, p) in tl.cases},
            "GBps": sum(tl.bytes_per_replay(c) for c in tl.cases) * 5 / tt / 1e9}
        tl.close()
        wide = Sweep(hc, torch, dev, g2, SWEEP_T, (True,), 12, CALLS, stream, tiles=True)
        tw, pc = time_cases(torch, wide, 5, 3, stream)
        extra["wide_d4096_K512_pend_down_tiles"] = {
            f"T{T}": {"us_per_read": 1e6 * pc[(T, p)] / (5 * CALLS),
                      "GBps": read_bytes(g2, T, p) * 5 * CALLS / pc[(T, p)] / 1e9} for (T, p) in wide.cases}
        wide.close()

    if rank != 0:
        if pg:
            pg.barrier()
            pg.destroy_process_group()
        return 0

    peaks = measured_peaks()
    # the read (down kernel + up kernel) is the unit; reads of the batch
    # overlap, so its time is the case's time over its reads (T=1, pending off)
    t1 = per_case[(1, False)] / (args.steps * calls)
    achieved = read_bytes(g, 1, False) / t1 / 1e9
    traffic = profiled_traffic()
    roofline = {"bound": "hbm", "achieved": achieved, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                "frac": achieved / peaks["hbm_gbs"],
                "traffic": traffic["dram_bytes_per_read_T1"] if traffic else None,
                "peak_nominal": NOMINAL_HBM_GBS, "frac_of_nominal": achieved / NOMINAL_HBM_GBS,
                "unit_of_work": "one read (down + up kernel) at T=1, pending off: algorithmic bytes "
                                "over the 300-read batch's time per read (reads overlap on the "
                                "library's streams)",
                "peak_source": peaks["source"]}

    cpu = None
    if world == 1 and not args.no_cpu_baseline:
        b, n, el = OracleWork().sample(args.cpu_seconds, sweep_cases())
        cpu = {"value": b / el / 1e9, "unit": "GB/s", "cores": 1, "kind": "oracle",
               "sample": f"{n} FP64 oracle reads cycling the sweep's 14 cases ({el:.1f} s, 1 thread)",
               "us_per_read": 1e6 * el / n}

    line = {
        "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * total / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f32 (bf16 weights)", "data": "synthetic",
        "config": {"workload": "cold read sweep: n=4 streams, d=2560, K=320, T in (1,2,3,4,5,6,8), "
                               "pending write off and on, 300 independent reads per case rotated over "
                               "16 weight sets, own inputs and outputs per read, one hc_read_batch per "
                               "case, CUDA-graph replay",
                   "weight_layout": "each weight set's W_down and W_up also registered in tile order "
                                    "with the handle before capture (hc_read_register_down_tiles, "
                                    "hc_read_register_up_tiles; outside the timed region): the kernels "
                                    "fetch their tiles from it, bit-identical to the weights as given "
                                    "(extra.sweep_weights_as_given)",
                   "batch_plan": sorted(plans),
                   "l2": "inputs larger than L2 (16 x 13.1 MB weight sets rotated)",
                   "parallelism": f"replicas x{world}"},
        "us_per_read": us_per_read, "GBps_per_case": gbs_per_case,
        "roofline": roofline, "cpu_baseline": cpu,
        "e2e": {"value": e2e_value, "unit": "GB/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "steps": e2e_steps,
                "note": "per step, every read's own R (and P) copied in from pinned host memory and "
                        "every read's out and mean copied back, around the same graph replays; copies in, "
                        "reads and copies out on three streams ordered per case by events, so one case's "
                        "copies overlap another case's reads"},
        "gpu_launches": 2 * calls * len(sweep_cases()) * args.steps,
        "clocks": clocks.summary(),
        "extra": extra,
        "kernel_hash": kernel_source_hash(),
    }
    print(json.dumps(line), flush=True)
    if pg:
        pg.barrier()
        pg.destroy_process_group()
    return 0


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=("gb300", "reference"), default="gb300")
    ap.add_argument("--quick", action="store_true", help="skip the extra configurations")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--calls", type=int, default=CALLS, help="reads per case (default 300)")
    ap.add_argument("--profile", action="store_true",
                    help="no timing: a few cold direct reads at T=1 and T=8 (L2 flushed "
                         "before each), a small case for ncu captures")
    ap.add_argument("--profile-q2", action="store_true",
                    help="run the small Q2_0 product case used for ncu captures and exit")
    ap.add_argument("--profile-wide", action="store_true",
                    help="no timing: cold direct reads at T=16 and T=64 on the wide tensor-memory "
                         "pair, a small case for ncu captures")
    ap.add_argument("--profile-q8", action="store_true",
                    help="no timing: cold direct reads, BF16 and Q8_0 at T=4, Q8_0 at T=1 and T=8, "
                         "a small case for ncu captures")
    args = ap.parse_args(argv)
    args.warmup = max(3, args.warmup)  # at least three untimed warm-up steps
    if args.impl == "reference":
        return run_reference(args)
    if args.profile:
        return run_profile_case()
    if args.profile_q8:
        return run_profile_q8_case()
    if args.profile_wide:
        return run_profile_wide_case()
    if args.profile_q2:
        return run_profile_q2_case()
    return run_gpu(args)


if __name__ == "__main__":
    sys.exit(main())
