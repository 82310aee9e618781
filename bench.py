#!/usr/bin/env python3
"""Route-step benchmark (one JSON line on rank 0).

A step is one MoE layer's route step -- latent down projection, router
logits, top-16 and routing weights -- for the workload's token rows, with
every input resident in HBM.  The headline workload is the 8-row decode step
over 8 distinct weight banks cycled layer by layer (64.2 MB of weights each,
513 MB in total, so the weights never stay in the 129 MB L2).  Steps run as
replays of a CUDA graph of 64 layer steps; the timed region is exactly K
steps, bracketed by a barrier and a device synchronise on both sides and
timed with CUDA events on the launching stream.

The other row counts (1, 9, 12, 16, 20 decode; 1024 and 3072 prefill, the
latter per 92-layer chunk) are measured the same way and reported under
"sweep".  `e2e` repeats the headline through the host-buffer call (hidden
rows read from pinned host memory and all results written back to it, every
step): three `HostStep`s (the checked-once form of route_step_host) of one
plan with three batches in flight, with one and two in flight and the plain
route_step_host call timed beside it.
`cpu_baseline` times the oracle on the host cores on a bounded sample.

Multi-GPU: the step this benchmark times runs on one GPU (the weights are per
layer and the rows are few), so N GPUs run N independent replicas ("scaling":
"weak").  The library's column-shard plans are the sharded form; their
exchange is the caller's collective and is not timed here.

`--impl reference` times the oracle itself (the only reference this work
has), on a bounded sample per step, and prints the same line.
"""

from __future__ import annotations

import argparse
import hashlib
import json
import math
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

METRIC = "route-step us/layer and rows/s at 1-20 rows and 3072 rows; % HBM / tensor roofline"
K_HIDDEN, N_LATENT, N_EXPERTS, TOPK = 7168, 3584, 896, 16
WEIGHT_BYTES = K_HIDDEN * (N_LATENT + N_EXPERTS) * 2           # 64,225,280
ROW_BYTES = K_HIDDEN * 2 + N_LATENT * 2 + N_EXPERTS * 4 + TOPK * 8   # 25,216
FLOP_PER_ROW = 2 * K_HIDDEN * (N_LATENT + N_EXPERTS)          # 64,225,280
GRAPH_LEN = 64
SPIN_CYCLES = 200_000  # ~0.1 ms at 2 GHz
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
_CSRC = "latent_projection_top_gb300/csrc/"
# the sources each profiled kernel is built from: a recorded DRAM traffic
# figure stands only while these files are unchanged
KERNEL_SOURCES = {
    "decode_stream_kernel": [_CSRC + f for f in ("decode_kernel.cu", "topk16.cuh", "sm103_ptx.cuh",
                                                 "common.cuh", "twofloat.cuh")],
    "prefill_pair_kernel": [_CSRC + f for f in ("prefill_kernel.cu", "sm103_ptx.cuh", "common.cuh")],
}


def parse_args():
    p = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=64 * 1024)
    p.add_argument("--warmup", type=int, default=640)
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--workload", default="decode_r8",
                   choices=["decode_r1", "decode_r8", "decode_sweep", "prefill_r1024",
                            "prefill_r3072"])
    p.add_argument("--rows", type=int, default=None, help="rows (decode_sweep: 9/12/16/20)")
    p.add_argument("--no-sweep", action="store_true")
    p.add_argument("--no-e2e", action="store_true")
    p.add_argument("--no-cpu", action="store_true")
    p.add_argument("--no-spread", action="store_true",
                   help="skip the 5-run spread and the no-overlap figure (profiling runs)")
    p.add_argument("--prefill-banks", type=int, default=92,
                   help="distinct weight banks of a prefill chunk (one per layer)")
    p.add_argument("--no-overlap", action="store_true",
                   help="read each step's hidden rows only after the previous step has finished")
    return p.parse_args()


# ---------------------------------------------------------------- plumbing

def whole_job_rows_per_s(world: int, steps: int, rows: int, ms: float) -> float:
    """Rows of every replica over the slowest replica's time (ms, max over
    ranks): each of the `world` ranks runs `steps` layers of `rows` rows."""
    return world * steps * rows / (ms / 1e3)


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return {k: float(d[k]) for k in FALLBACK_PEAKS}, "measured"
    except (OSError, KeyError, ValueError):
        return dict(FALLBACK_PEAKS), "fallback"


_COMMENT = re.compile(r"//[^\n]*|/\*.*?\*/", re.S)


def kernel_source_sha(kernel: str):
    """Hash of a kernel's sources with comments and whitespace removed, so
    that an edit of a comment keeps a recorded ncu figure valid and any change
    of the code voids it."""
    h = hashlib.sha256()
    for rel in KERNEL_SOURCES[kernel]:
        with open(os.path.join(ROOT, rel), encoding="utf-8") as f:
            code = _COMMENT.sub(" ", f.read())
        h.update(" ".join(code.split()).encode())
    return h.hexdigest()[:16]


def recorded_traffic(kernel: str, workload: str):
    """DRAM bytes per launch from a committed ncu summary, if it was taken
    on the current kernel sources; else None."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            d = json.load(f)
        e = d[f"{kernel}:{workload}"]
        if e.get("source_sha") != kernel_source_sha(kernel):
            return None
        return float(e["dram_bytes_per_launch"])
    except (OSError, KeyError, ValueError):
        return None


class ClockSampler:
    """nvidia-smi clock / throttle samples while the timed region runs."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    NAMES = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100", "-i", str(self.index)],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except OSError:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.time(), line.strip()))

    def stop(self, t0: float, t1: float):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        sm, smax, reasons, n_in = [], [], set(), 0
        for t, line in self.lines:
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 8:
                continue
            inside = t0 - 0.15 <= t <= t1 + 0.15
            if not inside:
                continue
            n_in += 1
            try:
                sm.append(float(parts[0]))
                smax.append(float(parts[1]))
            except ValueError:
                pass
            for name, v in zip(self.NAMES, parts[4:8]):
                if v.lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": n_in}


class NvmlClocks:
    """In-process, read-only NVML queries of the SM clock and the active
    clock-event reasons, polled every millisecond: nvidia-smi samples every
    100 ms at best, which can miss a timed region of a fraction of a
    millisecond altogether.  Nothing is set; unavailable NVML reads as None."""

    REASONS = {0x8: "hw_slowdown", 0x40: "hw_thermal_slowdown", 0x20: "sw_thermal_slowdown",
               0x4: "sw_power_cap"}

    def __init__(self, index: int):
        import ctypes
        self.ok = False
        self.samples = []
        try:
            lib = ctypes.CDLL("libnvidia-ml.so.1")
            if lib.nvmlInit_v2() != 0:
                return
            h = ctypes.c_void_p()
            if lib.nvmlDeviceGetHandleByIndex_v2(ctypes.c_uint(index), ctypes.byref(h)) != 0:
                return
            self.lib, self.h, self.ct = lib, h, ctypes
            fn = getattr(lib, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
                getattr(lib, "nvmlDeviceGetCurrentClocksThrottleReasons")
            self.reasons_fn = fn
            self.max_mhz = self._clock(lib.nvmlDeviceGetMaxClockInfo)
            self.ok = True
        except (OSError, AttributeError):
            self.ok = False

    def _clock(self, fn):
        v = self.ct.c_uint()
        return v.value if fn(self.h, self.ct.c_uint(1), self.ct.byref(v)) == 0 else None  # 1 = SM

    def read(self):
        if not self.ok:
            return None
        r = self.ct.c_ulonglong()
        reasons = r.value if self.reasons_fn(self.h, self.ct.byref(r)) == 0 else 0
        return (self._clock(self.lib.nvmlDeviceGetClockInfo), reasons)

    def start(self):
        self.stop_flag = False
        if self.ok:
            self.samples.append(self.read())
            self.thread = threading.Thread(target=self._poll, daemon=True)
            self.thread.start()
        return self

    def _poll(self):
        while not self.stop_flag:
            self.samples.append(self.read())
            time.sleep(0.001)

    def stop(self):
        self.stop_flag = True
        if not self.ok:
            return None
        self.thread.join(timeout=1)
        self.samples.append(self.read())
        sm = [s[0] for s in self.samples if s and s[0]]
        bits = 0
        for s in self.samples:
            if s:
                bits |= s[1]
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": self.max_mhz,
                "reasons": sorted(n for b, n in self.REASONS.items() if bits & b),
                "samples": len(self.samples), "source": "NVML (in process, read only), 1 ms poll"}


# ----------------------------------------------------------- distributed

class Dist:
    def __init__(self):
        import torch
        self.torch = torch
        self.world = int(os.environ.get("WORLD_SIZE", "1"))
        self.rank = int(os.environ.get("RANK", "0"))
        self.local = int(os.environ.get("LOCAL_RANK", "0"))
        if self.world > 1:
            import torch.distributed as dist
            os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
            backend = "nccl" if torch.cuda.is_available() else "gloo"
            if backend == "nccl":
                torch.cuda.set_device(self.local)
            dist.init_process_group(backend)
            self.dist = dist
        else:
            self.dist = None

    def barrier(self):
        if self.dist is not None:
            self.dist.barrier()

    def max(self, x: float) -> float:
        if self.dist is None:
            return x
        t = self.torch.tensor([x], dtype=self.torch.float64,
                              device=f"cuda:{self.local}" if self.torch.cuda.is_available() else "cpu")
        self.dist.all_reduce(t, op=self.dist.ReduceOp.MAX)
        return float(t.item())

    def close(self):
        if self.dist is not None:
            self.dist.destroy_process_group()


# ------------------------------------------------------------- watchdog

class Watchdog:
    """Ends the process if a GPU phase runs far past any plausible time, so
    that a kernel that never completes cannot hold the GPU: the process exits
    with status 3 and a message naming the phase (its context is torn down)."""

    def __init__(self, limit_s: float = 180.0):
        self.limit = limit_s
        self.phase = None
        self.t0 = 0.0
        threading.Thread(target=self._watch, daemon=True).start()

    def _watch(self):
        while True:
            time.sleep(1.0)
            ph = self.phase
            if ph is not None and time.time() - self.t0 > self.limit:
                sys.stderr.write(f"bench: GPU phase '{ph}' exceeded {self.limit:.0f} s; exiting\n")
                sys.stderr.flush()
                os._exit(3)

    def __call__(self, phase: str):
        wd = self

        class _Phase:
            def __enter__(self):
                wd.phase, wd.t0 = phase, time.time()

            def __exit__(self, *exc):
                wd.phase = None
        return _Phase()


WATCHDOG = None


def guarded(phase: str):
    global WATCHDOG
    if WATCHDOG is None:
        WATCHDOG = Watchdog()
    return WATCHDOG(phase)


# ---------------------------------------------------------------- our arm

class RouteBench:
    def __init__(self, device: int):
        import numpy as np
        import torch
        import latent_projection_top_gb300 as route
        import synth
        self.np, self.torch, self.route, self.synth = np, torch, route, synth
        self.dev = f"cuda:{device}"
        self.device = device
        self.banks = {}

    def d(self, bits):
        np, torch = self.np, self.torch
        return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).to(self.dev).view(
            torch.bfloat16)

    def weight_banks(self, kind: str, n: int):
        key = (kind, n)
        if key not in self.banks:
            wk = self.synth.WORKLOADS["decode_r8" if kind == "decode" else "prefill_r3072"]
            out = []
            for b in range(n):
                wl, wr = self.synth.weight_bank(wk.seed, b)
                out.append((self.d(wl), self.d(wr)))
            self.banks[key] = out
        return self.banks[key]

    def hidden(self, workload: str, rows: int, nb: int):
        # at most 8 distinct hidden inputs: the weights (distinct per layer) are
        # what defeats L2; the hidden values do not change the timing
        wk = self.synth.WORKLOADS[workload]
        distinct = [self.d(wk.hidden(b, rows)) for b in range(min(wk.banks, 8, nb))]
        return [distinct[b % len(distinct)] for b in range(nb)]

    def outputs(self, rows: int):
        torch, route = self.torch, self.route
        return (torch.empty((rows, route.N_LATENT), dtype=torch.bfloat16, device=self.dev),
                torch.empty((rows, route.N_EXPERTS), dtype=torch.float32, device=self.dev),
                torch.empty((rows, route.TOPK), dtype=torch.int32, device=self.dev),
                torch.empty((rows, route.TOPK), dtype=torch.float32, device=self.dev))

    def make_steps(self, workload: str, rows: int, nbanks: int, gemm_only: bool = False,
                   overlap: bool = False, sumsq: bool = False, ksplit: bool = False,
                   producer: str | None = None):
        """Closures, one per bank, each enqueuing one layer's route step.

        producer="before": each step is preceded on the stream by a plain
        copy kernel (torch's) that writes the step's hidden rows from a
        source buffer -- a stand-in for the norm that precedes routing in a
        model; it triggers no programmatic launch, so the route step starts
        only once it has finished.  producer="alone": the copies only (their
        time is subtracted from the pair's)."""
        route = self.route
        mode = route.DECODE if workload.startswith("decode") else route.PREFILL
        plan = route.Plan(mode, rows, self.device)
        if overlap:
            route.route_set_overlap(plan, True)
        if ksplit:
            route.route_set_latent_ksplit(plan, True)
        banks = self.weight_banks("decode" if mode == route.DECODE else "prefill", nbanks)
        hs = self.hidden(workload, rows, nbanks)
        outs = [self.outputs(rows) for _ in range(nbanks)]
        steps = []
        for (wl, wr), h, o in zip(banks, hs, outs):
            if producer is not None:
                dst = self.torch.empty_like(h)
                if producer == "alone":
                    steps.append(lambda s, h=h, dst=dst: dst.copy_(h))
                else:
                    def step(s, h=h, dst=dst, wl=wl, wr=wr, o=o):
                        dst.copy_(h)
                        route.route_step(plan, dst, wl, wr, *o, stream=s)
                    steps.append(step)
            elif gemm_only:
                steps.append(lambda s, h=h, wl=wl, wr=wr, o=o:
                             route.latent_router_forward(plan, h, wl, wr, o[0], o[1], stream=s))
            elif sumsq:
                ss = self.torch.empty((rows,), dtype=self.torch.float32, device=self.dev)
                steps.append(lambda s, h=h, wl=wl, wr=wr, o=o, ss=ss:
                             route.route_step_sumsq(plan, h, wl, wr, *o, ss, stream=s))
            else:
                steps.append(lambda s, h=h, wl=wl, wr=wr, o=o:
                             route.route_step(plan, h, wl, wr, *o, stream=s))
        launches = 1 if (mode == route.PREFILL and gemm_only) else 2
        return plan, steps, launches

    def spread(self, steps, runs: int = 5, replays: int = 200, graph_len: int = GRAPH_LEN,
               warm_replays: int = 20, dist=None):
        """The timing method of the decode page ("Kimi K3.1 recipe ...",
        commit message): `runs` runs of `replays` replays of a graph of
        `graph_len` layer steps.  Returns the per-step time of each run (us)."""
        with guarded(f"spread {runs}x{replays}"):
            torch = self.torch
            s = torch.cuda.Stream(device=self.dev)
            s.wait_stream(torch.cuda.current_stream(self.dev))
            g = self.graph(steps, graph_len, 0, s)
            torch.cuda.synchronize(self.dev)
            with torch.cuda.stream(s):
                for _ in range(warm_replays):
                    g.replay()
            torch.cuda.synchronize(self.dev)
            out = []
            for _ in range(runs):
                if dist is not None:
                    dist.barrier()
                e0 = torch.cuda.Event(enable_timing=True)
                e1 = torch.cuda.Event(enable_timing=True)
                with torch.cuda.stream(s):
                    e0.record(s)
                    for _ in range(replays):
                        g.replay()
                    e1.record(s)
                e1.synchronize()
                ms = e0.elapsed_time(e1)
                if dist is not None:
                    ms = dist.max(ms)
                out.append(ms * 1e3 / (replays * graph_len))
            del g
            return out

    def ab(self, steps_a, steps_b, rounds: int = 5, replays: int = 200,
           graph_len: int = GRAPH_LEN, warm_replays: int = 20, dist=None):
        """Interleaved A/B: one graph of `graph_len` steps for each side, then
        `rounds` times a run of `replays` replays of each side, A first in
        even rounds and B first in odd ones, so that both sides see the same
        drift of the part's power state.  Returns the per-step times of each
        side's runs (us)."""
        with guarded(f"a/b {rounds}x{replays}"):
            torch = self.torch
            s = torch.cuda.Stream(device=self.dev)
            s.wait_stream(torch.cuda.current_stream(self.dev))
            graphs = [self.graph(st, graph_len, 0, s) for st in (steps_a, steps_b)]
            torch.cuda.synchronize(self.dev)
            with torch.cuda.stream(s):
                for g in graphs:
                    for _ in range(warm_replays):
                        g.replay()
            torch.cuda.synchronize(self.dev)
            out = ([], [])
            for r in range(rounds):
                for side in ((0, 1) if r % 2 == 0 else (1, 0)):
                    g = graphs[side]
                    if dist is not None:
                        dist.barrier()
                    e0 = torch.cuda.Event(enable_timing=True)
                    e1 = torch.cuda.Event(enable_timing=True)
                    with torch.cuda.stream(s):
                        e0.record(s)
                        for _ in range(replays):
                            g.replay()
                        e1.record(s)
                    e1.synchronize()
                    ms = e0.elapsed_time(e1)
                    if dist is not None:
                        ms = dist.max(ms)
                    out[side].append(ms * 1e3 / (replays * graph_len))
            del graphs
            return out

    def per_layer_us(self, steps, dist):
        """One chunk launched eagerly with an event between consecutive layers:
        per-layer time (median, min, max) and the chunk total, from the second
        of two passes."""
        torch = self.torch
        s = torch.cuda.Stream(device=self.dev)
        ev = [torch.cuda.Event(enable_timing=True) for _ in range(len(steps) + 1)]
        for _ in range(2):
            torch.cuda.synchronize(self.dev)
            with torch.cuda.stream(s):
                ev[0].record(s)
                for i, st in enumerate(steps):
                    st(s)
                    ev[i + 1].record(s)
            ev[-1].synchronize()
        per = sorted(ev[i].elapsed_time(ev[i + 1]) * 1e3 for i in range(len(steps)))
        total = ev[0].elapsed_time(ev[-1]) * 1e3
        return {"layers": len(steps), "median": round(per[len(per) // 2], 3),
                "min": round(per[0], 3), "max": round(per[-1], 3),
                "chunk_us": round(dist.max(total), 3),
                "note": "eager launches with an event between layers"}

    def graph(self, steps, n: int, offset: int, stream):
        torch = self.torch
        g = torch.cuda.CUDAGraph()
        with torch.cuda.stream(stream):
            with torch.cuda.graph(g, stream=stream):
                for i in range(n):
                    steps[(offset + i) % len(steps)](stream)
        return g

    def run(self, steps, k: int, warmup: int, dist=None, sampler_index=None, graph_len=GRAPH_LEN):
        """Time exactly k steps (after `warmup` steps) as graph replays.
        Returns (elapsed_ms, clocks)."""
        with guarded(f"{k} timed steps"):
            return self._run(steps, k, warmup, dist, sampler_index, graph_len)

    def _run(self, steps, k, warmup, dist, sampler_index, graph_len):
        torch = self.torch
        s = torch.cuda.Stream(device=self.dev)
        s.wait_stream(torch.cuda.current_stream(self.dev))
        L = min(graph_len, max(k, 1))
        g_full = self.graph(steps, L, 0, s)
        rem = k % L
        g_rem = self.graph(steps, rem, 0, s) if rem else None
        # the timed graphs go to the device now: a graph's first replay would
        # otherwise carry the upload (0.1-0.3 us a layer of a 20-layer graph)
        self.graphs_uploaded = upload_graphs([g for g in (g_full, g_rem) if g is not None], s)
        w_full, w_rem = divmod(warmup, L)
        g_wrem = self.graph(steps, w_rem, 0, s) if w_rem else None
        torch.cuda.synchronize(self.dev)
        sampler = ClockSampler(sampler_index).start() if sampler_index is not None else None
        nvml = NvmlClocks(sampler_index) if sampler_index is not None else None
        with torch.cuda.stream(s):
            for _ in range(w_full):
                g_full.replay()
            if g_wrem is not None:
                g_wrem.replay()
        torch.cuda.synchronize(self.dev)
        if dist is not None:
            dist.barrier()
        torch.cuda.synchronize(self.dev)
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        if nvml is not None:
            nvml.start()
        t0 = time.time()
        with torch.cuda.stream(s):
            # A short device-side wait ahead of the start event keeps the GPU
            # busy while the host submits the timed graphs, so that the host's
            # submission latency is not timed as device time (it is in e2e).
            torch.cuda._sleep(SPIN_CYCLES)
            e0.record(s)
            for _ in range(k // L):
                g_full.replay()
            if g_rem is not None:
                g_rem.replay()
            e1.record(s)
        e1.synchronize()
        torch.cuda.synchronize(self.dev)
        t1 = time.time()
        nv = nvml.stop() if nvml is not None else None
        if dist is not None:
            dist.barrier()
        clocks = sampler.stop(t0, t1) if sampler is not None else None
        if clocks is not None and not clocks.get("samples") and nv is not None:
            # a timed region shorter than nvidia-smi's sampling interval
            nv["note"] = (f"timed region {1e3 * (t1 - t0):.2f} ms is shorter than nvidia-smi's "
                          "100 ms sampling interval; clocks from in-process NVML reads")
            clocks = nv
        return e0.elapsed_time(e1), clocks

    def e2e(self, workload: str, rows: int, k: int, dist):
        """route_step_host: H2D hidden + step + D2H results, every step."""
        with guarded("e2e"):
            return self._e2e(workload, rows, k, dist)

    def _e2e(self, workload: str, rows: int, k: int, dist):
        torch, route, np = self.torch, self.route, self.np
        mode = route.DECODE if workload.startswith("decode") else route.PREFILL
        wl, wr = self.weight_banks("decode" if mode == route.DECODE else "prefill", 8)[0]
        wk = self.synth.WORKLOADS[workload]
        def host_bufs(b):
            return (torch.from_numpy(wk.hidden(b, rows).view(np.int16)).view(torch.bfloat16)
                    .pin_memory(),
                    torch.empty((rows, route.N_LATENT), dtype=torch.bfloat16).pin_memory(),
                    torch.empty((rows, route.N_EXPERTS), dtype=torch.float32).pin_memory(),
                    torch.empty((rows, route.TOPK), dtype=torch.int32).pin_memory(),
                    torch.empty((rows, route.TOPK), dtype=torch.float32).pin_memory())

        (hid, lat, lg, ids, w), others = host_bufs(0), [host_bufs(b) for b in (1, 2)]
        s = torch.cuda.Stream(device=self.dev)
        with route.Plan(mode, rows, self.device) as plan:
            # route_step_host checks its tensors on every call; HostStep (the
            # serving-loop form of the same call) checks them once and launches
            # a captured graph; HostSteps on buffers of their own keep several
            # batches in flight through launch / wait
            step = route.HostStep(plan, hid, wl, wr, lat, lg, ids, w, stream=s)
            ring = [step] + [route.HostStep(plan, o[0], wl, wr, *o[1:], stream=s) for o in others]
            for _ in range(5):
                route.route_step_host(plan, hid, wl, wr, lat, lg, ids, w, stream=s)
                for st in ring:
                    st()
                    st.launch()
                    st.wait()
            dist.barrier()
            torch.cuda.synchronize(self.dev)
            t0 = time.perf_counter()
            for _ in range(k):
                route.route_step_host(plan, hid, wl, wr, lat, lg, ids, w, stream=s)
            torch.cuda.synchronize(self.dev)
            t_checked = time.perf_counter() - t0
            dist.barrier()
            torch.cuda.synchronize(self.dev)
            t0 = time.perf_counter()
            for _ in range(k):
                step()
            torch.cuda.synchronize(self.dev)
            t_sync = time.perf_counter() - t0
            by_depth = {}
            for depth in (2, 3):
                dist.barrier()
                torch.cuda.synchronize(self.dev)
                t0 = time.perf_counter()
                for i in range(depth - 1):
                    ring[i].launch()
                for i in range(k):
                    if i + depth - 1 < k:
                        ring[(i + depth - 1) % depth].launch()
                    ring[i % depth].wait()
                torch.cuda.synchronize(self.dev)
                by_depth[depth] = dist.max(time.perf_counter() - t0)
            dist.barrier()
        t_sync, t_checked = dist.max(t_sync), dist.max(t_checked)
        depth = E2E_DEPTH
        t = by_depth[depth]
        h2d = hid.numel() * 2
        d2h = lat.numel() * 2 + lg.numel() * 4 + ids.numel() * 4 + w.numel() * 4
        return {"value": round(dist.world * k * rows / t, 1), "unit": "rows/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "us_per_step": round(t / k * 1e6, 3), "steps": k, "in_flight": depth,
                "path": f"{depth} HostSteps of one plan on one stream, each on its own pinned "
                        f"host buffers, launched and waited for in turn with {depth} batches in "
                        "flight (launch C, wait A, launch A, wait B, ...); every step reads its "
                        "hidden rows from host memory and its wait returns once that step's "
                        "results are in its host buffers",
                "us_per_step_by_in_flight": {"1 (HostStep call, CUDA graph)":
                                             round(t_sync / k * 1e6, 3),
                                             **{str(d): round(v / k * 1e6, 3)
                                                for d, v in by_depth.items()}},
                "us_per_step_route_step_host": round(t_checked / k * 1e6, 3)}


def upload_graphs(graphs, stream) -> bool:
    """cudaGraphUpload of each instantiated graph on `stream`, through the CUDA
    runtime this process already uses (found in its memory map), so that the
    graphs' first replays do not include the upload.  Executes nothing.
    Returns False (and uploads nothing) where that runtime or the graphs'
    handles are not reachable."""
    import ctypes
    path = None
    try:
        with open("/proc/self/maps") as f:
            for line in f:
                name = line.split()[-1] if line.strip() else ""
                if os.path.basename(name).startswith("libcudart.so"):
                    path = name
                    break
    except OSError:
        return False
    if path is None or not all(hasattr(g, "raw_cuda_graph_exec") for g in graphs):
        return False
    rt = ctypes.CDLL(path)
    for g in graphs:
        rc = rt.cudaGraphUpload(ctypes.c_void_p(g.raw_cuda_graph_exec()),
                                ctypes.c_void_p(stream.cuda_stream))
        if rc != 0:
            return False
    return True


def oracle_rows_per_s(workload: str, rows: int, budget_s: float = 10.0):
    """The oracle, as it stands, on whole layer steps of the workload until the
    budget is spent (at least one step).  Single-threaded."""
    import oracle
    import synth
    wk = synth.WORKLOADS[workload]
    hid = wk.hidden(0, rows)
    wl, wr = synth.weight_bank(wk.seed, 0)
    oracle.build()
    n, t0 = 0, time.perf_counter()
    while True:
        _, lg, _, _ = oracle.latent_router(hid, wl, wr)
        oracle.topk(lg)
        n += 1
        if time.perf_counter() - t0 >= budget_s:
            break
    t = time.perf_counter() - t0
    return {"value": round(n * rows / t, 3), "unit": "rows/s", "cores": 1,
            "host_cores": os.cpu_count(), "kind": "oracle",
            "sample": f"{n} full layer step(s) of {rows} rows of {workload} (bank 0), "
                      f"{t:.1f} s, single-threaded float64 C"}


def oracle_rows_per_s_all_cores(workload: str, rows: int, budget_s: float = 10.0):
    """A second CPU figure, labelled apart from `cpu_baseline`: the same
    single-threaded oracle run as independent whole layer steps on every host
    core at once (one thread per core; each ctypes call releases the
    interpreter lock), rows of all threads over the wall time."""
    import oracle
    import synth
    from concurrent.futures import ThreadPoolExecutor
    wk = synth.WORKLOADS[workload]
    hid = wk.hidden(0, rows)
    wl, wr = synth.weight_bank(wk.seed, 0)
    oracle.build()
    cores = os.cpu_count() or 1
    t0 = time.perf_counter()

    def worker(_):
        n = 0
        while True:
            _, lg, _, _ = oracle.latent_router(hid, wl, wr)
            oracle.topk(lg)
            n += 1
            if time.perf_counter() - t0 >= budget_s:
                return n

    with ThreadPoolExecutor(cores) as ex:
        steps = sum(ex.map(worker, range(cores)))
    t = time.perf_counter() - t0
    return {"value": round(steps * rows / t, 3), "unit": "rows/s", "cores": cores,
            "kind": "oracle, all cores",
            "sample": f"{steps} full layer steps of {rows} rows of {workload} (bank 0) on "
                      f"{cores} threads, {t:.1f} s wall"}


def main_ours(args):
    import torch
    dist = Dist()
    dev = dist.local if torch.cuda.is_available() else 0
    torch.cuda.set_device(dev)
    peaks, peak_src = load_peaks()
    rb = RouteBench(dev)
    wk = args.workload
    rows = args.rows or (8 if wk == "decode_r8" else 1 if wk == "decode_r1" else 20 if
                         wk == "decode_sweep" else 1024 if wk == "prefill_r1024" else 3072)
    decode = wk.startswith("decode")
    nbanks = 8 if decode else args.prefill_banks
    overlap = not args.no_overlap
    plan, steps, launches = rb.make_steps(wk, rows, nbanks, overlap=overlap)
    ms, clocks = rb.run(steps, args.steps, args.warmup, dist, sampler_index=dev)
    rb.route.route_device_status(plan)  # raises if any launch hit a bounded-wait timeout
    ms = dist.max(ms)
    step_s = ms / 1e3 / args.steps
    value = whole_job_rows_per_s(dist.world, args.steps, rows, ms)

    # roofline of the dominant kernel
    if decode:
        # The step is the weight-streaming kernel plus the small kernel that
        # finishes the split-K sums and runs the top-16; the whole step time
        # (average launch period over the timed region) is charged to the
        # streaming kernel, which is conservative.
        kern_s = step_s
        algo = WEIGHT_BYTES + rows * ROW_BYTES
        achieved = algo / kern_s / 1e9
        roof = {"bound": "hbm",
                "kernel": f"decode_stream_kernel<{16 if rows <= 16 else 32}> (+ decode_finish_kernel)",
                "achieved": round(achieved, 1), "peak": peaks["hbm_gbs"], "unit": "GB/s",
                "frac": round(achieved / peaks["hbm_gbs"], 4),
                "peak_source": f"{peak_src} hbm_gbs",
                "algorithmic_bytes_per_launch": algo,
                "traffic": recorded_traffic("decode_stream_kernel", wk)}
    else:
        p2, gsteps, _ = rb.make_steps(wk, rows, nbanks, gemm_only=True, overlap=overlap)
        gms, _ = rb.run(gsteps, 92, 3 * 92, dist)
        kern_s = dist.max(gms) / 1e3 / 92
        flop = FLOP_PER_ROW * rows
        achieved = flop / kern_s / 1e12
        roof = {"bound": "tensor", "kernel": "prefill_pair_kernel (prefill GEMM, CTA pairs)",
                "achieved": round(achieved, 1), "peak": peaks["bf16_tflops"], "unit": "TFLOP/s",
                "frac": round(achieved / peaks["bf16_tflops"], 4),
                "peak_source": f"{peak_src} bf16_tflops (burst)",
                "algorithmic_flop_per_launch": flop,
                "traffic": recorded_traffic("prefill_pair_kernel", wk)}
        p2.close()

    out = {"metric": METRIC, "value": round(value, 1), "unit": "rows/s", "n_gpus": dist.world,
           "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(step_s * 1e3, 6),
           "us_per_layer": round(step_s * 1e6, 3),
           "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
           "data": "synthetic (seeded N(0,1) hidden, N(0,1/7168) weights; no real Kimi weights here)",
           "config": {"workload": wk, "rows": rows, "weight_banks": nbanks,
                      "layers_per_graph": GRAPH_LEN,
                      "overlap": overlap,
                      "timing": "CUDA events on the launching stream around exactly the timed steps; "
                                "a ~0.1 ms device-side wait precedes the start event so that the "
                                "host's graph submission is not timed",
                      "l2": f"inputs larger than L2: {nbanks} distinct weight banks x 64.2 MB, "
                            "one per layer, cycled",
                      "parallelism": f"replicas x{dist.world} (no sharding, no collectives)"},
           "roofline": roof, "clocks": clocks, "gpu_launches": launches * args.steps,
           "timed_graphs_uploaded": bool(getattr(rb, "graphs_uploaded", False))}

    # the same configuration timed the decode page's way: median (min, max)
    # over 5 runs of many graph replays (steady state, no pipeline fill)
    sp = DECODE_SPREAD if decode else PREFILL_SPREAD
    if not args.no_spread:
        out["spread"] = dict(summarise(rb.spread(steps, dist=dist, **sp)), method=SPREAD_METHOD)
    if overlap and not args.no_spread:
        # the same workload with each step held behind the previous one's tail
        p3, s3, _ = rb.make_steps(wk, rows, nbanks, overlap=False)
        sm = summarise(rb.spread(s3, dist=dist, **sp))
        rb.route.route_device_status(p3)
        t3 = sm["median"] / 1e6
        out["without_overlap"] = {"us_per_layer": sm["median"], "us_spread": sm,
                                  "rows_per_s": round(dist.world * rows / t3, 1)}
        if decode:
            algo = WEIGHT_BYTES + rows * ROW_BYTES
            out["without_overlap"]["hbm_frac"] = round(algo / t3 / 1e9 / peaks["hbm_gbs"], 4)
        p3.close()
    if not args.no_e2e:
        out["e2e"] = rb.e2e(wk, rows, min(args.steps, 4096), dist)
    if not args.no_sweep:
        smp = ClockSampler(dev).start()
        t0 = time.time()
        out["sweep"] = sweep(rb, dist, peaks, args)
        out["sweep_clocks"] = smp.stop(t0, time.time())
        out["sweep_method"] = SPREAD_METHOD
    if dist.rank == 0 and dist.world == 1 and not args.no_cpu:
        out["cpu_baseline"] = oracle_rows_per_s(wk, rows)
        out["cpu_all_cores"] = oracle_rows_per_s_all_cores(wk, rows)
    plan.close()
    if dist.rank == 0:
        print(json.dumps(out), flush=True)
    dist.close()


def summarise(us):
    """median / min / max of per-run per-layer times (us)."""
    srt = sorted(us)
    return {"median": round(statistics.median(srt), 3), "min": round(srt[0], 3),
            "max": round(srt[-1], 3), "runs": len(srt)}


# batches in flight in the e2e figure: three keep the device busy (two leave
# it idle between steps, a step's own latency being about 25 us)
E2E_DEPTH = 3
DECODE_SPREAD = dict(runs=5, replays=200, graph_len=GRAPH_LEN)
PREFILL_SPREAD = dict(runs=5, replays=10, graph_len=92)
SPREAD_METHOD = ("per-layer us: median (min, max) over 5 runs; decode: 200 replays of a "
                 "64-layer graph per run, prefill: 10 replays of a 92-layer graph per run")


def sweep(rb, dist, peaks, args):
    res = []
    for wk, rows in [("decode_r1", 1), ("decode_r8", 8), ("decode_sweep", 9), ("decode_sweep", 12),
                     ("decode_sweep", 16), ("decode_sweep", 20)]:
        algo = WEIGHT_BYTES + rows * ROW_BYTES
        entry = {"workload": wk, "rows": rows, "bound": "hbm"}
        for ov in (True, False):
            plan, steps, _ = rb.make_steps(wk, rows, 8, overlap=ov)
            sm = summarise(rb.spread(steps, dist=dist, **DECODE_SPREAD))
            rb.route.route_device_status(plan)
            plan.close()
            t = sm["median"] / 1e6
            sfx = "" if ov else "_without_overlap"
            entry.update({"us_per_layer" + sfx: sm["median"], "us_spread" + sfx: sm,
                          "rows_per_s" + sfx: round(rows / t, 1),
                          "achieved_gbs" + sfx: round(algo / t / 1e9, 1),
                          "frac" + sfx: round(algo / t / 1e9 / peaks["hbm_gbs"], 4)})
        res.append(entry)
    # the regime of a model: each route step follows a kernel that writes its
    # hidden rows and does not trigger a programmatic launch (overlap off)
    for wk, rows in [("decode_r1", 1), ("decode_r8", 8), ("decode_sweep", 12),
                     ("decode_sweep", 16), ("decode_sweep", 20)]:
        algo = WEIGHT_BYTES + rows * ROW_BYTES
        plan, pair, _ = rb.make_steps(wk, rows, 8, producer="before")
        us_pair = summarise(rb.spread(pair, dist=dist, **DECODE_SPREAD))
        rb.route.route_device_status(plan)
        plan.close()
        p2, alone, _ = rb.make_steps(wk, rows, 8, producer="alone")
        us_prod = summarise(rb.spread(alone, dist=dist, **DECODE_SPREAD))
        p2.close()
        t = (us_pair["median"] - us_prod["median"]) / 1e6
        res.append({"workload": wk, "rows": rows, "bound": "hbm",
                    "regime": "after a producer kernel (copy of the hidden rows, no programmatic "
                              "launch trigger), overlap off",
                    "us_per_layer": round(t * 1e6, 3), "rows_per_s": round(rows / t, 1),
                    "frac": round(algo / t / 1e9 / peaks["hbm_gbs"], 4),
                    "us_producer_and_step": us_pair, "us_producer_alone": us_prod,
                    "note": "us_per_layer = median(producer + step) - median(producer alone)"})
    for wk, rows in [("prefill_r1024", 1024), ("prefill_r3072", 3072)]:
        nb = args.prefill_banks
        flop = FLOP_PER_ROW * rows
        e = {"workload": wk, "rows": rows, "bound": "tensor", "weight_banks": nb,
             "note": "burst: one 92-layer graph after two (against the burst bf16 peak); "
                     "sustained: 5 runs of 10 such graphs back to back, under the power cap "
                     "(against the sustained peak)"}
        # the plain mode first (always valid); overlap beside it: for prefill
        # its gain varies from box to box and has been negative
        for ov in (False, True):
            plan, steps, _ = rb.make_steps(wk, rows, nb, overlap=ov)
            p2, gsteps, _ = rb.make_steps(wk, rows, nb, gemm_only=True, overlap=ov)
            tb = dist.max(rb.run(steps, 92, 2 * 92, dist, graph_len=92)[0]) / 1e3 / 92
            tgb = dist.max(rb.run(gsteps, 92, 2 * 92, dist, graph_len=92)[0]) / 1e3 / 92
            st = summarise(rb.spread(steps, dist=dist, **PREFILL_SPREAD))
            gm = summarise(rb.spread(gsteps, dist=dist, **PREFILL_SPREAD))
            rb.route.route_device_status(plan)
            rb.route.route_device_status(p2)
            t, tg = st["median"] / 1e6, gm["median"] / 1e6
            sfx = "_with_overlap" if ov else ""
            e.update({"us_per_layer" + sfx: round(tb * 1e6, 3),
                      "chunk_ms_92_layers" + sfx: round(tb * 92 * 1e3, 3),
                      "rows_per_s" + sfx: round(rows / tb, 1),
                      "gemm_us" + sfx: round(tgb * 1e6, 3),
                      "gemm_tflops" + sfx: round(flop / tgb / 1e12, 1),
                      "frac" + sfx: round(flop / tgb / 1e12 / peaks["bf16_tflops"], 4),
                      "us_per_layer_sustained" + sfx: st["median"], "us_spread_sustained" + sfx: st,
                      "gemm_us_sustained" + sfx: gm["median"], "gemm_us_spread_sustained" + sfx: gm,
                      "frac_sustained" + sfx: round(
                          flop / tg / 1e12 / peaks["bf16_tflops_sustained"], 4)})
            if rows == 3072 and not ov:
                e["per_layer_us"] = rb.per_layer_us(steps[:92], dist)
            plan.close()
            p2.close()
        res.append(e)
    # the route step that also returns each latent row's sum of squares, and
    # the step with the general path's K-split latent arithmetic
    # each timed against the plain route step in interleaved runs (A/B), so
    # that the difference is not the drift of the part's power state
    variants = [dict(sumsq=True), dict(ksplit=True)]
    for var in variants:
        for wk, rows in [("decode_r8", 8), ("decode_sweep", 20), ("prefill_r1024", 1024),
                         ("prefill_r3072", 3072)]:
            decode = wk.startswith("decode")
            nb = 8 if decode else args.prefill_banks
            ov = decode
            base, bsteps, _ = rb.make_steps(wk, rows, nb, overlap=ov)
            plan, steps, _ = rb.make_steps(wk, rows, nb, overlap=ov, **var)
            kw = dict(DECODE_SPREAD if decode else PREFILL_SPREAD)
            kw["rounds"] = kw.pop("runs")
            ua, ub = rb.ab(bsteps, steps, dist=dist, **kw)
            rb.route.route_device_status(base)
            rb.route.route_device_status(plan)
            base.close()
            plan.close()
            sm = summarise(ub)
            t = sm["median"] / 1e6
            e = {"workload": wk, "rows": rows, "overlap": ov, "us_per_layer": sm["median"],
                 "us_spread": sm, "rows_per_s": round(rows / t, 1),
                 "us_plain_step_interleaved": summarise(ua),
                 "us_added": summarise([b - a for a, b in zip(ua, ub)]),
                 "ab": "runs alternate with the plain route step's (ABBA order), same "
                       "workload and mode; us_added = per-round difference (median, min, max)"}
            if var.get("sumsq"):
                e["call"] = "route_step_sumsq"
            else:
                e["latent"] = "k-split (8 BF16 partials)"
            if decode:
                algo = WEIGHT_BYTES + rows * (ROW_BYTES + (4 if var.get("sumsq") else 0))
                e.update({"bound": "hbm", "frac": round(algo / t / 1e9 / peaks["hbm_gbs"], 4)})
            res.append(e)
    res += eager_sweep(rb, dist)
    res += shard_sweep(rb, dist)
    return res


def eager_sweep(rb, dist, n: int = 4096):
    """Decode layers launched eagerly (no graph), 8 weight banks cycled,
    overlap on: through route_step (tensors checked on every call) and
    through Step objects (checked once).  Per-layer time = CUDA events around
    the n launches; the host's enqueue time per layer beside it."""
    torch, route = rb.torch, rb.route
    out = []
    rows, wk = 8, "decode_r8"
    for how in ("route_step", "Step"):
        with guarded(f"eager {how}"):
            plan = route.Plan(route.DECODE, rows, rb.device)
            route.route_set_overlap(plan, True)
            banks = rb.weight_banks("decode", 8)
            hs = rb.hidden(wk, rows, 8)
            outs = [rb.outputs(rows) for _ in range(8)]
            s = torch.cuda.Stream(device=rb.dev)
            s.wait_stream(torch.cuda.current_stream(rb.dev))
            if how == "Step":
                calls = [route.Step(plan, h, wl, wr, *o, stream=s)
                         for (wl, wr), h, o in zip(banks, hs, outs)]
            else:
                calls = [(lambda h=h, wl=wl, wr=wr, o=o:
                          route.route_step(plan, h, wl, wr, *o, stream=s))
                         for (wl, wr), h, o in zip(banks, hs, outs)]
            for i in range(64):
                calls[i % 8]()
            torch.cuda.synchronize(rb.dev)
            dist.barrier()
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            with torch.cuda.stream(s):
                e0.record(s)
                t0 = time.perf_counter()
                for i in range(n):
                    calls[i % 8]()
                t1 = time.perf_counter()
                e1.record(s)
            e1.synchronize()
            us = dist.max(e0.elapsed_time(e1)) * 1e3 / n
            route.route_device_status(plan)
            plan.close()
        out.append({"workload": wk, "rows": rows, "overlap": True, "launch": f"eager, {how}",
                    "us_per_layer": round(us, 3), "host_us_per_layer": round((t1 - t0) / n * 1e6, 3),
                    "layers": n})
    return out


def shard_sweep(rb, dist):
    """One rank's share of a column-sharded decode step (shard 0 of W; its
    weights cycled over 32 banks so that they do not stay in L2), both
    regimes.  The exchange between ranks is not part of it."""
    route, torch = rb.route, rb.torch
    banks = rb.weight_banks("decode", 32)
    res = []
    for W, rows in ((8, 8), (16, 8)):
        NL, NE = route.shard_columns(W)
        sb = [(wl[:, :NL].contiguous(), wr[:, :NE].contiguous()) for wl, wr in banks]
        h = rb.hidden("decode_r8", rows, 1)[0]
        outs = [(torch.empty((rows, NL), dtype=torch.bfloat16, device=rb.dev),
                 torch.empty((rows, NE), dtype=torch.float32, device=rb.dev),
                 torch.empty((rows, TOPK), dtype=torch.int32, device=rb.dev),
                 torch.empty((rows, TOPK), dtype=torch.float32, device=rb.dev)) for _ in sb]
        for ov in (True, False):
            plan = route.ShardPlan(rows, 0, W, rb.device)
            route.route_set_overlap(plan, ov)
            steps = [lambda s, wl=wl, wr=wr, o=o: route.route_shard_step(plan, h, wl, wr, *o, stream=s)
                     for (wl, wr), o in zip(sb, outs)]
            sm = summarise(rb.spread(steps, dist=dist, runs=3, replays=100))
            route.route_device_status(plan)
            byt = (NL + NE) * K_HIDDEN * 2
            res.append({"workload": f"column shard 0 of {W} (decode_r8 rows)", "rows": rows,
                        "overlap": ov, "shard_latent_cols": NL, "shard_experts": NE,
                        "us_per_layer": sm["median"], "us_spread": sm, "grid": plan.grid,
                        "weight_bytes": byt, "achieved_gbs": round(byt / sm["median"] / 1e3, 1),
                        "note": "one rank's compute on one GPU; the candidate exchange is not timed"})
            plan.close()
        del sb
    return res


# --------------------------------------------------------- reference arm

def main_reference(args):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return  # the oracle runs once, on rank 0
    import numpy as np
    import oracle
    import synth
    wk = synth.WORKLOADS[args.workload]
    rows = args.rows or max(wk.rows) if args.workload != "decode_sweep" else (args.rows or 20)
    if args.workload == "decode_r8" and args.rows is None:
        rows = 8
    hid = wk.hidden(0, rows)
    wl, wr = synth.weight_bank(wk.seed, 0)
    oracle.build()
    full_cols = N_LATENT + N_EXPERTS
    # size the per-step sample so that warm-up + timed steps take ~120 s
    per_row_col_s = 0.23 / full_cols  # rough single-core cost of one row x one column
    budget = 120.0 / max(1, args.steps + args.warmup)
    cols = int(max(1, min(full_cols, budget / (per_row_col_s * rows))))
    W = np.ascontiguousarray(np.concatenate([wl, wr], axis=1)[:, :cols])
    _, lg_full, _, _ = oracle.latent_router(hid, wl[:, :1].copy(), wr)
    for _ in range(args.warmup):
        oracle.dot64(hid, W)
        oracle.topk(lg_full)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle.dot64(hid, W)
        oracle.topk(lg_full)
    t = time.perf_counter() - t0
    frac = cols / full_cols
    value = rows * frac * args.steps / t
    sample = (f"{rows} rows x {cols} of {full_cols} weight columns (float64 dot products) + "
              f"top-16 of {rows} rows per step, scaled to a full layer")
    out = {"metric": METRIC, "impl": "reference", "value": round(value, 4), "unit": "rows/s",
           "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
           "ms_per_step": round(t / args.steps * 1e3, 6),
           "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
           "data": "synthetic", "config": {"workload": args.workload, "rows": rows},
           "cpu_baseline": {"value": round(value, 4), "unit": "rows/s", "cores": 1,
                            "kind": "oracle", "sample": sample},
           "e2e": {"value": round(value, 4), "unit": "rows/s", "h2d_bytes_per_step": 0,
                   "d2h_bytes_per_step": 0}}
    print(json.dumps(out), flush=True)


if __name__ == "__main__":
    a = parse_args()
    if a.impl == "reference":
        main_reference(a)
    else:
        main_ours(a)
