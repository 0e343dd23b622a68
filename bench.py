"""Benchmark of the top-k index selector.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload decode_1m_masked]

A step is one tks_topk_indices call over one batch of the named workload
(batch=1, N=1048576 fp32 logits, k=2048 by default).  Steps read rotating
copies of the input whose total size exceeds twice the L2 cache, so every
step reads its logits from HBM.  K steps are captured in CUDA graphs and
timed with CUDA events on the launching stream.

Prints one JSON line.  `value` is microseconds per row over the whole job
(lower is better).  `roofline` compares the one-pass algorithmic read bytes
per launch with the measured HBM copy bandwidth.  `e2e` repeats the
measurement through the public API with host buffers (pinned host -> device
copy of the logits, the call, device -> host copy of the indices) inside the
timed region.  `cpu_baseline` times the CPU oracle on a bounded sample.

--impl reference times the CPU oracle itself (the only reference that exists
for this method) on the same workload, as a bounded sample per step.

With torchrun (--gpus N > 1) every rank runs an independent replica on its
own GPU (rows are independent; there is no data exchange); the time is the
maximum over ranks and `value` divides it by the rows all ranks processed.
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

import numpy as np  # noqa: E402

import workloads as W  # noqa: E402

METRIC = "TopK-select µs/row and HBM GB/s (batch=1, N=128K–1M, k=2048) vs roofline"
UNIT = "us/row"
# every file that is compiled into libtks.so
KERNEL_SOURCES = [
    os.path.join(ROOT, "sparse_attention_topk_gb300", "csrc", name)
    for name in ("tks_select.cu", "tks_select512.cu", "tks_order.cu", "tks_device.cuh",
                 "tks_kernel.cuh", "tks_internal.h")
] + [os.path.join(ROOT, "include", "tks.h")]
PROFILES = os.path.join(ROOT, "profiles")
FALLBACK_HBM_GBS = 6800.0


def kernel_source_hash() -> str:
    h = hashlib.sha256()
    for p in KERNEL_SOURCES:
        with open(p, "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def measured_peaks() -> tuple[float, str]:
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, "fallback"


def recorded_traffic(workload: str) -> float | None:
    """DRAM bytes per launch from the committed ncu summary, if it was taken on
    the current kernel source (else None)."""
    path = os.path.join(PROFILES, f"tks_select_{workload}.md")
    try:
        text = open(path).read()
    except OSError:
        return None
    m_hash = re.search(r"kernel source hash:\s*`?([0-9a-f]{16})", text)
    m_tr = re.search(r"dram bytes per launch:\s*([0-9]+)", text)
    if not (m_hash and m_tr) or m_hash.group(1) != kernel_source_hash():
        return None
    return float(m_tr.group(1))


# ---------------------------------------------------------------------------
# distributed helpers (replicas only)
# ---------------------------------------------------------------------------

def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def init_dist(world: int, backend: str):
    if world <= 1:
        return None
    import torch.distributed as dist
    os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
    dist.init_process_group(backend=backend)
    return dist


def barrier(dist, device=None):
    if dist is not None:
        if device is not None and dist.get_backend() == "nccl":
            dist.barrier(device_ids=[device.index])
        else:
            dist.barrier()


def max_over_ranks(dist, value: float, device=None) -> float:
    """Largest value over all ranks (the job's time is its slowest rank's)."""
    if dist is None:
        return value
    import torch
    t = torch.tensor([value], dtype=torch.float64,
                     device=device if (device is not None and dist.get_backend() == "nccl") else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ---------------------------------------------------------------------------
# clocks sampled during the timed region
# ---------------------------------------------------------------------------

class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id: str):
        self.gpu = gpu_id
        self.proc = None
        self.lines: list[str] = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self._t = threading.Thread(target=self._read, daemon=True)
            self._t.start()
            time.sleep(0.3)
        except OSError:
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
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self) -> dict:
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                mx = float(parts[1])
            except ValueError:
                continue
            for name, flag in zip(names, parts[4:8]):
                if flag.lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": mx,
                "reasons": sorted(reasons), "samples": len(sm)}


# ---------------------------------------------------------------------------
# the CPU oracle as baseline
# ---------------------------------------------------------------------------

class OneCore:
    """Pins the calling thread to one host core for the duration (Linux), so
    the single-threaded oracle timing does not migrate between cores."""

    def __enter__(self):
        self.saved = None
        try:
            self.saved = os.sched_getaffinity(0)
            os.sched_setaffinity(0, {max(self.saved)})
        except (AttributeError, OSError):
            self.saved = None
        return self

    def __exit__(self, *exc):
        if self.saved is not None:
            os.sched_setaffinity(0, self.saved)


def cpu_oracle_time(w, budget_s: float = 10.0) -> dict:
    """The oracle (single thread, pinned to one core) on whole rows of the
    workload, repeated until about budget_s of CPU work; microseconds per row."""
    with OneCore():
        return _cpu_oracle_time(w, budget_s)


def _cpu_oracle_time(w, budget_s: float) -> dict:
    import oracle
    lib = oracle.load()
    times = []
    t_start = time.perf_counter()
    r = 0
    while True:
        row = r % w.batch
        L = int(w.row_len[row])
        t0 = time.perf_counter()
        oracle.topk_indices(w.values[row:row + 1, :L], w.k, None, w.dtype, lib=lib)
        times.append(time.perf_counter() - t0)
        r += 1
        if time.perf_counter() - t_start > budget_s and r >= 3:
            break
    lo, hi = int(w.row_len.min()), int(w.row_len.max())
    lens = f"N={lo}" if lo == hi else f"rows taken in turn, N={lo}..{hi}"
    return {"value": round(statistics.median(times) * 1e6, 3), "unit": UNIT, "cores": 1,
            "kind": "oracle",
            "sample": f"{r} whole rows of {w.name} ({lens}), median of single-thread "
                      f"C oracle runs pinned to one of {os.cpu_count()} host cores"}


def reference_arm(args, w):
    """--impl reference: the CPU oracle per step on a bounded prefix sample of
    the row, scaled to a whole row by n log n (one pinned core)."""
    with OneCore():
        _reference_arm(args, w)


def _reference_arm(args, w):
    import oracle
    lib = oracle.load()
    steps, warmup = args.steps, args.warmup
    budget = 90.0  # seconds for the whole run
    N = int(w.row_len[0])
    # one full-row timing fixes the per-element cost, then size the sample
    t0 = time.perf_counter()
    oracle.topk_indices(w.values[0:1, :N], w.k, None, w.dtype, lib=lib)
    full = time.perf_counter() - t0
    per = budget / max(1, steps + warmup)
    n = N
    while n > 4096 and full * (n * math.log2(n)) / (N * math.log2(N)) > per:
        n //= 2
    kk = min(w.k, max(1, n // 8))
    sample = w.values[0:1, :n]
    for _ in range(warmup):
        oracle.topk_indices(sample, kk, None, w.dtype, lib=lib)
    t0 = time.perf_counter()
    for _ in range(steps):
        oracle.topk_indices(sample, kk, None, w.dtype, lib=lib)
    dt = time.perf_counter() - t0
    scale = (N * math.log2(N)) / (n * math.log2(n))
    us_row = dt / steps * 1e6 * scale
    line = {
        "impl": "reference", "metric": METRIC, "value": round(us_row, 3), "unit": UNIT,
        "n_gpus": args.gpus, "steps": steps, "warmup": warmup, "ms_per_step": round(us_row / 1e3, 6),
        "higher_is_better": False, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic",
        "config": {"workload": w.name, "batch": w.batch, "n": N, "k": w.k},
        "cpu_baseline": {"value": round(us_row, 3), "unit": UNIT, "cores": 1, "kind": "oracle",
                         "sample": f"first {n} positions of the row, k={kk}, per step; "
                                   f"scaled to N={N} by n*log2(n) (merge sort)"},
        "e2e": {"value": round(us_row, 3), "unit": UNIT, "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)



# ---------------------------------------------------------------------------
# device timing of one workload
# ---------------------------------------------------------------------------

class DeviceTiming:
    """Back-to-back and cold timing of tks_topk_indices on one workload.

    Steps read rotating copies of the input whose total size exceeds 2.5x the
    L2 cache; L2 is flushed just before the timed region (then three calls on
    a spare input bring the kernel's code and workspace back) and a copy is
    read again only after all the others, so every step reads its logits
    from HBM.
    Steps are captured in CUDA graphs of up to 512 calls (graph j reads the
    copies from j * 512 on); the warm-up replays each graph the timed region
    uses at least once (a graph's first launch uploads it), and a short spin
    kernel ahead of the first event keeps the device busy while the host
    submits the graphs, so the timed region holds the K calls and nothing else.
    """

    SPIN_CYCLES = 2_000_000  # ~1 ms at the GB300's clocks: longer than the host needs to submit

    def __init__(self, tks, torch, w, stream, device, l2):
        self.tks, self.torch, self.w, self.stream, self.device, self.l2 = tks, torch, w, stream, device, l2
        x_host = torch.from_numpy(w.values.copy())
        if w.dtype == W.BF16:
            x_host = x_host.view(torch.bfloat16)
        self.x_host = x_host
        self.nbytes = x_host.numel() * x_host.element_size()
        self.ncopies = max(2, math.ceil(2.5 * l2 / self.nbytes))
        self.base = x_host.to(device)
        self.copies = [self.base.clone() for _ in range(self.ncopies)]
        self.spare = self.base.clone()  # read only between the L2 flush and the timed region
        self.full_rows = bool(np.all(w.row_len == w.row_stride))
        self.rl = None if self.full_rows else torch.from_numpy(w.row_len.copy()).to(device)
        self.out = torch.empty((w.batch, w.k), dtype=torch.int32, device=device)
        self.flush = torch.empty(2 * l2 // 4 + 1, dtype=torch.float32, device=device)
        self.graphs = {}
        self.G = 1
        with torch.cuda.stream(stream):
            self.call(0)  # sets up the stream's workspace before capture
        stream.synchronize()
        st = tks.device_status(stream)
        if st != tks.TKS_OK:
            raise RuntimeError(f"device status after set-up: {tks.status_string(st)}")

    def call(self, i):
        self.tks.topk_indices(self.copies[i % self.ncopies], self.w.k, row_len=self.rl, out=self.out,
                              stream=self.stream)

    def graph_calls(self, steps):
        self.G = min(512, max(1, steps))
        return self.G

    def _keys(self, k):
        """(calls, first copy) of the graphs that run k steps."""
        n_off = 1 if self.ncopies <= self.G else math.ceil(self.ncopies / self.G)
        keys, j = [], 0
        while k > 0:
            n = min(self.G, k)
            keys.append((n, (j % n_off) * self.G))
            k -= n
            j += 1
        return keys

    def _graph(self, key):
        if key not in self.graphs:
            torch = self.torch
            n, off = key
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=self.stream):
                for i in range(n):
                    self.call(off + i)
            self.graphs[key] = g
        return self.graphs[key]

    def run(self, k):
        with self.torch.cuda.stream(self.stream):
            for key in self._keys(k):
                self._graph(key).replay()

    def warm(self, steps, warmup):
        """Replays every graph that run(steps) uses once, then more steps up to
        `warmup` in all; returns the number of warm-up steps made."""
        done = 0
        with self.torch.cuda.stream(self.stream):
            for key in dict.fromkeys(self._keys(steps)):
                self._graph(key).replay()
                done += key[0]
        if done < max(3, warmup):
            self.run(max(3, warmup) - done)
            done = max(3, warmup)
        self.stream.synchronize()
        return done

    def timed(self, steps):
        """Device time of exactly `steps` calls (ms), CUDA events on the stream."""
        torch = self.torch
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(self.stream):
            self.flush.fill_(1.0)
            # the flush also evicted the kernel's code and workspace: three calls
            # on an input outside the rotation bring those back
            for _ in range(3):
                self.tks.topk_indices(self.spare, self.w.k, row_len=self.rl, out=self.out,
                                      stream=self.stream)
            torch.cuda._sleep(self.SPIN_CYCLES)
            e0.record(self.stream)
        self.run(steps)
        e1.record(self.stream)
        e1.synchronize()
        return e0.elapsed_time(e1)

    def cold(self, calls=16, pairs=7):
        """Latency of one call that follows another kernel with L2 flushed.

        One CUDA graph holds `calls` x [a write of twice the L2 size, one call],
        another the same writes alone; they are replayed in turn, and the
        difference over `calls` (median over `pairs` replays of each) is the
        call's latency after the write kernel, its launch included.  Beside it,
        `event_us_per_call`: one host-launched call between two CUDA events
        after the write (median over `calls`), which adds the gap the event
        record leaves before the launch; event timestamps on this GPU advance
        in steps of about 1 us, so single calls read on that grid."""
        torch = self.torch
        flush = self.flush
        g_call, g_flush = torch.cuda.CUDAGraph(), torch.cuda.CUDAGraph()
        with torch.cuda.graph(g_call, stream=self.stream):
            for i in range(calls):
                flush.fill_(float(i))
                self.call(i)
        with torch.cuda.graph(g_flush, stream=self.stream):
            for i in range(calls):
                flush.fill_(float(i))

        def replay_ms(g):
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            with torch.cuda.stream(self.stream):
                torch.cuda._sleep(self.SPIN_CYCLES)
                e0.record(self.stream)
                g.replay()
                e1.record(self.stream)
            e1.synchronize()
            return e0.elapsed_time(e1)

        replay_ms(g_call)  # a graph's first launch uploads it
        replay_ms(g_flush)
        diffs = []
        for _ in range(pairs):
            a = replay_ms(g_call)
            b = replay_ms(g_flush)
            diffs.append((a - b) * 1e3 / calls)
        del g_call, g_flush

        event_us = []
        for i in range(calls):
            c0 = torch.cuda.Event(enable_timing=True)
            c1 = torch.cuda.Event(enable_timing=True)
            with torch.cuda.stream(self.stream):
                flush.fill_(float(i))
                c0.record(self.stream)
                self.call(i)
                c1.record(self.stream)
            c1.synchronize()
            event_us.append(c0.elapsed_time(c1) * 1e3)
        st = self.tks.device_status(self.stream)
        if st != self.tks.TKS_OK:
            raise RuntimeError(f"device status after the cold calls: {self.tks.status_string(st)}")
        return {"us_per_call": round(statistics.median(diffs), 3),
                "spread": [round(min(diffs), 3), round(max(diffs), 3)],
                "calls": calls, "pairs": pairs,
                "how": f"graph of {calls} x [{2 * self.l2 // 2**20} MiB write, call] minus graph of "
                       f"the writes alone, over {calls}; median of {pairs} pairs of replays",
                "event_us_per_call": round(statistics.median(event_us), 3)}

    def release(self):
        self.graphs.clear()
        self.copies = []
        self.spare = None
        self.flush = None


def other_configs(tks, torch, args, main_name, stream, device, l2, peak, gpu_id):
    """µs per row, GB/s, fraction of peak and cold latency of the other named
    workloads, each timed like the headline (back to back in CUDA graphs over
    rotating copies larger than L2) and checked against the oracle."""
    import oracle
    res = {}
    steps = max(3, min(args.steps, 2048))
    with ClockSampler(gpu_id) as clk:
        for name in W.NAMED:
            if name == main_name:
                continue
            w = W.named(name)
            dev = DeviceTiming(tks, torch, w, stream, device, l2)
            dev.graph_calls(steps)
            dev.warm(steps, args.warmup)
            ms = dev.timed(steps)
            st = tks.device_status(stream)
            if st != tks.TKS_OK:
                raise RuntimeError(f"{name}: device status {tks.status_string(st)}")
            got = dev.out.cpu().numpy()
            want = oracle.topk_workload(w)
            ok = all(np.array_equal(np.sort(got[r, :min(w.k, int(w.row_len[r]))]),
                                    want[r, :min(w.k, int(w.row_len[r]))]) for r in range(w.batch))
            if not ok:
                raise RuntimeError(f"{name}: GPU result differs from the oracle")
            us_call = ms * 1e3 / steps
            cold = dev.cold()
            gbs = w.algorithmic_bytes / (us_call * 1e-6) / 1e9
            res[name] = {"us_per_row": round(us_call / w.batch, 4), "us_per_call": round(us_call, 3),
                         "batch": w.batch, "n": int(w.row_stride), "k": w.k, "logits": w.dtype,
                         "gbs": round(gbs, 1), "frac": round(gbs / peak, 5), "steps": steps,
                         "cold_us_per_call": cold["us_per_call"],
                         "cold_event_us_per_call": cold["event_us_per_call"], "matches_oracle": True,
                         "plan": dict(zip(("blocks_per_row", "grid"),
                                          tks.plan(w.batch, w.row_stride, w.k, 0 if w.dtype == W.F32 else 1)))}
            dev.release()
            del dev
            torch.cuda.empty_cache()
    res["clocks"] = clk.summary()
    return res

# ---------------------------------------------------------------------------
# the GPU arm
# ---------------------------------------------------------------------------

def gpu_arm(args, w, dist, rank, world, device):
    import torch

    import sparse_attention_topk_gb300 as tks

    tks.load()
    if args.hist_variant == "aggregated":
        # the measurement build: warp-aggregated first-round adds
        from sparse_attention_topk_gb300 import _build
        tks.use(_build.build(hist_aggregate=True))
    torch.cuda.set_device(device)
    stream = torch.cuda.Stream(device)
    props = torch.cuda.get_device_properties(device)
    l2 = int(getattr(props, "L2_cache_size", 126 * 2**20))
    dev = DeviceTiming(tks, torch, w, stream, device, l2)
    x_host, nbytes, ncopies = dev.x_host, dev.nbytes, dev.ncopies
    copies, out, rl, full_rows, base = dev.copies, dev.out, dev.rl, dev.full_rows, dev.base
    G = dev.graph_calls(args.steps)
    warm_steps = dev.warm(args.steps, args.warmup)

    # timed: exactly K steps
    barrier(dist, device)
    torch.cuda.synchronize(device)
    uuid = getattr(props, "uuid", None)
    gpu_id = f"GPU-{uuid}" if uuid is not None and not str(uuid).startswith("GPU-") else str(uuid or device.index)
    with ClockSampler(gpu_id) as clk:
        ms = dev.timed(args.steps)
    torch.cuda.synchronize(device)
    barrier(dist, device)
    st = tks.device_status(stream)
    if st != tks.TKS_OK:
        raise RuntimeError(f"device status after the timed run: {tks.status_string(st)}")
    ms_max = max_over_ranks(dist, ms, device)
    call = dev.call

    rows_total = args.steps * w.batch * world
    us_per_row = ms_max * 1e3 / rows_total
    launch_us = ms * 1e3 / args.steps  # one kernel launch per step on this rank
    alg_bytes = w.algorithmic_bytes
    achieved = alg_bytes / (launch_us * 1e-6) / 1e9
    peak, peak_src = measured_peaks()

    cold = dev.cold()

    # a read-only streaming probe for context: a sum over 1 GiB
    probe = torch.ones(2**28, dtype=torch.float32, device=device)
    probe_ms = []
    for _ in range(7):
        p0 = torch.cuda.Event(enable_timing=True)
        p1 = torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            p0.record(stream)
            probe.sum()
            p1.record(stream)
        p1.synchronize()
        probe_ms.append(p0.elapsed_time(p1))
    del probe
    read_probe_gbs = 2**30 / (statistics.median(probe_ms) * 1e-3) / 1e9

    # end to end through the public API with host buffers: page-locked logits
    # in, indices out, the kernel reading the logits across the host link and
    # writing the indices back (tks_topk_indices_host); rotating host copies
    # larger than L2 so no step is served from a cache
    k_e2e = min(args.steps, 2000)
    ncop_host = max(2, math.ceil(2.5 * l2 / nbytes))
    x_pins = [x_host.pin_memory() for _ in range(ncop_host)]
    rl_pin = None if full_rows else torch.from_numpy(w.row_len.copy()).pin_memory()
    out_pin = torch.empty((w.batch, w.k), dtype=torch.int32).pin_memory()

    def host_call(i):
        tks.topk_indices(x_pins[i % ncop_host], w.k, row_len=rl_pin, out=out_pin, stream=stream)

    def timed_e2e(step):
        for i in range(3):
            step(i)
        stream.synchronize()
        barrier(dist, device)
        f0 = torch.cuda.Event(enable_timing=True)
        f1 = torch.cuda.Event(enable_timing=True)
        f0.record(stream)
        for i in range(k_e2e):
            step(i)
        f1.record(stream)
        f1.synchronize()
        barrier(dist, device)
        return max_over_ranks(dist, f0.elapsed_time(f1), device) * 1e3 / (k_e2e * w.batch * world)

    e2e_us_row = timed_e2e(host_call)
    st = tks.device_status(stream)
    if st != tks.TKS_OK:
        raise RuntimeError(f"device status after the host-buffer run: {tks.status_string(st)}")
    host_result = out_pin.numpy().copy()

    # the same through device buffers with copy-engine copies on either side
    x_dev = torch.empty_like(base)

    def staged_call(i):
        with torch.cuda.stream(stream):
            x_dev.copy_(x_pins[i % ncop_host], non_blocking=True)
            tks.topk_indices(x_dev, w.k, row_len=rl, out=out, stream=stream)
            out_pin.copy_(out, non_blocking=True)

    staged_us_row = timed_e2e(staged_call)
    del x_pins

    # the rank-ordered variant (tks_topk_indices_sorted: selection + on-chip
    # ordering kernel), same rotating inputs, outside the headline timing
    sorted_line = None
    if w.k <= tks.TKS_SORTED_K_MAX:
        out_s = torch.empty((w.batch, w.k), dtype=torch.int32, device=device)

        def call_sorted(i):
            tks.topk_indices(copies[i % ncopies], w.k, row_len=rl, out=out_s, stream=stream,
                             sorted=True)

        with torch.cuda.stream(stream):
            call_sorted(0)
        stream.synchronize()
        gs = torch.cuda.CUDAGraph()
        with torch.cuda.graph(gs, stream=stream):
            for i in range(G):
                call_sorted(i)
        reps = max(1, min(args.steps, 4096) // G)
        with torch.cuda.stream(stream):
            gs.replay()
        stream.synchronize()
        s0 = torch.cuda.Event(enable_timing=True)
        s1 = torch.cuda.Event(enable_timing=True)
        s0.record(stream)
        with torch.cuda.stream(stream):
            for _ in range(reps):
                gs.replay()
        s1.record(stream)
        s1.synchronize()
        st = tks.device_status(stream)
        if st != tks.TKS_OK:
            raise RuntimeError(f"device status after the sorted run: {tks.status_string(st)}")
        sorted_us_row = s0.elapsed_time(s1) * 1e3 / (reps * G * w.batch)
        sorted_line = {"value": round(sorted_us_row, 4), "unit": UNIT, "steps": reps * G,
                       "launches_per_step": 2, "what": "tks_topk_indices_sorted (rank order)"}
        if rank == 0:
            import oracle
            if not np.array_equal(out_s.cpu().numpy(), oracle.topk_workload(w, ordered=True)):
                raise RuntimeError("sorted GPU result differs from the oracle's rank order")

    # the results of the last steps are correct (cheap spot check on rank 0)
    if rank == 0:
        import oracle
        want = oracle.topk_workload(w)
        for what, res in (("host-buffer", host_result), ("staged", out_pin.numpy())):
            for r in range(w.batch):
                take = min(w.k, int(w.row_len[r]))
                if not (np.array_equal(np.sort(res[r, :take]), want[r, :take])
                        and np.all(res[r, take:] == -1)):
                    raise RuntimeError(f"{what} GPU result differs from the oracle in row {r}")

    if rank != 0:
        return
    line = {
        "metric": METRIC, "value": round(us_per_row, 4), "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": warm_steps,
        "ms_per_step": round(ms_max / args.steps, 6), "higher_is_better": False,
        "scaling": "weak", "vs_baseline": None, "dtype": "u32",
        "data": "synthetic",
        "config": {
            "workload": w.name, "batch": w.batch, "n": int(w.row_stride), "k": w.k,
            "logits": w.dtype, "row_len": "full rows" if full_rows else "ragged (device row_len)",
            "l2": f"inputs larger than L2: {ncopies} rotating copies of {nbytes} B "
                  f"({ncopies * nbytes / 2**20:.0f} MiB > 2x {l2 / 2**20:.0f} MiB L2)",
            "graph": f"{G} calls per CUDA graph; warm-up replays every timed graph first; a "
                     f"spin kernel ahead of the first event hides the graph's submission",
            "value_is": "back to back: calls queued one after another on one stream, the next "
                        "call's blocks resident while this call finishes (programmatic dependent "
                        "launch); `cold` is one call right after a kernel that flushed L2 "
                        "(graph difference, launch included)",
            "parallelism": f"replicas x{world}",
            "first_round_histogram": "plain shared-memory adds" if args.hist_variant == "plain"
                                     else "warp-aggregated adds (measurement build)",
            "plan": dict(zip(("blocks_per_row", "grid"), tks.plan(w.batch, w.row_stride, w.k,
                                                                  0 if w.dtype == W.F32 else 1))),
        },
        "roofline": {
            "bound": "hbm", "achieved": round(achieved, 2), "peak": peak, "unit": "GB/s",
            "frac": round(achieved / peak, 5), "peak_source": peak_src,
            "algorithmic_bytes_per_launch": alg_bytes,
            "traffic": recorded_traffic(w.name),
            "frac_of_nominal_8000": round(achieved / 8000.0, 5),
            "read_probe": {"gbs": round(read_probe_gbs, 1), "frac": round(achieved / read_probe_gbs, 5),
                           "what": "torch sum over a 1 GiB fp32 buffer (library kernel, read only)"},
        },
        "cold": cold,
        "latency": {"back_to_back_us_per_call": round(ms_max * 1e3 / args.steps, 3),
                    "cold_us_per_call": cold["us_per_call"],
                    "cold_event_us_per_call": cold["event_us_per_call"]},
        "gpu_launches": args.steps,
        "e2e": {"value": round(e2e_us_row, 4), "unit": UNIT,
                "h2d_bytes_per_step": int(alg_bytes + (0 if full_rows else 4 * w.batch)),
                "d2h_bytes_per_step": int(w.batch * w.k * 4), "steps": k_e2e,
                "via": "tks_topk_indices_host: page-locked host logits read by the kernel, "
                       f"indices written to page-locked host memory; {ncop_host} rotating host copies",
                "staged_copies": {"value": round(staged_us_row, 4), "unit": UNIT,
                                  "via": "cudaMemcpyAsync of the logits in, tks_topk_indices on "
                                         "device buffers, cudaMemcpyAsync of the indices out",
                                  "h2d_bytes_per_step": int(nbytes)}},
        "clocks": clk.summary(),
    }
    if sorted_line is not None:
        line["sorted"] = sorted_line
    if world == 1 and not args.no_configs:
        line["configs"] = other_configs(tks, torch, args, w.name, stream, device, l2, peak, gpu_id)
    if rank == 0 and world == 1:  # (the CPU baseline is taken at N=1 only)
        line["cpu_baseline"] = cpu_oracle_time(w, budget_s=args.cpu_budget)
    print(json.dumps(line), flush=True)


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=40000)
    ap.add_argument("--warmup", type=int, default=2000)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="decode_1m_masked", choices=sorted(W.NAMED) + sorted(W.EXTRA))
    ap.add_argument("--hist-variant", choices=["plain", "aggregated"], default="plain",
                    help="aggregated: the measurement build whose first-round histogram "
                         "uses warp-aggregated (match_any) adds")
    ap.add_argument("--no-configs", action="store_true",
                    help="skip the timing of the other named workloads")
    ap.add_argument("--cpu-budget", type=float, default=10.0,
                    help="seconds of CPU oracle work for cpu_baseline")
    args = ap.parse_args(argv)
    world, rank, local = dist_env()
    w = W.named(args.workload)
    if args.impl == "reference":
        if rank == 0:
            reference_arm(args, w)
        return 0
    import torch
    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA device (the CPU oracle alone: --impl reference)")
    device = torch.device("cuda", local)
    dist = init_dist(world, "nccl")
    try:
        gpu_arm(args, w, dist, rank, world, device)
    finally:
        if dist is not None:
            dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
