"""Benchmark of the 1-bit Adam compression-stage step on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload bertL]
                    [--phase compressed|warmup|loco] [--W 8] [--impl reference]

One "step" is one pass of the whole hot path over one batch of synthetic gradients:
worker compress (momentum, error compensation, chunk RMS, sign packing), server average
and recompress, and the preconditioned update -- three kernels of the CUDA library,
called through its C ABI. The default workload is the BERT-Large-sized buffer (390
tensors fused, n = 333,496,320, W = 8 simulated workers, chunk = n/W, float16 grads).

Printed: one JSON line (rank 0) with the metric in params*workers/s, the step time, the
HBM roofline fraction of the dominant kernel (the worker pass) from CUDA events recorded
by the library on its launch stream during the timed region, the end-to-end rate through
the host-buffer entry point (gradients copied from pinned host memory every step, the
server's compressed message copied back) beside the same copy timed alone, sampled SM
clocks, and the CPU oracle timed on a bounded sample of the same workload. Every timed
loop cycles through three seeded per-step gradient draws made before timing starts.

With the default headline, a "workloads" object follows with the same measurements for
every other workload of the recipe, run one after another with memory freed between
them: the BERT-Base-sized step (masked, after its warm-up steps) and its warm-up step,
the 2^28-element sweep at W = 2, 4, 8, 16 (compressed and warm-up steps), the GPT-like
buffer's LoCo step and 1-bit step, and the tiny buffer (eager and from a CUDA graph).

With --gpus N > 1 (launched by torchrun) every rank runs an independent replica on its
own GPU (the path does not shard: the W workers already live on one GPU); the value is
the units of all ranks over the slowest rank's time. --impl reference times the CPU
oracle (the reference the kernels are checked against) on the same workload.
"""
import argparse
import hashlib
import json
import os
import platform
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "params*workers/sec and achieved HBM GB/s (% of roofline) per compressed step"
UNIT = "params*workers/s"


def parse():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=200)
    p.add_argument("--warmup", type=int, default=5)
    p.add_argument("--workload", default="bertL", choices=["tiny", "bertB", "bertL", "sweep", "loco"])
    p.add_argument("--phase", default="compressed", choices=["compressed", "warmup", "loco"])
    p.add_argument("--W", type=int, default=None, help="workers (sweep workload)")
    p.add_argument("--n", type=int, default=None,
                   help="elements (default: the workload's own size; smaller cases are for profiling)")
    p.add_argument("--chunk", type=int, default=None, help="elements per scale (default n/W)")
    p.add_argument("--impl", default="ours", choices=["ours", "reference"])
    p.add_argument("--e2e-steps", type=int, default=10)
    p.add_argument("--cpu-seconds", type=float, default=15.0)
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--graph", action="store_true",
                   help="time replays of one step captured in a CUDA graph (small, launch-bound buffers)")
    p.add_argument("--workloads", default="default",
                   help="after the headline line's own workload, also time the other workloads: "
                        "'default' (only when the headline is the default bertL step), 'all', 'none', "
                        "or comma-separated substrings of their keys (e.g. 'sweep_W16,loco')")
    return p.parse_args()


# ---- byte model (algorithmic bytes per element; the state read and written once) ----

def bytes_per_elem(phase, W, s_g, masked=False, bits=4):
    if phase == "compressed":
        return W * (s_g + 8.25) + 28.25 + (0.125 if masked else 0.0)
    if phase == "warmup":
        return W * s_g + 24.0
    return W * (s_g + 8.5) + W / 2 + 24.0           # LoCo, 4-bit


def worker_bytes_per_elem(W, s_g):
    """The worker pass: W rows of grads read, z read and written, sign bits written; m read."""
    return W * (s_g + 8.125) + 4.0


L2_BYTES = 129 * 1000 * 1000        # GB300 L2 (129 MB)


# the worker kernel's sources (its DRAM traffic record is valid only while they match)
WORKER_SOURCES = ["ob_worker.cuh", "ob_worker_f32.cu", "ob_worker_f16.cu", "ob_worker_bf16.cu",
                  "ob_common.cuh", "ob_tma.cuh", "ob_internal.h"]


def kernel_source_hash(files):
    h = hashlib.sha256()
    for f in files:
        h.update(open(os.path.join(ROOT, "error_compensated_bit_gb300", "csrc", f), "rb").read())
    return h.hexdigest()[:16]


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        pk = json.load(open(path))
        return float(pk["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


def load_traffic(workload, W, kernel_hash):
    """DRAM bytes per worker launch from a committed ncu capture, if it matches the kernel."""
    path = os.path.join(ROOT, "profiles", "worker_dram_traffic.json")
    if not os.path.exists(path):
        return None
    rec = json.load(open(path))
    if rec.get("kernel_hash") != kernel_hash:
        return None
    entry = rec.get("per_launch", {}).get("%s_W%d" % (workload, W))
    return entry


# ---- clocks during the timed region -----------------------------------------------

class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), "--query-gpu=" + self.FIELDS,
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except (OSError, FileNotFoundError):
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if not self.proc:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.t.join(timeout=2)
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx = float(parts[2])
            except ValueError:
                continue
            for nm, val in zip(names, parts[5:9]):
                if val.lower() == "active":
                    reasons.add(nm)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


# ---- distributed plumbing (timing only; the path itself has no collective) ---------

def dist_init(args):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("gloo")
        return dist, dist.get_rank(), world, int(os.environ.get("LOCAL_RANK", "0"))
    return None, 0, 1, 0


def max_over_ranks(dist, value):
    if dist is None:
        return value
    import torch
    t = torch.tensor([value], dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(dist):
    if dist is not None:
        dist.barrier()


# ---- CPU baseline / reference arm (the oracle on a bounded sample) ------------------

def oracle_sample_run(wl, phase, n_sample, seconds, min_steps=2, max_steps=None):
    """Time the oracle on the first n_sample elements of the workload's recipe.

    Returns (seconds per step, steps timed, sample description)."""
    import numpy as np
    import oracle as O
    from error_compensated_bit_gb300 import synth
    sw = synth.workload(wl.name, W=wl.W, n=n_sample)
    sw.n_real = n_sample - n_sample % (sw.W * 256)
    sw.chunk = 0
    n = sw.n
    ora = O.default()
    st = O.OracleState(n, sw.W, sw.C, x=synth.params(sw).numpy(), m=np.zeros(n),
                       v=synth.variance(sw).numpy(), b1=sw.b1, b2=sw.b2, eps=sw.eps, lr=sw.lr)
    if sw.zero_frac > 0 and phase == "compressed":
        st.mask = synth.mask(sw).numpy().astype(np.uint8)
    g = synth.to_numpy_grads(synth.grads(sw, 0))
    err = np.zeros((sw.W, n), np.float32)
    fn = {"compressed": lambda: ora.compressed_step(st, g),
          "warmup": lambda: ora.warmup_step(st, g),
          "loco": lambda: ora.loco_step(st, g, err, 0.9, 4)}[phase]
    fn()                                    # untimed first step (page-in)
    times = []
    t_end = time.perf_counter() + seconds
    while (len(times) < min_steps or time.perf_counter() < t_end) and (max_steps is None or len(times) < max_steps):
        t0 = time.perf_counter()
        fn()
        times.append(time.perf_counter() - t0)
    per = sum(times) / len(times)
    desc = ("%s recipe, first %d elements (n=%d, W=%d, chunk=n/W), %s grads, %d %s steps "
            "single-threaded on %s" % (wl.name, sw.n_real, n, sw.W, str(sw.grad_dtype).split(".")[-1],
                                       len(times), phase, platform.machine()))
    return per, len(times), n * sw.W, desc


def reference_arm(args, wl):
    dist, rank, world, _ = dist_init(args)
    if rank != 0:
        return 0
    # size the sample so that warmup + steps finish in about two minutes
    per_small, _, units_small, _ = oracle_sample_run(wl, args.phase, wl.W * 256 * 256, 1.0, 1, 3)
    per_unit = per_small / units_small
    budget = 120.0 / max(1, args.steps + args.warmup)
    n_sample = int(budget / per_unit / wl.W)
    n_sample = max(wl.W * 256 * 16, min(n_sample, 1 << 23))
    import numpy as np  # noqa: F401
    per, steps, units, desc = oracle_sample_run(wl, args.phase, n_sample, 0.0,
                                                min_steps=args.steps, max_steps=args.steps)
    value = units / per
    line = {"metric": METRIC, "value": value, "unit": UNIT, "impl": "reference",
            "n_gpus": args.gpus, "steps": steps, "warmup": args.warmup, "ms_per_step": per * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
            "data": "synthetic",
            "config": {"workload": workload_desc(wl, args.phase), "sample_elements": units // wl.W},
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": 1, "kind": "oracle",
                             "sample": desc},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line))
    return 0


def workload_desc(wl, phase):
    what = {"compressed": "1-bit compressed step", "warmup": "full-precision Adam warm-up step",
            "loco": "LoCo 4-bit step"}[phase]
    return "%s: %s, n=%d, W=%d, chunk=%d, %s grads" % (
        wl.name, what, wl.n, wl.W, wl.C, str(wl.grad_dtype).split(".")[-1])


# ---- the GPU arm ----------------------------------------------------------------------

KERNEL_OF_PHASE = {"compressed": "worker", "warmup": "warmup", "loco": "loco_quant"}
GRAD_BUFFERS = 3        # per-step gradient draws, cycled through in every timed loop


LOCO_ONE_PASS_MAX_CHUNK = 4096    # LoCo chunks up to this long: absmax and quantize in one pass


def dominant_kernel_bytes(phase, n, W, s_g, chunk=None):
    """Algorithmic bytes of one launch of the phase's dominant kernel."""
    if phase == "compressed":
        return n * worker_bytes_per_elem(W, s_g)
    if phase == "warmup":
        return n * (W * s_g + 24.0)
    if chunk is not None and chunk > LOCO_ONE_PASS_MAX_CHUNK:
        # LoCo, long chunks: quantize every row and take the Adam step in one pass
        # (g, e read and e written per row; x, m, v read and written; codes kept in registers)
        return n * (W * (s_g + 8.0) + 24.0)
    return n * W * (s_g + 8.5)                     # LoCo quantize: g, e read; e, codes written


class Run:
    """One workload's device state, set up, warmed and timed through the C ABI.

    Gradients for GRAD_BUFFERS steps (the recipe's seeded per-step draws) are drawn on the
    device before anything is timed, and step t uses draw t mod GRAD_BUFFERS."""

    def __init__(self, torch, ob, synth, dev, wl, phase):
        self.torch, self.ob, self.synth, self.dev, self.wl, self.phase = torch, ob, synth, dev, wl, phase
        n, W, C = wl.n, wl.W, wl.C
        self.masked = wl.zero_frac > 0 and phase == "compressed"
        self.ctx = ob.Context(n, W, C, wl.b1, wl.b2, wl.eps, wl.lr)
        self.x = synth.params(wl, dev)
        self.v = synth.variance(wl, dev)
        self.m = torch.zeros(n, dtype=torch.float32, device=dev)
        self.ew = torch.zeros(W, n, dtype=torch.float32, device=dev)
        self.es = torch.zeros(n, dtype=torch.float32, device=dev)
        self.ws = torch.empty(self.ctx.workspace_bytes(), dtype=torch.uint8, device=dev)
        self.ctx.workspace_init(self.ws)
        self.lws = None
        if phase == "loco":
            self.lws = torch.zeros(self.ctx.loco_workspace_bytes(4), dtype=torch.uint8, device=dev)
        self.stream = torch.cuda.current_stream(dev)
        # the BERT-Base recipe runs its warm-up Adam steps before the compressed ones
        self.grads = [synth.grads(wl, 1000 + t, dev) for t in range(GRAD_BUFFERS)]
        if phase == "compressed" and wl.warmup_steps:
            for t in range(wl.warmup_steps):
                self.ctx.warmup_step(self.grads[t % GRAD_BUFFERS], self.x, self.m, self.v, self.ws, self.stream)
        self.grads = [synth.grads(wl, t, dev, out=self.grads[t]) for t in range(GRAD_BUFFERS)]
        if self.masked:
            self.ctx.set_mask(synth.mask(wl, dev), self.ws)
        self.t = 0

    def step(self, stream=None):
        s = stream or self.stream
        g = self.grads[self.t % GRAD_BUFFERS]
        self.t += 1
        if self.phase == "compressed":
            self.ctx.compressed_step(g, self.x, self.m, self.v, self.ew, self.es, self.ws, s)
        elif self.phase == "warmup":
            self.ctx.warmup_step(g, self.x, self.m, self.v, self.ws, s)
        else:
            self.ctx.loco_step(g, self.x, self.m, self.v, self.ew, self.lws, 0.9, 4, s)

    def bytes_per_step(self):
        return self.wl.n * bytes_per_elem(self.phase, self.wl.W, self.wl.grad_bytes, self.masked)

    def measure(self, steps, warmup, graph=False, clocks=None, barrier_fn=None):
        """Warm up, then time `steps` steps with CUDA events on the launch stream."""
        torch, dev, ctx = self.torch, self.dev, self.ctx
        for _ in range(max(3, warmup)):
            self.step()
        torch.cuda.synchronize(dev)
        cuda_graph = None
        graph_launches = 0
        if graph:
            # one captured graph per gradient buffer, replayed in turn
            side = torch.cuda.Stream(dev)
            side.wait_stream(self.stream)
            cuda_graph = []
            for b in range(GRAD_BUFFERS):
                gr = torch.cuda.CUDAGraph()
                cap0 = ctx.launch_count()
                with torch.cuda.graph(gr, stream=side):
                    self.t = b
                    self.step(torch.cuda.current_stream(dev))
                graph_launches = ctx.launch_count() - cap0
                cuda_graph.append(gr)
            for gr in cuda_graph:
                gr.replay()
            torch.cuda.synchronize(dev)
        b_step = self.bytes_per_step()
        # a step that streams less than 8x the L2 could be served partly from it: then the
        # L2 is flushed (a 2x-L2 buffer written) before every step, outside per-step events
        flush = b_step < 8 * L2_BYTES
        scratch = torch.empty(2 * L2_BYTES // 4, dtype=torch.float32, device=dev) if flush else None
        s = self.stream

        def timed_loop(kernel_events):
            """`steps` steps; per-step events when flushing, else one pair around all."""
            ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                  for _ in range(steps if flush else 1)]
            ctx.profile(kernel_events)
            launches0 = ctx.launch_count()
            if barrier_fn:
                barrier_fn()
            torch.cuda.synchronize(dev)
            if clocks:
                clocks.start()
                time.sleep(0.3)
            if not flush:
                ev[0][0].record(s)
            for t in range(steps):
                if flush:
                    scratch.fill_(float(t))
                    ev[t][0].record(s)
                if cuda_graph is not None:
                    cuda_graph[t % GRAD_BUFFERS].replay()
                else:
                    self.step()
                if flush:
                    ev[t][1].record(s)
            if not flush:
                ev[0][1].record(s)
            torch.cuda.synchronize(dev)
            clk = clocks.stop() if clocks else None
            if barrier_fn:
                barrier_fn()
            return sum(a.elapsed_time(b) for a, b in ev), ctx.launch_count() - launches0, clk

        # Per-kernel events (recorded by the library around each launch) time the kernels;
        # on a step of a few tens of microseconds they also lengthen it (each pair splits
        # the launch chain), so a flushed small step is timed once without them for the
        # step time and once with them for the kernel times.
        separate = flush and cuda_graph is None
        if separate:
            ms_total, launches, clk = timed_loop(False)
            kernels_ms, _, _ = timed_loop(True)
        else:
            ms_total, launches, clk = timed_loop(cuda_graph is None)
            kernels_ms = ms_total
        if cuda_graph is not None:   # replays launch the captured kernels without the library's counter
            launches = steps * graph_launches
        per_kernel = {}
        for k, name in self.ob.KERNEL_NAMES.items():
            t_ms, cnt = ctx.profile_read(k)
            if cnt:
                per_kernel[name] = {"launches": cnt, "avg_us": 1e3 * t_ms / cnt, "share": t_ms / kernels_ms}
        ctx.profile(False)
        del scratch
        dom = KERNEL_OF_PHASE[self.phase]
        k_bytes = dominant_kernel_bytes(self.phase, self.wl.n, self.wl.W, self.wl.grad_bytes, self.wl.C)
        k_avg_us = per_kernel[dom]["avg_us"] if dom in per_kernel else None
        return {"ms_total": ms_total, "steps": steps, "b_step": b_step, "flush": flush,
                "kernel_events_pass": "separate" if separate else "same",
                "kernels": per_kernel, "launches": launches, "clocks": clk,
                "cuda_graph": cuda_graph is not None, "dominant": dom, "k_bytes": k_bytes,
                "k_avg_us": k_avg_us}

    def free(self):
        for name in ("x", "v", "m", "ew", "es", "ws", "lws", "grads"):
            setattr(self, name, None)
        self.ctx.close()
        self.torch.cuda.synchronize(self.dev)
        self.torch.cuda.empty_cache()


def summarize(run, res, peak):
    """One workload's entry: step time, rate, the step's algorithmic GB/s against the peak,
    the dominant kernel's roofline and every kernel's share of the step."""
    wl = run.wl
    ms_step = res["ms_total"] / res["steps"]
    gbs = res["b_step"] / (ms_step / 1e3) / 1e9
    dom = None
    if res["k_avg_us"]:
        ach = res["k_bytes"] / (res["k_avg_us"] / 1e6) / 1e9
        dom = {"kernel": res["dominant"], "avg_us": res["k_avg_us"], "achieved_gbs": ach,
               "frac": ach / peak, "algorithmic_bytes_per_launch": res["k_bytes"]}
    return {"workload": workload_desc(wl, run.phase), "n": wl.n, "W": wl.W, "chunk": wl.C,
            "grad_dtype": str(wl.grad_dtype).split(".")[-1], "masked": run.masked,
            "steps": res["steps"], "ms_per_step": ms_step, "value": wl.n * wl.W / (ms_step / 1e3),
            "unit": UNIT, "hbm_gbs_step": gbs, "hbm_frac_step": gbs / peak,
            "bytes_per_step": res["b_step"], "dominant": dom,
            "kernels": {k: {"avg_us": v["avg_us"], "share": v["share"]} for k, v in res["kernels"].items()},
            "cuda_graph": res["cuda_graph"], "l2": "flushed before every step" if res["flush"] else "streamed (step >> L2)",
            "kernel_times": ("a second timed pass with per-kernel events (shares of that pass)"
                             if res["kernel_events_pass"] == "separate" else "per-kernel events in the timed pass"),
            "gpu_launches": res["launches"], "clocks": res["clocks"]}


# The workloads other than the headline, run in sequence after it (memory freed between):
# (name, phase, workers or None for the recipe's, replayed from a CUDA graph[, chunk]).
# The last two are the headline and LoCo buffers with 256-element chunks (the recipes
# use chunk = n/W), the short-chunk paths of the worker and of LoCo.
EXTRA_WORKLOADS = [
    ("bertB", "compressed", None, False), ("bertB", "warmup", None, False),
    ("sweep", "compressed", 2, False), ("sweep", "warmup", 2, False),
    ("sweep", "compressed", 4, False), ("sweep", "warmup", 4, False),
    ("sweep", "compressed", 8, False), ("sweep", "warmup", 8, False),
    ("sweep", "compressed", 16, False), ("sweep", "warmup", 16, False),
    ("loco", "loco", None, False), ("loco", "compressed", None, False),
    ("tiny", "compressed", None, False), ("tiny", "compressed", None, True),
    ("bertL", "compressed", None, False, 256), ("loco", "loco", None, False, 256),
]


def run_extra_workloads(torch, ob, synth, dev, steps, warmup, peak, only=None):
    out = {}
    for entry in EXTRA_WORKLOADS:
        name, phase, W, graph = entry[:4]
        chunk = entry[4] if len(entry) > 4 else None
        key = "%s%s_%s%s%s" % (name, "_W%d" % W if W else "", phase, "_graph" if graph else "",
                               "_c%d" % chunk if chunk else "")
        if only and not any(o in key for o in only):
            continue
        wl = synth.workload(name, W=W, chunk=chunk)
        run = Run(torch, ob, synth, dev, wl, phase)
        n_steps = max(steps, 50) if name == "tiny" else steps
        res = run.measure(n_steps, warmup, graph=graph, clocks=ClockSampler(_gpu_index(dev)))
        out[key] = summarize(run, res, peak)
        run.free()
        del run
    return out


def _gpu_index(dev):
    vis = os.environ.get("CUDA_VISIBLE_DEVICES")
    return vis.split(",")[dev.index] if vis else dev.index


def e2e_leg(torch, run, steps, dist, world):
    """End to end through ob_compressed_step_host, plus the same host-to-device copy alone."""
    wl, dev, ctx, stream = run.wl, run.dev, run.ctx, run.stream
    n, W, C = wl.n, wl.W, wl.C
    g0 = run.grads[0]
    g_host = torch.empty(g0.shape, dtype=g0.dtype, pin_memory=True)
    g_host.copy_(g0)
    sb_host = torch.empty(n // 32, dtype=torch.int32, pin_memory=True)
    ss_host = torch.empty(n // C, dtype=torch.float32, pin_memory=True)
    # two device gradient buffers, alternated, so that the next step's host copy overlaps
    # this step's kernels (the library orders each copy after the last worker pass that
    # read the buffer); the timed draws are released to make room
    g_dev = [run.grads[0], run.grads[1]]
    run.grads = g_dev
    x, m, v, ew, es, ws = run.x, run.m, run.v, run.ew, run.es, run.ws
    for i in range(2):
        ctx.compressed_step_host(g_host, g_dev[i % 2], x, m, v, ew, es, ws, sb_host, ss_host, stream)
    torch.cuda.synchronize(dev)
    barrier(dist)
    t0 = time.perf_counter()
    for i in range(steps):
        ctx.compressed_step_host(g_host, g_dev[i % 2], x, m, v, ew, es, ws, sb_host, ss_host, stream)
    torch.cuda.synchronize(dev)
    e_ms = max_over_ranks(dist, (time.perf_counter() - t0) * 1e3)
    h2d = int(g_host.numel() * g_host.element_size())
    # the copy alone: the same pinned bytes, host to device, back to back on one stream,
    # each copy timed by its own events (the host link's rate varies from copy to copy:
    # the median and the fastest are reported)
    side = torch.cuda.Stream(dev)
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(steps + 1)]
    with torch.cuda.stream(side):
        g_dev[0].copy_(g_host, non_blocking=True)
        ev[0].record(side)
        for i in range(steps):
            g_dev[i % 2].copy_(g_host, non_blocking=True)
            ev[i + 1].record(side)
    side.synchronize()
    per_copy = sorted(ev[i].elapsed_time(ev[i + 1]) for i in range(steps))
    copy_ms = per_copy[len(per_copy) // 2]
    out = {"value": n * W * steps * world / (e_ms / 1e3), "unit": UNIT,
           "ms_per_step": e_ms / steps,
           "h2d_bytes_per_step": h2d,
           "d2h_bytes_per_step": int(n // 8 + (n // C) * 4),
           "copy_only": {"ms_per_step": copy_ms, "h2d_gbs": h2d / (copy_ms / 1e3) / 1e9,
                         "fastest_ms": per_copy[0], "fastest_h2d_gbs": h2d / (per_copy[0] / 1e3) / 1e9,
                         "what": "the same pinned host-to-device gradient copy alone, back to back, "
                                 "CUDA events on its stream around each copy (median and fastest "
                                 "of the copies): the link bound of the end-to-end step"},
           "path": "ob_compressed_step_host each step: pinned host grads -> device (library copy "
                   "stream, overlapped with the previous step's kernels), the step, server "
                   "signs+scales -> pinned host; host wall clock with device syncs at both ends"}
    del g_host, sb_host, ss_host
    return out


def gpu_arm(args, wl):
    import torch
    from error_compensated_bit_gb300 import build, ob, synth

    dist, rank, world, local = dist_init(args)
    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA device for the GPU arm")
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    build.build()
    ob.load()
    peak, peak_kind = load_peaks()

    run = Run(torch, ob, synth, dev, wl, args.phase)
    res = run.measure(args.steps, args.warmup, graph=args.graph, clocks=ClockSampler(_gpu_index(dev)),
                      barrier_fn=lambda: barrier(dist))
    n, W, C = wl.n, wl.W, wl.C
    ms_total = max_over_ranks(dist, res["ms_total"])
    ms_step = ms_total / args.steps
    value = n * W * args.steps * world / (ms_total / 1e3)
    b_step = res["b_step"]
    k_avg_s = res["k_avg_us"] / 1e6 if res["k_avg_us"] else None
    achieved = res["k_bytes"] / k_avg_s / 1e9 if k_avg_s else None
    if args.phase == "compressed":
        khash = kernel_source_hash(WORKER_SOURCES)
    elif args.phase == "warmup":
        khash = kernel_source_hash(["ob_warmup.cu", "ob_common.cuh"])
    else:
        khash = kernel_source_hash(["ob_loco.cu", "ob_common.cuh"])
    traffic = load_traffic(wl.name, W, khash) if args.phase == "compressed" else None

    e2e = None
    if args.phase == "compressed" and args.e2e_steps > 0:
        e2e = e2e_leg(torch, run, args.e2e_steps, dist, world)
    run.free()
    del run

    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": max(3, args.warmup), "ms_per_step": ms_step, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": {"workload": workload_desc(wl, args.phase), "n": n, "W": W, "chunk": C,
                   "grad_dtype": str(wl.grad_dtype).split(".")[-1], "masked": wl.zero_frac > 0 and args.phase == "compressed",
                   "cuda_graph": res["cuda_graph"], "grad_buffers": GRAD_BUFFERS,
                   "parallelism": "replicas" if world > 1 else "single GPU",
                   "l2": ("flushed: a %d MB buffer written before every step, steps timed one by one "
                          "(each streams %.2f GB, under 8x the 129 MB L2)" % (2 * L2_BYTES // 10**6, b_step / 1e9)
                          if res["flush"] else
                          "no flush: each step streams %.1f GB, far more than the 129 MB L2" % (b_step / 1e9))},
        "hbm_gbs_step": b_step / (ms_step / 1e3) / 1e9,
        "hbm_frac_step": b_step / (ms_step / 1e3) / 1e9 / peak,
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak if achieved else None, "traffic": traffic,
                     "kernel": res["dominant"],
                     "algorithmic_bytes_per_launch": res["k_bytes"], "avg_launch_us": res["k_avg_us"],
                     "peak_kind": "%s hbm_gbs (STREAM-style copy)" % peak_kind},
        "kernels": res["kernels"],
        "clocks": res["clocks"], "gpu_launches": res["launches"], "e2e": e2e,
    }
    default_run = args.workload == "bertL" and args.phase == "compressed" and args.n is None and args.chunk is None
    if args.workloads != "none" and (default_run or args.workloads != "default"):
        if world == 1:
            only = None if args.workloads in ("default", "all") else args.workloads.split(",")
            line["workloads"] = run_extra_workloads(torch, ob, synth, dev, args.steps, args.warmup, peak, only)
        else:
            line["workloads"] = "run at N=1 only (replicas add nothing per GPU)"
    if rank == 0 and not args.no_cpu_baseline:
        n_s = wl.W * 256 * 4096
        per, steps, u, desc = oracle_sample_run(wl, args.phase, n_s, args.cpu_seconds)
        line["cpu_baseline"] = {"value": u / per, "unit": UNIT, "cores": 1, "kind": "oracle",
                                "sample": desc}
    if rank == 0:
        print(json.dumps(line))
    if dist is not None:
        dist.destroy_process_group()
    return 0


def main():
    args = parse()
    from error_compensated_bit_gb300 import synth
    wl = synth.workload(args.workload, W=args.W, n=args.n, chunk=args.chunk)
    if args.phase == "loco" and args.workload != "loco":
        pass
    if args.impl == "reference":
        return reference_arm(args, wl)
    return gpu_arm(args, wl)


if __name__ == "__main__":
    sys.exit(main())
