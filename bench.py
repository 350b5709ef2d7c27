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
server's compressed message copied back), sampled SM clocks, and the CPU oracle timed on
a bounded sample of the same workload.

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

    n, W, C = wl.n, wl.W, wl.C
    s_g = wl.grad_bytes
    masked = wl.zero_frac > 0 and args.phase == "compressed"
    ctx = ob.Context(n, W, C, wl.b1, wl.b2, wl.eps, wl.lr)
    x = synth.params(wl, dev)
    v = synth.variance(wl, dev)
    m = torch.zeros(n, dtype=torch.float32, device=dev)
    ew = torch.zeros(W, n, dtype=torch.float32, device=dev)
    es = torch.zeros(n, dtype=torch.float32, device=dev)
    ws = torch.empty(ctx.workspace_bytes(), dtype=torch.uint8, device=dev)
    ctx.workspace_init(ws)
    g = synth.grads(wl, 0, dev)
    mask = None
    if masked:
        mask = synth.mask(wl, dev)
        ctx.set_mask(mask, ws)
    lws = None
    if args.phase == "loco":
        lws = torch.zeros(ctx.loco_workspace_bytes(4), dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)

    def one_step():
        if args.phase == "compressed":
            ctx.compressed_step(g, x, m, v, ew, es, ws, stream)
        elif args.phase == "warmup":
            ctx.warmup_step(g, x, m, v, ws, stream)
        else:
            ctx.loco_step(g, x, m, v, ew, lws, 0.9, 4, stream)

    # the BERT-Base recipe runs its warm-up steps before the compressed ones
    if args.phase == "compressed" and wl.warmup_steps:
        for t in range(wl.warmup_steps):
            ctx.warmup_step(synth.grads(wl, t + 1, dev, out=g), x, m, v, ws, stream)
        synth.grads(wl, 0, dev, out=g)
    for _ in range(max(3, args.warmup)):
        one_step()
    torch.cuda.synchronize(dev)
    graph = None
    if args.graph:
        side = torch.cuda.Stream(dev)
        side.wait_stream(stream)
        graph = torch.cuda.CUDAGraph()
        cap0 = ctx.launch_count()
        with torch.cuda.graph(graph, stream=side):
            cap = torch.cuda.current_stream(dev)
            if args.phase == "compressed":
                ctx.compressed_step(g, x, m, v, ew, es, ws, cap)
            elif args.phase == "warmup":
                ctx.warmup_step(g, x, m, v, ws, cap)
            else:
                ctx.loco_step(g, x, m, v, ew, lws, 0.9, 4, cap)
        graph_launches = ctx.launch_count() - cap0     # kernels captured per step
        graph.replay()
        torch.cuda.synchronize(dev)

    # timed region
    clocks = ClockSampler(dev.index if "CUDA_VISIBLE_DEVICES" not in os.environ else
                          os.environ["CUDA_VISIBLE_DEVICES"].split(",")[dev.index])
    # A step that streams less than 8x the L2 could be served partly from it: then the L2
    # is flushed (a 2x-L2 buffer written) before every step, outside per-step events.
    b_step = n * bytes_per_elem(args.phase, W, s_g, masked)
    flush = b_step < 8 * L2_BYTES
    scratch = torch.empty(2 * L2_BYTES // 4, dtype=torch.float32, device=dev) if flush else None
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(args.steps if flush else 1)]
    launches0 = ctx.launch_count()
    ctx.profile(True)
    barrier(dist)
    torch.cuda.synchronize(dev)
    clocks.start()
    time.sleep(0.3)
    if not flush:
        ev[0][0].record(stream)
    for t in range(args.steps):
        if flush:
            scratch.fill_(float(t))
            ev[t][0].record(stream)
        if graph is not None:
            graph.replay()
        else:
            one_step()
        if flush:
            ev[t][1].record(stream)
    if not flush:
        ev[0][1].record(stream)
    torch.cuda.synchronize(dev)
    clk = clocks.stop()
    barrier(dist)
    ms_total = sum(a.elapsed_time(b) for a, b in ev)
    launches = ctx.launch_count() - launches0
    if graph is not None:     # replays launch the captured kernels without the library's counter
        launches = args.steps * graph_launches
    kid = {"compressed": ob.OB_K_WORKER, "warmup": ob.OB_K_WARMUP, "loco": ob.OB_K_LOCO_QUANT}[args.phase]
    k_ms, k_n = ctx.profile_read(kid)
    per_kernel = {}
    for k, name in ob.KERNEL_NAMES.items():
        t_ms, cnt = ctx.profile_read(k)
        if cnt:
            per_kernel[name] = {"launches": cnt, "avg_us": 1e3 * t_ms / cnt,
                                "share": t_ms / ms_total}
    ctx.profile(False)
    ms_total = max_over_ranks(dist, ms_total)

    ms_step = ms_total / args.steps
    units = n * W * args.steps * world
    value = units / (ms_total / 1e3)
    peak, peak_kind = load_peaks()
    if args.phase == "compressed":
        k_bytes = n * worker_bytes_per_elem(W, s_g)
        khash = kernel_source_hash(["ob_worker.cu", "ob_common.cuh", "ob_tma.cuh"])
    elif args.phase == "warmup":
        k_bytes = n * (W * s_g + 24.0)
        khash = kernel_source_hash(["ob_warmup.cu", "ob_common.cuh"])
    else:
        k_bytes = n * W * (s_g + 8.5)
        khash = kernel_source_hash(["ob_loco.cu", "ob_common.cuh"])
    # per-kernel events exist only for direct launches (not for graph replays)
    k_avg_s = (k_ms / k_n) / 1e3 if k_n else None
    achieved = k_bytes / k_avg_s / 1e9 if k_avg_s else None
    traffic = load_traffic(wl.name, W, khash) if args.phase == "compressed" else None

    # end to end through the host-buffer entry point (compressed phase only)
    e2e = None
    if args.phase == "compressed" and args.e2e_steps > 0:
        g_host = torch.empty(g.shape, dtype=g.dtype, pin_memory=True)
        g_host.copy_(g)
        sb_host = torch.empty(n // 32, dtype=torch.int32, pin_memory=True)
        ss_host = torch.empty(n // C, dtype=torch.float32, pin_memory=True)
        # two device gradient buffers, alternated, so that the next step's host copy
        # overlaps this step's kernels (the library orders each copy after the last
        # worker pass that read the buffer)
        g_dev = [torch.empty_like(g), torch.empty_like(g)]
        del g
        for i in range(2):
            ctx.compressed_step_host(g_host, g_dev[i % 2], x, m, v, ew, es, ws, sb_host, ss_host, stream)
        torch.cuda.synchronize(dev)
        barrier(dist)
        t0 = time.perf_counter()
        for i in range(args.e2e_steps):
            ctx.compressed_step_host(g_host, g_dev[i % 2], x, m, v, ew, es, ws, sb_host, ss_host, stream)
        torch.cuda.synchronize(dev)
        e_ms = max_over_ranks(dist, (time.perf_counter() - t0) * 1e3)
        e2e = {"value": n * W * args.e2e_steps * world / (e_ms / 1e3), "unit": UNIT,
               "ms_per_step": e_ms / args.e2e_steps,
               "h2d_bytes_per_step": int(g_host.numel() * g_host.element_size()),
               "d2h_bytes_per_step": int(n // 8 + (n // C) * 4),
               "path": "ob_compressed_step_host each step: pinned host grads -> device (library copy "
                       "stream, overlapped with the previous step's kernels), the step, server "
                       "signs+scales -> pinned host; host wall clock with device syncs at both ends"}
        del g_host, g_dev

    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": max(3, args.warmup), "ms_per_step": ms_step, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": {"workload": workload_desc(wl, args.phase), "n": n, "W": W, "chunk": C,
                   "grad_dtype": str(wl.grad_dtype).split(".")[-1], "masked": masked,
                   "cuda_graph": graph is not None,
                   "parallelism": "replicas" if world > 1 else "single GPU",
                   "l2": ("flushed: a %d MB buffer written before every step, steps timed one by one "
                          "(each streams %.2f GB, under 8x the 129 MB L2)" % (2 * L2_BYTES // 10**6, b_step / 1e9)
                          if flush else
                          "no flush: each step streams %.1f GB, far more than the 129 MB L2" % (b_step / 1e9))},
        "hbm_gbs_step": b_step / (ms_step / 1e3) / 1e9,
        "hbm_frac_step": b_step / (ms_step / 1e3) / 1e9 / peak,
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak if achieved else None, "traffic": traffic,
                     "kernel": {"compressed": "worker", "warmup": "warmup", "loco": "loco_quant"}[args.phase],
                     "algorithmic_bytes_per_launch": k_bytes, "avg_launch_us": k_avg_s * 1e6 if k_avg_s else None,
                     "peak_kind": "%s hbm_gbs (STREAM-style copy)" % peak_kind},
        "kernels": per_kernel,
        "clocks": clk, "gpu_launches": launches, "e2e": e2e,
    }
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
