#!/usr/bin/env python
"""Benchmark of the channel-wise (UVU) CG tensor-product graph convolution on GB300.

One step = one pass of the hot path over the workload: the forward (uvu_fwd) and the full VJP
(uvu_bwd_edge for dw and dY, then dx).  The graph preparation (receiver CSR and its transpose)
is done once before timing, as in "Receiver-streaming convolutions for channel-wise UVU tensor
products" (opening post, benchmark paragraph: graph construction outside the timed region), and
reported separately.

Prints one JSON line.  `value` is whole-job fwd+VJP edges/s with inputs resident in HBM;
`e2e` is the same metric through the C ABI with the inputs copied from pinned host memory and
all outputs copied back inside the timed region.  The roofline object describes the kernel with
the largest share of the step: algorithmic bytes per launch / its CUDA-event duration.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--config 1] [--dx-mode sender|atomic]
  python bench.py --impl reference ...   # the fp64 CPU oracle on bounded samples
Under torchrun (N > 1) every rank runs an independent replica of the workload on its own GPU
(the operation is not sharded); timings are max-reduced over ranks.
"""

from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "edges/sec fwd & fwd+VJP UVU conv (5k nodes/280k edges); % of HBM roofline"


def parse_args(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="uvu", choices=["uvu", "reference"])
    ap.add_argument("--config", type=int, default=1)
    ap.add_argument("--nodes", type=int, default=None,
                    help="node count of the workload (default: the config's); smaller graphs of the "
                         "same plan serve ncu captures, which must stay a few GB on the device")
    ap.add_argument("--dx-mode", default="staged", choices=["staged", "sender", "atomic"])
    ap.add_argument("--e2e-steps", type=int, default=5)
    ap.add_argument("--e2e-chunks", type=int, default=16)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-hvp", action="store_true", help="skip the double-backward measurement")
    ap.add_argument("--no-tp", action="store_true", help="skip the batched tensor-product measurement")
    ap.add_argument("--no-radial", action="store_true", help="skip the fused-radial-weight measurement")
    ap.add_argument("--no-configs", action="store_true",
                    help="skip the fwd and fwd+VJP measurement of the other four workloads")
    ap.add_argument("--tp-batch", type=int, default=100000, help="samples of the batched tensor product")
    ap.add_argument("--no-clocks", action="store_true", help="do not sample nvidia-smi clocks")
    ap.add_argument("--single-mode", action="store_true",
                    help="warm up and time only --dx-mode (profiling runs)")
    return ap.parse_args(argv)


# ------------------------------------------------------------------------- bytes and units

def algorithmic_bytes(N, E, U, P, Dx, Dy, Do, s):
    """Compulsory bytes per launch of each kernel: its share of the operation's inputs read once
    and outputs written once (x, Y, w, out or d_out, the indices; dx, dY, dw).  Intermediates a
    design chooses to keep in memory (the staged per-edge dx partials, an atomic dx
    read-modify-write) are not algorithmic bytes: ``overhead_bytes`` lists them."""
    idx_r = 4 * (N + 1) + 4 * E          # recv_offsets + src
    idx_s = 4 * (N + 1) + 8 * E          # send_offsets + send_eids + send_recv
    x, Y, w, out = N * U * Dx * s, E * Dy * s, E * P * U * s, N * U * Do * s
    return {
        "uvu_fwd": x + Y + w + out + idx_r,
        "uvu_bwd_edge": x + Y + w + out + idx_r + Y + w,        # reads x,Y,w,d_out; writes dY,dw
        "uvu_bwd_edge+atomic_dx": x + Y + w + out + idx_r + Y + w + x,
        "uvu_bwd_dx": Y + w + out + idx_s + x,                  # reads Y,w,d_out; writes dx
        "uvu_bwd_dx_reduce": 4 * (N + 1) + 4 * E + x,           # reads the send CSR; writes dx
        "fwd": x + Y + w + out + idx_r,
        "vjp": (x + Y + w + out + idx_r + idx_s) + (x + Y + w),
    }


def overhead_bytes(N, E, U, Dx, s):
    """Bytes a kernel moves beyond its compulsory share, by dx mode: the staged mode writes and
    reads back one dx partial row per (edge, channel)."""
    part = E * U * Dx * s
    return {"staged": {"uvu_bwd_edge": part, "uvu_bwd_dx_reduce": part},
            "atomic": {}, "sender": {}}


def describe(spec, info, E, N=None):
    return (f"{spec.name}: {N or spec.n_nodes} nodes, {E} edges, x {spec.irreps_x}, "
            f"SH {spec.irreps_sh}, l3<={spec.lmax_out} ({info.n_paths} paths), {spec.dtype}")


def fp64_ops_per_edge_channel(plan):
    """FP64 instructions the plan's generated forward executed per (edge, channel), from an ncu
    count committed under profiles/ for this exact generated source (None when the source has
    changed since the count was taken)."""
    path = os.path.join(ROOT, "profiles", "fp64_ops.json")
    if not os.path.exists(path):
        return None
    import hashlib
    tab = json.load(open(path))
    h = hashlib.sha256(plan.source()[0].encode()).hexdigest()[:16]
    ent = tab.get("uvu_fwd")
    if not ent or ent.get("source_sha") != h:
        return None
    return ent


def measure_alu_peaks(uvu, torch, dev, stream):
    """FP32 and FP64 FMA rates of this GPU, measured now with the library's FMA-chain probe
    (8 independent chains per thread, 8 blocks of 256 threads per SM): the best of five launches,
    timed with CUDA events on the launching stream.  TFLOP/s at 2 flop per FMA."""
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    blocks = sms * 8
    res = {}
    for name, f64, iters in (("fp32", False, 1024), ("fp64", True, 64)):
        buf = torch.empty(blocks * 256, dtype=torch.float64 if f64 else torch.float32, device=dev)
        uvu.fma_rate_probe(buf, f64, blocks, iters, stream)
        best = None
        fmas = 0.0
        for _ in range(5):
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            fmas = uvu.fma_rate_probe(buf, f64, blocks, iters, stream)
            b.record(stream)
            torch.cuda.synchronize()
            ms = a.elapsed_time(b)
            best = ms if best is None else min(best, ms)
        res[name + "_tflops"] = 2.0 * fmas / (best / 1000.0) / 1e12
        res[name + "_probe_ms"] = best
    res["method"] = ("library FMA-chain probe (uvu_fma_rate_probe): %d blocks x 256 threads x 8 chains, "
                     "best of 5 launches, CUDA events; 2 flop per FMA" % blocks)
    return res


# ------------------------------------------------------------------------- clocks sampling

class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.proc = None
        self.gpu = gpu_index
        # raw nvidia-smi samples (the JSON line carries their summary); UVU_BENCH_CLOCKS_DIR
        # chooses where they are kept
        import tempfile
        d = os.environ.get("UVU_BENCH_CLOCKS_DIR") or tempfile.gettempdir()
        self.path = os.path.join(d, f"uvu_bench_clocks_rank{gpu_index}.csv")

    def start(self):
        try:
            os.makedirs(os.path.dirname(self.path), exist_ok=True)
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=self.f, stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None

    def stop(self):
        if not self.proc:
            return None
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.f.close()
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax),
                "reasons": sorted(reasons), "samples": len(sm)}


# ------------------------------------------------------------------------- distributed

def dist_env():
    return (int(os.environ.get("RANK", 0)), int(os.environ.get("LOCAL_RANK", 0)),
            int(os.environ.get("WORLD_SIZE", 1)))


def max_over_ranks(value: float, world: int, device=None) -> float:
    """Max of a per-rank float over the process group (identity for one process)."""
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


# ------------------------------------------------------------------------- CPU oracle leg

def cpu_model():
    """The host CPU's model name (lscpu, else /proc/cpuinfo)."""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.lower().startswith("model name"):
                return line.split(":", 1)[1].strip()
    except (OSError, subprocess.SubprocessError):
        pass
    try:
        for line in open("/proc/cpuinfo"):
            if line.lower().startswith(("model name", "cpu part")):
                return line.split(":", 1)[1].strip()
    except OSError:
        pass
    return "unknown"


class OracleSampler:
    """Times the fp64 CPU oracle (oracle.conv, as it stands) on bounded samples of one workload.

    fwd: the oracle's receiver-stationary loops over the edges of a random set of receivers;
    VJP: dY and dw over the same receivers' edges, plus dx over a random set of senders, which
    covers each of their out-edges.  A sample is a compact sub-problem: the sampled receivers
    with their incoming edges (global sender ids, the full x), or the sampled senders with their
    out-edges and the d_out rows those edges reach, so every edge is computed exactly as in the
    full problem.  w and d_out values of the sampled rows are drawn here (the oracle's time does
    not depend on them).  Each measurement repeats samples until at least `min_s` seconds of wall
    time have passed and reports edges per second over that time."""

    def __init__(self, key, wl=None, seed=0):
        import numpy as np
        from clebsch_gordan_tensor_receiver_gb300 import workloads
        from oracle import graph, paths
        self.np = np
        self.spec = workloads.SPECS[key]
        self.wl = wl if wl is not None else workloads.make_workload(key)
        self.lay = paths.layout(self.spec.irreps_x, self.spec.irreps_sh, self.spec.lmax_out)
        self.N, self.E = self.wl.n_nodes, self.wl.n_edges
        self.off = graph.recv_offsets(self.wl.recv, self.N).astype(np.int64)
        self.dt = np.float64 if self.spec.dtype == "float64" else np.float32
        self.rng = np.random.default_rng(seed)
        self.P, self.U = len(self.lay.paths), self.lay.mul
        self.nr = max(1, min(self.N, 8))
        self.ns = max(1, min(self.N, 8))

    def _normal(self, shape, scale=1.0):
        return (self.rng.standard_normal(shape) * scale).astype(self.dt)

    def _recv_sample(self, n):
        np = self.np
        rs = np.sort(self.rng.choice(self.N, size=min(n, self.N), replace=False))
        segs = [np.arange(self.off[r], self.off[r + 1]) for r in rs]
        eidx = np.concatenate(segs) if segs else np.zeros(0, np.int64)
        loff = np.zeros(rs.size + 1, np.int64)
        np.cumsum([a.size for a in segs], out=loff[1:])
        w = self._normal((eidx.size, self.P, self.U), 1.0 / self.spec.w_scale_degree ** 0.5)
        g = self._normal((rs.size, self.U, self.lay.dim_out))
        return loff, self.wl.src[eidx], self.wl.Y[eidx], w, g, eidx.size

    def _send_sample(self, n):
        np = self.np
        from oracle import graph
        ss = np.sort(self.rng.choice(self.N, size=min(n, self.N), replace=False))
        eidx = np.nonzero(np.isin(self.wl.src, ss))[0]
        recv = graph.recv_of_edges(self.off)[eidx]
        # compact node ids: the sampled senders and the receivers their edges reach
        nodes, inv = np.unique(np.concatenate([ss, recv, self.wl.src[eidx]]), return_inverse=True)
        crecv = inv[ss.size:ss.size + eidx.size]
        csrc = inv[ss.size + eidx.size:]
        csend = inv[:ss.size]
        coff = graph.recv_offsets(crecv, nodes.size)  # edges stay receiver-sorted
        w = self._normal((eidx.size, self.P, self.U), 1.0 / self.spec.w_scale_degree ** 0.5)
        g = self._normal((nodes.size, self.U, self.lay.dim_out))
        return coff, csrc, self.wl.Y[eidx], w, g, nodes.size, csend, eidx.size

    def _rate(self, kind, min_s, threads):
        """edges/s of one measurement of `kind` ("fwd" or "vjp") lasting >= min_s seconds."""
        from oracle import conv
        done_e, spent = 0.0, 0.0
        per_edge_vjp = []
        while spent < min_s:
            loff, src, Y, w, g, ne = self._recv_sample(self.nr)
            if kind == "fwd":
                t0 = time.perf_counter()
                conv.fwd(self.lay, loff, src, self.wl.x, Y, w, nthreads=threads)
                dt = time.perf_counter() - t0
                done_e += ne
                spent += dt
                if dt < 0.5 and self.nr < self.N:  # grow the sample towards ~0.5 s per call
                    self.nr = min(self.N, max(self.nr + 1, int(self.nr * 0.6 / max(dt, 1e-3))))
                continue
            t0 = time.perf_counter()
            conv.bwd_edges(self.lay, loff, src, self.wl.x, Y, w, g, nthreads=threads)
            t1 = time.perf_counter()
            coff, csrc, Ys, ws, gs, nn, csend, nse = self._send_sample(self.ns)
            t2 = time.perf_counter()
            conv.bwd_dx(self.lay, coff, csrc, Ys, ws, gs, nn, senders=csend, nthreads=threads)
            t3 = time.perf_counter()
            spent += (t1 - t0) + (t3 - t2)
            per_edge_vjp.append(((t1 - t0) / max(ne, 1) + (t3 - t2) / max(nse, 1), (t1 - t0) + (t3 - t2)))
            if t1 - t0 < 0.3 and self.nr < self.N:
                self.nr = min(self.N, max(self.nr + 1, int(self.nr * 0.4 / max(t1 - t0, 1e-3))))
            if t3 - t2 < 0.3 and self.ns < self.N:
                self.ns = min(self.N, max(self.ns + 1, int(self.ns * 0.4 / max(t3 - t2, 1e-3))))
        if kind == "fwd":
            return done_e / spent
        # time-weighted mean of the per-edge VJP cost over the samples of this measurement
        tot = sum(t for _, t in per_edge_vjp)
        return 1.0 / (sum(c * t for c, t in per_edge_vjp) / tot)

    def measure(self, threads, min_s=2.0, reps=3):
        """Median of `reps` measurements: fwd edges/s, VJP edges/s and fwd+VJP edges/s."""
        import statistics as st
        self._rate("fwd", 0.3, threads)   # calibrate the sample sizes (untimed)
        self._rate("vjp", 0.3, threads)
        f = [self._rate("fwd", min_s, threads) for _ in range(reps)]
        v = [self._rate("vjp", min_s, threads) for _ in range(reps)]
        fm, vm = st.median(f), st.median(v)
        return {"fwd_edges_per_s": fm, "vjp_edges_per_s": vm, "fwd_vjp_edges_per_s": 1.0 / (1.0 / fm + 1.0 / vm),
                "fwd_runs": f, "vjp_runs": v, "threads": threads,
                "sample": f"fwd: {self.nr} random receivers with their in-edges per call; VJP: dY, dw over "
                          f"{self.nr} receivers' in-edges and dx over {self.ns} random senders' out-edges per call; "
                          f"each run repeats calls for >= {min_s:.1f} s wall; median of {reps} runs"}


def cpu_baseline_protocol(keys_wl, threads):
    """The oracle on the host cores for every workload (fwd, VJP and fwd+VJP edges/s, median of
    three runs of >= 2 s), plus single-threaded runs of the tiny and MACE-medium workloads."""
    per = {}
    for key, wl in keys_wl:
        smp = OracleSampler(key, wl, seed=31 + key)
        ent = {"workload": smp.spec.name, "all_cores": smp.measure(threads)}
        if key in (0, 1):
            ent["single_thread"] = OracleSampler(key, wl, seed=41 + key).measure(1)
        per[smp.spec.name] = ent
    return per


def run_reference(args):
    rank, local_rank, world = dist_env()
    if world > 1 and rank != 0:
        return 0
    from oracle import conv
    smp = OracleSampler(args.config, seed=900)
    thr = conv.default_threads()
    smp._rate("fwd", 0.3, thr)
    smp._rate("vjp", 0.3, thr)
    for _ in range(args.warmup):
        smp._rate("fwd", 0.5, thr)
    rates, fw, vj = [], [], []
    t0 = time.perf_counter()
    for _ in range(args.steps):
        f = smp._rate("fwd", 1.0, thr)
        v = smp._rate("vjp", 1.0, thr)
        fw.append(f)
        vj.append(v)
        rates.append(1.0 / (1.0 / f + 1.0 / v))
    wall = time.perf_counter() - t0
    value = statistics.median(rates)
    sample = ("each step: the oracle's fwd, then its VJP (dY, dw over sampled receivers' in-edges; dx over "
              "sampled senders' out-edges), each repeated for >= 1 s wall on samples of %d receivers / %d senders; "
              "value = median over steps of fwd+VJP edges/s" % (smp.nr, smp.ns))
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "edges/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1000 * wall / max(args.steps, 1), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": describe(smp.spec, type("I", (), {"n_paths": smp.P}), smp.E),
                   "parallelism": "replicas"},
        "fwd_edges_per_s": statistics.median(fw), "vjp_edges_per_s": statistics.median(vj),
        "cpu_baseline": {"value": value, "unit": "edges/s", "cores": thr, "kind": "oracle",
                         "cpu_model": cpu_model(), "sample": sample},
        "e2e": {"value": value, "unit": "edges/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line))
    return 0


# ------------------------------------------------------------------------- GPU leg

def main(argv=None):
    args = parse_args(argv)
    if args.impl == "reference":
        return run_reference(args)

    # More hardware work queues than the default eight, set before the CUDA context exists: the
    # e2e leg's copy-in and copy-out streams otherwise can share a queue with each other or with
    # streams created earlier in the run, and then the two copy directions run one after the
    # other (measured: 26 ms per step instead of 13 on the same box and buffers).
    os.environ.setdefault("CUDA_DEVICE_MAX_CONNECTIONS", "32")
    import numpy as np
    import torch

    rank, local_rank, world = dist_env()
    torch.cuda.set_device(local_rank)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local_rank))
    dev = torch.device("cuda", local_rank)

    from clebsch_gordan_tensor_receiver_gb300 import uvu, workloads
    spec = workloads.SPECS[args.config]
    wl = workloads.make_workload(spec, args.nodes)
    wl_cache = {args.config: wl} if args.nodes is None else {}
    plan = uvu.Plan(spec.irreps_x, spec.irreps_sh, spec.lmax_out, spec.dtype)
    info = plan.info
    N, E, U, P = wl.n_nodes, wl.n_edges, info.mul, info.n_paths
    Dx, Dy, Do = info.dim_x, info.dim_sh, info.dim_out
    w_h = workloads.make_weights(spec, E, P)
    g_h = workloads.make_cotangent(spec, N, Do)
    tdt = torch.float64 if spec.dtype == "float64" else torch.float32
    s = 8 if spec.dtype == "float64" else 4

    def to_dev(a):
        return torch.from_numpy(np.ascontiguousarray(a)).to(dev)

    x, Y, w, g = to_dev(wl.x), to_dev(wl.Y), to_dev(w_h), to_dev(g_h)
    recv, src = to_dev(wl.recv), to_dev(wl.src)
    stream = torch.cuda.current_stream(dev)

    # graph preparation (untimed in the metric; reported separately)
    torch.cuda.synchronize()
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    t0.record(stream)
    G = uvu.Graph(N, recv, src)
    t1.record(stream)
    torch.cuda.synchronize()
    csr_ms = t0.elapsed_time(t1)

    out = torch.empty(N, U, Do, dtype=tdt, device=dev)
    dx = torch.empty(N, U, Dx, dtype=tdt, device=dev)
    dY = torch.empty(E, Dy, dtype=tdt, device=dev)
    dw = torch.empty(E, P, U, dtype=tdt, device=dev)
    modes = [args.dx_mode] + ([] if args.single_mode else
                              [m for m in ("staged", "sender", "atomic") if m != args.dx_mode])
    ws = None
    if "staged" in modes:
        ws = torch.empty(max(plan.workspace_bytes(N, E, uvu.UVU_DX_STAGED), 16), dtype=torch.uint8,
                         device=dev)
    dx_kernel = {"sender": "uvu_bwd_dx", "staged": "uvu_bwd_dx_reduce", "atomic": None}

    def step(mode, evs=None):
        if evs:
            evs[0].record(stream)
        plan.fwd(N, x, Y, w, G.recv_offsets, src, out, stream)
        if evs:
            evs[1].record(stream)
        plan.bwd_edge(N, x, Y, w, G.recv_offsets, src, g, dY=dY, dw=dw,
                      dx_atomic=dx if mode == "atomic" else None,
                      dx_edge=ws if mode == "staged" else None, stream=stream)
        if evs:
            evs[2].record(stream)
        if mode == "sender":
            plan.bwd_dx(N, E, Y, w, G.send_offsets, G.send_eids, G.send_recv, g, dx, stream)
        elif mode == "staged":
            plan.bwd_dx_reduce(N, E, G.send_offsets, G.send_eids, ws, dx, stream)
        if evs:
            evs[3].record(stream)

    def timed(mode, K):
        evs = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(K)]
        start = torch.cuda.Event(enable_timing=True)
        end = torch.cuda.Event(enable_timing=True)
        barrier(world)
        torch.cuda.synchronize()
        start.record(stream)
        for k in range(K):
            step(mode, evs[k])
        end.record(stream)
        torch.cuda.synchronize()
        barrier(world)
        total = start.elapsed_time(end)
        per = {"uvu_fwd": [], "uvu_bwd_edge": []}
        if dx_kernel[mode]:
            per[dx_kernel[mode]] = []
        for e in evs:
            per["uvu_fwd"].append(e[0].elapsed_time(e[1]))
            per["uvu_bwd_edge"].append(e[1].elapsed_time(e[2]))
            if dx_kernel[mode]:
                per[dx_kernel[mode]].append(e[2].elapsed_time(e[3]))
        spread[mode] = {k: {"median": statistics.median(v), "min": min(v), "max": max(v)}
                        for k, v in per.items()}
        return total, {k: statistics.mean(v) for k, v in per.items()}

    for _ in range(max(args.warmup, 3)):
        for m in modes:
            step(m)
    torch.cuda.synchronize()

    spread = {}
    clocks = ClockSampler(local_rank)
    if not args.no_clocks:
        clocks.start()
    results = {m: timed(m, args.steps) for m in modes}
    clk = clocks.stop()
    assert plan.device_status() == 0, "a kernel reported a bounded-wait timeout"
    alu = measure_alu_peaks(uvu, torch, dev, stream)
    alu_peak = alu["fp32_tflops"]

    total_ms, kern_ms = results[args.dx_mode]
    total_ms = max_over_ranks(total_ms, world, dev)
    ms_step = total_ms / args.steps
    value = world * E / (ms_step / 1000.0)

    B = algorithmic_bytes(N, E, U, P, Dx, Dy, Do, s)
    peaks = {}
    pk_path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(pk_path):
        peaks = json.load(open(pk_path))
    hbm_peak = peaks.get("hbm_gbs")
    peak_src = "measured" if hbm_peak else "fallback"
    hbm_peak = hbm_peak or 6800.0

    def frac(bytes_, ms):
        gbs = bytes_ / (ms / 1000.0) / 1e9
        return gbs, gbs / hbm_peak

    edge_key = {"atomic": "uvu_bwd_edge+atomic_dx", "staged": "uvu_bwd_edge", "sender": "uvu_bwd_edge"}
    OV = overhead_bytes(N, E, U, Dx, s)

    def mode_summary(mode):
        tot, km = results[mode]
        vjp = sum(v for k, v in km.items() if k != "uvu_fwd")
        gbs, fr = frac(B["vjp"], vjp)
        return {"vjp_ms": vjp, "vjp_edges_per_s": world * E / (vjp / 1000), "vjp_GB_s": gbs,
                "vjp_hbm_frac": fr, "fwd_vjp_edges_per_s": world * E / (tot / args.steps / 1000),
                "deterministic": mode != "atomic", "overhead_bytes": sum(OV[mode].values()),
                "kernels_ms": km}

    # per kernel: compulsory bytes (its share of the operation's inputs and outputs) over its
    # time against the HBM peak; the intermediates the design adds are listed beside them
    kernels = {}
    for k, ms in kern_ms.items():
        key = edge_key[args.dx_mode] if k == "uvu_bwd_edge" else k
        gbs, fr = frac(B[key], ms)
        ov = OV[args.dx_mode].get(k, 0)
        kernels[k] = {"ms": ms, "bytes": B[key], "GB_s": gbs, "frac": fr, "overhead_bytes": ov,
                      "moved_GB_s": (B[key] + ov) / (ms / 1000.0) / 1e9}
    dom = max(kernels, key=lambda k: kernels[k]["ms"])
    traffic = None
    tpath = os.path.join(ROOT, "profiles", "traffic.json")
    if os.path.exists(tpath):
        import hashlib
        tj = json.load(open(tpath))
        h = hashlib.sha256(plan.source()[0].encode()).hexdigest()[:16]
        ent = tj.get(f"{spec.name}:{dom}:{args.dx_mode}")
        if ent and ent.get("source_sha") == h:
            traffic = ent["dram_bytes_per_launch"]
    fwd_ms = kern_ms["uvu_fwd"]
    vjp_ms = sum(v for k, v in kern_ms.items() if k != "uvu_fwd")
    fwd_gbs, fwd_fr = frac(B["fwd"], fwd_ms)
    vjp_gbs, vjp_fr = frac(B["vjp"], vjp_ms)
    line = {
        "metric": METRIC, "value": value, "unit": "edges/s", "n_gpus": world,
        "steps": args.steps, "warmup": max(args.warmup, 3), "ms_per_step": ms_step,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f64" if s == 8 else "f32", "data": "synthetic",
        "config": {"workload": describe(spec, info, E, N), "n_nodes": N, "n_edges": E,
                   "dx_mode": args.dx_mode, "parallelism": "replicas" if world > 1 else "single",
                   "l2": "inputs larger than L2 (w alone is %.2f GB), no flush" % (E * P * U * s / 1e9)},
        "fwd": {"edges_per_s": world * E / (fwd_ms / 1000), "ms": fwd_ms, "GB_s": fwd_gbs,
                "hbm_frac": fwd_fr, "bytes": B["fwd"]},
        "vjp": {"edges_per_s": world * E / (vjp_ms / 1000), "ms": vjp_ms, "GB_s": vjp_gbs,
                "hbm_frac": vjp_fr, "bytes": B["vjp"], "dx_mode": args.dx_mode},
        "dx_modes": {m: mode_summary(m) for m in modes},
        "kernels": kernels,
        "roofline": {"kernel": dom, "bound": "hbm", "achieved": kernels[dom]["GB_s"],
                     "peak": hbm_peak, "unit": "GB/s", "frac": kernels[dom]["frac"],
                     "traffic": traffic, "algorithmic_bytes": kernels[dom]["bytes"],
                     "overhead_bytes": kernels[dom]["overhead_bytes"],
                     "traffic_over_algorithmic": (traffic / kernels[dom]["bytes"]) if traffic else None,
                     "peak_source": peak_src + " hbm_gbs (copy)",
                     "note": "achieved = compulsory bytes of the kernel (x, Y, w, d_out, indices read; dY, dw "
                             "written) / its CUDA-event time; traffic = ncu DRAM read+write per launch"},
        "kernel_ms_spread": spread,
        "csr_build_ms": csr_ms,
        "alu_peaks": alu,
        "clocks": clk,
        "gpu_launches": args.steps * (2 if args.dx_mode == "atomic" else 3),
    }

    # receiver- vs sender-stationary forward: the data-movement model's bytes and choice, and both
    # forwards timed on this workload
    if world == 1 and not args.single_mode:
        choice, br, bs = plan.fwd_model(N, E)
        fs_out = torch.empty_like(out)

        def ev_med(fn, reps=5):
            for _ in range(2):
                fn()
            ts = []
            for _ in range(reps):
                a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                a.record(stream)
                fn()
                b.record(stream)
                ts.append((a, b))
            torch.cuda.synchronize()
            return statistics.median(a.elapsed_time(b) for a, b in ts)

        r_ms = ev_med(lambda: plan.fwd(N, x, Y, w, G.recv_offsets, src, fs_out, stream=stream))
        s_ms = ev_med(lambda: plan.fwd_sender(N, E, x, Y, w, G.send_offsets, G.send_eids, G.send_recv,
                                              fs_out, stream=stream))
        line["fwd_modes"] = {"model_choice": {uvu.UVU_FWD_RECEIVER: "receiver", uvu.UVU_FWD_SENDER: "sender"}[choice],
                             "model_bytes": {"receiver": br, "sender": bs},
                             "measured_ms": {"receiver": r_ms, "sender": s_ms},
                             "measured_choice": "receiver" if r_ms <= s_ms else "sender"}
        assert plan.device_status() == 0
        del fs_out

    # channel mixing of the UVU output (the factorised UVW convolution's second step), W = U:
    # a dense contraction over the channel index, bound by the FP32 FMA pipe (its bytes are the
    # UVU output in and the mixed output out)
    if world == 1 and not args.single_mode:
        Wm = U
        mgen = torch.Generator(device=dev).manual_seed(77)
        Mm = torch.randn((P, U, Wm), generator=mgen, device=dev, dtype=tdt) / (U ** 0.5)
        mo = torch.empty((N, Wm, Do), device=dev, dtype=tdt)
        mg = torch.randn((N, Wm, Do), generator=mgen, device=dev, dtype=tdt)
        md_in, mdM = torch.empty_like(out), torch.empty_like(Mm)
        mws = torch.empty(max(plan.mix_workspace_bytes(N, Wm)), dtype=torch.uint8, device=dev)

        def ev_mix(fn, reps=10):
            for _ in range(3):
                fn()
            ts = []
            for _ in range(reps):
                a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                a.record(stream)
                fn()
                b.record(stream)
                ts.append((a, b))
            torch.cuda.synchronize()
            return statistics.median(a.elapsed_time(b) for a, b in ts)

        mf = ev_mix(lambda: plan.mix_fwd(N, Wm, out, Mm, mo, workspace=mws, stream=stream))
        mi = ev_mix(lambda: plan.mix_bwd(N, Wm, out, Mm, mg, d_in=md_in, workspace=mws, stream=stream))
        mM = ev_mix(lambda: plan.mix_bwd(N, Wm, out, Mm, mg, dM=mdM, workspace=mws, stream=stream))
        flops = 2.0 * N * U * Wm * Do
        line["mix"] = {"w_out": Wm, "flops_per_launch": flops,
                       "fwd_ms": mf, "bwd_d_in_ms": mi, "bwd_dM_ms": mM,
                       "fwd_tflops": flops / (mf / 1000) / 1e12, "bwd_d_in_tflops": flops / (mi / 1000) / 1e12,
                       "bwd_dM_tflops": flops / (mM / 1000) / 1e12,
                       "alu_peak_tflops": alu_peak, "fwd_alu_frac": flops / (mf / 1000) / 1e12 / alu_peak,
                       "note": "bound alu: fraction of the FP32 FMA rate measured in this run (alu_peaks)"}
        assert plan.device_status() == 0
        del Mm, mo, mg, md_in, mdM, mws

    # convolution with fused radial weights: the radial network (edge lengths -> hidden features
    # h, enveloped Bessel basis of 8 functions, three SiLU layers of 64) and the forward that forms
    # w = h W_last per (edge, channel) in registers.  Beside them the materialised alternative on
    # the same h: the last layer as one cuBLAS GEMM writing w [E][P][U] (FP32, and TF32 tensor
    # cores), then uvu_fwd reading it.  Inputs drawn on the device (seeded).
    if not args.no_radial and world == 1 and not args.single_mode:
        Hr, widths = 64, [8, 64, 64, 64]
        rgen = torch.Generator(device=dev).manual_seed(515)
        a3 = (0.75 / 5.0) ** 3
        rr = 5.0 * (a3 + (1 - a3) * torch.rand(E, generator=rgen, device=dev, dtype=torch.float64)) ** (1.0 / 3.0)
        rr = rr.to(tdt)
        Wn = torch.cat([(torch.randn((widths[i], widths[i + 1]), generator=rgen, device=dev, dtype=tdt)
                         / widths[i] ** 0.5).reshape(-1) for i in range(3)])
        Wlast = torch.randn((Hr, P, U), generator=rgen, device=dev, dtype=tdt) / Hr ** 0.5 / spec.w_scale_degree ** 0.5
        hbuf = torch.empty((E, Hr), device=dev, dtype=tdt)
        rout = torch.empty_like(out)
        reps = max(5, args.steps // 2)
        hid_ms = ev_mix(lambda: plan.radial_hidden(rr, 5.0, 5, widths, Wn, hbuf, stream=stream), reps)
        fus_ms = ev_mix(lambda: plan.fwd_radial(N, x, Y, hbuf, Wlast, G.recv_offsets, src, rout, stream=stream), reps)
        wmat = torch.empty((E, P * U), device=dev, dtype=tdt)
        tf32_prev = torch.backends.cuda.matmul.allow_tf32
        gemm = {}
        for name, tf in (("fp32", False), ("tf32", True)):
            torch.backends.cuda.matmul.allow_tf32 = tf
            gemm[name] = ev_mix(lambda: torch.matmul(hbuf, Wlast.view(Hr, P * U), out=wmat), reps)
        torch.backends.cuda.matmul.allow_tf32 = False
        torch.matmul(hbuf, Wlast.view(Hr, P * U), out=wmat)
        torch.backends.cuda.matmul.allow_tf32 = tf32_prev
        conv_ms = ev_mix(lambda: plan.fwd(N, x, Y, wmat.view(E, P, U), G.recv_offsets, src, out, stream), reps)
        torch.cuda.synchronize()
        rel = float(torch.linalg.vector_norm((rout - out).double()) / torch.linalg.vector_norm(out.double()))
        # the tensor-core path: the last layer materialised by uvu_radial_weights (3xTF32), then the
        # convolution; its VJP: uvu_conv_bwd's kernels with w, then the last layer's gradients (dh on
        # the tensor cores, dW_last on CUDA cores) and the network's reverse pass (dr, dW_i)
        rw_ws = torch.empty(max(16, plan.radial_weights_workspace(Hr)), dtype=torch.uint8, device=dev)
        tc_w_ms = ev_mix(lambda: plan.radial_weights(hbuf, Wlast, wmat.view(E, P, U), workspace=rw_ws, stream=stream), reps)
        wv = wmat.view(E, P, U)
        plan.radial_weights(hbuf, Wlast, wv, workspace=rw_ws, stream=stream)
        tc_conv_ms = ev_mix(lambda: plan.fwd(N, x, Y, wv, G.recv_offsets, src, out, stream), reps)
        rdw = torch.empty_like(wv)
        rdh = torch.empty_like(hbuf)
        rdWl = torch.empty_like(Wlast)
        rdr = torch.empty_like(rr)
        rdW = torch.empty_like(Wn)
        rws = torch.empty(max(16, plan.radial_weights_bwd_workspace(E, Hr)), dtype=torch.uint8, device=dev)
        rhws = torch.empty(max(16, plan.radial_hidden_bwd_workspace(E, widths)), dtype=torch.uint8, device=dev)

        def conv_vjp():
            plan.bwd_edge(N, x, Y, wv, G.recv_offsets, src, g, dY=dY, dw=rdw, dx_edge=ws, stream=stream)
            plan.bwd_dx_reduce(N, E, G.send_offsets, G.send_eids, ws, dx, stream)
        vjp_conv_ms = ev_mix(conv_vjp, reps)
        dh_ms = ev_mix(lambda: plan.radial_weights_bwd(hbuf, Wlast, rdw, dh=rdh, workspace=rws, stream=stream), reps)
        dWl_ms = ev_mix(lambda: plan.radial_weights_bwd(hbuf, Wlast, rdw, dw_last=rdWl, workspace=rws, stream=stream), reps)
        hb_ms = ev_mix(lambda: plan.radial_hidden_bwd(rr, 5.0, 5, widths, Wn, rdh, rdr, rdW, workspace=rhws,
                                                      stream=stream), reps)
        torch.backends.cuda.matmul.allow_tf32 = False
        cb_dh = ev_mix(lambda: torch.matmul(rdw.view(E, P * U), Wlast.view(Hr, P * U).t(), out=rdh), reps)
        cb_dWl = ev_mix(lambda: torch.matmul(hbuf.t(), rdw.view(E, P * U), out=rdWl.view(Hr, P * U)), reps)
        torch.backends.cuda.matmul.allow_tf32 = tf32_prev
        assert plan.device_status() == 0
        flops_last = 2.0 * E * U * P * Hr
        tf32_peak = float(peaks.get("bf16_tflops", 0.0)) / 2.0 if peaks.get("bf16_tflops") else None
        tc = {
            "weights_ms": tc_w_ms, "weights_GB_s": (E * P * U * s + E * Hr * s) / (tc_w_ms / 1000) / 1e9,
            "weights_hbm_frac": (E * P * U * s + E * Hr * s) / (tc_w_ms / 1000) / 1e9 / hbm_peak,
            "weights_tensor_tflops": 3 * flops_last / (tc_w_ms / 1000) / 1e12,
            "tf32_peak_tflops": tf32_peak,
            "conv_fwd_ms": tc_conv_ms, "fwd_total_ms": hid_ms + tc_w_ms + tc_conv_ms,
            "conv_vjp_ms": vjp_conv_ms, "dh_ms": dh_ms, "dw_last_ms": dWl_ms, "hidden_bwd_ms": hb_ms,
            "vjp_total_ms": vjp_conv_ms + dh_ms + dWl_ms + hb_ms,
            "fwd_vjp_total_ms": hid_ms + tc_w_ms + tc_conv_ms + vjp_conv_ms + dh_ms + dWl_ms + hb_ms,
            "cublas_fp32": {"weights_ms": gemm["fp32"], "dh_ms": cb_dh, "dw_last_ms": cb_dWl,
                            "fwd_vjp_total_ms": hid_ms + gemm["fp32"] + conv_ms + vjp_conv_ms + cb_dh + cb_dWl + hb_ms},
            "note": ("weights and dh on the tensor cores (tcgen05 kind::tf32, operands split hi + lo, three products "
                     "per term: fp32 accuracy; tensor flops = 3 x 2 E H P U); dW_last and the network's reverse pass "
                     "on CUDA cores (compensated sums over all edges); tf32 peak = measured bf16 dense / 2 (nominal "
                     "ratio); cublas_fp32 replaces the three products with cuBLAS FP32 GEMMs (library, comparison only)")}
        hid_flops = 2.0 * E * sum(widths[i] * widths[i + 1] for i in range(3))
        fused_bytes = E * U * Dx * s + E * Dy * s + E * Hr * s + N * U * Do * s + 4 * (N + 1) + 4 * E
        line["radial"] = {
            "hidden": widths, "r_cut": 5.0, "p_env": 5,
            "hidden_ms": hid_ms, "hidden_tflops": hid_flops / (hid_ms / 1000) / 1e12,
            "fused_fwd_ms": fus_ms, "fused_edges_per_s": E / (fus_ms / 1000),
            "fused_last_layer_tflops": flops_last / (fus_ms / 1000) / 1e12,
            "fused_last_layer_alu_frac": flops_last / (fus_ms / 1000) / 1e12 / alu_peak,
            "fused_bytes": fused_bytes, "fused_GB_s": fused_bytes / (fus_ms / 1000) / 1e9,
            "materialised": {"gemm_fp32_ms": gemm["fp32"], "gemm_tf32_ms": gemm["tf32"], "uvu_fwd_ms": conv_ms,
                             "w_bytes": E * P * U * s,
                             "total_fp32_ms": hid_ms + gemm["fp32"] + conv_ms,
                             "total_tf32_ms": hid_ms + gemm["tf32"] + conv_ms},
            "fused_total_ms": hid_ms + fus_ms,
            "tensor_core_path": tc,
            "rel_frobenius_vs_materialised_fp32": rel,
            "note": "alu bound: last-layer FMAs (2 E U P H flop) over the FP32 rate measured in this run; "
                    "the materialised GEMMs are cuBLAS (library), shown for comparison only"}
        assert plan.device_status() == 0
        del rr, Wn, Wlast, hbuf, rout, wmat, rdw, rdh, rdWl, rdr, rdW, rws, rhws, rw_ws

    # fwd and fwd+VJP (staged dx) of the other four workloads, each on its own plan and graph:
    # edges/s, GB/s of the compulsory bytes and the fraction of the HBM peak; for the fp64
    # workload also the FP64 arithmetic rate against the nominal FP64 peak.  w and d_out are
    # drawn on the device (seeded); inputs of workloads 2-4 exceed L2, workload 0 fits in it.
    if not args.no_configs and world == 1 and not args.single_mode and args.nodes is None:
        cfg_line = {}
        for key in [k for k in sorted(workloads.SPECS) if k != args.config]:
            sp = workloads.SPECS[key]
            wk = workloads.make_workload(key)
            wl_cache[key] = wk
            pk = uvu.Plan(sp.irreps_x, sp.irreps_sh, sp.lmax_out, sp.dtype)
            ik = pk.info
            Nk, Ek, Uk, Pk = wk.n_nodes, wk.n_edges, ik.mul, ik.n_paths
            dtk = torch.float64 if sp.dtype == "float64" else torch.float32
            sk = 8 if sp.dtype == "float64" else 4
            cgen = torch.Generator(device=dev).manual_seed(600 + key)
            xk, Yk = to_dev(wk.x), to_dev(wk.Y)
            srck = to_dev(wk.src)
            Gk = uvu.Graph(Nk, to_dev(wk.recv), srck)
            wkd = torch.randn((Ek, Pk, Uk), generator=cgen, device=dev, dtype=dtk) / sp.w_scale_degree ** 0.5
            gk = torch.randn((Nk, Uk, ik.dim_out), generator=cgen, device=dev, dtype=dtk)
            ok_, dxk = torch.empty((Nk, Uk, ik.dim_out), device=dev, dtype=dtk), torch.empty((Nk, Uk, ik.dim_x), device=dev, dtype=dtk)
            dYk, dwk = torch.empty((Ek, ik.dim_sh), device=dev, dtype=dtk), torch.empty_like(wkd)
            wsk = torch.empty(max(16, pk.workspace_bytes(Nk, Ek, uvu.UVU_DX_STAGED)), dtype=torch.uint8, device=dev)
            f_ms = ev_mix(lambda: pk.fwd(Nk, xk, Yk, wkd, Gk.recv_offsets, srck, ok_, stream), 10)

            def vjp_k():
                pk.bwd_edge(Nk, xk, Yk, wkd, Gk.recv_offsets, srck, gk, dY=dYk, dw=dwk, dx_edge=wsk, stream=stream)
                pk.bwd_dx_reduce(Nk, Ek, Gk.send_offsets, Gk.send_eids, wsk, dxk, stream)
            v_ms = ev_mix(vjp_k, 10)
            assert pk.device_status() == 0
            Bk = algorithmic_bytes(Nk, Ek, Uk, Pk, ik.dim_x, ik.dim_sh, ik.dim_out, sk)
            ent = {"workload": describe(sp, ik, Ek, Nk), "n_edges": Ek,
                   "fwd_ms": f_ms, "fwd_edges_per_s": Ek / (f_ms / 1000), "fwd_GB_s": frac(Bk["fwd"], f_ms)[0],
                   "fwd_hbm_frac": frac(Bk["fwd"], f_ms)[1], "vjp_ms": v_ms, "vjp_edges_per_s": Ek / (v_ms / 1000),
                   "vjp_GB_s": frac(Bk["vjp"], v_ms)[0], "vjp_hbm_frac": frac(Bk["vjp"], v_ms)[1],
                   "fwd_vjp_edges_per_s": Ek / ((f_ms + v_ms) / 1000), "fwd_bytes": Bk["fwd"], "vjp_bytes": Bk["vjp"],
                   "l2_resident": Bk["fwd"] < 129e6}
            if sp.dtype == "float64":
                # forward arithmetic from the plan's own CG: 2 flop per non-zero and per output
                # component (a nominal count: the generated forward executes fewer operations
                # where column scales turn coefficients into +-1)
                nnz = 0
                for pth in range(Pk):
                    nnz += int((pk.cg(pth) != 0).sum())
                ffl = 2.0 * Ek * Uk * (nnz + ik.dim_out)
                ent["fwd_fp64_tflops_estimate"] = ffl / (f_ms / 1000) / 1e12
                ent["fwd_fp64_frac_of_measured"] = ent["fwd_fp64_tflops_estimate"] / alu["fp64_tflops"]
                ent["fp64_peak_tflops_measured"] = alu["fp64_tflops"]
                ops = fp64_ops_per_edge_channel(pk)
                if ops:
                    ent["fwd_fp64_executed"] = {
                        "dfma_per_edge_channel": ops["dfma"], "dmul_dadd_per_edge_channel": ops["dmul"] + ops["dadd"],
                        "tflops": Ek * Uk * (2 * ops["dfma"] + ops["dmul"] + ops["dadd"]) / (f_ms / 1000) / 1e12,
                        "pipe_frac_of_measured": Ek * Uk * (ops["dfma"] + ops["dmul"] + ops["dadd"]) /
                                                 (f_ms / 1000) / (alu["fp64_tflops"] / 2 * 1e12),
                        "source": ops["source"]}
                ent["fp64_note"] = ("estimate = 2 E U (nnz + D_out) flop; fraction of the FP64 FMA rate measured "
                                    "in this run (alu_peaks)")
            cfg_line[sp.name] = ent
            del xk, Yk, srck, Gk, wkd, gk, ok_, dxk, dYk, dwk, wsk, pk
            torch.cuda.empty_cache()
        line["configs"] = cfg_line

    # batched (non-convolution) tensor product on the same irreps: B samples, per-sample and
    # batch-shared weights, forward and VJP (dx, dy, dw); inputs drawn on the device (seeded)
    if not args.no_tp and world == 1 and info.mul >= 32:
        Bt = args.tp_batch
        gen = torch.Generator(device=dev).manual_seed(4242)
        tx = torch.randn((Bt, U, Dx), generator=gen, device=dev, dtype=tdt)
        ty = torch.randn((Bt, Dy), generator=gen, device=dev, dtype=tdt)
        tg = torch.randn((Bt, U, Do), generator=gen, device=dev, dtype=tdt)
        tout, tdx, tdy = torch.empty_like(tg), torch.empty_like(tx), torch.empty_like(ty)

        def ev_ms(fn, reps):
            for _ in range(3):
                fn()
            ts = []
            for _ in range(reps):
                a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                a.record(stream)
                fn()
                b.record(stream)
                ts.append((a, b))
            torch.cuda.synchronize()
            return statistics.median(a.elapsed_time(b) for a, b in ts)

        xs_, ys_, os_ = Bt * U * Dx * s, Bt * Dy * s, Bt * U * Do * s
        tp_line = {"batch": Bt, "note": "x [B][U][D_x], y [B][D_Y], d_out ~ N(0,1) drawn on the device; "
                   "compulsory bytes: fwd reads x, y, w and writes out; VJP reads x, y, w, d_out and "
                   "writes dx, dy, dw"}
        reps = max(5, args.steps // 2)
        for mode, shared in (("per_sample", False), ("shared", True)):
            tw = torch.randn((P, U) if shared else (Bt, P, U), generator=gen, device=dev, dtype=tdt)
            tdw = torch.empty_like(tw)
            tws = torch.empty(max(16, plan.tp_workspace_bytes(Bt, shared)), dtype=torch.uint8, device=dev)
            wb = tw.numel() * s
            f_ms = ev_ms(lambda: plan.tp_fwd(Bt, tx, ty, tw, tout, w_shared=shared, stream=stream), reps)
            b_ms = ev_ms(lambda: plan.tp_bwd(Bt, tx, ty, tw, tg, dx=tdx, dy=tdy, dw=tdw, w_shared=shared,
                                             workspace=tws, stream=stream), reps)
            fb, bb = xs_ + ys_ + wb + os_, xs_ + ys_ + wb + os_ + xs_ + ys_ + wb
            f_gbs, f_fr = frac(fb, f_ms)
            b_gbs, b_fr = frac(bb, b_ms)
            tp_line[mode] = {"fwd_ms": f_ms, "fwd_samples_per_s": Bt / (f_ms / 1000), "fwd_GB_s": f_gbs,
                             "fwd_hbm_frac": f_fr, "vjp_ms": b_ms, "vjp_samples_per_s": Bt / (b_ms / 1000),
                             "vjp_GB_s": b_gbs, "vjp_hbm_frac": b_fr, "fwd_bytes": fb, "vjp_bytes": bb}
            del tw, tdw, tws
        assert plan.device_status() == 0
        line["tp"] = tp_line
        del tx, ty, tg, tout, tdx, tdy

    # double backward (HVP): gradients of <ax,dx> + <aY,dY> + <aw,dw>, timed on the same workload
    if not args.no_hvp and world == 1:
        gen = torch.Generator(device=dev).manual_seed(2026)
        ax = torch.randn(x.shape, generator=gen, device=dev, dtype=tdt)
        aY = torch.randn(Y.shape, generator=gen, device=dev, dtype=tdt)
        aw = torch.randn(w.shape, generator=gen, device=dev, dtype=tdt)
        hg, hx = torch.empty_like(out), torch.empty_like(dx)
        hY, hw = torch.empty_like(dY), torch.empty_like(dw)
        hws = torch.empty(max(1, plan.workspace_bytes(N, E, uvu.UVU_DX_STAGED)), dtype=torch.uint8, device=dev)

        def hvp_call(**outs):
            plan.hvp(N, x, Y, w, G.recv_offsets, src, G.send_offsets, G.send_eids, g, ax=ax, aY=aY,
                     aw=aw, workspace=hws, stream=stream, **outs)

        def ev_time(fn, reps):
            for _ in range(2):
                fn()
            ts = []
            for _ in range(reps):
                a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                a.record(stream)
                fn()
                b.record(stream)
                ts.append((a, b))
            torch.cuda.synchronize()
            return statistics.median(a.elapsed_time(b) for a, b in ts)

        reps = max(3, args.steps // 2)
        t_all = ev_time(lambda: hvp_call(grad_d_out=hg, grad_x=hx, grad_Y=hY, grad_w=hw), reps)
        t_fwd = ev_time(lambda: hvp_call(grad_d_out=hg), reps)
        t_edge = ev_time(lambda: hvp_call(grad_Y=hY, grad_w=hw), reps)
        xb, Yb, wb, ob = N * U * Dx * s, E * Dy * s, E * P * U * s, N * U * Do * s
        hvp_bytes = (2 * xb + 2 * Yb + 2 * wb + ob + 4 * (N + 1) * 2 + 8 * E) + (ob + xb + Yb + wb)
        gbs, fr = frac(hvp_bytes, t_all)
        line["hvp"] = {"ms": t_all, "edges_per_s": E / (t_all / 1000), "GB_s": gbs, "hbm_frac": fr,
                       "bytes": hvp_bytes, "kernels_ms": {"uvu_hvp_fwd": t_fwd, "uvu_hvp_edge": t_edge,
                                                          "uvu_bwd_dx_reduce": max(0.0, t_all - t_fwd - t_edge)},
                       "note": "gradients of <ax,dx>+<aY,dY>+<aw,dw> w.r.t. d_out, x, Y, w; compulsory "
                               "bytes: reads x,ax,Y,aY,w,aw,d_out,CSRs; writes the four gradients"}
        assert plan.device_status() == 0
        del ax, aY, aw, hg, hx, hY, hw, hws

    # end-to-end through the C ABI from pinned host buffers: every step copies its inputs (x, Y,
    # w, d_out and the graph arrays) in and its results (out, dx, dY, dw) out.  The receivers are
    # split into chunks whose copies and kernels are pipelined over three streams (copy in,
    # compute, copy out), using receiver sub-ranges of the same entry points (offsets are absolute
    # edge indices, so recv_offsets + r0 with n_nodes = r1 - r0 is a valid CSR for the chunk).
    if not args.no_e2e:
        pin = lambda t: t.cpu().pin_memory()
        hin = {"x": pin(x), "Y": pin(Y), "w": pin(w), "g": pin(g), "roff": pin(G.recv_offsets),
               "src": pin(src), "soff": pin(G.send_offsets), "seid": pin(G.send_eids),
               "srecv": pin(G.send_recv)}
        dbuf = {k: torch.empty_like(v, device=dev) for k, v in hin.items()}
        hout = {"out": pin(out), "dx": pin(dx), "dY": pin(dY), "dw": pin(dw)}
        h2d = sum(v.numel() * v.element_size() for v in hin.values())
        d2h = sum(v.numel() * v.element_size() for v in hout.values())
        roff_h = hin["roff"].numpy()
        # atomic dx is zeroed by the edge-kernel call, so that mode runs as one chunk
        K = 1 if args.dx_mode == "atomic" else max(1, min(args.e2e_chunks, N))
        cuts = [0]
        for i in range(1, K):  # equal edge counts per chunk
            cuts.append(int(np.searchsorted(roff_h, i * E / K)))
        cuts.append(N)
        cuts = sorted(set(cuts))
        s_in, s_cmp, s_out = torch.cuda.Stream(dev), stream, torch.cuda.Stream(dev)
        mode_e2e = args.dx_mode

        def e2e_step(s_cmp=s_cmp, capture=False):
            # s_cmp: the compute stream (the capturing stream when recorded into a CUDA graph);
            # the copy streams fork from it and join it again at the end
            ev_in, ev_cmp = [], []
            with torch.cuda.stream(s_in):
                if capture:
                    s_in.wait_stream(s_cmp)  # fork; replays of the graph run one after another
                else:
                    s_in.wait_stream(s_out)  # previous step's results are out before buffers are reused
                for k in ("x", "roff", "src", "soff", "seid", "srecv"):
                    dbuf[k].copy_(hin[k], non_blocking=True)
                for a, b in zip(cuts[:-1], cuts[1:]):
                    e0, e1 = int(roff_h[a]), int(roff_h[b])
                    dbuf["Y"][e0:e1].copy_(hin["Y"][e0:e1], non_blocking=True)
                    dbuf["w"][e0:e1].copy_(hin["w"][e0:e1], non_blocking=True)
                    dbuf["g"][a:b].copy_(hin["g"][a:b], non_blocking=True)
                    ev = torch.cuda.Event()
                    ev.record(s_in)
                    ev_in.append(ev)
            d = dbuf
            for i, (a, b) in enumerate(zip(cuts[:-1], cuts[1:])):
                s_cmp.wait_event(ev_in[i])
                n = b - a
                ro = d["roff"][a:]
                plan.fwd(n, d["x"], d["Y"], d["w"], ro, d["src"], out[a:], s_cmp)
                plan.bwd_edge(n, d["x"], d["Y"], d["w"], ro, d["src"], d["g"][a:], dY=dY, dw=dw,
                              dx_atomic=dx if mode_e2e == "atomic" else None,
                              dx_edge=ws if mode_e2e == "staged" else None, stream=s_cmp)
                ev = torch.cuda.Event()
                ev.record(s_cmp)
                ev_cmp.append(ev)
            if mode_e2e == "staged":
                plan.bwd_dx_reduce(N, E, d["soff"], d["seid"], ws, dx, s_cmp)
            elif mode_e2e == "sender":
                plan.bwd_dx(N, E, d["Y"], d["w"], d["soff"], d["seid"], d["srecv"], d["g"], dx, s_cmp)
            ev_dx = torch.cuda.Event()
            ev_dx.record(s_cmp)
            with torch.cuda.stream(s_out):
                for i, (a, b) in enumerate(zip(cuts[:-1], cuts[1:])):
                    s_out.wait_event(ev_cmp[i])
                    e0, e1 = int(roff_h[a]), int(roff_h[b])
                    hout["out"][a:b].copy_(out[a:b], non_blocking=True)
                    hout["dY"][e0:e1].copy_(dY[e0:e1], non_blocking=True)
                    hout["dw"][e0:e1].copy_(dw[e0:e1], non_blocking=True)
                s_out.wait_event(ev_dx)
                hout["dx"].copy_(dx, non_blocking=True)
            s_cmp.wait_stream(s_out)

        # device-resident results of one ordinary step, to check the chunked host path against
        step(args.dx_mode)
        torch.cuda.synchronize()
        ref = {k: v.clone() for k, v in dict(out=out, dx=dx, dY=dY, dw=dw).items()}
        for _ in range(2):
            e2e_step()
        torch.cuda.synchronize()
        same = all(torch.equal(hout[k], ref[k].cpu()) for k in ref) if args.dx_mode != "atomic" else None
        barrier(world)
        tw = time.perf_counter()
        issue = 0.0
        for _ in range(args.e2e_steps):
            ti = time.perf_counter()
            e2e_step()
            issue += time.perf_counter() - ti
        torch.cuda.synchronize()
        eager_ms = (time.perf_counter() - tw) * 1000 / args.e2e_steps
        issue_ms = issue * 1000 / args.e2e_steps
        # The same step recorded once into a CUDA graph (copies, the library's kernels and the
        # stream fork/join) and replayed: the host then issues one launch per step instead of
        # about a hundred, so a slow or busy host CPU no longer sets the step time.
        graph_ms, graph_err, graph_same = None, None, None
        try:
            cg = torch.cuda.CUDAGraph()
            cap = torch.cuda.Stream(dev)
            cap.wait_stream(stream)
            with torch.cuda.graph(cg, stream=cap):
                e2e_step(s_cmp=cap, capture=True)
            torch.cuda.synchronize()
            for v in hout.values():
                v.zero_()
            cg.replay()
            torch.cuda.synchronize()
            graph_same = all(torch.equal(hout[k], ref[k].cpu()) for k in ref) if args.dx_mode != "atomic" else None
            barrier(world)
            tw = time.perf_counter()
            for _ in range(args.e2e_steps):
                cg.replay()
            torch.cuda.synchronize()
            graph_ms = (time.perf_counter() - tw) * 1000 / args.e2e_steps
            del cg
        except Exception as ex:  # capture unsupported here: the eager step stands
            graph_err = f"{type(ex).__name__}: {ex}"[:200]
            torch.cuda.synchronize()
        del ref
        # The faster of the two launch modes is the step time (both are reported): on some boxes
        # the replayed graph's copy nodes ran the two copy directions one after the other
        # (20.6 ms against 13.1 ms eager in one driver run), on others replay was the faster.
        use_graph = graph_ms is not None and graph_same is not False and graph_ms <= eager_ms
        e_ms = max_over_ranks(graph_ms if use_graph else eager_ms, world, dev)
        # the results that came back are the full outputs of the step
        line["e2e"] = {"value": world * E / (e_ms / 1000), "unit": "edges/s",
                       "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": e_ms,
                       "launch": "cuda_graph" if use_graph else "eager",
                       "eager_ms_per_step": eager_ms, "eager_host_issue_ms_per_step": issue_ms,
                       "graph_ms_per_step": graph_ms, "graph_error": graph_err,
                       "chunks": len(cuts) - 1, "dx_mode": mode_e2e, "bitwise_equal_to_resident": same,
                       "graph_bitwise_equal_to_resident": graph_same,
                       "h2d_GB_s": h2d / (e_ms / 1000) / 1e9, "d2h_GB_s": d2h / (e_ms / 1000) / 1e9}

        # this machine's host link, measured the same way (pinned buffers, one large copy each way,
        # alone and concurrently): the ceiling the end-to-end step is bound by
        def link(fn, reps=3):
            fn()
            torch.cuda.synchronize()
            t0 = time.perf_counter()
            for _ in range(reps):
                fn()
            torch.cuda.synchronize()
            return (time.perf_counter() - t0) / reps

        wb = hin["w"].numel() * hin["w"].element_size()

        def h2d_only():
            with torch.cuda.stream(s_in):
                dbuf["w"].copy_(hin["w"], non_blocking=True)

        def d2h_only():
            with torch.cuda.stream(s_out):
                hout["dw"].copy_(dw, non_blocking=True)

        def both():
            h2d_only()
            d2h_only()

        t_h, t_d, t_b = link(h2d_only), link(d2h_only), link(both)
        line["e2e"]["link"] = {"h2d_GB_s": wb / t_h / 1e9, "d2h_GB_s": wb / t_d / 1e9,
                               "concurrent_each_way_GB_s": wb / t_b / 1e9, "bytes_per_copy": wb}
        line["e2e"]["frac_of_concurrent_link"] = ((h2d + d2h) / 2 / (e_ms / 1000)) / (wb / t_b)
        assert plan.device_status() == 0

    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        # the fp64 CPU oracle on this host's cores, per workload (fwd, VJP, fwd+VJP; median of
        # three runs of >= 2 s each), single-threaded too for the tiny and MACE-medium workloads
        from oracle import conv
        thr = conv.default_threads()
        keys = [args.config] + [k for k in sorted(workloads.SPECS) if k != args.config]
        per = cpu_baseline_protocol([(k, wl_cache.get(k)) for k in keys], thr)
        main = per[spec.name]["all_cores"]
        line["cpu_baseline"] = {"value": main["fwd_vjp_edges_per_s"], "unit": "edges/s", "cores": thr,
                                "kind": "oracle", "cpu_model": cpu_model(),
                                "sample": f"{spec.name}: " + main["sample"],
                                "per_workload": per}
    if rank == 0:
        print(json.dumps(line))
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
