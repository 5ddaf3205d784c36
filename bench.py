"""Benchmark of the INSTANT low-rank linear backward on one GB300 (or N replicas).

Headline workload: the long-sequence wide linear (4096 -> 11008, B=4, L=2048,
Rx=Ry=16, bf16 with fp32 accumulation, planted spectrum sigma_i ~ 1/i).  A step
is one training step of the layer through every row of the hot path:
activation compression (x_hat = P x), the one-read gradient projection, g_w,
g_hat_x and the rank-R expansion, captured as CUDA graphs over rotating buffer
sets.  Every N_t steps (default 100) the calibration phase runs eagerly: the
autocorrelation statistics of 64 samples (the step's batch plus resident
calibration samples) and the two eigen-solves that rewrite [P; Q].  It is
charged at 1/N_t of its measured time per step; the oracle arm charges its own
calibration the same way.

The BERT-base block, the BERT FFN pair and the ViT-MLP pair are measured the
same way (without the end-to-end and CPU legs) and reported under
``detail.workloads``.

Output: one JSON line (rank 0).  ``--impl reference`` times the fp64 CPU oracle
on a bounded sample of the same workload instead.
"""

from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "low-rank linear-backward layers/s and achieved HBM GB/s (% of roofline) on 1 GB300"
UNIT = "layers/s"
HEADLINE = "long_seq_4096_11008"
DETAIL_WORKLOADS = "bert_base_block,bert_ffn_pair,vit_mlp_pair_49"
L2_BYTES = 129 << 20


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=HEADLINE)
    ap.add_argument("--detail-workloads", default=DETAIL_WORKLOADS,
                    help="comma-separated workloads measured for detail.workloads ('' for none)")
    ap.add_argument("--nt", type=int, default=100, help="recalibration period N_t")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--kernel-iters", type=int, default=400)
    ap.add_argument("--e2e-steps", type=int, default=60)
    ap.add_argument("--cpu-baseline-only", action="store_true",
                    help="print the oracle's cpu_baseline object and exit (no GPU)")
    ap.add_argument("--mode", choices=["bench", "kernels", "profile", "drift"], default="bench",
                    help="kernels: after a first (cold) calibration, run one recalibration "
                         "period eagerly -- a warm-started calibration and N_t steps -- and "
                         "exit (the case ncu captures); prints the number of library launches "
                         "before the period as 'skip=N'; profile: each step kernel of the "
                         "workload's first layer and one accumulation of both statistics of "
                         "its batch, launched twice (a warm-up group, then the group a profiler "
                         "captures), with no calibration samples resident; drift: the "
                         "oversampling study on the "
                         "drifting ViT-MLP workload (reconstruction error per step for p in "
                         "0,2,4 and N_t in 5,10,100)")
    return ap.parse_args()


# ---------------------------------------------------------------------------
# distributed helpers (one process per GPU; replicas, no data-path collective)
# ---------------------------------------------------------------------------
def dist_env():
    return (int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")),
            int(os.environ.get("LOCAL_RANK", "0")))


def dist_init(backend: str):
    import torch.distributed as dist

    rank, world, _ = dist_env()
    if world > 1 and not dist.is_initialized():
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        dist.init_process_group(backend, rank=rank, world_size=world)
    return rank, world


def barrier():
    import torch.distributed as dist

    if dist.is_available() and dist.is_initialized():
        dist.barrier()


def max_over_ranks(x: float, device=None) -> float:
    import torch
    import torch.distributed as dist

    if not (dist.is_available() and dist.is_initialized()):
        return x
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def aggregate(elapsed_s: float, units_per_rank: float, world: int, device=None):
    """Whole-job throughput: all ranks' units over the slowest rank's time."""
    slowest = max_over_ranks(elapsed_s, device)
    return units_per_rank * world / slowest, slowest


# ---------------------------------------------------------------------------
# algorithmic bytes and flops per launch (compulsory reads + writes, bf16
# tensors and fp32 g_w; the intermediates Sx, Sq, g_hat_x count where a
# launch reads or writes them through HBM)
# ---------------------------------------------------------------------------
def layer_bytes(B, L, Cx, Cy, Rx, Ry):
    return {
        "compress_act": B * L * Cx * 2 + Rx * L * 2 + B * Rx * Cx * 2,
        "project_grad": B * L * Cy * 2 + (Rx + Ry) * L * 2 + B * (Rx + Ry) * Cy * 2,
        "grad_w": B * Rx * (Cy + Cx) * 2 + Cy * Cx * 4,
        "grad_x_core": B * Ry * Cy * 2 + Cy * Cx * 2 + B * Ry * Cx * 2,
        "expand": B * Ry * Cx * 2 + Ry * L * 2 + B * L * Cx * 2,
        "grad_x": B * Ry * Cy * 2 + Cy * Cx * 2 + Ry * L * 2 + B * L * Cx * 2,
        "grad_w_x": (B * Rx * (Cy + Cx) * 2 + Cy * Cx * 4
                     + B * Ry * Cy * 2 + Cy * Cx * 2 + Ry * L * 2 + B * L * Cx * 2),
        "backward": (B * L * Cy * 2 + (Rx + Ry) * L * 2 + B * (Rx + Ry) * Cy * 2
                     + B * Rx * Cx * 2 + Cy * Cx * 2 + Cy * Cx * 4 + B * L * Cx * 2),
    }


def layer_flops(B, L, Cx, Cy, Rx, Ry):
    return {
        "compress_act": 2 * B * Rx * L * Cx,
        "project_grad": 2 * B * (Rx + Ry) * L * Cy,
        "grad_w": 2 * B * Rx * Cy * Cx,
        "grad_x_core": 2 * B * Ry * Cy * Cx,
        "expand": 2 * B * Ry * L * Cx,
        "grad_x": 2 * B * Ry * Cy * Cx + 2 * B * Ry * L * Cx,
        "grad_w_x": 2 * B * Rx * Cy * Cx + 2 * B * Ry * Cy * Cx + 2 * B * Ry * L * Cx,
        "backward": (2 * B * (Rx + Ry) * L * Cy + 2 * B * Rx * Cy * Cx + 2 * B * Ry * Cy * Cx
                     + 2 * B * Ry * L * Cx),
    }


def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return {"hbm_gbs": float(d["hbm_gbs"]), "bf16_tflops": float(d["bf16_tflops"]),
                "bf16_tflops_sustained": float(d.get("bf16_tflops_sustained", d["bf16_tflops"])),
                "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
            "source": "fallback"}


KERNEL_SOURCES = {
    "compress_act": ("project.cu", "project_tile.cuh"),
    "project_grad": ("project.cu", "project_tile.cuh"),
    "grad_w": ("gemm.cu", "gradw_stream.cu"), "grad_x_core": ("gemm.cu",), "expand": ("expand.cu",),
    "grad_x": ("gradx_fused.cu", "project_tile.cuh"),
    "grad_w_x": ("gradx_fused.cu", "project_tile.cuh"),
    "backward": ("gradx_fused.cu", "project_tile.cuh"),
}


def source_hash(kernel: str) -> str:
    d = os.path.join(ROOT, "rank_compressed_backprop_gb300", "csrc")
    h = hashlib.sha256()
    for f in (*KERNEL_SOURCES[kernel], "tc.cuh", "kernels.h"):
        h.update(open(os.path.join(d, f), "rb").read())
    return h.hexdigest()[:16]


def ncu_traffic(kernel: str, workload: str):
    """DRAM bytes per launch recorded from an ncu capture of this kernel on
    this workload, if the kernel's sources are unchanged since; else None."""
    p = os.path.join(ROOT, "profiles", "ncu_traffic.txt")
    if not os.path.exists(p):
        return None
    for line in open(p):
        parts = line.split()
        if len(parts) >= 4 and parts[0] == kernel and parts[1] == workload:
            if parts[3] != source_hash(kernel):
                return None
            return float(parts[2])
    return None


class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons during a region."""

    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        # raw samples: $INSTANT_BENCH_CLOCKS_DIR if set (to keep them), else a temp file
        d = os.environ.get("INSTANT_BENCH_CLOCKS_DIR") or tempfile.gettempdir()
        self.path = os.path.join(d, f"instant_clocks_rank{index}_{os.getpid()}.csv")

    def __enter__(self):
        try:
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.Q}", "--format=csv,noheader",
                 "-lms", "50"], stdout=self.f, stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except (OSError, FileNotFoundError):
            self.proc = None
        return self

    def __exit__(self, *a):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.f.close()

    def summary(self):
        if self.proc is None or not os.path.exists(self.path):
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        sm, smax, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in open(self.path):
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1].split()[0]))
                smax = float(f[2].split()[0])
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": smax,
                "samples": len(sm), "reasons": sorted(reasons)}


# ---------------------------------------------------------------------------
# workloads
# ---------------------------------------------------------------------------
def workload_config(name: str, nt: int, world: int) -> dict:
    """The `config` object, identical in both arms."""
    import workloads as W

    wl = W.workload(name)
    layers = [list(c) for c in wl.layers]
    li = W.LayerInputs(wl, 0)
    step_bytes = sum(layer_bytes(wl.B, wl.L, cx, cy, wl.Rx, wl.Ry)["compress_act"]
                     + layer_bytes(wl.B, wl.L, cx, cy, wl.Rx, wl.Ry)["backward"]
                     for cx, cy in wl.layers)
    return {
        "workload": f"{wl.name}: B={wl.B} L={wl.L} layers {layers} (Cx, Cy) Rx=Ry={wl.Rx}, bf16 "
                    f"with fp32 accumulation, planted spectrum",
        "name": name,
        "B": wl.B, "L": wl.L, "Cx": li.Cx, "Cy": li.Cy, "Rx": wl.Rx, "Ry": wl.Ry,
        "layers": layers,
        "step": "per layer: compress_act + backward (the projection of g_y, then g_w and g_x)",
        "calibration_every": nt,
        "calibration_samples": wl.calib_samples, "calibration_p": wl.p, "eps": wl.eps,
        "calibration_charge": "1/N_t of the calibration phase's measured time per step",
        "l2": f"inputs larger than L2: one step reads and writes {step_bytes / 1e6:.0f} MB "
              f"of compulsory traffic (L2 {L2_BYTES >> 20} MB); rotating buffer sets",
        "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
    }


def to_dev(a, dev):
    import numpy as np
    import torch

    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).to(dev)


def resident_calibration(li, wl):
    """Host chunks of the calibration samples beyond the step's own batch:
    calib_samples - B samples in chunks of B (seeds j = 1, 2, ...)."""
    rest = max(0, wl.calib_samples - wl.B)
    xs, gs = [], []
    j = 1
    while rest > 0:
        n = min(wl.B, rest)
        xs.append(li.calib_x(j, n))
        gs.append(li.calib_g(j, n))
        rest -= n
        j += 1
    return xs, gs


class LayerBench:
    """One layer of a workload on the GPU: its InstantLinear, rotating buffer
    sets and resident calibration samples."""

    def __init__(self, wl, layer, dev, nsets_hint=None):
        import numpy as np
        import torch
        import workloads as W
        from rank_compressed_backprop_gb300 import InstantLinear

        li = W.LayerInputs(wl, layer)
        self.wl, self.li = wl, li
        self.B, self.L, self.Rx, self.Ry = wl.B, wl.L, wl.Rx, wl.Ry
        self.Cx, self.Cy = li.Cx, li.Cy
        bf = torch.bfloat16
        self.host = {"x": li.x(), "g": li.g_y(), "w": li.w()}
        self.w = to_dev(self.host["w"], dev)
        self.lay = InstantLinear(self.w, B=self.B, L=self.L, Rx=self.Rx, Ry=self.Ry, n_t=100,
                                 eps=wl.eps, p=wl.p)
        xs, gs = resident_calibration(li, wl)
        self.xc = torch.cat([to_dev(a, dev) for a in xs]) if xs else None
        self.gc = torch.cat([to_dev(a, dev) for a in gs]) if gs else None
        x0, g0 = to_dev(self.host["x"], dev), to_dev(self.host["g"], dev)
        B, L, Cx, Cy, Rx = self.B, self.L, self.Cx, self.Cy, self.Rx
        per_set = (B * L * (Cx + Cy) * 2 + B * Rx * Cx * 2 + Cy * Cx * 4 + B * L * Cx * 2)
        n = nsets_hint or int(min(8, max(3, math.ceil(600e6 / per_set))))
        self.sets = []
        for _ in range(n):
            self.sets.append({
                "x": x0.clone(), "g": g0.clone(),
                "xhat": torch.empty(B, Rx, Cx, dtype=bf, device=dev),
                "gw": torch.empty(Cy, Cx, dtype=torch.float32, device=dev),
                "gx": torch.empty(B, L, Cx, dtype=bf, device=dev),
            })
        del x0, g0
        self.set_bytes = per_set

    def accumulate(self, s):
        """The statistics of the step's batch and of the resident calibration
        samples."""
        self.lay.accumulate(s["x"], s["g"])
        if self.xc is not None:
            self.lay.accumulate(self.xc, self.gc)

    def calibrate(self, s):
        self.accumulate(s)
        return self.lay.recalibrate()

    def step(self, s):
        self.lay.compress(s["x"], out=s["xhat"])
        self.lay.backward(s["g"], xhat=s["xhat"], gw=s["gw"], gx=s["gx"])

    def kernels(self):
        """The library calls of the step, each alone (for per-kernel timing)."""
        from rank_compressed_backprop_gb300 import api

        lay, w, B, Rx, Ry, Cy = self.lay, self.w, self.B, self.Rx, self.Ry, self.Cy
        ws = lay.ws_gx
        return {
            "compress_act": lambda s: api.compress_act(s["x"], lay.P, s["xhat"]),
            "project_grad": lambda s: api.project_grad(s["g"], lay.PQ, lay.Sx, lay.Sq, Rx, Ry),
            "grad_w": lambda s: api.grad_w(lay.Sx, s["xhat"], s["gw"], B),
            "grad_x": lambda s: api.grad_x(lay.Sq, w, lay.Q, s["gx"], ws),
            "grad_w_x": lambda s: api.grad_w_x(lay.Sx, s["xhat"], s["gw"], lay.Sq, w, lay.Q, s["gx"],
                                               ws, B),
            "backward": lambda s: api.backward(s["g"], lay.PQ, s["xhat"], w, lay.Sx, lay.Sq, s["gw"],
                                               s["gx"], lay.ws_bw, Rx),
            "grad_x_core": lambda s: api.grad_x_core(lay.Sq, w, ws, B),
            "expand": lambda s: api.expand(lay.Q, s["gx"], ws, Cy),
        }


def graph_time_us(fn, sets, iters, stream):
    """Device time per call of `fn` from a CUDA graph of back-to-back calls over
    the rotating sets (no host launch overhead)."""
    import torch

    n = len(sets)
    per_graph = 5 * n
    for i in range(n):
        fn(sets[i])
    cs = torch.cuda.Stream()
    cs.wait_stream(torch.cuda.current_stream())
    kg = torch.cuda.CUDAGraph()
    with torch.cuda.stream(cs):
        with torch.cuda.graph(kg, stream=cs):
            for i in range(per_graph):
                fn(sets[i % n])
    torch.cuda.current_stream().wait_stream(cs)
    kg.replay()
    torch.cuda.synchronize()
    reps = max(1, iters // per_graph)
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(stream)
    for _ in range(reps):
        kg.replay()
    b.record(stream)
    torch.cuda.synchronize()
    return a.elapsed_time(b) * 1e3 / (reps * per_graph)


def kernel_figures(lb, kus, peaks):
    """Per-kernel achieved GB/s, TFLOP/s and roofline fractions: HBM fraction
    for every kernel, and for the two dense products the fraction of
    min(P_tc, AI * BW)."""
    nb = layer_bytes(lb.B, lb.L, lb.Cx, lb.Cy, lb.Rx, lb.Ry)
    nf = layer_flops(lb.B, lb.L, lb.Cx, lb.Cy, lb.Rx, lb.Ry)
    out = {}
    for k, us in kus.items():
        gbs = nb[k] / (us * 1e-6) / 1e9
        tf = nf[k] / (us * 1e-6) / 1e12
        d = {"us": round(us, 3), "gbs": round(gbs, 1), "hbm_frac": round(gbs / peaks["hbm_gbs"], 4),
             "tflops": round(tf, 2)}
        if k in ("grad_w", "grad_x_core"):
            ai = nf[k] / nb[k]
            bound = min(peaks["bf16_tflops"], ai * peaks["hbm_gbs"] / 1e3)
            d["ai_flop_per_byte"] = round(ai, 1)
            d["bound_tflops"] = round(bound, 1)
            d["bound_frac"] = round(tf / bound, 4)
        out[k] = d
    return out


def forward_figures(lb, args, stream, peaks):
    """The layer's forward y = x w^T with x_hat = P x from the same x tiles
    (one launch), against the same GEMM without the side output followed by
    compress_act (two launches); cuBLAS (torch.matmul) for context."""
    import torch
    from rank_compressed_backprop_gb300 import api

    B, L, Cx, Cy, Rx = lb.B, lb.L, lb.Cx, lb.Cy, lb.Rx
    lay = lb.lay
    y = torch.empty(B, L, Cy, dtype=torch.bfloat16, device=lay.w.device)
    ws = api.forward_workspace(B, L, Cx, Rx, torch.bfloat16, lay.w.device)
    sets = lb.sets
    fused = lambda s: api.forward(s["x"], lay.w, y, lay.P, s["xhat"], ws)  # noqa: E731
    alone = lambda s: api.forward(s["x"], lay.w, y)  # noqa: E731

    def separate(s):
        api.forward(s["x"], lay.w, y)
        api.compress_act(s["x"], lay.P, s["xhat"])

    def cublas(s):
        torch.matmul(s["x"].view(B * L, Cx), lay.w.t(), out=y.view(B * L, Cy))

    n0 = api.launch_count()
    fused(sets[0])
    fused_launches = api.launch_count() - n0
    iters = max(20, args.kernel_iters // 10)
    us = {k: graph_time_us(f, sets, iters, stream)
          for k, f in (("fused", fused), ("gemm_alone", alone), ("gemm_then_compress", separate),
                       ("cublas_matmul", cublas))}
    flops = 2.0 * B * L * Cx * Cy
    out = {"launches_fused": fused_launches}
    for k, v in us.items():
        tf = flops / (v * 1e-6) / 1e12
        out[k] = {"us": round(v, 2), "tflops": round(tf, 1),
                  "tensor_frac": round(tf / peaks["bf16_tflops"], 4)}
    return out


def step_kernels_of(lb):
    """The launches one step of this layer makes (compress, projection, and the
    single fused g_w+g_x launch or its three-launch form)."""
    from rank_compressed_backprop_gb300 import api

    s = lb.sets[0]
    c0 = api.launch_count()
    lb.kernels()["grad_w_x"](s)
    n = api.launch_count() - c0
    return ["compress_act", "project_grad"] + (["grad_w_x"] if n == 1 else
                                               ["grad_w", "grad_x_core", "expand"])


# ---------------------------------------------------------------------------
# our implementation
# ---------------------------------------------------------------------------
def measure_workload(name, args, dev, world, stream, full: bool):
    """Builds the workload's layers and measures: the timed loop (K steps,
    calibration every N_t charged at 1/N_t), per-kernel graph timings and the
    calibration's parts.  Returns a dict of results (plus the layer benches)."""
    import torch
    import workloads as W
    from rank_compressed_backprop_gb300 import api

    wl = W.workload(name)
    lbs = [LayerBench(wl, i, dev) for i in range(len(wl.layers))]
    nsets = min(len(lb.sets) for lb in lbs)

    # the layers of a model recalibrate at the same step: their statistics are
    # solved together (one batched call for all layers)
    from rank_compressed_backprop_gb300 import LayerCalibration
    layer_cal = LayerCalibration([lb.lay for lb in lbs])

    def calibrate(i):
        for lb in lbs:
            lb.accumulate(lb.sets[i % nsets])
        return layer_cal.recalibrate()

    def step(i):
        for lb in lbs:
            lb.step(lb.sets[i % nsets])

    cal0 = calibrate(0)
    for i in range(nsets):
        step(i)
    torch.cuda.synchronize()
    if args.mode == "kernels":
        print(f"skip={api.launch_count()}", flush=True)
        calibrate(0)
        for i in range(args.nt):
            step(i)
        torch.cuda.synchronize()
        if api.device_status() != 0:
            raise RuntimeError("device status set")
        print(f"period_launches={api.launch_count()}", flush=True)
        return None
    c0 = api.launch_count()
    step(0)
    launches_per_step = api.launch_count() - c0

    # one graph runs the step on each buffer set in turn; single-step graphs
    # cover a remainder
    cs = torch.cuda.Stream()
    cs.wait_stream(torch.cuda.current_stream())
    graphs = []
    with torch.cuda.stream(cs):
        gall = torch.cuda.CUDAGraph()
        with torch.cuda.graph(gall, stream=cs):
            for i in range(nsets):
                step(i)
        for i in range(nsets):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=cs):
                step(i)
            graphs.append(g)
    torch.cuda.current_stream().wait_stream(cs)
    torch.cuda.synchronize()

    def run_steps(first, count, cal_events=None):
        """Steps first..first+count-1; with cal_events, the calibration phase
        runs before the group holding a multiple of N_t, between two events."""
        i, end = first, first + count
        while i < end:
            n = nsets if (i % nsets == 0 and end - i >= nsets) else 1
            if cal_events is not None and any((j % args.nt) == 0 for j in range(i, i + n)):
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record(stream)
                calibrate(i)
                e1.record(stream)
                cal_events.append((e0, e1))
            if n == nsets:
                gall.replay()
            else:
                graphs[i % nsets].replay()
            i += n

    run_steps(0, max(args.warmup, 3))
    calibrate(0)  # warm path of the calibration (warm-started solve)
    torch.cuda.synchronize()

    # ---- timed region ----
    res = {"wl": wl, "lbs": lbs, "cal0": cal0, "nsets": nsets, "launches_per_step": launches_per_step}
    cal_events = []
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    clk = ClockSampler(torch.cuda.current_device()) if full else None
    if clk:
        clk.__enter__()
    barrier()
    torch.cuda.synchronize()
    lc0 = api.launch_count()
    start.record(stream)
    run_steps(0, args.steps, cal_events)
    end.record(stream)
    torch.cuda.synchronize()
    lc1 = api.launch_count()
    barrier()
    if clk:
        clk.__exit__(None, None, None)
        res["clocks"] = clk.summary()
    elapsed = start.elapsed_time(end) / 1e3
    cal_s = sum(a.elapsed_time(b) for a, b in cal_events) / 1e3
    n_cal = len(cal_events)
    step_s = elapsed - cal_s
    cal_avg = cal_s / n_cal
    charged = step_s + cal_avg * args.steps / args.nt
    res.update(elapsed_s=elapsed, cal_s=cal_s, n_cal=n_cal, step_s=step_s, cal_avg_s=cal_avg,
               charged_s=charged,
               gpu_launches=(lc1 - lc0) + launches_per_step * args.steps)
    res["value"], res["slowest_s"] = aggregate(charged, float(args.steps), world, dev)

    # ---- per-kernel device times (graphs of back-to-back launches) ----
    peaks = measured_peaks()
    per_layer = []
    for li, lb in enumerate(lbs):
        kus = {k: graph_time_us(fn, lb.sets[:nsets], args.kernel_iters, stream)
               for k, fn in lb.kernels().items()}
        per_layer.append({"layer": [lb.Cx, lb.Cy], "step_kernels": step_kernels_of(lb),
                          "kernels": kernel_figures(lb, kus, peaks)})
    res["per_layer"] = per_layer

    # ---- the step graph alone ----
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    nstep = max(nsets, int(200e3 / max(1.0, step_s * 1e6 / args.steps)) // nsets * nsets)
    a.record(stream)
    run_steps(0, nstep)
    b.record(stream)
    torch.cuda.synchronize()
    res["step_graph_us"] = a.elapsed_time(b) * 1e3 / nstep

    # ---- calibration parts: accumulation of every statistic (the tensor-bound
    # step) and the solves ----
    s0 = [lb.sets[0] for lb in lbs]
    for lb, s in zip(lbs, s0):
        lb.lay.accumulate(s["x"], s["g"])
        if lb.xc is not None:
            lb.lay.accumulate(lb.xc, lb.gc)
    reps = 5
    a.record(stream)
    for _ in range(reps):
        for lb, s in zip(lbs, s0):
            lb.lay.accumulate(s["x"], s["g"])
            if lb.xc is not None:
                lb.lay.accumulate(lb.xc, lb.gc)
    b.record(stream)
    torch.cuda.synchronize()
    acc_us = a.elapsed_time(b) * 1e3 / reps
    acc_flops = sum(wl.calib_samples * wl.L * (wl.L + 1) * (lb.Cx + lb.Cy) for lb in lbs)
    t0 = time.perf_counter()
    layer_cal.recalibrate()
    solve_ms = (time.perf_counter() - t0) * 1e3
    res["calibration_parts"] = {
        "accumulate_all_statistics_us": round(acc_us, 2),
        # upper triangle incl. the diagonal: L(L+1) flops per channel and sample
        "accumulate_tflops": round(acc_flops / (acc_us * 1e-6) / 1e12, 1),
        "accumulate_tensor_frac": round(acc_flops / (acc_us * 1e-6) / 1e12 / peaks["bf16_tflops"], 4),
        "accumulate_tensor_frac_of_sustained": round(
            acc_flops / (acc_us * 1e-6) / 1e12 / peaks["bf16_tflops_sustained"], 4),
        "solve_all_wall_ms": round(solve_ms, 3),
        "calibration_phase_ms": round(cal_avg * 1e3, 3),
    }
    if api.device_status() != 0:
        raise RuntimeError("device status set")
    return res


def run_ours(args):
    import torch

    rank, world, local = dist_env()
    if world > 1:
        torch.cuda.set_device(local)
    dist_init("nccl" if world > 1 else "gloo")
    dev = torch.device("cuda", torch.cuda.current_device())
    from rank_compressed_backprop_gb300.build import build

    build()
    import workloads as W

    stream = torch.cuda.current_stream()
    r = measure_workload(args.workload, args, dev, world, stream, full=True)
    if r is None:
        return
    wl, lbs = r["wl"], r["lbs"]
    peaks = measured_peaks()
    # roofline: the longest launch of the step (all of them HBM-bound here)
    cands = []
    for pl, lb in zip(r["per_layer"], lbs):
        for k in pl["step_kernels"]:
            cands.append((pl["kernels"][k]["us"], k, lb))
    _, dom, dlb = max(cands, key=lambda c: c[0])
    nbytes = layer_bytes(dlb.B, dlb.L, dlb.Cx, dlb.Cy, dlb.Rx, dlb.Ry)[dom]
    dus = [pl for pl in r["per_layer"] if pl["layer"] == [dlb.Cx, dlb.Cy]][0]["kernels"][dom]["us"]
    achieved = nbytes / (dus * 1e-6) / 1e9
    roofline = {"bound": "hbm", "kernel": dom, "achieved": round(achieved, 1),
                "peak": peaks["hbm_gbs"], "unit": "GB/s", "frac": round(achieved / peaks["hbm_gbs"], 4),
                "peak_source": peaks["source"] + " (burst copy)",
                "bytes_per_launch": nbytes, "us_per_launch": dus,
                "traffic": ncu_traffic(dom, args.workload)}

    e2e = run_e2e(args, lbs[0], dev) if len(lbs) == 1 else None
    fwd = forward_figures(lbs[0], args, stream, peaks)

    cpu = cpu1 = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline(args.workload, args.nt)
        cpu1 = cpu_baseline_1thread(args.workload, args.nt)

    details = {}
    for name in [n for n in args.detail_workloads.split(",") if n and n != args.workload]:
        d = measure_workload(name, args, dev, world, stream, full=False)
        details[name] = {
            "layers_per_s": round(d["value"] * len(d["lbs"]), 2),
            "steps_per_s": round(d["value"], 2),
            "ms_per_step": round(d["charged_s"] * 1e3 / args.steps, 5),
            "step_graph_us": round(d["step_graph_us"], 3),
            "calibration_phase_ms": round(d["cal_avg_s"] * 1e3, 3),
            "calibration_parts": d["calibration_parts"],
            "per_layer": d["per_layer"],
            "calibration_k": [[c.k for c in cl] for cl in d["cal0"]],
        }
        del d
        torch.cuda.empty_cache()

    lb = lbs[0]
    B, L, Cx, Cy, Rx, Ry = lb.B, lb.L, lb.Cx, lb.Cy, lb.Rx, lb.Ry
    nl = len(lbs)
    out = {
        "metric": METRIC, "value": round(r["value"] * nl, 2), "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(r["slowest_s"] * 1e3 / args.steps, 5),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded planted-spectrum activations and gradients)",
        "config": workload_config(args.workload, args.nt, world),
        "roofline": roofline,
        "cpu_baseline": cpu,
        "e2e": e2e,
        "gpu_launches": int(r["gpu_launches"]),
        "clocks": r.get("clocks"),
        "detail": {
            "per_layer": r["per_layer"],
            "step_graph_us": round(r["step_graph_us"], 3),
            "step_graph_layers_per_s": round(1e6 * nl / r["step_graph_us"], 1),
            "timed_region": {"elapsed_s": round(r["elapsed_s"], 5), "steps_s": round(r["step_s"], 5),
                             "calibrations": r["n_cal"], "calibration_s": round(r["cal_s"], 5),
                             "charged_s": round(r["charged_s"], 5)},
            "buffer_sets": r["nsets"], "set_bytes": lb.set_bytes,
            "calibration_parts": r["calibration_parts"],
            "cpu_baseline_1thread": cpu1,
            "launches_per_step": r["launches_per_step"],
            "calibration_k": [c.k for c in r["cal0"][0]],
            "flops_vanilla_per_layer": 4 * B * L * Cx * Cy,
            "flops_low_rank_per_layer": 2 * B * (Rx + Ry) * (Cx * Cy + L * Cx + L * Cy),
            "activation_memory_ratio": L / Rx,
            "peaks": peaks,
            "forward": fwd,
            "workloads": details,
        },
    }
    if rank == 0:
        print(json.dumps(out), flush=True)


def run_e2e(args, lb, dev):
    """Same metric through the public API, inputs from pinned host memory and
    results read back every step.  Three streams form a pipeline over two
    device buffer sets: while step i computes (InstantLinear.compress and
    .backward), the inputs of step i+1 go up and the results of step i-1 come
    down; events keep every buffer from being overwritten before it is
    consumed.  The calibration phase runs every N_t steps as in the timed
    loop and is charged the same way (1/N_t of its time per step)."""
    import numpy as np
    import torch

    lay = lb.lay
    x_h = torch.from_numpy(np.ascontiguousarray(lb.host["x"]).view(np.int16)).view(torch.bfloat16).pin_memory()
    g_h = torch.from_numpy(np.ascontiguousarray(lb.host["g"]).view(np.int16)).view(torch.bfloat16).pin_memory()
    nbuf = 2
    xs = [torch.empty_like(x_h, device=dev) for _ in range(nbuf)]
    gs = [torch.empty_like(g_h, device=dev) for _ in range(nbuf)]
    xh = [torch.empty_like(lay.xhat) for _ in range(nbuf)]
    gws = [torch.empty_like(lay.gw) for _ in range(nbuf)]
    gxs = [torch.empty_like(lay.gx) for _ in range(nbuf)]
    gw_h = [torch.empty(lay.gw.shape, dtype=torch.float32).pin_memory() for _ in range(nbuf)]
    gx_h = [torch.empty(lay.gx.shape, dtype=torch.bfloat16).pin_memory() for _ in range(nbuf)]
    s_c = torch.cuda.current_stream()
    s_in, s_out = torch.cuda.Stream(), torch.cuda.Stream()
    ev_in = [torch.cuda.Event() for _ in range(nbuf)]
    ev_c = [torch.cuda.Event() for _ in range(nbuf)]
    ev_out = [torch.cuda.Event() for _ in range(nbuf)]
    steps = args.e2e_steps
    cal_events = []

    def upload(i):
        k = i % nbuf
        with torch.cuda.stream(s_in):
            if i >= nbuf:
                s_in.wait_event(ev_c[k])  # step i-2 no longer reads set k
            xs[k].copy_(x_h, non_blocking=True)
            gs[k].copy_(g_h, non_blocking=True)
            ev_in[k].record(s_in)

    def compute(i, timed):
        k = i % nbuf
        s_c.wait_event(ev_in[k])
        if i >= nbuf:
            s_c.wait_event(ev_out[k])  # step i-2's results have been read back
        if i % args.nt == 0:
            # the step's batch plus the resident calibration samples, then the solve
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(s_c)
            lay.accumulate(xs[k], gs[k])
            if lb.xc is not None:
                lay.accumulate(lb.xc, lb.gc)
            lay.recalibrate()
            e1.record(s_c)
            if timed:
                cal_events.append((e0, e1))
        lay.compress(xs[k], out=xh[k])
        lay.backward(gs[k], xhat=xh[k], gw=gws[k], gx=gxs[k])
        ev_c[k].record(s_c)
        with torch.cuda.stream(s_out):
            s_out.wait_event(ev_c[k])
            gw_h[k].copy_(gws[k], non_blocking=True)
            gx_h[k].copy_(gxs[k], non_blocking=True)
            ev_out[k].record(s_out)

    def run(n, first, timed):
        upload(first)
        for i in range(first, first + n):
            if i + 1 < first + n:
                upload(i + 1)
            compute(i, timed)
        s_c.wait_event(ev_out[(first + n - 1) % nbuf])

    run(4, 1, False)
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier()
    torch.cuda.synchronize()
    a.record(s_c)
    s_in.wait_stream(s_c)
    s_out.wait_stream(s_c)
    run(steps, 0, True)
    b.record(s_c)
    torch.cuda.synchronize()
    el = a.elapsed_time(b) / 1e3
    cal = sum(e0.elapsed_time(e1) for e0, e1 in cal_events) / 1e3
    charged = el - cal + (cal / max(1, len(cal_events))) * steps / args.nt
    _, world, _ = dist_env()
    val, _ = aggregate(charged, float(steps), world, dev)
    return {"value": round(val, 2), "unit": UNIT,
            "h2d_bytes_per_step": x_h.numel() * 2 + g_h.numel() * 2,
            "d2h_bytes_per_step": gw_h[0].numel() * 4 + gx_h[0].numel() * 2,
            "steps": steps, "elapsed_s": round(el, 5), "calibration_s": round(cal, 5),
            "api": "InstantLinear.compress/backward (eager); per step the inputs are copied from "
                   "pinned host memory and g_w, g_x read back into pinned host memory, pipelined "
                   "over two buffer sets on separate copy streams; calibration every N_t charged "
                   "at 1/N_t"}


# ---------------------------------------------------------------------------
# the oracle on the host (cpu_baseline and the reference arm)
# ---------------------------------------------------------------------------
def _cores():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count()


class OracleSample:
    """The oracle's share of a workload: one sample of each layer's batch for
    the step, and one sample of x and g_y for the accumulation."""

    def __init__(self, name):
        import workloads as W

        self.wl = W.workload(name)
        self.layers = []
        for i in range(len(self.wl.layers)):
            li = W.LayerInputs(self.wl, i, B=1)
            self.layers.append({"x": li.x(), "g": li.g_y(), "w": li.w()})
        self.bs = 1

    def calibration(self, O, W):
        """Accumulation time per sample (both statistics of every layer) and
        the solve time; returns (acc_s_per_sample, solve_s, projectors)."""
        wl = self.wl
        t0 = time.perf_counter()
        Cs = [(O.accumulate_autocorrelation(d["x"]), O.accumulate_autocorrelation(d["g"]))
              for d in self.layers]
        t_acc = time.perf_counter() - t0
        t0 = time.perf_counter()
        proj = []
        for CX, CG in Cs:
            cx = O.calibrate(CX, self.bs, eps=wl.eps, p=wl.p, r_override=wl.Rx)
            cg = O.calibrate(CG, self.bs, eps=wl.eps, p=wl.p, r_override=wl.Ry)
            proj.append((W.f32_to_bf16_bits(cx["rows"]), W.f32_to_bf16_bits(cg["rows"])))
        t_solve = time.perf_counter() - t0
        return t_acc / self.bs, t_solve, proj

    def step(self, O, proj):
        for d, (Pb, Qb) in zip(self.layers, proj):
            O.low_rank_backward(d["x"], d["g"], d["w"], Pb, Qb)

    @property
    def frac(self):
        return self.bs / self.wl.B


def oracle_rates(name, nt, budget_s):
    """Oracle time of one whole step (scaled from the sample) and of one whole
    calibration phase (the accumulation scaled to calib_samples, plus the
    solve), on the host cores."""
    import oracle as O
    import workloads as W

    smp = OracleSample(name)
    acc_ps, t_solve, proj = smp.calibration(O, W)
    t_cal = acc_ps * smp.wl.calib_samples + t_solve
    smp.step(O, proj)  # warm
    n, t1 = 0, time.perf_counter()
    while True:
        smp.step(O, proj)
        n += 1
        if time.perf_counter() - t1 > budget_s or n >= 200:
            break
    t_step = (time.perf_counter() - t1) / n / smp.frac
    return smp, t_step, t_cal, acc_ps, t_solve, n


def cpu_baseline(name, nt, budget_s: float = 10.0):
    smp, t_step, t_cal, acc_ps, t_solve, n = oracle_rates(name, nt, budget_s)
    per_step = t_step + t_cal / nt
    nl = len(smp.wl.layers)
    return {"value": round(nl / per_step, 4), "unit": UNIT, "cores": _cores(), "kind": "oracle",
            "sample": f"fp64 numpy oracle: {n} steps on {smp.bs} of {smp.wl.B} samples per layer "
                      f"({t_step * smp.frac:.3f} s each, scaled to the batch); calibration: "
                      f"accumulation of one sample ({acc_ps:.2f} s) scaled to "
                      f"{smp.wl.calib_samples} + the solves ({t_solve:.2f} s), charged at 1/N_t "
                      f"(N_t={nt})"}


def cpu_baseline_1thread(name, nt: int):
    """The same oracle sample on one host thread (BLAS and OpenMP pinned to
    one thread in a child process, so that the parent's pools are untouched)."""
    env = dict(os.environ, OMP_NUM_THREADS="1", OPENBLAS_NUM_THREADS="1", MKL_NUM_THREADS="1",
               NUMEXPR_NUM_THREADS="1")
    cmd = [sys.executable, os.path.abspath(__file__), "--cpu-baseline-only", "--nt", str(nt),
           "--workload", name]
    try:
        r = subprocess.run(cmd, env=env, capture_output=True, text=True, timeout=600)
        line = [ln for ln in r.stdout.splitlines() if ln.startswith("{")][-1]
        d = json.loads(line)
        d["cores"] = 1
        return d
    except Exception as e:  # reported, not fatal: the all-core figure is the baseline
        return {"unavailable": f"{type(e).__name__}: {e}"[:200]}


def run_reference(args):
    """The oracle arm: same metric, config, unit and warm-up, on the host
    cores; K oracle steps on a one-sample share of each batch, plus the
    calibration phase (accumulation of a sample scaled to the calibration
    samples, and the solves) charged at 1/N_t per step as in the GPU arm."""
    rank, world, _ = dist_env()
    if rank != 0:
        return
    import oracle as O
    import workloads as W

    smp = OracleSample(args.workload)
    acc_ps, t_solve, proj = smp.calibration(O, W)
    t_cal = acc_ps * smp.wl.calib_samples + t_solve
    for _ in range(args.warmup):
        smp.step(O, proj)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        smp.step(O, proj)
    t_steps = (time.perf_counter() - t0) / smp.frac
    charged = t_steps + t_cal * args.steps / args.nt
    nl = len(smp.wl.layers)
    value = nl * args.steps / charged
    sample = (f"{args.steps} oracle steps on {smp.bs} of {smp.wl.B} samples per layer "
              f"({t_steps * smp.frac / args.steps:.3f} s each, scaled to the batch); calibration: "
              f"accumulation of one sample ({acc_ps:.2f} s) scaled to {smp.wl.calib_samples} + the "
              f"solves ({t_solve:.2f} s), charged at 1/N_t (N_t={args.nt})")
    out = {"impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": UNIT,
           "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
           "ms_per_step": round(charged * 1e3 / args.steps, 3), "higher_is_better": True,
           "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
           "config": workload_config(args.workload, args.nt, world),
           "cpu_baseline": {"value": round(value, 4), "unit": UNIT, "cores": _cores(),
                            "kind": "oracle", "sample": sample},
           "e2e": {"value": round(value, 4), "unit": UNIT, "h2d_bytes_per_step": 0,
                   "d2h_bytes_per_step": 0}}
    print(json.dumps(out), flush=True)


def run_profile(args):
    """Two groups of the step's launches on the first layer of the workload
    (compress_act, project_grad, grad_w, grad_x_core, expand, one accumulation
    of both statistics of the step's batch, and the forward with x_hat), the
    second for a profiler to capture; the projector is the one calibrated from
    the step's own batch."""
    import torch
    import workloads as W
    from rank_compressed_backprop_gb300.build import build

    build()
    from rank_compressed_backprop_gb300 import InstantLinear, api

    wl = W.workload(args.workload)
    li = W.LayerInputs(wl, 0)
    dev = torch.device("cuda", torch.cuda.current_device())
    x, g, w = to_dev(li.x(), dev), to_dev(li.g_y(), dev), to_dev(li.w(), dev)
    B, L, Cx, Cy, Rx, Ry = wl.B, wl.L, li.Cx, li.Cy, wl.Rx, wl.Ry
    lay = InstantLinear(w, B=B, L=L, Rx=Rx, Ry=Ry, eps=wl.eps, p=wl.p)
    lay.accumulate(x, g)
    lay.recalibrate()
    y = torch.empty(B, L, Cy, dtype=torch.bfloat16, device=dev)
    wsf = api.forward_workspace(B, L, Cx, Rx, torch.bfloat16, dev)
    order = ["compress_act", "project_grad", "grad_w", "grad_x_core", "expand", "accumulate",
             "forward"]

    def group():
        api.compress_act(x, lay.P, lay.xhat)
        api.project_grad(g, lay.PQ, lay.Sx, lay.Sq, Rx, Ry)
        api.grad_w(lay.Sx, lay.xhat, lay.gw, B)
        api.grad_x_core(lay.Sq, w, lay.ws_gx, B)
        api.expand(lay.Q, lay.gx, lay.ws_gx, Cy)
        api.calib_accumulate_batch([(x, lay.C_X), (g, lay.C_G)])
        api.forward(x, w, y, lay.P, lay.xhat, wsf)

    torch.cuda.synchronize()
    c0 = api.launch_count()
    group()
    torch.cuda.synchronize()
    per_group = api.launch_count() - c0
    group()
    torch.cuda.synchronize()
    if api.device_status() != 0:
        raise RuntimeError("device status set")
    print(json.dumps({"mode": "profile", "workload": args.workload, "order": order,
                      "launches_per_group": per_group}), flush=True)


def run_drift(args):
    """Oversampling under subspace drift: per-step ||g - Q^T Q g|| / ||g|| on the
    first layer of the drifting ViT-MLP workload, for p in {0, 2, 4} and
    N_t in {5, 10, 100}, every computation in the CUDA library."""
    import torch
    import workloads as W
    from rank_compressed_backprop_gb300.build import build

    build()
    from rank_compressed_backprop_gb300 import api
    from rank_compressed_backprop_gb300.drift import drift_errors

    wl = W.workload("vit_mlp_pair_49")
    li = W.LayerInputs(wl)
    dev = torch.device("cuda", torch.cuda.current_device())
    steps = wl.steps
    batches = [to_dev(li.g_y(t), dev) for t in range(steps)]
    B, L, C = batches[0].shape
    table = {}
    for p in (0, 2, 4):
        for n_t in (5, 10, 100):
            drift_errors(lambda t: batches[t], 2, n_t, p, eps=wl.eps)  # warm-up
            torch.cuda.synchronize()
            t0 = time.perf_counter()
            run = drift_errors(lambda t: batches[t], steps, n_t, p, eps=wl.eps)
            torch.cuda.synchronize()
            el = time.perf_counter() - t0
            table[f"p={p},N_t={n_t}"] = {
                "errors": [round(e, 5) for e in run.errors],
                "mean": round(sum(run.errors) / len(run.errors), 5),
                "last": round(run.errors[-1], 5),
                "calibrations": [list(c) for c in run.calibrations],
                "ms_per_step": round(el * 1e3 / steps, 3),
            }
    # the reconstruction-error kernel alone (reads g once plus the projected rows)
    Q = torch.zeros(8, L, dtype=batches[0].dtype, device=dev)
    Q[:, :8] = torch.eye(8, dtype=batches[0].dtype, device=dev)
    S = torch.empty(B, 8, C, dtype=batches[0].dtype, device=dev)
    ws = torch.empty(16, dtype=torch.uint8, device=dev)
    api.compress_act(batches[0], Q, S)
    reps = 20
    for i in range(3):
        api.reconstruction_error(batches[i], Q, S.view(B * 8, C), ws)
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record()
    for i in range(reps):
        api.reconstruction_error(batches[i % steps], Q, S.view(B * 8, C), ws)
    b.record()
    torch.cuda.synchronize()
    us = a.elapsed_time(b) * 1e3 / reps
    nbytes = B * L * C * 2 + B * 8 * C * 2
    print(json.dumps({
        "mode": "drift",
        "workload": f"ViT-MLP first layer g_y [{B}, {L}, {C}] bf16, planted rank-6 spectrum plus "
                    f"noise, token basis rotated by a seeded Givens angle of {wl.drift_angle} rad "
                    f"per step, {steps} steps, eps={wl.eps}",
        "table": table,
        "recon_kernel": {"us_per_call_incl_sync": round(us, 2), "bytes": nbytes,
                         "gbs_incl_sync": round(nbytes / (us * 1e-6) / 1e9, 1)},
    }), flush=True)


def main():
    args = parse()
    if args.cpu_baseline_only:
        print(json.dumps(cpu_baseline(args.workload, args.nt, budget_s=8.0)))
        return
    if args.mode == "drift":
        run_drift(args)
    elif args.mode == "profile":
        run_profile(args)
    elif args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
