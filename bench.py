#!/usr/bin/env python
"""Benchmark of the weight-only quantized matmul + AddRmsNorm on one B300.

A step is one call of the fused operator (dequant-matmul + bias + residual +
RMSNorm, through the C ABI) on one batch of seeded synthetic inputs whose packed
INT4/INT8 weights are already resident, as a deployed layer's weights are. The
INT32 -> INT4 pack runs once per weight; it is timed in the same run and
reported under "pack".

Default workload: the largest single-GPU configuration, the M-sweep's
M = 16384 point (bf16, 16384 x 8192 x 28672, INT4 per-group g = 128).
``--config`` picks another: tiny, decode, w8a16, prefill, sweep:<M>,
sweep_pt:<M>. Unless ``--no-extra``, the same line also carries short
device-timed runs of the other named workloads (decode, prefill, W8A16 and the
sweep's M = 1 and 16) under "workloads".

L2: every step uses the next of R distinct input sets (weights included) whose
total size exceeds twice the L2 size, so no step finds its weights in L2; a
set larger than that is used alone.

Timing: W eager warm-up steps, then the K timed steps are replayed from a CUDA
graph (capture of the same C-ABI calls), bracketed by a barrier and a device
synchronize, timed with CUDA events on the launching stream; max over ranks.
``e2e`` repeats the steps with each step's inputs copied from pinned host
memory and both outputs copied back inside the timed region, captured into
CUDA graphs with the copies in, the call and the copies out on three streams
(step i+1's inputs travel while step i computes; event edges keep every input
set until its call and its outputs have been read), as a serving loop issues
them; eager calls on one stream if the capture is refused.

Multi-GPU (torchrun): "replicas only" -- each rank runs its own copy of the
workload, with no collective on the data path; value = all ranks' FLOPs / the
slowest rank's time.

``--impl reference`` times the fp64 CPU oracle (the plain restatement of the
operator used by the tests) on a bounded row sample of the same workload.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import torch  # noqa: E402

METRIC = "dequant-GEMM+AddRmsNorm TFLOP/s, weight GB/s, % of B300 roofline"
PEAKS_FALLBACK = {"hbm_gbs": 6400.0, "bf16_tflops": 1800.0, "bf16_tflops_sustained": 1400.0}


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=None)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--config", default="sweep:16384")
    ap.add_argument("--kernel", choices=["auto", "generic", "decode", "prefill"], default="auto")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-pack", action="store_true")
    ap.add_argument("--no-extra", action="store_true")
    return ap.parse_args()


# ------------------------------------------------------------------ workload

def make_problem(config: str, device):
    from weight_only_bit_pack_b300 import inputs
    config = config.split("@")[0]  # "@tiled", "@transposed": same workload, weight layout
    if config in inputs.CONFIGS:
        return inputs.CONFIGS[config](device)
    if config.startswith("sweep_pt:"):
        return inputs.sweep(int(config.split(":")[1]), per_tensor=True, device=device)
    if config.startswith("sweep:"):
        return inputs.sweep(int(config.split(":")[1]), device=device)
    raise SystemExit(f"unknown config {config}")


def default_steps(config: str) -> int:
    if config in ("sweep:16384", "sweep_pt:16384"):
        return 30
    return {"tiny": 2000, "decode": 20000, "w8a16": 200, "prefill": 40}.get(
        config, 20000 if config.endswith(":1") or config.endswith(":16") else 100)


def alg_bytes(p) -> dict:
    """Algorithmic bytes of one call: every input read once, every output written once."""
    dt = 2
    w = p.K * p.N * p.wbits // 8
    so = p.scale.numel() * dt * (2 if p.offset is not None else 1)
    vec = p.N * dt * (2 if p.bias is not None else 1)
    act = p.M * p.K * dt + p.M * p.N * dt * 3  # x1, residual, y, normOut
    return {"weight": w, "scale_offset": so, "vectors": vec, "activations": act,
            "total": w + so + vec + act}


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return d, "measured"
    except OSError:
        return dict(PEAKS_FALLBACK), "fallback"


# ------------------------------------------------------------------ clocks

class ClockSampler:
    """Samples SM clock and throttle reasons through NVML while running."""

    REASONS = {0x8: "hw_slowdown", 0x40: "hw_thermal_slowdown", 0x20: "sw_thermal_slowdown",
               0x4: "sw_power_cap", 0x80: "hw_power_brake_slowdown", 0x1: "gpu_idle"}

    def __init__(self, device, period_s: float = 0.005):
        self.samples = []
        self.reasons = set()
        self.period = period_s
        self.stop_ev = threading.Event()
        self.max_mhz = None
        self.err = None
        self.proc = None
        uuid = str(torch.cuda.get_device_properties(device).uuid)
        self.uuid = uuid if uuid.startswith("GPU-") else "GPU-" + uuid
        try:
            import pynvml
            pynvml.nvmlInit()
            self.nv = pynvml
            self.h = pynvml.nvmlDeviceGetHandleByUUID(self.uuid)
            self.max_mhz = pynvml.nvmlDeviceGetMaxClockInfo(self.h, pynvml.NVML_CLOCK_SM)
        except Exception as e:  # noqa: BLE001 - no NVML binding: sample nvidia-smi instead
            self.nv = None
            self.err = f"pynvml unavailable ({e}); sampled nvidia-smi"
        self.th = threading.Thread(target=self._run, daemon=True)

    def _sample(self):
        mhz = self.nv.nvmlDeviceGetClockInfo(self.h, self.nv.NVML_CLOCK_SM)
        r = self.nv.nvmlDeviceGetCurrentClocksEventReasons(self.h)
        self.samples.append(mhz)
        for bit, name in self.REASONS.items():
            if r & bit and name != "gpu_idle":
                self.reasons.add(name)

    def _run(self):
        while not self.stop_ev.is_set():
            try:
                self._sample()
            except Exception:  # noqa: BLE001
                break
            time.sleep(self.period)

    SMI_FIELDS = ("clocks.sm,clocks.max.sm,clocks_event_reasons.hw_slowdown,"
                  "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
                  "clocks_event_reasons.sw_power_cap")

    def _smi_cmd(self, loop):
        cmd = ["nvidia-smi", "-i", self.uuid, f"--query-gpu={self.SMI_FIELDS}",
               "--format=csv,noheader,nounits"]
        return cmd + (["-lms", "20"] if loop else [])

    def _parse_smi(self, text):
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in text.splitlines():
            f = [x.strip() for x in line.split(",")]
            if len(f) < 6:
                continue
            try:
                self.samples.append(float(f[0]))
                self.max_mhz = float(f[1])
            except ValueError:
                continue
            for name, v in zip(names, f[2:6]):
                if v.lower() == "active":
                    self.reasons.add(name)

    def __enter__(self):
        if self.nv:
            self.th.start()
        else:
            import subprocess
            try:
                self.proc = subprocess.Popen(self._smi_cmd(True), stdout=subprocess.PIPE,
                                             stderr=subprocess.DEVNULL, text=True)
            except OSError as e:
                self.err = f"no NVML and no nvidia-smi: {e}"
        return self

    def __exit__(self, *a):
        if self.nv:
            self.stop_ev.set()
            self.th.join()
            if not self.samples:
                try:
                    self._sample()
                except Exception:  # noqa: BLE001
                    pass
        elif self.proc is not None:
            import subprocess
            self.proc.terminate()
            out, _ = self.proc.communicate(timeout=10)
            self._parse_smi(out)
            if not self.samples:  # region shorter than one sampling period
                r = subprocess.run(self._smi_cmd(False), capture_output=True, text=True)
                self._parse_smi(r.stdout)

    def summary(self):
        d = {"sm_mhz": statistics.median(self.samples) if self.samples else None,
             "sm_max_mhz": self.max_mhz, "reasons": sorted(self.reasons),
             "samples": len(self.samples)}
        if self.err:
            d["note"] = self.err
        return d


# ------------------------------------------------------------------ distributed

def dist_setup(args):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        return world, rank, local  # rank 0 alone runs the CPU oracle; no process group
    torch.cuda.set_device(local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group(backend="nccl")
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(world, value: float) -> float:
    if world == 1:
        return value
    import torch.distributed as dist
    dev = "cuda" if torch.cuda.is_available() and dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([value], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ------------------------------------------------------------------ CPU oracle

def oracle_sample(p, target_flops: float):
    """Row sample of the workload whose fp64 oracle cost is about target_flops."""
    per_row = 2.0 * p.K * p.N
    rows = max(1, min(p.M, int(target_flops // per_row)))
    return list(range(rows))


def run_oracle_rows(p, rows, cpu_cache):
    import oracle
    if "x2" not in cpu_cache:
        cpu_cache["x2"] = p.x2.to("cpu").to(torch.int32)
        for f in ("scale", "offset", "bias", "gamma"):
            v = getattr(p, f)
            cpu_cache[f] = None if v is None else v.to("cpu")
        cpu_cache["x1"] = p.x1.reshape(-1, p.K)[: max(rows) + 1].to("cpu")
        cpu_cache["res"] = p.residual.reshape(-1, p.N)[: max(rows) + 1].to("cpu")
    c = cpu_cache
    return oracle.matmul_add_rmsnorm(c["x1"][rows], c["x2"], c["scale"], c["offset"], c["bias"],
                                     c["res"][rows], c["gamma"], p.eps, p.group)


def cores_used():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count()


def cpu_baseline(p, seconds=10.0, max_reps=200):
    rows = oracle_sample(p, 2e9)
    cache = {}
    run_oracle_rows(p, rows, cache)  # load + first call (untimed)
    t0 = time.perf_counter()
    reps = 0
    while True:
        run_oracle_rows(p, rows, cache)
        reps += 1
        el = time.perf_counter() - t0
        if el >= seconds or reps >= max_reps:
            break
    flops = 2.0 * len(rows) * p.K * p.N * reps
    return {"value": flops / el / 1e12, "unit": "TFLOP/s", "cores": cores_used(), "kind": "oracle",
            "sample": f"{len(rows)} of {p.M} rows x {reps} repetitions ({el:.1f} s, fp64 C oracle)"}


# ------------------------------------------------------------------ our arm

def layout_of(config):
    """Weight layout named by a config's suffix: "@tiled", "@transposed", else dense."""
    return config.split("@")[1] if "@" in config else "dense"


def layout_suffix(layout):
    return "" if layout == "dense" else "_" + layout


class Runner:
    """R distinct input sets of one workload on the device (weights packed once,
    then copied), a zeroed workspace, and step(i) = one C-ABI call on set i % R."""

    def __init__(self, wq, p, kernel, dev, stream, layout="dense"):
        self.p, self.kernel, self.stream = p, kernel, stream
        self.layout, self.tiled = layout, layout == "tiled"
        tiled = self.tiled
        self.w_src = p.x2
        if tiled:
            self.w0 = wq.pack_int4_tiled(p.x2)
        elif layout == "transposed":
            self.w0 = wq.TransposedWeight(wq.pack_int4(p.x2.t().contiguous()), 4)
        else:
            self.w0 = wq.pack_int4(p.x2) if p.wbits == 4 else p.x2.contiguous()
        self.ab = alg_bytes(p)
        l2 = torch.cuda.get_device_properties(dev).L2_cache_size
        self.set_bytes = self.ab["total"]
        R = 1 if self.set_bytes > 2 * l2 else int(math.ceil(2 * l2 / self.set_bytes)) + 1
        self.R = max(1, min(R, 64))
        self.sets = []
        for i in range(self.R):
            if tiled:
                w = wq.TiledInt4(self.w0.data.clone(), self.w0.K, self.w0.N)
            elif layout == "transposed":
                w = wq.TransposedWeight(self.w0.data.clone(), 4)
            else:
                w = self.w0.clone()
            s = {"x1": p.x1.clone(), "w": w, "scale": p.scale.clone(),
                 "offset": None if p.offset is None else p.offset.clone(),
                 "bias": None if p.bias is None else p.bias.clone(),
                 "residual": p.residual.clone(), "gamma": p.gamma.clone(),
                 "y": torch.empty_like(p.residual), "normOut": torch.empty_like(p.residual)}
            self.sets.append(s)
        ws_bytes = wq.matmul_add_rmsnorm_get_workspace(p.x1, self.w0, p.scale, p.offset, p.bias,
                                                       p.residual, p.gamma, p.eps, p.group,
                                                       kernel=kernel)
        self.ws = torch.zeros(max(ws_bytes, 2048), dtype=torch.uint8, device=dev)  # header zeroed once
        self.chosen = int(wq.select_kernel(p.x1, self.w0, p.scale, p.offset, p.bias, p.residual,
                                           p.gamma, p.eps, p.group)) if kernel == 0 else kernel
        self.wq = wq

    def step(self, i):
        s, p = self.sets[i % self.R], self.p
        self.wq.matmul_add_rmsnorm(s["x1"], s["w"], s["scale"], s["offset"], s["bias"],
                                   s["residual"], s["gamma"], p.eps, p.group, y=s["y"],
                                   normOut=s["normOut"], workspace=self.ws, kernel=self.kernel,
                                   stream=self.stream)

    def kernels_per_call(self) -> int:
        """Our kernel launches per call: generic = matmul + epilogue; decode = one;
        prefill = the tcgen05 kernel plus its row pre-pass (per-group scales, or an
        offset) and its scale pre-pass (per-group scales)."""
        p = self.p
        if self.chosen == 3:
            return 1 + (1 if (p.group or p.offset is not None) else 0) + (1 if p.group else 0)
        return {1: 2, 2: 1}.get(self.chosen, 2)

    def l2_note(self) -> str:
        if self.R > 1:
            return f"rotating {self.R} distinct input sets, {self.R * self.set_bytes / 1e6:.0f} MB > 2x L2"
        return f"one input set of {self.set_bytes / 1e6:.0f} MB > 2x L2"


def capture_graphs(runner, K):
    """The K steps captured into CUDA graphs (chunks of at most 1000 calls)."""
    graphs, done = [], 0
    while done < K:
        n = min(1000, K - done)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=runner.stream):
            for i in range(done, done + n):
                runner.step(i)
        graphs.append(g)
        done += n
    return graphs


def roofline(p, ms_step, peaks):
    ab = alg_bytes(p)
    t_s = ms_step * 1e-3
    flops = 2.0 * p.M * p.K * p.N
    if ab["total"] / (peaks["hbm_gbs"] * 1e9) >= flops / (peaks["bf16_tflops"] * 1e12):
        roof = {"bound": "hbm", "achieved": ab["total"] / t_s / 1e9, "peak": peaks["hbm_gbs"],
                "unit": "GB/s"}
    else:
        roof = {"bound": "tensor", "achieved": flops / t_s / 1e12, "peak": peaks["bf16_tflops"],
                "unit": "TFLOP/s"}
    roof["frac"] = roof["achieved"] / roof["peak"]
    return roof


def time_extra(wq, config, dev, stream, steps, warmup, peaks):
    """Device time of one named workload (graph replay, CUDA events), for the
    line's "workloads" key."""
    p = make_problem(config, dev)
    r = Runner(wq, p, 0, dev, stream, layout=layout_of(config))
    for i in range(warmup):
        r.step(i)
    graphs = capture_graphs(r, steps)
    for g in graphs:
        g.replay()
    torch.cuda.synchronize(dev)
    ev0 = torch.cuda.Event(enable_timing=True)
    ev1 = torch.cuda.Event(enable_timing=True)
    ev0.record(stream)
    for g in graphs:
        g.replay()
    ev1.record(stream)
    torch.cuda.synchronize(dev)
    ms = ev0.elapsed_time(ev1) / steps
    roof = roofline(p, ms, peaks)
    out = {"workload": p.name + layout_suffix(r.layout), "M": p.M, "K": p.K, "N": p.N,
           "kernel":
           ["auto", "generic", "decode", "prefill"][r.chosen], "steps": steps, "ms_per_step": ms,
           "TFLOP/s": 2.0 * p.M * p.K * p.N / (ms * 1e-3) / 1e12,
           "weight_GBps": r.ab["weight"] / (ms * 1e-3) / 1e9,
           "roofline_bound": roof["bound"], "roofline_frac": roof["frac"], "l2": r.l2_note()}
    del graphs, r, p
    torch.cuda.synchronize(dev)
    torch.cuda.empty_cache()
    return out


def time_dynamic_quant(wq, dev, stream, bits, steps, warmup, peaks, M=8192, K=8192):
    """Device time of the per-token dynamic quantization of a bf16 (M, K) activation."""
    g = torch.Generator(device=dev).manual_seed(6)
    R = 3  # distinct inputs, 3 x 134 MB > 2x L2
    xs = [torch.randn((M, K), generator=g, device=dev).to(torch.bfloat16) for _ in range(R)]
    ys = [torch.empty((M, K if bits == 8 else K // 2), dtype=torch.int8 if bits == 8 else torch.uint8,
                      device=dev) for _ in range(R)]
    ss = [torch.empty(M, dtype=torch.float32, device=dev) for _ in range(R)]
    for i in range(warmup):
        wq.dynamic_quant(xs[i % R], None, bits, y=ys[i % R], scale=ss[i % R], stream=stream)
    gr = torch.cuda.CUDAGraph()
    with torch.cuda.graph(gr, stream=stream):
        for i in range(steps):
            wq.dynamic_quant(xs[i % R], None, bits, y=ys[i % R], scale=ss[i % R], stream=stream)
    gr.replay()
    torch.cuda.synchronize(dev)
    ev0 = torch.cuda.Event(enable_timing=True)
    ev1 = torch.cuda.Event(enable_timing=True)
    ev0.record(stream)
    gr.replay()
    ev1.record(stream)
    torch.cuda.synchronize(dev)
    ms = ev0.elapsed_time(ev1) / steps
    nbytes = M * K * 2 + M * K * bits // 8 + M * 4
    out = {"workload": f"dynamic_quant_bf16_int{bits}_M{M}_K{K}", "kernel": "dynamic_quant",
           "steps": steps, "ms_per_step": ms, "GB/s": nbytes / (ms * 1e-3) / 1e9,
           "roofline_bound": "hbm", "roofline_frac": nbytes / (ms * 1e-3) / 1e9 / peaks["hbm_gbs"],
           "l2": f"rotating {R} distinct inputs, {R * M * K * 2 / 1e6:.0f} MB > 2x L2"}
    del gr, xs, ys, ss
    torch.cuda.synchronize(dev)
    torch.cuda.empty_cache()
    return out


def _graph_time(stream, dev, fn, steps, warmup):
    """Per-call device time (ms) of fn(i) replayed from a CUDA graph of `steps` calls."""
    for i in range(warmup):
        fn(i)
    gr = torch.cuda.CUDAGraph()
    with torch.cuda.graph(gr, stream=stream):
        for i in range(steps):
            fn(i)
    gr.replay()
    torch.cuda.synchronize(dev)
    ev0 = torch.cuda.Event(enable_timing=True)
    ev1 = torch.cuda.Event(enable_timing=True)
    ev0.record(stream)
    gr.replay()
    ev1.record(stream)
    torch.cuda.synchronize(dev)
    del gr
    return ev0.elapsed_time(ev1) / steps


# fp32 FMA peak of the CUDA cores: 148 SMs x 128 lanes x 2 FLOP x 2.032 GHz (unit
# counts and maximum SM clock of the part)
FP32_FMA_TFLOPS = 148 * 128 * 2 * 2.032e9 / 1e12


def time_fp4(wq, dev, stream, steps, warmup, peaks):
    """FP4 E2M1 pack of a float32 (8192, 28672) weight, and the mx block-scaled
    matmul with in-place add on a gradient-accumulation shape: y (4096, 4096) +=
    x1^T-stored (8192 tokens, 4096) @ x2 (8192, 4096), FP4 operands, E8M0 scales."""
    out = []
    g = torch.Generator(device=dev).manual_seed(7)
    K, N = 8192, 28672
    R = 2  # 2 x 940 MB of float32 input > 2x L2
    ws = [torch.randn((K, N), generator=g, device=dev) * 3 for _ in range(R)]
    os_ = [torch.empty((K, N // 2), dtype=torch.uint8, device=dev) for _ in range(R)]
    ms = _graph_time(stream, dev, lambda i: wq.pack_fp4(ws[i % R], out=os_[i % R], stream=stream),
                     steps, warmup)
    nbytes = K * N * 4 + K * N // 2
    out.append({"workload": f"pack_fp4_f32_K{K}_N{N}", "kernel": "pack_fp4", "ms_per_step": ms,
                "GB/s": nbytes / (ms * 1e-3) / 1e9, "roofline_bound": "hbm",
                "roofline_frac": nbytes / (ms * 1e-3) / 1e9 / peaks["hbm_gbs"],
                "l2": f"rotating {R} inputs of {K * N * 4 / 1e6:.0f} MB"})
    del ws, os_
    M, KT, N2 = 4096, 8192, 4096
    J = KT // 32
    x1 = torch.randint(0, 256, (KT, M // 2), generator=g, device=dev, dtype=torch.uint8)
    s1 = torch.randint(120, 134, (J, M), generator=g, device=dev, dtype=torch.uint8)
    x2 = torch.randint(0, 256, (KT, N2 // 2), generator=g, device=dev, dtype=torch.uint8)
    s2 = torch.randint(120, 134, (J, N2), generator=g, device=dev, dtype=torch.uint8)
    y = torch.zeros((M, N2), dtype=torch.float32, device=dev)
    ms = _graph_time(stream, dev, lambda i: wq.mx_matmul_add(x1, s1, x2, s2, y, x1_transposed=True,
                                                             stream=stream), 10, 2)
    tf = 2.0 * M * N2 * KT / (ms * 1e-3) / 1e12
    out.append({"workload": f"mx_matmul_add_fp4_M{M}_K{KT}_N{N2}_x1T", "kernel": "mx_matmul_add (tensor cores)",
                "ms_per_step": ms, "TFLOP/s": tf, "roofline_bound": "tensor",
                "roofline_peak": peaks["bf16_tflops"], "roofline_frac": tf / peaks["bf16_tflops"]})
    ms = _graph_time(stream, dev, lambda i: wq.mx_matmul_add(x1, s1, x2, s2, y, x1_transposed=True,
                                                             kernel="exact", stream=stream), 2, 1)
    tf = 2.0 * M * N2 * KT / (ms * 1e-3) / 1e12
    out.append({"workload": f"mx_matmul_add_fp4_M{M}_K{KT}_N{N2}_x1T", "kernel": "mx_matmul_add (exact, CUDA cores)",
                "ms_per_step": ms, "TFLOP/s": tf, "roofline_bound": "alu",
                "roofline_peak": FP32_FMA_TFLOPS, "roofline_frac": tf / FP32_FMA_TFLOPS})
    del x1, s1, x2, s2, y
    torch.cuda.synchronize(dev)
    torch.cuda.empty_cache()
    return out


EXTRA = (("decode", 2000), ("decode@tiled", 2000), ("sweep:1", 1000), ("sweep:1@tiled", 1000),
         ("sweep:16", 1000), ("sweep:16@tiled", 1000), ("sweep:64", 500), ("sweep:64@tiled", 500),
         ("w8a16", 50), ("prefill", 20), ("sweep:4096@transposed", 10))


def traffic_record(kernel_name, workload):
    """DRAM bytes per launch of the dominant kernel from the committed ncu summary
    (profiles/traffic.md), or None when no capture matches this workload or the
    kernel's source has changed since the capture (sha256 of its .cu file)."""
    import hashlib
    import re
    path = os.path.join(ROOT, "profiles", "traffic.md")
    try:
        text = open(path).read()
    except OSError:
        return None
    for m in re.finditer(r"^traffic: (.*)$", text, flags=re.M):
        kv = dict(x.split("=", 1) for x in m.group(1).split())
        if kv.get("kernel") != kernel_name or kv.get("workload") != workload:
            continue
        src = os.path.join(ROOT, "weight_only_bit_pack_b300", "csrc", kv.get("source", ""))
        try:
            sha = hashlib.sha256(open(src, "rb").read()).hexdigest()[:16]
        except OSError:
            return None
        if sha != kv.get("source_sha"):
            return None
        return float(kv["dram_bytes_per_launch"])
    return None


def run_ours(args, world, rank, local):
    import weight_only_bit_pack_b300 as wq
    from weight_only_bit_pack_b300 import build as wqbuild
    wqbuild.build()
    dev = torch.device("cuda", local)
    kernel = {"auto": 0, "generic": 1, "decode": 2, "prefill": 3}[args.kernel]
    p = make_problem(args.config, dev)
    K = args.steps if args.steps is not None else default_steps(args.config)
    W = max(3, args.warmup)

    stream = torch.cuda.Stream(device=dev)
    torch.cuda.set_stream(stream)
    runner = Runner(wq, p, kernel, dev, stream, layout=layout_of(args.config))
    w_src, w0, ab, R, sets = runner.w_src, runner.w0, runner.ab, runner.R, runner.sets
    chosen = runner.chosen
    step = runner.step

    for i in range(W):
        step(i)
    torch.cuda.synchronize(dev)

    # capture the K timed steps (in chunks so a graph stays small), replay once untimed
    graphs = capture_graphs(runner, K)
    for g in graphs:
        g.replay()
    torch.cuda.synchronize(dev)

    ev0 = torch.cuda.Event(enable_timing=True)
    ev1 = torch.cuda.Event(enable_timing=True)
    barrier(world)
    torch.cuda.synchronize(dev)
    with ClockSampler(dev) as clk:
        ev0.record(stream)
        for g in graphs:
            g.replay()
        ev1.record(stream)
        torch.cuda.synchronize(dev)
    barrier(world)
    t_ms = ev0.elapsed_time(ev1)
    t_ms = max_over_ranks(world, t_ms)
    ms_step = t_ms / K
    flops = 2.0 * p.M * p.K * p.N
    tflops = flops / (ms_step * 1e-3) / 1e12 * world
    w_gbs = ab["weight"] / (ms_step * 1e-3) / 1e9
    del graphs

    # end-to-end: pinned host inputs -> device, call, outputs -> pinned host
    e2e = None
    if not args.no_e2e:
        hx = [p.x1.cpu().pin_memory() for _ in range(2)]
        hr = [p.residual.cpu().pin_memory() for _ in range(2)]
        hy = torch.empty(p.residual.shape, dtype=p.residual.dtype).pin_memory()
        hn = torch.empty(p.residual.shape, dtype=p.residual.dtype).pin_memory()
        Ke = min(K, 2000 if ms_step < 0.1 else 50)
        # at least two device sets of the per-step tensors (x1, residual, y,
        # normOut; the weight operands are shared), so that one step's copies
        # travel while the next step computes
        esets = list(sets)
        if len(esets) < 2:
            e = dict(sets[0])
            for key in ("x1", "residual", "y", "normOut"):
                e[key] = torch.empty_like(sets[0][key])
            e["x1"].copy_(sets[0]["x1"])
            e["residual"].copy_(sets[0]["residual"])
            esets.append(e)
        Re = len(esets)

        def estep(i):
            s = esets[i % Re]
            wq.matmul_add_rmsnorm(s["x1"], s["w"], s["scale"], s["offset"], s["bias"],
                                  s["residual"], s["gamma"], p.eps, p.group, y=s["y"],
                                  normOut=s["normOut"], workspace=runner.ws, kernel=runner.kernel,
                                  stream=stream)

        def e2e_step(i):
            s = esets[i % Re]
            s["x1"].copy_(hx[i % 2], non_blocking=True)
            s["residual"].copy_(hr[i % 2], non_blocking=True)
            estep(i)
            hy.copy_(s["y"], non_blocking=True)
            hn.copy_(s["normOut"], non_blocking=True)

        # The per-step sequence (two copies in, the call, two copies out) is
        # captured into CUDA graphs, as a serving loop would issue it: copies in
        # on one stream, the call on the launch stream, copies out on a third,
        # so that step i+1's inputs travel while step i computes. Step i waits
        # for its own inputs and for the copy-out of the step that last used
        # its device set (i - Re); its copy-in waits for that step's call. If
        # the capture is refused the same sequence runs eagerly on one stream.
        s_in = torch.cuda.Stream(device=dev)
        s_out = torch.cuda.Stream(device=dev)

        def capture_pipelined(lo, hi):
            ev_k, ev_out = {}, {}
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                s_in.wait_stream(stream)
                s_out.wait_stream(stream)
                for i in range(lo, hi):
                    s = esets[i % Re]
                    with torch.cuda.stream(s_in):
                        if i - Re >= lo:
                            s_in.wait_event(ev_k[i - Re])
                        s["x1"].copy_(hx[i % 2], non_blocking=True)
                        s["residual"].copy_(hr[i % 2], non_blocking=True)
                        ev_in = torch.cuda.Event()
                        ev_in.record(s_in)
                    stream.wait_event(ev_in)
                    if i - Re >= lo:
                        stream.wait_event(ev_out[i - Re])
                    estep(i)
                    ev_k[i] = torch.cuda.Event()
                    ev_k[i].record(stream)
                    with torch.cuda.stream(s_out):
                        s_out.wait_event(ev_k[i])
                        hy.copy_(s["y"], non_blocking=True)
                        hn.copy_(s["normOut"], non_blocking=True)
                        ev_out[i] = torch.cuda.Event()
                        ev_out[i].record(s_out)
                stream.wait_stream(s_in)
                stream.wait_stream(s_out)
            return g

        def capture_serial(lo, hi):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                for i in range(lo, hi):
                    e2e_step(i)
            return g

        launch = "cuda_graph_pipelined"
        try:
            egraphs = []
            done = 0
            while done < Ke:
                n = min(200, Ke - done)
                try:
                    g = capture_pipelined(done, done + n) if launch == "cuda_graph_pipelined" \
                        else capture_serial(done, done + n)
                except Exception as ex:
                    if launch != "cuda_graph_pipelined":
                        raise
                    print(f"e2e pipelined capture failed ({ex}); one stream", file=sys.stderr)
                    torch.cuda.synchronize(dev)
                    launch, egraphs, done = "cuda_graph", [], 0
                    continue
                egraphs.append(g)
                done += n
            for g in egraphs:
                g.replay()
            torch.cuda.synchronize(dev)
            barrier(world)
            torch.cuda.synchronize(dev)
            ev0.record(stream)
            for g in egraphs:
                g.replay()
            ev1.record(stream)
            torch.cuda.synchronize(dev)
        except Exception as ex:  # capture refused: time the eager sequence instead
            print(f"e2e graph capture failed ({ex}); timing eager calls", file=sys.stderr)
            launch = "eager"
            torch.cuda.synchronize(dev)
            for i in range(W + Ke):
                if i == W:
                    barrier(world)
                    torch.cuda.synchronize(dev)
                    ev0.record(stream)
                e2e_step(i)
            ev1.record(stream)
            torch.cuda.synchronize(dev)
        te = max_over_ranks(world, ev0.elapsed_time(ev1)) / Ke
        h2d = hx[0].numel() * hx[0].element_size() + hr[0].numel() * hr[0].element_size()
        d2h = 2 * hy.numel() * hy.element_size()
        e2e = {"value": flops / (te * 1e-3) / 1e12 * world, "unit": "TFLOP/s",
               "ms_per_step": te, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
               "steps": Ke, "launch": launch}

    # INT32 -> INT4 pack of this workload's weight (once per weight in deployment)
    pack = None
    if not args.no_pack and p.wbits == 4 and runner.layout != "transposed":
        if runner.tiled:
            out = wq.TiledInt4(torch.empty_like(w0.data), w0.K, w0.N)
            pack_fn = lambda: wq.pack_int4_tiled(w_src, out=out, stream=stream)  # noqa: E731
        else:
            out = torch.empty_like(w0)
            pack_fn = lambda: wq.pack_int4(w_src, out=out, stream=stream)  # noqa: E731
        for _ in range(3):
            pack_fn()
        torch.cuda.synchronize(dev)
        reps = 20
        ev0.record(stream)
        for _ in range(reps):
            pack_fn()
        ev1.record(stream)
        torch.cuda.synchronize(dev)
        tp = ev0.elapsed_time(ev1) / reps
        ob = out.data if runner.tiled else out
        pbytes = w_src.numel() * 4 + ob.numel()
        peaks, _src = load_peaks()
        pack = {"layout": "tiled" if runner.tiled else "dense", "ms": tp,
                "GB/s": pbytes / (tp * 1e-3) / 1e9, "bytes": pbytes,
                "frac_of_measured_hbm": pbytes / (tp * 1e-3) / 1e9 / peaks["hbm_gbs"],
                "bit_exact": bool(torch.equal(ob, w0.data if runner.tiled else w0))}

    peaks, peak_src = load_peaks()
    roof = roofline(p, ms_step, peaks)
    # the dominant kernel's DRAM bytes per launch, from the committed ncu capture
    kname = {3: "prefill_kernel", 2: "decode_kernel"}.get(chosen, "generic_gemm_kernel")
    wname = p.name + layout_suffix(runner.layout)
    roof["traffic"] = traffic_record(kname, wname)
    roof["traffic_source"] = ("profiles/traffic.md (ncu dram__bytes_read.sum + "
                              "dram__bytes_write.sum of one launch)"
                              if roof["traffic"] is not None else
                              "none: no capture of this kernel source on this workload")
    roof["peak_source"] = f"{peak_src} (MEASURED_PEAKS.json)" if peak_src == "measured" else \
        "fallback 6.4 TB/s / 1.8 PFLOP/s"
    roof["kernel"] = (f"{kname}: achieved over the whole call (its pre-pass launches included), "
                      f"kernel choice {['auto', 'generic', 'decode', 'prefill'][chosen]}")
    roof["alg_bytes_per_launch"] = ab["total"]
    roof["flops_per_launch"] = flops

    line = {
        "metric": METRIC, "value": tflops, "unit": "TFLOP/s", "n_gpus": world, "steps": K,
        "warmup": W, "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": {torch.bfloat16: "bf16", torch.float16: "f16"}[p.dtype],
        "data": "synthetic (seeded; weights random INT4/INT8, activations N(0,1))",
        "config": {"workload": wname, "M": p.M, "K": p.K, "N": p.N, "wbits": p.wbits,
                   "group": p.group, "offset": p.offset is not None, "bias": p.bias is not None,
                   "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
                   "l2": runner.l2_note(),
                   "timing": "CUDA graph replay of the K steps, CUDA events on the launch stream",
                   "kernel": ["auto", "generic", "decode", "prefill"][chosen]},
        "weight_GBps": w_gbs,
        "roofline": roof,
        "e2e": e2e,
        "gpu_launches": K * runner.kernels_per_call(),
        "pack": pack,
    }
    if rank == 0:
        line["clocks"] = clk.summary()
        if not args.no_cpu_baseline and world == 1:
            line["cpu_baseline"] = cpu_baseline(p)
        elif not args.no_cpu_baseline:
            line["cpu_baseline"] = None
    if not args.no_extra and world == 1:
        del runner, sets, w0, p
        torch.cuda.synchronize(dev)
        torch.cuda.empty_cache()
        extras = []
        for cfg, n in EXTRA:
            if cfg == args.config:
                continue
            extras.append(time_extra(wq, cfg, dev, stream, n, W, peaks))
        for bits in (8, 4):
            extras.append(time_dynamic_quant(wq, dev, stream, bits, 50, W, peaks))
        extras += time_fp4(wq, dev, stream, 20, W, peaks)
        line["workloads"] = extras
    if rank == 0:
        print(json.dumps(line), flush=True)


# ------------------------------------------------------------------ reference arm (CPU oracle)

def run_reference(args, world, rank):
    if rank != 0:
        return
    p = make_problem(args.config, "cpu")
    K = args.steps if args.steps is not None else 10
    W = max(3, args.warmup)
    rows = oracle_sample(p, 1e9)
    cache = {}
    for _ in range(W):
        run_oracle_rows(p, rows, cache)
    t0 = time.perf_counter()
    for _ in range(K):
        run_oracle_rows(p, rows, cache)
    el = time.perf_counter() - t0
    flops = 2.0 * len(rows) * p.K * p.N
    val = flops * K / el / 1e12
    sample = f"{len(rows)} of {p.M} rows per step (fp64 C oracle, OpenMP)"
    line = {"impl": "reference", "metric": METRIC, "value": val, "unit": "TFLOP/s",
            "n_gpus": world, "steps": K, "warmup": W, "ms_per_step": el / K * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "f64", "data": "synthetic (seeded)",
            "config": {"workload": p.name, "M": p.M, "K": p.K, "N": p.N, "rows_per_step": len(rows)},
            "cpu_baseline": {"value": val, "unit": "TFLOP/s", "cores": cores_used(),
                             "kind": "oracle", "sample": sample},
            "e2e": {"value": val, "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def main():
    args = parse_args()
    world, rank, local = dist_setup(args)
    if args.impl == "reference":
        run_reference(args, world, rank)
    else:
        run_ours(args, world, rank, local)
    if world > 1 and args.impl == "ours":
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
