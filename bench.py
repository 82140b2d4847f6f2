#!/usr/bin/env python
"""Benchmark of the MoE layer (router -> schedule -> pull dispatch -> grouped SwiGLU FFN ->
weighted combine, and its backward) on GB300.

One step = one forward + one backward of the DeepSeek-V3-shaped layer (T=4096 tokens,
hidden 7168, 256 experts of intermediate 2048, top-8 sigmoid router with renormalised
gates) on seeded synthetic bf16 data, inputs resident in HBM.  Prints one JSON line.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl mok|reference]

--impl reference times the float64 CPU oracle (the deliberately slow, obviously correct
restatement of the layer) on a bounded sample of the same workload on the host cores.
Under torchrun (N > 1) every rank runs an independent replica on its own GPU and batch
(weak scaling, no collective on the data path); rank 0 prints the line.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "MoE-layer tokens/s, fwd+bwd, 1xGB300 (grouped-GEMM % of tensor peak reported alongside)"
UNIT = "tokens/s"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
CPU_SAMPLE = {"T": 1536, "E": 16}       # cpu_baseline: 1536 tokens of the DSV3 shape over 16 experts (~10 s)
REF_SAMPLE = {"T": 256, "E": 16}        # --impl reference: per step


def _workloads():
    from mixture_experts_layer_table_gb300 import workloads as W
    return {"dsv3": W.DSV3, "dsv3_e16_t256": W.DSV3.scaled(name="dsv3_e16_t256", T=256, E=16),
            "dsv3_e16_t1024": W.DSV3.scaled(name="dsv3_e16_t1024", T=1024, E=16),
            "dsv3_skew": W.DSV3_SKEW}


WORKLOADS = _workloads()
# forward expert GEMMs: library choice, CTA pairs (256-row tiles) or single CTAs (128-row tiles)
GEMM_FLAGS = {"auto": 0, "pair": 2, "single": 4}
# Kernels per traced library call where one call launches several: the schedule table is a
# histogram, a scan and a placement kernel.
KERNELS_PER_CALL = {"schedule": 3}


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            p = json.load(f)
        return p, "measured"
    return FALLBACK_PEAKS, "fallback"


def kernel_bytes(s, wgrad_bytes=4):
    """Algorithmic HBM bytes of one launch of each kernel: reads + writes of distinct data in the
    layouts the kernels use (bf16 inputs and weights; h|u, expert outputs and dX rows in fp32;
    a, dh|du and g*a as bf16 hi + lo pairs; weight gradients in fp32 by default)."""
    T, H, I, E, k = s.T, s.H, s.I, s.E, s.k
    R = T * k
    return {
        "router_gemm": T * H * 2 + E * H * 2 + T * E * 4,
        "topk": T * E * 4 * 2 + T * k * 8,
        "schedule": R * 4 * 5 + E * 8,
        "gather_x": T * H * 2 + R * H * 2 + R * 4,
        "gemm1_swiglu": E * 2 * I * H * 2 + R * H * 2 + R * 2 * I * 4 + R * I * 4,
        "gemm2": E * H * I * 2 + R * I * 4 + R * H * 4,
        "combine": R * H * 4 + T * H * 2 + R * 8,
        "gather_dy": T * H * 2 + R * H * 2 + R * 4,
        "dgrad_swiglu": E * H * I * 2 + R * H * 2 + R * 2 * I * 4 + R * 2 * I * 4 + R * I * 4 + R * (I // 256) * 4,
        "dgrad_x": E * 2 * I * H * 2 + R * 2 * I * 4 + R * H * 4,
        "wgrad_w2": R * H * 2 + R * I * 4 + E * H * I * wgrad_bytes,
        "wgrad_w13": R * 2 * I * 4 + R * H * 2 + E * 2 * I * H * wgrad_bytes,
        "router_dlogits": R * (I // 256) * 4 + R * 12 + T * E * 8,
        "router_wgrad": T * H * 2 + E * H * 4 + T * E * 4,
        "combine_dx": R * H * 4 + E * H * 2 + T * H * 2 + T * E * 4,
    }


def kernel_flops(s):
    """Dense tensor-core FLOPs of one launch of each GEMM kernel."""
    T, H, I, E, k = s.T, s.H, s.I, s.E, s.k
    R = T * k
    return {"router_gemm": 2 * T * E * H, "gemm1_swiglu": 2 * R * 2 * I * H, "gemm2": 2 * R * H * I,
            "dgrad_swiglu": 2 * R * H * I, "dgrad_x": 2 * R * 2 * I * H, "wgrad_w2": 2 * R * H * I,
            "wgrad_w13": 2 * R * 2 * I * H}


def load_traffic():
    """Per-launch DRAM bytes (dram__bytes_read.sum + dram__bytes_write.sum) from the committed
    ncu summary, keyed by kernel; only entries marked current for the present kernels."""
    path = os.path.join(ROOT, "profiles", "dram_traffic_dsv3.txt")
    out = {}
    if os.path.exists(path):
        with open(path) as f:
            for line in f:
                parts = line.split()
                if len(parts) >= 3 and not line.startswith("#") and parts[2] == "current":
                    out[parts[0]] = float(parts[1])
    return out


class ClockSampler:
    """nvidia-smi clocks and throttle reasons, sampled every 100 ms while running."""

    FIELDS = "index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active," \
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown," \
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap"

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.15)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as f:
            for line in f:
                p = [x.strip() for x in line.split(",")]
                if len(p) < 9:
                    continue
                try:
                    sm.append(float(p[1]))
                    mx.append(float(p[2]))
                except ValueError:
                    continue
                for n, v in zip(names, p[5:9]):
                    if v.lower() == "active":
                        reasons.add(n)
        os.unlink(self.path)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


def cpu_sample_run(T, E, repeats=1):
    """Times the float64 oracle (forward + backward) on T tokens of the DSV3 shape over E experts."""
    import numpy as np
    from mixture_experts_layer_table_gb300 import workloads as W
    from oracle import moe_oracle as O
    shp = W.DSV3.scaled(T=T, E=E)
    inp = W.make_inputs(shp, seed=0, device="cpu")
    f = {k: (v.double().numpy() if v is not None else None) for k, v in inp.items()}
    times = []
    for _ in range(repeats):
        t0 = time.perf_counter()
        fwd = O.forward(f["x"], f["w_router"], f["w13"], f["w2"], kind=shp.router, k=shp.k, renorm=shp.renorm)
        O.backward(fwd, f["dy"], f["x"], f["w_router"], f["w13"], f["w2"], kind=shp.router, k=shp.k,
                   renorm=shp.renorm)
        times.append(time.perf_counter() - t0)
    return times


def cpu_sample_subprocess(T, E, repeats=1):
    cores = os.cpu_count() or 1
    env = dict(os.environ, OPENBLAS_NUM_THREADS=str(cores), OMP_NUM_THREADS=str(cores), MKL_NUM_THREADS=str(cores),
               CUDA_VISIBLE_DEVICES="")
    r = subprocess.run([sys.executable, os.path.abspath(__file__), "--cpu-sample", str(T), str(E), str(repeats)],
                       env=env, capture_output=True, text=True, timeout=1800)
    if r.returncode != 0:
        raise RuntimeError(r.stderr[-2000:])
    times = json.loads(r.stdout.strip().splitlines()[-1])
    return times, cores


class LazyExperts:
    """[E][rows][cols] float64 view of a host bf16 tensor that widens one expert at a time, so
    that the oracle can stream the experts of a full-size layer (45 GB in float64) through host
    memory.  Indexing only: w[e], w[e, a:b]."""

    def __init__(self, t):
        self.t = t
        self.shape = tuple(t.shape)

    def __getitem__(self, idx):
        if isinstance(idx, tuple):
            return self.t[idx[0]].double().numpy()[idx[1:]]
        return self.t[idx].double().numpy()


def mem_available_gb():
    try:
        with open("/proc/meminfo") as f:
            for line in f:
                if line.startswith("MemAvailable:"):
                    return int(line.split()[1]) / 2**20
    except OSError:
        pass
    return None


def cpu_planned_timings(inp, shp):
    """The float64 oracle, as it stands, at the full sizes of the workloads, on the host cores
    after the GPU runs: the DSV3 layer forward (near-uniform routing) and the skewed DSV3 layer
    forward + backward on all cores (numpy / OpenBLAS default threads, one per core), each
    streaming one expert's weights in float64 at a time (LazyExperts), and the tiny layer forward
    + backward on one thread.  The inputs are this run's (copied from the GPU).  The skewed
    forward + backward holds the layer's float64 weight gradients (45 GB): it is skipped, with
    the reason, when the host has less than 150 GB available."""
    import numpy as np
    from mixture_experts_layer_table_gb300 import workloads as W
    from oracle import moe_oracle as O

    cores = os.cpu_count() or 1
    out = {"cores": cores, "threads": "OpenBLAS default (one per core); tiny: 1", "cpu_model": cpu_model()}
    host = {k: v.cpu() for k, v in inp.items() if v is not None}
    x, wr, dy = (host[n].double().numpy() for n in ("x", "w_router", "dy"))
    w13, w2 = LazyExperts(host["w13"]), LazyExperts(host["w2"])
    T = shp.T
    t0 = time.perf_counter()
    O.forward(x, wr, w13, w2, kind=shp.router, k=shp.k, renorm=shp.renorm)
    sec = time.perf_counter() - t0
    out["dsv3_fwd"] = {"seconds": round(sec, 2), "tokens_per_s": round(T / sec, 1),
                       "workload": shp.name + ", forward, full size"}
    avail = mem_available_gb()
    skew = W.DSV3_SKEW
    if avail is not None and avail < 150:
        out["dsv3_skew_fwd_bwd"] = {"skipped": f"needs ~120 GB of host memory, {avail:.0f} GB available"}
    else:
        bias = W.skew_bias(skew.E).double().numpy()
        t0 = time.perf_counter()
        f = O.forward(x, wr, w13, w2, kind=skew.router, k=skew.k, renorm=skew.renorm, router_bias=bias)
        O.backward(f, dy, x, wr, w13, w2, kind=skew.router, k=skew.k, renorm=skew.renorm)
        sec = time.perf_counter() - t0
        del f
        out["dsv3_skew_fwd_bwd"] = {"seconds": round(sec, 2), "tokens_per_s": round(T / sec, 1),
                                    "workload": skew.name + ", forward + backward, full size"}
    del x, wr, dy, w13, w2, host
    env = dict(os.environ, OPENBLAS_NUM_THREADS="1", OMP_NUM_THREADS="1", MKL_NUM_THREADS="1",
               CUDA_VISIBLE_DEVICES="")
    r = subprocess.run([sys.executable, os.path.abspath(__file__), "--cpu-tiny"], env=env, capture_output=True,
                       text=True, timeout=600)
    if r.returncode == 0:
        sec = json.loads(r.stdout.strip().splitlines()[-1])
        out["tiny_fwd_bwd_1thread"] = {"seconds": round(sec, 4), "tokens_per_s": round(W.TINY.T / sec, 1),
                                       "workload": W.TINY.name + ", forward + backward, one thread"}
    else:
        out["tiny_fwd_bwd_1thread"] = {"skipped": r.stderr[-300:]}
    return out


def cpu_tiny_run():
    """Seconds of the float64 oracle's forward + backward of the tiny layer (one thread when the
    caller sets the BLAS thread count to 1)."""
    from mixture_experts_layer_table_gb300 import workloads as W
    from oracle import moe_oracle as O
    shp = W.TINY
    inp = W.make_inputs(shp, seed=0, device="cpu")
    f = {k: (v.double().numpy() if v is not None else None) for k, v in inp.items()}
    best = None
    for _ in range(3):
        t0 = time.perf_counter()
        fwd = O.forward(f["x"], f["w_router"], f["w13"], f["w2"], kind=shp.router, k=shp.k, renorm=shp.renorm)
        O.backward(fwd, f["dy"], f["x"], f["w_router"], f["w13"], f["w2"], kind=shp.router, k=shp.k,
                   renorm=shp.renorm)
        sec = time.perf_counter() - t0
        best = sec if best is None else min(best, sec)
    return best


def fwd_gemm_hbm(trace, kb, peaks):
    """Forward expert GEMMs at the DSV3 layer against the measured HBM copy bandwidth: algorithmic
    bytes (weights, rows in and out) over their traced time."""
    names = [n for n in ("gemm1_swiglu", "gemm2") if n in trace and n in kb]
    if not names:
        return None
    ms = sum(trace[n]["total_ms"] / trace[n]["launches"] for n in names)
    gbps = sum(kb[n] for n in names) / (ms * 1e-3) / 1e9
    return {"kernels": names, "ms": round(ms, 4), "GBps": round(gbps, 1), "frac": round(gbps / peaks["hbm_gbs"], 4),
            "peak": peaks["hbm_gbs"]}


def ring_sweep(shp, x, w_router, w13, w2, y_plain, steps, warmup):
    """The ring forward at `shp` (a fixed 512 MiB token ring) for each minibatch of the sweep, with
    GEMM2 and the merge as separate launches and in the persistent launch (`persistent`): ms per
    forward over K forwards after W warm-ups, and whether y is bitwise the plain forward's."""
    from mixture_experts_layer_table_gb300 import _native as N
    from mixture_experts_layer_table_gb300 import workloads as W

    sweep = {}
    for m in W.RING_MINIBATCHES:
        sweep[str(m)] = ring_point(shp, x, w_router, w13, w2, y_plain, steps, warmup, m, 0)
        sweep[str(m)]["persistent"] = ring_point(shp, x, w_router, w13, w2, y_plain, steps, warmup, m,
                                                 N.FLAG_RING_PERSISTENT)
    return sweep


def ring_point(shp, x, w_router, w13, w2, y_plain, steps, warmup, m, flags):
    """One point of the ring sweep: minibatch m with the given descriptor flags."""
    import torch

    import mixture_experts_layer_table_gb300 as mok
    from mixture_experts_layer_table_gb300 import _native as N
    from mixture_experts_layer_table_gb300 import workloads as W

    stream = torch.cuda.current_stream()
    y = torch.empty_like(y_plain)
    layer = mok.MoELayer(mok.desc_from_shape(shp, minibatch=m, ring_bytes=W.RING_BYTES, flags=flags), device=x.device)
    for _ in range(warmup):
        layer.forward(x, w_router, w13, w2, y=y)
    torch.cuda.synchronize()
    if layer.status() != (0, 0):
        raise RuntimeError("device status set during the ring warm-up")
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    N.trace_start(16 * steps + 16)
    e0.record(stream)
    for _ in range(steps):
        layer.forward(x, w_router, w13, w2, y=y)
    e1.record(stream)
    torch.cuda.synchronize()
    trace = N.trace_stop()
    if layer.status() != (0, 0):
        raise RuntimeError("device status set in the ring forward")
    ms = e0.elapsed_time(e1) / steps
    return {"fwd_ms": round(ms, 4), "tokens_per_s": round(shp.T / (ms * 1e-3), 1),
            "ring_slots": min(W.RING_BYTES // (m * shp.H * 2), -(-shp.R // m)),
            "bitwise_equal_to_plain": bool(torch.equal(y, y_plain)),
            "kernels": {n: round(t["total_ms"] / t["launches"], 4) for n, t in trace.items()}}


def ring_fwd_bwd(shp, x, w_router, w13, w2, steps, warmup, minibatch=2368):
    """Forward + backward at `shp` with and without the 512 MiB ring (minibatch `minibatch`): ms per
    step over K steps after W warm-ups, the backward's replay of the dispatched rows (the ring-based
    backward gathers only the minibatches the ring overwrote), and whether every gradient is
    bitwise the plain layer's."""
    import torch

    import mixture_experts_layer_table_gb300 as mok
    from mixture_experts_layer_table_gb300 import _native as N
    from mixture_experts_layer_table_gb300 import workloads as W

    g = torch.Generator(device=x.device).manual_seed(4)
    dy = torch.empty((shp.T, shp.H), dtype=torch.float32, device=x.device).normal_(0.0, 1.0, generator=g)
    dy = dy.to(torch.bfloat16)
    stream = torch.cuda.current_stream()
    out = {"minibatch": minibatch, "ring_bytes": W.RING_BYTES}
    grads = {}
    for name, kw in (("plain", {}), ("ring", {"minibatch": minibatch, "ring_bytes": W.RING_BYTES})):
        layer = mok.MoELayer(mok.desc_from_shape(shp, **kw), device=x.device)
        for _ in range(warmup):
            layer.forward(x, w_router, w13, w2)
            gr = layer.backward(dy, x, w_router, w13, w2)
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        N.trace_start(40 * steps + 16)
        e0.record(stream)
        for _ in range(steps):
            layer.forward(x, w_router, w13, w2)
            layer.backward(dy, x, w_router, w13, w2, out=gr)
        e1.record(stream)
        torch.cuda.synchronize()
        trace = N.trace_stop()
        if layer.status() != (0, 0):
            raise RuntimeError(f"device status set in the {name} forward + backward")
        ms = e0.elapsed_time(e1) / steps
        out[name] = {"fwd_bwd_ms": round(ms, 4), "tokens_per_s": round(shp.T / (ms * 1e-3), 1)}
        if "gather_x_replay" in trace:
            t = trace["gather_x_replay"]
            out[name]["replay_ms"] = round(t["total_ms"] / t["launches"], 4)
        grads[name] = gr
        del layer
        torch.cuda.empty_cache()
    out["bitwise_equal_gradients"] = all(torch.equal(grads["plain"][n], grads["ring"][n]) for n in grads["plain"])
    R = shp.R
    n_mb = -(-R // minibatch)
    slots = min(W.RING_BYTES // (minibatch * shp.H * 2), n_mb)
    out["rows_replayed"] = (n_mb - slots) * minibatch
    out["rows_resident"] = R - out["rows_replayed"]
    del grads, dy
    torch.cuda.empty_cache()
    return out


def tensor_sha256(t):
    """SHA-256 of a tensor's bit pattern (row-major bytes), read back to the host."""
    import hashlib
    import torch
    b = t.detach().contiguous().cpu().reshape(-1).view(torch.uint8)
    return hashlib.sha256(b.numpy().tobytes()).hexdigest()


def cpu_model():
    """The host CPU's model name (/proc/cpuinfo, else lscpu, else the machine type)."""
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                if line.lower().startswith("model name"):
                    return line.split(":", 1)[1].strip()
    except OSError:
        pass
    try:
        r = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10)
        for line in r.stdout.splitlines():
            if line.lower().startswith("model name"):
                return line.split(":", 1)[1].strip()
    except (OSError, subprocess.SubprocessError):
        pass
    import platform
    return platform.machine()


def sample_desc(T, E):
    return (f"float64 oracle forward+backward on {T} tokens of the same layer shape (hidden 7168, "
            f"intermediate 2048, top-8 sigmoid router, renormalised) restricted to {E} experts, "
            f"seeded CPU draws; tokens/s = {T} / seconds")


# ---- replicas (bench.py --gpus N under torchrun): one independent layer per GPU, no collective
# on the data path; the ranks only meet at barriers around the timed region and to take the
# slowest rank's time, and the whole-job rate counts every rank's tokens.

def replica_barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def replica_max(value, world, device):
    """The largest value over the ranks (every rank gets it)."""
    if world <= 1:
        return value
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_rate(tokens_per_rank, world, ms_per_step):
    """tokens/s of the whole job: every rank's tokens over the slowest rank's step time."""
    return tokens_per_rank * world / (ms_per_step * 1e-3)


def run_reference(args, rank, world):
    if rank != 0:
        return
    T, E = REF_SAMPLE["T"], REF_SAMPLE["E"]
    times, cores = cpu_sample_subprocess(T, E, repeats=args.warmup + args.steps)
    timed = times[args.warmup:]
    sec = sum(timed)
    value = T * len(timed) / sec
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * sec / len(timed),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic (seeded Gaussian activations and weights)",
            "config": {"workload": "dsv3_T4096_H7168_E256_I2048_top8_sigmoid (sampled: %d tokens, %d experts)" % (T, E),
                       "passes": "fwd+bwd"},
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle",
                             "sample": sample_desc(T, E), "cpu_model": cpu_model()},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def run_mok(args, rank, world, local_rank):
    import torch
    import torch.distributed as dist

    import mixture_experts_layer_table_gb300 as mok
    from mixture_experts_layer_table_gb300 import _native as N
    from mixture_experts_layer_table_gb300 import workloads as W

    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    mok.load()
    shp = WORKLOADS[args.workload]
    T, H, I, E, k = shp.T, shp.H, shp.I, shp.E, shp.k
    inp = W.make_inputs(shp, seed=1000 * rank, device=str(dev))
    layer = mok.MoELayer(mok.desc_from_shape(shp, flags=GEMM_FLAGS[args.gemm]), device=dev)
    grads = {"dx": torch.empty((T, H), dtype=torch.bfloat16, device=dev),
             "dw_router": torch.empty((E, H), dtype=torch.float32, device=dev),
             "dw13": torch.empty((E, 2 * I, H), dtype=torch.float32, device=dev),
             "dw2": torch.empty((E, H, I), dtype=torch.float32, device=dev),
             "dgates": torch.empty((T, k), dtype=torch.float32, device=dev)}
    y = torch.empty((T, H), dtype=torch.bfloat16, device=dev)
    x, wr, w13, w2, dy = inp["x"], inp["w_router"], inp["w13"], inp["w2"], inp["dy"]
    bias0 = inp["router_bias"]  # the skewed workload's selection bias, else None

    def fwd():
        layer.forward(x, wr, w13, w2, router_bias=bias0, y=y)

    def step():
        layer.forward(x, wr, w13, w2, router_bias=bias0, y=y)
        layer.backward(dy, x, wr, w13, w2, out=grads)

    def barrier():
        replica_barrier(world)

    def max_over_ranks(v):
        return replica_max(v, world, dev)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    code, site = layer.status()
    if code != 0:
        raise RuntimeError(f"device status {code} at site {site} during warm-up")
    counts = layer.view("counts").cpu()

    # ---- timed region: K steps of forward + backward, per-kernel events on the launching stream
    sampler = ClockSampler(torch.cuda.current_device())
    stream = torch.cuda.current_stream()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier()
    torch.cuda.synchronize()
    sampler.start()
    N.trace_start(40 * args.steps + 16)
    ev0.record(stream)
    for _ in range(args.steps):
        step()
    ev1.record(stream)
    torch.cuda.synchronize()
    barrier()
    trace = N.trace_stop()
    clocks = sampler.stop()
    ms = max_over_ranks(ev0.elapsed_time(ev1) / args.steps)
    code, site = layer.status()
    if code != 0:
        raise RuntimeError(f"device status {code} at site {site}")

    # ---- forward only
    for _ in range(2):
        fwd()
    barrier()
    torch.cuda.synchronize()
    ev0.record(stream)
    for _ in range(args.steps):
        fwd()
    ev1.record(stream)
    torch.cuda.synchronize()
    fwd_ms = max_over_ranks(ev0.elapsed_time(ev1) / args.steps)

    # ---- the same step with bf16 weight gradients (MOK_FLAG_WGRAD_BF16): what the fp32 reading
    #      of dW13 / dW2 costs (the bf16 result is the fp32 one rounded to nearest even)
    wgrad_bf16_ms = None
    if not args.no_wgrad_bf16:
        layer16 = mok.MoELayer(mok.desc_from_shape(shp, flags=GEMM_FLAGS[args.gemm] | N.FLAG_WGRAD_BF16), device=dev)
        g16 = dict(grads)
        g16["dw13"] = torch.empty((E, 2 * I, H), dtype=torch.bfloat16, device=dev)
        g16["dw2"] = torch.empty((E, H, I), dtype=torch.bfloat16, device=dev)
        for _ in range(2):
            layer16.forward(x, wr, w13, w2, y=y)
            layer16.backward(dy, x, wr, w13, w2, out=g16)
        barrier()
        torch.cuda.synchronize()
        N.trace_start(40 * args.steps + 16)
        ev0.record(stream)
        for _ in range(args.steps):
            layer16.forward(x, wr, w13, w2, y=y)
            layer16.backward(dy, x, wr, w13, w2, out=g16)
        ev1.record(stream)
        torch.cuda.synchronize()
        trace16 = N.trace_stop()
        wgrad_bf16_ms = max_over_ranks(ev0.elapsed_time(ev1) / args.steps)
        if layer16.status() != (0, 0):
            raise RuntimeError("device status set in the bf16 weight-gradient step")
        wgrad_bf16 = {"fwd_bwd_ms": round(wgrad_bf16_ms, 4),
                      "tokens_per_s": round(whole_job_rate(T, world, wgrad_bf16_ms), 1),
                      "kernels": {n: round(trace16[n]["total_ms"] / trace16[n]["launches"], 4)
                                  for n in ("wgrad_w2", "wgrad_w13") if n in trace16}}
        del layer16, g16

    # ---- the skewed-routing layer: the same tokens and weights with the Zipf-Mandelbrot router
    #      bias (hottest expert ~10x the mean load), forward + backward
    skew = None
    if not args.no_skew:
        bias = W.skew_bias(E).to(dev)

        def skew_step():
            layer.forward(x, wr, w13, w2, router_bias=bias, y=y)
            layer.backward(dy, x, wr, w13, w2, out=grads)

        for _ in range(2):
            skew_step()
        barrier()
        torch.cuda.synchronize()
        N.trace_start(40 * args.steps + 16)
        ev0.record(stream)
        for _ in range(args.steps):
            skew_step()
        ev1.record(stream)
        torch.cuda.synchronize()
        skew_trace = N.trace_stop()
        skew_ms = max_over_ranks(ev0.elapsed_time(ev1) / args.steps)
        if layer.status() != (0, 0):
            raise RuntimeError("device status set in the skewed step")
        sc = layer.view("counts").cpu()
        skew = {"workload": W.DSV3_SKEW.name + " (same tokens and weights, Zipf-Mandelbrot router bias)",
                "fwd_bwd_ms": round(skew_ms, 4), "tokens_per_s": round(whole_job_rate(T, world, skew_ms), 1),
                "expert_rows_min_max": [int(sc.min()), int(sc.max())],
                "kernels": {n: round(t["total_ms"] / t["launches"], 4) for n, t in skew_trace.items()}}

    # ---- the tiny layer (T=256, H=256, 8 experts, I=512, top-2 softmax): launch-bound, so timed
    #      eager and as one CUDA graph of the whole forward + backward, replayed
    tiny = None
    if not args.no_tiny:
        tiny = tiny_layer_step(args.steps, args.warmup, dev, stream, max_over_ranks, barrier)

    # ---- end to end through the public API with host buffers (pinned), copies timed.  Every
    #      step copies its own x and dY in and its y and dX out; a copy stream moves step i+1's
    #      inputs and step i-1's outputs while step i computes (two device buffer sets).
    x_h = [x.cpu().pin_memory() for _ in range(2)]
    dy_h = [dy.cpu().pin_memory() for _ in range(2)]
    y_h = [torch.empty((T, H), dtype=torch.bfloat16).pin_memory() for _ in range(2)]
    dx_h = [torch.empty((T, H), dtype=torch.bfloat16).pin_memory() for _ in range(2)]
    x_d = [torch.empty_like(x) for _ in range(2)]
    dy_d = [torch.empty_like(dy) for _ in range(2)]
    y_d = [torch.empty_like(y) for _ in range(2)]
    dx_d = [torch.empty_like(grads["dx"]) for _ in range(2)]
    copy_stream = torch.cuda.Stream(device=dev)
    ready = [torch.cuda.Event() for _ in range(2)]   # inputs of buffer b are on the device
    done = [torch.cuda.Event() for _ in range(2)]    # step on buffer b has finished computing
    g_e2e = dict(grads)

    def copy_in(b):
        with torch.cuda.stream(copy_stream):
            x_d[b].copy_(x_h[b], non_blocking=True)
            dy_d[b].copy_(dy_h[b], non_blocking=True)
            ready[b].record(copy_stream)

    def copy_out(b):
        with torch.cuda.stream(copy_stream):
            copy_stream.wait_event(done[b])
            y_h[b].copy_(y_d[b], non_blocking=True)
            dx_h[b].copy_(dx_d[b], non_blocking=True)

    def e2e_run(n):
        copy_in(0)
        for i in range(n):
            b = i % 2
            stream.wait_event(ready[b])
            layer.forward(x_d[b], wr, w13, w2, router_bias=bias0, y=y_d[b])
            g_e2e["dx"] = dx_d[b]
            layer.backward(dy_d[b], x_d[b], wr, w13, w2, out=g_e2e)
            done[b].record(stream)
            if i + 1 < n:
                with torch.cuda.stream(copy_stream):
                    if i >= 1:
                        copy_stream.wait_event(done[1 - b])  # buffer 1-b was used by step i-1
                copy_in(1 - b)
            copy_out(b)
        stream.wait_stream(copy_stream)

    e2e_run(2)
    barrier()
    torch.cuda.synchronize()
    ev0.record(stream)
    e2e_run(args.steps)
    ev1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks(ev0.elapsed_time(ev1) / args.steps)

    # ---- MXFP8 forward (weights quantised once, outside the timed region)
    mx = None
    if not args.no_mxfp8:
        wq = mok.quantize_weights(layer.desc, w13, w2)
        mx_desc = mok.desc_from_shape(shp.scaled(mxfp8=True))
        mx_layer = mok.MoELayer(mx_desc, device=dev)
        for _ in range(2):
            mok.moe_forward_mxfp8(mx_desc, x, wr, None, None, wq, y, mx_layer.ctx, mx_layer.ws)
        barrier()
        torch.cuda.synchronize()
        N.trace_start(16 * args.steps + 16)
        ev0.record(stream)
        for _ in range(args.steps):
            mok.moe_forward_mxfp8(mx_desc, x, wr, None, None, wq, y, mx_layer.ctx, mx_layer.ws)
        ev1.record(stream)
        torch.cuda.synchronize()
        mx_trace = N.trace_stop()
        mx_ms = max_over_ranks(ev0.elapsed_time(ev1) / args.steps)
        if mx_layer.status() != (0, 0):
            raise RuntimeError("device status set in the MXFP8 forward")
        # MXFP8 forward + backward (backward-direction weights quantised once, outside the timing)
        wb = mok.quantize_weights_backward(layer.desc, w13, w2)

        def mx_step():
            mok.moe_forward_mxfp8(mx_desc, x, wr, None, None, wq, y, mx_layer.ctx, mx_layer.ws)
            mx_layer.backward_mxfp8(dy, x, wr, wb, out=grads)

        for _ in range(2):
            mx_step()
        barrier()
        torch.cuda.synchronize()
        N.trace_start(40 * args.steps + 16)
        ev0.record(stream)
        for _ in range(args.steps):
            mx_step()
        ev1.record(stream)
        torch.cuda.synchronize()
        mxb_trace = N.trace_stop()
        mxb_ms = max_over_ranks(ev0.elapsed_time(ev1) / args.steps)
        if mx_layer.status() != (0, 0):
            raise RuntimeError("device status set in the MXFP8 backward")
        # the same step with bf16 weight gradients (MOK_FLAG_WGRAD_BF16: the fp32 ones rounded once;
        # the MXFP8 tolerance is a relative Frobenius error, which that rounding barely moves)
        mx_desc16 = mok.desc_from_shape(shp.scaled(mxfp8=True), flags=N.FLAG_WGRAD_BF16)
        mx_layer16 = mok.MoELayer(mx_desc16, device=dev)
        g16 = dict(grads)
        g16["dw13"] = torch.empty((E, 2 * I, H), dtype=torch.bfloat16, device=dev)
        g16["dw2"] = torch.empty((E, H, I), dtype=torch.bfloat16, device=dev)

        def mx_step16():
            mok.moe_forward_mxfp8(mx_desc16, x, wr, None, None, wq, y, mx_layer16.ctx, mx_layer16.ws)
            mx_layer16.backward_mxfp8(dy, x, wr, wb, out=g16)

        for _ in range(2):
            mx_step16()
        barrier()
        torch.cuda.synchronize()
        ev0.record(stream)
        for _ in range(args.steps):
            mx_step16()
        ev1.record(stream)
        torch.cuda.synchronize()
        mxb16_ms = max_over_ranks(ev0.elapsed_time(ev1) / args.steps)
        if mx_layer16.status() != (0, 0):
            raise RuntimeError("device status set in the MXFP8 backward with bf16 weight gradients")
        del mx_layer16, g16
        mx = {"fwd_ms": round(mx_ms, 4), "tokens_per_s": round(whole_job_rate(T, world, mx_ms), 1),
              "kernels": {n: round(t["total_ms"] / t["launches"], 4) for n, t in mx_trace.items()},
              "fwd_bwd_ms": round(mxb_ms, 4), "fwd_bwd_tokens_per_s": round(whole_job_rate(T, world, mxb_ms), 1),
              "fwd_bwd_kernels": {n: round(t["total_ms"] / t["launches"], 4) for n, t in mxb_trace.items()},
              "fwd_bwd_ms_wgrad_bf16": round(mxb16_ms, 4),
              "fwd_bwd_tokens_per_s_wgrad_bf16": round(whole_job_rate(T, world, mxb16_ms), 1),
              "weights": "forward: E4M3 + E8M0 per 32 along K (11.3 GB + 0.35 GB of scales); backward: W2 "
                         "and W13 transposed, E4M3 + E8M0 along H and 2I (11.3 GB + 0.35 GB); GEMM1, GEMM2, dA' "
                         "and dX_g on the FP8 tensor path (block-scaled MMAs), the weight gradients on the "
                         "exact values of their row-quantised operands (bf16 tensor path); activations and "
                         "gradients quantised along each GEMM's reduction"}
        del mx_layer, wq, wb

    # ---- the same weights at T=16384 (512 rows per expert): the forward GEMMs become
    #      tensor-bound; their fraction of the measured bf16 peak is graded there
    tb = None
    if not args.no_tensor_bound:
        shp_tb = W.RING
        g = torch.Generator(device=dev).manual_seed(12345 + rank)
        x_tb = torch.randn((shp_tb.T, H), generator=g, device=dev, dtype=torch.float32).to(torch.bfloat16)
        tb_ms, tb_kernels, tb_grouped, tb_layer, y_tb = tensor_bound_forward(shp_tb, x_tb, wr, w13, w2, args.steps,
                                                                            args.warmup, GEMM_FLAGS[args.gemm])
        tb = {"workload": shp_tb.name + " (same weights, x ~ N(0, 1))", "fwd_ms": round(tb_ms, 4),
              "tokens_per_s": round(whole_job_rate(shp_tb.T, world, tb_ms), 1),
              "grouped_gemm": tb_grouped,
              "kernels": {n: v for n, v in tb_kernels.items()}}
        del tb_layer
        if not args.no_fp16_w2:
            # the same forward on an fp16 copy of W2 (converted once, outside the timing): a kept as
            # one fp16 value, one GEMM2 MMA per K step instead of the bf16 hi / lo pair
            w2_f16 = mok.convert_f16(w2)
            f_ms, f_kernels, f_grouped, f_layer, _ = tensor_bound_forward(
                shp_tb, x_tb, wr, w13, w2_f16, args.steps, args.warmup, GEMM_FLAGS[args.gemm] | N.FLAG_W2_F16)
            tb["fp16_w2"] = {"fwd_ms": round(f_ms, 4), "tokens_per_s": round(whole_job_rate(shp_tb.T, world, f_ms), 1),
                             "grouped_gemm": f_grouped, "kernels": f_kernels,
                             "what": "MOK_FLAG_W2_F16: W2 as IEEE fp16 (exact for these bf16 weights), a as one "
                                     "fp16 value (11 significant bits) instead of a bf16 hi / lo pair"}
            del f_layer, w2_f16
            torch.cuda.empty_cache()
        if not args.no_ring_sweep:
            tb["ring_sweep"] = ring_sweep(shp_tb, x_tb, wr, w13, w2, y_tb.clone(), args.steps, args.warmup)
            tb["ring_fwd_bwd"] = ring_fwd_bwd(shp_tb, x_tb, wr, w13, w2, args.steps, args.warmup)
        del x_tb, y_tb

    if rank != 0:
        return
    peaks, peak_kind = load_peaks()
    kb = kernel_bytes(shp)
    kf = kernel_flops(shp)
    per_kernel = {}
    for name, t in trace.items():
        avg = t["total_ms"] / t["launches"]
        e = {"launches": t["launches"], "avg_ms": round(avg, 4), "share": None}
        if name in kb:
            e["GBps"] = round(kb[name] / (avg * 1e-3) / 1e9, 1)
        if name in kf:
            e["TFLOPs"] = round(kf[name] / (avg * 1e-3) / 1e12, 1)
        per_kernel[name] = e
    tot = sum(t["total_ms"] for t in trace.values())
    for name, t in trace.items():
        per_kernel[name]["share"] = round(t["total_ms"] / tot, 4)
    dom = max(trace, key=lambda n: trace[n]["total_ms"])
    dom_avg_s = trace[dom]["total_ms"] / trace[dom]["launches"] * 1e-3
    achieved = kb[dom] / dom_avg_s / 1e9
    # the committed DRAM counters were taken on the DSV3 layer with near-uniform routing
    traffic = load_traffic().get(dom) if args.workload == "dsv3" else None
    roofline = {"bound": "hbm", "achieved": round(achieved, 1), "peak": peaks["hbm_gbs"], "unit": "GB/s",
                "frac": round(achieved / peaks["hbm_gbs"], 4), "traffic": traffic, "kernel": dom,
                "peak_source": peak_kind}
    gemm_names = [n for n in kf if n in trace]
    gemm_ms = sum(trace[n]["total_ms"] / trace[n]["launches"] for n in gemm_names)
    gemm_flop = sum(kf[n] for n in gemm_names)
    gemm_tflops = gemm_flop / (gemm_ms * 1e-3) / 1e12
    fwd_gemm = [n for n in ("router_gemm", "gemm1_swiglu", "gemm2") if n in trace]
    fwd_gemm_ms = sum(trace[n]["total_ms"] / trace[n]["launches"] for n in fwd_gemm)
    fwd_gemm_tflops = sum(kf[n] for n in fwd_gemm) / (fwd_gemm_ms * 1e-3) / 1e12
    launches = sum(t["launches"] * KERNELS_PER_CALL.get(n, 1) for n, t in trace.items())

    cpu = None
    if world == 1 and not args.no_cpu_baseline:
        times, cores = cpu_sample_subprocess(CPU_SAMPLE["T"], CPU_SAMPLE["E"], repeats=1)
        cpu = {"value": CPU_SAMPLE["T"] / times[0], "unit": UNIT, "cores": cores, "kind": "oracle",
               "sample": sample_desc(CPU_SAMPLE["T"], CPU_SAMPLE["E"]), "seconds": round(times[0], 2),
               "cpu_model": cpu_model()}
        if not args.no_cpu_full:
            cpu["planned"] = cpu_planned_timings(inp, shp)

    step_bytes = 2 * T * H * 2
    line = {
        "metric": METRIC, "value": round(whole_job_rate(T, world, ms), 1), "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms, 4), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded Gaussian bf16 activations and weights; no dataset)",
        "config": {"workload": shp.name, "T": T, "hidden": H, "experts": E, "intermediate": I, "top_k": k,
                   "expert_gemm": args.gemm,
                   "router": "sigmoid+renorm", "passes": "fwd+bwd",
                   "parallelism": "replicas" if world > 1 else "single-gpu",
                   "l2": "inputs larger than L2 (22.5 GB of expert weights streamed per pass)",
                   "expert_rows_min_max": [int(counts.min()), int(counts.max())]},
        "fwd_tokens_per_s": round(whole_job_rate(T, world, fwd_ms), 1), "fwd_ms": round(fwd_ms, 4),
        "tflops_fwd_bwd": round(W.algorithmic_flops(shp, "fwd+bwd") / (ms * 1e-3) / 1e12, 1),
        "grouped_gemm": {"tflops_fwd_bwd": round(gemm_tflops, 1),
                         "frac_bf16_peak": round(gemm_tflops / peaks["bf16_tflops_sustained"], 4),
                         "tflops_fwd": round(fwd_gemm_tflops, 1),
                         "frac_bf16_peak_fwd": round(fwd_gemm_tflops / peaks["bf16_tflops_sustained"], 4),
                         "peak": peaks["bf16_tflops_sustained"], "peak_source": peak_kind + " (sustained)",
                         "frac_bf16_peak_fwd_burst": round(fwd_gemm_tflops / peaks["bf16_tflops"], 4),
                         "fwd_hbm": fwd_gemm_hbm(trace, kb, peaks),
                         "note": "at this shape (128 rows per expert) the forward GEMMs stream 22.5 GB of "
                                 "weights: HBM-bound, their HBM fraction is the one that applies"},
        "roofline": roofline,
        "kernels": per_kernel,
        "e2e": {"value": round(whole_job_rate(T, world, e2e_ms), 1), "unit": UNIT, "h2d_bytes_per_step": step_bytes,
                "d2h_bytes_per_step": step_bytes, "ms_per_step": round(e2e_ms, 4),
                "what": "pinned host x and dY copied in, forward + backward, y and dX copied out, every step; "
                        "the copies of neighbouring steps overlap the compute on a second stream"},
        "wgrad_bf16": wgrad_bf16 if wgrad_bf16_ms is not None else None,
        "skew_fwd_bwd": skew,
        "tiny_fwd_bwd": tiny,
        "fwd_bwd_ms_wgrad_bf16": round(wgrad_bf16_ms, 4) if wgrad_bf16_ms is not None else None,
        "mxfp8_fwd": mx,
        "tensor_bound_fwd": tb,
        "inputs": {"seed": 1000 * rank, "generators": "x, W_r, W13, W2, dY from seeds seed+0..4 (fp32 draws "
                   "rounded to bf16)", "sha256": {"x": tensor_sha256(x), "w_router": tensor_sha256(wr),
                                                  "dy": tensor_sha256(dy)}},
        "gpu_launches": launches,
        "clocks": clocks,
        "cpu_baseline": cpu,
    }
    print(json.dumps(line), flush=True)


def tiny_layer_step(steps, warmup, dev, stream, max_over_ranks, barrier):
    """The tiny layer's forward + backward: ms per step eager and as a replayed CUDA graph (the
    captured step is checked bitwise against the eager one)."""
    import torch

    import mixture_experts_layer_table_gb300 as mok
    from mixture_experts_layer_table_gb300 import workloads as W

    shp = W.TINY
    T, H, E, I, k = shp.T, shp.H, shp.E, shp.I, shp.k
    inp = W.make_inputs(shp, seed=0, device=str(dev))
    layer = mok.MoELayer(mok.desc_from_shape(shp), device=dev)
    y = torch.empty((T, H), dtype=torch.bfloat16, device=dev)
    g = {"dx": torch.empty((T, H), dtype=torch.bfloat16, device=dev),
         "dw_router": torch.empty((E, H), dtype=torch.float32, device=dev),
         "dw13": torch.empty((E, 2 * I, H), dtype=torch.float32, device=dev),
         "dw2": torch.empty((E, H, I), dtype=torch.float32, device=dev),
         "dgates": torch.empty((T, k), dtype=torch.float32, device=dev)}

    def step():
        layer.forward(inp["x"], inp["w_router"], inp["w13"], inp["w2"], y=y)
        layer.backward(inp["dy"], inp["x"], inp["w_router"], inp["w13"], inp["w2"], out=g)

    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    n = max(steps, 100)  # each step is tens of microseconds

    def timed(run):
        for _ in range(warmup):
            run()
        barrier()
        torch.cuda.synchronize()
        e0.record(stream)
        for _ in range(n):
            run()
        e1.record(stream)
        torch.cuda.synchronize()
        return max_over_ranks(e0.elapsed_time(e1) / n)

    eager_ms = timed(step)
    y0, g0 = y.clone(), {name: t.clone() for name, t in g.items()}
    side = torch.cuda.Stream(device=dev)
    side.wait_stream(stream)
    with torch.cuda.stream(side):
        step()
    stream.wait_stream(side)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        step()
    graph_ms = timed(graph.replay)
    if layer.status() != (0, 0):
        raise RuntimeError("device status set in the tiny layer")
    same = bool(torch.equal(y, y0) and all(torch.equal(g[name], g0[name]) for name in g))
    return {"workload": shp.name, "steps": n, "eager_ms": round(eager_ms, 4), "graph_ms": round(graph_ms, 4),
            "tokens_per_s_eager": round(T / (eager_ms * 1e-3), 1), "tokens_per_s_graph": round(T / (graph_ms * 1e-3), 1),
            "graph_bitwise_equal_to_eager": same}


def tensor_bound_forward(shp, x, w_router, w13, w2, steps, warmup, flags=0):
    """The plain forward at a tensor-bound shape (512 rows per expert): K forwards timed between
    CUDA events after W warm-ups, then K more with the per-kernel trace, SM clocks sampled
    throughout.  Returns (ms per forward, per-kernel dict, grouped-GEMM dict, layer, y)."""
    import torch

    import mixture_experts_layer_table_gb300 as mok
    from mixture_experts_layer_table_gb300 import _native as N

    y = torch.empty((shp.T, shp.H), dtype=torch.bfloat16, device=x.device)
    stream = torch.cuda.current_stream()
    layer = mok.MoELayer(mok.desc_from_shape(shp, flags=flags), device=x.device)
    sampler = ClockSampler(torch.cuda.current_device())
    sampler.start()
    for _ in range(warmup):
        layer.forward(x, w_router, w13, w2, y=y)
    torch.cuda.synchronize()
    if layer.status() != (0, 0):
        raise RuntimeError("device status set during warm-up")
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(steps):
        layer.forward(x, w_router, w13, w2, y=y)
    e1.record(stream)
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / steps
    N.trace_start(16 * steps + 16)
    for _ in range(steps):
        layer.forward(x, w_router, w13, w2, y=y)
    torch.cuda.synchronize()
    trace = N.trace_stop()
    clocks = sampler.stop()
    if layer.status() != (0, 0):
        raise RuntimeError("device status set")
    peaks, peak_kind = load_peaks()
    kf = kernel_flops(shp)
    kernels = {}
    for name, t in trace.items():
        avg = t["total_ms"] / t["launches"]
        kernels[name] = {"avg_ms": round(avg, 4)}
        if name in kf:
            kernels[name]["TFLOPs"] = round(kf[name] / (avg * 1e-3) / 1e12, 1)
    fwd_gemm = [n for n in ("gemm1_swiglu", "gemm2") if n in trace]
    g_ms = sum(trace[n]["total_ms"] / trace[n]["launches"] for n in fwd_gemm)
    g_tf = sum(kf[n] for n in fwd_gemm) / (g_ms * 1e-3) / 1e12
    # the GEMMs run inside back-to-back forwards (a long step): the sustained (power-capped)
    # measured peak is the denominator; the burst one is given too, with the SM clocks seen
    grouped = {"kernels": fwd_gemm, "ms": round(g_ms, 4), "tflops": round(g_tf, 1),
               "frac_bf16_peak_sustained": round(g_tf / peaks["bf16_tflops_sustained"], 4),
               "peak_sustained": peaks["bf16_tflops_sustained"],
               "frac_bf16_peak": round(g_tf / peaks["bf16_tflops"], 4), "peak": peaks["bf16_tflops"],
               "peak_source": peak_kind, "flops": "algorithmic: 2*R*2I*H (GEMM1) + 2*R*H*I (GEMM2)",
               "clocks": clocks}
    if clocks and clocks.get("sm_mhz") and peaks.get("sm_max_mhz"):
        # the burst peak scaled to this run's median SM clock (taking the burst figure as measured
        # at the maximum clock): how close the kernels come at the clock the power cap allowed
        scale = clocks["sm_mhz"] / peaks["sm_max_mhz"]
        grouped["frac_bf16_peak_clock_normalised"] = round(g_tf / (peaks["bf16_tflops"] * scale), 4)
    # Timed alone, as the burst peak was (the best of 10 single GEMMs): the best of 5 single
    # forwards, each after half a second of idle (the power cap lets the clocks recover), GEMM1 +
    # GEMM2 of that forward from the per-kernel trace, against the burst peak.
    sampler = ClockSampler(torch.cuda.current_device())
    sampler.start()
    best = None
    for _ in range(5):
        time.sleep(0.5)
        N.trace_start(32)
        layer.forward(x, w_router, w13, w2, y=y)
        torch.cuda.synchronize()
        tr = N.trace_stop()
        g = sum(tr[n]["total_ms"] / tr[n]["launches"] for n in fwd_gemm)
        best = g if best is None else min(best, g)
    bclocks = sampler.stop()
    if layer.status() != (0, 0):
        raise RuntimeError("device status set")
    b_tf = sum(kf[n] for n in fwd_gemm) / (best * 1e-3) / 1e12
    grouped["burst"] = {"ms": round(best, 4), "tflops": round(b_tf, 1),
                        "frac_bf16_peak": round(b_tf / peaks["bf16_tflops"], 4), "peak": peaks["bf16_tflops"],
                        "what": "best of 5 single forwards, each after 0.5 s idle (the burst peak is the best "
                                "of 10 single GEMMs)", "clocks": bclocks}
    return ms, kernels, grouped, layer, y


def run_macrobatch_study(args):
    """Macrobatch interleaving on one GPU: the T=16384 forward (256 experts, top-8, hidden 7168) as
    one call, then as M = 2 and 4 macrobatches of T/M tokens each, (a) back to back on one stream
    and (b) interleaved over two streams with a workspace each, so that the combine of macrobatch i
    can run beside the router, schedule and dispatch of macrobatch i+1.  Each macrobatch streams
    all expert weights again.  K forwards after W warm-ups, CUDA events around the whole loop.
    One JSON line."""
    import torch

    import mixture_experts_layer_table_gb300 as mok
    from mixture_experts_layer_table_gb300 import workloads as W

    mok.load()
    shp = W.RING
    inp = W.make_inputs(shp, seed=0, device="cuda", with_dy=False)
    x, wr, w13, w2 = inp["x"], inp["w_router"], inp["w13"], inp["w2"]
    y = torch.empty((shp.T, shp.H), dtype=torch.bfloat16, device="cuda")
    main = torch.cuda.current_stream()
    side = torch.cuda.Stream()

    def timed(run):
        for _ in range(args.warmup):
            run()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(main)
        for _ in range(args.steps):
            run()
        main.wait_stream(side)
        e1.record(main)
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) / args.steps

    one = mok.MoELayer(mok.desc_from_shape(shp))
    y_one = None

    def run_one():
        one.forward(x, wr, w13, w2, y=y)

    out = {"one_call_ms": round(timed(run_one), 4)}
    y_one = y.clone()
    del one
    torch.cuda.empty_cache()
    for M in (2, 4):
        tm = shp.T // M
        sub = shp.scaled(T=tm)
        layers = [mok.MoELayer(mok.desc_from_shape(sub)) for _ in range(2)]
        streams = [main, side]

        def run_seq():
            for i in range(M):
                sl = slice(i * tm, (i + 1) * tm)
                layers[0].forward(x[sl], wr, w13, w2, y=y[sl])

        def run_inter():
            # macrobatch i on stream i % 2 with workspace i % 2; a stream waits for the other's
            # previous macrobatch only through the workspace it reuses (two back)
            for i in range(M):
                st = streams[i % 2]
                sl = slice(i * tm, (i + 1) * tm)
                with torch.cuda.stream(st):
                    layers[i % 2].forward(x[sl], wr, w13, w2, y=y[sl], stream=st)

        seq_ms = timed(run_seq)
        seq_equal = bool(torch.equal(y, y_one))
        inter_ms = timed(run_inter)
        inter_equal = bool(torch.equal(y, y_one))
        ok = all(l.status() == (0, 0) for l in layers)
        out[f"M{M}"] = {"macrobatch_tokens": tm, "back_to_back_ms": round(seq_ms, 4),
                        "interleaved_two_streams_ms": round(inter_ms, 4),
                        "y_bitwise_equal_to_one_call": [seq_equal, inter_equal], "status_ok": ok}
        del layers
        torch.cuda.empty_cache()
    line = {"metric": "macrobatch study: forward ms at T=16384 (one call vs M macrobatches)",
            "value": out["one_call_ms"], "unit": "ms", "n_gpus": 1, "steps": args.steps, "warmup": args.warmup,
            "higher_is_better": False, "dtype": "bf16",
            "data": "synthetic (seeded Gaussian bf16 activations and weights; no dataset)",
            "config": {"workload": shp.name, "weights_bytes_per_pass": shp.E * 3 * shp.H * shp.I * 2},
            "study": out}
    print(json.dumps(line), flush=True)


def run_ring_sweep(args):
    """Ring forward at T=16384 (256 experts, top-8, hidden 7168): a fixed 512 MiB token ring
    and the minibatch sizes 512 / 1024 / 2368 / 2560 / 4096, each timed over K forwards after
    W warm-ups, against the same forward without the ring.  One JSON line."""
    import torch

    import mixture_experts_layer_table_gb300 as mok
    from mixture_experts_layer_table_gb300 import workloads as W

    mok.load()
    shp = W.RING
    inp = W.make_inputs(shp, seed=0, device="cuda", with_dy=False)
    plain_ms, kernels, grouped, plain, y = tensor_bound_forward(shp, inp["x"], inp["w_router"], inp["w13"], inp["w2"],
                                                                args.steps, args.warmup, GEMM_FLAGS[args.gemm])
    y_plain = y.clone()
    del plain
    sweep = ring_sweep(shp, inp["x"], inp["w_router"], inp["w13"], inp["w2"], y_plain, args.steps, args.warmup)
    best = min(sweep.values(), key=lambda v: v["fwd_ms"])
    line = {"metric": "ring forward tokens/s (fixed 512 MiB token ring, minibatch sweep)",
            "value": best["tokens_per_s"], "unit": UNIT, "n_gpus": 1, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": best["fwd_ms"], "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "bf16", "data": "synthetic (seeded Gaussian bf16 activations and weights; no dataset)",
            "config": {"workload": shp.name, "ring_bytes": W.RING_BYTES, "comm_sms": 12, "passes": "fwd",
                       "expert_gemm": args.gemm,
                       "min_minibatch_two_waves": mok.min_minibatch(0, shp.I)},
            "plain_forward_ms": round(plain_ms, 4), "plain_forward_kernels": kernels,
            "grouped_gemm_fwd": grouped, "sweep": sweep}
    print(json.dumps(line), flush=True)


def main():
    if len(sys.argv) >= 2 and sys.argv[1] == "--cpu-tiny":
        print(json.dumps(cpu_tiny_run()))
        return
    if len(sys.argv) >= 2 and sys.argv[1] == "--cpu-sample":
        T, E, rep = int(sys.argv[2]), int(sys.argv[3]), int(sys.argv[4])
        print(json.dumps(cpu_sample_run(T, E, rep)))
        return
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=30)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["mok", "reference"], default="mok")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-cpu-full", action="store_true",
                    help="skip the full-size oracle timings (DSV3 forward, skewed DSV3 forward + backward; ~1 min)")
    ap.add_argument("--no-wgrad-bf16", action="store_true", help="skip the step with bf16 weight gradients")
    ap.add_argument("--no-fp16-w2", action="store_true",
                    help="skip the T=16384 forward on an fp16 copy of W2 (MOK_FLAG_W2_F16)")
    ap.add_argument("--no-ring-sweep", action="store_true",
                    help="skip the ring-forward minibatch sweep at T=16384 in the default line")
    ap.add_argument("--no-mxfp8", action="store_true", help="skip the MXFP8 forward and forward+backward timing")
    ap.add_argument("--no-skew", action="store_true", help="skip the skewed-routing forward+backward timing")
    ap.add_argument("--no-tiny", action="store_true", help="skip the tiny layer (eager and CUDA-graph) timing")
    ap.add_argument("--no-tensor-bound", action="store_true",
                    help="skip the forward at T=16384 (tensor-bound grouped GEMMs)")
    ap.add_argument("--ring-sweep", action="store_true",
                    help="time the ring forward at T=16384 over the minibatch sweep instead")
    ap.add_argument("--macrobatch", action="store_true",
                    help="time the T=16384 forward as one call against 2 and 4 macrobatches (back to back, "
                         "and interleaved over two streams) instead")
    ap.add_argument("--gemm", choices=sorted(GEMM_FLAGS), default="auto",
                    help="expert GEMM kernels: pair / single = the row-tile kernels on CTA pairs / single "
                         "CTAs; auto = the library's default (narrow-segment pair kernel: expert rows as the MMA's N)")
    ap.add_argument("--workload", choices=sorted(WORKLOADS), default="dsv3",
                    help="dsv3: the benchmarked layer; dsv3_e16_t256 / dsv3_e16_t1024: the same "
                         "layer on 16 experts and 256 / 1024 tokens (128 / 512 rows per expert, a few "
                         "GB, for profiler captures)")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        run_reference(args, rank, world)
        return
    if args.ring_sweep:
        if rank == 0:
            run_ring_sweep(args)
        return
    if args.macrobatch:
        if rank == 0:
            run_macrobatch_study(args)
        return
    if world > 1:
        import torch
        import torch.distributed as dist
        torch.cuda.set_device(local_rank)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local_rank))
    try:
        run_mok(args, rank, world, local_rank)
    finally:
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()


if __name__ == "__main__":
    main()
