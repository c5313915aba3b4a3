"""Benchmark: batch-1 decode step through a quantized decoder stack.

One step = every quantized linear of every layer (4 dependent launches per
layer), replayed from a CUDA graph.  The stack (several GB) is far larger
than the 129 MB L2, so no flush is needed between steps.  The headline is
the 70B-shaped outlier-aware INT4 stack (80 layers, 35.3 GB, the largest
configuration on one GPU); the line also carries one sub-result per other
configuration (Gemma-2-9B INT8 at batch 1/16, Llama-3.2-3B INT4, 7B INT4 at
batch 1/4/16/64, 7B and 70B INT8, the 256 x 256 INT8 check, the Gemma INT8
stack paged from pinned host memory) under "workloads".

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
                  [--impl ours|reference] [--no-sub] [--head] [--paged] [--tiered]
                  [--stream-quant] [--no-cpu]

Prints ONE JSON line.  Under torchrun (N > 1) every rank runs an independent
replica (the method targets one GPU; no collectives) and rank 0 prints.
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

METRIC = "quantized GEMV achieved HBM GB/s (% of GB300 peak); batch-1 us per decoder layer"
FALLBACK_HBM_GBS = 6800.0
FALLBACK_TENSOR_TFLOPS = 1900.0   # dense bf16/fp16, one earlier GB300 measurement
DOMINANT_GROUP = 2  # {gate, up}: the largest launch of every layer


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=600)  # ~1 s timed: several clock samples
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", default="llama_70b_int4o")
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-sub", action="store_true",
                    help="skip the sub-results of the other configurations ('workloads')")
    ap.add_argument("--no-cpu", action="store_true", help="skip the CPU oracle baseline")
    ap.add_argument("--paged", action="store_true",
                    help="also stream the 70B and Gemma stacks through the pager")
    ap.add_argument("--head", action="store_true",
                    help="also time the 3B vocabulary lookup + lm_head (tied INT8, untied INT4)")
    ap.add_argument("--tiered", action="store_true",
                    help="also time the 70B stack with its first 40 (60) layers in HBM and "
                         "the rest streamed from pinned host memory, and with 0 (40) layers "
                         "in HBM and the rest read in place from pinned host memory")
    ap.add_argument("--stream-quant", action="store_true",
                    help="also time the streaming quantizer (checkpoint file -> pool file)")
    ap.add_argument("--fused", action="store_true",
                    help="one sequence launch per layer (the four products) instead of four")
    ap.add_argument("--no-overlap", action="store_true",
                    help="launch without programmatic dependent launch")
    ap.add_argument("--batch", type=int, default=1,
                    help="batch of the measured stack (1 = the decode headline)")
    ap.add_argument("--layers", type=int, default=None,
                    help="first L layers only (small case for profiling; not a bench line)")
    a = ap.parse_args()
    a.warmup = max(a.warmup, 3)
    return a


def profiled_traffic(profile_md: str, kernel_src: str):
    """DRAM bytes per launch of the dominant kernel, from the committed ncu
    summary, if it was taken on the kernel source as it is now (else None).
    The summary carries 'traffic_bytes_per_launch: N' and 'source_sha256: H'."""
    import hashlib
    path = os.path.join(ROOT, "profiles", profile_md)
    src = os.path.join(ROOT, kernel_src)
    if not (os.path.exists(path) and os.path.exists(src)):
        return None
    want = hashlib.sha256(open(src, "rb").read()).hexdigest()
    got, traffic = None, None
    for line in open(path):
        line = line.strip().strip("`- ")
        if line.startswith("source_sha256:"):
            got = line.split(":", 1)[1].strip()
        elif line.startswith("traffic_bytes_per_launch:"):
            traffic = int(line.split(":", 1)[1].strip().replace(",", ""))
    return traffic if got == want else None


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        try:
            d = json.load(open(p))
            for k in ("hbm_gbs", "hbm_GBps", "hbm"):
                if k in d and isinstance(d[k], (int, float)):
                    return float(d[k]), "measured"
        except Exception:
            pass
    return FALLBACK_HBM_GBS, "fallback"


def tensor_peak():
    """Dense fp16/bf16 tensor peak (TFLOP/s): the measured cuBLAS bf16 burst
    figure (fp16 runs at the bf16 rate), else the fallback."""
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        try:
            d = json.load(open(p))
            for k in ("bf16_tflops", "bf16_TFLOPs", "bf16"):
                if k in d and isinstance(d[k], (int, float)):
                    return float(d[k]), "measured"
        except Exception:
            pass
    return FALLBACK_TENSOR_TFLOPS, "fallback"


class Clocks:
    """SM clocks and throttle reasons sampled while timing.

    Samples come from NVML (libnvidia-ml, read-only queries: SM clock, its
    maximum, the active clock-event reasons) every 10 ms on a host thread,
    else from an `nvidia-smi -lms 200` child.  The summary keeps the samples
    taken inside the window between mark_start() and mark_end() (the timed
    region), and says how many there were."""
    Q = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    # NVML clock-event reason bits
    REASON_BITS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown",
                   0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown"}
    PERIOD_S = 0.01

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.window = None
        self.samples = []
        self.backend = None
        self._stop = None
        self._thread = None
        self.f = None

    def mark_start(self):
        self.window = [time.time(), None]

    def mark_end(self):
        if self.window:
            self.window[1] = time.time()

    @classmethod
    def decode(cls, mask: int) -> set:
        return {n for bit, n in cls.REASON_BITS.items() if mask & bit}

    def _nvml_open(self):
        import ctypes
        lib = ctypes.CDLL("libnvidia-ml.so.1")
        if lib.nvmlInit_v2() != 0:
            raise OSError("nvmlInit failed")
        h = ctypes.c_void_p()
        rc = -1
        try:  # the device torch calls `index`, by UUID (robust to CUDA_VISIBLE_DEVICES)
            import torch
            u = getattr(torch.cuda.get_device_properties(self.index), "uuid", None)
            if u is not None:
                rc = lib.nvmlDeviceGetHandleByUUID(("GPU-" + str(u)).encode(), ctypes.byref(h))
        except Exception:
            rc = -1
        if rc != 0 and lib.nvmlDeviceGetHandleByIndex_v2(ctypes.c_uint(self.index),
                                                         ctypes.byref(h)) != 0:
            raise OSError("no NVML handle")
        reasons = getattr(lib, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            lib.nvmlDeviceGetCurrentClocksThrottleReasons
        mx = ctypes.c_uint()
        if lib.nvmlDeviceGetMaxClockInfo(h, 1, ctypes.byref(mx)) != 0:   # 1 = SM clock
            raise OSError("no max clock")

        def sample():
            mhz, r = ctypes.c_uint(), ctypes.c_ulonglong()
            if lib.nvmlDeviceGetClockInfo(h, 1, ctypes.byref(mhz)) != 0:
                return None
            if reasons(h, ctypes.byref(r)) != 0:
                return None
            return (time.time(), float(mhz.value), float(mx.value), self.decode(r.value))
        return sample

    def __enter__(self):
        import threading
        try:
            sample = self._nvml_open()
            self.backend = "nvml"
            self._stop = threading.Event()

            def loop():
                while not self._stop.is_set():
                    x = sample()
                    if x is not None:
                        self.samples.append(x)
                    self._stop.wait(self.PERIOD_S)
            self._thread = threading.Thread(target=loop, daemon=True)
            self._thread.start()
            return self
        except Exception:
            pass
        try:
            self.f = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.Q}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=self.f, stderr=subprocess.DEVNULL)
            self.backend = "nvidia-smi"
        except (FileNotFoundError, OSError):
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self._thread:
            self._stop.set()
            self._thread.join(timeout=5)
        if self.proc:
            self.proc.terminate()
            self.proc.wait(timeout=10)

    def summary(self):
        if self.backend == "nvml":
            out = self.summarize(list(self.samples), self.window, slack=0.0)
        elif self.proc:
            self.f.flush()
            out = self.parse(open(self.f.name).read(), self.window)
        else:
            return None
        if out:
            out["source"] = self.backend
        return out

    @staticmethod
    def parse(text: str, window=None):
        """nvidia-smi CSV lines to samples, then summarize()."""
        import datetime
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        samples = []
        for line in text.strip().splitlines():
            r = [c.strip() for c in line.split(",")]
            if len(r) < 10:
                continue
            try:
                t = datetime.datetime.strptime(r[0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
                samples.append((t, float(r[2]), float(r[3]),
                                {n for n, v in zip(names, r[6:10]) if v.lower() == "active"}))
            except ValueError:
                continue
        return Clocks.summarize(samples, window)

    @staticmethod
    def summarize(samples, window=None, slack=0.05):
        """Median SM clock, the maximum clock and the throttle reasons seen,
        over the samples (t, sm_mhz, max_mhz, reasons) inside window = [t0, t1]
        (host epoch seconds, widened by `slack` for nvidia-smi's coarser
        timestamps) when there are any, else over all samples."""
        if not samples:
            return None
        inside, in_region = samples, 0
        if window and window[1] is not None:
            w = [x for x in samples if window[0] - slack <= x[0] <= window[1] + slack]
            if w:
                inside, in_region = w, len(w)
        reasons = set()
        for x in inside:
            reasons |= x[3]
        return {"sm_mhz": statistics.median(x[1] for x in inside),
                "sm_max_mhz": max(x[2] for x in inside), "reasons": sorted(reasons),
                "samples": len(inside), "samples_in_timed_region": in_region,
                "samples_total": len(samples)}


def cpu_baseline_one_thread(wl_name: str):
    """The same oracle on one host thread (BLAS pinned to one thread in a
    child process, since the thread count is fixed when numpy loads), on the
    gate matrix of layer 0 (k for the 70B layer): (GB/s, sample text), or
    None if it fails."""
    one = ("k",) if wl_name in CPU_SAMPLE else ("gate",)
    code = ("import json, bench; g, t, smp, th = bench.cpu_baseline(%r, 4.0, %r); "
            "print(json.dumps([g, smp]))" % (wl_name, one))
    env = dict(os.environ, OMP_NUM_THREADS="1", OPENBLAS_NUM_THREADS="1", MKL_NUM_THREADS="1")
    try:
        out = subprocess.run([sys.executable, "-c", code], cwd=ROOT, env=env, capture_output=True,
                             text=True, timeout=120)
        g, smp = json.loads(out.stdout.strip().splitlines()[-1])
        return g, smp
    except Exception:
        return None


# Matrices of layer 0 the CPU baseline samples per workload (the 70B layer's
# 28672-wide matrices would take minutes to generate and quantize in fp64 on
# the host; its k and v projections are the same format at a bounded size).
CPU_SAMPLE = {"llama_70b_int4o": ("k", "v")}


def cpu_baseline(wl_name: str, budget_s: float = 12.0, only=None):
    """The CPU oracle, as it stands, on a bounded sample: the products of one
    layer's matrices (quantized by the oracle itself; `only`: a subset of
    them), repeated until about budget_s of CPU work.  Returns (GB/s,
    seconds, sample text, threads)."""
    import numpy as np

    from oracle import qz_oracle as O
    from weight_only_quantized_dequant_gb300 import synthetic as S

    wl = S.WORKLOADS[wl_name]
    if only is None:
        only = CPU_SAMPLE.get(wl_name)
    mats = []
    for m in S.MATS:
        if only is not None and m not in only:
            continue
        N, K = wl.shape(m)
        W = S.weight(N, K, S.matrix_seed(wl, 0, m), dist=wl.dist).numpy()
        x = S.activation(1, K, 11 + len(mats)).numpy()
        if wl.fmt == "int8":
            q, s = O.int8_quantize(W)
            mats.append(("int8", (q, s), x, O.int8_weight_bytes(N, K)))
        else:
            n_out = O.default_n_out(K)
            perm = O.select_outliers(O.saliency_fixed(W), np.abs(x[0]).astype(np.float32), n_out)
            wo, q4, s = O.int4o_quantize(W, perm, n_out)
            mats.append(("int4o", (wo, q4, s, perm, n_out, K), x, O.int4o_weight_bytes(N, K, n_out)))
    done_bytes, t_total, reps = 0, 0.0, 0
    while t_total < budget_s and reps < 50:
        for kind, w, x, nbytes in mats:
            t0 = time.perf_counter()
            if kind == "int8":
                O.int8_product_ref(w[0], w[1], x)
            else:
                O.int4o_product_ref(*w, x)
            t_total += time.perf_counter() - t0
            done_bytes += nbytes
        reps += 1
    threads = len(os.sched_getaffinity(0))
    try:
        from threadpoolctl import threadpool_info
        info = threadpool_info()
        if info:
            threads = max(i.get("num_threads", 1) for i in info)
    except Exception:
        pass
    which = "all 7 matrices" if only is None else "+".join(only)
    sample = (f"oracle fp64 products of {which} of layer 0 of {wl_name}, "
              f"{reps} pass(es), {done_bytes / 1e9:.2f} GB of packed weights")
    return done_bytes / t_total / 1e9, t_total, sample, threads


def max_over_ranks(dist_ctx, values, device=None):
    """Each timing's largest value over all ranks: the slowest replica sets
    the job's time.  Without a process group, the values themselves."""
    if dist_ctx is None:
        return [float(v) for v in values]
    import torch
    t = torch.tensor([float(v) for v in values], dtype=torch.float64, device=device)
    dist_ctx.all_reduce(t, op=dist_ctx.ReduceOp.MAX)
    return [float(v) for v in t.tolist()]


def job_gbs(world: int, bytes_per_step: float, ms_per_step: float) -> float:
    """Whole-job GB/s: each of the world replicas moves bytes_per_step per
    step, and the job's step takes ms_per_step (the slowest rank)."""
    return world * bytes_per_step / (ms_per_step * 1e-3) / 1e9


def run_reference(a):
    """--impl reference: the CPU oracle timed on the host cores."""
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    import numpy as np  # noqa: F401

    from oracle import qz_oracle as O
    from weight_only_quantized_dequant_gb300 import synthetic as S

    wl = S.WORKLOADS[a.workload]
    N, K = wl.shape("down")
    # a bounded sample: at most 16 M weights of the down projection's rows
    # (all of them but for the 70B layer, 512 of its 8192 rows)
    N = min(N, max(1, (1 << 24) // K))
    W = S.weight(N, K, S.matrix_seed(wl, 0, "down"), dist=wl.dist).numpy()
    x = S.activation(1, K, 5).numpy()
    if wl.fmt == "int8":
        q, s = O.int8_quantize(W)
        step = lambda: O.int8_product_ref(q, s, x)  # noqa: E731
        nbytes = O.int8_weight_bytes(N, K)
    else:
        n_out = O.default_n_out(K)
        perm = O.select_outliers(O.saliency_fixed(W), np.abs(x[0]).astype(np.float32), n_out)
        wo, q4, s4 = O.int4o_quantize(W, perm, n_out)
        step = lambda: O.int4o_product_ref(wo, q4, s4, perm, n_out, K, x)  # noqa: E731
        nbytes = O.int4o_weight_bytes(N, K, n_out)
    for _ in range(a.warmup):
        step()
    t0 = time.perf_counter()
    for _ in range(a.steps):
        step()
    dt = (time.perf_counter() - t0) / a.steps
    gbs = nbytes / dt / 1e9
    cores = len(os.sched_getaffinity(0))
    rows = "" if N == wl.shape("down")[0] else f", {N} of its {wl.shape('down')[0]} rows"
    sample = f"oracle fp64 product of the down projection ({N}x{K}{rows}) of layer 0, per step"
    out = {"impl": "reference", "metric": METRIC, "value": round(gbs, 4), "unit": "GB/s",
           "n_gpus": a.gpus, "steps": a.steps, "warmup": a.warmup,
           "ms_per_step": round(dt * 1e3, 3), "higher_is_better": True, "scaling": "weak",
           "vs_baseline": None, "dtype": "f64", "data": "synthetic",
           "config": {"workload": a.workload, "sample": f"down projection of layer 0{rows}"},
           "cpu_baseline": {"value": round(gbs, 4), "unit": "GB/s", "cores": cores,
                            "kind": "oracle", "sample": sample},
           "e2e": {"value": round(gbs, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                   "d2h_bytes_per_step": 0}}
    print(json.dumps(out), flush=True)


def copy_probe_gbs(device) -> float:
    """Device-to-device copy of 2 GiB with torch (read + write bytes / time):
    context for the HBM fallback peak, not a roofline denominator."""
    import torch
    a = torch.empty((1 << 31,), dtype=torch.uint8, device=device)
    b = torch.empty_like(a)
    for _ in range(3):
        b.copy_(a)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(10):
        b.copy_(a)
    e1.record()
    torch.cuda.synchronize(device)
    gbs = 2 * a.numel() * 10 / (e0.elapsed_time(e1) * 1e-3) / 1e9
    del a, b
    torch.cuda.empty_cache()
    return gbs


# The other configurations, reported as sub-results of the headline line.
SUB_CONFIGS = [("gemma2_9b_int8", 1), ("gemma2_9b_int8", 16), ("llama32_3b_int4o", 1),
               ("llama_7b_int4o", 1), ("llama_7b_int4o", 4), ("llama_7b_int4o", 16),
               ("llama_7b_int4o", 64), ("llama_7b_int8", 1), ("llama_70b_int8", 1),
               ("llama_70b_int4o", 1)]


def measure_tiny(steps: int, warmup: int, device, peak: float) -> dict:
    """The 256 x 256 INT8 check (W ~ N(0, 0.02^2), x ~ N(0, 1), CPU seed 0):
    quantized on the GPU, one GEMV launch per step replayed from a CUDA
    graph of `steps` launches.  The 64 KiB matrix stays in L2, so this is a
    launch-latency figure, not an HBM one."""
    import torch

    from weight_only_quantized_dequant_gb300 import api
    from weight_only_quantized_dequant_gb300 import synthetic as S

    W, x = S.tiny_int8_inputs()
    w = api.quantize_int8(W.to(device))
    xd = x[0].to(device)
    y = torch.empty((256,), dtype=torch.float16, device=device)
    s = torch.cuda.Stream(device=device)
    s.wait_stream(torch.cuda.current_stream(device))
    with torch.cuda.stream(s):
        for _ in range(warmup):
            api.gemv_int8(w, xd, y, stream=s)
    torch.cuda.synchronize(device)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        for _ in range(steps):
            api.gemv_int8(w, xd, y, stream=s)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(s):
        g.replay()
        e0.record(s)
        g.replay()
        e1.record(s)
    torch.cuda.synchronize(device)
    us = e0.elapsed_time(e1) * 1e3 / steps
    nbytes = w.nbytes() + 2 * 256 + 2 * 256
    return {"batch": 1, "layers": 1, "us_per_launch": round(us, 3),
            "ms_per_step": round(us * 1e-3, 6), "gbs": round(nbytes / (us * 1e-6) / 1e9, 2),
            "pct_of_peak": round(100.0 * nbytes / (us * 1e-6) / 1e9 / peak, 3),
            "note": "64 KiB matrix, L2-resident: launch-bound"}


def measure(wl_name: str, batch: int, steps: int, warmup: int, dist_ctx=None,
            clocks=False, device=None, layers=None, overlap=True, fused=False, e2e=True):
    """Build the stack, capture one step, time it.  Returns a dict (e2e:
    also time the step with its host copies)."""
    import torch

    from weight_only_quantized_dequant_gb300 import stack as ST
    from weight_only_quantized_dequant_gb300 import synthetic as S

    wl = S.WORKLOADS[wl_name]
    t_build = time.perf_counter()
    st = ST.LayerStack(wl, layers=layers, batch=batch, device=device, fused=fused)
    torch.cuda.synchronize()
    t_build = time.perf_counter() - t_build

    # one contiguous host<->device staging area per direction for e2e
    xs = [x for xs in st.x for x in xs]
    ys = [y for ys in st.y for yy in ys for y in yy]
    x_dev = torch.cat([x.reshape(-1) for x in xs])
    y_dev = torch.empty((sum(y.numel() for y in ys),), dtype=torch.float16, device=device)
    off = 0
    for l in range(st.n_layers):           # re-point inputs/outputs into the staging areas
        for g in range(len(st.x[l])):
            n = st.x[l][g].numel()
            st.x[l][g] = x_dev[off:off + n].view_as(st.x[l][g])
            off += n
    off = 0
    for l in range(st.n_layers):
        for g in range(len(st.y[l])):
            for k in range(len(st.y[l][g])):
                n = st.y[l][g][k].numel()
                st.y[l][g][k] = y_dev[off:off + n].view_as(st.y[l][g][k])
                off += n
    x_host = x_dev.cpu().pin_memory()
    y_host = torch.empty(y_dev.shape, dtype=torch.float16).pin_memory()

    # Two graphs of one step: the plain one is the timed step; the second
    # brackets every launch of the dominant group with timing events (event
    # nodes serialise their neighbours, so it is timed separately).
    from weight_only_quantized_dequant_gb300 import api
    s = torch.cuda.Stream(device=device)

    def _ev():  # external: a timing node inside the captured graph
        try:
            return torch.cuda.Event(enable_timing=True, external=True)
        except TypeError:
            return torch.cuda.Event(enable_timing=True)
    ev = [(_ev(), _ev()) for _ in range(st.n_layers)]

    def step(stream, events):
        for l in range(st.n_layers):
            if st.fused:  # one launch per layer: that launch is the timed kernel
                if events:
                    ev[l][0].record(stream)
                st.run_layer_fused(l, stream)
                if events:
                    ev[l][1].record(stream)
                continue
            for g in range(len(S.GROUPS)):
                if events and g == DOMINANT_GROUP:
                    ev[l][0].record(stream)
                st.run_group(l, g, stream)
                if events and g == DOMINANT_GROUP:
                    ev[l][1].record(stream)

    api.set_overlap(overlap)
    s.wait_stream(torch.cuda.current_stream(device))
    with torch.cuda.stream(s):
        step(s, False)
    torch.cuda.synchronize(device)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=s):
        step(s, False)
    graph_ev = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph_ev, stream=s):
        step(s, True)
    api.set_overlap(False)
    torch.cuda.synchronize(device)

    def barrier():
        if dist_ctx is not None:
            dist_ctx.barrier()
        torch.cuda.synchronize(device)

    with torch.cuda.stream(s):
        for _ in range(warmup):
            graph.replay()
    barrier()
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    clk = Clocks(device.index if device is not None else 0) if clocks else None
    if clk:
        clk.__enter__()
        time.sleep(0.3)
    if clk:
        clk.mark_start()
    with torch.cuda.stream(s):
        t0.record(s)
        for _ in range(steps):
            graph.replay()
        t1.record(s)
    barrier()
    if clk:
        clk.mark_end()
        clk.__exit__(None, None, None)
    ms = t0.elapsed_time(t1) / steps
    # instrumented graph: same warm-up and step count, dominant launches timed
    with torch.cuda.stream(s):
        for _ in range(warmup):
            graph_ev.replay()
    barrier()
    dom_sum, n_dom = 0.0, 0
    with torch.cuda.stream(s):
        for _ in range(steps):
            graph_ev.replay()
            s.synchronize()
            dom_sum += sum(a.elapsed_time(b) for a, b in ev)
            n_dom += len(ev)
    barrier()
    dom_avg_ms = dom_sum / n_dom

    # e2e: pinned host inputs -> device, step, outputs -> pinned host
    e2e_serial_ms = e2e_ms = float("nan")
    if e2e:
        with torch.cuda.stream(s):
            for _ in range(warmup):
                x_dev.copy_(x_host, non_blocking=True)
                graph.replay()
                y_host.copy_(y_dev, non_blocking=True)
        barrier()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(s):
            e0.record(s)
            for _ in range(steps):
                x_dev.copy_(x_host, non_blocking=True)
                graph.replay()
                y_host.copy_(y_dev, non_blocking=True)
            e1.record(s)
        barrier()
        e2e_serial_ms = e0.elapsed_time(e1) / steps
        e2e_ms = e2e_pipelined(st, s, graph, x_dev, x_host, y_dev, y_host, steps, warmup, barrier,
                               overlap, device)

    dom_names = S.GROUPS[DOMINANT_GROUP]
    dom_bytes = sum(st.layers[0].mats[m].nbytes() for m in dom_names)
    dom_wbytes = dom_bytes
    K_dom = wl.shape(dom_names[0])[1]
    dom_bytes += 2 * batch * K_dom + sum(2 * batch * wl.shape(m)[0] for m in dom_names)
    if wl.fmt == "int4o":
        dom_bytes += 4 * K_dom
    if st.fused:
        dom_names = ("layer",)
        dom_bytes = st.weight_bytes_per_layer() + st.io_bytes_per_layer()
    out = {
        "workload": wl_name, "batch": batch, "layers": st.n_layers,
        "bytes_per_step": st.bytes_per_step(),
        "padded_bytes_per_step": st.n_layers * (st.padded_weight_bytes_per_layer() +
                                                st.io_bytes_per_layer()),
        "weight_bytes_per_layer": st.weight_bytes_per_layer(),
        "ms_per_step": ms, "us_per_layer": ms * 1e3 / st.n_layers,
        "gbs": st.bytes_per_step() / (ms * 1e-3) / 1e9,
        "dominant": {"group": "+".join(dom_names), "bytes_per_launch": dom_bytes,
                     "weight_bytes": dom_wbytes,
                     "avg_ms": dom_avg_ms, "gbs": dom_bytes / (dom_avg_ms * 1e-3) / 1e9,
                     # multiply-adds of the launch (every weight times every input row)
                     "flops_per_launch": 2.0 * batch * sum(
                         wl.shape(m)[0] * wl.shape(m)[1] for m in dom_names) if not st.fused else 0.0},
        "e2e_ms": e2e_ms, "e2e_gbs": st.bytes_per_step() / (e2e_ms * 1e-3) / 1e9,
        "e2e_serial_ms": e2e_serial_ms,
        "h2d": st.h2d_bytes_per_step(), "d2h": st.d2h_bytes_per_step(),
        "launches_per_step": st.launches_per_step(), "build_s": t_build,
        "stack_gb": st.n_layers * st.weight_bytes_per_layer() / 1e9,
    }
    if clk:
        out["clocks"] = clk.summary()
    del graph, st
    torch.cuda.empty_cache()
    return out


def e2e_pipelined(st, s, graph, x_dev, x_host, y_dev, y_host, steps, warmup, barrier, overlap,
                  device, chunks: int = 6) -> float:
    """End to end with the host copies overlapped: one graph per step in
    which the inputs go up in `chunks` layer ranges on one copy stream, each
    range's layers wait only for their own inputs, and each range's outputs
    go down on a second copy stream as soon as its last layer is done.
    Checked once against the serial step's outputs (bit for bit); returns ms
    per step."""
    import torch

    from weight_only_quantized_dequant_gb300 import api
    from weight_only_quantized_dequant_gb300 import synthetic as S
    L = st.n_layers
    xo, yo = [0], [0]
    for l in range(L):
        xo.append(xo[-1] + sum(x.numel() for x in st.x[l]))
        yo.append(yo[-1] + sum(y.numel() for yy in st.y[l] for y in yy))
    C = max(1, min(chunks, L))
    b = [L * c // C for c in range(C + 1)]
    cin = torch.cuda.Stream(device=device)
    cout = torch.cuda.Stream(device=device)
    ev_in = [torch.cuda.Event() for _ in range(C)]
    ev_out = [torch.cuda.Event() for _ in range(C)]

    def step():
        cin.wait_stream(s)
        cout.wait_stream(s)
        with torch.cuda.stream(cin):
            for c in range(C):
                x_dev[xo[b[c]]:xo[b[c + 1]]].copy_(x_host[xo[b[c]]:xo[b[c + 1]]],
                                                   non_blocking=True)
                ev_in[c].record(cin)
        for c in range(C):
            s.wait_event(ev_in[c])
            for l in range(b[c], b[c + 1]):
                if st.fused:
                    st.run_layer_fused(l, s)
                else:
                    for g in range(len(S.GROUPS)):
                        st.run_group(l, g, s)
            ev_out[c].record(s)
            cout.wait_event(ev_out[c])
            with torch.cuda.stream(cout):
                y_host[yo[b[c]]:yo[b[c + 1]]].copy_(y_dev[yo[b[c]]:yo[b[c + 1]]],
                                                    non_blocking=True)
        s.wait_stream(cin)
        s.wait_stream(cout)

    y_ref = y_host.clone()  # the serial step's outputs (the last timed step)
    api.set_overlap(overlap)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        step()
    api.set_overlap(False)
    y_host.zero_()
    with torch.cuda.stream(s):
        g.replay()
    barrier()
    if not torch.equal(y_host, y_ref):
        raise RuntimeError("pipelined end-to-end step differs from the serial one")
    with torch.cuda.stream(s):
        for _ in range(warmup):
            g.replay()
    barrier()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(s):
        e0.record(s)
        for _ in range(steps):
            g.replay()
        e1.record(s)
    barrier()
    del g
    return e0.elapsed_time(e1) / steps


def h2d_probe_gbs(device, nbytes=1 << 30) -> float:
    """Pinned host -> device copy bandwidth of the link on this machine."""
    import torch
    h = torch.empty((nbytes,), dtype=torch.uint8).pin_memory()
    d = torch.empty((nbytes,), dtype=torch.uint8, device=device)
    for _ in range(2):
        d.copy_(h, non_blocking=True)
    torch.cuda.synchronize(device)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(5):
        d.copy_(h, non_blocking=True)
    e1.record()
    torch.cuda.synchronize(device)
    return nbytes * 5 / (e0.elapsed_time(e1) * 1e-3) / 1e9


def paged_parts(ps, device, layers: int = 8) -> dict:
    """The pager's two halves timed alone, per layer: the host->device copy
    of a packed layer into a slot (copy stream, no GEMVs) and the layer's
    GEMV launches from a filled slot (compute stream, no copies).  A paged
    layer that overlaps them perfectly takes max(t_copy, t_gemv)."""
    import torch
    n = max(2, layers)
    cp, cs = ps.copy_stream, ps.compute_stream
    torch.cuda.synchronize(device)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(cp):
        e0.record(cp)
        for l in range(n):
            ps.slots[l % 2].copy_(ps.blobs[l % ps.distinct], non_blocking=True)
        e1.record(cp)
    torch.cuda.synchronize(device)
    t_copy = e0.elapsed_time(e1) / n
    # slot j <- host layer j, then the GEMVs of those two layers alternately
    with torch.cuda.stream(cp):
        for j in range(2):
            ps.slots[j].copy_(ps.blobs[j % ps.distinct], non_blocking=True)
    torch.cuda.synchronize(device)
    for l in range(2):                                   # warm-up
        ps.run_layer(ps._views[l % 2], l % 2 % ps.distinct, cs)
    torch.cuda.synchronize(device)
    e0.record(cs)
    for l in range(n):
        ps.run_layer(ps._views[l % 2], l % 2 % ps.distinct, cs)
    e1.record(cs)
    torch.cuda.synchronize(device)
    t_gemv = e0.elapsed_time(e1) / n
    return {"t_copy_us": round(t_copy * 1e3, 2), "t_gemv_us": round(t_gemv * 1e3, 2),
            "copy_gbs": round(ps.blob_bytes / (t_copy * 1e-3) / 1e9, 1)}


def measure_paged(wl_name: str, steps: int, warmup: int, device, distinct: int = 4):
    """Stack streamed layer by layer from pinned host memory through the
    pager (two device slots, copy stream + compute stream)."""
    import torch

    from weight_only_quantized_dequant_gb300 import stack as ST
    from weight_only_quantized_dequant_gb300 import synthetic as S

    ps = ST.PagedStack(S.WORKLOADS[wl_name], distinct=distinct, device=device)
    torch.cuda.synchronize(device)
    cs = ps.compute_stream
    for _ in range(warmup):
        ps.run_step()
    torch.cuda.synchronize(device)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(cs)
    for _ in range(steps):
        ps.run_step()
    e1.record(cs)
    torch.cuda.synchronize(device)
    ms = e0.elapsed_time(e1) / steps
    out = {"workload": wl_name, "layers": ps.n_layers, "distinct_host_layers": ps.distinct,
           "layer_bytes": ps.blob_bytes, "ms_per_step": round(ms, 3),
           "us_per_layer": round(ms * 1e3 / ps.n_layers, 2),
           "h2d_gbs": round(ps.n_layers * ps.blob_bytes / (ms * 1e-3) / 1e9, 1),
           "link_probe_gbs": round(h2d_probe_gbs(device), 1),
           "link": "pinned host -> device cudaMemcpyAsync, 1 GiB, 5 copies"}
    out["link_frac"] = round(out["h2d_gbs"] / out["link_probe_gbs"], 4)
    parts = paged_parts(ps, device)
    out.update(parts)
    t_layer = ms * 1e3 / ps.n_layers
    # 1.0 = the layer costs exactly its slower half (copy and GEMVs fully overlapped)
    out["t_layer_over_max_copy_gemv"] = round(t_layer / max(parts["t_copy_us"],
                                                            parts["t_gemv_us"]), 4)
    ps.close()
    del ps
    torch.cuda.empty_cache()
    return out


def measure_head(name: str, steps: int, warmup: int, device):
    """The steps either side of the stack: INT8 vocabulary lookup of one
    token plus the output projection over the whole vocabulary, tied (the
    INT8 table) or untied (outlier-aware INT4).  Each variant is one captured
    graph (lookup + lm_head GEMV) replayed `steps` times."""
    import torch

    from weight_only_quantized_dequant_gb300 import api
    from weight_only_quantized_dequant_gb300 import synthetic as S

    hd = S.HEADS[name]
    V, H = hd.vocab, hd.hidden
    W = S.weight(V, H, hd.seed_base, device=device)
    table = api.quantize_int8(W)
    del W
    n_out = api.default_n_out(H)
    W2 = S.weight(V, H, hd.seed_base + 1, device=device)
    colsum = torch.zeros((H,), dtype=torch.int64, device=device)
    api.saliency_accumulate(W2, colsum)
    perm = api.select_outliers(colsum, S.x_profile(H, n_out, hd.seed_base + 2, device=device), n_out)
    w4 = api.quantize_int4_outlier(W2, perm, n_out)
    del W2
    tok = S.tokens(1, V, hd.seed_base + 4, device=device)
    h = S.activation(1, H, hd.seed_base + 3, device=device)[0]
    emb = torch.empty((1, H), dtype=torch.float16, device=device)
    logits = torch.empty((V,), dtype=torch.float16, device=device)
    torch.cuda.synchronize(device)
    s = torch.cuda.Stream(device=device)
    io = 4 + 2 * H + 2 * H + 2 * V       # token, looked-up row, hidden state, logits
    variants = {"tied_int8": (lambda st: api.gemv_int8(table, h, logits, stream=st),
                              H + 4 + table.nbytes() + io),
                "untied_int4o": (lambda st: api.gemv_int4_outlier(w4, h, logits, stream=st),
                                 H + 4 + w4.nbytes() + 4 * H + io)}
    out = {"vocab": V, "hidden": H}
    for key, (head, nbytes) in variants.items():
        def step(st):
            api.embed_int8(table, tok, emb, stream=st)
            head(st)
        s.wait_stream(torch.cuda.current_stream(device))
        with torch.cuda.stream(s):
            step(s)
        torch.cuda.synchronize(device)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            step(s)
        with torch.cuda.stream(s):
            for _ in range(warmup):
                g.replay()
        torch.cuda.synchronize(device)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(s):
            e0.record(s)
            for _ in range(steps):
                g.replay()
            e1.record(s)
        torch.cuda.synchronize(device)
        ms = e0.elapsed_time(e1) / steps
        out[key] = {"us_per_token": round(ms * 1e3, 3), "bytes": nbytes,
                    "gbs": round(nbytes / (ms * 1e-3) / 1e9, 1)}
        del g
    assert api.device_error() == 0
    del table, w4
    torch.cuda.empty_cache()
    return out


def measure_tiered(wl_name: str, resident: int, steps: int, warmup: int, device,
                   distinct: int = 4, mode: str = "paged"):
    """First `resident` layers in HBM, the rest in pinned host memory,
    streamed through the pager (mode "paged") or read in place by the
    zero-copy GEMV (mode "zero_copy")."""
    import torch

    from weight_only_quantized_dequant_gb300 import api
    from weight_only_quantized_dequant_gb300 import stack as ST
    from weight_only_quantized_dequant_gb300 import synthetic as S

    ts = ST.TieredStack(S.WORKLOADS[wl_name], resident, distinct=distinct, device=device,
                        mode=mode)
    torch.cuda.synchronize(device)
    cs = ts.stream
    for _ in range(warmup):
        ts.run_step()
    torch.cuda.synchronize(device)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(cs)
    for _ in range(steps):
        ts.run_step()
    e1.record(cs)
    torch.cuda.synchronize(device)
    assert api.device_error() == 0
    ms = e0.elapsed_time(e1) / steps
    tier_b = ts.n_layers - ts.resident
    out = {"workload": wl_name, "mode": mode, "layers": ts.n_layers, "resident": ts.resident,
           "ms_per_step": round(ms, 3), "us_per_layer": round(ms * 1e3 / ts.n_layers, 2),
           "gbs": round(ts.bytes_per_step() / (ms * 1e-3) / 1e9, 1),
           "host_layer_bytes": ts.weight_bytes_per_layer}
    if tier_b and mode == "zero_copy" and ts.resident == 0:
        # every weight byte crossed the host link once: the in-place read rate
        out["host_read_gbs"] = round(tier_b * ts.weight_bytes_per_layer / (ms * 1e-3) / 1e9, 1)
    if tier_b and mode == "paged":
        parts = paged_parts(ts.host, device)
        out.update(parts)
        # resident layers cost their GEMVs; paged ones the slower half
        ideal_ms = (ts.resident * parts["t_gemv_us"] +
                    tier_b * max(parts["t_copy_us"], parts["t_gemv_us"])) * 1e-3
        out["t_step_over_ideal"] = round(ms / ideal_ms, 4)
    ts.close()
    del ts
    torch.cuda.empty_cache()
    return out


def measure_stream_quant(wl_name: str, layers: int, device) -> dict:
    """Offline side: a synthetic checkpoint of `layers` layers written to a
    temporary directory, quantized layer by layer into a pool file (timed, with
    the host memory it held), then the pool read back into pinned memory."""
    import resource
    import shutil

    import torch

    from weight_only_quantized_dequant_gb300 import checkpoint as C
    from weight_only_quantized_dequant_gb300 import synthetic as S

    wl = S.WORKLOADS[wl_name]
    tmp = tempfile.mkdtemp(prefix="qz_ckpt_")
    try:
        ck, pool = os.path.join(tmp, "w.safetensors"), os.path.join(tmp, "w.qz")
        t = time.perf_counter()
        size = C.write_synthetic_checkpoint(ck, wl, layers, device=device)
        t_write = time.perf_counter() - t
        rss0 = resource.getrusage(resource.RUSAGE_SELF).ru_maxrss
        torch.cuda.synchronize(device)
        t = time.perf_counter()
        st = C.quantize_stream(ck, wl, layers, pool, device=device)
        t_q = time.perf_counter() - t
        rss1 = resource.getrusage(resource.RUSAGE_SELF).ru_maxrss
        t = time.perf_counter()
        hdr, blobs = C.load_pool(pool)
        t_load = time.perf_counter() - t
        return {"workload": wl_name, "layers": layers, "checkpoint_gb": round(size / 1e9, 3),
                "write_s": round(t_write, 2), "quantize_s": round(t_q, 2),
                "quantize_gbs": round(st["checkpoint_bytes"] / t_q / 1e9, 2),
                "host_buffers_mb": round(st["host_buffer_bytes"] / 2**20, 1),
                "peak_rss_growth_mb": round(max(0, rss1 - rss0) / 1024, 1),
                "pool_gb": round(st["pool_bytes"] / 1e9, 3),
                "pool_load_gbs": round(st["pool_bytes"] / t_load / 1e9, 2),
                "note": "checkpoint freshly written: its pages are likely in the page cache"}
    finally:
        shutil.rmtree(tmp, ignore_errors=True)


def main():
    a = parse()
    if a.impl == "reference":
        return run_reference(a)
    import torch

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if not torch.cuda.is_available():
        print(json.dumps({"error": "no CUDA device"}))
        return 1
    device = torch.device("cuda", local)
    torch.cuda.set_device(device)
    dist_ctx = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=device)
        dist_ctx = dist

    from weight_only_quantized_dequant_gb300 import build
    if rank == 0:
        build.build()
    if dist_ctx is not None:
        dist_ctx.barrier()

    r = measure(a.workload, a.batch, a.steps, a.warmup, dist_ctx, clocks=(rank == 0), device=device,
                layers=a.layers, overlap=not a.no_overlap, fused=a.fused)
    ms_all, e2e_all = max_over_ranks(dist_ctx, [r["ms_per_step"], r["e2e_ms"]], device)

    extra = {}
    if not a.no_sub and rank == 0 and a.layers is None:
        peak_sub, _ = peaks()
        for name, b in SUB_CONFIGS:
            if (name, b) == (a.workload, a.batch):
                continue
            e = measure(name, b, max(20, a.steps // 4), a.warmup, None, device=device,
                        overlap=not a.no_overlap, e2e=False)
            extra[f"{name}_b{b}"] = {
                "batch": b, "layers": e["layers"], "ms_per_step": round(e["ms_per_step"], 4),
                "us_per_layer": round(e["us_per_layer"], 3), "gbs": round(e["gbs"], 2),
                "pct_of_peak": round(100.0 * e["gbs"] / peak_sub, 2),
                "dominant_gbs": round(e["dominant"]["gbs"], 2),
                "stack_gb": round(e["stack_gb"], 3)}
        extra["tiny_int8_b1"] = measure_tiny(max(100, a.steps), a.warmup, device, peak_sub)
        # the Gemma INT8 stack as the ELG page runs it: every layer streamed
        # from pinned host memory through the pager
        extra["gemma2_9b_int8_paged"] = measure_paged("gemma2_9b_int8", 3, 1, device)

    if a.head and rank == 0:
        extra["llama32_3b_head"] = measure_head("llama32_3b_head", max(10, a.steps), a.warmup,
                                                device)

    if a.tiered and rank == 0:
        wl70 = "llama_70b_int4o"
        for res, mode in ((40, "paged"), (60, "paged"), (0, "zero_copy"), (40, "zero_copy")):
            extra[f"{wl70}_tiered_{res}_{mode}"] = measure_tiered(
                wl70, res, max(2, a.steps // 10), 1, device, mode=mode)
        extra["link_probe_gbs"] = round(h2d_probe_gbs(device), 1)

    if a.stream_quant and rank == 0:
        extra["stream_quant_llama32_3b"] = measure_stream_quant("llama32_3b_int4o", 4, device)
        extra["stream_quant_gemma2_9b"] = measure_stream_quant("gemma2_9b_int8", 2, device)

    if a.paged and rank == 0:
        for name in ("llama_70b_int4o",) + (("gemma2_9b_int8",) if a.no_sub else ()):
            extra[f"{name}_paged"] = measure_paged(name, max(2, a.steps // 10), 1, device)

    cpu = None
    if rank == 0 and not a.no_cpu:
        gbs_cpu, t_cpu, sample, threads = cpu_baseline(a.workload)
        cpu = {"value": round(gbs_cpu, 4), "unit": "GB/s", "cores": threads, "kind": "oracle",
               "sample": sample, "seconds": round(t_cpu, 2)}
        one = cpu_baseline_one_thread(a.workload)
        if one is not None:
            cpu["single_thread"] = {"value": round(one[0], 4), "unit": "GB/s", "cores": 1,
                                    "sample": one[1]}

    if rank != 0:
        if dist_ctx is not None:
            dist_ctx.destroy_process_group()
        return 0
    peak, peak_src = peaks()
    value = job_gbs(world, r["bytes_per_step"], ms_all)
    dom = r["dominant"]
    if a.batch <= 8:
        # the library's dispatch: batch 1 on the CUDA-core GEMV, batches 2..8
        # on the warp-MMA GEMV (when the staged inputs fit)
        mv = a.batch > 1
        prof, src = ((f"mv_{a.workload}_gateup_b{a.batch}.md", "k_mv.cu") if mv
                     else (f"gemv_{a.workload}_gateup.md", "k_gemv.cu"))
        roofline = {"bound": "hbm", "achieved": round(dom["gbs"], 2), "peak": peak,
                    "unit": "GB/s", "frac": round(dom["gbs"] / peak, 4),
                    "traffic": profiled_traffic(
                        prof, "weight_only_quantized_dequant_gb300/csrc/" + src),
                    "kernel": ("gemv sequence (one layer per launch)" if a.fused
                               else f"{'mv_kernel (warp MMA)' if mv else 'gemv_kernel'} "
                                    f"({dom['group']} grouped launch)"),
                    "bytes_per_launch": dom["bytes_per_launch"],
                    "avg_launch_us": round(dom["avg_ms"] * 1e3, 3),
                    "peak_kind": peak_src}
    else:
        # tensor-core GEMM: fp16 x fp16 MMAs of N = batch rounded up to 16.
        # An N-wide MMA does N/256 of the work of the N-256 shape the dense
        # peak is quoted for; frac_of_n_scaled_peak assumes the MMA issue
        # rate does not depend on N (an assumption, not a measurement)
        tpk, tpk_src = tensor_peak()
        tflops = dom["flops_per_launch"] / (dom["avg_ms"] * 1e-3) / 1e12
        np_ = (a.batch + 15) // 16 * 16
        roofline = {"bound": "tensor", "achieved": round(tflops, 2), "peak": tpk,
                    "unit": "TFLOP/s", "frac": round(tflops / tpk, 4),
                    "traffic": profiled_traffic(
                        f"tc_{a.workload}_gateup_b{a.batch}.md",
                        "weight_only_quantized_dequant_gb300/csrc/k_tc.cu"),
                    "kernel": f"tc_gemm ({dom['group']} grouped launch)",
                    "flops_per_launch": dom["flops_per_launch"],
                    "bytes_per_launch": dom["bytes_per_launch"],
                    "weight_gbs": round(dom["gbs"], 2),
                    "avg_launch_us": round(dom["avg_ms"] * 1e3, 3),
                    "mma_n": np_, "frac_of_n_scaled_peak": round(tflops / (tpk * np_ / 256), 4),
                    "peak_kind": tpk_src}
    out = {
        "metric": METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": world,
        "steps": a.steps, "warmup": a.warmup, "ms_per_step": round(ms_all, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f32", "data": "synthetic",
        "config": {"workload": a.workload,
                   "format": "int8 per-tensor" if "int8" in a.workload else "int4 outlier-aware",
                   "batch": a.batch,
                   "layers": r["layers"], "launches_per_layer": 1 if a.fused else 4,
                   "graph": True,
                   "overlap": not a.no_overlap,
                   "l2": f"inputs larger than L2 ({r['stack_gb']:.2f} GB stack > 129 MB)",
                   "parallelism": f"replicas x{world}" if world > 1 else "single GPU"},
        "us_per_layer": round(ms_all * 1e3 / r["layers"], 3),
        "pct_of_peak": round(100.0 * value / world / peak, 2),
        # the same step counted in bytes as stored (rows padded to 16 bytes)
        "padded_gbs": round(job_gbs(world, r["padded_bytes_per_step"], ms_all), 2),
        "peak_source": f"{peak:.0f} GB/s of {peak_src}",
        "roofline": roofline,
        "cpu_baseline": cpu,
        "e2e": {"value": round(job_gbs(world, r["bytes_per_step"], e2e_all), 2),
                "unit": "GB/s", "h2d_bytes_per_step": r["h2d"], "d2h_bytes_per_step": r["d2h"],
                "ms_per_step": round(e2e_all, 4),
                # inputs up and outputs down in 6 layer ranges, overlapped with
                # the products; the copies strictly before/after the step:
                "pipelined": True, "serial_ms_per_step": round(r["e2e_serial_ms"], 4)},
        "gpu_launches": r["launches_per_step"] * a.steps,
        "copy_probe_gbs": round(copy_probe_gbs(device), 1) if a.layers is None else None,
        "clocks": r.get("clocks"),
    }
    if extra:
        out["workloads"] = extra
    print(json.dumps(out), flush=True)
    if dist_ctx is not None:
        dist_ctx.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main() or 0)
