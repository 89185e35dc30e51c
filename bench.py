#!/usr/bin/env python3
"""Bench: batch-1 VBQ decode step on the 9B-shaped stack (one JSON line on stdout).

value    whole-job effective HBM GB/s of the decode step:
         algorithmic bytes of all projections per step / device time per step.
         The device is timed with CUDA events on the launching stream over
         exactly --steps steps. A barrier and a synchronize bracket the timed
         region on both sides, and the max over ranks is taken.
extra    decode-step microseconds at the 9B and 1B shapes, the dominant kernel's
         roofline, a dense bf16 GEMV over the same shapes (distinct weights per
         layer), the 768x768 config-0 GEMV hot and cold, the batch sweep, the C++
         CPU oracle timed on one host core, and an end-to-end number through
         host buffers.

--impl reference times the C++ CPU oracle (the only reference implementation,
single-threaded) on a bounded sample of the same workload, with the same metric.

Launch: python bench.py [--gpus N --steps K --warmup W]; for N > 1 under
torchrun, each rank runs an independent replica (the path has no data-path
exchange), and value sums the ranks' bytes over the max time.
"""

from __future__ import annotations

import argparse
import json
import os
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "mixed-bit dequant-GEMV HBM GB/s (% of peak); decode-step µs at 1B/9B shapes"
GROUP_META_BYTES = 2.25  # fp16 scale + 2-bit class per group


def parse():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=20)
    p.add_argument("--warmup", type=int, default=5)
    p.add_argument("--impl", choices=["vbq", "reference"], default="vbq")
    p.add_argument("--no-1b", action="store_true", help="skip the 1B-shaped step")
    p.add_argument("--no-dense", action="store_true", help="skip the dense bf16 baseline")
    p.add_argument("--cpu-seconds", type=float, default=15.0, help="budget of the CPU-oracle sample")
    p.add_argument("--no-sweep", action="store_true", help="skip the batch sweep and the stress matrices")
    p.add_argument("--workload", choices=["9b", "1b"], default="9b",
                   help="decode-step shape of the headline (1b: a smaller case for profiling)")
    return p.parse_args()


# --------------------------------------------------------------------------- distributed

def dist_setup(args):
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if ws > 1:
        import torch.distributed as dist
        backend = "nccl" if args.impl == "vbq" else "gloo"
        if backend == "nccl":
            import torch
            torch.cuda.set_device(local)
        dist.init_process_group(backend)
    return ws, rank, local


def barrier(ws):
    if ws > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(v: float, ws: int) -> float:
    if ws == 1:
        return v
    import torch
    import torch.distributed as dist
    t = torch.tensor([v], dtype=torch.float64, device="cuda" if dist.get_backend() == "nccl" else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# --------------------------------------------------------------------------- workload

def algorithmic_bytes(n: int, k: int, code_bytes: int) -> float:
    """Codes + 2.25 B per group (fp16 scale + 2-bit class) + bf16 x + fp32 y."""
    groups = n * (k // 64)
    return code_bytes + GROUP_META_BYTES * groups + 2.0 * k + 4.0 * n


class PackedModel:
    def __init__(self, V, shape, seed=0):
        from synth import gen_model_matrix, model_matrix_list
        self.shape = shape
        self.handles = []
        self.alg_bytes = 0.0
        self.code_bytes = 0
        self.total_bytes = 0
        self.weights = 0
        self.per_matrix = []  # (layer, proj, N, K, algorithmic bytes, handle)
        for (layer, proj) in model_matrix_list(shape):
            m = gen_model_matrix(shape, layer, proj, seed=seed)
            h = V.Matrix(m.codes, m.bits, m.scales)
            info = h.info()
            ab = algorithmic_bytes(m.N, m.K, info["code_bytes"])
            self.alg_bytes += ab
            self.code_bytes += info["code_bytes"]
            self.total_bytes += info["total_bytes"]
            self.weights += m.N * m.K
            self.per_matrix.append((layer, proj, m.N, m.K, ab, h))
            self.handles.append(h)
            del m
        desc = V.make_model_desc(shape.n_layers, shape.d, shape.n_heads, shape.n_kv_heads, shape.head_dim,
                                 shape.d_ff, shape.vocab, 1e-5)
        self.model = V.Model(desc, self.handles)

    def close(self):
        self.model.close()
        for h in self.handles:
            h.close()


# --------------------------------------------------------------------------- clocks

class ClockSampler:
    """SM clock and clock-event reasons over the timed region.

    NVML (pynvml) is sampled every 2 ms from a thread when it is importable.
    Otherwise nvidia-smi runs with a 20 ms period from before the warm-up
    (prepare()), and only the samples that arrive inside the timed region, plus
    the first one after it, are kept."""
    REASONS = {"hw_slowdown": 0x8, "sw_thermal_slowdown": 0x20, "hw_thermal_slowdown": 0x40, "sw_power_cap": 0x4}
    SMI_FIELDS = ("clocks.sm,clocks.max.sm,clocks_event_reasons.hw_slowdown,"
                  "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
                  "clocks_event_reasons.sw_power_cap")

    def __init__(self, cuda_index: int):
        self.cuda_index = cuda_index
        self.samples = []      # (host time, sm MHz, set of reasons)
        self.max_mhz = None
        self.err = None
        self.mode = None
        self.t0 = self.t1 = None
        self._stop = threading.Event()
        self.thread = None
        self.proc = None

    # -- NVML
    def _nvml(self):
        import pynvml as N
        import torch
        N.nvmlInit()
        try:
            p = torch.cuda.get_device_properties(self.cuda_index)
            h = N.nvmlDeviceGetHandleByPciBusId(f"{p.pci_domain_id:08x}:{p.pci_bus_id:02x}:{p.pci_device_id:02x}.0")
        except Exception:
            h = N.nvmlDeviceGetHandleByIndex(self.cuda_index)
        self.max_mhz = float(N.nvmlDeviceGetMaxClockInfo(h, N.NVML_CLOCK_SM))
        get_r = getattr(N, "nvmlDeviceGetCurrentClocksEventReasons", None) or N.nvmlDeviceGetCurrentClocksThrottleReasons

        def sample():
            sm = float(N.nvmlDeviceGetClockInfo(h, N.NVML_CLOCK_SM))
            r = int(get_r(h))
            self.samples.append((time.perf_counter(), sm, {n for n, b in self.REASONS.items() if r & b}))

        def run():
            while not self._stop.is_set():
                try:
                    sample()
                except Exception as e:
                    self.err = str(e)
                    return
                self._stop.wait(0.002)
        self.thread = threading.Thread(target=run, daemon=True)
        self.thread.start()

    # -- nvidia-smi
    def _smi(self):
        import subprocess
        import torch
        try:
            p = torch.cuda.get_device_properties(self.cuda_index)
            dev = f"--id={p.pci_domain_id:08x}:{p.pci_bus_id:02x}:{p.pci_device_id:02x}.0"
        except Exception:
            dev = f"--id={self.cuda_index}"
        self.proc = subprocess.Popen(["nvidia-smi", dev, f"--query-gpu={self.SMI_FIELDS}",
                                      "--format=csv,noheader,nounits", "-lms", "20"],
                                     stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]

        def run():
            for line in self.proc.stdout:
                parts = [q.strip() for q in line.split(",")]
                if len(parts) < 6:
                    continue
                try:
                    sm, mx = float(parts[0]), float(parts[1])
                except ValueError:
                    continue
                self.max_mhz = mx
                self.samples.append((time.perf_counter(), sm,
                                     {n for n, v in zip(names, parts[2:6]) if v.lower().startswith("active")}))
        self.thread = threading.Thread(target=run, daemon=True)
        self.thread.start()

    def prepare(self):
        """Starts sampling (call before the warm-up)."""
        try:
            self._nvml()
            self.mode = "nvml, every 2 ms"
        except Exception as e:
            self.err = f"nvml: {e}"
            try:
                self._smi()
                self.mode = "nvidia-smi, every 20 ms"
                deadline = time.perf_counter() + 10.0
                while not self.samples and time.perf_counter() < deadline:
                    time.sleep(0.01)
            except OSError as e2:
                self.err += f"; nvidia-smi: {e2}"

    def start(self):
        self.t0 = time.perf_counter()

    def stop(self) -> dict:
        self.t1 = time.perf_counter()
        if self.mode is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "error": self.err}
        if self.mode.startswith("nvidia-smi"):
            deadline = time.perf_counter() + 1.0
            while not any(t > self.t1 for t, _, _ in self.samples) and time.perf_counter() < deadline:
                time.sleep(0.005)
        self._stop.set()
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
        if self.thread is not None:
            self.thread.join(timeout=2)
        inside = [q for q in self.samples if self.t0 <= q[0] <= self.t1]
        after = [q for q in self.samples if q[0] > self.t1][:1]
        use = inside + after
        sm = [q[1] for q in use]
        reasons = sorted(set().union(*[q[2] for q in use])) if use else []
        return {"sm_mhz": float(np.median(sm)) if sm else None, "sm_max_mhz": self.max_mhz, "reasons": reasons,
                "samples": len(sm), "source": self.mode}


# --------------------------------------------------------------------------- GPU timings

def time_steps(fn, steps, warmup, stream, ws):
    import torch
    for _ in range(warmup):
        fn()
    torch.cuda.synchronize()
    barrier(ws)
    torch.cuda.synchronize()
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    start.record(stream)
    for _ in range(steps):
        fn()
    end.record(stream)
    torch.cuda.synchronize()
    barrier(ws)
    ms = start.elapsed_time(end) / steps
    return ms


# DRAM traffic (dram__bytes_read.sum + dram__bytes_write.sum) of one decode-kernel
# launch on the 9B-shaped step, from an ncu capture of the build whose kernel
# sources hash to the key; any other build reports null.
DECODE_TRAFFIC = {
    "0b70fcb5670b620b": 2098673920,  # 2,092,879,104 B read + 5,794,816 B written in one launch
    "53b0ad5d05c397fc": 2098785536,  # 2,093,091,840 B read + 5,693,696 B written in one launch
}
KERNEL_SOURCES = ("decode.cuh", "gemv.cuh", "ptx.cuh", "layout.h", "model.cu", "plan.cpp", "plan.h", "pack.cpp")


def kernel_source_hash() -> str:
    import hashlib
    h = hashlib.sha256()
    for f in KERNEL_SOURCES:
        with open(os.path.join(ROOT, "mixed_precision_weight_bit_b300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def decode_kernel_roofline(V, pm, x, logits, stream, peak_gbs, ms_step, steps, workload):
    """Roofline of vbq_decode_kernel, the only kernel of a step: algorithmic bytes per launch over the average
    launch time of the timed region (one launch per step). A second pass brackets each launch with events on
    its stream, as a check of the spread."""
    import torch
    ev = []
    with torch.cuda.stream(stream):
        for _ in range(steps):
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            V.vbq_decode_step(pm.model.handle, x, logits, stream)
            b.record(stream)
            ev.append((a, b))
    torch.cuda.synchronize()
    ms = [a.elapsed_time(b) for a, b in ev]
    achieved = pm.alg_bytes / (ms_step * 1e-3) / 1e9
    key = kernel_source_hash()
    traffic = DECODE_TRAFFIC.get(key) if workload == "9b" else None
    return {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak_gbs, "unit": "GB/s",
            "frac": round(achieved / peak_gbs, 4), "traffic": traffic,
            "kernel": "vbq_decode_kernel", "launches_timed": steps,
            "avg_launch_us": round(ms_step * 1e3, 2),
            "bracketed_launch_us": {"min": round(min(ms) * 1e3, 2), "avg": round(sum(ms) / len(ms) * 1e3, 2)},
            "alg_bytes_per_launch": round(pm.alg_bytes), "kernel_source_hash": key,
            "note": "one launch per decode step; algorithmic bytes = sum over the projections of "
                    "codes + 2.25 B/group + 2K + 4N; traffic = DRAM bytes of one launch from ncu (null "
                    "unless captured on this build)"}


def context_step(V, pm, shape, x, logits, stream, peak_gbs, ctx, steps=10):
    """The decode step at position ctx - 1 (vbq_decode_step_at): every layer's rotary append and
    attention over ctx cached positions (seeded bf16 keys and values) between the projections."""
    import torch
    from cuda.bindings import runtime as rt
    V.vbq_model_set_context(pm.model.handle, ctx)
    g = torch.Generator(device="cuda")
    g.manual_seed(0)
    for layer in range(shape.n_layers):
        kp, vp, stride = V.vbq_model_kv_cache(pm.model.handle, layer)
        for ptr in (kp, vp):
            t = torch.randn(shape.n_kv_heads, stride, shape.head_dim, device="cuda", generator=g).to(torch.bfloat16)
            (err,) = rt.cudaMemcpy(ptr, t.data_ptr(), t.numel() * 2, rt.cudaMemcpyKind.cudaMemcpyDeviceToDevice)
            assert int(err) == 0
    torch.cuda.synchronize()

    def step():
        V.vbq_decode_step_at(pm.model.handle, x, ctx - 1, logits, stream)

    with torch.cuda.stream(stream):
        ms = time_steps(step, steps, 3, stream, 1)
    assert V.vbq_device_check() == 0
    kv_bytes = 2.0 * shape.n_layers * shape.n_kv_heads * ctx * shape.head_dim * 2
    V.vbq_model_set_context(pm.model.handle, 0)
    return {"us": round(ms * 1e3, 1), "context": ctx, "kv_bytes": kv_bytes,
            "GB/s": round((pm.alg_bytes + kv_bytes) / (ms * 1e-3) / 1e9, 1),
            "frac": round((pm.alg_bytes + kv_bytes) / (ms * 1e-3) / 1e9 / peak_gbs, 4),
            "launches_per_step": 3 * shape.n_layers + 1,
            "note": "vbq_decode_step_at at position ctx - 1: n_layers + 1 decode-kernel launches with each "
                    "layer's rotary append and attention between them; bytes = the step's algorithmic bytes + "
                    "the K and V caches read"}


def standalone_gemv(V, pm, stream, peak_gbs, reps=3):
    """Each projection as its own vbq_gemv launch, bracketed by events on the launching stream."""
    import torch
    from synth import gen_x
    xs = {}
    ys = {}
    for (_, proj, n, k, ab, h) in pm.per_matrix:
        if k not in xs:
            xs[k] = torch.from_numpy(gen_x(k, seed=9).view(np.int16)).cuda()
        if n not in ys:
            ys[n] = torch.empty(n, dtype=torch.float32, device="cuda")
    ev = []
    with torch.cuda.stream(stream):
        for (_, _, n, k, ab, h) in pm.per_matrix:  # warm
            V.vbq_gemv(h.handle, xs[k], ys[n], stream)
        for _ in range(reps):
            for (_, _, n, k, ab, h) in pm.per_matrix:
                a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                a.record(stream)
                V.vbq_gemv(h.handle, xs[k], ys[n], stream)
                b.record(stream)
                ev.append((a, b, ab))
    torch.cuda.synchronize()
    tot_ms = sum(a.elapsed_time(b) for a, b, _ in ev)
    tot_b = sum(ab for _, _, ab in ev)
    launches = len(ev)
    achieved = tot_b / (tot_ms * 1e-3) / 1e9
    return {"achieved": round(achieved, 1), "unit": "GB/s", "frac": round(achieved / peak_gbs, 4),
            "kernel": "vbq_gemv1_kernel", "launches": launches,
            "avg_launch_us": round(tot_ms * 1e3 / launches, 2),
            "alg_bytes_per_launch": round(tot_b / launches),
            "note": "each projection of the step's stack launched alone through vbq_gemv"}


def dense_baseline(V, shape, stream, steps=3):
    """Dense bf16 GEMV (same codebase) over every projection of the stack, with distinct weights per layer
    (n_layers x 7 matrices + the head, as the VBQ step streams them), on the launching stream."""
    import torch
    from synth import PROJS, model_matrix_shape
    g = torch.Generator(device="cuda")
    g.manual_seed(0)
    mats = []
    for _ in range(shape.n_layers):
        for p in PROJS:
            n, k = model_matrix_shape(shape, p)
            mats.append((torch.randn(n, k, device="cuda", dtype=torch.bfloat16, generator=g) * 0.02, n, k))
    n, k = model_matrix_shape(shape, "head")
    mats.append((torch.randn(n, k, device="cuda", dtype=torch.bfloat16, generator=g) * 0.02, n, k))
    xs = {k: torch.randn(k, device="cuda", dtype=torch.bfloat16, generator=g) for (_, _, k) in mats}
    ys = {n: torch.empty(n, device="cuda") for (_, n, _) in mats}

    jobs = [(W, xs[k], ys[n], n, k) for (W, n, k) in mats]

    def step_many():
        V.vbq_dense_gemv_bf16_many(jobs, stream)

    def step_each():
        for (W, n, k) in mats:
            V.vbq_dense_gemv_bf16(W, xs[k], ys[n], n, k, stream)

    with torch.cuda.stream(stream):
        ms = time_steps(step_many, steps, 1, stream, 1)
        ms_each = time_steps(step_each, steps, 1, stream, 1)
    nbytes = sum(2.0 * n * k + 2.0 * k + 4.0 * n for (_, n, k) in mats)
    del mats, jobs
    torch.cuda.empty_cache()
    return {"us_per_step": round(ms * 1e3, 1), "GB/s": round(nbytes / (ms * 1e-3) / 1e9, 1),
            "weight_bytes": nbytes, "launches_per_step": 1,
            "one_launch_per_matrix": {"us_per_step": round(ms_each * 1e3, 1),
                                      "GB/s": round(nbytes / (ms_each * 1e-3) / 1e9, 1),
                                      "launches_per_step": shape.n_layers * len(PROJS) + 1},
            "note": "bf16 W and x, fp32 accumulate; bytes = 2NK + 2K + 4N per matrix; "
                    "every matrix of the step in one launch (vbq_dense_gemv_bf16_many)"}


def config0_gemv(V, stream, peak_gbs):
    """The 768x768 config-0 linear, batch 1: one vbq_gemv launch, hot (repeated, L2-resident) and cold
    (512 MiB written between launches)."""
    import torch
    from synth import CONFIG0_PROBS, gen_matrix, gen_x
    m = gen_matrix(768, 768, CONFIG0_PROBS, seed=0)
    mat = V.Matrix(m.codes, m.bits, m.scales)
    info = mat.info()
    x = torch.from_numpy(gen_x(768, seed=0).view(np.int16)).cuda()
    y = torch.empty(768, device="cuda")
    cold = time_cold(lambda: V.vbq_gemv(mat.handle, x, y, stream), stream)
    with torch.cuda.stream(stream):
        for _ in range(5):
            V.vbq_gemv(mat.handle, x, y, stream)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for _ in range(100):
            V.vbq_gemv(mat.handle, x, y, stream)
        b.record(stream)
    torch.cuda.synchronize()
    hot = a.elapsed_time(b) / 100 * 1e3
    alg = algorithmic_bytes(768, 768, info["code_bytes"])
    mat.close()
    return {"cold_us": round(cold, 2), "hot_us": round(hot, 2), "alg_bytes": round(alg),
            "GB/s_cold": round(alg / cold / 1e3, 1), "frac_cold": round(alg / cold / 1e3 / peak_gbs, 5),
            "note": "one launch per call; at 211 KB the call is bound by launch and synchronization latency"}


def time_cold(fn, stream, reps=10):
    """Median device time of fn() over reps runs, with a 512 MiB write between runs to evict L2."""
    import torch
    flush = torch.empty(512 << 20, dtype=torch.uint8, device="cuda")
    for _ in range(2):
        fn()
    ts = []
    for _ in range(reps):
        with torch.cuda.stream(stream):   # the flush is ordered before the timed call on the same stream
            flush.zero_()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        fn()
        b.record(stream)
        torch.cuda.synchronize()
        ts.append(a.elapsed_time(b))
    del flush
    return float(np.median(ts)) * 1e3


def batch_sweep(V, stream):
    """14336x4096 at the config-0 allocation, batch 1..64 and 128, 256, cold L2 (CUDA cores up to 3 columns,
    tensor cores from 4)."""
    import torch
    from synth import CONFIG0_PROBS, gen_matrix, gen_x
    m = gen_matrix(14336, 4096, CONFIG0_PROBS, seed=0)
    mat = V.Matrix(m.codes, m.bits, m.scales)
    info = mat.info()
    out = {}
    for B in (1, 2, 4, 8, 16, 32, 64):
        X = torch.from_numpy(gen_x(4096, seed=100 + B, batch=B).view(np.int16)).cuda()
        Y = torch.empty(B, 14336, device="cuda")
        us = time_cold(lambda: V.vbq_gemm_smallbatch(mat.handle, X, B, Y, stream), stream)
        alg = algorithmic_bytes(14336, 4096, info["code_bytes"]) + 2.0 * 4096 * (B - 1) + 4.0 * 14336 * (B - 1)
        out[str(B)] = {"us": round(us, 1), "GB/s": round(alg / us / 1e3, 1),
                       "TFLOP/s": round(2.0 * 14336 * 4096 * B / us / 1e6, 2)}
    for B in (128, 256):  # prefill-sized batches through vbq_gemm (blocks of 64 columns)
        X = torch.from_numpy(gen_x(4096, seed=100 + B, batch=B).view(np.int16)).cuda()
        Y = torch.empty(B, 14336, device="cuda")
        us = time_cold(lambda: V.vbq_gemm(mat.handle, X, B, Y, stream), stream)
        out[str(B)] = {"us": round(us, 1), "TFLOP/s": round(2.0 * 14336 * 4096 * B / us / 1e6, 2),
                       "note": "vbq_gemm: one tensor-core call per 64 columns"}
    mat.close()
    return out


def attention_decode_sweep(V, stream, peak_gbs):
    """Decode attention of one token over a bf16 KV cache at the 9B shape (32 query heads, 8 kv heads,
    head_dim 128), cold L2: the cache bytes read per call over the call's time."""
    import torch
    H, Hkv, d = 32, 8, 128
    g = torch.Generator(device="cuda")
    g.manual_seed(0)
    out = {}
    for T in (1024, 4096, 16384, 65536):
        q = (torch.randn(H, d, device="cuda", generator=g) * 0.5).to(torch.bfloat16)
        kc = (torch.randn(Hkv, T, d, device="cuda", generator=g) * 0.5).to(torch.bfloat16)
        vc = torch.randn(Hkv, T, d, device="cuda", generator=g).to(torch.bfloat16)
        o = torch.empty(H, d, device="cuda")
        us = time_cold(lambda: V.vbq_attention_decode(q, kc, vc, H, Hkv, d, T, T, o, stream), stream)
        nbytes = 2.0 * Hkv * T * d * 2 + H * d * 2 + H * d * 4
        out[str(T)] = {"us": round(us, 2), "GB/s": round(nbytes / us / 1e3, 1),
                       "frac": round(nbytes / us / 1e3 / peak_gbs, 4)}
        del kc, vc
    kn = torch.zeros(Hkv, d, device="cuda", dtype=torch.bfloat16)
    kc = torch.zeros(Hkv, 4096, d, device="cuda", dtype=torch.bfloat16)
    vc = torch.zeros_like(kc)
    q = torch.zeros(H, d, device="cuda", dtype=torch.bfloat16)
    us = time_cold(lambda: V.vbq_rope_append(q, kn, kn, kc, vc, H, Hkv, d, 4096, 1000, 10000.0, stream), stream)
    out["rope_append_us"] = round(us, 2)
    out["note"] = ("vbq_attention_decode, 32 q heads over 8 kv heads, head_dim 128, T positions, up to 64 spans per kv head; "
                   "bytes = K and V of the T positions + q + out")
    return out


def dense_chain(W, shape, x_bits, eps=1e-5):
    """Logits of the dense model over the same glue as the decode step (unit-gain RMSNorm, attention at
    position 0, SwiGLU, bf16 at every projection input), in fp64 torch on the host: the dense side of the
    divergence measurement."""
    import torch
    def bf16(t):
        return t.to(torch.bfloat16).to(torch.float64)
    def rms(h):
        return h / torch.sqrt((h * h).mean() + eps)
    def mm(layer, proj, u):
        return torch.from_numpy(W[(layer, proj)]).to(torch.float64) @ u
    h = torch.from_numpy(x_bits.view(np.int16)).view(torch.bfloat16).to(torch.float64)
    group = shape.n_heads // shape.n_kv_heads
    for layer in range(shape.n_layers):
        u = bf16(rms(h))
        v = mm(layer, "v", u).view(shape.n_kv_heads, shape.head_dim)
        a = bf16(torch.cat([v[i // group] for i in range(shape.n_heads)]))
        h = h + mm(layer, "o", a)
        u = bf16(rms(h))
        g, up = mm(layer, "gate", u), mm(layer, "up", u)
        h = h + mm(layer, "down", bf16(g / (1.0 + torch.exp(-g)) * up))
    return mm(shape.n_layers, "head", bf16(rms(h))).numpy()


def divergence_tiny(V, n_inputs=16):
    """KL divergence and argmax flips between a dense synthetic model (the tiny shape, Gaussian weights
    of variance 1/K) and its VBQ encodings (vbq_quantize_rtn) at three allocations, over seeded inputs."""
    import torch
    from synth import CONFIG0_PROBS, gen_x, model_matrix_list, model_matrix_shape, model_tiny
    shape = model_tiny()
    rng = np.random.default_rng(11)
    W = {}
    for (layer, proj) in model_matrix_list(shape):
        n, k = model_matrix_shape(shape, proj)
        W[(layer, proj)] = (rng.standard_normal((n, k)) / np.sqrt(k)).astype(np.float32)
    xs = [gen_x(shape.d, seed=100 + i) for i in range(n_inputs)]
    ref = np.array([dense_chain(W, shape, x) for x in xs])

    def log_softmax(z):
        m = z.max(axis=-1, keepdims=True)
        return z - m - np.log(np.exp(z - m).sum(axis=-1, keepdims=True))
    out = {}
    for name, probs in [("all_8bit", {8: 1.0}), ("config0_mix", CONFIG0_PROBS), ("all_1bit", {1: 1.0})]:
        brng = np.random.default_rng(12)
        handles = []
        bits_total = 0
        n_groups = 0
        for (layer, proj) in model_matrix_list(shape):
            w = W[(layer, proj)]
            bits = brng.choice(list(probs.keys()), size=(w.shape[0], w.shape[1] // 64),
                               p=list(probs.values())).astype(np.uint8)
            bits_total += int(bits.astype(np.int64).sum())
            n_groups += bits.size
            codes, scales = V.vbq_quantize_rtn(w, bits)
            handles.append(V.Matrix(codes, bits, scales))
        desc = V.make_model_desc(shape.n_layers, shape.d, shape.n_heads, shape.n_kv_heads, shape.head_dim,
                                 shape.d_ff, shape.vocab, 1e-5)
        model = V.Model(desc, handles)
        got = []
        for x in xs:
            lg = torch.empty(shape.vocab, device="cuda")
            V.vbq_decode_step(model.handle, torch.from_numpy(x.view(np.int16)).cuda(), lg)
            torch.cuda.synchronize()
            got.append(lg.cpu().numpy().astype(np.float64))
        model.close()
        for h in handles:
            h.close()
        lp, lq = log_softmax(ref), log_softmax(np.array(got))
        kl = (np.exp(lp) * (lp - lq)).sum(axis=-1)
        flips = np.argmax(ref, axis=-1) != np.argmax(np.array(got), axis=-1)
        out[name] = {"mean_bits": round(bits_total / n_groups, 3), "kl_mean": float(kl.mean()),
                     "kl_max": float(kl.max()), "argmax_flip_rate": float(flips.mean())}
    out["note"] = (f"tiny shape, {n_inputs} seeded inputs; the dense model's fp64 chain (same glue) vs the VBQ "
                   "decode step on its round-to-nearest encodings; KL(dense || VBQ) of the next-token distributions")
    return out


def fakequant_bench(V, stream, peak_gbs, n=8192, k=8192):
    """The training-side fake quantization on an fp32 [n][k] weight (Gumbel-Softmax mixture over
    {1,2,4,8} bits per group, straight-through backward), cold L2: bytes streamed over the call's time."""
    import torch
    g = torch.Generator(device="cuda")
    g.manual_seed(0)
    W = torch.randn(n, k, device="cuda", generator=g) * 0.1
    alpha = torch.randn(n, k // 64, 4, device="cuda", generator=g)
    u = torch.rand(n, k // 64, 4, device="cuda", generator=g) * 0.98 + 0.01
    G = torch.randn(n, k, device="cuda", generator=g)
    out, dW, da = torch.empty_like(W), torch.empty_like(W), torch.empty_like(alpha)
    fwd = time_cold(lambda: V.vbq_fakequant_forward(W, alpha, u, 0.7, n, k, out, stream), stream)
    bwd = time_cold(lambda: V.vbq_fakequant_backward(W, alpha, u, 0.7, G, n, k, dW, da, stream), stream)
    groups = n * (k // 64)
    fb = 8.0 * n * k + 32.0 * groups          # W in, W_mix out; alpha and u
    bb = 12.0 * n * k + 48.0 * groups         # W and G in, dW out; alpha, u in, dalpha out
    return {"shape": [n, k], "forward_us": round(fwd, 1), "forward_GB/s": round(fb / fwd / 1e3, 1),
            "forward_frac": round(fb / fwd / 1e3 / peak_gbs, 4), "backward_us": round(bwd, 1),
            "backward_GB/s": round(bb / bwd / 1e3, 1), "backward_frac": round(bb / bwd / 1e3 / peak_gbs, 4)}


def stress_8192(V, stream):
    """The 8192x8192 allocation-stress matrices (a)-(e), batch 1, cold L2."""
    import torch
    from synth import gen_stress, gen_x
    x = torch.from_numpy(gen_x(8192, seed=21).view(np.int16)).cuda()
    y = torch.empty(8192, device="cuda")
    out = {}
    for case in "abcde":
        m = gen_stress(case, 8192, 8192)
        mat = V.Matrix(m.codes, m.bits, m.scales)
        info = mat.info()
        us = time_cold(lambda: V.vbq_gemv(mat.handle, x, y, stream), stream)
        alg = algorithmic_bytes(8192, 8192, info["code_bytes"])
        out[case] = {"us": round(us, 1), "GB/s": round(alg / us / 1e3, 1), "mean_bits": round(info["mean_bits"], 3)}
        mat.close()
    return out


# --------------------------------------------------------------------------- CPU oracle

def host_cpu():
    """Logical CPUs of the host (nproc) and the CPU model (lscpu, else /proc/cpuinfo)."""
    cores = os.cpu_count()
    model = None
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.strip().startswith("Model name:"):
                model = line.split(":", 1)[1].strip()
                break
    except Exception:
        pass
    if not model:
        try:
            with open("/proc/cpuinfo") as f:
                for line in f:
                    if line.startswith("model name"):
                        model = line.split(":", 1)[1].strip()
                        break
        except Exception:
            pass
    return cores, model


def step_weights(shape) -> int:
    from synth import model_matrix_list, model_matrix_shape
    return sum(int(np.prod(model_matrix_shape(shape, p))) for (_, p) in model_matrix_list(shape))


def cpu_oracle_sample(shape, budget_s: float):
    """The C++ oracle's GEMV (one core: fp32 dequant, fp64 sums) over the stack's projections in step
    order, until the time budget is spent. The per-weight rate of the sample gives the seconds of a
    whole decode step."""
    from oracle import vbq_oracle_cpp as C
    from synth import gen_model_matrix, gen_x, model_matrix_list
    C.build()
    done_bytes, spent, n_mats, weights = 0.0, 0.0, 0, 0
    for (layer, proj) in model_matrix_list(shape):
        m = gen_model_matrix(shape, layer, proj, seed=0)
        x = gen_x(m.K, seed=9)
        code_bytes = int((8 * m.bits.astype(np.int64)).sum())
        t0 = time.perf_counter()
        C.gemv(m.codes, m.bits, m.scales, x)
        spent += time.perf_counter() - t0
        done_bytes += algorithmic_bytes(m.N, m.K, code_bytes)
        weights += m.N * m.K
        n_mats += 1
        if spent >= budget_s:
            break
    per_step = step_weights(shape) * spent / weights
    return {"value": round(done_bytes / spent / 1e9, 4), "unit": "GB/s", "seconds": round(spent, 2),
            "seconds_per_step": round(per_step, 2), "weights": weights, "n_mats": n_mats,
            "sample": f"C++ oracle gemv over the first {n_mats} projections of the {shape.name} stack "
                      f"({weights / 1e6:.0f}M weights, {done_bytes / 1e6:.0f} MB algorithmic, {spent:.1f} s)"}


def cpu_baseline(shape, budget_s: float):
    """The cpu_baseline object: the oracle on one core, with the host described and the seconds of one
    decode step at both model shapes (from each shape's sample rate)."""
    from synth import model_1b, model_9b
    cores_total, cpu_model = host_cpu()
    main = cpu_oracle_sample(shape, budget_s)
    other = model_1b() if shape.name == "vbq-9b" else model_9b()
    side = cpu_oracle_sample(other, budget_s / 3.0)
    per = {shape.name: main, other.name: side}
    return {"value": main["value"], "unit": "GB/s", "cores": 1, "cores_total": cores_total,
            "cpu_model": cpu_model, "kind": "oracle",
            "threads": "1 core used: the C++ oracle is single-threaded (no BLAS)",
            "sample": main["sample"],
            "seconds_per_step_9b": per["vbq-9b"]["seconds_per_step"],
            "seconds_per_step_1b": per["vbq-1b"]["seconds_per_step"],
            "seconds_per_step_note": "sample seconds x (weights of one step / weights sampled)"}


# --------------------------------------------------------------------------- main arms

def peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), "measured"
    except Exception:
        return 6400.0, "fallback"


def workload_text(shape):
    size = {"vbq-9b": "9B", "vbq-1b": "1B"}.get(shape.name, shape.name)
    att = (f"GQA {shape.n_heads}/{shape.n_kv_heads}x{shape.head_dim}" if shape.n_kv_heads != shape.n_heads
           else f"MHA {shape.n_heads}x{shape.head_dim}")
    return (f"{size}-shaped decode step, batch 1 ({shape.n_layers} layers, d={shape.d}, {att}, SwiGLU "
            f"{shape.d_ff}, vocab {shape.vocab}), per-group {{1,2,4,8}}-bit weights, seed 0")


def run_reference(args, ws, rank):
    """The C++ oracle arm: the first projections of the stack (about one second of oracle work) are drawn
    once; each step times the oracle's GEMV over all of them."""
    if rank != 0:
        return
    from oracle import vbq_oracle_cpp as C
    from synth import gen_model_matrix, gen_x, model_1b, model_9b, model_matrix_list
    shape = model_9b() if args.workload == "9b" else model_1b()
    cores_total, cpu_model = host_cpu()
    C.build()
    per_step_s = max(0.5, min(2.0, args.cpu_seconds / max(1, args.steps + args.warmup)))
    target = per_step_s / 3e-9  # weights, at about 3 ns per weight on one core
    mats, weights = [], 0
    for (layer, proj) in model_matrix_list(shape):
        m = gen_model_matrix(shape, layer, proj, seed=0)
        mats.append((m, gen_x(m.K, seed=9), algorithmic_bytes(m.N, m.K, int((8 * m.bits.astype(np.int64)).sum()))))
        weights += m.N * m.K
        if weights >= target:
            break

    def step():
        t0 = time.perf_counter()
        for m, x, _ in mats:
            C.gemv(m.codes, m.bits, m.scales, x)
        return time.perf_counter() - t0

    for _ in range(args.warmup):
        step()
    secs = [step() for _ in range(args.steps)]
    t = float(np.median(secs))
    v = sum(ab for _, _, ab in mats) / t / 1e9
    per_step = step_weights(shape) * t / weights
    sample = (f"C++ oracle gemv over the first {len(mats)} projections of the {shape.name} stack "
              f"({weights / 1e6:.0f}M weights), median of {args.steps} timed passes")
    line = {"metric": METRIC, "value": round(v, 4), "unit": "GB/s", "n_gpus": args.gpus, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": round(per_step * 1e3, 1),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "impl": "reference", "config": {"workload": workload_text(shape)},
            "cpu_baseline": {"value": round(v, 4), "unit": "GB/s", "cores": 1, "cores_total": cores_total,
                             "cpu_model": cpu_model, "kind": "oracle", "sample": sample,
                             "seconds_per_step": round(per_step, 2)},
            "e2e": {"value": round(v, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def run_vbq(args, ws, rank, local):
    import torch
    import mixed_precision_weight_bit_b300 as V
    from synth import gen_x, model_1b, model_9b

    torch.cuda.set_device(local)
    stream = torch.cuda.Stream()
    peak, peak_kind = peaks()

    shape = model_9b() if args.workload == "9b" else model_1b()
    t0 = time.perf_counter()
    pm = PackedModel(V, shape, seed=0)
    pack_s = time.perf_counter() - t0
    x = torch.from_numpy(gen_x(shape.d, seed=7).view(np.int16)).cuda()
    logits = torch.empty(shape.vocab, dtype=torch.float32, device="cuda")

    def step():
        V.vbq_decode_step(pm.model.handle, x, logits, stream)

    clocks = ClockSampler(local)
    clocks.prepare()
    with torch.cuda.stream(stream):
        for _ in range(max(args.warmup, 3)):
            step()
        torch.cuda.synchronize()
        clocks.start()
        launches0 = V.vbq_launch_count()
        ms = time_steps(step, args.steps, 0, stream, ws)
        launches = V.vbq_launch_count() - launches0
        clk = clocks.stop()
    assert V.vbq_device_check() == 0
    ms_max = max_over_ranks(ms, ws)
    value = ws * pm.alg_bytes / (ms_max * 1e-3) / 1e9

    # end to end through host buffers (pinned): H2D of x, D2H of logits, every step
    xh = torch.from_numpy(gen_x(shape.d, seed=7).view(np.int16)).pin_memory()
    lh = torch.empty(shape.vocab, dtype=torch.float32).pin_memory()
    for _ in range(3):
        V.vbq_decode_step_host(pm.model.handle, xh, lh, stream)
    barrier(ws)
    t1 = time.perf_counter()
    for _ in range(args.steps):
        V.vbq_decode_step_host(pm.model.handle, xh, lh, stream)
    e2e_s = (time.perf_counter() - t1) / args.steps
    e2e_s = max_over_ranks(e2e_s, ws)

    roof = decode_kernel_roofline(V, pm, x, logits, stream, peak, ms, args.steps, args.workload)
    roof["peak_kind"] = peak_kind
    standalone = standalone_gemv(V, pm, stream, peak)
    w = "_" + args.workload
    alg_step = pm.alg_bytes
    extra = {"decode_step_us" + w: round(ms * 1e3, 1), "pack_seconds" + w: round(pack_s, 1),
             "weights" + w: pm.weights, "alg_bytes_per_step" + w: round(pm.alg_bytes),
             "device_bytes" + w: pm.total_bytes, "code_bytes" + w: pm.code_bytes,
             "standalone_gemv" + w: standalone,
             "decode_step_ctx4096" + w: context_step(V, pm, shape, x, logits, stream, peak, 4096)}
    pm.close()
    torch.cuda.empty_cache()

    if not args.no_1b and args.workload == "9b":
        s1 = model_1b()
        pm1 = PackedModel(V, s1, seed=0)
        x1 = torch.from_numpy(gen_x(s1.d, seed=7).view(np.int16)).cuda()
        l1 = torch.empty(s1.vocab, dtype=torch.float32, device="cuda")
        with torch.cuda.stream(stream):
            ms1 = time_steps(lambda: V.vbq_decode_step(pm1.model.handle, x1, l1, stream), args.steps,
                             max(args.warmup, 3), stream, 1)
        extra["decode_step_us_1b"] = round(ms1 * 1e3, 1)
        extra["alg_bytes_per_step_1b"] = round(pm1.alg_bytes)
        extra["GB/s_1b"] = round(pm1.alg_bytes / (ms1 * 1e-3) / 1e9, 1)
        pm1.close()
        torch.cuda.empty_cache()
    extra["config0_768x768"] = config0_gemv(V, stream, peak)
    if not args.no_sweep:
        extra["batch_sweep_14336x4096"] = batch_sweep(V, stream)
        extra["stress_8192"] = stress_8192(V, stream)
        extra["attention_decode_9b_heads"] = attention_decode_sweep(V, stream, peak)
        extra["divergence_tiny"] = divergence_tiny(V)
        extra["fakequant_8192x8192"] = fakequant_bench(V, stream, peak)
    if not args.no_dense:
        extra["dense_bf16" + w] = dense_baseline(V, shape, stream)
        extra["dense_bf16" + w]["speedup_vbq"] = round(extra["dense_bf16" + w]["us_per_step"] / (ms * 1e3), 2)

    cpu = None
    if rank == 0:
        cpu = cpu_baseline(shape, args.cpu_seconds)

    if rank == 0:
        line = {"metric": METRIC, "value": round(value, 1), "unit": "GB/s", "n_gpus": ws, "steps": args.steps,
                "warmup": max(args.warmup, 3), "ms_per_step": round(ms_max, 4), "higher_is_better": True,
                "scaling": "weak", "vs_baseline": None,
                "dtype": "f32 accumulate (bf16 x, packed 1/2/4/8-bit codes, fp16 scales)", "data": "synthetic",
                "config": {"workload": workload_text(shape),
                           "l2": f"inputs larger than L2: {pm.total_bytes / 1e9:.2f} GB of packed weights "
                                 "streamed per step",
                           "parallelism": f"replicas x{ws}"},
                "frac_of_peak": round(value / ws / peak, 4), "peak_gbs": peak,
                "roofline": roof,
                "cpu_baseline": cpu,
                "e2e": {"value": round(ws * alg_step / e2e_s / 1e9, 1), "unit": "GB/s",
                        "h2d_bytes_per_step": 2 * shape.d, "d2h_bytes_per_step": 4 * shape.vocab,
                        "us_per_step": round(e2e_s * 1e6, 1)},
                "gpu_launches": int(launches),
                "clocks": clk,
                **extra}
        print(json.dumps(line), flush=True)


def main():
    args = parse()
    ws, rank, local = dist_setup(args)
    if args.impl == "reference":
        run_reference(args, ws, rank)
    else:
        run_vbq(args, ws, rank, local)
    if ws > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
