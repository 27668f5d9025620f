"""Benchmark of the single-GPU MoE layer forward (router -> align -> GEMM1 +
SwiGLU -> GEMM2 + weight -> finalize) on one GB300, one JSON line on stdout.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                  [--workload dsv3] [--T 4096] [--no-sweep] [--no-cpu]

A step is one pass of the whole hot path over one batch of T synthetic tokens
(seeded inputs of the workload's shapes, random-init weights): the layer
captured as one CUDA graph (moe_layer: router, align, GEMM1, GEMM2,
finalize), replayed K times between CUDA events on the launching stream.  The
headline (`value`) is the largest single-GPU workload, the DeepSeek-V3-shaped
layer (22.5 GB of bf16 experts) at T = 4096 tokens.  Each stage is also
captured in its own graph and replayed with events between them, which gives
every kernel's own time (the dominant kernel's roofline).

The same line carries every other workload, each timed as its own graphs
with L2 flushed before every replay: the Qwen3-shaped layer at T = 1, 64,
512 and 4096, DeepSeek-V3 at T = 1 and 256, the low-bit DeepSeek-V4-Flash
layer at T = 512 and 4096, the GLM router and align (alone and together,
BLOCK_M 16 / 64 / 128, T = 1 .. 4096), and each gate's floor (an empty kernel
and a kernel that reads the gate once, "How an MoE Model Picks Its Experts
During LLM Inference" §3.3) against which the router's time is reported.

With --gpus N (N > 1) and no torchrun environment, N replica processes are
started here, one per GPU; under torchrun every rank is such a replica.  The
layer has no collective: each rank runs the headline workload on its own GPU
and the step time is the maximum over ranks (one all-reduce MAX of a float).

--impl reference times the CPU oracle (the test-infrastructure reference of
the method) on a bounded token sample of the same workload.
"""
from __future__ import annotations

import argparse
import ctypes
import json
import math
import os
import socket
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = ("MoE layer µs/layer & tokens/s vs T (1..4096); router µs; "
          "% HBM/tensor roofline")
UNIT = "tokens/s"
HEADLINE = ("dsv3", 4096)


# --------------------------------------------------------------------------
# peaks, clocks, distributed helpers
# --------------------------------------------------------------------------
def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        p = json.load(open(path))
        return {"hbm_gbs": float(p["hbm_gbs"]), "bf16_tflops": float(p["bf16_tflops"]),
                "bf16_tflops_sustained": float(p.get("bf16_tflops_sustained", p["bf16_tflops"])),
                "source": "measured"}
    except Exception:
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
                "source": "fallback"}


# clocks-event reason bits of NVML (nvml.h, nvmlClocksEventReason*)
_REASON_BITS = {"sw_power_cap": 0x4, "hw_slowdown": 0x8, "sw_thermal_slowdown": 0x20,
                "hw_thermal_slowdown": 0x40}


class ClockSampler:
    """SM clock, power and clocks-event reasons sampled every few milliseconds
    in a thread for the whole run (NVML through ctypes; nvidia-smi at 20 ms if
    NVML cannot be loaded).  summary(t0, t1) covers the samples taken between
    two host times, e.g. around a timed region."""

    def __init__(self, smi_id: str, period_s: float = 0.005):
        self.smi_id = smi_id
        self.period_s = period_s
        self.samples = []        # (host time, sm MHz, reasons bitmask, power W)
        self.max_mhz = None
        self.source = None
        self._stop = threading.Event()
        self._thread = None
        self._proc = None

    def _nvml(self):
        lib = ctypes.CDLL("libnvidia-ml.so.1")
        if lib.nvmlInit_v2() != 0:
            raise RuntimeError("nvmlInit failed")
        h = ctypes.c_void_p()
        if self.smi_id.startswith("GPU-") or self.smi_id.startswith("MIG-"):
            rc = lib.nvmlDeviceGetHandleByUUID(self.smi_id.encode(), ctypes.byref(h))
        else:
            rc = lib.nvmlDeviceGetHandleByIndex_v2(int(self.smi_id), ctypes.byref(h))
        if rc != 0:
            raise RuntimeError("nvml handle")
        mx = ctypes.c_uint(0)
        if lib.nvmlDeviceGetMaxClockInfo(h, 1, ctypes.byref(mx)) == 0:
            self.max_mhz = float(mx.value)
        reasons_fn = getattr(lib, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            lib.nvmlDeviceGetCurrentClocksThrottleReasons
        return lib, h, reasons_fn

    def start(self):
        try:
            lib, h, reasons_fn = self._nvml()
            self.source = "nvml, %d ms" % round(self.period_s * 1e3)

            def loop():
                clk, rs, pw = ctypes.c_uint(0), ctypes.c_ulonglong(0), ctypes.c_uint(0)
                while not self._stop.is_set():
                    t = time.perf_counter()
                    if lib.nvmlDeviceGetClockInfo(h, 1, ctypes.byref(clk)) == 0:
                        reasons_fn(h, ctypes.byref(rs))
                        lib.nvmlDeviceGetPowerUsage(h, ctypes.byref(pw))
                        self.samples.append((t, float(clk.value), int(rs.value),
                                             pw.value / 1e3))
                    time.sleep(self.period_s)

            self._thread = threading.Thread(target=loop, daemon=True)
            self._thread.start()
        except Exception:
            self._start_smi()
        return self

    def _start_smi(self):
        fields = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.sw_power_cap,"
                  "clocks_event_reasons.hw_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
                  "clocks_event_reasons.hw_thermal_slowdown")
        try:
            self._proc = subprocess.Popen(
                ["nvidia-smi", "-i", self.smi_id, f"--query-gpu={fields}",
                 "--format=csv,noheader,nounits", "-lms=20"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.source = "nvidia-smi, 20 ms"

            def read():
                bits = [_REASON_BITS[n] for n in ("sw_power_cap", "hw_slowdown",
                                                   "sw_thermal_slowdown", "hw_thermal_slowdown")]
                for line in self._proc.stdout:
                    parts = [x.strip() for x in line.split(",")]
                    try:
                        sm, mx, pw = float(parts[0]), float(parts[1]), float(parts[2])
                    except (ValueError, IndexError):
                        continue
                    r = sum(b for b, v in zip(bits, parts[3:7]) if v.lower().startswith("active"))
                    self.max_mhz = mx
                    self.samples.append((time.perf_counter(), sm, r, pw))

            self._thread = threading.Thread(target=read, daemon=True)
            self._thread.start()
        except Exception:
            self._proc = None

    def stop(self):
        self._stop.set()
        if self._proc is not None:
            self._proc.terminate()
            try:
                self._proc.wait(timeout=5)
            except Exception:
                self._proc.kill()
        if self._thread is not None:
            self._thread.join(timeout=5)

    def summary(self, t0=None, t1=None):
        s = [x for x in list(self.samples) if (t0 is None or x[0] >= t0) and
             (t1 is None or x[0] <= t1)]
        if not s:
            return {"sm_mhz": None, "sm_max_mhz": self.max_mhz, "reasons": [], "samples": 0,
                    "source": self.source}
        reasons = sorted(n for n, b in _REASON_BITS.items() if any(x[2] & b for x in s))
        return {"sm_mhz": statistics.median(x[1] for x in s), "sm_max_mhz": self.max_mhz,
                "sm_mhz_min": min(x[1] for x in s), "power_w_max": round(max(x[3] for x in s), 1),
                "reasons": reasons, "samples": len(s), "source": self.source}


def smi_index(local: int) -> str:
    """nvidia-smi -i argument of this process's device (honours CUDA_VISIBLE_DEVICES)."""
    cvd = os.environ.get("CUDA_VISIBLE_DEVICES", "").strip()
    if cvd:
        parts = [p.strip() for p in cvd.split(",") if p.strip()]
        if local < len(parts):
            return parts[local]
    return str(local)


def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def reduce_max(value: float, world: int, device=None) -> float:
    """Maximum of a float over the ranks of the default process group."""
    if world <= 1:
        return value
    import torch
    import torch.distributed as dist
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(world: int, device=None):
    if world > 1:
        import torch.distributed as dist
        if device is not None and dist.get_backend() == "nccl":
            dist.barrier(device_ids=[device.index])
        else:
            dist.barrier()


def free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def launch_replicas(n: int, argv: list) -> int:
    """Start n replicas of this script, one per GPU (rank r on local device
    r), with the rendezvous environment torchrun would give them; rank 0's
    stdout is this process's.  Returns the first non-zero exit code, else 0."""
    port = free_port()
    procs = []
    for r in range(n):
        env = dict(os.environ, RANK=str(r), LOCAL_RANK=str(r), WORLD_SIZE=str(n),
                   LOCAL_WORLD_SIZE=str(n), MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
        procs.append(subprocess.Popen([sys.executable, os.path.abspath(__file__)] + list(argv),
                                      env=env, stdout=None if r == 0 else subprocess.DEVNULL))
    rcs = [p.wait() for p in procs]
    return next((rc for rc in rcs if rc != 0), 0)


# --------------------------------------------------------------------------
# algorithmic bytes / FLOPs (the method's own, padding and round trips apart)
# --------------------------------------------------------------------------
def work_model(w, T, touched, block_m, b_x=None, b_w=None, b_g=None):
    """Bytes per element: bf16 2; low-bit workload: e4m3 activations and the
    re-quantised intermediate 1 + 1/32 (scale byte per 32), e2m1 weights
    0.5 + 1/32, fp32 gate 4."""
    H, E, k, F = w.H, w.E, w.k, w.F
    if b_x is None:
        b_x = (1 + 1 / 32) if w.lowbit else 2
    if b_w is None:
        b_w = (0.5 + 1 / 32) if w.lowbit else 2
    if b_g is None:
        b_g = 4 if w.lowbit else 2
    b_i = (1 + 1 / 32) if w.lowbit else 2   # intermediate
    cap = T * k + E * (block_m - 1)
    st = {
        "router": {"bytes": E * H * b_g + T * H * b_x + 8 * T * k, "flops": 2 * T * E * H},
        "align": {"bytes": 4 * T * k + 4 * cap + 4 * math.ceil(cap / block_m), "flops": 0},
        "gemm1": {"bytes": touched * 2 * F * H * b_w + T * H * b_x + T * k * F * b_i,
                  "flops": 2 * T * k * 2 * F * H},
        "gemm2": {"bytes": touched * H * F * b_w + T * k * F * b_i + T * k * H * 2,
                  "flops": 2 * T * k * H * F},
        "finalize": {"bytes": T * k * H * 2 + T * H * 2, "flops": 0},
    }
    layer = {"bytes": touched * 3 * H * F * b_w + T * H * b_x + T * H * 2 + st["router"]["bytes"],
             "flops": 6 * T * k * H * F + st["router"]["flops"]}
    return st, layer


# nominal dense-rate ratio fp8 : bf16 on the tensor cores (4.5 : 2.25 PFLOP/s),
# used only when the fp8 rate could not be measured in the run
FP8_OVER_BF16 = 2.0


def roofline_of(bytes_, flops, seconds, peaks, fp8=False):
    """Binding roofline of a kernel or the layer.  The tensor peak is the
    measured bf16 figure, or for the block-scaled fp8 contractions of the
    low-bit workload the fp8 rate measured in the run (else the bf16 figure
    times the nominal fp8 : bf16 ratio)."""
    if fp8:
        tc = peaks.get("fp8_tflops") or peaks["bf16_tflops"] * FP8_OVER_BF16
        tdt = ("fp8 (measured in this run: torch._scaled_mm e4m3 8192^3)"
               if peaks.get("fp8_tflops") else "fp8 (bf16 measured x 2, nominal ratio)")
    else:
        tc, tdt = peaks["bf16_tflops"], "bf16"
    t_hbm = bytes_ / (peaks["hbm_gbs"] * 1e9)
    t_tc = flops / (tc * 1e12)
    if t_hbm >= t_tc:
        ach = bytes_ / seconds / 1e9
        return {"bound": "hbm", "achieved": ach, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                "frac": ach / peaks["hbm_gbs"]}
    ach = flops / seconds / 1e12
    return {"bound": "tensor", "achieved": ach, "peak": tc, "unit": "TFLOP/s",
            "frac": ach / tc, "tensor_dtype": tdt}


def rounded(d):
    return {k: (round(v, 4) if isinstance(v, float) else v) for k, v in d.items()}


class L2Flush:
    """Evicts the workload from L2 between timed replays: writes a 512 MB
    buffer (4x L2), then reads a separate 256 MB buffer so the dirty lines of
    the write are written back before the timed region instead of inside it."""

    def __init__(self, torch, dev):
        self.w = torch.empty(512 << 20, dtype=torch.uint8, device=dev)
        self.r = torch.zeros((256 << 20) // 4, dtype=torch.int32, device=dev)
        self.acc = torch.zeros((), dtype=torch.int64, device=dev)
        self.torch = torch

    def __call__(self):
        self.w.zero_()
        self.torch.sum(self.r, (0,), dtype=self.torch.int64, out=self.acc)


def measure_fp8_peak(torch, dev):
    """Dense fp8 tensor rate of this GPU: torch._scaled_mm (cuBLASLt) e4m3 x
    e4m3 -> bf16 at 8192^3, best of 10.  The block-scaled MMA of the low-bit
    kernels issues at the fp8 rate."""
    try:
        n = 8192
        a = torch.randn((n, n), device=dev).to(torch.float8_e4m3fn)
        b = torch.randn((n, n), device=dev).to(torch.float8_e4m3fn).t()
        one = torch.ones((), device=dev, dtype=torch.float32)

        def f():
            return torch._scaled_mm(a, b, scale_a=one, scale_b=one, out_dtype=torch.bfloat16)

        for _ in range(3):
            f()
        torch.cuda.synchronize()
        best = float("inf")
        for _ in range(10):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            f()
            e1.record()
            torch.cuda.synchronize()
            best = min(best, e0.elapsed_time(e1))
        del a, b
        return 2.0 * n ** 3 / (best / 1e3) / 1e12, None
    except Exception as e:  # the tensor-core rate then falls back to the nominal ratio
        return None, f"{type(e).__name__}: {e}"[:200]


# --------------------------------------------------------------------------
# CPU oracle leg
# --------------------------------------------------------------------------
def oracle_sample_step(w, d_host, T, tokens):
    """One pass of the oracle's hot path over a token sample: router, align of
    the sample's assignments, naive per-expert FFN and weighted sum."""
    import numpy as np
    import oracle
    x_dt = "e4m3" if w.lowbit else "bf16"
    g_dt = "f32" if w.lowbit else "bf16"
    ids, wts, gap = oracle.router(d_host["hidden"], x_dt, d_host["gate"], g_dt,
                                  d_host.get("bias"), T, w.H, w.E, w.k, w.scoring, w.n_group,
                                  w.topk_group, w.renormalize, w.scaling,
                                  x_scale=d_host.get("hidden_scale"), tokens=tokens)
    from router_experts_gb300 import workloads as W
    oracle.align(ids, len(tokens), w.k, w.E, W.block_m_for(T, w.k, w.E))
    full_ids = np.zeros((T, w.k), np.int32)
    full_w = np.zeros((T, w.k), np.float64)
    full_ids[tokens] = ids
    full_w[tokens] = wts
    oracle.moe_ffn(d_host["hidden"], x_dt, d_host["w13"], d_host["w2"],
                   "e2m1" if w.lowbit else "bf16", T, w.H, w.F, w.E, w.k, full_ids, full_w,
                   x_scale=d_host.get("hidden_scale"), w13_scale=d_host.get("w13_scale"),
                   w2_scale=d_host.get("w2_scale"), tokens=tokens)


def host_inputs(d):
    from router_experts_gb300 import workloads as W
    out = {}
    for k, v in d.items():
        out[k] = v.cpu().numpy() if k == "bias" else W.to_host_raw(v)
    return out


def time_oracle(w, d_host, T, n_tokens, steps=1, seed=0):
    import numpy as np
    rng = np.random.default_rng(seed)
    times = []
    for s in range(steps):
        tokens = np.sort(rng.choice(T, n_tokens, replace=False)).astype(np.int32)
        t0 = time.perf_counter()
        oracle_sample_step(w, d_host, T, tokens)
        times.append(time.perf_counter() - t0)
    return times


def workload_label(w, T, BM=None):
    grp = f", groups {w.n_group}/{w.topk_group}" if w.n_group > 1 else ""
    bm = f", BLOCK_M={BM}" if BM else ""
    kind = "e4m3 x e2m1 experts" if w.lowbit else "bf16 experts"
    return (f"{w.name} MoE layer forward (H={w.H}, E={w.E}, k={w.k}, F={w.F}, {w.scoring}"
            f"{grp}, {kind}), T={T} tokens{bm}, random-init weights")


# --------------------------------------------------------------------------
# GPU leg
# --------------------------------------------------------------------------
class LayerBench:
    """Graphs and timings of one layer workload on one device."""

    names = ["router", "align", "gemm1", "gemm2", "finalize"]

    def __init__(self, torch, moe, W, w, d, dev, peaks, Ts):
        self.torch, self.moe, self.W, self.w, self.d, self.dev = torch, moe, W, w, d, dev
        self.peaks = peaks
        self.stream = torch.cuda.current_stream(dev)
        # One workspace, sized once for every call below: a CUDA graph keeps
        # the buffer it was captured with, so the buffer must never be replaced.
        lib = moe.load()
        k, E, H, F = w.k, w.E, w.H, w.F
        adt = moe.DT_E4M3 if w.lowbit else moe.DT_BF16
        need = 0
        for Tn in Ts:
            bmn = moe.pick_block_m(Tn, k, E)
            need = max(need, moe.layer_workspace_bytes(Tn, H, F, E, k, 0, adt),
                       lib.moe_router_workspace_bytes(Tn, H, E), lib.moe_align_workspace_bytes(),
                       lib.moe_ffn_workspace_bytes(Tn, H, F, E, k, bmn, adt))
        self.ws = moe.Workspace(dev)
        self.ws.get(need)

    def lowbit_kw(self, xs=None):
        d = self.d
        if not self.w.lowbit:
            return {}
        return dict(hidden_scale=d["hidden_scale"] if xs is None else xs,
                    w13_scale=d["w13_scale"], w2_scale=d["w2_scale"])

    def layer_args(self, x):
        w, d = self.w, self.d
        return (x, d["gate"], d.get("bias"), d["w13"], d["w2"], w.k, w.scoring, w.n_group,
                w.topk_group, w.renormalize, w.scaling)

    def stage_graphs(self, x, xs=None):
        """One CUDA graph per kernel for the batch x (xs: its scales for the
        low-bit workload); returns graphs + routing facts."""
        torch, moe, w, d, ws = self.torch, self.moe, self.w, self.d, self.ws
        k, E = w.k, w.E
        Tn = x.shape[0]
        bm = moe.pick_block_m(Tn, k, E)
        a_r = (x, d["gate"], d.get("bias"), k, w.scoring, w.n_group, w.topk_group,
               w.renormalize, w.scaling)
        lb = dict(x_scale=xs, w13_scale=d.get("w13_scale")) if w.lowbit else {}
        lb2 = dict(w2_scale=d.get("w2_scale")) if w.lowbit else {}

        def g1(s_ids, blk, npp):
            return moe.expert_gemm1(x, d["w13"], bm, s_ids, blk, npp, k, ws=ws, **lb)

        def g2(inter, s_ids, blk, npp):
            if w.lowbit:
                return moe.expert_gemm2(inter[0], d["w2"], Tn, k, bm, s_ids, blk, npp, wts, ws=ws,
                                        inter_scale=inter[1], **lb2)
            return moe.expert_gemm2(inter, d["w2"], Tn, k, bm, s_ids, blk, npp, wts, ws=ws)

        ids, wts = moe.router(*a_r, hidden_scale=xs, ws=ws)
        s_ids, blk, npp = moe.align(ids, E, bm, ws=ws)
        inter = g1(s_ids, blk, npp)
        st = g2(inter, s_ids, blk, npp)
        y = moe.finalize(st, Tn, k)
        torch.cuda.synchronize()
        gs, outs = {}, {}

        def cap(name, fn):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g):
                outs[name] = fn()
            gs[name] = g

        cap("router", lambda: moe.router(*a_r, hidden_scale=xs, ws=ws, out=(ids, wts)))
        cap("align", lambda: moe.align(ids, E, bm, ws=ws))
        s2, b2, n2 = outs["align"]
        cap("gemm1", lambda: g1(s2, b2, n2))
        i2 = outs["gemm1"]
        cap("gemm2", lambda: g2(i2, s2, b2, n2))
        st2 = outs["gemm2"]
        cap("finalize", lambda: moe.finalize(st2, Tn, k, out=y))
        for n in self.names:
            gs[n].replay()
        torch.cuda.synchronize()
        facts = {"touched": int(torch.unique(ids).numel()), "block_m": bm,
                 "max_rows": int(torch.bincount(ids.reshape(-1).long(), minlength=E).max()),
                 "padded_rows": int(n2.item())}
        return gs, facts, outs

    def layer_graph(self, x, xs=None, out=None):
        torch, moe = self.torch, self.moe
        out = out if out is not None else torch.empty((x.shape[0], self.w.H),
                                                      dtype=torch.bfloat16, device=self.dev)
        kw = self.lowbit_kw(xs)
        moe.layer(*self.layer_args(x), ws=self.ws, out=out, **kw)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            moe.layer(*self.layer_args(x), ws=self.ws, out=out, **kw)
        return g, out

    def stage_times(self, gs, reps, flush=None):
        """Mean (flush None) or median (flushed) µs of every stage graph."""
        torch, names = self.torch, self.names
        for _ in range(3):
            if flush is not None:
                flush()
            for n in names:
                gs[n].replay()
        times = {n: [] for n in names}
        evs = [[torch.cuda.Event(enable_timing=True) for _ in range(len(names) + 1)]
               for _ in range(reps)]
        torch.cuda.synchronize()
        for i in range(reps):
            if flush is not None:
                flush()
            for j, n in enumerate(names):
                evs[i][j].record(self.stream)
                gs[n].replay()
            evs[i][-1].record(self.stream)
            if flush is not None:
                torch.cuda.synchronize()
        torch.cuda.synchronize()
        for i in range(reps):
            for j, n in enumerate(names):
                times[n].append(evs[i][j].elapsed_time(evs[i][j + 1]) * 1e3)
        agg = statistics.mean if flush is None else statistics.median
        return {n: agg(v) for n, v in times.items()}

    def graph_us(self, g, reps, flush):
        """Median µs of a graph replayed after an L2 flush."""
        torch = self.torch
        for _ in range(3):
            flush()
            g.replay()
        lt = []
        for _ in range(reps):
            flush()
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record(self.stream)
            g.replay()
            e1.record(self.stream)
            torch.cuda.synchronize()
            lt.append(e0.elapsed_time(e1) * 1e3)
        return statistics.median(lt)

    def sweep_point(self, T, flush, reps=25):
        """The layer at T tokens (a prefix of the workload's batch) as one graph
        and as stage graphs, L2 flushed before every replay."""
        d, w = self.d, self.w
        x = d["hidden"][:T].contiguous()
        xs = d["hidden_scale"][:T].contiguous() if w.lowbit else None
        gs, fs, ka = self.stage_graphs(x, xs)
        us = self.stage_times(gs, reps, flush)
        lg, _ = self.layer_graph(x, xs)
        tot = self.graph_us(lg, reps, flush)
        del lg, gs, ka
        # the whole layer in one persistent kernel (small bf16 batches)
        pers = None
        if not w.lowbit and self.moe.layer_persistent_workspace_bytes(T, w.H, w.F, w.E, w.k):
            torch = self.torch
            wsp = self.moe.Workspace(self.dev)
            out = torch.empty((T, w.H), dtype=torch.bfloat16, device=self.dev)
            pa = self.layer_args(x)

            def run_p():
                self.moe.layer_persistent(pa[0], pa[1], pa[2], pa[3], pa[4], pa[5], pa[6], pa[7],
                                          pa[8], pa[9], pa[10], ws=wsp, out=out)

            run_p()
            pg = torch.cuda.CUDAGraph()
            with torch.cuda.graph(pg):
                run_p()
            pers = self.graph_us(pg, reps, flush)
            del pg, wsp
        sm_, lm = work_model(w, T, fs["touched"], fs["block_m"])
        lr = roofline_of(lm["bytes"], lm["flops"], tot / 1e6, self.peaks, fp8=w.lowbit)
        stage_roof = {}
        for n in self.names:
            r = roofline_of(sm_[n]["bytes"], sm_[n]["flops"], us[n] / 1e6, self.peaks,
                            fp8=w.lowbit and n in ("gemm1", "gemm2"))
            stage_roof[n] = {"bound": r["bound"], "frac": round(r["frac"], 4)}
        res = {"us_per_layer": round(tot, 2), "tokens_per_s": round(T / (tot / 1e6), 1),
                "stage_us": {n: round(v, 2) for n, v in us.items()},
                "stage_roofline": stage_roof,
                "touched_experts": fs["touched"], "block_m": fs["block_m"],
                "max_rows_per_expert": fs["max_rows"],
                "roofline": {"bound": lr["bound"], "frac": round(lr["frac"], 4),
                             "achieved": round(lr["achieved"], 1), "unit": lr["unit"]}}
        if pers is not None:
            pr = roofline_of(lm["bytes"], lm["flops"], pers / 1e6, self.peaks)
            res["persistent"] = {"us_per_layer": round(pers, 2),
                                 "roofline": {"bound": pr["bound"], "frac": round(pr["frac"], 4)},
                                 "note": "moe_layer_persistent: the whole layer in one kernel"}
        return res


def kernel_name(w, stage, BM, H):
    gw1 = 4 if (BM == 128 and H <= 4096) else 2
    if stage in ("gemm1", "gemm2"):
        kind = 0 if stage == "gemm1" else 1
        if w.lowbit:
            return "lowbit_gemm_kernel<%d>" % kind
        if BM == 128 and H > 4096:  # 128-row tiles on CTA pairs above H = 4096
            return "ffn_pair_kernel<%d,%d>" % (kind, 4 if kind == 0 else 2)
        return "ffn_gemm_kernel<%d,%d,%d>" % ((0, BM, gw1) if kind == 0 else (1, BM, 2))
    return {"router": "router_gemm_kernel + router_select_kernel", "align": "align_kernel",
            "finalize": "finalize_kernel"}[stage]


def floor_probe(torch, moe, dev, stream, gate, flush, reps=25):
    """"How an MoE Model Picks Its Experts During LLM Inference" §3.3: an
    empty kernel of one block, an empty kernel of as many 512-thread blocks as
    the read, and a kernel whose every thread loads 16 bytes of the gate (the
    whole matrix once), each one graph replayed after an L2 flush."""
    nbytes = gate.numel() * gate.element_size()
    blocks = max(1, -(-nbytes // (16 * 512)))
    sink = torch.zeros((1,), dtype=torch.int32, device=dev)
    out = {}
    for name, fn in (("empty_1_block_us", lambda: moe.probe_empty(1, 512, dev)),
                     ("empty_%d_blocks_us" % blocks, lambda: moe.probe_empty(blocks, 512, dev)),
                     ("read_gate_us", lambda: moe.probe_read(gate, sink))):
        fn()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            fn()
        for _ in range(3):
            flush()
            g.replay()
        lt = []
        for _ in range(reps):
            flush()
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            g.replay()
            e1.record(stream)
            torch.cuda.synchronize()
            lt.append(e0.elapsed_time(e1) * 1e3)
        out[name] = round(statistics.median(lt), 2)
        del g
    out["gate_bytes"] = nbytes
    return out


def glm_router_align(torch, moe, W, dev, stream, flush, reps=25):
    """Configuration "router + align only" (GLM-style gate): router alone, align
    alone and the two in one graph, BLOCK_M 16 / 64 / 128, T = 1 .. 4096,
    each graph replayed after an L2 flush (median µs)."""
    w = W.WORKLOADS["glm"]
    Tmax = max(w.Ts)
    d = W.make_inputs(w, Tmax, seed=0, device=dev, experts=False)
    ws = moe.Workspace(dev)
    lib = moe.load()
    ws.get(max(lib.moe_router_workspace_bytes(Tmax, w.H, w.E), lib.moe_align_workspace_bytes()))
    res = {"router_us": {}, "align_us": {}, "router_align_us": {},
           "router_kernels": {}, "shape": f"H={w.H}, E={w.E}, k={w.k}, sigmoid + bias"}

    def timed(fn):
        fn()
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            keep = fn()
        for _ in range(3):
            flush()
            g.replay()
        lt = []
        for _ in range(reps):
            flush()
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            g.replay()
            e1.record(stream)
            torch.cuda.synchronize()
            lt.append(e0.elapsed_time(e1) * 1e3)
        del g, keep
        return round(statistics.median(lt), 2)

    for T in w.Ts:
        x = d["hidden"][:T].contiguous()
        args = (x, d["gate"], d["bias"], w.k, w.scoring)
        ids, wts = moe.router(*args, ws=ws)
        res["router_us"][str(T)] = timed(lambda: moe.router(*args, ws=ws, out=(ids, wts)))
        res["router_kernels"][str(T)] = moe.router_kernel_count(T, w.H, w.E)
        for bm in w.block_ms:
            res["align_us"].setdefault(str(bm), {})[str(T)] = timed(
                lambda: moe.align(ids, w.E, bm, ws=ws))

            def both():
                moe.router(*args, ws=ws, out=(ids, wts))
                return moe.align(ids, w.E, bm, ws=ws)

            res["router_align_us"].setdefault(str(bm), {})[str(T)] = timed(both)
    floor = floor_probe(torch, moe, dev, stream, d["gate"], flush, reps)
    res["floor"] = floor
    res["router_over_floor"] = {T: round(v / floor["read_gate_us"], 2)
                                for T, v in res["router_us"].items()}
    del d, ws
    return res


def run_ours(args):
    import numpy as np
    import torch

    from router_experts_gb300 import build as B
    from router_experts_gb300 import moe
    from router_experts_gb300 import workloads as W

    world, rank, local = dist_env()
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    B.build()
    moe.load()
    peaks = load_peaks()
    clk = ClockSampler(smi_index(local)).start()
    stream = torch.cuda.current_stream(dev)
    run_sweeps = world == 1 and not args.no_sweep
    if run_sweeps:
        fp8, fp8_err = measure_fp8_peak(torch, dev)
        peaks["fp8_tflops"] = fp8
        if fp8_err:
            peaks["fp8_error"] = fp8_err

    w = W.WORKLOADS[args.workload]
    if args.experts:
        # fewer experts of the same shape: a smaller device footprint for
        # profiler captures (the sweeps and the other workloads are skipped)
        import dataclasses
        w = dataclasses.replace(w, E=args.experts)
        run_sweeps = False
    T = args.T
    k, E, H, F = w.k, w.E, w.H, w.F
    d = W.make_inputs(w, T, seed=args.seed, device=dev)
    torch.cuda.synchronize()
    sweep_Ts = [t for t in w.Ts if t < T] if run_sweeps else []
    lb = LayerBench(torch, moe, W, w, d, dev, peaks, [T] + sweep_Ts)

    # ---- stage graphs (each holds exactly one kernel of the library) ----
    graphs, facts, keep_alive = lb.stage_graphs(d["hidden"], d.get("hidden_scale"))
    BM, touched = facts["block_m"], facts["touched"]

    # the bytes a step reads are the touched experts' weights (plus scales), not
    # the whole weight tensors: only inputs larger than L2 make a flush needless
    weights_bytes = ((d["w13"].numel() + d["w2"].numel()) * d["w13"].element_size()
                     + sum(d[s].numel() for s in ("w13_scale", "w2_scale") if s in d))
    weights_bytes = weights_bytes * touched // E
    l2_note = ("inputs larger than L2 (weights of the touched experts %.2f GB)" % (weights_bytes / 1e9)
               if weights_bytes > 256e6 else "L2 flushed between steps (512 MB write, then 256 MB read)")
    flush = None if weights_bytes > 256e6 else L2Flush(torch, dev)

    # the layer as a user runs it: one CUDA graph holding every kernel; this
    # is the timed step
    y_layer = torch.empty((T, H), dtype=torch.bfloat16, device=dev)
    layer_graph, _ = lb.layer_graph(d["hidden"], d.get("hidden_scale"), out=y_layer)
    for _ in range(args.warmup):
        if flush is not None:
            flush()
        layer_graph.replay()
    torch.cuda.synchronize()

    K = args.steps
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(K)]
    barrier(world, dev)
    torch.cuda.synchronize()
    h0 = time.perf_counter()
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    if flush is None:
        t_start.record(stream)
    for i in range(K):
        if flush is not None:
            flush()
            ev[i][0].record(stream)
        layer_graph.replay()
        if flush is not None:
            ev[i][1].record(stream)
    if flush is None:
        t_end.record(stream)
    torch.cuda.synchronize()
    h1 = time.perf_counter()
    barrier(world, dev)
    if flush is None:
        total_ms = t_start.elapsed_time(t_end)
    else:
        total_ms = sum(ev[i][0].elapsed_time(ev[i][1]) for i in range(K))
    total_ms = reduce_max(total_ms, world, dev)
    ms_per_step = total_ms / K
    value = world * T * K / (total_ms / 1e3)
    clocks = clk.summary(h0, h1)
    del layer_graph

    # ---- per-kernel times: each stage graph replayed with events between them ----
    Ks = max(3, min(K, 500))
    stage_us = lb.stage_times(graphs, Ks, flush)
    st_model, layer_model = work_model(w, T, touched, BM)
    names = LayerBench.names
    dom = max(names, key=lambda n: stage_us[n])
    roof = roofline_of(st_model[dom]["bytes"], st_model[dom]["flops"], stage_us[dom] / 1e6, peaks,
                       fp8=w.lowbit and dom in ("gemm1", "gemm2"))
    roof["kernel"] = kernel_name(w, dom, BM, H)
    roof["launch_us"] = round(stage_us[dom], 2)
    roof["algorithmic_bytes"] = st_model[dom]["bytes"]
    roof["algorithmic_flops"] = st_model[dom]["flops"]
    # DRAM bytes per launch come only from an ncu capture of this same run's
    # kernel (--traffic-csv); without one the field stays null
    roof["traffic"] = None
    if args.traffic_csv:
        roof["traffic"] = traffic_from_csv(args.traffic_csv, roof["kernel"])
    roof["peak_source"] = peaks["source"] + " (burst)"
    layer_roof = roofline_of(layer_model["bytes"], layer_model["flops"], ms_per_step / 1e3, peaks,
                             fp8=w.lowbit)
    stage_roof = {}
    for n in names:
        r = roofline_of(st_model[n]["bytes"], st_model[n]["flops"], stage_us[n] / 1e6, peaks,
                        fp8=w.lowbit and n in ("gemm1", "gemm2"))
        stage_roof[n] = {"bound": r["bound"], "frac": round(r["frac"], 4)}
    del graphs, keep_alive

    # ---- the headline workload's other batch sizes ----
    workloads = {}
    if run_sweeps:
        fl = L2Flush(torch, dev)
        sw = {}
        for Ts in sweep_Ts:
            sw[str(Ts)] = lb.sweep_point(Ts, fl)
        sw[str(T)] = {"us_per_layer": round(ms_per_step * 1e3, 2),
                      "tokens_per_s": round(T / (ms_per_step / 1e3), 1),
                      "stage_us": {n: round(v, 2) for n, v in stage_us.items()},
                      "stage_roofline": stage_roof,
                      "touched_experts": touched, "block_m": BM,
                      "max_rows_per_expert": facts["max_rows"],
                      "roofline": {"bound": layer_roof["bound"],
                                   "frac": round(layer_roof["frac"], 4),
                                   "achieved": round(layer_roof["achieved"], 1),
                                   "unit": layer_roof["unit"]},
                      "note": "the headline run (K timed steps)"}
        workloads[w.name] = {"shape": workload_label(w, T).split(", T=")[0], "T": sw}
        workloads[w.name]["floor"] = floor_probe(torch, moe, dev, stream, d["gate"], fl)
        del fl

    # ---- end to end through the public API, host buffers ----
    # A serving loop: every step copies its hidden rows from pinned host
    # memory, runs moe.layer and copies its output back to pinned host memory.
    # With at least 1 MiB to copy per step the copies run on their own streams
    # (one per direction, two device buffers each), so step i+1's input copy
    # and step i-1's output copy overlap step i's layer; events order each
    # buffer's reuse.  Smaller steps run the three in order on one stream (the
    # cross-stream events would cost more than the copies they hide).
    lbk = lb.lowbit_kw()
    x_host = d["hidden"].cpu().pin_memory()
    xs_host = d["hidden_scale"].cpu().pin_memory() if w.lowbit else None
    y_host = [torch.empty((T, H), dtype=torch.bfloat16).pin_memory() for _ in range(2)]
    x_dev = [torch.empty_like(d["hidden"]) for _ in range(2)]
    xs_dev = [torch.empty_like(d["hidden_scale"]) for _ in range(2)] if w.lowbit else None
    y_dev = [torch.empty((T, H), dtype=torch.bfloat16, device=dev) for _ in range(2)]
    s_comp, s_in, s_out = (torch.cuda.Stream(dev) for _ in range(3))
    h2d = x_host.numel() * x_host.element_size() + (xs_host.numel() if w.lowbit else 0)
    overlap = h2d >= (1 << 20)

    def serve(n):
        """n steps; returns (start, end) events on the current stream."""
        main = torch.cuda.current_stream(dev)
        t0 = torch.cuda.Event(enable_timing=True)
        t1 = torch.cuda.Event(enable_timing=True)
        if not overlap:
            t0.record(main)
            for _ in range(n):
                x_dev[0].copy_(x_host, non_blocking=True)
                if w.lowbit:
                    xs_dev[0].copy_(xs_host, non_blocking=True)
                lbe = dict(lbk, hidden_scale=xs_dev[0]) if w.lowbit else {}
                moe.layer(*lb.layer_args(x_dev[0]), ws=lb.ws, out=y_dev[0], **lbe)
                y_host[0].copy_(y_dev[0], non_blocking=True)
            t1.record(main)
            return t0, t1
        landed = [torch.cuda.Event() for _ in range(2)]   # input of the buffer copied in
        used = [torch.cuda.Event() for _ in range(2)]     # layer of the buffer done
        taken = [torch.cuda.Event() for _ in range(2)]    # output of the buffer copied out
        t0.record(main)
        for st in (s_comp, s_in, s_out):
            st.wait_event(t0)
        for i in range(n):
            b = i % 2
            with torch.cuda.stream(s_in):
                if i >= 2:
                    s_in.wait_event(used[b])      # step i-2's layer has read x_dev[b]
                x_dev[b].copy_(x_host, non_blocking=True)
                if w.lowbit:
                    xs_dev[b].copy_(xs_host, non_blocking=True)
                landed[b].record(s_in)
            with torch.cuda.stream(s_comp):
                s_comp.wait_event(landed[b])
                if i >= 2:
                    s_comp.wait_event(taken[b])   # step i-2's output has left y_dev[b]
                lbe = dict(lbk, hidden_scale=xs_dev[b]) if w.lowbit else {}
                moe.layer(*lb.layer_args(x_dev[b]), ws=lb.ws, out=y_dev[b], **lbe)
                used[b].record(s_comp)
            with torch.cuda.stream(s_out):
                s_out.wait_event(used[b])
                y_host[b].copy_(y_dev[b], non_blocking=True)
                taken[b].record(s_out)
        for st in (s_comp, s_in, s_out):
            main.wait_stream(st)
        t1.record(main)
        return t0, t1

    K2 = max(3, min(K, 50))
    serve(4)
    torch.cuda.synchronize()
    barrier(world, dev)
    a, b = serve(K2)
    torch.cuda.synchronize()
    e2e_ms = reduce_max(a.elapsed_time(b), world, dev)
    e2e = {"value": round(world * T * K2 / (e2e_ms / 1e3), 1), "unit": UNIT,
           "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": T * H * 2, "steps": K2,
           "overlap": ("copies of neighbouring steps overlap the layer (copy stream per "
                       "direction, two buffers each)") if overlap else
                      "none (copy in, layer, copy out in order on one stream)"}
    code = moe.read_device_error(lb.ws.buf)
    del x_dev, xs_dev, y_dev, y_host, x_host, xs_host

    # ---- CPU oracle baseline (rank 0, N = 1 only) ----
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu:
        import oracle
        oracle.build()
        dh = host_inputs(d)
        # a pilot pass sizes the sample to about 15 s of CPU work
        pilot = min(T, 8)
        tp = time_oracle(w, dh, T, pilot, steps=1, seed=2)[0]
        n_tok = int(max(pilot, min(T, args.cpu_tokens if args.cpu_tokens > 0 else
                                   pilot * 15.0 / max(tp, 1e-6))))
        times = time_oracle(w, dh, T, n_tok, steps=1, seed=1)
        cpu = {"value": round(n_tok / times[0], 3), "unit": UNIT, "cores": oracle.num_threads(),
               "kind": "oracle",
               "sample": f"{n_tok} of the {T} tokens (router, align of their assignments, "
                         f"naive per-expert FFN, combine), one pass, {times[0]:.1f} s"}
        del dh
    lb = None
    del d
    torch.cuda.empty_cache()

    # ---- the other workloads, each on its own inputs ----
    if run_sweeps:
        fl = L2Flush(torch, dev)
        for name in ("qwen3", "dsv3", "v4lo"):
            if name == w.name:
                continue
            wo = W.WORKLOADS[name]
            Tm = max(wo.Ts)
            do = W.make_inputs(wo, Tm, seed=args.seed, device=dev)
            lbo = LayerBench(torch, moe, W, wo, do, dev, peaks, list(wo.Ts))
            sw = {str(Ts): lbo.sweep_point(Ts, fl) for Ts in wo.Ts}
            workloads[name] = {"shape": workload_label(wo, Tm).split(", T=")[0], "T": sw,
                               "floor": floor_probe(torch, moe, dev, stream, do["gate"], fl)}
            del lbo, do
            torch.cuda.empty_cache()
        workloads["glm"] = glm_router_align(torch, moe, W, dev, stream, fl)
        for name, v in workloads.items():
            if name == "glm" or "1" not in v["T"]:
                continue
            r1 = v["T"]["1"]["stage_us"]["router"]
            v["router_T1_over_floor"] = round(r1 / v["floor"]["read_gate_us"], 2)
        del fl
        torch.cuda.empty_cache()
    clk.stop()

    line = {
        "metric": METRIC, "value": round(value, 1), "unit": UNIT, "n_gpus": world, "steps": K,
        "warmup": args.warmup, "ms_per_step": round(ms_per_step, 4), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None,
        "dtype": ("e4m3 x e2m1 (block-scaled MMA kind::mxf8f6f4, fp32 accumulate)"
                  if w.lowbit else "bf16"),
        "data": "synthetic",
        "config": {"workload": workload_label(w, T, BM),
                   "T": T, "block_m": BM, "touched_experts": touched,
                   "max_rows_per_expert": facts["max_rows"],
                   "padded_rows": facts["padded_rows"], "l2": l2_note,
                   "parallelism": f"replicas x{world}" if world > 1 else "single GPU"},
        "roofline": rounded(roof),
        "layer_roofline": rounded(layer_roof),
        "stage_us": {n: round(v, 2) for n, v in stage_us.items()},
        "stage_roofline": stage_roof,
        "stage_note": "each kernel as its own graph, %d replays with events between them" % Ks,
        "workloads": workloads,
        "peaks": {k2: (round(v, 1) if isinstance(v, float) else v) for k2, v in peaks.items()},
        "e2e": e2e,
        "gpu_launches": K * moe.layer_kernel_count(
            T, H, F, E, k, "e4m3" if w.lowbit else "bf16", "f32" if w.lowbit else "bf16",
            "e2m1" if w.lowbit else "bf16"),
        "cpu_baseline": cpu,
        "device_error_word": code,
        "clocks": clocks,
        "clocks_run": clk.summary(),
    }
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


def traffic_from_csv(path, kernel):
    """dram__bytes_read.sum + dram__bytes_write.sum of the first launch of
    `kernel` in an ncu --csv capture (ncu's raw page), or None."""
    import csv
    try:
        rows = list(csv.DictReader(open(path)))
    except Exception:
        return None
    base = kernel.split("<")[0]
    tot = {}
    for r in rows:
        name = r.get("Kernel Name", "")
        if base not in name:
            continue
        m, v = r.get("Metric Name", ""), r.get("Metric Value", "").replace(",", "")
        if m in ("dram__bytes_read.sum", "dram__bytes_write.sum"):
            try:
                scale = {"byte": 1, "Kbyte": 1e3, "Mbyte": 1e6, "Gbyte": 1e9}.get(
                    r.get("Metric Unit", "byte"), 1)
                tot.setdefault(r.get("ID", "0"), {})[m] = float(v) * scale
            except ValueError:
                pass
    for _, mm in sorted(tot.items()):
        if len(mm) == 2:
            return sum(mm.values())
    return None


def run_dry(args):
    """The replica launch and the max-over-ranks reduction without a GPU (gloo
    process group): every rank reports a step time of rank + 1 ms."""
    world, rank, _ = dist_env()
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("gloo")
    ms = reduce_max(float(rank + 1), world)
    barrier(world)
    if rank == 0:
        print(json.dumps({"dry_run": True, "n_gpus": world, "ms_per_step": ms,
                          "steps": args.steps, "warmup": args.warmup, "scaling": "weak"}),
              flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


def run_reference(args):
    """The CPU oracle as the reference arm, on a bounded token sample."""
    world, rank, local = dist_env()
    if rank != 0:
        return
    import torch

    import oracle
    from router_experts_gb300 import workloads as W
    oracle.build()
    w = W.WORKLOADS[args.workload]
    T = args.T
    # the seeded inputs are drawn with the same generators as the GPU arm's
    # (on the GPU when there is one, then copied to host); only the oracle's
    # work on the host cores is timed
    gen_dev = torch.device("cuda", local) if torch.cuda.is_available() else torch.device("cpu")
    d = W.make_inputs(w, T, seed=args.seed, device=gen_dev)
    dh = host_inputs(d)
    del d
    if gen_dev.type == "cuda":
        torch.cuda.empty_cache()
    # size the per-step sample so that the W warm-up and K timed steps take
    # about two minutes together
    t1 = time_oracle(w, dh, T, 1, steps=1, seed=100)[0]
    budget = 120.0 / max(1, args.steps + args.warmup)
    n_tok = int(max(1, min(T, args.ref_tokens, budget // max(t1, 1e-6))))
    time_oracle(w, dh, T, n_tok, steps=args.warmup, seed=101)
    times = time_oracle(w, dh, T, n_tok, steps=args.steps, seed=0)
    tot = sum(times)
    value = n_tok * len(times) / tot
    sample = (f"{n_tok} of the {T} tokens per step (router, align of their assignments, "
              f"naive per-expert FFN, combine)")
    line = {
        "impl": "reference", "metric": METRIC, "value": round(value, 3), "unit": UNIT,
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(tot / len(times) * 1e3, 2), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": workload_label(w, T), "T": T},
        "cpu_baseline": {"value": round(value, 3), "unit": UNIT, "cores": oracle.num_threads(),
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": round(value, 3), "unit": UNIT, "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def main(argv=None):
    argv = list(sys.argv[1:] if argv is None else argv)
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=HEADLINE[0])
    ap.add_argument("--T", type=int, default=HEADLINE[1])
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--no-sweep", action="store_true",
                    help="time only the headline workload")
    ap.add_argument("--no-cpu", action="store_true")
    ap.add_argument("--cpu-tokens", type=int, default=0,
                    help="oracle sample size for cpu_baseline (0: about 15 s of CPU work)")
    ap.add_argument("--ref-tokens", type=int, default=64)
    ap.add_argument("--experts", type=int, default=0,
                    help="override the workload's expert count (profiler captures of a "
                         "smaller device footprint; implies --no-sweep)")
    ap.add_argument("--traffic-csv", default="",
                    help="ncu --csv raw capture of this command's dominant kernel")
    ap.add_argument("--dry-run", action="store_true",
                    help="replica launch and max-over-ranks reduction only (no GPU)")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        if "--steps" not in argv:
            args.steps = 5
        run_reference(args)
        return 0
    if args.gpus > 1 and "WORLD_SIZE" not in os.environ:
        return launch_replicas(args.gpus, argv)
    if args.dry_run:
        run_dry(args)
    else:
        run_ours(args)
    return 0


if __name__ == "__main__":
    sys.exit(main())
