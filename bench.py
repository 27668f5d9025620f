"""Benchmark of the single-GPU MoE layer forward (router -> align -> GEMM1 +
SwiGLU -> GEMM2 + weight -> finalize) on one GB300, one JSON line on stdout.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                  [--workload qwen3] [--T 4096] [--no-sweep] [--no-cpu]

A step is one pass of the whole hot path over one batch of T synthetic tokens
(seeded inputs of the workload's shapes, random-init weights): the layer
captured as one CUDA graph (moe_layer: router, align, GEMM1, GEMM2,
finalize), replayed K times between CUDA events on the launching stream.  Each stage is also captured in its own graph and replayed
with events between them, which gives every kernel's own time (the dominant
kernel's roofline).
Under torchrun every rank runs an independent replica (the layer has no
collective); the step time is the maximum over ranks.

--impl reference times the CPU oracle (the test-infrastructure reference of
the method) on a bounded token sample of the same workload.
"""
from __future__ import annotations

import argparse
import json
import math
import os
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


class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons during a region."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int, period_ms: int = 100):
        self.gpu_index = gpu_index
        self.period_ms = period_ms
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu_index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", f"-lms={self.period_ms}"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self._t = threading.Thread(target=self._read, daemon=True)
            self._t.start()
        except Exception:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *a):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
            self._t.join(timeout=5)

    def summary(self):
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [x.strip() for x in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx = float(parts[2])
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": mx, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


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


# DRAM bytes (read + write) per launch of a dominant kernel, from one ncu
# capture of the same workload and kernel build (the profile that records it);
# an entry is dropped whenever its kernel changes.
MEASURED_TRAFFIC = {
    ("qwen3", 4096, "ffn_gemm_kernel<0,128,4>"): (979.1e6, "profiles/ffn_gemm_qwen3_T4096.md"),
    ("v4lo", 4096, "lowbit_gemm_kernel<0>"): (2338.2e6, "profiles/lowbit_gemm_v4lo_T4096.md"),
}

# nominal dense-rate ratio fp8 : bf16 on the tensor cores (4.5 : 2.25 PFLOP/s)
FP8_OVER_BF16 = 2.0


def roofline_of(bytes_, flops, seconds, peaks, fp8=False):
    """Binding roofline of a kernel or the layer.  The tensor peak is the
    measured bf16 figure, times the nominal fp8/bf16 ratio for the block-scaled
    fp8 contractions of the low-bit workload."""
    tc = peaks["bf16_tflops"] * (FP8_OVER_BF16 if fp8 else 1.0)
    t_hbm = bytes_ / (peaks["hbm_gbs"] * 1e9)
    t_tc = flops / (tc * 1e12)
    if t_hbm >= t_tc:
        ach = bytes_ / seconds / 1e9
        return {"bound": "hbm", "achieved": ach, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                "frac": ach / peaks["hbm_gbs"]}
    ach = flops / seconds / 1e12
    return {"bound": "tensor", "achieved": ach, "peak": tc, "unit": "TFLOP/s",
            "frac": ach / tc, "tensor_dtype": "fp8 (bf16 measured x 2, nominal ratio)" if fp8
            else "bf16"}


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


# --------------------------------------------------------------------------
# GPU leg
# --------------------------------------------------------------------------
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
    w = W.WORKLOADS[args.workload]
    T = args.T
    k, E, H, F = w.k, w.E, w.H, w.F
    BM = moe.pick_block_m(T, k, E)
    d = W.make_inputs(w, T, seed=args.seed, device=dev)
    torch.cuda.synchronize()
    stream = torch.cuda.current_stream(dev)

    # ---- stage graphs (each holds exactly one kernel of the library) ----
    ws = moe.Workspace(dev)
    # One workspace, sized once for every call below: a CUDA graph keeps the
    # buffer it was captured with, so the buffer must never be replaced.
    lib = moe.load()
    adt = moe.DT_E4M3 if w.lowbit else moe.DT_BF16
    ws_need = 0
    for Tn in set([T] + list(w.Ts)):
        bmn = moe.pick_block_m(Tn, k, E)
        ws_need = max(ws_need, moe.layer_workspace_bytes(Tn, H, F, E, k, 0, adt),
                      lib.moe_router_workspace_bytes(Tn, H, E), lib.moe_align_workspace_bytes(),
                      lib.moe_ffn_workspace_bytes(Tn, H, F, E, k, bmn, adt))
    ws.get(ws_need)
    names = ["router", "align", "gemm1", "gemm2", "finalize"]

    def stage_graphs(x, xs=None):
        """One CUDA graph per kernel for the batch x (xs: its scales for the
        low-bit workload); returns graphs + routing facts."""
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
        for n in names:
            gs[n].replay()
        torch.cuda.synchronize()
        facts = {"touched": int(torch.unique(ids).numel()), "block_m": bm,
                 "max_rows": int(torch.bincount(ids.reshape(-1).long(), minlength=E).max()),
                 "padded_rows": int(n2.item())}
        return gs, facts, outs

    graphs, facts, keep_alive = stage_graphs(d["hidden"], d.get("hidden_scale"))
    BM, touched = facts["block_m"], facts["touched"]

    # the bytes a step reads are the touched experts' weights (plus scales), not
    # the whole weight tensors: only inputs larger than L2 make a flush needless
    weights_bytes = ((d["w13"].numel() + d["w2"].numel()) * d["w13"].element_size()
                     + sum(d[s].numel() for s in ("w13_scale", "w2_scale") if s in d))
    weights_bytes = weights_bytes * touched // E
    lbk = dict(hidden_scale=d.get("hidden_scale"), w13_scale=d.get("w13_scale"),
               w2_scale=d.get("w2_scale")) if w.lowbit else {}
    l2_note = ("inputs larger than L2 (weights of the touched experts %.2f GB)" % (weights_bytes / 1e9)
               if weights_bytes > 256e6 else "L2 flushed between steps (512 MB write, then 256 MB read)")
    flush = None if weights_bytes > 256e6 else L2Flush(torch, dev)

    # the layer as a user runs it: one CUDA graph holding every kernel; this
    # is the timed step
    layer_args = (d["hidden"], d["gate"], d.get("bias"), d["w13"], d["w2"], k, w.scoring,
                  w.n_group, w.topk_group, w.renormalize, w.scaling)
    y_layer = torch.empty((T, H), dtype=torch.bfloat16, device=dev)
    moe.layer(*layer_args, ws=ws, out=y_layer, **lbk)
    layer_graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(layer_graph):
        moe.layer(*layer_args, ws=ws, out=y_layer, **lbk)

    for _ in range(args.warmup):
        if flush is not None:
            flush()
        layer_graph.replay()
    torch.cuda.synchronize()

    K = args.steps
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(K)]
    barrier(world, dev)
    torch.cuda.synchronize()
    with ClockSampler(smi_index(local)) as clk:
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
    barrier(world, dev)
    if flush is None:
        total_ms = t_start.elapsed_time(t_end)
    else:
        total_ms = sum(ev[i][0].elapsed_time(ev[i][1]) for i in range(K))
    total_ms = reduce_max(total_ms, world, dev)
    ms_per_step = total_ms / K
    value = world * T * K / (total_ms / 1e3)
    del layer_graph

    # ---- per-kernel times: each stage graph replayed with events between them ----
    Ks = max(3, min(K, 500))
    for _ in range(3):
        if flush is not None:
            flush()
        for n in names:
            graphs[n].replay()
    sev = [[torch.cuda.Event(enable_timing=True) for _ in range(len(names) + 1)] for _ in range(Ks)]
    torch.cuda.synchronize()
    for i in range(Ks):
        if flush is not None:
            flush()
        for j, n in enumerate(names):
            sev[i][j].record(stream)
            graphs[n].replay()
        sev[i][len(names)].record(stream)
    torch.cuda.synchronize()
    per_stage = {n: [sev[i][j].elapsed_time(sev[i][j + 1]) for i in range(Ks)]
                 for j, n in enumerate(names)}
    stage_ms = {n: sum(v) / len(v) for n, v in per_stage.items()}
    st_model, layer_model = work_model(w, T, touched, BM)
    dom = max(names, key=lambda n: stage_ms[n])
    roof = roofline_of(st_model[dom]["bytes"], st_model[dom]["flops"], stage_ms[dom] / 1e3, peaks,
                       fp8=w.lowbit and dom in ("gemm1", "gemm2"))
    # GEMM1 row tiles (BLOCK_M 128) gather the token rows with four warps up
    # to H = 4096, with two otherwise (third template argument)
    gw1 = 4 if (BM == 128 and H <= 4096) else 2
    gk = ("lowbit_gemm_kernel<%d>", "lowbit_gemm_kernel<%d>") if w.lowbit else \
        ("ffn_gemm_kernel<%d," + str(BM) + "," + str(gw1) + ">",
         "ffn_gemm_kernel<%d," + str(BM) + ",2>")
    roof["kernel"] = {"router": "router_kernel", "align": "align_kernel",
                      "gemm1": gk[0] % 0, "gemm2": gk[1] % 1,
                      "finalize": "finalize_kernel"}[dom]
    tr = MEASURED_TRAFFIC.get((w.name, T, roof["kernel"]))
    roof["traffic"] = tr[0] if tr else None
    roof["traffic_unit"] = "bytes per launch"
    roof["traffic_source"] = tr[1] if tr else None
    roof["peak_source"] = peaks["source"] + " (burst)"
    layer_roof = roofline_of(layer_model["bytes"], layer_model["flops"], ms_per_step / 1e3, peaks,
                             fp8=w.lowbit)
    del graphs, keep_alive

    # ---- sweep over T: per-kernel times, L2 flushed before each replay ----
    sweep = {}
    if not args.no_sweep and rank == 0:
        fl = L2Flush(torch, dev)
        for Ts in w.Ts:
            if Ts >= T:
                continue
            xs = d["hidden"][:Ts].contiguous()
            xsc = d["hidden_scale"][:Ts].contiguous() if w.lowbit else None
            gs, fs, ka = stage_graphs(xs, xsc)
            lbs = dict(lbk, hidden_scale=xsc) if w.lowbit else {}
            times = {n: [] for n in names}
            for it in range(25):
                fl()
                evs = [torch.cuda.Event(enable_timing=True) for _ in range(len(names) + 1)]
                for j, n in enumerate(names):
                    evs[j].record(stream)
                    gs[n].replay()
                evs[-1].record(stream)
                torch.cuda.synchronize()
                if it >= 3:
                    for j, n in enumerate(names):
                        times[n].append(evs[j].elapsed_time(evs[j + 1]) * 1e3)
            us = {n: statistics.median(v) for n, v in times.items()}
            # the layer as a user runs it: one graph holding the five kernels
            lg = torch.cuda.CUDAGraph()
            moe.layer(xs, d["gate"], d.get("bias"), d["w13"], d["w2"], k, w.scoring, w.n_group,
                      w.topk_group, w.renormalize, w.scaling, ws=ws, **lbs)
            with torch.cuda.graph(lg):
                moe.layer(xs, d["gate"], d.get("bias"), d["w13"], d["w2"], k, w.scoring,
                          w.n_group, w.topk_group, w.renormalize, w.scaling, ws=ws, **lbs)
            lt = []
            for it in range(25):
                fl()
                e0 = torch.cuda.Event(enable_timing=True)
                e1 = torch.cuda.Event(enable_timing=True)
                e0.record(stream)
                lg.replay()
                e1.record(stream)
                torch.cuda.synchronize()
                if it >= 3:
                    lt.append(e0.elapsed_time(e1) * 1e3)
            tot = statistics.median(lt)
            del lg
            sm_, lm = work_model(w, Ts, fs["touched"], fs["block_m"])
            lr = roofline_of(lm["bytes"], lm["flops"], tot / 1e6, peaks, fp8=w.lowbit)
            sweep[str(Ts)] = {"us_per_layer": round(tot, 2),
                              "tokens_per_s": round(Ts / (tot / 1e6), 1),
                              "stage_us": {n: round(v, 2) for n, v in us.items()},
                              "stage_note": "each kernel as its own graph (incl. launch gaps)",
                              "touched_experts": fs["touched"], "block_m": fs["block_m"],
                              "roofline": {"bound": lr["bound"], "frac": round(lr["frac"], 4)}}
            del gs, ka
        sweep[str(T)] = {"us_per_layer": round(ms_per_step * 1e3, 2),
                         "tokens_per_s": round(T / (ms_per_step / 1e3), 1),
                         "stage_us": {n: round(v * 1e3, 2) for n, v in stage_ms.items()},
                         "touched_experts": touched, "block_m": BM,
                         "roofline": {"bound": layer_roof["bound"],
                                      "frac": round(layer_roof["frac"], 4)}}
        del fl

    # ---- end to end through the public API, host buffers ----
    # A serving loop: every step copies its hidden rows from pinned host
    # memory, runs moe.layer and copies its output back to pinned host memory.
    # With at least 1 MiB to copy per step the copies run on their own streams
    # (one per direction, two device buffers each), so step i+1's input copy
    # and step i-1's output copy overlap step i's layer; events order each
    # buffer's reuse.  Smaller steps run the three in order on one stream (the
    # cross-stream events would cost more than the copies they hide).
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
                moe.layer(x_dev[0], d["gate"], d.get("bias"), d["w13"], d["w2"], k, w.scoring,
                          w.n_group, w.topk_group, w.renormalize, w.scaling, ws=ws, out=y_dev[0],
                          **lbe)
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
                moe.layer(x_dev[b], d["gate"], d.get("bias"), d["w13"], d["w2"], k, w.scoring,
                          w.n_group, w.topk_group, w.renormalize, w.scaling, ws=ws, out=y_dev[b],
                          **lbe)
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
    code = moe.read_device_error(ws.buf)

    # ---- CPU oracle baseline (rank 0, N = 1 only) ----
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu:
        import oracle
        oracle.build()
        dh = host_inputs(d)
        # a pilot pass sizes the sample to about 15 s of CPU work
        pilot = min(T, 16)
        tp = time_oracle(w, dh, T, pilot, steps=1, seed=2)[0]
        n_tok = int(max(pilot, min(T, args.cpu_tokens if args.cpu_tokens > 0 else
                                   pilot * 15.0 / max(tp, 1e-6))))
        times = time_oracle(w, dh, T, n_tok, steps=1, seed=1)
        cpu = {"value": round(n_tok / times[0], 3), "unit": UNIT, "cores": oracle.num_threads(),
               "kind": "oracle",
               "sample": f"{n_tok} of the {T} tokens (router, align of their assignments, "
                         f"naive per-expert FFN, combine), one pass, {times[0]:.1f} s"}

    line = {
        "metric": METRIC, "value": round(value, 1), "unit": UNIT, "n_gpus": world, "steps": K,
        "warmup": args.warmup, "ms_per_step": round(ms_per_step, 4), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None,
        "dtype": "e4m3 x e2m1 (f16 MMA, fp32 accumulate)" if w.lowbit else "bf16",
        "data": "synthetic",
        "config": {"workload": f"{w.name} MoE layer forward (H={H}, E={E}, k={k}, F={F}, "
                               f"{w.scoring}{', groups %d/%d' % (w.n_group, w.topk_group) if w.n_group > 1 else ''}), "
                               f"T={T} tokens, BLOCK_M={BM}, random-init weights",
                   "T": T, "block_m": BM, "touched_experts": touched,
                   "max_rows_per_expert": facts["max_rows"],
                   "padded_rows": facts["padded_rows"], "l2": l2_note,
                   "parallelism": f"replicas x{world}" if world > 1 else "single GPU"},
        "roofline": {k2: (round(v, 4) if isinstance(v, float) else v) for k2, v in roof.items()},
        "layer_roofline": {k2: (round(v, 4) if isinstance(v, float) else v)
                           for k2, v in layer_roof.items()},
        "stage_us": {n: round(v * 1e3, 2) for n, v in stage_ms.items()},
        "stage_note": "each kernel as its own graph, %d replays with events between them" % Ks,
        "sweep": sweep,
        "e2e": e2e,
        "gpu_launches": K * moe.layer_kernel_count(
            T, H, F, E, k, "e4m3" if w.lowbit else "bf16", "f32" if w.lowbit else "bf16",
            "e2m1" if w.lowbit else "bf16"),
        "cpu_baseline": cpu,
        "device_error_word": code,
    }
    clocks = clk.summary()
    line["clocks"] = clocks
    if rank == 0:
        print(json.dumps(line), flush=True)
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
    d = W.make_inputs(w, T, seed=args.seed, device="cpu")
    dh = host_inputs(d)
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
        "config": {"workload": f"{w.name} MoE layer forward (H={w.H}, E={w.E}, k={w.k}, "
                               f"F={w.F}), T={T} tokens, random-init weights", "T": T},
        "cpu_baseline": {"value": round(value, 3), "unit": UNIT, "cores": oracle.num_threads(),
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": round(value, 3), "unit": UNIT, "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="qwen3")
    ap.add_argument("--T", type=int, default=4096)
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--no-sweep", action="store_true")
    ap.add_argument("--no-cpu", action="store_true")
    ap.add_argument("--cpu-tokens", type=int, default=0,
                    help="oracle sample size for cpu_baseline (0: about 15 s of CPU work)")
    ap.add_argument("--ref-tokens", type=int, default=32)
    args = ap.parse_args(argv)
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        if "--steps" not in (argv if argv is not None else sys.argv):
            args.steps = 5
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
