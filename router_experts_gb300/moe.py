"""Python binding of the C ABI in ``include/moe.h`` (argument marshalling only).

Every step runs in the CUDA library ``libmoe.so``; this module passes torch
tensors' device pointers and sizes through ctypes and raises on any non-zero
status.  There is no fallback: if the library is not built, every call raises.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "_build", "libmoe.so")

MOE_OK, MOE_ERR_ARG, MOE_ERR_UNSUPPORTED, MOE_ERR_CUDA, MOE_ERR_DEVICE = 0, 1, 2, 3, 4
SOFTMAX, SIGMOID, SQRT_SOFTPLUS = 0, 1, 2
SCORING = {"softmax": SOFTMAX, "sigmoid": SIGMOID, "sqrt_softplus": SQRT_SOFTPLUS}
DT_BF16, DT_F32, DT_E4M3, DT_E2M1 = 0, 1, 2, 3
DEVERR_BAD_EXPERT_ID, DEVERR_WAIT_TIMEOUT, DEVERR_BAD_TABLE = 1, 2, 4
# workspace header words a test may set (include/moe.h)
WS_ALIGN_BARRIER_OFFSET, WS_WAIT_LIMIT_OFFSET = 5120, 5376

_lock = threading.Lock()
_lib = None


class MoeError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        lib = load()
        msg = lib.moe_status_string(status).decode()
        cuda = lib.moe_last_cuda_error_string().decode()
        super().__init__(f"{where}: {msg}" + (f" ({cuda})" if cuda and status == MOE_ERR_CUDA else ""))


def load():
    """Load libmoe.so (raises if it has not been built)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"CUDA library not built: {LIB_PATH} is missing "
                               "(run router_experts_gb300.build.build())")
        lib = ctypes.CDLL(LIB_PATH)
        P, I, I64, F, SZ = (ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_float,
                            ctypes.c_size_t)
        sig = {
            "moe_router_workspace_bytes": (SZ, [I, I, I]),
            "moe_router_cast_e4m3": (I, [P, P, I, P, I, I, I, I, I, I, I, I, F, P, P, P, P, P, SZ,
                                         P]),
            "moe_router_kernel_count": (I, [I, I, I, I, I]),
            "moe_layer_kernel_count": (I, [I, I, I, I, I, I, I, I]),
            "moe_cast_e4m3": (I, [P, I, I, P, P, P]),
            "moe_router": (I, [P, I, P, P, I, P, I, I, I, I, I, I, I, I, F, P, P, P, SZ, P]),
            "moe_align_workspace_bytes": (SZ, []),
            "moe_align": (I, [P, I, I, I, I, P, I64, P, P, P, SZ, P]),
            "moe_ffn_workspace_bytes": (SZ, [I, I, I, I, I, I, I]),
            "moe_expert_gemm1": (I, [P, I, P, P, P, I, I, I, I, I, I, I, P, P, P, I64, P, P, P, SZ,
                                     P]),
            "moe_expert_gemm2": (I, [P, P, I, P, P, I, I, I, I, I, I, I, P, P, P, I64, P, P, P, SZ,
                                     P]),
            "moe_grouped_ffn": (I, [P, P, I, P, P, P, P, I, I, I, I, I, I, I, P, P, P, I64, P, P, P,
                                    SZ, P]),
            "moe_finalize": (I, [P, I, I, I, P, P]),
            "moe_layer_workspace_bytes": (SZ, [I, I, I, I, I, I, I]),
            "moe_layer": (I, [P, I, P, P, I, P, P, P, P, P, I, I, I, I, I, I, I, I, I, I, F, I, P, P,
                              SZ, P]),
            "moe_pick_block_m": (I, [I, I, I]),
            "moe_layer_persistent_workspace_bytes": (SZ, [I, I, I, I, I]),
            "moe_layer_persistent": (I, [P, P, P, P, P, I, I, I, I, I, I, I, I, I, F, P, P, P, P,
                                         SZ, P]),
            "moe_probe_empty": (I, [I, I, P]),
            "moe_probe_read": (I, [P, SZ, P, P]),
            "moe_workspace_init": (I, [P, SZ, P]),
            "moe_read_device_error": (I, [P, P, I, P]),
            "moe_status_string": (ctypes.c_char_p, [I]),
            "moe_last_cuda_error_string": (ctypes.c_char_p, []),
        }
        for name, (res, args) in sig.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _lib = lib
        return lib


def _p(t):
    """Device pointer of a tensor argument.  The library reads every tensor as
    a dense row-major CUDA buffer, so anything else is refused here instead of
    reaching a kernel as a host address or in the wrong layout."""
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError(f"expected a CUDA tensor, got one on {t.device}")
    if not t.is_contiguous():
        raise ValueError(f"expected a contiguous tensor, got strides {t.stride()}")
    return ctypes.c_void_p(t.data_ptr())


def _stream(device=None):
    return ctypes.c_void_p(torch.cuda.current_stream(device).cuda_stream)


def _check(rc: int, where: str):
    if rc != MOE_OK:
        raise MoeError(rc, where)


def _dt(t: torch.Tensor, scale) -> int:
    if t.dtype == torch.bfloat16:
        return DT_BF16
    if t.dtype == torch.float32:
        return DT_F32
    if t.dtype in (torch.uint8, torch.float8_e4m3fn) and scale is not None:
        return DT_E4M3
    raise ValueError(f"unsupported dtype {t.dtype}")


class Workspace:
    """A device workspace, zeroed when (re)allocated, reused across calls."""

    def __init__(self, device=None):
        self.device = torch.device(device or "cuda")
        self.buf = None

    def get(self, nbytes: int) -> torch.Tensor:
        nbytes = max(int(nbytes), 1)
        if self.buf is None or self.buf.numel() < nbytes:
            self.buf = None
            self.buf = torch.zeros(nbytes, dtype=torch.uint8, device=self.device)
        return self.buf


_default_ws = {}


def default_workspace(device) -> Workspace:
    d = torch.device(device)
    key = (d.type, d.index if d.index is not None else torch.cuda.current_device())
    if key not in _default_ws:
        _default_ws[key] = Workspace(torch.device(key[0], key[1]))
    return _default_ws[key]


def read_device_error(ws: torch.Tensor, clear: bool = True) -> int:
    """Synchronising read of the sticky device error word."""
    code = ctypes.c_int32(0)
    rc = load().moe_read_device_error(_p(ws), ctypes.byref(code), int(clear), _stream(ws.device))
    if rc not in (MOE_OK, MOE_ERR_DEVICE):
        _check(rc, "moe_read_device_error")
    return int(code.value)


def pick_block_m(T: int, k: int, E: int) -> int:
    return int(load().moe_pick_block_m(T, k, E))


def router_kernel_count(T: int, H: int, E: int, hidden_dtype="bf16", gate_dtype="bf16") -> int:
    """Kernels moe_router enqueues for these shapes and types."""
    dt = {"bf16": DT_BF16, "f32": DT_F32, "e4m3": DT_E4M3}
    return int(load().moe_router_kernel_count(T, H, E, dt[hidden_dtype], dt[gate_dtype]))


def layer_kernel_count(T: int, H: int, F: int, E: int, k: int, act_dtype="bf16",
                       gate_dtype="bf16", weight_dtype="bf16") -> int:
    """Kernels moe_layer enqueues for these shapes and types."""
    dt = {"bf16": DT_BF16, "f32": DT_F32, "e4m3": DT_E4M3, "e2m1": DT_E2M1}
    return int(load().moe_layer_kernel_count(T, H, F, E, k, dt[act_dtype], dt[gate_dtype],
                                             dt[weight_dtype]))


def cast_e4m3(x):
    """bf16 [T, H] -> (e4m3 codes [T, H] uint8, UE8M0 scale bytes [T, H/32] uint8)."""
    lib = load()
    T, H = x.shape
    codes = torch.empty((T, H), dtype=torch.uint8, device=x.device)
    scales = torch.empty((T, H // 32), dtype=torch.uint8, device=x.device)
    _check(lib.moe_cast_e4m3(_p(x), T, H, _p(codes), _p(scales), _stream(x.device)),
           "moe_cast_e4m3")
    return codes, scales


def probe_empty(blocks: int = 1, threads: int = 512, device=None):
    """Enqueue an empty kernel (the launch part of a router's floor)."""
    _check(load().moe_probe_empty(int(blocks), int(threads), _stream(device)), "moe_probe_empty")


def probe_read(t: torch.Tensor, sink: torch.Tensor):
    """Enqueue a kernel whose threads each load 16 bytes of t (the whole
    tensor once): the cold-read part of a router's floor."""
    _check(load().moe_probe_read(_p(t), t.numel() * t.element_size(), _p(sink),
                                 _stream(t.device)), "moe_probe_read")


# ---- entry points ---------------------------------------------------------------

def router(hidden, gate, bias, k, scoring="softmax", n_group=1, topk_group=1, renormalize=True,
           scaling=1.0, hidden_scale=None, ws: Workspace | None = None, out=None):
    """-> (topk_ids [T,k] int32, topk_weights [T,k] float32)."""
    lib = load()
    T, H = hidden.shape
    E = gate.shape[0]
    dev = hidden.device
    ids, wts = out if out is not None else (
        torch.empty((T, k), dtype=torch.int32, device=dev),
        torch.empty((T, k), dtype=torch.float32, device=dev))
    ws = ws or default_workspace(dev)
    buf = ws.get(lib.moe_router_workspace_bytes(T, H, E))
    rc = lib.moe_router(_p(hidden), _dt(hidden, hidden_scale), _p(hidden_scale), _p(gate),
                        _dt(gate, None), _p(bias), T, H, E, k,
                        SCORING[scoring], n_group, topk_group,
                        int(bool(renormalize)), float(scaling), _p(ids), _p(wts), _p(buf),
                        buf.numel(), _stream(dev))
    _check(rc, "moe_router")
    return ids, wts


def router_cast_e4m3(hidden, gate, bias, k, scoring="softmax", n_group=1, topk_group=1,
                     renormalize=True, scaling=1.0, ws: Workspace | None = None):
    """Router on a bf16 hidden that also writes its FP8 cast -> (topk_ids [T,k]
    int32, topk_weights [T,k] float32, e4m3 codes [T,H] uint8, UE8M0 scales
    [T,H/32] uint8)."""
    lib = load()
    T, H = hidden.shape
    E = gate.shape[0]
    dev = hidden.device
    ids = torch.empty((T, k), dtype=torch.int32, device=dev)
    wts = torch.empty((T, k), dtype=torch.float32, device=dev)
    codes = torch.empty((T, H), dtype=torch.uint8, device=dev)
    scales = torch.empty((T, H // 32), dtype=torch.uint8, device=dev)
    ws = ws or default_workspace(dev)
    buf = ws.get(lib.moe_router_workspace_bytes(T, H, E))
    rc = lib.moe_router_cast_e4m3(_p(hidden), _p(gate), _dt(gate, None), _p(bias), T, H, E, k,
                                  SCORING[scoring], n_group, topk_group, int(bool(renormalize)),
                                  float(scaling), _p(ids), _p(wts), _p(codes), _p(scales),
                                  _p(buf), buf.numel(), _stream(dev))
    _check(rc, "moe_router_cast_e4m3")
    return ids, wts, codes, scales


def align(topk_ids, E, block_m, cap_rows=None, ws: Workspace | None = None):
    """-> (sorted_ids [cap], block_expert [ceil(cap/BM)], num_post_padded [1]) int32."""
    lib = load()
    T, k = topk_ids.shape
    dev = topk_ids.device
    cap = T * k + E * (block_m - 1) if cap_rows is None else int(cap_rows)
    sorted_ids = torch.empty((cap,), dtype=torch.int32, device=dev)
    block_expert = torch.empty(((cap + block_m - 1) // block_m,), dtype=torch.int32, device=dev)
    npp = torch.empty((1,), dtype=torch.int32, device=dev)
    ws = ws or default_workspace(dev)
    buf = ws.get(lib.moe_align_workspace_bytes())
    rc = lib.moe_align(_p(topk_ids), T, k, E, block_m, _p(sorted_ids), cap, _p(block_expert),
                       _p(npp), _p(buf), buf.numel(), _stream(dev))
    _check(rc, "moe_align")
    return sorted_ids, block_expert, npp


def _wdt(w):
    return DT_BF16 if w.dtype == torch.bfloat16 else DT_E2M1


def _is_lowbit(w):
    return w.dtype == torch.uint8


def expert_gemm1(x, w13, block_m, sorted_ids, block_expert, npp, k, cap_rows=None,
                 ws: Workspace | None = None, x_scale=None, w13_scale=None):
    """bf16: -> inter [cap, F] bf16.  Low-bit (uint8 e4m3 x with x_scale, packed
    e2m1 w13 with w13_scale): -> (inter codes [cap, F] uint8, scales [cap, F/32])."""
    lib = load()
    T, H = x.shape
    E, F2, _ = w13.shape
    F = F2 // 2
    cap = sorted_ids.numel() if cap_rows is None else int(cap_rows)
    act_dt = _dt(x, x_scale)
    ws = ws or default_workspace(x.device)
    buf = ws.get(lib.moe_ffn_workspace_bytes(T, H, F, E, k, block_m, act_dt))
    if act_dt == DT_E4M3:
        inter = torch.empty((cap, F), dtype=torch.uint8, device=x.device)
        isc = torch.empty((cap, F // 32), dtype=torch.uint8, device=x.device)
    else:
        inter = torch.empty((cap, F), dtype=torch.bfloat16, device=x.device)
        isc = None
    rc = lib.moe_expert_gemm1(_p(x), act_dt, _p(x_scale), _p(w13), _p(w13_scale), _wdt(w13), T, H,
                              F, E, k, block_m, _p(sorted_ids), _p(block_expert), _p(npp), cap,
                              _p(inter), _p(isc), _p(buf), buf.numel(), _stream(x.device))
    _check(rc, "moe_expert_gemm1")
    return (inter, isc) if act_dt == DT_E4M3 else inter


def expert_gemm2(inter, w2, T, k, block_m, sorted_ids, block_expert, npp, topk_weights,
                 ws: Workspace | None = None, inter_scale=None, w2_scale=None):
    """-> stage [T*k, H] bf16 (rows weighted by topk_weights)."""
    lib = load()
    E, H, Fw = w2.shape
    F = Fw * 2 if _is_lowbit(w2) else Fw
    cap = inter.shape[0]
    act_dt = DT_E4M3 if inter_scale is not None else DT_BF16
    stage = torch.empty((T * k, H), dtype=torch.bfloat16, device=inter.device)
    ws = ws or default_workspace(inter.device)
    buf = ws.get(lib.moe_ffn_workspace_bytes(T, H, F, E, k, block_m, act_dt))
    rc = lib.moe_expert_gemm2(_p(inter), _p(inter_scale), act_dt, _p(w2), _p(w2_scale), _wdt(w2),
                              T, H, F, E, k, block_m, _p(sorted_ids), _p(block_expert), _p(npp),
                              cap, _p(topk_weights), _p(stage), _p(buf), buf.numel(),
                              _stream(inter.device))
    _check(rc, "moe_expert_gemm2")
    return stage


def grouped_ffn(x, w13, w2, k, block_m, sorted_ids, block_expert, npp, topk_weights,
                ws: Workspace | None = None, x_scale=None, w13_scale=None, w2_scale=None):
    """GEMM1 + SwiGLU and GEMM2 + weight -> stage [T*k, H] bf16."""
    lib = load()
    T, H = x.shape
    E, F2, _ = w13.shape
    F = F2 // 2
    cap = sorted_ids.numel()
    act_dt = _dt(x, x_scale)
    stage = torch.empty((T * k, H), dtype=torch.bfloat16, device=x.device)
    ws = ws or default_workspace(x.device)
    buf = ws.get(lib.moe_ffn_workspace_bytes(T, H, F, E, k, block_m, act_dt))
    rc = lib.moe_grouped_ffn(_p(x), _p(x_scale), act_dt, _p(w13), _p(w13_scale), _p(w2),
                             _p(w2_scale), _wdt(w13), T, H, F, E, k, block_m, _p(sorted_ids),
                             _p(block_expert), _p(npp), cap, _p(topk_weights), _p(stage),
                             _p(buf), buf.numel(), _stream(x.device))
    _check(rc, "moe_grouped_ffn")
    return stage


def finalize(stage, T, k, out=None):
    """stage [T*k, H] bf16 -> out [T, H] bf16."""
    lib = load()
    H = stage.shape[1]
    out = torch.empty((T, H), dtype=torch.bfloat16, device=stage.device) if out is None else out
    rc = lib.moe_finalize(_p(stage), T, k, H, _p(out), _stream(stage.device))
    _check(rc, "moe_finalize")
    return out


def layer_workspace_bytes(T, H, F, E, k, block_m=0, act_dt=DT_BF16) -> int:
    return int(load().moe_layer_workspace_bytes(T, H, F, E, k, block_m, act_dt))


def layer(hidden, gate, bias, w13, w2, k, scoring="softmax", n_group=1, topk_group=1,
          renormalize=True, scaling=1.0, block_m=0, hidden_scale=None, w13_scale=None,
          w2_scale=None, ws: Workspace | None = None, out=None):
    """The whole MoE layer forward -> out [T, H] bf16."""
    lib = load()
    T = hidden.shape[0]
    E, H = gate.shape
    F = w2.shape[2] * (2 if _is_lowbit(w2) else 1)
    act_dt = _dt(hidden, hidden_scale)
    dev = hidden.device
    out = torch.empty((T, H), dtype=torch.bfloat16, device=dev) if out is None else out
    ws = ws or default_workspace(dev)
    buf = ws.get(lib.moe_layer_workspace_bytes(T, H, F, E, k, block_m, act_dt))
    rc = lib.moe_layer(_p(hidden), act_dt, _p(hidden_scale), _p(gate), _dt(gate, None), _p(bias),
                       _p(w13), _p(w13_scale), _p(w2), _p(w2_scale), _wdt(w13), T, H, F, E, k,
                       SCORING[scoring], n_group, topk_group,
                       int(bool(renormalize)), float(scaling), block_m, _p(out), _p(buf),
                       buf.numel(), _stream(dev))
    _check(rc, "moe_layer")
    return out


def layer_persistent_workspace_bytes(T, H, F, E, k) -> int:
    return int(load().moe_layer_persistent_workspace_bytes(T, H, F, E, k))


def layer_persistent(hidden, gate, bias, w13, w2, k, scoring="softmax", n_group=1, topk_group=1,
                     renormalize=True, scaling=1.0, ws: Workspace | None = None, out=None,
                     routing=None):
    """The whole layer in one persistent kernel (small batches, bf16) -> out
    [T, H] bf16.  routing=(topk_ids [T,k] int32, topk_weights [T,k] f32): also
    keep the router's selection there."""
    lib = load()
    T, H = hidden.shape
    E = gate.shape[0]
    F = w2.shape[2]
    dev = hidden.device
    out = torch.empty((T, H), dtype=torch.bfloat16, device=dev) if out is None else out
    if T == 0:
        return out
    need = lib.moe_layer_persistent_workspace_bytes(T, H, F, E, k)
    if need == 0:
        raise MoeError(MOE_ERR_ARG, "moe_layer_persistent_workspace_bytes")
    ws = ws or default_workspace(dev)
    buf = ws.get(need)
    ids, wts = routing if routing is not None else (None, None)
    rc = lib.moe_layer_persistent(_p(hidden), _p(gate), _p(bias), _p(w13), _p(w2), T, H, F, E, k,
                                  SCORING[scoring], n_group, topk_group, int(bool(renormalize)),
                                  float(scaling), _p(out), _p(ids), _p(wts), _p(buf), buf.numel(),
                                  _stream(dev))
    _check(rc, "moe_layer_persistent")
    return out
