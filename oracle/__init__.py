"""CPU oracle of the single-GPU MoE layer forward -- TEST INFRASTRUCTURE.

Only ``tests/``, ``__graft_entry__.smoke()`` and the ``cpu_baseline`` /
``--impl reference`` legs of ``bench.py`` may import this package.  The
product path (``router_experts_gb300``) never imports it and shares no code
with it: the oracle is plain C (``moe_oracle.c``) in double precision that
decodes its own input formats, wrapped here with ctypes and numpy.

Every function follows a passage of the pages (cited in ``moe_oracle.c``):
  * router     -- "How an MoE Model Picks Its Experts During LLM Inference"
                  §1 (rank key vs weight, Fig. 3), §4 (reference router),
                  §5.3 (k rounds, lowest id wins); "Mixture of Experts"
                  (grouped, bias-corrected routing; routed scaling factor).
  * align      -- "MoE Kernels, in depth", "Alignment: making ragged routing
                  tileable"; "Mixture of Experts", worked moe_align example.
  * expert FFN -- "MoE Kernels, in depth" (naive per-expert loop, SwiGLU on
                  the fused gate/up matrix); "How GPUs Fuse Communication and
                  Computation During LLM Inference" §1.1 and §3.5.
The whole layer has no printed end-to-end value on the pages; its composition
(router -> experts -> weighted combine) is pinned by hand-derived closed-form
cases in ``tests/test_oracle_layer.py`` (grouped sigmoid routing with a bias,
renormalisation and scaling; softmax routing with and without
renormalisation).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "moe_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "libmoe_oracle.so")
_lock = threading.Lock()
_lib = None

DT = {"bf16": 0, "f32": 1, "e4m3": 2, "e2m1": 3}


def build(force: bool = False) -> str:
    """Compile moe_oracle.c with the host C compiler (portable C, OpenMP)."""
    os.makedirs(_BUILD, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".{os.getpid()}.tmp"
    subprocess.check_call(["gcc", "-O2", "-std=c11", "-fopenmp", "-fPIC", "-shared",
                           "-o", tmp, _SRC, "-lm"])
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB_PATH)
            P = ctypes.c_void_p
            i32, i64, f64 = ctypes.c_int, ctypes.c_int64, ctypes.c_double
            lib.orc_bf16_to_double.restype = f64
            lib.orc_bf16_to_double.argtypes = [ctypes.c_uint16]
            lib.orc_e4m3_to_double.restype = f64
            lib.orc_e4m3_to_double.argtypes = [ctypes.c_uint8]
            lib.orc_e2m1_to_double.restype = f64
            lib.orc_e2m1_to_double.argtypes = [ctypes.c_uint8]
            lib.orc_ue8m0_to_double.restype = f64
            lib.orc_ue8m0_to_double.argtypes = [ctypes.c_uint8]
            lib.orc_round_bf16.restype = f64
            lib.orc_round_bf16.argtypes = [f64]
            lib.orc_round_e4m3.restype = f64
            lib.orc_round_e4m3.argtypes = [f64]
            lib.orc_decode.restype = None
            lib.orc_decode.argtypes = [P, i32, P, i64, i64, i64, P]
            lib.orc_router.restype = i32
            lib.orc_router.argtypes = [P, i32, P, P, i32, P, i32, i32, i32, i32, i32, i32, i32,
                                       i32, f64, P, i32, P, P, P, P]
            lib.orc_align.restype = i32
            lib.orc_align.argtypes = [P, i32, i32, i32, i32, i64, P, P, P]
            lib.orc_expert_ffn.restype = None
            lib.orc_expert_ffn.argtypes = [P, P, P, P, P, i32, i32, i32, i32, i32, P]
            lib.orc_moe_ffn.restype = i32
            lib.orc_moe_ffn.argtypes = [P, i32, P, P, P, P, P, i32, i32, i32, i32, i32, i32,
                                        P, P, P, i32, i32, P]
            lib.orc_quantize_e4m3.restype = i32
            lib.orc_quantize_e4m3.argtypes = [P, i32, i32, i32, P, P]
            lib.orc_num_threads.restype = i32
            lib.orc_num_threads.argtypes = []
            _lib = lib
    return _lib


def _ptr(a):
    return None if a is None else ctypes.c_void_p(a.ctypes.data)


def _raw(a):
    """Raw little-endian bytes of a host array, kept C-contiguous."""
    return None if a is None else np.ascontiguousarray(a)


def num_threads() -> int:
    return int(_load().orc_num_threads())


# --- number formats ---------------------------------------------------------

def bf16_to_double(bits: int) -> float:
    return _load().orc_bf16_to_double(int(bits))


def e4m3_to_double(code: int) -> float:
    return _load().orc_e4m3_to_double(int(code))


def e2m1_to_double(nibble: int) -> float:
    return _load().orc_e2m1_to_double(int(nibble))


def ue8m0_to_double(code: int) -> float:
    return _load().orc_ue8m0_to_double(int(code))


def round_bf16(v: float) -> float:
    return _load().orc_round_bf16(float(v))


def round_e4m3(v: float) -> float:
    return _load().orc_round_e4m3(float(v))


def decode(raw: np.ndarray, dtype: str, rows: int, cols: int, scale=None) -> np.ndarray:
    """Decode a row-major [rows, cols] matrix held as raw bytes/words."""
    raw = _raw(raw)
    scale = _raw(scale)
    out = np.empty((rows, cols), dtype=np.float64)
    _load().orc_decode(_ptr(raw), DT[dtype], _ptr(scale), 0, rows, cols, _ptr(out))
    return out


# --- the method -------------------------------------------------------------

SCORING = {"softmax": 0, "sigmoid": 1, "sqrt_softplus": 2}


def router(x, x_dt, gate, gate_dt, bias, T, H, E, k, scoring, n_group=1, topk_group=1,
           renormalize=True, scaling=1.0, x_scale=None, tokens=None, want_logits=False):
    """Routing of the listed tokens. scoring: 'softmax' | 'sigmoid' | 'sqrt_softplus'.

    Returns (ids [n,k] int32, weights [n,k] f64, gap [n] f64[, logits [n,E]])."""
    lib = _load()
    x, gate, x_scale = _raw(x), _raw(gate), _raw(x_scale)
    b = None if bias is None else np.ascontiguousarray(bias, dtype=np.float32)
    tl = None if tokens is None else np.ascontiguousarray(tokens, dtype=np.int32)
    n = T if tl is None else len(tl)
    ids = np.empty((n, k), dtype=np.int32)
    w = np.empty((n, k), dtype=np.float64)
    gap = np.empty((n,), dtype=np.float64)
    logits = np.empty((n, E), dtype=np.float64) if want_logits else None
    rc = lib.orc_router(_ptr(x), DT[x_dt], _ptr(x_scale), _ptr(gate), DT[gate_dt], _ptr(b),
                        T, H, E, k, SCORING[scoring], n_group, topk_group,
                        int(bool(renormalize)), float(scaling), _ptr(tl), n, _ptr(ids), _ptr(w),
                        _ptr(logits), _ptr(gap))
    if rc != 0:
        raise ValueError("oracle router: invalid arguments")
    return (ids, w, gap, logits) if want_logits else (ids, w, gap)


def quantize_e4m3(x, x_dt, T, H):
    """FP8 cast of a [T, H] bf16 or f32 array: (codes [T, H] uint8, scale bytes
    [T, H/32] uint8), per 32 values the smallest 2^s with amax / 2^s <= 448."""
    x = _raw(x)
    codes = np.empty((T, H), dtype=np.uint8)
    scales = np.empty((T, H // 32), dtype=np.uint8)
    if _load().orc_quantize_e4m3(_ptr(x), DT[x_dt], T, H, _ptr(codes), _ptr(scales)) != 0:
        raise ValueError("oracle quantize_e4m3: invalid arguments")
    return codes, scales


def align(topk_ids, T, k, E, block_m, cap_rows=None):
    """Returns (sorted_ids [cap], block_expert [ceil(cap/BM)], num_post_padded)."""
    ids = np.ascontiguousarray(topk_ids, dtype=np.int32).reshape(-1)
    if cap_rows is None:
        cap_rows = T * k + E * (block_m - 1)
    sorted_ids = np.empty((cap_rows,), dtype=np.int32)
    block_expert = np.empty(((cap_rows + block_m - 1) // block_m,), dtype=np.int32)
    npp = np.zeros((1,), dtype=np.int32)
    rc = _load().orc_align(_ptr(ids), T, k, E, block_m, cap_rows, _ptr(sorted_ids),
                           _ptr(block_expert), _ptr(npp))
    if rc != 0:
        raise ValueError("oracle align: invalid arguments")
    return sorted_ids, block_expert, int(npp[0])


def expert_ffn(x_row, w13, w2, w_dt, H, F, e, w13_scale=None, w2_scale=None, emulate=0):
    """One expert on one decoded hidden row (float64 [H]) -> float64 [H]."""
    xr = np.ascontiguousarray(x_row, dtype=np.float64)
    w13, w2, w13_scale, w2_scale = _raw(w13), _raw(w2), _raw(w13_scale), _raw(w2_scale)
    out = np.empty((H,), dtype=np.float64)
    _load().orc_expert_ffn(_ptr(xr), _ptr(w13), _ptr(w13_scale), _ptr(w2), _ptr(w2_scale),
                           DT[w_dt], H, F, e, emulate, _ptr(out))
    return out


def moe_ffn(x, x_dt, w13, w2, w_dt, T, H, F, E, k, ids, weights, x_scale=None,
            w13_scale=None, w2_scale=None, tokens=None, emulate=0):
    """Naive per-expert loop + weighted sum for the listed tokens -> [n, H] f64."""
    x, w13, w2 = _raw(x), _raw(w13), _raw(w2)
    x_scale, w13_scale, w2_scale = _raw(x_scale), _raw(w13_scale), _raw(w2_scale)
    ids = np.ascontiguousarray(ids, dtype=np.int32)
    weights = np.ascontiguousarray(weights, dtype=np.float64)
    tl = None if tokens is None else np.ascontiguousarray(tokens, dtype=np.int32)
    n = T if tl is None else len(tl)
    y = np.empty((n, H), dtype=np.float64)
    rc = _load().orc_moe_ffn(_ptr(x), DT[x_dt], _ptr(x_scale), _ptr(w13), _ptr(w13_scale),
                             _ptr(w2), _ptr(w2_scale), DT[w_dt], T, H, F, E, k, _ptr(ids),
                             _ptr(weights), _ptr(tl), n, emulate, _ptr(y))
    if rc != 0:
        raise ValueError("oracle moe_ffn: invalid arguments")
    return y


def moe_layer(x, x_dt, gate, gate_dt, bias, w13, w2, w_dt, T, H, F, E, k, scoring,
              n_group=1, topk_group=1, renormalize=True, scaling=1.0, x_scale=None,
              router_x=None, router_x_dt=None, w13_scale=None, w2_scale=None, tokens=None,
              emulate=0):
    """Router + expert FFN + combine for the listed tokens.

    router_x/router_x_dt: the router's view of the hidden state when it differs
    from the experts' (the low-bit layer routes on the dequantised fp32 rows).
    Returns (y [n,H], ids [n,k], weights [n,k], gap [n])."""
    rx = x if router_x is None else router_x
    rdt = x_dt if router_x_dt is None else router_x_dt
    rsc = x_scale if router_x is None else None
    ids, w, gap = router(rx, rdt, gate, gate_dt, bias, T, H, E, k, scoring, n_group,
                         topk_group, renormalize, scaling, x_scale=rsc, tokens=tokens)
    # expand the listed tokens' routing into [T, k] tables for the FFN call
    tl = np.arange(T, dtype=np.int32) if tokens is None else np.asarray(tokens, dtype=np.int32)
    full_ids = np.zeros((T, k), dtype=np.int32)
    full_w = np.zeros((T, k), dtype=np.float64)
    full_ids[tl] = ids
    full_w[tl] = w
    y = moe_ffn(x, x_dt, w13, w2, w_dt, T, H, F, E, k, full_ids, full_w, x_scale=x_scale,
                w13_scale=w13_scale, w2_scale=w2_scale, tokens=tl, emulate=emulate)
    return y, ids, w, gap
