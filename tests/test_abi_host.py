"""Host-side checks of the C ABI (no GPU needed): the library loads, exports
every entry point include/moe.h declares, and rejects invalid arguments on the
host before launching anything."""
import ctypes
import os
import re

import pytest
import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    from router_experts_gb300 import build, moe
    build.build()
    return moe.load()


def declared_functions():
    src = open(os.path.join(ROOT, "include", "moe.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    names = re.findall(r"^\s*(?:const\s+)?\w+\s*\*?\s*(moe_\w+)\s*\(", src, flags=re.M)
    return sorted(set(names))


def test_header_declares_the_entry_points():
    names = declared_functions()
    for want in ["moe_router", "moe_align", "moe_expert_gemm1", "moe_expert_gemm2",
                 "moe_grouped_ffn", "moe_finalize", "moe_layer", "moe_read_device_error"]:
        assert want in names


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name


def test_status_strings(lib):
    assert lib.moe_status_string(0) == b"ok"
    assert lib.moe_status_string(1) == b"invalid argument"
    assert lib.moe_status_string(2) == b"unsupported combination"


def test_pick_block_m_rule(lib):
    # mean rows per expert T*k/E: < 8 -> 16, < 64 -> 64, else 128
    assert lib.moe_pick_block_m(1, 8, 128) == 16
    assert lib.moe_pick_block_m(64, 8, 128) == 16
    assert lib.moe_pick_block_m(128, 8, 128) == 64
    assert lib.moe_pick_block_m(512, 8, 128) == 64
    assert lib.moe_pick_block_m(1024, 8, 128) == 128
    assert lib.moe_pick_block_m(256, 8, 256) == 64
    assert lib.moe_pick_block_m(4096, 8, 256) == 128


def test_workspace_sizes_grow_with_shape(lib):
    a = lib.moe_layer_workspace_bytes(1, 2048, 768, 128, 8, 0, 0)
    b = lib.moe_layer_workspace_bytes(4096, 2048, 768, 128, 8, 0, 0)
    assert 0 < a < b
    assert lib.moe_layer_workspace_bytes(16, 64, 32, 8, 2, 33, 0) == 0  # bad block_m
    assert lib.moe_router_workspace_bytes(1, 4096, 288) > 0
    assert lib.moe_align_workspace_bytes() > 0


# The validation tests below pass placeholder addresses that host checks must
# reject; they are CPU tests and never run where a CUDA device is present.
no_device = pytest.mark.skipif(torch.cuda.is_available(),
                               reason="placeholder pointers: host-only test")


def call_router(lib, T=4, H=64, E=8, k=2, scoring=0, n_group=1, topk_group=1, hidden_dt=0,
                gate_dt=0, hidden=1 << 12, gate=1 << 12, ws=1 << 12, ws_bytes=1 << 30):
    P = ctypes.c_void_p
    return lib.moe_router(P(hidden), hidden_dt, None, P(gate), gate_dt, None, T, H, E, k, scoring,
                          n_group, topk_group, 1, ctypes.c_float(1.0), P(1 << 12), P(1 << 12),
                          P(ws), ws_bytes, None)


@no_device
def test_router_rejects_bad_arguments_without_launching(lib):
    # these all fail host validation, so no device pointer is touched
    assert call_router(lib, k=9) == 1             # k > E
    assert call_router(lib, H=48) == 1            # H % 32
    assert call_router(lib, E=513, k=2) == 1      # E > 512
    assert call_router(lib, n_group=3) == 1       # E % n_group
    assert call_router(lib, E=8, k=4, n_group=4, topk_group=1) == 1  # too few experts kept
    assert call_router(lib, scoring=5) == 1
    assert call_router(lib, hidden_dt=3) == 2     # e2m1 hidden: unsupported
    assert call_router(lib, gate_dt=2) == 2
    assert call_router(lib, hidden=(1 << 12) + 2) == 1  # misaligned
    assert call_router(lib, T=0) == 0             # T = 0 is a no-op


@no_device
def test_align_and_ffn_reject_bad_arguments(lib):
    P = ctypes.c_void_p
    # capacity below T*k + E*(BM-1)
    rc = lib.moe_align(P(4096), 4, 2, 8, 16, P(4096), 8 + 8 * 15 - 1, P(4096), P(4096), P(4096),
                       1 << 20, None)
    assert rc == 1
    rc = lib.moe_align(P(4096), 4, 2, 8, 32, P(4096), 1000, P(4096), P(4096), P(4096), 1 << 20,
                       None)
    assert rc == 1  # block_m not in {16, 64, 128}
    # H not a multiple of 64
    rc = lib.moe_expert_gemm1(P(4096), 0, None, P(4096), None, 0, 4, 96, 32, 8, 2, 16, P(4096),
                              P(4096), P(4096), 200, P(4096), None, P(4096), 1 << 30, None)
    assert rc == 1
    # mixed bf16 activations with fp4 weights: unsupported
    rc = lib.moe_expert_gemm1(P(4096), 0, None, P(4096), None, 3, 4, 64, 32, 8, 2, 16, P(4096),
                              P(4096), P(4096), 200, P(4096), None, P(4096), 1 << 30, None)
    assert rc == 2
    assert lib.moe_finalize(P(4096), 4, 2, 60, P(4096), None) == 1  # H % 8
    assert lib.moe_finalize(P(4096), 0, 2, 64, P(4096), None) == 0  # T = 0


def call_layer(lib, T=4, H=64, F=32, E=8, k=2, act_dt=0, gate_dt=0, w_dt=0, block_m=16,
               out=1 << 12, ws=1 << 12, ws_bytes=1 << 30, hidden=1 << 12):
    P = ctypes.c_void_p
    return lib.moe_layer(P(hidden), act_dt, None, P(1 << 12), gate_dt, None, P(1 << 12), None,
                         P(1 << 12), None, w_dt, T, H, F, E, k, 0, 1, 1, 1, ctypes.c_float(1.0),
                         block_m, P(out) if out else None, P(ws), ws_bytes, None)


@no_device
def test_layer_and_cast_reject_bad_arguments(lib):
    # every case fails host validation before anything is launched
    assert call_layer(lib, k=9) == 1              # k > E
    assert call_layer(lib, block_m=32) == 1       # tile height not in {16, 64, 128}
    assert call_layer(lib, H=96) == 1             # H % 64 for the expert GEMMs
    assert call_layer(lib, F=48) == 1             # F % 32
    assert call_layer(lib, ws_bytes=1024) == 1    # workspace too small
    assert call_layer(lib, ws=(1 << 12) + 8) == 1  # workspace not 256-byte aligned
    assert call_layer(lib, out=0) == 1            # no output
    assert call_layer(lib, w_dt=3) == 1           # e2m1 experts need H, F % 128
    assert call_layer(lib, act_dt=1) == 2         # fp32 activations into the expert GEMMs
    assert call_layer(lib, T=0) == 0              # T = 0 is a no-op
    P = ctypes.c_void_p
    assert lib.moe_cast_e4m3(P(1 << 12), 4, 48, P(1 << 12), P(1 << 12), None) == 1  # H % 32
    assert lib.moe_cast_e4m3(P(1 << 12), -1, 64, P(1 << 12), P(1 << 12), None) == 1
    assert lib.moe_cast_e4m3(P((1 << 12) + 2), 4, 64, P(1 << 12), P(1 << 12), None) == 1
    assert lib.moe_cast_e4m3(P(1 << 12), 0, 64, P(1 << 12), P(1 << 12), None) == 0


def test_layer_kernel_count(lib):
    # router launches (bf16 hidden and gate: the gate GEMM, whose last CTA
    # selects up to 4 tokens, then a selection kernel above that; one below 8
    # tokens for an fp32 gate; + a conversion for e4m3 hidden with an fp32
    # gate; one for more experts than the tensor-core router covers), align
    # except for one token (single-assignment blocks), GEMM1, GEMM2, finalize
    assert lib.moe_layer_kernel_count(1, 2048, 768, 128, 8, 0, 0, 0) == 4
    assert lib.moe_layer_kernel_count(2, 2048, 768, 128, 8, 0, 0, 0) == 5
    assert lib.moe_layer_kernel_count(4, 2048, 768, 128, 8, 0, 0, 0) == 5
    assert lib.moe_layer_kernel_count(5, 2048, 768, 128, 8, 0, 0, 0) == 6
    assert lib.moe_layer_kernel_count(4096, 2048, 768, 128, 8, 0, 0, 0) == 6
    assert lib.moe_router_kernel_count(4, 2048, 128, 0, 0) == 1
    assert lib.moe_router_kernel_count(5, 2048, 128, 0, 0) == 2
    # (an e4m3 hidden with e2m1 experts: + the permutation of its rows)
    assert lib.moe_layer_kernel_count(1, 4096, 2048, 256, 6, 2, 1, 3) == 5
    assert lib.moe_layer_kernel_count(8, 4096, 2048, 256, 6, 2, 1, 3) == 8
    assert lib.moe_layer_kernel_count(4096, 4096, 2048, 256, 6, 2, 1, 3) == 8
    assert lib.moe_layer_kernel_count(1, 2048, 768, 640, 8, 0, 0, 0) == 4
    assert lib.moe_layer_kernel_count(0, 2048, 768, 128, 8, 0, 0, 0) == 0
    # a bf16 hidden with e2m1 experts: the FP8 cast rides in the router's
    # selection launch (no launch of its own)
    assert lib.moe_layer_kernel_count(4096, 4096, 2048, 256, 6, 0, 1, 3) == 7


def test_binding_refuses_host_tensors():
    # every tensor is handed to the kernels as a device address: a host tensor
    # is refused in the binding instead of reaching a kernel
    import torch
    from router_experts_gb300 import moe
    with pytest.raises(ValueError, match="CUDA tensor"):
        moe._p(torch.zeros((4, 64), dtype=torch.bfloat16))
    assert moe._p(None) is None


def test_header_offsets_match_the_binding():
    # the workspace header words a test may set, as moe.h defines them
    from router_experts_gb300 import moe
    src = open(os.path.join(ROOT, "include", "moe.h")).read()
    defs = dict(re.findall(r"#define\s+(MOE_WS_\w+)\s+(\d+)", src))
    assert int(defs["MOE_WS_ALIGN_BARRIER_OFFSET"]) == moe.WS_ALIGN_BARRIER_OFFSET
    assert int(defs["MOE_WS_WAIT_LIMIT_OFFSET"]) == moe.WS_WAIT_LIMIT_OFFSET


def test_probe_arguments_rejected_on_host(lib):
    lib.moe_probe_empty.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_void_p]
    lib.moe_probe_read.argtypes = [ctypes.c_void_p, ctypes.c_size_t, ctypes.c_void_p,
                                   ctypes.c_void_p]
    assert lib.moe_probe_empty(0, 512, None) == 1
    assert lib.moe_probe_empty(1, 1024, None) == 1
    assert lib.moe_probe_read(None, 4096, None, None) == 1
    # a size that is not a whole number of 16-byte loads
    assert lib.moe_probe_read(ctypes.c_void_p(256), 4008, ctypes.c_void_p(512), None) == 1


def test_persistent_layer_limits_checked_on_host(lib):
    P, I = ctypes.c_void_p, ctypes.c_int
    lib.moe_layer_persistent_workspace_bytes.restype = ctypes.c_size_t
    lib.moe_layer_persistent_workspace_bytes.argtypes = [I, I, I, I, I]
    fn = lib.moe_layer_persistent
    fn.restype = I
    fn.argtypes = [P, P, P, P, P, I, I, I, I, I, I, I, I, I, ctypes.c_float, P, P, P, P,
                   ctypes.c_size_t, P]
    # Qwen3 shapes: up to 64 tokens (T*k <= 512); F and H whole 64-wide K steps
    assert lib.moe_layer_persistent_workspace_bytes(64, 2048, 768, 128, 8) > 0
    assert lib.moe_layer_persistent_workspace_bytes(65, 2048, 768, 128, 8) == 0
    assert lib.moe_layer_persistent_workspace_bytes(4, 2048, 96, 128, 8) == 0
    assert lib.moe_layer_persistent_workspace_bytes(4, 2048, 768, 640, 8) == 0
    a = P(1 << 12)
    big = ctypes.c_size_t(1 << 40)
    # nothing is launched for invalid arguments (the pointers are never read)
    assert fn(a, a, None, a, a, 65, 2048, 768, 128, 8, 0, 1, 1, 1, 1.0, a, None, None, a, big,
              None) == 1
    assert fn(a, a, None, a, a, 4, 2048, 96, 128, 8, 0, 1, 1, 1, 1.0, a, None, None, a, big,
              None) == 1
    # ids without weights
    assert fn(a, a, None, a, a, 4, 2048, 768, 128, 8, 0, 1, 1, 1, 1.0, a, a, None, a, big,
              None) == 1
    assert fn(a, a, None, a, a, 0, 2048, 768, 128, 8, 0, 1, 1, 1, 1.0, a, None, None, a, big,
              None) == 0
