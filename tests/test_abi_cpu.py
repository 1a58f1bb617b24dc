"""The C ABI library builds, loads and exports every declared symbol; host-side
argument validation answers before any device work (no GPU needed)."""
import ctypes
import glob
import os
import re

import pytest

import __graft_entry__
from nvfp4_mixture_experts_moe_gb300 import binding as B

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    __graft_entry__.build()
    return B.lib()


def declared_functions():
    names = set()
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        text = open(h).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        for m in re.finditer(r"\b(moe_\w+)\s*\(", text):
            names.add(m.group(1))
    return sorted(names)


def test_every_declared_symbol_is_exported(lib):
    names = declared_functions()
    assert "moe_nvfp4_forward" in names and len(names) >= 15
    for n in names:
        assert hasattr(lib, n), n
        assert ctypes.cast(getattr(lib, n), ctypes.c_void_p).value


def test_status_strings(lib):
    assert B.status_string(0) == "MOE_OK"
    assert B.status_string(6) == "MOE_ERR_DEVICE"


def test_host_validation_before_device_work(lib):
    L = lib
    assert L.moe_route_topk(None, 4, 0, 1, None, None, None) == B.MOE_ERR_INVALID_ARG
    assert L.moe_route_topk(None, 4, 8, 9, None, None, None) == B.MOE_ERR_UNSUPPORTED
    assert L.moe_route_topk(None, 4, 2048, 2, None, None, None) == B.MOE_ERR_UNSUPPORTED
    assert L.moe_route_topk(None, 0, 8, 2, None, None, None) == B.MOE_OK  # empty batch: no-op
    assert L.moe_permute(256, 4, 2, 8, 256, 256, 256, 256, None, 0, None) == B.MOE_ERR_WORKSPACE
    assert L.moe_permute(256, 4, 2, 8, 256, 256, 256, 256, 256 * 3, 0, None) == B.MOE_ERR_WORKSPACE
    # a zero or non-finite global scale is refused (it would silently zero an expert)
    for bad in (0.0, -1.0, float("inf"), float("nan")):
        gs = (ctypes.c_float * 1)(bad)
        assert L.moe_nvfp4_prepare_weights(256, 256, ctypes.cast(gs, ctypes.c_void_p), 128, 64, 0, 0, 256,
                                           None) == B.MOE_ERR_INVALID_ARG
    gs = (ctypes.c_float * 1)(1.0)
    assert L.moe_nvfp4_prepare_weights(256, 256, ctypes.cast(gs, ctypes.c_void_p), 100, 64, 0, 0, 256,
                                       None) == B.MOE_ERR_INVALID_ARG
    # grouped GEMM: a negative row count is refused on the host
    ga = B.MoeGemmArgs(mode=0, gate_up=1, num_groups=2, N=256, K=64, rows=-1)
    assert L.moe_nvfp4_grouped_gemm(ctypes.byref(ga), 256, 4096, None) == B.MOE_ERR_INVALID_ARG
    assert L.moe_nvfp4_quantize(256, 4, 24, 256, 256, 256, 256, 256, None) == B.MOE_ERR_INVALID_ARG
    assert L.moe_combine(256, 256, None, None, 4, 2, 12, 256, None) == B.MOE_ERR_INVALID_ARG
    assert L.moe_combine(256, 256, None, 8, 4, 2, 16, 256, None) == B.MOE_ERR_INVALID_ARG  # misaligned


def test_sizes(lib):
    assert B.moe_prepare_size(3072, 4096, 0, 1) == 256 + 3072 * 4096 * 9 // 16
    d = B.MoeLayerDesc(T=8, H=4096, I=1536, I_shared=1536, E=320, k=8, mode=0, w13=256, w2=256,
                       w13_shared=256, w2_shared=256)
    n8 = B.moe_workspace_size(d)
    d.T = 4096
    n4096 = B.moe_workspace_size(d)
    assert 0 < n8 < n4096
    d.H = 100
    assert B.moe_workspace_size(d) == 0
    # grouped GEMM: header, then the f16 rows and their multipliers (256-byte aligned pieces)
    base = B.moe_gemm_workspace_size(9)
    assert B.moe_gemm_workspace_size_rows(9, 0, 64) == base
    assert B.moe_gemm_workspace_size_rows(9, 100, 64) == base + 12800 + 512
    assert B.moe_gemm_workspace_size_rows(9, -1, 64) == 0
    assert B.moe_gemm_workspace_size_rows(9, 100, 0) == 0
    # K % 256 == 0: also room for the W4A4 codes and per-tile scale atoms; the larger need counts
    assert B.moe_gemm_workspace_size_rows(9, 100, 256) == base + 51200 + 512
    assert B.moe_gemm_workspace_size_rows(1000, 100, 256) == B.moe_gemm_workspace_size(1000) + 12800 + 1000 * 2048


def test_import_global_scale_host_only(lib):
    # host-only entry point: runs here without a GPU; checked against the
    # worked pair of the GLM thread (golden file) and the oracle
    import numpy as np
    from oracle import nvfp4
    gold = {}
    with open(os.path.join(ROOT, "tests", "golden", "global_scale_worked_example.txt")) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                key, val = line.split()
                gold[key] = float(val)
    assert B.moe_import_global_scale(gold["dequant_scale"], B.MOE_SCALE_DEQUANT) == gold["quant_scale"]
    assert B.moe_import_global_scale(gold["quant_scale"], B.MOE_SCALE_QUANT) == gold["quant_scale"]
    vals = np.random.default_rng(3).uniform(1e-7, 1e5, 500).astype(np.float32)
    for v in vals:
        got = np.float32(B.moe_import_global_scale(float(v), B.MOE_SCALE_DEQUANT))
        assert got == nvfp4.import_global_scale(v, "dequant")
    out = ctypes.c_float(0)
    for bad in (0.0, -1.0, float("inf"), float("nan")):
        assert lib.moe_import_global_scale(bad, B.MOE_SCALE_DEQUANT, ctypes.byref(out)) == B.MOE_ERR_INVALID_ARG
    assert lib.moe_import_global_scale(1.0, 7, ctypes.byref(out)) == B.MOE_ERR_INVALID_ARG


def test_new_entry_points_validate_on_host(lib):
    L = lib
    # router GEMM: H must be a multiple of 8, pointers set; T = 0 is a no-op
    assert L.moe_router_gemm(256, 256, 4, 12, 8, 256, None) == B.MOE_ERR_INVALID_ARG
    assert L.moe_router_gemm(None, None, 0, 64, 8, None, None) == B.MOE_OK
    assert L.moe_router_gemm(None, 256, 4, 64, 8, 256, None) == B.MOE_ERR_INVALID_ARG
    # static quantisation: the scale must be positive and finite
    for bad in (0.0, -2.0, float("inf"), float("nan")):
        assert L.moe_nvfp4_quantize_static(256, 4, 64, bad, 256, 256, None) == B.MOE_ERR_INVALID_ARG
    # fold: ratio must be positive and finite; n = 0 is a no-op
    for bad in (0.0, -1.0, float("inf")):
        assert L.moe_nvfp4_fold_scales(256, 16, bad, 256, None) == B.MOE_ERR_INVALID_ARG
    assert L.moe_nvfp4_fold_scales(256, 0, 1.0, 256, None) == B.MOE_OK
    # static scales on a W4A16 layer, or negative ones, are refused
    d = B.MoeLayerDesc(T=8, H=4096, I=1536, I_shared=1536, E=320, k=8, mode=0, w13=256, w2=256,
                       w13_shared=256, w2_shared=256)
    assert B.moe_workspace_size(d) > 0
    d.x_global_scale = 100.0
    assert B.moe_workspace_size(d) == 0
    d.mode = 1
    d.H, d.I = 4096, 1536
    assert B.moe_workspace_size(d) > 0
    d.h_global_scale = -1.0
    assert B.moe_workspace_size(d) == 0
    d.h_global_scale = 0.0
    # the router matrix adds the [T, E] logits to the workspace
    n0 = B.moe_workspace_size(d)
    d.w_router = 256
    assert B.moe_workspace_size(d) >= n0 + 8 * 320 * 4
    d.w_router = 258
    assert B.moe_workspace_size(d) == 0


def test_empty_batches_are_host_no_ops(lib):
    # T = 0 (or rows = 0) returns MOE_OK before any device work
    d = B.MoeLayerDesc(T=0, H=4096, I=1536, I_shared=1536, E=320, k=8, mode=0, w13=256, w2=256,
                       w13_shared=256, w2_shared=256)
    assert lib.moe_nvfp4_forward(ctypes.byref(d), None, None, None, None, None, 0, None) == B.MOE_OK
    assert lib.moe_nvfp4_quantize_static(None, 0, 64, 1.0, None, None, None) == B.MOE_OK
    assert lib.moe_combine(None, None, None, None, 0, 8, 4096, None, None) == B.MOE_OK
    assert lib.moe_swiglu(None, 0, 128, None, None) == B.MOE_OK


def test_debug_hooks_validate_keys(lib):
    assert lib.moe_debug_set(99, 1) == B.MOE_ERR_INVALID_ARG
    for key in (B.MOE_DEBUG_WAIT_LIMIT, B.MOE_DEBUG_EXTRA_ARRIVALS, B.MOE_DEBUG_DISABLE_DECODE_FUSED,
                B.MOE_DEBUG_DECODE_STAGE_KB, B.MOE_DEBUG_FP4_TILE, B.MOE_DEBUG_F16_TILE):
        assert lib.moe_debug_set(key, 0) == B.MOE_OK   # 0 restores every default
    for bad in (-1, 6, 16, 56, 60, 100):   # FP4 tile shapes: two digits, each 0..5
        assert lib.moe_debug_set(B.MOE_DEBUG_FP4_TILE, bad) == B.MOE_ERR_INVALID_ARG
    assert lib.moe_debug_set(B.MOE_DEBUG_FP4_TILE, 23) == B.MOE_OK
    assert lib.moe_debug_set(B.MOE_DEBUG_FP4_TILE, 0) == B.MOE_OK
    for bad in (-1, 2, 10):   # W4A16 tile shapes: 0 (default) or 1 (128-row tiles only)
        assert lib.moe_debug_set(B.MOE_DEBUG_F16_TILE, bad) == B.MOE_ERR_INVALID_ARG
    assert lib.moe_debug_set(B.MOE_DEBUG_F16_TILE, 1) == B.MOE_OK
    assert lib.moe_debug_set(B.MOE_DEBUG_F16_TILE, 0) == B.MOE_OK


def test_binding_structs_match_the_header(tmp_path):
    """The binding's ctypes structs have the C header's field offsets and
    sizes (compiled here with the host C compiler)."""
    import shutil
    import subprocess
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no host C compiler")
    structs = {"moe_gemm_args": B.MoeGemmArgs, "moe_layer_desc": B.MoeLayerDesc}
    lines = ["#include <stddef.h>", "#include <stdio.h>", '#include "moe_nvfp4.h"', "int main(void) {"]
    for cname, py in structs.items():
        lines.append(f'  printf("{cname} size %zu\\n", sizeof({cname}));')
        for name, _ in py._fields_:
            lines.append(f'  printf("{cname} {name} %zu\\n", offsetof({cname}, {name}));')
    lines += ["  return 0;", "}"]
    src = tmp_path / "layout.c"
    src.write_text("\n".join(lines) + "\n")
    exe = tmp_path / "layout"
    inc = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include")
    subprocess.run([cc, "-std=c99", "-I", inc, str(src), "-o", str(exe)], check=True)
    got = {}
    for line in subprocess.run([str(exe)], check=True, capture_output=True, text=True).stdout.splitlines():
        cname, field, value = line.split()
        got[(cname, field)] = int(value)
    for cname, py in structs.items():
        assert got[(cname, "size")] == ctypes.sizeof(py), cname
        for name, _ in py._fields_:
            assert got[(cname, name)] == getattr(py, name).offset, (cname, name)
