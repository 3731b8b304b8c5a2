"""The C ABI library: builds, loads, exports what include/moe.h declares, and
validates arguments on the host (no GPU needed: every call below is rejected
before the library touches CUDA)."""
import ctypes
import os
import re

import pytest

import mixture_experts_layer_12_gb300 as moe
from mixture_experts_layer_12_gb300 import build as moe_build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    moe_build.build()
    return moe.load_library()


def declared_symbols():
    with open(os.path.join(ROOT, "include", "moe.h")) as f:
        src = f.read()
    return set(re.findall(r"MOE_API\s+[\w\s\*]+?\b(moe_\w+)\s*\(", src))


def exported_symbols(path):
    import subprocess
    out = subprocess.run(["nm", "-D", "--defined-only", path], capture_output=True, text=True,
                         check=True).stdout
    return {line.split()[-1] for line in out.splitlines() if line.strip()}


def test_exports_match_header(lib):
    decl = declared_symbols()
    assert len(decl) == 19
    assert decl == set(moe.EXPORTS)
    exported = {s for s in exported_symbols(moe.LIB_PATH) if s.startswith("moe_")}
    assert exported == decl
    for name in decl:
        assert getattr(lib, name) is not None


def test_version(lib):
    assert moe.moe_version() >> 16 == 1


def _al(v, a=1024):
    return -(-v // a) * a


def fused_route_bytes(T, H, E):
    """The fused route's workspace region (T > 128 or E > 64, at most 128
    tiles of 128 tokens): per-CTA counts [ctas, E16] bytes, ctas <=
    min(ceil(T / 64) * min(8, H / 64), 256) (64-token tiles, clusters of up
    to 8 K splits)."""
    if (T <= 128 and E <= 64) or -(-T // 128) > 128:
        return 0
    ctas = min(-(-T // 64) * min(8, -(-H // 64)), 256)
    e16 = -(-E // 16) * 16
    return _al(ctas * e16)


def test_workspace_size_and_capacity_host_only(lib):
    s = moe.make_shape(4096, 4096, 14336, 8, 2)
    # status block + per-128-token expert counts + the fused route's regions
    # + h [T*k, F] + Y [T*k, H], bf16
    route = 1024 + 1024 + fused_route_bytes(4096, 4096, 8)
    assert fused_route_bytes(4096, 4096, 8) == 4096
    assert moe.moe_workspace_size(s) == route + 8192 * 14336 * 2 + 8192 * 4096 * 2
    assert moe.moe_route_workspace_size(s) == route  # 32 tiles x 8 experts x 4 B of counts
    s3 = moe.make_shape(2048, 4096, 0, 128, 8)
    assert moe.moe_route_workspace_size(s3) == 1024 + 16 * 128 * 4 + 256 * 128
    # past 128 tiles the route is router + dispatch kernels: no fused regions
    s4 = moe.make_shape(40000, 256, 0, 8, 2)
    assert moe.moe_route_workspace_size(s4) == 1024 + _al(313 * 8 * 4)
    assert moe.moe_expert_capacity(moe.make_shape(8192, 2048, 1408, 64, 4, 1.2)) == 615
    assert moe.moe_expert_capacity(moe.make_shape(8192, 2048, 1408, 64, 4, None)) == -1
    assert moe.moe_expert_capacity(moe.make_shape(64, 128, 256, 8, 2, 1.0)) == 16


def test_any_expert_count_is_accepted_and_pads_w_router(lib):
    # E % 8 != 0: the route reads a copy of W_router with its rows padded to
    # a multiple of 8 experts, [H, E rounded up to 8] bf16, in the workspace
    for E in (1, 2, 4, 6, 13, 250):
        k = min(E, 2)
        s = moe.make_shape(300, 4096, 256, E, k)
        pad = _al(4096 * (-(-E // 8) * 8) * 2)
        hist = _al(3 * E * 4)
        route = 1024 + hist + pad + fused_route_bytes(300, 4096, E)
        assert moe.moe_route_workspace_size(s) == route
        assert moe.moe_workspace_size(s) == route + 300 * k * (256 + 4096) * 2
    s8 = moe.make_shape(300, 4096, 256, 16, 2)
    # no copy when E % 8 == 0
    assert moe.moe_route_workspace_size(s8) == 1024 + 1024 + fused_route_bytes(300, 4096, 16)


@pytest.mark.parametrize("T,k,E,cf", [(8192, 4, 64, 1.2), (64, 2, 8, 1.0), (10, 1, 8, 0.8),
                                      (3, 2, 8, 1.0), (100, 8, 256, 0.37), (7, 3, 16, float("nan"))])
def test_capacity_matches_oracle(lib, T, k, E, cf):
    import oracle
    assert moe.moe_expert_capacity(moe.make_shape(T, 8, 8, E, k, cf)) == oracle.capacity(T, k, E, cf)


@pytest.mark.parametrize("kw,code", [
    (dict(E=0), moe.MOE_ERR_UNSUPPORTED), (dict(E=264), moe.MOE_ERR_UNSUPPORTED),
    (dict(k=9), moe.MOE_ERR_UNSUPPORTED), (dict(k=0), moe.MOE_ERR_UNSUPPORTED),
    (dict(H=100), moe.MOE_ERR_UNSUPPORTED), (dict(F=12), moe.MOE_ERR_UNSUPPORTED),
    (dict(T=-1), moe.MOE_ERR_INVALID_ARG), (dict(T=1 << 22, k=8), moe.MOE_ERR_UNSUPPORTED),
    (dict(gating=3), moe.MOE_ERR_INVALID_ARG), (dict(gating=-1), moe.MOE_ERR_INVALID_ARG),
])
def test_bad_shapes_rejected_before_launch(lib, kw, code):
    base = dict(T=64, H=128, F=256, E=8, k=2)
    base.update(kw)
    s = moe.make_shape(**base)
    assert lib.moe_workspace_size(ctypes.byref(s)) == 0
    rc = lib.moe_forward(ctypes.byref(s), *([None] * 13), 0, None)
    assert rc == code
    assert lib.moe_last_error_string()


def test_null_and_misaligned_pointers_rejected(lib):
    s = moe.make_shape(64, 128, 256, 8, 2)
    ws_need = lib.moe_workspace_size(ctypes.byref(s))
    # null workspace
    rc = lib.moe_forward(ctypes.byref(s), *([None] * 13), ws_need, None)
    assert rc == moe.MOE_ERR_INVALID_ARG
    assert b"ws" in lib.moe_last_error_string()
    # misaligned workspace pointer (never dereferenced: rejected on the host)
    rc = lib.moe_forward(ctypes.byref(s), *([None] * 12), ctypes.c_void_p(0x1008), ws_need, None)
    assert rc == moe.MOE_ERR_INVALID_ARG
    # workspace too small
    rc = lib.moe_forward(ctypes.byref(s), *([None] * 12), ctypes.c_void_p(0x1000), ws_need - 16, None)
    assert rc == moe.MOE_ERR_INVALID_ARG
    assert b"workspace" in lib.moe_last_error_string()
    # route: null counts
    rc = lib.moe_route(ctypes.byref(s), *([None] * 9), ctypes.c_void_p(0x1000), 4096, None)
    assert rc == moe.MOE_ERR_INVALID_ARG
    # route: workspace smaller than moe_route_workspace_size
    rc = lib.moe_route(ctypes.byref(s), *([None] * 9), ctypes.c_void_p(0x1000), 1024, None)
    assert rc == moe.MOE_ERR_INVALID_ARG and b"moe_route_workspace_size" in lib.moe_last_error_string()
    # self-test limit outside its range
    rc = lib.moe_selftest_wait_timeout(ctypes.c_void_p(0x1000), 4096, 10, None)
    assert rc == moe.MOE_ERR_INVALID_ARG


def test_python_binding_rejects_host_tensors(lib):
    import torch
    s = moe.make_shape(4, 8, 8, 8, 2)
    with pytest.raises((ValueError, TypeError)):
        moe.moe_dispatch(s, torch.zeros(4, 2, dtype=torch.int32), torch.zeros(8, dtype=torch.int32),
                         torch.zeros(9, dtype=torch.int32), torch.zeros(8, dtype=torch.int32),
                         torch.zeros(4, 2, dtype=torch.int32), torch.zeros(256, dtype=torch.uint8))


def test_unknown_expert_act_rejected(lib):
    s = moe.make_shape(64, 128, 256, 8, 2)
    s.expert_act = 7
    assert lib.moe_workspace_size(ctypes.byref(s)) == 0
    assert lib.moe_forward(ctypes.byref(s), *([None] * 13), 0, None) == moe.MOE_ERR_INVALID_ARG


def test_step_entry_points_validate_before_touching_the_device(lib):
    s = moe.make_shape(64, 128, 256, 8, 1)
    ws = ctypes.c_void_p(16)
    for n in (0, 257, -3):
        assert lib.moe_expert_ffn(ctypes.byref(s), n, None, None, None, None, None, ws, 1 << 30,
                                  None) == moe.MOE_ERR_INVALID_ARG
    bad = moe.make_shape(64, 128, 256, 300, 1)  # more experts than the limit
    assert lib.moe_dispatch_rows(ctypes.byref(bad), None, None, None, None, None) == \
        moe.MOE_ERR_UNSUPPORTED
    assert lib.moe_combine(ctypes.byref(bad), None, None, None, None, None) == \
        moe.MOE_ERR_UNSUPPORTED


def test_forward_plan_is_a_host_only_shape_rule(lib):
    import moe_synth
    # the route runs as one launch up to 128 tiles of 128 tokens (CUDA cores
    # for T <= 128 with E <= 64, the fused tensor-core route otherwise)
    for cfg, want in [(moe_synth.DECODE, (True, False)), (moe_synth.TINY, (True, False)),
                      (moe_synth.PREFILL, (True, False)), (moe_synth.PREFILL_K1, (True, True)),
                      (moe_synth.SKEWED, (True, False))]:
        s = moe.make_shape(cfg.T, cfg.H, cfg.F, cfg.E, cfg.k, cfg.capacity_factor)
        assert moe.moe_forward_plan(s) == want, cfg.name
    assert moe.moe_forward_plan(moe.make_shape(128, 64, 64, 64, 2)) == (True, False)
    assert moe.moe_forward_plan(moe.make_shape(16384, 64, 64, 64, 2)) == (True, False)
    assert moe.moe_forward_plan(moe.make_shape(16385, 64, 64, 72, 2)) == (False, False)
    c = ctypes.c_int32(0)
    good = moe.make_shape(64, 128, 256, 8, 2)
    assert lib.moe_forward_plan(ctypes.byref(good), None, ctypes.byref(c)) == moe.MOE_ERR_INVALID_ARG


def test_route_plan_validates_before_the_device(lib):
    # bad shapes and null outputs are refused on the host; a good shape needs
    # a device (without one the call reports a CUDA error, never a crash)
    tm, sp = ctypes.c_int32(-1), ctypes.c_int32(-1)
    bad = moe.make_shape(64, 100, 256, 8, 2)  # H not a multiple of 8
    assert lib.moe_route_plan(ctypes.byref(bad), ctypes.byref(tm), ctypes.byref(sp)) == moe.MOE_ERR_UNSUPPORTED
    good = moe.make_shape(2048, 4096, 0, 128, 1)
    assert lib.moe_route_plan(ctypes.byref(good), None, ctypes.byref(sp)) == moe.MOE_ERR_INVALID_ARG
    import torch
    if not torch.cuda.is_available():
        rc = lib.moe_route_plan(ctypes.byref(good), ctypes.byref(tm), ctypes.byref(sp))
        assert rc == moe.MOE_ERR_CUDA and (tm.value, sp.value) == (0, 0)


def test_plain_c_caller(lib, tmp_path):
    # tests/c_abi_check.c: a C program built with gcc against include/moe.h
    # and linked to libmoe.so, calling the host-answered entry points
    import subprocess
    exe = tmp_path / "c_abi_check"
    libdir = os.path.dirname(moe.LIB_PATH)
    subprocess.run(["gcc", "-std=c11", "-Wall", "-Wextra", "-Werror",
                    "-I", os.path.join(ROOT, "include"), os.path.join(ROOT, "tests", "c_abi_check.c"),
                    "-L", libdir, "-l:libmoe.so", f"-Wl,-rpath,{libdir}", "-lm", "-o", str(exe)],
                   check=True)
    r = subprocess.run([str(exe)], capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    assert r.stdout.strip() == "ok"
