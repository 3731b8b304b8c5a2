"""The allocation-free expert FFN + combine entry point.

moe_expert_ffn_combine_noalloc serves callers that cannot allocate device
memory (for example a runtime that reserves all device memory up front and
forbids cudaMalloc afterwards, or a plain C host that owns only its inputs
and outputs): instead of a caller workspace it uses a static scratch array
inside the library.  These tests call it through the C ABI and check that
it gives bit for bit the same y as the workspace entry point (both run the
same kernels, so any difference -- stale scratch from the previous call in
a few rows, say -- is a fault), on calls in a row of different shapes, that
its status word reads back clean, and that shapes beyond the scratch are
refused with a clear error.  This file is collected last so that a failure
here cannot hide another test's result.
"""
import ctypes

import pytest
import torch

import moe_synth
import mixture_experts_layer_12_gb300 as moe

pytestmark = pytest.mark.gpu

DEV = "cuda:0"


@pytest.fixture(scope="module", autouse=True)
def _built():
    from mixture_experts_layer_12_gb300 import build
    build.build()
    moe.load_library()


def _routed(cfg):
    inputs = {k: (None if v is None else v.to(DEV)) for k, v in moe_synth.make_inputs(cfg).items()}
    s = moe.make_shape(cfg.T, cfg.H, cfg.F, cfg.E, cfg.k, cfg.capacity_factor)
    r = moe.alloc_routing(cfg.T, cfg.E, cfg.k, DEV)
    ws = moe.alloc_workspace(s, DEV)
    moe.moe_route(s, inputs["x"], inputs["w_router"], inputs["bias"], r.ids, r.weights, r.counts,
                  r.offsets, r.perm, r.slot, ws)
    return s, inputs, r, ws


def test_noalloc_matches_workspace_entry_point_on_two_calls():
    # two different shapes in a row: a decode-sized batch, then a smaller one
    # with a capacity limit, so stale scratch from the first call would show
    cfgs = [moe_synth.DECODE,
            moe_synth.MoEConfig("small", T=96, H=256, F=384, E=16, k=4, seed=31,
                                capacity_factor=0.8),
            moe_synth.MoEConfig("top1", T=200, H=256, F=384, E=8, k=1, seed=32,
                                capacity_factor=0.6)]
    for cfg in cfgs:
        s, inp, r, ws = _routed(cfg)
        y_ref = torch.empty(cfg.T, cfg.H, dtype=torch.bfloat16, device=DEV)
        moe.moe_expert_ffn_combine(s, inp["x"], inp["w1"], inp["w2"], r.weights, r.offsets, r.perm,
                                   r.slot, y_ref, ws)
        assert moe.moe_get_device_status(ws) == 0
        y = torch.full((cfg.T, cfg.H), float("nan"), dtype=torch.bfloat16, device=DEV)
        moe.moe_expert_ffn_combine_noalloc(s, inp["x"], inp["w1"], inp["w2"], r.weights, r.offsets,
                                           r.perm, r.slot, y)
        assert moe.moe_noalloc_device_status() == 0
        assert torch.isfinite(y.float()).all()
        assert torch.equal(y, y_ref), cfg.name


def test_noalloc_refuses_shapes_beyond_its_scratch():
    # through the C ABI directly: the shape is refused on the host before any
    # pointer is looked at, so placeholder addresses are never dereferenced
    s = moe.make_shape(4096, 4096, 14336, 8, 2)  # ~300 MB of intermediates
    assert moe.moe_workspace_size(s) > moe.MOE_NOALLOC_SCRATCH_BYTES
    lib = moe.load_library()
    rc = lib.moe_expert_ffn_combine_noalloc(ctypes.byref(s), *([ctypes.c_void_p(256)] * 8), None)
    assert rc == moe.MOE_ERR_UNSUPPORTED
    assert b"scratch" in lib.moe_last_error_string()
