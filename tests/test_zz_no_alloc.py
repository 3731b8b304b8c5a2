"""The allocation-free expert FFN + combine entry point.

moe_expert_ffn_combine_noalloc serves callers that cannot allocate device
memory (for example a runtime that reserves all device memory up front and
forbids cudaMalloc afterwards, or a plain C host that owns only its inputs
and outputs): instead of a caller workspace it uses a static scratch array
inside the library.  These tests call it through the C ABI and check that
it gives the same y as the workspace entry point, on two calls in a row
(the second call must not see the first one's leftovers), and that shapes
beyond the scratch are refused with a clear error.  This file is collected
last so that a failure here cannot hide another test's result.
"""
import pytest
import torch

import moe_synth
import mixture_experts_layer_12_gb300 as moe

pytestmark = pytest.mark.gpu

DEV = "cuda:0"
Y_MAX_REL = 1e-2  # same acceptance as the oracle parity tests
Y_MEAN_REL = 5e-3


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


def _close(y, y_ref):
    d = (y.float() - y_ref.float()).abs()
    ref = y_ref.float().abs()
    assert d.max().item() <= Y_MAX_REL * ref.max().item()
    assert d.mean().item() <= Y_MEAN_REL * ref.mean().item()


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
        torch.cuda.synchronize()
        assert torch.isfinite(y.float()).all()
        _close(y, y_ref)


def test_noalloc_refuses_shapes_beyond_its_scratch():
    s = moe.make_shape(4096, 4096, 14336, 8, 2)  # ~300 MB of intermediates
    assert moe.moe_workspace_size(s) > moe.MOE_NOALLOC_SCRATCH_BYTES
    bf = torch.empty(8, dtype=torch.bfloat16, device=DEV)
    f32 = torch.empty(4, dtype=torch.float32, device=DEV)
    i32 = torch.empty(4, dtype=torch.int32, device=DEV)
    with pytest.raises(moe.MoEError) as e:  # refused on the host, nothing is launched
        moe.moe_expert_ffn_combine_noalloc(s, bf, bf, bf, f32, i32, i32, i32, bf)
    assert e.value.code == moe.MOE_ERR_UNSUPPORTED
    assert "scratch" in str(e.value)
