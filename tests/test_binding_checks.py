"""Host-side argument checks of the Python binding (no GPU needed).

The library indexes every buffer from the shape alone, so a tensor with too
few elements, or one on another GPU than the current device, would turn into
out-of-bounds device accesses.  The binding refuses both before anything is
launched.  These tests check the rule itself on duck-typed stand-ins, and
that every wrapper asks, per argument, for the element count its C entry
point reads (sizes derived here by hand from include/moe.h).
"""
import ctypes
from types import SimpleNamespace

import pytest
import torch

import mixture_experts_layer_12_gb300 as moe


class FakeTensor:
    def __init__(self, numel, dtype=torch.bfloat16, device="cuda:0", contiguous=True):
        self._n, self.dtype, self.device, self._c = numel, dtype, torch.device(device), contiguous

    def numel(self):
        return self._n

    def is_contiguous(self):
        return self._c


def test_check_tensor_rules():
    ok = FakeTensor(100)
    moe.check_tensor(ok, torch.bfloat16, "x", 100, 0)
    with pytest.raises(ValueError, match="at least 101"):
        moe.check_tensor(ok, torch.bfloat16, "x", 101, 0)
    with pytest.raises(ValueError, match="cuda:1"):
        moe.check_tensor(FakeTensor(100, device="cuda:1"), torch.bfloat16, "x", 10, 0)
    with pytest.raises(ValueError, match="CUDA tensor"):
        moe.check_tensor(FakeTensor(100, device="cpu"), torch.bfloat16, "x", 10, 0)
    with pytest.raises(TypeError):
        moe.check_tensor(FakeTensor(100, dtype=torch.float32), torch.bfloat16, "x", 10, 0)
    with pytest.raises(ValueError, match="contiguous"):
        moe.check_tensor(FakeTensor(100, contiguous=False), torch.bfloat16, "x", 10, 0)
    # an empty tensor needs no device (a T = 0 call passes empty buffers)
    moe.check_tensor(FakeTensor(0, device="cpu"), torch.bfloat16, "x", 0, 0)


def test_undersized_host_tensor_raises_before_the_library_is_touched():
    s = moe.make_shape(4, 8, 8, 8, 2)
    with pytest.raises(ValueError, match="ids holds 7"):
        moe.moe_dispatch(s, torch.zeros(7, dtype=torch.int32), torch.zeros(8, dtype=torch.int32),
                         torch.zeros(9, dtype=torch.int32), torch.zeros(8, dtype=torch.int32),
                         torch.zeros(8, dtype=torch.int32), torch.zeros(256, dtype=torch.uint8))


@pytest.fixture
def recorded(monkeypatch):
    """Replaces pointer marshalling and the library: records the minimum
    element count each wrapper demands for each named argument."""
    seen = {}

    def fake_ptr(t, dtype=None, name="tensor", min_numel=0):
        seen[name] = min_numel
        return ctypes.c_void_p(16)

    lib = SimpleNamespace()
    for n in moe.EXPORTS:
        setattr(lib, n, lambda *a, **k: moe.MOE_OK)
    monkeypatch.setattr(moe, "_ptr", fake_ptr)
    monkeypatch.setattr(moe, "load_library", lambda path=None: lib)
    return seen


def _t():
    return torch.zeros(1, dtype=torch.uint8)


def test_wrappers_demand_the_sizes_the_entry_points_read(recorded):
    T, H, F, E, k = 5, 16, 24, 8, 3
    s = moe.make_shape(T, H, F, E, k)
    z = _t()
    moe.moe_forward(s, *([z] * 12), z, stream=0)
    want = dict(x=T * H, w_router=H * E, b_router=E, w1=E * H * F, w2=E * F * H, y=T * H,
                ids=T * k, weights=T * k, counts=E, offsets=E + 1, perm=T * k, slot=T * k)
    assert {n: recorded[n] for n in want} == want
    recorded.clear()
    moe.moe_expert_ffn_combine(s, *([z] * 8), z, stream=0)
    assert {n: recorded[n] for n in ("x", "w1", "w2", "weights", "offsets", "perm", "slot", "y")} == \
        dict(x=T * H, w1=E * H * F, w2=E * F * H, weights=T * k, offsets=E + 1, perm=T * k,
             slot=T * k, y=T * H)
    recorded.clear()
    moe.moe_expert_ffn_combine_noalloc(s, *([z] * 8), stream=0)
    assert recorded["y"] == T * H and recorded["w1"] == E * H * F
    recorded.clear()
    moe.moe_dispatch_rows(s, z, z, z, z, stream=0)
    assert recorded == dict(x=T * H, perm=T * k, offsets=E + 1, xp=T * k * H)
    recorded.clear()
    moe.moe_combine(s, z, z, z, z, stream=0)
    assert recorded == dict(Y=T * k * H, weights=T * k, slot=T * k, y=T * H)
    recorded.clear()
    moe.moe_expert_ffn(s, 6, z, z, z, z, z, z, stream=0)
    assert {n: recorded[n] for n in ("xp", "w1", "w2", "seg_offsets", "Y")} == \
        dict(xp=T * k * H, w1=E * H * F, w2=E * F * H, seg_offsets=7, Y=T * k * H)
    recorded.clear()
    moe.moe_route(s, *([z] * 9), z, stream=0)
    assert {n: recorded[n] for n in ("x", "w_router", "ids", "perm", "slot", "counts")} == \
        dict(x=T * H, w_router=H * E, ids=T * k, perm=T * k, slot=T * k, counts=E)
    recorded.clear()
    moe.moe_dispatch(s, *([z] * 5), z, stream=0)
    assert recorded["ids"] == T * k and recorded["offsets"] == E + 1
    # gated experts: W1 holds [W_gate | W_up], 2F columns
    g = moe.make_shape(T, H, F, E, k, act="swiglu")
    recorded.clear()
    moe.moe_forward(g, *([z] * 12), z, stream=0)
    assert recorded["w1"] == E * H * 2 * F and recorded["w2"] == E * F * H
