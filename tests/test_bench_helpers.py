"""bench.py's bookkeeping on the host: which kernels a forward step launches,
the algorithmic work each one is measured against, and when an ncu traffic
figure still applies (no GPU needed)."""
import pytest

import bench
import moe_synth
import mixture_experts_layer_12_gb300 as moe
from mixture_experts_layer_12_gb300 import build as moe_build


@pytest.fixture(scope="module", autouse=True)
def lib():
    moe_build.build()
    return moe.load_library()


def _shape(cfg):
    return moe.make_shape(cfg.T, cfg.H, cfg.F, cfg.E, cfg.k, cfg.capacity_factor)


def test_launched_kernels_follow_the_forward_plan():
    every = set(moe.KERNEL_NAMES)
    # large batch, k = 2: all six steps are kernels of their own
    assert set(bench.launched_kernels(_shape(moe_synth.PREFILL))) == every
    # small batch: the router also dispatches
    assert set(bench.launched_kernels(_shape(moe_synth.DECODE))) == every - {"dispatch"}
    # k = 1: the second GEMM also combines
    assert set(bench.launched_kernels(_shape(moe_synth.PREFILL_K1))) == every - {"combine"}
    for name in every - set(bench.launched_kernels(_shape(moe_synth.DECODE))):
        assert name in bench.FUSED_INTO


def test_kernel_work_formulas():
    cfg = moe_synth.PREFILL
    n_rows, hit = cfg.T * cfg.k, cfg.E
    w = bench.kernel_work(cfg, n_rows, hit)
    # each expert GEMM: 2 * rows * H * F FLOPs; prefill's pair is 1.924 TFLOP
    assert w["expert_gemm1"]["flops"] == 2.0 * n_rows * cfg.H * cfg.F
    assert w["expert_gemm2"]["flops"] == w["expert_gemm1"]["flops"]
    assert abs(2 * w["expert_gemm1"]["flops"] - 1.924e12) < 1e9
    # router bytes: x once, W_router once, ids + weights out
    assert w["router"]["bytes"] == 2.0 * cfg.T * cfg.H + 2.0 * cfg.H * cfg.E + 8.0 * cfg.T * cfg.k
    # gated experts: W1 holds gate and up, twice the columns
    g = bench.kernel_work(moe_synth.PREFILL_SWIGLU, n_rows, hit)
    assert g["expert_gemm1"]["flops"] == 2 * w["expert_gemm1"]["flops"]
    assert g["expert_gemm2"]["flops"] == w["expert_gemm2"]["flops"]


def test_ncu_traffic_only_for_the_sources_it_was_taken_on(monkeypatch):
    key = "prefill/expert_gemm1"
    entry = dict(bench.NCU_TRAFFIC[key])
    # the figure applies exactly while the source file hashes to the recorded value
    monkeypatch.setitem(bench.NCU_TRAFFIC, key, dict(entry, src_sha=bench.src_sha(entry["src"])))
    assert bench.ncu_traffic(key) == entry["bytes"]
    monkeypatch.setitem(bench.NCU_TRAFFIC, key, dict(entry, src_sha="0" * 16))
    assert bench.ncu_traffic(key) is None
    # several sources: every one must match
    multi = "router_k1/router+dispatch"
    m = dict(bench.NCU_TRAFFIC[multi])
    shas = [bench.src_sha(f) for f in m["src"]]
    monkeypatch.setitem(bench.NCU_TRAFFIC, multi, dict(m, src_sha=shas))
    assert bench.ncu_traffic(multi) == m["bytes"]
    monkeypatch.setitem(bench.NCU_TRAFFIC, multi, dict(m, src_sha=[shas[0], "0" * 16]))
    assert bench.ncu_traffic(multi) is None
    assert bench.ncu_traffic("no/such") is None
