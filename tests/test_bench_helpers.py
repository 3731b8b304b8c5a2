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
    # up to 128 tiles of 128 tokens the route (router + dispatch) is one launch
    assert set(bench.launched_kernels(_shape(moe_synth.PREFILL))) == every - {"dispatch"}
    assert set(bench.launched_kernels(_shape(moe_synth.DECODE))) == every - {"dispatch"}
    # past that, all six steps are kernels of their own
    assert set(bench.launched_kernels(_shape(moe_synth.PREFILL.with_(T=20000)))) == every
    # k = 1: the second GEMM also combines
    assert set(bench.launched_kernels(_shape(moe_synth.PREFILL_K1))) == \
        every - {"combine", "dispatch"}
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


def test_tensor_peak_follows_the_timed_region_and_clocks():
    peaks = {"hbm_gbs": 6000.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
    full = {"sm_mhz": 2070.0, "sm_max_mhz": 2070.0, "reasons": []}
    capped = {"sm_mhz": 1650.0, "sm_max_mhz": 2070.0, "reasons": ["sw_power_cap"]}
    flagged_full = {"sm_mhz": 2070.0, "sm_max_mhz": 2070.0, "reasons": ["sw_power_cap"]}
    # a short region at full clocks is a burst (a momentary cap flag included);
    # a long one, or one whose clock the power cap held down, runs at the
    # sustained rate
    assert bench.tensor_peak(peaks, 25.0, full) == (1900.0, "burst")
    assert bench.tensor_peak(peaks, 25.0, flagged_full) == (1900.0, "burst")
    assert bench.tensor_peak(peaks, 25.0, capped) == (1700.0, "sustained")
    assert bench.tensor_peak(peaks, 1400.0, full) == (1700.0, "sustained")
    assert bench.tensor_peak(peaks, 25.0, None) == (1900.0, "burst")


def test_roofline_reports_both_tensor_fractions():
    peaks = {"hbm_gbs": 6000.0, "bf16_tflops": 2000.0, "bf16_tflops_sustained": 1600.0}
    gemm = {"flops": 1.0e12, "bytes": 1.0e9}  # intensity 1000 FLOP/B > ridge
    r = bench.roofline(gemm, 1.0, peaks, "measured", 20.0, {"reasons": []}, "expert_gemm1")
    assert r["bound"] == "tensor" and r["achieved"] == 1000.0
    assert r["frac"] == 0.5 and r["frac_of_burst"] == 0.5 and r["frac_of_sustained"] == 0.625
    assert "burst" in r["peak_kind"]
    stream = {"flops": 1.0e9, "bytes": 3.0e9}
    h = bench.roofline(stream, 1.0, peaks, "measured", 20.0, None, "route")
    assert h["bound"] == "hbm" and h["achieved"] == 3000.0 and h["frac"] == 0.5


def test_cpu_baseline_is_the_oracle_equivalent_full_time():
    import oracle
    oracle.build()
    cfg = moe_synth.TINY
    inputs = moe_synth.make_inputs(cfg)
    cb = bench.cpu_baseline(inputs, cfg, 16)
    assert cb["kind"] == "oracle" and cb["unit"] == "tokens/s" and cb["value"] > 0
    assert "every 16-th token (4 tokens" in cb["sample"] and cb["nproc"] >= 1
    route_only = bench.cpu_baseline(moe_synth.make_inputs(moe_synth.ROUTER[2].with_(T=64, H=128),
                                                          with_ffn=False),
                                    moe_synth.ROUTER[2].with_(T=64, H=128), 16)
    assert "FFN" not in route_only["sample"]
