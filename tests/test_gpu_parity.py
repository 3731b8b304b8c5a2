"""CUDA path vs the oracle, element by element, through the C ABI.

Small workloads compare every row; the full-size workloads compare routing
and dispatch for every token and y on every 16th token (tokens are
independent once routed and dispatched), in the same launch configuration
bench.py times.
"""
import numpy as np
import pytest
import torch

import moe_synth
import oracle
import mixture_experts_layer_12_gb300 as moe
from parity import check_dispatch, check_routing, check_y, reference_y

pytestmark = pytest.mark.gpu

DEV = "cuda:0"
# the seeded workloads whose oracle routing figures tests/golden/routing_stats.json holds
STATS_WORKLOADS = ("tiny", "prefill", "router_k1", "router_k2", "router_k4", "router_k8", "skewed",
                   "skewed_cf1.2", "decode", "prefill_k1")


@pytest.fixture(scope="module", autouse=True)
def _built():
    from mixture_experts_layer_12_gb300 import build
    build.build()
    oracle.build()
    moe.load_library()


def to_dev(inputs):
    return {k: (None if v is None else v.to(DEV)) for k, v in inputs.items()}


def gpu_route(cfg, dev_in, gating=0):
    s = moe.make_shape(cfg.T, cfg.H, max(cfg.F, 8), cfg.E, cfg.k, cfg.capacity_factor, gating)
    r = moe.alloc_routing(cfg.T, cfg.E, cfg.k, DEV)
    ws = moe.alloc_route_workspace(s, DEV)
    moe.moe_route(s, dev_in["x"], dev_in["w_router"], dev_in["bias"], r.ids, r.weights, r.counts,
                  r.offsets, r.perm, r.slot, ws)
    assert moe.moe_get_device_status(ws) == 0
    return r


def gpu_forward(cfg, dev_in, gating=0):
    layer = moe.MoELayer(dev_in["w_router"], dev_in["w1"], dev_in["w2"], cfg.k, bias=dev_in["bias"],
                         capacity_factor=cfg.capacity_factor, gating=gating, act=cfg.act)
    y = layer(dev_in["x"])
    assert moe.moe_get_device_status(layer.ws) == 0
    return layer, y


def np_(t):
    return t.detach().cpu().numpy()


def routing_parity(cfg, inputs, r, nthreads=0, gating=0):
    logits = oracle.router_logits(inputs["x"], inputs["w_router"], inputs["bias"], nthreads)
    o_ids, o_vals = oracle.topk(logits, cfg.k)
    o_w = oracle.gate_weights(logits, o_ids, o_vals, gating)
    gids = np_(r.ids)
    rep = check_routing(logits, o_ids, o_w, gids, np_(r.weights), gating)
    rep.update(check_dispatch(gids, cfg.E, cfg.capacity_factor, np_(r.counts), np_(r.offsets),
                              np_(r.perm), np_(r.slot)))
    rep["ids_equal_oracle_everywhere"] = bool(np.array_equal(gids, o_ids))
    if cfg.name in STATS_WORKLOADS and gating == 0:
        check_stats(cfg, rep, gids, o_ids)
    return logits, rep


def check_stats(cfg, rep, gpu_ids, ora_ids):
    """The GPU's routing against the oracle's figures stored in
    tests/golden/routing_stats.json (written from the oracle alone): the
    near-tie count, and the kept / dropped assignments -- exactly when the
    GPU chose the oracle's experts for every token, else within the tokens
    whose expert set may differ."""
    import json
    import os
    with open(os.path.join(os.path.dirname(__file__), "golden", "routing_stats.json")) as f:
        st = json.load(f)["workloads"][cfg.name]
    assert rep["near_tie_tokens"] == st["near_tie_tokens"]
    if np.array_equal(gpu_ids, ora_ids):
        assert (rep["kept"], rep["dropped"]) == (st["kept_assignments"], st["dropped_assignments"])
    else:
        assert abs(rep["dropped"] - st["dropped_assignments"]) <= cfg.k * st["membership_ties"]
    return st


def forward_parity(cfg, stride=1, nthreads=0, gating=0):
    inputs = moe_synth.make_inputs(cfg)
    dev_in = to_dev(inputs)
    layer, y = gpu_forward(cfg, dev_in, gating)
    logits, rep = routing_parity(cfg, inputs, layer.routing, nthreads, gating)
    rows = np.arange(0, cfg.T, stride, dtype=np.int32)
    y_ref = reference_y(inputs, logits, np_(layer.routing.ids), np_(layer.routing.slot), rows, nthreads,
                        gating)
    y_gpu = y.float().cpu().numpy()[rows]
    rep.update(check_y(y_gpu, y_ref))
    print(cfg.name, rep)
    return rep


# ------------------------------------------------------------- self test --

def test_bounded_wait_times_out_and_reports():
    ws = torch.empty(1024, dtype=torch.uint8, device=DEV)
    moe.moe_selftest_wait_timeout(ws, 2_000_000)  # 2 ms
    with pytest.raises(moe.MoEError) as e:
        moe.moe_get_device_status(ws)
    assert e.value.code == moe.MOE_ERR_TIMEOUT
    # the context stays usable and the status word was cleared
    assert moe.moe_get_device_status(ws) == 0
    assert torch.ones(4, device=DEV).sum().item() == 4.0


# --------------------------------------------------------------- dispatch --

@pytest.mark.parametrize("T,E,k,cf,skew", [
    (1, 8, 1, None, False), (7, 8, 2, None, False), (1000, 64, 4, 1.0, True),
    (8192, 64, 4, 1.2, True), (3000, 256, 8, None, False), (2048, 128, 8, 0.5, False),
    (4096, 8, 2, None, True), (513, 16, 3, 0.05, False), (20000, 32, 8, 0.9, True),
    (129, 256, 8, 0.3, False),
])
def test_dispatch_fed_oracle_ids(T, E, k, cf, skew):
    rng = np.random.default_rng(T + E + k)
    if skew:
        p = np.full(E, 1.0)
        p[0] = 20.0 * E
        p /= p.sum()
    else:
        p = None
    ids = np.stack([rng.choice(E, size=k, replace=False, p=p) for _ in range(T)]).astype(np.int32)
    s = moe.make_shape(T, 8, 8, E, k, cf)
    r = moe.alloc_routing(T, E, k, DEV)
    ws = moe.alloc_route_workspace(s, DEV)
    moe.moe_dispatch(s, torch.from_numpy(ids).to(DEV), r.counts, r.offsets, r.perm, r.slot, ws)
    assert moe.moe_get_device_status(ws) == 0
    check_dispatch(ids, E, cf, np_(r.counts), np_(r.offsets), np_(r.perm), np_(r.slot))


def test_dispatch_bad_ids_flagged():
    ids = torch.tensor([[0, 9], [3, 1]], dtype=torch.int32, device=DEV)
    s = moe.make_shape(2, 8, 8, 8, 2)
    r = moe.alloc_routing(2, 8, 2, DEV)
    ws = moe.alloc_route_workspace(s, DEV)
    moe.moe_dispatch(s, ids, r.counts, r.offsets, r.perm, r.slot, ws)
    with pytest.raises(moe.MoEError) as e:
        moe.moe_get_device_status(ws)
    assert e.value.code == moe.MOE_ERR_DEVICE
    assert np_(r.slot)[0, 1] == -1 and np_(r.counts).sum() == 3


# ----------------------------------------------------------------- router --

def test_router_tiny():
    cfg = moe_synth.TINY
    inputs = moe_synth.make_inputs(cfg, with_ffn=False)
    r = gpu_route(cfg, to_dev(inputs))
    _, rep = routing_parity(cfg, inputs, r)
    print(rep)


@pytest.mark.parametrize("k", [1, 2, 4, 8])
def test_router_sweep_full_size(k):
    cfg = moe_synth.ROUTER[k]
    inputs = moe_synth.make_inputs(cfg, with_ffn=False)
    r = gpu_route(cfg, to_dev(inputs))
    _, rep = routing_parity(cfg, inputs, r)
    print(cfg.name, moe.moe_route_plan(moe.make_shape(cfg.T, cfg.H, 8, cfg.E, cfg.k)), rep)


@pytest.mark.parametrize("T,E,k,cf", [(16384, 128, 2, None), (16384, 8, 1, 0.7),
                                      (3000, 200, 8, 0.3), (9000, 64, 4, None),
                                      (16384, 256, 8, 1.1),   # widest accumulator, most tiles
                                      (129, 256, 8, None),    # 2 tiles x 8 K splits, E > 64
                                      (256, 96, 3, 0.5)])     # 2 tiles, E = 96 (E16 = 96)
def test_route_in_one_launch_at_scale(T, E, k, cf):
    # the fused route: 128 tiles (the most it takes: one K split each), E that
    # fills an uneven number of count chunks (200 -> 13), drops, many tiles
    cfg = moe_synth.MoEConfig("fused", T=T, H=512, F=0, E=E, k=k, seed=28, capacity_factor=cf)
    assert moe.moe_forward_plan(moe.make_shape(T, cfg.H, 8, E, k, cf))[0]
    inputs = moe_synth.make_inputs(cfg, with_ffn=False)
    r = gpu_route(cfg, to_dev(inputs))
    _, rep = routing_parity(cfg, inputs, r)
    if cf is not None:
        assert rep["dropped"] > 0


@pytest.mark.parametrize("gating", [moe.MOE_GATE_SOFTMAX_TOPK, moe.MOE_GATE_SOFTMAX_TOPK_RENORM])
@pytest.mark.parametrize("T,E,k", [(4096, 8, 2), (2048, 128, 8), (700, 13, 4)])
def test_route_in_one_launch_gating_and_bias(gating, T, E, k):
    # the fused route with the softmax-over-all-experts gate modes, a bias and
    # E % 8 != 0 (padded W_router)
    cfg = moe_synth.MoEConfig("fusedgate", T=T, H=256, F=0, E=E, k=k, seed=33, bias0=1.5)
    assert moe.moe_forward_plan(moe.make_shape(T, cfg.H, 8, E, k, None, gating))[0]
    inputs = moe_synth.make_inputs(cfg, with_ffn=False)
    r = gpu_route(cfg, to_dev(inputs), gating)
    routing_parity(cfg, inputs, r, gating=gating)


def test_route_plans_cover_tile_heights_and_splits():
    # the one-launch route picks 64- or 128-token tiles and clusters of 1, 2,
    # 4 or 8 K splits by shape; every pair these shapes select is checked
    # against the oracle, and together they take both heights and all splits
    shapes = [(300, 4096, 16, 2),    # few tiles, long K: 64-token tiles x 8
              (2048, 1024, 8, 2),    # 16 tiles
              (4096, 1024, 8, 2),    # 32 tiles
              (8192, 1024, 64, 4),   # 64 tiles
              (12000, 512, 8, 1),    # 94 tiles: one CTA each
              (129, 64, 8, 2)]       # one K block: 64-token tiles, no split
    seen = set()
    for i, (T, H, E, k) in enumerate(shapes):
        cfg = moe_synth.MoEConfig("plans", T=T, H=H, F=0, E=E, k=k, seed=40 + i)
        plan = moe.moe_route_plan(moe.make_shape(T, H, 8, E, k))
        assert plan[0] in (64, 128) and plan[1] in (1, 2, 4, 8), plan
        seen.add(plan)
        inputs = moe_synth.make_inputs(cfg, with_ffn=False)
        r = gpu_route(cfg, to_dev(inputs))
        _, rep = routing_parity(cfg, inputs, r)
        print(T, H, E, k, plan, rep)
    assert {tm for tm, _ in seen} == {64, 128}, seen
    assert {sp for _, sp in seen} == {1, 2, 4, 8}, seen


@pytest.mark.parametrize("T,H,E,k", [(1, 1000, 128, 8), (63, 1000, 96, 2), (65, 1000, 96, 3),
                                     (191, 1000, 200, 4), (320, 1000, 72, 2), (2100, 1000, 128, 1)])
def test_route_ragged_tokens_and_k_blocks(T, H, E, k):
    # the one-launch route at token counts off the 64- and 128-token tiles and
    # with H = 1000 (a last K block of 40 columns, zero-filled by TMA), so the
    # K splits of a cluster hold different numbers of K blocks
    cfg = moe_synth.MoEConfig("ragged", T=T, H=H, F=0, E=E, k=k, seed=50)
    plan = moe.moe_route_plan(moe.make_shape(T, H, 8, E, k))
    assert plan != (0, 0), plan
    inputs = moe_synth.make_inputs(cfg, with_ffn=False)
    r = gpu_route(cfg, to_dev(inputs))
    _, rep = routing_parity(cfg, inputs, r)
    print(T, H, E, k, plan, rep)


def test_route_plan_outside_the_fused_route():
    # small batches and batches past 128 tiles of 128 tokens route otherwise
    assert moe.moe_route_plan(moe.make_shape(32, 4096, 8, 8, 2)) == (0, 0)
    assert moe.moe_route_plan(moe.make_shape(17000, 256, 8, 128, 4)) == (0, 0)


def test_router_kernels_past_128_tiles_wide_experts():
    # 133 tiles, E = 128: the cluster router + dispatch kernel path
    cfg = moe_synth.MoEConfig("wide128", T=17000, H=256, F=0, E=128, k=4, seed=29)
    assert not moe.moe_forward_plan(moe.make_shape(cfg.T, cfg.H, 8, cfg.E, cfg.k))[0]
    inputs = moe_synth.make_inputs(cfg, with_ffn=False)
    r = gpu_route(cfg, to_dev(inputs))
    routing_parity(cfg, inputs, r)


@pytest.mark.parametrize("cf", [None, 0.9])
def test_router_more_tiles_than_one_wave(cf):
    # 313 tiles of 128 tokens: more router clusters than fit on the GPU at
    # once, and 313 segments for the scan of the per-tile counts
    cfg = moe_synth.MoEConfig("wide", T=40000, H=256, F=0, E=8, k=2, seed=27, capacity_factor=cf)
    assert not moe.moe_forward_plan(moe.make_shape(cfg.T, cfg.H, 8, cfg.E, cfg.k, cf))[0]
    inputs = moe_synth.make_inputs(cfg, with_ffn=False)
    r = gpu_route(cfg, to_dev(inputs))
    _, rep = routing_parity(cfg, inputs, r)
    if cf is not None:
        assert rep["dropped"] > 0


@pytest.mark.parametrize("T,E,k,cf,gating,bias", [
    (128, 64, 8, 0.5, 0, None),      # the largest small batch, 64 experts, drops
    (100, 16, 3, None, 1, 0.5),      # softmax over all experts
    (37, 32, 4, 1.0, 2, None),       # renormalised
    (1, 8, 2, None, 0, None),        # one token
    (128, 8, 2, 0.3, 0, 3.0),        # skewed, heavy drops
])
def test_small_batch_route_in_one_launch(T, E, k, cf, gating, bias):
    # T <= 128 and E <= 64: logits on the CUDA cores, dispatch by the last CTA
    cfg = moe_synth.MoEConfig("small", T=T, H=264, F=0, E=E, k=k, seed=29, capacity_factor=cf,
                              bias0=bias)
    assert moe.moe_forward_plan(moe.make_shape(T, cfg.H, 8, E, k, cf, gating))[0]
    inputs = moe_synth.make_inputs(cfg, with_ffn=False)
    r = gpu_route(cfg, to_dev(inputs), gating)
    _, rep = routing_parity(cfg, inputs, r, gating=gating)
    if cf == 0.3:
        assert rep["dropped"] > 0


@pytest.mark.parametrize("T,H,E,k,bias", [(1, 64, 8, 1, None), (130, 200, 16, 3, 0.5),
                                          (257, 520, 256, 8, None), (64, 4096, 40, 5, 2.0),
                                          (300, 72, 192, 2, None),
                                          # E % 8 != 0 (W_router read from a padded copy):
                                          # small-batch and tensor-core routers
                                          (100, 256, 1, 1, None), (64, 264, 4, 3, 1.0),
                                          (128, 136, 6, 6, None), (200, 136, 2, 2, None),
                                          (300, 520, 6, 4, 0.5), (1000, 256, 13, 5, None),
                                          (300, 128, 250, 8, None), (129, 64, 1, 1, None)])
def test_router_edge_shapes(T, H, E, k, bias):
    cfg = moe_synth.MoEConfig("edge", T=T, H=H, F=0, E=E, k=k, seed=11, bias0=bias)
    inputs = moe_synth.make_inputs(cfg, with_ffn=False)
    r = gpu_route(cfg, to_dev(inputs))
    routing_parity(cfg, inputs, r)


@pytest.mark.parametrize("T,E,k", [(2048, 128, 2), (2688, 64, 3), (3840, 128, 1), (6400, 16, 2),
                                   (2688, 192, 2)])
def test_router_tile_counts(T, E, k):
    # 16, 21, 30 and 50 tiles of 128 tokens: the K split per tile (the most,
    # up to 8, whose clusters all fit in one wave) changes across these
    # counts, and with it the rows each rank reduces; E = 192 takes the
    # widest accumulator (three 64-expert column blocks)
    cfg = moe_synth.MoEConfig("tiles", T=T, H=1024, F=0, E=E, k=k, seed=31)
    inputs = moe_synth.make_inputs(cfg, with_ffn=False)
    r = gpu_route(cfg, to_dev(inputs))
    routing_parity(cfg, inputs, r)


def test_router_duplicate_columns_tie_to_lower_index():
    cfg = moe_synth.MoEConfig("ties", T=200, H=256, F=0, E=16, k=4, seed=12)
    inputs = moe_synth.make_inputs(cfg, with_ffn=False)
    inputs["w_router"][:, 9] = inputs["w_router"][:, 4]  # experts 4 and 9 tie exactly
    r = gpu_route(cfg, to_dev(inputs))
    ids = np_(r.ids)
    seen = 0
    for t in range(cfg.T):
        row = ids[t].tolist()
        if 4 in row and 9 in row:
            assert row.index(4) + 1 == row.index(9)
            seen += 1
        elif 9 in row:
            raise AssertionError(f"token {t} picked 9 without 4: {row}")
    assert seen > 0


# ---------------------------------------------------------------- forward --

def test_forward_tiny_all_rows():
    forward_parity(moe_synth.TINY)


def test_forward_decode_all_rows():
    cfg = moe_synth.DECODE
    rep = forward_parity(cfg)
    # every expert is hit at least once on this seed
    inputs = moe_synth.make_inputs(cfg, with_ffn=False)
    _, ids, _, _ = oracle.route(inputs["x"], inputs["w_router"], cfg.k)
    assert len(np.unique(ids)) == cfg.E
    assert rep["near_tie_tokens"] >= 0


def test_forward_prefill_sampled():
    forward_parity(moe_synth.PREFILL, stride=16)


@pytest.mark.parametrize("cfg", [moe_synth.SKEWED, moe_synth.SKEWED_CF], ids=lambda c: c.name)
def test_forward_skewed_sampled(cfg):
    rep = forward_parity(cfg, stride=16)
    if cfg.capacity_factor is not None:
        assert rep["dropped"] > 0


@pytest.mark.parametrize("T,H,F,E,k,cf,bias", [
    (1, 64, 64, 8, 1, None, None),          # one token
    (7, 136, 200, 8, 2, None, None),        # ragged H, F (not multiples of 64 / 256)
    (300, 128, 520, 16, 8, None, None),     # k = 8, many ragged row blocks
    (200, 256, 264, 8, 2, 0.3, 3.0),        # heavy drops, skewed
    (150, 64, 128, 8, 1, None, 50.0),       # all tokens to expert 0, others empty
    (33, 512, 1408, 64, 4, 1.0, None),      # many experts with 0-3 rows
    (129, 72, 8, 8, 3, None, None),         # F = 8
    (50, 128, 256, 1, 1, None, None),       # one expert
    (200, 64, 128, 2, 2, None, None),       # two experts, both chosen by every token
    (129, 256, 264, 4, 3, None, 1.0),       # four experts, tensor-core router
    (300, 136, 200, 6, 4, 0.8, None),       # six experts, drops
    (500, 256, 256, 13, 2, None, None),     # thirteen experts
    (190, 1000, 264, 96, 2, None, None),    # one-launch route, 64-token tiles x 8 K splits, ragged K
    (2100, 1024, 256, 128, 1, 1.1, None),   # 64-token tiles x 4 splits, k = 1 combine in GEMM2, drops
])
def test_forward_edge_shapes(T, H, F, E, k, cf, bias):
    cfg = moe_synth.MoEConfig("edge", T=T, H=H, F=F, E=E, k=k, seed=21, capacity_factor=cf,
                              bias0=bias)
    forward_parity(cfg)


def test_forward_all_dropped_rows_are_zero():
    cfg = moe_synth.MoEConfig("drop", T=256, H=64, F=64, E=8, k=2, seed=22, capacity_factor=0.05,
                              bias0=8.0)
    inputs = moe_synth.make_inputs(cfg)
    layer, y = gpu_forward(cfg, to_dev(inputs))
    slot = np_(layer.routing.slot)
    dead = np.all(slot < 0, axis=1)
    assert dead.any()
    assert torch.all(y[torch.from_numpy(dead).to(DEV)] == 0)
    forward_parity(cfg)


def test_forward_empty_batch():
    cfg = moe_synth.TINY
    inputs = to_dev(moe_synth.make_inputs(cfg))
    s = moe.make_shape(0, cfg.H, cfg.F, cfg.E, cfg.k)
    r = moe.alloc_routing(0, cfg.E, cfg.k, DEV)
    r.counts.fill_(7)
    r.offsets.fill_(7)
    ws = torch.empty(1024, dtype=torch.uint8, device=DEV)
    y = torch.empty(0, cfg.H, dtype=torch.bfloat16, device=DEV)
    x0 = torch.empty(0, cfg.H, dtype=torch.bfloat16, device=DEV)
    moe.moe_forward(s, x0, inputs["w_router"], None, inputs["w1"], inputs["w2"], y, r.ids, r.weights,
                    r.counts, r.offsets, r.perm, r.slot, ws)
    assert moe.moe_get_device_status(ws) == 0
    assert np_(r.counts).tolist() == [0] * cfg.E and np_(r.offsets).tolist() == [0] * (cfg.E + 1)


def test_forward_is_deterministic_and_graph_capturable():
    cfg = moe_synth.MoEConfig("det", T=512, H=256, F=512, E=16, k=4, seed=23)
    dev_in = to_dev(moe_synth.make_inputs(cfg))
    layer, y = gpu_forward(cfg, dev_in)
    y1 = y.clone()
    ids1 = layer.routing.ids.clone()
    y.zero_()
    layer(dev_in["x"])
    torch.cuda.synchronize()
    assert torch.equal(y1, layer.y) and torch.equal(ids1, layer.routing.ids)
    # the same call captured in a CUDA graph and replayed gives the same bits
    stream = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    layer.y.zero_()
    with torch.cuda.graph(g, stream=stream):
        layer(dev_in["x"])
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(y1, layer.y)


def test_split_entry_points_match_forward():
    cfg = moe_synth.MoEConfig("split", T=300, H=192, F=320, E=16, k=2, seed=24, capacity_factor=0.9)
    dev_in = to_dev(moe_synth.make_inputs(cfg))
    layer, y = gpu_forward(cfg, dev_in)
    s = moe.make_shape(cfg.T, cfg.H, cfg.F, cfg.E, cfg.k, cfg.capacity_factor)
    r = moe.alloc_routing(cfg.T, cfg.E, cfg.k, DEV)
    ws = moe.alloc_workspace(s, DEV)
    moe.moe_route(s, dev_in["x"], dev_in["w_router"], None, r.ids, r.weights, r.counts, r.offsets,
                  r.perm, r.slot, ws)
    y2 = torch.empty_like(y)
    moe.moe_expert_ffn_combine(s, dev_in["x"], dev_in["w1"], dev_in["w2"], r.weights, r.offsets,
                               r.perm, r.slot, y2, ws)
    assert moe.moe_get_device_status(ws) == 0
    assert torch.equal(y, y2)
    for a, b in [(r.ids, layer.routing.ids), (r.slot, layer.routing.slot), (r.perm, layer.routing.perm)]:
        assert torch.equal(a, b)


def test_back_to_back_steps_with_overlapped_launch():
    # consecutive forwards share the routing buffers and the workspace; the
    # kernels after the first of each call start early (programmatic
    # dependent launch), so alternate two inputs into two outputs inside one
    # graph and compare each with a lone eager call
    cfg = moe_synth.MoEConfig("chain", T=384, H=256, F=512, E=16, k=2, seed=26)
    dev_in = to_dev(moe_synth.make_inputs(cfg))
    xb = torch.roll(dev_in["x"], 7, dims=0) * -0.5
    layer, _ = gpu_forward(cfg, dev_in)
    r = layer.routing
    ys = [torch.empty_like(layer.y) for _ in range(2)]
    refs = []
    for x in (dev_in["x"], xb):
        moe.moe_forward(layer.shape, x, layer.w_router, layer.bias, layer.w1, layer.w2, layer.y,
                        r.ids, r.weights, r.counts, r.offsets, r.perm, r.slot, layer.ws)
        refs.append(layer.y.clone())
    assert not torch.equal(refs[0], refs[1])
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=torch.cuda.Stream()):
        for i in range(12):
            moe.moe_forward(layer.shape, (dev_in["x"], xb)[i % 2], layer.w_router, layer.bias,
                            layer.w1, layer.w2, ys[i % 2], r.ids, r.weights, r.counts, r.offsets,
                            r.perm, r.slot, layer.ws)
    for _ in range(3):
        ys[0].zero_()
        ys[1].zero_()
        g.replay()
        torch.cuda.synchronize()
        assert moe.moe_get_device_status(layer.ws) == 0
        assert torch.equal(ys[0], refs[0]) and torch.equal(ys[1], refs[1])


def test_profiled_forward_eager_and_captured():
    cfg = moe_synth.MoEConfig("prof", T=256, H=128, F=256, E=8, k=2, seed=25)
    dev_in = to_dev(moe_synth.make_inputs(cfg))
    layer, y_ref = gpu_forward(cfg, dev_in)
    y_ref = y_ref.clone()
    r = layer.routing
    nk = len(moe.KERNEL_NAMES)
    evs = [torch.cuda.Event(enable_timing=True) for _ in range(nk + 1)]
    for e in evs:
        e.record()
    args = (layer.shape, dev_in["x"], layer.w_router, layer.bias, layer.w1, layer.w2, layer.y, r.ids,
            r.weights, r.counts, r.offsets, r.perm, r.slot, layer.ws)
    moe.moe_forward_profiled(*args, evs)  # eager
    torch.cuda.synchronize()
    times = [evs[i].elapsed_time(evs[i + 1]) for i in range(nk)]
    assert all(t >= 0 for t in times)
    assert torch.equal(layer.y, y_ref)
    g = torch.cuda.CUDAGraph()  # captured: events become timed graph nodes
    with torch.cuda.graph(g, stream=torch.cuda.Stream()):
        moe.moe_forward_profiled(*args, evs)
    layer.y.zero_()
    g.replay()
    torch.cuda.synchronize()
    assert all(evs[i].elapsed_time(evs[i + 1]) >= 0 for i in range(nk))
    assert torch.equal(layer.y, y_ref)


# ------------------------------------------------------- gating variants --

@pytest.mark.parametrize("gating", [moe.MOE_GATE_SOFTMAX_TOPK, moe.MOE_GATE_SOFTMAX_TOPK_RENORM])
@pytest.mark.parametrize("E,k", [(8, 2), (64, 4), (128, 8), (16, 16)])
def test_router_softmax_over_all_experts(gating, E, k):
    if k > 8:
        k = 8
    cfg = moe_synth.MoEConfig("gate", T=300, H=256, F=0, E=E, k=k, seed=40 + E, bias0=0.5)
    inputs = moe_synth.make_inputs(cfg, with_ffn=False)
    r = gpu_route(cfg, to_dev(inputs), gating)
    routing_parity(cfg, inputs, r, gating=gating)
    w = np_(r.weights).astype(np.float64).sum(1)
    if gating == moe.MOE_GATE_SOFTMAX_TOPK:
        assert np.all(w <= 1 + 1e-5) and (k == E or np.all(w < 1))
    else:
        np.testing.assert_allclose(w, 1.0, atol=1e-5)


@pytest.mark.parametrize("gating", [moe.MOE_GATE_SOFTMAX_TOPK, moe.MOE_GATE_SOFTMAX_TOPK_RENORM])
def test_forward_softmax_over_all_experts(gating):
    cfg = moe_synth.MoEConfig("gatefwd", T=200, H=256, F=384, E=16, k=4, seed=44,
                              capacity_factor=1.1)
    forward_parity(cfg, gating=gating)


def test_load_cv_diagnostic():
    cfg = moe_synth.SKEWED
    inputs = moe_synth.make_inputs(cfg, with_ffn=False)
    r = gpu_route(cfg, to_dev(inputs))
    counts = np_(r.counts).astype(np.float64)
    assert moe.load_cv(r.counts) == pytest.approx(counts.std() / counts.mean(), rel=1e-9)
    assert moe.load_cv(r.counts) > 1.0  # expert 0 takes ~99% of the tokens


# ------------------------------------------------------ gated (SwiGLU) experts --

@pytest.mark.parametrize("T,H,F,E,k,cf", [
    (64, 128, 256, 8, 2, None),      # tiny shape
    (300, 136, 200, 16, 4, 0.8),     # ragged H and F (F not a multiple of 128), drops
    (7, 64, 64, 8, 1, None),         # a few tokens
])
def test_forward_swiglu_edge_shapes(T, H, F, E, k, cf):
    cfg = moe_synth.MoEConfig("swiglu", T=T, H=H, F=F, E=E, k=k, seed=50, capacity_factor=cf,
                              act="swiglu")
    forward_parity(cfg)


def test_forward_swiglu_decode_all_rows():
    forward_parity(moe_synth.DECODE_SWIGLU)


def test_forward_swiglu_prefill_sampled():
    forward_parity(moe_synth.PREFILL_SWIGLU, stride=16)


# ------------------------------------------- k = 1: combine fused into GEMM2 --

@pytest.mark.parametrize("act", ["gelu", "swiglu"])
def test_forward_k1_drops_zero_rows_written(act):
    # y starts as NaN everywhere: dropped tokens must be written as 0 and
    # kept tokens as w * expert output, with no combine kernel
    cfg = moe_synth.MoEConfig("k1drop", T=300, H=136, F=264, E=8, k=1, seed=60,
                              capacity_factor=0.5, bias0=2.0, act=act)
    inputs = moe_synth.make_inputs(cfg)
    dev_in = to_dev(inputs)
    layer = moe.MoELayer(dev_in["w_router"], dev_in["w1"], dev_in["w2"], 1, bias=dev_in["bias"],
                         capacity_factor=cfg.capacity_factor, act=act)
    layer._ensure(cfg.T, dev_in["x"].device)
    layer.y.view(torch.int16).fill_(0x7FC0)  # bf16 NaN
    r = layer.routing
    moe.moe_forward(layer.shape, dev_in["x"], layer.w_router, layer.bias, layer.w1, layer.w2, layer.y,
                    r.ids, r.weights, r.counts, r.offsets, r.perm, r.slot, layer.ws)
    assert moe.moe_get_device_status(layer.ws) == 0
    y = layer.y
    assert not torch.isnan(y).any()
    dead = torch.from_numpy(np_(r.slot)[:, 0] < 0).to(DEV)
    assert dead.any() and (~dead).any()
    assert torch.all(y[dead] == 0)
    logits, rep = routing_parity(cfg, inputs, r)
    rows = np.arange(cfg.T, dtype=np.int32)
    y_ref = reference_y(inputs, logits, np_(r.ids), np_(r.slot), rows)
    check_y(y.float().cpu().numpy(), y_ref)


def test_forward_k1_softmax_over_all_experts():
    # the gate weight of the single expert is below 1 here, so a missing
    # scale would show
    cfg = moe_synth.MoEConfig("k1gate", T=200, H=256, F=384, E=16, k=1, seed=61)
    rep = forward_parity(cfg, gating=moe.MOE_GATE_SOFTMAX_TOPK)
    assert rep["dropped"] == 0


def test_forward_k1_prefill_sampled():
    forward_parity(moe_synth.PREFILL_K1, stride=16)


# ------------------------------------------- expert parallelism (simulated) --

def _exchange_locally(layers, routed, padded):
    """The two all-to-alls of an expert-parallel step for G ranks held in
    one process: slices of the senders' rows, concatenated per receiver."""
    G = len(layers)
    backs = [None] * G
    if padded:
        cap = routed[0].rows.shape[0] // G
        outs = []
        for d in range(G):
            recv = torch.cat([routed[s].rows[d * cap:(d + 1) * cap] for s in range(G)])
            counts = torch.stack([routed[s].send_counts[d] for s in range(G)])
            outs.append(layers[d].compute(recv, counts).clone())
        for s in range(G):
            backs[s] = torch.cat([outs[d][s * cap:(s + 1) * cap] for d in range(G)])
        return backs
    splits = [r.send_counts.sum(dim=1).tolist() for r in routed]   # splits[s][d]
    starts = [np.concatenate([[0], np.cumsum(sp)]).tolist() for sp in splits]
    outs = []
    for d in range(G):
        counts = torch.stack([routed[s].send_counts[d] for s in range(G)])
        rows = torch.cat([routed[s].rows[starts[s][d]:starts[s][d + 1]] for s in range(G)])
        outs.append((layers[d].compute(rows, counts).clone(), [splits[s][d] for s in range(G)]))
    for s in range(G):
        parts = []
        for d in range(G):
            Y, recv = outs[d]
            off = int(sum(recv[:s]))
            parts.append(Y[off:off + recv[s]])
        backs[s] = torch.cat(parts)
    return backs


@pytest.mark.parametrize("padded", [False, True], ids=["exact", "padded"])
@pytest.mark.parametrize("G,T,H,F,E,k,cf,bias,act", [
    (2, 512, 256, 512, 8, 2, None, None, "gelu"),
    (4, 700, 256, 384, 8, 4, 0.8, 2.0, "gelu"),      # drops, skew, ragged
    (2, 300, 128, 256, 16, 2, None, None, "swiglu"),
    (2, 256, 128, 256, 8, 1, 0.7, 1.0, "gelu"),      # k = 1 (the whole layer fuses its combine)
])
def test_expert_parallel_ranks_match_whole_layer(G, T, H, F, E, k, cf, bias, act, padded):
    from mixture_experts_layer_12_gb300.expert_parallel import CudaOps, ExpertParallelMoE
    cfg = moe_synth.MoEConfig("ep", T=T, H=H, F=F, E=E, k=k, seed=80, capacity_factor=cf,
                              bias0=bias, act=act)
    full = to_dev(moe_synth.make_inputs(cfg))
    xs = [to_dev(moe_synth.make_inputs(cfg.with_(seed=90 + r), with_ffn=False))["x"]
          for r in range(G)]
    El = E // G
    layers = [ExpertParallelMoE(CudaOps(full["w_router"], full["w1"][r * El:(r + 1) * El],
                                        full["w2"][r * El:(r + 1) * El], k, E, bias=full["bias"],
                                        capacity_factor=cf, act=act), r, G, padded=padded)
              for r in range(G)]
    routed = [layers[r].send(xs[r]) for r in range(G)]
    backs = _exchange_locally(layers, routed, padded)
    whole = moe.MoELayer(full["w_router"], full["w1"], full["w2"], k, bias=full["bias"],
                         capacity_factor=cf, act=act)
    full_cpu = moe_synth.make_inputs(cfg)
    for r in range(G):
        y = layers[r].finish(routed[r], backs[r]).clone()
        # against the oracle: each rank's routing and dispatch over its own
        # tokens, and its y from the oracle's combine on those decisions
        inputs_r = dict(full_cpu, x=xs[r].cpu())
        logits, _ = routing_parity(cfg, inputs_r, routed[r])
        y_ora = reference_y(inputs_r, logits, np_(routed[r].ids), np_(routed[r].slot),
                            np.arange(T, dtype=np.int32))
        check_y(y.float().cpu().numpy(), y_ora)
        # and against the single-GPU layer on the same tokens
        y_ref = whole(xs[r]).clone()
        assert moe.moe_get_device_status(whole.ws) == 0
        if k > 1:
            assert torch.equal(y, y_ref), f"rank {r}"
        else:  # the whole layer rounds w * acc once; here Y is rounded first
            check_y(y.float().cpu().numpy(), y_ref.double().cpu().numpy())


def test_expert_parallel_padded_phases_need_no_host_sync():
    # the padded mode's local phases -- routing and send blocks, expert FFN of
    # the received blocks, return to dispatch order and combine -- captured
    # in CUDA graphs (a device-to-host read would fail the capture) and
    # replayed: the replay reproduces the eager result
    from mixture_experts_layer_12_gb300.expert_parallel import CudaOps, ExpertParallelMoE
    G, cfg = 2, moe_synth.MoEConfig("epg", T=64, H=256, F=512, E=8, k=2, seed=81)
    full = to_dev(moe_synth.make_inputs(cfg))
    xs = [to_dev(moe_synth.make_inputs(cfg.with_(seed=95 + r), with_ffn=False))["x"]
          for r in range(G)]
    El = cfg.E // G
    layers = [ExpertParallelMoE(CudaOps(full["w_router"], full["w1"][r * El:(r + 1) * El],
                                        full["w2"][r * El:(r + 1) * El], cfg.k, cfg.E), r, G,
                                padded=True) for r in range(G)]
    routed = [layers[r].send(xs[r]) for r in range(G)]  # eager warm-up allocates the buffers
    backs = _exchange_locally(layers, routed, True)
    y_eager = [layers[r].finish(routed[r], backs[r]).clone() for r in range(G)]
    st = torch.cuda.Stream()
    gs = [torch.cuda.CUDAGraph() for _ in range(3)]
    with torch.cuda.graph(gs[0], stream=st):
        routed = [layers[r].send(xs[r]) for r in range(G)]
        recv = [torch.cat([routed[s].rows.chunk(G)[d] for s in range(G)]) for d in range(G)]
        counts = [torch.stack([routed[s].send_counts[d] for s in range(G)]) for d in range(G)]
    with torch.cuda.graph(gs[1], stream=st):
        outs = [layers[d].compute(recv[d], counts[d]) for d in range(G)]
        back = [torch.cat([outs[d].chunk(G)[s] for d in range(G)]) for s in range(G)]
    with torch.cuda.graph(gs[2], stream=st):
        ys = [layers[r].finish(routed[r], back[r]) for r in range(G)]
    for y in ys:
        y.zero_()
    for g in gs:
        g.replay()
    torch.cuda.synchronize()
    for r in range(G):
        assert torch.equal(ys[r], y_eager[r]), f"rank {r}"


# ------------------------------------------- the step entry points, one by one --

@pytest.mark.parametrize("T,H,E,k,cf", [(300, 256, 16, 3, 0.7), (64, 136, 8, 1, None),
                                        (1000, 64, 32, 8, 0.4)])
def test_combine_entry_point_against_oracle(T, H, E, k, cf):
    # moe_combine alone on random expert outputs Y and a dispatch with drops:
    # y[t] = sum over kept j of w[t, j] * Y[slot[t, j]] against the oracle
    rng = np.random.default_rng(T + H)
    ids = np.stack([rng.choice(E, size=k, replace=False) for _ in range(T)]).astype(np.int32)
    _, offsets, _, slot = oracle.dispatch(ids, E, cf)
    g = torch.Generator().manual_seed(T)
    Y = torch.randn(T * k, H, generator=g).to(torch.bfloat16)
    w = rng.uniform(0.0, 1.0, size=(T, k)).astype(np.float32)
    y = torch.full((T, H), float("nan"), dtype=torch.bfloat16, device=DEV)
    moe.moe_combine(moe.make_shape(T, H, 8, E, k, cf), Y.to(DEV), torch.from_numpy(w).to(DEV),
                    torch.from_numpy(slot).to(DEV), y)
    torch.cuda.synchronize()
    ref = oracle.combine_given(Y, w, slot)
    got = y.double().cpu().numpy()
    check_y(got, ref)
    # an fp32 sum of at most k products, rounded once to bf16: within half a
    # bf16 step of the exact sum, plus the fp32 rounding of the terms
    absum = oracle.combine_given(Y.abs(), np.abs(w), slot)
    bound = 2.0 ** -8 * np.abs(ref) + 1e-6 * absum
    assert np.all(np.abs(got - ref) <= bound)
    assert np.all(got[np.all(slot < 0, axis=1)] == 0.0)


@pytest.mark.parametrize("T,H,F,E,k,cf,act", [(500, 256, 384, 16, 2, 0.8, "gelu"),
                                              (96, 128, 256, 8, 4, None, "swiglu")])
def test_step_entry_points_against_oracle(T, H, F, E, k, cf, act):
    # moe_route -> moe_dispatch_rows -> moe_expert_ffn -> moe_combine: the
    # regrouped rows are x[perm // k] bit for bit, and y is the oracle's
    # combine on the GPU's routing decisions
    cfg = moe_synth.MoEConfig("steps", T=T, H=H, F=F, E=E, k=k, seed=85, capacity_factor=cf,
                              act=act)
    inputs = moe_synth.make_inputs(cfg)
    dev_in = to_dev(inputs)
    s = moe.make_shape(T, H, F, E, k, cf, act=act)
    r = moe.alloc_routing(T, E, k, DEV)
    ws = moe.alloc_workspace(s, DEV)
    moe.moe_route(s, dev_in["x"], dev_in["w_router"], None, r.ids, r.weights, r.counts, r.offsets,
                  r.perm, r.slot, ws)
    logits, rep = routing_parity(cfg, inputs, r)
    kept = rep["kept"]
    xp = torch.zeros(T * k, H, dtype=torch.bfloat16, device=DEV)
    moe.moe_dispatch_rows(s, dev_in["x"], r.perm, r.offsets, xp)
    perm = np_(r.perm)[:kept].astype(np.int64)
    assert torch.equal(xp[:kept].cpu(), inputs["x"][perm // k])
    Y = torch.empty(T * k, H, dtype=torch.bfloat16, device=DEV)
    moe.moe_expert_ffn(s, E, xp, dev_in["w1"], dev_in["w2"], r.offsets, Y, ws)
    y = torch.empty(T, H, dtype=torch.bfloat16, device=DEV)
    moe.moe_combine(s, Y, r.weights, r.slot, y)
    assert moe.moe_get_device_status(ws) == 0
    y_ref = reference_y(inputs, logits, np_(r.ids), np_(r.slot), np.arange(T, dtype=np.int32))
    check_y(y.float().cpu().numpy(), y_ref)
    # and moe_expert_ffn_combine, the same steps in one call, against the oracle too
    y2 = torch.full((T, H), float("nan"), dtype=torch.bfloat16, device=DEV)
    moe.moe_expert_ffn_combine(s, dev_in["x"], dev_in["w1"], dev_in["w2"], r.weights, r.offsets,
                               r.perm, r.slot, y2, ws)
    assert moe.moe_get_device_status(ws) == 0
    check_y(y2.float().cpu().numpy(), y_ref)


# ---------------------------------------------- host batches, copies overlapped --

@pytest.mark.parametrize("graphs", [False, True], ids=["launches", "graphs"])
def test_host_pipeline_matches_one_call_at_a_time(graphs):
    from mixture_experts_layer_12_gb300.host_pipeline import HostPipeline
    cfg = moe_synth.MoEConfig("pipe", T=256, H=256, F=512, E=8, k=2, seed=28)
    dev_in = to_dev(moe_synth.make_inputs(cfg))
    layer = moe.MoELayer(dev_in["w_router"], dev_in["w1"], dev_in["w2"], cfg.k)
    xs = [moe_synth.make_inputs(cfg.with_(seed=100 + i), with_ffn=False)["x"].pin_memory()
          for i in range(5)]
    refs = [layer(x.to(DEV)).cpu() for x in xs]
    ys = [torch.full((cfg.T, cfg.H), float("nan"), dtype=torch.bfloat16).pin_memory()
          for _ in range(5)]
    HostPipeline(layer, cfg.T, DEV, graphs=graphs).run(xs, ys)
    torch.cuda.synchronize()
    assert moe.moe_get_device_status(layer.ws) == 0
    for y, ref in zip(ys, refs):
        assert torch.equal(y, ref)


# ------------------------------------------------- the GEMM1 epilogue's GELU --

def _gelu_reference_check(x, Y):
    import math
    zz = x.double().cpu().reshape(-1).numpy()
    ref = np.array([0.5 * v * math.erfc(-v / math.sqrt(2.0)) for v in zz])
    got = Y.double().cpu().reshape(-1).numpy()
    err = np.abs(got - ref)
    near = zz >= -5.0  # |GELU| > 1.4e-6: within one bf16 step of the exact value
    assert np.all(err[near] <= 2.0 ** -7 * np.abs(ref[near]))
    # z < -5 (|GELU| < 1.4e-6): Abramowitz & Stegun 7.1.26's relative error
    # grows to 2.0% at z = -10 (|GELU| ~ 1e-18), plus half a bf16 step
    assert np.all(err[~near] <= 0.03 * np.abs(ref[~near]))
    assert np.all(np.sign(got) == np.sign(ref))
    return zz, got


def test_gelu_epilogue_elementwise_against_fp64():
    # W1 = W2 = I (one expert, H = F = 64): Y = h = bf16(GELU(x)) element by
    # element, so the epilogue's GELU is seen directly for z in [-10, 10]
    T, H = 1024, 64
    eye = torch.eye(H, dtype=torch.bfloat16, device=DEV).reshape(1, H, H).contiguous()
    z = torch.linspace(-10.0, 10.0, T * H, dtype=torch.float64)
    z[T * H // 2] = 0.0
    x = z.to(torch.bfloat16).reshape(T, H).to(DEV)
    s = moe.make_shape(T, H, H, 1, 1)
    ws = moe.alloc_workspace(s, DEV)
    Y = torch.empty(T, H, dtype=torch.bfloat16, device=DEV)
    seg = torch.tensor([0, T], dtype=torch.int32, device=DEV)
    moe.moe_expert_ffn(s, 1, x, eye, eye, seg, Y, ws)
    assert moe.moe_get_device_status(ws) == 0
    _, got = _gelu_reference_check(x, Y)
    assert got[T * H // 2] == 0.0


def test_gelu_epilogue_small_batch_kernel():
    # 64 rows in 64 one-row segments of one expert, F = 10240: 2560 column
    # tiles, so GEMM1 runs on the small-batch kernel (weights as the MMA's M
    # operand); W1 = [I | 0] and W2 = [I ; 0] expose h[:, :64] = GELU(x)
    T, H, F = 64, 64, 10240
    w1 = torch.zeros(1, H, F, dtype=torch.bfloat16, device=DEV)
    w1[0, :, :H] = torch.eye(H, dtype=torch.bfloat16, device=DEV)
    w2 = torch.zeros(1, F, H, dtype=torch.bfloat16, device=DEV)
    w2[0, :H, :] = torch.eye(H, dtype=torch.bfloat16, device=DEV)
    z = torch.linspace(-10.0, 10.0, T * H, dtype=torch.float64)
    x = z.to(torch.bfloat16).reshape(T, H).to(DEV)
    s = moe.make_shape(T, H, F, 1, 1)
    ws = moe.alloc_workspace(s, DEV)
    Y = torch.empty(T, H, dtype=torch.bfloat16, device=DEV)
    seg = torch.arange(T + 1, dtype=torch.int32, device=DEV)
    moe.moe_expert_ffn(s, T, x, w1, w2, seg, Y, ws)
    assert moe.moe_get_device_status(ws) == 0
    _gelu_reference_check(x, Y)


def test_expert_ffn_row_block_boundaries():
    # segments of 0, 1, 64, 127, 128, 129, 255, 256, 257, 384 and 385 rows
    # (segment i on expert i % 4): every kind of last row block -- none, at
    # most 128 rows (an M = 128 tile, 64 rows per CTA), a full 256-row tile
    # -- checked row by row against the oracle
    sizes = [0, 1, 64, 127, 128, 129, 255, 256, 257, 384, 385]
    rows = sum(sizes)
    cfg = moe_synth.MoEConfig("tailblocks", T=rows, H=256, F=384, E=4, k=1, seed=37)
    inp = moe_synth.make_inputs(cfg)
    s = moe.make_shape(rows, cfg.H, cfg.F, cfg.E, 1)
    ws = moe.alloc_workspace(s, DEV)
    seg = torch.tensor(np.concatenate([[0], np.cumsum(sizes)]), dtype=torch.int32, device=DEV)
    Y = torch.empty(rows, cfg.H, dtype=torch.bfloat16, device=DEV)
    moe.moe_expert_ffn(s, len(sizes), inp["x"].to(DEV), inp["w1"].to(DEV), inp["w2"].to(DEV), seg,
                       Y, ws)
    assert moe.moe_get_device_status(ws) == 0
    ref = np.empty((rows, cfg.H))
    r = 0
    for i, n in enumerate(sizes):
        for _ in range(n):
            ref[r] = oracle.expert_ffn(inp["x"][r], inp["w1"][i % cfg.E], inp["w2"][i % cfg.E])
            r += 1
    check_y(Y.float().cpu().numpy(), ref)


# ----------------------------------------------- small batches (T*k <= 64 rows) --

# The small-batch kernel runs a GEMM when it has at least two waves of column
# tiles (2 x 76 pairs on a GB300): F = 5120 over 8 experts gives GEMM1 160
# tiles, H = 5120 gives GEMM2 160; the other shapes stay on the main kernel.
@pytest.mark.parametrize("T,H,F,E,k,cf,bias", [
    (16, 256, 5120, 8, 4, None, None),   # GEMM1 small: 64 rows over 8 experts
    (40, 5120, 512, 8, 1, 0.5, None),    # GEMM2 small with the k = 1 combine; drops
    (21, 264, 1408, 16, 3, 0.7, None),   # ragged H and F, drops (main kernel)
    (64, 256, 296, 8, 1, None, 50.0),    # every row on one expert (main kernel)
])
def test_forward_small_batch_weights_as_m_operand(T, H, F, E, k, cf, bias):
    cfg = moe_synth.MoEConfig("smallgemm", T=T, H=H, F=F, E=E, k=k, seed=33, capacity_factor=cf,
                              bias0=bias)
    forward_parity(cfg)
