"""Pins of the CPU oracle against what the pages and the mathematics fix.

None of these re-types an oracle formula: each compares the oracle with an
independent construction (hand-derived closed forms, brute force, a second
formulation, a library routine used as a step, or an exact identity), chosen
so that a dropped term, a wrong sign or index, or a transposed operand in
``oracle/moe_oracle.c`` fails at least one of them.
"""
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
import moe_synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "worked_example.json")


def bf16(a) -> torch.Tensor:
    return torch.as_tensor(np.asarray(a, dtype=np.float32)).to(torch.bfloat16)


def f64(t: torch.Tensor) -> np.ndarray:
    return t.to(torch.float64).numpy()


def rand_bf16(shape, std, seed):
    g = torch.Generator().manual_seed(seed)
    return (torch.randn(*shape, generator=g) * std).to(torch.bfloat16)


def gelu_np(z):
    return 0.5 * z * (1.0 + np.vectorize(math.erf)(z / math.sqrt(2.0)))


# ---------------------------------------------------------------- golden ----

@pytest.fixture(scope="module")
def golden():
    with open(GOLDEN) as f:
        return json.load(f)


def _golden_inputs(g):
    return (bf16(g["x"]), bf16(g["w_router"]), bf16(g["w1"]), bf16(g["w2"]))


def test_golden_routing(golden):
    x, wr, _, _ = _golden_inputs(golden)
    logits, ids, vals, w = oracle.route(x, wr, golden["k"])
    np.testing.assert_array_equal(logits, np.array(golden["expected"]["logits"], np.float32))
    np.testing.assert_array_equal(ids, golden["expected"]["ids"])
    np.testing.assert_allclose(w, golden["expected"]["w"], rtol=0, atol=1e-7)


@pytest.mark.parametrize("case,cf", [("no_cap", None), ("cf_1.0", 1.0)])
def test_golden_dispatch_and_combine(golden, case, cf):
    x, wr, w1, w2 = _golden_inputs(golden)
    exp = golden["expected"][case]
    out = oracle.moe_forward(x, wr, w1, w2, golden["k"], capacity_factor=cf)
    if cf is not None:
        assert oracle.capacity(golden["T"], golden["k"], golden["E"], cf) == exp["capacity"]
    np.testing.assert_array_equal(out["counts"], exp["counts"])
    np.testing.assert_array_equal(out["offsets"], exp["offsets"])
    n = exp["offsets"][-1]
    np.testing.assert_array_equal(out["perm"][:n], exp["perm"])
    np.testing.assert_array_equal(out["slot"], exp["slot"])
    # w is fp32 (rounded once from double), so y matches to fp32 resolution.
    np.testing.assert_allclose(out["y"], exp["y"], rtol=2e-7, atol=1e-12)


def test_golden_gelu_fixed_points(golden):
    # 1x1 expert: y = GELU(x) for x in {1, -1, 0}; GELU(-z) = GELU(z) - z.
    one = bf16([[1.0]])
    for xv, want in [(1.0, golden["expected"]["gelu_1"]),
                     (-1.0, golden["expected"]["gelu_1"] - 1.0),
                     (0.0, 0.0)]:
        y = oracle.expert_ffn(bf16([xv]), one, one)
        assert abs(y[0] - want) < 1e-15


# ------------------------------------------------------------ router GEMM ---

@pytest.mark.parametrize("T,H,E,with_bias", [(7, 24, 5, False), (33, 136, 16, True), (5, 8, 1, True)])
def test_logits_against_fp64_matmul(T, H, E, with_bias):
    x = rand_bf16((T, H), 1.0, 1)
    wr = rand_bf16((H, E), 1.0 / math.sqrt(H), 2)
    bias = np.linspace(-3, 3, E).astype(np.float32) if with_bias else None
    got = oracle.router_logits(x, wr, bias)
    ref = (f64(x) @ f64(wr)).astype(np.float32)  # one fp64 library matmul, one rounding
    if bias is not None:
        ref = ref + bias
    # Same double sum up to summation order, then one rounding to fp32.
    np.testing.assert_allclose(got, ref, rtol=1.2e-7, atol=1e-30)
    # A transposed operand would not even be shape-compatible when H != E;
    # check the orientation explicitly with a one-hot router.
    onehot = torch.zeros(H, E, dtype=torch.bfloat16)
    onehot[H - 1, E - 1] = 1.0
    lg = oracle.router_logits(x, onehot)
    np.testing.assert_array_equal(lg[:, E - 1], f64(x)[:, H - 1].astype(np.float32))
    if E > 1:
        assert np.all(lg[:, : E - 1] == 0)


# ------------------------------------------------------------------ TopK ----

def _brute_topk(lg, k):
    # Full sort of (-logit, expert) pairs: descending logit, ties -> lower index.
    return np.array([[e for _, e in sorted((-float(v), e) for e, v in enumerate(row))][:k]
                     for row in lg], dtype=np.int32)


def _argmax_passes(lg, k):
    # k passes of a strict '>' argmax (the first maximum wins), masking winners.
    out = []
    for row in lg:
        taken, ids = set(), []
        for _ in range(k):
            best, bi = None, -1
            for e, v in enumerate(row):
                if e in taken:
                    continue
                if best is None or v > best:
                    best, bi = v, e
            taken.add(bi)
            ids.append(bi)
        out.append(ids)
    return np.array(out, dtype=np.int32)


@pytest.mark.parametrize("E", [1, 2, 3, 8, 16])
def test_topk_brute_force_with_ties(E):
    rng = np.random.default_rng(E)
    # small integer logits: many exact ties
    lg = rng.integers(-3, 4, size=(200, E)).astype(np.float32)
    for k in range(1, min(8, E) + 1):
        ids, vals = oracle.topk(lg, k)
        np.testing.assert_array_equal(ids, _brute_topk(lg, k))
        np.testing.assert_array_equal(ids, _argmax_passes(lg, k))
        np.testing.assert_array_equal(vals, np.take_along_axis(lg, ids, axis=1))


def test_topk_duplicate_router_columns_pick_lower_index():
    T, H, E = 40, 64, 8
    x = rand_bf16((T, H), 1.0, 3)
    wr = rand_bf16((H, E), 0.125, 4)
    wr[:, 5] = wr[:, 2]  # experts 2 and 5 always tie exactly
    _, ids, _, w = oracle.route(x, wr, k=8)
    pos = {e: np.argmax(ids == e, axis=1) for e in (2, 5)}
    assert np.all(pos[2] + 1 == pos[5])  # adjacent, lower index first
    rows = np.arange(T)
    np.testing.assert_array_equal(w[rows, pos[2]], w[rows, pos[5]])


# ----------------------------------------------------------- gate softmax ---

def test_softmax_closed_forms_and_invariants():
    rng = np.random.default_rng(0)
    for k in range(1, 9):
        s = -np.sort(-rng.normal(size=(50, k)).astype(np.float32), axis=1)
        w = oracle.gate_softmax(s)
        np.testing.assert_allclose(w.astype(np.float64).sum(1), 1.0, atol=1e-6)
        if k == 1:
            assert np.all(w == 1.0)
        if k == 2:  # w0 = 1 / (1 + exp(s1 - s0))
            ref = 1.0 / (1.0 + np.exp(s[:, 1].astype(np.float64) - s[:, 0]))
            np.testing.assert_allclose(w[:, 0], ref, rtol=1e-7)
        # shift invariance (exact fp32 shift by a power of two)
        np.testing.assert_allclose(oracle.gate_softmax(s + np.float32(8.0)), w, rtol=0, atol=2e-7)
    eq = np.full((3, 2), 0.75, np.float32)
    assert np.all(oracle.gate_softmax(eq) == 0.5)
    # larger logit -> larger weight, and the order is kept
    w = oracle.gate_softmax(np.array([[3.0, 1.0, -2.0]], np.float32))
    assert w[0, 0] > w[0, 1] > w[0, 2]


def test_bias_shift_leaves_routing_unchanged():
    T, H, E = 30, 32, 6
    x = rand_bf16((T, H), 1.0, 5)
    wr = rand_bf16((H, E), 0.25, 6)
    _, ids0, _, w0 = oracle.route(x, wr, k=3, bias=np.zeros(E, np.float32))
    _, ids1, _, w1 = oracle.route(x, wr, k=3, bias=np.full(E, 0.5, np.float32))
    np.testing.assert_array_equal(ids0, ids1)
    np.testing.assert_allclose(w0, w1, atol=1e-6)


def test_softmax_over_all_experts_variant():
    special = pytest.importorskip("scipy.special")
    rng = np.random.default_rng(3)
    lg = rng.normal(size=(60, 12)).astype(np.float32)
    for k in (1, 3, 12):
        ids, vals = oracle.topk(lg, k)
        w1 = oracle.gate_softmax_all(lg, ids, 1)
        p = special.softmax(lg.astype(np.float64), axis=1)  # library softmax over all E
        np.testing.assert_allclose(w1, np.take_along_axis(p, ids.astype(np.int64), 1), rtol=1e-6)
        assert np.all(w1.astype(np.float64).sum(1) <= 1 + 1e-6)
        w2 = oracle.gate_softmax_all(lg, ids, 2)
        np.testing.assert_allclose(w2, oracle.gate_softmax(vals), rtol=0, atol=2e-7)
        if k == 12:  # selecting every expert: no renormalisation needed
            np.testing.assert_allclose(w1, oracle.gate_softmax(vals), rtol=0, atol=2e-7)
    with pytest.raises(RuntimeError):
        oracle.gate_softmax_all(lg, ids, 0)


# -------------------------------------------------------------- capacity ----

def test_capacity_values():
    assert oracle.capacity(8192, 4, 64, 1.2) == 615      # ceil(614.4)
    assert oracle.capacity(64, 2, 8, 1.0) == 16          # exact integer, no round-up
    assert oracle.capacity(10, 1, 3, 1.0) == 4           # ceil(3.33)
    assert oracle.capacity(3, 2, 3, 1.0) == 2
    assert oracle.capacity(6, 1, 4, 0.5) == 1            # ceil(0.75)
    assert oracle.capacity(100, 2, 8, None) == -1
    assert oracle.capacity(100, 2, 8, 0.0) == -1
    assert oracle.capacity(100, 2, 8, float("nan")) == -1
    assert oracle.capacity(100, 2, 8, 1e9) == 200        # clamped to T*k


# -------------------------------------------------------------- dispatch ----

def _brute_dispatch(ids, E, cap):
    T, k = ids.shape
    # enumerate all (t, j), stable-sort by expert, then keep the first cap of each
    entries = sorted(range(T * k), key=lambda i: ids.flat[i])
    counts = np.zeros(E, np.int32)
    kept = []
    for i in entries:
        e = ids.flat[i]
        if cap < 0 or counts[e] < cap:
            counts[e] += 1
            kept.append(i)
    offsets = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    slot = np.full(T * k, -1, np.int32)
    for r, i in enumerate(kept):
        slot[i] = r
    return counts, offsets, np.array(kept, np.int32), slot.reshape(T, k)


def _random_ids(T, E, k, rng, skew=False):
    ids = np.empty((T, k), np.int32)
    for t in range(T):
        p = None
        if skew:
            p = np.full(E, 1.0)
            p[0] = 8.0 * E
            p /= p.sum()
        ids[t] = rng.choice(E, size=k, replace=False, p=p)
    return ids


@pytest.mark.parametrize("T,E,k,cf,skew", [(1, 1, 1, None, False), (17, 4, 2, None, False),
                                           (50, 8, 3, 1.0, False), (64, 8, 2, 0.5, True),
                                           (33, 16, 4, 1.25, True), (20, 3, 3, 0.1, False)])
def test_dispatch_brute_force_and_invariants(T, E, k, cf, skew):
    rng = np.random.default_rng(T * 131 + E)
    ids = _random_ids(T, E, k, rng, skew)
    counts, offsets, perm, slot = oracle.dispatch(ids, E, cf)
    cap = oracle.capacity(T, k, E, cf)
    bc, bo, bp, bs = _brute_dispatch(ids, E, cap)
    np.testing.assert_array_equal(counts, bc)
    np.testing.assert_array_equal(offsets, bo)
    n = offsets[-1]
    np.testing.assert_array_equal(perm[:n], bp)
    np.testing.assert_array_equal(slot, bs)
    # invariants
    pre = np.bincount(ids.ravel(), minlength=E)
    np.testing.assert_array_equal(counts, pre if cap < 0 else np.minimum(pre, cap))
    assert n == counts.sum()
    assert len(set(perm[:n].tolist())) == n
    for r in range(n):
        assert slot.flat[perm[r]] == r  # slot o perm = identity
    for e in range(E):
        toks = perm[offsets[e]:offsets[e + 1]] // k
        assert np.all(np.diff(toks) > 0)  # ascending tokens within an expert
        assert np.all(ids.flat[perm[offsets[e]:offsets[e + 1]]] == e)
    if cap >= 0:  # dropped ones are exactly the later-token overflow
        for e in range(E):
            mine = [i for i in range(T * k) if ids.flat[i] == e]
            assert all(slot.flat[i] >= 0 for i in mine[:cap])
            assert all(slot.flat[i] == -1 for i in mine[cap:])


def test_dispatch_huge_capacity_equals_no_limit():
    rng = np.random.default_rng(9)
    ids = _random_ids(40, 8, 2, rng, skew=True)
    a = oracle.dispatch(ids, 8, None)
    b = oracle.dispatch(ids, 8, 1e6)
    for u, v in zip(a, b):
        np.testing.assert_array_equal(u, v)


def test_dispatch_rejects_bad_ids():
    with pytest.raises(RuntimeError):
        oracle.dispatch(np.array([[0, 5]], np.int32), 4)


# ------------------------------------------------------------ expert FFN ----

def test_identity_experts_reproduce_input():
    # F = 2H, W1 = [I | -I], W2 = [I ; -I]: GELU(z) - GELU(-z) = z, so the
    # expert is the identity; with k = 1 the gate weight is 1 and y = x.
    T, H, E = 12, 16, 3
    x = rand_bf16((T, H), 1.0, 7)
    eye = np.eye(H, dtype=np.float32)
    w1 = bf16(np.stack([np.concatenate([eye, -eye], 1)] * E))
    w2 = bf16(np.stack([np.concatenate([eye, -eye], 0)] * E))
    wr = rand_bf16((H, E), 0.25, 8)
    out = oracle.moe_forward(x, wr, w1, w2, k=1)
    np.testing.assert_allclose(out["y"], f64(x), rtol=0, atol=1e-12)


@pytest.mark.parametrize("H,F", [(8, 24), (40, 12)])
def test_expert_ffn_against_numpy(H, F):
    x = rand_bf16((H,), 1.0, 10)
    w1 = rand_bf16((H, F), 1.0 / math.sqrt(H), 11)
    w2 = rand_bf16((F, H), 1.0 / math.sqrt(F), 12)
    got = oracle.expert_ffn(x, w1, w2)
    ref = gelu_np(f64(x) @ f64(w1)) @ f64(w2)
    np.testing.assert_allclose(got, ref, rtol=1e-12, atol=1e-14)


def _silu_np(z):
    return z / (1.0 + np.exp(-z))


@pytest.mark.parametrize("H,F", [(8, 24), (40, 12)])
def test_expert_swiglu_against_numpy(H, F):
    x = rand_bf16((H,), 1.0, 13)
    w1 = rand_bf16((H, 2 * F), 1.0 / math.sqrt(H), 14)  # [gate | up]
    w2 = rand_bf16((F, H), 1.0 / math.sqrt(F), 15)
    got = oracle.expert_swiglu(x, w1, w2)
    X, W1, W2 = f64(x), f64(w1), f64(w2)
    ref = (_silu_np(X @ W1[:, :F]) * (X @ W1[:, F:])) @ W2
    np.testing.assert_allclose(got, ref, rtol=1e-12, atol=1e-14)
    # the halves are not interchangeable: swapping gate and up changes y
    swapped = torch.cat([w1[:, F:], w1[:, :F]], dim=1)
    assert not np.allclose(oracle.expert_swiglu(x, swapped, w2), got)
    # a zero gate (SiLU(0) = 0) or a zero up projection silences the expert
    for half in (slice(0, F), slice(F, 2 * F)):
        z = w1.clone()
        z[:, half] = 0
        assert np.all(oracle.expert_swiglu(x, z, w2) == 0.0)


def test_swiglu_fixed_points():
    # 1x1: y = SiLU(g) * u with g = x * wg, u = x * wu; SiLU(1) = 1/(1+e^-1)
    x = bf16([1.0])
    y = oracle.expert_swiglu(x, bf16([[1.0, 2.0]]), bf16([[1.0]]))
    assert abs(y[0] - 2.0 / (1.0 + math.exp(-1.0))) < 1e-15
    y = oracle.expert_swiglu(bf16([-2.0]), bf16([[1.0, 1.0]]), bf16([[1.0]]))
    assert abs(y[0] - (-2.0 / (1.0 + math.exp(2.0))) * -2.0) < 1e-15


def test_swiglu_combine_dense_masked():
    cfg = moe_synth.MoEConfig("t", T=20, H=16, F=24, E=4, k=2, seed=9)
    inp = moe_synth.make_inputs(cfg)
    g = torch.Generator().manual_seed(5)
    w1 = (torch.randn(cfg.E, cfg.H, 2 * cfg.F, generator=g) / math.sqrt(cfg.H)).to(torch.bfloat16)
    out = oracle.moe_forward(inp["x"], inp["w_router"], w1, inp["w2"], cfg.k, act="swiglu")
    X = f64(inp["x"])
    ref = np.zeros_like(X)
    for t in range(cfg.T):
        for j in range(cfg.k):
            e = out["ids"][t, j]
            W1, W2 = f64(w1[e]), f64(inp["w2"][e])
            ref[t] += out["w"][t, j] * ((_silu_np(X[t] @ W1[:, :cfg.F]) * (X[t] @ W1[:, cfg.F:])) @ W2)
    np.testing.assert_allclose(out["y"], ref, rtol=1e-10, atol=1e-12)


# --------------------------------------------------------------- combine ----

def _dense_masked(x, w1, w2, ids, w, slot, E):
    # second formulation: every expert on every token, gated by a dense mask
    X = f64(x)
    T = X.shape[0]
    gate = np.zeros((T, E))
    for t in range(T):
        for j in range(ids.shape[1]):
            if slot[t, j] >= 0:
                gate[t, ids[t, j]] += w[t, j]
    y = np.zeros_like(X)
    for e in range(E):
        y += gate[:, e:e + 1] * (gelu_np(X @ f64(w1[e])) @ f64(w2[e]))
    return y


@pytest.mark.parametrize("cf", [None, 0.75])
def test_combine_dense_masked_formulation(cf):
    cfg = moe_synth.MoEConfig("t", T=24, H=16, F=40, E=5, k=2, seed=3, bias0=1.5)
    inp = moe_synth.make_inputs(cfg)
    out = oracle.moe_forward(inp["x"], inp["w_router"], inp["w1"], inp["w2"], cfg.k,
                             bias=inp["bias"], capacity_factor=cf)
    ref = _dense_masked(inp["x"], inp["w1"], inp["w2"], out["ids"], out["w"], out["slot"], cfg.E)
    np.testing.assert_allclose(out["y"], ref, rtol=1e-10, atol=1e-12)
    if cf is not None:
        assert (out["slot"] < 0).any()  # the cap does drop something here


def test_identical_experts_ignore_routing():
    cfg = moe_synth.MoEConfig("t", T=16, H=8, F=12, E=4, k=3, seed=4)
    inp = moe_synth.make_inputs(cfg)
    w1 = inp["w1"][:1].repeat(cfg.E, 1, 1)
    w2 = inp["w2"][:1].repeat(cfg.E, 1, 1)
    out = oracle.moe_forward(inp["x"], inp["w_router"], w1, w2, cfg.k)
    ref = gelu_np(f64(inp["x"]) @ f64(w1[0])) @ f64(w2[0])
    np.testing.assert_allclose(out["y"], ref, rtol=2e-7, atol=1e-9)  # sum w = 1 in fp32


def test_token_permutation_permutes_output():
    cfg = moe_synth.MoEConfig("t", T=20, H=8, F=16, E=4, k=2, seed=5)
    inp = moe_synth.make_inputs(cfg)
    p = np.random.default_rng(1).permutation(cfg.T)
    a = oracle.moe_forward(inp["x"], inp["w_router"], inp["w1"], inp["w2"], cfg.k)
    b = oracle.moe_forward(inp["x"][p], inp["w_router"], inp["w1"], inp["w2"], cfg.k)
    np.testing.assert_array_equal(b["ids"], a["ids"][p])
    np.testing.assert_allclose(b["y"], a["y"][p], rtol=0, atol=0)


def test_all_slots_dropped_gives_zero_and_rows_subset():
    cfg = moe_synth.MoEConfig("t", T=30, H=8, F=8, E=4, k=2, seed=6, bias0=6.0)
    inp = moe_synth.make_inputs(cfg)
    out = oracle.moe_forward(inp["x"], inp["w_router"], inp["w1"], inp["w2"], cfg.k,
                             bias=inp["bias"], capacity_factor=0.2)
    dead = np.all(out["slot"] < 0, axis=1)
    assert dead.any()
    assert np.all(out["y"][dead] == 0.0)
    rows = np.arange(0, cfg.T, 7)
    sub = oracle.combine_rows(inp["x"], inp["w1"], inp["w2"], out["ids"], out["w"], out["slot"], rows)
    np.testing.assert_array_equal(sub, out["y"][rows])


def test_thread_count_does_not_change_results():
    cfg = moe_synth.MoEConfig("t", T=40, H=32, F=48, E=4, k=2, seed=8)
    inp = moe_synth.make_inputs(cfg)
    a = oracle.moe_forward(inp["x"], inp["w_router"], inp["w1"], inp["w2"], cfg.k, nthreads=1)
    b = oracle.moe_forward(inp["x"], inp["w_router"], inp["w1"], inp["w2"], cfg.k, nthreads=4)
    np.testing.assert_array_equal(a["y"], b["y"])
    np.testing.assert_array_equal(a["logits"], b["logits"])


# ------------------------------------------- combine of given expert outputs --

@pytest.mark.parametrize("T,H,k,cf", [(9, 16, 3, None), (40, 8, 2, 0.6), (1, 24, 1, None)])
def test_combine_given_dense_gate_matrix(T, H, k, cf):
    # a second formulation: the gates as a dense [T, rows] matrix G with
    # G[t, slot[t, j]] = w[t, j], and y = G Y by numpy's matmul
    rng = np.random.default_rng(T * 7 + k)
    E = 4
    ids = np.stack([rng.choice(E, size=k, replace=False) for _ in range(T)]).astype(np.int32)
    _, offsets, _, slot = oracle.dispatch(ids, E, cf)
    n = int(offsets[-1])
    Y = rand_bf16((max(n, 1), H), 1.0, T + H)
    w = rng.uniform(0.05, 1.0, size=(T, k)).astype(np.float32)
    G = np.zeros((T, Y.shape[0]))
    for t in range(T):
        for j in range(k):
            if slot[t, j] >= 0:
                G[t, slot[t, j]] = w[t, j]
    np.testing.assert_allclose(oracle.combine_given(Y, w, slot), G @ f64(Y), rtol=1e-12, atol=1e-12)


def test_combine_given_copies_rows_and_zeroes_dropped_tokens():
    Y = rand_bf16((5, 8), 1.0, 3)
    slot = np.array([[4], [-1], [0], [2], [-1]], dtype=np.int32)
    w = np.ones((5, 1), dtype=np.float32)
    y = oracle.combine_given(Y, w, slot)
    Yd = f64(Y)
    for t, r in enumerate(slot[:, 0]):
        np.testing.assert_array_equal(y[t], Yd[r] if r >= 0 else np.zeros(8))
    with pytest.raises(RuntimeError):
        oracle.combine_given(Y, w, np.array([[5], [0], [0], [0], [0]], dtype=np.int32))


def test_stored_routing_stats_match_the_oracle():
    # tests/golden/routing_stats.json is written by make_routing_stats.py
    # from the oracle; recompute the small workloads' rows
    import importlib.util
    path = os.path.join(os.path.dirname(__file__), "golden", "make_routing_stats.py")
    spec = importlib.util.spec_from_file_location("make_routing_stats", path)
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    with open(os.path.join(os.path.dirname(__file__), "golden", "routing_stats.json")) as f:
        stored = json.load(f)["workloads"]
    for name in ("tiny", "decode"):
        assert mod.stats(moe_synth.ALL[name]) == stored[name]


def test_seeded_inputs_are_the_same_bits_on_every_machine():
    # tests/golden/synth_checksums.json: sha256 of seeded tensors' bf16 bits
    # (make_synth_checksums.py); the generator is integer streams + float64
    # Box-Muller, so x86-64 and aarch64 hosts draw identical inputs
    import importlib.util
    path = os.path.join(os.path.dirname(__file__), "golden", "make_synth_checksums.py")
    spec = importlib.util.spec_from_file_location("make_synth_checksums", path)
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    with open(os.path.join(os.path.dirname(__file__), "golden", "synth_checksums.json")) as f:
        stored = json.load(f)
    assert {n: mod.digest(fn()) for n, fn in mod.CASES.items()} == stored
