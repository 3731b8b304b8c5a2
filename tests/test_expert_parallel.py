"""Expert parallelism on CPU ranks: the exchange plan and the all-to-all
sequence of mixture_experts_layer_12_gb300.expert_parallel.

Two gloo ranks each hold their own tokens and half of the experts.  The
compute steps are stand-ins written from the oracle (fp64), so the test
checks only what the expert-parallel module adds -- which rows go where,
the segment layout of the received rows, and the return to dispatch order --
against the oracle's whole layer on each rank's tokens with every expert.
"""
import os
import sys
from types import SimpleNamespace

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_send_splits_follow_expert_major_dispatch_order():
    from mixture_experts_layer_12_gb300.expert_parallel import segment_offsets, send_splits
    offsets = [0, 3, 3, 7, 12, 12, 13, 20, 21]  # E = 8
    assert send_splits(offsets, 2) == [12, 9]
    assert send_splits(offsets, 4) == [3, 9, 1, 8]
    assert send_splits(offsets, 1) == [21]
    rc = torch.tensor([[2, 0, 5], [1, 4, 0]])  # [sources, local experts]
    so = segment_offsets(rc)
    assert so.dtype == torch.int32 and so.tolist() == [0, 2, 2, 7, 8, 12, 12]


class OracleOps:
    """fp64 stand-ins for the library's compute steps (test only)."""

    def __init__(self, w_router, w1_local, w2_local, k, E, bias, cf, act):
        self.w_router, self.w1, self.w2, self.bias = w_router, w1_local, w2_local, bias
        self.k, self.E, self.cf, self.act = k, E, cf, act
        self.El, self.H = w2_local.shape[0], w2_local.shape[2]

    def route(self, x):
        import oracle
        _, ids, _, w = oracle.route(x, self.w_router, self.k, bias=self.bias)
        counts, offsets, perm, slot = oracle.dispatch(ids, self.E, self.cf)
        t = torch.from_numpy
        return SimpleNamespace(ids=t(ids), weights=t(w), counts=t(counts), offsets=t(offsets),
                               perm=t(perm), slot=t(slot))

    def dispatch_rows(self, x, r):
        kept = int(r.offsets[-1])
        xp = torch.zeros(x.shape[0] * self.k, self.H, dtype=x.dtype)
        xp[:kept] = x[r.perm[:kept].long() // self.k]
        return xp

    def max_rows_to_one_rank(self, T):
        import oracle
        c = oracle.capacity(T, self.k, self.E, self.cf)
        return T * self.k if c < 0 else min(T * self.k, self.El * c)

    def expert_ffn(self, rows, seg_offsets, n_segments):
        import oracle
        f = oracle.expert_swiglu if self.act == "swiglu" else oracle.expert_ffn
        so = seg_offsets.tolist()
        assert len(so) == n_segments + 1
        Y = torch.full((rows.shape[0], self.H), float("nan"), dtype=torch.float64)
        for i in range(n_segments):
            e = i % self.El
            for rr in range(so[i], so[i + 1]):
                Y[rr] = torch.from_numpy(f(rows[rr], self.w1[e], self.w2[e]))
        return Y

    def combine(self, Y, r, T):
        y = torch.zeros(T, self.H, dtype=torch.float64)
        for t in range(T):
            for j in range(self.k):
                s = int(r.slot[t, j])
                if s >= 0:
                    y[t] += float(r.weights[t, j]) * Y[s]
        return y


def _worker(rank, world, port, out_dir, cfg_kw, padded):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import moe_synth
    import oracle
    from mixture_experts_layer_12_gb300.expert_parallel import ExpertParallelMoE, TorchExchange
    oracle.build()
    cfg = moe_synth.MoEConfig("ep", **cfg_kw)
    full = moe_synth.make_inputs(cfg)                       # same weights on every rank
    x = moe_synth.make_inputs(cfg.with_(seed=cfg.seed + 100 + rank), with_ffn=False)["x"]
    El = cfg.E // world
    sl = slice(rank * El, (rank + 1) * El)
    ops = OracleOps(full["w_router"], full["w1"][sl], full["w2"][sl], cfg.k, cfg.E, full["bias"],
                    cfg.capacity_factor, cfg.act)
    layer = ExpertParallelMoE(ops, rank, world, TorchExchange(), padded=padded)
    y = layer.forward(x)
    ref = oracle.moe_forward(x, full["w_router"], full["w1"], full["w2"], cfg.k, bias=full["bias"],
                             capacity_factor=cfg.capacity_factor, act=cfg.act)
    routed = layer.send(x)
    torch.save(dict(y=y, ref=torch.from_numpy(np.asarray(ref["y"])),
                    sent=routed.send_counts.sum(dim=1).tolist(),
                    dropped=int((routed.slot < 0).sum())),
               os.path.join(out_dir, f"rank{rank}.pt"))
    dist.barrier()
    dist.destroy_process_group()


@pytest.mark.parametrize("cfg_kw", [
    dict(T=48, H=16, F=24, E=8, k=2, seed=70),
    dict(T=40, H=16, F=24, E=8, k=3, seed=71, capacity_factor=0.6, bias0=2.0),  # drops, skew
    dict(T=32, H=16, F=8, E=4, k=1, seed=72, act="swiglu"),
], ids=["k2", "k3_drops", "k1_swiglu"])
@pytest.mark.parametrize("padded", [False, True], ids=["exact", "padded"])
def test_two_rank_expert_parallel_matches_whole_layer(tmp_path, cfg_kw, padded):
    # exact: row all-to-alls of exactly the rows (split sizes read once);
    # padded: equal-split blocks, every index step on the device
    world = 2
    port = 29600 + (os.getpid() % 1500) + (7 if padded else 0)
    mp.start_processes(_worker, args=(world, port, str(tmp_path), cfg_kw, padded), nprocs=world,
                       join=True, start_method="spawn")
    for r in range(world):
        res = torch.load(tmp_path / f"rank{r}.pt")
        np.testing.assert_allclose(res["y"].numpy(), res["ref"].numpy(), rtol=1e-10, atol=1e-12)
        assert sum(res["sent"]) > 0 and len(res["sent"]) == world
        if cfg_kw.get("capacity_factor"):
            assert res["dropped"] > 0
