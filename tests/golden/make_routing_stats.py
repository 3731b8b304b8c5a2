"""Writes routing_stats.json: per seeded workload, what the oracle's routing
and dispatch give -- near-tie tokens (the acceptance rule's exemption),
kept and dropped assignments, and how much of the load the most popular
expert takes.  Calls only the oracle (and the seeded input generators).

    python tests/golden/make_routing_stats.py

Near-tie token: two adjacent values among its k+1 largest oracle logits
differ by less than 1e-4 (tests/parity.py).  "membership_ties" counts the
subset whose k-th and (k+1)-th logits are that close -- the only tokens
whose expert SET may legitimately differ; the rest can only swap columns.
"""
import json
import os
import sys

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(os.path.dirname(HERE))
sys.path.insert(0, ROOT)
sys.path.insert(0, os.path.dirname(HERE))

import moe_synth  # noqa: E402
import oracle  # noqa: E402
from parity import NEAR_TIE, near_tie_tokens  # noqa: E402

WORKLOADS = ["tiny", "prefill", "router_k1", "router_k2", "router_k4", "router_k8", "skewed",
             "skewed_cf1.2", "decode", "prefill_k1"]


def stats(cfg) -> dict:
    inputs = moe_synth.make_inputs(cfg, with_ffn=False)
    logits, ids, _, _ = oracle.route(inputs["x"], inputs["w_router"], cfg.k, bias=inputs["bias"])
    counts, offsets, _, slot = oracle.dispatch(ids, cfg.E, cfg.capacity_factor)
    srt = -np.sort(-logits.astype(np.float64), axis=1)
    member = (srt[:, cfg.k - 1] - srt[:, cfg.k] < NEAR_TIE) if cfg.k < cfg.E else \
        np.zeros(cfg.T, bool)
    pre = np.bincount(ids.reshape(-1), minlength=cfg.E)
    c = counts.astype(np.float64)
    return {
        "T": cfg.T, "E": cfg.E, "k": cfg.k,
        "capacity": oracle.capacity(cfg.T, cfg.k, cfg.E, cfg.capacity_factor),
        "near_tie_tokens": int(near_tie_tokens(logits, cfg.k).sum()),
        "membership_ties": int(member.sum()),
        "kept_assignments": int(offsets[-1]),
        "dropped_assignments": int((slot < 0).sum()),
        "tokens_all_dropped": int(np.all(slot < 0, axis=1).sum()),
        "expert0_token_fraction": round(float(np.mean(np.any(ids == 0, axis=1))), 6),
        "max_expert_assignments": int(pre.max()),
        "load_cv_kept": round(float(c.std() / c.mean()), 6) if c.mean() > 0 else 0.0,
    }


def main():
    out = {"rule": f"near-tie: adjacent gap < {NEAR_TIE} among the k+1 largest oracle logits",
           "workloads": {name: stats(moe_synth.ALL[name]) for name in WORKLOADS}}
    with open(os.path.join(HERE, "routing_stats.json"), "w") as f:
        json.dump(out, f, indent=1)
        f.write("\n")
    for n, v in out["workloads"].items():
        print(n, v)


if __name__ == "__main__":
    main()
