"""Writes synth_checksums.json: sha256 of the bf16 bits of seeded inputs
(moe_synth), so any machine can check that it draws the same tensors.

    python tests/golden/make_synth_checksums.py
"""
import hashlib
import json
import os
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(os.path.dirname(HERE)))

import torch  # noqa: E402

import moe_synth  # noqa: E402

CASES = {
    "router_k2.x": lambda: moe_synth.make_x(moe_synth.ROUTER[2]),
    "router_k2.w_router": lambda: moe_synth.make_w_router(moe_synth.ROUTER[2]),
    "tiny.w1[3]": lambda: moe_synth.make_w1_expert(moe_synth.TINY, 3),
    "decode.w2[5]": lambda: moe_synth.make_w2_expert(moe_synth.DECODE, 5),
}


def digest(t: torch.Tensor) -> str:
    return hashlib.sha256(t.contiguous().view(torch.int16).numpy().tobytes()).hexdigest()


def main():
    out = {name: digest(fn()) for name, fn in CASES.items()}
    with open(os.path.join(HERE, "synth_checksums.json"), "w") as f:
        json.dump(out, f, indent=1)
        f.write("\n")
    print(out)


if __name__ == "__main__":
    main()
