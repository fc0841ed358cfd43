"""Writes tests/golden/tiny_seed0.json: the oracle's routing and output for
the tiny MoE layer (M=2, H=256, E=8, top_k=2, I=SI=128; seed 0).

Calls only the oracle and the seeded input generator.  The pages print no
worked example, so this file is a regression anchor for the oracle itself:
the pins in tests/test_oracle_pins.py are what tie the oracle to the pages.
Run from the repository root: python tests/golden/make_golden.py
"""
import json
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
sys.path.insert(0, ROOT)

import oracle  # noqa: E402
from nvfp4_w4a16_mixture_gb300 import synth  # noqa: E402


def main():
    shape = synth.CONFIGS["tiny"]
    M, H, E, k, I, SI = shape
    x, layer = synth.make_problem(M, H, E, k, I, SI, seed=0)
    r = oracle.forward(x, layer, k)
    gold = {"shape": list(shape), "seed": 0, "ids": r["ids"].tolist(), "tw": r["tw"].tolist(),
            "out_bf16_bits": r["out"].astype(int).tolist()}
    path = os.path.join(os.path.dirname(os.path.abspath(__file__)), "tiny_seed0.json")
    with open(path, "w") as f:
        json.dump(gold, f)
        f.write("\n")


if __name__ == "__main__":
    main()
