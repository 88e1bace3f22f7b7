"""Writes tiny_decode_oracle.json: sampled oracle outputs for the tiny decode
workload (seed 0).  Calls only the oracle and the seeded input generator."""
import json
import os
import sys

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(os.path.dirname(HERE)))

import oracle  # noqa: E402
import workloads  # noqa: E402


def main():
    seed = 0
    inp = workloads.tiny_decode(seed=seed)
    out, lse, _ = oracle.forward(inp)
    rng = np.random.default_rng(1234)
    idx = [(int(h), int(d)) for h, d in zip(rng.integers(0, 16, 64), rng.integers(0, 512, 64))]
    fx = dict(seed=seed, workload="tiny_decode", out_index=idx,
              out_values=[float(out[0, h, d]) for h, d in idx], lse=[float(x) for x in lse[0]])
    with open(os.path.join(HERE, "tiny_decode_oracle.json"), "w") as f:
        json.dump(fx, f, indent=1)


if __name__ == "__main__":
    main()
