"""Writes tests/golden/tiny_T8_oracle.json by calling only the CPU oracle.

The fixture is a regression record of the oracle on the tiny layer (T=8,
H=256, I=128, E=8, top_k=2, rank 8, 2 adapters, seed 0): routing ids and
weights, the permutation, and a hash plus a few rows of the output.  The
pages print no worked example for this layer, so no stored value here comes
from them; the oracle itself is pinned by tests/test_oracle_pins.py.

Run from the repository root:  python tests/golden/make_golden.py
"""
import hashlib
import json
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

import oracle  # noqa: E402
import workloads  # noqa: E402


def main():
    wl = workloads.WORKLOADS["tiny_T8"]
    inp = workloads.make_inputs(wl)
    res = oracle.forward_inputs(inp)
    off, e2p, p2e = oracle.permute(res["ids"], wl.E)
    doc = {
        "workload": wl.name,
        "generator": "workloads.make_inputs(WORKLOADS['tiny_T8'])",
        "topk_ids": res["ids"].tolist(),
        "topk_w": [[float(v) for v in row] for row in res["w"]],
        "expert_offsets": off.tolist(),
        "expanded_to_permuted": e2p.tolist(),
        "out_bf16_sha256": hashlib.sha256(res["out_bf16"].tobytes()).hexdigest(),
        "out64_rows_0_1": [[float(v) for v in row] for row in res["out64"][:2]],
    }
    path = os.path.join(ROOT, "tests", "golden", "tiny_T8_oracle.json")
    with open(path, "w") as f:
        json.dump(doc, f, indent=1)
    print("wrote", path)


if __name__ == "__main__":
    main()
