"""The oracle against the fixture that tests/golden/make_golden.py wrote from it.

A change of the oracle's arithmetic shows up here; it must then be justified
by a reading of the pages and the fixture regenerated with that script.
"""
import hashlib
import json
import os

import numpy as np

import oracle
import workloads

HERE = os.path.dirname(os.path.abspath(__file__))


def test_tiny_fixture():
    with open(os.path.join(HERE, "golden", "tiny_T8_oracle.json")) as f:
        doc = json.load(f)
    wl = workloads.WORKLOADS[doc["workload"]]
    inp = workloads.make_inputs(wl)
    res = oracle.forward_inputs(inp)
    assert res["ids"].tolist() == doc["topk_ids"]
    np.testing.assert_allclose(res["w"], doc["topk_w"], rtol=0, atol=0)
    off, e2p, _ = oracle.permute(res["ids"], wl.E)
    assert off.tolist() == doc["expert_offsets"]
    assert e2p.tolist() == doc["expanded_to_permuted"]
    assert hashlib.sha256(res["out_bf16"].tobytes()).hexdigest() == doc["out_bf16_sha256"]
    np.testing.assert_allclose(res["out64"][:2], doc["out64_rows_0_1"], rtol=1e-15)
