"""The oracle reproduces its stored tiny-workload fixture (tests/golden/tiny_oracle.json,
written by tests/golden/make_golden.py, which runs only the oracle)."""
import json
import os

import numpy as np

from tests.golden.make_golden import run

HERE = os.path.dirname(os.path.abspath(__file__))


def test_tiny_oracle_fixture():
    want = json.load(open(os.path.join(HERE, "golden", "tiny_oracle.json")))
    got = run()
    assert got["prompt"] == want["prompt"]
    assert got["argmax_per_step"] == want["argmax_per_step"]
    for k, v in want["logits_head_at_pos"].items():
        np.testing.assert_allclose(got["logits_head_at_pos"][k], v, rtol=1e-12, atol=1e-14)
