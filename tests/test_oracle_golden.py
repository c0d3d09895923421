"""Regression pin: the oracle reproduces its stored tiny-workload output
(written by tests/golden/make_oracle_golden.py, which calls only oracle/)."""
import json
import os

import pytest

from tests.golden.make_oracle_golden import compute

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "oracle_tiny_step.json")


def test_oracle_matches_stored_tiny_step():
    ref = json.load(open(GOLDEN))
    got = compute()
    assert got["loss"] == pytest.approx(ref["loss"], rel=1e-12)
    for k, v in ref["grad_norms"].items():
        assert got["grad_norms"][k] == pytest.approx(v, rel=1e-10), k
