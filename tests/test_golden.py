"""The oracle still reproduces the stored tiny-workload result bit for bit
(tests/golden/tiny_oracle.json, written by tests/golden/make_golden.py)."""
import json
import os

from tests.golden.make_golden import tiny_oracle

HERE = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def test_tiny_oracle_matches_golden():
    with open(os.path.join(HERE, "tiny_oracle.json")) as f:
        stored = json.load(f)
    assert tiny_oracle() == stored
