"""Regression fixture of the oracle's verify side and FP8 loop, written by
tests/golden/make_golden.py (oracle only): uniforms, probabilistic accept,
logits to probabilities, the FP8 quantiser and the FP8 loop's tokens on
seeded inputs must reproduce exactly."""
import json
import os

from tests.golden.make_golden import verify_golden

HERE = os.path.dirname(os.path.abspath(__file__))


def test_verify_side_golden():
    with open(os.path.join(HERE, "golden", "verify_side.json")) as f:
        want = json.load(f)
    got = verify_golden()
    for key in want:
        if key != "source":
            assert got[key] == want[key], key
