"""Guards the oracle against unintended drift: compares it with digests
that tests/golden/make_oracle_regression.py wrote from the oracle itself.
This is not a pin (the pins are in test_oracle_pins.py); it only makes any
change to the oracle's arithmetic visible."""
import json
import os
import sys

import pytest

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.join(HERE, "golden"))

import make_oracle_regression as mk  # noqa: E402

with open(os.path.join(HERE, "golden", "oracle_regression.json")) as f:
    CASES = json.load(f)["cases"]


@pytest.mark.parametrize("case", CASES, ids=lambda c: "-".join(map(str, c["args"])))
def test_oracle_unchanged(orc, case):
    got = mk.run_case(*case["args"])
    want = case["expect"]
    for k in ("vals", "idx", "scale", "zero"):
        assert got[k] == want[k], k
    assert got["y"] == want["y"]
