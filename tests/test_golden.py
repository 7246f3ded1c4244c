"""The oracle still reproduces its frozen fixtures (tests/golden/*.json)."""
import json
import os

import numpy as np
import pytest

HERE = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


@pytest.mark.parametrize("name", ["decode_tiny", "verify_tiny"])
def test_oracle_matches_fixture(name):
    import sys
    sys.path.insert(0, HERE)
    import make_golden

    got = getattr(make_golden, name)()
    with open(os.path.join(HERE, name + ".json")) as f:
        ref = json.load(f)
    assert got["case"] == ref["case"]
    for key in ref:
        if key == "case":
            continue
        np.testing.assert_allclose(np.array(got[key]), np.array(ref[key]), rtol=1e-12, atol=1e-14)
