"""The stored oracle outputs under tests/golden/ (written by
tests/golden/make_golden.py from oracle/ only) against a fresh run of the same
oracle calls: an unintended change to the oracle's arithmetic shows up here.
Codes must agree exactly, real values to 1e-12 relative (fp64 BLAS may order
sums differently on another machine)."""

import os
import sys

import numpy as np
import pytest

HERE = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")
sys.path.insert(0, HERE)
import make_golden as G  # noqa: E402

CASES = G.cases()


@pytest.mark.parametrize("name", sorted(CASES))
def test_oracle_matches_stored_outputs(name):
    stored = G.read(os.path.join(HERE, name + ".txt"))
    fresh = CASES[name]
    assert set(stored) == set(fresh)
    for key, want in stored.items():
        got = np.asarray(fresh[key], dtype=np.float64)
        assert got.shape == want.shape, (name, key)
        if key == "codes":
            np.testing.assert_array_equal(got, want, err_msg="%s %s" % (name, key))
        else:
            np.testing.assert_allclose(got, want, rtol=1e-12, atol=0, err_msg="%s %s" % (name, key))


def test_stored_files_cite_their_source():
    for name in CASES:
        with open(os.path.join(HERE, name + ".txt")) as f:
            head = f.read(400)
        assert "make_golden.py" in head and "oracle" in head and "Theorem 3.2" in head
