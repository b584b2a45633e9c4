"""The oracle against its stored regression fixture (tests/golden/oracle_small.json).

The fixture holds small fixed inputs and the fp64 outputs the oracle gave for them
when it was written by tests/golden/make_golden.py (which calls only oracle/).  The
pages print no worked numeric example, so these values pin the oracle to its own
earlier state, not to the pages: they make any later change of its arithmetic
visible.  The pins against the pages and the mathematics are in test_oracle_pins.py.
"""
import json
import os
import sys

import numpy as np
import pytest

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.join(HERE, "golden"))

import make_golden  # noqa: E402

FIXTURE = os.path.join(HERE, "golden", "oracle_small.json")


def _load():
    with open(FIXTURE) as f:
        return json.load(f)["cases"]


def _arr(x, dtype=np.float64):
    return None if x is None else np.asarray(x, dtype=dtype)


@pytest.mark.parametrize("case", _load(), ids=lambda c: c["name"])
def test_oracle_reproduces_stored_values(case):
    x = {k: _arr(v, np.int64 if k == "cu_seqlens" else np.float64) for k, v in case["inputs"].items()}
    got = make_golden.run_oracle(x, case["options"])
    want = case["outputs"]
    assert sorted(got) == sorted(want)
    for name, ref in want.items():
        ref = np.asarray(ref)
        g = np.asarray(got[name])
        assert g.shape == ref.shape, name
        # summation order is fixed in the oracle; allow only last-bit differences
        # from the compiler's choice of fused multiply-adds across machines
        np.testing.assert_allclose(g, ref, rtol=1e-12, atol=1e-13, err_msg=name)


def test_fixture_covers_the_options():
    names = [c["name"] for c in _load()]
    assert any("longhorn" in n for n in names)
    assert any("packed" in n for n in names)
    packed = [c for c in _load() if c["inputs"]["cu_seqlens"] is not None][0]
    lengths = np.diff(packed["inputs"]["cu_seqlens"])
    assert (lengths == 0).any(), "an empty packed sequence is part of the fixture"
