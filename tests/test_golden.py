"""The oracle reproduces its stored output on the tiny workload (tests/golden/tiny_oracle.json,
written by tests/golden/make_golden.py from the oracle alone; the pages print no worked
example)."""
import json
import os

import pytest

from tests.golden import make_golden

HERE = os.path.dirname(os.path.abspath(__file__))


def test_tiny_golden():
    with open(os.path.join(HERE, "golden", "tiny_oracle.json")) as f:
        want = json.load(f)
    got = make_golden.compute()
    assert got["c32"] == want["c32"] and got["count"] == want["count"]
    assert got["c_exact"] == pytest.approx(want["c_exact"], rel=1e-14)
    assert got["resident"] == want["resident"]
    for gq, wq in zip(got["queries"], want["queries"]):
        assert gq["fetch_ids"] == wq["fetch_ids"]
        for gh, wh in zip(gq["heads"], wq["heads"]):
            assert gh["certified"] == wh["certified"] and gh["k_star"] == wh["k_star"]
            assert gh["F"] == wh["F"]
            for k in ["eps_L", "beta", "D", "lse"]:
                assert gh[k] == pytest.approx(wh[k], rel=1e-12, abs=1e-300)
            assert gh["o"] == pytest.approx(wh["o"], rel=1e-12, abs=1e-14)
