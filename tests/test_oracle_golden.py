"""The oracle reproduces its stored regression fixtures bit for bit (see
tests/golden/README.md: fixtures of the pinned oracle, written by
tests/golden/make_golden.py, which calls only the oracle and the generator)."""
import json
import os

import pytest

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def test_oracle_matches_its_regression_fixtures(oracle_lib):
    import importlib.util
    spec = importlib.util.spec_from_file_location("make_golden", os.path.join(GOLDEN, "make_golden.py"))
    mk = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mk)
    stored = json.load(open(os.path.join(GOLDEN, "oracle_regression.json")))
    now = mk.cases()
    assert sorted(stored) == sorted(now)
    for name in stored:
        assert stored[name] == now[name], name
