"""The oracle still reproduces the stored outputs of tests/golden/make_golden.py."""
import json
import os
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.join(HERE, "golden"))


def test_oracle_matches_stored_golden(oracle_mod):
    import make_golden
    stored = json.load(open(os.path.join(HERE, "golden", "oracle_small.json")))
    now = make_golden.make()
    for name in stored:
        if name.startswith("_"):
            continue
        assert now[name] == stored[name], name
