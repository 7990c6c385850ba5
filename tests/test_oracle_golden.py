"""The oracle still reproduces its stored regression fixtures (see tests/golden/README.md)."""
import json
import os
import sys

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.join(HERE, "golden"))

import make_golden  # noqa: E402


def _load(name):
    with open(os.path.join(HERE, "golden", name)) as f:
        return json.load(f)


def test_oracle_chain_fixture():
    ref = _load("oracle_tiny_chain.json")
    now = make_golden.chain_fixture()
    for k in ("cluster_ids", "shortlist_len", "tokens", "token_idx", "accepted", "correction"):
        assert now[k] == ref[k], k
    np.testing.assert_allclose(np.array(now["logits_head"]), np.array(ref["logits_head"]),
                               rtol=1e-12, atol=1e-12)


def test_oracle_tree_fixture():
    ref = _load("oracle_tiny_tree.json")
    now = make_golden.tree_fixture()
    for k in ("tokens", "accepted", "correction", "path"):
        assert now[k] == ref[k], k
