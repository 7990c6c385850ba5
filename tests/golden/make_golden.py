"""Write the oracle regression fixtures in this folder.

Runs the CPU oracle (and nothing else) on the seeded Tiny chain and tiny-tree workloads and
stores its integer outputs and a few logits.  The pages print no worked example for this
path, so these fixtures pin nothing to the pages: they only freeze the oracle against
accidental change.  Regenerate with ``python tests/golden/make_golden.py`` and name, in the
commit message, the passage or reading that justified the change.
"""
import json
import os
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(os.path.dirname(HERE)))

import oracle            # noqa: E402
import workloads as wl   # noqa: E402


def chain_fixture():
    inp = wl.chain_inputs(wl.config("tiny"), 0)
    r = oracle.chain_step(inp)[0]
    return dict(
        config="tiny", seed=0,
        cluster_ids=[p["ids"].tolist() for p in r["positions"]],
        shortlist_len=[int(len(p["S"])) for p in r["positions"]],
        tokens=[p["token"] for p in r["positions"]],
        token_idx=[p["idx"] for p in r["positions"]],
        logits_head=[[float(x) for x in p["logits"][:4]] for p in r["positions"]],
        accepted=r["accepted"], correction=r["correction"])


def tree_fixture():
    inp = wl.tree_inputs(wl.config("tiny_tree"), 0)
    r = oracle.tree_step(inp)
    return dict(
        config="tiny_tree", seed=0,
        tokens=[[n["token"] for d in r[b]["depths"] for n in d["nodes"]] for b in sorted(r)],
        accepted=[r[b]["accepted"] for b in sorted(r)],
        correction=[r[b]["correction"] for b in sorted(r)],
        path=[r[b]["path"] for b in sorted(r)])


if __name__ == "__main__":
    for name, fn in (("oracle_tiny_chain.json", chain_fixture), ("oracle_tiny_tree.json", tree_fixture)):
        with open(os.path.join(HERE, name), "w") as f:
            json.dump(fn(), f, indent=1)
        print("wrote", name)
