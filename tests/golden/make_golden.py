"""Writes the golden snapshots of the oracle (tests/golden/*.json).

The pages print no worked-example values, only their test configurations, so these files
are regression snapshots of the oracle, not independent pins: they fix its outputs at the
two shapes of lattice-inference 0.6.0's gradient checks (src/attention/gdn_backward.rs,
tests `gradcheck_gdn_backward`: 8 tokens, 1 key head, 1 value head, key and value dim 8;
`gradcheck_gdn_backward_multi_head`: 4 tokens, 2 key heads, 4 value heads, dims 6) on
seeded inputs from workloads/, so that an unintended change of the oracle's arithmetic
shows.  Calls nothing but the oracle and the seeded generator.

    python tests/golden/make_golden.py
"""
import json
import os
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(os.path.dirname(HERE)))

import numpy as np  # noqa: E402

import oracle  # noqa: E402
import workloads as W  # noqa: E402

CASES = {
    "gradcheck_single_head": dict(Hk=1, Hv=1, Dk=8, Dv=8, seqlens=(8,), seed=42),
    "gradcheck_multi_head": dict(Hk=2, Hv=4, Dk=6, Dv=6, seqlens=(4,), seed=2024),
}


def case_inputs(name):
    kw = CASES[name]
    wl = W.custom(dtype="f32", packed=False, S0_std=0.5, dST_std=0.5, dt_bias_std=0.3, **kw)
    return wl, W.generate(wl)


def compute(name):
    wl, inp = case_inputs(name)
    fwd, bwd = oracle.run_inputs(inp, n_threads=1)
    out = {k: np.asarray(v).tolist() for k, v in list(fwd.items()) + list(bwd.items())}
    return {"case": name, "shape": CASES[name], "source": __doc__.split("\n\n")[1].strip(),
            "values": out}


if __name__ == "__main__":
    for name in CASES:
        path = os.path.join(HERE, name + ".json")
        with open(path, "w") as f:
            json.dump(compute(name), f, indent=None, separators=(",", ":"))
        print("wrote", path)
