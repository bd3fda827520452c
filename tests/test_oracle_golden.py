"""The oracle against its stored snapshots (tests/golden/, written by
tests/golden/make_golden.py at the shapes of lattice-inference's gradient checks):
a regression check that its outputs have not moved, to 1e-12."""
import json
import os

import numpy as np
import pytest

HERE = os.path.dirname(os.path.abspath(__file__))
GOLDEN = os.path.join(HERE, "golden")


@pytest.mark.parametrize("name", ["gradcheck_single_head", "gradcheck_multi_head"])
def test_oracle_matches_its_snapshot(name):
    import importlib.util
    spec = importlib.util.spec_from_file_location("make_golden", os.path.join(GOLDEN,
                                                                               "make_golden.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    stored = json.load(open(os.path.join(GOLDEN, name + ".json")))
    now = mod.compute(name)
    assert stored["shape"] == json.loads(json.dumps(now["shape"]))
    for key, ref in stored["values"].items():
        got = np.asarray(now["values"][key])
        ref = np.asarray(ref)
        assert got.shape == ref.shape, key
        assert np.allclose(got, ref, rtol=1e-12, atol=1e-14), key
