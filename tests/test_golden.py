"""The generator + oracle pair reproduces its stored results on this machine.

tests/golden/tiny_oracle.json was written by tests/golden/make_golden.py, which
calls only the oracle and the seeded generator (the pages print no worked
example to store instead).  A mismatch means the inputs or the float64 results
drifted between machines or after an edit of the oracle.
"""

import json
import os

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))


def test_tiny_golden_reproduces():
    import importlib.util
    spec = importlib.util.spec_from_file_location("make_golden", os.path.join(HERE, "golden", "make_golden.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    live = mod.tiny_record()
    with open(os.path.join(HERE, "golden", "tiny_oracle.json")) as f:
        ref = json.load(f)
    assert live["inputs_sha256"] == ref["inputs_sha256"]
    for key in ("doff", "accept_len", "bonus_token", "n_clipped"):
        assert live[key] == ref[key], key
    assert live["accept_rate"] == ref["accept_rate"]
    for key in ("kl", "ce", "lse_z", "lse_t", "S", "grad_l1"):
        np.testing.assert_allclose(live[key], ref[key], rtol=1e-12, atol=1e-13, err_msg=key)
    assert abs(live["loss"] - ref["loss"]) <= 1e-12 * abs(ref["loss"])
