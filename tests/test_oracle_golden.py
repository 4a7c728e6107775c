"""The oracle reproduces its stored tiny-layer record on this host.

tests/golden/tiny_layer.json was written by tests/golden/make_golden.py,
which calls only the oracle; it stores its inputs, so this check holds on any
host whatever its random generator.  It catches a build of the oracle that
computes differently here (compiler, libm, OpenMP) from where it was written.
"""
import json
import os

import numpy as np

import oracle

PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden", "tiny_layer.json")


def _arr(d):
    return np.array([float.fromhex(h) for h in d["hex"]]).reshape(d["shape"])


def test_oracle_reproduces_golden_record():
    doc = json.load(open(PATH))
    s = doc["shape"]
    inp = {k: _arr(v) for k, v in doc["inputs"].items()}
    cu = np.cumsum([0] + doc["lengths"])
    out, cs, ss = oracle.layer(h_k=s["h_k"], h_v=s["h_v"], d_k=s["d_k"], d_v=s["d_v"],
                               conv_w_width=s["conv_w"], l2_eps=s["l2_eps"],
                               rms_eps=s["rms_eps"], cu_seqlens=cu, **inp)
    exp = {k: _arr(v) for k, v in doc["expected"].items()}
    np.testing.assert_allclose(out, exp["out"], rtol=0, atol=1e-13)
    np.testing.assert_allclose(ss, exp["ssm_state"], rtol=0, atol=1e-13)
    np.testing.assert_array_equal(cs, exp["conv_state"])
