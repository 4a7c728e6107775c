"""Writes tests/golden/tiny_layer.json: one tiny packed layer case.

The inputs are stored with the outputs, so the fixture does not depend on the
random generator of the machine that reads it.  Every value is written by the
fp64 oracle (and nothing else).  The source pages print no worked example of
the layer; this fixture is the oracle's own regression record, used to check
that the oracle builds and computes the same numbers on every host
(x86 build machine, Arm GPU host).

Run from the repository root:  python tests/golden/make_golden.py
"""
import json
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
sys.path.insert(0, ROOT)

import torch  # noqa: E402

import gdn_inputs as gi  # noqa: E402
import oracle  # noqa: E402

SHAPE = gi.Shape(h_k=1, h_v=2, d_k=4, d_v=3)
LENGTHS = [5, 2]


def main():
    p = gi.make_params(SHAPE, 99, dtype=torch.float32, norm_w="uniform")
    x = gi.make_tokens(SHAPE, sum(LENGTHS), 99, dtype=torch.float32)
    st = gi.make_states(SHAPE, len(LENGTHS), 99, ssm_std=0.3, conv_std=1.0)
    inp = {"qkv": x["qkv"], "z": x["z"], "a": x["a"], "b": x["b"], **p, **st}
    out, cs, ss = oracle.layer(h_k=SHAPE.h_k, h_v=SHAPE.h_v, d_k=SHAPE.d_k, d_v=SHAPE.d_v,
                               conv_w_width=SHAPE.conv_w, cu_seqlens=gi.cu_seqlens(LENGTHS),
                               **inp)
    hexl = lambda t: [float(v).hex() for v in torch.as_tensor(t).double().flatten().tolist()]
    doc = {
        "what": "tiny packed Gated DeltaNet layer, fp64 oracle outputs",
        "shape": {"h_k": SHAPE.h_k, "h_v": SHAPE.h_v, "d_k": SHAPE.d_k, "d_v": SHAPE.d_v,
                  "conv_w": SHAPE.conv_w, "l2_eps": 1e-6, "rms_eps": 1e-6},
        "lengths": LENGTHS,
        "inputs": {k: {"shape": list(v.shape), "hex": hexl(v)} for k, v in inp.items()},
        "expected": {"out": {"shape": list(out.shape), "hex": hexl(out)},
                     "conv_state": {"shape": list(cs.shape), "hex": hexl(cs)},
                     "ssm_state": {"shape": list(ss.shape), "hex": hexl(ss)}},
    }
    path = os.path.join(os.path.dirname(os.path.abspath(__file__)), "tiny_layer.json")
    with open(path, "w") as f:
        json.dump(doc, f, indent=0)
    print("wrote", path)


if __name__ == "__main__":
    main()
