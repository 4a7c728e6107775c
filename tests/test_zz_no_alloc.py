"""gdn_prefill_noalloc, the prefill for callers that cannot allocate, agrees
with gdn_prefill.

Some callers cannot give the library a device workspace when they run the
layer (a fixed memory budget, an allocator closed after start-up, a host
framework with no allocation hook).  gdn_prefill_noalloc takes the same
inputs and outputs and keeps its scratch in a fixed device array inside the
library.  Here it runs twice in a row through the C ABI, on different batch
shapes (so the second call finds the first call's contents in the shared
array), and each result is compared with gdn_prefill's on identical inputs
and initial states, within the prefill tolerance.  The first batch is also
compared with the fp64 oracle directly, and a call with a rejected cu_seqlens
must report GDN_ERR_DEVICE_BOUNDS through its status word and write nothing.
"""
import numpy as np
import pytest
import torch

import gated_deltanet_linear_06_gb300 as gdn
import gdn_inputs as gi
from gpu_util import DEV, PREFILL_TOL, dims_of, oracle_layer, rel_err, to_dev

pytestmark = pytest.mark.gpu
SH = gi.LAYER


def _inputs(lengths, seed, sh=SH):
    T = sum(lengths)
    params = gi.make_params(sh, seed, norm_w="uniform")
    tok = gi.make_tokens(sh, T, seed)
    gc = gi.gate_controlled(sh, T, seed)
    tok["a"], tok["b"] = gc["a"], gc["b"]
    params["A_log"], params["dt_bias"] = gc["A_log"], gc["dt_bias"]
    st = gi.make_states(sh, len(lengths), seed, ssm_std=0.1 ** 0.5, conv_std=1.0)
    return to_dev(params), to_dev(tok), st


def _both(lengths, seed, bitwise=False, sh=SH, against_oracle=False):
    dims = dims_of(sh)
    p, x, st = _inputs(lengths, seed, sh)
    N, T = len(lengths), sum(lengths)
    cu = gi.cu_seqlens(lengths).to(DEV)
    res = {}
    for which in ("workspace", "noalloc"):
        conv, ssm = st["conv_state"].clone().to(DEV), st["ssm_state"].clone().to(DEV)
        out = torch.full((T, sh.h_v, sh.d_v), float("nan"), dtype=torch.bfloat16, device=DEV)
        if which == "workspace":
            ws = torch.empty(gdn.gdn_workspace_bytes(dims, N, T), dtype=torch.uint8, device=DEV)
            gdn.gdn_prefill(dims, x["qkv"], x["z"], x["a"], x["b"], p["A_log"], p["dt_bias"],
                            p["conv_w"], p["norm_w"], cu, conv, ssm, out, ws)
            status = gdn.gdn_read_device_status(ws)
        else:
            word = torch.full((1,), -1, dtype=torch.int32, device=DEV)
            gdn.gdn_prefill_noalloc(dims, x["qkv"], x["z"], x["a"], x["b"], p["A_log"],
                                    p["dt_bias"], p["conv_w"], p["norm_w"], cu, conv, ssm, out,
                                    device_status=word)
            status = gdn.gdn_read_device_status(word)
        assert status == 0, (which, status)
        res[which] = (out, conv, ssm)
    (o_w, c_w, s_w), (o_n, c_n, s_n) = res["workspace"], res["noalloc"]
    assert not torch.isnan(o_n.float()).any()
    e_out, e_ssm = rel_err(o_n, o_w), rel_err(s_n, s_w)
    assert e_out <= PREFILL_TOL and e_ssm <= PREFILL_TOL, (e_out, e_ssm)
    np.testing.assert_array_equal(c_n.cpu().numpy(), c_w.cpu().numpy())
    if bitwise:
        assert torch.equal(o_n.view(torch.int16), o_w.view(torch.int16))
        assert torch.equal(s_n, s_w)
    if against_oracle:
        # the allocation-free result against the fp64 definition itself
        tok = {k: v.cpu() for k, v in x.items()}
        ref, r_conv, r_ssm = oracle_layer(sh, tok, {k: v.cpu() for k, v in p.items()}, cu.cpu(),
                                          conv_state=st["conv_state"], ssm_state=st["ssm_state"])
        eo, es = rel_err(o_n, ref), rel_err(s_n, r_ssm)
        assert eo <= PREFILL_TOL and es <= PREFILL_TOL, (eo, es)
        np.testing.assert_array_equal(c_n.cpu().numpy(), r_conv)
    return e_out, e_ssm


def test_noalloc_matches_prefill_on_two_calls_in_a_row():
    # call 1: gdn_prefill splits the 2500-token sequence into parallel
    # segments, the allocation-free entry point scans it whole
    e1 = _both([2500, 70, 1], seed=21, against_oracle=True)
    # call 2: a different batch; the shared array still holds call 1's list.
    # No sequence is longer than one segment, and then gdn_prefill's prep and
    # scan passes do exactly the single pass's arithmetic: bit-identical results
    e2 = _both([64, 129, 0, 33], seed=22, bitwise=True)
    print(f"call 1 rel diff out {e1[0]:.2e} state {e1[1]:.2e}; "
          f"call 2 out {e2[0]:.2e} state {e2[1]:.2e}")


@pytest.mark.parametrize("h_k,h_v", [(32, 32), (8, 32)])
def test_noalloc_matches_prefill_bitwise_at_other_head_groupings(h_k, h_v):
    # 1 and 4 value heads per key head, no sequence longer than one segment:
    # the two entry points do the same arithmetic
    _both([300, 64, 5], seed=23, bitwise=True, sh=gi.Shape(h_k=h_k, h_v=h_v))


def test_noalloc_reports_a_rejected_cu_seqlens_through_its_status_word():
    # a decreasing cu_seqlens is caught on the device: the status word copied
    # out reads GDN_ERR_DEVICE_BOUNDS and nothing is written; the next good call
    # clears the library's word again
    dims = dims_of(SH)
    p, x, st = _inputs([60, 40], seed=24)
    conv, ssm = st["conv_state"].clone().to(DEV), st["ssm_state"].clone().to(DEV)
    out = torch.full((100, SH.h_v, SH.d_v), float("nan"), dtype=torch.bfloat16, device=DEV)
    word = torch.full((1,), -1, dtype=torch.int32, device=DEV)
    bad = torch.tensor([0, 70, 40], dtype=torch.int32, device=DEV)
    gdn.gdn_prefill_noalloc(dims, x["qkv"], x["z"], x["a"], x["b"], p["A_log"], p["dt_bias"],
                            p["conv_w"], p["norm_w"], bad, conv, ssm, out, device_status=word,
                            total_tokens=100)
    assert gdn.gdn_read_device_status(word) == gdn.GDN_ERR_DEVICE_BOUNDS
    assert torch.isnan(out.float()).all()
    assert torch.equal(conv.cpu(), st["conv_state"]) and torch.equal(ssm.cpu(), st["ssm_state"])
    good = gi.cu_seqlens([60, 40]).to(DEV)
    gdn.gdn_prefill_noalloc(dims, x["qkv"], x["z"], x["a"], x["b"], p["A_log"], p["dt_bias"],
                            p["conv_w"], p["norm_w"], good, conv, ssm, out, device_status=word)
    assert gdn.gdn_read_device_status(word) == 0
    assert not torch.isnan(out.float()).any()
