"""GPU checks of gdn_decode_multi (several tokens per sequence in one call), through the C ABI.

Bars: outputs, states and traces bit-identical to the same tokens fed one
gdn_decode_step call at a time; against the fp64 oracle the same 1e-4 bar as
the single step (max |gpu - oracle| / max |oracle| on fp32 output and state).
"""
import numpy as np
import pytest
import torch

import gated_deltanet_linear_06_gb300 as gdn
import gdn_inputs as gi
from gpu_util import DECODE_TOL, DEV, dims_of, oracle_layer, rel_err, to_dev

pytestmark = pytest.mark.gpu
SH = gi.LAYER


def _seq_major(toks):
    """[steps][B][...] host tokens -> contiguous [B][steps][...]."""
    return {k: v.transpose(0, 1).contiguous() for k, v in toks.items()}


def _tokens(sh, steps, B, seed, offset=0):
    t = gi.make_tokens(sh, steps * B, seed, offset=offset * B)
    return {k: v.reshape(steps, B, *v.shape[1:]) for k, v in t.items()}


def _multi(dims, tok, params, conv, ssm, out, steps, slot=None, n_slots=None, ssm_trace=None,
           conv_trace=None, status=None):
    gdn.gdn_decode_multi(dims, tok["qkv"], tok["z"], tok["a"], tok["b"], params["A_log"],
                         params["dt_bias"], params["conv_w"], params["norm_w"], slot,
                         n_slots if n_slots is not None else conv.shape[0], conv, ssm, out, steps,
                         ssm_trace=ssm_trace, conv_trace=conv_trace, device_status=status,
                         batch=out.shape[0])


def _single(dims, tok, params, conv, ssm, out, slot=None, n_slots=None, status=None):
    gdn.gdn_decode_step(dims, tok["qkv"], tok["z"], tok["a"], tok["b"], params["A_log"],
                        params["dt_bias"], params["conv_w"], params["norm_w"], slot,
                        n_slots if n_slots is not None else conv.shape[0], conv, ssm, out,
                        device_status=status)


@pytest.mark.parametrize("h_k,h_v", [(16, 32), (16, 16), (8, 32)])   # G = 2, 1, 4
@pytest.mark.parametrize("steps", [1, 3, 8])
@pytest.mark.parametrize("use_slot", [False, True])
def test_decode_multi_equals_successive_single_steps_bitwise(h_k, h_v, steps, use_slot):
    # B = 37 sequences (not a multiple of any launch unit), states ~ N(0, 0.3)
    # and N(0, 1), seed 61; with use_slot the batch maps into a pool of 45
    # states in a scrambled order.
    sh = gi.Shape(h_k=h_k, h_v=h_v)
    B, pool = 37, 45
    params = to_dev(gi.make_params(sh, 61, norm_w="uniform"))
    dims = dims_of(sh)
    n = pool if use_slot else B
    st = gi.make_states(sh, n, 61, ssm_std=0.3, conv_std=1.0)
    perm = torch.randperm(pool, generator=torch.Generator().manual_seed(61))[:B]
    slot = perm.to(torch.int32).to(DEV) if use_slot else None
    toks = _tokens(sh, steps, B, 61)
    f32 = torch.float32
    for out_dtype in (f32, torch.bfloat16):
        conv_m, ssm_m = st["conv_state"].to(DEV), st["ssm_state"].to(DEV)
        conv_s, ssm_s = conv_m.clone(), ssm_m.clone()
        out_m = torch.full((B, steps, sh.h_v, sh.d_v), float("nan"), dtype=out_dtype, device=DEV)
        ssm_tr = torch.full((B, steps, sh.h_v, sh.d_v, sh.d_k), float("nan"), device=DEV)
        Cc = 2 * sh.h_k * sh.d_k + sh.h_v * sh.d_v
        conv_tr = torch.full((B, steps, sh.conv_w - 1, Cc), float("nan"), device=DEV)
        status = torch.zeros(1, dtype=torch.int32, device=DEV)
        _multi(dims, to_dev(_seq_major(toks)), params, conv_m, ssm_m, out_m, steps, slot=slot,
               n_slots=n, ssm_trace=ssm_tr, conv_trace=conv_tr, status=status)
        assert gdn.gdn_read_device_status(status) == 0
        rows = perm.tolist() if use_slot else list(range(B))
        for t in range(steps):
            out_s = torch.empty(B, sh.h_v, sh.d_v, dtype=out_dtype, device=DEV)
            _single(dims, to_dev({k: v[t] for k, v in toks.items()}), params, conv_s, ssm_s, out_s,
                    slot=slot, n_slots=n)
            assert torch.equal(out_m[:, t], out_s), f"token {t}: output differs"
            assert torch.equal(ssm_tr[:, t], ssm_s[rows]), f"token {t}: SSM trace differs"
            assert torch.equal(conv_tr[:, t], conv_s[rows]), f"token {t}: conv trace differs"
        assert torch.equal(ssm_m, ssm_s) and torch.equal(conv_m, conv_s)


def test_decode_multi_without_traces_matches_with_traces():
    # the trace writes are optional stores beside the same arithmetic: the
    # outputs and final states must not depend on them
    B, steps = 19, 5
    params = to_dev(gi.make_params(SH, 62))
    st = gi.make_states(SH, B, 62, ssm_std=0.3, conv_std=1.0)
    td = to_dev(_seq_major(_tokens(SH, steps, B, 62)))
    dims = dims_of(SH)
    res = []
    for traced in (False, True):
        conv, ssm = st["conv_state"].to(DEV), st["ssm_state"].to(DEV)
        out = torch.empty(B, steps, SH.h_v, SH.d_v, dtype=torch.bfloat16, device=DEV)
        tr = torch.empty(B, steps, SH.h_v, SH.d_v, SH.d_k, device=DEV) if traced else None
        _multi(dims, td, params, conv, ssm, out, steps, ssm_trace=tr)
        res.append((out, ssm, conv))
    for x, y in zip(*res):
        assert torch.equal(x, y)


def test_decode_multi_matches_oracle_over_32_tokens():
    # 4 sequences x 4 calls of 8 tokens, against the oracle's 32-token
    # sequences from the same starting states; fp32 output and state within 1e-4
    B, steps, calls = 4, 8, 4
    params = gi.make_params(SH, 63)
    st = gi.make_states(SH, B, 63, ssm_std=0.1 ** 0.5, conv_std=1.0)
    dims = dims_of(SH)
    pd = to_dev(params)
    conv, ssm = st["conv_state"].to(DEV), st["ssm_state"].to(DEV)
    toks = _tokens(SH, steps * calls, B, 63)
    out = torch.empty(B, steps * calls, SH.h_v, SH.d_v, device=DEV)
    for c in range(calls):
        chunk = {k: v[c * steps:(c + 1) * steps] for k, v in toks.items()}
        o = torch.empty(B, steps, SH.h_v, SH.d_v, device=DEV)
        _multi(dims, to_dev(_seq_major(chunk)), pd, conv, ssm, o, steps)
        out[:, c * steps:(c + 1) * steps] = o
    packed = {k: v.transpose(0, 1).reshape(B * steps * calls, *v.shape[2:]) for k, v in toks.items()}
    cu = np.arange(B + 1) * steps * calls
    ref, ref_conv, ref_ssm = oracle_layer(SH, packed, params, cu, conv_state=st["conv_state"],
                                          ssm_state=st["ssm_state"])
    assert rel_err(out.reshape(-1, SH.h_v, SH.d_v), ref) <= DECODE_TOL
    assert rel_err(ssm, ref_ssm) <= DECODE_TOL
    np.testing.assert_array_equal(conv.cpu().double().numpy(), ref_conv)


def test_decode_multi_flags_bad_slots_and_leaves_other_states():
    B, pool, steps = 4, 9, 3
    params = to_dev(gi.make_params(SH, 64))
    st = gi.make_states(SH, pool, 64, ssm_std=0.3, conv_std=1.0)
    td = to_dev(_seq_major(_tokens(SH, steps, B, 64)))
    dims = dims_of(SH)
    good = torch.tensor([7, 2, 8, 0], dtype=torch.int32, device=DEV)
    conv_g, ssm_g = st["conv_state"].to(DEV), st["ssm_state"].to(DEV)
    out_g = torch.empty(B, steps, SH.h_v, SH.d_v, device=DEV)
    _multi(dims, td, params, conv_g, ssm_g, out_g, steps, slot=good, n_slots=pool)
    conv_p, ssm_p = st["conv_state"].to(DEV), st["ssm_state"].to(DEV)
    out_p = torch.full((B, steps, SH.h_v, SH.d_v), float("nan"), device=DEV)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    bad = torch.tensor([7, pool, 8, -1], dtype=torch.int32, device=DEV)
    _multi(dims, td, params, conv_p, ssm_p, out_p, steps, slot=bad, n_slots=pool, status=status)
    assert gdn.gdn_read_device_status(status) == 6
    assert torch.equal(out_p[[0, 2]], out_g[[0, 2]])
    assert torch.isnan(out_p[[1, 3]]).all()
    assert torch.equal(ssm_p[[7, 8]], ssm_g[[7, 8]])
    keep = [0, 1, 2, 3, 4, 5, 6]
    assert torch.equal(ssm_p[keep].cpu(), st["ssm_state"][keep])
    assert torch.equal(conv_p[keep].cpu(), st["conv_state"][keep])


def test_decode_multi_one_token_without_traces_equals_single_step():
    # one token and no trace runs the single-step kernel; with a trace, the
    # multi-token kernel: both must give the single step's bits
    B = 11
    params = to_dev(gi.make_params(SH, 65))
    st = gi.make_states(SH, B, 65, ssm_std=0.3, conv_std=1.0)
    toks = _tokens(SH, 1, B, 65)
    dims = dims_of(SH)
    res = []
    for mode in ("single", "multi", "multi_traced"):
        conv, ssm = st["conv_state"].to(DEV), st["ssm_state"].to(DEV)
        if mode == "single":
            out = torch.empty(B, SH.h_v, SH.d_v, device=DEV)
            _single(dims, to_dev({k: v[0] for k, v in toks.items()}), params, conv, ssm, out)
        else:
            out = torch.empty(B, 1, SH.h_v, SH.d_v, device=DEV)
            tr = torch.empty(B, 1, SH.h_v, SH.d_v, SH.d_k, device=DEV) if mode == "multi_traced" else None
            _multi(dims, to_dev(_seq_major(toks)), params, conv, ssm, out, 1, ssm_trace=tr)
            out = out[:, 0]
        res.append((out, ssm, conv))
    for other in res[1:]:
        for x, y in zip(res[0], other):
            assert torch.equal(x, y)
