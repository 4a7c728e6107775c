"""GPU checks of the captured decode chain (gdn_decode_graph_*), through the C ABI.

Bars: a graph launch is bit-identical to the same gdn_decode_step calls made
one by one (outputs and states), also after the caller refills the bound
buffers; over the 3-sequence x 1024-step decode workload the graph path meets
the single step's 1e-4 bar against the fp64 oracle.
"""
import numpy as np
import pytest
import torch

import gated_deltanet_linear_06_gb300 as gdn
import gdn_inputs as gi
from gpu_util import DECODE_TOL, DEV, dims_of, oracle_layer, rel_err, to_dev

pytestmark = pytest.mark.gpu
SH = gi.LAYER


def _tokens(steps, B, seed, offset=0):
    t = gi.make_tokens(SH, steps * B, seed, offset=offset * B)
    return {k: v.reshape(steps, B, *v.shape[1:]) for k, v in t.items()}


def _eager(dims, toks, params, conv, ssm, out, slot=None, n_slots=None):
    for t in range(toks["qkv"].shape[0]):
        gdn.gdn_decode_step(dims, toks["qkv"][t], toks["z"][t], toks["a"][t], toks["b"][t],
                            params["A_log"], params["dt_bias"], params["conv_w"], params["norm_w"],
                            slot, n_slots if n_slots is not None else conv.shape[0], conv, ssm,
                            out[t])


@pytest.mark.parametrize("use_slot,out_dtype", [(False, torch.float32), (True, torch.bfloat16)])
def test_graph_launch_equals_eager_steps_bitwise(use_slot, out_dtype):
    # B = 3 sequences x 64 steps per launch (seed 81), two launches with the
    # buffers refilled in between; with use_slot the 3 sequences live in slots
    # 4, 0, 2 of a 5-slot pool
    B, S = 3, 64
    dims = dims_of(SH)
    params = to_dev(gi.make_params(SH, 81))
    n = 5 if use_slot else B
    st = gi.make_states(SH, n, 81, ssm_std=0.1 ** 0.5, conv_std=1.0)
    slot = torch.tensor([4, 0, 2], dtype=torch.int32, device=DEV) if use_slot else None
    conv_g, ssm_g = st["conv_state"].to(DEV), st["ssm_state"].to(DEV)
    conv_e, ssm_e = conv_g.clone(), ssm_g.clone()
    bound = to_dev(_tokens(S, B, 81))
    out_g = torch.empty(S, B, SH.h_v, SH.d_v, dtype=out_dtype, device=DEV)
    out_e = torch.empty_like(out_g)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    g = gdn.gdn_decode_graph_create(dims, S, bound["qkv"], bound["z"], bound["a"], bound["b"],
                                    params["A_log"], params["dt_bias"], params["conv_w"],
                                    params["norm_w"], slot, n, conv_g, ssm_g, out_g,
                                    device_status=status)
    try:
        for launch in range(2):
            if launch:
                for k, v in to_dev(_tokens(S, B, 81, offset=S)).items():
                    bound[k].copy_(v)
            g.launch()
            _eager(dims, bound, params, conv_e, ssm_e, out_e, slot=slot, n_slots=n)
            assert torch.equal(out_g, out_e), f"launch {launch}: outputs differ"
            assert torch.equal(ssm_g, ssm_e) and torch.equal(conv_g, conv_e)
        assert gdn.gdn_read_device_status(status) == 0
    finally:
        g.close()


def test_graph_path_three_sequences_1024_steps_matches_oracle():
    # the 3-sequence decode workload (state ~ N(0, 0.1), conv state ~ N(0, 1),
    # seed 1) run as 16 launches of one 64-step graph, the caller refilling the
    # bound token buffers before each; checked against the oracle after every
    # launch
    B, S, launches = 3, 64, 16
    dims = dims_of(SH)
    params = gi.make_params(SH, 1)
    pd = to_dev(params)
    st = gi.make_states(SH, B, 1, ssm_std=0.1 ** 0.5, conv_std=1.0)
    conv, ssm = st["conv_state"].to(DEV), st["ssm_state"].to(DEV)
    ref_conv, ref_ssm = st["conv_state"].double().numpy(), st["ssm_state"].double().numpy()
    bound = to_dev(_tokens(S, B, 1))
    out = torch.empty(S, B, SH.h_v, SH.d_v, device=DEV)
    g = gdn.gdn_decode_graph_create(dims, S, bound["qkv"], bound["z"], bound["a"], bound["b"],
                                    pd["A_log"], pd["dt_bias"], pd["conv_w"], pd["norm_w"], None,
                                    B, conv, ssm, out)
    try:
        for L in range(launches):
            toks = _tokens(S, B, 1, offset=L * S)
            for k, v in to_dev(toks).items():
                bound[k].copy_(v)
            g.launch()
            packed = {k: v.transpose(0, 1).reshape(B * S, *v.shape[2:]) for k, v in toks.items()}
            ref, ref_conv, ref_ssm = oracle_layer(SH, packed, params, np.arange(B + 1) * S,
                                                  conv_state=ref_conv, ssm_state=ref_ssm)
            ref = ref.reshape(B, S, SH.h_v, SH.d_v).transpose(1, 0, 2, 3)
            assert rel_err(out, ref) <= DECODE_TOL, f"launch {L}"
            assert rel_err(ssm, ref_ssm) <= DECODE_TOL, f"launch {L}"
            np.testing.assert_array_equal(conv.cpu().double().numpy(), ref_conv)
    finally:
        g.close()


@pytest.mark.parametrize("S,h_k,h_v,B", [(1, 16, 32, 2), (2, 32, 32, 2), (5, 8, 32, 2), (3, 16, 32, 2),
                                         (6, 16, 32, 48)])
def test_short_chains_and_head_groupings_equal_eager_steps_bitwise(S, h_k, h_v, B):
    # chains shorter than the conv window (the conv state after the chain then
    # keeps rows of the starting one), 1, 2 and 4 value heads per key head, and
    # a batch of 48 whose 3072 CTAs run in several waves
    sh = gi.Shape(h_k=h_k, h_v=h_v)
    dims = dims_of(sh)
    params = to_dev(gi.make_params(sh, 82))
    st = gi.make_states(sh, B, 82, ssm_std=0.1 ** 0.5, conv_std=1.0)
    conv_g, ssm_g = st["conv_state"].to(DEV), st["ssm_state"].to(DEV)
    conv_e, ssm_e = conv_g.clone(), ssm_g.clone()
    t = gi.make_tokens(sh, S * B, 82)
    bound = to_dev({k: v.reshape(S, B, *v.shape[1:]) for k, v in t.items()})
    out_g = torch.empty(S, B, sh.h_v, sh.d_v, device=DEV)
    out_e = torch.empty_like(out_g)
    g = gdn.gdn_decode_graph_create(dims, S, bound["qkv"], bound["z"], bound["a"], bound["b"],
                                    params["A_log"], params["dt_bias"], params["conv_w"],
                                    params["norm_w"], None, B, conv_g, ssm_g, out_g)
    try:
        for launch in range(2):
            g.launch()
            for s in range(S):
                gdn.gdn_decode_step(dims, bound["qkv"][s], bound["z"][s], bound["a"][s], bound["b"][s],
                                    params["A_log"], params["dt_bias"], params["conv_w"],
                                    params["norm_w"], None, B, conv_e, ssm_e, out_e[s])
            assert torch.equal(out_g, out_e), f"launch {launch}"
            assert torch.equal(ssm_g, ssm_e) and torch.equal(conv_g, conv_e), f"launch {launch}"
    finally:
        g.close()


def test_graph_with_a_bad_slot_reports_it_and_leaves_that_entry_alone():
    # entry 1's slot is out of range: it is skipped on the device (its output
    # rows keep their NaN canary), the others decode as eager steps do
    B, S, n = 3, 4, 3
    dims = dims_of(SH)
    params = to_dev(gi.make_params(SH, 83))
    st = gi.make_states(SH, n, 83, ssm_std=0.1 ** 0.5, conv_std=1.0)
    slot = torch.tensor([2, 7, 0], dtype=torch.int32, device=DEV)
    conv_g, ssm_g = st["conv_state"].to(DEV), st["ssm_state"].to(DEV)
    conv_e, ssm_e = conv_g.clone(), ssm_g.clone()
    t = gi.make_tokens(SH, S * B, 83)
    bound = to_dev({k: v.reshape(S, B, *v.shape[1:]) for k, v in t.items()})
    out_g = torch.full((S, B, SH.h_v, SH.d_v), float("nan"), device=DEV)
    out_e = out_g.clone()
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    g = gdn.gdn_decode_graph_create(dims, S, bound["qkv"], bound["z"], bound["a"], bound["b"],
                                    params["A_log"], params["dt_bias"], params["conv_w"],
                                    params["norm_w"], slot, n, conv_g, ssm_g, out_g,
                                    device_status=status)
    try:
        g.launch()
    finally:
        g.close()
    assert gdn.gdn_read_device_status(status) == gdn.GDN_ERR_DEVICE_BOUNDS
    _eager(dims, bound, params, conv_e, ssm_e, out_e, slot=slot, n_slots=n)
    assert torch.isnan(out_g[:, 1]).all()
    assert torch.equal(out_g[:, [0, 2]], out_e[:, [0, 2]])
    assert torch.equal(ssm_g, ssm_e) and torch.equal(conv_g, conv_e)
