"""GPU parity of the dense projections around the layer (gdn_in_proj,
gdn_out_proj) and of the whole projected layer, against the fp64 oracle.

The projections are y = x w^T on the tensor cores: bf16 operands, fp32
accumulation, bf16 result.  Each element is checked against the oracle's
fp64 product as |gpu - ref| <= 1 bf16 ulp(ref) + 1e-4 max|ref| (the rounding
of the stored result, plus the fp32 accumulation).  The projected layer
(input projection, prefill or decode, output projection) is checked at the
prefill bar, 1e-2 of max|ref|.  Outputs start as NaN, so an element the
kernel never writes fails.
"""
import numpy as np
import pytest
import torch

import gated_deltanet_linear_06_gb300 as gdn
import gdn_inputs as gi
import oracle
from gpu_util import DEV, PREFILL_TOL, assert_bf16_close, dims_of, oracle_layer, rel_err

pytestmark = pytest.mark.gpu
SMALL = gi.Shape(h_k=2, h_v=8)     # 4 value heads per key head; 2576 input-projection features
PROJ_TOL = 1e-4


def _nan(*shape):
    return torch.full(shape, float("nan"), dtype=torch.bfloat16, device=DEV)


def _in_proj_gpu(sh, hidden, x, w_in):
    dims = dims_of(sh)
    T = x.shape[0]
    qkv, z, a, b = _nan(T, sh.cc), _nan(T, sh.h_v, sh.d_v), _nan(T, sh.h_v), _nan(T, sh.h_v)
    word = torch.zeros(1, dtype=torch.int32, device=DEV)
    gdn.gdn_in_proj(dims, hidden, x.to(DEV), w_in.to(DEV), qkv, z, a, b, device_status=word)
    assert gdn.gdn_read_device_status(word) == 0
    return qkv, z, a, b


@pytest.mark.parametrize("T,hidden", [(300, 192), (1, 64), (129, 256)])
def test_in_proj_matches_oracle(T, hidden):
    # 300 tokens: three row tiles with a ragged tail; 2576 features: eleven
    # column tiles, the last one partial, and every destination run
    sh = SMALL
    x = gi.make_hidden(T, hidden, seed=40)
    w = gi.make_proj_weights(sh, hidden, seed=40)["w_in"]
    got = _in_proj_gpu(sh, hidden, x, w)
    ref = oracle.linear(x, w)
    Cc, Cv = sh.cc, sh.cv
    parts = (ref[:, :Cc], ref[:, Cc:Cc + Cv].reshape(T, sh.h_v, sh.d_v), ref[:, Cc + Cv:Cc + Cv + sh.h_v],
             ref[:, Cc + Cv + sh.h_v:])
    for g, r in zip(got, parts):
        assert_bf16_close(g, r, tol=PROJ_TOL)


def test_in_proj_full_layer_shape_sampled_rows():
    # the 16/32-head layer at hidden 2048 over 32768 tokens (the size the bench
    # times), one launch; the oracle recomputes 48 sampled rows
    sh, hidden, T = gi.LAYER, 2048, 32768
    x = gi.make_hidden(T, hidden, seed=41)
    w = gi.make_proj_weights(sh, hidden, seed=41)["w_in"]
    qkv, z, a, b = _in_proj_gpu(sh, hidden, x, w)
    rows = np.sort(np.random.default_rng(41).choice(T, 48, replace=False))
    rows[-1] = T - 1
    ref = oracle.linear(x[rows], w)
    got = torch.cat([qkv[rows], z[rows].reshape(len(rows), -1), a[rows], b[rows]], 1)
    assert_bf16_close(got, ref, tol=PROJ_TOL)
    for t in (qkv, z, a, b):
        assert not torch.isnan(t.float()).any()


@pytest.mark.parametrize("T,hidden", [(300, 192), (1, 64), (200, 2048)])
def test_out_proj_matches_oracle(T, hidden):
    sh = SMALL
    dims = dims_of(sh)
    o = gi.make_hidden(T, sh.cv, seed=42).reshape(T, sh.h_v, sh.d_v)
    w = gi.make_proj_weights(sh, hidden, seed=42)["w_out"]
    y = _nan(T, hidden)
    gdn.gdn_out_proj(dims, hidden, o.to(DEV), w.to(DEV), y)
    assert_bf16_close(y, oracle.out_proj(o, w), tol=PROJ_TOL)


def test_out_proj_full_layer_shape_sampled_rows():
    sh, hidden, T = gi.LAYER, 2048, 32768
    dims = dims_of(sh)
    o = gi.make_hidden(T, sh.cv, seed=43).reshape(T, sh.h_v, sh.d_v)
    w = gi.make_proj_weights(sh, hidden, seed=43)["w_out"]
    y = _nan(T, hidden)
    gdn.gdn_out_proj(dims, hidden, o.to(DEV), w.to(DEV), y)
    rows = np.sort(np.random.default_rng(43).choice(T, 48, replace=False))
    rows[-1] = T - 1
    assert_bf16_close(y[rows], oracle.out_proj(o[rows], w), tol=PROJ_TOL)
    assert not torch.isnan(y.float()).any()


def _projected_prefill(sh, hidden, lengths, seed):
    dims = dims_of(sh)
    T, N = sum(lengths), len(lengths)
    x = gi.make_hidden(T, hidden, seed)
    w = gi.make_proj_weights(sh, hidden, seed)
    p = gi.make_params(sh, seed, norm_w="uniform")
    st = gi.make_states(sh, N, seed, ssm_std=0.1 ** 0.5, conv_std=1.0)
    # GPU: in_proj -> gdn_prefill -> out_proj, nothing reshaped in between
    qkv, z, a, b = _in_proj_gpu(sh, hidden, x, w["w_in"])
    pd = {k: v.to(DEV) for k, v in p.items()}
    conv, ssm = st["conv_state"].clone().to(DEV), st["ssm_state"].clone().to(DEV)
    out = _nan(T, sh.h_v, sh.d_v)
    cu = gi.cu_seqlens(lengths)
    ws = torch.empty(gdn.gdn_workspace_bytes(dims, N, T), dtype=torch.uint8, device=DEV)
    gdn.gdn_prefill(dims, qkv, z, a, b, pd["A_log"], pd["dt_bias"], pd["conv_w"], pd["norm_w"],
                    cu.to(DEV), conv, ssm, out, ws)
    assert gdn.gdn_read_device_status(ws) == 0
    y = _nan(T, hidden)
    gdn.gdn_out_proj(dims, hidden, out, w["w_out"].to(DEV), y)
    # oracle: the same chain in fp64, the layer's bf16 inputs and output rounded as stored
    r_qkv, r_z, r_a, r_b = oracle.in_proj(x, w["w_in"], h_k=sh.h_k, h_v=sh.h_v, d_k=sh.d_k, d_v=sh.d_v)
    r_out, _, r_ssm = oracle_layer(sh, {"qkv": r_qkv, "z": r_z, "a": r_a, "b": r_b}, p, cu,
                                   conv_state=st["conv_state"], ssm_state=st["ssm_state"])
    r_y = oracle.out_proj(oracle.round_bf16(r_out), w["w_out"])
    return rel_err(y, r_y), rel_err(ssm, r_ssm)


@pytest.mark.parametrize("sh,hidden,lengths", [(SMALL, 256, [300, 77, 0, 5]),
                                               (gi.LAYER, 2048, [640, 130])])
def test_projected_prefill_matches_oracle(sh, hidden, lengths):
    e_y, e_ssm = _projected_prefill(sh, hidden, lengths, seed=44)
    print(f"projected prefill: y {e_y:.2e}, state {e_ssm:.2e}")
    assert e_y <= PREFILL_TOL and e_ssm <= PREFILL_TOL, (e_y, e_ssm)


def test_projected_decode_steps_match_oracle():
    # 3 sequences, 2 tokens each: in_proj -> gdn_decode_step (bf16 out) -> out_proj per step
    sh, hidden, B, steps = gi.LAYER, 2048, 3, 2
    dims = dims_of(sh)
    x = gi.make_hidden(B * steps, hidden, seed=45)     # row s * B + n: step s, sequence n
    w = gi.make_proj_weights(sh, hidden, seed=45)
    p = gi.make_params(sh, 45)
    st = gi.make_states(sh, B, 45, ssm_std=0.1 ** 0.5, conv_std=1.0)
    pd = {k: v.to(DEV) for k, v in p.items()}
    conv, ssm = st["conv_state"].clone().to(DEV), st["ssm_state"].clone().to(DEV)
    ys = []
    for s in range(steps):
        qkv, z, a, b = _in_proj_gpu(sh, hidden, x[s * B:(s + 1) * B], w["w_in"])
        out = _nan(B, sh.h_v, sh.d_v)
        gdn.gdn_decode_step(dims, qkv, z, a, b, pd["A_log"], pd["dt_bias"], pd["conv_w"], pd["norm_w"],
                            None, B, conv, ssm, out)
        y = _nan(B, hidden)
        gdn.gdn_out_proj(dims, hidden, out, w["w_out"].to(DEV), y)
        ys.append(y.float().cpu())
    order = [s * B + n for n in range(B) for s in range(steps)]     # sequence-major packing
    r_qkv, r_z, r_a, r_b = oracle.in_proj(x[order], w["w_in"], h_k=sh.h_k, h_v=sh.h_v, d_k=sh.d_k,
                                          d_v=sh.d_v)
    r_out, _, r_ssm = oracle_layer(sh, {"qkv": r_qkv, "z": r_z, "a": r_a, "b": r_b}, p,
                                   [n * steps for n in range(B + 1)],
                                   conv_state=st["conv_state"], ssm_state=st["ssm_state"])
    r_y = oracle.out_proj(oracle.round_bf16(r_out), w["w_out"])
    got = torch.stack(ys, 1).reshape(B * steps, hidden)
    # the bar is the prefill's: the fp32-accumulated projection and the oracle's
    # fp64 one can round a few of the layer's bf16 inputs to neighbouring values
    e_y, e_ssm = rel_err(got, r_y), rel_err(ssm, r_ssm)
    assert e_y <= PREFILL_TOL and e_ssm <= PREFILL_TOL, (e_y, e_ssm)
