"""The tiny configuration (1 sequence of 64 tokens, 2 key / 2 value heads,
d_k = d_v = 32) on the GPU, through an exact embedding into the compiled
d = 128 kernels, against the fp64 oracle run at d = 32.

The kernels are compiled for head size 128 only.  A head-size-32 layer embeds
into them exactly: every q, k and v block, z and the conv weights get zero
channels 32 .. 127.  Zero channels stay zero through the conv and SiLU
(SiLU(0) = 0), add nothing to the q and k sums of squares, leave the padded
rows and columns of the state at zero (v and k^ are zero there) and give zero
outputs.  Two constants depend on the width:
  - q^ carries 1/sqrt(128) instead of 1/sqrt(32), so o is halved;
  - the RMSNorm's mean runs over 128 outputs, 96 of them zero.
Together the normalised output becomes 2 o / sqrt(sum(o^2)/32 + 16 eps) * w,
so the embedded layer runs with rms_eps / 16 and norm_w / 2, which makes it
equal to the d = 32 layer.  The activations are bf16 here (the GPU path's
input type) and the oracle reads the same bf16 values; the state is fp32.
"""
import numpy as np
import pytest
import torch

import gated_deltanet_linear_06_gb300 as gdn
import gdn_inputs as gi
import oracle
from gpu_util import DECODE_TOL, DEV, PREFILL_TOL, rel_err

pytestmark = pytest.mark.gpu
TINY = gi.TINY          # h_k = h_v = 2, d = 32
WIDE = 128
EPS = 1e-6


def _pad_blocks(x, n_blocks, d, axis=-1):
    """[..., n_blocks * d] -> [..., n_blocks * WIDE], block b's d channels first."""
    shp = x.shape[:-1]
    xb = x.reshape(*shp, n_blocks, d)
    out = torch.zeros(*shp, n_blocks, WIDE, dtype=x.dtype)
    out[..., :d] = xb
    return out.reshape(*shp, n_blocks * WIDE)


def _inputs(seed, slow):
    T = 64
    p = gi.make_params(TINY, seed)          # bf16 conv weights
    tok = gi.make_tokens(TINY, T, seed)
    if slow:
        gc = gi.gate_controlled(TINY, T, seed)
        tok["a"], tok["b"] = gc["a"], gc["b"]
        p["A_log"], p["dt_bias"] = gc["A_log"], gc["dt_bias"]
    return p, tok


def _padded(p, tok):
    d, hk, hv = TINY.d_k, TINY.h_k, TINY.h_v
    T = tok["qkv"].shape[0]
    q, k, v = tok["qkv"][:, :hk * d], tok["qkv"][:, hk * d:2 * hk * d], tok["qkv"][:, 2 * hk * d:]
    qkv = torch.cat([_pad_blocks(q, hk, d), _pad_blocks(k, hk, d), _pad_blocks(v, hv, d)], 1)
    z = _pad_blocks(tok["z"].reshape(T, hv * d), hv, d).reshape(T, hv, WIDE)
    cw = p["conv_w"]                                     # [Cc][W], channels as qkv
    cq, ck, cv = cw[:hk * d], cw[hk * d:2 * hk * d], cw[2 * hk * d:]
    pad_w = lambda w, nb: _pad_blocks(w.t().contiguous(), nb, d).t().contiguous()
    conv_w = torch.cat([pad_w(cq, hk), pad_w(ck, hk), pad_w(cv, hv)], 0)
    norm_w = torch.zeros(WIDE)
    norm_w[:d] = p["norm_w"] / 2
    return ({"qkv": qkv.contiguous(), "z": z.contiguous(), "a": tok["a"], "b": tok["b"]},
            {"A_log": p["A_log"], "dt_bias": p["dt_bias"], "conv_w": conv_w, "norm_w": norm_w})


def _oracle(p, tok):
    return oracle.layer(h_k=TINY.h_k, h_v=TINY.h_v, d_k=TINY.d_k, d_v=TINY.d_v, qkv=tok["qkv"],
                        z=tok["z"], a=tok["a"], b=tok["b"], A_log=p["A_log"], dt_bias=p["dt_bias"],
                        conv_w=p["conv_w"], norm_w=p["norm_w"], cu_seqlens=[0, 64],
                        l2_eps=EPS, rms_eps=EPS)


def _dims():
    return gdn.make_dims(h_k=TINY.h_k, h_v=TINY.h_v, d_k=WIDE, d_v=WIDE, l2_eps=EPS, rms_eps=EPS / 16)


@pytest.mark.parametrize("slow", [False, True])
def test_tiny_config_prefill_through_the_embedding(slow):
    p, tok = _inputs(0, slow)
    ref, ref_conv, ref_ssm = _oracle(p, tok)
    xt, pp = _padded(p, tok)
    xt, pp = {k: v.to(DEV) for k, v in xt.items()}, {k: v.to(DEV) for k, v in pp.items()}
    dims = _dims()
    cc = 2 * TINY.h_k * WIDE + TINY.h_v * WIDE
    conv = torch.zeros(1, 3, cc, device=DEV)
    ssm = torch.zeros(1, TINY.h_v, WIDE, WIDE, device=DEV)
    out = torch.full((64, TINY.h_v, WIDE), float("nan"), dtype=torch.bfloat16, device=DEV)
    ws = torch.empty(gdn.gdn_workspace_bytes(dims, 1, 64), dtype=torch.uint8, device=DEV)
    gdn.gdn_prefill(dims, xt["qkv"], xt["z"], xt["a"], xt["b"], pp["A_log"], pp["dt_bias"],
                    pp["conv_w"], pp["norm_w"], gi.cu_seqlens([64]).to(DEV), conv, ssm, out, ws)
    assert gdn.gdn_read_device_status(ws) == 0
    d = TINY.d_k
    e_out = rel_err(out[:, :, :d], ref)
    e_ssm = rel_err(ssm[:, :, :d, :d], ref_ssm)
    assert e_out <= PREFILL_TOL and e_ssm <= PREFILL_TOL, (e_out, e_ssm)
    # the padding stays exactly zero
    assert not out[:, :, d:].float().any() and not ssm[:, :, d:, :].any() and not ssm[:, :, :, d:].any()
    # the conv state holds the last three raw inputs of the real channels
    conv_real = torch.cat([conv[0, :, blk * WIDE: blk * WIDE + d] for blk in range(cc // WIDE)], 1)
    np.testing.assert_array_equal(conv_real.cpu().double().numpy(), ref_conv[0])


def test_tiny_config_decode_through_the_embedding():
    # the same 64 tokens fed one decode step at a time, fp32 output
    p, tok = _inputs(0, slow=True)
    ref, _, ref_ssm = _oracle(p, tok)
    xt, pp = _padded(p, tok)
    xt, pp = {k: v.to(DEV) for k, v in xt.items()}, {k: v.to(DEV) for k, v in pp.items()}
    dims = _dims()
    cc = 2 * TINY.h_k * WIDE + TINY.h_v * WIDE
    conv = torch.zeros(1, 3, cc, device=DEV)
    ssm = torch.zeros(1, TINY.h_v, WIDE, WIDE, device=DEV)
    outs = []
    for t in range(64):
        o = torch.empty(1, TINY.h_v, WIDE, device=DEV)
        # one token's rows, each in its own (16-byte aligned) buffer
        tk = {k: v[t:t + 1].clone() for k, v in xt.items()}
        gdn.gdn_decode_step(dims, tk["qkv"], tk["z"], tk["a"], tk["b"], pp["A_log"], pp["dt_bias"],
                            pp["conv_w"], pp["norm_w"], None, 1, conv, ssm, o)
        outs.append(o)
    got = torch.cat(outs, 0)
    d = TINY.d_k
    e_out = rel_err(got[:, :, :d], ref)
    e_ssm = rel_err(ssm[:, :, :d, :d], ref_ssm)
    assert e_out <= DECODE_TOL and e_ssm <= DECODE_TOL, (e_out, e_ssm)
    assert not got[:, :, d:].any()
