"""GPU checks of gdn_prefill_host (host activations, copies overlapped with compute), through the C ABI.

Bars: bit-identical to the same segments fed to gdn_prefill one after another
on device copies of the inputs; one segment covering everything is
bit-identical to a single gdn_prefill call; against the fp64 oracle the
prefill's 1e-2 bar on the output and the final state, the conv state exact.
"""
import numpy as np
import pytest
import torch

import gated_deltanet_linear_06_gb300 as gdn
import gdn_inputs as gi
from gpu_util import DEV, PREFILL_TOL, dims_of, oracle_layer, rel_err, to_dev

pytestmark = pytest.mark.gpu
SH = gi.LAYER


def _segments(cu, T, seg):
    """The library's segmentation: token ranges of `seg`, each with the range of
    sequences holding its tokens and their local cu_seqlens."""
    out, j = [], 0
    for s0 in range(0, T, seg):
        s1 = min(T, s0 + seg)
        while cu[j + 1] <= s0:
            j += 1
        jb = j
        while cu[jb + 1] < s1:
            jb += 1
        local = [0] + [min(cu[q + 1], s1) - s0 for q in range(j, jb + 1)]
        out.append((s0, s1, j, jb - j + 1, local))
    return out


def _host_call(dims, tok, pd, cu_list, st, seg, pinned=True):
    # page-locked buffers let the library's copies run asynchronously; pageable ones still work
    T = tok["qkv"].shape[0]
    N = len(cu_list) - 1
    host_mem = (lambda t: t.pin_memory()) if pinned else (lambda t: t.clone())
    host = {k: host_mem(v.contiguous()) for k, v in tok.items()}
    out = host_mem(torch.full((T, SH.h_v, SH.d_v), float("nan"), dtype=torch.bfloat16))
    conv, ssm = st["conv_state"].clone().to(DEV), st["ssm_state"].clone().to(DEV)
    ws = torch.empty(gdn.gdn_prefill_host_workspace_bytes(dims, N, T, seg), dtype=torch.uint8,
                     device=DEV)
    gdn.gdn_prefill_host(dims, host["qkv"], host["z"], host["a"], host["b"], pd["A_log"],
                         pd["dt_bias"], pd["conv_w"], pd["norm_w"],
                         torch.tensor(cu_list, dtype=torch.int32), conv, ssm, out, ws,
                         seg_tokens=seg)
    torch.cuda.synchronize()
    assert gdn.gdn_read_device_status(ws) == 0
    return out, conv, ssm


def _segmented_device_calls(dims, tok, pd, cu_list, st, seg):
    T = tok["qkv"].shape[0]
    td = to_dev(tok)
    out = torch.empty(T, SH.h_v, SH.d_v, dtype=torch.bfloat16, device=DEV)
    conv, ssm = st["conv_state"].clone().to(DEV), st["ssm_state"].clone().to(DEV)
    for s0, s1, ja, nj, local in _segments(cu_list, T, seg):
        ws = torch.empty(gdn.gdn_workspace_bytes(dims, nj, s1 - s0), dtype=torch.uint8, device=DEV)
        gdn.gdn_prefill(dims, td["qkv"][s0:s1], td["z"][s0:s1], td["a"][s0:s1], td["b"][s0:s1],
                        pd["A_log"], pd["dt_bias"], pd["conv_w"], pd["norm_w"],
                        torch.tensor(local, dtype=torch.int32, device=DEV),
                        conv[ja:ja + nj], ssm[ja:ja + nj], out[s0:s1], ws)
        assert gdn.gdn_read_device_status(ws) == 0
    return out.cpu(), conv, ssm


def _problem(lengths, seed):
    cu_list = [0]
    for n in lengths:
        cu_list.append(cu_list[-1] + n)
    T = cu_list[-1]
    params = gi.make_params(SH, seed)
    tok = gi.make_tokens(SH, T, seed)
    st = gi.make_states(SH, len(lengths), seed, ssm_std=0.1 ** 0.5, conv_std=1.0)
    return cu_list, params, tok, st


@pytest.mark.parametrize("seg,pinned", [(1024, True), (320, True), (320, False), (100, True)])
def test_prefill_host_equals_segmented_device_calls_and_matches_oracle(seg, pinned):
    # lengths 5000, 3, 0, 1200, 2500 (seed 91, carried states): segment
    # boundaries cut sequences, a 3-token sequence and an empty one sit inside;
    # 100-token segments start at token offsets that are no multiple of 8
    lengths = [5000, 3, 0, 1200, 2500]
    cu_list, params, tok, st = _problem(lengths, 91)
    dims = dims_of(SH)
    pd = to_dev(params)
    out_h, conv_h, ssm_h = _host_call(dims, tok, pd, cu_list, st, seg, pinned)
    out_d, conv_d, ssm_d = _segmented_device_calls(dims, tok, pd, cu_list, st, seg)
    assert torch.equal(out_h, out_d)
    assert torch.equal(ssm_h, ssm_d) and torch.equal(conv_h, conv_d)
    if seg == 1024:
        ref, ref_conv, ref_ssm = oracle_layer(SH, tok, params, np.array(cu_list),
                                              conv_state=st["conv_state"], ssm_state=st["ssm_state"])
        assert rel_err(out_h, ref) <= PREFILL_TOL
        assert rel_err(ssm_h, ref_ssm) <= PREFILL_TOL
        np.testing.assert_array_equal(conv_h.cpu().double().numpy(), ref_conv)


def test_prefill_host_one_segment_equals_one_device_call():
    lengths = [700, 1, 900]
    cu_list, params, tok, st = _problem(lengths, 92)
    dims = dims_of(SH)
    pd = to_dev(params)
    T = cu_list[-1]
    out_h, conv_h, ssm_h = _host_call(dims, tok, pd, cu_list, st, 4096)
    out_d, conv_d, ssm_d = _segmented_device_calls(dims, tok, pd, cu_list, st, T)
    assert len(_segments(cu_list, T, T)) == 1
    assert torch.equal(out_h, out_d)
    assert torch.equal(ssm_h, ssm_d) and torch.equal(conv_h, conv_d)
