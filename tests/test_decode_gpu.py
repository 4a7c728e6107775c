"""GPU parity of gdn_decode_step against the fp64 oracle, through the C ABI.

Bars: max |gpu - oracle| / max |oracle| <= 1e-4 on the fp32 state and the
fp32 output; the bf16 output within one bf16 ulp of the oracle plus that
same 1e-4 carried through the rounding; a sequence bit-identical alone and
inside a batch.
"""
import numpy as np
import pytest
import torch

import gated_deltanet_linear_06_gb300 as gdn
import gdn_inputs as gi
from gpu_util import DECODE_TOL, DEV, assert_bf16_close, dims_of, oracle_layer, rel_err, to_dev

pytestmark = pytest.mark.gpu
SH = gi.LAYER


def _step(dims, tok, params, conv, ssm, out, slot=None, n_slots=None, status=None):
    gdn.gdn_decode_step(dims, tok["qkv"], tok["z"], tok["a"], tok["b"], params["A_log"],
                        params["dt_bias"], params["conv_w"], params["norm_w"], slot,
                        n_slots if n_slots is not None else conv.shape[0], conv, ssm, out,
                        device_status=status)


def _oracle_steps(sh, toks, params, conv0, ssm0, seq_ids=None):
    """Oracle over S steps of B sequences: toks[k] is [S, B, ...]; each
    sequence's S tokens form one packed sequence of length S."""
    S, B = toks["qkv"].shape[:2]
    ids = list(range(B)) if seq_ids is None else list(seq_ids)
    packed = {k: v[:, ids].transpose(0, 1).reshape(len(ids) * S, *v.shape[2:]) for k, v in toks.items()}
    cu = np.arange(len(ids) + 1) * S
    return oracle_layer(sh, packed, params, cu, conv_state=conv0[ids], ssm_state=ssm0[ids])


def _tokens(sh, steps, B, seed, offset=0, gates=None):
    t = gi.make_tokens(sh, steps * B, seed, offset=offset * B)
    if gates is not None:
        g = gi.gate_controlled(sh, steps * B, seed, decay=gates[0], beta=gates[1], offset=offset)
        t["a"], t["b"] = g["a"], g["b"]
    return {k: v.reshape(steps, B, *v.shape[1:]) for k, v in t.items()}


@pytest.mark.parametrize("slow", [False, True])
def test_decode_three_sequences_1024_steps(slow):
    # 3 sequences, 1024 successive tokens each; state ~ N(0, 0.1), conv state
    # ~ N(0, 1), seed 1.  Checked every 64th step and at the last step.
    B, steps, block = 3, (1024 if not slow else 256), 64
    params = gi.make_params(SH, 1)
    gates = ((0.9, 1.0), (0.0, 0.3)) if slow else None
    if slow:
        gc = gi.gate_controlled(SH, 1, 1)
        params["A_log"], params["dt_bias"] = gc["A_log"], gc["dt_bias"]
    st = gi.make_states(SH, B, 1, ssm_std=0.1 ** 0.5, conv_std=1.0)
    dims = dims_of(SH)
    pd = to_dev(params)
    conv, ssm = st["conv_state"].to(DEV), st["ssm_state"].to(DEV)
    ref_conv, ref_ssm = st["conv_state"].double().numpy(), st["ssm_state"].double().numpy()
    out = torch.empty(B, SH.h_v, SH.d_v, device=DEV)
    worst = 0.0
    for b0 in range(0, steps, block):
        toks = _tokens(SH, block, B, 1, offset=b0, gates=gates)
        for s in range(block):
            _step(dims, to_dev({k: v[s] for k, v in toks.items()}), pd, conv, ssm, out)
        ref_out, ref_conv, ref_ssm = _oracle_steps(SH, toks, params, ref_conv, ref_ssm)
        ref_last = ref_out.reshape(B, block, SH.h_v, SH.d_v)[:, -1]
        e = max(rel_err(out, ref_last), rel_err(ssm, ref_ssm))
        np.testing.assert_array_equal(conv.cpu().double().numpy(), ref_conv)
        worst = max(worst, e)
        assert e <= DECODE_TOL, f"step {b0 + block}: rel err {e:.3e}"
    print(f"worst rel err over {steps} steps: {worst:.3e}")


def test_decode_bf16_output_within_one_ulp():
    B, steps = 5, 4
    params = gi.make_params(SH, 11, norm_w="uniform")
    st = gi.make_states(SH, B, 11, ssm_std=0.1 ** 0.5, conv_std=1.0)
    dims = dims_of(SH)
    pd = to_dev(params)
    conv, ssm = st["conv_state"].to(DEV), st["ssm_state"].to(DEV)
    toks = _tokens(SH, steps, B, 11)
    out = torch.empty(steps, B, SH.h_v, SH.d_v, dtype=torch.bfloat16, device=DEV)
    for s in range(steps):
        _step(dims, to_dev({k: v[s] for k, v in toks.items()}), pd, conv, ssm, out[s])
    ref, _, _ = _oracle_steps(SH, toks, params, st["conv_state"], st["ssm_state"])
    ref = ref.reshape(B, steps, SH.h_v, SH.d_v).transpose(1, 0, 2, 3)
    assert_bf16_close(out, ref)


def test_decode_solo_equals_batched_bitwise_256x256():
    # B = 256 sequences x 256 steps, exp(g) ~ U(0.5, 1), seed 4: sequence 0
    # alone and sequence 0 inside the batch must agree bit for bit after every
    # step (output and state); sampled sequences also match the oracle.
    B, steps = 256, 256
    params = gi.make_params(SH, 4)
    gc = gi.gate_controlled(SH, 1, 4)
    params["A_log"], params["dt_bias"] = gc["A_log"], gc["dt_bias"]
    st = gi.make_states(SH, B, 4, ssm_std=0.1 ** 0.5, conv_std=1.0)
    dims = dims_of(SH)
    pd = to_dev(params)
    conv, ssm = st["conv_state"].to(DEV), st["ssm_state"].to(DEV)
    conv1, ssm1 = conv[:1].clone(), ssm[:1].clone()
    out = torch.empty(B, SH.h_v, SH.d_v, dtype=torch.bfloat16, device=DEV)
    out1 = torch.empty(1, SH.h_v, SH.d_v, dtype=torch.bfloat16, device=DEV)
    sample = [0, 131, 255]
    kept = {k: [] for k in ("qkv", "z", "a", "b")}
    outs = []
    for s in range(steps):
        t = _tokens(SH, 1, B, 4, offset=s, gates=((0.5, 1.0), (0.0, 1.0)))
        t = {k: v[0] for k, v in t.items()}
        td = to_dev(t)
        _step(dims, td, pd, conv, ssm, out)
        _step(dims, {k: v[:1] for k, v in td.items()}, pd, conv1, ssm1, out1)
        assert torch.equal(out[:1], out1), f"step {s}: output differs solo vs batched"
        assert torch.equal(ssm[:1], ssm1), f"step {s}: state differs solo vs batched"
        assert torch.equal(conv[:1], conv1), f"step {s}: conv state differs"
        for k in kept:
            kept[k].append(t[k][sample])
        outs.append(out[sample].float().cpu())
    toks = {k: torch.stack(v) for k, v in kept.items()}
    ref, _, ref_ssm = _oracle_steps(SH, toks, params, st["conv_state"][sample],
                                    st["ssm_state"][sample])
    got = torch.stack(outs, 1).reshape(len(sample) * steps, SH.h_v, SH.d_v)
    assert rel_err(ssm[sample], ref_ssm) <= DECODE_TOL
    assert_bf16_close(got, ref)


def test_decode_slot_indirection_matches_dense_and_flags_bad_slots():
    B, pool = 4, 9
    params = gi.make_params(SH, 21)
    st = gi.make_states(SH, pool, 21, ssm_std=0.3, conv_std=1.0)
    dims = dims_of(SH)
    pd = to_dev(params)
    toks = {k: v[0] for k, v in _tokens(SH, 1, B, 21).items()}
    td = to_dev(toks)
    slots = [7, 2, 8, 0]
    # dense reference: states gathered into batch order
    conv_d = st["conv_state"][slots].to(DEV)
    ssm_d = st["ssm_state"][slots].to(DEV)
    out_d = torch.empty(B, SH.h_v, SH.d_v, device=DEV)
    _step(dims, td, pd, conv_d, ssm_d, out_d)
    conv_p, ssm_p = st["conv_state"].to(DEV), st["ssm_state"].to(DEV)
    out_p = torch.empty(B, SH.h_v, SH.d_v, device=DEV)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    _step(dims, td, pd, conv_p, ssm_p, out_p, slot=torch.tensor(slots, dtype=torch.int32, device=DEV),
          n_slots=pool, status=status)
    assert gdn.gdn_read_device_status(status) == 0
    assert torch.equal(out_p, out_d)
    assert torch.equal(ssm_p[slots], ssm_d) and torch.equal(conv_p[slots], conv_d)
    untouched = [i for i in range(pool) if i not in slots]
    assert torch.equal(ssm_p[untouched].cpu(), st["ssm_state"][untouched])
    # an out-of-range slot: that entry is skipped and the status word says so
    conv_p, ssm_p = st["conv_state"].to(DEV), st["ssm_state"].to(DEV)
    out_p = torch.full((B, SH.h_v, SH.d_v), float("nan"), device=DEV)
    bad = torch.tensor([7, pool, 8, -1], dtype=torch.int32, device=DEV)
    _step(dims, td, pd, conv_p, ssm_p, out_p, slot=bad, n_slots=pool, status=status)
    assert gdn.gdn_read_device_status(status) == 6
    assert torch.equal(out_p[[0, 2]], out_d[[0, 2]])
    assert torch.isnan(out_p[[1, 3]]).all()
    assert torch.equal(ssm_p[[0, 2, 1, 3, 4, 5, 6]].cpu(), st["ssm_state"][[0, 2, 1, 3, 4, 5, 6]])


@pytest.mark.parametrize("h_k,h_v", [(32, 32), (8, 32), (2, 4)])
def test_decode_other_head_groupings(h_k, h_v):
    sh = gi.Shape(h_k=h_k, h_v=h_v)
    B, steps = 3, 3
    params = gi.make_params(sh, 31, norm_w="uniform")
    st = gi.make_states(sh, B, 31, ssm_std=0.3, conv_std=1.0)
    dims = dims_of(sh)
    pd = to_dev(params)
    conv, ssm = st["conv_state"].to(DEV), st["ssm_state"].to(DEV)
    toks = _tokens(sh, steps, B, 31)
    out = torch.empty(steps, B, sh.h_v, sh.d_v, device=DEV)
    for s in range(steps):
        _step(dims, to_dev({k: v[s] for k, v in toks.items()}), pd, conv, ssm, out[s])
    ref, ref_conv, ref_ssm = _oracle_steps(sh, toks, params, st["conv_state"], st["ssm_state"])
    ref = ref.reshape(B, steps, sh.h_v, sh.d_v).transpose(1, 0, 2, 3)
    assert rel_err(out, ref) <= DECODE_TOL
    assert rel_err(ssm, ref_ssm) <= DECODE_TOL
    np.testing.assert_array_equal(conv.cpu().double().numpy(), ref_conv)


def test_decode_zero_write_and_no_decay_keeps_state_bitwise():
    # beta = 0 and exp(g) = 1 (A_log very negative, b very negative): the
    # state must come back bit for bit, and the output is S q^ normalised
    B = 2
    params = gi.make_params(SH, 41)
    params["A_log"] = torch.full((SH.h_v,), -100.0)
    st = gi.make_states(SH, B, 41, ssm_std=0.3, conv_std=1.0)
    toks = {k: v[0] for k, v in _tokens(SH, 1, B, 41).items()}
    toks["b"] = torch.full_like(toks["b"], -100.0)
    dims = dims_of(SH)
    conv, ssm = st["conv_state"].to(DEV), st["ssm_state"].to(DEV)
    out = torch.empty(B, SH.h_v, SH.d_v, device=DEV)
    _step(dims, to_dev(toks), to_dev(params), conv, ssm, out)
    assert torch.equal(ssm.cpu(), st["ssm_state"])
    ref, _, _ = _oracle_steps(SH, {k: v[None] for k, v in toks.items()}, params,
                              st["conv_state"], st["ssm_state"])
    assert rel_err(out, ref) <= DECODE_TOL


def test_decode_is_deterministic():
    B = 7
    params = to_dev(gi.make_params(SH, 51))
    st = gi.make_states(SH, B, 51, ssm_std=0.3, conv_std=1.0)
    td = to_dev({k: v[0] for k, v in _tokens(SH, 1, B, 51).items()})
    dims = dims_of(SH)
    res = []
    for _ in range(2):
        conv, ssm = st["conv_state"].to(DEV), st["ssm_state"].to(DEV)
        out = torch.empty(B, SH.h_v, SH.d_v, dtype=torch.bfloat16, device=DEV)
        _step(dims, td, params, conv, ssm, out)
        res.append((out, ssm, conv))
    for x, y in zip(*res):
        assert torch.equal(x, y)


@pytest.mark.parametrize("out_dtype,use_slot,B,pinned", [(torch.float32, False, 6, True),
                                                         (torch.bfloat16, True, 6, True),
                                                         (torch.bfloat16, False, 70, True),
                                                         (torch.float32, True, 100, False),
                                                         (torch.bfloat16, False, 6, False)])
def test_decode_from_host_buffers_equals_device_step_bitwise(out_dtype, use_slot, B, pinned):
    # gdn_decode_step_host (host qkv/z/a/b/out) against gdn_decode_step on device
    # copies of the same tokens: 8 steps of B sequences (seed 86); with use_slot
    # the sequences live in slots B+1..2 of a (B+2)-slot pool.  Page-locked
    # buffers are read and written in place by the kernel, pageable ones go
    # through the staging copies.  The output starts as NaN on the host.
    S, n = 8, B + 2
    dims = dims_of(SH)
    params = to_dev(gi.make_params(SH, 86))
    st = gi.make_states(SH, n, 86, ssm_std=0.1 ** 0.5, conv_std=1.0)
    slot = torch.arange(B + 1, 1, -1, dtype=torch.int32, device=DEV) if use_slot else None
    conv_h, ssm_h = st["conv_state"].to(DEV), st["ssm_state"].to(DEV)
    conv_d, ssm_d = conv_h.clone(), ssm_h.clone()
    toks = _tokens(SH, S, B, 86)
    ws = torch.empty(gdn.gdn_decode_step_host_workspace_bytes(dims, B, out_dtype), dtype=torch.uint8,
                     device=DEV)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    # steps 4..7 through a prepared call on fixed pinned buffers refilled in place
    host_mem = (lambda t: t.pin_memory()) if pinned else (lambda t: t.clone())
    fixed = {k: host_mem(torch.empty(v[0].shape, dtype=v.dtype)) for k, v in toks.items()}
    out_fixed = host_mem(torch.empty(B, SH.h_v, SH.d_v, dtype=out_dtype))
    prepared = gdn.prepare_decode_step_host(dims, fixed["qkv"], fixed["z"], fixed["a"], fixed["b"],
                                            params["A_log"], params["dt_bias"], params["conv_w"],
                                            params["norm_w"], slot, n, conv_h, ssm_h, out_fixed, ws,
                                            device_status=status)
    for s in range(S):
        if s < 4:
            host = {k: host_mem(v[s].contiguous()) for k, v in toks.items()}
            out_h = host_mem(torch.full((B, SH.h_v, SH.d_v), float("nan"), dtype=out_dtype))
            gdn.gdn_decode_step_host(dims, host["qkv"], host["z"], host["a"], host["b"], params["A_log"],
                                     params["dt_bias"], params["conv_w"], params["norm_w"], slot, n,
                                     conv_h, ssm_h, out_h, ws, device_status=status)
        else:
            for k, v in toks.items():
                fixed[k].copy_(v[s])
            out_fixed.fill_(float("nan"))
            prepared()
            out_h = out_fixed
        out_d = torch.empty(B, SH.h_v, SH.d_v, dtype=out_dtype, device=DEV)
        _step(dims, {k: v[s].to(DEV) for k, v in toks.items()}, params, conv_d, ssm_d, out_d, slot=slot,
              n_slots=n)
        torch.cuda.synchronize()
        assert torch.equal(out_h, out_d.cpu()), f"step {s}"
    assert torch.equal(ssm_h, ssm_d) and torch.equal(conv_h, conv_d)
    assert gdn.gdn_read_device_status(status) == 0


def test_decode_from_host_buffers_flags_a_bad_slot():
    # entry 1's slot is out of range: skipped on the device (its host output
    # rows keep their NaN canary) and reported in the status word; the other
    # entries decode as the device step does
    B, n = 3, 4
    dims = dims_of(SH)
    params = to_dev(gi.make_params(SH, 87))
    st = gi.make_states(SH, n, 87, ssm_std=0.1 ** 0.5, conv_std=1.0)
    slot = torch.tensor([3, 9, 0], dtype=torch.int32, device=DEV)
    conv_h, ssm_h = st["conv_state"].to(DEV), st["ssm_state"].to(DEV)
    conv_d, ssm_d = conv_h.clone(), ssm_h.clone()
    tok = gi.make_tokens(SH, B, 87)
    host = {k: v.pin_memory() for k, v in tok.items()}
    out_h = torch.full((B, SH.h_v, SH.d_v), float("nan")).pin_memory()
    out_d = torch.full((B, SH.h_v, SH.d_v), float("nan"), device=DEV)
    ws = torch.empty(gdn.gdn_decode_step_host_workspace_bytes(dims, B, torch.float32), dtype=torch.uint8,
                     device=DEV)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    gdn.gdn_decode_step_host(dims, host["qkv"], host["z"], host["a"], host["b"], params["A_log"],
                             params["dt_bias"], params["conv_w"], params["norm_w"], slot, n, conv_h, ssm_h,
                             out_h, ws, device_status=status)
    _step(dims, to_dev(tok), params, conv_d, ssm_d, out_d, slot=slot, n_slots=n)
    torch.cuda.synchronize()
    assert gdn.gdn_read_device_status(status) == gdn.GDN_ERR_DEVICE_BOUNDS
    assert torch.isnan(out_h[1]).all()
    assert torch.equal(out_h[[0, 2]], out_d[[0, 2]].cpu())
    assert torch.equal(ssm_h, ssm_d) and torch.equal(conv_h, conv_d)
