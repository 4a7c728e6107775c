"""GPU checks of the state pool primitives gdn_state_copy and gdn_state_reset, through the C ABI.

Bars: copies are bit-exact; a sequence continued from a restored snapshot
(prefill of its own tail, then decode steps) is bit-identical to the same
sequence continued without the snapshot; bad slot indices are skipped and
reported through the device status word.
"""
import pytest
import torch

import gated_deltanet_linear_06_gb300 as gdn
import gdn_inputs as gi
from gpu_util import DEV, dims_of, to_dev

pytestmark = pytest.mark.gpu
SH = gi.LAYER


def _pool(n, seed, fill=None):
    if fill is not None:
        conv = torch.full((n, SH.conv_w - 1, SH.cc), fill, device=DEV)
        ssm = torch.full((n, SH.h_v, SH.d_v, SH.d_k), fill, device=DEV)
        return conv, ssm
    st = gi.make_states(SH, n, seed, ssm_std=0.3, conv_std=1.0)
    return st["conv_state"].to(DEV), st["ssm_state"].to(DEV)


def _idx(v):
    return torch.tensor(v, dtype=torch.int32, device=DEV)


def test_state_copy_is_exact_and_touches_only_its_slots():
    # pool of 9 random states (seed 71) -> bank of 5 NaN-filled slots
    dims = dims_of(SH)
    conv, ssm = _pool(9, 71)
    bconv, bssm = _pool(5, 0, fill=float("nan"))
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    gdn.gdn_state_copy(dims, conv, ssm, bconv, bssm, src_slot=_idx([7, 2, 5]),
                       dst_slot=_idx([4, 0, 2]), device_status=status)
    assert gdn.gdn_read_device_status(status) == 0
    for s, d in ((7, 4), (2, 0), (5, 2)):
        assert torch.equal(bconv[d], conv[s]) and torch.equal(bssm[d], ssm[s])
    assert torch.isnan(bssm[[1, 3]]).all() and torch.isnan(bconv[[1, 3]]).all()
    # dense form: slot i -> slot i for the first n
    d2c, d2s = _pool(3, 0, fill=-1.0)
    gdn.gdn_state_copy(dims, conv, ssm, d2c, d2s, n=3)
    assert torch.equal(d2c, conv[:3]) and torch.equal(d2s, ssm[:3])


def test_state_copy_and_reset_flag_bad_slots():
    dims = dims_of(SH)
    conv, ssm = _pool(4, 72)
    bconv, bssm = _pool(3, 0, fill=2.0)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    gdn.gdn_state_copy(dims, conv, ssm, bconv, bssm, src_slot=_idx([1, 4, 3]),
                       dst_slot=_idx([0, 1, 3]), device_status=status)
    assert gdn.gdn_read_device_status(status) == 6
    assert torch.equal(bssm[0], ssm[1]) and torch.equal(bconv[0], conv[1])
    assert (bssm[[1, 2]] == 2.0).all() and (bconv[[1, 2]] == 2.0).all()   # skipped pairs
    status.zero_()
    keep_c, keep_s = conv.clone(), ssm.clone()
    gdn.gdn_state_reset(dims, conv, ssm, slot=_idx([2, -1, 0]), device_status=status)
    assert gdn.gdn_read_device_status(status) == 6
    assert (ssm[[0, 2]] == 0).all() and (conv[[0, 2]] == 0).all()
    assert torch.equal(ssm[[1, 3]], keep_s[[1, 3]]) and torch.equal(conv[[1, 3]], keep_c[[1, 3]])


def test_state_reset_equals_a_fresh_zero_state():
    dims = dims_of(SH)
    conv, ssm = _pool(3, 73)
    gdn.gdn_state_reset(dims, conv, ssm)
    assert (conv == 0).all() and (ssm == 0).all()


def test_restore_and_continue_is_bitwise_the_uninterrupted_run():
    # A 1,100-token prefix (seed 74) is prefilled from zero states and
    # snapshotted into bank slot 3.  Run A continues directly: a 300-token tail
    # (prefill), then 4 decode steps.  Run B restores the snapshot into another
    # state pair and feeds the same tail and steps.  Every output and the final
    # states must agree bit for bit.  Then three forks restored from the same
    # snapshot into slots of one decode pool continue with different tokens; the
    # fork fed run A's tokens matches run A bit for bit.
    dims = dims_of(SH)
    params = to_dev(gi.make_params(SH, 74))
    P, T = 1100, 300
    tok = to_dev(gi.make_tokens(SH, P + T, 74))
    steps = 4
    dec = gi.make_tokens(SH, steps * 3, 75)
    dec = to_dev({k: v.reshape(steps, 3, *v.shape[1:]) for k, v in dec.items()})

    def prefill(conv, ssm, lo, hi):
        n = hi - lo
        out = torch.empty(n, SH.h_v, SH.d_v, dtype=torch.bfloat16, device=DEV)
        ws = torch.empty(gdn.gdn_workspace_bytes(dims, 1, n), dtype=torch.uint8, device=DEV)
        gdn.gdn_prefill(dims, tok["qkv"][lo:hi], tok["z"][lo:hi], tok["a"][lo:hi],
                        tok["b"][lo:hi], params["A_log"], params["dt_bias"], params["conv_w"],
                        params["norm_w"], gi.cu_seqlens([n]).to(DEV), conv, ssm, out, ws)
        assert gdn.gdn_read_device_status(ws) == 0
        return out

    def decode(conv, ssm, t, col, slot=None, n_slots=None):
        B = 1 if slot is None else slot.numel()
        cols = [col] if slot is None else col
        out = torch.empty(B, SH.h_v, SH.d_v, device=DEV)
        gdn.gdn_decode_step(dims, *(dec[k][t, cols].contiguous() for k in ("qkv", "z", "a", "b")),
                            params["A_log"], params["dt_bias"], params["conv_w"], params["norm_w"],
                            slot, n_slots if n_slots is not None else conv.shape[0], conv, ssm, out)
        return out

    conv_a, ssm_a = _pool(1, 0, fill=0.0)
    prefill(conv_a, ssm_a, 0, P)
    bank_c, bank_s = _pool(4, 0, fill=float("nan"))
    gdn.gdn_state_copy(dims, conv_a, ssm_a, bank_c, bank_s, dst_slot=_idx([3]))
    out_a = prefill(conv_a, ssm_a, P, P + T)
    dec_a = [decode(conv_a, ssm_a, t, 0) for t in range(steps)]

    conv_b, ssm_b = _pool(1, 0, fill=5.0)
    gdn.gdn_state_copy(dims, bank_c, bank_s, conv_b, ssm_b, src_slot=_idx([3]))
    out_b = prefill(conv_b, ssm_b, P, P + T)
    dec_b = [decode(conv_b, ssm_b, t, 0) for t in range(steps)]
    assert torch.equal(out_a, out_b)
    for x, y in zip(dec_a, dec_b):
        assert torch.equal(x, y)
    assert torch.equal(ssm_a, ssm_b) and torch.equal(conv_a, conv_b)

    # forks: the prefix snapshot restored into slots 5, 1, 6 of a 7-slot pool,
    # which then decode 4 steps straight after the prefix, batched
    pool_c, pool_s = _pool(7, 76)
    slots = _idx([5, 1, 6])
    gdn.gdn_state_copy(dims, bank_c, bank_s, pool_c, pool_s, src_slot=_idx([3, 3, 3]),
                       dst_slot=slots)
    conv_c, ssm_c = _pool(1, 0, fill=0.0)
    gdn.gdn_state_copy(dims, bank_c, bank_s, conv_c, ssm_c, src_slot=_idx([3]))
    for t in range(steps):
        o3 = decode(pool_c, pool_s, t, [0, 1, 2], slot=slots, n_slots=7)
        o1 = decode(conv_c, ssm_c, t, 1)
        assert torch.equal(o3[1:2], o1)
    assert torch.equal(pool_s[1], ssm_c[0]) and torch.equal(pool_c[1], conv_c[0])
    assert not torch.equal(pool_s[5], pool_s[1])       # the forks diverged
