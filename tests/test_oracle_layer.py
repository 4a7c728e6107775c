"""Whole-layer pins of the fp64 oracle: structure, state carry, head mapping.

The scalar and vector pieces are pinned in test_oracle_pins.py; these tests
pin how the layer wires them together (which channel block is q, k and v,
which key head a value head reads, how the conv and SSM states carry across
calls, how packed sequences stay independent).
"""
import math

import numpy as np
import pytest
import torch

import gdn_inputs as gi
import oracle

TOL = 1e-12
SMALL = gi.Shape(h_k=2, h_v=4, d_k=8, d_v=6)


def _inputs(shape, lengths, seed, dtype=torch.float32, slow=False, ssm_std=0.3,
            conv_std=1.0):
    T = sum(lengths)
    p = gi.make_params(shape, seed, dtype=dtype, norm_w="uniform")
    x = gi.make_tokens(shape, T, seed, dtype=dtype)
    st = gi.make_states(shape, len(lengths), seed, ssm_std=ssm_std, conv_std=conv_std)
    if slow:
        gc = gi.gate_controlled(shape, T, seed, dtype=dtype)
        x["a"], x["b"] = gc["a"], gc["b"]
        p["A_log"], p["dt_bias"] = gc["A_log"], gc["dt_bias"]
    return dict(h_k=shape.h_k, h_v=shape.h_v, d_k=shape.d_k, d_v=shape.d_v,
                conv_w_width=shape.conv_w, qkv=x["qkv"], z=x["z"], a=x["a"],
                b=x["b"], A_log=p["A_log"], dt_bias=p["dt_bias"],
                conv_w=p["conv_w"], norm_w=p["norm_w"],
                cu_seqlens=gi.cu_seqlens(lengths), conv_state=st["conv_state"],
                ssm_state=st["ssm_state"])


def _close(a, b, tol=TOL):
    np.testing.assert_allclose(a, b, rtol=0, atol=tol * max(1.0, float(np.nanmax(np.abs(b)))))


@pytest.mark.parametrize("slow", [False, True])
def test_tiny_fp32_sequential_equals_chunked16(slow):
    # the tiny fp32 layer: 1 sequence, T = 64, 2 key / 2 value heads, d = 32
    kw = _inputs(gi.TINY, [64], seed=0, slow=slow, ssm_std=0.0, conv_std=0.0)
    o1, c1, s1 = oracle.layer(**kw)
    o2, c2, s2 = oracle.layer(**kw, chunk=16)
    _close(o2, o1)
    _close(s2, s1)
    np.testing.assert_array_equal(c1, c2)


@pytest.mark.parametrize("C", [3, 64])
def test_layer_chunked_equals_sequential_varlen(C):
    kw = _inputs(SMALL, [70, 0, 1, 9, 130], seed=5, slow=True)
    o1, _, s1 = oracle.layer(**kw)
    o2, _, s2 = oracle.layer(**kw, chunk=C)
    _close(o2, o1)
    _close(s2, s1)


def test_prefill_then_decode_equals_longer_prefill():
    T = 23
    kw = _inputs(SMALL, [T + 1], seed=6, slow=True)
    out_full, cs_full, ss_full = oracle.layer(**kw)
    head = dict(kw, qkv=kw["qkv"][:T], z=kw["z"][:T], a=kw["a"][:T], b=kw["b"][:T],
                cu_seqlens=gi.cu_seqlens([T]))
    out_h, cs_h, ss_h = oracle.layer(**head)
    tail = dict(kw, qkv=kw["qkv"][T:], z=kw["z"][T:], a=kw["a"][T:], b=kw["b"][T:],
                cu_seqlens=gi.cu_seqlens([1]), conv_state=cs_h, ssm_state=ss_h)
    out_t, cs_t, ss_t = oracle.layer(**tail)
    _close(out_h, out_full[:T])
    _close(out_t, out_full[T:])
    _close(ss_t, ss_full)
    np.testing.assert_array_equal(cs_t, cs_full)


def test_segmented_equals_unsegmented():
    segs = [5, 1, 2, 31, 64, 1]
    T = sum(segs)
    kw = _inputs(SMALL, [T], seed=7, slow=True)
    out_full, cs_full, ss_full = oracle.layer(**kw)
    cs, ss = kw["conv_state"], kw["ssm_state"]
    outs = []
    t = 0
    for n in segs:
        part = dict(kw, qkv=kw["qkv"][t:t + n], z=kw["z"][t:t + n], a=kw["a"][t:t + n],
                    b=kw["b"][t:t + n], cu_seqlens=gi.cu_seqlens([n]),
                    conv_state=cs, ssm_state=ss)
        o, cs, ss = oracle.layer(**part, chunk=4)
        outs.append(o)
        t += n
    _close(np.concatenate(outs), out_full)
    _close(ss, ss_full)
    np.testing.assert_array_equal(cs, cs_full)


def test_packed_sequences_are_independent_and_permute():
    lengths = [7, 0, 3, 12]
    kw = _inputs(SMALL, lengths, seed=8)
    out, cs, ss = oracle.layer(**kw)
    cu = np.cumsum([0] + lengths)
    perm = [3, 1, 0, 2]
    rows = np.concatenate([np.arange(cu[i], cu[i + 1]) for i in perm]).astype(np.int64)
    pk = dict(kw, qkv=kw["qkv"][rows], z=kw["z"][rows], a=kw["a"][rows], b=kw["b"][rows],
              cu_seqlens=gi.cu_seqlens([lengths[i] for i in perm]),
              conv_state=kw["conv_state"][perm], ssm_state=kw["ssm_state"][perm])
    out_p, cs_p, ss_p = oracle.layer(**pk)
    np.testing.assert_array_equal(out_p, out[rows])
    np.testing.assert_array_equal(cs_p, cs[perm])
    np.testing.assert_array_equal(ss_p, ss[perm])
    # the empty sequence keeps both of its states
    np.testing.assert_array_equal(cs[1], kw["conv_state"][1].double().numpy())
    np.testing.assert_array_equal(ss[1], kw["ssm_state"][1].double().numpy())


def test_gqa_equals_duplicated_key_heads():
    # G = 2 (value head h reads key head h // 2) equals G = 1 with each key
    # head's q and k channels copied next to itself
    sh = SMALL
    kw = _inputs(sh, [17, 4], seed=9)
    out, cs, ss = oracle.layer(**kw)
    dup = gi.Shape(h_k=sh.h_v, h_v=sh.h_v, d_k=sh.d_k, d_v=sh.d_v)
    q = kw["qkv"][:, :sh.cq].reshape(-1, sh.h_k, sh.d_k)
    k = kw["qkv"][:, sh.cq:2 * sh.cq].reshape(-1, sh.h_k, sh.d_k)
    v = kw["qkv"][:, 2 * sh.cq:]
    qd = q.repeat_interleave(2, dim=1).reshape(q.shape[0], -1)
    kd = k.repeat_interleave(2, dim=1).reshape(k.shape[0], -1)

    def dup_ch(t):                 # [..., cc] -> [..., cc of the duplicated shape]
        qq = t[..., :sh.cq].unflatten(-1, (sh.h_k, sh.d_k)).repeat_interleave(2, dim=-2)
        kk = t[..., sh.cq:2 * sh.cq].unflatten(-1, (sh.h_k, sh.d_k)).repeat_interleave(2, dim=-2)
        return torch.cat([qq.flatten(-2), kk.flatten(-2), t[..., 2 * sh.cq:]], dim=-1)

    kd_all = dict(kw, h_k=dup.h_k, qkv=torch.cat([qd, kd, v], dim=1),
                  conv_w=dup_ch(kw["conv_w"].T).T.contiguous(),
                  conv_state=dup_ch(kw["conv_state"]))
    out_d, cs_d, ss_d = oracle.layer(**kd_all)
    _close(out_d, out)
    _close(ss_d, ss)


def test_value_head_reads_key_head_floor_h_over_G():
    # zero key head 0's q conv taps: q^ = 0 there, so exactly value heads 0
    # and 1 (floor(h / 2) = 0) output zero; heads 2 and 3 do not
    kw = _inputs(SMALL, [9], seed=10)
    w = kw["conv_w"].clone()
    w[:SMALL.d_k] = 0.0
    out, _, _ = oracle.layer(**dict(kw, conv_w=w))
    np.testing.assert_array_equal(out[:, :2], 0.0)
    assert np.all(np.abs(out[:, 2:]).max(axis=(0, 2)) > 1e-3)


def test_zero_key_block_leaves_pure_decay():
    # with k^ = 0 the state only decays: o_t = exp(gamma_t) S0 q^_t.  Use the
    # identity conv tap (w = [0, 0, 0, 1]) so q = silu(x_q).
    sh = SMALL
    kw = _inputs(sh, [6], seed=11)
    w = torch.zeros(sh.cc, 4)
    w[:, 3] = 1.0
    w[sh.cq:2 * sh.cq] = 0.0
    # a large RMS epsilon keeps the scale of o (and so the 1/sqrt(d_k) on q)
    # visible in the output
    kw = dict(kw, conv_w=w, rms_eps=0.5)
    out, _, ss = oracle.layer(**kw)
    x = kw["qkv"].double().numpy()
    A_log = kw["A_log"].double().numpy()
    a = kw["a"].double().numpy()
    S0 = kw["ssm_state"][0].double().numpy()
    gam = np.zeros(sh.h_v)
    zz = kw["z"].double().numpy()
    nw = kw["norm_w"].double().numpy()
    for t in range(6):
        for h in range(sh.h_v):
            kh = h // 2
            qr = x[t, kh * sh.d_k:(kh + 1) * sh.d_k]
            qs = qr / (1 + np.exp(-qr))
            qh = qs / math.sqrt(qs @ qs + 1e-6) / math.sqrt(sh.d_k)
            gam[h] += -math.exp(A_log[h]) * math.log1p(math.exp(a[t, h]))
            o = math.exp(gam[h]) * (S0[h] @ qh)
            r = o / math.sqrt(np.mean(o * o) + 0.5)
            exp_out = r * nw * zz[t, h] / (1 + np.exp(-zz[t, h]))
            np.testing.assert_allclose(out[t, h], exp_out, rtol=0, atol=1e-12)
    for h in range(sh.h_v):
        np.testing.assert_allclose(ss[0, h], math.exp(gam[h]) * S0[h], rtol=1e-12, atol=0)


def test_write_gate_one_overwrites_key_direction():
    # beta = 1 (b = 40 rounds sigmoid to 1.0) with the identity conv tap:
    # after one token S k^ = v exactly, where k^ = silu(x_k) / |silu(x_k)| is
    # a unit vector and v = silu(x_v)
    sh = SMALL
    kw = _inputs(sh, [1], seed=17)
    w = torch.zeros(sh.cc, 4)
    w[:, 3] = 1.0
    kw = dict(kw, conv_w=w, l2_eps=0.0, b=torch.full((1, sh.h_v), 40.0))
    _, _, ss = oracle.layer(**kw)
    x = kw["qkv"][0].double().numpy()
    y = x / (1 + np.exp(-x))
    for h in range(sh.h_v):
        kh = h // 2
        k = y[sh.cq + kh * sh.d_k:sh.cq + (kh + 1) * sh.d_k]
        k = k / math.sqrt(k @ k)
        v = y[2 * sh.cq + h * sh.d_v:2 * sh.cq + (h + 1) * sh.d_v]
        np.testing.assert_allclose(ss[0, h] @ k, v, rtol=0, atol=1e-12)


def test_first_token_from_zero_state_closed_form():
    # S0 = 0, one token: o = beta (k^.q^) v, so after the RMSNorm (eps = 0)
    # out = sign(k^.q^) v / rms(v) * w * silu(z), independent of beta and g
    sh = SMALL
    kw = _inputs(sh, [1], seed=12, ssm_std=0.0)
    w = torch.zeros(sh.cc, 4)
    w[:, 3] = 1.0
    kw = dict(kw, conv_w=w, rms_eps=0.0, l2_eps=0.0)
    out, _, _ = oracle.layer(**kw)
    x = kw["qkv"][0].double().numpy()
    y = x / (1 + np.exp(-x))
    zz = kw["z"][0].double().numpy()
    nw = kw["norm_w"].double().numpy()
    for h in range(sh.h_v):
        kh = h // 2
        qk = y[kh * sh.d_k:(kh + 1) * sh.d_k] @ y[sh.cq + kh * sh.d_k:sh.cq + (kh + 1) * sh.d_k]
        v = y[2 * sh.cq + h * sh.d_v:2 * sh.cq + (h + 1) * sh.d_v]
        exp_out = np.sign(qk) * v / math.sqrt(np.mean(v * v)) * nw * zz[h] / (1 + np.exp(-zz[h]))
        np.testing.assert_allclose(out[0, h], exp_out, rtol=0, atol=1e-12)


def test_zero_gate_input_zeroes_only_that_head():
    kw = _inputs(SMALL, [5], seed=13)
    z = kw["z"].clone()
    z[:, 1] = 0.0
    out, _, _ = oracle.layer(**dict(kw, z=z))
    np.testing.assert_array_equal(out[:, 1], 0.0)
    assert np.abs(out[:, [0, 2, 3]]).min(axis=(0, 2)).max() >= 0.0
    assert np.all(np.abs(out[:, [0, 2, 3]]).max(axis=(0, 2)) > 1e-3)


def test_head_mask_samples_the_same_values():
    kw = _inputs(SMALL, [11, 3], seed=14)
    out, _, ss = oracle.layer(**kw)
    mask = [0, 1, 0, 1]
    out_m, _, ss_m = oracle.layer(**kw, head_mask=mask)
    np.testing.assert_array_equal(out_m[:, [1, 3]], out[:, [1, 3]])
    np.testing.assert_array_equal(ss_m[:, [1, 3]], ss[:, [1, 3]])
    assert np.all(np.isnan(out_m[:, [0, 2]]))
    np.testing.assert_array_equal(ss_m[:, [0, 2]], kw["ssm_state"][:, [0, 2]].double().numpy())


def test_threads_do_not_change_results():
    kw = _inputs(SMALL, [19, 2, 40], seed=15)
    o1, c1, s1 = oracle.layer(**kw, n_threads=1)
    o2, c2, s2 = oracle.layer(**kw, n_threads=4)
    np.testing.assert_array_equal(o1, o2)
    np.testing.assert_array_equal(s1, s2)
    np.testing.assert_array_equal(c1, c2)


def test_bad_cu_seqlens_rejected():
    kw = _inputs(SMALL, [4, 4], seed=16)
    with pytest.raises(ValueError):
        oracle.layer(**dict(kw, cu_seqlens=np.array([0, 5, 3])))
