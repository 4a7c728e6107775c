"""GPU parity of gdn_prefill against the fp64 oracle, through the C ABI.

Bar: max |gpu - oracle| / max |oracle| <= 1e-2 over the bf16 output and over
the fp32 final state (bf16 tensor-core operands, fp32 accumulation); the
conv state, a copy of raw inputs, must match exactly.
"""
import numpy as np
import pytest
import torch

import gated_deltanet_linear_06_gb300 as gdn
import gdn_inputs as gi
from gpu_util import DECODE_TOL, DEV, PREFILL_TOL, dims_of, oracle_layer, rel_err, to_dev

pytestmark = pytest.mark.gpu
SH = gi.LAYER


def _inputs(sh, lengths, seed, slow=False, ssm_std=0.0, conv_std=0.0, norm_w="ones"):
    T = sum(lengths)
    params = gi.make_params(sh, seed, norm_w=norm_w)
    tok = gi.make_tokens(sh, T, seed)
    if slow:
        gc = gi.gate_controlled(sh, T, seed)
        tok["a"], tok["b"] = gc["a"], gc["b"]
        params["A_log"], params["dt_bias"] = gc["A_log"], gc["dt_bias"]
    st = gi.make_states(sh, len(lengths), seed, ssm_std=ssm_std, conv_std=conv_std)
    return params, tok, st


def _run(sh, lengths, params, tok, st, out_fill=None):
    dims = dims_of(sh)
    N, T = len(lengths), sum(lengths)
    conv = st["conv_state"].clone().to(DEV)
    ssm = st["ssm_state"].clone().to(DEV)
    out = torch.empty(T, sh.h_v, sh.d_v, dtype=torch.bfloat16, device=DEV)
    if out_fill is not None:
        out.fill_(out_fill)
    ws = torch.empty(gdn.gdn_workspace_bytes(dims, N, T), dtype=torch.uint8, device=DEV)
    pd, td = to_dev(params), to_dev(tok)
    gdn.gdn_prefill(dims, td["qkv"], td["z"], td["a"], td["b"], pd["A_log"], pd["dt_bias"],
                    pd["conv_w"], pd["norm_w"], gi.cu_seqlens(lengths).to(DEV), conv, ssm, out, ws)
    status = gdn.gdn_read_device_status(ws)
    return out, conv, ssm, status


def _check(sh, lengths, params, tok, st, head_mask=None, tol=PREFILL_TOL):
    out, conv, ssm, status = _run(sh, lengths, params, tok, st)
    assert status == 0
    ref, ref_conv, ref_ssm = oracle_layer(sh, tok, params, gi.cu_seqlens(lengths),
                                          conv_state=st["conv_state"], ssm_state=st["ssm_state"],
                                          head_mask=head_mask)
    heads = slice(None) if head_mask is None else [i for i, m in enumerate(head_mask) if m]
    e_out = rel_err(out[:, heads], ref[:, heads])
    e_ssm = rel_err(ssm[:, heads], ref_ssm[:, heads])
    np.testing.assert_array_equal(conv.cpu().double().numpy(), ref_conv)
    assert e_out <= tol and e_ssm <= tol, (e_out, e_ssm)
    return e_out, e_ssm


@pytest.mark.parametrize("slow", [False, True])
def test_prefill_varlen_ragged_short_and_empty(slow):
    lengths = [70, 33, 1, 2, 128, 0, 64, 200]
    params, tok, st = _inputs(SH, lengths, 5, slow=slow, ssm_std=0.1 ** 0.5, conv_std=1.0,
                              norm_w="uniform")
    e = _check(SH, lengths, params, tok, st)
    print(f"rel err out {e[0]:.2e} state {e[1]:.2e}")


@pytest.mark.parametrize("slow", [False, True])
def test_prefill_segment_boundaries(slow):
    # sequences longer than one segment are scanned in parallel segments whose
    # start states are composed from per-segment transfer maps.  The lengths
    # straddle the segment length this call uses (exactly one segment, one and a
    # token, two and a ragged tail); the slow-decay variant makes the state carry
    # across every boundary
    T, n = 16384, 5
    L = gdn.gdn_prefill_segment_tokens(dims_of(SH), n, T)
    assert L >= 1024 and L % 64 == 0
    lengths = [L, L + 1, 2 * L + 67, 5]
    lengths.append(T - sum(lengths))
    assert lengths[-1] > 0
    params, tok, st = _inputs(SH, lengths, 12, slow=slow, ssm_std=0.1 ** 0.5, conv_std=1.0,
                              norm_w="uniform")
    e = _check(SH, lengths, params, tok, st)
    print(f"rel err out {e[0]:.2e} state {e[1]:.2e}")


def test_prefill_segments_carry_state_with_near_unit_decay():
    # with exp(g) in (0.999, 1) and small write gates the state a segment starts
    # from still matters a thousand tokens later, so a wrong transfer map or a
    # wrong composition of maps shows in the outputs and the final state
    lengths = [3000, 1500, 10]
    T = sum(lengths)
    params = gi.make_params(SH, 14, norm_w="uniform")
    tok = gi.make_tokens(SH, T, 14)
    gc = gi.gate_controlled(SH, T, 14, decay=(0.999, 1.0), beta=(0.0, 0.05))
    tok["a"], tok["b"] = gc["a"], gc["b"]
    params["A_log"], params["dt_bias"] = gc["A_log"], gc["dt_bias"]
    st = gi.make_states(SH, len(lengths), 14, ssm_std=1.0, conv_std=1.0)
    e = _check(SH, lengths, params, tok, st)
    print(f"rel err out {e[0]:.2e} state {e[1]:.2e}")


def test_prefill_segments_with_fast_and_slow_decay_heads():
    # value heads 0-15 decay fast (the default gate distribution: a segment's
    # total log-decay is far below -160, so the transfer scan starts near the
    # segment's end and the map is zero), heads 16-31 slowly (exp(g) in
    # (0.99, 1): the whole segment is scanned); one call, both kinds of head
    lengths = [6000, 37]
    T = sum(lengths)
    params, tok, st = _inputs(SH, lengths, 16, ssm_std=0.1 ** 0.5, conv_std=1.0, norm_w="uniform")
    gc = gi.gate_controlled(SH, T, 16, decay=(0.99, 1.0), beta=(0.0, 0.2))
    slow = slice(16, 32)
    tok["a"][:, slow], tok["b"][:, slow] = gc["a"][:, slow], gc["b"][:, slow]
    params["A_log"][slow], params["dt_bias"][slow] = gc["A_log"][slow], gc["dt_bias"][slow]
    e = _check(SH, lengths, params, tok, st)
    print(f"rel err out {e[0]:.2e} state {e[1]:.2e}")


def test_prefill_zero_write_no_decay_keeps_state_bitwise_across_segments():
    # beta = 0 and exp(g) = 1: every chunk and every segment's transfer map is
    # exactly the identity, so the state comes back bit for bit, whether or not
    # the sequence was split
    lengths = [2600, 40]
    params, tok, st = _inputs(SH, lengths, 15, ssm_std=0.3, conv_std=1.0)
    params["A_log"] = torch.full((SH.h_v,), -100.0)
    tok["b"] = torch.full_like(tok["b"], -100.0)
    out, conv, ssm, status = _run(SH, lengths, params, tok, st)
    assert status == 0
    assert torch.equal(ssm.cpu(), st["ssm_state"])
    ref, _, _ = oracle_layer(SH, tok, params, gi.cu_seqlens(lengths),
                             conv_state=st["conv_state"], ssm_state=st["ssm_state"])
    assert rel_err(out, ref) <= PREFILL_TOL


def test_prefill_many_sequences_unsegmented():
    # 20 sequences x 32 value heads fill the GPU, so no sequence is split, even
    # those longer than a segment; a mix of long, short and empty sequences
    lengths = [1500, 30, 0, 1100, 64, 65, 3, 700, 1030, 128] * 2
    assert gdn.gdn_prefill_segment_tokens(dims_of(SH), len(lengths), sum(lengths)) == 0
    params, tok, st = _inputs(SH, lengths, 13, slow=True, ssm_std=0.1 ** 0.5, conv_std=1.0)
    e = _check(SH, lengths, params, tok, st)
    print(f"rel err out {e[0]:.2e} state {e[1]:.2e}")


def test_prefill_single_sequence_4096():
    # T = 4096, zero initial state, seed 2
    params, tok, st = _inputs(SH, [4096], 2)
    e = _check(SH, [4096], params, tok, st)
    print(f"rel err out {e[0]:.2e} state {e[1]:.2e}")


def test_prefill_long_varlen_with_carried_segments():
    # packed {32768, 8192, 2048, 512, 131072 split into 4 x 32768 segments
    # carrying state}, seed 3.  Call 1 packs the four sequences and the first
    # segment; calls 2-4 continue the segmented sequence from its states.  The
    # outputs and the final states are compared with the oracle run on the
    # unsegmented sequences, on a sample of value heads.
    seg = 32768
    lengths = [32768, 8192, 2048, 512, 4 * seg]
    params, tok, st = _inputs(SH, lengths, 3)
    mask = [1 if h in (0, 13, 31) else 0 for h in range(SH.h_v)]
    heads = [0, 13, 31]
    ref, ref_conv, ref_ssm = oracle_layer(SH, tok, params, gi.cu_seqlens(lengths),
                                          conv_state=st["conv_state"], ssm_state=st["ssm_state"],
                                          head_mask=mask)
    T1 = sum(lengths[:4]) + seg
    first = {k: v[:T1] for k, v in tok.items()}
    out1, conv, ssm, status = _run(SH, lengths[:4] + [seg], params, first, st)
    assert status == 0
    outs = [out1[:, heads].float().cpu()]
    for k in range(1, 4):
        part = {kk: v[T1 + (k - 1) * seg:T1 + k * seg] for kk, v in tok.items()}
        sk = {"conv_state": conv[4:5].cpu(), "ssm_state": ssm[4:5].cpu()}
        o, c, s, status = _run(SH, [seg], params, part, sk)
        assert status == 0
        outs.append(o[:, heads].float().cpu())
        conv[4:5], ssm[4:5] = c, s
    got = torch.cat(outs)
    e_out = rel_err(got, ref[:, heads])
    e_ssm = rel_err(ssm[:, heads], ref_ssm[:, heads])
    np.testing.assert_array_equal(conv.cpu().double().numpy(), ref_conv)
    print(f"rel err out {e_out:.2e} state {e_ssm:.2e}")
    assert e_out <= PREFILL_TOL and e_ssm <= PREFILL_TOL


def test_prefill_then_decode_equals_longer_prefill():
    T = 77
    params, tok, st = _inputs(SH, [T + 1], 6, slow=True, ssm_std=0.3, conv_std=1.0)
    ref, ref_conv, ref_ssm = oracle_layer(SH, tok, params, gi.cu_seqlens([T + 1]),
                                          conv_state=st["conv_state"], ssm_state=st["ssm_state"])
    head = {k: v[:T] for k, v in tok.items()}
    out, conv, ssm, status = _run(SH, [T], params, head, st)
    assert status == 0
    last = to_dev({k: v[T:] for k, v in tok.items()})
    pd = to_dev(params)
    o1 = torch.empty(1, SH.h_v, SH.d_v, device=DEV)
    gdn.gdn_decode_step(dims_of(SH), last["qkv"], last["z"], last["a"], last["b"], pd["A_log"],
                        pd["dt_bias"], pd["conv_w"], pd["norm_w"], None, 1, conv, ssm, o1)
    assert rel_err(out, ref[:T]) <= PREFILL_TOL
    assert rel_err(o1, ref[T:]) <= PREFILL_TOL
    assert rel_err(ssm, ref_ssm) <= PREFILL_TOL
    np.testing.assert_array_equal(conv.cpu().double().numpy(), ref_conv)


@pytest.mark.parametrize("h_k,h_v", [(32, 32), (8, 32), (2, 4)])
def test_prefill_other_head_groupings(h_k, h_v):
    sh = gi.Shape(h_k=h_k, h_v=h_v)
    lengths = [100, 7, 64]
    params, tok, st = _inputs(sh, lengths, 7, ssm_std=0.3, conv_std=1.0, norm_w="uniform")
    _check(sh, lengths, params, tok, st)


@pytest.mark.parametrize("h_k,h_v", [(32, 32), (8, 32), (6, 12)])
def test_prefill_segmented_other_head_groupings(h_k, h_v):
    # a sequence longer than one segment with 1, 4 and 2 value heads per key
    # head: the prep pass's head groups, both transfer tracks and the combine
    # at groupings other than 2; 6 key heads do not split into the launcher's
    # four stream groups, so that call runs as one group
    sh = gi.Shape(h_k=h_k, h_v=h_v)
    lengths = [2100, 30]
    params, tok, st = _inputs(sh, lengths, 16, slow=True, ssm_std=0.3, conv_std=1.0, norm_w="uniform")
    e = _check(sh, lengths, params, tok, st)
    print(f"rel err out {e[0]:.2e} state {e[1]:.2e}")


def test_prefill_extreme_decay_stays_finite():
    # a = 30 gives g ~ -30 exp(A_log) per token: the cumulative decay of a
    # chunk is far below fp32's range, and every exponential must stay finite
    lengths = [130]
    params, tok, st = _inputs(SH, lengths, 8, ssm_std=0.3)
    tok["a"] = torch.full_like(tok["a"], 30.0)
    _check(SH, lengths, params, tok, st)


def test_prefill_bad_cu_seqlens_writes_nothing():
    lengths = [40, 24]
    params, tok, st = _inputs(SH, lengths, 9, ssm_std=0.3, conv_std=1.0)
    dims = dims_of(SH)
    conv, ssm = st["conv_state"].clone().to(DEV), st["ssm_state"].clone().to(DEV)
    out = torch.full((64, SH.h_v, SH.d_v), float("nan"), dtype=torch.bfloat16, device=DEV)
    ws = torch.empty(gdn.gdn_workspace_bytes(dims, 2, 64), dtype=torch.uint8, device=DEV)
    pd, td = to_dev(params), to_dev(tok)
    for bad in ([0, 50, 40], [0, 40, 65], [1, 40, 64]):
        gdn.gdn_prefill(dims, td["qkv"], td["z"], td["a"], td["b"], pd["A_log"], pd["dt_bias"],
                        pd["conv_w"], pd["norm_w"], torch.tensor(bad, dtype=torch.int32, device=DEV),
                        conv, ssm, out, ws)
        assert gdn.gdn_read_device_status(ws) == 6
        assert torch.isnan(out.float()).all()
        assert torch.equal(ssm.cpu(), st["ssm_state"]) and torch.equal(conv.cpu(), st["conv_state"])


def test_prefill_writes_every_output_and_is_deterministic():
    lengths = [65, 3, 190]
    params, tok, st = _inputs(SH, lengths, 10, ssm_std=0.3, conv_std=1.0)
    a = _run(SH, lengths, params, tok, st, out_fill=float("nan"))
    b = _run(SH, lengths, params, tok, st, out_fill=0.0)
    assert not torch.isnan(a[0].float()).any()
    for x, y in zip(a[:3], b[:3]):
        assert torch.equal(x, y)


def test_prefill_cuda_graph_replay_is_bitwise_eager():
    # a segmented call -- its head groups fork from the caller's stream to the
    # library's side streams and join back -- captured into a CUDA graph and
    # replayed twice gives the eager call's output and states bit for bit
    lengths = [2100, 30]
    params, tok, st = _inputs(SH, lengths, 18, ssm_std=0.3, conv_std=1.0)
    e_out, e_conv, e_ssm, status = _run(SH, lengths, params, tok, st)
    assert status == 0
    dims = dims_of(SH)
    T = sum(lengths)
    pd, td = to_dev(params), to_dev(tok)
    cu = gi.cu_seqlens(lengths).to(DEV)
    conv0, ssm0 = st["conv_state"].to(DEV), st["ssm_state"].to(DEV)
    conv, ssm = conv0.clone(), ssm0.clone()
    out = torch.empty(T, SH.h_v, SH.d_v, dtype=torch.bfloat16, device=DEV)
    ws = torch.empty(gdn.gdn_workspace_bytes(dims, len(lengths), T), dtype=torch.uint8, device=DEV)

    def call():
        gdn.gdn_prefill(dims, td["qkv"], td["z"], td["a"], td["b"], pd["A_log"], pd["dt_bias"],
                        pd["conv_w"], pd["norm_w"], cu, conv, ssm, out, ws)

    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):   # warm-up off the default stream, as capture wants
        call()
    torch.cuda.current_stream().wait_stream(side)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        call()
    for _ in range(2):
        conv.copy_(conv0)
        ssm.copy_(ssm0)
        out.fill_(float("nan"))
        graph.replay()
        torch.cuda.synchronize()
        assert gdn.gdn_read_device_status(ws) == 0
        assert torch.equal(out, e_out) and torch.equal(conv, e_conv) and torch.equal(ssm, e_ssm)
