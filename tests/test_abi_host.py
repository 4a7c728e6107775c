"""Host-side checks of the C ABI: the library loads, exports what the header
declares, and rejects bad arguments before it touches a device.

No call here reaches the GPU: every call either returns from host-side
validation or launches nothing (empty batch), so these run without a device.
"""
import ctypes
import os
import re
import subprocess

import numpy as np
import pytest
import torch

import gated_deltanet_linear_06_gb300 as gdn
from gated_deltanet_linear_06_gb300 import build as gbuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "gdn.h")
FAKE = 0x10000          # a 16-byte-aligned address that is never dereferenced on this path


@pytest.fixture(scope="module")
def L():
    gbuild.build()
    return gdn.lib()


def _declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(gdn_[a-z_]+)\s*\(", text)))


def test_header_declares_the_entry_points():
    names = _declared_functions()
    for want in ("gdn_prefill", "gdn_decode_step", "gdn_workspace_bytes", "gdn_state_bytes",
                 "gdn_read_device_status", "gdn_status_string", "gdn_version",
                 "gdn_decode_multi", "gdn_prefill_noalloc", "gdn_prefill_segment_tokens",
                 "gdn_state_copy", "gdn_state_reset", "gdn_decode_graph_create",
                 "gdn_decode_graph_launch", "gdn_decode_graph_destroy", "gdn_prefill_host",
                 "gdn_prefill_host_workspace_bytes", "gdn_prefill_host_segments",
                 "gdn_prefill_segment_tokens_for", "gdn_selftest_wait_timeout",
                 "gdn_in_proj", "gdn_out_proj", "gdn_decode_step_host",
                 "gdn_decode_step_host_workspace_bytes"):
        assert want in names


def test_library_exports_every_declared_symbol(L):
    for name in _declared_functions():
        assert hasattr(L, name), name
    out = subprocess.run(["nm", "-D", "--defined-only", gdn.LIB_PATH], capture_output=True,
                         text=True, check=True).stdout
    exported = set(re.findall(r"\bT (gdn_[a-z_]+)\b", out))
    assert set(_declared_functions()) <= exported


def test_version_and_status_strings(L):
    assert gdn.gdn_version() >= 200
    for code in range(7):
        s = gdn.gdn_status_string(code)
        assert s.startswith(gdn.STATUS_NAMES[code])
    assert "unknown" in gdn.gdn_status_string(99)


def test_state_bytes_matches_the_pages_state_size(L):
    # 32 value heads x 128 x 128 fp32 = 2 MiB of SSM state per layer; over
    # 30 Gated DeltaNet layers that is the ~60 MiB per sequence the llmxabe
    # README states.  The conv state adds 3 rows of 8192 fp32 channels.
    d = gdn.make_dims()
    assert gdn.gdn_state_bytes(d) == 2 * 2**20 + 3 * 8192 * 4
    assert 30 * 32 * 128 * 128 * 4 == 60 * 2**20
    assert gdn.gdn_state_bytes(gdn.make_dims(h_k=0)) == 0


def test_prefill_segment_tokens_rejects_bad_arguments(L):
    # argument checks come before any device query, so they hold without a GPU
    assert gdn.gdn_prefill_segment_tokens(gdn.make_dims(d_k=64), 1, 4096) == -1
    assert gdn.gdn_prefill_segment_tokens(gdn.make_dims(), -1, 4096) == -1
    assert gdn.gdn_prefill_segment_tokens(gdn.make_dims(), 1, -5) == -1


def test_workspace_bytes(L):
    d = gdn.make_dims()
    assert gdn.gdn_workspace_bytes(d, 1, 4096) >= 256
    assert gdn.gdn_workspace_bytes(d, -1, 4096) == 0
    assert gdn.gdn_workspace_bytes(gdn.make_dims(d_k=64), 1, 64) == 0


def _decode(L, dims, **kw):
    args = dict(qkv=FAKE, z=FAKE, a=FAKE, b=FAKE, A_log=FAKE, dt_bias=FAKE, conv_w=FAKE,
                norm_w=FAKE, slot=None, n_slots=4, batch=4, conv_state=FAKE, ssm_state=FAKE,
                out=FAKE, out_dtype=0, status=None, stream=None)
    args.update(kw)
    return L.gdn_decode_step(ctypes.byref(dims) if dims is not None else None, args["qkv"],
                             args["z"], args["a"], args["b"], args["A_log"], args["dt_bias"],
                             args["conv_w"], args["norm_w"], args["slot"], args["n_slots"],
                             args["batch"], args["conv_state"], args["ssm_state"], args["out"],
                             args["out_dtype"], args["status"], args["stream"])


def _decode_host(L, dims, **kw):
    args = dict(qkv=FAKE, z=FAKE, a=FAKE, b=FAKE, A_log=FAKE, dt_bias=FAKE, conv_w=FAKE,
                norm_w=FAKE, slot=None, n_slots=4, batch=4, conv_state=FAKE, ssm_state=FAKE,
                out=FAKE, out_dtype=0, status=None, ws=0x100000, ws_bytes=1 << 40, stream=None)
    args.update(kw)
    return L.gdn_decode_step_host(ctypes.byref(dims) if dims is not None else None, args["qkv"],
                                  args["z"], args["a"], args["b"], args["A_log"], args["dt_bias"],
                                  args["conv_w"], args["norm_w"], args["slot"], args["n_slots"],
                                  args["batch"], args["conv_state"], args["ssm_state"], args["out"],
                                  args["out_dtype"], args["status"], args["ws"], args["ws_bytes"],
                                  args["stream"])


def _prefill(L, dims, **kw):
    args = dict(qkv=FAKE, z=FAKE, a=FAKE, b=FAKE, A_log=FAKE, dt_bias=FAKE, conv_w=FAKE,
                norm_w=FAKE, cu=FAKE, n_seqs=2, T=100, conv_state=FAKE, ssm_state=FAKE,
                out=FAKE, ws=0x100000, ws_bytes=1 << 40, stream=None)
    args.update(kw)
    return L.gdn_prefill(ctypes.byref(dims) if dims is not None else None, args["qkv"],
                         args["z"], args["a"], args["b"], args["A_log"], args["dt_bias"],
                         args["conv_w"], args["norm_w"], args["cu"], args["n_seqs"], args["T"],
                         args["conv_state"], args["ssm_state"], args["out"], args["ws"],
                         args["ws_bytes"], args["stream"])


OK, INVALID, UNSUP, WS = 0, 1, 2, 3


def test_decode_rejects_bad_dims(L):
    assert _decode(L, None) == INVALID
    assert _decode(L, gdn.make_dims(h_k=3, h_v=32)) == INVALID        # h_v % h_k
    assert _decode(L, gdn.make_dims(h_k=0)) == INVALID
    assert _decode(L, gdn.make_dims(l2_eps=-1.0)) == INVALID
    assert _decode(L, gdn.make_dims(l2_eps=float("nan"))) == INVALID
    assert _decode(L, gdn.make_dims(d_k=64, d_v=64)) == UNSUP
    assert _decode(L, gdn.make_dims(conv_w=3)) == UNSUP
    assert _decode(L, gdn.make_dims(h_k=4, h_v=32)) == UNSUP           # G = 8
    assert _decode(L, gdn.make_dims(h_k=128, h_v=128)) == UNSUP        # h_k > 64


def test_decode_host_workspace_and_rejections(L):
    # staging for qkv, z, a, b and the output, each 256-byte aligned; every
    # rejection below returns before anything is enqueued (no GPU needed)
    d = gdn.make_dims()
    B = 5
    cc, zv = 2 * 16 * 128 + 32 * 128, 32 * 128
    r = lambda x: (x + 255) // 256 * 256
    want = r(B * cc * 2) + r(B * zv * 2) + 2 * r(B * 32 * 2)
    assert L.gdn_decode_step_host_workspace_bytes(ctypes.byref(d), B, 0) == want + r(B * zv * 2)
    assert L.gdn_decode_step_host_workspace_bytes(ctypes.byref(d), B, 1) == want + r(B * zv * 4)
    assert L.gdn_decode_step_host_workspace_bytes(ctypes.byref(d), -1, 0) == 0
    assert L.gdn_decode_step_host_workspace_bytes(ctypes.byref(d), B, 2) == 0
    assert L.gdn_decode_step_host_workspace_bytes(ctypes.byref(gdn.make_dims(d_k=64, d_v=64)), B, 0) == 0
    assert _decode_host(L, None) == INVALID
    assert _decode_host(L, gdn.make_dims(d_k=64, d_v=64)) == UNSUP
    assert _decode_host(L, d, out_dtype=2) == INVALID
    assert _decode_host(L, d, batch=-1) == INVALID
    assert _decode_host(L, d, batch=0, qkv=None) == OK                  # nothing to do
    for host in ("qkv", "z", "a", "b", "out"):
        assert _decode_host(L, d, **{host: None}) == INVALID
    assert _decode_host(L, d, ws=None) == WS
    assert _decode_host(L, d, ws=0x100010) == WS                        # not 256-byte aligned
    need = L.gdn_decode_step_host_workspace_bytes(ctypes.byref(d), 4, 0)
    assert _decode_host(L, d, ws_bytes=need - 1) == WS
    # the device arguments are checked as gdn_decode_step checks them
    assert _decode_host(L, d, ws_bytes=need, A_log=None) == INVALID
    assert _decode_host(L, d, ws_bytes=need, ssm_state=FAKE + 4) == INVALID
    assert _decode_host(L, d, ws_bytes=need, n_slots=3) == INVALID     # fewer states than entries
    assert _decode_host(L, d, ws_bytes=need, slot=FAKE + 8) == INVALID
    assert _decode_host(L, d, ws_bytes=need, status=FAKE + 2) == INVALID


def test_decode_rejects_bad_pointers_and_sizes(L):
    d = gdn.make_dims()
    assert _decode(L, d, qkv=None) == INVALID
    assert _decode(L, d, ssm_state=FAKE + 4) == INVALID               # misaligned
    assert _decode(L, d, out=FAKE + 8) == INVALID
    assert _decode(L, d, slot=FAKE + 4) == INVALID
    assert _decode(L, d, status=FAKE + 2) == INVALID
    assert _decode(L, d, batch=-1) == INVALID
    assert _decode(L, d, n_slots=3) == INVALID                         # fewer states than batch
    assert _decode(L, d, out_dtype=7) == INVALID
    assert _decode(L, d, batch=0) == OK                                # nothing to launch


def _decode_multi(L, dims, **kw):
    args = dict(qkv=FAKE, z=FAKE, a=FAKE, b=FAKE, A_log=FAKE, dt_bias=FAKE, conv_w=FAKE,
                norm_w=FAKE, slot=None, n_slots=4, batch=4, steps=4, conv_state=FAKE,
                ssm_state=FAKE, out=FAKE, out_dtype=0, ssm_trace=None, conv_trace=None,
                status=None, stream=None)
    args.update(kw)
    return L.gdn_decode_multi(ctypes.byref(dims) if dims is not None else None, args["qkv"],
                              args["z"], args["a"], args["b"], args["A_log"], args["dt_bias"],
                              args["conv_w"], args["norm_w"], args["slot"], args["n_slots"],
                              args["batch"], args["steps"], args["conv_state"],
                              args["ssm_state"], args["out"], args["out_dtype"],
                              args["ssm_trace"], args["conv_trace"], args["status"],
                              args["stream"])


def test_decode_multi_rejects_bad_arguments(L):
    d = gdn.make_dims()
    assert gdn.GDN_DECODE_MAX_STEPS == 8
    assert _decode_multi(L, None) == INVALID
    assert _decode_multi(L, gdn.make_dims(h_k=3, h_v=32)) == INVALID
    assert _decode_multi(L, gdn.make_dims(d_k=64, d_v=64)) == UNSUP
    assert _decode_multi(L, gdn.make_dims(h_k=4, h_v=32)) == UNSUP     # G = 8
    assert _decode_multi(L, d, steps=0) == INVALID
    assert _decode_multi(L, d, steps=9) == INVALID                     # above the limit
    assert _decode_multi(L, d, steps=-3) == INVALID
    assert _decode_multi(L, d, qkv=None) == INVALID
    assert _decode_multi(L, d, ssm_state=FAKE + 4) == INVALID
    assert _decode_multi(L, d, ssm_trace=FAKE + 8) == INVALID          # misaligned trace
    assert _decode_multi(L, d, conv_trace=FAKE + 4) == INVALID
    assert _decode_multi(L, d, slot=FAKE + 4) == INVALID
    assert _decode_multi(L, d, status=FAKE + 2) == INVALID
    assert _decode_multi(L, d, batch=-1) == INVALID
    assert _decode_multi(L, d, n_slots=3) == INVALID
    assert _decode_multi(L, d, out_dtype=5) == INVALID
    assert _decode_multi(L, d, batch=0) == OK
    assert _decode_multi(L, d, batch=0, steps=8) == OK


def _copy(L, dims, **kw):
    args = dict(sc=FAKE, ss=FAKE, ns=4, si=None, dc=FAKE, ds=FAKE, nd=4, di=None, n=4,
                status=None, stream=None)
    args.update(kw)
    return L.gdn_state_copy(ctypes.byref(dims) if dims is not None else None, args["sc"],
                            args["ss"], args["ns"], args["si"], args["dc"], args["ds"],
                            args["nd"], args["di"], args["n"], args["status"], args["stream"])


def test_state_copy_and_reset_reject_bad_arguments(L):
    d = gdn.make_dims()
    assert _copy(L, None) == INVALID
    assert _copy(L, gdn.make_dims(d_k=64, d_v=64)) == UNSUP
    assert _copy(L, d, sc=None) == INVALID                  # a copy needs a source
    assert _copy(L, d, ss=None) == INVALID
    assert _copy(L, d, dc=None) == INVALID
    assert _copy(L, d, ds=FAKE + 4) == INVALID              # misaligned
    assert _copy(L, d, si=FAKE + 4) == INVALID
    assert _copy(L, d, di=FAKE + 8) == INVALID
    assert _copy(L, d, status=FAKE + 2) == INVALID
    assert _copy(L, d, ns=3) == INVALID                     # fewer source slots than pairs
    assert _copy(L, d, nd=3) == INVALID
    assert _copy(L, d, ns=0, si=FAKE) == INVALID            # an index array into no slots
    assert _copy(L, d, n=-1) == INVALID
    assert _copy(L, d, n=65536, ns=1 << 20, nd=1 << 20) == INVALID
    assert _copy(L, d, n=0) == OK                           # nothing to launch
    rst = lambda **kw: L.gdn_state_reset(ctypes.byref(d), kw.get("c", FAKE), kw.get("s", FAKE),
                                         kw.get("ns", 4), kw.get("slot"), kw.get("n", 4),
                                         None, None)
    assert rst(c=None) == INVALID
    assert rst(s=FAKE + 4) == INVALID
    assert rst(ns=2) == INVALID
    assert rst(slot=FAKE + 4) == INVALID
    assert rst(n=0) == OK


def test_decode_graph_create_rejects_bad_arguments_without_a_device(L):
    d = gdn.make_dims()

    def create(dims=d, steps=4, batch=3, n_slots=3, out=FAKE, graph=True, **kw):
        h = ctypes.c_void_p(12345)
        st = L.gdn_decode_graph_create(ctypes.byref(dims) if dims is not None else None, steps,
                                       FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE,
                                       kw.get("slot"), n_slots, batch, FAKE, FAKE, out, 0, None,
                                       ctypes.byref(h) if graph else None)
        return st, h.value
    assert create(graph=False)[0] == INVALID
    assert create(dims=None) == (INVALID, None)         # the handle is cleared on failure
    assert create(steps=0)[0] == INVALID
    assert create(batch=0)[0] == INVALID
    assert create(n_slots=2)[0] == INVALID
    assert create(out=FAKE + 4)[0] == INVALID
    assert create(slot=FAKE + 4)[0] == INVALID
    assert create(dims=gdn.make_dims(h_k=4, h_v=32))[0] == UNSUP
    assert L.gdn_decode_graph_launch(None, None) == INVALID
    L.gdn_decode_graph_destroy(None)                    # a no-op


def test_prefill_host_rejects_bad_arguments_before_any_device_call(L):
    d = gdn.make_dims()
    cu_ok = (ctypes.c_int32 * 3)(0, 100, 250)
    need = L.gdn_prefill_host_workspace_bytes(ctypes.byref(d), 2, 250, 64)
    assert need > 0
    assert L.gdn_prefill_host_workspace_bytes(ctypes.byref(d), 2, 250, 32) == 0   # seg < 64
    assert L.gdn_prefill_host_workspace_bytes(None, 2, 250, 0) == 0

    def call(dims=d, cu=cu_ok, n=2, T=250, seg=64, ws=0x100000, ws_bytes=None):
        return L.gdn_prefill_host(ctypes.byref(dims) if dims is not None else None, FAKE, FAKE,
                                  FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, cu, n, T, FAKE, FAKE, FAKE,
                                  seg, ws, need if ws_bytes is None else ws_bytes, None)
    assert call(dims=None) == INVALID
    assert call(dims=gdn.make_dims(d_k=64, d_v=64)) == UNSUP
    assert call(cu=None) == INVALID
    assert call(cu=(ctypes.c_int32 * 3)(0, 100, 249)) == INVALID        # last != total
    assert call(cu=(ctypes.c_int32 * 3)(1, 100, 250)) == INVALID        # first != 0
    assert call(cu=(ctypes.c_int32 * 3)(0, 200, 150), T=150) == INVALID  # decreasing
    assert call(seg=10) == INVALID
    assert call(seg=-1) == INVALID
    assert call(ws_bytes=need - 1) == WS
    assert call(ws=0x100010) == WS                                      # not 256-aligned

    def call_dev(**bad):                        # device pointers, checked before any copy
        p = dict(A_log=FAKE, dt_bias=FAKE, conv_w=FAKE, norm_w=FAKE, conv=FAKE, ssm=FAKE)
        p.update(bad)
        return L.gdn_prefill_host(ctypes.byref(d), FAKE, FAKE, FAKE, FAKE, p["A_log"],
                                  p["dt_bias"], p["conv_w"], p["norm_w"], cu_ok, 2, 250, p["conv"],
                                  p["ssm"], FAKE, 64, 0x100000, need, None)
    for name in ("A_log", "dt_bias", "conv_w", "norm_w", "conv", "ssm"):
        assert call_dev(**{name: None}) == INVALID, name
        assert call_dev(**{name: FAKE + 4}) == INVALID, name
    assert call(cu=(ctypes.c_int32 * 1)(0), n=0, T=0) == OK             # nothing to do


def _segments_model(cu, T, seg):
    """Plain restatement of the segmentation: tokens [s0, s1) and the
    sequences from the one holding s0 to the one holding s1 - 1."""
    holder = lambda t: max(q for q in range(len(cu) - 1) if cu[q] <= t < cu[q + 1])
    out = []
    for s0 in range(0, T, seg):
        s1 = min(T, s0 + seg)
        ja, jb = holder(s0), holder(s1 - 1)
        out.append((s0, s1, ja, jb - ja + 1))
    return out


def test_prefill_host_segments_match_the_plain_model_and_tile_the_batch(L):
    # 300 random packed batches (seed 5): 1-12 sequences of 0-3000 tokens,
    # with empty sequences and lengths at and around segment boundaries
    rng = np.random.default_rng(5)
    for trial in range(300):
        n = int(rng.integers(1, 13))
        pick = rng.integers(0, 4, size=n)
        lens = np.where(pick == 0, 0, np.where(pick == 1, rng.integers(1, 70, size=n),
                                               rng.integers(1, 3000, size=n)))
        if lens.sum() == 0:
            lens[0] = 1
        seg = int(rng.choice([0, 64, 100, 1024, 4096]))
        cu = [0] + list(np.cumsum(lens).astype(int))
        T = cu[-1]
        got = gdn.gdn_prefill_host_segments(torch.tensor(cu, dtype=torch.int32), seg)
        eff = min(seg if seg else 5120, T)
        assert got == _segments_model(cu, T, eff), (trial, cu, seg)
        # the segments tile [0, T) and each holds every token of its sequences' overlap
        assert got[0][0] == 0 and got[-1][1] == T
        assert all(a[1] == b[0] for a, b in zip(got, got[1:]))
        for s0, s1, ja, nj in got:
            held = [q for q in range(n) if cu[q] < s1 and cu[q + 1] > s0]
            assert held and held[0] == ja and held[-1] == ja + nj - 1
    bad = torch.tensor([0, 5, 3], dtype=torch.int32)
    with pytest.raises(gdn.GdnError):
        gdn.gdn_prefill_host_segments(bad)
    with pytest.raises(gdn.GdnError):
        gdn.gdn_prefill_host_segments(torch.tensor([0, 100], dtype=torch.int32), 32)


def test_selftest_wait_timeout_rejects_bad_arguments(L):
    assert L.gdn_selftest_wait_timeout(None, 1 << 20, None) == INVALID
    assert L.gdn_selftest_wait_timeout(FAKE + 2, 1 << 20, None) == INVALID     # misaligned
    assert L.gdn_selftest_wait_timeout(FAKE, 0, None) == INVALID
    assert L.gdn_selftest_wait_timeout(FAKE, (1 << 31) + 1, None) == INVALID    # over ~1 s


def test_workspace_grows_with_sequences_and_tokens(L):
    # gdn_prefill_host sizes one gdn_prefill workspace for (all sequences, one
    # segment of tokens) and reuses it for every segment's call, whose counts
    # are no larger: that needs gdn_workspace_bytes non-decreasing in both
    d = gdn.make_dims()
    ns = [1, 2, 3, 5, 8, 19, 64, 300]
    Ts = [1, 63, 64, 1024, 1025, 4096, 4100, 32768, 100000]
    for n in ns:
        row = [gdn.gdn_workspace_bytes(d, n, T) for T in Ts]
        assert all(x > 0 for x in row) and row == sorted(row), (n, row)
    for T in Ts:
        col = [gdn.gdn_workspace_bytes(d, n, T) for n in ns]
        assert col == sorted(col), (T, col)
    # and the host-fed call's own workspace holds at least that much
    assert (gdn.gdn_prefill_host_workspace_bytes(d, 5, 100000, 4096)
            > gdn.gdn_workspace_bytes(d, 5, 4096))


def test_prefill_segment_length_cost_model(L):
    # the choices measured on a 152-SM GB300 (32 value heads): 3648 tokens at
    # 32K (9 segments, the fastest of the lengths timed), 3456 at 64K, 2048 at 8K
    d = gdn.make_dims()
    seg = lambda n, T, sms=152: gdn.gdn_prefill_segment_tokens_for(d, n, T, sms)
    assert seg(1, 32768) == 3648 and seg(1, 65536) == 3456 and seg(1, 8192) == 2048
    assert seg(1, 1024) == 0                  # no longer than the shortest segment
    assert seg(19, 100000) == 0               # 19 x 32 heads >= 4 x 152: the GPU is full
    for n in (1, 2, 5, 18):
        for T in (1025, 5000, 32768, 131072, 262144):
            L_ = seg(n, T)
            assert L_ % 64 == 0 and 1024 <= L_ < T, (n, T, L_)
    assert seg(1, 32768, sms=0) == -1
    assert gdn.gdn_prefill_segment_tokens_for(gdn.make_dims(d_k=64, d_v=64), 1, 32768, 152) == -1


def test_prefill_rejects_bad_arguments(L):
    d = gdn.make_dims()
    assert _prefill(L, None) == INVALID
    assert _prefill(L, gdn.make_dims(chunk=32)) == UNSUP
    assert _prefill(L, d, cu=None) == INVALID
    assert _prefill(L, d, z=FAKE + 2) == INVALID
    assert _prefill(L, d, n_seqs=-1) == INVALID
    assert _prefill(L, d, T=-5) == INVALID
    assert _prefill(L, d, T=1 << 31) == INVALID
    assert _prefill(L, d, ws=None) == WS
    assert _prefill(L, d, ws=0x100010) == WS                           # not 256-aligned
    assert _prefill(L, d, ws_bytes=16) == WS
    assert _prefill(L, d, n_seqs=0) == OK                              # nothing to launch
    assert _prefill(L, d, T=0) == OK


def test_projections_reject_bad_arguments(L):
    d = gdn.make_dims()
    inp = lambda dims, H, T, *ptrs: L.gdn_in_proj(dims, H, T, *ptrs, None, None)
    outp = lambda dims, H, T, *ptrs: L.gdn_out_proj(dims, H, T, *ptrs, None, None)
    six, three = [FAKE] * 6, [FAKE] * 3
    D = ctypes.byref(d)
    assert inp(None, 2048, 5, *six) == INVALID
    assert inp(ctypes.byref(gdn.make_dims(d_k=64, d_v=64)), 2048, 5, *six) == UNSUP
    assert inp(D, 0, 5, *six) == INVALID                   # hidden
    assert inp(D, 2000, 5, *six) == UNSUP                  # not a multiple of 64
    assert inp(D, 65536 + 64, 5, *six) == UNSUP
    assert inp(D, 2048, -1, *six) == INVALID
    assert inp(D, 2048, 1 << 31, *six) == INVALID
    assert inp(D, 2048, 0, *six) == OK                     # nothing to launch
    assert inp(D, 2048, 5, FAKE, FAKE, FAKE + 8, FAKE, FAKE, FAKE) == INVALID   # misaligned qkv
    assert inp(D, 2048, 5, FAKE, None, FAKE, FAKE, FAKE, FAKE) == INVALID
    # h_v must be a multiple of 8 (the a and b runs are 16-byte stores)
    assert inp(ctypes.byref(gdn.make_dims(h_k=2, h_v=4)), 2048, 5, *six) == UNSUP
    assert L.gdn_in_proj(D, 2048, 5, *six, FAKE + 2, None) == INVALID             # status word alignment
    assert outp(D, 2048, 0, *three) == OK
    assert outp(D, 2048, 5, FAKE, FAKE, None) == INVALID
    assert outp(D, 96, 5, *three) == UNSUP
    assert outp(ctypes.byref(gdn.make_dims(conv_w=3)), 2048, 5, *three) == UNSUP


def test_noalloc_prefill_rejects_more_sequences_than_its_fixed_scratch(L):
    d = gdn.make_dims()
    text = open(HEADER).read()
    max_seqs = int(re.search(r"#define GDN_NOALLOC_MAX_SEQS (\d+)", text).group(1))
    args = [FAKE] * 9
    call = lambda n, T: L.gdn_prefill_noalloc(ctypes.byref(d), *args, n, T, FAKE, FAKE, FAKE, None, None)
    assert call(max_seqs + 1, 1 << 20) == UNSUP
    assert call(0, 100) == OK                        # nothing to launch
    assert L.gdn_prefill_noalloc(None, *args, 1, 1, FAKE, FAKE, FAKE, None, None) == INVALID
    assert L.gdn_prefill_noalloc(ctypes.byref(gdn.make_dims(d_k=64, d_v=64)), *args, 1, 1, FAKE,
                                 FAKE, FAKE, None, None) == UNSUP


def test_binding_checks_tensor_arguments(L):
    import torch
    d = gdn.make_dims()
    cpu = torch.zeros(4, 8192, dtype=torch.bfloat16)
    with pytest.raises(ValueError):
        gdn.gdn_decode_step(d, cpu, cpu, cpu, cpu, cpu, cpu, cpu, cpu, None, 4, cpu, cpu,
                            torch.zeros(4, 32, 128), stream=0)
    # the host-fed prefill wants host activations of the right dtype and size,
    # before anything reaches the library
    T = 64
    qkv = torch.zeros(T, 8192, dtype=torch.bfloat16)
    z = torch.zeros(T, 32, 128, dtype=torch.bfloat16)
    ab = torch.zeros(T, 32, dtype=torch.bfloat16)
    out = torch.zeros(T, 32, 128, dtype=torch.bfloat16)
    cu = torch.tensor([0, T], dtype=torch.int32)
    for bad in (dict(qkv=qkv.float()), dict(z=z[:, :16]), dict(out=out[: T - 1]),
                dict(cu=cu.long()), dict(qkv=qkv.t())):
        a = dict(qkv=qkv, z=z, out=out, cu=cu)
        a.update(bad)
        with pytest.raises(ValueError):
            gdn.gdn_prefill_host(d, a["qkv"], a["z"], ab, ab, None, None, None, None, a["cu"],
                                 None, None, a["out"], None)
    with pytest.raises(ValueError):
        gdn.gdn_prefill_host_segments(cu.long())


C_CONSUMER = r"""
#include <stdio.h>
#include "gdn.h"
int main(void) {
  gdn_dims d = {16, 32, 128, 128, 4, 64, 1e-6f, 1e-6f};
  int32_t cu[4] = {0, 5000, 5000, 9000};
  long long info[16];
  long long n = gdn_prefill_host_segments(cu, 3, 9000, 4096, info, 4);
  gdn_decode_graph* g = NULL;
  gdn_status bad = gdn_decode_graph_create(&d, 0, 0, 0, 0, 0, 0, 0, 0, 0, 0, 1, 1, 0, 0, 0, 0, 0, &g);
  printf("%d %zu %lld %lld %lld %lld %lld %d\n", gdn_version(), gdn_state_bytes(&d), n,
         info[4], info[5], info[6], info[7], (int)bad);
  return 0;
}
"""


def test_header_is_plain_c_and_a_c_program_links_the_library(L, tmp_path):
    # the ABI is for C callers: the header must compile as strict C99, and a C
    # program must link libgdn.so and get the host-only answers without a GPU
    inc = os.path.dirname(HEADER)
    subprocess.run(["gcc", "-std=c99", "-Wall", "-Wextra", "-Werror", "-pedantic", "-x", "c",
                    "-fsyntax-only", HEADER], check=True)
    src = tmp_path / "consumer.c"
    src.write_text(C_CONSUMER)
    exe = tmp_path / "consumer"
    libdir = os.path.dirname(gdn.LIB_PATH)
    subprocess.run(["gcc", "-std=c99", "-Wall", "-Werror", "-I", inc, str(src), "-L", libdir,
                    "-lgdn", f"-Wl,-rpath,{libdir}", "-o", str(exe)], check=True)
    out = subprocess.run([str(exe)], capture_output=True, text=True, check=True).stdout.split()
    version, state, nseg, s0, s1, ja, nj, bad = map(int, out)
    assert version == gdn.gdn_version() and state == gdn.gdn_state_bytes(gdn.make_dims())
    # 9000 tokens in 4096-token segments: the second covers tokens 4096-8191, from
    # sequence 0 (tokens 0-4999) through sequence 2 (5000-8999), the empty one between
    assert (nseg, s0, s1, ja, nj) == (3, 4096, 8192, 0, 3)
    assert bad == INVALID     # steps = 0
