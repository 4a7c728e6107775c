"""Python binding of libgdn, the Gated DeltaNet layer for GB300 (sm_103a).

Argument marshalling only: every function here has the name of the C entry
point it calls (include/gdn.h), turns torch tensors into device pointers and
the current torch stream into a cudaStream_t, and raises ``GdnError`` on a
non-OK status.  All arithmetic runs in the CUDA kernels of libgdn.so; there
is no CPU path.  If libgdn.so has not been built, loading fails loudly.

Shapes (see include/gdn.h for the full contract):
  qkv [T, Cc] bf16 (Cc = 2 h_k 128 + h_v 128), z [T, h_v, 128] bf16,
  a, b [T, h_v] bf16, A_log, dt_bias [h_v] fp32, conv_w [Cc, 4] bf16,
  norm_w [128] fp32, conv_state [N, 3, Cc] fp32, ssm_state [N, h_v, 128, 128]
  fp32, out [T, h_v, 128].
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libgdn.so")

GDN_OK = 0
GDN_ERR_DEVICE_TIMEOUT = 5
GDN_ERR_DEVICE_BOUNDS = 6
GDN_DTYPE_BF16 = 0
GDN_DTYPE_F32 = 1
GDN_DECODE_MAX_STEPS = 8   # most tokens one gdn_decode_multi call takes per sequence
STATUS_NAMES = {0: "GDN_OK", 1: "GDN_ERR_INVALID_ARG", 2: "GDN_ERR_UNSUPPORTED",
                3: "GDN_ERR_WORKSPACE", 4: "GDN_ERR_CUDA", 5: "GDN_ERR_DEVICE_TIMEOUT",
                6: "GDN_ERR_DEVICE_BOUNDS"}


class GdnError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {gdn_status_string(status)}")


class Dims(ctypes.Structure):
    """gdn_dims."""
    _fields_ = [("h_k", ctypes.c_int), ("h_v", ctypes.c_int), ("d_k", ctypes.c_int),
                ("d_v", ctypes.c_int), ("conv_w", ctypes.c_int), ("chunk", ctypes.c_int),
                ("l2_eps", ctypes.c_float), ("rms_eps", ctypes.c_float)]


def make_dims(h_k=16, h_v=32, d_k=128, d_v=128, conv_w=4, chunk=64, l2_eps=1e-6,
              rms_eps=1e-6) -> Dims:
    return Dims(h_k, h_v, d_k, d_v, conv_w, chunk, l2_eps, rms_eps)


_lib = None
_lock = threading.Lock()
_P = ctypes.c_void_p


def lib() -> ctypes.CDLL:
    """The loaded libgdn.so (raises if it was never built)."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise RuntimeError(
                    f"{LIB_PATH} is missing: build it first "
                    "(python -c 'import __graft_entry__ as g; g.build()')")
            L = ctypes.CDLL(LIB_PATH)
            DP = ctypes.POINTER(Dims)
            L.gdn_version.restype = ctypes.c_int
            L.gdn_version.argtypes = []
            L.gdn_status_string.restype = ctypes.c_char_p
            L.gdn_status_string.argtypes = [ctypes.c_int]
            L.gdn_state_bytes.restype = ctypes.c_size_t
            L.gdn_state_bytes.argtypes = [DP]
            L.gdn_workspace_bytes.restype = ctypes.c_size_t
            L.gdn_workspace_bytes.argtypes = [DP, ctypes.c_int, ctypes.c_longlong]
            L.gdn_prefill_segment_tokens.restype = ctypes.c_longlong
            L.gdn_prefill_segment_tokens.argtypes = [DP, ctypes.c_int, ctypes.c_longlong]
            L.gdn_prefill_segment_tokens_for.restype = ctypes.c_longlong
            L.gdn_prefill_segment_tokens_for.argtypes = [DP, ctypes.c_int, ctypes.c_longlong,
                                                         ctypes.c_int]
            L.gdn_prefill.restype = ctypes.c_int
            L.gdn_prefill.argtypes = [DP] + [_P] * 9 + [ctypes.c_int, ctypes.c_longlong] + \
                [_P] * 4 + [ctypes.c_size_t, _P]
            L.gdn_decode_step.restype = ctypes.c_int
            L.gdn_decode_step.argtypes = [DP] + [_P] * 9 + [ctypes.c_int, ctypes.c_int] + \
                [_P] * 3 + [ctypes.c_int, _P, _P]
            L.gdn_decode_step_host_workspace_bytes.restype = ctypes.c_size_t
            L.gdn_decode_step_host_workspace_bytes.argtypes = [DP, ctypes.c_int, ctypes.c_int]
            L.gdn_decode_step_host.restype = ctypes.c_int
            L.gdn_decode_step_host.argtypes = [DP] + [_P] * 9 + [ctypes.c_int, ctypes.c_int] + \
                [_P] * 3 + [ctypes.c_int, _P, _P, ctypes.c_size_t, _P]
            L.gdn_decode_multi.restype = ctypes.c_int
            L.gdn_decode_multi.argtypes = [DP] + [_P] * 9 + [ctypes.c_int] * 3 + [_P] * 3 + \
                [ctypes.c_int] + [_P] * 4
            L.gdn_state_copy.restype = ctypes.c_int
            L.gdn_state_copy.argtypes = [DP, _P, _P, ctypes.c_int, _P, _P, _P, ctypes.c_int, _P,
                                         ctypes.c_int, _P, _P]
            L.gdn_state_reset.restype = ctypes.c_int
            L.gdn_state_reset.argtypes = [DP, _P, _P, ctypes.c_int, _P, ctypes.c_int, _P, _P]
            L.gdn_decode_graph_create.restype = ctypes.c_int
            L.gdn_decode_graph_create.argtypes = [DP, ctypes.c_int] + [_P] * 9 + \
                [ctypes.c_int, ctypes.c_int] + [_P] * 3 + [ctypes.c_int, _P,
                                                           ctypes.POINTER(ctypes.c_void_p)]
            L.gdn_decode_graph_launch.restype = ctypes.c_int
            L.gdn_decode_graph_launch.argtypes = [ctypes.c_void_p, _P]
            L.gdn_decode_graph_destroy.restype = None
            L.gdn_decode_graph_destroy.argtypes = [ctypes.c_void_p]
            L.gdn_prefill_host_workspace_bytes.restype = ctypes.c_size_t
            L.gdn_prefill_host_workspace_bytes.argtypes = [DP, ctypes.c_int, ctypes.c_longlong,
                                                           ctypes.c_int]
            L.gdn_prefill_host_segments.restype = ctypes.c_longlong
            L.gdn_prefill_host_segments.argtypes = [_P, ctypes.c_int, ctypes.c_longlong,
                                                    ctypes.c_int, _P, ctypes.c_longlong]
            L.gdn_prefill_host.restype = ctypes.c_int
            L.gdn_prefill_host.argtypes = [DP] + [_P] * 9 + [ctypes.c_int, ctypes.c_longlong] + \
                [_P] * 3 + [ctypes.c_int, _P, ctypes.c_size_t, _P]
            L.gdn_prefill_noalloc.restype = ctypes.c_int
            L.gdn_prefill_noalloc.argtypes = [DP] + [_P] * 9 + [ctypes.c_int, ctypes.c_longlong] + \
                [_P] * 5
            L.gdn_selftest_wait_timeout.restype = ctypes.c_int
            L.gdn_selftest_wait_timeout.argtypes = [_P, ctypes.c_longlong, _P]
            L.gdn_in_proj.restype = ctypes.c_int
            L.gdn_in_proj.argtypes = [DP, ctypes.c_int, ctypes.c_longlong] + [_P] * 8
            L.gdn_out_proj.restype = ctypes.c_int
            L.gdn_out_proj.argtypes = [DP, ctypes.c_int, ctypes.c_longlong] + [_P] * 5
            L.gdn_read_device_status.restype = ctypes.c_int
            L.gdn_read_device_status.argtypes = [_P, _P, ctypes.POINTER(ctypes.c_int32)]
            _lib = L
    return _lib


def gdn_version() -> int:
    return lib().gdn_version()


def gdn_status_string(status: int) -> str:
    return lib().gdn_status_string(int(status)).decode()


def gdn_state_bytes(dims: Dims) -> int:
    return lib().gdn_state_bytes(ctypes.byref(dims))


def gdn_workspace_bytes(dims: Dims, n_seqs: int, total_tokens: int) -> int:
    return lib().gdn_workspace_bytes(ctypes.byref(dims), int(n_seqs), int(total_tokens))


def gdn_prefill_segment_tokens(dims: Dims, n_seqs: int, total_tokens: int) -> int:
    return lib().gdn_prefill_segment_tokens(ctypes.byref(dims), int(n_seqs), int(total_tokens))


def gdn_prefill_segment_tokens_for(dims: Dims, n_seqs: int, total_tokens: int, sms: int) -> int:
    """gdn_prefill's segment length on a GPU with `sms` SMs (no device needed)."""
    return lib().gdn_prefill_segment_tokens_for(ctypes.byref(dims), int(n_seqs),
                                                int(total_tokens), int(sms))


def _stream(stream) -> int | None:
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else stream


def _ptr(t, dtype, name, numel=None):
    if t is None:
        return None
    if not isinstance(t, torch.Tensor):
        return t                       # a raw device address, passed through
    if not t.is_cuda or t.dtype != dtype or not t.is_contiguous():
        raise ValueError(f"{name}: want a contiguous CUDA {dtype} tensor, "
                         f"got {t.dtype} on {t.device} (contiguous={t.is_contiguous()})")
    if numel is not None and t.numel() != numel:
        raise ValueError(f"{name}: want {numel} elements, got {t.numel()}")
    return t.data_ptr()


def _hptr(t, dtype, name, numel=None):
    """Address of a contiguous HOST tensor (pinned memory lets copies overlap)."""
    if not isinstance(t, torch.Tensor) or t.is_cuda or t.dtype != dtype or not t.is_contiguous():
        raise ValueError(f"{name}: want a contiguous host {dtype} tensor")
    if numel is not None and t.numel() != numel:
        raise ValueError(f"{name}: want {numel} elements, got {t.numel()}")
    return t.data_ptr()


def _check(status: int, where: str):
    if status != GDN_OK:
        raise GdnError(status, where)


def gdn_prefill(dims: Dims, qkv, z, a, b, A_log, dt_bias, conv_w, norm_w, cu_seqlens,
                conv_state, ssm_state, out, workspace, stream=None, n_seqs=None,
                total_tokens=None):
    """Chunked prefill over cu_seqlens-packed sequences (states updated in place)."""
    bf, f32 = torch.bfloat16, torch.float32
    N = int(n_seqs if n_seqs is not None else cu_seqlens.numel() - 1)
    T = int(total_tokens if total_tokens is not None else qkv.shape[0])
    Cc = 2 * dims.h_k * dims.d_k + dims.h_v * dims.d_v
    ws_bytes = workspace.numel() * workspace.element_size()
    st = lib().gdn_prefill(
        ctypes.byref(dims), _ptr(qkv, bf, "qkv", T * Cc), _ptr(z, bf, "z", T * dims.h_v * dims.d_v),
        _ptr(a, bf, "a", T * dims.h_v), _ptr(b, bf, "b", T * dims.h_v),
        _ptr(A_log, f32, "A_log", dims.h_v), _ptr(dt_bias, f32, "dt_bias", dims.h_v),
        _ptr(conv_w, bf, "conv_w", Cc * dims.conv_w), _ptr(norm_w, f32, "norm_w", dims.d_v),
        _ptr(cu_seqlens, torch.int32, "cu_seqlens", N + 1), N, T,
        _ptr(conv_state, f32, "conv_state", N * (dims.conv_w - 1) * Cc),
        _ptr(ssm_state, f32, "ssm_state", N * dims.h_v * dims.d_v * dims.d_k),
        _ptr(out, bf, "out", T * dims.h_v * dims.d_v), _ptr(workspace, workspace.dtype, "workspace"),
        ws_bytes, _stream(stream))
    _check(st, "gdn_prefill")


def gdn_prefill_noalloc(dims: Dims, qkv, z, a, b, A_log, dt_bias, conv_w, norm_w, cu_seqlens,
                        conv_state, ssm_state, out, device_status=None, stream=None, n_seqs=None,
                        total_tokens=None):
    """gdn_prefill for callers that cannot allocate: no workspace argument; the
    library's own fixed device array holds the scratch (see include/gdn.h)."""
    bf, f32 = torch.bfloat16, torch.float32
    N = int(n_seqs if n_seqs is not None else cu_seqlens.numel() - 1)
    T = int(total_tokens if total_tokens is not None else qkv.shape[0])
    Cc = 2 * dims.h_k * dims.d_k + dims.h_v * dims.d_v
    st = lib().gdn_prefill_noalloc(
        ctypes.byref(dims), _ptr(qkv, bf, "qkv", T * Cc), _ptr(z, bf, "z", T * dims.h_v * dims.d_v),
        _ptr(a, bf, "a", T * dims.h_v), _ptr(b, bf, "b", T * dims.h_v),
        _ptr(A_log, f32, "A_log", dims.h_v), _ptr(dt_bias, f32, "dt_bias", dims.h_v),
        _ptr(conv_w, bf, "conv_w", Cc * dims.conv_w), _ptr(norm_w, f32, "norm_w", dims.d_v),
        _ptr(cu_seqlens, torch.int32, "cu_seqlens", N + 1), N, T,
        _ptr(conv_state, f32, "conv_state", N * (dims.conv_w - 1) * Cc),
        _ptr(ssm_state, f32, "ssm_state", N * dims.h_v * dims.d_v * dims.d_k),
        _ptr(out, bf, "out", T * dims.h_v * dims.d_v),
        _ptr(device_status, torch.int32, "device_status", 1), _stream(stream))
    _check(st, "gdn_prefill_noalloc")


def gdn_decode_step(dims: Dims, qkv, z, a, b, A_log, dt_bias, conv_w, norm_w, slot, n_slots,
                    conv_state, ssm_state, out, device_status=None, stream=None, batch=None):
    """One decode step for ``batch`` sequences (states updated in place)."""
    bf, f32 = torch.bfloat16, torch.float32
    B = int(batch if batch is not None else qkv.shape[0])
    Cc = 2 * dims.h_k * dims.d_k + dims.h_v * dims.d_v
    out_dtype = GDN_DTYPE_F32 if out.dtype == f32 else GDN_DTYPE_BF16
    st = lib().gdn_decode_step(
        ctypes.byref(dims), _ptr(qkv, bf, "qkv", B * Cc), _ptr(z, bf, "z", B * dims.h_v * dims.d_v),
        _ptr(a, bf, "a", B * dims.h_v), _ptr(b, bf, "b", B * dims.h_v),
        _ptr(A_log, f32, "A_log", dims.h_v), _ptr(dt_bias, f32, "dt_bias", dims.h_v),
        _ptr(conv_w, bf, "conv_w", Cc * dims.conv_w), _ptr(norm_w, f32, "norm_w", dims.d_v),
        _ptr(slot, torch.int32, "slot", B), int(n_slots),
        B, _ptr(conv_state, f32, "conv_state", int(n_slots) * (dims.conv_w - 1) * Cc),
        _ptr(ssm_state, f32, "ssm_state", int(n_slots) * dims.h_v * dims.d_v * dims.d_k),
        _ptr(out, out.dtype, "out", B * dims.h_v * dims.d_v), out_dtype,
        _ptr(device_status, torch.int32, "device_status", 1), _stream(stream))
    _check(st, "gdn_decode_step")


def gdn_decode_step_host_workspace_bytes(dims: Dims, batch: int, out_dtype=torch.bfloat16) -> int:
    code = GDN_DTYPE_F32 if out_dtype == torch.float32 else GDN_DTYPE_BF16
    return lib().gdn_decode_step_host_workspace_bytes(ctypes.byref(dims), int(batch), code)


def _decode_step_host_args(dims, qkv, z, a, b, A_log, dt_bias, conv_w, norm_w, slot, n_slots,
                           conv_state, ssm_state, out, workspace, device_status, stream):
    bf, f32 = torch.bfloat16, torch.float32
    B = int(qkv.shape[0])
    Cc = 2 * dims.h_k * dims.d_k + dims.h_v * dims.d_v
    if out.dtype not in (bf, f32):
        raise ValueError("out: want a host bfloat16 or float32 tensor")
    out_dtype = GDN_DTYPE_F32 if out.dtype == f32 else GDN_DTYPE_BF16
    return (ctypes.byref(dims), _hptr(qkv, bf, "qkv", B * Cc), _hptr(z, bf, "z", B * dims.h_v * dims.d_v),
            _hptr(a, bf, "a", B * dims.h_v), _hptr(b, bf, "b", B * dims.h_v),
            _ptr(A_log, f32, "A_log", dims.h_v), _ptr(dt_bias, f32, "dt_bias", dims.h_v),
            _ptr(conv_w, bf, "conv_w", Cc * dims.conv_w), _ptr(norm_w, f32, "norm_w", dims.d_v),
            _ptr(slot, torch.int32, "slot", B), int(n_slots),
            B, _ptr(conv_state, f32, "conv_state", int(n_slots) * (dims.conv_w - 1) * Cc),
            _ptr(ssm_state, f32, "ssm_state", int(n_slots) * dims.h_v * dims.d_v * dims.d_k),
            _hptr(out, out.dtype, "out", B * dims.h_v * dims.d_v), out_dtype,
            _ptr(device_status, torch.int32, "device_status", 1), _ptr(workspace, torch.uint8, "workspace"),
            workspace.numel() if isinstance(workspace, torch.Tensor) else 0, _stream(stream))


def gdn_decode_step_host(dims: Dims, qkv, z, a, b, A_log, dt_bias, conv_w, norm_w, slot, n_slots,
                         conv_state, ssm_state, out, workspace, device_status=None, stream=None):
    """gdn_decode_step with qkv, z, a, b and out in (pinned) HOST memory: the
    call copies them in and out on the stream itself."""
    _check(lib().gdn_decode_step_host(*_decode_step_host_args(
        dims, qkv, z, a, b, A_log, dt_bias, conv_w, norm_w, slot, n_slots, conv_state, ssm_state, out,
        workspace, device_status, stream)), "gdn_decode_step_host")


class PreparedCall:
    """One library call whose arguments were checked and marshalled once:
    calling the object runs the same C function on the same buffers again
    (refill them in place between calls), at the cost of one ctypes call.
    The tensors it was prepared with must outlive it."""
    __slots__ = ("_fn", "_args", "_where", "_keep")

    def __init__(self, fn, args, where, keep):
        self._fn, self._args, self._where, self._keep = fn, args, where, keep

    def __call__(self) -> None:
        st = self._fn(*self._args)
        if st != GDN_OK:
            raise GdnError(st, self._where)


def prepare_decode_step_host(dims: Dims, qkv, z, a, b, A_log, dt_bias, conv_w, norm_w, slot, n_slots,
                             conv_state, ssm_state, out, workspace, device_status=None,
                             stream=None) -> PreparedCall:
    """gdn_decode_step_host on these buffers and this stream, ready to call
    once per step (a serving loop that refills the same pinned buffers)."""
    args = _decode_step_host_args(dims, qkv, z, a, b, A_log, dt_bias, conv_w, norm_w, slot, n_slots,
                                  conv_state, ssm_state, out, workspace, device_status, stream)
    keep = (dims, qkv, z, a, b, A_log, dt_bias, conv_w, norm_w, slot, conv_state, ssm_state, out,
            workspace, device_status)
    return PreparedCall(lib().gdn_decode_step_host, args, "gdn_decode_step_host", keep)


def gdn_decode_multi(dims: Dims, qkv, z, a, b, A_log, dt_bias, conv_w, norm_w, slot, n_slots,
                     conv_state, ssm_state, out, steps, ssm_trace=None, conv_trace=None,
                     device_status=None, stream=None, batch=None):
    """``steps`` decode steps per sequence for ``batch`` sequences in one call
    (token-major activations [batch][steps][...]; states updated in place)."""
    bf, f32 = torch.bfloat16, torch.float32
    K = int(steps)
    B = int(batch if batch is not None else out.shape[0])
    Cc = 2 * dims.h_k * dims.d_k + dims.h_v * dims.d_v
    out_dtype = GDN_DTYPE_F32 if out.dtype == f32 else GDN_DTYPE_BF16
    st = lib().gdn_decode_multi(
        ctypes.byref(dims), _ptr(qkv, bf, "qkv", B * K * Cc), _ptr(z, bf, "z", B * K * dims.h_v * dims.d_v),
        _ptr(a, bf, "a", B * K * dims.h_v), _ptr(b, bf, "b", B * K * dims.h_v),
        _ptr(A_log, f32, "A_log", dims.h_v), _ptr(dt_bias, f32, "dt_bias", dims.h_v),
        _ptr(conv_w, bf, "conv_w", Cc * dims.conv_w), _ptr(norm_w, f32, "norm_w", dims.d_v),
        _ptr(slot, torch.int32, "slot", B), int(n_slots), B, K,
        _ptr(conv_state, f32, "conv_state", int(n_slots) * (dims.conv_w - 1) * Cc),
        _ptr(ssm_state, f32, "ssm_state", int(n_slots) * dims.h_v * dims.d_v * dims.d_k),
        _ptr(out, out.dtype, "out", B * K * dims.h_v * dims.d_v), out_dtype,
        _ptr(ssm_trace, f32, "ssm_trace", B * K * dims.h_v * dims.d_v * dims.d_k),
        _ptr(conv_trace, f32, "conv_trace", B * K * (dims.conv_w - 1) * Cc),
        _ptr(device_status, torch.int32, "device_status", 1), _stream(stream))
    _check(st, "gdn_decode_multi")


def gdn_prefill_host_workspace_bytes(dims: Dims, n_seqs: int, total_tokens: int,
                                     seg_tokens: int = 0) -> int:
    return lib().gdn_prefill_host_workspace_bytes(ctypes.byref(dims), int(n_seqs),
                                                  int(total_tokens), int(seg_tokens))


def gdn_prefill_host_segments(cu_seqlens, seg_tokens: int = 0) -> list[tuple[int, int, int, int]]:
    """gdn_prefill_host's segments for a host int32 cu_seqlens: a list of
    (first token, end token, first sequence, sequence count)."""
    N = int(cu_seqlens.numel()) - 1
    cu = _hptr(cu_seqlens, torch.int32, "cu_seqlens", N + 1)
    T = int(cu_seqlens[-1])
    n = lib().gdn_prefill_host_segments(cu, N, T, int(seg_tokens), None, 0)
    if n < 0:
        raise GdnError(1, "gdn_prefill_host_segments")
    info = (ctypes.c_longlong * (4 * max(n, 1)))()
    lib().gdn_prefill_host_segments(cu, N, T, int(seg_tokens), info, n)
    return [tuple(info[4 * i: 4 * i + 4]) for i in range(n)]


def gdn_prefill_host(dims: Dims, qkv, z, a, b, A_log, dt_bias, conv_w, norm_w, cu_seqlens,
                     conv_state, ssm_state, out, workspace, seg_tokens=0, stream=None):
    """gdn_prefill from host activations (qkv, z, a, b, cu_seqlens, out on the host;
    parameters, states and workspace on the device), copies overlapped with compute."""
    bf, f32 = torch.bfloat16, torch.float32
    N = int(cu_seqlens.numel()) - 1
    T = int(qkv.shape[0])
    Cc = 2 * dims.h_k * dims.d_k + dims.h_v * dims.d_v
    st = lib().gdn_prefill_host(
        ctypes.byref(dims), _hptr(qkv, bf, "qkv", T * Cc), _hptr(z, bf, "z", T * dims.h_v * dims.d_v),
        _hptr(a, bf, "a", T * dims.h_v), _hptr(b, bf, "b", T * dims.h_v),
        _ptr(A_log, f32, "A_log", dims.h_v), _ptr(dt_bias, f32, "dt_bias", dims.h_v),
        _ptr(conv_w, bf, "conv_w", Cc * dims.conv_w), _ptr(norm_w, f32, "norm_w", dims.d_v),
        _hptr(cu_seqlens, torch.int32, "cu_seqlens", N + 1), N, T,
        _ptr(conv_state, f32, "conv_state", N * (dims.conv_w - 1) * Cc),
        _ptr(ssm_state, f32, "ssm_state", N * dims.h_v * dims.d_v * dims.d_k),
        _hptr(out, bf, "out", T * dims.h_v * dims.d_v), int(seg_tokens),
        _ptr(workspace, torch.uint8, "workspace"), workspace.numel(), _stream(stream))
    _check(st, "gdn_prefill_host")


class DecodeGraph:
    """A CUDA graph of ``steps`` successive decode steps over bound buffers
    (gdn_decode_graph_create); ``launch()`` runs them all, ``close()`` frees it."""

    def __init__(self, handle, keep):
        self._h = handle
        self._keep = keep              # the bound tensors stay alive with the graph

    def launch(self, stream=None):
        if not self._h:
            raise ValueError("gdn_decode_graph: closed")
        _check(lib().gdn_decode_graph_launch(self._h, _stream(stream)), "gdn_decode_graph_launch")

    def close(self):
        if self._h:
            lib().gdn_decode_graph_destroy(self._h)
            self._h = None
            self._keep = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def gdn_decode_graph_create(dims: Dims, steps, qkv, z, a, b, A_log, dt_bias, conv_w, norm_w,
                            slot, n_slots, conv_state, ssm_state, out, device_status=None):
    """Capture ``steps`` decode steps over step-major buffers ([steps][batch][...])."""
    bf, f32 = torch.bfloat16, torch.float32
    S, B = int(steps), int(out.shape[1])
    Cc = 2 * dims.h_k * dims.d_k + dims.h_v * dims.d_v
    out_dtype = GDN_DTYPE_F32 if out.dtype == f32 else GDN_DTYPE_BF16
    h = ctypes.c_void_p()
    st = lib().gdn_decode_graph_create(
        ctypes.byref(dims), S, _ptr(qkv, bf, "qkv", S * B * Cc),
        _ptr(z, bf, "z", S * B * dims.h_v * dims.d_v), _ptr(a, bf, "a", S * B * dims.h_v),
        _ptr(b, bf, "b", S * B * dims.h_v), _ptr(A_log, f32, "A_log", dims.h_v),
        _ptr(dt_bias, f32, "dt_bias", dims.h_v), _ptr(conv_w, bf, "conv_w", Cc * dims.conv_w),
        _ptr(norm_w, f32, "norm_w", dims.d_v), _ptr(slot, torch.int32, "slot", B), int(n_slots), B,
        _ptr(conv_state, f32, "conv_state", int(n_slots) * (dims.conv_w - 1) * Cc),
        _ptr(ssm_state, f32, "ssm_state", int(n_slots) * dims.h_v * dims.d_v * dims.d_k),
        _ptr(out, out.dtype, "out", S * B * dims.h_v * dims.d_v), out_dtype,
        _ptr(device_status, torch.int32, "device_status", 1), ctypes.byref(h))
    _check(st, "gdn_decode_graph_create")
    keep = (qkv, z, a, b, A_log, dt_bias, conv_w, norm_w, slot, conv_state, ssm_state, out,
            device_status)
    return DecodeGraph(h.value, keep)


def _pool(dims: Dims, conv_state, ssm_state, name):
    """Slot count of a state pool ([slots][W-1][Cc] and [slots][h_v][d_v][d_k] fp32)."""
    n = int(ssm_state.shape[0])
    Cc = 2 * dims.h_k * dims.d_k + dims.h_v * dims.d_v
    f32 = torch.float32
    return n, (_ptr(conv_state, f32, name + " conv_state", n * (dims.conv_w - 1) * Cc),
               _ptr(ssm_state, f32, name + " ssm_state", n * dims.h_v * dims.d_v * dims.d_k))


def gdn_state_copy(dims: Dims, src_conv_state, src_ssm_state, dst_conv_state, dst_ssm_state,
                   src_slot=None, dst_slot=None, n=None, device_status=None, stream=None):
    """Copy n whole states from one state pool's slots into another's (snapshot / restore)."""
    ns, (sc, ss) = _pool(dims, src_conv_state, src_ssm_state, "source")
    nd, (dc, ds) = _pool(dims, dst_conv_state, dst_ssm_state, "destination")
    if n is None:
        n = int(src_slot.numel()) if src_slot is not None else (
            int(dst_slot.numel()) if dst_slot is not None else min(ns, nd))
    st = lib().gdn_state_copy(
        ctypes.byref(dims), sc, ss, ns, _ptr(src_slot, torch.int32, "src_slot", n), dc, ds, nd,
        _ptr(dst_slot, torch.int32, "dst_slot", n), int(n),
        _ptr(device_status, torch.int32, "device_status", 1), _stream(stream))
    _check(st, "gdn_state_copy")


def gdn_state_reset(dims: Dims, conv_state, ssm_state, slot=None, n=None, device_status=None,
                    stream=None):
    """Zero the states of n slots of a state pool."""
    ns, (c, s) = _pool(dims, conv_state, ssm_state, "pool")
    if n is None:
        n = int(slot.numel()) if slot is not None else ns
    st = lib().gdn_state_reset(ctypes.byref(dims), c, s, ns, _ptr(slot, torch.int32, "slot", n),
                               int(n), _ptr(device_status, torch.int32, "device_status", 1),
                               _stream(stream))
    _check(st, "gdn_state_reset")


def gdn_selftest_wait_timeout(device_status, budget_cycles: int = 1 << 22, stream=None):
    """Run the bounded-wait self-test (the kernel times out on purpose and
    writes GDN_ERR_DEVICE_TIMEOUT into ``device_status``)."""
    st = lib().gdn_selftest_wait_timeout(_ptr(device_status, torch.int32, "device_status", 1),
                                         int(budget_cycles), _stream(stream))
    _check(st, "gdn_selftest_wait_timeout")


def in_proj_features(dims: Dims) -> int:
    """Rows of gdn_in_proj's weight: Cc conv channels, z, a, b."""
    return 2 * dims.h_k * dims.d_k + 2 * dims.h_v * dims.d_v + 2 * dims.h_v


def gdn_in_proj(dims: Dims, hidden: int, x, w_in, qkv, z, a, b, device_status=None, stream=None,
                tokens=None):
    """Input projection x [T, hidden] -> the layer's qkv, z, a, b (bf16, written in place)."""
    bf = torch.bfloat16
    T = int(tokens if tokens is not None else x.shape[0])
    H = int(hidden)
    Cc = 2 * dims.h_k * dims.d_k + dims.h_v * dims.d_v
    st = lib().gdn_in_proj(
        ctypes.byref(dims), H, T, _ptr(x, bf, "x", T * H),
        _ptr(w_in, bf, "w_in", in_proj_features(dims) * H), _ptr(qkv, bf, "qkv", T * Cc),
        _ptr(z, bf, "z", T * dims.h_v * dims.d_v), _ptr(a, bf, "a", T * dims.h_v),
        _ptr(b, bf, "b", T * dims.h_v), _ptr(device_status, torch.int32, "device_status", 1),
        _stream(stream))
    _check(st, "gdn_in_proj")


def gdn_out_proj(dims: Dims, hidden: int, o, w_out, y, device_status=None, stream=None,
                 tokens=None):
    """Output projection o [T, h_v, d_v] -> y [T, hidden] (bf16)."""
    bf = torch.bfloat16
    T = int(tokens if tokens is not None else o.shape[0])
    H = int(hidden)
    Cv = dims.h_v * dims.d_v
    st = lib().gdn_out_proj(
        ctypes.byref(dims), H, T, _ptr(o, bf, "o", T * Cv), _ptr(w_out, bf, "w_out", H * Cv),
        _ptr(y, bf, "y", T * H), _ptr(device_status, torch.int32, "device_status", 1),
        _stream(stream))
    _check(st, "gdn_out_proj")


def gdn_read_device_status(status_word, stream=None) -> int:
    """Waits for the stream and returns the device status word's value."""
    code = ctypes.c_int32(0)
    addr = status_word.data_ptr() if isinstance(status_word, torch.Tensor) else status_word
    _check(lib().gdn_read_device_status(addr, _stream(stream), ctypes.byref(code)),
           "gdn_read_device_status")
    return code.value
