"""fp64 CPU oracle of the Gated DeltaNet layer -- test infrastructure only.

Only the tests, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline
leg may import this package.  The CUDA library never loads it, and it shares
no code with the CUDA library: the arithmetic lives in ``gdn_oracle.c``
(plain C, fp64), and this module only marshals numpy arrays into it.

Every array handed over is converted to float64 first; bf16 and fp32 values
convert exactly, so the oracle sees the very bits the GPU path sees.

The layer definition the C file follows is written out at its top (conv +
SiLU, q/k L2 norm, decay and write gates, gated delta rule, gated RMSNorm).
"""
from __future__ import annotations

import contextlib
import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "gdn_oracle.c")
_LIB_PATH = os.path.join(_HERE, "libgdn_oracle.so")
_lib = None
_lock = threading.Lock()


def build(force: bool = False) -> str:
    """Compile gdn_oracle.c into libgdn_oracle.so with gcc (-O2, OpenMP)."""
    stale = (not os.path.exists(_LIB_PATH)
             or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC))
    if force or stale:
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O2", "-fPIC", "-shared", "-fopenmp", "-std=c11",
               "-o", tmp, _SRC, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


class OrDims(ctypes.Structure):
    _fields_ = [("h_k", ctypes.c_int), ("h_v", ctypes.c_int),
                ("d_k", ctypes.c_int), ("d_v", ctypes.c_int),
                ("conv_w", ctypes.c_int), ("l2_eps", ctypes.c_double),
                ("rms_eps", ctypes.c_double)]


_D = ctypes.POINTER(ctypes.c_double)
_I64 = ctypes.POINTER(ctypes.c_int64)
_I32 = ctypes.POINTER(ctypes.c_int32)


def _configure(L):
    for name in ("or_silu", "or_sigmoid", "or_softplus"):
        getattr(L, name).restype = ctypes.c_double
        getattr(L, name).argtypes = [ctypes.c_double]
    L.or_gates.restype = None
    L.or_gates.argtypes = [ctypes.c_double] * 4 + [_D, _D]
    L.or_conv_silu.restype = None
    L.or_conv_silu.argtypes = [ctypes.c_long, ctypes.c_int, ctypes.c_int,
                               _D, ctypes.c_long, _D, _D, _D, _D]
    L.or_l2norm.restype = None
    L.or_l2norm.argtypes = [ctypes.c_int, _D, ctypes.c_double, ctypes.c_double, _D]
    L.or_gated_rmsnorm.restype = None
    L.or_gated_rmsnorm.argtypes = [ctypes.c_int, _D, _D, _D, ctypes.c_double, _D]
    for name in ("or_recurrence_seq", "or_recurrence_products"):
        getattr(L, name).restype = None
        getattr(L, name).argtypes = [ctypes.c_long, ctypes.c_int, ctypes.c_int] + [_D] * 7
    L.or_recurrence_chunked.restype = None
    L.or_recurrence_chunked.argtypes = [ctypes.c_long, ctypes.c_int, ctypes.c_int,
                                        ctypes.c_int] + [_D] * 7
    L.or_layer.restype = ctypes.c_int
    L.or_layer.argtypes = [ctypes.POINTER(OrDims)] + [_D] * 8 + [
        _I64, ctypes.c_int, _D, _D, _D, _I32, ctypes.c_int, ctypes.c_int]
    L.or_max_threads.restype = ctypes.c_int
    L.or_max_threads.argtypes = []
    L.or_linear.restype = None
    L.or_linear.argtypes = [ctypes.c_long] * 3 + [_D] * 3
    L.or_round_bf16.restype = None
    L.or_round_bf16.argtypes = [ctypes.c_long, _D, _D]
    return L


def lib():
    global _lib
    with _lock:
        if _lib is None:
            _lib = _configure(ctypes.CDLL(build()))
    return _lib


@contextlib.contextmanager
def using_library(path: str):
    """Route every call of this module to another build of gdn_oracle.c for
    the duration of the block (the mutation tests load deliberately broken
    copies this way)."""
    global _lib
    lib()
    with _lock:
        saved = _lib
        _lib = _configure(ctypes.CDLL(path))
    try:
        yield
    finally:
        with _lock:
            _lib = saved


def _f64(x) -> np.ndarray:
    """Contiguous float64 copy of a numpy array or a CPU torch tensor."""
    if hasattr(x, "detach"):
        x = x.detach().to("cpu")
        import torch  # only when a tensor was passed
        x = x.to(torch.float64).numpy()
    return np.ascontiguousarray(np.asarray(x, dtype=np.float64))


def _p(x: np.ndarray):
    return x.ctypes.data_as(_D)


# ---- scalar pieces -----------------------------------------------------------

def silu(x: float) -> float:
    return lib().or_silu(float(x))


def sigmoid(x: float) -> float:
    return lib().or_sigmoid(float(x))


def softplus(x: float) -> float:
    return lib().or_softplus(float(x))


def gates(a: float, b: float, A_log: float, dt_bias: float):
    """(g, beta) of one token of one value head."""
    g = ctypes.c_double()
    beta = ctypes.c_double()
    lib().or_gates(float(a), float(b), float(A_log), float(dt_bias),
                   ctypes.byref(g), ctypes.byref(beta))
    return g.value, beta.value


# ---- vector pieces -----------------------------------------------------------

def conv_silu(x, w, state=None):
    """Causal depthwise conv + SiLU of one sequence.

    x: [T, n_ch]; w: [n_ch, W]; state: [W-1, n_ch] or None (zeros).
    Returns (y [T, n_ch], state_out [W-1, n_ch]).
    """
    x = _f64(x)
    w = _f64(w)
    T, n_ch = x.shape
    W = w.shape[1]
    st = _f64(state) if state is not None else None
    y = np.empty((T, n_ch))
    st_out = np.empty((max(W - 1, 0), n_ch))
    lib().or_conv_silu(T, n_ch, W, _p(x), n_ch, _p(w),
                       _p(st) if st is not None else None, _p(y),
                       _p(st_out) if W > 1 else None)
    return y, st_out


def l2norm(v, eps: float, scale: float = 1.0):
    v = _f64(v)
    out = np.empty_like(v)
    lib().or_l2norm(v.shape[0], _p(v), eps, scale, _p(out))
    return out


def gated_rmsnorm(o, z, w, eps: float):
    o, z, w = _f64(o), _f64(z), _f64(w)
    out = np.empty_like(o)
    lib().or_gated_rmsnorm(o.shape[0], _p(o), _p(z), _p(w), eps, _p(out))
    return out


# ---- the recurrence of one (sequence, value head) -----------------------------

def _rec_args(q, k, v, g, beta, S0):
    q, k, v, g, beta = (_f64(t) for t in (q, k, v, g, beta))
    T, d_k = q.shape
    d_v = v.shape[1]
    S = _f64(S0).copy() if S0 is not None else np.zeros((d_v, d_k))
    o = np.empty((T, d_v))
    return q, k, v, g, beta, S, o, T, d_k, d_v


def recurrence_seq(q, k, v, g, beta, S0=None):
    """Sequential gated delta rule.  Returns (o [T, d_v], S [d_v, d_k])."""
    q, k, v, g, beta, S, o, T, d_k, d_v = _rec_args(q, k, v, g, beta, S0)
    lib().or_recurrence_seq(T, d_k, d_v, _p(q), _p(k), _p(v), _p(g), _p(beta),
                            _p(S), _p(o))
    return o, S


def recurrence_chunked(q, k, v, g, beta, S0=None, chunk: int = 64):
    """Chunked WY/UT form of the same recurrence."""
    q, k, v, g, beta, S, o, T, d_k, d_v = _rec_args(q, k, v, g, beta, S0)
    lib().or_recurrence_chunked(T, d_k, d_v, int(chunk), _p(q), _p(k), _p(v),
                                _p(g), _p(beta), _p(S), _p(o))
    return o, S


def recurrence_products(q, k, v, g, beta, S0=None):
    """Explicit product form (short sequences only)."""
    q, k, v, g, beta, S, o, T, d_k, d_v = _rec_args(q, k, v, g, beta, S0)
    lib().or_recurrence_products(T, d_k, d_v, _p(q), _p(k), _p(v), _p(g),
                                 _p(beta), _p(S), _p(o))
    return o, S


# ---- the whole layer -----------------------------------------------------------

def max_threads() -> int:
    return lib().or_max_threads()


def layer(*, h_k, h_v, d_k, d_v, conv_w_width=4, l2_eps=1e-6, rms_eps=1e-6,
          qkv, z, a, b, A_log, dt_bias, conv_w, norm_w, cu_seqlens,
          conv_state=None, ssm_state=None, head_mask=None, chunk=0,
          n_threads=0):
    """The layer over cu_seqlens-packed sequences, in fp64.

    Shapes: qkv [T, Cc]; z [T, h_v, d_v]; a, b [T, h_v]; A_log, dt_bias [h_v];
    conv_w [Cc, W]; norm_w [d_v]; cu_seqlens [N+1]; conv_state [N, W-1, Cc];
    ssm_state [N, h_v, d_v, d_k] (both None = zeros).
    Returns (out [T, h_v, d_v], conv_state_out, ssm_state_out); heads masked
    out by ``head_mask`` keep NaN in ``out`` and their input state.
    """
    cu = np.ascontiguousarray(np.asarray(
        cu_seqlens.cpu().numpy() if hasattr(cu_seqlens, "cpu") else cu_seqlens,
        dtype=np.int64))
    N = cu.shape[0] - 1
    Cc = 2 * h_k * d_k + h_v * d_v
    W = conv_w_width
    qkv = _f64(qkv).reshape(-1, Cc)
    T = qkv.shape[0]
    z = _f64(z).reshape(T, h_v, d_v)
    a = _f64(a).reshape(T, h_v)
    b = _f64(b).reshape(T, h_v)
    A_log, dt_bias = _f64(A_log), _f64(dt_bias)
    conv_w = _f64(conv_w).reshape(Cc, W)
    norm_w = _f64(norm_w)
    cs = (_f64(conv_state).reshape(N, W - 1, Cc).copy() if conv_state is not None
          else np.zeros((N, W - 1, Cc)))
    ss = (_f64(ssm_state).reshape(N, h_v, d_v, d_k).copy() if ssm_state is not None
          else np.zeros((N, h_v, d_v, d_k)))
    out = np.full((T, h_v, d_v), np.nan)
    mask = None
    if head_mask is not None:
        mask = np.ascontiguousarray(np.asarray(head_mask, dtype=np.int32))
        assert mask.shape == (h_v,)
    dims = OrDims(h_k, h_v, d_k, d_v, W, l2_eps, rms_eps)
    rc = lib().or_layer(ctypes.byref(dims), _p(qkv), _p(z), _p(a), _p(b),
                        _p(A_log), _p(dt_bias), _p(conv_w), _p(norm_w),
                        cu.ctypes.data_as(_I64), N, _p(cs), _p(ss), _p(out),
                        mask.ctypes.data_as(_I32) if mask is not None else None,
                        int(chunk), int(n_threads))
    if rc != 0:
        raise ValueError("oracle: inconsistent arguments")
    return out, cs, ss


# ---- the dense projections around the layer -----------------------------------

def linear(x, w):
    """y = x w^T in fp64 (x [M, K], w [N, K] output features by input features)."""
    x, w = _f64(x), _f64(w)
    M, K = x.shape
    N = w.shape[0]
    assert w.shape[1] == K
    y = np.empty((M, N))
    lib().or_linear(M, N, K, _p(x), _p(w), _p(y))
    return y


def round_bf16(x):
    """Each value rounded to bf16 (nearest, ties to even), as fp64."""
    x = _f64(x)
    y = np.empty_like(x)
    lib().or_round_bf16(x.size, _p(x), _p(y))
    return y


def in_proj(x, w_in, *, h_k, h_v, d_k, d_v):
    """The input projection, stored as the layer's bf16 inputs.

    x [T, hidden]; w_in [Cc + h_v d_v + 2 h_v, hidden], its rows (output
    features) in the order: the Cc mixed q|k|v conv channels, z (value head
    major), a, b.  Returns (qkv [T, Cc], z [T, h_v, d_v], a [T, h_v],
    b [T, h_v]), each the fp64 product rounded to bf16.
    """
    Cc = 2 * h_k * d_k + h_v * d_v
    y = round_bf16(linear(x, w_in))
    assert y.shape[1] == Cc + h_v * d_v + 2 * h_v
    T = y.shape[0]
    qkv = y[:, :Cc]
    z = y[:, Cc:Cc + h_v * d_v].reshape(T, h_v, d_v)
    a = y[:, Cc + h_v * d_v:Cc + h_v * d_v + h_v]
    b = y[:, Cc + h_v * d_v + h_v:]
    return (np.ascontiguousarray(qkv), np.ascontiguousarray(z), np.ascontiguousarray(a),
            np.ascontiguousarray(b))


def out_proj(o, w_out):
    """The output projection of the layer's output o [T, h_v, d_v] (or [T, h_v d_v]),
    w_out [hidden, h_v d_v]: fp64 [T, hidden]."""
    o = _f64(o)
    return linear(o.reshape(o.shape[0], -1), w_out)
