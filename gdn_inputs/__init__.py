"""Seeded synthetic inputs for the Gated DeltaNet layer.

Shared by the tests, the benchmark and the oracle's callers; it holds none of
the layer's arithmetic.  Every tensor comes from a torch CPU generator seeded
per (seed, stream), is drawn in fp32 and then rounded to the storage dtype
(bf16 rounds to nearest even), so the GPU path and the oracle read the same
bits.

Default distributions (the small fp32 case and the bf16 layer cases):
  q, k, v, z, a, b ~ N(0, 1);  A_log ~ U(0, ln 16);  dt_bias = 0;
  conv weights ~ N(0, variance 1/4);  RMSNorm weight = 1;
  SSM state ~ N(0, variance 0.1) or 0;  conv state ~ N(0, 1) or 0.
The second parameter of N(.,.) is read as the variance.

Projection inputs: the hidden state x ~ N(0, 1); projection weights
~ N(0, variance 1 / fan-in), so each projected value is about N(0, 1).

Controlled-gate variants pick the decay and write gates directly:
``gate_controlled`` draws u ~ U(lo, hi) and beta ~ U(blo, bhi), then sets
A_log = 0, dt_bias = 0, a = ln(1/u - 1) and b = ln(beta / (1 - beta)).
With those settings softplus(a) = -ln u, so the layer's exp(g) equals u up to
the bf16 rounding of a (the rounded a is what both sides read).
"""
from __future__ import annotations

import math
from dataclasses import dataclass

import torch


@dataclass(frozen=True)
class Shape:
    h_k: int = 16
    h_v: int = 32
    d_k: int = 128
    d_v: int = 128
    conv_w: int = 4

    @property
    def cq(self) -> int:
        return self.h_k * self.d_k

    @property
    def cv(self) -> int:
        return self.h_v * self.d_v

    @property
    def cc(self) -> int:
        """Mixed conv channels: q | k | v."""
        return 2 * self.cq + self.cv


LAYER = Shape()                      # 16 key heads, 32 value heads, d = 128
TINY = Shape(h_k=2, h_v=2, d_k=32, d_v=32)

_STREAMS = {"params": 1, "tokens": 2, "states": 3, "gates": 4, "norm_w": 5, "hidden": 6,
            "proj": 7}
_BLOCK = 2048                        # rows drawn per block (bounds fp32 temps)


def _gen(seed: int, stream: str, block: int = 0) -> torch.Generator:
    g = torch.Generator(device="cpu")
    g.manual_seed((seed * 1_000_003 + _STREAMS[stream] * 10_007 + block) & 0x7FFF_FFFF_FFFF)
    return g


def _randn(shape, gen, std: float, dtype) -> torch.Tensor:
    x = torch.randn(shape, generator=gen, dtype=torch.float32)
    if std != 1.0:
        x.mul_(std)
    return x.to(dtype)


def _randn_rows(rows: int, cols, seed: int, stream: str, std: float, dtype,
                offset: int = 0) -> torch.Tensor:
    """[rows, *cols] drawn in blocks, so huge tensors need no huge fp32 temp.

    Block b of the stream always holds the same values, whatever ``rows`` is,
    so a prefix of a long draw equals a shorter draw (used by the tests that
    split one sequence into segments)."""
    cols = tuple(cols) if isinstance(cols, (tuple, list)) else (cols,)
    out = torch.empty((rows,) + cols, dtype=dtype)
    r = 0
    while r < rows:
        blk = (offset + r) // _BLOCK
        lo = (offset + r) - blk * _BLOCK
        n = min(_BLOCK - lo, rows - r)
        full = _randn((_BLOCK,) + cols, _gen(seed, stream, blk), std, dtype)
        out[r:r + n] = full[lo:lo + n]
        r += n
    return out


def make_params(shape: Shape, seed: int, dtype=torch.bfloat16,
                norm_w: str = "ones") -> dict:
    """Per-layer parameters.  conv_w has ``dtype``; the rest are fp32."""
    g = _gen(seed, "params")
    A_log = torch.rand(shape.h_v, generator=g) * math.log(16.0)
    dt_bias = torch.zeros(shape.h_v)
    conv_w = _randn((shape.cc, shape.conv_w), g, 0.5, dtype)
    if norm_w == "ones":
        nw = torch.ones(shape.d_v)
    elif norm_w == "uniform":
        nw = 0.5 + torch.rand(shape.d_v, generator=_gen(seed, "norm_w"))
    else:
        raise ValueError(norm_w)
    return {"A_log": A_log.float(), "dt_bias": dt_bias.float(),
            "conv_w": conv_w, "norm_w": nw.float()}


def make_tokens(shape: Shape, T: int, seed: int, dtype=torch.bfloat16,
                offset: int = 0) -> dict:
    """Per-token activations for T tokens (rows ``offset`` .. ``offset+T`` of
    the seed's stream): qkv [T, cc], z [T, h_v, d_v], a [T, h_v], b [T, h_v]."""
    qkv = _randn_rows(T, shape.cc, seed, "tokens", 1.0, dtype, offset)
    z = _randn_rows(T, (shape.h_v, shape.d_v), seed + 7_777, "tokens", 1.0, dtype, offset)
    ab = _randn_rows(T, (2, shape.h_v), seed + 15_551, "tokens", 1.0, dtype, offset)
    return {"qkv": qkv, "z": z, "a": ab[:, 0].contiguous(), "b": ab[:, 1].contiguous()}


def make_states(shape: Shape, n: int, seed: int, ssm_std: float = 0.0,
                conv_std: float = 0.0) -> dict:
    """conv_state [n, W-1, cc] and ssm_state [n, h_v, d_v, d_k], fp32."""
    g = _gen(seed, "states")
    W1 = shape.conv_w - 1
    conv = (_randn((n, W1, shape.cc), g, conv_std, torch.float32) if conv_std
            else torch.zeros((n, W1, shape.cc)))
    ssm = (_randn_rows(n * shape.h_v, (shape.d_v, shape.d_k), seed, "states",
                       ssm_std, torch.float32).reshape(n, shape.h_v, shape.d_v, shape.d_k)
           if ssm_std else torch.zeros((n, shape.h_v, shape.d_v, shape.d_k)))
    return {"conv_state": conv, "ssm_state": ssm}


def gate_controlled(shape: Shape, T: int, seed: int, decay=(0.9, 1.0),
                    beta=(0.0, 0.3), dtype=torch.bfloat16, offset: int = 0) -> dict:
    """a, b [T, h_v] and A_log, dt_bias [h_v] such that exp(g) ~ U(decay) and
    beta ~ U(beta), per the recipe in the module docstring."""
    lo, hi = decay
    blo, bhi = beta
    n = T * shape.h_v
    g = _gen(seed, "gates", offset)
    u = lo + (hi - lo) * torch.rand(n, generator=g, dtype=torch.float64)
    u = u.clamp(min=1e-12, max=1.0 - 1e-7)
    bt = blo + (bhi - blo) * torch.rand(n, generator=g, dtype=torch.float64)
    bt = bt.clamp(min=1e-6, max=1.0 - 1e-6)
    a = torch.log(1.0 / u - 1.0).reshape(T, shape.h_v)
    b = torch.log(bt / (1.0 - bt)).reshape(T, shape.h_v)
    return {"a": a.to(torch.float32).to(dtype), "b": b.to(torch.float32).to(dtype),
            "A_log": torch.zeros(shape.h_v), "dt_bias": torch.zeros(shape.h_v)}


def cu_seqlens(lengths) -> torch.Tensor:
    """int32 [N+1] prefix sums of ``lengths`` (packed, no padding)."""
    c = [0]
    for n in lengths:
        c.append(c[-1] + int(n))
    return torch.tensor(c, dtype=torch.int32)


def make_hidden(T: int, hidden: int, seed: int, dtype=torch.bfloat16, offset: int = 0) -> torch.Tensor:
    """Hidden states x [T, hidden] ~ N(0, 1) (rows ``offset`` .. ``offset+T``)."""
    return _randn_rows(T, hidden, seed, "hidden", 1.0, dtype, offset)


def make_proj_weights(shape: Shape, hidden: int, seed: int, dtype=torch.bfloat16) -> dict:
    """The projections' weights, output features by input features:
    w_in [cc + cv + 2 h_v, hidden] ~ N(0, 1/hidden) (rows: q|k|v channels, z,
    a, b) and w_out [hidden, cv] ~ N(0, 1/cv)."""
    n_in = shape.cc + shape.cv + 2 * shape.h_v
    w_in = _randn_rows(n_in, hidden, seed, "proj", hidden ** -0.5, dtype)
    w_out = _randn_rows(hidden, shape.cv, seed + 31_337, "proj", shape.cv ** -0.5, dtype)
    return {"w_in": w_in, "w_out": w_out}
