"""Shared helpers of the GPU parity tests (not a test module)."""
import numpy as np
import torch

import gated_deltanet_linear_06_gb300 as gdn
import gdn_inputs as gi
import oracle

DEV = torch.device("cuda:0")

# The acceptance bars: max |gpu - oracle| / max |oracle| over a whole tensor.
DECODE_TOL = 1e-4     # fp32 state and fp32 output of a decode step
PREFILL_TOL = 1e-2    # bf16-operand prefill: bf16 output and the fp32 final state


def rel_err(got, ref) -> float:
    got = got.detach().double().cpu().numpy() if isinstance(got, torch.Tensor) else np.asarray(got, np.float64)
    ref = ref.detach().double().cpu().numpy() if isinstance(ref, torch.Tensor) else np.asarray(ref, np.float64)
    assert got.shape == ref.shape, (got.shape, ref.shape)
    assert np.all(np.isfinite(got)), "non-finite values in the GPU result"
    return float(np.abs(got - ref).max() / max(np.abs(ref).max(), 1e-30))


def bf16_round(x: np.ndarray) -> np.ndarray:
    """fp64 -> bf16 (round to nearest even) -> fp64."""
    return torch.from_numpy(np.asarray(x, np.float64)).to(torch.float32).to(torch.bfloat16).double().numpy()


def bf16_ulp(x: np.ndarray) -> np.ndarray:
    """Spacing of bf16 numbers at |x| (8 significant bits)."""
    ax = np.maximum(np.abs(x), 1e-38)
    return 2.0 ** (np.floor(np.log2(ax)) - 7)


def dims_of(sh: gi.Shape):
    return gdn.make_dims(h_k=sh.h_k, h_v=sh.h_v, d_k=sh.d_k, d_v=sh.d_v, conv_w=sh.conv_w)


def oracle_layer(sh: gi.Shape, tok: dict, params: dict, cu, conv_state=None, ssm_state=None,
                 head_mask=None, n_threads=0):
    return oracle.layer(h_k=sh.h_k, h_v=sh.h_v, d_k=sh.d_k, d_v=sh.d_v, conv_w_width=sh.conv_w,
                        qkv=tok["qkv"], z=tok["z"], a=tok["a"], b=tok["b"],
                        A_log=params["A_log"], dt_bias=params["dt_bias"],
                        conv_w=params["conv_w"], norm_w=params["norm_w"], cu_seqlens=cu,
                        conv_state=conv_state, ssm_state=ssm_state, head_mask=head_mask,
                        n_threads=n_threads)


def to_dev(d: dict) -> dict:
    return {k: v.to(DEV) for k, v in d.items()}


def assert_bf16_close(got_bf16, ref, tol=DECODE_TOL):
    """bf16 output check: |got - ref| <= 1 bf16 ulp of ref + tol * max|ref|.

    A bf16 result of an fp32 computation that meets ``tol`` differs from the
    exact value by its rounding (at most one ulp once the fp32 error can push
    it across a rounding boundary) plus the fp32 error itself; near-zero
    outputs are dominated by the second term."""
    got = got_bf16.detach().float().cpu().double().numpy() if isinstance(got_bf16, torch.Tensor) \
        else np.asarray(got_bf16, np.float64)
    ref = np.asarray(ref, np.float64)
    bound = bf16_ulp(ref) + tol * np.abs(ref).max()
    excess = np.abs(got - ref) - bound
    worst_ulps = float((np.abs(got - bf16_round(ref)) / bf16_ulp(ref)).max())
    assert np.all(excess <= 0), f"bf16 output off by up to {worst_ulps:.1f} ulp beyond the bound"
    return worst_ulps
