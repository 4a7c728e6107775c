"""GPU check of the device-side failure path, without a fault.

A bounded wait that runs out (a barrier nothing completes) must end the
kernel with GDN_ERR_DEVICE_TIMEOUT in the status word, keep a code already
recorded, and leave the context usable for the kernels that follow.
"""
import time

import pytest
import torch

import gated_deltanet_linear_06_gb300 as gdn
import gdn_inputs as gi
from gpu_util import DEV, dims_of, to_dev

pytestmark = pytest.mark.gpu
SH = gi.LAYER
TIMEOUT, BOUNDS = 5, 6


def test_bounded_wait_times_out_reports_and_the_context_stays_usable():
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    t0 = time.monotonic()
    gdn.gdn_selftest_wait_timeout(status, 1 << 22)        # ~2 ms of clock cycles
    assert gdn.gdn_read_device_status(status) == TIMEOUT
    assert time.monotonic() - t0 < 30
    # a code already in the word is kept
    status.fill_(BOUNDS)
    gdn.gdn_selftest_wait_timeout(status, 1 << 20)
    assert gdn.gdn_read_device_status(status) == BOUNDS
    # the kernels that follow run normally: two decode steps from the same
    # states agree bit for bit, and a state reset zeroes its slots
    dims = dims_of(SH)
    params = to_dev(gi.make_params(SH, 97))
    st = gi.make_states(SH, 3, 97, ssm_std=0.3, conv_std=1.0)
    tok = to_dev(gi.make_tokens(SH, 3, 97))
    outs = []
    for _ in range(2):
        conv, ssm = st["conv_state"].to(DEV), st["ssm_state"].to(DEV)
        out = torch.empty(3, SH.h_v, SH.d_v, device=DEV)
        gdn.gdn_decode_step(dims, tok["qkv"], tok["z"], tok["a"], tok["b"], params["A_log"],
                            params["dt_bias"], params["conv_w"], params["norm_w"], None, 3, conv,
                            ssm, out)
        outs.append((out, ssm))
    assert torch.isfinite(outs[0][0]).all()
    assert torch.equal(outs[0][0], outs[1][0]) and torch.equal(outs[0][1], outs[1][1])
    gdn.gdn_state_reset(dims, conv, ssm)
    torch.cuda.synchronize()
    assert (ssm == 0).all() and (conv == 0).all()
