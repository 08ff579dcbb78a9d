"""Failure detection on the GPU without a fault: a bounded wait that runs out is reported to
the host as CBR_ERR_TIMEOUT by cbr_stream_status, the error word is cleared, and the context
stays usable for the next training step (through the C ABI)."""
import time

import numpy as np
import pytest
import torch

import oracle
from conv_batchnorm_relu_gb300 import cbr
from conv_batchnorm_relu_gb300.inputs import CONFIGS, make_inputs, seed_for
from parity import max_err_ok, oracle_inputs, to_np

pytestmark = pytest.mark.gpu

CBR_ERR_TIMEOUT = 7


def test_expired_bounded_wait_is_reported_and_context_stays_usable():
    torch.cuda.synchronize()
    assert cbr.stream_status_code() == cbr.CBR_OK
    t0 = time.perf_counter()
    cbr.selftest_bounded_wait(20000)  # 20 ms on a barrier that nothing completes
    assert cbr.stream_status_code() == CBR_ERR_TIMEOUT
    assert time.perf_counter() - t0 >= 0.015
    # the word was cleared by the read, and nothing else is pending
    assert cbr.stream_status_code() == cbr.CBR_OK

    # the next training step runs normally
    spec = CONFIGS[1]
    inp = make_inputs(spec, seed_for(1), with_dy=False)
    layer = cbr.Layer.from_spec(spec)
    g = {k: v.cuda() for k, v in inp.items()}
    fwd_ws, _ = cbr.workspace_size(layer)
    out = cbr.forward_train(layer, g["x"], g["w"], g["gamma"], g["beta"], g["running_mean"],
                            g["running_var"], spec.momentum, spec.eps, ws=cbr.new_workspace(fwd_ws))
    assert cbr.stream_status_code() == cbr.CBR_OK
    o = oracle_inputs(inp)
    ref = oracle.forward_train(o["x"], o["w"], o["gamma"], o["beta"], o["running_mean"],
                               o["running_var"], spec.momentum, spec.eps, spec.stride, spec.pad)
    max_err_ok(to_np(out["y"]), ref["y"], "y after a reported timeout")
