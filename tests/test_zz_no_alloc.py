"""The allocation-free training forward, cbr_forward_train_noalloc, against cbr_forward_train.

Some callers cannot allocate device memory where they run: plug-ins called from another
framework's execution loop without access to its allocator, or latency-critical loops that
cannot pay for cudaMalloc's cost and implicit synchronisation.  This entry point serves them
from scratch compiled into the library.  The test calls it through the C ABI twice in a row,
so the second call runs on scratch left behind by the first, and compares each call's
outputs with those of the workspace-based entry point on the same inputs, using the parity
tolerances of the other GPU tests; the first call is also checked against the CPU oracle
directly, so the test does not rest on the other entry point alone.  It runs last so that a
failure here cannot hide others.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
from conv_batchnorm_relu_gb300 import build, cbr
from conv_batchnorm_relu_gb300.inputs import CONFIGS, CBRSpec, make_inputs
from parity import mask_ok, max_err_ok, oracle_inputs, rel_close, stat_close, to_np, unpack_mask

pytestmark = pytest.mark.gpu

CASES = {
    "n3_56_64_f16": (CONFIGS[3].with_(n=3), 2001),
    "c128_bf16": (CBRSpec("c128", n=2, h=24, w=24, c_in=128, c_out=128, dtype="bf16"), 2004),
}


def _lib():
    build.build()
    lib = cbr.load()
    vp, fp = ctypes.c_void_p, ctypes.c_float
    f = lib.cbr_forward_train_noalloc
    f.argtypes = [ctypes.POINTER(cbr.Desc), vp, vp, vp, vp, vp, vp, fp, fp, vp, vp, vp, vp, vp, vp]
    f.restype = ctypes.c_int32
    return lib


def _outputs(layer, spec, dev):
    y = torch.empty((spec.n, spec.p, spec.q, spec.c_out), dtype=spec.torch_dtype, device=dev)
    return {"y": y, "z": torch.empty_like(y),
            "mask": torch.empty(cbr.mask_words(layer), dtype=torch.int32, device=dev),
            "saved_mean": torch.empty(spec.c_out, device=dev),
            "saved_inv_var": torch.empty(spec.c_out, device=dev)}


@pytest.mark.parametrize("case", list(CASES))
def test_noalloc_forward_matches_workspace_forward_twice(case):
    spec, seed = CASES[case]
    lib = _lib()
    dev = torch.device("cuda", 0)
    layer = cbr.Layer.from_spec(spec)
    inp = make_inputs(spec, seed, with_dy=False)
    g = {k: v.to(dev) for k, v in inp.items()}
    fwd_bytes, _ = cbr.workspace_size(layer)
    ws = cbr.new_workspace(fwd_bytes, dev)
    d = layer.desc()
    for call in range(2):
        # the workspace-based entry point, from a copy of the running statistics
        rm_ref, rv_ref = g["running_mean"].clone(), g["running_var"].clone()
        ref = cbr.forward_train(layer, g["x"], g["w"], g["gamma"], g["beta"], rm_ref, rv_ref,
                                spec.momentum, spec.eps, ws=ws)
        # the allocation-free entry point, from another copy
        rm, rv = g["running_mean"].clone(), g["running_var"].clone()
        o = _outputs(layer, spec, dev)
        st = lib.cbr_forward_train_noalloc(
            ctypes.byref(d), g["x"].data_ptr(), g["w"].data_ptr(), g["gamma"].data_ptr(),
            g["beta"].data_ptr(), rm.data_ptr(), rv.data_ptr(), spec.momentum, spec.eps,
            o["y"].data_ptr(), o["mask"].data_ptr(), o["z"].data_ptr(), o["saved_mean"].data_ptr(),
            o["saved_inv_var"].data_ptr(), torch.cuda.current_stream().cuda_stream)
        assert st == 0, f"call {call}: {cbr.STATUS_NAMES.get(st, st)}"
        cbr.stream_status()
        max_err_ok(to_np(o["y"]), to_np(ref["y"]), f"y (call {call})")
        max_err_ok(to_np(o["z"]), to_np(ref["z"]), f"z (call {call})")
        assert torch.equal(o["mask"], ref["mask"]), f"mask (call {call})"
        sd = 1.0 / to_np(ref["saved_inv_var"])
        stat_close(to_np(o["saved_mean"]), to_np(ref["saved_mean"]), sd, f"saved_mean (call {call})")
        rel_close(to_np(o["saved_inv_var"]), to_np(ref["saved_inv_var"]), f"saved_inv_var (call {call})")
        stat_close(to_np(rm), to_np(rm_ref), spec.momentum * sd, f"running_mean (call {call})")
        rel_close(to_np(rv), to_np(rv_ref), f"running_var (call {call})")
        if call == 0:
            o_np = oracle_inputs(inp)
            want = oracle.forward_train(o_np["x"], o_np["w"], o_np["gamma"], o_np["beta"],
                                        o_np["running_mean"], o_np["running_var"], spec.momentum,
                                        spec.eps, spec.stride, spec.pad)
            max_err_ok(to_np(o["y"]), want["y"], "y vs oracle")
            max_err_ok(to_np(o["z"]), want["z"], "z vs oracle")
            mask_ok(unpack_mask(o["mask"], want["pre"].size), want["pre"], "mask vs oracle")
            sd = np.sqrt(want["var"])
            stat_close(to_np(o["saved_mean"]), want["mean"], sd, "saved_mean vs oracle")
            rel_close(to_np(o["saved_inv_var"]), want["inv_std"], "saved_inv_var vs oracle")
