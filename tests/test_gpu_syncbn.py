"""GPU tests of the synchronised-BN split calls (BatchNorm CUDA page, section 7.1), with two
ranks simulated on one GPU: each half of a batch runs the first-half calls, the "collective" is
a concatenation (moments) or a sum (backward sums) on the device, and each half then runs the
second-half calls.  The statistics, y, dx, dgamma, dbeta and the summed dW must match one
training step over the whole batch, and the oracle over the whole batch."""
import numpy as np
import pytest
import torch

import oracle
from conv_batchnorm_relu_gb300 import cbr
from conv_batchnorm_relu_gb300.inputs import CBRSpec, make_inputs
from parity import max_err_ok, oracle_inputs, rel_close, stat_close, to_np

pytestmark = pytest.mark.gpu

CASES = {
    "fused_64": (CBRSpec("syncbn 64", n=4, h=14, w=18, c_in=64, c_out=64), 2301),
    "c128_bf16": (CBRSpec("syncbn 128", n=4, h=10, w=12, c_in=128, c_out=128, dtype="bf16"), 2302),
    "first": (CBRSpec("syncbn first", n=4, h=24, w=24, c_in=3, c_out=64, r=7, s=7, stride=2, pad=3,
                      x_dist="uniform2.5", first_layer=True), 2303),
}


@pytest.mark.parametrize("case", list(CASES))
def test_two_rank_syncbn_matches_one_whole_batch_step(case):
    spec, seed = CASES[case]
    inp = make_inputs(spec, seed)
    g = {k: v.cuda() for k, v in inp.items()}
    need_dx = not spec.first_layer
    whole = cbr.Layer.from_spec(spec)
    half = cbr.Layer.from_spec(spec.with_(n=spec.n // 2))
    fwd_b, bwd_b = cbr.workspace_size(whole)

    # one step over the whole batch
    rm_w, rv_w = g["running_mean"].clone(), g["running_var"].clone()
    ref = cbr.forward_train(whole, g["x"], g["w"], g["gamma"], g["beta"], rm_w, rv_w, spec.momentum, spec.eps,
                            ws=cbr.new_workspace(fwd_b))
    rb = cbr.backward(whole, g["dy"], g["x"], g["w"], ref["mask"], cbr.CBR_MASK_BITS, ref["z"], g["gamma"],
                      ref["saved_mean"], ref["saved_inv_var"], ws=cbr.new_workspace(bwd_b), need_dx=need_dx)

    # two ranks: images [0, n/2) and [n/2, n)
    parts = [slice(0, spec.n // 2), slice(spec.n // 2, spec.n)]
    wsf = [cbr.new_workspace(fwd_b) for _ in parts]
    wsb = [cbr.new_workspace(bwd_b) for _ in parts]
    zs, moms = zip(*[cbr.forward_train_stats(half, g["x"][p], g["w"], ws=wsf[i]) for i, p in enumerate(parts)])
    moments_all = torch.stack(moms)                       # the all-gather, in rank order
    rms = [g["running_mean"].clone() for _ in parts]
    rvs = [g["running_var"].clone() for _ in parts]
    fo = [cbr.forward_train_finish(half, moments_all, g["gamma"], g["beta"], rms[i], rvs[i], spec.momentum,
                                   spec.eps, zs[i], ws=wsf[i]) for i in range(2)]
    assert fo[0]["m_total"] == spec.m
    sums = [cbr.backward_sums(half, g["dy"][p], fo[i]["mask"], cbr.CBR_MASK_BITS, zs[i], fo[i]["saved_mean"],
                              ws=wsb[i]) for i, p in enumerate(parts)]
    total = sums[0] + sums[1]                              # the all-reduce
    bo = [cbr.backward_finish(half, total, spec.m, g["dy"][p], g["x"][p], g["w"], fo[i]["mask"], cbr.CBR_MASK_BITS,
                              zs[i], g["gamma"], fo[i]["saved_mean"], fo[i]["saved_inv_var"], ws=wsb[i],
                              need_dx=need_dx) for i, p in enumerate(parts)]
    cbr.stream_status()

    # both ranks hold the same statistics, and they are the whole batch's
    for i in range(2):
        assert torch.equal(fo[i]["saved_mean"], fo[0]["saved_mean"])
        assert torch.equal(fo[i]["saved_inv_var"], fo[0]["saved_inv_var"])
        assert torch.equal(bo[i]["dgamma"], bo[0]["dgamma"]) and torch.equal(bo[i]["dbeta"], bo[0]["dbeta"])
    o = oracle_inputs(inp)
    want = oracle.forward_train(o["x"], o["w"], o["gamma"], o["beta"], o["running_mean"], o["running_var"],
                                spec.momentum, spec.eps, spec.stride, spec.pad)
    sd = np.sqrt(want["var"])
    stat_close(to_np(fo[0]["saved_mean"]), want["mean"], sd, "saved_mean vs oracle")
    rel_close(to_np(fo[0]["saved_inv_var"]), want["inv_std"], "saved_inv_var vs oracle")
    stat_close(to_np(rms[0]), want["running_mean"], spec.momentum * sd, "running_mean vs oracle")
    rel_close(to_np(rvs[0]), want["running_var"], "running_var vs oracle")
    stat_close(to_np(fo[0]["saved_mean"]), to_np(ref["saved_mean"]), sd, "saved_mean vs one step")
    rel_close(to_np(fo[0]["saved_inv_var"]), to_np(ref["saved_inv_var"]), "saved_inv_var vs one step")

    # each rank's y and dx are its share of the whole batch's; dW summed over ranks is the whole's
    y = torch.cat([fo[0]["y"], fo[1]["y"]])
    max_err_ok(to_np(y), to_np(ref["y"]), "y vs one step")
    max_err_ok(to_np(y), want["y"], "y vs oracle")
    for k in ("dgamma", "dbeta"):
        scale = np.abs(to_np(rb[k])).max()
        assert np.allclose(to_np(bo[0][k]), to_np(rb[k]), rtol=1e-3, atol=1e-3 * scale), k
    max_err_ok(to_np(bo[0]["dw"] + bo[1]["dw"]), to_np(rb["dw"]), "dw (summed over ranks) vs one step")
    if need_dx:
        max_err_ok(to_np(torch.cat([bo[0]["dx"], bo[1]["dx"]])), to_np(rb["dx"]), "dx vs one step")
