"""CPU checks of the parity helpers: the ambiguous-mask allowance covers every valid choice of
mask at |pre| <= margin, and does not cover a flip at a decided position."""
import numpy as np

import oracle
from conv_batchnorm_relu_gb300.inputs import CONFIGS, make_inputs
from parity import mask_slack, oracle_inputs


def _backward_with_mask(o, ref, mask, spec):
    K = ref["z"].shape[-1]
    dz, dg, db = oracle.bn_relu_bwd(o["dy"].reshape(-1, K), mask.reshape(-1, K).astype(np.uint8),
                                    ref["xhat"].reshape(-1, K), ref["var"], o["gamma"], spec.eps)
    dz = dz.reshape(ref["z"].shape)
    dx = oracle.conv2d_dgrad(dz, o["w"], (spec.h, spec.w), spec.stride, spec.pad)
    dw = oracle.conv2d_wgrad(dz, o["x"], (spec.r, spec.s), spec.stride, spec.pad)
    return dict(dx=dx, dw=dw, dgamma=dg, dbeta=db)


def _case(spec, seed):
    o = oracle_inputs(make_inputs(spec, seed))
    ref = oracle.forward_train(o["x"], o["w"], o["gamma"], o["beta"], o["running_mean"],
                               o["running_var"], spec.momentum, spec.eps, spec.stride, spec.pad)
    rb = oracle.backward(o["dy"], o["x"], o["w"], ref, o["gamma"], spec.eps, spec.stride, spec.pad)
    return o, ref, rb


def test_mask_slack_covers_ambiguous_flips():
    spec = CONFIGS[1]
    o, ref, rb = _case(spec, 1235)
    margin = 0.15  # wide margin: many ambiguous positions
    sl = mask_slack(spec, o, ref, rb, margin=margin)
    assert sl["count"] > 20
    rng = np.random.default_rng(0)
    amb = np.abs(ref["pre"]) <= margin
    for trial in range(5):
        flip = amb & (rng.random(amb.shape) < 0.5)
        m2 = np.where(flip, 1 - ref["mask"], ref["mask"])
        alt = _backward_with_mask(o, ref, m2, spec)
        for k in ("dx", "dw", "dgamma", "dbeta"):
            assert np.all(np.abs(alt[k] - rb[k]) <= sl[k] * (1 + 1e-9) + 1e-12), (trial, k)


def test_mask_slack_does_not_cover_decided_flips():
    spec = CONFIGS[1].with_(n=4, h=12, w=12)
    o, ref, rb = _case(spec, 77)
    sl = mask_slack(spec, o, ref, rb)  # the real margin, 1e-3
    decided = np.argwhere((np.abs(ref["pre"]) > 0.3) & (np.abs(o["dy"]) > 0.5))
    rng = np.random.default_rng(1)
    for j in rng.choice(len(decided), 5, replace=False):
        i = tuple(decided[j])
        m3 = ref["mask"].copy()
        m3[i] = 1 - m3[i]
        alt = _backward_with_mask(o, ref, m3, spec)
        assert np.any(np.abs(alt["dx"] - rb["dx"]) > sl["dx"] + 2e-2), i
        assert np.any(np.abs(alt["dw"] - rb["dw"]) > sl["dw"] + 2e-2), i
