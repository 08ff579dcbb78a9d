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


def test_sampled_slack_equals_full_slack_at_the_samples():
    """mask_slack_core evaluated only at listed pixels and taps (the full-size tests' form)
    gives the full allowance's values there."""
    from parity import mask_slack_core
    spec = CONFIGS[1]
    o, ref, rb = _case(spec, 1240)
    full = mask_slack(spec, o, ref, rb, margin=0.2)  # a wide margin so many points are ambiguous
    pre = ref["pre"]
    amb = np.abs(pre) <= 0.2
    K = pre.shape[-1]
    a = o["gamma"] * ref["inv_std"]
    idx = np.argwhere(amb)
    vals = np.abs(a[idx[:, 3]] * o["dy"][amb])
    M = pre.shape[0] * pre.shape[1] * pre.shape[2]
    s1 = np.where(amb, np.abs(o["dy"]), 0.0).reshape(-1, K).sum(0)
    s2 = np.where(amb, np.abs(o["dy"] * ref["xhat"]), 0.0).reshape(-1, K).sum(0)
    u = a * (s1 + np.abs(ref["xhat"]).reshape(-1, K).max(0) * s2) / M
    pix = np.array([(0, 0, 0), (1, 7, 7), (0, 3, 5), (1, 0, 7)])
    taps = np.array([(0, 0, 0), (15, 2, 2), (7, 1, 0)])
    sl = mask_slack_core(idx, vals, u, o["x"], o["w"], spec.stride, spec.pad, taps=taps, pixels=pix)
    assert full["count"] > 0
    np.testing.assert_allclose(sl["dx"], full["dx"][pix[:, 0], pix[:, 1], pix[:, 2]], rtol=1e-12, atol=0)
    np.testing.assert_allclose(sl["dw"], full["dw"][taps[:, 0], taps[:, 1], taps[:, 2]], rtol=1e-12, atol=0)
    only_taps = mask_slack_core(idx, vals, u, o["x"], o["w"], spec.stride, spec.pad, taps=taps)
    assert only_taps["dx"] is None
