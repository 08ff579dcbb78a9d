"""Pins for the CPU oracle: each test checks the oracle against something other than itself.

The pins are:
* closed forms: the CBR page's feature-map size, running statistics, x-hat moments;
* exact identities of BN backward: sum(dz) = 0 and sum(dz*xhat) = gamma*inv*dgamma*eps/(var+eps);
* special cases that reduce to a textbook routine: 1x1 conv = GEMM, delta filters = shifts;
* central finite differences on tiny inputs for every gradient;
* BN folding equals conv -> BN(running) -> ReLU;
* a library cross-check against PyTorch CPU float64 (conv2d + batch_norm + autograd).

The mutation tests at the end plant plausible mistakes in oracle outputs, on the CPU, and check
that some pin rejects each one.
"""
import json
import os

import numpy as np
import pytest
import torch

import oracle
from conv_batchnorm_relu_gb300.inputs import CONFIGS, CBRSpec, make_inputs

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _rng(seed):
    return np.random.default_rng(seed)


def _rand_case(seed, N, H, W, C, K, R, S):
    g = _rng(seed)
    x = g.standard_normal((N, H, W, C))
    w = g.standard_normal((K, R, S, C)) * (2.0 / (C * R * S)) ** 0.5
    gamma = g.uniform(0.5, 1.5, K)
    beta = g.normal(0.0, 0.1, K)
    return x, w, gamma, beta


# ------------------------------------------------------------------- page numbers
def test_feature_map_size_from_cbr_page():
    """CBR page section 1 works the size of one fp16 N=256, 56x56, C=64 feature map:
    about 102 MB; unfused, about 200 MB of extra traffic per layer (one write + one read)."""
    with open(os.path.join(GOLDEN, "cbr_page_numbers.json")) as f:
        g = json.load(f)
    spec = CONFIGS[3]
    nbytes = spec.n * spec.p * spec.q * spec.c_out * 2
    assert nbytes == g["feature_map_bytes"]
    assert abs(nbytes / 1e6 - g["feature_map_mb_printed"]) < 1.0
    assert abs(2 * nbytes / 1e6 - g["extra_traffic_mb_printed"]) < 6.0
    assert spec.m == g["n_ac"]


# ------------------------------------------------------------------- convolution
@pytest.mark.parametrize("stride,pad", [(1, 0), (2, 0)])
def test_conv_1x1_is_gemm(stride, pad):
    x, w, _, _ = _rand_case(1, 2, 5, 6, 7, 9, 1, 1)
    z = oracle.conv2d_fwd(x, w, stride, pad)
    xs = x[:, ::stride, ::stride, :]
    ref = xs.reshape(-1, 7) @ w.reshape(9, 7).T
    np.testing.assert_allclose(z.reshape(-1, 9), ref, rtol=1e-13, atol=1e-13)


@pytest.mark.parametrize("R,S,stride,pad", [(3, 3, 1, 1), (7, 7, 2, 3), (3, 3, 2, 1), (5, 3, 1, 2)])
def test_conv_delta_filter_is_shift(R, S, stride, pad):
    """A filter with a single one at (k0,r0,s0,c0) reproduces the input sampled at
    (p*stride-pad+r0, q*stride-pad+s0): cross-correlation, no flip, zero padding."""
    N, H, W, C, K = 2, 9, 8, 3, 2
    x = _rng(2).standard_normal((N, H, W, C))
    P = (H + 2 * pad - R) // stride + 1
    Q = (W + 2 * pad - S) // stride + 1
    for r0 in range(R):
        for s0 in range(S):
            w = np.zeros((K, R, S, C))
            w[1, r0, s0, 2] = 1.0
            z = oracle.conv2d_fwd(x, w, stride, pad)
            assert z.shape == (N, P, Q, K)
            assert np.all(z[..., 0] == 0.0)
            for p in range(P):
                for q in range(Q):
                    h, ww = p * stride - pad + r0, q * stride - pad + s0
                    exp = x[:, h, ww, 2] if (0 <= h < H and 0 <= ww < W) else np.zeros(N)
                    assert np.array_equal(z[:, p, q, 1], exp)


# ------------------------------------------------------------------- BN forward
def test_xhat_moments():
    """Per channel over N*P*Q: mean(xhat) = 0 and mean(xhat^2) = var/(var+eps) exactly,
    i.e. the normalised output has mean ~0 and variance ~1 before the affine."""
    x, w, gamma, beta = _rand_case(3, 3, 7, 6, 5, 4, 3, 3)
    f = oracle.forward_train(x, w, gamma, beta, np.zeros(4), np.ones(4), 0.1, 1e-5, 1, 1)
    xh = f["xhat"].reshape(-1, 4)
    assert np.max(np.abs(xh.mean(0))) < 1e-12
    np.testing.assert_allclose((xh ** 2).mean(0), f["var"] / (f["var"] + 1e-5), rtol=1e-12)


def test_running_stats_closed_form():
    """1x1 identity conv so z = x; channel c alternates (c+0.5) -/+ 1, so the batch mean is
    c+0.5 and the biased variance 1.  CBR page section 4.2 update with momentum = weight of
    the new batch, unbiased variance for the running estimate."""
    C, N, H, W = 4, 2, 3, 4
    M = N * H * W
    x = np.empty((N, H, W, C))
    sign = np.where(np.arange(M) % 2 == 0, -1.0, 1.0).reshape(N, H, W)
    for c in range(C):
        x[..., c] = c + 0.5 + sign
    w = np.eye(C).reshape(C, 1, 1, C)
    rm0, rv0 = np.array([0.3, -0.2, 1.0, 0.0]), np.array([1.0, 2.0, 0.5, 1.5])
    f = oracle.forward_train(x, w, np.ones(C), np.zeros(C), rm0, rv0, 0.1, 1e-5, 1, 0)
    np.testing.assert_allclose(f["mean"], np.arange(C) + 0.5, rtol=1e-15)
    np.testing.assert_allclose(f["var"], np.ones(C), rtol=1e-14)
    np.testing.assert_allclose(f["running_mean"], 0.9 * rm0 + 0.1 * (np.arange(C) + 0.5), rtol=1e-15)
    np.testing.assert_allclose(f["running_var"], 0.9 * rv0 + 0.1 * M / (M - 1), rtol=1e-15)
    np.testing.assert_allclose(f["inv_std"], 1.0 / np.sqrt(1.0 + 1e-5), rtol=1e-15)


def test_mask_is_strictly_greater_than_zero():
    """CMP_GT: a pre-activation of exactly 0 gives mask 0, y 0 and no gradient."""
    C = 2
    vals = np.array([-1.0, 0.0, 1.0] * 4)
    x = np.stack([vals, vals], axis=-1).reshape(1, 3, 4, C)
    w = np.eye(C).reshape(C, 1, 1, C)
    f = oracle.forward_train(x, w, np.ones(C), np.zeros(C), np.zeros(C), np.ones(C), 0.1, 1e-5, 1, 0)
    zero_pos = f["pre"] == 0.0
    assert zero_pos.sum() == 8
    assert np.all(f["mask"][zero_pos] == 0) and np.all(f["y"][zero_pos] == 0.0)
    dy = np.ones_like(f["y"])
    b = oracle.backward(dy, x, w, f, np.ones(C), 1e-5, 1, 0)
    # with dy = 1 on the masked-on positions only: dbeta = count(pre > 0)
    np.testing.assert_allclose(b["dbeta"], [4.0, 4.0])


# ------------------------------------------------------------------- BN backward identities
def test_bn_backward_identities():
    """sum(dz) = 0 and sum(dz*xhat) = gamma*inv_std*dgamma*eps/(var+eps), per channel."""
    x, w, gamma, beta = _rand_case(4, 2, 6, 6, 4, 5, 3, 3)
    eps = 1e-5
    f = oracle.forward_train(x, w, gamma, beta, np.zeros(5), np.ones(5), 0.1, eps, 1, 1)
    dy = _rng(5).standard_normal(f["y"].shape)
    b = oracle.backward(dy, x, w, f, gamma, eps, 1, 1)
    dz = b["dz"].reshape(-1, 5)
    xh = f["xhat"].reshape(-1, 5)
    scale = np.abs(dz).sum(0)
    assert np.max(np.abs(dz.sum(0)) / scale) < 1e-13
    exp = gamma * f["inv_std"] * b["dgamma"] * eps / (f["var"] + eps)
    np.testing.assert_allclose((dz * xh).sum(0), exp, rtol=1e-6, atol=1e-13 * scale.max())


# ------------------------------------------------------------------- finite differences
def _loss(x, w, gamma, beta, dy, stride, pad, eps):
    f = oracle.forward_train(x, w, gamma, beta, np.zeros(len(gamma)), np.ones(len(gamma)), 0.1,
                             eps, stride, pad)
    return float((dy * f["y"]).sum()), f["pre"]


def _fd_check(x, w, gamma, beta, stride, pad, seed, max_coords=None, h=1e-6):
    eps = 1e-5
    f = oracle.forward_train(x, w, gamma, beta, np.zeros(len(gamma)), np.ones(len(gamma)), 0.1,
                             eps, stride, pad)
    dy = _rng(seed).standard_normal(f["y"].shape)
    b = oracle.backward(dy, x, w, f, gamma, eps, stride, pad)
    analytic = {"x": b["dx"], "w": b["dw"], "gamma": b["dgamma"], "beta": b["dbeta"]}
    params = {"x": x, "w": w, "gamma": gamma, "beta": beta}
    g = _rng(seed + 1)
    checked, worst = 0, 0.0
    for name, arr in params.items():
        idxs = list(np.ndindex(arr.shape))
        if max_coords and len(idxs) > max_coords:
            idxs = [idxs[i] for i in g.choice(len(idxs), max_coords, replace=False)]
        for idx in idxs:
            vals = {}
            masks = []
            for sgn in (1, -1):
                p2 = {k: v.copy() for k, v in params.items()}
                p2[name][idx] += sgn * h
                L, pre = _loss(p2["x"], p2["w"], p2["gamma"], p2["beta"], dy, stride, pad, eps)
                vals[sgn] = L
                masks.append(pre > 0)
            if not (np.array_equal(masks[0], f["mask"] > 0) and np.array_equal(masks[1], f["mask"] > 0)):
                continue  # the +-h step crosses a ReLU kink
            fd = (vals[1] - vals[-1]) / (2 * h)
            an = analytic[name][idx]
            err = abs(fd - an) / (1e-1 + abs(an))
            worst = max(worst, err)
            checked += 1
    return checked, worst


@pytest.mark.parametrize("shape", [
    dict(N=2, H=4, W=4, C=2, K=3, R=3, S=3, stride=1, pad=1),
    dict(N=1, H=7, W=6, C=3, K=4, R=3, S=3, stride=2, pad=1),
    dict(N=2, H=9, W=9, C=3, K=2, R=7, S=7, stride=2, pad=3),
])
def test_finite_differences_small(shape):
    x, w, gamma, beta = _rand_case(6, shape["N"], shape["H"], shape["W"], shape["C"], shape["K"],
                                   shape["R"], shape["S"])
    checked, worst = _fd_check(x, w, gamma, beta, shape["stride"], shape["pad"], seed=7)
    assert checked > 0.8 * (x.size + w.size + gamma.size + beta.size)
    assert worst < 1e-6, worst


def test_finite_differences_config1():
    spec = CONFIGS[1]
    inp = make_inputs(spec, 1235)
    x = inp["x"].double().numpy()
    w = inp["w"].double().numpy()
    checked, worst = _fd_check(x, w, inp["gamma"].double().numpy(), inp["beta"].double().numpy(),
                               1, 1, seed=8, max_coords=40)
    assert checked > 100
    assert worst < 1e-6, worst


# ------------------------------------------------------------------- inference fold
def test_fold_equals_conv_bn_running_relu():
    """conv(x, W_fold) + b_fold -> ReLU equals conv -> BN(running stats) -> ReLU."""
    x, w, gamma, beta = _rand_case(9, 2, 6, 5, 4, 6, 3, 3)
    g = _rng(10)
    rm, rv = g.normal(0, 0.5, 6), g.uniform(0.5, 2.0, 6)
    bias = g.normal(0, 0.3, 6)
    for cb in (None, bias):
        inf = oracle.forward_infer(x, w, gamma, beta, rm, rv, 1e-5, 1, 1, conv_bias=cb)
        z = oracle.conv2d_fwd(x, w, 1, 1).reshape(-1, 6)
        if cb is not None:
            z = z + cb
        pre = oracle.bn_infer(z, rm, rv, gamma, beta, 1e-5)
        ref = np.maximum(pre, 0.0).reshape(inf["y"].shape)
        np.testing.assert_allclose(inf["y"], ref, rtol=1e-12, atol=1e-12 * np.abs(ref).max())


def test_scale_invariance_of_train_forward():
    """BN removes the scale of W: y(x, a*W) = y(x, W) for a > 0 when eps = 0."""
    x, w, gamma, beta = _rand_case(11, 2, 5, 5, 3, 4, 3, 3)
    f1 = oracle.forward_train(x, w, gamma, beta, np.zeros(4), np.ones(4), 0.1, 0.0, 1, 1)
    f2 = oracle.forward_train(x, 3.7 * w, gamma, beta, np.zeros(4), np.ones(4), 0.1, 0.0, 1, 1)
    np.testing.assert_allclose(f1["y"], f2["y"], rtol=1e-11, atol=1e-12)


# ------------------------------------------------------------------- library cross-check
def _torch_reference(x, w, gamma, beta, dy, stride, pad, eps, momentum, rm0, rv0):
    xt = torch.tensor(x).permute(0, 3, 1, 2).contiguous().requires_grad_(True)
    wt = torch.tensor(w).permute(0, 3, 1, 2).contiguous().requires_grad_(True)
    gt = torch.tensor(gamma).requires_grad_(True)
    bt = torch.tensor(beta).requires_grad_(True)
    rm, rv = torch.tensor(rm0).clone(), torch.tensor(rv0).clone()
    z = torch.nn.functional.conv2d(xt, wt, stride=stride, padding=pad)
    y = torch.relu(torch.nn.functional.batch_norm(z, rm, rv, gt, bt, training=True,
                                                  momentum=momentum, eps=eps))
    dyt = torch.tensor(dy).permute(0, 3, 1, 2)
    (y * dyt).sum().backward()
    nhwc = lambda t: t.detach().permute(0, 2, 3, 1).numpy()
    return dict(y=nhwc(y), dx=nhwc(xt.grad), dw=wt.grad.permute(0, 2, 3, 1).numpy(),
                dgamma=gt.grad.numpy(), dbeta=bt.grad.numpy(), rm=rm.numpy(), rv=rv.numpy())


@pytest.mark.parametrize("shape", [
    dict(N=2, H=8, W=8, C=8, K=16, R=3, S=3, stride=1, pad=1),
    dict(N=2, H=11, W=13, C=3, K=8, R=7, S=7, stride=2, pad=3),
    dict(N=3, H=9, W=7, C=16, K=8, R=3, S=3, stride=1, pad=1),
])
def test_against_torch_cpu_float64(shape):
    x, w, gamma, beta = _rand_case(12, shape["N"], shape["H"], shape["W"], shape["C"], shape["K"],
                                   shape["R"], shape["S"])
    K = shape["K"]
    g = _rng(13)
    rm0, rv0 = g.normal(0, 0.1, K), g.uniform(0.5, 1.5, K)
    f = oracle.forward_train(x, w, gamma, beta, rm0, rv0, 0.1, 1e-5, shape["stride"], shape["pad"])
    dy = g.standard_normal(f["y"].shape)
    b = oracle.backward(dy, x, w, f, gamma, 1e-5, shape["stride"], shape["pad"])
    t = _torch_reference(x, w, gamma, beta, dy, shape["stride"], shape["pad"], 1e-5, 0.1, rm0, rv0)
    for got, ref in [(f["y"], t["y"]), (b["dx"], t["dx"]), (b["dw"], t["dw"]),
                     (b["dgamma"], t["dgamma"]), (b["dbeta"], t["dbeta"]),
                     (f["running_mean"], t["rm"]), (f["running_var"], t["rv"])]:
        np.testing.assert_allclose(got, ref, rtol=1e-9, atol=1e-11 * max(1.0, np.abs(ref).max()))


def test_dgrad_at_matches_full_dgrad():
    x, w, gamma, beta = _rand_case(14, 2, 7, 9, 8, 16, 3, 3)
    dz = _rng(15).standard_normal((2, 7, 9, 16))
    full = oracle.conv2d_dgrad(dz, w, (7, 9), 1, 1)
    pix = [(0, 0, 0), (1, 6, 8), (0, 3, 4), (1, 0, 8)]
    at = oracle.conv2d_dgrad_at(dz, w, (7, 9), 1, 1, pix)
    for i, (n, h, ww) in enumerate(pix):
        assert np.array_equal(at[i], full[n, h, ww])


def test_fwd_at_and_wgrad_at_match_full_forms():
    """The sampled fprop and wgrad evaluate the same sums as the full forms (stride 2 with
    padding, so out-of-range taps and strided rows are exercised)."""
    x, w, gamma, beta = _rand_case(18, 2, 9, 11, 3, 8, 5, 5)
    full = oracle.conv2d_fwd(x, w, 2, 2)
    pix = [(0, 0, 0), (1, full.shape[1] - 1, full.shape[2] - 1), (0, 2, 3), (1, 0, full.shape[2] - 1)]
    at = oracle.conv2d_fwd_at(x, w, 2, 2, pix)
    for i, (n, p, q) in enumerate(pix):
        assert np.array_equal(at[i], full[n, p, q])
    dz = _rng(19).standard_normal(full.shape)
    dw = oracle.conv2d_wgrad(dz, x, (5, 5), 2, 2)
    taps = [(0, 0, 0), (7, 4, 4), (3, 2, 1), (5, 0, 4)]
    at = oracle.conv2d_wgrad_at(dz, x, (5, 5), 2, 2, taps)
    for i, (k, r, s_) in enumerate(taps):
        assert np.array_equal(at[i], dw[k, r, s_])


# ------------------------------------------------------------------- mutation tests
def test_pins_reject_planted_mistakes():
    """Plant plausible oracle mistakes on the CPU and check that a pin rejects each."""
    x, w, gamma, beta = _rand_case(16, 2, 5, 5, 3, 4, 3, 3)
    eps = 1e-5
    f = oracle.forward_train(x, w, gamma, beta, np.zeros(4), np.ones(4), 0.1, eps, 1, 1)
    dy = _rng(17).standard_normal(f["y"].shape)
    b = oracle.backward(dy, x, w, f, gamma, eps, 1, 1)
    t = _torch_reference(x, w, gamma, beta, dy, 1, 1, eps, 0.1, np.zeros(4), np.ones(4))
    rel = lambda a, r: np.max(np.abs(a - r)) / np.max(np.abs(r))
    # (a) gamma dropped from dz (the garbled form of the BN page's first dx formula)
    dz_nog = b["dz"] / gamma
    assert rel(oracle.conv2d_dgrad(dz_nog, w, (5, 5), 1, 1), t["dx"]) > 1e-2
    # (b) convolution instead of cross-correlation (flipped filter)
    z_flip = oracle.conv2d_fwd(x, w[:, ::-1, ::-1, :], 1, 1)
    assert rel(z_flip, oracle.conv2d_fwd(x, w, 1, 1)) > 1e-2
    # (c) biased variance in the running estimate
    M = f["z"].reshape(-1, 4).shape[0]
    assert abs((0.9 + 0.1 * f["var"][0]) - f["running_var"][0]) > 1e-3 / M
    # (d) dgamma sign or missing mask
    assert rel(-b["dgamma"], t["dgamma"]) > 1.0
    dz_nomask, dg_nomask, db_nomask = oracle.bn_relu_bwd(
        dy.reshape(-1, 4), np.ones_like(f["mask"]).reshape(-1, 4), f["xhat"].reshape(-1, 4),
        f["var"], gamma, eps)
    assert rel(db_nomask, t["dbeta"]) > 1e-2
    # (e) transposed wgrad (dW indexed [c,r,s,k] instead of [k,r,s,c]) on a square case
    xs, ws, gs, bs = _rand_case(18, 2, 5, 5, 4, 4, 3, 3)
    fs = oracle.forward_train(xs, ws, gs, bs, np.zeros(4), np.ones(4), 0.1, eps, 1, 1)
    dys = _rng(19).standard_normal(fs["y"].shape)
    bsq = oracle.backward(dys, xs, ws, fs, gs, eps, 1, 1)
    ts = _torch_reference(xs, ws, gs, bs, dys, 1, 1, eps, 0.1, np.zeros(4), np.ones(4))
    assert rel(bsq["dw"].transpose(3, 1, 2, 0), ts["dw"]) > 1e-2
