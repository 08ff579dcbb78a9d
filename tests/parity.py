"""Parity helpers: the tolerances every GPU-vs-oracle comparison uses.

Tolerances (stated for this operator):
  * y, z, dx, dW (fp16/bf16 tensors and the fp32 dW): max|err| <= 2e-2 + 1e-2 * max|ref|
    (the absolute + relative-to-max form of the TileLang page's allclose check);
  * saved_mean, running_mean: |err_c| <= 1e-3 * max(|ref_c|, sd_c) per channel (sd_c = the
    channel's batch standard deviation, times momentum for the running mean);
  * dgamma, dbeta (sums over M rows that may cancel): |err_c| <= 1e-3 * max(|ref_c|, rss_c),
    rss_c = sqrt(sum of the squared summed terms) -- g*xhat for dgamma, g for dbeta;
  * saved_inv_var, running_var: relative error <= 1e-3;
  * ReLU mask: exact wherever |pre-activation| > 1e-3.

Two derived allowances, both computed from oracle data only:
  * Ambiguous mask positions.  Where |pre| <= 1e-3 either mask value is a valid result (the
    GPU decides on the rounded z).  A different decision there changes dz by a*dy at that
    position and, through dbeta/dgamma, every dz of the channel by a tiny amount; `mask_slack`
    bounds the resulting change of dx, dW, dgamma and dbeta element by element, and the
    comparisons add it to their tolerance.
  * dgamma reads the stored z.  sum g*(z - mean)*inv_std over the fp16/bf16-rounded z carries
    the storage rounding: 4 standard deviations of that error, 4*(u/sqrt(3))*inv_std*
    sqrt(sum (g*z)^2) with unit roundoff u = 2^-11 (fp16) or 2^-8 (bf16), are added to
    dgamma's tolerance.
"""
from __future__ import annotations

import numpy as np
import torch

import oracle

ATOL, RTOL_MAX = 2e-2, 1e-2
STAT_RTOL = 1e-3
MASK_MARGIN = 1e-3


def to_np(t: torch.Tensor) -> np.ndarray:
    return t.detach().float().cpu().double().numpy()


def max_err_ok(got, ref, name: str) -> float:
    got, ref = np.asarray(got, dtype=np.float64), np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape, (name, got.shape, ref.shape)
    err = float(np.max(np.abs(got - ref))) if got.size else 0.0
    bound = ATOL + RTOL_MAX * (float(np.max(np.abs(ref))) if ref.size else 0.0)
    assert np.all(np.isfinite(got)), f"{name}: non-finite values"
    assert err <= bound, f"{name}: max|err| {err:.4g} > {bound:.4g}"
    return err


def stat_close(got, ref, scale, name: str) -> float:
    got, ref, scale = (np.asarray(a, dtype=np.float64) for a in (got, ref, scale))
    denom = np.maximum(np.abs(ref), scale)
    rel = np.abs(got - ref) / denom
    worst = float(rel.max())
    assert worst <= STAT_RTOL, f"{name}: worst scaled error {worst:.3g} > {STAT_RTOL}"
    return worst


def rel_close(got, ref, name: str, floor: float = 0.0) -> float:
    got, ref = np.asarray(got, dtype=np.float64), np.asarray(ref, dtype=np.float64)
    denom = np.maximum(np.abs(ref), floor)
    worst = float((np.abs(got - ref) / denom).max())
    assert worst <= STAT_RTOL, f"{name}: worst relative error {worst:.3g} > {STAT_RTOL}"
    return worst


def unpack_mask(words: torch.Tensor, total: int) -> np.ndarray:
    b = words.detach().cpu().numpy().view(np.uint8)
    return np.unpackbits(b, bitorder="little")[:total].astype(bool)


def mask_ok(got_bits: np.ndarray, pre_ref: np.ndarray, name: str = "mask", margin=MASK_MARGIN) -> int:
    """The mask agrees exactly wherever |pre| > margin (a scalar, or one value per element)."""
    pre = pre_ref.reshape(-1)
    decided = np.abs(pre) > np.broadcast_to(margin, pre_ref.shape).reshape(-1)
    bad = int(np.count_nonzero(got_bits[decided] != (pre[decided] > 0)))
    assert bad == 0, f"{name}: {bad} decided positions differ"
    return bad


def oracle_inputs(inp: dict) -> dict:
    """fp64 numpy copies of the (already rounded) inputs."""
    return {k: v.double().numpy() for k, v in inp.items()}


def grad_sum_scales(dy: np.ndarray, mask: np.ndarray, xhat: np.ndarray) -> tuple[np.ndarray, np.ndarray]:
    """Root-sum-square scales of the dgamma (g*xhat) and dbeta (g) sums, per channel."""
    c = dy.shape[-1]
    g = (dy * (mask > 0)).reshape(-1, c)
    xh = xhat.reshape(-1, c)
    return np.sqrt(((g * xh) ** 2).sum(0)), np.sqrt((g ** 2).sum(0))


UNIT_ROUNDOFF = {"f16": 2.0 ** -11, "bf16": 2.0 ** -8}


def mask_slack(spec, o: dict, ref: dict, rb: dict, margin=MASK_MARGIN) -> dict:
    """Element-wise bounds on how much the backward outputs may move when the ReLU mask is
    decided either way at the ambiguous positions |pre| <= margin (a scalar or one value per
    element; oracle data only)."""
    pre = ref["pre"]
    amb = np.abs(pre) <= margin
    N, P, Q, K = pre.shape
    a = np.asarray(o["gamma"]) * ref["inv_std"]                     # dz = a*g + ...
    dy = o["dy"]
    M = N * P * Q
    s1 = np.where(amb, np.abs(dy), 0.0).reshape(-1, K).sum(0)        # bound on |delta dbeta|
    s2 = np.where(amb, np.abs(dy * ref["xhat"]), 0.0).reshape(-1, K).sum(0)  # |delta dgamma|
    xh_max = np.abs(ref["xhat"]).reshape(-1, K).max(0)
    u = a * (s1 + xh_max * s2) / M                                   # |delta dz| everywhere, per channel
    idx = np.argwhere(amb)
    vals = np.abs(a[idx[:, 3]] * dy[amb])                            # |delta dz| at ambiguous points
    sl = mask_slack_core(idx, vals, u, o["x"], o["w"], spec.stride, spec.pad)
    return dict(dx=sl["dx"], dw=sl["dw"], dbeta=s1, dgamma=s2, count=int(amb.sum()))


def mask_slack_core(idx, vals, u, x, w, stride: int, pad: int, taps=None, pixels=None,
                    need_dx: bool | None = None) -> dict:
    """Propagate per-point dz changes through both backward convolutions.

    idx: (n, p, q, k) rows of the ambiguous output points; vals: the bound on |delta dz| at
    each; u[k]: the bound on |delta dz| at every point of channel k (through dbeta/dgamma).
    Returns the dx bound (all input pixels, or the listed (n, h, w) pixels; None when neither
    pixels nor a full dx is wanted, i.e. taps given without pixels, or need_dx is False) and the
    dW bound (all taps, or the listed (k, r, s) taps)."""
    _, H, W, C = x.shape
    K, R, S = w.shape[0], w.shape[1], w.shape[2]
    want_dx = (pixels is not None or taps is None) if need_dx is None else need_dx
    dx_sl = np.zeros_like(x) if want_dx else None
    dw_sl = np.zeros_like(w)
    aw, ax = np.abs(w), np.abs(x)
    for r in range(R):
        for s_ in range(S):
            h = idx[:, 1] * stride - pad + r
            ww = idx[:, 2] * stride - pad + s_
            ok = (h >= 0) & (h < H) & (ww >= 0) & (ww < W)
            n_, k_ = idx[ok, 0], idx[ok, 3]
            vv = vals[ok][:, None]
            if want_dx:
                np.add.at(dx_sl, (n_, h[ok], ww[ok]), vv * aw[k_, r, s_, :])
            np.add.at(dw_sl[:, r, s_, :], k_, vv * ax[n_, h[ok], ww[ok], :])
    # second order: every dz of channel k may move by u[k]
    if want_dx:
        dx_sl += (u[:, None] * aw.reshape(K, -1, C).sum(1)).sum(0)[None, None, None, :]
    dw_sl += u[:, None, None, None] * ax.reshape(-1, C).sum(0)[None, None, None, :]
    if pixels is not None:
        pixels = np.asarray(pixels)
        dx_sl = dx_sl[pixels[:, 0], pixels[:, 1], pixels[:, 2]]
    if taps is not None:
        taps = np.asarray(taps)
        dw_sl = dw_sl[taps[:, 0], taps[:, 1], taps[:, 2]]
    return dict(dx=dx_sl, dw=dw_sl)


def max_err_ok_slack(got, ref, slack, name: str) -> float:
    """max_err_ok with an element-wise allowance added to the bound; returns max|err|."""
    got, ref = np.asarray(got, dtype=np.float64), np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape, (name, got.shape, ref.shape)
    assert np.all(np.isfinite(got)), f"{name}: non-finite values"
    bound = ATOL + RTOL_MAX * float(np.max(np.abs(ref)))
    worst = float((np.abs(got - ref) - slack).max())
    assert worst <= bound, f"{name}: max(|err| - slack) {worst:.4g} > {bound:.4g}"
    return float(np.max(np.abs(got - ref)))


def stat_close_slack(got, ref, scale, slack, name: str, extra=None) -> float:
    """Per-channel |err| <= 1e-3*max(|ref|, scale) + slack (+ extra); returns the worst ratio of
    error to that widened tolerance."""
    got, ref, scale = (np.asarray(a, dtype=np.float64) for a in (got, ref, scale))
    tol = STAT_RTOL * np.maximum(np.abs(ref), scale) + slack
    if extra is not None:
        tol = tol + extra
    worst = float((np.abs(got - ref) / tol).max())
    assert worst <= 1.0, f"{name}: worst error / tolerance {worst:.3g} > 1"
    return worst


def scaled_error(got, ref, scale) -> float:
    """The unwidened per-channel error |err| / max(|ref|, scale), worst over channels (the bare
    1e-3 criterion, before any allowance is added)."""
    got, ref, scale = (np.asarray(a, dtype=np.float64) for a in (got, ref, scale))
    return float((np.abs(got - ref) / np.maximum(np.abs(ref), scale)).max())


def storage_rounding_margin(spec, ref: dict, o: dict) -> np.ndarray:
    """Per-element bound on how far the GPU's pre-activation, computed from z rounded to the
    storage dtype, may lie from the oracle's: gamma*inv_std*|z|*u (at least the 1e-3 margin).
    Negligible when z is centred near 0, it dominates when |mean/std| of z is large."""
    u = UNIT_ROUNDOFF[spec.dtype]
    a = np.asarray(o["gamma"]) * ref["inv_std"]
    return np.maximum(MASK_MARGIN, a * np.abs(ref["z"]) * u)


def dgamma_storage_rounding(spec, o: dict, ref: dict) -> np.ndarray:
    """4-sigma bound of dgamma's error from reading the stored (rounded) z."""
    u = UNIT_ROUNDOFF[spec.dtype]
    K = ref["z"].shape[-1]
    g = (o["dy"] * (ref["mask"] > 0)).reshape(-1, K)
    z = ref["z"].reshape(-1, K)
    return 4.0 * (u / np.sqrt(3.0)) * ref["inv_std"] * np.sqrt(((g * z) ** 2).sum(0))
