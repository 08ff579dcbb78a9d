"""Parity helpers: the tolerances every GPU-vs-oracle comparison uses.

Tolerances (stated for this operator):
  * y, z, dx, dW (fp16/bf16 tensors and the fp32 dW): max|err| <= 2e-2 + 1e-2 * max|ref|
    (the absolute + relative-to-max form of the TileLang page's allclose check);
  * saved_mean, running_mean, dbeta: |err_c| <= 1e-3 * max(|ref_c|, scale_c) per channel, where
    scale_c is the channel's standard deviation for means and max_c |ref| for dbeta;
  * saved_inv_var, running_var, dgamma: relative error <= 1e-3 (dgamma against
    max(|ref_c|, 1e-3 * max|ref|));
  * ReLU mask: exact wherever |pre-activation| > 1e-3.
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


def mask_ok(got_bits: np.ndarray, pre_ref: np.ndarray, name: str = "mask") -> int:
    pre = pre_ref.reshape(-1)
    decided = np.abs(pre) > MASK_MARGIN
    bad = int(np.count_nonzero(got_bits[decided] != (pre[decided] > 0)))
    assert bad == 0, f"{name}: {bad} decided positions differ"
    return bad


def oracle_inputs(inp: dict) -> dict:
    """fp64 numpy copies of the (already rounded) inputs."""
    return {k: v.double().numpy() for k, v in inp.items()}
