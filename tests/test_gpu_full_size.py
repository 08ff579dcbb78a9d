"""GPU parity at the full benchmark workloads (the N=256 56x56 64->64 layer, the N=256 224x224
3->64 7x7 stride-2 first layer, and the N=64 112x112 128->128 bf16 layer), on the benchmark's
seeded inputs and in the launch configuration it times: training forward with z kept and the
bit-packed ReLU mask, then the backward from them (no dx for the first layer).

The oracle computes the forward in full: the 7-loop convolution over every output pixel, the
two-pass batch statistics, and the normalise/affine/ReLU step.  z, y and the mask are compared
element by element (in chunks of images, to bound host memory), the statistics and the running
statistics channel by channel, and dgamma/dbeta from the oracle's full BN backward.  The two
backward convolutions are compared in full: every element of dx and of dW against the
oracle's 7-loop data and weight gradients of its own dz.  dgamma's error is also printed
before the allowances are added.  The 128->128 layer also checks the folded inference path
(fold in full, y at sampled output pixels).  Tolerances and the mask-ambiguity allowance are
those of tests/parity.py.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
from conv_batchnorm_relu_gb300 import cbr
from conv_batchnorm_relu_gb300.inputs import CONFIGS, make_inputs, seed_for
from parity import (ATOL, MASK_MARGIN, RTOL_MAX, UNIT_ROUNDOFF, mask_slack_core, max_err_ok,
                    max_err_ok_slack, rel_close, scaled_error, stat_close, stat_close_slack)

pytestmark = pytest.mark.gpu

CHUNK_ELEMS = 1 << 24     # output elements per comparison chunk


def host_bytes_available() -> int:
    """MemAvailable, capped by the cgroup limit when one is set."""
    avail = None
    with open("/proc/meminfo") as f:
        for line in f:
            if line.startswith("MemAvailable:"):
                avail = int(line.split()[1]) * 1024
    for p in ("/sys/fs/cgroup/memory.max", "/sys/fs/cgroup/memory/memory.limit_in_bytes"):
        try:
            with open(p) as f:
                v = f.read().strip()
            if v != "max":
                lim = int(v)
                try:
                    with open(p.replace("memory.max", "memory.current").replace(
                            "memory.limit_in_bytes", "memory.usage_in_bytes")) as f:
                        lim -= int(f.read().strip())
                except OSError:
                    pass
                avail = lim if avail is None else min(avail, lim)
        except (OSError, ValueError):
            pass
    return avail if avail is not None else 0


def host_bytes_needed(spec) -> int:
    """Peak fp64 host memory of this check: x, z, xhat, dy, dz and the full dx comparison, bytes."""
    out = spec.m * spec.c_out
    inp = spec.n * spec.h * spec.w * spec.c_in
    dx_bufs = 0 if spec.first_layer else 3 * inp  # dx: oracle, allowance, GPU result
    return 8 * (4 * out + 3 * inp + dx_bufs) + 2 * out + 8 * CHUNK_ELEMS * 8


def sample_pixels(rng, n, h, w, count):
    """(n, h, w) triples: the four corners and four edge midpoints of the first and last image,
    then uniform samples."""
    fixed = []
    for img in (0, n - 1):
        for hh, ww in ((0, 0), (0, w - 1), (h - 1, 0), (h - 1, w - 1),
                       (0, w // 2), (h - 1, w // 2), (h // 2, 0), (h // 2, w - 1)):
            fixed.append((img, hh, ww))
    rnd = np.stack([rng.integers(0, n, count), rng.integers(0, h, count),
                    rng.integers(0, w, count)], axis=1)
    return np.unique(np.concatenate([np.array(fixed), rnd]), axis=0).astype(np.int32)


class MaxErr:
    """Running max|got - ref| and max|ref| over chunks of one tensor."""

    def __init__(self, name):
        self.name, self.err, self.ref = name, 0.0, 0.0

    def add(self, got, ref):
        assert np.all(np.isfinite(got)), f"{self.name}: non-finite values"
        self.err = max(self.err, float(np.max(np.abs(got - ref))))
        self.ref = max(self.ref, float(np.max(np.abs(ref))))

    def check(self):
        bound = ATOL + RTOL_MAX * self.ref
        assert self.err <= bound, f"{self.name}: max|err| {self.err:.4g} > {bound:.4g}"


def check_full_size(spec, inp, gpu):
    """Compare one full-size GPU training step against the oracle.  ``gpu`` maps names to
    fp64 numpy results: per-channel vectors and dW whole; z, y (and the unpacked mask) through
    ``gpu["chunk"](name, n0, n1)``; dx through ``gpu["dx"]()``."""
    K, st, pad = spec.c_out, spec.stride, spec.pad
    x = inp["x"].double().numpy()
    w = inp["w"].double().numpy()
    gamma = inp["gamma"].double().numpy()
    beta = inp["beta"].double().numpy()

    # ---- forward: conv over every output pixel, batch statistics, running statistics
    z = oracle.conv2d_fwd(x, w, st, pad)
    mean, var = oracle.bn_batch_stats(z.reshape(-1, K))
    M = z.shape[0] * z.shape[1] * z.shape[2]
    rm, rv, inv = oracle.bn_finalize(mean, var, M, spec.eps, spec.momentum,
                                     inp["running_mean"].double().numpy(),
                                     inp["running_var"].double().numpy())
    sd = np.sqrt(var)
    stat_close(gpu["saved_mean"], mean, sd, "saved_mean")
    rel_close(gpu["saved_inv_var"], inv, "saved_inv_var")
    stat_close(gpu["running_mean"], rm, spec.momentum * sd, "running_mean")
    rel_close(gpu["running_var"], rv, "running_var")

    # ---- forward elementwise (per chunk of images) and the per-channel sums the backward
    # checks need, so that pre and y are never held in full
    dy = inp["dy"].double().numpy()
    xhat = np.empty_like(z)
    mask = np.empty(z.shape, dtype=np.uint8)
    amb_idx, amb_dy = [], []
    s1 = np.zeros(K)            # sum over ambiguous points of |dy|
    s2 = np.zeros(K)            # sum over ambiguous points of |dy * xhat|
    rss_g2, rss_b2, gz2 = np.zeros(K), np.zeros(K), np.zeros(K)
    xh_max = np.zeros(K)
    ez, ey = MaxErr("z"), MaxErr("y")
    per_img = z.shape[1] * z.shape[2] * K
    step = max(1, CHUNK_ELEMS // per_img)
    for n0 in range(0, spec.n, step):
        n1 = min(spec.n, n0 + step)
        zc = z[n0:n1]
        xh, pre, y, m = oracle.bn_relu_fwd(zc.reshape(-1, K), mean, var, gamma, beta, spec.eps)
        ez.add(gpu["chunk"]("z", n0, n1).reshape(-1, K), zc.reshape(-1, K))
        ey.add(gpu["chunk"]("y", n0, n1).reshape(-1, K), y)
        decided = np.abs(pre) > MASK_MARGIN
        got_m = gpu["chunk"]("mask", n0, n1).reshape(-1, K)
        bad = int(np.count_nonzero(got_m[decided] != (pre[decided] > 0)))
        assert bad == 0, f"mask: {bad} decided positions differ in images {n0}..{n1 - 1}"
        xhat[n0:n1] = xh.reshape(zc.shape)
        mask[n0:n1] = m.reshape(zc.shape)
        dyc = dy[n0:n1].reshape(-1, K)
        g = dyc * (m > 0)
        rss_g2 += ((g * xh) ** 2).sum(0)
        rss_b2 += (g ** 2).sum(0)
        gz2 += ((g * zc.reshape(-1, K)) ** 2).sum(0)
        xh_max = np.maximum(xh_max, np.abs(xh).max(0))
        amb = ~decided
        s1 += np.where(amb, np.abs(dyc), 0.0).sum(0)
        s2 += np.where(amb, np.abs(dyc * xh), 0.0).sum(0)
        rows, ks = np.nonzero(amb)
        q_ = z.shape[2]
        pq = z.shape[1] * q_
        amb_idx.append(np.stack([n0 + rows // pq, (rows % pq) // q_, rows % q_, ks], axis=1))
        amb_dy.append(dyc[rows, ks])
        del xh, pre, y, m, g, got_m
    ez.check()
    ey.check()
    del z

    # ---- BN backward in full (oracle), dgamma / dbeta
    dz, dgamma, dbeta = oracle.bn_relu_bwd(dy.reshape(-1, K), mask.reshape(-1, K),
                                           xhat.reshape(-1, K), var, gamma, spec.eps)
    del xhat, mask, dy
    dz = dz.reshape(spec.n, spec.p, spec.q, K)
    idx = np.concatenate(amb_idx)
    a = gamma * inv
    vals = np.abs(a[idx[:, 3]] * np.concatenate(amb_dy))
    u = a * (s1 + xh_max * s2) / M
    u_rounding = UNIT_ROUNDOFF[spec.dtype]
    db_ratio = stat_close_slack(gpu["dbeta"], dbeta, np.sqrt(rss_b2), s1, "dbeta")
    dg_ratio = stat_close_slack(gpu["dgamma"], dgamma, np.sqrt(rss_g2), s2, "dgamma",
                                extra=4.0 * (u_rounding / np.sqrt(3.0)) * inv * np.sqrt(gz2))
    # the bare 1e-3 criterion, before the mask and storage-rounding allowances, reported beside
    db_bare = scaled_error(gpu["dbeta"], dbeta, np.sqrt(rss_b2))
    dg_bare = scaled_error(gpu["dgamma"], dgamma, np.sqrt(rss_g2))
    print(f"\n{spec.name}: dgamma unwidened error {dg_bare:.3g} (of the 1e-3 bound: {dg_bare / 1e-3:.2f}x), "
          f"error / widened tolerance {dg_ratio:.3g}; dbeta unwidened {db_bare:.3g}, ratio {db_ratio:.3g}")

    # ---- dW and dx in full (oracle 7-loop convolutions over every output)
    need_dx = not spec.first_layer
    sl = mask_slack_core(idx, vals, u, x, w, st, pad, need_dx=need_dx)
    dw_ref = oracle.conv2d_wgrad(dz, x, (spec.r, spec.s), st, pad)
    err_dw = max_err_ok_slack(gpu["dw"], dw_ref, sl["dw"], "dw")
    err_dx = None
    if need_dx:
        dx_ref = oracle.conv2d_dgrad(dz, w, (spec.h, spec.w), st, pad)
        err_dx = max_err_ok_slack(gpu["dx"](), dx_ref, sl["dx"], "dx")
    return dict(ambiguous=int(idx.shape[0]), err_dw=err_dw, err_dx=err_dx,
                dgamma_unwidened=dg_bare, dbeta_unwidened=db_bare,
                dgamma_ratio=dg_ratio, dbeta_ratio=db_ratio)


def _unpack_chunk(words: torch.Tensor, e0: int, e1: int) -> np.ndarray:
    """Mask bits of NHWC elements [e0, e1) (e0, e1 multiples of 32) from the packed words."""
    b = words[e0 // 32:e1 // 32].cpu().numpy().view(np.uint8)
    return np.unpackbits(b, bitorder="little").astype(bool)


def run_full_step(spec):
    """One training step through the C ABI in the benchmark's launch configuration."""
    inp = make_inputs(spec, seed_for_spec(spec))
    layer = cbr.Layer.from_spec(spec)
    g = {k: v.cuda() for k, v in inp.items()}
    fwd_ws, bwd_ws = cbr.workspace_size(layer)
    ws_f, ws_b = cbr.new_workspace(fwd_ws), cbr.new_workspace(bwd_ws)
    need_dx = not spec.first_layer
    out = cbr.forward_train(layer, g["x"], g["w"], g["gamma"], g["beta"], g["running_mean"],
                            g["running_var"], spec.momentum, spec.eps, ws=ws_f, save_z=True)
    bwd = cbr.backward(layer, g["dy"], g["x"], g["w"], out["mask"], cbr.CBR_MASK_BITS, out["z"],
                       g["gamma"], out["saved_mean"], out["saved_inv_var"], ws=ws_b,
                       need_dx=need_dx)
    cbr.stream_status()
    del ws_f, ws_b
    vec = lambda t: t.detach().double().cpu().numpy()
    per_img = spec.p * spec.q * spec.c_out

    def chunk(name, n0, n1):
        if name == "mask":
            return _unpack_chunk(out["mask"], n0 * per_img, n1 * per_img)
        return out[name][n0:n1].double().cpu().numpy()

    def dx_all():
        return bwd["dx"].double().cpu().numpy()

    res = dict(saved_mean=vec(out["saved_mean"]), saved_inv_var=vec(out["saved_inv_var"]),
               running_mean=vec(g["running_mean"]), running_var=vec(g["running_var"]),
               dgamma=vec(bwd["dgamma"]), dbeta=vec(bwd["dbeta"]), dw=vec(bwd["dw"]),
               chunk=chunk, dx=dx_all)
    return inp, g, res


def seed_for_spec(spec) -> int:
    for i, c in CONFIGS.items():
        if c == spec:
            return seed_for(i)
    raise KeyError(spec.name)


@pytest.mark.parametrize("cfg", [3, 4, 5])
def test_full_size_training_step(cfg):
    spec = CONFIGS[cfg]
    need = host_bytes_needed(spec)
    have = host_bytes_available()
    if have < 2 * need:
        pytest.skip(f"host memory: {have / 2**30:.1f} GiB available, {2 * need / 2**30:.1f} GiB wanted")
    inp, g, res = run_full_step(spec)
    info = check_full_size(spec, inp, res)
    assert info["err_dw"] is not None and (spec.first_layer or info["err_dx"] is not None)


def test_full_size_folded_inference():
    """The 128->128 bf16 layer's inference path: fold in full, y at sampled output pixels."""
    spec = CONFIGS[5]
    inp = make_inputs(spec, seed_for(5), with_dy=False)
    gen = torch.Generator().manual_seed(seed_for(5) + 7)
    rm = torch.randn(spec.c_out, generator=gen) * 0.2
    rv = torch.rand(spec.c_out, generator=gen) + 0.5
    layer = cbr.Layer.from_spec(spec)
    g = {k: v.cuda() for k, v in inp.items()}
    w_fold, b_fold = cbr.fold_bn(layer, g["w"], g["gamma"], g["beta"], rm.cuda(), rv.cuda(), spec.eps)
    y = cbr.forward_infer(layer, g["x"], w_fold, b_fold)
    cbr.stream_status()
    w_ref, b_ref = oracle.fold(inp["w"].double().numpy(), inp["gamma"].double().numpy(),
                               inp["beta"].double().numpy(), rm.double().numpy(),
                               rv.double().numpy(), spec.eps)
    max_err_ok(w_fold.double().cpu().numpy(), w_ref, "w_fold")
    max_err_ok(b_fold.double().cpu().numpy(), b_ref, "b_fold")
    rng = np.random.default_rng(seed_for(5) + 1)
    pix = sample_pixels(rng, spec.n, spec.p, spec.q, 512)
    z_at = oracle.conv2d_fwd_at(inp["x"].double().numpy(), w_ref, spec.stride, spec.pad, pix)
    y_ref = oracle.bias_relu(z_at, b_ref)
    t = torch.as_tensor(pix, dtype=torch.long).cuda()
    y_got = y[t[:, 0], t[:, 1], t[:, 2]].double().cpu().numpy()
    max_err_ok(y_got, y_ref, "y_infer (sampled pixels)")
