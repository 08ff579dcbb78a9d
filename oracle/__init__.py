"""Plain fp64 CPU oracle for the training-mode Conv -> BatchNorm -> ReLU operator.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline
arm of ``bench.py`` may import this package.  The CUDA library and its Python binding never
import it.  The two sides share no code; they share only the seeded input generator, which
holds none of the method's arithmetic.

The arithmetic lives in ``cbr_oracle.c``.  It is a direct 7-loop convolution, a two-pass
BatchNorm, ReLU and the hand-derived backward, all in fp64.  This module only marshals numpy
arrays and composes the C steps in the order the pages give them:

* forward (Tech-Renaissance CBR page, sections 4.1-4.3): conv -> batch stats -> finalize ->
  normalise + affine + ReLU + mask;
* backward (same page, sections 5.1-5.2; BatchNorm CUDA page, section 3.1): mask -> BN
  backward -> DGrad and WGrad;
* inference (CBR page sections 2 and 6; BatchNorm CUDA page section 4.4): fold BN into
  W_fold / b_fold, then conv + bias + ReLU.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "cbr_oracle.c")
_LIB = os.path.join(_HERE, "libcbr_oracle.so")
_lock = threading.Lock()
_lib = None

_D = ctypes.POINTER(ctypes.c_double)
_U8 = ctypes.POINTER(ctypes.c_uint8)
_I32 = ctypes.POINTER(ctypes.c_int32)


def build_lib(force: bool = False) -> str:
    """Compile cbr_oracle.c with gcc (-O2, OpenMP, no FP contraction) into libcbr_oracle.so."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O2", "-std=c11", "-fopenmp", "-fPIC", "-shared", "-ffp-contract=off",
               "-o", tmp, _SRC, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build_lib()
            lib = ctypes.CDLL(_LIB)
            i, i64, d = ctypes.c_int, ctypes.c_int64, ctypes.c_double
            conv_args = [i] * 9
            lib.cbr_oracle_out_dim.argtypes = [i, i, i, i]
            lib.cbr_oracle_out_dim.restype = i
            lib.cbr_oracle_conv2d_fwd.argtypes = conv_args + [_D, _D, _D]
            lib.cbr_oracle_conv2d_fwd_at.argtypes = conv_args + [_D, _D, i, _I32, _D]
            lib.cbr_oracle_conv2d_dgrad.argtypes = conv_args + [_D, _D, _D]
            lib.cbr_oracle_conv2d_dgrad_at.argtypes = conv_args + [_D, _D, i, _I32, _D]
            lib.cbr_oracle_conv2d_wgrad.argtypes = conv_args + [_D, _D, _D]
            lib.cbr_oracle_conv2d_wgrad_at.argtypes = conv_args + [_D, _D, i, _I32, _D]
            lib.cbr_oracle_bn_batch_stats.argtypes = [i64, i, _D, _D, _D]
            lib.cbr_oracle_bn_relu_fwd.argtypes = [i64, i, _D, _D, _D, _D, _D, d, _D, _D, _D, _U8]
            lib.cbr_oracle_bn_finalize.argtypes = [i, i64, _D, _D, d, d, _D, _D, _D]
            lib.cbr_oracle_bn_relu_bwd.argtypes = [i64, i, _D, _U8, _D, _D, _D, d, _D, _D, _D]
            lib.cbr_oracle_bn_infer.argtypes = [i64, i, _D, _D, _D, _D, _D, d, _D]
            lib.cbr_oracle_fold.argtypes = [i, i, _D, _D, _D, _D, _D, _D, d, _D, _D]
            lib.cbr_oracle_bias_relu.argtypes = [i64, i, _D, _D, _D]
            lib.cbr_oracle_num_threads.argtypes = []
            lib.cbr_oracle_num_threads.restype = i
            _lib = lib
    return _lib


def _f64(a) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(a, dtype=np.float64))


def _p(a: np.ndarray | None):
    if a is None:
        return None
    if a.dtype == np.float64:
        return a.ctypes.data_as(_D)
    if a.dtype == np.uint8:
        return a.ctypes.data_as(_U8)
    if a.dtype == np.int32:
        return a.ctypes.data_as(_I32)
    raise TypeError(a.dtype)


def num_threads() -> int:
    return _load().cbr_oracle_num_threads()


def out_dim(n: int, k: int, stride: int, pad: int) -> int:
    return _load().cbr_oracle_out_dim(n, k, stride, pad)


# ----------------------------------------------------------------------------- conv steps
def conv2d_fwd(x, w, stride: int, pad: int) -> np.ndarray:
    """x NHWC [N,H,W,C], w KRSC [K,R,S,C] -> z NPQK (direct 7-loop cross-correlation)."""
    x, w = _f64(x), _f64(w)
    N, H, W, C = x.shape
    K, R, S, C2 = w.shape
    assert C == C2
    P, Q = out_dim(H, R, stride, pad), out_dim(W, S, stride, pad)
    z = np.empty((N, P, Q, K), dtype=np.float64)
    _load().cbr_oracle_conv2d_fwd(N, H, W, C, K, R, S, stride, pad, _p(x), _p(w), _p(z))
    return z


def conv2d_fwd_at(x, w, stride: int, pad: int, pixels) -> np.ndarray:
    """z at the listed output pixels ((n,p,q) rows) -> [len(pixels), K]."""
    x, w = _f64(x), _f64(w)
    N, H, W, C = x.shape
    K, R, S, C2 = w.shape
    assert C == C2
    pix = np.ascontiguousarray(np.asarray(pixels, dtype=np.int32).reshape(-1, 3))
    out = np.empty((pix.shape[0], K), dtype=np.float64)
    _load().cbr_oracle_conv2d_fwd_at(N, H, W, C, K, R, S, stride, pad, _p(x), _p(w),
                                     pix.shape[0], _p(pix), _p(out))
    return out


def conv2d_dgrad(dz, w, in_hw: tuple[int, int], stride: int, pad: int) -> np.ndarray:
    dz, w = _f64(dz), _f64(w)
    N, P, Q, K = dz.shape
    K2, R, S, C = w.shape
    assert K == K2
    H, W = in_hw
    assert (P, Q) == (out_dim(H, R, stride, pad), out_dim(W, S, stride, pad))
    dx = np.empty((N, H, W, C), dtype=np.float64)
    _load().cbr_oracle_conv2d_dgrad(N, H, W, C, K, R, S, stride, pad, _p(dz), _p(w), _p(dx))
    return dx


def conv2d_dgrad_at(dz, w, in_hw: tuple[int, int], stride: int, pad: int, pixels) -> np.ndarray:
    """dx at the listed input pixels ((n,h,w) rows) -> [len(pixels), C]."""
    dz, w = _f64(dz), _f64(w)
    N, P, Q, K = dz.shape
    _, R, S, C = w.shape
    H, W = in_hw
    pix = np.ascontiguousarray(np.asarray(pixels, dtype=np.int32).reshape(-1, 3))
    out = np.empty((pix.shape[0], C), dtype=np.float64)
    _load().cbr_oracle_conv2d_dgrad_at(N, H, W, C, K, R, S, stride, pad, _p(dz), _p(w),
                                       pix.shape[0], _p(pix), _p(out))
    return out


def conv2d_wgrad(dz, x, filter_rs: tuple[int, int], stride: int, pad: int) -> np.ndarray:
    dz, x = _f64(dz), _f64(x)
    N, H, W, C = x.shape
    N2, P, Q, K = dz.shape
    R, S = filter_rs
    assert N == N2 and (P, Q) == (out_dim(H, R, stride, pad), out_dim(W, S, stride, pad))
    dw = np.empty((K, R, S, C), dtype=np.float64)
    _load().cbr_oracle_conv2d_wgrad(N, H, W, C, K, R, S, stride, pad, _p(dz), _p(x), _p(dw))
    return dw


def conv2d_wgrad_at(dz, x, filter_rs: tuple[int, int], stride: int, pad: int, taps) -> np.ndarray:
    """dW at the listed filter taps ((k,r,s) rows) -> [len(taps), C]."""
    dz, x = _f64(dz), _f64(x)
    N, H, W, C = x.shape
    N2, P, Q, K = dz.shape
    R, S = filter_rs
    assert N == N2 and (P, Q) == (out_dim(H, R, stride, pad), out_dim(W, S, stride, pad))
    tap = np.ascontiguousarray(np.asarray(taps, dtype=np.int32).reshape(-1, 3))
    out = np.empty((tap.shape[0], C), dtype=np.float64)
    _load().cbr_oracle_conv2d_wgrad_at(N, H, W, C, K, R, S, stride, pad, _p(dz), _p(x),
                                       tap.shape[0], _p(tap), _p(out))
    return out


# ----------------------------------------------------------------------------- BN steps
def bn_batch_stats(z2d) -> tuple[np.ndarray, np.ndarray]:
    z2d = _f64(z2d)
    M, C = z2d.shape
    mean, var = np.empty(C), np.empty(C)
    _load().cbr_oracle_bn_batch_stats(M, C, _p(z2d), _p(mean), _p(var))
    return mean, var


def bn_relu_fwd(z2d, mean, var, gamma, beta, eps: float):
    z2d = _f64(z2d)
    M, C = z2d.shape
    xhat, pre, y = (np.empty((M, C)) for _ in range(3))
    mask = np.empty((M, C), dtype=np.uint8)
    _load().cbr_oracle_bn_relu_fwd(M, C, _p(z2d), _p(_f64(mean)), _p(_f64(var)), _p(_f64(gamma)),
                                   _p(_f64(beta)), eps, _p(xhat), _p(pre), _p(y), _p(mask))
    return xhat, pre, y, mask


def bn_finalize(mean, var, M: int, eps: float, momentum: float, running_mean, running_var):
    C = len(mean)
    rm, rv = _f64(running_mean).copy(), _f64(running_var).copy()
    inv = np.empty(C)
    _load().cbr_oracle_bn_finalize(C, M, _p(_f64(mean)), _p(_f64(var)), eps, momentum, _p(rm),
                                   _p(rv), _p(inv))
    return rm, rv, inv


def bn_relu_bwd(dy2d, mask2d, xhat2d, var, gamma, eps: float, want_dz: bool = True):
    dy2d, xhat2d = _f64(dy2d), _f64(xhat2d)
    mask2d = np.ascontiguousarray(mask2d, dtype=np.uint8)
    M, C = dy2d.shape
    dz = np.empty((M, C)) if want_dz else None
    dgamma, dbeta = np.empty(C), np.empty(C)
    _load().cbr_oracle_bn_relu_bwd(M, C, _p(dy2d), _p(mask2d), _p(xhat2d), _p(_f64(var)),
                                   _p(_f64(gamma)), eps, _p(dz), _p(dgamma), _p(dbeta))
    return dz, dgamma, dbeta


def bn_infer(z2d, running_mean, running_var, gamma, beta, eps: float) -> np.ndarray:
    z2d = _f64(z2d)
    M, C = z2d.shape
    pre = np.empty((M, C))
    _load().cbr_oracle_bn_infer(M, C, _p(z2d), _p(_f64(running_mean)), _p(_f64(running_var)),
                                _p(_f64(gamma)), _p(_f64(beta)), eps, _p(pre))
    return pre


def fold(w, gamma, beta, running_mean, running_var, eps: float, conv_bias=None):
    w = _f64(w)
    K = w.shape[0]
    RSC = int(np.prod(w.shape[1:]))
    w_fold = np.empty_like(w)
    b_fold = np.empty(K)
    cb = None if conv_bias is None else _f64(conv_bias)
    _load().cbr_oracle_fold(K, RSC, _p(w), _p(cb), _p(_f64(gamma)), _p(_f64(beta)),
                            _p(_f64(running_mean)), _p(_f64(running_var)), eps, _p(w_fold),
                            _p(b_fold))
    return w_fold, b_fold


def bias_relu(z2d, bias) -> np.ndarray:
    z2d = _f64(z2d)
    M, C = z2d.shape
    out = np.empty((M, C))
    _load().cbr_oracle_bias_relu(M, C, _p(z2d), _p(_f64(bias)), _p(out))
    return out


# ----------------------------------------------------------------------------- composed
def forward_train(x, w, gamma, beta, running_mean, running_var, momentum: float, eps: float,
                  stride: int, pad: int) -> dict:
    """The training forward in the order of the CBR page, sections 4.1-4.3."""
    z = conv2d_fwd(x, w, stride, pad)
    N, P, Q, K = z.shape
    z2 = z.reshape(-1, K)
    mean, var = bn_batch_stats(z2)
    rm, rv, inv_std = bn_finalize(mean, var, z2.shape[0], eps, momentum, running_mean, running_var)
    xhat, pre, y, mask = bn_relu_fwd(z2, mean, var, gamma, beta, eps)
    shp = (N, P, Q, K)
    return dict(z=z, mean=mean, var=var, inv_std=inv_std, running_mean=rm, running_var=rv,
                xhat=xhat.reshape(shp), pre=pre.reshape(shp), y=y.reshape(shp),
                mask=mask.reshape(shp))


def backward(dy, x, w, fwd: dict, gamma, eps: float, stride: int, pad: int,
             need_dx: bool = True, dx_pixels=None) -> dict:
    """Backward in the order of the CBR page, sections 5.1-5.2: mask, BN backward, then WGrad
    and DGrad.  With dx_pixels, dx is evaluated only at those (n,h,w) input pixels."""
    dy = _f64(dy)
    K = dy.shape[-1]
    dz, dgamma, dbeta = bn_relu_bwd(dy.reshape(-1, K), fwd["mask"].reshape(-1, K),
                                    fwd["xhat"].reshape(-1, K), fwd["var"], gamma, eps)
    dz = dz.reshape(dy.shape)
    R, S = w.shape[1], w.shape[2]
    out = dict(dz=dz, dgamma=dgamma, dbeta=dbeta)
    out["dw"] = conv2d_wgrad(dz, x, (R, S), stride, pad)
    hw = (x.shape[1], x.shape[2])
    if need_dx:
        if dx_pixels is None:
            out["dx"] = conv2d_dgrad(dz, w, hw, stride, pad)
        else:
            out["dx_at"] = conv2d_dgrad_at(dz, w, hw, stride, pad, dx_pixels)
    return out


def forward_infer(x, w, gamma, beta, running_mean, running_var, eps: float, stride: int,
                  pad: int, conv_bias=None) -> dict:
    """Folded inference (CBR page section 2): relu(conv(x, W_fold) + b_fold)."""
    w_fold, b_fold = fold(w, gamma, beta, running_mean, running_var, eps, conv_bias)
    z = conv2d_fwd(x, w_fold, stride, pad)
    K = z.shape[-1]
    y = bias_relu(z.reshape(-1, K), b_fold).reshape(z.shape)
    return dict(w_fold=w_fold, b_fold=b_fold, y=y)
