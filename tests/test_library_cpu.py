"""Host-side tests of libcbr.so that need no GPU: the library builds and loads, exports every
function include/cbr.h declares, sizes workspaces, and rejects bad arguments with the
documented status codes before anything is launched.

Pointer arguments here are fake addresses: every call below fails validation (or the device
check) on the host, so nothing is dereferenced and no kernel is launched."""
import ctypes

import pytest
import torch

from conv_batchnorm_relu_gb300 import build, cbr
from conv_batchnorm_relu_gb300.inputs import CONFIGS


@pytest.fixture(scope="module")
def lib():
    build.build()
    lib = cbr.load()
    lib.cbr_forward_infer_bn.argtypes = [ctypes.POINTER(cbr.Desc)] + [ctypes.c_void_p] * 7 + [ctypes.c_float] + \
        [ctypes.c_void_p] * 2
    lib.cbr_forward_infer_bn.restype = ctypes.c_int32
    return lib


def _desc(**kw):
    base = dict(n=2, h=8, w=8, c_in=8, c_out=16, r=3, s=3, stride=1, pad=1, dtype=0)
    base.update(kw)
    return cbr.Desc(*[base[k] for k in ("n", "h", "w", "c_in", "c_out", "r", "s", "stride", "pad", "dtype")])


P = 0x10000  # fake, 16-byte aligned "device" address


def _fwd(lib, d, **over):
    args = dict(x=P, w=P, gamma=P, beta=P, rm=P, rv=P, mom=0.1, eps=1e-5, y=P, mask=P, z=P,
                sm=P, siv=P, ws=P, ws_bytes=1 << 40)
    args.update(over)
    return lib.cbr_forward_train(ctypes.byref(d) if d is not None else None, args["x"], args["w"],
                                 args["gamma"], args["beta"], args["rm"], args["rv"], args["mom"],
                                 args["eps"], args["y"], args["mask"], args["z"], args["sm"],
                                 args["siv"], args["ws"], args["ws_bytes"], None)


def test_exports_every_declared_function(lib):
    names = cbr.declared_functions()
    assert {"cbr_forward_train", "cbr_backward", "cbr_forward_infer", "cbr_fold_bn",
            "cbr_workspace_size", "cbr_stream_status"} <= set(names)
    for n in names:
        assert hasattr(lib, n), n
    assert lib.cbr_version() >= 100
    assert lib.cbr_status_string(3) == b"CBR_ERR_UNSUPPORTED"


def test_workspace_sizes(lib):
    for i, spec in CONFIGS.items():
        d = cbr.Layer.from_spec(spec).desc()
        f, b = ctypes.c_size_t(), ctypes.c_size_t()
        assert lib.cbr_workspace_size(ctypes.byref(d), ctypes.byref(f), ctypes.byref(b)) == 0
        act = spec.n * spec.p * spec.q * spec.c_out * 2
        # fwd: z when the caller does not save it; bwd: z if recomputed (and the materialised dz
        # for layers the fused backward kernel does not take)
        assert f.value >= act and b.value >= act
        assert f.value < act + (64 << 20) and b.value < 2 * act + (256 << 20)


@pytest.mark.parametrize("kw,status", [
    (dict(c_out=12), 1),        # Cout % 8 != 0 (CBR page, section 8)
    (dict(dtype=2), 3),         # fp32 is not an AMP dtype
    (dict(n=0), 1),
    (dict(pad=-1), 1),
    (dict(h=1, w=1, pad=0), 1),  # 3x3 does not fit
    (dict(n=1, h=1, w=1, r=1, s=1, pad=0), 1),  # M = 1: unbiased variance undefined
])
def test_desc_validation(lib, kw, status):
    assert _fwd(lib, _desc(**kw)) == status


def test_null_and_scalar_checks(lib):
    d = _desc()
    assert _fwd(lib, None) == 1
    for k in ("x", "w", "gamma", "beta", "rm", "rv", "y", "sm", "siv", "ws"):
        assert _fwd(lib, d, **{k: None}) == 1, k
    assert _fwd(lib, d, mom=1.5) == 1
    assert _fwd(lib, d, eps=0.0) == 1
    assert _fwd(lib, d, eps=float("nan")) == 1


def test_alignment_checks(lib):
    d = _desc()
    assert _fwd(lib, d, x=P + 2) == 2
    assert _fwd(lib, d, y=P + 8) == 2
    assert _fwd(lib, d, gamma=P + 2) == 2


def test_unsupported_shapes(lib):
    assert _fwd(lib, _desc(c_out=24)) == 3               # Cout not in {16,32,64,128}
    assert _fwd(lib, _desc(c_in=12)) == 3                # Cin not a multiple of 8
    assert _fwd(lib, _desc(c_in=256, c_out=64)) == 3     # Cin > 128
    assert _fwd(lib, _desc(w=300, h=4)) == 3             # padded width > 256


def test_workspace_too_small(lib):
    d = _desc()
    f = ctypes.c_size_t()
    lib.cbr_workspace_size(ctypes.byref(d), ctypes.byref(f), None)
    assert _fwd(lib, d, z=None, ws_bytes=f.value - 1) == 4


def test_backward_rejects_dx_aliasing_x(lib):
    d = _desc()
    st = lib.cbr_backward(ctypes.byref(d), P, P, P, P, 0, P, P, P, P, P, P, P, P, P, 1 << 40, None)
    assert st == 1
    st = lib.cbr_backward(ctypes.byref(d), P, P, P, P, 7, P, P, P, P, P + (1 << 20), P, P, P, P,
                          1 << 40, None)
    assert st == 1  # bad mask kind


@pytest.mark.skipif(torch.cuda.is_available(), reason="checks the no-device path")
def test_no_device_is_reported(lib):
    assert _fwd(lib, _desc()) == 5


def test_noalloc_forward_requires_z_saved(lib):
    f = lib.cbr_forward_train_noalloc
    vp, fp = ctypes.c_void_p, ctypes.c_float
    f.argtypes = [ctypes.POINTER(cbr.Desc), vp, vp, vp, vp, vp, vp, fp, fp, vp, vp, vp, vp, vp, vp]
    f.restype = ctypes.c_int32
    d = _desc()
    assert f(ctypes.byref(d), P, P, P, P, P, P, 0.1, 1e-5, P, P, None, P, P, None) == 1
    bad = _desc(c_out=12)
    assert f(ctypes.byref(bad), P, P, P, P, P, P, 0.1, 1e-5, P, P, P, P, P, None) == 1


def test_noalloc_forward_rejects_before_touching_scratch(lib):
    """Argument, alignment and shape errors come back with the same codes as cbr_forward_train,
    before the device check and before anything is enqueued on the shared scratch."""
    f = lib.cbr_forward_train_noalloc
    vp, fp = ctypes.c_void_p, ctypes.c_float
    f.argtypes = [ctypes.POINTER(cbr.Desc), vp, vp, vp, vp, vp, vp, fp, fp, vp, vp, vp, vp, vp, vp]
    f.restype = ctypes.c_int32
    d = _desc()
    assert f(ctypes.byref(d), P, P, P, P, P, P, 1.5, 1e-5, P, P, P, P, P, None) == 1   # momentum
    assert f(ctypes.byref(d), P, P, P, P, P, P, 0.1, 0.0, P, P, P, P, P, None) == 1    # eps
    assert f(ctypes.byref(d), P + 2, P, P, P, P, P, 0.1, 1e-5, P, P, P, P, P, None) == 2  # x misaligned
    assert f(ctypes.byref(d), P, P, P, P, P, P, 0.1, 1e-5, P, P, P + 8, P, P, None) == 2  # z misaligned
    assert f(ctypes.byref(_desc(c_out=24)), P, P, P, P, P, P, 0.1, 1e-5, P, P, P, P, P, None) == 3
    if not torch.cuda.is_available():
        # valid arguments reach the device check, which reports the missing GPU
        assert f(ctypes.byref(d), P, P, P, P, P, P, 0.1, 1e-5, P, P, P, P, P, None) == 5


def test_selftest_limit_checked_before_device(lib):
    for bad in (0, -5, 1000001):
        assert lib.cbr_selftest_bounded_wait(bad, None) == 1
    # a valid limit gets as far as the device check (no GPU here)
    assert lib.cbr_selftest_bounded_wait(1000, None) == 5


def test_mask_transcoding_validation(lib):
    """Argument checks of cbr_mask_bits_to_bytes / cbr_mask_bytes_to_bits, before any launch."""
    for f in (lib.cbr_mask_bits_to_bytes, lib.cbr_mask_bytes_to_bits):
        assert f(P, P, -1, None) == 1            # negative count
        assert f(None, P, 64, None) == 1         # NULL buffer
        assert f(P, None, 64, None) == 1
        assert f(None, None, 0, None) == 0       # empty: nothing to do
    assert lib.cbr_mask_bits_to_bytes(P + 2, P, 64, None) == 2   # words must be 4-byte aligned
    assert lib.cbr_mask_bits_to_bytes(P, P + 4, 64, None) == 2   # bytes must be 16-byte aligned
    assert lib.cbr_mask_bytes_to_bits(P + 8, P, 64, None) == 2
    if not torch.cuda.is_available():
        assert lib.cbr_mask_bits_to_bytes(P, P, 64, None) == 5


def test_backward_accepts_byte_mask_kind(lib):
    d = _desc()
    # CBR_MASK_BYTES (2) wants a 16-byte aligned mask; kinds past it are rejected
    st = lib.cbr_backward(ctypes.byref(d), P, P, P, P + 4, 2, P, P, P, P, P + (1 << 20), P, P, P, P,
                          1 << 40, None)
    assert st == 2
    st = lib.cbr_backward(ctypes.byref(d), P, P, P, P, 3, P, P, P, P, P + (1 << 20), P, P, P, P,
                          1 << 40, None)
    assert st == 1


def test_infer_bn_validation(lib):
    d = _desc()
    f = lib.cbr_forward_infer_bn
    assert f(ctypes.byref(d), P, P, None, P, P, P, P, 1e-5, None, None) == 1     # no y
    assert f(ctypes.byref(d), P, P, None, P, P, P, P, 0.0, P, None) == 1         # eps
    assert f(ctypes.byref(d), P + 2, P, None, P, P, P, P, 1e-5, P, None) == 2    # x misaligned
    first = _desc(c_in=3, c_out=64, r=7, s=7, stride=2, pad=3, h=32, w=32)
    assert f(ctypes.byref(first), P, P, None, P, P, P, P, 1e-5, P, None) == 3     # first layer: fold it
