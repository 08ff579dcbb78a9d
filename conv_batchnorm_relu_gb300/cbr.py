"""Python binding of libcbr.so: argument marshalling only.

Every step of the operator runs in the CUDA library's kernels; this module allocates the
output tensors with torch (the caller-owns-memory convention of the C ABI), passes raw
pointers and the current CUDA stream, and raises :class:`CBRError` on a non-OK status.
There is no fallback: if the library is missing or the device is not a GB300 (sm_103),
calls raise.
"""
from __future__ import annotations

import ctypes
import os
import re
import threading
from dataclasses import dataclass

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libcbr.so")
HEADER_PATH = os.path.join(os.path.dirname(_PKG), "include", "cbr.h")

CBR_OK = 0
STATUS_NAMES = {0: "CBR_OK", 1: "CBR_ERR_INVALID_ARG", 2: "CBR_ERR_MISALIGNED",
                3: "CBR_ERR_UNSUPPORTED", 4: "CBR_ERR_WORKSPACE", 5: "CBR_ERR_DEVICE",
                6: "CBR_ERR_CUDA", 7: "CBR_ERR_TIMEOUT"}
CBR_F16, CBR_BF16 = 0, 1
CBR_MASK_BITS, CBR_MASK_FROM_Y, CBR_MASK_BYTES = 0, 1, 2


class CBRError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {STATUS_NAMES.get(status, status)}")


class Desc(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in
                ("n", "h", "w", "c_in", "c_out", "r", "s", "stride", "pad", "dtype")]


_lock = threading.Lock()
_lib = None


def load(path: str | None = None) -> ctypes.CDLL:
    """Open libcbr.so (raises if it has not been built)."""
    global _lib
    with _lock:
        if _lib is None:
            p = path or LIB_PATH
            if not os.path.exists(p):
                raise RuntimeError(f"libcbr.so not built ({p}); run conv_batchnorm_relu_gb300/build.py")
            lib = ctypes.CDLL(p)
            vp, sz, i32, fp = ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int32, ctypes.c_float
            D = ctypes.POINTER(Desc)
            lib.cbr_version.restype = i32
            lib.cbr_status_string.argtypes = [i32]
            lib.cbr_status_string.restype = ctypes.c_char_p
            lib.cbr_workspace_size.argtypes = [D, ctypes.POINTER(sz), ctypes.POINTER(sz)]
            lib.cbr_forward_train.argtypes = [D, vp, vp, vp, vp, vp, vp, fp, fp, vp, vp, vp, vp,
                                              vp, vp, sz, vp]
            lib.cbr_forward_train_persistent.argtypes = lib.cbr_forward_train.argtypes
            lib.cbr_backward.argtypes = [D, vp, vp, vp, vp, i32, vp, vp, vp, vp, vp, vp, vp, vp,
                                         vp, sz, vp]
            lib.cbr_fold_bn.argtypes = [D, vp, vp, vp, vp, vp, vp, fp, vp, vp, vp]
            lib.cbr_forward_infer.argtypes = [D, vp, vp, vp, vp, vp]
            lib.cbr_forward_infer_bn.argtypes = [D, vp, vp, vp, vp, vp, vp, vp, fp, vp, vp]
            lib.cbr_stream_status.argtypes = [vp]
            lib.cbr_forward_train_stats.argtypes = [D, vp, vp, vp, vp, vp, sz, vp]
            lib.cbr_forward_train_finish.argtypes = [D, vp, i32, vp, vp, vp, vp, fp, fp, vp, vp, vp, vp, vp,
                                                     vp, sz, vp]
            lib.cbr_backward_sums.argtypes = [D, vp, vp, i32, vp, vp, vp, vp, sz, vp]
            lib.cbr_backward_finish.argtypes = [D, vp, ctypes.c_int64, vp, vp, vp, vp, i32, vp, vp, vp, vp, vp,
                                                vp, vp, vp, vp, sz, vp]
            lib.cbr_mask_bits_to_bytes.argtypes = [vp, vp, ctypes.c_int64, vp]
            lib.cbr_mask_bytes_to_bits.argtypes = [vp, vp, ctypes.c_int64, vp]
            lib.cbr_selftest_bounded_wait.argtypes = [i32, vp]
            lib.cbr_profile_next_call.argtypes = [ctypes.POINTER(vp), i32]
            lib.cbr_profile_last_count.restype = i32
            for f in ("cbr_workspace_size", "cbr_forward_train", "cbr_forward_train_persistent", "cbr_backward",
                      "cbr_fold_bn",
                      "cbr_forward_infer", "cbr_forward_infer_bn", "cbr_stream_status", "cbr_profile_next_call",
                      "cbr_selftest_bounded_wait", "cbr_mask_bits_to_bytes", "cbr_mask_bytes_to_bits",
                      "cbr_forward_train_stats", "cbr_forward_train_finish", "cbr_backward_sums",
                      "cbr_backward_finish"):
                getattr(lib, f).restype = i32
            _lib = lib
    return _lib


def declared_functions() -> list[str]:
    """Names of the functions include/cbr.h declares."""
    with open(HEADER_PATH) as f:
        text = f.read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(cbr_[a-z_]+)\s*\(", text)))


def _check(status: int, what: str) -> None:
    if status != CBR_OK:
        raise CBRError(status, what)


def _ptr(t: torch.Tensor | None) -> int | None:
    return None if t is None else t.data_ptr()


def _stream() -> int:
    return torch.cuda.current_stream().cuda_stream


@dataclass(frozen=True)
class Layer:
    n: int
    h: int
    w: int
    c_in: int
    c_out: int
    r: int = 3
    s: int = 3
    stride: int = 1
    pad: int = 1
    dtype: torch.dtype = torch.float16

    @property
    def p(self) -> int:
        return (self.h + 2 * self.pad - self.r) // self.stride + 1

    @property
    def q(self) -> int:
        return (self.w + 2 * self.pad - self.s) // self.stride + 1

    def desc(self) -> Desc:
        return Desc(self.n, self.h, self.w, self.c_in, self.c_out, self.r, self.s, self.stride,
                    self.pad, CBR_BF16 if self.dtype == torch.bfloat16 else CBR_F16)

    @staticmethod
    def from_spec(spec) -> "Layer":
        return Layer(spec.n, spec.h, spec.w, spec.c_in, spec.c_out, spec.r, spec.s, spec.stride,
                     spec.pad, spec.torch_dtype)


def workspace_size(layer: Layer) -> tuple[int, int]:
    f, b = ctypes.c_size_t(), ctypes.c_size_t()
    d = layer.desc()
    _check(load().cbr_workspace_size(ctypes.byref(d), ctypes.byref(f), ctypes.byref(b)),
           "cbr_workspace_size")
    return f.value, b.value


def new_workspace(nbytes: int, device="cuda") -> torch.Tensor:
    """Zero-filled workspace (its arrival counters must start at zero)."""
    return torch.zeros(nbytes, dtype=torch.uint8, device=device)


def mask_words(layer: Layer) -> int:
    return (layer.n * layer.p * layer.q * layer.c_out + 31) // 32


def forward_train(layer: Layer, x, w, gamma, beta, running_mean, running_var, momentum=0.1,
                  eps=1e-5, *, ws, want_mask=True, save_z=True, out=None, persistent=False) -> dict:
    """cbr_forward_train (persistent: cbr_forward_train_persistent, the one-launch form).
    running_mean / running_var are updated in place."""
    dev = x.device
    o = dict(out or {})
    if "y" not in o:
        o["y"] = torch.empty((layer.n, layer.p, layer.q, layer.c_out), dtype=layer.dtype, device=dev)
    if want_mask and "mask" not in o:
        o["mask"] = torch.empty(mask_words(layer), dtype=torch.int32, device=dev)
    if save_z and "z" not in o:
        o["z"] = torch.empty_like(o["y"])
    for k in ("saved_mean", "saved_inv_var"):
        if k not in o:
            o[k] = torch.empty(layer.c_out, dtype=torch.float32, device=dev)
    d = layer.desc()
    name = "cbr_forward_train_persistent" if persistent else "cbr_forward_train"
    st = getattr(load(), name)(
        ctypes.byref(d), _ptr(x), _ptr(w), _ptr(gamma), _ptr(beta), _ptr(running_mean),
        _ptr(running_var), float(momentum), float(eps), _ptr(o["y"]), _ptr(o.get("mask")),
        _ptr(o.get("z")), _ptr(o["saved_mean"]), _ptr(o["saved_inv_var"]), _ptr(ws),
        ws.numel(), _stream())
    _check(st, name)
    return o


def backward(layer: Layer, dy, x, w, y_or_mask, mask_kind, z_saved, gamma, saved_mean,
             saved_inv_var, *, ws, need_dx=True, out=None) -> dict:
    """cbr_backward -> dict(dx (or None), dw, dgamma, dbeta)."""
    dev = dy.device
    o = dict(out or {})
    if need_dx and "dx" not in o:
        o["dx"] = torch.empty((layer.n, layer.h, layer.w, layer.c_in), dtype=layer.dtype, device=dev)
    if "dw" not in o:
        o["dw"] = torch.empty((layer.c_out, layer.r, layer.s, layer.c_in), dtype=torch.float32, device=dev)
    for k in ("dgamma", "dbeta"):
        if k not in o:
            o[k] = torch.empty(layer.c_out, dtype=torch.float32, device=dev)
    d = layer.desc()
    st = load().cbr_backward(
        ctypes.byref(d), _ptr(dy), _ptr(x), _ptr(w), _ptr(y_or_mask), int(mask_kind),
        _ptr(z_saved), _ptr(gamma), _ptr(saved_mean), _ptr(saved_inv_var),
        _ptr(o.get("dx")) if need_dx else None, _ptr(o["dw"]), _ptr(o["dgamma"]),
        _ptr(o["dbeta"]), _ptr(ws), ws.numel(), _stream())
    _check(st, "cbr_backward")
    if not need_dx:
        o["dx"] = None
    return o


# ----------------------------------------------------------------------------- synchronised BN
# The split calls bracket one collective each; the collectives run through torch.distributed
# (NCCL on GPUs), the arithmetic on both sides of them in the library's kernels.

def moments_floats(layer: Layer) -> int:
    """Floats of one rank's moments: mean [c_out], M2 [c_out], row count."""
    return 2 * layer.c_out + 1


def forward_train_stats(layer: Layer, x, w, *, ws, z=None):
    """cbr_forward_train_stats -> (z, moments [2*c_out + 1])."""
    if z is None:
        z = torch.empty((layer.n, layer.p, layer.q, layer.c_out), dtype=layer.dtype, device=x.device)
    mom = torch.empty(moments_floats(layer), dtype=torch.float32, device=x.device)
    d = layer.desc()
    _check(load().cbr_forward_train_stats(ctypes.byref(d), _ptr(x), _ptr(w), _ptr(z), _ptr(mom), _ptr(ws),
                                          ws.numel(), _stream()), "cbr_forward_train_stats")
    return z, mom


def forward_train_finish(layer: Layer, moments_all, gamma, beta, running_mean, running_var, momentum, eps, z, *,
                         ws, want_mask=True, out=None) -> dict:
    """cbr_forward_train_finish: moments_all [world][2*c_out + 1] in rank order."""
    dev = z.device
    o = dict(out or {})
    if "y" not in o:
        o["y"] = torch.empty_like(z)
    if want_mask and "mask" not in o:
        o["mask"] = torch.empty(mask_words(layer), dtype=torch.int32, device=dev)
    for k in ("saved_mean", "saved_inv_var"):
        if k not in o:
            o[k] = torch.empty(layer.c_out, dtype=torch.float32, device=dev)
    world = moments_all.shape[0]
    d = layer.desc()
    _check(load().cbr_forward_train_finish(
        ctypes.byref(d), _ptr(moments_all), int(world), _ptr(gamma), _ptr(beta), _ptr(running_mean),
        _ptr(running_var), float(momentum), float(eps), _ptr(z), _ptr(o["y"]), _ptr(o.get("mask")),
        _ptr(o["saved_mean"]), _ptr(o["saved_inv_var"]), _ptr(ws), ws.numel(), _stream()),
        "cbr_forward_train_finish")
    o["z"] = z
    o["m_total"] = int(round(float(moments_all[:, -1].double().sum())))
    return o


def backward_sums(layer: Layer, dy, y_or_mask, mask_kind, z, saved_mean, *, ws) -> torch.Tensor:
    """cbr_backward_sums -> [sum g (c_out)][sum g*(z - mean) (c_out)] of this rank."""
    sums = torch.empty(2 * layer.c_out, dtype=torch.float32, device=dy.device)
    d = layer.desc()
    _check(load().cbr_backward_sums(ctypes.byref(d), _ptr(dy), _ptr(y_or_mask), int(mask_kind), _ptr(z),
                                    _ptr(saved_mean), _ptr(sums), _ptr(ws), ws.numel(), _stream()),
           "cbr_backward_sums")
    return sums


def backward_finish(layer: Layer, sums_all, m_total: int, dy, x, w, y_or_mask, mask_kind, z, gamma,
                    saved_mean, saved_inv_var, *, ws, need_dx=True, out=None) -> dict:
    """cbr_backward_finish -> dict(dx (or None), dw, dgamma, dbeta)."""
    dev = dy.device
    o = dict(out or {})
    if need_dx and "dx" not in o:
        o["dx"] = torch.empty((layer.n, layer.h, layer.w, layer.c_in), dtype=layer.dtype, device=dev)
    if "dw" not in o:
        o["dw"] = torch.empty((layer.c_out, layer.r, layer.s, layer.c_in), dtype=torch.float32, device=dev)
    for k in ("dgamma", "dbeta"):
        if k not in o:
            o[k] = torch.empty(layer.c_out, dtype=torch.float32, device=dev)
    d = layer.desc()
    _check(load().cbr_backward_finish(
        ctypes.byref(d), _ptr(sums_all), int(m_total), _ptr(dy), _ptr(x), _ptr(w), _ptr(y_or_mask),
        int(mask_kind), _ptr(z), _ptr(gamma), _ptr(saved_mean), _ptr(saved_inv_var),
        _ptr(o.get("dx")) if need_dx else None, _ptr(o["dw"]), _ptr(o["dgamma"]), _ptr(o["dbeta"]), _ptr(ws),
        ws.numel(), _stream()), "cbr_backward_finish")
    if not need_dx:
        o["dx"] = None
    return o


def gather_moments(moments: torch.Tensor, group=None) -> torch.Tensor:
    """Every rank's moments in rank order, [world][2*c_out + 1] (an all-gather: moments are merged,
    not summed).  Without an initialised process group this rank is the whole batch."""
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()):
        return moments.unsqueeze(0)
    world = dist.get_world_size(group)
    out = [torch.empty_like(moments) for _ in range(world)]
    dist.all_gather(out, moments.contiguous(), group=group)
    return torch.stack(out)


def reduce_sums(sums: torch.Tensor, group=None) -> torch.Tensor:
    """The backward's per-channel sums added over all ranks (an all-reduce)."""
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()):
        return sums
    out = sums.clone()
    dist.all_reduce(out, op=dist.ReduceOp.SUM, group=group)
    return out


def syncbn_forward_train(layer: Layer, x, w, gamma, beta, running_mean, running_var, momentum=0.1,
                         eps=1e-5, *, ws, group=None, want_mask=True, out=None) -> dict:
    """Synchronised training forward: statistics over every rank's share of the batch."""
    z, mom = forward_train_stats(layer, x, w, ws=ws, z=(out or {}).get("z"))
    gathered = gather_moments(mom, group)
    return forward_train_finish(layer, gathered, gamma, beta, running_mean, running_var, momentum, eps, z,
                                ws=ws, want_mask=want_mask, out=out)


def syncbn_backward(layer: Layer, dy, x, w, y_or_mask, mask_kind, z, gamma, saved_mean, saved_inv_var,
                    m_total: int, *, ws, group=None, need_dx=True, out=None) -> dict:
    """Synchronised training backward: dgamma, dbeta and the BN data gradient over the global
    batch of m_total rows (from syncbn_forward_train's "m_total")."""
    sums = reduce_sums(backward_sums(layer, dy, y_or_mask, mask_kind, z, saved_mean, ws=ws), group)
    return backward_finish(layer, sums, m_total, dy, x, w, y_or_mask, mask_kind, z, gamma, saved_mean,
                           saved_inv_var, ws=ws, need_dx=need_dx, out=out)


def fold_bn(layer: Layer, w, gamma, beta, running_mean, running_var, eps=1e-5, conv_bias=None):
    w_fold = torch.empty_like(w)
    b_fold = torch.empty(layer.c_out, dtype=torch.float32, device=w.device)
    d = layer.desc()
    st = load().cbr_fold_bn(ctypes.byref(d), _ptr(w), _ptr(conv_bias), _ptr(gamma), _ptr(beta),
                            _ptr(running_mean), _ptr(running_var), float(eps), _ptr(w_fold),
                            _ptr(b_fold), _stream())
    _check(st, "cbr_fold_bn")
    return w_fold, b_fold


def forward_infer(layer: Layer, x, w_fold, b_fold, out=None):
    y = out if out is not None else torch.empty((layer.n, layer.p, layer.q, layer.c_out),
                                                dtype=layer.dtype, device=x.device)
    d = layer.desc()
    _check(load().cbr_forward_infer(ctypes.byref(d), _ptr(x), _ptr(w_fold), _ptr(b_fold),
                                    _ptr(y), _stream()), "cbr_forward_infer")
    return y


def mask_bits_to_bytes(bits: torch.Tensor, count: int, out: torch.Tensor | None = None) -> torch.Tensor:
    """cbr_mask_bits_to_bytes: the bit-packed mask (int32 words) as one uint8 (0/1) per element."""
    out = out if out is not None else torch.empty(count, dtype=torch.uint8, device=bits.device)
    _check(load().cbr_mask_bits_to_bytes(_ptr(bits), _ptr(out), int(count), _stream()), "cbr_mask_bits_to_bytes")
    return out


def mask_bytes_to_bits(mask_bytes: torch.Tensor, count: int, out: torch.Tensor | None = None) -> torch.Tensor:
    """cbr_mask_bytes_to_bits: a byte-per-element mask (non-zero = set) as bit-packed int32 words."""
    out = out if out is not None else torch.empty((count + 31) // 32, dtype=torch.int32, device=mask_bytes.device)
    _check(load().cbr_mask_bytes_to_bits(_ptr(mask_bytes), _ptr(out), int(count), _stream()), "cbr_mask_bytes_to_bits")
    return out


def forward_infer_bn(layer: Layer, x, w, gamma, beta, running_mean, running_var, eps=1e-5, conv_bias=None,
                     out=None):
    """cbr_forward_infer_bn: relu(conv(x, w)*scale + shift) with BatchNorm on the accumulator."""
    y = out if out is not None else torch.empty((layer.n, layer.p, layer.q, layer.c_out),
                                                dtype=layer.dtype, device=x.device)
    d = layer.desc()
    _check(load().cbr_forward_infer_bn(ctypes.byref(d), _ptr(x), _ptr(w), _ptr(conv_bias), _ptr(gamma),
                                       _ptr(beta), _ptr(running_mean), _ptr(running_var), float(eps), _ptr(y),
                                       _stream()), "cbr_forward_infer_bn")
    return y


def stream_status(stream: int | None = None) -> None:
    """Synchronise the stream and raise if a kernel reported a device-side error."""
    _check(load().cbr_stream_status(stream if stream is not None else _stream()),
           "cbr_stream_status")


def stream_status_code(stream: int | None = None) -> int:
    """cbr_stream_status's raw status code (0 = CBR_OK), without raising."""
    return load().cbr_stream_status(stream if stream is not None else _stream())


def selftest_bounded_wait(limit_us: int) -> None:
    """Launch the library's bounded-wait self-test on the current stream (see include/cbr.h)."""
    _check(load().cbr_selftest_bounded_wait(int(limit_us), _stream()), "cbr_selftest_bounded_wait")


def profile_next_call(events: list) -> None:
    """Record the given torch.cuda.Event objects at the kernel boundaries of the next call."""
    arr = (ctypes.c_void_p * len(events))(*[e.cuda_event for e in events])
    profile_next_call._keep = arr  # keep alive until the call consumes it
    _check(load().cbr_profile_next_call(arr, len(events)), "cbr_profile_next_call")


def profile_last_count() -> int:
    return load().cbr_profile_last_count()
