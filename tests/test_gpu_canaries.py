"""Out-of-bounds write detection without a sanitizer: every buffer the library writes (outputs,
in-place running statistics, workspaces) is placed inside a larger allocation whose guard bytes
before and after are filled with a pattern, and the guards must be intact after a training
step and a folded inference call.  Small and ragged shapes exercise the tile tails, the
padded dz rows and the first-layer kernels (through the C ABI)."""
import pytest
import torch

from conv_batchnorm_relu_gb300 import cbr
from conv_batchnorm_relu_gb300.inputs import CONFIGS, CBRSpec, make_inputs

pytestmark = pytest.mark.gpu

GUARD = 4096
PATTERN = 0xA5

CASES = {
    "cfg1": (CONFIGS[1], 31),
    "ragged_13x29": (CBRSpec("ragged", n=2, h=13, w=29, c_in=64, c_out=64), 32),
    "c128_odd_bf16": (CBRSpec("c128 odd", n=1, h=17, w=30, c_in=128, c_out=128, dtype="bf16"), 33),
    "k5x5_c32": (CBRSpec("5x5", n=2, h=11, w=19, c_in=32, c_out=64, r=5, s=5, pad=2), 34),
    "first_ragged_bf16": (CBRSpec("first ragged", n=3, h=45, w=61, c_in=3, c_out=16, r=7, s=7, stride=2,
                                  pad=3, x_dist="uniform2.5", first_layer=True, dtype="bf16"), 35),
    "first_odd64": (CBRSpec("first odd 64", n=2, h=29, w=37, c_in=3, c_out=64, r=7, s=7, stride=2, pad=3,
                            x_dist="uniform2.5", first_layer=True), 36),
}


class Guarded:
    """Tensors carved out of guarded device allocations."""

    def __init__(self):
        self.bufs = []

    def new(self, shape, dtype, fill=None):
        n = 1
        for d in shape:
            n *= d
        nbytes = n * torch.empty((), dtype=dtype).element_size()
        buf = torch.full((GUARD + nbytes + GUARD,), PATTERN, dtype=torch.uint8, device="cuda")
        t = buf[GUARD:GUARD + nbytes].view(dtype).view(shape)
        if fill is not None:
            t.copy_(fill)
        self.bufs.append((buf, nbytes))
        return t

    def workspace(self, nbytes):
        t = self.new((nbytes,), torch.uint8)
        t.zero_()  # arrival counters must start at zero
        return t

    def check(self):
        for i, (buf, nbytes) in enumerate(self.bufs):
            head = buf[:GUARD]
            tail = buf[GUARD + nbytes:]
            assert bool((head == PATTERN).all()), f"buffer {i}: bytes before it were written"
            assert bool((tail == PATTERN).all()), f"buffer {i}: bytes after it were written"


@pytest.mark.parametrize("case", list(CASES))
def test_no_writes_outside_any_buffer(case):
    spec, seed = CASES[case]
    inp = make_inputs(spec, seed)
    layer = cbr.Layer.from_spec(spec)
    G = Guarded()
    dt = spec.torch_dtype
    x = G.new(tuple(inp["x"].shape), dt, inp["x"].cuda())
    w = G.new(tuple(inp["w"].shape), dt, inp["w"].cuda())
    dy = G.new(tuple(inp["dy"].shape), dt, inp["dy"].cuda())
    gamma = G.new((spec.c_out,), torch.float32, inp["gamma"].cuda())
    beta = G.new((spec.c_out,), torch.float32, inp["beta"].cuda())
    rm = G.new((spec.c_out,), torch.float32, inp["running_mean"].cuda())
    rv = G.new((spec.c_out,), torch.float32, inp["running_var"].cuda())
    out_shape = (spec.n, spec.p, spec.q, spec.c_out)
    fo = {"y": G.new(out_shape, dt), "z": G.new(out_shape, dt),
          "mask": G.new((cbr.mask_words(layer),), torch.int32),
          "saved_mean": G.new((spec.c_out,), torch.float32),
          "saved_inv_var": G.new((spec.c_out,), torch.float32)}
    need_dx = not spec.first_layer
    bo = {"dw": G.new((spec.c_out, spec.r, spec.s, spec.c_in), torch.float32),
          "dgamma": G.new((spec.c_out,), torch.float32), "dbeta": G.new((spec.c_out,), torch.float32)}
    if need_dx:
        bo["dx"] = G.new(tuple(inp["x"].shape), dt)
    fwd_ws, bwd_ws = cbr.workspace_size(layer)
    ws_f, ws_b = G.workspace(fwd_ws), G.workspace(bwd_ws)
    cbr.forward_train(layer, x, w, gamma, beta, rm, rv, spec.momentum, spec.eps, ws=ws_f, out=fo)
    cbr.backward(layer, dy, x, w, fo["mask"], cbr.CBR_MASK_BITS, fo["z"], gamma, fo["saved_mean"],
                 fo["saved_inv_var"], ws=ws_b, need_dx=need_dx, out=bo)
    # the backward again without a kept z (z recomputed into the workspace)
    ws_b2 = G.workspace(bwd_ws)
    cbr.backward(layer, dy, x, w, fo["y"], cbr.CBR_MASK_FROM_Y, None, gamma, fo["saved_mean"],
                 fo["saved_inv_var"], ws=ws_b2, need_dx=need_dx, out=bo)
    # folded inference
    w_fold = G.new(tuple(inp["w"].shape), dt)
    b_fold = G.new((spec.c_out,), torch.float32)
    st = cbr.load().cbr_fold_bn(cbr.ctypes.byref(layer.desc()), w.data_ptr(), None, gamma.data_ptr(),
                                beta.data_ptr(), rm.data_ptr(), rv.data_ptr(), float(spec.eps),
                                w_fold.data_ptr(), b_fold.data_ptr(), torch.cuda.current_stream().cuda_stream)
    assert st == cbr.CBR_OK
    y_inf = G.new(out_shape, dt)
    cbr.forward_infer(layer, x, w_fold, b_fold, out=y_inf)
    cbr.stream_status()
    torch.cuda.synchronize()
    G.check()
