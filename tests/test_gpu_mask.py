"""GPU tests of the ReLU-mask transcoding (bit-packed <-> one byte per element, the CBR page's
BOOLEAN mask against a standalone ReLU's INT8 mask, sections 8 and 9) and of cbr_backward fed
a byte-per-element mask (CBR_MASK_BYTES), through the C ABI."""
import numpy as np
import pytest
import torch

from conv_batchnorm_relu_gb300 import cbr
from conv_batchnorm_relu_gb300.inputs import CBRSpec, make_inputs

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("count", [1, 31, 32, 33, 1000, 32 * 4096 + 17])
def test_bits_to_bytes_matches_unpack(count):
    gen = torch.Generator().manual_seed(count)
    words = torch.randint(-2**31, 2**31 - 1, ((count + 31) // 32,), generator=gen, dtype=torch.int64).to(torch.int32)
    got = cbr.mask_bits_to_bytes(words.cuda(), count)
    cbr.stream_status()
    want = np.unpackbits(words.numpy().view(np.uint8), bitorder="little")[:count]
    assert np.array_equal(got.cpu().numpy(), want)


@pytest.mark.parametrize("count", [1, 31, 32, 33, 1000, 32 * 4096 + 17])
def test_bytes_to_bits_sets_nonzero_and_clears_the_tail(count):
    gen = torch.Generator().manual_seed(count + 1)
    # values other than 0 and 1 count as set, as in an INT8 mask that stores the activation flag
    vals = torch.randint(0, 4, (count,), generator=gen, dtype=torch.int64)
    mask_bytes = torch.where(vals == 3, torch.full_like(vals, 255), vals).to(torch.uint8)
    out = torch.full(((count + 31) // 32,), -1, dtype=torch.int32).cuda()  # tail bits must be cleared
    got = cbr.mask_bytes_to_bits(mask_bytes.cuda(), count, out=out)
    cbr.stream_status()
    bits = (mask_bytes.numpy() != 0).astype(np.uint8)
    padded = np.zeros(((count + 31) // 32) * 32, dtype=np.uint8)
    padded[:count] = bits
    want = np.packbits(padded, bitorder="little").view(np.int32)
    assert np.array_equal(got.cpu().numpy(), want)


def test_round_trip_of_a_forward_mask():
    spec = CBRSpec("ragged", n=2, h=13, w=29, c_in=64, c_out=64)
    inp = make_inputs(spec, 2201, with_dy=False)
    layer = cbr.Layer.from_spec(spec)
    g = {k: v.cuda() for k, v in inp.items()}
    fwd, _ = cbr.workspace_size(layer)
    out = cbr.forward_train(layer, g["x"], g["w"], g["gamma"], g["beta"], g["running_mean"],
                            g["running_var"], ws=cbr.new_workspace(fwd))
    count = spec.m * spec.c_out
    as_bytes = cbr.mask_bits_to_bytes(out["mask"], count)
    back = cbr.mask_bytes_to_bits(as_bytes, count)
    cbr.stream_status()
    # the forward leaves the bits past the last element unspecified; compare the defined ones
    full = count // 32
    assert torch.equal(back[:full], out["mask"][:full])
    # a set mask bit means the pre-activation was positive, so y > 0 wherever a byte is 1 (the
    # converse can fail only where a positive pre-activation rounds to zero in the storage dtype)
    assert bool(((out["y"].reshape(-1) > 0) | ~as_bytes.bool()).all())


@pytest.mark.parametrize("spec,seed", [
    (CBRSpec("ragged", n=2, h=13, w=29, c_in=64, c_out=64), 2202),           # fused backward
    (CBRSpec("c128", n=1, h=17, w=30, c_in=128, c_out=128), 2203),           # materialised dz
    (CBRSpec("first", n=2, h=32, w=32, c_in=3, c_out=64, r=7, s=7, stride=2, pad=3,
             x_dist="uniform2.5", first_layer=True), 2204),                  # first layer
])
def test_backward_with_byte_mask_equals_bit_mask(spec, seed):
    inp = make_inputs(spec, seed)
    layer = cbr.Layer.from_spec(spec)
    g = {k: v.cuda() for k, v in inp.items()}
    fwd, bwd = cbr.workspace_size(layer)
    out = cbr.forward_train(layer, g["x"], g["w"], g["gamma"], g["beta"], g["running_mean"],
                            g["running_var"], ws=cbr.new_workspace(fwd))
    need_dx = not spec.first_layer
    a = cbr.backward(layer, g["dy"], g["x"], g["w"], out["mask"], cbr.CBR_MASK_BITS, out["z"], g["gamma"],
                     out["saved_mean"], out["saved_inv_var"], ws=cbr.new_workspace(bwd), need_dx=need_dx)
    as_bytes = cbr.mask_bits_to_bytes(out["mask"], spec.m * spec.c_out)
    b = cbr.backward(layer, g["dy"], g["x"], g["w"], as_bytes, cbr.CBR_MASK_BYTES, out["z"], g["gamma"],
                     out["saved_mean"], out["saved_inv_var"], ws=cbr.new_workspace(bwd), need_dx=need_dx)
    cbr.stream_status()
    for k in ("dw", "dgamma", "dbeta") + (("dx",) if need_dx else ()):
        assert torch.equal(a[k], b[k]), k
