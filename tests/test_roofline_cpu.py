"""The roofline ledger the benchmark reports against (host logic, no GPU): per-pass minimum
bytes and algorithmic FLOPs for the benchmark workloads, checked against the closed forms
(activation sizes of the CBR page's 102,760,448-byte feature map, 2*M*K_red*Cout per
convolution) and against the per-pass roofs computed by hand from the same peaks."""
import pytest

from conv_batchnorm_relu_gb300 import roofline
from conv_batchnorm_relu_gb300.inputs import CONFIGS

S3 = 256 * 56 * 56 * 64 * 2          # one fp16 activation of the N=256 56x56 64-channel layer
MASK3 = S3 // 16                      # one bit per element
W3 = 64 * 3 * 3 * 64 * 2
DW3 = 64 * 3 * 3 * 64 * 4


def test_ledger_bytes_and_flops_n256_56x56_c64():
    assert S3 == 102_760_448
    passes = {p.name: p for p in roofline.ledger(CONFIGS[3])}
    assert passes["conv_fprop_genstats"].bytes == 2 * S3 + W3
    assert passes["bn_apply_relu"].bytes == 2 * S3 + MASK3
    assert passes["bn_bwd_reduce"].bytes == 2 * S3 + MASK3
    assert passes["conv_wgrad"].bytes == 3 * S3 + MASK3 + DW3
    assert passes["conv_dgrad"].bytes == 3 * S3 + MASK3 + W3
    flops = 2 * (256 * 56 * 56) * (3 * 3 * 64) * 64
    assert flops == 59_190_018_048
    for name in ("conv_fprop_genstats", "conv_wgrad", "conv_dgrad"):
        assert passes[name].flops == flops
    assert passes["bn_apply_relu"].flops == passes["bn_bwd_reduce"].flops == 0


def test_first_layer_has_no_dgrad_pass():
    names = [p.name for p in roofline.ledger(CONFIGS[4], need_dx=False)]
    assert "conv_dgrad" not in names and len(names) == 4
    fl = 2 * (256 * 112 * 112) * (7 * 7 * 3) * 64
    assert all(p.flops in (0, fl) for p in roofline.ledger(CONFIGS[4], need_dx=False))


def test_step_roof_matches_hand_sum():
    # the per-pass roofs of the N=256 56x56 64->64 step at 6774.2 GB/s and 1921.0 TFLOP/s,
    # computed by hand: K1 30.81 (tensor), apply 31.29, reduce 31.29, wgrad 46.48, dgrad 46.47
    peaks = {"hbm_gbs": 6774.2, "bf16_tflops": 1921.0, "bf16_tflops_sustained": 1921.0}
    by_hand = {"conv_fprop_genstats": 30.81, "bn_apply_relu": 31.29, "bn_bwd_reduce": 31.29,
               "conv_wgrad": 46.48, "conv_dgrad": 46.47}
    for p in roofline.ledger(CONFIGS[3]):
        us, bound = p.roof_us(peaks)
        assert us == pytest.approx(by_hand[p.name], abs=0.01), p.name
        assert bound == ("tensor" if p.name == "conv_fprop_genstats" else "hbm")
    assert roofline.step_roof_us(CONFIGS[3], peaks) == pytest.approx(sum(by_hand.values()), abs=0.03)


def test_inference_pass_is_tensor_bound_at_128_channels():
    spec = CONFIGS[5]
    p = roofline.infer_pass(spec)
    act = 64 * 112 * 112 * 128 * 2
    assert p.bytes == 2 * act + 128 * 3 * 3 * 128 * 2 + 128 * 4
    assert p.flops == 2 * (64 * 112 * 112) * (3 * 3 * 128) * 128
    peaks = {"hbm_gbs": 6795.1, "bf16_tflops": 1900.2, "bf16_tflops_sustained": 1719.8}
    us, bound = p.roof_us(peaks)
    assert bound == "tensor" and us == pytest.approx(236.76e9 / 1900.2e12 * 1e6, rel=1e-4)
    us_s, _ = p.roof_us(peaks, sustained=True)
    assert us_s == pytest.approx(236.76e9 / 1719.8e12 * 1e6, rel=1e-4)


def test_kernel_passes_of_the_fused_backward():
    """The fused dgrad + wgrad kernel reads dy, z, the mask, x and W once and writes dx and dW:
    3 activations of the N=256 56x56 64-channel layer plus dx, two convolutions' FLOPs."""
    ks = {p.name: p for p in roofline.kernel_passes(CONFIGS[3], need_dx=True, fused=True)}
    assert set(ks) == {"conv_fprop_genstats", "bn_apply_relu", "bn_bwd_reduce", "conv_bwd_fused"}
    assert ks["conv_bwd_fused"].bytes == 4 * S3 + MASK3 + W3 + DW3
    assert ks["conv_bwd_fused"].flops == 2 * 59_190_018_048
    # without dx (weight gradient only): no dx write, no filter read, one convolution
    ks = {p.name: p for p in roofline.kernel_passes(CONFIGS[3], need_dx=False, fused=True)}
    assert ks["conv_bwd_fused"].bytes == 3 * S3 + MASK3 + DW3
    assert ks["conv_bwd_fused"].flops == 59_190_018_048
    # materialised dz: the dz pass writes one activation more than it reads beyond the reduction
    ks = {p.name: p for p in roofline.kernel_passes(CONFIGS[3], need_dx=True, fused=False)}
    assert ks["bn_dz"].bytes == 3 * S3 + MASK3
    assert ks["conv_wgrad"].bytes == 2 * S3 + DW3 and ks["conv_dgrad"].bytes == 2 * S3 + W3


def test_kernel_passes_of_the_persistent_forward():
    """The persistent forward reads x and W once and writes z, y and the mask in one kernel."""
    ks = {p.name: p for p in roofline.kernel_passes(CONFIGS[2], need_dx=True, fused=True, persist=True)}
    assert set(ks) == {"conv_fprop_apply", "bn_bwd_reduce", "conv_bwd_fused"}
    s2 = 32 * 56 * 56 * 64 * 2
    x2 = 32 * 56 * 56 * 64 * 2
    assert ks["conv_fprop_apply"].bytes == x2 + W3 + 2 * s2 + s2 // 16
    assert ks["conv_fprop_apply"].flops == 59_190_018_048 // 8
