"""The seeded input recipe shared by the GPU tests, the oracle and the benchmark (CPU only):
shapes and dtypes of the five workloads, determinism per seed, and the stated distributions
(x ~ N(0,1) or U(-2.5,2.5), Kaiming-normal W, gamma ~ U(0.5,1.5), beta ~ N(0,0.1^2),
running statistics 0/1, dy ~ N(0,1)), checked on draws large enough for tight bounds."""
import math

import pytest
import torch

from conv_batchnorm_relu_gb300.inputs import CONFIGS, CBRSpec, make_inputs, seed_for


def test_workload_shapes_and_dtypes():
    expect = {1: ((2, 8, 8, 8), (16, 3, 3, 8), torch.float16),
              2: ((32, 56, 56, 64), (64, 3, 3, 64), torch.float16),
              3: ((256, 56, 56, 64), (64, 3, 3, 64), torch.float16),
              4: ((256, 224, 224, 3), (64, 7, 7, 3), torch.float16),
              5: ((64, 112, 112, 128), (128, 3, 3, 128), torch.bfloat16)}
    outs = {1: (8, 8), 2: (56, 56), 3: (56, 56), 4: (112, 112), 5: (112, 112)}
    for k, (xs, ws, dt) in expect.items():
        spec = CONFIGS[k]
        assert (spec.n, spec.h, spec.w, spec.c_in) == xs
        assert (spec.c_out, spec.r, spec.s, spec.c_in) == ws
        assert spec.torch_dtype == dt
        assert (spec.p, spec.q) == outs[k]
        assert seed_for(k) == 1234 + k
    assert CONFIGS[4].first_layer and CONFIGS[4].stride == 2 and CONFIGS[4].pad == 3
    assert CONFIGS[5].infer


def test_draws_are_deterministic_per_seed():
    spec = CONFIGS[1]
    a, b, c = make_inputs(spec, 7), make_inputs(spec, 7), make_inputs(spec, 8)
    for k in a:
        assert torch.equal(a[k], b[k]), k
    assert not torch.equal(a["x"], c["x"])


def test_distributions_follow_the_recipe():
    spec = CBRSpec("stats", n=8, h=32, w=32, c_in=64, c_out=128)
    d = make_inputs(spec, 99)
    x = d["x"].float()
    assert abs(x.mean().item()) < 0.01 and abs(x.std().item() - 1.0) < 0.01
    w = d["w"].float()
    kaiming = math.sqrt(2.0 / (64 * 3 * 3))
    assert abs(w.std().item() / kaiming - 1.0) < 0.02
    g = d["gamma"]
    assert g.dtype == torch.float32 and g.min().item() >= 0.5 and g.max().item() <= 1.5
    assert abs(d["beta"].std().item() - 0.1) < 0.03
    assert torch.equal(d["running_mean"], torch.zeros(128)) and torch.equal(d["running_var"], torch.ones(128))
    dy = d["dy"].float()
    assert dy.shape == (8, 32, 32, 128) and abs(dy.std().item() - 1.0) < 0.01
    first = make_inputs(CBRSpec("img", n=2, h=64, w=64, c_in=3, c_out=64, r=7, s=7, stride=2, pad=3,
                                x_dist="uniform2.5", first_layer=True), 5, with_dy=False)
    xf = first["x"].float()
    assert xf.min().item() >= -2.5 and xf.max().item() <= 2.5
    assert abs(xf.std().item() - 5.0 / math.sqrt(12.0)) < 0.02
    assert "dy" not in first


@pytest.mark.parametrize("dt", ["f16", "bf16"])
def test_x_is_the_first_draw_rounded_to_the_storage_dtype(dt):
    """x is drawn first from the seeded generator and cast (RNE) to the storage dtype."""
    spec = CBRSpec("r", n=1, h=4, w=4, c_in=8, c_out=16, dtype=dt)
    d = make_inputs(spec, 3)
    g = torch.Generator("cpu").manual_seed(3)
    x32 = torch.randn((1, 4, 4, 8), generator=g, dtype=torch.float32)
    assert torch.equal(d["x"], x32.to(spec.torch_dtype))
