"""The seeded input generator: determinism, slice regeneration, distribution, recipes."""

import math

import numpy as np
import torch

import synth


def test_same_seed_same_bits_and_slices_regenerate():
    a = synth.normal((4096,), 7, 2, synth.W_UP)
    b = synth.normal((4096,), 7, 2, synth.W_UP)
    assert torch.equal(a, b)
    part = synth.normal_f64(1000, 500, 7, 2, synth.W_UP).float()
    assert torch.equal(a[1000:1500], part)


def test_streams_differ_by_seed_layer_and_tensor():
    base = synth.normal((256,), 0, 0, 0)
    for args in ((1, 0, 0), (0, 1, 0), (0, 0, 1)):
        other = synth.normal((256,), *args)
        assert not torch.equal(base, other)
        assert abs(float(torch.corrcoef(torch.stack([base, other]))[0, 1])) < 0.2


def test_standard_normal_moments():
    v = synth.normal_f64(0, 1 << 20, 11, 0, 0).numpy()
    n = v.size
    assert abs(v.mean()) < 5 / math.sqrt(n)
    assert abs(v.var() - 1.0) < 5 * math.sqrt(2.0 / n)
    assert abs(np.mean(v ** 3)) < 5 * math.sqrt(15.0 / n)
    assert abs(np.mean(v ** 4) - 3.0) < 5 * math.sqrt(96.0 / n)
    # tail mass beyond 3 sigma: 0.0027
    assert abs(np.mean(np.abs(v) > 3.0) - 0.0026998) < 0.0005


def test_weight_scales_follow_fan_in():
    shape = synth.LayerShape("t", 256, 512, 4, 2, "bf16")
    wg, wu, wd = synth.expert_weights(shape, 0)
    assert wg.dtype == torch.bfloat16 and wg.shape == (4, 256, 512) and wd.shape == (4, 512, 256)
    assert abs(wg.float().std().item() - 1 / 16) < 1e-3
    assert abs(wd.float().std().item() - 1 / math.sqrt(512)) < 1e-3
    wr = synth.router_weight(shape, 0)
    assert wr.shape == (256, 4)


def test_router_offset_recipes():
    z = synth.router_offset(synth.QWEN2)
    assert z.shape == (64,) and z[0].item() == 0.0
    assert z[9].item() == np.float32(-1.1 * math.log(10.0))
    assert torch.all(z[1:] < z[:-1])
    m = synth.router_offset(synth.DEEPSEEK_MASKED)
    assert int(torch.isinf(m).sum()) == 32 and torch.all(torch.isinf(m[3::4]))
    assert synth.router_offset(synth.DEEPSEEK) is None
