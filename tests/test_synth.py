"""The seeded input generator: bf16 rounding and planted needles."""
import math

import numpy as np
import torch

import kv_synth as ks


def test_bf16_rounding_matches_torch():
    rng = np.random.default_rng(0)
    x = np.concatenate([rng.standard_normal(100000).astype(np.float32) * 10,
                        np.array([0.0, -0.0, 1e-40, -1e-40, 3.0e38, 1.00390625, 1.01171875], np.float32)])
    ours = ks.f32_to_bf16_bits(x)
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    np.testing.assert_array_equal(ours, ref)
    np.testing.assert_array_equal(ks.bf16_bits_to_f32(ours),
                                  torch.from_numpy(ours.view(np.int16)).view(torch.bfloat16).float().numpy())


def test_tiny_generator_deterministic_and_needles():
    a = ks.gen_kv2(ks.TINY)
    b = ks.gen_kv2(ks.TINY, threads=1)
    np.testing.assert_array_equal(a.K, b.K)
    np.testing.assert_array_equal(a.Q, b.Q)
    assert a.K.shape == (1, 1, 4096, 128) and a.Q.shape == (1, 4, 4096, 128)
    assert len(a.needles[0]) == 8
    G = ks.TINY.G
    for g, pq, pk in a.needles[0]:
        q = ks.bf16_bits_to_f32(a.Q[0, g, pq]).astype(np.float64)
        for t in range(4):
            k = ks.bf16_bits_to_f32(a.K[0, g // G, pk + t]).astype(np.float64)
            assert abs(q @ k / math.sqrt(128) - ks.NEEDLE_LOGIT) < 0.1
        assert pk >= ks.TINY.sinks


def test_layers_regenerate_independently():
    cfg = ks.scaled(ks.TINY, L=3, N=512, needles_per_layer=4)
    allk = ks.gen_kv2(cfg)
    one = ks.gen_layer(cfg, 2)
    np.testing.assert_array_equal(allk.K[2], one.K)


def test_sensitivity_range():
    s = ks.gen_sensitivity(ks.EPI_3B)
    assert s.shape == (28,) and s.min() >= 0.5 and s.max() <= 1.5
