"""Pins of the Q4 codec oracle (persistent Q4 KV cache page, "방법론 및
시스템 설계"): bf16 directed rounding against brute force and torch, a
hand-worked row with a rounding tie, exact integer and constant groups, nibble
order, grid coverage and the error bound."""
import json
import os

import numpy as np
import torch

from oracle import q4

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def bf16_neighbours(x):
    """All bf16 values within two ulps of float32 x (brute force)."""
    b = np.float32(x).view(np.uint32) & np.uint32(0xFFFF0000)
    cands = []
    for k in range(-2, 3):
        v = (np.int64(b) + k * 0x10000) & 0xFFFFFFFF
        cands.append(np.uint32(v).view(np.float32))
    return [float(c) for c in cands if np.isfinite(c)]


def test_bf16_rounding_against_brute_force_and_torch():
    rng = np.random.default_rng(0)
    x = (rng.standard_normal(3000) * np.exp(rng.uniform(-20, 20, 3000))).astype(np.float32)
    x[:10] = [0.0, -0.0, 1.0, -1.0, 0.2, -0.2, 3.0, 1e-30, -1e-30, 65504.0]
    dn, up, rn = q4.bf16_round_down(x), q4.bf16_round_up(x), q4.bf16_round_nearest(x)
    for i, xi in enumerate(x):
        nb = bf16_neighbours(xi)
        assert dn[i] == max(v for v in nb if v <= xi)
        assert up[i] == min(v for v in nb if v >= xi)
    ref = torch.from_numpy(x).to(torch.bfloat16).float().numpy()
    np.testing.assert_array_equal(rn, ref)


def test_hand_worked_row_with_tie():
    g = json.load(open(os.path.join(GOLD, "q4_small.json")))
    row = np.full(128, g["group0_fill"], np.float32)
    row[:3] = g["group0_values"]
    row[64:] = g["group1_const"]
    c, s, lo = q4.encode(row[None])
    assert s[0].tolist() == g["step"] and lo[0].tolist() == g["offset"]
    assert c[0, :3].tolist() == g["group0_codes"] and np.all(c[0, 64:] == 0)
    x = q4.decode(c, s, lo)
    assert x[0, :3].tolist() == g["group0_decoded"] and np.all(x[0, 64:] == g["group1_const"])
    assert q4.pack_codes(c)[0, :2].tolist() == g["packed_first_bytes"]


def test_integer_group_is_exact():
    row = np.tile(np.arange(16, dtype=np.float32), 8)[None]
    c, s, lo = q4.encode(row)
    assert np.all(s == 1.0) and np.all(lo == 0.0)
    assert c[0].tolist() == row[0].astype(int).tolist()
    np.testing.assert_array_equal(q4.decode(c, s, lo), row)


def test_pack_round_trip_and_nibble_order():
    rng = np.random.default_rng(1)
    c = rng.integers(0, 16, size=(5, 128), dtype=np.uint8)
    p = q4.pack_codes(c)
    assert p.shape == (5, 64) and p[0, 0] == (c[0, 0] | (c[0, 1] << 4))
    np.testing.assert_array_equal(q4.unpack_codes(p), c)


def test_grid_covers_group_and_error_bound():
    rng = np.random.default_rng(2)
    X = (rng.standard_normal((400, 128)) * np.exp(rng.uniform(-3, 3, (400, 1)))).astype(np.float32)
    X = q4.bf16_round_nearest(X)                       # cache values are bf16
    c, s, lo = q4.encode(X)
    Xg = X.reshape(400, 2, 64)
    assert np.all(lo <= Xg.min(axis=2)) and np.all(lo + 15 * s.astype(np.float64) >= Xg.max(axis=2))
    assert np.all(c <= 15)
    Y = q4.decode(c, s, lo).reshape(400, 2, 64)
    err = np.abs(Y.astype(np.float64) - Xg)
    bound = s[:, :, None] / 2 * (1 + 1e-6) + np.abs(Y) * 2.0 ** -8 + 1e-30
    assert np.all(err <= bound)
