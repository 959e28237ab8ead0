"""Pins of the decode-attention oracle (compact serving backend of the KV²
page, "전제와 한계") against closed forms, a library attention routine, the
compaction layout of the compression oracle, and hand-worked segment tables.
"""
import math

import numpy as np
import pytest
import torch
from scipy.special import logsumexp, softmax

from oracle import decode, kv2


def test_equal_keys_give_mean_of_values():
    rng = np.random.default_rng(1)
    d, n = 16, 37
    k = rng.standard_normal(d)
    K = np.tile(k, (n, 1))
    V = rng.standard_normal((n, d))
    q = rng.standard_normal(d)
    out, lse = decode.attend_one(K, V, q, 0.25)
    np.testing.assert_allclose(out, V.mean(axis=0), rtol=1e-13, atol=1e-15)
    assert lse == pytest.approx(0.25 * float(q @ k) + math.log(n), abs=1e-12)


def test_single_key_returns_its_value():
    rng = np.random.default_rng(2)
    K, V, q = rng.standard_normal((1, 8)), rng.standard_normal((1, 8)), rng.standard_normal(8)
    out, lse = decode.attend_one(K, V, q, 1 / math.sqrt(8))
    np.testing.assert_array_equal(out, V[0])
    assert lse == pytest.approx(float(K[0] @ q) / math.sqrt(8), abs=1e-14)


def test_needle_dominates():
    rng = np.random.default_rng(3)
    d, n = 32, 500
    K = rng.standard_normal((n, d)) * 0.01
    q = rng.standard_normal(d)
    K[123] = 80.0 * q / (q @ q)                 # logit 80 at scale 1, others ~0
    V = rng.standard_normal((n, d))
    out, _ = decode.attend_one(K, V, q, 1.0)
    np.testing.assert_allclose(out, V[123], rtol=0, atol=n * math.exp(-75) * np.abs(V).max())


def test_identity_values_expose_the_weights():
    rng = np.random.default_rng(4)
    n = 12
    K = rng.standard_normal((n, n))
    q = rng.standard_normal(n)
    out, lse = decode.attend_one(K, np.eye(n), q, 0.3)
    np.testing.assert_allclose(out, softmax(0.3 * (K @ q)), rtol=1e-13)
    assert lse == pytest.approx(float(logsumexp(0.3 * (K @ q))), abs=1e-13)
    assert out.sum() == pytest.approx(1.0, abs=1e-14)


def test_empty_segment():
    out, lse = decode.decode_attention(np.zeros((4, 8)), np.zeros((4, 8)), [2], [0], np.ones((1, 3, 8)))
    assert np.all(out == 0) and np.all(np.isneginf(lse))


@pytest.mark.parametrize("G", [1, 3, 4])
def test_against_torch_sdpa_gqa(G):
    """GQA decode over ragged segments equals torch's scaled_dot_product_attention
    (float64, math kernel) run segment by segment."""
    rng = np.random.default_rng(10 + G)
    d = 16
    lens = [5, 1, 40, 17]
    off = np.concatenate([[0], np.cumsum(lens)[:-1]]) + 3   # leading unused rows
    rows = int(off[-1] + lens[-1] + 2)
    Kc, Vc = rng.standard_normal((rows, d)), rng.standard_normal((rows, d))
    q = rng.standard_normal((len(lens), G, d))
    out, lse = decode.decode_attention(Kc, Vc, off, lens, q)
    for s, (o, n) in enumerate(zip(off, lens)):
        Kt = torch.from_numpy(Kc[o:o + n]).expand(G, n, d)[None]
        Vt = torch.from_numpy(Vc[o:o + n]).expand(G, n, d)[None]
        qt = torch.from_numpy(q[s])[None, :, None, :]
        ref = torch.nn.functional.scaled_dot_product_attention(qt, Kt, Vt)[0, :, 0].numpy()
        np.testing.assert_allclose(out[s], ref, rtol=1e-12, atol=1e-13)
        ref_lse = torch.logsumexp(qt[0, :, 0] @ Kt[0, 0].T / math.sqrt(d), dim=-1).numpy()
        np.testing.assert_allclose(lse[s], ref_lse, rtol=1e-13)


def test_segment_table_hand_worked():
    off, ln = decode.compact_segments(2, 2, [3, 5])
    assert off.tolist() == [0, 3, 6, 11] and ln.tolist() == [3, 3, 5, 5]


def test_segment_table_indexes_the_compaction():
    """Rows of a segment are exactly that (layer, head)'s compacted rows as the
    compression oracle lays them out (layer-major, head-major, ascending)."""
    rng = np.random.default_rng(5)
    L, H, N, d = 3, 2, 20, 4
    X = rng.standard_normal((L, H, N, d))
    score = rng.random((L, H, N))
    kl = [6, 4, 9]
    kept = kv2.evict(score, 2, kl)
    Xc = kv2.compact(X, kept)
    flat = np.concatenate([Xc[l].reshape(-1, d) for l in range(L)])
    off, ln = decode.compact_segments(L, H, kl)
    for l in range(L):
        for h in range(H):
            s = l * H + h
            np.testing.assert_array_equal(flat[off[s]:off[s] + ln[s]], X[l, h][kept[l][h]])


def test_abs_weighted_bounds_output():
    rng = np.random.default_rng(6)
    Kc, Vc = rng.standard_normal((50, 8)), rng.standard_normal((50, 8))
    q = rng.standard_normal((2, 2, 8))
    out, _ = decode.decode_attention(Kc, Vc, [0, 20], [20, 30], q)
    bound = decode.abs_weighted(Kc, Vc, [0, 20], [20, 30], q)
    assert np.all(np.abs(out) <= bound + 1e-15)
