"""Pins of the EpiCache per-turn oracle ("[26'ICML] EpiCache", "방법: 3단계"
step ③, Fig. 3): question-to-episode matching and the packed episode cache."""
import json
import os

import numpy as np
import pytest
from scipy.spatial.distance import cdist

from oracle import decode, episode, kv2

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def test_match_hand_worked():
    g = json.load(open(os.path.join(GOLD, "episode_match_small.json")))
    Q, C = np.array(g["queries"], float), np.array(g["centroids"], float)
    ep, d2 = episode.nearest_episode(Q, C)
    np.testing.assert_array_equal(d2, g["d2"])
    assert ep.tolist() == g["episode"]
    ep_t, _ = episode.nearest_episode(Q, C, tau=g["tau"])
    assert ep_t.tolist() == g["episode_tau"]


def test_match_against_scipy_and_argmin():
    rng = np.random.default_rng(0)
    Q, C = rng.standard_normal((40, 64)), rng.standard_normal((7, 64))
    ep, d2 = episode.nearest_episode(Q, C)
    np.testing.assert_allclose(d2, cdist(Q, C, "sqeuclidean"), rtol=1e-12)
    assert ep.tolist() == np.argmin(cdist(Q, C), axis=1).tolist()


def test_ties_go_to_lower_index_and_threshold_is_inclusive():
    C = np.array([[1.0, 0.0], [0.0, 1.0], [1.0, 0.0]])
    ep, _ = episode.nearest_episode(np.array([[0.5, 0.5], [2.0, 0.0]]), C)
    assert ep.tolist() == [0, 0]
    ep, _ = episode.nearest_episode(np.array([[4.0, 0.0]]), C, tau=3.0)      # distance exactly 3
    assert ep.tolist() == [0]
    ep, _ = episode.nearest_episode(np.array([[4.0 + 1e-9, 0.0]]), C, tau=3.0)
    assert ep.tolist() == [-1]


def test_unit_vectors_match_by_cosine():
    rng = np.random.default_rng(1)
    Q = rng.standard_normal((30, 16))
    C = rng.standard_normal((5, 16))
    Q /= np.linalg.norm(Q, axis=1, keepdims=True)
    C /= np.linalg.norm(C, axis=1, keepdims=True)
    ep, _ = episode.nearest_episode(Q, C)
    assert ep.tolist() == np.argmax(Q @ C.T, axis=1).tolist()


def test_pack_is_the_compacted_layout():
    rng = np.random.default_rng(2)
    L, H, N, d = 3, 2, 30, 8
    X = rng.standard_normal((L, H, N, d))
    kl = [5, 9, 4]
    kept = kv2.evict(rng.random((L, H, N)), 2, kl)
    Kc = kv2.compact(X, kept)
    K, V, P, lens = episode.pack_cache(Kc, Kc, [k for k in kept])
    assert lens == kl
    off, ln = decode.compact_segments(L, H, kl)
    for l in range(L):
        for h in range(H):
            s = l * H + h
            np.testing.assert_array_equal(K[off[s]:off[s] + ln[s]], X[l, h][kept[l][h]])
            np.testing.assert_array_equal(P[off[s]:off[s] + ln[s]], kept[l][h])
