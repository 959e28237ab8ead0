"""Float64 CPU oracle for EpiCache's per-turn path: matching a question to
its episode and packing an episode's compressed cache for the swap.

TEST INFRASTRUCTURE ONLY.  Nothing in the product path imports this module:
only ``tests/``, ``__graft_entry__.smoke()`` and the CPU legs of ``bench.py``
may call it.  It shares no code with the CUDA library.

Source: "[26'ICML] EpiCache" (juyoungkimmy-kim.github.io), section "방법:
3단계" steps ① and ③ and Fig. 3.  Conversation segments are embedded and
clustered with K-means into E episodes; each turn the new question is embedded
and the closest episode's compressed cache is brought in to answer (a
completely new topic gets a new cache); the idle caches wait in CPU memory or
storage, and the page times the swap (load + write back) separately from the
matching.

Readings (the page prints no formula):
* "closest" is the K-means assignment rule: the smallest Euclidean distance
  from the question embedding to an episode centroid; equal distances go to
  the lower episode index;
* "a completely new topic": the closest centroid is farther than a caller
  threshold tau (Euclidean); the match is then -1;
* the cache that is swapped is the episode's kept rows only, laid out as the
  headwise compaction lays them out (layer-major, then KV head, positions in
  cache order), with the global positions alongside.
"""
from __future__ import annotations

import numpy as np


def nearest_episode(queries: np.ndarray, centroids: np.ndarray, tau: float | None = None):
    """queries float64 [B][De], centroids [E][De] -> (episode int64 [B],
    squared distances float64 [B][E]).  Ties go to the lower index; with tau,
    a question farther than tau from every centroid gets -1."""
    B, E = queries.shape[0], centroids.shape[0]
    d2 = np.zeros((B, E))
    for b in range(B):
        for e in range(E):
            diff = queries[b] - centroids[e]
            d2[b, e] = float(diff @ diff)
    ep = np.full(B, -1, dtype=np.int64)
    for b in range(B):
        best = 0
        for e in range(1, E):
            if d2[b, e] < d2[b, best]:
                best = e
        if tau is None or d2[b, best] <= tau * tau:
            ep[b] = best
    return ep, d2


def pack_cache(layers_K, layers_V, layers_pos):
    """Concatenate an episode cache held per layer (arrays [Hkv][len_l][...])
    into the contiguous compacted layout: rows of (layer 0, head 0), (layer 0,
    head 1), ...; returns (K rows, V rows, positions, per-layer lengths)."""
    K = np.concatenate([k.reshape(-1, k.shape[-1]) for k in layers_K])
    V = np.concatenate([v.reshape(-1, v.shape[-1]) for v in layers_V])
    P = np.concatenate([p.reshape(-1) for p in layers_pos])
    return K, V, P, [k.shape[1] for k in layers_K]
