"""Float64 CPU oracle for decode attention over a compacted KV cache.

TEST INFRASTRUCTURE ONLY.  Nothing in the product path imports this module:
only ``tests/``, ``__graft_entry__.smoke()`` and the CPU legs of ``bench.py``
may call it.  It shares no code with the CUDA library.

Source: the KV² page ("KV²가 전체 문맥 재계산 없이 KV 캐시를 압축한다",
onedev.kr/papers/598), section "전제와 한계" (assumptions and limits): the
compression it reports is headwise masking, so the cache is not physically
smaller; real decode savings need a compact serving backend that attends over
the physically compacted cache, whose length differs per (layer, KV head).

What the step computes (a plain reading; the page prints no formula): one
decoding query per query head attends, with ordinary softmax attention, over
the kept rows of its KV head only.  A "segment" is the run of kept rows of one
(layer, KV head) -- rows ``off .. off+len-1`` of the compacted K and V -- and
the G query heads of that KV head read it (grouped-query attention, query head
g of segment s is row ``q[s, g]``):

    z_i   = scale * (q . k_i)             for the len kept rows i
    lse   = log sum_i exp(z_i)            (natural log; -inf when len = 0)
    out   = sum_i exp(z_i - lse) * v_i    (0 when len = 0)

with scale = 1/sqrt(d) unless given.  Segment tables follow the layout the
headwise compaction writes: layer l starts at row Hkv * sum_{l'<l} k_{l'} and
KV head h of layer l at that plus h * k_l.
"""
from __future__ import annotations

import math

import numpy as np


def compact_segments(L: int, Hkv: int, k_per_layer) -> tuple[np.ndarray, np.ndarray]:
    """(row offset, length) of every (layer, KV head) segment of a compacted
    cache, in (layer, head) order."""
    off = np.zeros(L * Hkv, dtype=np.int64)
    ln = np.zeros(L * Hkv, dtype=np.int32)
    row = 0
    for l in range(L):
        for h in range(Hkv):
            off[l * Hkv + h] = row
            ln[l * Hkv + h] = int(k_per_layer[l])
            row += int(k_per_layer[l])
    return off, ln


def attend_one(Kseg: np.ndarray, Vseg: np.ndarray, q: np.ndarray, scale: float) -> tuple[np.ndarray, float]:
    """Softmax attention of one query over one segment (float64)."""
    n = Kseg.shape[0]
    if n == 0:
        return np.zeros(Vseg.shape[1] if Vseg.ndim == 2 else q.shape[0]), -math.inf
    z = scale * (Kseg @ q)
    zmax = float(np.max(z))
    w = np.exp(z - zmax)
    lse = zmax + math.log(float(np.sum(w)))
    a = np.exp(z - lse)
    return a @ Vseg, lse


def decode_attention(Kc: np.ndarray, Vc: np.ndarray, seg_off, seg_len, q: np.ndarray, scale: float | None = None):
    """Decode attention of every segment.

    Kc, Vc: float64 [rows][d]; q: float64 [n_seg][G][d].
    Returns out float64 [n_seg][G][d] and lse float64 [n_seg][G]."""
    n_seg, G, d = q.shape
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    out = np.zeros((n_seg, G, d))
    lse = np.zeros((n_seg, G))
    for s in range(n_seg):
        o, n = int(seg_off[s]), int(seg_len[s])
        Ks, Vs = Kc[o:o + n], Vc[o:o + n]
        for g in range(G):
            out[s, g], lse[s, g] = attend_one(Ks, Vs, q[s, g], scale)
    return out, lse


def abs_weighted(Kc, Vc, seg_off, seg_len, q, scale=None):
    """sum_i softmax_i * |v_i| per output element: the natural scale of the
    rounding error of a weighted sum (used to set parity tolerances)."""
    n_seg, G, d = q.shape
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    res = np.zeros((n_seg, G, d))
    for s in range(n_seg):
        o, n = int(seg_off[s]), int(seg_len[s])
        if n == 0:
            continue
        for g in range(G):
            z = scale * (Kc[o:o + n] @ q[s, g])
            a = np.exp(z - z.max())
            a /= a.sum()
            res[s, g] = a @ np.abs(Vc[o:o + n])
    return res
