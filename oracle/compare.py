"""Parity checks between the CUDA path and the oracle (test infrastructure).

Tolerances follow the parity bar: scores within 1e-3 relative (bf16 inputs,
fp32 accumulation on the GPU, float64 here); selected / kept index sets exact
in count and exact as sets except for positions whose oracle score lies
within 1e-4 relative of the selection threshold; compacted rows bit-exact.
"""
from __future__ import annotations

import numpy as np

SCORE_RTOL = 1e-3
PROXY_FLOOR = 1e-3   # cosines cross zero: |gpu - ref| <= 1e-3 * max(|ref|, 1e-3)
TIE_REL = 1e-4


def score_errors(gpu: np.ndarray, ref: np.ndarray, rtol: float = SCORE_RTOL, floor: float = 0.0):
    """Indices where |gpu - ref| > rtol * max(|ref|, floor) (NaN in ref skipped)."""
    gpu = np.asarray(gpu, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    m = ~np.isnan(ref)
    bound = rtol * np.maximum(np.abs(ref), floor)
    bad = m & ~(np.abs(gpu - ref) <= bound)
    return np.nonzero(bad)


def assert_scores(gpu, ref, rtol=SCORE_RTOL, floor=0.0, what="scores"):
    bad = score_errors(gpu, ref, rtol, floor)
    if len(bad[0]):
        g = np.asarray(gpu, np.float64)[bad]
        r = np.asarray(ref, np.float64)[bad]
        k = np.argmax(np.abs(g - r) / np.maximum(np.abs(r), max(floor, 1e-300)))
        raise AssertionError(f"{what}: {len(bad[0])} entries outside rtol={rtol} (floor {floor}); "
                             f"worst at {tuple(int(b[k]) for b in bad)}: gpu={g[k]!r} ref={r[k]!r}")


def assert_topk_set(gpu_idx, ref_vals, lo: int, hi: int, n: int, forced=(), what="set", rel=TIE_REL):
    """The GPU's chosen positions of [lo, hi) (plus ``forced`` positions that
    must be present) against the oracle values: exact count, ascending, and
    the same set up to near-ties of the n-th largest oracle value."""
    gpu_idx = np.asarray(gpu_idx, dtype=np.int64)
    forced = list(forced)
    assert len(gpu_idx) == n + len(forced), f"{what}: count {len(gpu_idx)} != {n + len(forced)}"
    assert np.all(np.diff(gpu_idx) > 0), f"{what}: not strictly ascending"
    assert set(forced) <= set(gpu_idx.tolist()), f"{what}: forced positions missing"
    body = np.array([i for i in gpu_idx.tolist() if i not in set(forced)], dtype=np.int64)
    if n == 0:
        assert len(body) == 0
        return
    assert body.min() >= lo and body.max() < hi, f"{what}: index outside [{lo}, {hi})"
    v = np.asarray(ref_vals, dtype=np.float64)[lo:hi]
    v = np.where(np.isnan(v), -np.inf, v)
    order = sorted(range(hi - lo), key=lambda i: (-v[i], i))
    ref_set = set(lo + i for i in order[:n])
    tau = v[order[n - 1]]
    band = rel * abs(tau) if np.isfinite(tau) else 0.0
    got = set(body.tolist())
    for i in got - ref_set:
        assert v[i - lo] >= tau - band, f"{what}: kept {i} (ref {v[i - lo]!r}) below threshold {tau!r}"
    for i in ref_set - got:
        assert v[i - lo] <= tau + band, f"{what}: dropped {i} (ref {v[i - lo]!r}) above threshold {tau!r}"
