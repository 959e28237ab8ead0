"""Pins of the float64 oracle against closed forms, hand-worked fixtures,
library routines and brute force -- nothing here re-runs the oracle's own
formula to check itself.

Fixtures live in tests/golden/*.json, each citing the page section it follows.
"""
import itertools
import json
import math
import os

import numpy as np
import pytest
import torch

from oracle import kv2

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def gold(name):
    with open(os.path.join(GOLD, name)) as f:
        return json.load(f)


# ---------------------------------------------------------------------------
# KeyDiff proxy
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("case", gold("keydiff_closed_forms.json")["cases"], ids=lambda c: c["name"])
def test_keydiff_closed_forms(case):
    s = kv2.keydiff_head(np.array(case["keys"], dtype=np.float64))
    np.testing.assert_allclose(s, case["s"], atol=1e-15)


def test_keydiff_mean_over_heads():
    g = gold("keydiff_closed_forms.json")["mean_over_heads"]
    K = np.array(g["heads"], dtype=np.float64)[None]       # [L=1, H=2, N, d]
    p, s = kv2.proxy_scores(K)
    np.testing.assert_allclose(p, g["p"], atol=1e-15)
    # layers and heads are interchangeable in the mean
    p2, _ = kv2.proxy_scores(np.array(g["heads"], dtype=np.float64)[:, None])
    np.testing.assert_allclose(p2, g["p"], atol=1e-15)


def test_keydiff_parallel_keys_all_minus_one():
    rng = np.random.default_rng(1)
    v = rng.standard_normal(16)
    K = rng.uniform(0.1, 5.0, size=(50, 1)) * v[None]
    np.testing.assert_allclose(kv2.keydiff_head(K), -1.0, atol=1e-14)


def test_keydiff_per_token_scale_invariance():
    rng = np.random.default_rng(2)
    K = rng.standard_normal((64, 32))
    c = rng.uniform(0.01, 100.0, size=(64, 1))
    np.testing.assert_allclose(kv2.keydiff_head(K * c), kv2.keydiff_head(K), atol=1e-13)


def test_keydiff_bounded_and_sign():
    rng = np.random.default_rng(3)
    K = rng.standard_normal((200, 16)) + 3.0
    s = kv2.keydiff_head(K)
    assert np.all(s <= 1 + 1e-15) and np.all(s >= -1 - 1e-15)
    # a key pointing away from the common offset scores highest
    K[17] = -K[17]
    assert int(np.argmax(kv2.keydiff_head(K))) == 17


def test_keydiff_matches_cosine_library_routine():
    """scipy's cosine distance restates cos independently: s = cos_dist - 1."""
    from scipy.spatial.distance import cdist
    rng = np.random.default_rng(4)
    K = rng.standard_normal((40, 8)) + np.array([2.0] + [0.0] * 7)
    unit = K / np.linalg.norm(K, axis=1, keepdims=True)
    u = unit.mean(axis=0, keepdims=True)
    ref = cdist(K, u, metric="cosine")[:, 0] - 1.0
    np.testing.assert_allclose(kv2.keydiff_head(K), ref, atol=1e-13)


def test_knorm_closed_forms_and_aggregate():
    """Knorm: s = -|k|; 3-4-5 keys, a zero key, scaling a key scales its
    score, and p is the head mean."""
    K = np.array([[3.0, 4.0], [0.0, 0.0], [6.0, 8.0], [-1.0, 0.0]])
    np.testing.assert_allclose(kv2.knorm_head(K), [-5.0, 0.0, -10.0, -1.0], atol=0)
    rng = np.random.default_rng(8)
    X = rng.standard_normal((30, 16))
    c = rng.uniform(0.1, 10.0, size=(30, 1))
    np.testing.assert_allclose(kv2.knorm_head(X * c), kv2.knorm_head(X) * c[:, 0], rtol=1e-13)
    np.testing.assert_allclose(-kv2.knorm_head(X), np.linalg.norm(X, axis=1), rtol=1e-14)
    p, s = kv2.proxy_scores(np.stack([K[None], 2 * K[None]]), kind="knorm")
    np.testing.assert_allclose(p, [-7.5, 0.0, -15.0, -1.5], atol=0)


# ---------------------------------------------------------------------------
# Chunk plan and query selection
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("case", gold("nq_table.json")["cases"], ids=lambda c: f"N{c['N']}")
def test_chunk_plan_table(case):
    ch = kv2.chunk_plan(case["N"], case["S"], case["m"], case["rho"])
    assert [c.hi - c.lo for c in ch] == case["sizes"]
    assert [c.nq for c in ch] == case["nq"]
    assert sum(c.nq for c in ch) == case["Q"]
    assert ch[0].lo == case["S"] and ch[-1].hi == case["N"]
    assert [c.off for c in ch] == list(np.cumsum([0] + case["nq"][:-1]))


def test_select_small_golden():
    g = gold("select_small.json")
    sel, ch = kv2.select_queries(np.array(g["p"], dtype=np.float64), g["N"], g["S"], g["m"], g["rho"])
    assert [[c.lo, c.hi] for c in ch] == g["chunks"]
    assert [c.nq for c in ch] == g["nq"]
    assert sel.tolist() == g["sel"]


def _is_top_set(vals, lo, hi, chosen):
    """Brute-force characterisation: every chosen position outranks every
    unchosen one (higher value, or equal value and lower position)."""
    chosen = set(chosen)
    for i in chosen:
        for j in range(lo, hi):
            if j in chosen:
                continue
            if not (vals[i] > vals[j] or (vals[i] == vals[j] and i < j)):
                return False
    return True


@pytest.mark.parametrize("seed", range(6))
def test_select_brute_force_with_ties(seed):
    rng = np.random.default_rng(seed)
    N, S, m = 37, 3, 8
    p = rng.integers(0, 4, size=N).astype(np.float64)    # many ties
    rho = [0.25, 0.5, 0.8, 1.0, 0.01, 0.3][seed]
    sel, ch = kv2.select_queries(p, N, S, m, rho)
    for c in ch:
        got = sel[c.off:c.off + c.nq].tolist()
        assert got == sorted(got) and len(got) == c.nq
        assert _is_top_set(p, c.lo, c.hi, got)
        # library cross-check: stable argsort on -p
        ref = np.sort(c.lo + np.argsort(-p[c.lo:c.hi], kind="stable")[:c.nq])
        assert got == ref.tolist()


def test_select_exhaustive_tiny():
    """All n-subsets of a 6-position chunk: exactly one satisfies the rank
    property and it is the selected one."""
    rng = np.random.default_rng(11)
    for _ in range(20):
        p = rng.integers(0, 3, size=8).astype(np.float64)
        sel, ch = kv2.select_queries(p, 8, 2, 6, 0.5)
        winners = [c for c in itertools.combinations(range(2, 8), 3) if _is_top_set(p, 2, 8, c)]
        assert len(winners) == 1 and list(winners[0]) == sel.tolist()


def test_select_rho_one_is_whole_chunk():
    p = np.random.default_rng(5).standard_normal(50)
    sel, ch = kv2.select_queries(p, 50, 4, 16, 1.0)
    assert sel.tolist() == list(range(4, 50))


def test_select_nan_ranks_lowest():
    p = np.array([0, 0, np.nan, 1.0, np.nan, -5.0])
    sel, _ = kv2.select_queries(p, 6, 2, 4, 0.5)
    assert sel.tolist() == [3, 5]


# ---------------------------------------------------------------------------
# Reconstruction scoring
# ---------------------------------------------------------------------------
def _explicit_scores(K, Q, sel, chunks, G):
    """Independent restatement through torch's scaled_dot_product_attention
    (float64, math backend): for each chunk the appended sequence is
    [cache keys, appended keys]; V = identity recovers the attention matrix;
    the score is the max over the chunk's query rows and the group's heads."""
    H, N, d = K.shape
    out = np.full((H, N), np.nan)
    for h in range(H):
        for c in chunks:
            idx = sel[c.off:c.off + c.nq]
            keys = np.concatenate([K[h], K[h][idx]], axis=0)           # [N+nq, d]
            T = keys.shape[0]
            mask = np.ones((c.nq, T), dtype=bool)
            mask[:, N:] = np.tril(np.ones((c.nq, c.nq), dtype=bool))
            eye = torch.eye(T, dtype=torch.float64)
            best = np.zeros(c.hi - c.lo)
            for g in range(G):
                q = torch.from_numpy(Q[h * G + g][idx])
                A = torch.nn.functional.scaled_dot_product_attention(
                    q[None, None], torch.from_numpy(keys)[None, None], eye[None, None],
                    attn_mask=torch.from_numpy(mask)[None, None]).numpy()[0, 0]
                assert np.allclose(A.sum(axis=1), 1.0, atol=1e-12)
                best = np.maximum(best, A[:, c.lo:c.hi].max(axis=0))
            out[h, c.lo:c.hi] = best
    return out


@pytest.mark.parametrize("rho,G", [(0.25, 2), (1.0, 2), (0.5, 1), (0.4, 3)])
def test_recon_matches_explicit_attention(rho, G):
    rng = np.random.default_rng(int(rho * 100) + G)
    H, N, d, S, m = 2, 16, 8, 2, 5
    K = rng.standard_normal((1, H, N, d)) * 1.5
    Q = rng.standard_normal((1, H * G, N, d)) * 1.5
    p = rng.standard_normal(N)
    sel, ch = kv2.select_queries(p, N, S, m, rho)
    score, lse = kv2.recon_scores(K, Q, sel, ch)
    ref = _explicit_scores(K[0], Q[0], sel, ch, G)
    assert np.all(np.isnan(score[0, :, :S]))
    np.testing.assert_allclose(score[0, :, S:], ref[:, S:], rtol=1e-12, atol=0)


def test_recon_rho_one_full_query_scoring():
    """rho = 1: every chunk position reconstructs; each position's score is
    at least its own self-attention share among the chunk's queries."""
    rng = np.random.default_rng(9)
    H, G, N, d, S, m = 1, 2, 12, 4, 1, 4
    K = rng.standard_normal((1, H, N, d))
    Q = rng.standard_normal((1, H * G, N, d))
    sel, ch = kv2.select_queries(np.zeros(N), N, S, m, 1.0)
    assert sel.tolist() == list(range(S, N))
    score, _ = kv2.recon_scores(K, Q, sel, ch)
    ref = _explicit_scores(K[0], Q[0], sel, ch, G)
    np.testing.assert_allclose(score[0, 0, S:], ref[0, S:], rtol=1e-12)


def test_recon_lse_rows_sum_to_one():
    rng = np.random.default_rng(10)
    H, G, N, d, S, m = 1, 2, 30, 8, 2, 7
    K = rng.standard_normal((1, H, N, d)) * 2
    Q = rng.standard_normal((1, G, N, d)) * 2
    sel, ch = kv2.select_queries(rng.standard_normal(N), N, S, m, 0.5)
    _, lse = kv2.recon_scores(K, Q, sel, ch)
    for c in ch:
        for g in range(G):
            for j in range(c.nq):
                q = Q[0, g, sel[c.off + j]]
                keys = np.concatenate([K[0, 0], K[0, 0][sel[c.off:c.off + j + 1]]])
                z = keys @ q / math.sqrt(d)
                assert abs(np.exp(z - lse[0, g, c.off + j]).sum() - 1.0) < 1e-12


def test_recon_all_keys_equal_closed_form():
    """Equal keys give every query a uniform row: attention 1/(N+j+1) for
    query j, so each scored position gets 1/(N+1) (from j = 0)."""
    rng = np.random.default_rng(12)
    N, d, S, m = 40, 16, 4, 9
    k = rng.standard_normal(d)
    K = np.broadcast_to(k, (1, 1, N, d)).copy()
    Q = rng.standard_normal((1, 3, N, d))
    sel, ch = kv2.select_queries(rng.standard_normal(N), N, S, m, 0.3)
    score, lse = kv2.recon_scores(K, Q, sel, ch)
    np.testing.assert_allclose(score[0, 0, S:], 1.0 / (N + 1), rtol=1e-13)


def test_recon_single_needle():
    rng = np.random.default_rng(13)
    N, d, S, m = 64, 16, 4, 30
    K = rng.standard_normal((1, 1, N, d)) * 0.1
    Q = rng.standard_normal((1, 2, N, d)) * 0.1
    sel, ch = kv2.select_queries(rng.standard_normal(N), N, S, m, 0.2)
    q = Q[0, 1, sel[ch[1].off + 1]]
    K[0, 0, 50] = 80.0 * math.sqrt(d) * q / (q @ q)     # logit 80 for that query
    score, _ = kv2.recon_scores(K, Q, sel, ch)
    assert score[0, 0, 50] > 1 - 1e-12 and np.nanmax(np.delete(score[0, 0], 50)) < 0.5


def test_recon_chunk_isolation():
    rng = np.random.default_rng(14)
    N, d, S, m = 40, 8, 2, 10
    K = rng.standard_normal((1, 1, N, d))
    Q = rng.standard_normal((1, 2, N, d))
    sel, ch = kv2.select_queries(rng.standard_normal(N), N, S, m, 0.3)
    s0, _ = kv2.recon_scores(K, Q, sel, ch)
    Q2 = Q.copy()
    Q2[0, :, sel[ch[2].off:ch[2].off + ch[2].nq]] *= -3.0
    s1, _ = kv2.recon_scores(K, Q2, sel, ch)
    c2 = ch[2]
    same = np.r_[S:c2.lo, c2.hi:N]
    np.testing.assert_array_equal(s0[0, 0, same], s1[0, 0, same])
    assert not np.allclose(s0[0, 0, c2.lo:c2.hi], s1[0, 0, c2.lo:c2.hi])


def test_recon_gqa_group_mapping():
    """Query head g reads KV head g // G: duplicating a query head inside its
    group leaves the max unchanged, and a needle planted for head 3 (KV head
    1 when G = 2) shows only in KV head 1."""
    rng = np.random.default_rng(15)
    N, d, S, m, G = 32, 8, 2, 15, 2
    K = rng.standard_normal((1, 2, N, d)) * 0.2
    Q = rng.standard_normal((1, 4, N, d)) * 0.2
    sel, ch = kv2.select_queries(rng.standard_normal(N), N, S, m, 0.2)
    q = Q[0, 3, sel[ch[1].off]]        # a query of the chunk that holds position 20
    assert ch[1].lo <= 20 < ch[1].hi
    K[0, 1, 20] = 60.0 * math.sqrt(d) * q / (q @ q)
    K[0, 0, 20] = K[0, 1, 20]          # same key in KV head 0, but no head there sees that query
    sc, _ = kv2.recon_scores(K, Q, sel, ch)
    assert sc[0, 1, 20] > 0.999 and sc[0, 0, 20] < 0.5
    Qd = Q.copy(); Qd[0, 1] = Qd[0, 0]
    K1 = K[:, :1]
    a, _ = kv2.recon_scores(K1, Qd[:, :2], sel, ch)
    b, _ = kv2.recon_scores(K1, Qd[:, :1], sel, ch)
    np.testing.assert_array_equal(a, b)


# ---------------------------------------------------------------------------
# Eviction, compaction, refinement
# ---------------------------------------------------------------------------
def test_evict_small_golden():
    g = gold("evict_small.json")
    score = np.array(g["score"], dtype=np.float64)
    kept = kv2.evict(score, g["S"], g["k"])
    assert [k.tolist() for k in kept] == g["kept"]
    assert np.all(score[:, :, :g["S"]] == g["pinned"])


@pytest.mark.parametrize("seed", range(5))
def test_evict_brute_force_and_counts(seed):
    rng = np.random.default_rng(100 + seed)
    L, H, N, S = 3, 2, 29, 3
    score = rng.integers(0, 5, size=(L, H, N)).astype(np.float64)
    score[:, :, :S] = np.nan                     # sinks are not read
    ks = [S, 10, N]
    work = score.copy()
    kept = kv2.evict(work, S, ks)
    for l in range(L):
        assert kept[l].shape == (H, ks[l])
        for h in range(H):
            kk = kept[l][h].tolist()
            assert kk == sorted(kk) and set(range(S)) <= set(kk)
            assert _is_top_set(work[l, h], 0, N, kk)
    assert kept[2].tolist() == [list(range(N))] * H           # k = N keeps all


def test_compact_matches_numpy_take():
    rng = np.random.default_rng(7)
    X = rng.integers(0, 2**16, size=(2, 3, 20, 8)).astype(np.uint16)
    kept = [np.sort(rng.choice(20, size=(3, 5), replace=True), axis=1), np.tile(np.arange(20), (3, 1))]
    out = kv2.compact(X, kept)
    for l in range(2):
        for h in range(3):
            np.testing.assert_array_equal(out[l][h], np.take(X[l, h], kept[l][h], axis=0))


def test_refine_identical_rows_and_hand_example():
    row = np.array([0.0, 0.0, 0.3, 0.1, 0.6])
    score = np.broadcast_to(row, (3, 2, 5)).copy()
    np.testing.assert_allclose(kv2.refine_proxy(score, 2)[2:], row[2:], atol=0)
    sc = np.array([[[9, 9, 0.2, 0.4]], [[9, 9, 0.6, 0.0]]])
    np.testing.assert_allclose(kv2.refine_proxy(sc, 2), [0, 0, 0.4, 0.2])


def test_budget_count():
    assert kv2.budget_count(0.05, 4096) == 204
    assert kv2.budget_count(0.02, 16384) == 327
    assert kv2.budget_count(0.05, 32768) == 1638
    assert kv2.budget_count(0.10, 131072) == 13107


def test_compress_single_pass_equals_passes_one():
    rng = np.random.default_rng(21)
    L, H, G, N, d = 2, 2, 2, 40, 8
    K = rng.standard_normal((L, H, N, d)); V = rng.standard_normal((L, H, N, d))
    Q = rng.standard_normal((L, H * G, N, d))
    out = kv2.kv2_compress(K, V, Q, 2, 16, 0.25, [8, 8], passes=1)
    p, _ = kv2.proxy_scores(K)
    sel, ch = kv2.select_queries(p, N, 2, 16, 0.25)
    assert out["sel"][0].tolist() == sel.tolist()
    out3 = kv2.kv2_compress(K, V, Q, 2, 16, 0.25, [8, 8], passes=3)
    assert len(out3["sel"]) == 3 and out3["sel"][0].tolist() == sel.tolist()


def test_refinement_passes_follow_planted_needles():
    """KV² page, "무엇과 다른가" (refinement): each pass's scores replace the
    proxy for the next pass's selection.  Hand-built case with one chunk
    [1, 6) and one reconstruction query per pass (rho = 0.2):
      pass 1: KeyDiff ranks key 2 first -- it is the only key pointing against
              the mean unit key (-e1 against five keys near +e1);
      pass 2: the pool query at 2 is 100 e5, whose only nonzero logit is with
              key 4 (0.1 e5 component), so key 4 takes most of the attention
              and the refined proxy selects 4;
      pass 3: the pool query at 4 is 100 e3, a needle on key 1 -> selects 1.
    A dropped refinement (p kept), a refined p taken from the wrong pass or a
    selection of the lowest instead of the highest scores changes this
    sequence."""
    d, N = 8, 6
    e = np.eye(d)
    K = np.stack([e[0], e[0] + 0.1 * e[2], -e[0], e[0] + 0.1 * e[3], e[0] + 0.1 * e[4], e[0] + 0.1 * e[5]])
    Qp = np.zeros((N, d))
    Qp[2] = 100 * e[4]
    Qp[4] = 100 * e[2]
    K4 = K[None, None]                  # [L=1][Hkv=1][N][d]
    Q4 = Qp[None, None]                 # [L=1][Hq=1][N][d]
    out = kv2.kv2_compress(K4, K4.copy(), Q4, 1, 5, 0.2, [2], passes=3)
    assert [s.tolist() for s in out["sel"]] == [[2], [4], [1]]
    # the last pass scores with the all-zero query at 1: every logit is 0, the
    # attention is uniform, so the tie rule keeps the lowest non-sink position
    assert out["kept"][0].tolist() == [[0, 1]]


# ---------------------------------------------------------------------------
# EpiCache: layer budgets and block prefill
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("case", gold("layer_budgets.json")["cases"], ids=lambda c: str(c["sens"]) + str(c["alpha"]))
def test_layer_budgets_golden(case):
    got = kv2.layer_budgets(case["sens"], case["alpha"], case["M"], case["S"])
    assert got.tolist() == case["budgets"]


def test_layer_budgets_properties():
    rng = np.random.default_rng(3)
    sens = rng.uniform(0.5, 1.5, size=28)
    for alpha in (0, 1, 3, 8):
        b = kv2.layer_budgets(sens, alpha, 8192, 4)
        assert int(b.sum()) == 28 * 8192
        order = np.argsort(sens)
        assert np.all(np.diff(b[order]) >= 0)            # monotone in sensitivity
    assert np.all(kv2.layer_budgets(sens, 0, 8192, 4) == 8192)
    # sharper alpha concentrates budget
    assert kv2.layer_budgets(sens, 8, 8192, 4).max() > kv2.layer_budgets(sens, 2, 8192, 4).max()


def _epi_inputs(seed, H=2, G=2, n=50, d=8, P=4):
    rng = np.random.default_rng(seed)
    return (rng.standard_normal((H, n, d)), rng.standard_normal((H, n, d)),
            rng.standard_normal((H * G, P, d)), rng.standard_normal((H, P, d)))


def test_block_prefill_no_eviction_is_identity():
    Kh, Vh, Qp, Kp = _epi_inputs(1)
    Kc, Vc, pos, t0 = kv2.block_prefill_layer(Kh, Vh, Qp, Kp, block=64, M=50, sinks=2)
    np.testing.assert_array_equal(Kc, Kh); np.testing.assert_array_equal(Vc, Vh)
    assert t0 == 50 and pos.tolist() == [list(range(50))] * 2


def test_block_prefill_one_block_equals_single_shot():
    Kh, Vh, Qp, Kp = _epi_inputs(2)
    M, S = 17, 2
    Kc, Vc, pos, _ = kv2.block_prefill_layer(Kh, Vh, Qp, Kp, block=50, M=M, sinks=S)
    # single shot: the whole history is one chunk scored by the prompt
    sc = np.stack([_explicit_prompt_scores(Kh[h], Qp[2 * h:2 * h + 2], Kp[h], S) for h in range(2)])
    for h in range(2):
        order = sorted(range(S, 50), key=lambda i: (-sc[h, i], i))[:M - S]
        assert pos[h].tolist() == list(range(S)) + sorted(order)
        np.testing.assert_array_equal(Kc[h], Kh[h][pos[h]])


def _explicit_prompt_scores(Kh, Qg, Kp, S):
    """Prompt queries appended after the cache (causal among themselves);
    attention matrix through torch SDPA with V = identity."""
    n, d = Kh.shape
    P = Qg.shape[1]
    keys = torch.from_numpy(np.concatenate([Kh, Kp]))
    mask = np.ones((P, n + P), dtype=bool)
    mask[:, n:] = np.tril(np.ones((P, P), dtype=bool))
    eye = torch.eye(n + P, dtype=torch.float64)
    best = np.zeros(n)
    for g in range(Qg.shape[0]):
        A = torch.nn.functional.scaled_dot_product_attention(
            torch.from_numpy(Qg[g])[None, None], keys[None, None], eye[None, None],
            attn_mask=torch.from_numpy(mask)[None, None]).numpy()[0, 0]
        best = np.maximum(best, A[:, :n].max(axis=0))
    best[:S] = np.inf
    return best


def test_block_prefill_resume_and_bounded():
    Kh, Vh, Qp, Kp = _epi_inputs(3, n=90)
    full = kv2.block_prefill_layer(Kh, Vh, Qp, Kp, block=16, M=20, sinks=3)
    st = kv2.block_prefill_layer(Kh, Vh, Qp, Kp, block=16, M=20, sinks=3, n_blocks=2)
    assert st[0].shape[1] <= 20 + 16
    res = kv2.block_prefill_layer(Kh, Vh, Qp, Kp, block=16, M=20, sinks=3, state=st)
    for a, b in zip(full, res):
        np.testing.assert_array_equal(np.asarray(a), np.asarray(b))
    assert full[0].shape[1] == 20
    assert all(set(range(3)) <= set(r.tolist()) for r in full[2])
