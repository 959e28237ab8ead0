"""GPU parity of the top-n kernels on rows that span several CTAs.

KV² page, "어떻게 동작하나" (per-chunk selection of the reconstruction
queries) and "무엇과 다른가" (sink pin and eviction to the budget): every
(layer, KV head) row, or chunk of p, is split over a cluster of up to eight
CTAs that stage their parts in shared memory; rows longer than eight parts
fall back to the global-memory kernels.  Integer-valued scores make the tie
rule (lower position first) decide most of the set, so the kept positions
must equal the oracle's exactly.
"""
import numpy as np
import pytest
import torch

import kv_synth as ks
from oracle import compare, kv2

pytestmark = pytest.mark.gpu

DEV = "cuda:0"


@pytest.fixture(scope="module")
def qk():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    import __graft_entry__ as ge
    ge.build()
    import query_agnostic_kv_gb300 as q
    q.kvc_device_check()
    return q


def _ws(qk, shape, S):
    return torch.empty(4096, dtype=torch.uint8, device=DEV)   # eviction needs two words of it


def _evict_case(qk, L, H, N, S, ks_, sc):
    shape = (L, H, H, 128, N)
    score = torch.from_numpy(sc.reshape(-1).copy()).to(DEV)
    kept = torch.empty(H * sum(ks_), dtype=torch.int32, device=DEV)
    qk.kvc_evict_topk(shape, score, S, ks_, kept, ws=_ws(qk, shape, S))
    assert qk.kvc_stream_status() == 0
    ref = sc.astype(np.float64).copy()
    ref_kept = kv2.evict(ref, S, ks_)
    got = kept.cpu().numpy()
    off = 0
    for l in range(L):
        for h in range(H):
            assert got[off:off + ks_[l]].tolist() == ref_kept[l][h].tolist(), (l, h)
            off += ks_[l]
    pinned = score.cpu().numpy().reshape(L, H, N)[:, :, :S]
    assert np.all(pinned == np.nanmax(sc[:, :, S:]))


# (L, Hkv, N, budgets): candidates per row N - 4
EVICT_CASES = {
    "five-parts": (2, 2, 70000, [1500, 4]),            # 69996 -> 5 CTAs of 14000 keys
    "eight-wide-parts": (1, 1, 393220, [20000]),       # 393216 -> 8 CTAs of 49152 keys (192 KB each)
    "global-fallback": (1, 1, 400000, [1000]),         # longer than eight parts: global-memory kernel
    "keep-all-but-one": (1, 2, 33000, [32999]),        # threshold at the very bottom, 3 CTAs
}


@pytest.mark.parametrize("name", list(EVICT_CASES))
def test_evict_rows_over_several_ctas(qk, name):
    L, H, N, ks_ = EVICT_CASES[name]
    rng = np.random.default_rng(11)
    sc = rng.integers(0, 3000, size=(L, H, N)).astype(np.float32)   # many exact ties
    _evict_case(qk, L, H, N, 4, ks_, sc)


def test_evict_special_values(qk):
    """NaN ranks below -inf, -0 ties with +0, infinities order normally."""
    L, H, N, S = 1, 2, 20000, 4
    rng = np.random.default_rng(5)
    sc = rng.standard_normal((L, H, N)).astype(np.float32)
    idx = rng.choice(np.arange(S, N), size=400, replace=False)
    sc[0, 0, idx[:100]] = np.nan
    sc[0, 0, idx[100:200]] = -0.0
    sc[0, 0, idx[200:300]] = 0.0
    sc[0, 1, idx[300:340]] = np.inf
    sc[0, 1, idx[340:400]] = -np.inf
    _evict_case(qk, L, H, N, S, [3000], sc)
    # a budget reaching into the NaN tail keeps NaNs in position order
    sc2 = np.full((1, 1, 5000), np.nan, dtype=np.float32)
    sc2[0, 0, 100:200] = 1.0
    _evict_case(qk, 1, 1, 5000, S, [300], sc2)


@pytest.mark.parametrize("N,m,rho", [(50000, 50000, 0.013), (61234, 20000, 0.1), (4100, 4096, 0.5)])
def test_select_chunks_over_several_ctas(qk, N, m, rho):
    S = 4
    rng = np.random.default_rng(N)
    p = rng.integers(0, 500, size=N).astype(np.float32)               # ties everywhere
    off = qk.kvc_chunk_plan(N, S, m, rho)
    sel = torch.empty(off[-1], dtype=torch.int32, device=DEV)
    qk.kvc_select_queries(N, S, m, rho, torch.from_numpy(p).to(DEV), sel)
    assert qk.kvc_stream_status() == 0
    ref, _ = kv2.select_queries(p.astype(np.float64), N, S, m, rho)
    assert np.array_equal(sel.cpu().numpy().astype(np.int64), ref)


def test_compress_fused_compaction_over_several_ctas(qk):
    """kvc_compress chooses and copies the kept rows in one launch; with
    40000 positions every row spans three CTAs.  The kept set is checked on
    the GPU's own scores, the compacted rows bit for bit."""
    cfg = ks.scaled(ks.TINY, name="fused40k", L=1, Hkv=2, Hq=4, N=40000, m=4096, rho=0.02, budget=0.05,
                    needles_per_layer=8)
    x = ks.gen_kv2(cfg)
    L, H, Hq, N, S = cfg.L, cfg.Hkv, cfg.Hq, cfg.N, cfg.sinks
    shape = (L, H, Hq, 128, N)
    to_dev = lambda a: torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).to(DEV)
    K, V, Q = to_dev(x.K), to_dev(x.V), to_dev(x.Q)
    k = qk.kvc_budget_count(cfg.budget, N, S)
    ws = torch.empty(qk.kvc_workspace_size(shape, S, cfg.m, cfg.rho), dtype=torch.uint8, device=DEV)
    score = torch.empty(L * H * N, dtype=torch.float32, device=DEV)
    kept = torch.empty(L * H * k, dtype=torch.int32, device=DEV)
    Kc = torch.empty(L * H * k * 128, dtype=torch.bfloat16, device=DEV)
    Vc = torch.empty_like(Kc)
    qk.kvc_compress(shape, K, V, Q, S, cfg.m, cfg.rho, 1, [k] * L, kept, Kc, Vc, score=score, ws=ws)
    assert qk.kvc_stream_status() == 0
    sc = score.cpu().numpy().reshape(L, H, N).astype(np.float64)
    kept_g = kept.cpu().numpy().reshape(L, H, k)
    Kc_g = Kc.view(torch.int16).cpu().numpy().view(np.uint16).reshape(L, H, k, 128)
    Vc_g = Vc.view(torch.int16).cpu().numpy().view(np.uint16).reshape(L, H, k, 128)
    for h in range(H):
        compare.assert_topk_set(kept_g[0, h], sc[0, h], S, N, k - S, forced=range(S), what=f"kept h={h}")
        np.testing.assert_array_equal(Kc_g[0, h], x.K[0, h][kept_g[0, h]])
        np.testing.assert_array_equal(Vc_g[0, h], x.V[0, h][kept_g[0, h]])
    assert np.all(sc[:, :, :S] == np.float32(sc[:, :, S:].max()))


@pytest.mark.parametrize("N", [3000, 40000])
def test_evict_compact_equals_the_two_calls(qk, N):
    """The fused entry point keeps, pins and copies exactly what
    kvc_evict_topk followed by kvc_compact does."""
    L, H, S = 3, 2, 4
    ks_ = [S, N // 20, N // 3]
    rng = np.random.default_rng(N)
    sc = rng.random((L, H, N)).astype(np.float32)
    sc[:, :, 7::13] = 0.5                                            # exact ties
    shape = (L, H, 2 * H, 128, N)
    g = torch.Generator(device=DEV).manual_seed(1)
    K = torch.randn(L * H * N * 128, generator=g, device=DEV).to(torch.bfloat16)
    V = torch.randn(L * H * N * 128, generator=g, device=DEV).to(torch.bfloat16)
    outs = []
    for fused in (False, True):
        score = torch.from_numpy(sc.reshape(-1).copy()).to(DEV)
        kept = torch.empty(H * sum(ks_), dtype=torch.int32, device=DEV)
        Kc = torch.empty(H * sum(ks_) * 128, dtype=torch.bfloat16, device=DEV)
        Vc = torch.empty_like(Kc)
        ws = torch.empty(4096, dtype=torch.uint8, device=DEV)
        if fused:
            qk.kvc_evict_compact(shape, score, S, ks_, kept, K, V, Kc, Vc, ws=ws)
        else:
            qk.kvc_evict_topk(shape, score, S, ks_, kept, ws=ws)
            qk.kvc_compact(shape, K, V, kept, ks_, Kc, Vc)
        assert qk.kvc_stream_status() == 0
        outs.append((score.cpu(), kept.cpu(), Kc.view(torch.int16).cpu(), Vc.view(torch.int16).cpu()))
    for a, b in zip(*outs):
        assert torch.equal(a, b)
