"""GPU parity: every stage of the CUDA path, called through the C ABI,
against the float64 oracle on the same seeded inputs.

Each stage is checked on the GPU's own upstream output (the oracle's
selection runs on the GPU's p, its scoring on the GPU's selection, ...), so a
legitimate near-tie upstream cannot cascade into a false failure.
Tolerances: scores 1e-3 relative (proxy with a 1e-3 absolute floor), index
sets exact up to oracle near-ties within 1e-4 of the threshold, compacted rows
bit-exact.
"""
import dataclasses
import math

import numpy as np
import pytest
import torch

import kv_synth as ks
from oracle import compare, kv2

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def qk():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    import __graft_entry__ as ge
    ge.build()
    import query_agnostic_kv_gb300 as q
    q.kvc_device_check()
    return q


DEV = "cuda:0"


def to_dev(bits: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).to(DEV)


def bits_of(t: torch.Tensor) -> np.ndarray:
    return t.view(torch.int16).cpu().numpy().view(np.uint16)


def run_stages(qk, x, cfg, lse=False, Kapp=None):
    """Proxy -> select -> recon -> evict -> compact through the C ABI."""
    L, H, Hq, N, S = cfg.L, cfg.Hkv, cfg.Hq, cfg.N, cfg.sinks
    shape = (L, H, Hq, 128, N)
    K, V, Q = to_dev(x.K), to_dev(x.V), to_dev(x.Q)
    off = qk.kvc_chunk_plan(N, S, cfg.m, cfg.rho)
    Qn = off[-1]
    ws = torch.empty(qk.kvc_workspace_size(shape, S, cfg.m, cfg.rho), dtype=torch.uint8, device=DEV)
    out = {}
    p = torch.empty(N, dtype=torch.float32, device=DEV)
    s = torch.empty(L * H * N, dtype=torch.float32, device=DEV)
    qk.kvc_proxy_score(shape, K, p, s, ws=ws)
    sel = torch.empty(Qn, dtype=torch.int32, device=DEV)
    qk.kvc_select_queries(N, S, cfg.m, cfg.rho, p, sel)
    score = torch.full((L * H * N,), float("nan"), dtype=torch.float32, device=DEV)
    lse_t = torch.empty(L * Hq * Qn, dtype=torch.float32, device=DEV) if lse else None
    qk.kvc_recon_score(shape, K, Q, sel, S, cfg.m, cfg.rho, score, Kapp=Kapp, lse=lse_t, ws=ws)
    assert qk.kvc_stream_status() == 0
    out["score_raw"] = score.cpu().numpy().reshape(L, H, N).astype(np.float64)
    k = qk.kvc_budget_count(cfg.budget, N, S)
    kept = torch.empty(L * H * k, dtype=torch.int32, device=DEV)
    qk.kvc_evict_topk(shape, score, S, [k] * L, kept, ws=ws)
    Kc = torch.empty(L * H * k * 128, dtype=torch.bfloat16, device=DEV)
    Vc = torch.empty_like(Kc)
    qk.kvc_compact(shape, K, V, kept, [k] * L, Kc, Vc)
    assert qk.kvc_stream_status() == 0
    out.update(p=p.cpu().numpy().astype(np.float64), s=s.cpu().numpy().reshape(L, H, N).astype(np.float64),
               sel=sel.cpu().numpy().astype(np.int64), score=score.cpu().numpy().reshape(L, H, N).astype(np.float64),
               kept=kept.cpu().numpy().reshape(L, H, k), Kc=bits_of(Kc).reshape(L, H, k, 128),
               Vc=bits_of(Vc).reshape(L, H, k, 128), k=k)
    if lse:
        out["lse"] = lse_t.cpu().numpy().reshape(L, Hq, Qn).astype(np.float64)
    return out


def check_all(x, cfg, out, pairs=None, lse=False, score_floor=0.0):
    L, H, N, S = cfg.L, cfg.Hkv, cfg.N, cfg.sinks
    # proxy
    p_ref, s_ref = kv2.proxy_scores(x.K)
    compare.assert_scores(out["s"], s_ref, floor=compare.PROXY_FLOOR, what="per-head KeyDiff s")
    compare.assert_scores(out["p"], p_ref, floor=compare.PROXY_FLOOR, what="proxy p")
    # selection on the GPU's p
    chunks = kv2.chunk_plan(N, S, cfg.m, cfg.rho)
    sel_ref, _ = kv2.select_queries(out["p"], N, S, cfg.m, cfg.rho)
    assert np.array_equal(out["sel"], sel_ref), "selection differs from the oracle on the same p"
    # reconstruction scores on the GPU's selection
    sc_ref, lse_ref = kv2.recon_scores(x.K, x.Q, out["sel"], chunks, pairs=pairs)
    todo = pairs if pairs is not None else [(l, h) for l in range(L) for h in range(H)]
    for (l, h) in todo:
        compare.assert_scores(out["score_raw"][l, h, S:], sc_ref[l, h, S:], floor=score_floor,
                              what=f"recon score l={l} h={h}")
        if lse:
            G = cfg.G
            for g in range(G):
                hq = h * G + g
                compare.assert_scores(out["lse"][l, hq], lse_ref[l, hq], rtol=1e-4, floor=10.0,
                                      what=f"lse l={l} hq={hq}")
    # sinks pinned to the global max of the GPU scores
    gmax = np.nanmax(out["score_raw"][:, :, S:])
    assert np.all(out["score"][:, :, :S] == np.float32(gmax))
    # eviction on the GPU's scores
    k = out["k"]
    for l in range(L):
        for h in range(H):
            compare.assert_topk_set(out["kept"][l, h], out["score"][l, h], S, N, k - S, forced=range(S),
                                    what=f"kept l={l} h={h}")
            np.testing.assert_array_equal(out["Kc"][l, h], x.K[l, h][out["kept"][l, h]])
            np.testing.assert_array_equal(out["Vc"][l, h], x.V[l, h][out["kept"][l, h]])


CASES = {
    # name: config (kept small enough that the oracle checks every head)
    "tiny-4k": ks.TINY,
    "ragged-1000": ks.scaled(ks.TINY, name="ragged", L=2, Hkv=2, Hq=8, N=1000, m=300, rho=0.2, budget=0.1,
                             needles_per_layer=6),
    "rho1-mha": ks.scaled(ks.TINY, name="rho1", L=1, Hkv=2, Hq=2, N=700, m=128, rho=1.0, budget=0.3,
                          needles_per_layer=2),
    "gqa3-one-chunk": ks.scaled(ks.TINY, name="gqa3", L=2, Hkv=2, Hq=6, N=777, m=4096, rho=0.05, budget=0.02,
                                sinks=3, needles_per_layer=2),
    "tiny-nq1": ks.scaled(ks.TINY, name="nq1", L=1, Hkv=1, Hq=4, N=300, m=40, rho=0.001, budget=0.05,
                          needles_per_layer=0),
    # G = 8 (304 query rows per chunk: two column-max query tiles, the second ragged) and no sinks
    "g8-no-sinks": ks.scaled(ks.TINY, name="g8s0", L=1, Hkv=2, Hq=16, N=900, m=256, rho=0.15, budget=0.1, sinks=0,
                             needles_per_layer=3),
}


@pytest.mark.parametrize("name", list(CASES))
def test_stagewise_parity(qk, name):
    cfg = CASES[name]
    x = ks.gen_kv2(cfg)
    out = run_stages(qk, x, cfg, lse=True)
    check_all(x, cfg, out, lse=True)


def test_sharp_attention_scores(qk):
    """Keys and queries scaled by 4 (logits x16): sharp softmax rows whose
    LSE sits far above most logits, where the column-max pass's lse terms and
    fp32 cancellation matter most.  Scores below 1e-30 (fp32 exp2 flushes
    them to zero) compare against that absolute floor."""
    cfg = CASES["ragged-1000"]
    x = ks.gen_kv2(cfg)
    up = lambda b: ks.f32_to_bf16_bits(ks.bf16_bits_to_f32(b) * np.float32(4.0))
    x = dataclasses.replace(x, K=up(x.K), Q=up(x.Q))
    out = run_stages(qk, x, cfg, lse=True)
    check_all(x, cfg, out, lse=True, score_floor=1e-30)


@pytest.mark.parametrize("name", ["ragged-1000", "tiny-4k"])
def test_recon_phases_match_one_call(qk, name):
    """kvc_recon_gather, kvc_recon_rows and kvc_recon_cols on one workspace
    (the gather on a second stream, ordered by an event) give exactly
    kvc_recon_score's scores and lse."""
    cfg = CASES[name]
    x = ks.gen_kv2(cfg)
    L, H, Hq, N, S = cfg.L, cfg.Hkv, cfg.Hq, cfg.N, cfg.sinks
    shape = (L, H, Hq, 128, N)
    K, Q = to_dev(x.K), to_dev(x.Q)
    Qn = qk.kvc_chunk_plan(N, S, cfg.m, cfg.rho)[-1]
    wsz = qk.kvc_workspace_size(shape, S, cfg.m, cfg.rho)
    ws1 = torch.empty(wsz, dtype=torch.uint8, device=DEV)
    ws2 = torch.empty(wsz, dtype=torch.uint8, device=DEV)
    p = torch.empty(N, dtype=torch.float32, device=DEV)
    qk.kvc_proxy_score(shape, K, p, ws=ws1)
    sel = torch.empty(Qn, dtype=torch.int32, device=DEV)
    qk.kvc_select_queries(N, S, cfg.m, cfg.rho, p, sel)
    score1 = torch.full((L * H * N,), float("nan"), device=DEV)
    lse1 = torch.empty(L * Hq * Qn, device=DEV)
    qk.kvc_recon_score(shape, K, Q, sel, S, cfg.m, cfg.rho, score1, lse=lse1, ws=ws1)
    score2 = torch.full_like(score1, float("nan"))
    lse2 = torch.empty_like(lse1)
    main = torch.cuda.current_stream()
    side = torch.cuda.Stream(device=DEV)
    side.wait_stream(main)
    with torch.cuda.stream(side):
        qk.kvc_recon_gather(shape, K, Q, sel, S, cfg.m, cfg.rho, ws=ws2, stream=side)
        done = torch.cuda.Event()
        done.record(side)
    main.wait_event(done)
    qk.kvc_recon_rows(shape, K, S, cfg.m, cfg.rho, lse=lse2, ws=ws2)
    qk.kvc_recon_cols(shape, K, S, cfg.m, cfg.rho, score2, ws=ws2)
    assert qk.kvc_stream_status() == 0
    assert torch.equal(score1.view(L, H, N)[:, :, S:], score2.view(L, H, N)[:, :, S:])
    assert torch.equal(lse1, lse2)


def test_explicit_appended_keys(qk):
    """Appended keys supplied by the caller (e.g. from a real reconstruction
    forward) instead of the cache keys at the selected positions."""
    cfg = CASES["ragged-1000"]
    x = ks.gen_kv2(cfg)
    off = qk.kvc_chunk_plan(cfg.N, cfg.sinks, cfg.m, cfg.rho)
    rng = np.random.default_rng(5)
    kapp = ks.f32_to_bf16_bits(rng.standard_normal((cfg.L, cfg.Hkv, off[-1], 128)).astype(np.float32) * 3)
    out = run_stages(qk, x, cfg, Kapp=to_dev(kapp))
    chunks = kv2.chunk_plan(cfg.N, cfg.sinks, cfg.m, cfg.rho)
    sc_ref, _ = kv2.recon_scores(x.K, x.Q, out["sel"], chunks, Kapp=kapp)
    compare.assert_scores(out["score_raw"][:, :, cfg.sinks:], sc_ref[:, :, cfg.sinks:], what="recon with Kapp")


def test_compress_matches_stages_and_is_deterministic(qk):
    cfg = CASES["ragged-1000"]
    x = ks.gen_kv2(cfg)
    L, H, Hq, N, S = cfg.L, cfg.Hkv, cfg.Hq, cfg.N, cfg.sinks
    shape = (L, H, Hq, 128, N)
    K, V, Q = to_dev(x.K), to_dev(x.V), to_dev(x.Q)
    k = qk.kvc_budget_count(cfg.budget, N, S)
    ws = torch.empty(qk.kvc_workspace_size(shape, S, cfg.m, cfg.rho), dtype=torch.uint8, device=DEV)
    res = []
    for _ in range(2):
        kept = torch.empty(L * H * k, dtype=torch.int32, device=DEV)
        Kc = torch.empty(L * H * k * 128, dtype=torch.bfloat16, device=DEV)
        Vc = torch.empty_like(Kc)
        score = torch.empty(L * H * N, dtype=torch.float32, device=DEV)
        qk.kvc_compress(shape, K, V, Q, S, cfg.m, cfg.rho, 1, [k] * L, kept, Kc, Vc, score=score, ws=ws)
        assert qk.kvc_stream_status() == 0
        res.append((kept.cpu().numpy(), bits_of(Kc), score.cpu().numpy()))
    assert np.array_equal(res[0][0], res[1][0]) and np.array_equal(res[0][1], res[1][1])
    assert np.array_equal(res[0][2], res[1][2])  # bitwise deterministic
    stages = run_stages(qk, x, cfg)
    assert np.array_equal(res[0][0].reshape(L, H, k), stages["kept"])


def test_proxies_past_knorm_grid_cap(qk):
    """Both proxies on one head whose row count passes the Knorm kernel's
    grid cap (8 blocks of 128 rows per SM) by one row: there the first
    half-warp of the first warp takes one more trip through its loop than its
    partner.  Zero keys are planted (their score is 0 under both proxies)."""
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    N = sms * 8 * 128 + 1
    rng = np.random.default_rng(7)
    z = rng.standard_normal((1, 1, N, 128), dtype=np.float32)
    z[..., ::32] += 5.0
    z *= np.exp(0.3 * rng.standard_normal((1, 1, N, 1))).astype(np.float32)
    z[0, 0, [0, 5, N - 1]] = 0.0
    bits = ks.f32_to_bf16_bits(z)
    K = to_dev(bits)
    shape = (1, 1, 4, 128, N)
    ws = torch.empty(qk.kvc_workspace_size(shape, 4, 4096, 0.1), dtype=torch.uint8, device=DEV)
    p = torch.empty(N, dtype=torch.float32, device=DEV)
    s = torch.empty(N, dtype=torch.float32, device=DEV)
    for kind, floor in (("knorm", 0.0), ("keydiff", compare.PROXY_FLOOR)):
        s.fill_(float("nan"))
        qk.kvc_proxy_score_kind(shape, kind, K, p, s, ws=ws)
        assert qk.kvc_stream_status() == 0
        p_ref, s_ref = kv2.proxy_scores(bits, kind=kind)
        got = s.cpu().numpy().reshape(1, 1, N)
        compare.assert_scores(got, s_ref, rtol=1e-5 if kind == "knorm" else compare.SCORE_RTOL, floor=floor,
                              what=f"{kind} s")
        compare.assert_scores(p.cpu().numpy(), p_ref, rtol=1e-5 if kind == "knorm" else compare.SCORE_RTOL,
                              floor=floor, what=f"{kind} p")
        assert np.all(got[0, 0, [0, 5, N - 1]] == 0.0)


@pytest.mark.parametrize("name", ["tiny-4k", "ragged-1000"])
def test_knorm_proxy_and_pipeline(qk, name):
    """Knorm proxy (s = -|k|, mean over heads) against the oracle, and the
    whole pipeline with Knorm as stage 1: selection on the GPU's p, scores
    and eviction on the GPU's selection."""
    cfg = CASES[name]
    x = ks.gen_kv2(cfg)
    L, H, Hq, N, S = cfg.L, cfg.Hkv, cfg.Hq, cfg.N, cfg.sinks
    shape = (L, H, Hq, 128, N)
    K, V, Q = to_dev(x.K), to_dev(x.V), to_dev(x.Q)
    ws = torch.empty(qk.kvc_workspace_size(shape, S, cfg.m, cfg.rho), dtype=torch.uint8, device=DEV)
    p = torch.empty(N, dtype=torch.float32, device=DEV)
    s = torch.empty(L * H * N, dtype=torch.float32, device=DEV)
    qk.kvc_proxy_score_kind(shape, "knorm", K, p, s, ws=ws)
    p_ref, s_ref = kv2.proxy_scores(x.K, kind="knorm")
    compare.assert_scores(s.cpu().numpy().reshape(L, H, N), s_ref, rtol=1e-5, what="knorm s")
    compare.assert_scores(p.cpu().numpy(), p_ref, rtol=1e-5, what="knorm p")
    k = qk.kvc_budget_count(cfg.budget, N, S)
    off = qk.kvc_chunk_plan(N, S, cfg.m, cfg.rho)
    kept = torch.empty(L * H * k, dtype=torch.int32, device=DEV)
    Kc = torch.empty(L * H * k * 128, dtype=torch.bfloat16, device=DEV)
    Vc = torch.empty_like(Kc)
    p2 = torch.empty(N, dtype=torch.float32, device=DEV)
    sel = torch.empty(off[-1], dtype=torch.int32, device=DEV)
    score = torch.empty(L * H * N, dtype=torch.float32, device=DEV)
    qk.kvc_compress_ex(shape, "knorm", K, V, Q, S, cfg.m, cfg.rho, 1, [k] * L, kept, Kc, Vc, p=p2, sel=sel,
                       score=score, ws=ws)
    assert qk.kvc_stream_status() == 0
    assert torch.equal(p2, p)
    sel_np = sel.cpu().numpy().astype(np.int64)
    ref_sel, chunks = kv2.select_queries(p.cpu().numpy().astype(np.float64), N, S, cfg.m, cfg.rho)
    assert np.array_equal(sel_np, ref_sel)
    sc_ref, _ = kv2.recon_scores(x.K, x.Q, sel_np, chunks)
    sc = score.cpu().numpy().reshape(L, H, N).astype(np.float64)
    compare.assert_scores(sc[:, :, S:], sc_ref[:, :, S:], what="scores after knorm selection")
    kept_np = kept.cpu().numpy().reshape(L, H, k)
    for l in range(L):
        for h in range(H):
            compare.assert_topk_set(kept_np[l, h], sc[l, h], S, N, k - S, forced=range(S))


def test_pinned_host_pool_and_values(qk):
    """The query pool and V may stay in pinned host memory (mapped into the
    device address space): the outputs are bit-identical to the
    device-resident run."""
    cfg = CASES["ragged-1000"]
    x = ks.gen_kv2(cfg)
    L, H, Hq, N, S = cfg.L, cfg.Hkv, cfg.Hq, cfg.N, cfg.sinks
    shape = (L, H, Hq, 128, N)
    K, V, Q = to_dev(x.K), to_dev(x.V), to_dev(x.Q)
    hV = torch.from_numpy(x.V.view(np.int16)).view(torch.bfloat16).pin_memory()
    hQ = torch.from_numpy(x.Q.view(np.int16)).view(torch.bfloat16).pin_memory()
    k = qk.kvc_budget_count(cfg.budget, N, S)
    ws = torch.empty(qk.kvc_workspace_size(shape, S, cfg.m, cfg.rho), dtype=torch.uint8, device=DEV)
    outs = []
    for v_in, q_in in ((V, Q), (hV, hQ)):
        kept = torch.empty(L * H * k, dtype=torch.int32, device=DEV)
        Kc = torch.empty(L * H * k * 128, dtype=torch.bfloat16, device=DEV)
        Vc = torch.empty_like(Kc)
        score = torch.empty(L * H * N, dtype=torch.float32, device=DEV)
        qk.kvc_compress(shape, K, v_in, q_in, S, cfg.m, cfg.rho, 1, [k] * L, kept, Kc, Vc, score=score, ws=ws)
        assert qk.kvc_stream_status() == 0
        outs.append((kept.cpu(), bits_of(Kc), bits_of(Vc), score.cpu()))
    for a, b in zip(outs[0], outs[1]):
        assert np.array_equal(np.asarray(a), np.asarray(b))


def test_refinement_passes(qk):
    """passes=3: each pass's mean stage-2 score replaces the proxy."""
    cfg = ks.scaled(ks.TINY, name="refine", L=2, Hkv=2, Hq=4, N=900, m=256, rho=0.25, budget=0.05,
                    needles_per_layer=4)
    x = ks.gen_kv2(cfg)
    L, H, Hq, N, S = cfg.L, cfg.Hkv, cfg.Hq, cfg.N, cfg.sinks
    shape = (L, H, Hq, 128, N)
    K, V, Q = to_dev(x.K), to_dev(x.V), to_dev(x.Q)
    k = qk.kvc_budget_count(cfg.budget, N, S)
    ws = torch.empty(qk.kvc_workspace_size(shape, S, cfg.m, cfg.rho), dtype=torch.uint8, device=DEV)
    off = qk.kvc_chunk_plan(N, S, cfg.m, cfg.rho)
    chunks = kv2.chunk_plan(N, S, cfg.m, cfg.rho)
    # the pass loop, one stage at a time, checked against the oracle each pass
    p = torch.empty(N, dtype=torch.float32, device=DEV)
    qk.kvc_proxy_score(shape, K, p, ws=ws)
    score = torch.empty(L * H * N, dtype=torch.float32, device=DEV)
    sel = torch.empty(off[-1], dtype=torch.int32, device=DEV)
    for t in range(3):
        qk.kvc_select_queries(N, S, cfg.m, cfg.rho, p, sel)
        p_np = p.cpu().numpy().astype(np.float64)
        sel_np = sel.cpu().numpy().astype(np.int64)
        ref_sel, _ = kv2.select_queries(p_np, N, S, cfg.m, cfg.rho)
        assert np.array_equal(sel_np, ref_sel)
        qk.kvc_recon_score(shape, K, Q, sel, S, cfg.m, cfg.rho, score, ws=ws)
        sc = score.cpu().numpy().reshape(L, H, N).astype(np.float64)
        sc_ref, _ = kv2.recon_scores(x.K, x.Q, sel_np, chunks)
        compare.assert_scores(sc[:, :, S:], sc_ref[:, :, S:], what=f"pass {t} scores")
        if t < 2:
            qk.kvc_refine_proxy(shape, score, S, p)
            compare.assert_scores(p.cpu().numpy(), kv2.refine_proxy(sc, S), rtol=1e-5, what="refined p")
    # the one-call pipeline gives the same selection as the staged loop
    kept = torch.empty(L * H * k, dtype=torch.int32, device=DEV)
    Kc = torch.empty(L * H * k * 128, dtype=torch.bfloat16, device=DEV)
    Vc = torch.empty_like(Kc)
    sel2 = torch.empty_like(sel)
    qk.kvc_compress(shape, K, V, Q, S, cfg.m, cfg.rho, 3, [k] * L, kept, Kc, Vc, sel=sel2, ws=ws)
    assert qk.kvc_stream_status() == 0
    assert torch.equal(sel2, sel)


def test_evict_edge_budgets(qk):
    """k = sinks keeps only the sinks; k = N keeps everything (identity
    compaction); per-layer budgets differ."""
    cfg = ks.scaled(ks.TINY, name="edge", L=3, Hkv=2, Hq=4, N=333, m=100, rho=0.3, budget=0.1, needles_per_layer=0)
    x = ks.gen_kv2(cfg)
    L, H, Hq, N, S = cfg.L, cfg.Hkv, cfg.Hq, cfg.N, cfg.sinks
    shape = (L, H, Hq, 128, N)
    rng = np.random.default_rng(0)
    sc = rng.integers(0, 50, size=(L, H, N)).astype(np.float32)     # many exact ties
    score = torch.from_numpy(sc.reshape(-1).copy()).to(DEV)
    ks_ = [S, 57, N]
    kept = torch.empty(H * sum(ks_), dtype=torch.int32, device=DEV)
    ws = torch.empty(qk.kvc_workspace_size(shape, S, cfg.m, cfg.rho), dtype=torch.uint8, device=DEV)
    qk.kvc_evict_topk(shape, score, S, ks_, kept, ws=ws)
    K, V = to_dev(x.K), to_dev(x.V)
    Kc = torch.empty(H * sum(ks_) * 128, dtype=torch.bfloat16, device=DEV)
    Vc = torch.empty_like(Kc)
    qk.kvc_compact(shape, K, V, kept, ks_, Kc, Vc)
    assert qk.kvc_stream_status() == 0
    kept_np = kept.cpu().numpy()
    Kc_np = bits_of(Kc).reshape(-1, 128)
    ref = sc.astype(np.float64).copy()
    ref_kept = kv2.evict(ref, S, ks_)
    off = 0
    for l in range(L):
        for h in range(H):
            got = kept_np[off:off + ks_[l]]
            assert got.tolist() == ref_kept[l][h].tolist()      # integer scores: exact
            np.testing.assert_array_equal(Kc_np[off:off + ks_[l]], x.K[l, h][got])
            off += ks_[l]
    assert np.all(score.cpu().numpy().reshape(L, H, N)[:, :, :S] == sc[:, :, S:].max())


def test_timeout_status_path(qk):
    """A device-side wait on a barrier that nothing completes expires after
    its limit and is reported as KVC_ERR_TIMEOUT; the context stays usable."""
    qk.kvc_debug_expire_wait(2_000_000)  # 2 ms
    assert qk.kvc_stream_status() == 3
    assert qk.kvc_stream_status() == 0
    x = torch.ones(4, device=DEV)
    assert float(x.sum()) == 4.0


def test_bounds_status_path(qk):
    """An out-of-range kept index is skipped and reported, not dereferenced."""
    shape = (1, 1, 4, 128, 64)
    K = torch.zeros(64 * 128, dtype=torch.bfloat16, device=DEV)
    kept = torch.tensor([0, 1, 2, 999], dtype=torch.int32, device=DEV)
    Kc = torch.zeros(4 * 128, dtype=torch.bfloat16, device=DEV)
    qk.kvc_compact(shape, K, None, kept, [4], Kc, None)
    assert qk.kvc_stream_status() == 4


EPI_CASES = {
    "epi-small": dict(L=3, Hkv=2, Hq=6, mean_budget=300),
    # budgets above 4096: the kept rows move in a separate tiled compaction
    # launch (one launch for both slab directions)
    "epi-long-kept": dict(L=3, Hkv=2, Hq=6, mean_budget=5000, n_hist=14000, block=2048),
    # 20 x 8 over-budget heads at the last blocks: 160 row-LSE units of
    # different lengths on 152 SMs, so the second, reversed wave is taken
    "epi-20x8": dict(L=20, Hkv=8, Hq=24, mean_budget=600),
    # rows of up to 38K keys: eviction clusters of three CTAs
    "epi-wide-rows": dict(L=2, Hkv=2, Hq=4, mean_budget=28000, n_hist=70000, block=8192),
    # 140K history positions: the ordered pack of the one-slab state takes
    # two bitmap windows of 2^17 positions
    "epi-long-history": dict(L=2, Hkv=2, Hq=4, mean_budget=700, n_hist=140000, block=8192),
    # no sinks, blocks of 17 tokens, budgets down to a few rows
    "epi-no-sinks": dict(L=3, Hkv=2, Hq=4, mean_budget=40, n_hist=400, block=17, sinks=0),
    # one-token blocks: every step after the budget evicts exactly one row
    "epi-one-token": dict(L=2, Hkv=1, Hq=2, mean_budget=12, n_hist=60, block=1),
}


def test_tiny_unchained_pipeline(qk):
    """The tiny workload end to end: the GPU's final kept sets against the
    oracle's own pipeline (its proxy, selection, scoring and eviction, with no
    GPU output fed back).  Any difference must lie inside the tie band of the
    oracle's final scores; the number of differences is printed."""
    cfg = ks.TINY
    x = ks.gen_kv2(cfg)
    L, H, N, S = cfg.L, cfg.Hkv, cfg.N, cfg.sinks
    shape = (L, H, cfg.Hq, 128, N)
    K, V, Q = to_dev(x.K), to_dev(x.V), to_dev(x.Q)
    k = qk.kvc_budget_count(cfg.budget, N, S)
    ws = torch.empty(qk.kvc_workspace_size(shape, S, cfg.m, cfg.rho), dtype=torch.uint8, device=DEV)
    kept = torch.empty(L * H * k, dtype=torch.int32, device=DEV)
    Kc = torch.empty(L * H * k * 128, dtype=torch.bfloat16, device=DEV)
    Vc = torch.empty_like(Kc)
    qk.kvc_compress(shape, K, V, Q, S, cfg.m, cfg.rho, 1, [k] * L, kept, Kc, Vc, ws=ws)
    assert qk.kvc_stream_status() == 0
    ref = kv2.kv2_compress(kv2.bf16_to_f64(x.K), kv2.bf16_to_f64(x.V), kv2.bf16_to_f64(x.Q), S, cfg.m, cfg.rho,
                           [k] * L)
    got = kept.cpu().numpy().reshape(L, H, k)
    diff = 0
    for l in range(L):
        for h in range(H):
            compare.assert_topk_set(got[l, h], ref["score"][l, h], S, N, k - S, forced=range(S),
                                    what=f"unchained kept l={l} h={h}")
            diff += len(set(got[l, h].tolist()) ^ set(ref["kept"][l][h].tolist()))
    print(f"tiny-4k: {diff} kept positions differ from the oracle's own pipeline")


def _block_state(qk, L, H, Hq, cap, S, budgets, layout):
    """Block-prefill state in the two-slab or one-slab layout; returns the
    state, the K/V slabs [K0, V0, (K1, V1)] and the position arrays."""
    n_slab = 2 if layout == "two-slab" else 1
    slabs = [torch.zeros(L * H * cap * 128, dtype=torch.bfloat16, device=DEV) for _ in range(2 * n_slab)]
    pos = [torch.zeros(L * H * cap, dtype=torch.int32, device=DEV) for _ in range(n_slab)]
    if n_slab == 2:
        st = qk.kvc_block_state_init(L, H, Hq, cap, S, budgets, slabs[0], slabs[1], pos[0], slabs[2], slabs[3],
                                     pos[1])
    else:
        st = qk.kvc_block_state_init(L, H, Hq, cap, S, budgets, slabs[0], slabs[1], pos[0])
    return st, slabs, pos


@pytest.mark.parametrize("layout", ["two-slab", "one-slab"])
@pytest.mark.parametrize("name", list(EPI_CASES))
def test_block_prefill_matches_oracle(qk, name, layout):
    """EpiCache-style streaming with per-layer budgets, small shapes, checked
    step by step: every over-budget step of every layer is compared with one
    oracle step started from the GPU's state before it, in ascending position
    order -- the step's scores element-wise (1e-3 relative, read from the
    workspace), the kept set up to oracle near-ties within 1e-4 of the
    threshold, the kept K and V rows bit for bit; an under-budget step must
    append the block unchanged.  The one-slab layout holds the same rows in
    another order; its packed image must be in position order."""
    case = dict(n_hist=1500, block=256, sinks=4)
    case.update(EPI_CASES[name])
    cfg = ks.EpiConfig(name, d=128, episodes=1, prompt_len=24, alpha=3.0, **case)
    sens = ks.gen_sensitivity(cfg)
    budgets = qk.kvc_layer_budgets(sens.tolist(), cfg.alpha, cfg.mean_budget, cfg.sinks)
    assert budgets == kv2.layer_budgets(sens.astype(np.float64), cfg.alpha, cfg.mean_budget, cfg.sinks).tolist()
    L, H, Hq, B, P, S = cfg.L, cfg.Hkv, cfg.Hq, cfg.block, cfg.prompt_len, cfg.sinks
    hist = [ks.gen_epi_history_layer(cfg, l) for l in range(L)]
    Kh = np.stack([h[0] for h in hist]); Vh = np.stack([h[1] for h in hist])
    prm = [ks.gen_epi_prompt_layer(cfg, 0, l) for l in range(L)]
    Qp = np.stack([p[0] for p in prm]); Kp = np.stack([p[1] for p in prm])
    cap = max(budgets) + B
    st, slabs, pos = _block_state(qk, L, H, Hq, cap, S, budgets, layout)
    ws = torch.empty(qk.kvc_block_workspace_size(st, B, P), dtype=torch.uint8, device=DEV)
    Qp_d, Kp_d = to_dev(Qp), to_dev(Kp)
    Kf = [kv2.bf16_to_f64(Kh[l]) for l in range(L)]
    Qf = [kv2.bf16_to_f64(Qp[l]) for l in range(L)]
    Kpf = [kv2.bf16_to_f64(Kp[l]) for l in range(L)]
    scored = 0
    for t0 in range(0, cfg.n_hist, B):
        t1 = min(t0 + B, cfg.n_hist)
        prev = [pos[st.cur[l]].view(L, H, cap)[l, :, :st.len[l]].cpu().numpy().astype(np.int64) for l in range(L)]
        kb = to_dev(np.ascontiguousarray(Kh[:, :, t0:t1]))
        vb = to_dev(np.ascontiguousarray(Vh[:, :, t0:t1]))
        qk.kvc_block_prefill_step(st, kb, vb, t1 - t0, Qp_d, Kp_d, P, ws=ws)
        assert qk.kvc_stream_status() == 0
        step_scores = ws[:L * H * cap * 4].view(torch.float32).cpu().numpy().reshape(L, H, cap).astype(np.float64)
        for l in range(L):
            n = st.len[l]
            c = st.cur[l]
            got_pos = pos[c].view(L, H, cap)[l, :, :n].cpu().numpy().astype(np.int64)
            got_K = bits_of(slabs[2 * c]).reshape(L, H, cap, 128)[l, :, :n]
            got_V = bits_of(slabs[2 * c + 1]).reshape(L, H, cap, 128)[l, :, :n]
            cat_pos = np.concatenate([prev[l], np.broadcast_to(np.arange(t0, t1), (H, t1 - t0))], axis=1)
            n_cat = cat_pos.shape[1]
            for h in range(H):
                np.testing.assert_array_equal(got_K[h], Kh[l, h][got_pos[h]])
                np.testing.assert_array_equal(got_V[h], Vh[l, h][got_pos[h]])
            if layout == "two-slab":
                assert np.all(np.diff(got_pos, axis=1) > 0), (t0, l)
            if n_cat <= budgets[l]:
                assert np.array_equal(got_pos, cat_pos), (t0, l)
                continue
            # one oracle step from the GPU's previous state, in position order
            # (the GPU scored its rows in row order: order maps one to the other)
            order = np.argsort(cat_pos, axis=1, kind="stable")
            cat_sorted = np.take_along_axis(cat_pos, order, axis=1)
            assert np.all(cat_sorted[:, :S] == np.arange(S)), "sinks first in both orders"
            Kcat = np.stack([Kf[l][h][cat_sorted[h]] for h in range(H)])
            sc = kv2.block_step_scores(Kcat, Qf[l], Kpf[l], S)
            for h in range(H):
                compare.assert_scores(step_scores[l, h, :n_cat][order[h]][S:], sc[h, S:], floor=0.0,
                                      what=f"block {t0} layer {l} head {h} scores")
                kept_sorted = np.sort(got_pos[h])
                assert len(np.unique(kept_sorted)) == len(kept_sorted)
                idx = np.searchsorted(cat_sorted[h], kept_sorted)
                assert np.array_equal(cat_sorted[h][idx], kept_sorted)
                compare.assert_topk_set(idx, sc[h], S, n_cat, budgets[l] - S, forced=range(S),
                                        what=f"block {t0} layer {l} head {h} kept")
            scored += 1
    assert scored > 0
    # for information: the final caches against the unchained oracle
    diff = 0
    for l in range(L):
        ref = kv2.block_prefill_layer(Kf[l], kv2.bf16_to_f64(Vh[l]), Qf[l], Kpf[l], B, budgets[l], S)
        got = pos[st.cur[l]].view(L, H, cap)[l, :, :st.len[l]].cpu().numpy()
        diff += sum(len(set(got[h].tolist()) ^ set(ref[2][h].tolist())) for h in range(H))
    print(f"{name} ({layout}): {scored} scored layer steps; {diff} positions differ from the unchained oracle")
    # the packed image: every segment in ascending position order
    R = qk.kvc_episode_rows(st)
    Kpk = torch.empty(R * 128, dtype=torch.bfloat16, device=DEV)
    Vpk = torch.empty_like(Kpk)
    ppk = torch.empty(R, dtype=torch.int32, device=DEV)
    qk.kvc_episode_pack(st, Kpk, Vpk, ppk)
    assert qk.kvc_stream_status() == 0
    Kb_, Vb_, pb_ = bits_of(Kpk).reshape(R, 128), bits_of(Vpk).reshape(R, 128), ppk.cpu().numpy()
    row = 0
    for l in range(L):
        n = st.len[l]
        got = pos[st.cur[l]].view(L, H, cap)[l, :, :n].cpu().numpy()
        for h in range(H):
            want = np.sort(got[h])
            np.testing.assert_array_equal(pb_[row:row + n], want)
            np.testing.assert_array_equal(Kb_[row:row + n], Kh[l, h][want])
            np.testing.assert_array_equal(Vb_[row:row + n], Vh[l, h][want])
            row += n
    assert row == R


def test_block_prefill_one_slab_ties(qk):
    """Exact score ties: history keys drawn from 24 distinct rows, so rows
    with the same key score the same and the threshold falls inside groups of
    equal scores.  The one-slab layout, whose rows are not in position order,
    must keep the same positions as the two-slab layout (lower global position
    wins a tie) at every step."""
    cfg = ks.EpiConfig("epi-ties", L=3, Hkv=2, Hq=6, d=128, n_hist=1500, block=256, episodes=1, prompt_len=24,
                       mean_budget=300, alpha=3.0, sinks=4)
    sens = ks.gen_sensitivity(cfg)
    budgets = qk.kvc_layer_budgets(sens.tolist(), cfg.alpha, cfg.mean_budget, cfg.sinks)
    L, H, Hq, B, P, S = cfg.L, cfg.Hkv, cfg.Hq, cfg.block, cfg.prompt_len, cfg.sinks
    rng = np.random.default_rng(7)
    pool = ks.gen_epi_history_layer(cfg, 0)[0][0, :24]                       # 24 distinct bf16 key rows
    Kh = pool[rng.integers(0, 24, size=(L, H, cfg.n_hist))]
    Vh = np.stack([ks.gen_epi_history_layer(cfg, l)[1] for l in range(L)])
    prm = [ks.gen_epi_prompt_layer(cfg, 0, l) for l in range(L)]
    Qp_d = to_dev(np.stack([p[0] for p in prm]))
    Kp_d = to_dev(np.stack([p[1] for p in prm]))
    cap = max(budgets) + B
    runs = [_block_state(qk, L, H, Hq, cap, S, budgets, lay) for lay in ("two-slab", "one-slab")]
    wss = [torch.empty(qk.kvc_block_workspace_size(r[0], B, P), dtype=torch.uint8, device=DEV) for r in runs]
    tied = 0
    for t0 in range(0, cfg.n_hist, B):
        t1 = min(t0 + B, cfg.n_hist)
        st0, _, pos0 = runs[0]
        prev = [pos0[st0.cur[l]].view(L, H, cap)[l, :, :st0.len[l]].cpu().numpy() for l in range(L)]
        kb = to_dev(np.ascontiguousarray(Kh[:, :, t0:t1]))
        vb = to_dev(np.ascontiguousarray(Vh[:, :, t0:t1]))
        sets = []
        for (st, slabs, pos), ws in zip(runs, wss):
            qk.kvc_block_prefill_step(st, kb, vb, t1 - t0, Qp_d, Kp_d, P, ws=ws)
            assert qk.kvc_stream_status() == 0
            sets.append([pos[st.cur[l]].view(L, H, cap)[l, :, :st.len[l]].cpu().numpy() for l in range(L)])
            for l in range(L):
                Kg = bits_of(slabs[2 * st.cur[l]]).reshape(L, H, cap, 128)[l, :, :st.len[l]]
                Vg = bits_of(slabs[2 * st.cur[l] + 1]).reshape(L, H, cap, 128)[l, :, :st.len[l]]
                for h in range(H):
                    np.testing.assert_array_equal(Kg[h], Kh[l, h][sets[-1][l][h]])
                    np.testing.assert_array_equal(Vg[h], Vh[l, h][sets[-1][l][h]])
        sc = wss[0][:L * H * cap * 4].view(torch.float32).cpu().numpy().reshape(L, H, cap)
        for l in range(L):
            n_cat = prev[l].shape[1] + t1 - t0
            for h in range(H):
                assert np.array_equal(np.sort(sets[1][l][h]), sets[0][l][h]), (t0, l, h)
            if n_cat <= budgets[l]:
                continue
            for h in range(H):
                # a tie at the threshold: a score value both kept and evicted
                cat = np.concatenate([prev[l][h], np.arange(t0, t1)])
                keep = np.isin(cat, sets[0][l][h])
                keep[:S] = False
                thr = sc[l, h, :n_cat][keep].min()
                out = ~np.isin(cat, sets[0][l][h])
                tied += int(np.any(sc[l, h, :n_cat][out] == thr))
    assert tied > 0, "the case must exercise ties at the threshold"
    print(f"{tied} (step, layer, head) evictions had ties at the threshold")


@pytest.mark.slow
def test_full_size_llama16k_sampled(qk):
    """The headline workload at full size, in the launch configuration the
    bench times; the oracle checks every proxy value and selection, and the
    scores, eviction and compaction of sampled (layer, KV head) pairs."""
    cfg = ks.LLAMA_16K
    x = ks.gen_kv2(cfg)
    out = run_stages(qk, x, cfg)
    pairs = [(0, 0), (13, 5), (31, 7)]
    L, H, N, S = cfg.L, cfg.Hkv, cfg.N, cfg.sinks
    p_ref, _ = kv2.proxy_scores(x.K)
    compare.assert_scores(out["p"], p_ref, floor=compare.PROXY_FLOOR, what="proxy p")
    chunks = kv2.chunk_plan(N, S, cfg.m, cfg.rho)
    sel_ref, _ = kv2.select_queries(out["p"], N, S, cfg.m, cfg.rho)
    assert np.array_equal(out["sel"], sel_ref)
    sc_ref, _ = kv2.recon_scores(x.K, x.Q, out["sel"], chunks, pairs=pairs)
    k = out["k"]
    for (l, h) in pairs:
        compare.assert_scores(out["score_raw"][l, h, S:], sc_ref[l, h, S:], what=f"score {l},{h}")
        compare.assert_topk_set(out["kept"][l, h], out["score"][l, h], S, N, k - S, forced=range(S))
        np.testing.assert_array_equal(out["Kc"][l, h], x.K[l, h][out["kept"][l, h]])
    # properties that hold for every head at any size
    assert np.all(np.isfinite(out["score"])) and np.all(out["score"] > 0) and np.all(out["score"] <= 1.0 + 1e-6)
    assert np.all(np.diff(out["kept"], axis=2) > 0)


def test_compress_gather_done_event(qk):
    """The optional gather-done event is recorded and changes nothing."""
    cfg = ks.scaled(ks.TINY, L=2, Hkv=2, Hq=4, N=1024, m=256)
    x = ks.gen_kv2(cfg)
    L, H, Hq, N, S = cfg.L, cfg.Hkv, cfg.Hq, cfg.N, cfg.sinks
    shape = (L, H, Hq, 128, N)
    K, V, Q = to_dev(x.K), to_dev(x.V), to_dev(x.Q)
    k = qk.kvc_budget_count(cfg.budget, N, S)
    ws = torch.empty(qk.kvc_workspace_size(shape, S, cfg.m, cfg.rho), dtype=torch.uint8, device=DEV)
    outs = []
    ev = torch.cuda.Event()
    ev.record()
    torch.cuda.synchronize()
    for use in (False, True):
        kept = torch.empty(L * H * k, dtype=torch.int32, device=DEV)
        Kc = torch.empty(L * H * k * 128, dtype=torch.bfloat16, device=DEV)
        Vc = torch.empty_like(Kc)
        qk.kvc_compress_ex(shape, "keydiff", K, V, Q, S, cfg.m, cfg.rho, 2, [k] * L, kept, Kc, Vc, ws=ws,
                           gather_done=ev if use else None)
        torch.cuda.synchronize()
        assert qk.kvc_stream_status() == 0
        outs.append((kept.clone(), Kc.clone(), Vc.clone()))
    assert ev.query()
    assert all(torch.equal(a, b) for a, b in zip(*outs))
    with pytest.raises(ValueError):
        qk.kvc_compress_ex(shape, "keydiff", K, V, Q, S, cfg.m, cfg.rho, 1, [k] * L, kept, Kc, Vc, ws=ws,
                           gather_done=torch.cuda.Event())


def test_compress_in_cuda_graph(qk):
    """After one eager call the whole compression step can be captured into a
    CUDA graph; replays give the eager results bit for bit."""
    cfg = ks.scaled(ks.TINY, L=2, Hkv=2, Hq=4, N=1024, m=256)
    x = ks.gen_kv2(cfg)
    L, H, Hq, N, S = cfg.L, cfg.Hkv, cfg.Hq, cfg.N, cfg.sinks
    shape = (L, H, Hq, 128, N)
    K, V, Q = to_dev(x.K), to_dev(x.V), to_dev(x.Q)
    k = qk.kvc_budget_count(cfg.budget, N, S)
    ws = torch.empty(qk.kvc_workspace_size(shape, S, cfg.m, cfg.rho), dtype=torch.uint8, device=DEV)
    kept = torch.empty(L * H * k, dtype=torch.int32, device=DEV)
    Kc = torch.empty(L * H * k * 128, dtype=torch.bfloat16, device=DEV)
    Vc = torch.empty_like(Kc)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        qk.kvc_compress(shape, K, V, Q, S, cfg.m, cfg.rho, 1, [k] * L, kept, Kc, Vc, ws=ws, stream=s)
    torch.cuda.synchronize()
    ref = (kept.clone(), Kc.clone(), Vc.clone())
    kept.zero_(); Kc.zero_(); Vc.zero_()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        qk.kvc_compress(shape, K, V, Q, S, cfg.m, cfg.rho, 1, [k] * L, kept, Kc, Vc, ws=ws,
                        stream=torch.cuda.current_stream())
    for _ in range(2):
        kept.zero_(); Kc.zero_(); Vc.zero_()
        g.replay()
        torch.cuda.synchronize()
        assert qk.kvc_stream_status() == 0
        assert torch.equal(kept, ref[0]) and torch.equal(Kc, ref[1]) and torch.equal(Vc, ref[2])


def test_block_state_init_validation(qk):
    """The one-slab layout needs all three second-slab buffers absent and a
    capacity its eviction kernel covers; mixed or oversized states are refused
    on the host (KVC_ERR_INVALID) before any device work."""
    L, H, Hq, S = 2, 2, 4, 4
    small = [torch.zeros(L * H * 64 * 128, dtype=torch.bfloat16, device=DEV) for _ in range(4)]
    pos = [torch.zeros(L * H * 64, dtype=torch.int32, device=DEV) for _ in range(2)]
    st = qk.kvc_block_state_init(L, H, Hq, 64, S, [16, 32], small[0], small[1], pos[0])
    assert st.K[1] is None and st.cur[0] == 0
    with pytest.raises(qk.KVCError):      # a second K slab without its V and positions
        qk.kvc_block_state_init(L, H, Hq, 64, S, [16, 32], small[0], small[1], pos[0], small[2], None, None)
    with pytest.raises(qk.KVCError):      # a budget above the capacity
        qk.kvc_block_state_init(L, H, Hq, 64, S, [16, 65], small[0], small[1], pos[0])
    big = 393216 + 128                    # more rows than the in-place eviction covers
    kb = torch.zeros(1 * 1 * big * 128, dtype=torch.bfloat16, device=DEV)
    vb = torch.zeros_like(kb)
    pb = torch.zeros(big, dtype=torch.int32, device=DEV)
    with pytest.raises(qk.KVCError):
        qk.kvc_block_state_init(1, 1, 2, big, S, [1000], kb, vb, pb)
    # the same capacity is fine with two slabs (their eviction falls back to the global-memory kernels)
    kb2, vb2, pb2 = torch.zeros_like(kb), torch.zeros_like(vb), torch.zeros_like(pb)
    qk.kvc_block_state_init(1, 1, 2, big, S, [1000], kb, vb, pb, kb2, vb2, pb2)
