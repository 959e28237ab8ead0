"""Full-size parity of the remaining workloads (GPU, slow): Qwen3-8B shape at
32K with two refinement passes, Llama-3.1-8B shape at 128K, and the EpiCache
block prefill of a 90K-token history (LLaMA3.2-3B shape, 4 episodes).

At these sizes the oracle checks every value it can afford (proxy scores,
selections, refinement scores) and samples the rest: whole (layer, KV head)
pairs, or whole chunks of them, and whole layers of the block prefill (the
layers of a block prefill evolve independently).  Each check runs the oracle
on the GPU's own upstream output.
"""
import math
import time

import numpy as np
import pytest
import torch

import kv_synth as ks
from oracle import compare, kv2

pytestmark = [pytest.mark.gpu, pytest.mark.slow]
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


def to_dev(bits):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).to(DEV)


def bits_of(t):
    return t.view(torch.int16).cpu().numpy().view(np.uint16)


def check_chunks(x, cfg, sel, score_gpu, pairs, chunk_ids=None):
    """Oracle scores of the listed (layer, KV head) pairs (optionally only
    some chunks of them) on the GPU's selection."""
    chunks = kv2.chunk_plan(cfg.N, cfg.sinks, cfg.m, cfg.rho)
    G = cfg.G
    for (l, h) in pairs:
        Klh = kv2.bf16_to_f64(x.K[l, h])
        use = chunks if chunk_ids is None else [chunks[i] for i in chunk_ids]
        for c in use:
            idx = sel[c.off:c.off + c.nq]
            Qrows = np.stack([kv2.bf16_to_f64(x.Q[l, h * G + g][idx]) for g in range(G)])
            one = kv2.Chunk(c.lo, c.hi, 0, c.nq)
            sc, _ = kv2.recon_head(Klh, Qrows, Klh[idx], [one])
            compare.assert_scores(score_gpu[l, h, c.lo:c.hi], sc[c.lo:c.hi],
                                  what=f"scores l={l} h={h} chunk [{c.lo},{c.hi})")


def test_qwen32k_refinement_passes(qk):
    cfg = ks.QWEN_32K
    x = ks.gen_kv2(cfg, threads=8)
    L, H, Hq, N, S = cfg.L, cfg.Hkv, cfg.Hq, cfg.N, cfg.sinks
    shape = (L, H, Hq, 128, N)
    K, Q = to_dev(x.K), to_dev(x.Q)
    off = qk.kvc_chunk_plan(N, S, cfg.m, cfg.rho)
    assert off[-1] == 8191
    ws = torch.empty(qk.kvc_workspace_size(shape, S, cfg.m, cfg.rho), dtype=torch.uint8, device=DEV)
    p = torch.empty(N, dtype=torch.float32, device=DEV)
    sel = torch.empty(off[-1], dtype=torch.int32, device=DEV)
    score = torch.empty(L * H * N, dtype=torch.float32, device=DEV)
    qk.kvc_proxy_score(shape, K, p, ws=ws)
    p_ref, _ = kv2.proxy_scores(x.K)
    compare.assert_scores(p.cpu().numpy(), p_ref, floor=compare.PROXY_FLOOR, what="proxy p")
    pairs = [(0, 0), (35, 7)]
    for t in range(cfg.passes):
        qk.kvc_select_queries(N, S, cfg.m, cfg.rho, p, sel)
        p_np = p.cpu().numpy().astype(np.float64)
        sel_np = sel.cpu().numpy().astype(np.int64)
        ref_sel, _ = kv2.select_queries(p_np, N, S, cfg.m, cfg.rho)
        assert np.array_equal(sel_np, ref_sel), f"pass {t}: selection"
        qk.kvc_recon_score(shape, K, Q, sel, S, cfg.m, cfg.rho, score, ws=ws)
        assert qk.kvc_stream_status() == 0
        sc = score.cpu().numpy().reshape(L, H, N).astype(np.float64)
        check_chunks(x, cfg, sel_np, sc, pairs[t % 2:t % 2 + 1], chunk_ids=[0, 7] if t else None)
        if t + 1 < cfg.passes:
            qk.kvc_refine_proxy(shape, score, S, p)
            compare.assert_scores(p.cpu().numpy(), kv2.refine_proxy(sc, S), rtol=1e-5, what="refined p")
    k = qk.kvc_budget_count(cfg.budget, N, S)
    assert k == 1638
    kept = torch.empty(L * H * k, dtype=torch.int32, device=DEV)
    qk.kvc_evict_topk(shape, score, S, [k] * L, kept, ws=ws)
    V = to_dev(x.V)
    Kc = torch.empty(L * H * k * 128, dtype=torch.bfloat16, device=DEV)
    Vc = torch.empty_like(Kc)
    qk.kvc_compact(shape, K, V, kept, [k] * L, Kc, Vc)
    assert qk.kvc_stream_status() == 0
    sc = score.cpu().numpy().reshape(L, H, N).astype(np.float64)
    kept_np = kept.cpu().numpy().reshape(L, H, k)
    Kc_np = bits_of(Kc).reshape(L, H, k, 128)
    for (l, h) in [(0, 0), (17, 3), (35, 7)]:
        compare.assert_topk_set(kept_np[l, h], sc[l, h], S, N, k - S, forced=range(S), what=f"kept {l},{h}")
        np.testing.assert_array_equal(Kc_np[l, h], x.K[l, h][kept_np[l, h]])
    assert np.all(np.diff(kept_np, axis=2) > 0)


def test_llama128k_sampled(qk):
    cfg = ks.LLAMA_128K
    x = ks.gen_kv2(cfg, threads=4)
    L, H, Hq, N, S = cfg.L, cfg.Hkv, cfg.Hq, cfg.N, cfg.sinks
    shape = (L, H, Hq, 128, N)
    K, V, Q = to_dev(x.K), to_dev(x.V), to_dev(x.Q)
    off = qk.kvc_chunk_plan(N, S, cfg.m, cfg.rho)
    assert off[-1] == 65534
    k = qk.kvc_budget_count(cfg.budget, N, S)
    assert k == 13107
    ws = torch.empty(qk.kvc_workspace_size(shape, S, cfg.m, cfg.rho), dtype=torch.uint8, device=DEV)
    p = torch.empty(N, dtype=torch.float32, device=DEV)
    sel = torch.empty(off[-1], dtype=torch.int32, device=DEV)
    score = torch.empty(L * H * N, dtype=torch.float32, device=DEV)
    kept = torch.empty(L * H * k, dtype=torch.int32, device=DEV)
    Kc = torch.empty(L * H * k * 128, dtype=torch.bfloat16, device=DEV)
    Vc = torch.empty_like(Kc)
    t0 = time.perf_counter()
    qk.kvc_compress(shape, K, V, Q, S, cfg.m, cfg.rho, 1, [k] * L, kept, Kc, Vc, p=p, sel=sel, score=score, ws=ws)
    assert qk.kvc_stream_status() == 0
    print(f"128K compress (first call) {1e3 * (time.perf_counter() - t0):.1f} ms")
    p_ref, _ = kv2.proxy_scores(x.K)
    compare.assert_scores(p.cpu().numpy(), p_ref, floor=compare.PROXY_FLOOR, what="proxy p")
    sel_np = sel.cpu().numpy().astype(np.int64)
    ref_sel, _ = kv2.select_queries(p.cpu().numpy().astype(np.float64), N, S, cfg.m, cfg.rho)
    assert np.array_equal(sel_np, ref_sel)
    sc = score.cpu().numpy().reshape(L, H, N).astype(np.float64)
    check_chunks(x, cfg, sel_np, sc, [(13, 5)], chunk_ids=[0, 15, 31])
    kept_np = kept.cpu().numpy().reshape(L, H, k)
    Kc_np = bits_of(Kc).reshape(L, H, k, 128)
    Vc_np = bits_of(Vc).reshape(L, H, k, 128)
    for (l, h) in [(0, 0), (31, 7)]:
        compare.assert_topk_set(kept_np[l, h], sc[l, h], S, N, k - S, forced=range(S), what=f"kept {l},{h}")
        np.testing.assert_array_equal(Kc_np[l, h], x.K[l, h][kept_np[l, h]])
        np.testing.assert_array_equal(Vc_np[l, h], x.V[l, h][kept_np[l, h]])
    assert np.all(np.isfinite(sc)) and np.all(sc > 0) and np.all(sc <= 1.0 + 1e-6)
    assert np.all(np.diff(kept_np, axis=2) > 0)


def test_epicache_block_prefill_full(qk):
    """90K-token history in 2048-token blocks, 28 layers with sensitivity-
    weighted budgets (alpha = 3, mean 8192), 4 episodes.  For sampled layers
    every step is compared with one oracle step started from the GPU's state
    before that step."""
    cfg = ks.EPI_3B
    L, H, Hq, B, P, S = cfg.L, cfg.Hkv, cfg.Hq, cfg.block, cfg.prompt_len, cfg.sinks
    sens = ks.gen_sensitivity(cfg)
    budgets = qk.kvc_layer_budgets(sens.tolist(), cfg.alpha, cfg.mean_budget, S)
    assert budgets == kv2.layer_budgets(sens.astype(np.float64), cfg.alpha, cfg.mean_budget, S).tolist()
    assert sum(budgets) == L * cfg.mean_budget
    hist = [ks.gen_epi_history_layer(cfg, l) for l in range(L)]
    Kh = np.stack([h[0] for h in hist])
    Vh = np.stack([h[1] for h in hist])
    del hist
    cap = max(budgets) + B
    slabs = [torch.zeros(L * H * cap * 128, dtype=torch.bfloat16, device=DEV) for _ in range(4)]
    pos = [torch.zeros(L * H * cap, dtype=torch.int32, device=DEV) for _ in range(2)]
    Kh_d = to_dev(Kh)
    Vh_d = to_dev(Vh)
    sample = {0: [0, 27], 1: [13], 2: [5], 3: [20]}
    for e in range(cfg.episodes):
        prm = [ks.gen_epi_prompt_layer(cfg, e, l) for l in range(L)]
        Qp = np.stack([p[0] for p in prm])
        Kp = np.stack([p[1] for p in prm])
        Qp_d, Kp_d = to_dev(Qp), to_dev(Kp)
        st = qk.kvc_block_state_init(L, H, Hq, cap, S, budgets, slabs[0], slabs[1], pos[0], slabs[2], slabs[3],
                                     pos[1])
        ws = torch.empty(qk.kvc_block_workspace_size(st, B, P), dtype=torch.uint8, device=DEV)
        t_gpu = 0.0
        for t0 in range(0, cfg.n_hist, B):
            t1 = min(t0 + B, cfg.n_hist)
            kb = Kh_d.view(L, H, cfg.n_hist, 128)[:, :, t0:t1].contiguous()
            vb = Vh_d.view(L, H, cfg.n_hist, 128)[:, :, t0:t1].contiguous()
            before = {l: (st.cur[l], st.len[l]) for l in sample[e]}
            prev = {l: pos[st.cur[l]].view(L, H, cap)[l, :, :st.len[l]].cpu().numpy() for l in sample[e]}
            torch.cuda.synchronize()
            a = time.perf_counter()
            qk.kvc_block_prefill_step(st, kb, vb, t1 - t0, Qp_d, Kp_d, P, ws=ws)
            assert qk.kvc_stream_status() == 0
            t_gpu += time.perf_counter() - a
            for l in sample[e]:
                n = st.len[l]
                got_pos = pos[st.cur[l]].view(L, H, cap)[l, :, :n].cpu().numpy()
                got_K = bits_of(slabs[2 * st.cur[l]]).reshape(L, H, cap, 128)[l, :, :n]
                for h in range(H):
                    np.testing.assert_array_equal(got_K[h], Kh[l, h][got_pos[h]])
                # one oracle step from the GPU's previous state
                old = prev[l].astype(np.int64)
                Kc = np.stack([kv2.bf16_to_f64(Kh[l, h][old[h]]) for h in range(H)])
                cat_pos = np.concatenate([old, np.broadcast_to(np.arange(t0, t1), (H, t1 - t0))], axis=1)
                n_cat = cat_pos.shape[1]
                if n_cat <= budgets[l]:
                    assert np.array_equal(got_pos, cat_pos)
                    continue
                Kcat = np.concatenate([Kc, kv2.bf16_to_f64(Kh[l, :, t0:t1])], axis=1)
                sc = kv2.block_step_scores(Kcat, kv2.bf16_to_f64(Qp[l]), kv2.bf16_to_f64(Kp[l]), S)
                for h in range(H):
                    # kept rows as cache indices of the concatenated cache
                    idx = np.searchsorted(cat_pos[h], got_pos[h])
                    assert np.array_equal(cat_pos[h][idx], got_pos[h])
                    compare.assert_topk_set(idx, sc[h], S, n_cat, budgets[l] - S, forced=range(S),
                                            what=f"episode {e} layer {l} head {h} block at {t0}")
        print(f"episode {e}: {cfg.n_hist} tokens in {t_gpu * 1e3:.1f} ms of block steps (incl. host sync per step)")
