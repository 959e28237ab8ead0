"""The layer-sharded call sequence on one GPU.

The KV² page's proxy is a mean over every (layer, KV head) pair and the sink
pin takes the max over every score ("어떻게 동작하나", "무엇과 다른가"); the
rest of the path is per (layer, KV head).  A cache split by layers therefore
needs one sum of N floats per pass and one max.  Here two shards (the first
and second half of the layers) run one after the other on the same GPU, the
sums and the max taken on the device by plain tensor arithmetic in place of
the collective, and the result is compared with the unsharded kvc_compress.
"""
import numpy as np
import pytest
import torch

import kv_synth as ks
from oracle import compare

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


def _bf16(a):
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).to(DEV)


@pytest.mark.parametrize("proxy", ["keydiff", "knorm"])
def test_two_layer_shards_match_unsharded(qk, proxy):
    cfg = ks.scaled(ks.TINY, name="shard", L=4, Hkv=2, Hq=8, N=3000, m=1000, rho=0.1, budget=0.05,
                    needles_per_layer=6, passes=2)
    x = ks.gen_kv2(cfg)
    L, H, Hq, N, S, d = cfg.L, cfg.Hkv, cfg.Hq, cfg.N, cfg.sinks, 128
    K, V, Q = _bf16(x.K), _bf16(x.V), _bf16(x.Q)
    k = qk.kvc_budget_count(cfg.budget, N, S)
    off = qk.kvc_chunk_plan(N, S, cfg.m, cfg.rho)
    nq = off[-1]

    # ---- unsharded
    shape = (L, H, Hq, d, N)
    ws = torch.empty(qk.kvc_workspace_size(shape, S, cfg.m, cfg.rho), dtype=torch.uint8, device=DEV)
    kept_u = torch.empty(L * H * k, dtype=torch.int32, device=DEV)
    Kc_u = torch.empty(L * H * k * d, dtype=torch.bfloat16, device=DEV)
    Vc_u = torch.empty_like(Kc_u)
    score_u = torch.empty(L * H * N, dtype=torch.float32, device=DEV)
    sel_u = torch.empty(nq, dtype=torch.int32, device=DEV)
    p_u = torch.empty(N, dtype=torch.float32, device=DEV)
    qk.kvc_proxy_score_kind(shape, proxy, K, p_u, ws=ws)
    p1_u = p_u.clone()
    qk.kvc_compress_ex(shape, proxy, K, V, Q, S, cfg.m, cfg.rho, 2, [k] * L, kept_u, Kc_u, Vc_u, p=p_u, sel=sel_u,
                       score=score_u, ws=ws)
    assert qk.kvc_stream_status() == 0

    # ---- two shards of L/2 layers each
    Ls = L // 2
    shp = (Ls, H, Hq, d, N)
    Kv = K.view(L, -1)
    Vv = V.view(L, -1)
    Qv = Q.view(L, -1)
    score_s = torch.empty(L * H * N, dtype=torch.float32, device=DEV)
    sv = score_s.view(L, -1)
    wss = [torch.empty(qk.kvc_workspace_size(shp, S, cfg.m, cfg.rho), dtype=torch.uint8, device=DEV)
           for _ in range(2)]
    psum = [torch.empty(N, dtype=torch.float32, device=DEV) for _ in range(2)]
    shard = [slice(0, Ls), slice(Ls, L)]
    p_s = torch.empty(N, dtype=torch.float32, device=DEV)
    sel_s = torch.empty(nq, dtype=torch.int32, device=DEV)
    for t in range(2):
        for r in range(2):
            if t == 0:
                qk.kvc_proxy_partial(shp, proxy, Kv[shard[r]].reshape(-1), psum[r], ws=wss[r])
            else:
                qk.kvc_refine_partial(shp, sv[shard[r]].reshape(-1), S, psum[r])
        qk.kvc_proxy_from_sums(N, L * H, psum[0] + psum[1], p_s)       # the all-reduce(sum) of the N floats
        if t == 0:
            compare.assert_scores(p_s.cpu().numpy(), p1_u.cpu().numpy(), rtol=1e-5, floor=1e-6,
                                  what="proxy from shard sums")
        qk.kvc_select_queries(N, S, cfg.m, cfg.rho, p_s, sel_s)
        for r in range(2):
            qk.kvc_recon_score(shp, Kv[shard[r]].reshape(-1), Qv[shard[r]].reshape(-1), sel_s, S, cfg.m, cfg.rho,
                               sv[shard[r]].reshape(-1), ws=wss[r])
    kept_s = torch.empty(L * H * k, dtype=torch.int32, device=DEV)
    kv_ = kept_s.view(L, -1)
    Kc_s = torch.empty(L * H * k * d, dtype=torch.bfloat16, device=DEV)
    Vc_s = torch.empty_like(Kc_s)
    maxes = torch.empty(2, dtype=torch.float32, device=DEV)
    for r in range(2):
        qk.kvc_evict_compact(shp, sv[shard[r]].reshape(-1), S, [k] * Ls, kv_[shard[r]].reshape(-1),
                             Kv[shard[r]].reshape(-1), Vv[shard[r]].reshape(-1),
                             Kc_s.view(L, -1)[shard[r]].reshape(-1), Vc_s.view(L, -1)[shard[r]].reshape(-1),
                             ws=wss[r])
        qk.kvc_score_max(shp, sv[shard[r]].reshape(-1), S, maxes[r:r + 1], ws=wss[r])
    gmax = maxes.max().reshape(1)                                       # the all-reduce(max)
    for r in range(2):
        qk.kvc_pin_sinks(shp, sv[shard[r]].reshape(-1), S, gmax)
    assert qk.kvc_stream_status() == 0

    sc = score_s.cpu().numpy().reshape(L, H, N)
    assert np.all(sc[:, :, :S] == sc[:, :, S:].max())
    kept_g = kept_s.cpu().numpy().reshape(L, H, k)
    Kc_g = Kc_s.view(torch.int16).cpu().numpy().view(np.uint16).reshape(L, H, k, d)
    for l in range(L):
        for h in range(H):
            compare.assert_topk_set(kept_g[l, h], sc[l, h].astype(np.float64), S, N, k - S, forced=range(S),
                                    what=f"sharded kept l={l} h={h}")
            np.testing.assert_array_equal(Kc_g[l, h], x.K[l, h][kept_g[l, h]])
    if torch.equal(sel_s, sel_u):
        # the same queries: every per-layer result is the unsharded one, bit for bit
        assert torch.equal(score_s, score_u)
        assert torch.equal(kept_s, kept_u)
        assert torch.equal(Kc_s, Kc_u) and torch.equal(Vc_s, Vc_u)
    else:
        print("sharded selection differs from the unsharded one on a near-tie of p")
