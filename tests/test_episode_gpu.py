"""GPU parity of EpiCache's per-turn path ("[26'ICML] EpiCache", "방법: 3단계"
step ③, Fig. 3) through the C ABI: question-to-episode matching against the
float64 oracle, the packed episode image (bit copies of the state's kept
rows), decode attention over that image, and the pinned host <-> device swap.

Matching tolerance: squared distances within 1e-5 relative (fp32 sums over
De terms); the chosen episode must be a closest one up to that tolerance
(exact ties go to the lower index on both sides); the threshold decision
may differ only for questions within that tolerance of tau."""
import json
import os

import numpy as np
import pytest
import torch

import kv_synth as ks
from oracle import decode, episode, kv2

pytestmark = pytest.mark.gpu
DEV = "cuda:0"
GOLD = os.path.join(os.path.dirname(__file__), "golden")


@pytest.fixture(scope="module")
def qk():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    import __graft_entry__ as ge
    ge.build()
    import query_agnostic_kv_gb300 as q
    q.kvc_device_check()
    return q


def match(qk, Q, C, tau=0.0):
    q = torch.from_numpy(Q).to(DEV)
    c = torch.from_numpy(C).to(DEV)
    ep = torch.full((Q.shape[0],), -7, dtype=torch.int32, device=DEV)
    d2 = torch.empty(Q.shape[0], C.shape[0], dtype=torch.float32, device=DEV)
    qk.kvc_episode_match(q, c, ep, d2, tau=tau)
    assert qk.kvc_stream_status() == 0
    return ep.cpu().numpy(), d2.cpu().numpy()


def check_match(Q, C, ep_g, d2_g, tau=None):
    ep_r, d2_r = episode.nearest_episode(Q.astype(np.float64), C.astype(np.float64), tau)
    np.testing.assert_allclose(d2_g, d2_r, rtol=1e-5, atol=1e-6)
    mins = d2_r.min(axis=1)
    for b in range(len(ep_g)):
        tol = 1e-5 * mins[b] + 1e-6
        if tau is not None and abs(mins[b] - tau * tau) <= 1e-5 * tau * tau + 1e-6:
            continue                                   # threshold near-tie: either answer is valid
        if ep_r[b] == -1:
            assert ep_g[b] == -1, b
            continue
        assert ep_g[b] >= 0 and d2_r[b, ep_g[b]] <= mins[b] + tol, b
        if ep_g[b] != ep_r[b]:                         # only a near-tie may differ
            assert abs(d2_r[b, ep_g[b]] - d2_r[b, ep_r[b]]) <= tol, b


def test_match_hand_worked(qk):
    g = json.load(open(os.path.join(GOLD, "episode_match_small.json")))
    Q, C = np.array(g["queries"], np.float32), np.array(g["centroids"], np.float32)
    Q4, C4 = np.zeros((len(Q), 4), np.float32), np.zeros((len(C), 4), np.float32)   # De must be a multiple of 4
    Q4[:, :2], C4[:, :2] = Q, C
    ep, d2 = match(qk, Q4, C4)
    np.testing.assert_array_equal(d2, np.array(g["d2"], np.float32))
    assert ep.tolist() == g["episode"]
    ep, _ = match(qk, Q4, C4, tau=g["tau"])
    assert ep.tolist() == g["episode_tau"]


@pytest.mark.parametrize("E,De,B", [(4, 1024, 2000), (37, 260, 301), (1, 4, 5), (64, 4096, 64)])
def test_match_random(qk, E, De, B):
    C, Q = ks.gen_turn_embeddings(E, De, B, seed=E + De)
    ep, d2 = match(qk, Q, C)
    check_match(Q, C, ep, d2)
    tau = float(np.sqrt(np.median(d2.min(axis=1))))
    ep, d2 = match(qk, Q, C, tau=tau)
    check_match(Q, C, ep, d2, tau=tau)
    assert (ep == -1).any() and (ep >= 0).any()


def test_match_rejects_bad_arguments(qk):
    q = torch.zeros(3, 6, device=DEV)
    with pytest.raises(qk.KVCError):
        qk.kvc_episode_match(q, torch.zeros(2, 6, device=DEV), torch.empty(3, dtype=torch.int32, device=DEV))


def build_state(qk, L=3, H=2, Hq=6, n_hist=1300, B=256, mean_budget=280):
    cfg = ks.EpiConfig("epi-pack", L=L, Hkv=H, Hq=Hq, d=128, n_hist=n_hist, block=B, episodes=1, prompt_len=16,
                       mean_budget=mean_budget, alpha=3.0, sinks=4)
    budgets = qk.kvc_layer_budgets(ks.gen_sensitivity(cfg).tolist(), cfg.alpha, cfg.mean_budget, cfg.sinks)
    hist = [ks.gen_epi_history_layer(cfg, l) for l in range(L)]
    Kh = np.stack([h[0] for h in hist]); Vh = np.stack([h[1] for h in hist])
    prm = [ks.gen_epi_prompt_layer(cfg, 0, l) for l in range(L)]
    Qp = np.stack([p[0] for p in prm]); Kpr = np.stack([p[1] for p in prm])
    cap = max(budgets) + B

    def dev(bits):
        return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).to(DEV)

    slabs = [torch.zeros(L * H * cap * 128, dtype=torch.bfloat16, device=DEV) for _ in range(4)]
    pos = [torch.zeros(L * H * cap, dtype=torch.int32, device=DEV) for _ in range(2)]
    st = qk.kvc_block_state_init(L, H, Hq, cap, cfg.sinks, budgets, slabs[0], slabs[1], pos[0], slabs[2], slabs[3],
                                 pos[1])
    ws = torch.empty(qk.kvc_block_workspace_size(st, B, cfg.prompt_len), dtype=torch.uint8, device=DEV)
    Qd, Kd = dev(Qp), dev(Kpr)
    for t0 in range(0, n_hist, B):
        t1 = min(t0 + B, n_hist)
        qk.kvc_block_prefill_step(st, dev(Kh[:, :, t0:t1]), dev(Vh[:, :, t0:t1]), t1 - t0, Qd, Kd, cfg.prompt_len,
                                  ws=ws)
    assert qk.kvc_stream_status() == 0
    return st, slabs, pos, cap


def test_pack_is_bit_copy_of_the_state_and_decodes(qk):
    L, H = 3, 2
    st, slabs, pos, cap = build_state(qk, L=L, H=H)
    rows = qk.kvc_episode_rows(st)
    assert rows == H * sum(st.len[l] for l in range(L))
    Kp = torch.empty(rows, 128, dtype=torch.bfloat16, device=DEV)
    Vp = torch.empty_like(Kp)
    Pp = torch.empty(rows, dtype=torch.int32, device=DEV)
    qk.kvc_episode_pack(st, Kp, Vp, Pp)
    assert qk.kvc_stream_status() == 0
    layers_K, layers_V, layers_P = [], [], []
    for l in range(L):
        c, n = st.cur[l], st.len[l]
        K = slabs[2 * c].view(L, H, cap, 128)[l, :, :n]
        V = slabs[2 * c + 1].view(L, H, cap, 128)[l, :, :n]
        P = pos[c].view(L, H, cap)[l, :, :n]
        layers_K.append(K.view(torch.int16).cpu().numpy())
        layers_V.append(V.view(torch.int16).cpu().numpy())
        layers_P.append(P.cpu().numpy())
    K_r, V_r, P_r, lens = episode.pack_cache(layers_K, layers_V, layers_P)
    np.testing.assert_array_equal(Kp.view(torch.int16).cpu().numpy(), K_r)
    np.testing.assert_array_equal(Vp.view(torch.int16).cpu().numpy(), V_r)
    np.testing.assert_array_equal(Pp.cpu().numpy(), P_r)
    # the packed image is decoded in place through the compacted-layout segment table
    off, ln = qk.kvc_compact_segments(L, H, lens)
    G = 3
    q = torch.randn(L * H, G, 128, generator=torch.Generator(device=DEV).manual_seed(9), device=DEV)
    q = q.to(torch.bfloat16)
    out = torch.empty(L * H, G, 128, dtype=torch.float32, device=DEV)
    ws = torch.empty(qk.kvc_decode_workspace_size(L * H, G, max(lens)), dtype=torch.uint8, device=DEV)
    qk.kvc_decode_attention(Kp, Vp, torch.tensor(off, device=DEV), torch.tensor(ln, dtype=torch.int32, device=DEV),
                            max(lens), q, out, ws=ws)
    assert qk.kvc_stream_status() == 0
    Kf, Vf, qf = Kp.double().cpu().numpy(), Vp.double().cpu().numpy(), q.double().cpu().numpy()
    ref, _ = decode.decode_attention(Kf, Vf, off, ln, qf)
    aw = decode.abs_weighted(Kf, Vf, off, ln, qf)
    assert np.all(np.abs(out.cpu().numpy() - ref) <= 2e-4 * aw + 1e-6)


def test_swap_round_trip_on_two_streams(qk):
    n = 3 * 1024 * 1024 + 8                                     # bf16 elements, not a multiple of anything nice
    a = torch.randn(n, device=DEV).to(torch.bfloat16)
    b = torch.randn(n).to(torch.bfloat16).pin_memory()
    host_out = torch.empty(n, dtype=torch.bfloat16).pin_memory()
    dev_in = torch.empty(n, dtype=torch.bfloat16, device=DEV)
    s_out, s_in = torch.cuda.Stream(), torch.cuda.Stream()
    torch.cuda.synchronize()
    qk.kvc_episode_swap(a, host_out, b, dev_in, out_stream=s_out, in_stream=s_in)
    torch.cuda.synchronize()
    assert torch.equal(host_out, a.cpu()) and torch.equal(dev_in.cpu(), b)
    qk.kvc_episode_swap(host_in=host_out, dev_in=dev_in)      # load only
    torch.cuda.synchronize()
    assert torch.equal(dev_in, a)
    with pytest.raises(qk.KVCError):
        qk.kvc_episode_swap(a, torch.empty(n, dtype=torch.bfloat16), None, None)   # pageable host memory
