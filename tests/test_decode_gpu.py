"""GPU parity of decode attention over compacted-cache segments (the compact
serving backend of the KV² page, "전제와 한계"), called through the C ABI,
against the float64 oracle on the same seeded inputs.

Tolerance: |gpu - ref| <= 2e-4 * sum_i softmax_i |v_i| + 1e-6 per output
element (the natural scale of the rounding error of a weighted sum: fp32
logits from exact bf16 products, a 2-ulp exp2, fp32 accumulation over up to
~10^4 rows, observed errors ~1e-6 of that scale); lse within
1e-4 * max(1, |lse|).
"""
import math

import numpy as np
import pytest
import torch

import kv_synth as ks
from oracle import decode

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


def run(qk, x, max_len=None, scale=0.0, ws=None, lse=True):
    n_seg, G = x["q"].shape[0], x["q"].shape[1]
    if max_len is None:
        max_len = int(x["seg_len"].max().item()) if n_seg else 0
    if ws is None:
        ws = torch.empty(qk.kvc_decode_workspace_size(n_seg, G, max_len), dtype=torch.uint8, device=DEV)
    out = torch.full((n_seg, G, 128), float("nan"), dtype=torch.float32, device=DEV)
    l = torch.full((n_seg, G), float("nan"), dtype=torch.float32, device=DEV) if lse else None
    qk.kvc_decode_attention(x["K"], x["V"], x["seg_off"], x["seg_len"], max_len, x["q"], out, l, scale=scale, ws=ws)
    return out, l


def check(x, out, lse, segs=None, scale=None):
    K, V, q = (x[k].double().cpu().numpy() for k in ("K", "V", "q"))
    off, ln = x["seg_off"].cpu().numpy(), x["seg_len"].cpu().numpy()
    segs = range(len(ln)) if segs is None else segs
    o_g, l_g = out.cpu().numpy(), None if lse is None else lse.cpu().numpy()
    for s in segs:
        ref, rl = decode.decode_attention(K, V, off[s:s + 1], ln[s:s + 1], q[s:s + 1], scale)
        aw = decode.abs_weighted(K, V, off[s:s + 1], ln[s:s + 1], q[s:s + 1], scale)
        err = np.abs(o_g[s] - ref[0])
        tol = 2e-4 * aw[0] + 1e-6
        assert np.all(err <= tol), (s, int(ln[s]), float((err / tol).max()))
        if l_g is not None:
            if ln[s] == 0:
                assert np.all(np.isneginf(l_g[s]))
            else:
                assert np.all(np.abs(l_g[s] - rl[0]) <= 1e-4 * np.maximum(1.0, np.abs(rl[0]))), s


RAGGED = [0, 1, 2, 63, 64, 65, 95, 96, 97, 191, 192, 193, 577, 1000, 4097]


@pytest.mark.parametrize("G", [1, 2, 3, 4, 5, 8])
def test_ragged_segments(qk, G):
    cfg = ks.DecodeConfig("ragged", seqs=1, Hkv=1, G=G, kept=0, seed=20 + G)
    x = ks.gen_decode(cfg, DEV, lens=RAGGED, gap=5)
    out, lse = run(qk, x)
    assert qk.kvc_stream_status() == 0
    check(x, out, lse)


def test_split_merge_many_lengths(qk):
    """Few long segments -> many splits per segment, merged by the last CTA."""
    cfg = ks.DecodeConfig("split", seqs=1, Hkv=1, G=4, kept=0, seed=31)
    lens = [5000, 4999, 3, 2600, 12000, 577]
    x = ks.gen_decode(cfg, DEV, lens=lens, gap=1)
    out, lse = run(qk, x)
    assert qk.kvc_stream_status() == 0
    check(x, out, lse)
    # max_len larger than any segment changes the split plan, not the result
    out2, lse2 = run(qk, x, max_len=30000)
    assert qk.kvc_stream_status() == 0
    check(x, out2, lse2)


def test_deterministic_and_workspace_reuse(qk):
    cfg = ks.DecodeConfig("det", seqs=1, Hkv=1, G=4, kept=0, seed=32)
    x = ks.gen_decode(cfg, DEV, lens=[7000, 300, 9000, 1], gap=0)
    ws = torch.empty(qk.kvc_decode_workspace_size(4, 4, 9000), dtype=torch.uint8, device=DEV)
    a, la = run(qk, x, ws=ws)
    b, lb = run(qk, x, ws=ws)
    assert qk.kvc_stream_status() == 0
    assert torch.equal(a, b) and torch.equal(la, lb)


def test_custom_scale_and_no_lse(qk):
    cfg = ks.DecodeConfig("scale", seqs=1, Hkv=1, G=3, kept=0, seed=33)
    x = ks.gen_decode(cfg, DEV, lens=[129, 2000, 40], gap=2)
    out, _ = run(qk, x, scale=0.05, lse=False)
    assert qk.kvc_stream_status() == 0
    check(x, out, None, scale=0.05)


def test_bounds_reported_and_other_segments_intact(qk):
    cfg = ks.DecodeConfig("bounds", seqs=1, Hkv=1, G=4, kept=0, seed=34)
    x = ks.gen_decode(cfg, DEV, lens=[100, 200, 50], gap=0)
    x["seg_off"][1] = x["rows"] - 100          # runs past the end of the cache
    out, lse = run(qk, x)
    assert qk.kvc_stream_status() == 4
    assert qk.kvc_stream_status() == 0          # cleared by the read
    check(x, out, lse, segs=[0, 2])
    assert torch.isnan(out[1]).all()            # skipped: left unwritten


def test_decode_over_compress_output(qk):
    """The compacted cache written by kvc_compress is decoded directly through
    the segment table of its layout."""
    cfg = ks.scaled(ks.TINY, L=2, Hkv=2, Hq=8, N=2048, m=512)
    x = ks.gen_kv2(cfg)
    L, H, Hq, N, S = cfg.L, cfg.Hkv, cfg.Hq, cfg.N, cfg.sinks
    shape = (L, H, Hq, 128, N)

    def dev(bits):
        return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).to(DEV)

    K, V, Q = dev(x.K), dev(x.V), dev(x.Q)
    kl = [qk.kvc_budget_count(0.1, N, S), qk.kvc_budget_count(0.05, N, S)]
    rows = H * sum(kl)
    kept = torch.empty(rows, dtype=torch.int32, device=DEV)
    Kc = torch.empty(rows, 128, dtype=torch.bfloat16, device=DEV)
    Vc = torch.empty_like(Kc)
    ws = torch.empty(qk.kvc_workspace_size(shape, S, cfg.m, cfg.rho), dtype=torch.uint8, device=DEV)
    qk.kvc_compress(shape, K, V, Q, S, cfg.m, cfg.rho, 1, kl, kept, Kc, Vc, ws=ws)
    off, ln = qk.kvc_compact_segments(L, H, kl)
    G = Hq // H
    qdec = torch.randn(L * H, G, 128, generator=torch.Generator(device=DEV).manual_seed(5), device=DEV)
    y = dict(K=Kc, V=Vc, q=qdec.to(torch.bfloat16), rows=rows,
             seg_off=torch.tensor(off, dtype=torch.int64, device=DEV),
             seg_len=torch.tensor(ln, dtype=torch.int32, device=DEV))
    out, lse = run(qk, y)
    assert qk.kvc_stream_status() == 0
    check(y, out, lse)


def test_full_size_decode_batch(qk):
    """The bench's launch: 64 sequences x 8 KV heads x 13107 kept rows (Llama-
    3.1-8B shape, 128K at a 10% budget), G = 4: sampled segments against the
    oracle; every output finite and inside the convex hull bound."""
    cfg = ks.DECODE_128K
    x = ks.gen_decode(cfg, DEV)
    out, lse = run(qk, x)
    assert qk.kvc_stream_status() == 0
    assert torch.isfinite(out).all() and torch.isfinite(lse).all()
    vmax = x["V"].float().abs().max().item()
    assert out.abs().max().item() <= vmax * (1 + 1e-5)
    rng = np.random.default_rng(0)
    segs = sorted(rng.choice(cfg.n_seg, size=12, replace=False).tolist())
    # copy only the sampled segments back for the oracle
    sub = {"K": [], "V": [], "q": x["q"][segs], "off": [], "len": []}
    row = 0
    for s in segs:
        o, n = int(x["seg_off"][s]), int(x["seg_len"][s])
        sub["K"].append(x["K"][o:o + n])
        sub["V"].append(x["V"][o:o + n])
        sub["off"].append(row)
        sub["len"].append(n)
        row += n
    y = dict(K=torch.cat(sub["K"]), V=torch.cat(sub["V"]), q=sub["q"],
             seg_off=torch.tensor(sub["off"]), seg_len=torch.tensor(sub["len"]))
    check(y, out[segs], lse[segs])
