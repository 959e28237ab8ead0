"""The allocation-free KeyDiff entry point, kvc_proxy_score_noalloc.

It exists for callers that cannot allocate device memory when they need
the proxy -- a runtime that has handed all free HBM to its own pool, or a
latency-critical path where cudaMalloc (which can synchronise the device)
is not allowed.  It must give the same p as kvc_proxy_score, which takes its
scratch from a caller-allocated workspace, on consecutive calls that reuse
the library's built-in scratch, also for a shape exactly at that scratch's
size, and must refuse larger shapes before launching anything.

This file is named so that pytest collects it last; it needs no state from
the other test files.
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


def _dev_bf16(bits):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).to(DEV)


def test_noalloc_matches_workspace_entry_point_twice(qk):
    # two different caches back to back: the second call reuses the scratch
    cfgs = [ks.scaled(ks.LLAMA_16K, L=2, N=16384, needles_per_layer=8),
            ks.scaled(ks.TINY, L=3, Hkv=2, Hq=6, N=3001, seed=7, needles_per_layer=4)]
    for cfg in cfgs:
        x = ks.gen_kv2(cfg)
        shape = (cfg.L, cfg.Hkv, cfg.Hq, 128, cfg.N)
        K = _dev_bf16(x.K)
        p_ref = torch.empty(cfg.N, dtype=torch.float32, device=DEV)
        ws = torch.empty(qk.kvc_workspace_size(shape, cfg.sinks, cfg.m, cfg.rho), dtype=torch.uint8, device=DEV)
        qk.kvc_proxy_score(shape, K, p_ref, ws=ws)
        p = torch.full((cfg.N,), float("nan"), dtype=torch.float32, device=DEV)
        qk.kvc_proxy_score_noalloc(shape, K, p)
        assert qk.kvc_stream_status() == 0
        compare.assert_scores(p.cpu().numpy(), p_ref.cpu().numpy(), floor=compare.PROXY_FLOOR,
                              what="noalloc proxy p")


LIMIT = 16 << 20   # bytes of the library's built-in scratch


def _full_size_inputs(shape, seed):
    L, H, _, d, N = shape
    g = torch.Generator(device=DEV).manual_seed(seed)
    K = torch.randn(L * H * N * d, generator=g, device=DEV).to(torch.bfloat16)
    p = torch.full((N,), float("nan"), dtype=torch.float32, device=DEV)
    return K, p


def test_noalloc_at_its_limit_matches_workspace_entry_point(qk):
    # 32 x 8 heads of 16384 rows: L*Hkv*N = 4194304, exactly at the limit
    shape = (32, 8, 32, 128, 16384)
    need = qk.kvc_proxy_workspace_size(shape, True)
    assert need == LIMIT
    K, p = _full_size_inputs(shape, 3)
    ws = torch.empty(need, dtype=torch.uint8, device=DEV)
    p_ref = torch.empty_like(p)
    qk.kvc_proxy_score(shape, K, p_ref, ws=ws)
    qk.kvc_proxy_score_noalloc(shape, K, p)
    assert qk.kvc_stream_status() == 0
    compare.assert_scores(p.cpu().numpy(), p_ref.cpu().numpy(), floor=compare.PROXY_FLOOR, what="noalloc p at limit")


def test_noalloc_rejects_shapes_beyond_its_scratch(qk):
    shape = (32, 8, 32, 128, 16385)      # one row past the 16 MiB scratch
    assert qk.kvc_proxy_workspace_size(shape, True) > LIMIT
    # inputs at full size, so that nothing could read past them even if the
    # host-side check were missing
    K, p = _full_size_inputs(shape, 4)
    with pytest.raises(qk.KVCError) as e:
        qk.kvc_proxy_score_noalloc(shape, K, p)
    assert e.value.code == 5  # KVC_ERR_WORKSPACE, raised on the host before any launch
    assert torch.isnan(p).all()          # nothing was written
