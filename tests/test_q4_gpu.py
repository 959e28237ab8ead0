"""GPU parity of the Q4 codec (persistent Q4 KV cache page, "방법론 및 시스템
설계") through the C ABI: codes, steps and offsets bit-exact against the fp32
oracle; decoded rows bit-exact against the oracle's decoding of the same
codes; decoding from page-locked host memory read in place; a compacted cache
round trip feeding decode attention."""
import numpy as np
import pytest
import torch

import kv_synth as ks
from oracle import decode, q4

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


def encode_gpu(qk, X):
    rows = X.shape[0]
    codes = torch.empty(rows, 64, dtype=torch.uint8, device=DEV)
    params = torch.empty(rows, 2, 2, dtype=torch.bfloat16, device=DEV)
    qk.kvc_q4_encode(X, codes, params)
    assert qk.kvc_stream_status() == 0
    return codes, params


def check_codec(qk, X):
    codes, params = encode_gpu(qk, X)
    Xf = X.float().cpu().numpy()
    c_r, s_r, lo_r = q4.encode(Xf)
    np.testing.assert_array_equal(codes.cpu().numpy(), q4.pack_codes(c_r))
    pf = params.float().cpu().numpy()
    np.testing.assert_array_equal(pf[:, :, 0], s_r)
    np.testing.assert_array_equal(pf[:, :, 1], lo_r)
    np.testing.assert_array_equal(np.signbit(pf), np.signbit(np.stack([s_r, lo_r], -1)))
    Y = torch.empty_like(X)
    qk.kvc_q4_decode(codes, params, Y)
    assert qk.kvc_stream_status() == 0
    np.testing.assert_array_equal(Y.float().cpu().numpy(), q4.decode(c_r, s_r, lo_r))
    return codes, params, Y


@pytest.mark.parametrize("rows", [1, 2, 3, 17, 1000, 65537, 200003])
def test_random_rows(qk, rows):
    cfg = ks.DecodeConfig("q4", seqs=1, Hkv=1, G=1, kept=rows, seed=rows)
    x = ks.gen_decode(cfg, DEV)
    check_codec(qk, x["K"])
    check_codec(qk, x["V"])


def test_special_rows(qk):
    rows = []
    rows.append(np.full(128, 3.0))                                   # constant
    rows.append(np.tile(np.arange(16.0), 8))                         # exact integers
    r = np.zeros(128); r[::2] = -0.0; r[1::2] = 0.0; rows.append(r)  # signed zeros
    r = np.linspace(-1e30, 1e30, 128); rows.append(r)                # large range
    r = np.linspace(-1e-38, 1e-38, 128); rows.append(r)              # subnormal bf16 values
    r = np.full(128, -2.5); r[7] = -2.4921875; rows.append(r)        # one step above a constant
    X = torch.tensor(np.stack(rows), dtype=torch.float32).to(torch.bfloat16).to(DEV)
    check_codec(qk, X)


def test_decode_reads_pinned_host_in_place(qk):
    cfg = ks.DecodeConfig("q4h", seqs=1, Hkv=1, G=1, kept=4099, seed=3)
    X = ks.gen_decode(cfg, DEV)["K"]
    codes, params = encode_gpu(qk, X)
    hc, hp = codes.cpu().pin_memory(), params.cpu().pin_memory()
    Y1, Y2 = torch.empty_like(X), torch.empty_like(X)
    qk.kvc_q4_decode(codes, params, Y1)
    qk.kvc_q4_decode(hc, hp, Y2)
    assert qk.kvc_stream_status() == 0
    assert torch.equal(Y1, Y2)


def test_round_trip_feeds_decode_attention(qk):
    """A Q4 round trip of a compacted cache changes decode-attention outputs
    only by the codec's error (reported, loosely bounded)."""
    cfg = ks.DecodeConfig("q4att", seqs=2, Hkv=4, G=4, kept=3000, seed=4)
    x = ks.gen_decode(cfg, DEV)
    K2, V2 = torch.empty_like(x["K"]), torch.empty_like(x["V"])
    for src, dst in ((x["K"], K2), (x["V"], V2)):
        c, p = encode_gpu(qk, src)
        qk.kvc_q4_decode(c, p, dst)
    n_seg, G = cfg.n_seg, cfg.G
    ws = torch.empty(qk.kvc_decode_workspace_size(n_seg, G, cfg.kept), dtype=torch.uint8, device=DEV)
    outs = []
    for K, V in ((x["K"], x["V"]), (K2, V2)):
        o = torch.empty(n_seg, G, 128, dtype=torch.float32, device=DEV)
        qk.kvc_decode_attention(K, V, x["seg_off"], x["seg_len"], cfg.kept, x["q"], o, ws=ws)
        outs.append(o)
    assert qk.kvc_stream_status() == 0
    rel = ((outs[0] - outs[1]).norm() / outs[0].norm()).item()
    assert rel < 0.25, rel


def test_decode_refuses_or_reads_pageable_memory(qk):
    """Ordinary (pageable) host memory is either refused on the host before any
    launch, or -- when the device reads pageable memory through the host's
    page tables -- decoded correctly; it never reaches a kernel otherwise."""
    import ctypes
    cfg = ks.DecodeConfig("q4p", seqs=1, Hkv=1, G=1, kept=777, seed=5)
    X = ks.gen_decode(cfg, DEV)["K"]
    codes, params = encode_gpu(qk, X)
    hc, hp = codes.cpu(), params.cpu()            # pageable copies
    assert not hc.is_pinned()
    Y = torch.zeros_like(X)
    rc = qk.lib().kvc_q4_decode(X.shape[0], ctypes.c_void_p(hc.data_ptr()), ctypes.c_void_p(hp.data_ptr()),
                                ctypes.c_void_p(Y.data_ptr()), ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert rc in (0, 1)
    torch.cuda.synchronize()
    assert qk.kvc_stream_status() == 0
    if rc == 0:
        Y2 = torch.empty_like(X)
        qk.kvc_q4_decode(codes, params, Y2)
        assert torch.equal(Y, Y2)
    else:
        assert torch.count_nonzero(Y) == 0


def test_compress_refuses_host_keys(qk):
    import ctypes
    x = ks.gen_kv2(ks.scaled(ks.TINY, N=512, m=128))
    K = torch.from_numpy(x.K.view(np.int16)).view(torch.bfloat16)          # host, pageable
    Q = torch.from_numpy(x.Q.view(np.int16)).view(torch.bfloat16).to(DEV)
    shape = qk.shape_of(1, 1, 4, 512)
    kept = torch.empty(64, dtype=torch.int32, device=DEV)
    Kc = torch.empty(64 * 128, dtype=torch.bfloat16, device=DEV)
    ws = torch.empty(qk.kvc_workspace_size(shape, 4, 128, 0.1), dtype=torch.uint8, device=DEV)
    k = (ctypes.c_int32 * 1)(25)
    rc = qk.lib().kvc_compress(shape, ctypes.c_void_p(K.data_ptr()), None, ctypes.c_void_p(Q.data_ptr()), 4, 128,
                               0.1, 1, k, ctypes.c_void_p(kept.data_ptr()), ctypes.c_void_p(Kc.data_ptr()), None,
                               None, None, None, ctypes.c_void_p(ws.data_ptr()), ws.numel(),
                               ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert rc == 1
