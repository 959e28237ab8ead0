"""Python binding of libkvc.so -- attention-score KV-cache compression on
GB300 (KV² selective reconstruction and EpiCache block prefill).

Every function here has the name of the C entry point it calls and only
marshals arguments: tensors become device pointers, the current torch CUDA
stream becomes the library stream, and a non-OK status raises KVCError.  All
compute runs in the library's CUDA kernels; nothing falls back to the CPU.
If the library has not been built, the first call raises.
"""
from __future__ import annotations

import ctypes
import os
from typing import Sequence

import torch

from . import _build

__all__ = [
    "KVCError", "kvc_shape", "kvc_block_state", "lib", "shape_of",
    "kvc_status_string", "kvc_device_check", "kvc_stream_status", "kvc_set_wait_limit_ns",
    "kvc_debug_expire_wait", "kvc_chunk_plan", "kvc_budget_count", "kvc_workspace_size",
    "kvc_proxy_score", "kvc_proxy_workspace_size", "kvc_select_queries", "kvc_recon_score", "kvc_recon_gather", "kvc_recon_rows",
    "kvc_recon_cols", "kvc_refine_proxy", "kvc_evict_topk",
    "kvc_compact", "kvc_evict_compact", "kvc_compress", "kvc_proxy_partial", "kvc_refine_partial",
    "kvc_proxy_from_sums", "kvc_score_max", "kvc_pin_sinks", "kvc_layer_budgets", "kvc_block_state_init",
    "kvc_block_workspace_size", "kvc_block_prefill_step", "EXPORTED",
]

KVC_MAX_LAYERS = 128
c_i32, c_i64, c_sz, c_vp, c_dbl = ctypes.c_int32, ctypes.c_int64, ctypes.c_size_t, ctypes.c_void_p, ctypes.c_double


class kvc_shape(ctypes.Structure):
    _fields_ = [("L", c_i32), ("Hkv", c_i32), ("Hq", c_i32), ("d", c_i32), ("N", c_i32)]


class kvc_block_state(ctypes.Structure):
    _fields_ = [("L", c_i32), ("Hkv", c_i32), ("Hq", c_i32), ("d", c_i32), ("capacity", c_i32), ("sinks", c_i32),
                ("K", c_vp * 2), ("V", c_vp * 2), ("pos", c_vp * 2),
                ("cur", c_i32 * KVC_MAX_LAYERS), ("len", c_i32 * KVC_MAX_LAYERS),
                ("budget", c_i32 * KVC_MAX_LAYERS), ("consumed", c_i64)]


class kvc_kernel_time(ctypes.Structure):
    _fields_ = [("name", ctypes.c_char * 32), ("launches", c_i32), ("total_ms", c_dbl)]


class KVCError(RuntimeError):
    def __init__(self, func: str, code: int):
        self.code = code
        super().__init__(f"{func}: {_status_text(code)}")


# name -> (restype, argtypes)
_SIGS = {
    "kvc_status_string": (ctypes.c_char_p, [c_i32]),
    "kvc_device_check": (c_i32, []),
    "kvc_stream_status": (c_i32, [c_vp]),
    "kvc_set_wait_limit_ns": (c_i32, [ctypes.c_uint64]),
    "kvc_debug_expire_wait": (c_i32, [ctypes.c_uint64, c_vp]),
    "kvc_chunk_plan": (c_i32, [c_i32, c_i32, c_i32, c_dbl, ctypes.POINTER(c_i32), ctypes.POINTER(c_i32)]),
    "kvc_budget_count": (c_i32, [c_dbl, c_i32, c_i32, ctypes.POINTER(c_i32)]),
    "kvc_workspace_size": (c_sz, [kvc_shape, c_i32, c_i32, c_dbl]),
    "kvc_proxy_score": (c_i32, [kvc_shape, c_vp, c_vp, c_vp, c_vp, c_sz, c_vp]),
    "kvc_proxy_workspace_size": (c_sz, [kvc_shape, c_i32]),
    "kvc_select_queries": (c_i32, [c_i32, c_i32, c_i32, c_dbl, c_vp, c_vp, c_vp]),
    "kvc_recon_score": (c_i32, [kvc_shape, c_vp, c_vp, c_vp, c_i32, c_i32, c_dbl, c_vp, c_vp, c_vp, c_vp, c_sz,
                                c_vp]),
    "kvc_recon_gather": (c_i32, [kvc_shape, c_vp, c_vp, c_vp, c_i32, c_i32, c_dbl, c_vp, c_vp, c_sz, c_vp]),
    "kvc_recon_rows": (c_i32, [kvc_shape, c_vp, c_i32, c_i32, c_dbl, c_vp, c_vp, c_vp, c_sz, c_vp]),
    "kvc_recon_cols": (c_i32, [kvc_shape, c_vp, c_i32, c_i32, c_dbl, c_vp, c_vp, c_sz, c_vp]),
    "kvc_refine_proxy": (c_i32, [kvc_shape, c_vp, c_i32, c_vp, c_vp]),
    "kvc_evict_topk": (c_i32, [kvc_shape, c_vp, c_i32, ctypes.POINTER(c_i32), c_vp, c_vp, c_sz, c_vp]),
    "kvc_compact": (c_i32, [kvc_shape, c_vp, c_vp, c_vp, ctypes.POINTER(c_i32), c_vp, c_vp, c_vp]),
    "kvc_evict_compact": (c_i32, [kvc_shape, c_vp, c_i32, ctypes.POINTER(c_i32), c_vp, c_vp, c_vp, c_vp, c_vp, c_vp,
                                  c_sz, c_vp]),
    "kvc_compress": (c_i32, [kvc_shape, c_vp, c_vp, c_vp, c_i32, c_i32, c_dbl, c_i32, ctypes.POINTER(c_i32), c_vp,
                             c_vp, c_vp, c_vp, c_vp, c_vp, c_vp, c_sz, c_vp]),
    "kvc_layer_budgets": (c_i32, [ctypes.POINTER(ctypes.c_float), c_i32, c_dbl, c_i64, c_i32,
                                  ctypes.POINTER(c_i32)]),
    "kvc_block_state_init": (c_i32, [ctypes.POINTER(kvc_block_state), c_i32, c_i32, c_i32, c_i32, c_i32, c_i32,
                                     ctypes.POINTER(c_i32), c_vp, c_vp, c_vp, c_vp, c_vp, c_vp]),
    "kvc_block_workspace_size": (c_sz, [ctypes.POINTER(kvc_block_state), c_i32, c_i32]),
    "kvc_block_prefill_step": (c_i32, [ctypes.POINTER(kvc_block_state), c_vp, c_vp, c_i32, c_vp, c_vp, c_i32, c_vp,
                                       c_sz, c_vp]),
    "kvc_proxy_score_noalloc": (c_i32, [kvc_shape, c_vp, c_vp, c_vp]),
    "kvc_proxy_partial": (c_i32, [kvc_shape, c_i32, c_vp, c_vp, c_vp, c_vp, c_sz, c_vp]),
    "kvc_refine_partial": (c_i32, [kvc_shape, c_vp, c_i32, c_vp, c_vp]),
    "kvc_proxy_from_sums": (c_i32, [c_i32, c_i32, c_vp, c_vp, c_vp]),
    "kvc_score_max": (c_i32, [kvc_shape, c_vp, c_i32, c_vp, c_vp, c_sz, c_vp]),
    "kvc_pin_sinks": (c_i32, [kvc_shape, c_vp, c_i32, c_vp, c_vp]),
    "kvc_proxy_score_kind": (c_i32, [kvc_shape, c_i32, c_vp, c_vp, c_vp, c_vp, c_sz, c_vp]),
    "kvc_compress_ex": (c_i32, [kvc_shape, c_i32, c_vp, c_vp, c_vp, c_i32, c_i32, c_dbl, c_i32,
                                ctypes.POINTER(c_i32), c_vp, c_vp, c_vp, c_vp, c_vp, c_vp, c_vp, c_sz, c_vp, c_vp]),
    "kvc_decode_workspace_size": (c_sz, [c_i32, c_i32, c_i32]),
    "kvc_decode_attention": (c_i32, [c_i32, c_i32, c_vp, c_vp, c_i64, c_vp, c_vp, c_i32, c_vp, ctypes.c_float, c_vp,
                                     c_vp, c_vp, c_sz, c_vp]),
    "kvc_compact_segments": (c_i32, [c_i32, c_i32, ctypes.POINTER(c_i32), ctypes.POINTER(c_i64),
                                     ctypes.POINTER(c_i32)]),
    "kvc_episode_match": (c_i32, [c_i32, c_i32, c_i32, c_vp, c_vp, ctypes.c_float, c_vp, c_vp, c_vp]),
    "kvc_episode_rows": (c_i64, [ctypes.POINTER(kvc_block_state)]),
    "kvc_episode_pack": (c_i32, [ctypes.POINTER(kvc_block_state), c_vp, c_vp, c_vp, c_vp]),
    "kvc_episode_swap": (c_i32, [c_vp, c_vp, c_sz, c_vp, c_vp, c_sz, c_vp, c_vp]),
    "kvc_q4_encode": (c_i32, [c_i64, c_vp, c_vp, c_vp, c_vp]),
    "kvc_q4_decode": (c_i32, [c_i64, c_vp, c_vp, c_vp, c_vp]),
    "kvc_profile_begin": (c_i32, []),
    "kvc_profile_end": (c_i32, [ctypes.POINTER(kvc_kernel_time), c_i32, ctypes.POINTER(c_i32)]),
}
EXPORTED = tuple(_SIGS)

_lib = None


def lib() -> ctypes.CDLL:
    """The loaded libkvc.so (raises if it has not been built)."""
    global _lib
    if _lib is None:
        path = _build.LIB
        if not os.path.exists(path):
            raise RuntimeError(f"{path} is missing: build it with __graft_entry__.build() "
                               "(the CUDA library is required; there is no fallback)")
        L = ctypes.CDLL(path)
        for name, (res, args) in _SIGS.items():
            f = getattr(L, name)
            f.restype, f.argtypes = res, args
        _lib = L
    return _lib


def _status_text(code: int) -> str:
    try:
        return lib().kvc_status_string(int(code)).decode()
    except Exception:  # pragma: no cover
        return f"status {code}"


def _check(name: str, code: int) -> None:
    if code != 0:
        raise KVCError(name, code)


def shape_of(L: int, Hkv: int, Hq: int, N: int, d: int = 128) -> kvc_shape:
    return kvc_shape(L, Hkv, Hq, d, N)


def _shape(s) -> kvc_shape:
    if isinstance(s, kvc_shape):
        return s
    L, Hkv, Hq, d, N = s
    return kvc_shape(L, Hkv, Hq, d, N)


def _numel_ok(t, numel, name):
    if numel is not None and t.numel() < numel:
        raise ValueError(f"{name} holds {t.numel()} elements, the call reads or writes {numel}")


def _dev(t, dtype=None, name="tensor", numel=None):
    """Device pointer of a contiguous CUDA tensor (None -> NULL) holding at
    least `numel` elements when given."""
    if t is None:
        return None
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise TypeError(f"{name} must be a CUDA tensor")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name} must have dtype {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    _numel_ok(t, numel, name)
    return c_vp(t.data_ptr())


def _dev_or_pinned(t, dtype=None, name="tensor", numel=None):
    """Like _dev, but also accepts a pinned (page-locked) host tensor, which
    is mapped into the device address space: kernels then read only the rows
    they need across the host link instead of a full copy."""
    if t is not None and isinstance(t, torch.Tensor) and not t.is_cuda:
        if not t.is_pinned():
            raise TypeError(f"{name} must be a CUDA tensor or a pinned host tensor")
        if dtype is not None and t.dtype != dtype:
            raise TypeError(f"{name} must have dtype {dtype}, got {t.dtype}")
        if not t.is_contiguous():
            raise ValueError(f"{name} must be contiguous")
        _numel_ok(t, numel, name)
        return c_vp(t.data_ptr())
    return _dev(t, dtype, name, numel)


def _n(shape):
    """Element counts the KV² calls touch for a shape: keys/values, query
    pool, per-head scores, p."""
    L, Hkv, Hq, d, N = (shape.L, shape.Hkv, shape.Hq, shape.d, shape.N) if isinstance(shape, kvc_shape) else shape
    return {"K": L * Hkv * N * d, "Q": L * Hq * N * d, "S": L * Hkv * N, "N": N, "L": L, "Hkv": Hkv, "Hq": Hq,
            "d": d}


def _n_queries(N, sinks, m, rho):
    """Reconstruction queries of the chunk plan (None for a plan the library
    refuses; the call then reports it)."""
    n = c_i32(0)
    if lib().kvc_chunk_plan(N, sinks, m, float(rho), ctypes.byref(n), None) != 0:
        return None
    off = (c_i32 * (n.value + 1))()
    lib().kvc_chunk_plan(N, sinks, m, float(rho), ctypes.byref(n), off)
    return off[n.value]


def _ws(ws):
    if ws is None:
        return None, 0
    if not isinstance(ws, torch.Tensor) or not ws.is_cuda:
        raise TypeError("workspace must be a CUDA tensor")
    return c_vp(ws.data_ptr()), ws.numel() * ws.element_size()


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return c_vp(stream.cuda_stream)


def _i32_array(vals: Sequence[int]):
    return (c_i32 * len(vals))(*[int(v) for v in vals])


# ---------------------------------------------------------------- status
def kvc_status_string(code: int) -> str:
    return lib().kvc_status_string(int(code)).decode()


def kvc_device_check() -> None:
    _check("kvc_device_check", lib().kvc_device_check())


def kvc_stream_status(stream=None) -> int:
    """Synchronise and return (and clear) the device status code (0 = OK)."""
    return int(lib().kvc_stream_status(_stream(stream)))


def kvc_set_wait_limit_ns(limit_ns: int) -> None:
    _check("kvc_set_wait_limit_ns", lib().kvc_set_wait_limit_ns(int(limit_ns)))


def kvc_debug_expire_wait(limit_ns: int, stream=None) -> None:
    _check("kvc_debug_expire_wait", lib().kvc_debug_expire_wait(int(limit_ns), _stream(stream)))


def kvc_profile_begin() -> None:
    _check("kvc_profile_begin", lib().kvc_profile_begin())


def kvc_profile_end() -> dict:
    """Synchronise and return {kernel name: (launches, total ms)}."""
    arr = (kvc_kernel_time * 64)()
    n = c_i32(0)
    _check("kvc_profile_end", lib().kvc_profile_end(arr, 64, ctypes.byref(n)))
    return {arr[i].name.decode(): (int(arr[i].launches), float(arr[i].total_ms)) for i in range(min(n.value, 64))}


# ---------------------------------------------------------------- plans (host only)
def kvc_chunk_plan(N: int, sinks: int, m: int, rho: float) -> list[int]:
    """Prefix offsets of the per-chunk query counts (length M + 1)."""
    n = c_i32(0)
    _check("kvc_chunk_plan", lib().kvc_chunk_plan(N, sinks, m, float(rho), ctypes.byref(n), None))
    off = (c_i32 * (n.value + 1))()
    _check("kvc_chunk_plan", lib().kvc_chunk_plan(N, sinks, m, float(rho), ctypes.byref(n), off))
    return list(off)


def kvc_budget_count(b: float, N: int, sinks: int) -> int:
    k = c_i32(0)
    _check("kvc_budget_count", lib().kvc_budget_count(float(b), N, sinks, ctypes.byref(k)))
    return k.value


def kvc_workspace_size(shape, sinks: int, m: int, rho: float) -> int:
    return int(lib().kvc_workspace_size(_shape(shape), sinks, m, float(rho)))


def kvc_layer_budgets(sens: Sequence[float], alpha: float, mean_budget: int, sinks: int) -> list[int]:
    L = len(sens)
    s = (ctypes.c_float * L)(*[float(x) for x in sens])
    out = (c_i32 * L)()
    _check("kvc_layer_budgets", lib().kvc_layer_budgets(s, L, float(alpha), int(mean_budget), sinks, out))
    return list(out)


# ---------------------------------------------------------------- KV² stages
def kvc_proxy_workspace_size(shape, with_scores: bool = True) -> int:
    return int(lib().kvc_proxy_workspace_size(_shape(shape), 1 if with_scores else 0))


def kvc_proxy_score(shape, K, p, s=None, ws=None, stream=None) -> None:
    w, wb = _ws(ws)
    n = _n(shape)
    _check("kvc_proxy_score", lib().kvc_proxy_score(_shape(shape), _dev(K, torch.bfloat16, "K", n["K"]),
                                                    _dev(p, torch.float32, "p", n["N"]),
                                                    _dev(s, torch.float32, "s", n["S"]), w, wb, _stream(stream)))


KVC_PROXY_KEYDIFF = 0
KVC_PROXY_KNORM = 1
_PROXY = {"keydiff": KVC_PROXY_KEYDIFF, "knorm": KVC_PROXY_KNORM}


def _proxy_kind(kind) -> int:
    return _PROXY[kind] if isinstance(kind, str) else int(kind)


def kvc_proxy_score_kind(shape, kind, K, p, s=None, ws=None, stream=None) -> None:
    """kvc_proxy_score with a proxy kind: "keydiff" (default) or "knorm"."""
    w, wb = _ws(ws)
    n = _n(shape)
    _check("kvc_proxy_score_kind", lib().kvc_proxy_score_kind(
        _shape(shape), _proxy_kind(kind), _dev(K, torch.bfloat16, "K", n["K"]), _dev(p, torch.float32, "p", n["N"]),
        _dev(s, torch.float32, "s", n["S"]), w, wb, _stream(stream)))


def kvc_compress_ex(shape, proxy, K, V, Qpool, sinks, m, rho, passes, k_per_layer, kept, Kc, Vc, p=None, sel=None,
                    score=None, ws=None, stream=None, gather_done=None) -> None:
    """kvc_compress with a selectable stage-1 proxy ("keydiff" or "knorm");
    `gather_done` (a torch.cuda.Event that has been recorded once, so that it
    exists) is recorded right after the last query gather."""
    w, wb = _ws(ws)
    ev = None
    if gather_done is not None:
        if not gather_done.cuda_event:
            raise ValueError("gather_done must be a created event (record it once first)")
        ev = c_vp(gather_done.cuda_event)
    n = _n(shape)
    nk = n["Hkv"] * sum(int(k) for k in k_per_layer)
    nq = _n_queries(n["N"], sinks, m, rho)
    _check("kvc_compress_ex", lib().kvc_compress_ex(
        _shape(shape), _proxy_kind(proxy), _dev(K, torch.bfloat16, "K", n["K"]),
        _dev_or_pinned(V, torch.bfloat16, "V", n["K"]), _dev_or_pinned(Qpool, torch.bfloat16, "Qpool", n["Q"]), sinks,
        m, float(rho), passes, _i32_array(k_per_layer), _dev(kept, torch.int32, "kept", nk),
        _dev(Kc, torch.bfloat16, "Kc", nk * n["d"]), _dev(Vc, torch.bfloat16, "Vc", nk * n["d"]),
        _dev(p, torch.float32, "p", n["N"]), _dev(sel, torch.int32, "sel", nq), _dev(score, torch.float32, "score", n["S"]),
        w, wb, _stream(stream), ev))


def kvc_proxy_score_noalloc(shape, K, p, stream=None) -> None:
    """kvc_proxy_score without a workspace: for callers that cannot allocate
    device memory at this point (their runtime owns all free HBM, or the call
    sits on a path where cudaMalloc is not allowed).  Scratch comes from a
    16 MiB array inside the library; L*Hkv*N must not exceed 4194304 (32
    layers x 8 KV heads x 16K tokens is exactly at the limit)."""
    n = _n(shape)
    _check("kvc_proxy_score_noalloc", lib().kvc_proxy_score_noalloc(
        _shape(shape), _dev(K, torch.bfloat16, "K", n["K"]), _dev(p, torch.float32, "p", n["N"]), _stream(stream)))


# ---------------------------------------------------------------- layer-sharded calls
def kvc_proxy_partial(shape, kind, K, psum, s=None, ws=None, stream=None) -> None:
    """psum[i] = sum over this shard's (layer, KV head) pairs of the proxy s_i."""
    w, wb = _ws(ws)
    n = _n(shape)
    _check("kvc_proxy_partial", lib().kvc_proxy_partial(
        _shape(shape), _proxy_kind(kind), _dev(K, torch.bfloat16, "K", n["K"]), _dev(psum, torch.float32, "psum", n["N"]),
        _dev(s, torch.float32, "s", n["S"]), w, wb, _stream(stream)))


def kvc_refine_partial(shape, score, sinks, psum, stream=None) -> None:
    n = _n(shape)
    _check("kvc_refine_partial", lib().kvc_refine_partial(
        _shape(shape), _dev(score, torch.float32, "score", n["S"]), sinks, _dev(psum, torch.float32, "psum", n["N"]),
        _stream(stream)))


def kvc_proxy_from_sums(N, total_heads, psum, p, stream=None) -> None:
    _check("kvc_proxy_from_sums", lib().kvc_proxy_from_sums(
        N, total_heads, _dev(psum, torch.float32, "psum", N), _dev(p, torch.float32, "p", N), _stream(stream)))


def kvc_score_max(shape, score, sinks, max_out, ws=None, stream=None) -> None:
    w, wb = _ws(ws)
    n = _n(shape)
    _check("kvc_score_max", lib().kvc_score_max(
        _shape(shape), _dev(score, torch.float32, "score", n["S"]), sinks, _dev(max_out, torch.float32, "max_out", 1),
        w, wb, _stream(stream)))


def kvc_pin_sinks(shape, score, sinks, value, stream=None) -> None:
    n = _n(shape)
    _check("kvc_pin_sinks", lib().kvc_pin_sinks(
        _shape(shape), _dev(score, torch.float32, "score", n["S"]), sinks, _dev(value, torch.float32, "value", 1),
        _stream(stream)))


def kvc_select_queries(N, sinks, m, rho, p, sel, stream=None) -> None:
    _check("kvc_select_queries", lib().kvc_select_queries(N, sinks, m, float(rho), _dev(p, torch.float32, "p", N),
                                                          _dev(sel, torch.int32, "sel", _n_queries(N, sinks, m, rho)),
                                                          _stream(stream)))


def kvc_recon_score(shape, K, Qpool, sel, sinks, m, rho, score, Kapp=None, lse=None, ws=None, stream=None) -> None:
    w, wb = _ws(ws)
    n = _n(shape)
    nq = _n_queries(n["N"], sinks, m, rho) or 0
    _check("kvc_recon_score", lib().kvc_recon_score(
        _shape(shape), _dev(K, torch.bfloat16, "K", n["K"]), _dev_or_pinned(Qpool, torch.bfloat16, "Qpool", n["Q"]),
        _dev(sel, torch.int32, "sel", nq), sinks, m, float(rho),
        _dev(Kapp, torch.bfloat16, "Kapp", n["L"] * n["Hkv"] * nq * n["d"]), _dev(score, torch.float32, "score", n["S"]),
        _dev(lse, torch.float32, "lse", n["L"] * n["Hq"] * nq), w, wb, _stream(stream)))


def kvc_recon_gather(shape, K, Qpool, sel, sinks, m, rho, Kapp=None, ws=None, stream=None) -> None:
    """Phase 1 of kvc_recon_score: the query rows (and appended keys) into the workspace."""
    w, wb = _ws(ws)
    _check("kvc_recon_gather", lib().kvc_recon_gather(
        _shape(shape), _dev(K, torch.bfloat16, "K"), _dev_or_pinned(Qpool, torch.bfloat16, "Qpool"),
        _dev(sel, torch.int32, "sel"), sinks, m, float(rho), _dev(Kapp, torch.bfloat16, "Kapp"), w, wb,
        _stream(stream)))


def kvc_recon_rows(shape, K, sinks, m, rho, Kapp=None, lse=None, ws=None, stream=None) -> None:
    """Phase 2 of kvc_recon_score: the row log-sum-exp pass."""
    w, wb = _ws(ws)
    _check("kvc_recon_rows", lib().kvc_recon_rows(
        _shape(shape), _dev(K, torch.bfloat16, "K"), sinks, m, float(rho), _dev(Kapp, torch.bfloat16, "Kapp"),
        _dev(lse, torch.float32, "lse"), w, wb, _stream(stream)))


def kvc_recon_cols(shape, K, sinks, m, rho, score, ws=None, stream=None) -> None:
    """Phase 3 of kvc_recon_score: the column-max pass, writing score."""
    w, wb = _ws(ws)
    _check("kvc_recon_cols", lib().kvc_recon_cols(
        _shape(shape), _dev(K, torch.bfloat16, "K"), sinks, m, float(rho), _dev(score, torch.float32, "score"),
        w, wb, _stream(stream)))


def kvc_refine_proxy(shape, score, sinks, p, stream=None) -> None:
    n = _n(shape)
    _check("kvc_refine_proxy", lib().kvc_refine_proxy(_shape(shape), _dev(score, torch.float32, "score", n["S"]),
                                                      sinks, _dev(p, torch.float32, "p", n["N"]), _stream(stream)))


def kvc_evict_topk(shape, score, sinks, k_per_layer, kept, ws=None, stream=None) -> None:
    w, wb = _ws(ws)
    n = _n(shape)
    nk = n["Hkv"] * sum(int(k) for k in k_per_layer)
    _check("kvc_evict_topk", lib().kvc_evict_topk(_shape(shape), _dev(score, torch.float32, "score", n["S"]), sinks,
                                                  _i32_array(k_per_layer), _dev(kept, torch.int32, "kept", nk), w, wb,
                                                  _stream(stream)))


def kvc_compact(shape, K, V, kept, k_per_layer, Kc, Vc, stream=None) -> None:
    n = _n(shape)
    nk = n["Hkv"] * sum(int(k) for k in k_per_layer)
    _check("kvc_compact", lib().kvc_compact(_shape(shape), _dev_or_pinned(K, torch.bfloat16, "K", n["K"]),
                                            _dev_or_pinned(V, torch.bfloat16, "V", n["K"]),
                                            _dev(kept, torch.int32, "kept", nk), _i32_array(k_per_layer),
                                            _dev(Kc, torch.bfloat16, "Kc", nk * n["d"]),
                                            _dev(Vc, torch.bfloat16, "Vc", nk * n["d"]), _stream(stream)))


def kvc_evict_compact(shape, score, sinks, k_per_layer, kept, K, V, Kc, Vc, ws=None, stream=None) -> None:
    """kvc_evict_topk and kvc_compact in one launch."""
    w, wb = _ws(ws)
    n = _n(shape)
    nk = n["Hkv"] * sum(int(k) for k in k_per_layer)
    _check("kvc_evict_compact", lib().kvc_evict_compact(
        _shape(shape), _dev(score, torch.float32, "score", n["S"]), sinks, _i32_array(k_per_layer),
        _dev(kept, torch.int32, "kept", nk), _dev_or_pinned(K, torch.bfloat16, "K", n["K"]),
        _dev_or_pinned(V, torch.bfloat16, "V", n["K"]), _dev(Kc, torch.bfloat16, "Kc", nk * n["d"]),
        _dev(Vc, torch.bfloat16, "Vc", nk * n["d"]), w, wb, _stream(stream)))


def kvc_compress(shape, K, V, Qpool, sinks, m, rho, passes, k_per_layer, kept, Kc, Vc, p=None, sel=None,
                 score=None, ws=None, stream=None) -> None:
    w, wb = _ws(ws)
    n = _n(shape)
    nk = n["Hkv"] * sum(int(k) for k in k_per_layer)
    nq = _n_queries(n["N"], sinks, m, rho)
    _check("kvc_compress", lib().kvc_compress(
        _shape(shape), _dev(K, torch.bfloat16, "K", n["K"]), _dev_or_pinned(V, torch.bfloat16, "V", n["K"]),
        _dev_or_pinned(Qpool, torch.bfloat16, "Qpool", n["Q"]), sinks, m, float(rho), passes, _i32_array(k_per_layer),
        _dev(kept, torch.int32, "kept", nk), _dev(Kc, torch.bfloat16, "Kc", nk * n["d"]),
        _dev(Vc, torch.bfloat16, "Vc", nk * n["d"]), _dev(p, torch.float32, "p", n["N"]),
        _dev(sel, torch.int32, "sel", nq), _dev(score, torch.float32, "score", n["S"]), w, wb, _stream(stream)))


# ---------------------------------------------------------------- decode attention
def kvc_decode_workspace_size(n_seg: int, G: int, max_len: int) -> int:
    return int(lib().kvc_decode_workspace_size(n_seg, G, max_len))


def kvc_decode_attention(Kc, Vc, seg_off, seg_len, max_len, q, out, lse=None, scale=0.0, ws=None,
                         stream=None) -> None:
    """Decode attention of q [n_seg, G, 128] over the segments (seg_off,
    seg_len) of Kc/Vc [rows, 128]; writes out [n_seg, G, 128] (float32) and
    optionally lse [n_seg, G]."""
    if q.dim() != 3:
        raise ValueError("q must be [n_seg, G, 128]")
    n_seg, G = int(q.shape[0]), int(q.shape[1])
    if Kc.shape != Vc.shape or Kc.dim() != 2:
        raise ValueError("Kc and Vc must both be [rows, 128]")
    w, wb = _ws(ws)
    _check("kvc_decode_attention", lib().kvc_decode_attention(
        n_seg, G, _dev(Kc, torch.bfloat16, "Kc"), _dev(Vc, torch.bfloat16, "Vc"), int(Kc.shape[0]),
        _dev(seg_off, torch.int64, "seg_off"), _dev(seg_len, torch.int32, "seg_len"), int(max_len),
        _dev(q, torch.bfloat16, "q"), float(scale), _dev(out, torch.float32, "out"), _dev(lse, torch.float32, "lse"),
        w, wb, _stream(stream)))


def kvc_compact_segments(L: int, Hkv: int, k_per_layer) -> tuple[list[int], list[int]]:
    """(row offsets, lengths) of the (layer, KV head) segments of a compacted cache."""
    off = (c_i64 * (L * Hkv))()
    ln = (c_i32 * (L * Hkv))()
    _check("kvc_compact_segments", lib().kvc_compact_segments(L, Hkv, _i32_array(k_per_layer), off, ln))
    return list(off), list(ln)


# ---------------------------------------------------------------- EpiCache per turn
def kvc_episode_match(queries, centroids, episode, dist2=None, tau=0.0, stream=None) -> None:
    """Closest episode centroid of each question embedding (-1 past tau)."""
    B, De = int(queries.shape[0]), int(queries.shape[1])
    E = int(centroids.shape[0])
    _check("kvc_episode_match", lib().kvc_episode_match(
        B, E, De, _dev(queries, torch.float32, "queries"), _dev(centroids, torch.float32, "centroids"), float(tau),
        _dev(episode, torch.int32, "episode"), _dev(dist2, torch.float32, "dist2"), _stream(stream)))


def kvc_episode_rows(st) -> int:
    return int(lib().kvc_episode_rows(ctypes.byref(st)))


def kvc_episode_pack(st, Kp, Vp, pos=None, stream=None) -> None:
    _check("kvc_episode_pack", lib().kvc_episode_pack(
        ctypes.byref(st), _dev(Kp, torch.bfloat16, "Kp"), _dev(Vp, torch.bfloat16, "Vp"),
        _dev(pos, torch.int32, "pos"), _stream(stream)))


def kvc_episode_swap(dev_out=None, host_out=None, host_in=None, dev_in=None, out_stream=None, in_stream=None) -> None:
    """Write dev_out back into pinned host_out and bring pinned host_in into
    dev_in, on two streams (either pair may be None)."""
    def ptr(t):
        return None if t is None else c_vp(t.data_ptr())
    n_out = 0 if dev_out is None else dev_out.numel() * dev_out.element_size()
    n_in = 0 if host_in is None else host_in.numel() * host_in.element_size()
    if dev_out is not None and host_out.numel() * host_out.element_size() != n_out:
        raise ValueError("host_out must have the size of dev_out")
    if host_in is not None and dev_in.numel() * dev_in.element_size() != n_in:
        raise ValueError("dev_in must have the size of host_in")
    _check("kvc_episode_swap", lib().kvc_episode_swap(ptr(dev_out), ptr(host_out), n_out, ptr(host_in), ptr(dev_in),
                                                      n_in, _stream(out_stream), _stream(in_stream)))


# ---------------------------------------------------------------- Q4 codec
def kvc_q4_encode(X, codes, params, stream=None) -> None:
    """X bf16 [rows, 128] -> codes uint8 [rows, 64], params bf16 [rows, 2, 2]."""
    rows = int(X.shape[0])
    _check("kvc_q4_encode", lib().kvc_q4_encode(rows, _dev(X, torch.bfloat16, "X"), _dev(codes, torch.uint8, "codes"),
                                                _dev(params, torch.bfloat16, "params"), _stream(stream)))


def kvc_q4_decode(codes, params, X, stream=None) -> None:
    """codes/params (device or pinned host) -> X bf16 [rows, 128] on the device."""
    rows = int(X.shape[0])
    _check("kvc_q4_decode", lib().kvc_q4_decode(rows, _dev_or_pinned(codes, torch.uint8, "codes"),
                                                _dev_or_pinned(params, torch.bfloat16, "params"),
                                                _dev(X, torch.bfloat16, "X"), _stream(stream)))


# ---------------------------------------------------------------- EpiCache block prefill
def kvc_block_state_init(L, Hkv, Hq, capacity, sinks, budgets, K0, V0, pos0, K1=None, V1=None, pos1=None,
                         d: int = 128) -> kvc_block_state:
    """K1, V1, pos1 None: the one-slab layout (kept rows stay in place)."""
    st = kvc_block_state()
    _check("kvc_block_state_init", lib().kvc_block_state_init(
        ctypes.byref(st), L, Hkv, Hq, d, capacity, sinks, _i32_array(budgets),
        _dev(K0, torch.bfloat16, "K0"), _dev(V0, torch.bfloat16, "V0"), _dev(pos0, torch.int32, "pos0"),
        _dev(K1, torch.bfloat16, "K1"), _dev(V1, torch.bfloat16, "V1"), _dev(pos1, torch.int32, "pos1")))
    return st


def kvc_block_workspace_size(state: kvc_block_state, max_block: int, P: int) -> int:
    return int(lib().kvc_block_workspace_size(ctypes.byref(state), max_block, P))


def kvc_block_prefill_step(state: kvc_block_state, Kblk, Vblk, blk_len, Qprompt, Kprompt, P, ws=None,
                           stream=None) -> None:
    w, wb = _ws(ws)
    _check("kvc_block_prefill_step", lib().kvc_block_prefill_step(
        ctypes.byref(state), _dev(Kblk, torch.bfloat16, "Kblk"), _dev(Vblk, torch.bfloat16, "Vblk"), blk_len,
        _dev(Qprompt, torch.bfloat16, "Qprompt"), _dev(Kprompt, torch.bfloat16, "Kprompt"), P, w, wb,
        _stream(stream)))
