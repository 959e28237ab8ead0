"""CPU oracle of the 4-bit (Q4) codec for a compacted KV cache.

TEST INFRASTRUCTURE ONLY.  Nothing in the product path imports this module:
only ``tests/``, ``__graft_entry__.smoke()`` and the CPU legs of ``bench.py``
may call it.  It shares no code with the CUDA library.

Source: "Agent Memory Below the Prompt: Persistent Q4 KV Cache for
Multi-Agent LLM Inference on Edge Devices" (onedev.kr summary), sections
"방법론 및 시스템 설계" (each agent's KV cache is stored 4-bit quantized and
loaded straight back into attention instead of a re-prefill) and "실험 결과"
(about 4x more contexts than FP16 in the same memory).  The page names the
MLX framework but prints no format; the reading here, an affine group
quantiser, is:

* a row is one key or value vector of d = 128 bf16 values, split into
  G = 2 groups of 64 consecutive elements;
* per group, lo = min (a -0 minimum taken as +0) and hi = max (exact in
  fp32); the stored offset is lo
  rounded DOWN to bf16 and the stored step is (hi - lo_b) / 15 in fp32
  rounded UP to bf16, so the 16-level grid lo_b + c * s_b (c = 0..15) spans
  the whole group; a constant group stores s_b = 0;
* code c = clamp(rint((x - lo_b) / s_b), 0, 15) with IEEE fp32 subtraction
  and division and round-half-to-even (c = 0 when s_b = 0);
* two codes per byte, the even element in the low nibble: 64 bytes of codes
  plus 2 x (s_b, lo_b) bf16 = 72 bytes per row (256 bytes in bf16);
* decoding: x^ = bf16_rn(fp32(c * s_b) + lo_b), two separately rounded fp32
  operations (no fused multiply-add).

Every decision is taken in fp32, exactly as the device does it, so codes,
steps and offsets are bit-exact between the two sides.
"""
from __future__ import annotations

import numpy as np

D = 128
GROUP = 64


def _bits_f32(x):
    return np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)


def bf16_round_down(x: np.ndarray) -> np.ndarray:
    """Largest bf16 value <= x, as float32 (x finite)."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    b = _bits_f32(x)
    trunc = (b & np.uint32(0xFFFF0000)).view(np.float32)       # round toward zero
    exact = (b & np.uint32(0xFFFF)) == 0
    # negative values that were not exact need one more step away from zero
    step = ((b & np.uint32(0xFFFF0000)) + np.uint32(0x10000)).view(np.float32)
    return np.where(exact | (x >= 0), trunc, step).astype(np.float32)


def bf16_round_up(x: np.ndarray) -> np.ndarray:
    """Smallest bf16 value >= x, as float32 (x finite)."""
    return (-bf16_round_down(-np.asarray(x, dtype=np.float32))).astype(np.float32)


def bf16_round_nearest(x: np.ndarray) -> np.ndarray:
    """Round-to-nearest-even to bf16, as float32 (finite x)."""
    b = _bits_f32(x).astype(np.uint64)
    r = (b + 0x7FFF + ((b >> 16) & 1)) & 0xFFFF0000
    return r.astype(np.uint32).view(np.float32)


def encode(X: np.ndarray):
    """X float32 [rows][128] (bf16 values) -> (codes uint8 [rows][128],
    step float32 [rows][2], offset float32 [rows][2]); unpacked codes."""
    X = np.ascontiguousarray(X, dtype=np.float32)
    rows = X.shape[0]
    Xg = X.reshape(rows, D // GROUP, GROUP)
    lo = (Xg.min(axis=2) + np.float32(0.0)).astype(np.float32)   # -0 -> +0: a signed zero minimum is not unique
    hi = Xg.max(axis=2)
    lo_b = bf16_round_down(lo)
    s = ((hi - lo_b).astype(np.float32) / np.float32(15.0)).astype(np.float32)
    s_b = np.where(hi == lo, np.float32(0.0), bf16_round_up(s)).astype(np.float32)
    t = np.zeros_like(Xg)
    nz = s_b > 0
    diff = (Xg - lo_b[:, :, None]).astype(np.float32)
    with np.errstate(divide="ignore", invalid="ignore"):
        q = (diff / np.where(nz, s_b, np.float32(1.0))[:, :, None]).astype(np.float32)
    t = np.where(nz[:, :, None], q, np.float32(0.0))
    c = np.clip(np.rint(t), 0, 15).astype(np.uint8)
    return c.reshape(rows, D), s_b, lo_b


def pack_codes(c: np.ndarray) -> np.ndarray:
    """uint8 codes [rows][128] -> packed bytes [rows][64] (even element in the
    low nibble)."""
    c = np.asarray(c, dtype=np.uint8)
    return (c[:, 0::2] | (c[:, 1::2] << 4)).astype(np.uint8)


def unpack_codes(p: np.ndarray) -> np.ndarray:
    p = np.asarray(p, dtype=np.uint8)
    out = np.empty((p.shape[0], D), dtype=np.uint8)
    out[:, 0::2] = p & 0xF
    out[:, 1::2] = p >> 4
    return out


def decode(c: np.ndarray, s_b: np.ndarray, lo_b: np.ndarray) -> np.ndarray:
    """Unpacked codes + per-group step/offset -> float32 values of the decoded
    bf16 rows."""
    rows = c.shape[0]
    cg = c.reshape(rows, D // GROUP, GROUP).astype(np.float32)
    prod = (cg * s_b[:, :, None]).astype(np.float32)
    v = (prod + lo_b[:, :, None]).astype(np.float32)
    return bf16_round_nearest(v).reshape(rows, D)
