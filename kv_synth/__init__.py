"""Seeded synthetic KV caches and query pools.

This module only draws random inputs; it computes nothing of the compression
method itself.  Both the CUDA path (tests, bench) and the float64 oracle read
the tensors produced here, so the two sides see bit-identical bf16 inputs.

Workload shapes follow the pages' evaluation settings (Llama-3.1-8B / Qwen3-8B
GQA shapes at 4K-128K context, LLaMA3.2-3B with a 90K-token history streamed in
blocks); the datasets those pages evaluate on (RULER, LongBench, NIAH, LoCoMo,
RealTalk) are not used -- these generators stand in for their shapes only:

* keys     k = r * (z + 5 * 1_C), z ~ N(0, I_d), C = {0, 32, 64, 96},
           r = exp(N(0, 0.3^2)) drawn per (layer, kv head, position);
* values   N(0, I_d);
* queries  one per (layer, query head, position), N(0, I_d);
* needles  clusters of 4 consecutive keys in KV head g // G set to
           8 * sqrt(d) * q / |q|^2 for an anchor query q at (g, p_q), so the
           planted logit q.k / sqrt(d) is exactly 8 before bf16 rounding
           (sparse, anchor-like evidence, the regime KV^2 says it helps most).

Every draw uses numpy PCG64 with per-layer seeds (1000 * seed + layer), so a
layer can be regenerated alone, and layers can be generated in parallel.
All values are drawn in float32 and rounded to bfloat16 (round to nearest
even); they are returned as uint16 bit patterns (``*_bits``) together with the
exact float32 values.
"""
from __future__ import annotations

import math
from concurrent.futures import ThreadPoolExecutor
from dataclasses import dataclass, field
import os

import numpy as np

NEEDLE_LOGIT = 8.0
OFFSET_CHANNELS = (0, 32, 64, 96)
OFFSET_MEAN = 5.0
NORM_SIGMA = 0.3


# --------------------------------------------------------------------------
# bf16 helpers (storage format only)
# --------------------------------------------------------------------------
def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 to bfloat16 (nearest even); return uint16 bit patterns."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    u = x.view(np.uint32)
    # round to nearest even on the upper 16 bits; uint32 wrap-around only
    # affects NaN patterns, which are handled separately
    r = u + np.uint32(0x7FFF)
    r += (u >> np.uint32(16)) & np.uint32(1)
    r >>= np.uint32(16)
    out = r.astype(np.uint16)
    nan = np.isnan(x)
    if nan.any():
        out[nan] = 0x7FC0
    return out


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    """Exact float32 value of bfloat16 bit patterns."""
    return (np.ascontiguousarray(b, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def _threads() -> int:
    try:
        return max(1, len(os.sched_getaffinity(0)))
    except AttributeError:  # pragma: no cover
        return os.cpu_count() or 1


# --------------------------------------------------------------------------
# configs
# --------------------------------------------------------------------------
@dataclass(frozen=True)
class KV2Config:
    """One KV^2 compression workload (single pass unless passes > 1)."""
    name: str
    L: int
    Hkv: int
    Hq: int
    d: int
    N: int
    sinks: int
    m: int
    rho: float
    budget: float
    passes: int = 1
    needles_per_layer: int = 0
    needle_depths: bool = False
    seed: int = 0

    @property
    def G(self) -> int:
        return self.Hq // self.Hkv


@dataclass(frozen=True)
class EpiConfig:
    """EpiCache-style block prefill workload."""
    name: str
    L: int
    Hkv: int
    Hq: int
    d: int
    n_hist: int
    block: int
    episodes: int
    prompt_len: int
    mean_budget: int
    alpha: float
    sinks: int
    seed: int = 0

    @property
    def G(self) -> int:
        return self.Hq // self.Hkv


TINY = KV2Config("tiny-4k", L=1, Hkv=1, Hq=4, d=128, N=4096, sinks=4, m=1024,
                 rho=0.1, budget=0.05, needles_per_layer=8)
LLAMA_16K = KV2Config("llama3.1-8b-16k", L=32, Hkv=8, Hq=32, d=128, N=16384, sinks=4,
                      m=4096, rho=0.10, budget=0.02, needles_per_layer=256)
QWEN_32K = KV2Config("qwen3-8b-32k-3pass", L=36, Hkv=8, Hq=32, d=128, N=32768, sinks=4,
                     m=4096, rho=0.25, budget=0.05, passes=3, needles_per_layer=256)
LLAMA_128K = KV2Config("llama3.1-8b-128k", L=32, Hkv=8, Hq=32, d=128, N=131072, sinks=4,
                       m=4096, rho=0.5, budget=0.10, needles_per_layer=256, needle_depths=True)
EPI_3B = EpiConfig("epicache-llama3.2-3b-90k", L=28, Hkv=8, Hq=24, d=128, n_hist=90_000,
                   block=2048, episodes=4, prompt_len=64, mean_budget=8192, alpha=3.0, sinks=4)

KV2_CONFIGS = {c.name: c for c in (TINY, LLAMA_16K, QWEN_32K, LLAMA_128K)}


def scaled(cfg: KV2Config, **kw) -> KV2Config:
    """A copy of ``cfg`` with some fields replaced (small parity cases)."""
    d = dict(cfg.__dict__)
    d.update(kw)
    return KV2Config(**d)


# --------------------------------------------------------------------------
# generators
# --------------------------------------------------------------------------
def _layer_rng(seed: int, layer: int, salt: int = 0) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(1000 * seed + layer + salt))


def _needle_positions(rng, n_clusters, S, N, depths: bool):
    """Start positions of 4-key needle clusters, inside [S, N-4]."""
    if n_clusters == 0 or N - 4 <= S:
        return np.zeros(0, dtype=np.int64)
    lo, hi = S, N - 4
    starts = []
    used = np.zeros(N, dtype=bool)
    for c in range(n_clusters):
        for _attempt in range(64):
            if depths:
                dep = (c % 11) / 10.0
                base = lo + int(round(dep * (hi - lo)))
                p = base + int(rng.integers(-64, 65))
                p = min(max(p, lo), hi)
            else:
                p = int(rng.integers(lo, hi + 1))
            if not used[p:p + 4].any():
                break
        used[p:p + 4] = True
        starts.append(p)
    return np.asarray(starts, dtype=np.int64)


@dataclass
class LayerDraw:
    K: np.ndarray          # uint16 bits [Hkv][N][d]
    V: np.ndarray          # uint16 bits [Hkv][N][d]
    Q: np.ndarray          # uint16 bits [Hq][N][d]
    needles: list = field(default_factory=list)  # (g, p_q, p_k) triples


def gen_layer(cfg: KV2Config, layer: int, with_values: bool = True) -> LayerDraw:
    """Draw one layer of keys, values and the query pool for ``cfg``."""
    Hkv, Hq, N, d, G = cfg.Hkv, cfg.Hq, cfg.N, cfg.d, cfg.G
    rng = _layer_rng(cfg.seed, layer)
    z = rng.standard_normal((Hkv, N, d), dtype=np.float32)
    z[:, :, list(OFFSET_CHANNELS)] += np.float32(OFFSET_MEAN)
    r = np.exp(rng.standard_normal((Hkv, N, 1), dtype=np.float32) * np.float32(NORM_SIGMA))
    k = z * r
    q = rng.standard_normal((Hq, N, d), dtype=np.float32)
    needles = []
    if cfg.needles_per_layer:
        starts = _needle_positions(rng, cfg.needles_per_layer, cfg.sinks, N, cfg.needle_depths)
        for c, pk in enumerate(starts):
            g = int(rng.integers(0, Hq))
            pq = int(rng.integers(cfg.sinks, N))
            qv = bf16_bits_to_f32(f32_to_bf16_bits(q[g, pq])).astype(np.float64)
            kv = (NEEDLE_LOGIT * math.sqrt(d)) * qv / float(qv @ qv)
            k[g // G, pk:pk + 4, :] = kv.astype(np.float32)[None, :]
            needles.append((g, pq, int(pk)))
    Kb = f32_to_bf16_bits(k)
    Qb = f32_to_bf16_bits(q)
    if with_values:
        v = rng.standard_normal((Hkv, N, d), dtype=np.float32)
        Vb = f32_to_bf16_bits(v)
    else:
        Vb = np.zeros(0, dtype=np.uint16)
    return LayerDraw(K=Kb, V=Vb, Q=Qb, needles=needles)


@dataclass
class KV2Inputs:
    cfg: KV2Config
    K: np.ndarray   # uint16 [L][Hkv][N][d]
    V: np.ndarray   # uint16 [L][Hkv][N][d]
    Q: np.ndarray   # uint16 [L][Hq][N][d]
    needles: list   # per layer list of (g, p_q, p_k)


def gen_kv2(cfg: KV2Config, threads: int | None = None) -> KV2Inputs:
    """All layers of a KV^2 workload (bf16 bits), generated layer-parallel."""
    L, Hkv, Hq, N, d = cfg.L, cfg.Hkv, cfg.Hq, cfg.N, cfg.d
    K = np.empty((L, Hkv, N, d), dtype=np.uint16)
    V = np.empty((L, Hkv, N, d), dtype=np.uint16)
    Q = np.empty((L, Hq, N, d), dtype=np.uint16)
    needles = [None] * L

    def one(l):
        dr = gen_layer(cfg, l)
        K[l], V[l], Q[l] = dr.K, dr.V, dr.Q
        needles[l] = dr.needles

    nt = min(threads or _threads(), L)
    if nt <= 1:
        for l in range(L):
            one(l)
    else:
        with ThreadPoolExecutor(nt) as ex:
            list(ex.map(one, range(L)))
    return KV2Inputs(cfg, K, V, Q, needles)


# --------------------------------------------------------------------------
# EpiCache block-prefill inputs
# --------------------------------------------------------------------------
def gen_epi_history_layer(cfg: EpiConfig, layer: int):
    """History keys/values of one layer: uint16 bits [Hkv][n_hist][d] each."""
    c = KV2Config("epi-hist", L=cfg.L, Hkv=cfg.Hkv, Hq=cfg.Hq, d=cfg.d, N=cfg.n_hist,
                  sinks=cfg.sinks, m=cfg.block, rho=1.0, budget=1.0, seed=cfg.seed)
    rng = _layer_rng(c.seed, layer)
    z = rng.standard_normal((c.Hkv, c.N, c.d), dtype=np.float32)
    z[:, :, list(OFFSET_CHANNELS)] += np.float32(OFFSET_MEAN)
    r = np.exp(rng.standard_normal((c.Hkv, c.N, 1), dtype=np.float32) * np.float32(NORM_SIGMA))
    Kb = f32_to_bf16_bits(z * r)
    Vb = f32_to_bf16_bits(rng.standard_normal((c.Hkv, c.N, c.d), dtype=np.float32))
    return Kb, Vb


def gen_epi_prompt_layer(cfg: EpiConfig, episode: int, layer: int):
    """Patched-prompt queries [Hq][P][d] and keys [Hkv][P][d] (uint16 bits).

    Queries are drawn N(0, I) around a per-(layer, query head) episode
    centroid c_e ~ N(0, I); keys come from the key generator with the
    episode's seed.
    """
    rng = np.random.Generator(np.random.PCG64(10**6 + 1000 * episode + layer + 1000 * 1000 * cfg.seed))
    P, d = cfg.prompt_len, cfg.d
    cen = rng.standard_normal((cfg.Hq, 1, d), dtype=np.float32)
    q = cen + rng.standard_normal((cfg.Hq, P, d), dtype=np.float32)
    z = rng.standard_normal((cfg.Hkv, P, d), dtype=np.float32)
    z[:, :, list(OFFSET_CHANNELS)] += np.float32(OFFSET_MEAN)
    r = np.exp(rng.standard_normal((cfg.Hkv, P, 1), dtype=np.float32) * np.float32(NORM_SIGMA))
    return f32_to_bf16_bits(q), f32_to_bf16_bits(z * r)


def gen_sensitivity(cfg: EpiConfig) -> np.ndarray:
    """Seeded per-layer sensitivity vector sigma_l ~ U(0.5, 1.5) (float32)."""
    rng = np.random.Generator(np.random.PCG64(7_000_000 + cfg.seed))
    return rng.uniform(0.5, 1.5, size=cfg.L).astype(np.float32)


# --------------------------------------------------------------------------
# decode over compacted caches
# --------------------------------------------------------------------------
@dataclass(frozen=True)
class DecodeConfig:
    """Decode attention over compacted caches: `seqs` independent sequences,
    each with `kept` rows per KV head in the layer being decoded."""
    name: str
    seqs: int
    Hkv: int
    G: int
    kept: int
    needles_per_segment: int = 4
    seed: int = 7

    @property
    def n_seg(self) -> int:
        return self.seqs * self.Hkv


# Llama-3.1-8B shape, 128K context compressed to a 10% budget (k = 13107 per
# KV head), a batch of 64 sequences decoding one layer.
DECODE_128K = DecodeConfig("llama3.1-8b-128k-10pct-decode-b64", seqs=64, Hkv=8, G=4, kept=13107)
DECODE_128K_B16 = DecodeConfig("llama3.1-8b-128k-10pct-decode-b16", seqs=16, Hkv=8, G=4, kept=13107)
DECODE_TINY = DecodeConfig("decode-tiny", seqs=2, Hkv=2, G=4, kept=204)
DECODE_CONFIGS = {c.name: c for c in (DECODE_TINY, DECODE_128K_B16, DECODE_128K)}


def gen_decode(cfg: DecodeConfig, device="cpu", lens=None, gap: int = 0):
    """Seeded compacted-cache segments for decode attention, drawn with
    torch's generator on `device` (so large caches are made in place).

    Keys follow the compression workloads' recipe k = r (z + 5 * 1_C); values
    and queries are N(0, I); each segment holds `needles_per_segment` planted
    keys aligned to one of its queries (logit 8 at scale 1/sqrt(d)).  Rows of
    segment s are [off_s, off_s + len_s), with `gap` unused rows before each.
    Returns dict(K, V [rows, 128] bf16, q [n_seg, G, 128] bf16, seg_off int64,
    seg_len int32, rows)."""
    import torch

    d = 128
    n_seg = cfg.n_seg if lens is None else len(lens)
    lens = [cfg.kept] * n_seg if lens is None else [int(x) for x in lens]
    off, row = [], 0
    for n in lens:
        row += gap
        off.append(row)
        row += n
    rows = row
    g = torch.Generator(device=device)
    g.manual_seed(cfg.seed)
    K = torch.empty(rows, d, dtype=torch.bfloat16, device=device)
    V = torch.empty(rows, d, dtype=torch.bfloat16, device=device)
    bias = torch.zeros(d, device=device)
    bias[[0, 32, 64, 96]] = 5.0
    step = 1 << 20
    for r0 in range(0, rows, step):
        r1 = min(rows, r0 + step)
        z = torch.randn(r1 - r0, d, generator=g, device=device)
        r = torch.exp(0.3 * torch.randn(r1 - r0, 1, generator=g, device=device))
        K[r0:r1] = (r * (z + bias)).to(torch.bfloat16)
        V[r0:r1] = torch.randn(r1 - r0, d, generator=g, device=device).to(torch.bfloat16)
    q = torch.randn(n_seg, cfg.G, d, generator=g, device=device).to(torch.bfloat16)
    # needles: one per 1/NP of each segment (distinct rows), in segments of at least NP rows
    NP = cfg.needles_per_segment
    segs = [s for s, n in enumerate(lens) if n >= NP > 0]
    if segs:
        st = torch.tensor(segs, dtype=torch.int64, device=device)
        n_t = torch.tensor([lens[s] for s in segs], dtype=torch.float64, device=device)[:, None]
        o_t = torch.tensor([off[s] for s in segs], dtype=torch.int64, device=device)[:, None]
        u = torch.rand(len(segs), NP, generator=g, device=device, dtype=torch.float64)
        t = torch.arange(NP, device=device, dtype=torch.float64)[None, :]
        pos = torch.floor((t + u) * n_t / NP).to(torch.int64)
        qq = q.float()[st[:, None], (torch.arange(NP, device=device) % cfg.G)[None, :]]
        kn = 8.0 * math.sqrt(d) * qq / (qq * qq).sum(-1, keepdim=True)
        K[(o_t + pos).reshape(-1)] = kn.reshape(-1, d).to(torch.bfloat16)
    return dict(K=K, V=V, q=q, rows=rows,
                seg_off=torch.tensor(off, dtype=torch.int64, device=device),
                seg_len=torch.tensor(lens, dtype=torch.int32, device=device))


# --------------------------------------------------------------------------
# EpiCache per-turn matching inputs
# --------------------------------------------------------------------------
def gen_turn_embeddings(E: int, De: int, B: int, seed: int = 11, spread: float = 0.6, new_topic_frac: float = 0.1):
    """Episode centroids (N(0, I)) and B question embeddings: most drawn
    around a random centroid with per-dimension spread `spread`, a fraction
    `new_topic_frac` drawn far from all of them (3 N(0, I)).  float32."""
    rng = np.random.default_rng(seed)
    C = rng.standard_normal((E, De), dtype=np.float32)
    which = rng.integers(0, E, size=B)
    Q = C[which] + spread * rng.standard_normal((B, De), dtype=np.float32)
    far = rng.random(B) < new_topic_frac
    Q[far] = 3.0 * rng.standard_normal((int(far.sum()), De), dtype=np.float32)
    return C, Q.astype(np.float32)
