"""Float64 CPU oracle for attention-score-driven KV-cache compression.

TEST INFRASTRUCTURE ONLY.  Nothing in the product path imports this module:
only ``tests/``, ``__graft_entry__.smoke()`` and the ``cpu_baseline`` /
``--impl reference`` legs of ``bench.py`` may call it.  It shares no code with
the CUDA library (no kernels, headers, helpers or constants); both sides read
the same seeded bf16 inputs from ``kv_synth``, upcast exactly to float64 here.

Each function restates one step of the method as the pages describe it:

* "KV²가 전체 문맥 재계산 없이 KV 캐시를 압축한다" (onedev.kr/papers/598, the
  KV² page), sections "어떻게 동작하나" (how it works: sinks, chunks of m,
  KeyDiff proxy averaged over layers and KV heads, per-chunk top
  n_q = max(floor(rho |C_r|), 1) query selection) and "무엇과 다른가" (how it
  differs: appended reconstruction queries under a causal forward over the
  whole cache, chunk-restricted max-over-queries score, global gather, sink
  pinning to the max, bottom eviction to the budget, optional iterative
  refinement), "전제와 한계" (headwise compaction needed for serving).
* "[26'ICML] EpiCache" (juyoungkimmy-kim.github.io), section "방법: 3단계",
  step ② (block-wise prefill of 128-2048-token blocks scored against an
  episode's patched prompt, bounded peak memory; Fig. 1b/c) and "+α: 레이어별
  예산 배분" (per-layer budget from a sensitivity with sharpness alpha; Fig. 4).

The pages print no formulas.  Where they are silent this oracle takes the
plainest reading (listed in the design notes):

* KeyDiff: s_i = -cos(k_i, u) with u the mean of the L2-normalised keys of
  that (layer, KV head) over all positions; p_i = unweighted mean over all
  (layer, KV head) pairs.  A zero key has s = 0 and adds nothing to u.
* chunks C_r = [S + r m, min(S + (r+1) m, N)); n_q from the partial size;
  ties in every top-n are broken by the lower position; NaN ranks as -inf.
* appended reconstruction key of a selected position is the cache key at that
  position (KV²) or the prompt's own key (EpiCache); query j of chunk r sees
  all N cache keys and appended keys 0..j; softmax scale 1/sqrt(d); query
  head g reads KV head g // G; inputs are post-RoPE.
* sinks are pinned to the max over the whole score tensor; budgets count the
  sinks; kept positions are returned ascending.
* layer budgets: w_l = sigma_l^alpha / sum sigma^alpha, M_l = largest-remainder
  rounding of L*M*w_l, then at least S.
"""
from __future__ import annotations

import math
from dataclasses import dataclass

import numpy as np


# ---------------------------------------------------------------------------
# bf16 input decoding (storage format only)
# ---------------------------------------------------------------------------
def bf16_to_f64(bits: np.ndarray) -> np.ndarray:
    """Exact float64 value of bfloat16 bit patterns (uint16)."""
    b = np.ascontiguousarray(bits, dtype=np.uint16).astype(np.uint32) << 16
    return b.view(np.float32).astype(np.float64)


def _rank_value(x: float) -> float:
    """NaN ranks below every number (reading: NaN counts as -inf)."""
    return -math.inf if x != x else float(x)


# ---------------------------------------------------------------------------
# Stage 1: KeyDiff proxy  (KV² page, "어떻게 동작하나")
# ---------------------------------------------------------------------------
def keydiff_head(K: np.ndarray) -> np.ndarray:
    """KeyDiff score of every position of one (layer, KV head).

    K: float64 [N, d].  Returns s [N] with s_i = -(k_i . u) / (|k_i| |u|),
    u = mean_i k_i / |k_i| (zero keys excluded from the sum but counted in N).
    A higher score means the key is less like the typical key, i.e. more
    worth keeping.
    """
    K = np.asarray(K, dtype=np.float64)
    N = K.shape[0]
    norms = np.sqrt(np.sum(K * K, axis=1))
    unit = np.zeros_like(K)
    nz = norms > 0
    unit[nz] = K[nz] / norms[nz, None]
    u = unit.sum(axis=0) / N
    nu = math.sqrt(float(u @ u))
    s = np.zeros(N, dtype=np.float64)
    if nu == 0.0:
        return s
    s[nz] = -(unit[nz] @ u) / nu
    return s


def knorm_head(K: np.ndarray) -> np.ndarray:
    """Knorm proxy of one (layer, KV head): s_i = -|k_i| (the KV² page,
    "전제와 한계", names Knorm as the close alternative to KeyDiff; keys of
    smaller L2 norm rank higher)."""
    K = np.asarray(K, dtype=np.float64)
    return -np.sqrt(np.sum(K * K, axis=1))


def proxy_scores(K: np.ndarray, kind: str = "keydiff"):
    """Token-level proxy p_i = mean over (layer, KV head) of the per-head
    proxy (KeyDiff by default, or Knorm).

    K: float64 (or bf16 bits) [L, Hkv, N, d].  Returns (p [N], s [L, Hkv, N]).
    The pages report that the mean beat the max as the layer/head aggregate.
    """
    head = {"keydiff": keydiff_head, "knorm": knorm_head}[kind]
    L, H = K.shape[:2]
    if K.dtype == np.uint16:
        s = np.stack([np.stack([head(bf16_to_f64(K[l, h])) for h in range(H)]) for l in range(L)])
    else:
        s = np.stack([np.stack([head(K[l, h]) for h in range(H)]) for l in range(L)])
    p = s.reshape(L * H, -1).mean(axis=0)
    return p, s


# ---------------------------------------------------------------------------
# Stage 1: chunking and per-chunk query selection
# ---------------------------------------------------------------------------
@dataclass(frozen=True)
class Chunk:
    lo: int       # first cache position of C_r
    hi: int       # one past the last
    off: int      # offset of this chunk's queries in the concatenated selection
    nq: int       # n_q = max(floor(rho |C_r|), 1)


def chunk_plan(N: int, sinks: int, m: int, rho: float) -> list[Chunk]:
    """Chunks of size m over the non-sink part and their query counts."""
    if not (0 < rho <= 1) or m < 1 or sinks < 0 or sinks >= N:
        raise ValueError("invalid chunk plan arguments")
    out, off, lo = [], 0, sinks
    while lo < N:
        hi = min(lo + m, N)
        nq = max(int(math.floor(rho * (hi - lo) + 1e-9)), 1)
        out.append(Chunk(lo, hi, off, nq))
        off += nq
        lo = hi
    return out


def top_n_positions(values, lo: int, hi: int, n: int) -> list[int]:
    """The n positions in [lo, hi) with the largest values; the lower
    position wins a tie.  Returned in ascending position order."""
    order = sorted(range(lo, hi), key=lambda i: (-_rank_value(values[i]), i))
    return sorted(order[:n])


def select_queries(p: np.ndarray, N: int, sinks: int, m: int, rho: float):
    """Q_r = top n_q positions of p inside each chunk C_r (ascending).

    Returns (sel int64 [sum n_q], chunks).  The selected positions need not be
    contiguous.
    """
    chunks = chunk_plan(N, sinks, m, rho)
    sel = []
    for c in chunks:
        sel.extend(top_n_positions(p, c.lo, c.hi, c.nq))
    return np.asarray(sel, dtype=np.int64), chunks


# ---------------------------------------------------------------------------
# Stage 2: reconstruction scoring  (KV² page, "무엇과 다른가")
# ---------------------------------------------------------------------------
def recon_head(K: np.ndarray, Qrows: np.ndarray, Kapp: np.ndarray, chunks, cols=None):
    """Scores of one (layer, KV head) from its G query heads.

    K:     float64 [N, d]      prefilled cache keys of this KV head
    Qrows: float64 [G, Q, d]   reconstruction query vectors, chunk-major
                               (rows chunks[r].off .. off+nq of chunk r)
    Kapp:  float64 [Q, d]      keys of the appended reconstruction tokens
    chunks: list[Chunk]
    cols:  optional per-chunk (lo, hi) of scored cache positions (default:
           the chunk's own range)

    For query j of chunk r the logit row is
        z = [q.k_0 ... q.k_{N-1}, q.kapp_0 ... q.kapp_j] / sqrt(d)
    (the appended tokens follow the cache under a causal mask), lse = log sum
    exp z, and the attention paid to cache position i is exp(z_i - lse).  The
    score of i in C_r is the max of that attention over the chunk's queries
    and over the G query heads.  Returns (score [N] with NaN outside the
    chunks, lse [G, Q]).
    """
    N, d = K.shape
    G, Qn, _ = Qrows.shape
    scale = 1.0 / math.sqrt(d)
    score = np.full(N, np.nan)
    lse = np.zeros((G, Qn))
    for r, c in enumerate(chunks):
        lo, hi = (c.lo, c.hi) if cols is None else cols[r]
        ka = Kapp[c.off:c.off + c.nq]
        causal = np.tril(np.ones((c.nq, c.nq), dtype=bool))
        best = np.zeros(hi - lo)
        for g in range(G):
            q = Qrows[g, c.off:c.off + c.nq]
            zc = (q @ K.T) * scale                 # [nq, N] cache logits
            za = (q @ ka.T) * scale                # [nq, nq] appended logits
            za = np.where(causal, za, -np.inf)     # query j sees appended 0..j
            z = np.concatenate([zc, za], axis=1)
            mx = z.max(axis=1, keepdims=True)
            row_lse = mx[:, 0] + np.log(np.exp(z - mx).sum(axis=1))
            lse[g, c.off:c.off + c.nq] = row_lse
            att = np.exp(zc[:, lo:hi] - row_lse[:, None])   # attention to C_r
            best = np.maximum(best, att.max(axis=0))
        score[lo:hi] = best
    return score, lse


def recon_scores(K, Qpool, sel, chunks, Kapp=None, pairs=None):
    """Stage-2 scores for all (or the listed) (layer, KV head) pairs.

    K:     [L, Hkv, N, d] bf16 bits or float64
    Qpool: [L, Hq, Npool, d] query pool (one query per position per q head)
    sel:   [Q] source positions of the reconstruction tokens (chunk-major);
           query rows are Qpool[l, g, sel], appended keys K[l, h, sel] unless
           ``Kapp`` [L, Hkv, Q, d] gives them explicitly
    Returns (score [L, Hkv, N] (NaN at sinks), lse [L, Hq, Q]); with ``pairs``
    only those (l, h) entries are filled (others NaN).
    """
    L, H, N, d = K.shape
    Hq = Qpool.shape[1]
    G = Hq // H
    sel = np.asarray(sel, dtype=np.int64)
    f = (lambda a: bf16_to_f64(a)) if K.dtype == np.uint16 else (lambda a: np.asarray(a, np.float64))
    score = np.full((L, H, N), np.nan)
    lse = np.full((L, Hq, len(sel)), np.nan)
    todo = pairs if pairs is not None else [(l, h) for l in range(L) for h in range(H)]
    for (l, h) in todo:
        Klh = f(K[l, h])
        Qrows = np.stack([f(Qpool[l, h * G + g][sel]) for g in range(G)])
        ka = Klh[sel] if Kapp is None else f(Kapp[l, h])
        sc, ls = recon_head(Klh, Qrows, ka, chunks)
        score[l, h] = sc
        lse[l, h * G:(h + 1) * G] = ls
    return score, lse


def refine_proxy(score: np.ndarray, sinks: int) -> np.ndarray:
    """Iterative refinement: the next pass's token score is the mean over
    (layer, KV head) of this pass's stage-2 scores (same token granularity as
    the proxy).  Sink entries are not used by selection and are set to 0."""
    L, H, N = score.shape
    p = np.zeros(N)
    p[sinks:] = score[:, :, sinks:].reshape(L * H, -1).mean(axis=0)
    return p


# ---------------------------------------------------------------------------
# Eviction and compaction
# ---------------------------------------------------------------------------
def pin_sinks(score: np.ndarray, sinks: int) -> float:
    """Set every sink entry to the max of the gathered score tensor (in
    place); returns that max."""
    gmax = float(np.nanmax(score[..., sinks:])) if score.shape[-1] > sinks else 0.0
    score[..., :sinks] = gmax
    return gmax


def evict(score: np.ndarray, sinks: int, k_per_layer) -> list:
    """Pin sinks, then keep the k_l highest-scored positions of each
    (layer, KV head) (lower position wins a tie).  Returns kept[l] as int64
    [Hkv, k_l] ascending.  ``score`` is modified in place (sinks pinned)."""
    L, H, N = score.shape
    pin_sinks(score, sinks)
    kept = []
    for l in range(L):
        k = int(k_per_layer[l])
        if k < sinks or k > N:
            raise ValueError("budget must lie in [sinks, N]")
        kept.append(np.stack([np.asarray(top_n_positions(score[l, h], 0, N, k), dtype=np.int64)
                              for h in range(H)]) if k > 0 else np.zeros((H, 0), np.int64))
    return kept


def compact(X: np.ndarray, kept: list) -> list:
    """Headwise compaction: X_c[l][h, t] = X[l, h, kept[l][h, t]]."""
    out = []
    for l, kl in enumerate(kept):
        out.append(np.stack([X[l, h][kl[h]] for h in range(kl.shape[0])]))
    return out


def budget_count(b: float, N: int) -> int:
    """Kept tokens per (layer, KV head) for a budget fraction b (sinks
    included)."""
    return int(math.floor(b * N + 1e-9))


# ---------------------------------------------------------------------------
# Whole KV² pass (single or iterative)
# ---------------------------------------------------------------------------
def kv2_compress(K, V, Qpool, sinks, m, rho, k_per_layer, passes=1, proxy="keydiff"):
    """proxy -> passes x (select -> reconstruct -> [refine]) -> evict -> compact."""
    L, H, N, d = K.shape
    p, _ = proxy_scores(K, proxy)
    sel_hist = []
    for t in range(passes):
        sel, chunks = select_queries(p, N, sinks, m, rho)
        score, lse = recon_scores(K, Qpool, sel, chunks)
        sel_hist.append(sel)
        if t < passes - 1:
            p = refine_proxy(score, sinks)
    kept = evict(score, sinks, k_per_layer)
    return dict(p=p, sel=sel_hist, chunks=chunks, score=score, lse=lse, kept=kept,
                Kc=compact(K, kept), Vc=compact(V, kept))


# ---------------------------------------------------------------------------
# EpiCache: per-layer budgets and block prefill  ("[26'ICML] EpiCache")
# ---------------------------------------------------------------------------
def layer_budgets(sens, alpha: float, mean_budget: int, sinks: int) -> np.ndarray:
    """Per-layer budgets M_l from the sensitivity weighting with sharpness
    alpha (alpha = 0: uniform; larger alpha concentrates budget on sensitive
    layers).  The total L * mean_budget is split by largest remainder (ties
    to the lower layer), then each M_l is raised to at least ``sinks``."""
    sens = np.asarray(sens, dtype=np.float64)
    L = sens.shape[0]
    w = sens ** float(alpha)
    w = w / w.sum()
    total = L * int(mean_budget)
    quota = total * w
    base = np.floor(quota).astype(np.int64)
    rem = total - int(base.sum())
    frac = quota - base
    for l in sorted(range(L), key=lambda i: (-frac[i], i))[:max(rem, 0)]:
        base[l] += 1
    return np.maximum(base, sinks)


def block_step_scores(Kc: np.ndarray, Qprompt: np.ndarray, Kprompt: np.ndarray, sinks: int) -> np.ndarray:
    """Scores of every cache row of one layer against the episode prompt
    (the KV² max rule with the prompt's queries appended causally, one chunk
    covering all non-sink rows).  Kc: [Hkv, n, d]; returns [Hkv, n] with NaN
    at the sinks."""
    H, n, d = Kc.shape
    G = Qprompt.shape[0] // H
    P = Qprompt.shape[1]
    chunks = [Chunk(sinks, n, 0, P)]
    return np.stack([recon_head(Kc[h], Qprompt[h * G:(h + 1) * G], Kprompt[h], chunks)[0] for h in range(H)])


def block_step(Kc, Vc, pos, Kb, Vb, t0, Qprompt, Kprompt, M, sinks):
    """One block-prefill step of one layer: append the block (global
    positions t0..), and if the cache then exceeds M rows, keep the M best
    rows per KV head (sinks pinned, lower global position wins a tie) in
    position order.  Returns (Kc, Vc, pos, scores or None)."""
    H = Kb.shape[0]
    B = Kb.shape[1]
    Kc = np.concatenate([Kc, Kb], axis=1)
    Vc = np.concatenate([Vc, Vb], axis=1)
    pos = np.concatenate([pos, np.broadcast_to(np.arange(t0, t0 + B), (H, B))], axis=1)
    n = Kc.shape[1]
    if n <= M:
        return Kc, Vc, pos, None
    score = block_step_scores(Kc, Qprompt, Kprompt, sinks)
    work = score[None].copy()
    kept = evict(work, sinks, [M])[0]
    return (np.stack([Kc[h][kept[h]] for h in range(H)]), np.stack([Vc[h][kept[h]] for h in range(H)]),
            np.stack([pos[h][kept[h]] for h in range(H)]), score)


def block_prefill_layer(Kh: np.ndarray, Vh: np.ndarray, Qprompt: np.ndarray, Kprompt: np.ndarray,
                        block: int, M: int, sinks: int, state=None, n_blocks=None):
    """EpiCache block prefill of one layer for one episode.

    Kh, Vh:   float64 [Hkv, n_hist, d] history keys / values
    Qprompt:  float64 [Hq, P, d] patched-prompt queries of the episode
    Kprompt:  float64 [Hkv, P, d] the prompt's keys (appended causally)
    block:    tokens per block; M: this layer's budget
    state:    optional (Kc, Vc, pos, t0) to resume from; n_blocks limits how
              many blocks to process (resume tests).

    Each block is appended behind the kept cache.  When the cache then holds
    more than M tokens, every non-sink position is scored with the prompt
    (max attention over the prompt's queries and each KV head's G query
    heads), sinks are pinned, the M best positions per KV head are kept (lower
    global position wins a tie) in ascending order and the cache is
    compacted.  Returns (Kc, Vc, pos, t0) with pos the global positions.
    """
    H, n_hist, d = Kh.shape
    Hq, P, _ = Qprompt.shape
    G = Hq // H
    if state is None:
        Kc = np.zeros((H, 0, d)); Vc = np.zeros((H, 0, d))
        pos = np.zeros((H, 0), dtype=np.int64); t0 = 0
    else:
        Kc, Vc, pos, t0 = state
    done = 0
    while t0 < n_hist and (n_blocks is None or done < n_blocks):
        t1 = min(t0 + block, n_hist)
        Kc, Vc, pos, _ = block_step(Kc, Vc, pos, Kh[:, t0:t1], Vh[:, t0:t1], t0, Qprompt, Kprompt, M, sinks)
        t0 = t1
        done += 1
    return Kc, Vc, pos, t0
