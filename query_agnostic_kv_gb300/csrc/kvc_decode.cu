// Decode attention over a ragged, headwise-compacted KV cache (the compact
// serving backend the KV² page, section "전제와 한계", says real decode savings
// need).  A segment is the run of kept rows of one (layer, KV head); its G
// query heads each attend over it with ordinary softmax attention.
//
// The op is HBM-bound (every kept K and V row is read once; G = 1..8 queries
// per row, so there is no dense contraction worth a tensor core).  Design:
//  * persistent CTAs, one per SM; work items are (segment, split) pairs handed
//    out by an atomic counter, so a CTA that starts late simply takes fewer;
//  * one producer lane fetches items and streams each split's contiguous K and
//    V rows into a 4-stage shared-memory ring with 1-D bulk copies
//    (cp.async.bulk), completion counted in bytes on an mbarrier.  Each stage
//    carries a header (item, tile index) written by the producer, and the
//    first tile of an item also carries the item's queries, so consumers never
//    touch global memory on the way in;
//  * consumer warps split a tile; 16 lanes share one key (8 of its 128 dims,
//    one 16-byte shared-memory load per row), so a warp holds two keys at a
//    time; the G partial dot products are reduce-scattered across the 16
//    lanes, leaving one (key, query) logit per lane;
//  * packed f32x2 FMAs for q.k and p.v; base-2 online softmax with a lazily
//    updated reference max (rebased only when a logit exceeds it by 16);
//  * at the end of an item the warps' partials are merged through shared
//    memory (bounded mbarrier hand-offs); a one-split segment writes its
//    output, a split writes its (max, sum, unnormalised output) partial and a
//    second small kernel merges the splits.
// Every wait is bounded; on expiry the kernel records KVC_ERR_TIMEOUT and
// unwinds.  Segments whose (offset, length) fall outside the cache are
// reported as KVC_ERR_BOUNDS and skipped.
#include <cmath>

#include "kvc_internal.h"
#include "kvc_ptx.cuh"

namespace kvc {
namespace {

constexpr int D = kHeadDim;
constexpr int ROW_BYTES = D * 2;
constexpr int LPK = 16;                      // lanes per key
constexpr int LOG2_LPK = 4;
constexpr int KPW = 32 / LPK;                // keys per warp per batch
constexpr float REBASE = 16.f;               // log2 units
constexpr int kTargetItems = 4864;           // work items aimed for (32 per SM)
constexpr int kMinSplit = 512;               // keys
constexpr int HDR_BYTES = 128;


template <int GP>
struct DCfg {
  static constexpr int NW = GP <= 4 ? 15 : 8;        // consumer warps
  static constexpr int NB = GP <= 4 ? 4 : 2;        // batches per warp per tile
  static constexpr int STAGES = GP <= 4 ? 3 : 6;
  static constexpr int TK = KPW * NW * NB;                   // keys per stage
  static constexpr int TILE_BYTES = TK * ROW_BYTES;  // one of K or V
  static constexpr int QBYTES = GP * ROW_BYTES;      // the item's queries (first tile)
  static constexpr int STAGE_BYTES = HDR_BYTES + QBYTES + 2 * TILE_BYTES;
  static constexpr int THREADS = (NW + 1) * 32;
  static constexpr int ML_FLOATS = (2 * NW * GP + 3) / 4 * 4;   // sM, sL padded to whole float4s
  static constexpr int COMB_FLOATS = ML_FLOATS + NW * GP * D;
  static constexpr size_t SMEM = 128 + size_t(STAGES) * STAGE_BYTES + size_t(COMB_FLOATS) * 4 + 256;
};

// Written by the producer into each stage before it is released.
struct StageHdr {
  int32_t seg, c;      // segment, split
  int32_t t, nt;       // tile index within the item, tiles of the item
  int32_t rows;        // keys of the item
  int32_t ns;          // nonempty splits of the segment
  int32_t end;         // 1: no more items
  int32_t pad;
};

constexpr int MAX_STAGES = 8;
struct DBars {
  uint64_t full[MAX_STAGES];
  uint64_t empty[MAX_STAGES];
  uint64_t comb_full;   // every consumer warp has written its partial
  uint64_t comb_free;   // every consumer warp has read the merged partials
  int abort_flag;
};

__device__ __forceinline__ float ex2f(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ uint4 lds128(const void* p) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "r"(smem_u32(p)));
  return v;
}

// bf16 pair (one 32-bit word, low half = lower index) -> packed f32x2
__device__ __forceinline__ uint64_t bf2_to_f2(uint32_t w) {
  return pack2(__uint_as_float(w << 16), __uint_as_float(w & 0xffff0000u));
}

__device__ __forceinline__ float sum2(uint64_t a) {
  float x, y;
  unpack2(a, x, y);
  return x + y;
}

// Slot permutation of a lane: slot i of lane `lane` holds query i ^ qmask.
// With it every lane keeps the low half of its slots and sends the high half
// at each reduce-scatter step, so the exchange needs no selects.
template <int GP>
__device__ __forceinline__ int slot_mask(int lane) {
  return (lane & (LPK - 1)) / (LPK / GP);
}

// Reduce-scatter GP partial sums over the LPK lanes of a key (slots permuted
// by slot_mask): afterwards the lane holds the full sum of query
// (lane % LPK) / (LPK / GP).
template <int GP>
__device__ __forceinline__ float reduce_scatter(float (&v)[GP]) {
#pragma unroll
  for (int st = 0; st < LOG2_LPK; ++st) {
    const int o = (LPK / 2) >> st;
    const int n = GP >> st;
    if (n > 1) {
      const int h = n / 2;
#pragma unroll
      for (int i = 0; i < h; ++i) v[i] += __shfl_xor_sync(0xffffffffu, v[i + h], o);
    } else {
      v[0] += __shfl_xor_sync(0xffffffffu, v[0], o);
    }
  }
  return v[0];
}

// Segment bounds as both kernels check them.
__device__ __forceinline__ bool seg_ok(const DecodeParams& P, int seg, int& len, int64_t& off) {
  len = P.seg_len[seg];
  off = P.seg_off[seg];
  return !(len < 0 || len > P.max_len || off < 0 || off + len > P.kv_rows);
}

template <int GP>
__global__ void __launch_bounds__(DCfg<GP>::THREADS, 1) decode_kernel(const DecodeParams P) {
  using C = DCfg<GP>;
  constexpr int NW = C::NW;
  constexpr int NB = C::NB;
  constexpr int NCT = NW * 32;               // consumer threads
  constexpr int TK = C::TK;
  constexpr int TILE_BYTES = C::TILE_BYTES;
  constexpr int STAGE_BYTES = C::STAGE_BYTES;
  constexpr int STAGES = C::STAGES;
  static_assert(STAGES <= MAX_STAGES, "too many stages");
  static_assert(C::SMEM <= 232448, "shared memory per CTA exceeds 227 KB");
  static_assert(STAGE_BYTES % 16 == 0, "stages must stay 16-byte aligned");
  static_assert((HDR_BYTES + C::QBYTES) % 16 == 0 && TILE_BYTES % 16 == 0, "bulk-copy targets must be 16-byte aligned");
  static_assert((size_t(STAGES) * STAGE_BYTES) % 16 == 0, "combine area must be 16-byte aligned");
  static_assert(C::ML_FLOATS % 4 == 0 && (C::COMB_FLOATS * 4) % 8 == 0, "float4 partials and mbarriers alignment");
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sbase = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 127) & ~uintptr_t(127));
  float* sComb = reinterpret_cast<float*>(sbase + size_t(STAGES) * STAGE_BYTES);
  float* sM = sComb;                          // [NW][GP]
  float* sL = sM + NW * GP;                   // [NW][GP]
  float* sAcc = sComb + C::ML_FLOATS;         // [NW][GP][D], 16-byte aligned
  DBars* bars = reinterpret_cast<DBars*>(sComb + C::COMB_FLOATS);

  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  const int n_items = P.n_seg * P.n_split;

  if (tid == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&bars->full[s], 1);
      mbar_init(&bars->empty[s], NW);
    }
    mbar_init(&bars->comb_full, NCT);
    mbar_init(&bars->comb_free, NCT);
    bars->abort_flag = 0;
    fence_barrier_init();
  }
  __syncthreads();
  volatile int* abort_flag = &bars->abort_flag;

  if (warp == NW) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      int s = 0;
      uint32_t ph = 0;
      int64_t n_pushed = 0;
      bool stop = false;
      int i = atomicAdd(P.counter, 1);
      while (!stop) {
        if (i >= n_items) {
          // no more work: release one stage carrying the end marker
          if (!mbar_wait(&bars->empty[s], ph ^ 1u, P.limit_ns)) {
            *abort_flag = 1;
            record_status(P.status, DEV_TIMEOUT);
            break;
          }
          reinterpret_cast<StageHdr*>(sbase + size_t(s) * STAGE_BYTES)->end = 1;
          mbar_arrive(&bars->full[s]);
          ++n_pushed;
          break;
        }
        const int inext = atomicAdd(P.counter, 1);     // in flight while this item is issued
        const int seg = i / P.n_split;
        const int c = i - seg * P.n_split;
        int len;
        int64_t off;
        if (!seg_ok(P, seg, len, off)) {
          if (c == 0) record_status(P.status, DEV_BOUNDS);
          i = inext;
          continue;
        }
        const int r0 = c * P.CH;
        const int rows = min(P.CH, len - r0);
        if (rows <= 0) {
          if (c == 0 && len == 0) {   // empty segment: zero output, lse = -inf
            for (int x = 0; x < P.G * D; ++x) P.out[int64_t(seg) * P.G * D + x] = 0.f;
            if (P.lse)
              for (int g = 0; g < P.G; ++g) P.lse[int64_t(seg) * P.G + g] = -INFINITY;
          }
          i = inext;
          continue;
        }
        const int ns = (len + P.CH - 1) / P.CH;
        const int nt = (rows + TK - 1) / TK;
        for (int t = 0; t < nt; ++t) {
          if (*abort_flag) { stop = true; break; }
          if (!mbar_wait(&bars->empty[s], ph ^ 1u, P.limit_ns)) {
            *abort_flag = 1;
            record_status(P.status, DEV_TIMEOUT);
            stop = true;
            break;
          }
          uint8_t* st = sbase + size_t(s) * STAGE_BYTES;
          StageHdr* hd = reinterpret_cast<StageHdr*>(st);
          hd->seg = seg;
          hd->c = c;
          hd->t = t;
          hd->nt = nt;
          hd->rows = rows;
          hd->ns = ns;
          hd->end = 0;
          const int nr = min(TK, rows - t * TK);
          const uint32_t bytes = static_cast<uint32_t>(nr) * ROW_BYTES;
          const uint32_t qb = t == 0 ? static_cast<uint32_t>(P.G) * ROW_BYTES : 0u;
          const int64_t row = off + r0 + int64_t(t) * TK;
          mbar_arrive_expect_tx(&bars->full[s], 2 * bytes + qb);
          if (qb) bulk_load(st + HDR_BYTES, P.q + int64_t(seg) * P.G * D, qb, &bars->full[s]);
          bulk_load(st + HDR_BYTES + C::QBYTES, P.K + row * D, bytes, &bars->full[s]);
          bulk_load(st + HDR_BYTES + C::QBYTES + TILE_BYTES, P.V + row * D, bytes, &bars->full[s]);
          ++n_pushed;
          if (++s == STAGES) { s = 0; ph ^= 1u; }
        }
        i = inext;
      }
      // Wait for every copy this thread started before the CTA may exit.
      for (int k = 0; k < STAGES; ++k) {
        const int64_t nk = n_pushed / STAGES + (k < n_pushed % STAGES ? 1 : 0);   // phases of stage k
        if (nk > 0) mbar_wait(&bars->full[k], static_cast<uint32_t>(nk - 1) & 1u, P.limit_ns);
      }
    }
    return;
  }

  // -------------------------------------------------------------- consumers
  const int j = lane & (LPK - 1);            // 16-byte chunk of the row this lane owns
  const int kg = lane / LPK;                 // key within the warp's batch
  constexpr int DUP = LPK / GP;              // lanes holding the same (key, query) logit
  const int lq = j / DUP;                    // query index of this lane's logit
  const bool rep = (j % DUP) == 0;
  const int qmask = slot_mask<GP>(lane);
  int s = 0;
  uint32_t ph = 0, cph = 0;
  uint64_t qv[GP][4];
  uint64_t acc[GP][4];
  float m = -INFINITY, l = 0.f;

  while (true) {
    {
      const bool ok = !*abort_flag && mbar_wait(&bars->full[s], ph, P.limit_ns);
      if (__any_sync(0xffffffffu, !ok)) {   // the warp decides as one
        if (lane == 0) {
          *abort_flag = 1;
          record_status(P.status, DEV_TIMEOUT);
        }
        break;
      }
    }
    const uint8_t* st = sbase + size_t(s) * STAGE_BYTES;
    const StageHdr h = *reinterpret_cast<const StageHdr*>(st);
    if (h.end) break;
    if (h.t == 0) {
      // new item: its queries, pre-scaled to base-2 logits, in this lane's slot order
#pragma unroll
      for (int g = 0; g < GP; ++g) {
        const int qg = g ^ qmask;
        uint4 w = make_uint4(0u, 0u, 0u, 0u);
        if (qg < P.G) w = lds128(st + HDR_BYTES + qg * ROW_BYTES + j * 16);
        const uint32_t ww[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          float a, b;
          unpack2(bf2_to_f2(ww[k]), a, b);
          qv[g][k] = pack2(a * P.sc2, b * P.sc2);
          acc[g][k] = 0ull;
        }
      }
      m = -INFINITY;
      l = 0.f;
    }
    const int kb = warp * (KPW * NB);                    // first key of this warp in the tile
    const int nval = min(KPW * NB, h.rows - h.t * TK - kb);
    if (nval > 0) {
      const uint8_t* sK = st + HDR_BYTES + C::QBYTES;
      const uint8_t* sV = sK + TILE_BYTES;
      float sc[NB];
      // ---- logits
#pragma unroll
      for (int b = 0; b < NB; ++b) {
        const int e = b * KPW + kg;                      // key within this warp's block
        const bool valid = e < nval;
        uint4 kr = make_uint4(0u, 0u, 0u, 0u);
        if (valid) kr = lds128(sK + (kb + e) * ROW_BYTES + j * 16);
        const uint64_t k0 = bf2_to_f2(kr.x), k1 = bf2_to_f2(kr.y), k2 = bf2_to_f2(kr.z), k3 = bf2_to_f2(kr.w);
        float part[GP];
#pragma unroll
        for (int g = 0; g < GP; ++g) {
          uint64_t a = fma2(k0, qv[g][0], 0ull);
          a = fma2(k1, qv[g][1], a);
          a = fma2(k2, qv[g][2], a);
          a = fma2(k3, qv[g][3], a);
          part[g] = sum2(a);
        }
        const float z = reduce_scatter<GP>(part);
        sc[b] = valid ? z : -INFINITY;
      }
      // ---- online softmax (per warp, per query; lazily rebased)
      float mx = sc[0];
#pragma unroll
      for (int b = 1; b < NB; ++b) mx = fmaxf(mx, sc[b]);
#pragma unroll
      for (int o = LPK; o < 32; o <<= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
      if (m == -INFINITY) {
        m = mx;                                          // first keys of the item: exact max
      } else if (__any_sync(0xffffffffu, mx > m + REBASE)) {
        const float mn = fmaxf(m, mx);
        const float f = ex2f(m - mn);
        l *= f;
#pragma unroll
        for (int g = 0; g < GP; ++g) {
          const float fg = __shfl_sync(0xffffffffu, f, g * DUP);
          const uint64_t f2 = pack2(fg, fg);
#pragma unroll
          for (int k = 0; k < 4; ++k) acc[g][k] = fma2(acc[g][k], f2, 0ull);
        }
        m = mn;
      }
      float p[NB];
#pragma unroll
      for (int b = 0; b < NB; ++b) {
        p[b] = ex2f(sc[b] - m);
        if (rep) l += p[b];
      }
      // ---- p . v
#pragma unroll
      for (int b = 0; b < NB; ++b) {
        const int e = b * KPW + kg;
        uint4 vr = make_uint4(0u, 0u, 0u, 0u);
        if (e < nval) vr = lds128(sV + (kb + e) * ROW_BYTES + j * 16);
        const uint64_t v0 = bf2_to_f2(vr.x), v1 = bf2_to_f2(vr.y), v2 = bf2_to_f2(vr.z), v3 = bf2_to_f2(vr.w);
#pragma unroll
        for (int g = 0; g < GP; ++g) {
          const float pg = __shfl_sync(0xffffffffu, p[b], (lane & ~(LPK - 1)) | (g * DUP));
          const uint64_t p2 = pack2(pg, pg);
          acc[g][0] = fma2(p2, v0, acc[g][0]);
          acc[g][1] = fma2(p2, v1, acc[g][1]);
          acc[g][2] = fma2(p2, v2, acc[g][2]);
          acc[g][3] = fma2(p2, v3, acc[g][3]);
        }
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&bars->empty[s]);
    if (++s == STAGES) { s = 0; ph ^= 1u; }
    if (h.t != h.nt - 1) continue;

    // ---- end of the item: warp partial (m, l, acc) -> shared memory
#pragma unroll
    for (int o = LPK; o < 32; o <<= 1)
#pragma unroll
      for (int g = 0; g < GP; ++g)
#pragma unroll
        for (int k = 0; k < 4; ++k) acc[g][k] = add2(acc[g][k], __shfl_xor_sync(0xffffffffu, acc[g][k], o));
#pragma unroll
    for (int o = 1; o < DUP; o <<= 1) l += __shfl_xor_sync(0xffffffffu, l, o);
#pragma unroll
    for (int o = LPK; o < 32; o <<= 1) l += __shfl_xor_sync(0xffffffffu, l, o);
    {
      // the previous item's merged partials must have been read by everyone
      const bool ok = mbar_wait(&bars->comb_free, cph ^ 1u, P.limit_ns);
      if (__any_sync(0xffffffffu, !ok)) {
        if (lane == 0) {
          *abort_flag = 1;
          record_status(P.status, DEV_TIMEOUT);
        }
        break;
      }
    }
    if (lane < LPK) {
#pragma unroll
      for (int g = 0; g < GP; ++g) {
        float4 lo, hi;
        unpack2(acc[g][0], lo.x, lo.y);
        unpack2(acc[g][1], lo.z, lo.w);
        unpack2(acc[g][2], hi.x, hi.y);
        unpack2(acc[g][3], hi.z, hi.w);
        float4* dst = reinterpret_cast<float4*>(sAcc + (warp * GP + g) * D + j * 8);
        dst[0] = lo;
        dst[1] = hi;
      }
      if (rep) {
        sM[warp * GP + lq] = m;
        sL[warp * GP + lq] = l;
      }
    }
    mbar_arrive(&bars->comb_full);
    {
      const bool ok = mbar_wait(&bars->comb_full, cph, P.limit_ns);
      if (__any_sync(0xffffffffu, !ok)) {
        if (lane == 0) {
          *abort_flag = 1;
          record_status(P.status, DEV_TIMEOUT);
        }
        break;
      }
    }
    // ---- merge the warps; write the output or this split's partial
    const bool single = h.ns == 1;
    const int64_t pbase = (int64_t(h.seg) * P.n_split + h.c) * P.G;
    for (int idx = tid; idx < P.G * D; idx += NCT) {
      const int g = idx / D;
      const int dd = idx - g * D;
      float M = -INFINITY;
#pragma unroll
      for (int w = 0; w < NW; ++w) M = fmaxf(M, sM[w * GP + g]);
      float O = 0.f, Ls = 0.f;
#pragma unroll
      for (int w = 0; w < NW; ++w) {
        const float f = ex2f(sM[w * GP + g] - M);
        O = fmaf(f, sAcc[(w * GP + g) * D + dd], O);
        Ls = fmaf(f, sL[w * GP + g], Ls);
      }
      if (single) {
        P.out[(int64_t(h.seg) * P.G + g) * D + dd] = O / Ls;
        if (dd == 0 && P.lse) P.lse[int64_t(h.seg) * P.G + g] = (M + log2f(Ls)) * 0.69314718055994531f;
      } else {
        P.part_o[(pbase + g) * D + dd] = O;
        if (dd == 0) {
          P.part_ml[(pbase + g) * 2] = M;
          P.part_ml[(pbase + g) * 2 + 1] = Ls;
        }
      }
    }
    mbar_arrive(&bars->comb_free);
    cph ^= 1u;
  }
}

// Merges the splits of every multi-split segment: one warp per (segment,
// query head), four output dims per lane.
__global__ void __launch_bounds__(256) merge_kernel(const DecodeParams P) {
  const int gw = blockIdx.x * 8 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (gw >= P.n_seg * P.G) return;
  const int seg = gw / P.G;
  const int g = gw - seg * P.G;
  int len;
  int64_t off;
  if (!seg_ok(P, seg, len, off) || len == 0) return;
  const int ns = (len + P.CH - 1) / P.CH;
  if (ns == 1) return;
  const int64_t base = int64_t(seg) * P.n_split * P.G + g;
  float M = -INFINITY;
  for (int c = 0; c < ns; ++c) M = fmaxf(M, P.part_ml[(base + int64_t(c) * P.G) * 2]);
  float4 O = make_float4(0.f, 0.f, 0.f, 0.f);
  float Ls = 0.f;
  for (int c = 0; c < ns; ++c) {
    const int64_t r = base + int64_t(c) * P.G;
    const float f = ex2f(P.part_ml[r * 2] - M);
    const float4 o = reinterpret_cast<const float4*>(P.part_o + r * D)[lane];
    O.x = fmaf(f, o.x, O.x);
    O.y = fmaf(f, o.y, O.y);
    O.z = fmaf(f, o.z, O.z);
    O.w = fmaf(f, o.w, O.w);
    Ls = fmaf(f, P.part_ml[r * 2 + 1], Ls);
  }
  const float inv = 1.f / Ls;
  float* dst = P.out + (int64_t(seg) * P.G + g) * D + lane * 4;
  dst[0] = O.x * inv;
  dst[1] = O.y * inv;
  dst[2] = O.z * inv;
  dst[3] = O.w * inv;
  if (lane == 0 && P.lse) P.lse[int64_t(seg) * P.G + g] = (M + log2f(Ls)) * 0.69314718055994531f;
}

template <int GP>
cudaError_t launch_gp(const DecodeParams& p, int grid, cudaStream_t st) {
  using C = DCfg<GP>;
  cudaError_t e = cudaFuncSetAttribute(decode_kernel<GP>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(C::SMEM));
  if (e != cudaSuccess) return e;
  decode_kernel<GP><<<grid, C::THREADS, C::SMEM, st>>>(p);
  return cudaGetLastError();
}

}  // namespace
}  // namespace kvc

namespace kvc {

int32_t decode_tile_keys(int32_t G) {
  return G <= 1 ? DCfg<1>::TK : G <= 2 ? DCfg<2>::TK : G <= 4 ? DCfg<4>::TK : DCfg<8>::TK;
}

DecodePlan make_decode_plan(int32_t n_seg, int32_t G, int32_t max_len) {
  DecodePlan pl;
  const int32_t q = decode_tile_keys(G);   // splits are whole tiles
  if (n_seg < 1 || max_len < 1) {
    pl.CH = q;
    pl.n_split = 1;
    return pl;
  }
  int64_t want = (kTargetItems + n_seg - 1) / n_seg;                 // splits per segment for ~kTargetItems items
  const int64_t cap = (int64_t(max_len) + kMinSplit - 1) / kMinSplit;  // but no split below kMinSplit keys
  want = want < cap ? want : cap;
  if (want < 1) want = 1;
  int64_t ch = (int64_t(max_len) + want - 1) / want;
  ch = (ch + q - 1) / q * q;
  pl.CH = static_cast<int32_t>(ch);
  pl.n_split = static_cast<int32_t>((int64_t(max_len) + ch - 1) / ch);
  return pl;
}

cudaError_t launch_decode(const DecodeParams& p, cudaStream_t st) {
  const int64_t items = int64_t(p.n_seg) * p.n_split;
  if (items == 0) return cudaSuccess;
  cudaError_t e = cudaMemsetAsync(p.counter, 0, sizeof(int32_t), st);
  if (e != cudaSuccess) return e;
  const int grid = static_cast<int>(items < num_sms() ? items : num_sms());
  {
    ProfScope ps("decode_attn", st);
    if (p.G <= 1) e = launch_gp<1>(p, grid, st);
    else if (p.G <= 2) e = launch_gp<2>(p, grid, st);
    else if (p.G <= 4) e = launch_gp<4>(p, grid, st);
    else e = launch_gp<8>(p, grid, st);
  }
  if (e != cudaSuccess || p.n_split == 1) return e;
  ProfScope ps("decode_merge", st);
  const int64_t warps = int64_t(p.n_seg) * p.G;
  merge_kernel<<<static_cast<unsigned>((warps + 7) / 8), 256, 0, st>>>(p);
  return cudaGetLastError();
}

}  // namespace kvc
