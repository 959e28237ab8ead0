// Top-n selection with a deterministic tie rule, used twice on the path:
//  * KV² page, "어떻게 동작하나": inside each chunk C_r, the n_q positions with
//    the highest token score p become the reconstruction queries;
//  * KV² page, "무엇과 다른가": after gathering the scores, the sinks are
//    pinned to the max and the lowest-scored entries of every (layer, KV
//    head) are removed down to the budget.
// In both the lower position wins a tie and the output is in ascending
// position order.
//
// Main kernel (topk_cluster_kernel): one thread-block cluster of C CTAs per
// row (a chunk of p, or one (layer, KV head) score row).  Each CTA reads its
// contiguous part of the row from global memory ONCE, as order-preserving
// uint32 keys, into shared memory (float -> key: NaN below -inf, -0 -> +0).
// Everything after that runs out of shared memory:
//   1. the cluster's minimum and maximum key: their common leading bits are
//      shared by every key, so the radix select starts below them;
//   2. MSB-first radix select in 8-bit digits for the n-th largest key T:
//      per-warp histograms (shared-memory atomics), summed per CTA and then
//      over the cluster in rank order through distributed shared memory, so
//      every CTA finds the same digit;
//   3. ordered emit: every key > T plus the lowest-positioned keys == T, with
//      positions written through warp ballots and per-warp / per-CTA prefix
//      counts (the cluster's counts exchanged once);
//   4. eviction only: the kept K/V rows are copied into the compacted cache
//      in the same kernel (optional), and the last CTA to finish pins the
//      sinks to the global max score (when the caller reads the scores).
// A third use, EpiCache's block step ("[26'ICML] EpiCache", "방법: 3단계"
// step ②) on a one-slab state, evicts in place (a separate instance,
// INPLACE): instead of the ordered emit, the evicted rows below the budget
// and the kept rows at or above it are listed and the latter moved into the
// former; ties at the threshold are ranked by the rows' global positions.
// Rows longer than kMaxParts shared-memory parts use the global-memory radix
// kernels at the end of this file.
#include <cooperative_groups.h>

#include <algorithm>
#include <cstring>

#include "kvc_internal.h"
#include "kvc_ptx.cuh"

namespace cg = cooperative_groups;

namespace kvc {
namespace {

__device__ __forceinline__ uint32_t order_key(float x) {
  if (x != x) return 0u;                       // NaN ranks lowest
  uint32_t u = __float_as_uint(x + 0.0f);      // -0 -> +0
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
__device__ __forceinline__ float key_value(uint32_t k) {
  const uint32_t u = (k & 0x80000000u) ? (k & 0x7fffffffu) : ~k;
  return __uint_as_float(u);
}

// ====================================================================
// Cluster kernel
// ====================================================================
constexpr int CT = 512;               // threads per CTA
constexpr int CW = CT / 32;           // warps per CTA
constexpr int kPartKeys = 16384;      // keys per CTA in the common case (64 KB)
constexpr int kPartKeysMax = 49152;   // keys per CTA at most (192 KB)
constexpr int kMaxParts = 8;          // CTAs per row (portable cluster size)
static_assert(kEvictInPlaceRows == kMaxParts * kPartKeysMax, "in-place rows fit the shared-memory parts");

struct TopkArgs {
  int mode;                 // 0: per-chunk selection over p; 1: eviction over score rows; 2: eviction in place
  const float* vals;        // p (mode 0) or score (mode 1)
  // mode 0
  int N, sinks, m, n_chunks, nq_full, nq_last;
  int32_t* sel;
  // mode 1
  int32_t act[kMaxLayers];  // active layers, indexed by blockIdx.z
  int32_t* kept;
  float* score;             // the score rows again, writable (sink pin)
  uint32_t* gmax;           // [0] max order key, [1] arrivals; null: no pin
  int total_ctas;           // CTAs of the launch (last-arriver pin)
  int copy;                 // fused compaction of the kept rows
  int fill;                 // mode 2: entries per (l, h) of each pair list (holes, then movers)
  int* status;              // mode 2: KVC bounds status if holes and movers ever disagree
};

struct TopkShared {
  uint32_t whist[CW][256];  // per-warp histograms of one digit
  uint32_t chist[2][256];   // this CTA's histogram by pass parity (read by the cluster)
  uint32_t ghist[256];      // the cluster's histogram of the current digit
  uint32_t xch[6];          // min key, max key, gt count, eq count, holes, movers (read by the cluster)
  uint32_t wgt[CW], weq[CW];
  uint32_t wsel[CW], weqb[CW];  // per warp: first output slot, global eq rank of its first key
  uint32_t whol[CW], wmov[CW];  // in-place eviction, per warp: holes and movers
  uint32_t kmin, kmax;      // the cluster's candidate range
  uint32_t digit, rem;
  uint32_t lmin, lmax;      // this CTA's
  uint32_t sel_cta, sel_before;
  uint32_t eq_total;        // keys == T in the whole row
  int last;
};

struct RowDesc {
  const float* row;
  int lo, hi;         // candidate positions [lo, hi)
  uint32_t need;      // keys to select among them
  int32_t* out;       // selected positions go to out[nsink ...]; sinks to out[0 .. nsink)
  int nsink;
  int l, h;
};

__device__ __forceinline__ RowDesc row_of(const TopkArgs& A, const EvictParams& P) {
  RowDesc d;
  if (A.mode == 0) {
    const int r = blockIdx.y;
    d.row = A.vals;
    d.lo = A.sinks + r * A.m;   // below N for every chunk r
    d.hi = static_cast<int>(min(static_cast<int64_t>(d.lo) + A.m, static_cast<int64_t>(A.N)));
    d.need = static_cast<uint32_t>((r == A.n_chunks - 1) ? A.nq_last : A.nq_full);
    d.out = A.sel + static_cast<int64_t>(r) * A.nq_full;
    d.nsink = 0;
    d.l = 0;
    d.h = r;
  } else {
    const int l = A.act[blockIdx.z], h = blockIdx.y;
    d.row = A.vals + (static_cast<int64_t>(l) * P.Hkv + h) * P.ld;
    d.lo = P.sinks;
    d.hi = max(P.n[l], P.sinks);
    d.need = static_cast<uint32_t>(P.k[l] - P.sinks);
    d.out = A.kept + P.out_off[l] + static_cast<int64_t>(h) * P.k[l];
    d.nsink = P.sinks;
    d.l = l;
    d.h = h;
  }
  return d;
}

template <bool MULTI>
__device__ __forceinline__ void csync(cg::cluster_group& cl) {
  if (MULTI)
    cl.sync();
  else
    __syncthreads();
}

// MSB-first radix select over the cluster's staged keys: the need-th
// largest key T (every key of the cluster lies in [kmin, kmax]) and how many
// keys == T are taken.  Digits of 8 bits below the common prefix of kmin and
// kmax; per-warp histograms, summed per CTA and then over the cluster in rank
// order through distributed shared memory, so every CTA finds the same digit.
// Requires 1 <= need < number of keys.
template <bool MULTI>
__device__ void radix_select(cg::cluster_group& cl, TopkShared& sm, const uint32_t* keys, int cnt, int C,
                             uint32_t need, uint32_t kmin, uint32_t kmax, uint32_t& T, uint32_t& eq_need) {
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint32_t diff = kmin ^ kmax;
  int hb = diff ? 32 - __clz(diff) : 0;           // bits below the common prefix
  uint32_t prefix = hb >= 32 ? 0u : (kmax & ~((1u << hb) - 1u));
  uint32_t rem = need;
  int par = 0;
  while (hb > 0) {
    const int lb = max(hb - 8, 0);
    const uint32_t pmask = hb >= 32 ? 0u : (~0u << hb);
    const uint32_t dmask = (1u << (hb - lb)) - 1u;
#pragma unroll
    for (int t = 0; t < 8; ++t) sm.whist[warp][lane * 8 + t] = 0u;
    __syncwarp();
    for (int j = tid; j < cnt; j += CT) {
      const uint32_t k = keys[j];
      if ((k & pmask) == prefix) atomicAdd(&sm.whist[warp][(k >> lb) & dmask], 1u);
    }
    __syncthreads();
    if (tid < 256) {
      uint32_t t = 0;
#pragma unroll
      for (int w = 0; w < CW; ++w) t += sm.whist[w][tid];
      sm.chist[par][tid] = t;
    }
    const uint32_t* H = sm.chist[par];
    if (MULTI) {
      cl.sync();
      if (tid < 256) {
        uint32_t t = 0;
        for (int r = 0; r < C; ++r) t += cl.map_shared_rank(sm.chist[par], r)[tid];
        sm.ghist[tid] = t;
      }
      H = sm.ghist;
    }
    __syncthreads();
    if (warp == 0) {
      // bins from the top: lane l covers bins 255-8l .. 248-8l
      uint32_t c[8], tot = 0;
#pragma unroll
      for (int t = 0; t < 8; ++t) {
        c[t] = H[255 - (lane * 8 + t)];
        tot += c[t];
      }
      uint32_t incl = tot;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const uint32_t v = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += v;
      }
      const uint32_t excl = incl - tot;
      if (excl < rem && incl >= rem) {
        uint32_t run = excl;
        for (int t = 0; t < 8; ++t) {
          if (run + c[t] >= rem) {
            sm.digit = 255u - (lane * 8 + t);
            sm.rem = rem - run;
            break;
          }
          run += c[t];
        }
      }
    }
    __syncthreads();
    prefix |= sm.digit << lb;
    rem = sm.rem;
    hb = lb;
    par ^= 1;
  }
  T = prefix;
  eq_need = rem;
}

// Copy the kept rows t in [t0, t1) of (l, h) from the source slab into the
// destination.  Row t's position is t below nsink (a sink), else spos[t -
// s0] when the positions are in shared memory (spos non-null), else out[t].
// K and V rows form one stream of 256-byte row copies, half a warp per row,
// eight in flight per half-warp.
__device__ void copy_rows(const EvictParams& P, const EvictCopy& X, int l, int h, const int32_t* out,
                          const int32_t* spos, int s0, int nsink, int t0, int t1) {
  const int slab = X.slab[l];
  const uint4* K = static_cast<const uint4*>(X.K[slab]);
  const uint4* V = static_cast<const uint4*>(X.V[slab]);
  const int32_t* pos = X.pos[slab];
  uint4* Kd = static_cast<uint4*>(X.Kd[slab]);
  uint4* Vd = static_cast<uint4*>(X.Vd[slab]);
  int32_t* posd = X.posd[slab];
  const int64_t lh = static_cast<int64_t>(l) * P.Hkv + h;
  const int64_t src_base = lh * X.src_ld;
  const int64_t dst_base = X.dst_ld >= 0 ? lh * X.dst_ld : P.out_off[l] + static_cast<int64_t>(h) * P.k[l];
  const int sub = threadIdx.x & 15, hw = threadIdx.x >> 4;
  constexpr int HW = CT / 16;
  constexpr int R = 8;
  const int nt = t1 - t0;
  const int total = V ? 2 * nt : nt;    // row copies: K rows, then V rows
  for (int ub = hw; ub < total; ub += HW * R) {
    int32_t src[R];
    uint4 val[R];
#pragma unroll
    for (int u = 0; u < R; ++u) {
      const int w = ub + u * HW;
      src[u] = -1;
      if (w < total) {
        const int t = t0 + (w < nt ? w : w - nt);
        src[u] = t < nsink ? t : (spos ? spos[t - s0] : out[t]);
        const uint4* from = w < nt ? K : V;
        val[u] = __ldg(from + (src_base + src[u]) * 16 + sub);
      }
    }
#pragma unroll
    for (int u = 0; u < R; ++u) {
      const int w = ub + u * HW;
      if (src[u] < 0) continue;
      const bool isK = w < nt;
      const int t = t0 + (isK ? w : w - nt);
      (isK ? Kd : Vd)[(dst_base + t) * 16 + sub] = val[u];
      if (isK && posd && sub == 0) posd[dst_base + t] = pos ? pos[src_base + src[u]] : src[u];
    }
  }
}

// Row moves of an in-place eviction: rows movers[i] -> holes[i] for i in
// [p0, p1) of (l, h), K and V (and positions) in slab 0.  Holes lie below the
// budget and movers at or above it, so no row is both read and written.
// K and V rows form one stream of 256-byte row copies, half a warp per row,
// eight in flight per half-warp.
__device__ void move_rows(const EvictCopy& X, int l, int64_t lh, const int32_t* holes, const int32_t* movers,
                          int p0, int p1) {
  uint4* K = static_cast<uint4*>(X.Kd[0]);
  uint4* V = static_cast<uint4*>(X.Vd[0]);
  int32_t* pos = X.posd[0];
  const int64_t base = lh * X.src_ld;
  // V rows of movers come from the block when it is given (row r is block
  // row r - blk_row0[l])
  const uint4* Vsrc = X.Vblk ? static_cast<const uint4*>(X.Vblk) : V;
  const int64_t vbase = X.Vblk ? lh * X.blk_len - X.blk_row0[l] : base;
  const int sub = threadIdx.x & 15, hw = threadIdx.x >> 4;
  constexpr int HW = CT / 16;
  constexpr int R = 8;
  const int np = p1 - p0;
  const int total = 2 * np;             // K rows, then V rows
  for (int ub = hw; ub < total; ub += HW * R) {
    int32_t src[R];
    uint4 val[R];
#pragma unroll
    for (int u = 0; u < R; ++u) {
      const int w = ub + u * HW;
      src[u] = -1;
      if (w < total) {
        src[u] = movers[p0 + (w < np ? w : w - np)];
        val[u] = w < np ? K[(base + src[u]) * 16 + sub] : Vsrc[(vbase + src[u]) * 16 + sub];
      }
    }
#pragma unroll
    for (int u = 0; u < R; ++u) {
      const int w = ub + u * HW;
      if (src[u] < 0) continue;
      const bool isK = w < np;
      const int dst = holes[p0 + (isK ? w : w - np)];
      (isK ? K : V)[(base + dst) * 16 + sub] = val[u];
      if (isK && sub == 0) pos[base + dst] = pos[base + src[u]];
    }
  }
}

// Eviction in place (mode 2): the kept rows of (l, h) end up in rows [0, k)
// of slab 0 in no particular order.  A kept row at or above k (a "mover")
// moves into an evicted row below k (a "hole"); the i-th hole in row order
// takes the i-th mover, and there are as many of each.  Rows carry their
// global position (X.pos[0]), and a tie at the threshold is decided by it,
// lower position first, as in the ascending layout where row order is
// position order.
template <bool MULTI>
__device__ void evict_in_place(cg::cluster_group& cl, TopkShared& sm, uint32_t* keys, int cnt, int C, int rank,
                               const RowDesc& R, const TopkArgs& A, const EvictParams& P, const EvictCopy& X,
                               uint32_t T, uint32_t eq_need, int c0, int wb0, int wb1) {
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint32_t lt = (1u << lane) - 1u;
  const int64_t lh = static_cast<int64_t>(R.l) * P.Hkv + R.h;
  // a. more keys == T than are kept: rank them by position.  New keys: every
  // key > T above every tie, ties ordered by lower position (all distinct),
  // the rest at 0; the need-th largest of them is the new threshold and it
  // has no ties.
  const int kb = P.k[R.l];
  if (sm.eq_total > eq_need) {
    const int32_t* pos = X.pos[0] + lh * X.src_ld + c0;
    for (int j = tid; j < cnt; j += CT) {
      const uint32_t k = keys[j];
      keys[j] = k > T ? 0xffffffffu : (k == T ? 0x80000000u - static_cast<uint32_t>(pos[j]) : 0u);
    }
    __syncthreads();
    uint32_t one;
    radix_select<MULTI>(cl, sm, keys, cnt, C, R.need, 0u, 0xffffffffu, T, one);
    // the holes and movers counted with the counts assumed every tie kept:
    // count them again
    uint32_t nh = 0, nm = 0;
    for (int jb = wb0; jb < wb1; jb += 32) {
      const int j = jb + lane;
      const bool in = j < wb1;
      const bool take = in && keys[j] >= T;
      nh += __popc(__ballot_sync(0xffffffffu, in && !take && c0 + j < kb));
      nm += __popc(__ballot_sync(0xffffffffu, take && c0 + j >= kb));
    }
    if (lane == 0) {
      sm.whol[warp] = nh;
      sm.wmov[warp] = nm;
    }
    __syncthreads();
    if (tid == 0) {
      uint32_t h = 0, m = 0;
      for (int w = 0; w < CW; ++w) {
        h += sm.whol[w];
        m += sm.wmov[w];
      }
      sm.xch[4] = h;
      sm.xch[5] = m;
    }
    csync<MULTI>(cl);
  }
  // every key >= T is kept now
  // b. ranks of the holes and movers across the row
  if (tid == 0) {
    uint32_t hb = 0, mb = 0, ht = 0, mt = 0;
    for (int r = 0; r < C; ++r) {
      const uint32_t* x = MULTI ? cl.map_shared_rank(sm.xch, r) : sm.xch;
      if (r < rank) {
        hb += x[4];
        mb += x[5];
      }
      ht += x[4];
      mt += x[5];
    }
    for (int w = 0; w < CW; ++w) {
      sm.wsel[w] = hb;
      sm.weqb[w] = mb;
      hb += sm.whol[w];
      mb += sm.wmov[w];
    }
    // equal by construction (exactly need keys are kept); only the pairs
    // both lists hold are moved
    sm.sel_cta = min(min(ht, mt), static_cast<uint32_t>(A.fill));
    if ((ht != mt || mt > static_cast<uint32_t>(A.fill)) && rank == 0 && A.status)
      record_status(A.status, DEV_BOUNDS);
  }
  __syncthreads();
  int32_t* holes = A.kept + lh * 2 * A.fill;
  int32_t* movers = holes + A.fill;
  {
    uint32_t hr = sm.wsel[warp], mr = sm.weqb[warp];
    for (int jb = wb0; jb < wb1; jb += 32) {
      const int j = jb + lane;
      const bool in = j < wb1;
      const bool take = in && keys[j] >= T;
      const bool ho = in && !take && c0 + j < kb;
      const bool mo = take && c0 + j >= kb;
      const uint32_t hm = __ballot_sync(0xffffffffu, ho);
      const uint32_t mm = __ballot_sync(0xffffffffu, mo);
      const uint32_t hi = hr + __popc(hm & lt), mi = mr + __popc(mm & lt);
      if (ho && hi < static_cast<uint32_t>(A.fill)) holes[hi] = c0 + j;
      if (mo && mi < static_cast<uint32_t>(A.fill)) movers[mi] = c0 + j;
      hr += __popc(hm);
      mr += __popc(mm);
    }
  }
  // the lists are complete (and no peer reads this CTA's shared memory
  // after this point)
  __threadfence();
  if (MULTI) cl.sync();
  else __syncthreads();
  // c. this CTA's share of the pairs
  const int np = static_cast<int>(sm.sel_cta);
  const int per = (np + C - 1) / C;
  const int p0 = min(rank * per, np), p1 = min(p0 + per, np);
  move_rows(X, R.l, lh, holes, movers, p0, p1);
}

// INPLACE: the in-place eviction (mode 2) only; a separate instance keeps
// its registers out of the other modes.
template <bool MULTI, bool INPLACE>
__global__ void __launch_bounds__(CT, 2)
    topk_cluster_kernel(const __grid_constant__ TopkArgs A, const __grid_constant__ EvictParams P,
                        const __grid_constant__ EvictCopy X) {
  extern __shared__ __align__(16) uint32_t keys[];
  __shared__ TopkShared sm;
  cg::cluster_group cl = cg::this_cluster();
  const int C = MULTI ? static_cast<int>(cl.num_blocks()) : 1;
  const int rank = MULTI ? static_cast<int>(cl.block_rank()) : 0;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint32_t lt = (1u << lane) - 1u;

  const RowDesc R = row_of(A, P);
  const int cand = max(R.hi - R.lo, 0);
  const int part = (cand + C - 1) / C;
  const int c0 = R.lo + min(rank * part, cand);
  const int cnt = max(min(part, R.hi - c0), 0);

  if (tid == 0) {
    sm.lmin = 0xffffffffu;
    sm.lmax = 0u;
  }
  __syncthreads();
  // ---- 1. stage the part as order keys (sixteen loads in flight per thread)
  {
    uint32_t mn = 0xffffffffu, mx = 0u;
    for (int j0 = 0; j0 < cnt; j0 += CT * 16) {
      float v[16];
#pragma unroll
      for (int u = 0; u < 16; ++u) {
        const int j = j0 + u * CT + tid;
        v[u] = j < cnt ? R.row[c0 + j] : 0.f;
      }
#pragma unroll
      for (int u = 0; u < 16; ++u) {
        const int j = j0 + u * CT + tid;
        if (j < cnt) {
          const uint32_t k = order_key(v[u]);
          keys[j] = k;
          mn = min(mn, k);
          mx = max(mx, k);
        }
      }
    }
    mn = __reduce_min_sync(0xffffffffu, mn);
    mx = __reduce_max_sync(0xffffffffu, mx);
    if (lane == 0) {
      atomicMin(&sm.lmin, mn);
      atomicMax(&sm.lmax, mx);
    }
  }
  __syncthreads();
  if (tid == 0) {
    sm.xch[0] = sm.lmin;
    sm.xch[1] = sm.lmax;
    if (A.mode == 1 && A.gmax && cnt > 0) atomicMax(&A.gmax[0], sm.lmax);
  }
  csync<MULTI>(cl);
  if (tid == 0) {
    uint32_t mn = 0xffffffffu, mx = 0u;
    for (int r = 0; r < C; ++r) {
      const uint32_t* x = MULTI ? cl.map_shared_rank(sm.xch, r) : sm.xch;
      mn = min(mn, x[0]);
      mx = max(mx, x[1]);
    }
    sm.kmin = mn;
    sm.kmax = mx;
  }
  __syncthreads();

  // ---- 2. threshold T and the number of keys == T to take
  uint32_t T, eq_need;
  if (R.need == 0) {
    T = 0xffffffffu;          // no key reaches it (+inf maps to 0xff800000)
    eq_need = 0;
  } else if (R.need >= static_cast<uint32_t>(cand)) {
    T = 0u;                   // every key is >= 0: keep all
    eq_need = 0xffffffffu;
  } else {
    radix_select<MULTI>(cl, sm, keys, cnt, C, R.need, sm.kmin, sm.kmax, T, eq_need);
  }

  // ---- 3. counts per warp block (contiguous, whole multiples of 32 keys)
  const int WB = ((cnt + CW - 1) / CW + 31) & ~31;
  const int wb0 = min(warp * WB, cnt), wb1 = min(wb0 + WB, cnt);
  {
    // the in-place eviction also counts its holes and movers, assuming every
    // key == T is kept (true unless more keys tie at T than are kept)
    const int kb = INPLACE ? P.k[R.l] : 0;
    uint32_t g = 0, e = 0, nh = 0, nm = 0;
    for (int j = wb0 + lane; j < wb1; j += 32) {
      const uint32_t k = keys[j];
      g += k > T;
      e += k == T;
      if (INPLACE) {
        nh += (k < T && c0 + j < kb) ? 1u : 0u;
        nm += (k >= T && c0 + j >= kb) ? 1u : 0u;
      }
    }
    g = __reduce_add_sync(0xffffffffu, g);
    e = __reduce_add_sync(0xffffffffu, e);
    if (INPLACE) {
      nh = __reduce_add_sync(0xffffffffu, nh);
      nm = __reduce_add_sync(0xffffffffu, nm);
    }
    if (lane == 0) {
      sm.wgt[warp] = g;
      sm.weq[warp] = e;
      if (INPLACE) {
        sm.whol[warp] = nh;
        sm.wmov[warp] = nm;
      }
    }
  }
  __syncthreads();
  if (tid == 0) {
    uint32_t g = 0, e = 0, h = 0, m = 0;
    for (int w = 0; w < CW; ++w) {
      g += sm.wgt[w];
      e += sm.weq[w];
      if (INPLACE) {
        h += sm.whol[w];
        m += sm.wmov[w];
      }
    }
    sm.xch[2] = g;
    sm.xch[3] = e;
    sm.xch[4] = h;
    sm.xch[5] = m;
  }
  csync<MULTI>(cl);
  if (tid == 0) {
    // keys == T are taken in position order across the cluster, then the CTA
    uint32_t sel_before = 0, eq_before = 0, eq_total = 0;
    for (int r = 0; r < C; ++r) {
      const uint32_t* x = MULTI ? cl.map_shared_rank(sm.xch, r) : sm.xch;
      eq_total += x[3];
      if (r >= rank) continue;
      const uint32_t take = eq_need > eq_before ? min(eq_need - eq_before, x[3]) : 0u;
      sel_before += x[2] + take;
      eq_before += x[3];
    }
    sm.eq_total = eq_total;
    uint32_t s = sel_before;
    for (int w = 0; w < CW; ++w) {
      sm.wsel[w] = s;
      sm.weqb[w] = eq_before;
      const uint32_t take = eq_need > eq_before ? min(eq_need - eq_before, sm.weq[w]) : 0u;
      s += sm.wgt[w] + take;
      eq_before += sm.weq[w];
    }
    sm.sel_before = sel_before;
    sm.sel_cta = s - sel_before;
  }
  __syncthreads();
  if (INPLACE) {
    evict_in_place<MULTI>(cl, sm, keys, cnt, C, rank, R, A, P, X, T, eq_need, c0, wb0, wb1);
    return;
  }

  // ---- 4. ordered emit; for the fused copy the CTA's positions are also
  // kept in shared memory (in the histogram area, free by now) when they fit
  constexpr int kSposCap = CW * 256;
  static_assert(kSposCap >= kFusedCopyRows, "a fused copy keeps its positions in shared memory");
  int32_t* spos = (A.copy && sm.sel_cta <= static_cast<uint32_t>(kSposCap))
                      ? reinterpret_cast<int32_t*>(&sm.whist[0][0]) : nullptr;
  {
    uint32_t sel_run = sm.wsel[warp], eq_run = sm.weqb[warp];
    int32_t* out = R.out + R.nsink;
    for (int jb = wb0; jb < wb1; jb += 32) {
      const int j = jb + lane;
      const bool in = j < wb1;
      const uint32_t k = in ? keys[j] : 0u;
      const bool gt = in && k > T;
      const bool eq = in && k == T;
      const uint32_t em = __ballot_sync(0xffffffffu, eq);
      const bool take = gt || (eq && eq_run + __popc(em & lt) < eq_need);
      const uint32_t tm = __ballot_sync(0xffffffffu, take);
      if (take) {
        const uint32_t slot = sel_run + __popc(tm & lt);
        out[slot] = c0 + j;
        if (spos) spos[slot - sm.sel_before] = c0 + j;
      }
      sel_run += __popc(tm);
      eq_run += __popc(em);
    }
    if (rank == 0)
      for (int s = tid; s < R.nsink; s += CT) R.out[s] = s;
  }
  // no CTA leaves (or reuses its shared memory) while a peer may still read it
  if (MULTI) cl.sync();
  else __syncthreads();

  if (A.mode != 1) return;
  // ---- 5. fused compaction of this CTA's kept rows (and the sinks, rank 0)
  if (A.copy) {
    const int t0 = rank == 0 ? 0 : R.nsink + static_cast<int>(sm.sel_before);
    const int t1 = R.nsink + static_cast<int>(sm.sel_before + sm.sel_cta);
    copy_rows(P, X, R.l, R.h, R.out, spos, R.nsink + static_cast<int>(sm.sel_before), R.nsink, t0, t1);
  }
  // ---- 6. the last CTA to finish pins every sink to the global max
  if (A.gmax) {
    if (tid == 0) {
      __threadfence();
      const uint32_t prev = atomicAdd(&A.gmax[1], 1u);
      sm.last = prev + 1 == static_cast<uint32_t>(A.total_ctas);
    }
    __syncthreads();
    if (sm.last) {
      __threadfence();
      const float v = key_value(atomicOr(&A.gmax[0], 0u));
      const int S = P.sinks;
      const int per = P.Hkv * S;
      for (int a = 0; a < static_cast<int>(gridDim.z); ++a) {
        const int l = A.act[a];
        float* base = A.score + static_cast<int64_t>(l) * P.Hkv * P.ld;
        for (int i = tid; i < per; i += CT) {
          const int h = i / S, s = i - h * S;
          if (s < P.n[l]) base[static_cast<int64_t>(h) * P.ld + s] = v;
        }
      }
    }
  }
}

// ====================================================================
// Global-memory radix kernels: rows longer than kMaxParts shared-memory
// parts (and more chunks than a grid dimension holds).  One 1024-thread CTA
// per row makes four 8-bit digit passes and one ordered pass over the row
// in global memory.
// ====================================================================
constexpr int THREADS = 1024;
constexpr int WARPS = THREADS / 32;

struct SelectSmem {
  uint32_t hist[256];
  uint32_t warp_cnt[WARPS];
  uint32_t warp_eq[WARPS];
  uint32_t prefix, remaining, digit_out;
  uint32_t base_sel, base_eq;
  uint32_t maxkey;
};

// Find the n-th largest key of vals[lo, hi) (n >= 1, n <= hi - lo).
// Returns T; *cnt_gt receives how many keys are strictly greater.
__device__ uint32_t radix_threshold(const float* __restrict__ vals, int64_t lo, int64_t hi, uint32_t n,
                                    SelectSmem& sm, uint32_t* cnt_gt, bool want_max) {
  uint32_t prefix = 0, mask = 0, remaining = n;
  uint32_t localmax = 0;
  for (int shift = 24; shift >= 0; shift -= 8) {
    for (int b = threadIdx.x; b < 256; b += THREADS) sm.hist[b] = 0;
    __syncthreads();
    for (int64_t i = lo + threadIdx.x; i < hi; i += THREADS) {
      const uint32_t k = order_key(vals[i]);
      if (want_max && shift == 24) localmax = max(localmax, k);
      if ((k & mask) == prefix) atomicAdd(&sm.hist[(k >> shift) & 255u], 1u);
    }
    __syncthreads();
    if (threadIdx.x < 32) {
      uint32_t c[8], tot = 0;
#pragma unroll
      for (int t = 0; t < 8; ++t) {
        c[t] = sm.hist[255 - (threadIdx.x * 8 + t)];
        tot += c[t];
      }
      uint32_t incl = tot;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const uint32_t v = __shfl_up_sync(0xffffffffu, incl, o);
        if (threadIdx.x >= o) incl += v;
      }
      const uint32_t excl = incl - tot;
      if (excl < remaining && incl >= remaining) {
        uint32_t run = excl;
        for (int t = 0; t < 8; ++t) {
          if (run + c[t] >= remaining) {
            sm.digit_out = 255u - (threadIdx.x * 8 + t);
            sm.remaining = remaining - run;
            break;
          }
          run += c[t];
        }
      }
    }
    __syncthreads();
    const uint32_t dgt = sm.digit_out;
    remaining = sm.remaining;
    prefix |= dgt << shift;
    mask |= 255u << shift;
    __syncthreads();
  }
  if (want_max) {
    for (int o = 16; o > 0; o >>= 1) localmax = max(localmax, __shfl_xor_sync(0xffffffffu, localmax, o));
    if ((threadIdx.x & 31) == 0) atomicMax(&sm.maxkey, localmax);
  }
  *cnt_gt = n - remaining;
  return prefix;
}

// Writes, in ascending position order, every position of [lo, hi) whose key
// is > T plus the first `need_eq` positions whose key == T.
__device__ void emit_selected(const float* __restrict__ vals, int64_t lo, int64_t hi, uint32_t T, uint32_t need_eq,
                              int32_t* __restrict__ out, SelectSmem& sm) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    sm.base_sel = 0;
    sm.base_eq = 0;
  }
  __syncthreads();
  for (int64_t b0 = lo; b0 < hi; b0 += THREADS) {
    const int64_t i = b0 + threadIdx.x;
    uint32_t k = 0;
    const bool in = i < hi;
    if (in) k = order_key(vals[i]);
    const bool gt = in && k > T;
    const bool eq = in && k == T;
    const uint32_t eqmask = __ballot_sync(0xffffffffu, eq);
    if (lane == 0) sm.warp_eq[warp] = __popc(eqmask);
    __syncthreads();
    uint32_t eq_before = sm.base_eq;
    for (int w = 0; w < warp; ++w) eq_before += sm.warp_eq[w];
    eq_before += __popc(eqmask & ((1u << lane) - 1u));
    const bool take = gt || (eq && eq_before < need_eq);
    const uint32_t tmask = __ballot_sync(0xffffffffu, take);
    if (lane == 0) sm.warp_cnt[warp] = __popc(tmask);
    __syncthreads();
    uint32_t sel_before = sm.base_sel;
    for (int w = 0; w < warp; ++w) sel_before += sm.warp_cnt[w];
    sel_before += __popc(tmask & ((1u << lane) - 1u));
    if (take) out[sel_before] = static_cast<int32_t>(i);
    __syncthreads();
    if (threadIdx.x == 0) {
      uint32_t a = 0, e = 0;
      for (int w = 0; w < WARPS; ++w) {
        a += sm.warp_cnt[w];
        e += sm.warp_eq[w];
      }
      sm.base_sel += a;
      sm.base_eq += e;
    }
    __syncthreads();
  }
}

struct SelParams {
  int N, sinks, m, n_chunks, nq_full, nq_last;
};

__global__ void __launch_bounds__(THREADS) select_kernel(const float* __restrict__ p, SelParams P,
                                                         int32_t* __restrict__ sel) {
  __shared__ SelectSmem sm;
  const int r = blockIdx.x;
  const int64_t lo = P.sinks + static_cast<int64_t>(r) * P.m;
  const int64_t hi = min(lo + P.m, static_cast<int64_t>(P.N));
  const uint32_t n = (r == P.n_chunks - 1) ? P.nq_last : P.nq_full;
  int32_t* out = sel + static_cast<int64_t>(r) * P.nq_full;
  uint32_t gt;
  const uint32_t T = radix_threshold(p, lo, hi, n, sm, &gt, false);
  emit_selected(p, lo, hi, T, n - gt, out, sm);
}

__global__ void __launch_bounds__(THREADS) evict_kernel(float* __restrict__ score, const __grid_constant__ EvictParams P,
                                                        int32_t* __restrict__ kept, uint32_t* __restrict__ gmax) {
  __shared__ SelectSmem sm;
  const int l = blockIdx.y, h = blockIdx.x;
  if (!P.active[l]) return;
  const int n = P.n[l];
  const int k = P.k[l];
  const float* row = score + (static_cast<int64_t>(l) * P.Hkv + h) * P.ld;
  int32_t* out = kept + P.out_off[l] + static_cast<int64_t>(h) * k;
  if (threadIdx.x == 0) sm.maxkey = 0;
  for (int i = threadIdx.x; i < P.sinks; i += THREADS) out[i] = i;
  __syncthreads();
  const uint32_t need = static_cast<uint32_t>(k - P.sinks);
  const int lo = P.sinks;
  if (n > lo) {
    if (need > 0) {
      uint32_t gt;
      const uint32_t T = radix_threshold(row, lo, n, need, sm, &gt, true);
      emit_selected(row, lo, n, T, need - gt, out + P.sinks, sm);
    } else {
      uint32_t localmax = 0;
      for (int i = lo + threadIdx.x; i < n; i += THREADS) localmax = max(localmax, order_key(row[i]));
      for (int o = 16; o > 0; o >>= 1) localmax = max(localmax, __shfl_xor_sync(0xffffffffu, localmax, o));
      if ((threadIdx.x & 31) == 0) atomicMax(&sm.maxkey, localmax);
    }
    __syncthreads();
    if (threadIdx.x == 0 && gmax) atomicMax(gmax, sm.maxkey);
  }
}

// score[l][h][s] = max for s < sinks (every active layer).
__global__ void pin_kernel(float* __restrict__ score, const __grid_constant__ EvictParams P,
                           const uint32_t* __restrict__ gmax) {
  const int l = blockIdx.y, h = blockIdx.x;
  if (!P.active[l]) return;
  const float v = key_value(*gmax);
  float* row = score + (static_cast<int64_t>(l) * P.Hkv + h) * P.ld;
  for (int i = threadIdx.x; i < P.sinks && i < P.n[l]; i += blockDim.x) row[i] = v;
}

// Keys per CTA and CTAs per row for rows of up to `len` candidates, or
// false when a row needs more than kMaxParts shared-memory parts.
bool plan_parts(int64_t len, int* parts, int* part_keys) {
  if (len <= 0) {
    *parts = 1;
    *part_keys = 4;
    return true;
  }
  int64_t c = (len + kPartKeys - 1) / kPartKeys;
  int64_t pk = kPartKeys;
  if (c > kMaxParts) {
    c = kMaxParts;
    pk = ((len + kMaxParts - 1) / kMaxParts + 3) & ~int64_t(3);
    if (pk > kPartKeysMax) return false;
  } else {
    pk = ((len + c - 1) / c + 3) & ~int64_t(3);
  }
  *parts = static_cast<int>(c);
  *part_keys = static_cast<int>(pk);
  return true;
}

// Tiled compaction of the kept rows of every active layer, one launch.
cudaError_t compact_after(const EvictParams& ep, const int32_t* kept, const EvictCopy& copy, cudaStream_t st) {
  CompactParams cp;
  memset(&cp, 0, sizeof(cp));
  cp.L = ep.L;
  cp.Hkv = ep.Hkv;
  cp.src_ld = copy.src_ld;
  cp.dst_ld = copy.dst_ld;
  for (int l = 0; l < ep.L; ++l) {
    if (!ep.active[l]) continue;
    cp.n_src[l] = ep.n[l];
    cp.k[l] = ep.k[l];
    cp.idx_off[l] = ep.out_off[l];
    cp.dst_off[l] = ep.out_off[l];
    cp.active[l] = 1;
  }
  return launch_compact_slabs(kept, copy, cp, st);
}

cudaError_t launch_cluster(const TopkArgs& A, const EvictParams& P, const EvictCopy& X, int parts, int part_keys,
                           dim3 grid, cudaStream_t st) {
  const size_t smem = static_cast<size_t>(part_keys) * sizeof(uint32_t);
  cudaLaunchConfig_t cfg;
  memset(&cfg, 0, sizeof(cfg));
  cfg.gridDim = grid;
  cfg.blockDim = dim3(CT);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = parts;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  // The dynamic shared-memory limit is raised once per device (for the
  // largest part size), not on every launch.  No carveout preference: the
  // driver's choice already fits two CTAs of a 64 KB part per SM, and the L1
  // it leaves measured 3 us faster per 16K eviction than the largest
  // shared-memory carveout.
  static int attr_done[64][4];
  int d = 0;
  if (cudaGetDevice(&d) != cudaSuccess || d < 0 || d >= 64) return cudaErrorInvalidDevice;
  const int variant = (parts > 1 ? 1 : 0) + (A.mode == 2 ? 2 : 0);
  void (*const fns[4])(TopkArgs, EvictParams, EvictCopy) = {
      topk_cluster_kernel<false, false>, topk_cluster_kernel<true, false>, topk_cluster_kernel<false, true>,
      topk_cluster_kernel<true, true>};
  if (!attr_done[d][variant]) {
    const void* fn = reinterpret_cast<const void*>(fns[variant]);
    const cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                               static_cast<int>(kPartKeysMax * sizeof(uint32_t)));
    if (e != cudaSuccess) return e;
    attr_done[d][variant] = 1;
  }
  return cudaLaunchKernelEx(&cfg, fns[variant], A, P, X);
}

// Largest order key over the non-sink entries of LH rows of N scores.
__global__ void score_max_kernel(const float* __restrict__ score, int LH, int N, int sinks, uint32_t* key_word) {
  const int64_t total = static_cast<int64_t>(LH) * N;
  uint32_t m = 0;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < total;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x)
    if (i % N >= sinks) m = max(m, order_key(score[i]));
  m = __reduce_max_sync(0xffffffffu, m);
  if ((threadIdx.x & 31) == 0) atomicMax(key_word, m);
}
__global__ void key_to_float_kernel(const uint32_t* key_word, float* out) { *out = key_value(*key_word); }
__global__ void pin_value_kernel(float* __restrict__ score, int LH, int N, int sinks, const float* __restrict__ value) {
  const float v = *value;
  const int64_t total = static_cast<int64_t>(LH) * sinks;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < total;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x)
    score[(i / sinks) * N + i % sinks] = v;
}

}  // namespace

cudaError_t launch_score_max(const float* score, int LH, int N, int sinks, uint32_t* key_word, float* max_out,
                             cudaStream_t st) {
  cudaError_t e = cudaMemsetAsync(key_word, 0, sizeof(uint32_t), st);
  if (e != cudaSuccess) return e;
  ProfScope ps("score_max", st);
  score_max_kernel<<<2 * num_sms(), 256, 0, st>>>(score, LH, N, sinks, key_word);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  key_to_float_kernel<<<1, 1, 0, st>>>(key_word, max_out);
  return cudaGetLastError();
}

cudaError_t launch_pin_value(float* score, int LH, int N, int sinks, const float* value, cudaStream_t st) {
  if (sinks <= 0) return cudaSuccess;
  ProfScope ps("pin_sinks", st);
  pin_value_kernel<<<std::max(1, std::min(2 * num_sms(), (LH * sinks + 255) / 256)), 256, 0, st>>>(score, LH, N,
                                                                                                  sinks, value);
  return cudaGetLastError();
}

cudaError_t launch_select(const float* p, int N, int sinks, const ChunkPlan& plan, double rho, int32_t* sel,
                          cudaStream_t st) {
  (void)rho;
  int parts = 1, part_keys = 4;
  const int64_t longest = std::min<int64_t>(plan.m, static_cast<int64_t>(N) - sinks);
  const bool fits = plan.n_chunks <= 65535 && plan_parts(longest, &parts, &part_keys);
  ProfScope ps("select_topk", st);
  if (!fits) {
    SelParams sp{N, sinks, plan.m, plan.n_chunks, plan.nq_full, plan.nq_last};
    select_kernel<<<plan.n_chunks, THREADS, 0, st>>>(p, sp, sel);
    return cudaGetLastError();
  }
  TopkArgs A;
  memset(&A, 0, sizeof(A));
  A.mode = 0;
  A.vals = p;
  A.N = N;
  A.sinks = sinks;
  A.m = plan.m;
  A.n_chunks = plan.n_chunks;
  A.nq_full = plan.nq_full;
  A.nq_last = plan.nq_last;
  A.sel = sel;
  EvictParams P;
  memset(&P, 0, sizeof(P));
  EvictCopy X;
  memset(&X, 0, sizeof(X));
  cudaError_t e = launch_cluster(A, P, X, parts, part_keys, dim3(parts, plan.n_chunks, 1), st);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

cudaError_t launch_evict(float* score, const EvictParams& ep, int32_t* kept, uint32_t* gmax_word, bool pin,
                         const EvictCopy* copy, cudaStream_t st) {
  const bool want_pin = pin && gmax_word;
  if (want_pin) {
    cudaError_t e = cudaMemsetAsync(gmax_word, 0, 2 * sizeof(uint32_t), st);
    if (e != cudaSuccess) return e;
  }
  TopkArgs A;
  memset(&A, 0, sizeof(A));
  int n_act = 0;
  int64_t longest = 0;
  for (int l = 0; l < ep.L; ++l) {
    if (!ep.active[l]) continue;
    A.act[n_act++] = l;
    longest = std::max<int64_t>(longest, static_cast<int64_t>(ep.n[l]) - ep.sinks);
  }
  if (n_act == 0) return cudaSuccess;
  int kmax = 0;
  for (int a = 0; a < n_act; ++a) kmax = std::max(kmax, ep.k[A.act[a]]);
  const bool fuse = copy != nullptr && kmax <= kFusedCopyRows;
  int parts = 1, part_keys = 4;
  if (ep.Hkv <= 65535 && plan_parts(longest, &parts, &part_keys)) {
    A.mode = 1;
    A.vals = score;
    A.score = score;
    A.kept = kept;
    A.gmax = want_pin ? gmax_word : nullptr;
    A.total_ctas = parts * ep.Hkv * n_act;
    A.copy = fuse;
    EvictCopy X;
    if (copy)
      X = *copy;
    else
      memset(&X, 0, sizeof(X));
    {
      ProfScope ps(fuse ? "evict_compact" : "evict_topk", st);
      cudaError_t e = launch_cluster(A, ep, X, parts, part_keys, dim3(parts, ep.Hkv, n_act), st);
      if (e != cudaSuccess) return e;
      e = cudaGetLastError();
      if (e != cudaSuccess) return e;
    }
    if (!copy || fuse) return cudaSuccess;
    return compact_after(ep, kept, *copy, st);
  }
  // rows too long for the shared-memory parts
  dim3 grid(ep.Hkv, ep.L);
  {
    ProfScope ps("evict_topk", st);
    evict_kernel<<<grid, THREADS, 0, st>>>(score, ep, kept, want_pin ? gmax_word : nullptr);
  }
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  if (want_pin) {
    ProfScope ps("pin_sinks", st);
    pin_kernel<<<grid, 32, 0, st>>>(score, ep, gmax_word);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  if (!copy) return cudaSuccess;
  return compact_after(ep, kept, *copy, st);
}


cudaError_t launch_evict_in_place(const float* score, const EvictParams& ep, int32_t* lists, int list_stride,
                                  const EvictCopy& copy, cudaStream_t st) {
  TopkArgs A;
  memset(&A, 0, sizeof(A));
  int n_act = 0;
  int64_t longest = 0;
  for (int l = 0; l < ep.L; ++l) {
    if (!ep.active[l]) continue;
    A.act[n_act++] = l;
    longest = std::max<int64_t>(longest, static_cast<int64_t>(ep.n[l]) - ep.sinks);
  }
  if (n_act == 0) return cudaSuccess;
  int parts = 1, part_keys = 4;
  if (ep.Hkv > 65535 || !plan_parts(longest, &parts, &part_keys)) return cudaErrorInvalidValue;
  A.mode = 2;
  A.vals = score;
  A.kept = lists;
  A.fill = list_stride;
  A.status = status_word();
  A.total_ctas = parts * ep.Hkv * n_act;
  ProfScope ps("evict_in_place", st);
  cudaError_t e = launch_cluster(A, ep, copy, parts, part_keys, dim3(parts, ep.Hkv, n_act), st);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace kvc
