// Reconstruction scoring (KV² page, "무엇과 다른가"): the selected tokens are
// appended after the cache and attend causally over the whole cache; the
// score of a cache position of chunk C_r is the max, over the chunk's
// reconstruction queries and over the query heads sharing the KV head, of
// the softmax attention it receives.
//
// Two tensor-core passes per (layer, KV head), both on one warp-specialised
// skeleton (warp 0: TMA producer, warp 1: tcgen05.mma issuer and TMEM owner,
// warps 2-9: two consumer warpgroups):
//
//   pass 1 (row LSE)   A = 2 tiles of 128 reconstruction-query rows, B =
//                      streamed 128-key tiles of the cache, then the chunk's
//                      appended keys under the causal mask.  Each consumer
//                      thread owns one query row (one TMEM lane) and keeps an
//                      online max / sum of 2^x, ending with
//                      lse2 = max + log2(sum) (log2 units).
//   pass 2 (column max) A = 2 tiles of 128 cache keys of one chunk, B = the
//                      chunk's query rows.  Each consumer thread owns one key
//                      (TMEM lane) and folds max_j (x_ij - lse2_j) over every
//                      query column; exp2 is monotone, so one exp2 per key
//                      gives the max attention.  One store per position.
//
// Query rows are laid out per (layer, KV head) in a "row space": chunk r
// occupies rows [r*CR, r*CR + G*nq_r) ordered (query head g, query j), with
// CR = G*nq_full rounded up to 128 so that no 128-row tile straddles chunks.
// A gather kernel fills it (and the appended keys) from the query pool.
#include <cuda_bf16.h>

#include <cmath>
#include <cstring>

#include "kvc_internal.h"
#include "kvc_ptx.cuh"

namespace kvc {
namespace {

constexpr int TILE_ROWS = 128;                 // rows of every A and B tile
constexpr int TILE_BYTES = TILE_ROWS * 256;    // 128 rows x 128 bf16
constexpr int HALF_BYTES = TILE_BYTES / 2;     // one 64-column swizzled half
constexpr int KSTAGES = 3;                     // B-tile ring depth
constexpr int NUM_THREADS = 320;               // 10 warps
constexpr uint32_t TMEM_COLS = 512;            // 2 buffers x 2 accumulators x 128 columns
constexpr int SMEM_TILES = 4 + KSTAGES;        // A[2][2] + B ring
constexpr int SMEM_BYTES = 1024 + SMEM_TILES * TILE_BYTES + 256;

struct KParams {
  int Hkv, Hq, G, sinks;
  int n_active;
  int32_t layer[kMaxLayers];
  int32_t n[kMaxLayers];
  int32_t m[kMaxLayers];
  int32_t n_chunks[kMaxLayers];
  int32_t last_len[kMaxLayers];
  int32_t slab[kMaxLayers];
  int32_t unit_off[kMaxLayers + 1];   // pass-2 unit prefix over active layers
  int64_t ldK;
  int32_t nq_full, nq_last, Q;
  int32_t CR, Rpad;                   // row-space chunk stride and rows per (l, h)
  int32_t ldApp;                      // appended-key rows per (l, h)
  int32_t pairs1;                     // pass-1 units per (l, h): ceil(Rpad / 256)
  int n_units;
  float scale_log2;                   // log2(e) / sqrt(d)
  float* lse2;
  float* lse_out;
  float* score;
  int64_t ldS;
  int* status;
  uint64_t limit_ns;
};

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
__device__ __forceinline__ float lg2(float x) {
  float y;
  asm("lg2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ int nq_of(const KParams& P, int ai, int r) {
  return (r == P.n_chunks[ai] - 1) ? P.nq_last : P.nq_full;
}

// ----------------------------------------------------------------- units
struct Unit {
  int ai, layer, h, lh, slab, n;
  int has1;        // second A tile present
  // pass 1
  int R0, R1;      // row-space range [R0, R1] of the unit (inclusive)
  int ra, rb;      // chunk range touching the unit
  int nK;          // cache-key tiles
  // pass 2
  int r, lo, hi, key0;
  int nT;          // B tiles of the unit
};

template <int PASS>
__device__ __forceinline__ bool chunk_has_rows(const KParams& P, int ai, int r, int R0, int R1) {
  const int a = r * P.CR, b = r * P.CR + P.G * nq_of(P, ai, r) - 1;
  return a <= R1 && b >= R0;
}

template <int PASS>
__device__ Unit decode_unit(const KParams& P, int u) {
  Unit U;
  if (PASS == 1) {
    const int per_layer = P.Hkv * P.pairs1;
    U.ai = u / per_layer;
    const int rem = u - U.ai * per_layer;
    U.h = rem / P.pairs1;
    const int pp = rem - U.h * P.pairs1;
    U.layer = P.layer[U.ai];
    U.lh = U.layer * P.Hkv + U.h;
    U.slab = P.slab[U.ai];
    U.n = P.n[U.ai];
    U.R0 = pp * 2 * TILE_ROWS;
    U.R1 = min(U.R0 + 2 * TILE_ROWS, P.Rpad) - 1;
    U.has1 = (U.R0 + TILE_ROWS) < P.Rpad;
    const int nc = P.n_chunks[U.ai];
    U.ra = min(U.R0 / P.CR, nc - 1);
    U.rb = min(U.R1 / P.CR, nc - 1);
    U.nK = (U.n + TILE_ROWS - 1) / TILE_ROWS;
    int nt = U.nK;
    for (int r = U.ra; r <= U.rb; ++r)
      if (chunk_has_rows<1>(P, U.ai, r, U.R0, U.R1)) nt += (nq_of(P, U.ai, r) + TILE_ROWS - 1) / TILE_ROWS;
    U.nT = nt;
    U.r = U.lo = U.hi = U.key0 = 0;
  } else {
    int ai = 0;
    while (ai + 1 < P.n_active && u >= P.unit_off[ai + 1]) ++ai;
    U.ai = ai;
    U.layer = P.layer[ai];
    U.slab = P.slab[ai];
    U.n = P.n[ai];
    const int m = P.m[ai], nc = P.n_chunks[ai];
    const int pf = (m + 2 * TILE_ROWS - 1) / (2 * TILE_ROWS);
    const int pl = (P.last_len[ai] + 2 * TILE_ROWS - 1) / (2 * TILE_ROWS);
    const int per_head = (nc - 1) * pf + pl;
    const int rem = u - P.unit_off[ai];
    U.h = rem / per_head;
    const int q = rem - U.h * per_head;
    U.lh = U.layer * P.Hkv + U.h;
    int r, kp;
    if (q < (nc - 1) * pf) {
      r = q / pf;
      kp = q - r * pf;
    } else {
      r = nc - 1;
      kp = q - (nc - 1) * pf;
    }
    U.r = r;
    U.lo = P.sinks + r * m;
    U.hi = min(U.lo + m, U.n);
    U.key0 = U.lo + kp * 2 * TILE_ROWS;
    U.has1 = (U.key0 + TILE_ROWS) < U.hi;
    U.nT = (P.G * nq_of(P, ai, r) + TILE_ROWS - 1) / TILE_ROWS;
    U.R0 = U.R1 = U.ra = U.rb = U.nK = 0;
  }
  return U;
}

// Pass-1 B tile i of a unit: kind 0 = cache keys (t0 = first key), kind 1 =
// appended keys of chunk `chunk` (t0 = first appended index).
struct TileRef {
  int kind, t0, chunk;
};
__device__ __forceinline__ TileRef tile_at1(const KParams& P, const Unit& U, int i) {
  TileRef t;
  if (i < U.nK) {
    t.kind = 0;
    t.t0 = i * TILE_ROWS;
    t.chunk = -1;
    return t;
  }
  i -= U.nK;
  for (int r = U.ra; r <= U.rb; ++r) {
    if (!chunk_has_rows<1>(P, U.ai, r, U.R0, U.R1)) continue;
    const int na = (nq_of(P, U.ai, r) + TILE_ROWS - 1) / TILE_ROWS;
    if (i < na) {
      t.kind = 1;
      t.t0 = i * TILE_ROWS;
      t.chunk = r;
      return t;
    }
    i -= na;
  }
  t.kind = 1;
  t.t0 = 0;
  t.chunk = -2;  // unreachable for consistent callers
  return t;
}

// ----------------------------------------------------------------- kernel
struct __align__(8) Bars {
  uint64_t a_full[2], a_empty[2];
  uint64_t b_full[KSTAGES], b_empty[KSTAGES];
  uint64_t d_full[2], d_empty[2];
  uint64_t drain;
  uint32_t tmem_base;
  int abort_flag;
};

template <int PASS>
__global__ void __launch_bounds__(NUM_THREADS, 1)
    recon_kernel(const __grid_constant__ CUtensorMap tmQg, const __grid_constant__ CUtensorMap tmK0,
                 const __grid_constant__ CUtensorMap tmK1, const __grid_constant__ CUtensorMap tmApp,
                 const __grid_constant__ KParams P) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sA = smem;                              // [2 buffers][2 tiles]
  uint8_t* sB = smem + 4 * TILE_BYTES;             // [KSTAGES]
  Bars* bars = reinterpret_cast<Bars*>(smem + SMEM_TILES * TILE_BYTES);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int i = 0; i < 2; ++i) {
      mbar_init(&bars->a_full[i], 1);
      mbar_init(&bars->a_empty[i], 1);
      mbar_init(&bars->d_full[i], 1);
      mbar_init(&bars->d_empty[i], 8);
    }
    for (int i = 0; i < KSTAGES; ++i) {
      mbar_init(&bars->b_full[i], 1);
      mbar_init(&bars->b_empty[i], 1);
    }
    mbar_init(&bars->drain, 1);
    bars->abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 1) {
    tmem_alloc(&bars->tmem_base, TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = bars->tmem_base;
  volatile int* abort_flag = &bars->abort_flag;
  auto fail = [&](int where) {
    *abort_flag = 1;
    record_status(P.status, DEV_TIMEOUT);
    (void)where;
  };

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      tma_prefetch_desc(&tmQg);
      tma_prefetch_desc(&tmK0);
      tma_prefetch_desc(&tmK1);
      tma_prefetch_desc(&tmApp);
      int s = 0, ab = 0;
      uint32_t bph = 0, aph = 0;
      int issued_b[KSTAGES] = {};
      int issued_a[2] = {0, 0};
      for (int u = blockIdx.x; u < P.n_units && !*abort_flag; u += gridDim.x) {
        const Unit U = decode_unit<PASS>(P, u);
        // A tiles
        if (!mbar_wait(&bars->a_empty[ab], aph ^ 1, P.limit_ns)) { fail(1); break; }
        const uint32_t abytes = (1 + U.has1) * TILE_BYTES;
        mbar_arrive_expect_tx(&bars->a_full[ab], abytes);
        for (int t = 0; t <= U.has1; ++t) {
          uint8_t* dst = sA + (ab * 2 + t) * TILE_BYTES;
          const CUtensorMap* map;
          int32_t y;
          if (PASS == 1) {
            map = &tmQg;
            y = U.lh * P.Rpad + U.R0 + t * TILE_ROWS;
          } else {
            map = U.slab ? &tmK1 : &tmK0;
            y = static_cast<int32_t>(U.lh * P.ldK + U.key0 + t * TILE_ROWS);
          }
          tma_load_2d(dst, map, 0, y, &bars->a_full[ab]);
          tma_load_2d(dst + HALF_BYTES, map, 64, y, &bars->a_full[ab]);
        }
        issued_a[ab]++;
        if (++ab == 2) { ab = 0; aph ^= 1; }
        // B tiles
        for (int i = 0; i < U.nT; ++i) {
          if (*abort_flag) break;
          if (!mbar_wait(&bars->b_empty[s], bph ^ 1, P.limit_ns)) { fail(2); break; }
          mbar_arrive_expect_tx(&bars->b_full[s], TILE_BYTES);
          const CUtensorMap* map;
          int32_t y;
          if (PASS == 1) {
            const TileRef tr = tile_at1(P, U, i);
            if (tr.kind == 0) {
              map = U.slab ? &tmK1 : &tmK0;
              y = static_cast<int32_t>(U.lh * P.ldK + tr.t0);
            } else {
              map = &tmApp;
              y = U.lh * P.ldApp + tr.chunk * P.nq_full + tr.t0;
            }
          } else {
            map = &tmQg;
            y = U.lh * P.Rpad + U.r * P.CR + i * TILE_ROWS;
          }
          uint8_t* dst = sB + s * TILE_BYTES;
          tma_load_2d(dst, map, 0, y, &bars->b_full[s]);
          tma_load_2d(dst + HALF_BYTES, map, 64, y, &bars->b_full[s]);
          issued_b[s]++;
          if (++s == KSTAGES) { s = 0; bph ^= 1; }
        }
      }
      // Wait for every copy this thread started (normally already consumed).
      for (int i = 0; i < KSTAGES; ++i)
        if (issued_b[i] > 0) mbar_wait(&bars->b_full[i], (issued_b[i] - 1) & 1, P.limit_ns);
      for (int i = 0; i < 2; ++i)
        if (issued_a[i] > 0) mbar_wait(&bars->a_full[i], (issued_a[i] - 1) & 1, P.limit_ns);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc = idesc_bf16_f32(128, TILE_ROWS);
      int s = 0, ab = 0, db = 0;
      uint32_t bph = 0, aph = 0, dph = 0;
      for (int u = blockIdx.x; u < P.n_units && !*abort_flag; u += gridDim.x) {
        const Unit U = decode_unit<PASS>(P, u);
        if (!mbar_wait(&bars->a_full[ab], aph, P.limit_ns)) { fail(3); break; }
        tc_fence_after();
        const uint32_t a0 = smem_u32(sA + (ab * 2) * TILE_BYTES);
        for (int i = 0; i < U.nT; ++i) {
          if (*abort_flag) break;
          if (!mbar_wait(&bars->b_full[s], bph, P.limit_ns)) { fail(4); break; }
          if (!mbar_wait(&bars->d_empty[db], dph ^ 1, P.limit_ns)) { fail(5); break; }
          tc_fence_after();
          const uint32_t b0 = smem_u32(sB + s * TILE_BYTES);
          for (int t = 0; t <= U.has1; ++t) {
            const uint32_t d = tbase + db * 256 + t * 128;
            const uint32_t at = a0 + t * TILE_BYTES;
#pragma unroll
            for (int k = 0; k < 8; ++k) {
              const uint32_t koff = (k >> 2) * HALF_BYTES + (k & 3) * 32;
              mma_bf16(d, sdesc_kmajor_sw128(at + koff), sdesc_kmajor_sw128(b0 + koff), idesc, k > 0 ? 1u : 0u);
            }
          }
          mma_commit(&bars->b_empty[s]);
          mma_commit(&bars->d_full[db]);
          if (++s == KSTAGES) { s = 0; bph ^= 1; }
          if (++db == 2) { db = 0; dph ^= 1; }
        }
        mma_commit(&bars->a_empty[ab]);
        if (++ab == 2) { ab = 0; aph ^= 1; }
      }
      // All issued MMAs must finish before TMEM is released.
      mma_commit(&bars->drain);
      mbar_wait(&bars->drain, 0, P.limit_ns);
    }
  } else {
    // ------------------------------------------------------------ consumers
    const int wg = (warp - 2) >> 2;          // which A tile (accumulator)
    const int quarter = warp & 3;            // TMEM lane quarter this warp may access
    const int row = quarter * 32 + lane;     // row of the A tile
    const uint32_t lane_addr = tbase + (static_cast<uint32_t>(quarter * 32) << 16) + wg * 128;
    const float c = P.scale_log2;
    int db = 0;
    uint32_t dph = 0;
    for (int u = blockIdx.x; u < P.n_units && !*abort_flag; u += gridDim.x) {
      const Unit U = decode_unit<PASS>(P, u);
      if (PASS == 1) {
        // ---- row LSE over the cache and the chunk's appended keys
        const int R = U.R0 + wg * TILE_ROWS + row;
        const bool has_tile = (wg == 0) || U.has1;
        const int nc = P.n_chunks[U.ai];
        const int rr = min(R / P.CR, nc - 1);
        const int local = R - rr * P.CR;
        const int nq = nq_of(P, U.ai, rr);
        const bool valid = has_tile && local < P.G * nq && R < P.Rpad;
        const int g = valid ? local / nq : 0;
        const int j = valid ? local - g * nq : 0;
        float mrun = -INFINITY, ssum = 0.f;
        for (int i = 0; i < U.nT; ++i) {
          if (!mbar_wait(&bars->d_full[db], dph, P.limit_ns)) { fail(6); break; }
          tc_fence_after();
          const TileRef tr = tile_at1(P, U, i);
          int lim;
          if (tr.kind == 0) lim = U.n - tr.t0;
          else lim = (tr.chunk == rr) ? (j - tr.t0 + 1) : 0;
#pragma unroll 1
          for (int cb = 0; cb < 4; ++cb) {
            float v[32];
            __syncwarp();
            tmem_ld32(lane_addr + db * 256 + cb * 32, v);
            const int l32 = lim - cb * 32;
            if (l32 <= 0) continue;
            if (l32 < 32) {
#pragma unroll
              for (int k = 0; k < 32; ++k) v[k] = (k < l32) ? v[k] : -INFINITY;
            }
            float bm = v[0];
#pragma unroll
            for (int k = 1; k < 32; ++k) bm = fmaxf(bm, v[k]);
            const float mn = fmaxf(mrun, bm * c);
            if (mn > mrun) {
              ssum *= ex2(mrun - mn);
              mrun = mn;
            }
            float acc0 = 0.f, acc1 = 0.f;
#pragma unroll
            for (int k = 0; k < 32; k += 2) {
              acc0 += ex2(fmaf(v[k], c, -mrun));
              acc1 += ex2(fmaf(v[k + 1], c, -mrun));
            }
            ssum += acc0 + acc1;
          }
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&bars->d_empty[db]);
          if (++db == 2) { db = 0; dph ^= 1; }
        }
        if (*abort_flag) break;
        if (has_tile && R < P.Rpad) {
          const int64_t o = static_cast<int64_t>(U.lh) * P.Rpad + R;
          if (valid) {
            const float l2 = mrun + lg2(ssum);
            P.lse2[o] = l2;
            if (P.lse_out) {
              const int hq = U.h * P.G + g;
              P.lse_out[(static_cast<int64_t>(U.layer) * P.Hq + hq) * P.Q + rr * P.nq_full + j] =
                  l2 * 0.69314718055994531f;
            }
          } else {
            P.lse2[o] = INFINITY;  // padding rows never win the pass-2 max
          }
        }
      } else {
        // ---- column max over the chunk's queries for one key per thread
        const int pos = U.key0 + wg * TILE_ROWS + row;
        const bool valid = ((wg == 0) || U.has1) && pos < U.hi;
        const float* lrow = P.lse2 + static_cast<int64_t>(U.lh) * P.Rpad + U.r * P.CR;
        float vmax = -INFINITY;
        for (int i = 0; i < U.nT; ++i) {
          if (!mbar_wait(&bars->d_full[db], dph, P.limit_ns)) { fail(7); break; }
          tc_fence_after();
          const float4* lt = reinterpret_cast<const float4*>(lrow + i * TILE_ROWS);
#pragma unroll 1
          for (int cb = 0; cb < 4; ++cb) {
            float v[32];
            __syncwarp();
            tmem_ld32(lane_addr + db * 256 + cb * 32, v);
#pragma unroll
            for (int k4 = 0; k4 < 8; ++k4) {
              const float4 l = __ldg(lt + cb * 8 + k4);
              vmax = fmaxf(vmax, fmaf(v[4 * k4 + 0], c, -l.x));
              vmax = fmaxf(vmax, fmaf(v[4 * k4 + 1], c, -l.y));
              vmax = fmaxf(vmax, fmaf(v[4 * k4 + 2], c, -l.z));
              vmax = fmaxf(vmax, fmaf(v[4 * k4 + 3], c, -l.w));
            }
          }
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&bars->d_empty[db]);
          if (++db == 2) { db = 0; dph ^= 1; }
        }
        if (*abort_flag) break;
        if (valid) P.score[static_cast<int64_t>(U.lh) * P.ldS + pos] = ex2(vmax);
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tbase, TMEM_COLS);
  }
}

// ----------------------------------------------------------------- gather
// Fill the row space Qg (query rows, zero padding) and, for KV², the
// appended keys Kg = K[l, h, sel].  Half a warp moves one 256-byte row.
struct GParams {
  int Hkv, Hq, G;
  int n_active;
  int32_t layer[kMaxLayers];
  int32_t n[kMaxLayers];
  int32_t slab[kMaxLayers];
  int32_t n_chunks[kMaxLayers];
  int32_t nq_full, nq_last, Q, CR, Rpad;
  const int32_t* sel;
  const __nv_bfloat16* Qsrc;
  int64_t ldQ;
  const __nv_bfloat16* K[2];
  int64_t ldK;
  __nv_bfloat16* Qg;
  __nv_bfloat16* Kg;   // null: appended keys supplied by the caller
  int* status;
};

__global__ void __launch_bounds__(256) gather_kernel(const __grid_constant__ GParams P) {
  const int64_t rows_q = static_cast<int64_t>(P.n_active) * P.Hkv * P.Rpad;
  const int64_t rows_k = P.Kg ? static_cast<int64_t>(P.n_active) * P.Hkv * P.Q : 0;
  const int64_t total = rows_q + rows_k;
  const int sub = threadIdx.x & 15;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * (blockDim.x >> 4);
  for (int64_t w = static_cast<int64_t>(blockIdx.x) * (blockDim.x >> 4) + (threadIdx.x >> 4); w < total;
       w += stride) {
    uint4 val = make_uint4(0, 0, 0, 0);
    __nv_bfloat16* dst;
    if (w < rows_q) {
      const int64_t per = static_cast<int64_t>(P.Hkv) * P.Rpad;
      const int ai = static_cast<int>(w / per);
      const int64_t rem = w - ai * per;
      const int h = static_cast<int>(rem / P.Rpad);
      const int R = static_cast<int>(rem - static_cast<int64_t>(h) * P.Rpad);
      const int layer = P.layer[ai];
      const int nc = P.n_chunks[ai];
      const int r = min(R / P.CR, nc - 1);
      const int local = R - r * P.CR;
      const int nq = (r == nc - 1) ? P.nq_last : P.nq_full;
      dst = P.Qg + ((static_cast<int64_t>(layer) * P.Hkv + h) * P.Rpad + R) * kHeadDim;
      if (local < P.G * nq) {
        const int g = local / nq, j = local - g * nq;
        const int t = r * P.nq_full + j;
        const int src = P.sel ? P.sel[t] : t;
        if (src >= 0 && src < P.ldQ) {
          const __nv_bfloat16* s =
              P.Qsrc + ((static_cast<int64_t>(layer) * P.Hq + h * P.G + g) * P.ldQ + src) * kHeadDim;
          val = __ldg(reinterpret_cast<const uint4*>(s) + sub);
        } else if (sub == 0) {
          record_status(P.status, DEV_BOUNDS);
        }
      }
    } else {
      const int64_t w2 = w - rows_q;
      const int64_t per = static_cast<int64_t>(P.Hkv) * P.Q;
      const int ai = static_cast<int>(w2 / per);
      const int64_t rem = w2 - ai * per;
      const int h = static_cast<int>(rem / P.Q);
      const int t = static_cast<int>(rem - static_cast<int64_t>(h) * P.Q);
      const int layer = P.layer[ai];
      dst = P.Kg + ((static_cast<int64_t>(layer) * P.Hkv + h) * P.Q + t) * kHeadDim;
      const int src = P.sel ? P.sel[t] : t;
      if (src >= 0 && src < P.n[ai]) {
        const __nv_bfloat16* s =
            P.K[P.slab[ai]] + ((static_cast<int64_t>(layer) * P.Hkv + h) * P.ldK + src) * kHeadDim;
        val = __ldg(reinterpret_cast<const uint4*>(s) + sub);
      } else if (sub == 0) {
        record_status(P.status, DEV_BOUNDS);
      }
    }
    reinterpret_cast<uint4*>(dst)[sub] = val;
  }
}

int round_up(int a, int b) { return (a + b - 1) / b * b; }

}  // namespace

int32_t recon_rows(int G, int n_chunks, int nq_full, int nq_last) {
  const int CR = round_up(G * nq_full, TILE_ROWS);
  return (n_chunks - 1) * CR + round_up(G * nq_last, TILE_ROWS);
}

size_t recon_ws_bytes(int L, int Hkv, int G, int n_chunks, int nq_full, int nq_last, int Q, bool need_kg) {
  const int64_t Rpad = recon_rows(G, n_chunks, nq_full, nq_last);
  size_t b = 0;
  auto add = [&](size_t bytes) { b = ((b + 255) & ~size_t(255)) + bytes; };
  add(static_cast<size_t>(L) * Hkv * Rpad * kHeadDim * 2);      // Qg
  if (need_kg) add(static_cast<size_t>(L) * Hkv * Q * kHeadDim * 2);  // Kg
  add(static_cast<size_t>(L) * Hkv * Rpad * 4);                  // lse2
  return b + 256;
}

cudaError_t launch_recon(const ReconProblem& pr, const ReconWorkspace& ws, cudaStream_t st) {
  const int G = pr.G;
  // chunk layout is the same for every active layer in one call
  const int nc0 = pr.lay[0].n_chunks;
  const int CR = round_up(G * pr.nq_full, TILE_ROWS);
  const int Rpad = recon_rows(G, nc0, pr.nq_full, pr.nq_last);
  if (Rpad != ws.Rpad) return cudaErrorInvalidValue;

  // ---- gather
  GParams gp;
  memset(&gp, 0, sizeof(gp));
  gp.Hkv = pr.Hkv; gp.Hq = pr.Hq; gp.G = G; gp.n_active = pr.n_active;
  for (int a = 0; a < pr.n_active; ++a) {
    gp.layer[a] = pr.lay[a].layer;
    gp.n[a] = pr.lay[a].n;
    gp.slab[a] = pr.lay[a].slab;
    gp.n_chunks[a] = pr.lay[a].n_chunks;
  }
  gp.nq_full = pr.nq_full; gp.nq_last = pr.nq_last; gp.Q = pr.Q; gp.CR = CR; gp.Rpad = Rpad;
  gp.sel = pr.sel;
  gp.Qsrc = static_cast<const __nv_bfloat16*>(pr.Qsrc);
  gp.ldQ = pr.ldQ;
  gp.K[0] = static_cast<const __nv_bfloat16*>(pr.K[0]);
  gp.K[1] = static_cast<const __nv_bfloat16*>(pr.K[1] ? pr.K[1] : pr.K[0]);
  gp.ldK = pr.ldK;
  gp.Qg = static_cast<__nv_bfloat16*>(ws.Qg);
  gp.Kg = pr.Kapp ? nullptr : static_cast<__nv_bfloat16*>(ws.Kg);
  gp.status = status_word();
  {
    const int64_t rows = static_cast<int64_t>(pr.n_active) * pr.Hkv * (Rpad + (gp.Kg ? pr.Q : 0));
    int64_t blocks = (rows + 15) / 16;
    const int64_t cap = static_cast<int64_t>(num_sms()) * 8;
    if (blocks > cap) blocks = cap;
    if (blocks < 1) blocks = 1;
    {
      ProfScope ps("recon_gather", st);
      gather_kernel<<<static_cast<int>(blocks), 256, 0, st>>>(gp);
    }
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }

  // ---- tensor maps
  // Rows are addressed by model layer index, so the maps span all L layers.
  CUtensorMap tmQg, tmK0, tmK1, tmApp;
  const uint64_t LH = static_cast<uint64_t>(pr.L) * pr.Hkv;
  if (!make_tmap_rows(&tmQg, ws.Qg, LH * Rpad, TILE_ROWS)) return cudaErrorInvalidValue;
  if (!make_tmap_rows(&tmK0, pr.K[0], LH * pr.ldK, TILE_ROWS)) return cudaErrorInvalidValue;
  if (!make_tmap_rows(&tmK1, pr.K[1] ? pr.K[1] : pr.K[0], LH * pr.ldK, TILE_ROWS)) return cudaErrorInvalidValue;
  const void* app = pr.Kapp ? pr.Kapp : ws.Kg;
  const int64_t ldApp = pr.Kapp ? pr.ldApp : pr.Q;
  if (!make_tmap_rows(&tmApp, app, LH * ldApp, TILE_ROWS)) return cudaErrorInvalidValue;

  KParams kp;
  memset(&kp, 0, sizeof(kp));
  kp.Hkv = pr.Hkv; kp.Hq = pr.Hq; kp.G = G; kp.sinks = pr.sinks; kp.n_active = pr.n_active;
  int acc = 0;
  for (int a = 0; a < pr.n_active; ++a) {
    const ReconLayer& ly = pr.lay[a];
    kp.layer[a] = ly.layer; kp.n[a] = ly.n; kp.m[a] = ly.m; kp.n_chunks[a] = ly.n_chunks;
    kp.last_len[a] = ly.last_len; kp.slab[a] = ly.slab;
    kp.unit_off[a] = acc;
    const int pf = (ly.m + 255) / 256, pl = (ly.last_len + 255) / 256;
    acc += pr.Hkv * ((ly.n_chunks - 1) * pf + pl);
  }
  kp.unit_off[pr.n_active] = acc;
  kp.ldK = pr.ldK;
  kp.nq_full = pr.nq_full; kp.nq_last = pr.nq_last; kp.Q = pr.Q;
  kp.CR = CR; kp.Rpad = Rpad;
  kp.ldApp = static_cast<int32_t>(ldApp);
  kp.pairs1 = (Rpad + 255) / 256;
  kp.scale_log2 = static_cast<float>(1.4426950408889634 / std::sqrt(static_cast<double>(kHeadDim)));
  kp.lse2 = ws.lse2;
  kp.lse_out = pr.lse_out;
  kp.score = pr.score;
  kp.ldS = pr.ldS;
  kp.status = status_word();
  kp.limit_ns = wait_limit_ns();

  cudaError_t ea = cudaFuncSetAttribute(recon_kernel<1>, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
  if (ea != cudaSuccess) return ea;
  ea = cudaFuncSetAttribute(recon_kernel<2>, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
  if (ea != cudaSuccess) return ea;
  const int sms = num_sms();
  // pass 1
  kp.n_units = pr.n_active * pr.Hkv * kp.pairs1;
  if (kp.n_units > 0) {
    ProfScope ps("recon_lse", st);
    recon_kernel<1><<<kp.n_units < sms ? kp.n_units : sms, NUM_THREADS, SMEM_BYTES, st>>>(tmQg, tmK0, tmK1, tmApp, kp);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  // pass 2
  kp.n_units = acc;
  if (kp.n_units > 0) {
    ProfScope ps("recon_colmax", st);
    recon_kernel<2><<<kp.n_units < sms ? kp.n_units : sms, NUM_THREADS, SMEM_BYTES, st>>>(tmQg, tmK0, tmK1, tmApp, kp);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

}  // namespace kvc
