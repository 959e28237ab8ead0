// Reconstruction scoring (KV² page, "무엇과 다른가"): the selected tokens are
// appended after the cache and attend causally over the whole cache; the
// score of a cache position of chunk C_r is the max, over the chunk's
// reconstruction queries and over the query heads sharing the KV head, of
// the softmax attention it receives.
//
// Two tensor-core passes per (layer, KV head), both on one warp-specialised
// persistent skeleton (warp 0: TMA producer, warp 1: tcgen05.mma issuer and
// TMEM owner, then 4 warps per A tile as consumers):
//
//   pass 1 (row LSE)    A = 2 tiles of 128 reconstruction-query rows, B =
//                       streamed 256-key tiles of the cache, then the chunk's
//                       appended keys under the causal mask.  Each consumer
//                       thread owns half of one query row's columns (one TMEM
//                       lane) and keeps a sum of 2^x against a lazily moved
//                       reference: lse2 = reference + log2(sum).
//                       On GB300 the MUFU exp2 rate (32/clk/SM) equals the
//                       MMA logit rate at d = 128, so 16 consumer warps (4
//                       per SM sub-partition) keep the exponentials flowing
//                       while single-buffered accumulators are handed back to
//                       the MMA warp as soon as they are read.  Each row's
//                       -lse2/scale is written as three bf16 terms.
//   pass 2 (column max) A = 2 tiles of 128 cache keys of one chunk, B = the
//                       chunk's query rows in 256-row tiles.  A ninth K step
//                       multiplies a constant block of ones with the query
//                       rows' -lse2/scale terms, so each accumulator already
//                       holds x_ij - lse2_j/scale; each consumer thread owns
//                       one key (TMEM lane) and takes the max over the query
//                       columns.  exp2 is monotone, so one exp2 per key gives
//                       the max attention.  One store per position.
//
// Query rows are laid out per (layer, KV head) in a "row space": chunk r
// occupies rows [r*CR, r*CR + G*nq_r) ordered (query head g, query j), with
// CR = G*nq_full rounded up to 128 so that no 128-row tile straddles chunks.
// A gather kernel fills it (and the appended keys) from the query pool.
#include <cuda_bf16.h>

#include <algorithm>
#include <cmath>
#include <cstring>

#include "kvc_internal.h"
#include "kvc_ptx.cuh"

namespace kvc {
namespace {

constexpr int TILE_ROWS = 128;                  // rows of an A tile (TMEM lanes)
constexpr int TILE_BYTES = TILE_ROWS * 256;     // 128 rows x 128 bf16
constexpr uint32_t TMEM_COLS = 512;
constexpr int MAX_KST = 4;

// Per-pass shape of the pipeline.  B tiles of 256 rows (MMA N = 256) halve
// the A-operand re-reads from shared memory per FLOP; with N = 128 the
// shared-memory operand traffic, not the tensor core, caps the MMA rate.
// Pass 1 (8 layers of the 16K workload): two 128-column consumer groups per
// accumulator 1.27 ms, one 256-column group 1.42 ms; double-buffered
// accumulators on 128-key tiles 1.44-1.46 ms; 32-column TMEM loads
// 1.39-1.43 ms against 64-column loads.
template <int PASS>
struct Cfg;
template <>
struct Cfg<1> {
  static constexpr int NA = 2;          // A tiles (128 query rows each) per unit
  static constexpr int ABUF = 1;        // A buffers in shared memory
  static constexpr int DBUF = 1;        // accumulator buffers per A tile
  static constexpr int BN = 256;        // rows (keys) of a B tile = MMA N
  static constexpr int CSPLIT = 2;      // consumer warps sharing one TMEM lane quarter (column split)
  static constexpr int KST = 2;         // B-tile ring depth
};
// Pass 2: two 128-key A tiles per unit against 256-query B tiles (MMA
// N = 256, nine K steps: eight of d = 128, one for the lse), one consumer
// group per accumulator reading its 256 columns in four 64-column loads (the
// accumulator is released after the fourth).  With the lse subtraction inside
// the MMA this pass is bound by the tensor pipe (8 layers of the 16K
// workload: 0.295 ms, against 0.347 ms when the consumers subtracted a staged
// lse row, and the same 0.295 ms with two 128-column consumer groups per
// accumulator).  Also measured, all slower, while the consumers subtracted:
// 128-query tiles with the key tiles copied into TMEM, loads of the next
// column block issued before folding the current one, and the last query
// tile of a chunk multiplied at its own (smaller) N.
template <>
struct Cfg<2> {
  static constexpr int NA = 2;
  static constexpr int ABUF = 1;
  static constexpr int DBUF = 1;
  static constexpr int BN = 256;
  static constexpr int CSPLIT = 1;
  static constexpr int KST = 2;
};
// Pass 2 keeps one A buffer of two 128-key tiles with a barrier pair per
// tile: a tile is refilled (the next unit's keys, read once from HBM) as
// soon as the unit's last MMA on it is done, and the next unit's first B
// tile is issued before its key tiles so that it loads under the current
// unit's MMAs.  The producer also warms the next unit's key tiles in L2 once
// the unit's second B tile is on its way.
// Both passes' consumers read their accumulator in 64-column TMEM loads.
constexpr int P_BLK = 64;
template <int PASS>
constexpr int kThreads = 64 + 128 * Cfg<PASS>::NA * Cfg<PASS>::CSPLIT;
template <int PASS>
constexpr int kABytes = Cfg<PASS>::ABUF * Cfg<PASS>::NA * TILE_BYTES;
template <int PASS>
constexpr int kBStage = Cfg<PASS>::BN * 256;
template <int PASS>
constexpr int kCombBytes = Cfg<PASS>::CSPLIT > 1 ? Cfg<PASS>::NA * TILE_ROWS * 8 : 0;
// Pass 2 subtracts each query row's lse inside the MMA: a ninth K = 16 step
// multiplies a constant keys-side block (ones at K = 0..2) with a
// queries-side block holding -lse2/scale as three bf16 terms (about 24
// bits), so the accumulator already holds x_ij - lse2_j/scale and the
// consumers only take maxima.
template <int PASS>
constexpr int kBxStage = PASS == 2 ? Cfg<PASS>::BN * 32 : 0;   // the B tile's lse rows, 16 bf16 each
template <int PASS>
constexpr int kAxBytes = PASS == 2 ? TILE_ROWS * 32 : 0;       // the constant keys-side block
template <int PASS>
constexpr int kSmemBytes = 1024 + kABytes<PASS> + Cfg<PASS>::KST * (kBStage<PASS> + kBxStage<PASS>) +
                           kAxBytes<PASS> + kCombBytes<PASS> + 256;
static_assert(Cfg<1>::NA * Cfg<1>::DBUF * Cfg<1>::BN <= TMEM_COLS, "TMEM pass 1");
static_assert(Cfg<2>::NA * Cfg<2>::DBUF * Cfg<2>::BN <= TMEM_COLS, "TMEM pass 2");
static_assert(kSmemBytes<1> <= 232448 && kSmemBytes<2> <= 232448, "shared memory budget of one CTA");
static_assert(Cfg<1>::KST <= MAX_KST && Cfg<2>::KST <= MAX_KST, "ring depth");

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
  int32_t units1;                     // pass-1 units per (l, h)
  int32_t snake;                      // pass 1: odd waves in reverse CTA order
  int n_units;
  float scale_log2;                   // log2(e) / sqrt(d)
  __nv_bfloat16* lsx;                 // [rows][16]: -lse2/scale_log2 in three bf16 terms
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

// Row o of the lse rows: x = -lse2/scale as three bf16 terms (hi + mid + lo
// carries about 24 bits; each remainder is exact in fp32), then 13 zeros.
// -inf (padding rows) is stored as (-inf, 0, 0).
__device__ __forceinline__ uint32_t bf16x2_bits(__nv_bfloat16 a, __nv_bfloat16 b) {
  return static_cast<uint32_t>(__bfloat16_as_ushort(a)) | (static_cast<uint32_t>(__bfloat16_as_ushort(b)) << 16);
}
__device__ __forceinline__ void store_lse_row(__nv_bfloat16* lsx, int64_t o, float x) {
  const __nv_bfloat16 zero = __float2bfloat16_rn(0.f);
  __nv_bfloat16 hi = __float2bfloat16_rn(x), mid = zero, lo = zero;
  if (isfinite(x)) {
    const float r1 = x - __bfloat162float(hi);
    mid = __float2bfloat16_rn(r1);
    lo = __float2bfloat16_rn(r1 - __bfloat162float(mid));
  }
  uint4* dst = reinterpret_cast<uint4*>(lsx + o * 16);
  dst[0] = make_uint4(bf16x2_bits(hi, mid), bf16x2_bits(lo, zero), 0u, 0u);
  dst[1] = make_uint4(0u, 0u, 0u, 0u);
}

__device__ __forceinline__ int nq_of(const KParams& P, int ai, int r) {
  return (r == P.n_chunks[ai] - 1) ? P.nq_last : P.nq_full;
}

// ----------------------------------------------------------------- units
// The unit a CTA takes in wave k (units k*gridDim.x ... (k+1)*gridDim.x - 1),
// or -1 when it has none left (a wave that runs past n_units is the last
// one).  Pass-1 units differ in length when the active layers do (EpiCache
// budgets); then the host lists the longest layers first and sets P.snake,
// and odd waves go to the CTAs in reverse, so the CTAs that took the longest
// units in the first wave take the shortest ones in the second.
template <int PASS>
__device__ __forceinline__ int unit_of_wave(const KParams& P, int k) {
  const int c = (PASS == 1 && P.snake && (k & 1)) ? static_cast<int>(gridDim.x) - 1 - static_cast<int>(blockIdx.x)
                                                       : static_cast<int>(blockIdx.x);
  const int u = k * static_cast<int>(gridDim.x) + c;
  return u < P.n_units ? u : -1;
}

struct Unit {
  int ai, layer, h, lh, slab, n;
  int ntile;       // A tiles present (1..NA)
  // pass 1
  int R0, R1;      // row-space range [R0, R1] of the unit (inclusive)
  int ra, rb;      // chunk range touching the unit
  int nK;          // cache-key tiles
  // pass 2
  int r, lo, hi, key0;
  int nT;          // B tiles of the unit
};

__device__ __forceinline__ bool chunk_has_rows(const KParams& P, int ai, int r, int R0, int R1) {
  const int a = r * P.CR, b = r * P.CR + P.G * nq_of(P, ai, r) - 1;
  return a <= R1 && b >= R0;
}

template <int PASS>
__device__ Unit decode_unit(const KParams& P, int u) {
  constexpr int NA = Cfg<PASS>::NA;
  Unit U;
  if (PASS == 1) {
    const int per_layer = P.Hkv * P.units1;
    U.ai = u / per_layer;
    const int rem = u - U.ai * per_layer;
    U.h = rem / P.units1;
    const int q = rem - U.h * P.units1;
    U.layer = P.layer[U.ai];
    U.lh = U.layer * P.Hkv + U.h;
    U.slab = P.slab[U.ai];
    U.n = P.n[U.ai];
    U.R0 = q * NA * TILE_ROWS;
    U.R1 = min(U.R0 + NA * TILE_ROWS, P.Rpad) - 1;
    U.ntile = (U.R1 - U.R0) / TILE_ROWS + 1;
    const int nc = P.n_chunks[U.ai];
    U.ra = min(U.R0 / P.CR, nc - 1);
    U.rb = min(U.R1 / P.CR, nc - 1);
    constexpr int BN = Cfg<1>::BN;
    U.nK = (U.n + BN - 1) / BN;
    int nt = U.nK;
    for (int r = U.ra; r <= U.rb; ++r)
      if (chunk_has_rows(P, U.ai, r, U.R0, U.R1)) nt += (nq_of(P, U.ai, r) + BN - 1) / BN;
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
    constexpr int span = NA * TILE_ROWS;
    const int pf = (m + span - 1) / span;
    const int pl = (P.last_len[ai] + span - 1) / span;
    const int per_head = (nc - 1) * pf + pl;
    const int rem = u - P.unit_off[ai];
    U.h = rem / per_head;
    const int q = rem - U.h * per_head;
    U.lh = U.layer * P.Hkv + U.h;
    int r, kq;
    if (q < (nc - 1) * pf) {
      r = q / pf;
      kq = q - r * pf;
    } else {
      r = nc - 1;
      kq = q - (nc - 1) * pf;
    }
    U.r = r;
    U.lo = P.sinks + r * m;
    U.hi = min(U.lo + m, U.n);
    U.key0 = U.lo + kq * span;
    U.ntile = min(NA, (U.hi - U.key0 + TILE_ROWS - 1) / TILE_ROWS);
    U.nT = (P.G * nq_of(P, ai, r) + Cfg<2>::BN - 1) / Cfg<2>::BN;
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
  constexpr int BN = Cfg<1>::BN;
  TileRef t;
  if (i < U.nK) {
    t.kind = 0;
    t.t0 = i * BN;
    t.chunk = -1;
    return t;
  }
  i -= U.nK;
  for (int r = U.ra; r <= U.rb; ++r) {
    if (!chunk_has_rows(P, U.ai, r, U.R0, U.R1)) continue;
    const int na = (nq_of(P, U.ai, r) + BN - 1) / BN;
    if (i < na) {
      t.kind = 1;
      t.t0 = i * BN;
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
  uint64_t b_full[MAX_KST], b_empty[MAX_KST];
  uint64_t d_full[4], d_empty[4];  // per (accumulator buffer, A tile)
  uint64_t comb_full[2], comb_empty[2];  // pass 1: hand-off of the second column half per A tile
  uint64_t drain;
  uint32_t tmem_base;
  int abort_flag;
};

// Sum of 2^(v*c - m) over N logits (masked entries are -inf and add 0),
// in eight packed partial sums (measured 1.1% faster than four).
template <int N>
__device__ __forceinline__ float exp2_sum(const float (&v)[N], float c, float m) {
  constexpr int CH = 8;                                 // independent packed partial sums
  const uint64_t cc = pack2(c, c), nm = pack2(-m, -m);
  uint64_t acc[CH];
#pragma unroll
  for (int q = 0; q < CH; ++q) acc[q] = 0ull;
#pragma unroll
  for (int k = 0; k < N / 2; ++k) {
    float x0, x1;
    unpack2(fma2(pack2(v[2 * k], v[2 * k + 1]), cc, nm), x0, x1);
    acc[k % CH] = add2(acc[k % CH], pack2(ex2(x0), ex2(x1)));
  }
#pragma unroll
  for (int w = CH / 2; w >= 1; w /= 2)
#pragma unroll
    for (int q = 0; q < w; ++q) acc[q] = add2(acc[q], acc[q + w]);
  const uint64_t s2 = acc[0];
  float s0, s1;
  unpack2(s2, s0, s1);
  return s0 + s1;
}

template <int N>
__device__ __forceinline__ float block_max(const float (&v)[N]) {
  float t[8];
#pragma unroll
  for (int q = 0; q < 8; ++q) {
    float a = v[q];
#pragma unroll
    for (int k = q + 8; k + 8 < N; k += 16) a = fmax3(a, v[k], v[k + 8]);
    if ((N / 8) % 2 == 0) a = fmaxf(a, v[N - 8 + q]);
    t[q] = a;
  }
  return fmax3(fmax3(t[0], t[1], t[2]), fmax3(t[3], t[4], t[5]), fmaxf(t[6], t[7]));
}

// Log-sum-exp update with a lazily moved reference: sum_i 2^(x_i - mref) is
// exact for any reference, it only must not overflow.  The exact block max
// is taken for the row's first visible block; afterwards each block is summed
// against the current reference and only if that sum exceeds 2^40 (a logit
// more than ~34 above the reference, i.e. overflow is possible) the block is
// redone against its own max, with the running sum rescaled.  This drops the
// per-element max from the common path.
template <int N>
__device__ __forceinline__ void lse_update_lazy(float (&v)[N], int lim, float c, float& mref, float& ssum) {
  if (lim <= 0) return;
  if (lim < N) {
#pragma unroll
    for (int k = 0; k < N; ++k) v[k] = (k < lim) ? v[k] : -INFINITY;
  }
  if (mref == -INFINITY) mref = block_max<N>(v) * c;  // first visible block of the row
  float s = exp2_sum<N>(v, c, mref);
  if (!(s <= 1099511627776.0f)) {  // 2^40, also catches inf / NaN
    const float mn = fmaxf(mref, block_max<N>(v) * c);
    ssum *= ex2(mref - mn);
    mref = mn;
    s = exp2_sum<N>(v, c, mref);
  }
  ssum += s;
}


// EARLY (pass 2 only): units of at most two query tiles, whose first query
// tile is issued ahead of their key tiles, with a barrier pair per key tile.
template <int PASS, bool EARLY = false>
__global__ void __launch_bounds__(kThreads<PASS>, 1)
    recon_kernel(const __grid_constant__ CUtensorMap tmQg, const __grid_constant__ CUtensorMap tmK0,
                 const __grid_constant__ CUtensorMap tmK1, const __grid_constant__ CUtensorMap tmApp,
                 const __grid_constant__ KParams P) {
  constexpr int NA = Cfg<PASS>::NA, ABUF = Cfg<PASS>::ABUF, DBUF = Cfg<PASS>::DBUF;
  constexpr int BN = Cfg<PASS>::BN, CSPLIT = Cfg<PASS>::CSPLIT, KST = Cfg<PASS>::KST;
  constexpr int BSTAGE = kBStage<PASS>;            // bytes of one B tile
  constexpr int BHALF = BSTAGE / 2;                // one 64-column swizzled half of a B tile
  constexpr int AHALF = TILE_BYTES / 2;
  constexpr bool kEarly = PASS == 2 && EARLY;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sA = smem;                              // [ABUF][NA] tiles
  uint8_t* sB = smem + kABytes<PASS>;              // [KST] tiles of BN rows
  constexpr int BX_STAGE = kBxStage<PASS>;
  uint8_t* sBx = sB + KST * BSTAGE;                                     // [KST][BN][16] bf16 (pass 2)
  uint8_t* sAx = sBx + KST * BX_STAGE;                                  // [128][16] bf16 (pass 2)
  float2* sComb = reinterpret_cast<float2*>(sAx + kAxBytes<PASS>);      // [NA][128] column-half hand-off
  Bars* bars = reinterpret_cast<Bars*>(reinterpret_cast<uint8_t*>(sComb) + kCombBytes<PASS>);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    static_assert(ABUF <= 2 && (!kEarly || (ABUF == 1 && NA <= 2)), "A barriers");
    for (int i = 0; i < 2; ++i) {      // pass 1: per A buffer; pass 2: per A tile
      mbar_init(&bars->a_full[i], 1);
      mbar_init(&bars->a_empty[i], 1);
    }
    for (int i = 0; i < DBUF * NA; ++i) {
      mbar_init(&bars->d_full[i], 1);
      mbar_init(&bars->d_empty[i], 4 * CSPLIT);  // the warps reading this accumulator
    }
    for (int i = 0; i < KST; ++i) {
      mbar_init(&bars->b_full[i], 1);
      mbar_init(&bars->b_empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&bars->comb_full[i], 4);
      mbar_init(&bars->comb_empty[i], 4);
    }
    mbar_init(&bars->drain, 1);
    bars->abort_flag = 0;
    fence_barrier_init();
  }
  if (PASS == 2) {
    // keys-side block of the lse step: ones at K = 0..2, repeated at K = 8..10
    // so that the 32-byte swizzle (which may exchange a row's two 16-byte
    // halves) leaves it unchanged; the queries side is zero at K = 3..15
    uint4* ax = reinterpret_cast<uint4*>(sAx);
    for (int i = threadIdx.x; i < TILE_ROWS * 2; i += blockDim.x) ax[i] = make_uint4(0x3F803F80u, 0x00003F80u, 0u, 0u);
    fence_proxy_async_smem();
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
  auto fail = [&]() {
    *abort_flag = 1;
    record_status(P.status, DEV_TIMEOUT);
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
      int loads_b = 0, loads_a = 0;   // copies issued; copy j went to stage j % KST (buffer j % ABUF)
      // A tile t of a unit (128 rows; pass 2 reads them through the 128-row K maps)
      auto a_tile = [&](const Unit& W, int t, int32_t& y) -> const CUtensorMap* {
        if (PASS == 1) {
          y = W.lh * P.Rpad + W.R0 + t * TILE_ROWS;
          return &tmQg;
        }
        y = static_cast<int32_t>(W.lh * P.ldK + W.key0 + t * TILE_ROWS);
        return W.slab ? &tmK1 : &tmK0;
      };
      if constexpr (kEarly) {
        for (int k = 0, u; (u = unit_of_wave<PASS>(P, k)) >= 0 && !*abort_flag; ++k) {
          const Unit U = decode_unit<PASS>(P, u);
          auto prefetch_next = [&]() {
            const int un = unit_of_wave<PASS>(P, k + 1);
            if (un < 0) return;
            const Unit W = decode_unit<PASS>(P, un);
            for (int t = 0; t < W.ntile; ++t) {
              int32_t y;
              const CUtensorMap* map = a_tile(W, t, y);
              tma_prefetch_l2_2d(map, 0, y);
              tma_prefetch_l2_2d(map, 64, y);
            }
          };
          // B tile i (BN rows)
          auto issue_b = [&](int i) -> bool {
            if (*abort_flag) return false;
            if (!mbar_wait(&bars->b_empty[s], bph ^ 1, P.limit_ns)) { fail(); return false; }
            mbar_arrive_expect_tx(&bars->b_full[s], BSTAGE + BX_STAGE);
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
              y = U.lh * P.Rpad + U.r * P.CR + i * BN;
              // pass 2 receives the lse-row map in the appended-key slot
              tma_load_2d(sBx + s * BX_STAGE, &tmApp, 0, y, &bars->b_full[s]);
            }
            uint8_t* dst = sB + s * BSTAGE;
            tma_load_2d(dst, map, 0, y, &bars->b_full[s]);
            tma_load_2d(dst + BHALF, map, 64, y, &bars->b_full[s]);
            ++loads_b;
            if (PASS == 2 && i == min(1, U.nT - 1)) prefetch_next();
            if (++s == KST) { s = 0; bph ^= 1; }
            return true;
          };
          // The unit's first query tile goes out before its key tiles, so it
          // loads while the previous unit's MMAs still hold the A buffer, and
          // each key tile has its own barrier pair and is refilled as soon as
          // the previous unit's last MMA on it is done (EpiCache's one-tile
          // prompts: 0.157 -> 0.134 ms per step).  Units of many query tiles
          // use the buffer-wide loop below: there the reloads are rare, and
          // this one measured 3-7% slower at 32 layers of the 16K workload.
          {
            if (!issue_b(0)) break;
            bool ok = true;
            for (int t = 0; t < NA; ++t) {
              if (!mbar_wait(&bars->a_empty[t], aph ^ 1, P.limit_ns)) { fail(); ok = false; break; }
              if (t < U.ntile) {
                mbar_arrive_expect_tx(&bars->a_full[t], TILE_BYTES);
                uint8_t* dst = sA + t * TILE_BYTES;
                int32_t y;
                const CUtensorMap* map = a_tile(U, t, y);
                tma_load_2d(dst, map, 0, y, &bars->a_full[t]);
                tma_load_2d(dst + AHALF, map, 64, y, &bars->a_full[t]);
              } else {
                mbar_arrive(&bars->a_full[t]);    // a missing tile completes its phase empty
              }
            }
            if (!ok) break;
          }
          ++loads_a;
          if (++ab == ABUF) { ab = 0; aph ^= 1; }
          for (int i = 1; i < U.nT; ++i)
            if (!issue_b(i)) break;
        }
      } else {
        for (int k = 0, u; (u = unit_of_wave<PASS>(P, k)) >= 0 && !*abort_flag; ++k) {
          const Unit U = decode_unit<PASS>(P, u);
          if (!mbar_wait(&bars->a_empty[ab], aph ^ 1, P.limit_ns)) { fail(); break; }
          mbar_arrive_expect_tx(&bars->a_full[ab], U.ntile * TILE_BYTES);
          for (int t = 0; t < U.ntile; ++t) {
            uint8_t* dst = sA + (ab * NA + t) * TILE_BYTES;
            int32_t y;
            const CUtensorMap* map = a_tile(U, t, y);
            tma_load_2d(dst, map, 0, y, &bars->a_full[ab]);
            tma_load_2d(dst + AHALF, map, 64, y, &bars->a_full[ab]);
          }
          ++loads_a;
          auto prefetch_next = [&]() {
            const int un = unit_of_wave<PASS>(P, k + 1);
            if (un < 0) return;
            const Unit W = decode_unit<PASS>(P, un);
            for (int t = 0; t < W.ntile; ++t) {
              int32_t y;
              const CUtensorMap* map = a_tile(W, t, y);
              tma_prefetch_l2_2d(map, 0, y);
              tma_prefetch_l2_2d(map, 64, y);
            }
          };
          if (++ab == ABUF) { ab = 0; aph ^= 1; }
          // B tiles (BN rows each)
          for (int i = 0; i < U.nT; ++i) {
            if (*abort_flag) break;
            if (!mbar_wait(&bars->b_empty[s], bph ^ 1, P.limit_ns)) { fail(); break; }
            mbar_arrive_expect_tx(&bars->b_full[s], BSTAGE + BX_STAGE);
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
              y = U.lh * P.Rpad + U.r * P.CR + i * BN;
              // pass 2 receives the lse-row map in the appended-key slot
              tma_load_2d(sBx + s * BX_STAGE, &tmApp, 0, y, &bars->b_full[s]);
            }
            uint8_t* dst = sB + s * BSTAGE;
            tma_load_2d(dst, map, 0, y, &bars->b_full[s]);
            tma_load_2d(dst + BHALF, map, 64, y, &bars->b_full[s]);
            ++loads_b;
            if (PASS == 2 && i == min(1, U.nT - 1)) prefetch_next();
            if (++s == KST) { s = 0; bph ^= 1; }
          }
        }
      }
      // Wait for every copy this thread started (normally already consumed).
      for (int i = 0; i < KST; ++i)
        if (loads_b > i) mbar_wait(&bars->b_full[i], ((loads_b - 1 - i) / KST) & 1, P.limit_ns);
      if constexpr (kEarly) {
        for (int t = 0; t < NA; ++t)
          if (loads_a > 0) mbar_wait(&bars->a_full[t], (loads_a - 1) & 1, P.limit_ns);
      } else {
        for (int i = 0; i < ABUF; ++i)
          if (loads_a > i) mbar_wait(&bars->a_full[i], ((loads_a - 1 - i) / ABUF) & 1, P.limit_ns);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc = idesc_bf16_f32(128, BN);
      int s = 0, ab = 0, db = 0;
      uint32_t bph = 0, aph = 0, dph = 0;
      for (int k = 0, u; (u = unit_of_wave<PASS>(P, k)) >= 0 && !*abort_flag; ++k) {
        const Unit U = decode_unit<PASS>(P, u);
        constexpr bool per_tile = kEarly;
        if (!per_tile) {
          if (!mbar_wait(&bars->a_full[ab], aph, P.limit_ns)) { fail(); break; }
          tc_fence_after();
        }
        const uint32_t a0 = smem_u32(sA + (ab * NA) * TILE_BYTES);
        for (int i = 0; i < U.nT; ++i) {
          if (*abort_flag) break;
          if (!mbar_wait(&bars->b_full[s], bph, P.limit_ns)) { fail(); break; }
          const uint32_t b0 = smem_u32(sB + s * BSTAGE);
          bool ok = true;
          for (int t = 0; t < NA; ++t) {
            uint64_t* de = &bars->d_empty[db * NA + t];
            if (!mbar_wait(de, dph ^ 1, P.limit_ns)) { fail(); ok = false; break; }
            if (per_tile && i == 0) {    // A tile t, on its own barrier
              if (!mbar_wait(&bars->a_full[t], aph, P.limit_ns)) { fail(); ok = false; break; }
            }
            tc_fence_after();
            if (t < U.ntile) {
              const uint32_t d = tbase + (db * NA + t) * BN;
              const uint32_t at = a0 + t * TILE_BYTES;
#pragma unroll
              for (int k = 0; k < 8; ++k) {
                const uint32_t ka = (k >> 2) * AHALF + (k & 3) * 32;
                const uint32_t kb = (k >> 2) * BHALF + (k & 3) * 32;
                mma_bf16(d, sdesc_kmajor_sw128(at + ka), sdesc_kmajor_sw128(b0 + kb), idesc, k > 0 ? 1u : 0u);
              }
              if (PASS == 2)   // + (-lse2_j / scale) on every key row
                mma_bf16(d, sdesc_kmajor_sw32(smem_u32(sAx)), sdesc_kmajor_sw32(smem_u32(sBx + s * BX_STAGE)), idesc,
                         1u);
            }
            // accumulator t of this tile is complete (missing tiles commit nothing new)
            mma_commit(&bars->d_full[db * NA + t]);
            if (per_tile && i == U.nT - 1) mma_commit(&bars->a_empty[t]);   // A tile t is free again
          }
          if (!ok) break;
          mma_commit(&bars->b_empty[s]);
          if (++s == KST) { s = 0; bph ^= 1; }
          if (++db == DBUF) { db = 0; dph ^= 1; }
        }
        if (per_tile) {
          aph ^= 1;
        } else {
          mma_commit(&bars->a_empty[ab]);
          if (++ab == ABUF) { ab = 0; aph ^= 1; }
        }
      }
      // All issued MMAs must finish before TMEM is released.
      mma_commit(&bars->drain);
      mbar_wait(&bars->drain, 0, P.limit_ns);
    }
  } else {
    // ------------------------------------------------------------ consumers
    // consumer warps come in groups of 4 (one per TMEM lane quarter); group
    // `slot` reads accumulator wg = slot / CSPLIT, column part chalf
    const int slot = (warp - 2) >> 2;
    const int wg = slot / CSPLIT;            // which A tile (accumulator)
    const int chalf = slot % CSPLIT;         // which part of the accumulator's columns
    const int quarter = warp & 3;            // TMEM lane quarter this warp may access
    const int row = quarter * 32 + lane;     // row of the A tile
    const uint32_t lane_addr = tbase + (static_cast<uint32_t>(quarter * 32) << 16);
    const float c = P.scale_log2;
    int db = 0;
    uint32_t dph = 0;
    uint32_t comb_ph = 0;  // pass 1: phase of the per-unit half-row hand-off
    for (int k = 0, u; (u = unit_of_wave<PASS>(P, k)) >= 0 && !*abort_flag; ++k) {
      const Unit U = decode_unit<PASS>(P, u);
      const bool has_tile = wg < U.ntile;
      if (PASS == 1) {
        // ---- row LSE over the cache and the chunk's appended keys
        const int R = U.R0 + wg * TILE_ROWS + row;
        const int nc = P.n_chunks[U.ai];
        const int rr = min(R / P.CR, nc - 1);
        const int local = R - rr * P.CR;
        const int nq = nq_of(P, U.ai, rr);
        const bool valid = has_tile && local < P.G * nq && R < P.Rpad;
        const int g = valid ? local / nq : 0;
        const int j = valid ? local - g * nq : 0;
        float mrun = -INFINITY, ssum = 0.f;
        constexpr int COLS = BN / CSPLIT;  // columns of the tile this warp reads
        constexpr int PB = P_BLK;          // columns per TMEM load
        static_assert(COLS % PB == 0, "consumers read whole column blocks");
        for (int i = 0; i < U.nT; ++i) {
          uint64_t* df = &bars->d_full[db * NA + wg];
          if (!mbar_wait(df, dph, P.limit_ns)) { fail(); break; }
          tc_fence_after();
          const TileRef tr = tile_at1(P, U, i);
          const int lim = ((tr.kind == 0) ? U.n - tr.t0 : ((tr.chunk == rr) ? (j - tr.t0 + 1) : 0)) -
                          chalf * COLS;
          const uint32_t col = lane_addr + (db * NA + wg) * BN + chalf * COLS;
          // column blocks; the accumulator is handed back to the MMA warp
          // right after the last block is in registers
#pragma unroll
          for (int blk = 0; blk < COLS / PB; ++blk) {
            float v[PB];
            __syncwarp();
            tmem_ld64(col + blk * PB, v);
            if (blk == COLS / PB - 1) {
              tc_fence_before();
              __syncwarp();
              if (lane == 0) mbar_arrive(&bars->d_empty[db * NA + wg]);
            }
            lse_update_lazy<PB>(v, lim - blk * PB, c, mrun, ssum);
          }
          if (++db == DBUF) { db = 0; dph ^= 1; }
        }
        if (*abort_flag) break;
        if (CSPLIT > 1) {
          // fold the other column half's (max, sum) of this row into chalf 0
          if (chalf == 1) {
            if (!mbar_wait(&bars->comb_empty[wg], comb_ph ^ 1, P.limit_ns)) { fail(); break; }
            sComb[wg * TILE_ROWS + row] = make_float2(mrun, ssum);
            __syncwarp();
            if (lane == 0) mbar_arrive(&bars->comb_full[wg]);
          } else {
            if (!mbar_wait(&bars->comb_full[wg], comb_ph, P.limit_ns)) { fail(); break; }
            const float2 o = sComb[wg * TILE_ROWS + row];
            __syncwarp();
            if (lane == 0) mbar_arrive(&bars->comb_empty[wg]);
            const float m = fmaxf(mrun, o.x);
            const float s0 = (mrun == -INFINITY) ? 0.f : ssum * ex2(mrun - m);
            const float s1 = (o.x == -INFINITY) ? 0.f : o.y * ex2(o.x - m);
            mrun = m;
            ssum = s0 + s1;
          }
          comb_ph ^= 1;
        }
        if (chalf == 0 && has_tile && R < P.Rpad) {
          const int64_t o = static_cast<int64_t>(U.lh) * P.Rpad + R;
          if (valid) {
            const float l2 = mrun + lg2(ssum);
            store_lse_row(P.lsx, o, -l2 / c);
            if (P.lse_out) {
              const int hq = U.h * P.G + g;
              P.lse_out[(static_cast<int64_t>(U.layer) * P.Hq + hq) * P.Q + rr * P.nq_full + j] =
                  l2 * 0.69314718055994531f;
            }
          } else {
            store_lse_row(P.lsx, o, -INFINITY);   // padding rows never win the pass-2 max
          }
        }
      } else {
        // ---- column max over the chunk's queries: one key (TMEM lane) per
        // thread, this group's half of the accumulator's query columns
        constexpr int COLS = BN / CSPLIT;
        constexpr int PB = P_BLK;                        // columns per TMEM load
        static_assert(COLS % PB == 0, "pass-2 consumers read whole column blocks");
        const int pos = U.key0 + wg * TILE_ROWS + row;
        const bool valid = has_tile && pos < U.hi;
        const int rows_q = P.G * nq_of(P, U.ai, U.r);    // query rows of this chunk
        float vmax = -INFINITY;   // max_j (x_ij - lse2_j / scale) over this group's query columns
        for (int i = 0; i < U.nT; ++i) {
          uint64_t* df = &bars->d_full[db * NA + wg];
          if (!mbar_wait(df, dph, P.limit_ns)) { fail(); break; }
          tc_fence_after();
          // columns past the chunk's query rows belong to the next chunk
          const int lim = rows_q - i * BN - chalf * COLS;
          const uint32_t col = lane_addr + (db * NA + wg) * BN + chalf * COLS;
          float t[8];
#pragma unroll
          for (int q = 0; q < 8; ++q) t[q] = -INFINITY;
          // fold one block of query columns into t (bl: valid columns of the
          // block); the accumulator already holds x_ij - lse2_j / scale
          auto fold = [&](float (&v)[PB], int bl) {
            if (bl < PB) {
#pragma unroll
              for (int k = 0; k < PB; ++k) v[k] = (k < bl) ? v[k] : -INFINITY;
            }
#pragma unroll
            for (int k = 0; k < PB / 2; ++k) t[k & 7] = fmax3(t[k & 7], v[2 * k], v[2 * k + 1]);
          };
#pragma unroll
          for (int blk = 0; blk < COLS / PB; ++blk) {
            float v[PB];
            __syncwarp();
            tmem_ld64(col + blk * PB, v);
            if (blk == COLS / PB - 1) {
              // the accumulator goes back to the MMA warp once it is in registers
              tc_fence_before();
              __syncwarp();
              if (lane == 0) mbar_arrive(&bars->d_empty[db * NA + wg]);
            }
            const int bl = lim - blk * PB;
            if (bl > 0) fold(v, bl);
          }
          if (++db == DBUF) { db = 0; dph ^= 1; }
          vmax = fmax3(vmax, fmax3(t[0], t[1], t[2]), fmax3(t[3], t[4], t[5]));
          vmax = fmax3(vmax, t[6], t[7]);
        }
        if (*abort_flag) break;
        if (CSPLIT > 1) {
          // merge the column halves of this key's maximum into chalf 0
          if (chalf == 1) {
            if (!mbar_wait(&bars->comb_empty[wg], comb_ph ^ 1, P.limit_ns)) { fail(); break; }
            sComb[wg * TILE_ROWS + row].x = vmax;
            __syncwarp();
            if (lane == 0) mbar_arrive(&bars->comb_full[wg]);
          } else {
            if (!mbar_wait(&bars->comb_full[wg], comb_ph, P.limit_ns)) { fail(); break; }
            const float o = sComb[wg * TILE_ROWS + row].x;
            __syncwarp();
            if (lane == 0) mbar_arrive(&bars->comb_empty[wg]);
            vmax = fmaxf(vmax, o);
          }
          comb_ph ^= 1;
        }
        if (chalf == 0 && valid) P.score[static_cast<int64_t>(U.lh) * P.ldS + pos] = ex2(vmax * c);
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
// appended keys Kg = K[l, h, sel]: 256-byte rows, copied by half-warps
// (gather_rows_kernel).
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

// Source and destination of gathered row w (src null: zero row).  Index
// arithmetic in type I (32-bit whenever the row count allows).
template <class I>
__device__ __forceinline__ void gather_row(const GParams& P, I w, I rows_q, const uint4*& src, uint4*& dst) {
  src = nullptr;
  if (w < rows_q) {
    const I per = static_cast<I>(P.Hkv) * P.Rpad;
    const int ai = static_cast<int>(w / per);
    const I rem = w - static_cast<I>(ai) * per;
    const int h = static_cast<int>(rem / P.Rpad);
    const int R = static_cast<int>(rem - static_cast<I>(h) * P.Rpad);
    const int layer = P.layer[ai];
    const int nc = P.n_chunks[ai];
    const int r = min(R / P.CR, nc - 1);
    const int local = R - r * P.CR;
    const int nq = (r == nc - 1) ? P.nq_last : P.nq_full;
    dst = reinterpret_cast<uint4*>(P.Qg + ((static_cast<int64_t>(layer) * P.Hkv + h) * P.Rpad + R) * kHeadDim);
    if (local < P.G * nq) {
      const int g = local / nq, j = local - g * nq;
      const int t = r * P.nq_full + j;
      const int s = P.sel ? P.sel[t] : t;
      if (s >= 0 && s < P.ldQ)
        src = reinterpret_cast<const uint4*>(
            P.Qsrc + ((static_cast<int64_t>(layer) * P.Hq + h * P.G + g) * P.ldQ + s) * kHeadDim);
      else
        record_status(P.status, DEV_BOUNDS);
    }
  } else {
    const I w2 = w - rows_q;
    const I per = static_cast<I>(P.Hkv) * P.Q;
    const int ai = static_cast<int>(w2 / per);
    const I rem = w2 - static_cast<I>(ai) * per;
    const int h = static_cast<int>(rem / P.Q);
    const int t = static_cast<int>(rem - static_cast<I>(h) * P.Q);
    const int layer = P.layer[ai];
    dst = reinterpret_cast<uint4*>(P.Kg + ((static_cast<int64_t>(layer) * P.Hkv + h) * P.Q + t) * kHeadDim);
    const int s = P.sel ? P.sel[t] : t;
    if (s >= 0 && s < P.n[ai])
      src = reinterpret_cast<const uint4*>(P.K[P.slab[ai]] +
                                           ((static_cast<int64_t>(layer) * P.Hkv + h) * P.ldK + s) * kHeadDim);
    else
      record_status(P.status, DEV_BOUNDS);
  }
}

// Lane `sub` of a half-warp resolves row w0 + sub of 16 consecutive rows (one
// set of index divisions per row; with every lane resolving the same row the
// gather took 45% longer), and the half-warp then copies them four at a time,
// taking each row's addresses by shuffle: 16 lanes x 16 bytes per 256-byte
// row, four rows in flight.  Half-warps run independent loops, so the
// shuffles name only their own 16 lanes.
template <class I>
__global__ void __launch_bounds__(256) gather_rows_kernel(const __grid_constant__ GParams P) {
  const I rows_q = static_cast<I>(P.n_active) * P.Hkv * P.Rpad;
  const I rows_k = P.Kg ? static_cast<I>(P.n_active) * P.Hkv * P.Q : 0;
  const I total = rows_q + rows_k;
  const int sub = threadIdx.x & 15;
  const unsigned hmask = 0xffffu << (threadIdx.x & 16);
  const I hw = static_cast<I>(blockIdx.x) * (blockDim.x >> 4) + (threadIdx.x >> 4);
  const I stride = static_cast<I>(gridDim.x) * (blockDim.x >> 4) * 16;
  for (I w0 = hw * 16; w0 < total; w0 += stride) {
    const uint4* src = nullptr;
    uint4* dst = nullptr;
    const I w = w0 + sub;
    if (w < total) gather_row(P, w, rows_q, src, dst);
    const unsigned long long s64 = reinterpret_cast<unsigned long long>(src);
    const unsigned long long d64 = reinterpret_cast<unsigned long long>(dst);
#pragma unroll
    for (int b = 0; b < 16; b += 4) {
      uint4 val[4];
      uint4* d[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const uint4* sr = reinterpret_cast<const uint4*>(__shfl_sync(hmask, s64, b + u, 16));
        d[u] = reinterpret_cast<uint4*>(__shfl_sync(hmask, d64, b + u, 16));
        val[u] = sr ? __ldg(sr + sub) : make_uint4(0, 0, 0, 0);
      }
#pragma unroll
      for (int u = 0; u < 4; ++u)
        if (d[u]) d[u][sub] = val[u];
    }
  }
}

int round_up(int a, int b) { return (a + b - 1) / b * b; }

}  // namespace

int32_t recon_rows(int G, int n_chunks, int nq_full, int nq_last) {
  const int CR = round_up(G * nq_full, TILE_ROWS);
  return (n_chunks - 1) * CR + round_up(G * nq_last, TILE_ROWS);
}

cudaError_t launch_recon(const ReconProblem& pr, const ReconWorkspace& ws, cudaStream_t st, int phases) {
  const int G = pr.G;
  // chunk layout is the same for every active layer in one call
  const int nc0 = pr.lay[0].n_chunks;
  const int CR = round_up(G * pr.nq_full, TILE_ROWS);
  const int Rpad = recon_rows(G, nc0, pr.nq_full, pr.nq_last);
  if (Rpad != ws.Rpad) return cudaErrorInvalidValue;

  // ---- gather
  if (phases & RECON_GATHER) {
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
      int64_t blocks = (rows + 63) / 64;
      const int64_t cap = static_cast<int64_t>(num_sms()) * 8;
      if (blocks > cap) blocks = cap;
      if (blocks < 1) blocks = 1;
      {
        ProfScope ps("recon_gather", st);
        // 32-bit row arithmetic while every index (plus one grid stride of
        // look-ahead) stays below 2^31
        const int64_t slack = blocks * 16 * 16 * 2;
        if (rows + slack < (int64_t(1) << 31))
          gather_rows_kernel<int><<<static_cast<int>(blocks), 256, 0, st>>>(gp);
        else
          gather_rows_kernel<int64_t><<<static_cast<int>(blocks), 256, 0, st>>>(gp);
      }
      cudaError_t e = cudaGetLastError();
      if (e != cudaSuccess) return e;
      if (pr.gather_done) {
        e = cudaEventRecord(pr.gather_done, st);
        if (e != cudaSuccess) return e;
      }
    }
  }
  if (!(phases & (RECON_ROWS | RECON_COLS))) return cudaSuccess;

  // ---- tensor maps
  // Rows are addressed by model layer index, so the maps span all L layers.
  // Pass 1 streams keys in B tiles of Cfg<1>::BN rows; pass 2 reads keys as
  // 128-row A tiles and query rows as 128-row B tiles.
  CUtensorMap tmQg, tmQgB, tmK0a, tmK1a, tmK0b, tmK1b, tmApp;
  const uint64_t LH = static_cast<uint64_t>(pr.L) * pr.Hkv;
  const void* k1 = pr.K[1] ? pr.K[1] : pr.K[0];
  if (!make_tmap_rows(&tmQg, ws.Qg, LH * Rpad, TILE_ROWS)) return cudaErrorInvalidValue;
  if (!make_tmap_rows(&tmQgB, ws.Qg, LH * Rpad, Cfg<2>::BN)) return cudaErrorInvalidValue;
  if (!make_tmap_rows(&tmK0a, pr.K[0], LH * pr.ldK, TILE_ROWS)) return cudaErrorInvalidValue;
  if (!make_tmap_rows(&tmK1a, k1, LH * pr.ldK, TILE_ROWS)) return cudaErrorInvalidValue;
  if (!make_tmap_rows(&tmK0b, pr.K[0], LH * pr.ldK, Cfg<1>::BN)) return cudaErrorInvalidValue;
  if (!make_tmap_rows(&tmK1b, k1, LH * pr.ldK, Cfg<1>::BN)) return cudaErrorInvalidValue;
  const void* app = pr.Kapp ? pr.Kapp : ws.Kg;
  const int64_t ldApp = pr.Kapp ? pr.ldApp : pr.Q;
  if (!make_tmap_rows(&tmApp, app, LH * ldApp, Cfg<1>::BN)) return cudaErrorInvalidValue;
  CUtensorMap tmLx;   // pass 2 (fold): the lse rows, in the appended-key slot
  if (!make_tmap_rows16(&tmLx, ws.lsx, LH * Rpad, Cfg<2>::BN)) return cudaErrorInvalidValue;

  KParams kp;
  memset(&kp, 0, sizeof(kp));
  kp.Hkv = pr.Hkv; kp.Hq = pr.Hq; kp.G = G; kp.sinks = pr.sinks; kp.n_active = pr.n_active;
  constexpr int span2 = Cfg<2>::NA * TILE_ROWS;
  // Schedule order of the active layers: longest first (stable), so that the
  // pass-1 waves pair long units with short ones (see unit_of_wave).  Every
  // buffer is addressed by model layer, so the order changes no result.
  int ord[kMaxLayers];
  for (int a = 0; a < pr.n_active; ++a) ord[a] = a;
  std::stable_sort(ord, ord + pr.n_active, [&](int x, int y) { return pr.lay[x].n > pr.lay[y].n; });
  int acc = 0;
  for (int a = 0; a < pr.n_active; ++a) {
    const ReconLayer& ly = pr.lay[ord[a]];
    kp.layer[a] = ly.layer; kp.n[a] = ly.n; kp.m[a] = ly.m; kp.n_chunks[a] = ly.n_chunks;
    kp.last_len[a] = ly.last_len; kp.slab[a] = ly.slab;
    kp.unit_off[a] = acc;
    const int pf = (ly.m + span2 - 1) / span2, pl = (ly.last_len + span2 - 1) / span2;
    acc += pr.Hkv * ((ly.n_chunks - 1) * pf + pl);
  }
  kp.unit_off[pr.n_active] = acc;
  for (int a = 1; a < pr.n_active; ++a)
    if (pr.lay[a].n != pr.lay[0].n) kp.snake = 1;
  // pass-2 units of at most two query tiles: early B tiles, per-tile A barriers
  const bool early2 = static_cast<int64_t>(G) * std::max(pr.nq_full, pr.nq_last) <= 2 * Cfg<2>::BN;
  kp.ldK = pr.ldK;
  kp.nq_full = pr.nq_full; kp.nq_last = pr.nq_last; kp.Q = pr.Q;
  kp.CR = CR; kp.Rpad = Rpad;
  kp.ldApp = static_cast<int32_t>(ldApp);
  kp.units1 = (Rpad + Cfg<1>::NA * TILE_ROWS - 1) / (Cfg<1>::NA * TILE_ROWS);
  kp.scale_log2 = static_cast<float>(1.4426950408889634 / std::sqrt(static_cast<double>(kHeadDim)));
  kp.lsx = static_cast<__nv_bfloat16*>(ws.lsx);
  kp.lse_out = pr.lse_out;
  kp.score = pr.score;
  kp.ldS = pr.ldS;
  kp.status = status_word();
  kp.limit_ns = wait_limit_ns();

  cudaError_t ea = cudaFuncSetAttribute(recon_kernel<1>, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes<1>);
  if (ea != cudaSuccess) return ea;
  ea = cudaFuncSetAttribute(recon_kernel<2>, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes<2>);
  if (ea != cudaSuccess) return ea;
  ea = cudaFuncSetAttribute(recon_kernel<2, true>, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes<2>);
  if (ea != cudaSuccess) return ea;
  const int sms = num_sms();
  // pass 1
  kp.n_units = pr.n_active * pr.Hkv * kp.units1;
  if ((phases & RECON_ROWS) && kp.n_units > 0) {
    ProfScope ps("recon_lse", st);
    recon_kernel<1><<<kp.n_units < sms ? kp.n_units : sms, kThreads<1>, kSmemBytes<1>, st>>>(tmQg, tmK0b, tmK1b,
                                                                                            tmApp, kp);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  // pass 2
  kp.n_units = acc;
  if ((phases & RECON_COLS) && kp.n_units > 0) {
    ProfScope ps("recon_colmax", st);
    const unsigned grid2 = kp.n_units < sms ? kp.n_units : sms;
    if (early2)
      recon_kernel<2, true><<<grid2, kThreads<2>, kSmemBytes<2>, st>>>(tmQgB, tmK0a, tmK1a, tmLx, kp);
    else
      recon_kernel<2><<<grid2, kThreads<2>, kSmemBytes<2>, st>>>(tmQgB, tmK0a, tmK1a, tmLx, kp);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

}  // namespace kvc
