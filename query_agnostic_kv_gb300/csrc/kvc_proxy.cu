// KeyDiff proxy (KV² page, "어떻게 동작하나"): for each (layer, KV head)
// u = mean_i k_i / |k_i| and s_i = -cos(k_i, u); the token score p_i is the
// mean of s_i over all (layer, KV head) pairs.
//
// One thread-block cluster per (layer, KV head).  Each CTA owns a contiguous
// slice of positions: it sums the unit keys of its slice (pass A), the
// cluster exchanges the partial sums through distributed shared memory and
// every CTA adds them in rank order (so the result is deterministic and the
// same in every CTA), then each CTA re-reads its slice -- the first rows
// from a shared-memory copy kept during pass A, the rest from L2 -- and
// writes s (pass B).  Pass A also stores 1/|k_i| in s[i]; pass B reads it
// back on the same lane (the row -> lane mapping is the same in both passes),
// so it forms only k_i . U before overwriting s[i] with the score.  A second
// small kernel averages s over the heads.
//
// Each 256-byte key row is handled by half a warp: lane l16 owns channels
// [8*l16, 8*l16 + 8) as one 16-byte load.
#include <cooperative_groups.h>
#include <cuda_bf16.h>

#include "kvc_internal.h"
#include "kvc_ptx.cuh"

namespace cg = cooperative_groups;

namespace kvc {
namespace {

// 8 CTAs per head, two resident per SM (16K workload: 0.302 ms; clusters of
// 16, 4 and 2 CTAs measured 0.36, 0.32 and 0.33 ms; one 1024-thread CTA per
// SM 0.35 ms).
constexpr int CLUSTER = 8;
constexpr int THREADS = 512;
constexpr int CTAS_PER_SM = 2;            // two clusters' CTAs share an SM: one loads while the other waits
constexpr int HALVES = THREADS / 16;      // half-warps per CTA
constexpr int UNROLL = 8;                 // rows per half-warp in flight per step (64 KB per CTA)
constexpr int CACHE_ROWS = 256;           // rows of the slice kept in shared memory for pass B
// Pass B walks the slice backwards: the rows pass A loaded last are the
// likeliest to still be in L2, and the first rows come from the cache.
constexpr bool PASS_B_REVERSE = true;
constexpr int SMEM_BYTES = CACHE_ROWS * 256 + HALVES * 128 * 4;
// Steps ahead of the L2 prefetch of rows.  16K workload: none 0.311 ms, one
// step 0.302, two 0.355, three 0.388 (registers spill).
constexpr int KD_PREFETCH = 1;

// ---------------------------------------------------------------------------
// Per-row arithmetic of the KeyDiff kernel.  Channel products run on packed
// f32x2 pairs (measured 0.31 ms against 0.39 ms with scalar FMAs at 16K),
// and the eight rows a half-warp has in flight are reduced together: a
// transposing butterfly leaves row u's total on lanes 2u and 2u+1 of the
// half-warp after 15 shuffles for all eight rows (a butterfly per row takes
// 32).
__device__ __forceinline__ uint64_t bf2_to_f2(uint32_t w) {
  return pack2(__uint_as_float(w << 16), __uint_as_float(w & 0xffff0000u));
}
// The same pair built with byte permutes.  Pass A unpacks each row twice
// (for |k|^2, then for the unit-key sum once 1/|k| is known); spelling the
// second unpack differently keeps the compiler from holding all 64 unpacked
// values of the eight rows live across the reduction.
__device__ __forceinline__ uint64_t bf2_to_f2_prmt(uint32_t w) {
  return pack2(__uint_as_float(__byte_perm(w, 0u, 0x1044)), __uint_as_float(__byte_perm(w, 0u, 0x3244)));
}
__device__ __forceinline__ void unpack8(const uint4& q, float (&f)[8]) {
  const __nv_bfloat162* b = reinterpret_cast<const __nv_bfloat162*>(&q);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 t = __bfloat1622float2(b[i]);
    f[2 * i] = t.x;
    f[2 * i + 1] = t.y;
  }
}
__device__ __forceinline__ float sumsq8(const uint4& q) {
  const uint64_t x0 = bf2_to_f2(q.x), x1 = bf2_to_f2(q.y), x2 = bf2_to_f2(q.z), x3 = bf2_to_f2(q.w);
  uint64_t a = mul2(x0, x0);
  a = fma2(x1, x1, a);
  a = fma2(x2, x2, a);
  a = fma2(x3, x3, a);
  float lo, hi;
  unpack2(a, lo, hi);
  return lo + hi;
}
__device__ __forceinline__ float dot8(const uint4& q, const uint64_t (&u2)[4]) {
  uint64_t a = mul2(bf2_to_f2(q.x), u2[0]);
  a = fma2(bf2_to_f2(q.y), u2[1], a);
  a = fma2(bf2_to_f2(q.z), u2[2], a);
  a = fma2(bf2_to_f2(q.w), u2[3], a);
  float lo, hi;
  unpack2(a, lo, hi);
  return lo + hi;
}
// v[u] holds this lane's partial for row u (u = 0..7) of its half-warp.
// Returns the half-warp total of row (l16 >> 1), present on lanes 2u, 2u+1.
__device__ __forceinline__ float transpose_sum8(const float (&v)[8], int l16) {
  const bool b3 = (l16 & 8) != 0, b2 = (l16 & 4) != 0, b1 = (l16 & 2) != 0;
  float r[4];
#pragma unroll
  for (int k = 0; k < 4; ++k)   // keep rows k + 4*b3
    r[k] = (b3 ? v[k + 4] : v[k]) + __shfl_xor_sync(0xffffffffu, b3 ? v[k] : v[k + 4], 8);
  float r2[2];
#pragma unroll
  for (int k = 0; k < 2; ++k)   // keep rows k + 2*b2 + 4*b3
    r2[k] = (b2 ? r[k + 2] : r[k]) + __shfl_xor_sync(0xffffffffu, b2 ? r[k] : r[k + 2], 4);
  const float r3 = (b1 ? r2[1] : r2[0]) + __shfl_xor_sync(0xffffffffu, b1 ? r2[0] : r2[1], 2);
  return r3 + __shfl_xor_sync(0xffffffffu, r3, 1);
}

// Loads of rows that L2 will not serve again carry an L2 evict-first
// policy, so they leave L2 before the rows other heads' pass B still needs:
// every load of pass B (each row's last read), and pass A's loads of the
// rows kept in shared memory for pass B (16K workload: 0.303 -> 0.289 ->
// 0.280 ms; an evict-last policy on pass A's other loads changed nothing).
__device__ __forceinline__ uint64_t l2_policy_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}
__device__ __forceinline__ uint4 ld_nc_policy(const uint4* a, uint64_t pol) {
  uint4 r;
  asm volatile("ld.global.nc.L2::cache_hint.v4.u32 {%0, %1, %2, %3}, [%4], %5;"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "l"(a), "l"(pol));
  return r;
}

__global__ void __cluster_dims__(CLUSTER, 1, 1) __launch_bounds__(THREADS, CTAS_PER_SM)
    keydiff_kernel(const __nv_bfloat16* __restrict__ K, int N, float* __restrict__ s_out) {
  static_assert(UNROLL == 8, "rows are reduced in groups of eight");
  extern __shared__ __align__(16) uint8_t smem[];
  uint4* cache = reinterpret_cast<uint4*>(smem);                            // [CACHE_ROWS][16]
  float* red = reinterpret_cast<float*>(smem + CACHE_ROWS * 256);          // [HALVES][128]
  __shared__ float part[kHeadDim];
  __shared__ float U[kHeadDim];
  __shared__ float unorm_inv;

  cg::cluster_group cluster = cg::this_cluster();
  const int rank = static_cast<int>(cluster.block_rank());
  const int lh = blockIdx.y;
  const uint4* rows = reinterpret_cast<const uint4*>(K + static_cast<int64_t>(lh) * N * kHeadDim);
  float* srow = s_out + static_cast<int64_t>(lh) * N;

  const int slice = (N + CLUSTER - 1) / CLUSTER;
  const int i0 = min(rank * slice, N);
  const int i1 = min(i0 + slice, N);
  const int lane = threadIdx.x & 31;
  const int hw = threadIdx.x >> 4;
  const int l16 = threadIdx.x & 15;
  const int u_own = l16 >> 1;                 // row (of the eight) this lane ends up owning
  const bool writer = (l16 & 1) == 0;

  const uint64_t cached_read = l2_policy_evict_first();
  // ---- pass A: sum of unit keys over the slice; 1/|k_i| kept in s[i]
  uint64_t acc2[4] = {0ull, 0ull, 0ull, 0ull};
  for (int base = i0; base < i1; base += HALVES * UNROLL) {
    uint4 q[UNROLL];
#pragma unroll
    for (int u = 0; u < UNROLL; ++u) {
      const int i = base + u * HALVES + hw;
      // rows that pass B reads from the shared-memory copy are not needed in L2 again
      q[u] = (i < i1) ? ((i - i0 < CACHE_ROWS) ? ld_nc_policy(rows + static_cast<int64_t>(i) * 16 + l16, cached_read)
                                             : __ldg(rows + static_cast<int64_t>(i) * 16 + l16))
                      : make_uint4(0, 0, 0, 0);
    }
    if (KD_PREFETCH) {
      // warm L2 with the rows KD_PREFETCH steps ahead: lane l16 takes line (l16 & 1) of row (l16 >> 1)
      const int i = base + KD_PREFETCH * HALVES * UNROLL + u_own * HALVES + hw;
      if (i < i1) prefetch_l2(rows + static_cast<int64_t>(i) * 16 + (l16 & 1) * 8);
    }
    float ss[UNROLL];
#pragma unroll
    for (int u = 0; u < UNROLL; ++u) {
      const int i = base + u * HALVES + hw;
      if (i < i1 && i - i0 < CACHE_ROWS) cache[(i - i0) * 16 + l16] = q[u];
      ss[u] = sumsq8(q[u]);
    }
    const float tot = transpose_sum8(ss, l16);
    const float inv_own = tot > 0.f ? rsqrtf(tot) : 0.f;
    const int i_own = base + u_own * HALVES + hw;
    if (writer && i_own < i1) srow[i_own] = inv_own;
#pragma unroll
    for (int u = 0; u < UNROLL; ++u) {
      const float iv = __shfl_sync(0xffffffffu, inv_own, (lane & 16) | (u << 1));
      const uint64_t iv2 = pack2(iv, iv);
      acc2[0] = fma2(bf2_to_f2_prmt(q[u].x), iv2, acc2[0]);
      acc2[1] = fma2(bf2_to_f2_prmt(q[u].y), iv2, acc2[1]);
      acc2[2] = fma2(bf2_to_f2_prmt(q[u].z), iv2, acc2[2]);
      acc2[3] = fma2(bf2_to_f2_prmt(q[u].w), iv2, acc2[3]);
    }
  }
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    float a, b;
    unpack2(acc2[c], a, b);
    red[hw * 128 + l16 * 8 + 2 * c] = a;
    red[hw * 128 + l16 * 8 + 2 * c + 1] = b;
  }
  __syncthreads();
  if (threadIdx.x < kHeadDim) {
    float t = 0.f;
    for (int w = 0; w < HALVES; ++w) t += red[w * 128 + threadIdx.x];
    part[threadIdx.x] = t;
  }
  cluster.sync();
  // ---- exchange: U = sum of the cluster's partials in rank order
  if (threadIdx.x < kHeadDim) {
    float t = 0.f;
    for (int r = 0; r < CLUSTER; ++r) t += cluster.map_shared_rank(part, r)[threadIdx.x];
    U[threadIdx.x] = t;
  }
  cluster.sync();  // no CTA leaves while its partial may still be read
  if (threadIdx.x < 32) {
    float t = 0.f;
    for (int c = threadIdx.x; c < kHeadDim; c += 32) t = fmaf(U[c], U[c], t);
    for (int o = 16; o > 0; o >>= 1) t += __shfl_xor_sync(0xffffffffu, t, o);
    if (threadIdx.x == 0) unorm_inv = t > 0.f ? rsqrtf(t) : 0.f;
  }
  __syncthreads();

  // ---- pass B: s_i = -(k_i . U) / (|k_i| |U|)
  const uint64_t last_read = l2_policy_evict_first();
  uint64_t u2[4];
#pragma unroll
  for (int c = 0; c < 4; ++c) u2[c] = pack2(U[l16 * 8 + 2 * c], U[l16 * 8 + 2 * c + 1]);
  const float uinv = unorm_inv;
  const int nblk = (i1 - i0 + HALVES * UNROLL - 1) / (HALVES * UNROLL);
  for (int bi = 0; bi < nblk; ++bi) {
    const int base = i0 + (PASS_B_REVERSE ? nblk - 1 - bi : bi) * HALVES * UNROLL;
    const int i_own = base + u_own * HALVES + hw;
    if (KD_PREFETCH && bi + KD_PREFETCH < nblk) {
      // the rows KD_PREFETCH steps ahead that are not in the shared-memory copy
      const int nb = i0 + (PASS_B_REVERSE ? nblk - 1 - bi - KD_PREFETCH : bi + KD_PREFETCH) * HALVES * UNROLL;
      const int i = nb + u_own * HALVES + hw;
      if (i < i1 && i - i0 >= CACHE_ROWS) prefetch_l2(rows + static_cast<int64_t>(i) * 16 + (l16 & 1) * 8);
    }
    // 1/|k| of the owned row, written by this same lane in pass A
    const float inv_own = (writer && i_own < i1) ? srow[i_own] : 0.f;
    uint4 q[UNROLL];
#pragma unroll
    for (int u = 0; u < UNROLL; ++u) {
      const int i = base + u * HALVES + hw;
      if (i < i1)
        q[u] = (i - i0 < CACHE_ROWS) ? cache[(i - i0) * 16 + l16]
                                     : ld_nc_policy(rows + static_cast<int64_t>(i) * 16 + l16, last_read);
      else
        q[u] = make_uint4(0, 0, 0, 0);
    }
    float dt[UNROLL];
#pragma unroll
    for (int u = 0; u < UNROLL; ++u) dt[u] = dot8(q[u], u2);
    const float dot = transpose_sum8(dt, l16);
    if (writer && i_own < i1) srow[i_own] = (inv_own > 0.f && uinv > 0.f) ? -dot * inv_own * uinv : 0.f;
  }
}

// Knorm proxy (KV² page, "전제와 한계": the close alternative to KeyDiff):
// s_i = -|k_i| per (layer, KV head), one read of K.  Half a warp per 256-byte
// row, eight rows in flight per half-warp, one butterfly per row (for this
// single-pass kernel the transposed reduction measured slower: it holds all
// eight rows until the last arrives).  Each half-warp runs its own loop, so
// the shuffles name only the 16 lanes of the half-warp.
__global__ void __launch_bounds__(256) knorm_kernel(const uint4* __restrict__ K, int64_t rows,
                                                    float* __restrict__ s_out) {
  constexpr int R = 8;
  const int l16 = threadIdx.x & 15;
  const unsigned half_mask = 0xffffu << (threadIdx.x & 16);
  const int64_t hw = static_cast<int64_t>(blockIdx.x) * (blockDim.x >> 4) + (threadIdx.x >> 4);
  const int64_t stride = static_cast<int64_t>(gridDim.x) * (blockDim.x >> 4);
  for (int64_t r0 = hw; r0 < rows; r0 += stride * R) {
    uint4 q[R];
#pragma unroll
    for (int u = 0; u < R; ++u) {
      const int64_t r = r0 + u * stride;
      q[u] = (r < rows) ? __ldg(K + r * 16 + l16) : make_uint4(0, 0, 0, 0);
    }
#pragma unroll
    for (int u = 0; u < R; ++u) {
      float f[8];
      unpack8(q[u], f);
      float ss = 0.f;
#pragma unroll
      for (int c = 0; c < 8; ++c) ss = fmaf(f[c], f[c], ss);
#pragma unroll
      for (int o = 8; o > 0; o >>= 1) ss += __shfl_xor_sync(half_mask, ss, o);
      const int64_t r = r0 + u * stride;
      if (l16 == 0 && r < rows) s_out[r] = -sqrtf(ss);
    }
  }
}

// p[i] = (1/LH) sum_h x[h][i], 0 below `zero_below`; with `divide` 0 the
// plain sum (a shard's partial sum for the layer-sharded path).  A block
// covers 32 positions with 8 warps: warp w adds heads w, w + 8, ... of its
// lane's position (coalesced 128-byte rows), and the eight partial sums are
// then added in warp order, so the result does not depend on scheduling.
constexpr int MH_POS = 32, MH_SPLIT = 8;
__global__ void __launch_bounds__(MH_POS* MH_SPLIT)
    mean_heads_kernel(const float* __restrict__ x, int LH, int N, int64_t ld, int zero_below, int divide,
                      float* __restrict__ p) {
  __shared__ float part[MH_SPLIT][MH_POS];
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  const int i = blockIdx.x * MH_POS + lane;
  float t = 0.f;
  if (i < N && i >= zero_below)
    for (int h = w; h < LH; h += MH_SPLIT) t += x[static_cast<int64_t>(h) * ld + i];
  part[w][lane] = t;
  __syncthreads();
  if (w == 0 && i < N) {
    float s = 0.f;
#pragma unroll
    for (int q = 0; q < MH_SPLIT; ++q) s += part[q][lane];
    p[i] = i < zero_below ? 0.f : (divide ? s / static_cast<float>(LH) : s);
  }
}

// p[i] = psum[i] / heads (the division of the unsharded mean, applied to the
// shards' summed partials).
__global__ void sums_to_mean_kernel(const float* __restrict__ psum, int N, int heads, float* __restrict__ p) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i < N) p[i] = psum[i] / static_cast<float>(heads);
}

}  // namespace

// The cluster kernel needs no scratch beyond s.
size_t proxy_scratch_bytes(int LH, int N) {
  (void)LH;
  (void)N;
  return 0;
}

// The KeyDiff kernel's shared-memory attribute, set once per device.
cudaError_t keydiff_attr() {
  static int done[64];
  int d = 0;
  if (cudaGetDevice(&d) != cudaSuccess || d < 0 || d >= 64) return cudaErrorInvalidDevice;
  if (done[d]) return cudaSuccess;
  const cudaError_t e = cudaFuncSetAttribute(keydiff_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
  if (e == cudaSuccess) done[d] = 1;
  return e;
}

cudaError_t launch_proxy(const void* K, int LH, int N, float* s, float* p, void* scratch, cudaStream_t st) {
  (void)scratch;
  cudaError_t e = keydiff_attr();
  if (e != cudaSuccess) return e;
  dim3 grid(CLUSTER, LH);
  {
    ProfScope ps("keydiff", st);
    keydiff_kernel<<<grid, THREADS, SMEM_BYTES, st>>>(static_cast<const __nv_bfloat16*>(K), N, s);
  }
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  return launch_mean_heads(s, LH, N, N, 0, p, st);
}

cudaError_t launch_knorm(const void* K, int LH, int N, float* s, float* p, cudaStream_t st) {
  const int64_t rows = static_cast<int64_t>(LH) * N;
  int64_t blocks = (rows + 16 * 8 - 1) / (16 * 8);
  const int64_t cap = static_cast<int64_t>(num_sms()) * 8;
  if (blocks > cap) blocks = cap;
  {
    ProfScope ps("knorm", st);
    knorm_kernel<<<static_cast<int>(blocks), 256, 0, st>>>(static_cast<const uint4*>(K), rows, s);
  }
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  return launch_mean_heads(s, LH, N, N, 0, p, st);
}

cudaError_t launch_mean_heads(const float* x, int LH, int N, int64_t ld, int zero_below, float* p,
                              cudaStream_t st) {
  ProfScope ps("mean_heads", st);
  mean_heads_kernel<<<(N + MH_POS - 1) / MH_POS, MH_POS * MH_SPLIT, 0, st>>>(x, LH, N, ld, zero_below, 1, p);
  return cudaGetLastError();
}

cudaError_t launch_sum_heads(const float* x, int LH, int N, int64_t ld, int zero_below, float* psum,
                             cudaStream_t st) {
  ProfScope ps("sum_heads", st);
  mean_heads_kernel<<<(N + MH_POS - 1) / MH_POS, MH_POS * MH_SPLIT, 0, st>>>(x, LH, N, ld, zero_below, 0, psum);
  return cudaGetLastError();
}

cudaError_t launch_sums_to_mean(const float* psum, int N, int heads, float* p, cudaStream_t st) {
  ProfScope ps("sums_to_mean", st);
  sums_to_mean_kernel<<<(N + 255) / 256, 256, 0, st>>>(psum, N, heads, p);
  return cudaGetLastError();
}

// Per-head scores only (s[lh][i]), no average: the first half of launch_proxy
// / launch_knorm, for a shard that sums its heads itself.
cudaError_t launch_proxy_scores(int kind, const void* K, int LH, int N, float* s, cudaStream_t st) {
  if (kind == 1) {
    const int64_t rows = static_cast<int64_t>(LH) * N;
    int64_t blocks = (rows + 16 * 8 - 1) / (16 * 8);
    const int64_t cap = static_cast<int64_t>(num_sms()) * 8;
    if (blocks > cap) blocks = cap;
    ProfScope ps("knorm", st);
    knorm_kernel<<<static_cast<int>(blocks), 256, 0, st>>>(static_cast<const uint4*>(K), rows, s);
    return cudaGetLastError();
  }
  cudaError_t e = keydiff_attr();
  if (e != cudaSuccess) return e;
  ProfScope ps("keydiff", st);
  keydiff_kernel<<<dim3(CLUSTER, LH), THREADS, SMEM_BYTES, st>>>(static_cast<const __nv_bfloat16*>(K), N, s);
  return cudaGetLastError();
}

}  // namespace kvc
