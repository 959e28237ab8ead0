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
// writes s (pass B).  A second small kernel averages s over the heads.
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

#ifndef KVC_KD_CTAS
#define KVC_KD_CTAS 2
#endif
#ifndef KVC_KD_CACHE
#define KVC_KD_CACHE 256
#endif
#ifndef KVC_KD_REVERSE
#define KVC_KD_REVERSE 1
#endif
// 8 CTAs per head, two resident per SM (measured faster than 16-CTA clusters).
constexpr int CLUSTER = 8;
constexpr int THREADS = 512;
constexpr int CTAS_PER_SM = KVC_KD_CTAS;  // two clusters' CTAs share an SM: one loads while the other waits
constexpr int HALVES = THREADS / 16;      // half-warps per CTA
#ifndef KVC_KD_UNROLL
#define KVC_KD_UNROLL 8
#endif
constexpr int UNROLL = KVC_KD_UNROLL;      // rows per half-warp in flight per step (64 KB per CTA at 8)
constexpr int CACHE_ROWS = KVC_KD_CACHE;  // rows of the slice kept in shared memory for pass B
// Pass B walks the slice backwards: the rows pass A loaded last are the
// likeliest to still be in L2, and the first rows come from the cache.
constexpr bool PASS_B_REVERSE = KVC_KD_REVERSE != 0;
constexpr int SMEM_BYTES = CACHE_ROWS * 256 + HALVES * 128 * 4;

__device__ __forceinline__ void unpack8(const uint4& q, float (&f)[8]) {
  const __nv_bfloat162* b = reinterpret_cast<const __nv_bfloat162*>(&q);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 t = __bfloat1622float2(b[i]);
    f[2 * i] = t.x;
    f[2 * i + 1] = t.y;
  }
}

__device__ __forceinline__ float half_warp_sum(float v) {
  v += __shfl_xor_sync(0xffffffffu, v, 8);
  v += __shfl_xor_sync(0xffffffffu, v, 4);
  v += __shfl_xor_sync(0xffffffffu, v, 2);
  v += __shfl_xor_sync(0xffffffffu, v, 1);
  return v;
}

__global__ void __cluster_dims__(CLUSTER, 1, 1) __launch_bounds__(THREADS, CTAS_PER_SM)
    keydiff_kernel(const __nv_bfloat16* __restrict__ K, int N, float* __restrict__ s_out) {
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

  const int slice = (N + CLUSTER - 1) / CLUSTER;
  const int i0 = min(rank * slice, N);
  const int i1 = min(i0 + slice, N);
  const int hw = threadIdx.x >> 4;
  const int l16 = threadIdx.x & 15;

  // ---- pass A: sum of unit keys over the slice
  float acc[8];
#pragma unroll
  for (int c = 0; c < 8; ++c) acc[c] = 0.f;
  for (int base = i0; base < i1; base += HALVES * UNROLL) {
    uint4 q[UNROLL];
#pragma unroll
    for (int u = 0; u < UNROLL; ++u) {
      const int i = base + u * HALVES + hw;
      q[u] = (i < i1) ? __ldg(rows + static_cast<int64_t>(i) * 16 + l16) : make_uint4(0, 0, 0, 0);
    }
#pragma unroll
    for (int u = 0; u < UNROLL; ++u) {
      const int i = base + u * HALVES + hw;
      if (i < i1 && i - i0 < CACHE_ROWS) cache[(i - i0) * 16 + l16] = q[u];
      float f[8];
      unpack8(q[u], f);
      float ss = 0.f;
#pragma unroll
      for (int c = 0; c < 8; ++c) ss = fmaf(f[c], f[c], ss);
      ss = half_warp_sum(ss);
      const float inv = ss > 0.f ? rsqrtf(ss) : 0.f;
#pragma unroll
      for (int c = 0; c < 8; ++c) acc[c] = fmaf(f[c], inv, acc[c]);
    }
  }
#pragma unroll
  for (int c = 0; c < 8; ++c) red[hw * 128 + l16 * 8 + c] = acc[c];
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
  float uu[8];
#pragma unroll
  for (int c = 0; c < 8; ++c) uu[c] = U[l16 * 8 + c];
  const float uinv = unorm_inv;
  float* srow = s_out + static_cast<int64_t>(lh) * N;
  const int nblk = (i1 - i0 + HALVES * UNROLL - 1) / (HALVES * UNROLL);
  for (int bi = 0; bi < nblk; ++bi) {
    const int base = i0 + (PASS_B_REVERSE ? nblk - 1 - bi : bi) * HALVES * UNROLL;
    uint4 q[UNROLL];
#pragma unroll
    for (int u = 0; u < UNROLL; ++u) {
      const int i = base + u * HALVES + hw;
      if (i < i1)
        q[u] = (i - i0 < CACHE_ROWS) ? cache[(i - i0) * 16 + l16] : __ldg(rows + static_cast<int64_t>(i) * 16 + l16);
      else
        q[u] = make_uint4(0, 0, 0, 0);
    }
#pragma unroll
    for (int u = 0; u < UNROLL; ++u) {
      const int i = base + u * HALVES + hw;
      float f[8];
      unpack8(q[u], f);
      float ss = 0.f, dot = 0.f;
#pragma unroll
      for (int c = 0; c < 8; ++c) {
        ss = fmaf(f[c], f[c], ss);
        dot = fmaf(f[c], uu[c], dot);
      }
      ss = half_warp_sum(ss);
      dot = half_warp_sum(dot);
      if (l16 == 0 && i < i1) srow[i] = (ss > 0.f && uinv > 0.f) ? -dot * rsqrtf(ss) * uinv : 0.f;
    }
  }
}

// Knorm proxy (KV² page, "전제와 한계": the close alternative to KeyDiff):
// s_i = -|k_i| per (layer, KV head), one read of K.  Half a warp per 256-byte
// row, eight rows in flight per half-warp.
__global__ void __launch_bounds__(256) knorm_kernel(const uint4* __restrict__ K, int64_t rows,
                                                    float* __restrict__ s_out) {
  constexpr int R = 8;
  const int l16 = threadIdx.x & 15;
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
      ss = half_warp_sum(ss);
      const int64_t r = r0 + u * stride;
      if (l16 == 0 && r < rows) s_out[r] = -sqrtf(ss);
    }
  }
}

// p[i] = (1/LH) sum_h x[h][i] (fixed order), 0 below `zero_below`.
__global__ void mean_heads_kernel(const float* __restrict__ x, int LH, int N, int64_t ld, int zero_below,
                                  float* __restrict__ p) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= N) return;
  if (i < zero_below) {
    p[i] = 0.f;
    return;
  }
  float t = 0.f;
  for (int h = 0; h < LH; ++h) t += x[static_cast<int64_t>(h) * ld + i];
  p[i] = t / static_cast<float>(LH);
}

}  // namespace

cudaError_t launch_proxy(const void* K, int LH, int N, float* s, float* p, cudaStream_t st) {
  cudaError_t e = cudaFuncSetAttribute(keydiff_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
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
  mean_heads_kernel<<<(N + 255) / 256, 256, 0, st>>>(x, LH, N, ld, zero_below, p);
  return cudaGetLastError();
}

}  // namespace kvc
