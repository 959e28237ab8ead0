// EpiCache's per-turn path ("[26'ICML] EpiCache", "방법: 3단계" step ③ and
// Fig. 3): match each question embedding to its closest episode centroid, and
// pack an episode's compressed cache into one contiguous image so that the
// swap between pinned host memory and the device is a single copy per
// direction (the copies themselves go to the copy engines; see kvc_abi.cu).
//
// match_kernel: one warp per question; 16-byte loads of the question and of
// each centroid, squared differences in fp32, a butterfly sum, and a strict
// "<" scan over the centroids so equal distances keep the lower index.
// pack_kernel: the kept rows of every (layer, KV head) of a block-prefill
// state, taken from the slab that holds the layer, are copied in layer-major /
// head / row order; half a warp moves one 256-byte row as sixteen 16-byte
// loads and stores, four rows in flight per half warp.
#include "kvc_internal.h"
#include "kvc_ptx.cuh"

namespace kvc {
namespace {

constexpr int MATCH_WARPS = 8;
constexpr int PACK_THREADS = 256;
constexpr int PACK_ROWS = 64;      // rows per block: 16 half-warps x 4

__global__ void __launch_bounds__(MATCH_WARPS * 32) match_kernel(int B, int E, int De4, const float4* __restrict__ q,
                                                                 const float4* __restrict__ c, float tau2,
                                                                 int32_t* __restrict__ ep, float* __restrict__ d2out) {
  const int b = blockIdx.x * MATCH_WARPS + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (b >= B) return;
  const float4* qb = q + static_cast<int64_t>(b) * De4;
  int best = 0;
  float bestd = INFINITY;
  for (int e = 0; e < E; ++e) {
    const float4* ce = c + static_cast<int64_t>(e) * De4;
    float acc = 0.f;
    for (int i = lane; i < De4; i += 32) {
      const float4 a = qb[i], m = __ldg(ce + i);
      const float x = a.x - m.x, y = a.y - m.y, z = a.z - m.z, w = a.w - m.w;
      acc = fmaf(x, x, acc);
      acc = fmaf(y, y, acc);
      acc = fmaf(z, z, acc);
      acc = fmaf(w, w, acc);
    }
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
    if (d2out && lane == 0) d2out[static_cast<int64_t>(b) * E + e] = acc;
    if (acc < bestd) {    // strict: equal distances keep the lower index
      bestd = acc;
      best = e;
    }
  }
  if (lane == 0) ep[b] = (tau2 > 0.f && !(bestd <= tau2)) ? -1 : best;
}

__global__ void __launch_bounds__(PACK_THREADS) pack_kernel(const uint4* __restrict__ K0, const uint4* __restrict__ V0,
                                                            const int32_t* __restrict__ P0,
                                                            const uint4* __restrict__ K1, const uint4* __restrict__ V1,
                                                            const int32_t* __restrict__ P1, uint4* __restrict__ Kp,
                                                            uint4* __restrict__ Vp, int32_t* __restrict__ Pp,
                                                            const __grid_constant__ PackParams P) {
  const int l = blockIdx.z, h = blockIdx.y;
  const int n = P.len[l];
  const int t0 = blockIdx.x * PACK_ROWS;
  if (t0 >= n) return;
  const bool slab1 = P.cur[l] != 0;
  const uint4* Ks = slab1 ? K1 : K0;
  const uint4* Vs = slab1 ? V1 : V0;
  const int32_t* Ps = slab1 ? P1 : P0;
  const int64_t src_row = (static_cast<int64_t>(l) * P.Hkv + h) * P.cap;
  const int64_t dst_row = P.dst_off[l] + static_cast<int64_t>(h) * n;
  const int sub = threadIdx.x & 15;
  const int hw = threadIdx.x >> 4;
  uint4 kv[4], vv[4];
#pragma unroll
  for (int u = 0; u < 4; ++u) {
    const int t = t0 + u * 16 + hw;
    if (t < n) {
      kv[u] = Ks[(src_row + t) * 16 + sub];
      vv[u] = Vs[(src_row + t) * 16 + sub];
    }
  }
#pragma unroll
  for (int u = 0; u < 4; ++u) {
    const int t = t0 + u * 16 + hw;
    if (t < n) {
      Kp[(dst_row + t) * 16 + sub] = kv[u];
      Vp[(dst_row + t) * 16 + sub] = vv[u];
      if (Pp && sub == 0) Pp[dst_row + t] = Ps[src_row + t];
    }
  }
}

}  // namespace

cudaError_t launch_match(int B, int E, int De, const float* q, const float* c, float tau, int32_t* ep, float* d2,
                         cudaStream_t st) {
  if (B == 0) return cudaSuccess;
  ProfScope ps("episode_match", st);
  const float tau2 = tau > 0.f ? tau * tau : 0.f;
  match_kernel<<<(B + MATCH_WARPS - 1) / MATCH_WARPS, MATCH_WARPS * 32, 0, st>>>(
      B, E, De / 4, reinterpret_cast<const float4*>(q), reinterpret_cast<const float4*>(c), tau2, ep, d2);
  return cudaGetLastError();
}

cudaError_t launch_pack(const void* K0, const void* V0, const int32_t* P0, const void* K1, const void* V1,
                        const int32_t* P1, void* Kp, void* Vp, int32_t* Pp, const PackParams& pp, cudaStream_t st) {
  int max_len = 0;
  for (int l = 0; l < pp.L; ++l) max_len = pp.len[l] > max_len ? pp.len[l] : max_len;
  if (max_len == 0) return cudaSuccess;
  ProfScope ps("episode_pack", st);
  dim3 grid((max_len + PACK_ROWS - 1) / PACK_ROWS, pp.Hkv, pp.L);
  pack_kernel<<<grid, PACK_THREADS, 0, st>>>(
      static_cast<const uint4*>(K0), static_cast<const uint4*>(V0), P0, static_cast<const uint4*>(K1),
      static_cast<const uint4*>(V1), P1, static_cast<uint4*>(Kp), static_cast<uint4*>(Vp), Pp, pp);
  return cudaGetLastError();
}

}  // namespace kvc
