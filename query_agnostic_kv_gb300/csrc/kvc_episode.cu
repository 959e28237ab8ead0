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
// pack_ordered_kernel: the same image from a one-slab state, whose rows are
// in no particular order, written in ascending position order.  A row's
// packed index is the number of rows of its (layer, KV head) with a lower
// position: positions are distinct, so each CTA marks every position of its
// segment in a shared-memory bitmap (a window of 2^17 positions at a time),
// takes a prefix count over the bitmap's words, and reads each of its rows'
// ranks off it.
#include "kvc_internal.h"
#include "kvc_ptx.cuh"

namespace kvc {
namespace {

constexpr int MATCH_WARPS = 8;
constexpr int PACK_THREADS = 256;
constexpr int PACK_ROWS = 64;      // rows per block: 16 half-warps x 4
constexpr int OPACK_THREADS = 512;
constexpr int OPACK_ROWS = 1024;   // rows per block
constexpr int OPACK_WIN = 1 << 17; // positions per bitmap window
constexpr int OPACK_WORDS = OPACK_WIN / 32;

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


__global__ void __launch_bounds__(OPACK_THREADS) pack_ordered_kernel(const uint4* __restrict__ K0,
                                                                    const uint4* __restrict__ V0,
                                                                    const int32_t* __restrict__ P0,
                                                                    uint4* __restrict__ Kp, uint4* __restrict__ Vp,
                                                                    int32_t* __restrict__ Pp,
                                                                    const __grid_constant__ PackParams P) {
  __shared__ uint32_t bits[OPACK_WORDS];
  __shared__ uint32_t wpre[OPACK_WORDS];   // set bits in the words before each word
  __shared__ uint32_t tsum[OPACK_THREADS / 32];
  const int l = blockIdx.z, h = blockIdx.y;
  const int n = P.len[l];
  const int t0 = blockIdx.x * OPACK_ROWS;
  if (t0 >= n) return;
  const int t1 = min(t0 + OPACK_ROWS, n);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int64_t src_row = (static_cast<int64_t>(l) * P.Hkv + h) * P.cap;
  const int64_t dst_row = P.dst_off[l] + static_cast<int64_t>(h) * n;
  const int32_t* pos = P0 + src_row;
  const int sub = tid & 15, hw = tid >> 4;
  constexpr int HW = OPACK_THREADS / 16;
  constexpr int WPT = OPACK_WORDS / OPACK_THREADS;   // bitmap words per thread
  uint32_t base = 0;                                  // rows below the window
  for (int64_t w0 = 0; w0 < P.npos; w0 += OPACK_WIN) {
    for (int i = tid; i < OPACK_WORDS; i += OPACK_THREADS) bits[i] = 0u;
    __syncthreads();
    for (int t = tid; t < n; t += OPACK_THREADS) {
      const int64_t p = static_cast<int64_t>(pos[t]) - w0;
      if (p >= 0 && p < OPACK_WIN) atomicOr(&bits[p >> 5], 1u << (p & 31));
    }
    __syncthreads();
    // exclusive prefix of the words' popcounts: WPT consecutive words per
    // thread, then a scan over the threads
    uint32_t c[WPT], run = 0;
#pragma unroll
    for (int u = 0; u < WPT; ++u) {
      c[u] = run;
      run += __popc(bits[tid * WPT + u]);
    }
    uint32_t incl = run;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t v = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += v;
    }
    if (lane == 31) tsum[warp] = incl;
    __syncthreads();
    uint32_t before = 0, total = 0;
    for (int w = 0; w < OPACK_THREADS / 32; ++w) {
      before += w < warp ? tsum[w] : 0u;
      total += tsum[w];
    }
    const uint32_t excl = base + before + incl - run;
#pragma unroll
    for (int u = 0; u < WPT; ++u) wpre[tid * WPT + u] = excl + c[u];
    __syncthreads();
    // this block's rows whose position lies in the window; K rows, then V
    // rows, one half-warp per row, four in flight
    const int nt = t1 - t0;
    for (int ub = hw; ub < 2 * nt; ub += HW * 4) {
      int64_t dst[4];
      uint4 val[4];
      int32_t pv[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int w = ub + u * HW;
        dst[u] = -1;
        if (w < 2 * nt) {
          const int t = t0 + (w < nt ? w : w - nt);
          pv[u] = pos[t];
          const int64_t p = static_cast<int64_t>(pv[u]) - w0;
          if (p >= 0 && p < OPACK_WIN) {
            const int q = static_cast<int>(p);
            dst[u] = dst_row + wpre[q >> 5] + __popc(bits[q >> 5] & ((1u << (q & 31)) - 1u));
            val[u] = (w < nt ? K0 : V0)[(src_row + t) * 16 + sub];
          }
        }
      }
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        if (dst[u] < 0) continue;
        const bool isK = ub + u * HW < nt;
        (isK ? Kp : Vp)[dst[u] * 16 + sub] = val[u];
        if (isK && Pp && sub == 0) Pp[dst[u]] = pv[u];
      }
    }
    base += total;
    __syncthreads();    // the bitmap and prefix are rewritten for the next window
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
  if (pp.ordered) {
    static_assert(OPACK_WORDS % OPACK_THREADS == 0, "bitmap words split evenly over the threads");
    dim3 grid((max_len + OPACK_ROWS - 1) / OPACK_ROWS, pp.Hkv, pp.L);
    pack_ordered_kernel<<<grid, OPACK_THREADS, 0, st>>>(static_cast<const uint4*>(K0), static_cast<const uint4*>(V0),
                                                        P0, static_cast<uint4*>(Kp), static_cast<uint4*>(Vp), Pp, pp);
    return cudaGetLastError();
  }
  dim3 grid((max_len + PACK_ROWS - 1) / PACK_ROWS, pp.Hkv, pp.L);
  pack_kernel<<<grid, PACK_THREADS, 0, st>>>(
      static_cast<const uint4*>(K0), static_cast<const uint4*>(V0), P0, static_cast<const uint4*>(K1),
      static_cast<const uint4*>(V1), P1, static_cast<uint4*>(Kp), static_cast<uint4*>(Vp), Pp, pp);
  return cudaGetLastError();
}

}  // namespace kvc
