// Top-n selection with a deterministic tie rule, used twice on the path:
//  * KV² page, "어떻게 동작하나": inside each chunk C_r, the n_q positions with
//    the highest token score p become the reconstruction queries;
//  * KV² page, "무엇과 다른가": after gathering the scores, the sinks are
//    pinned to the max and the lowest-scored entries of every (layer, KV
//    head) are removed down to the budget.
// In both the lower position wins a tie and the output is in ascending
// position order.
//
// One CTA per segment: a 4-digit (8-bit) MSB-first radix select finds the
// n-th largest key T over the segment (float -> order-preserving uint32;
// NaN maps below -inf, -0 to +0), then one ordered pass keeps every key > T
// and the lowest-positioned keys == T, writing positions through a
// block-wide prefix count.
#include <cstring>

#include "kvc_internal.h"
#include "kvc_ptx.cuh"

namespace kvc {
namespace {

constexpr int THREADS = 1024;
constexpr int WARPS = THREADS / 32;

__device__ __forceinline__ uint32_t order_key(float x) {
  if (x != x) return 0u;                       // NaN ranks lowest
  uint32_t u = __float_as_uint(x + 0.0f);      // -0 -> +0
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
__device__ __forceinline__ float key_value(uint32_t k) {
  const uint32_t u = (k & 0x80000000u) ? (k & 0x7fffffffu) : ~k;
  return __uint_as_float(u);
}

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
__device__ uint32_t radix_threshold(const float* __restrict__ vals, int lo, int hi, uint32_t n, SelectSmem& sm,
                                    uint32_t* cnt_gt, bool want_max) {
  uint32_t prefix = 0, mask = 0, remaining = n;
  uint32_t localmax = 0;
  for (int shift = 24; shift >= 0; shift -= 8) {
    for (int b = threadIdx.x; b < 256; b += THREADS) sm.hist[b] = 0;
    __syncthreads();
    for (int i = lo + threadIdx.x; i < hi; i += THREADS) {
      const uint32_t k = order_key(vals[i]);
      if (want_max && shift == 24) localmax = max(localmax, k);
      if ((k & mask) == prefix) atomicAdd(&sm.hist[(k >> shift) & 255u], 1u);
    }
    __syncthreads();
    if (threadIdx.x < 32) {
      // bins from the top: lane l covers bins 255-8l .. 248-8l
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
      const bool here = excl < remaining && incl >= remaining;
      if (here) {
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
  *cnt_gt = n - remaining;  // keys strictly above T
  return prefix;
}

// Writes, in ascending position order, every position of [lo, hi) whose key
// is > T plus the first `need_eq` positions whose key == T.
__device__ void emit_selected(const float* __restrict__ vals, int lo, int hi, uint32_t T, uint32_t need_eq,
                              int32_t* __restrict__ out, SelectSmem& sm) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    sm.base_sel = 0;
    sm.base_eq = 0;
  }
  __syncthreads();
  for (int b0 = lo; b0 < hi; b0 += THREADS) {
    const int i = b0 + threadIdx.x;
    uint32_t k = 0;
    bool in = i < hi;
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
    if (take) out[sel_before] = i;
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

// ---------------------------------------------------------------- select
struct SelParams {
  int N, sinks, m, n_chunks, nq_full, nq_last;
};

__global__ void __launch_bounds__(THREADS) select_kernel(const float* __restrict__ p, SelParams P,
                                                         int32_t* __restrict__ sel) {
  __shared__ SelectSmem sm;
  const int r = blockIdx.x;
  const int lo = P.sinks + r * P.m;
  const int hi = min(lo + P.m, P.N);
  const uint32_t n = (r == P.n_chunks - 1) ? P.nq_last : P.nq_full;
  int32_t* out = sel + static_cast<int64_t>(r) * P.nq_full;
  uint32_t gt;
  const uint32_t T = radix_threshold(p, lo, hi, n, sm, &gt, false);
  emit_selected(p, lo, hi, T, n - gt, out, sm);
}

// ---------------------------------------------------------------- evict
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

}  // namespace

cudaError_t launch_select(const float* p, int N, int sinks, const ChunkPlan& plan, double rho, int32_t* sel,
                          cudaStream_t st) {
  (void)rho;
  SelParams sp{N, sinks, plan.m, plan.n_chunks, plan.nq_full, plan.nq_last};
  ProfScope ps("select_topk", st);
  select_kernel<<<plan.n_chunks, THREADS, 0, st>>>(p, sp, sel);
  return cudaGetLastError();
}

cudaError_t launch_evict(float* score, const EvictParams& ep, int32_t* kept, uint32_t* gmax_word, bool pin,
                         cudaStream_t st) {
  if (gmax_word) {
    cudaError_t e = cudaMemsetAsync(gmax_word, 0, sizeof(uint32_t), st);
    if (e != cudaSuccess) return e;
  }
  dim3 grid(ep.Hkv, ep.L);
  {
    ProfScope ps("evict_topk", st);
    evict_kernel<<<grid, THREADS, 0, st>>>(score, ep, kept, gmax_word);
  }
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess || !pin || !gmax_word) return e;
  ProfScope ps("pin_sinks", st);
  pin_kernel<<<grid, 32, 0, st>>>(score, ep, gmax_word);
  return cudaGetLastError();
}

}  // namespace kvc
