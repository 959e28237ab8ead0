// Headwise compaction (KV² page, "전제와 한계": serving needs the masked cache
// physically compacted per head) and the block append of EpiCache's
// block-wise prefill ("[26'ICML] EpiCache", "방법: 3단계" step ②).
//
// Both are row copies of 256-byte bf16 rows: half a warp moves one row as
// sixteen 16-byte loads and stores, rows of one (layer, KV head) per grid
// row, so reads and writes stay fully coalesced.
#include <cuda_bf16.h>

#include <cstring>

#include "kvc_internal.h"
#include "kvc_ptx.cuh"

namespace kvc {
namespace {

constexpr int THREADS = 256;
constexpr int ROWS_PER_BLOCK = 64;  // 16 half-warps x 4 rows

// Source and destination of layer l: the single buffers of a plain
// compaction, or (per-layer slabs) slab[l] -> its other slab.
struct CompactBufs {
  const uint4* K[2];
  const uint4* V[2];
  const int32_t* pos[2];
  uint4* Kd[2];
  uint4* Vd[2];
  int32_t* posd[2];
  int32_t slab[kMaxLayers];
};

__global__ void __launch_bounds__(THREADS) compact_kernel(const int32_t* __restrict__ idx,
                                                          const __grid_constant__ CompactBufs X,
                                                          const __grid_constant__ CompactParams P, int* status) {
  // One block per (layer, KV head, 64-row tile) of the active layers only:
  // layer l owns blocks [unit_off[l], unit_off[l+1]), head-major.  Budgets
  // that differ per layer leave no empty blocks behind (a (k_max/64, Hkv, L)
  // grid spent 8% of the EpiCache compaction on blocks that exit at once).
  const int u = blockIdx.x;
  int l = 0, hi = P.L;  // invariant: unit_off[l] <= u < unit_off[hi]
  while (hi - l > 1) {
    const int mid = (l + hi) >> 1;
    if (P.unit_off[mid] <= u) l = mid; else hi = mid;
  }
  const int k = P.k[l];
  const int sl = X.slab[l];
  const uint4* K = X.K[sl];
  const uint4* V = X.V[sl];
  const int32_t* pos_src = X.pos[sl];
  uint4* Kc = X.Kd[sl];
  uint4* Vc = X.Vd[sl];
  int32_t* pos_dst = X.posd[sl];
  const int tiles = (k + ROWS_PER_BLOCK - 1) / ROWS_PER_BLOCK;
  const int r = u - P.unit_off[l];
  const int h = r / tiles;
  const int t0 = (r - h * tiles) * ROWS_PER_BLOCK;
  const int64_t lh = static_cast<int64_t>(l) * P.Hkv + h;
  const int32_t* id = idx + P.idx_off[l] + static_cast<int64_t>(h) * k;
  const int64_t dst_base = (P.dst_ld >= 0) ? lh * P.dst_ld : P.dst_off[l] + static_cast<int64_t>(h) * k;
  const int64_t src_base = lh * P.src_ld;
  const int sub = threadIdx.x & 15;
  const int hw = threadIdx.x >> 4;
  int32_t src[4];
  uint4 kv[4], vv[4];
#pragma unroll
  for (int u = 0; u < 4; ++u) {
    const int t = t0 + u * 16 + hw;
    src[u] = -1;
    if (t < k) {
      const int s = id[t];
      if (s >= 0 && s < P.n_src[l]) {
        src[u] = s;
      } else if (sub == 0) {
        record_status(status, DEV_BOUNDS);
      }
    }
    if (src[u] >= 0) {
      kv[u] = __ldg(K + (src_base + src[u]) * 16 + sub);
      if (V) vv[u] = __ldg(V + (src_base + src[u]) * 16 + sub);
    }
  }
#pragma unroll
  for (int u = 0; u < 4; ++u) {
    const int t = t0 + u * 16 + hw;
    if (src[u] < 0) continue;
    Kc[(dst_base + t) * 16 + sub] = kv[u];
    if (V) Vc[(dst_base + t) * 16 + sub] = vv[u];
    if (pos_dst && sub == 0) pos_dst[dst_base + t] = pos_src ? pos_src[src_base + src[u]] : src[u];
  }
}

__global__ void __launch_bounds__(THREADS) append_kernel(const uint4* __restrict__ Kb, const uint4* __restrict__ Vb,
                                                         uint4* K0, uint4* V0, int32_t* pos0, uint4* K1, uint4* V1,
                                                         int32_t* pos1, const __grid_constant__ AppendParams P) {
  const int l = blockIdx.z, h = blockIdx.y;
  const int t0 = blockIdx.x * ROWS_PER_BLOCK;
  if (t0 >= P.B) return;
  const int64_t lh = static_cast<int64_t>(l) * P.Hkv + h;
  uint4* K = P.cur[l] ? K1 : K0;
  uint4* V = P.cur[l] ? V1 : V0;
  int32_t* pos = P.cur[l] ? pos1 : pos0;
  const int sub = threadIdx.x & 15;
  const int hw = threadIdx.x >> 4;
#pragma unroll
  for (int u = 0; u < 4; ++u) {
    const int t = t0 + u * 16 + hw;
    if (t >= P.B) continue;
    const int64_t src = (lh * P.B + t) * 16 + sub;
    const int64_t dst = (lh * P.ld + P.len[l] + t);
    K[dst * 16 + sub] = __ldg(Kb + src);
    if (t < P.vrows[l]) V[dst * 16 + sub] = __ldg(Vb + src);
    if (sub == 0) pos[dst] = static_cast<int32_t>(P.pos0 + t);
  }
}

}  // namespace

namespace {
cudaError_t launch_compact_bufs(const int32_t* idx, const CompactBufs& X, const CompactParams& cp, cudaStream_t st) {
  CompactParams p = cp;
  int64_t units = 0;
  for (int l = 0; l < p.L; ++l) {
    p.unit_off[l] = static_cast<int32_t>(units);
    if (p.active[l] && p.k[l] > 0) {
      units += static_cast<int64_t>(p.Hkv) * ((p.k[l] + ROWS_PER_BLOCK - 1) / ROWS_PER_BLOCK);
    }
  }
  if (units > 0x7fffffff) return cudaErrorInvalidValue;
  p.unit_off[p.L] = static_cast<int32_t>(units);
  if (units == 0) return cudaSuccess;
  const dim3 grid(static_cast<unsigned>(units));
  ProfScope ps("compact", st);
  compact_kernel<<<grid, THREADS, 0, st>>>(idx, X, p, status_word());
  return cudaGetLastError();
}
}  // namespace

cudaError_t launch_compact(const void* K, const void* V, const int32_t* idx, const int32_t* pos_src,
                           int32_t* pos_dst, void* Kc, void* Vc, const CompactParams& cp, cudaStream_t st) {
  CompactBufs X;
  memset(&X, 0, sizeof(X));
  X.K[0] = static_cast<const uint4*>(K);
  X.V[0] = static_cast<const uint4*>(V);
  X.pos[0] = pos_src;
  X.Kd[0] = static_cast<uint4*>(Kc);
  X.Vd[0] = static_cast<uint4*>(Vc);
  X.posd[0] = pos_dst;
  return launch_compact_bufs(idx, X, cp, st);
}

cudaError_t launch_compact_slabs(const int32_t* idx, const EvictCopy& copy, const CompactParams& cp, cudaStream_t st) {
  CompactBufs X;
  memset(&X, 0, sizeof(X));
  for (int i = 0; i < 2; ++i) {
    X.K[i] = static_cast<const uint4*>(copy.K[i]);
    X.V[i] = static_cast<const uint4*>(copy.V[i]);
    X.pos[i] = copy.pos[i];
    X.Kd[i] = static_cast<uint4*>(copy.Kd[i]);
    X.Vd[i] = static_cast<uint4*>(copy.Vd[i]);
    X.posd[i] = copy.posd[i];
  }
  for (int l = 0; l < cp.L; ++l) X.slab[l] = copy.slab[l];
  return launch_compact_bufs(idx, X, cp, st);
}

cudaError_t launch_append(const void* Kblk, const void* Vblk, void* K0, void* V0, int32_t* pos0, void* K1, void* V1,
                          int32_t* pos1, const AppendParams& ap, cudaStream_t st) {
  if (ap.B <= 0) return cudaSuccess;
  dim3 grid((ap.B + ROWS_PER_BLOCK - 1) / ROWS_PER_BLOCK, ap.Hkv, ap.L);
  ProfScope ps("block_append", st);
  append_kernel<<<grid, THREADS, 0, st>>>(static_cast<const uint4*>(Kblk), static_cast<const uint4*>(Vblk),
                                          static_cast<uint4*>(K0), static_cast<uint4*>(V0), pos0,
                                          static_cast<uint4*>(K1), static_cast<uint4*>(V1), pos1, ap);
  return cudaGetLastError();
}

}  // namespace kvc
