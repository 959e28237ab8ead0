// 4-bit (Q4) codec of a compacted KV cache ("Agent Memory Below the Prompt:
// Persistent Q4 KV Cache for Multi-Agent LLM Inference on Edge Devices",
// "방법론 및 시스템 설계": each agent's cache is kept 4-bit quantized and loaded
// straight back into attention).  The page fixes no format; this codec is an
// affine group quantiser over groups of 64 values of a 128-value row:
//   offset = min rounded down to bf16, step = (max - offset) / 15 rounded up
//   to bf16 (0 for a constant group), code = clamp(rint((x - offset) / step),
//   0, 15), two codes per byte (even element in the low nibble);
//   decode = bf16_rn(c * step + offset) with separately rounded fp32 ops.
// Every decision uses IEEE-rounded fp32 intrinsics (no contraction), and the
// code division is resolved exactly (see the encoder), so results are
// bit-exact with a plain fp32 restatement.
//
// Both kernels: 8 lanes per group (one 16-byte load or store of 8 bf16 each),
// a warp covers 2 rows, grid-stride over rows.  The decoder's inputs may be
// page-locked host memory read in place (72 bytes per row cross the link,
// 256 bytes per row are written to HBM).
#include <cuda_bf16.h>

#include "kvc_internal.h"
#include "kvc_ptx.cuh"

namespace kvc {
namespace {

constexpr int THREADS = 256;
constexpr int ROWS_PER_BLOCK = THREADS / 16;   // 16 lanes per row

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

constexpr int PAIRS = 4;   // row pairs a warp loads before it computes (memory parallelism)

// bf16x2 minimum of two packed pairs (exact: a selection per half).
__device__ __forceinline__ uint32_t bmin2(uint32_t a, uint32_t b) {
  const __nv_bfloat162 r = __hmin2(*reinterpret_cast<const __nv_bfloat162*>(&a),
                                   *reinterpret_cast<const __nv_bfloat162*>(&b));
  return *reinterpret_cast<const uint32_t*>(&r);
}

// One group of 64 values held by 8 lanes (8 values each): step, offset and
// the lane's 8 codes packed into 32 bits.
__device__ __forceinline__ void encode_group(const uint4 w, uint32_t& packed, uint32_t& param) {
  const uint32_t ww[4] = {w.x, w.y, w.z, w.w};
  // min and max travel together as the packed pair (min, -max): one bf16x2
  // minimum updates both, one shuffle moves both
  uint32_t mm;
  {
    const uint32_t m01 = bmin2(ww[0], ww[1]), m23 = bmin2(ww[2], ww[3]);
    const uint32_t n01 = bmin2(ww[0] ^ 0x80008000u, ww[1] ^ 0x80008000u);
    const uint32_t n23 = bmin2(ww[2] ^ 0x80008000u, ww[3] ^ 0x80008000u);
    const uint32_t lo2 = bmin2(m01, m23), nhi2 = bmin2(n01, n23);   // (min, min) and (-max, -max) of the halves
    const uint32_t a = __byte_perm(lo2, nhi2, 0x5410);              // (lo2.lo, nhi2.lo)
    const uint32_t b = __byte_perm(lo2, nhi2, 0x7632);              // (lo2.hi, nhi2.hi)
    mm = bmin2(a, b);
  }
#pragma unroll
  for (int o = 1; o < 8; o <<= 1) mm = bmin2(mm, __shfl_xor_sync(0xffffffffu, mm, o));
  float mn = bf16_lo(mm);
  const float mx = -bf16_hi(mm);
  mn = __fadd_rn(mn, 0.f);                  // -0 -> +0: min over {-0, +0} may give either
  const __nv_bfloat16 lo_h = __float2bfloat16_rd(mn);
  const float lo = __bfloat162float(lo_h);
  __nv_bfloat16 s_h = __float2bfloat16_rn(0.f);
  if (mx != mn) s_h = __float2bfloat16_ru(__fdiv_rn(__fsub_rn(mx, lo), 15.f));
  const float s = __bfloat162float(s_h);
  // code = rint(RN(a / s)) with a = x - offset in [0, 15 s].  The product
  // t = RN(a * RN(1/s)) is within 2^-23 |a/s| <= 1.9e-6 of a/s, and RN(a/s)
  // within 9.3e-7 of it, so unless t lies within 1e-4 of a half-integer
  // both round to the same integer; inside that window the IEEE quotient
  // itself is taken.  Subnormal steps (1/s would overflow) always divide.
  const bool fast = s >= 1.17549435e-38f;              // 2^-126, the smallest normal float
  const float rs = fast ? __frcp_rn(s) : 0.f;
  // rint(t) for 0 <= t < 2^22: RN(t + 2^23) holds it, ties to even, in its
  // low mantissa bits (a >= 0 because the offset is at most the minimum).
  // Both values of a 32-bit word are processed as one packed f32x2 pair
  // (IEEE round-to-nearest like the scalar operations); t - rint(t) is one
  // fused a*b+c with b = -1 (exact negation, one rounding).  a <= 15 s up to
  // one rounding, so t < 15.5 and rint(t) <= 15: the low 4 bits are the code.
  constexpr float kMagic = 8388608.f;                  // 2^23
  const uint64_t nlo2 = pack2(-lo, -lo), rs2 = pack2(rs, rs);
  const uint64_t mg2 = pack2(kMagic, kMagic), nmg2 = pack2(-kMagic, -kMagic), m1 = pack2(-1.f, -1.f);
  uint64_t a2[4], m2[4];
  bool near = false;
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    a2[k] = add2(pack2(bf16_lo(ww[k]), bf16_hi(ww[k])), nlo2);
    const uint64_t t2 = mul2(a2[k], rs2);
    m2[k] = add2(t2, mg2);
    const uint64_t d2 = fma2(add2(m2[k], nmg2), m1, t2);   // t - rint(t)
    float d0, d1;
    unpack2(d2, d0, d1);
    near |= (fabsf(d0) > 0.4999f) | (fabsf(d1) > 0.4999f);
  }
  near = (near || !fast) && s > 0.f;
  if (__any_sync(0xffffffffu, near)) {                 // rare: resolve near-ties with the IEEE quotient
    if (near) {
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        float a0, a1, mm0, mm1;
        unpack2(a2[k], a0, a1);
        unpack2(m2[k], mm0, mm1);
        const float t0 = __fmul_rn(a0, rs), t1 = __fmul_rn(a1, rs);
        if (!fast || fabsf(__fsub_rn(t0, __fsub_rn(mm0, kMagic))) > 0.4999f) mm0 = __fadd_rn(__fdiv_rn(a0, s), kMagic);
        if (!fast || fabsf(__fsub_rn(t1, __fsub_rn(mm1, kMagic))) > 0.4999f) mm1 = __fadd_rn(__fdiv_rn(a1, s), kMagic);
        m2[k] = pack2(mm0, mm1);
      }
    }
  }
  packed = 0;
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    float mm0, mm1;
    unpack2(m2[k], mm0, mm1);
    packed |= ((__float_as_uint(mm0) & 0xfu) | ((__float_as_uint(mm1) & 0xfu) << 4)) << (8 * k);
  }
  param = static_cast<uint32_t>(__bfloat16_as_ushort(s_h)) | (static_cast<uint32_t>(__bfloat16_as_ushort(lo_h)) << 16);
}

__global__ void __launch_bounds__(THREADS) q4_encode_kernel(int64_t rows, const uint4* __restrict__ X,
                                                            uint32_t* __restrict__ codes,
                                                            uint32_t* __restrict__ params) {
  const int li = threadIdx.x & 7;           // lane within the group
  const int g = (threadIdx.x >> 3) & 1;     // group within the row
  const int half = (threadIdx.x >> 4) & 1;  // row of the pair
  const int64_t warp_rows = 2 * PAIRS;
  const int64_t stride = int64_t(gridDim.x) * (THREADS / 32) * warp_rows;
  // The loop runs over the warp's block of rows, so every lane takes the
  // same trips and the shuffles always see the full warp.
  for (int64_t base = (int64_t(blockIdx.x) * (THREADS / 32) + (threadIdx.x >> 5)) * warp_rows; base < rows;
       base += stride) {
    uint4 w[PAIRS];
#pragma unroll
    for (int p = 0; p < PAIRS; ++p) {
      const int64_t r = base + 2 * p + half;
      w[p] = r < rows ? X[r * 16 + g * 8 + li] : make_uint4(0u, 0u, 0u, 0u);
    }
#pragma unroll
    for (int p = 0; p < PAIRS; ++p) {
      const int64_t r = base + 2 * p + half;
      uint32_t packed, param;
      encode_group(w[p], packed, param);
      if (r < rows) {
        codes[r * 16 + g * 8 + li] = packed;
        if (li == 0) params[r * 2 + g] = param;
      }
    }
  }
}

__global__ void __launch_bounds__(THREADS) q4_decode_kernel(int64_t rows, const uint32_t* __restrict__ codes,
                                                            const uint32_t* __restrict__ params,
                                                            uint4* __restrict__ X) {
  const int li = threadIdx.x & 7;
  const int g = (threadIdx.x >> 3) & 1;
  const int rs = threadIdx.x >> 4;
  for (int64_t r = int64_t(blockIdx.x) * ROWS_PER_BLOCK + rs; r < rows;
       r += int64_t(gridDim.x) * ROWS_PER_BLOCK) {
    const uint32_t packed = codes[r * 16 + g * 8 + li];
    const uint32_t pr = params[r * 2 + g];
    const float s = bf16_lo(pr);
    const float lo = bf16_hi(pr);
    uint32_t out[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const float c0 = static_cast<float>((packed >> (8 * k)) & 0xfu);
      const float c1 = static_cast<float>((packed >> (8 * k + 4)) & 0xfu);
      const __nv_bfloat16 a = __float2bfloat16_rn(__fadd_rn(__fmul_rn(c0, s), lo));
      const __nv_bfloat16 b = __float2bfloat16_rn(__fadd_rn(__fmul_rn(c1, s), lo));
      out[k] = static_cast<uint32_t>(__bfloat16_as_ushort(a)) | (static_cast<uint32_t>(__bfloat16_as_ushort(b)) << 16);
    }
    X[r * 16 + g * 8 + li] = make_uint4(out[0], out[1], out[2], out[3]);
  }
}

int grid_for(int64_t rows, int rows_per_block) {
  const int64_t need = (rows + rows_per_block - 1) / rows_per_block;
  const int64_t cap = int64_t(num_sms()) * 8;     // 8 blocks of 256 threads per SM
  return static_cast<int>(need < cap ? need : cap);
}

}  // namespace

cudaError_t launch_q4_encode(int64_t rows, const void* X, void* codes, void* params, cudaStream_t st) {
  if (rows == 0) return cudaSuccess;
  ProfScope ps("q4_encode", st);
  q4_encode_kernel<<<grid_for(rows, (THREADS / 32) * 2 * PAIRS), THREADS, 0, st>>>(rows, static_cast<const uint4*>(X),
                                                       static_cast<uint32_t*>(codes), static_cast<uint32_t*>(params));
  return cudaGetLastError();
}

cudaError_t launch_q4_decode(int64_t rows, const void* codes, const void* params, void* X, cudaStream_t st) {
  if (rows == 0) return cudaSuccess;
  ProfScope ps("q4_decode", st);
  q4_decode_kernel<<<grid_for(rows, ROWS_PER_BLOCK), THREADS, 0, st>>>(rows, static_cast<const uint32_t*>(codes),
                                                       static_cast<const uint32_t*>(params), static_cast<uint4*>(X));
  return cudaGetLastError();
}

}  // namespace kvc
