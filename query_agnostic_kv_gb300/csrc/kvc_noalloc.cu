// Allocation-free variant of the KeyDiff proxy entry point.
//
// kvc_proxy_score needs L*Hkv*N floats of scratch for the per-head scores
// before they are averaged into p; normally the caller passes that in a
// workspace it allocated.  Some callers cannot allocate device memory at the
// point where they want the proxy: serving runtimes that hand all free HBM
// to their own block pool at start-up, and latency-critical paths that may
// not call cudaMalloc because it can synchronise the whole device.  For
// them this file keeps the scratch in a fixed-size array in the library's
// own device memory instead.
//
// The array is reserved on a GPU when this module is first loaded there and
// stays reserved until the process exits (16 MiB per GPU).  Calls on the
// same device share it, so calls that overlap on the GPU (different streams
// without ordering between them) race on it.  Nothing in it needs clearing:
// every call overwrites all L*Hkv*N entries it reads.
#include <mutex>

#include "../../include/kvc.h"
#include "kvc_internal.h"

namespace kvc {
namespace {

constexpr size_t kScratchFloats = size_t(1) << 22;  // 4 Mi floats = 16 MiB
static __device__ __align__(256) float g_proxy_scratch[kScratchFloats];

constexpr int kMaxDev = 64;
std::mutex g_mu_noalloc;
float* g_scratch_ptr[kMaxDev];

}  // namespace
}  // namespace kvc

extern "C" kvc_status kvc_proxy_score_noalloc(kvc_shape shape, const void* K, float* p, kvc_stream stream) {
  using namespace kvc;
  if (shape.L < 1 || shape.Hkv < 1 || shape.Hq < shape.Hkv || shape.Hq % shape.Hkv != 0 || shape.d != kHeadDim ||
      shape.N < 1 || !K || !p || (reinterpret_cast<uintptr_t>(K) & 15u) != 0)
    return KVC_ERR_INVALID;
  if (!device_can_read(K) || !device_can_read(p)) return KVC_ERR_INVALID;
  const size_t need = static_cast<size_t>(shape.L) * shape.Hkv * shape.N;
  if (need > kScratchFloats) return KVC_ERR_WORKSPACE;  // larger than the built-in scratch
  const kvc_status dc = kvc_device_check();
  if (dc != KVC_OK) return dc;
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDev) return KVC_ERR_CUDA;
  float* scratch = nullptr;
  {
    // Set-up, once per device, with that device current: the host-side name
    // of the array is not a device address, so ask the runtime for it.
    std::lock_guard<std::mutex> lk(g_mu_noalloc);
    if (!g_scratch_ptr[dev]) {
      void* q = nullptr;
      if (cudaGetSymbolAddress(&q, g_proxy_scratch) != cudaSuccess || !q) return KVC_ERR_CUDA;
      g_scratch_ptr[dev] = static_cast<float*>(q);
    }
    scratch = g_scratch_ptr[dev];
  }
  const cudaError_t e = launch_proxy(K, shape.L * shape.Hkv, shape.N, scratch, p,
                                     reinterpret_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? KVC_OK : KVC_ERR_CUDA;
}
