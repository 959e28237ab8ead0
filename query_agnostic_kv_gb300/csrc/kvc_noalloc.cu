// Allocation-free variant of the KeyDiff proxy entry point.
//
// kvc_proxy_score needs scratch device memory -- the L*Hkv*N per-head scores
// before they are averaged into p -- which the caller normally passes as a
// workspace it allocated.  Some callers cannot allocate device memory at the point
// where they want the proxy: serving runtimes that hand all free HBM to
// their own block pool at start-up, and latency-critical paths that may not
// call cudaMalloc because it can synchronise the whole device.  For them
// this file keeps the scratch in a fixed-size array in the library's own
// device memory instead.
//
// The array is reserved on a GPU when this module is first loaded there and
// stays reserved until the process exits (16 MiB per GPU).  Calls on the
// same device share it, so calls that overlap on the GPU (different streams
// without ordering between them) race on it.  Nothing in it needs clearing:
// every call overwrites all the entries it reads.
#include "../../include/kvc.h"
#include "kvc_internal.h"

namespace kvc {
namespace {

constexpr size_t kScratchBytes = size_t(16) << 20;  // 16 MiB
static __device__ __align__(256) unsigned char g_proxy_scratch[kScratchBytes];

// the array's device address per device, keyed by context (see symbol_address)
SymbolSlot g_scratch_slot[64];

}  // namespace
}  // namespace kvc

extern "C" kvc_status kvc_proxy_score_noalloc(kvc_shape shape, const void* K, float* p, kvc_stream stream) {
  using namespace kvc;
  if (!shape_ok(shape) || !K || !p || (reinterpret_cast<uintptr_t>(K) & 15u) != 0) return KVC_ERR_INVALID;
  if (!device_can_read(K) || !device_can_read(p)) return KVC_ERR_INVALID;
  const int LH = shape.L * shape.Hkv;
  const size_t s_bytes = (static_cast<size_t>(LH) * shape.N * sizeof(float) + 255) & ~size_t(255);
  if (s_bytes + proxy_scratch_bytes(LH, shape.N) > kScratchBytes)
    return KVC_ERR_WORKSPACE;  // larger than the built-in scratch
  const kvc_status dc = kvc_device_check();
  if (dc != KVC_OK) return dc;
  // The host-side name of the array is not a device address: ask the
  // runtime for the address on the current device (cached per device and
  // context; the first call on a device does the lookup).
  char* base = static_cast<char*>(symbol_address(g_proxy_scratch, g_scratch_slot));
  if (!base) return KVC_ERR_CUDA;
  const cudaError_t e = launch_proxy(K, LH, shape.N, reinterpret_cast<float*>(base), p, base + s_bytes,
                                     reinterpret_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? KVC_OK : KVC_ERR_CUDA;
}
