// C ABI: argument validation, status plumbing, host-side plans and the
// orchestration of the KV² pipeline and EpiCache block prefill.  All device
// work happens in the kernels of the other translation units.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstring>
#include <mutex>
#include <vector>

#include "../../include/kvc.h"
#include "kvc_internal.h"
#include "kvc_ptx.cuh"

namespace kvc {

__device__ int g_status_word;

namespace {
constexpr int kMaxDevices = 64;
std::mutex g_mu;
SymbolSlot g_status_slot[kMaxDevices];
int g_sms[kMaxDevices];
int g_cc_ok[kMaxDevices];  // 0 unknown, 1 ok, -1 unsupported
uint64_t g_limit_ns = 1000000000ull;
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

int current_device() {
  int d = 0;
  if (cudaGetDevice(&d) != cudaSuccess) return -1;
  return (d >= 0 && d < kMaxDevices) ? d : -1;
}

__global__ void expire_kernel(uint64_t limit_ns, int* status) {
  __shared__ uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    fence_barrier_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    // nothing ever arrives on `bar`: the wait must expire
    if (!mbar_wait(&bar, 0, limit_ns)) record_status(status, DEV_TIMEOUT);
  }
}
// ---- profiling state
struct ProfRecord {
  const char* name;
  cudaEvent_t ev0, ev1;
};
bool g_prof_on = false;
std::vector<ProfRecord> g_prof;
std::vector<cudaEvent_t> g_event_pool;
size_t g_event_next = 0;

cudaEvent_t pooled_event() {
  if (g_event_next < g_event_pool.size()) return g_event_pool[g_event_next++];
  cudaEvent_t e = nullptr;
  if (cudaEventCreate(&e) != cudaSuccess) return nullptr;
  g_event_pool.push_back(e);
  ++g_event_next;
  return e;
}
}  // namespace

ProfScope::ProfScope(const char* name, cudaStream_t st) : stream(st) {
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_prof_on) return;
  cudaEvent_t a = pooled_event(), b = pooled_event();
  if (!a || !b) return;
  cudaEventRecord(a, st);
  g_prof.push_back({name, a, b});
  slot = static_cast<int>(g_prof.size()) - 1;
}

ProfScope::~ProfScope() {
  if (slot < 0) return;
  std::lock_guard<std::mutex> lk(g_mu);
  if (slot < static_cast<int>(g_prof.size())) cudaEventRecord(g_prof[slot].ev1, stream);
}

namespace {
PFN_cuCtxGetCurrent_v4000 g_ctx_current = nullptr;
PFN_cuCtxGetId_v12000 g_ctx_id = nullptr;
std::once_flag g_ctx_once;

// Unique ID of the calling thread's current context (false when there is
// none yet, or the driver lacks the query).
bool context_id(unsigned long long* id) {
  std::call_once(g_ctx_once, [] {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &fn, 4000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_ctx_current = reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(fn);
    fn = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &fn, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_ctx_id = reinterpret_cast<PFN_cuCtxGetId_v12000>(fn);
    cudaGetLastError();
  });
  if (!g_ctx_current || !g_ctx_id) return false;
  CUcontext ctx = nullptr;
  if (g_ctx_current(&ctx) != CUDA_SUCCESS || !ctx) return false;
  return g_ctx_id(ctx, id) == CUDA_SUCCESS;
}
}  // namespace

void* symbol_address(const void* symbol, SymbolSlot* slots) {
  const int d = current_device();
  if (d < 0) return nullptr;
  unsigned long long id = 0;
  const bool have_id = context_id(&id);
  {
    std::lock_guard<std::mutex> lk(g_mu);
    if (have_id && slots[d].ptr && slots[d].ctx == id) return slots[d].ptr;
  }
  void* p = nullptr;
  if (cudaGetSymbolAddress(&p, symbol) != cudaSuccess || !p) {
    cudaGetLastError();
    return nullptr;
  }
  // cudaGetSymbolAddress made the primary context current if it was not yet
  unsigned long long id2 = 0;
  std::lock_guard<std::mutex> lk(g_mu);
  if (context_id(&id2)) {
    slots[d].ctx = id2;
    slots[d].ptr = p;
  } else {
    slots[d].ptr = nullptr;   // no context ID to key it by: look it up every time
  }
  return p;
}

int* status_word() { return static_cast<int*>(symbol_address(&g_status_word, g_status_slot)); }

uint64_t wait_limit_ns() { return g_limit_ns; }

int num_sms() {
  const int d = current_device();
  if (d < 0) return 1;
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_sms[d]) {
    int v = 0;
    cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, d);
    g_sms[d] = v > 0 ? v : 1;
  }
  return g_sms[d];
}

namespace {
bool encode_fn_ready() {
  std::lock_guard<std::mutex> lk(g_mu);
  if (g_encode) return true;
  void* fn = nullptr;
  cudaDriverEntryPointQueryResult q;
  if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) != cudaSuccess ||
      q != cudaDriverEntryPointSuccess || !fn)
    return false;
  g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  return true;
}
}  // namespace

bool make_tmap_rows16(CUtensorMap* map, const void* base, uint64_t rows, uint32_t box_rows) {
  if (!encode_fn_ready()) return false;
  if (rows == 0) rows = 1;
  cuuint64_t dims[2] = {16, static_cast<cuuint64_t>(rows)};
  cuuint64_t strides[1] = {32};
  cuuint32_t box[2] = {16, box_rows};
  cuuint32_t es[2] = {1, 1};
  const CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box,
                              es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_32B,
                              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

bool make_tmap_rows(CUtensorMap* map, const void* base, uint64_t rows, uint32_t box_rows) {
  if (!encode_fn_ready()) return false;
  if (rows == 0) rows = 1;
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(kHeadDim), static_cast<cuuint64_t>(rows)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(kHeadDim) * 2};
  cuuint32_t box[2] = {64, box_rows};
  cuuint32_t es[2] = {1, 1};
  const CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box,
                              es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

bool make_plan(int32_t N, int32_t sinks, int32_t m, double rho, ChunkPlan* plan) {
  if (N < 1 || sinks < 0 || sinks >= N || m < 1 || !(rho > 0.0) || !(rho <= 1.0)) return false;
  const int64_t body = static_cast<int64_t>(N) - sinks;
  const int64_t nc = (body + m - 1) / m;
  if (nc > (int64_t(1) << 30)) return false;
  auto nq = [&](int64_t len) {
    const int64_t v = static_cast<int64_t>(std::floor(rho * static_cast<double>(len) + 1e-9));
    return static_cast<int32_t>(v < 1 ? 1 : v);
  };
  plan->n_chunks = static_cast<int32_t>(nc);
  plan->m = static_cast<int32_t>(std::min<int64_t>(m, body));
  plan->last_len = static_cast<int32_t>(body - (nc - 1) * static_cast<int64_t>(m));
  plan->nq_full = nc > 1 ? nq(m) : nq(plan->last_len);
  plan->nq_last = nq(plan->last_len);
  const int64_t Q = (nc - 1) * static_cast<int64_t>(plan->nq_full) + plan->nq_last;
  if (Q > (int64_t(1) << 30)) return false;
  plan->Q = static_cast<int32_t>(Q);
  if (nc == 1) plan->m = m;  // keep the caller's chunk size for the single-chunk case
  return true;
}

}  // namespace kvc

using namespace kvc;

namespace {

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
}  // namespace

namespace kvc {

// Memory kind of `p` as the runtime sees it (cudaMemoryTypeUnregistered for
// ordinary host memory or an unknown address).
cudaMemoryType memory_type(const void* p, const void** device_view = nullptr) {
  cudaPointerAttributes a{};
  if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
    cudaGetLastError();
    return cudaMemoryTypeUnregistered;
  }
  if (device_view) *device_view = a.devicePointer;
  return a.type;
}

// Device or managed memory (what the tensor-map and device-only inputs need).
bool is_device_memory(const void* p) {
  const cudaMemoryType t = memory_type(p);
  return t == cudaMemoryTypeDevice || t == cudaMemoryTypeManaged;
}

// Whether the current device's kernels may read `p` in place: device or
// managed memory, page-locked host memory mapped at the same address, or
// ordinary host memory when the device reads pageable memory through the
// host's page tables (cudaDevAttrPageableMemoryAccess).  Anything else would
// make a kernel touch an unmapped address, so the call is refused instead.
bool device_can_read(const void* p) {
  const void* view = nullptr;
  const cudaMemoryType t = memory_type(p, &view);
  if (t == cudaMemoryTypeDevice || t == cudaMemoryTypeManaged) return true;
  if (t == cudaMemoryTypeHost) return view == p;
  int d = 0, pageable = 0;
  if (cudaGetDevice(&d) != cudaSuccess ||
      cudaDeviceGetAttribute(&pageable, cudaDevAttrPageableMemoryAccess, d) != cudaSuccess) {
    cudaGetLastError();
    return false;
  }
  return pageable != 0;
}

}  // namespace kvc

namespace {


kvc_status cuda_status(cudaError_t e) { return e == cudaSuccess ? KVC_OK : KVC_ERR_CUDA; }

// Every non-null pointer argument a kernel will dereference must be memory the
// device can reach (see device_can_read); otherwise the call is refused before
// any launch.
bool reachable() { return true; }
template <class T, class... R>
bool reachable(const T* p, const R*... rest) {
  return (p == nullptr || device_can_read(p)) && reachable(rest...);
}

}  // namespace

namespace kvc {
bool shape_ok(const kvc_shape& s) {
  if (s.L < 1 || s.L > kMaxLayers || s.Hkv < 1 || s.Hq < s.Hkv || s.Hq % s.Hkv != 0 || s.d != kHeadDim || s.N < 1)
    return false;
  // (layer, KV head) pairs index a grid dimension of the proxy and eviction kernels
  if (static_cast<int64_t>(s.L) * s.Hkv > 65535) return false;
  // row coordinates of TMA boxes are int32
  const int64_t rows = static_cast<int64_t>(s.L) * s.Hq * s.N;
  return rows < (int64_t(1) << 31);
}
}  // namespace kvc

namespace {

kvc_status device_ok() {
  const int d = current_device();
  if (d < 0) return KVC_ERR_CUDA;
  {
    std::lock_guard<std::mutex> lk(g_mu);
    if (g_cc_ok[d] == 1) return KVC_OK;
    if (g_cc_ok[d] == -1) return KVC_ERR_UNSUPPORTED;
  }
  int major = 0, minor = 0;
  if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, d) != cudaSuccess ||
      cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, d) != cudaSuccess)
    return KVC_ERR_CUDA;
  const bool ok = (major == 10 && minor == 3);
  std::lock_guard<std::mutex> lk(g_mu);
  g_cc_ok[d] = ok ? 1 : -1;
  return ok ? KVC_OK : KVC_ERR_UNSUPPORTED;
}

// The one workspace layout every KV² entry point carves.
struct KV2Workspace {
  uint32_t* gmax = nullptr;
  float* p = nullptr;
  int32_t* sel = nullptr;
  float* score = nullptr;  // also the per-head proxy scores
  void* pscratch = nullptr;  // KeyDiff work list and partial sums
  ReconWorkspace rw{};
  size_t bytes = 0;
  bool ok = false;
};

KV2Workspace carve_kv2(const kvc_shape& s, const ChunkPlan& plan, void* base, size_t cap) {
  KV2Workspace w;
  Carver c(base, base ? cap : 0);
  const int G = s.Hq / s.Hkv;
  const int64_t LH = static_cast<int64_t>(s.L) * s.Hkv;
  w.gmax = c.take<uint32_t>(64);
  w.p = c.take<float>(s.N);
  w.sel = c.take<int32_t>(plan.Q);
  w.score = c.take<float>(LH * s.N);
  w.pscratch = c.take<uint8_t>(proxy_scratch_bytes(static_cast<int>(LH), s.N));
  w.rw.Rpad = recon_rows(G, plan.n_chunks, plan.nq_full, plan.nq_last);
  w.rw.Qg = c.take<uint16_t>(LH * w.rw.Rpad * kHeadDim);
  w.rw.Kg = c.take<uint16_t>(LH * plan.Q * kHeadDim);
  w.rw.lsx = c.take<uint16_t>(LH * w.rw.Rpad * 16);
  w.bytes = ((c.used + 255) & ~size_t(255)) + 256;
  w.ok = c.ok;
  return w;
}

kvc_status check_ws(void* ws, size_t ws_bytes, size_t need) {
  if (!ws || (reinterpret_cast<uintptr_t>(ws) & 255u) != 0 || ws_bytes < need) return KVC_ERR_WORKSPACE;
  return KVC_OK;
}

cudaStream_t cs(kvc_stream s) { return reinterpret_cast<cudaStream_t>(s); }

// Caller-supplied appended keys are a tensor-map source like K: device
// memory, 16-byte aligned (or absent).
bool kapp_ok(const void* Kapp) { return !Kapp || (aligned16(Kapp) && is_device_memory(Kapp)); }

kvc_status run_recon(const kvc_shape& s, const ChunkPlan& plan, int32_t sinks, const void* K, const void* Qpool,
                     const int32_t* sel, const void* Kapp, float* score, float* lse_out, const KV2Workspace& w,
                     cudaStream_t st, cudaEvent_t gather_done = nullptr, int phases = RECON_ALL) {
  ReconProblem pr;
  memset(&pr, 0, sizeof(pr));
  pr.L = s.L;
  pr.Hkv = s.Hkv;
  pr.Hq = s.Hq;
  pr.G = s.Hq / s.Hkv;
  pr.sinks = sinks;
  pr.n_active = s.L;
  for (int l = 0; l < s.L; ++l) {
    pr.lay[l].layer = l;
    pr.lay[l].n = s.N;
    pr.lay[l].m = plan.m;
    pr.lay[l].n_chunks = plan.n_chunks;
    pr.lay[l].last_len = plan.last_len;
    pr.lay[l].slab = 0;
  }
  pr.K[0] = K;
  pr.K[1] = nullptr;
  pr.ldK = s.N;
  pr.Qsrc = Qpool;
  pr.ldQ = s.N;
  pr.sel = sel;
  pr.Kapp = Kapp;
  pr.ldApp = plan.Q;
  pr.nq_full = plan.nq_full;
  pr.nq_last = plan.nq_last;
  pr.Q = plan.Q;
  pr.score = score;
  pr.ldS = s.N;
  pr.lse_out = lse_out;
  pr.gather_done = gather_done;
  return cuda_status(launch_recon(pr, w.rw, st, phases));
}

kvc_status run_evict(const kvc_shape& s, float* score, int32_t sinks, const int32_t* k_per_layer, int32_t* kept,
                     uint32_t* gmax, cudaStream_t st, const EvictCopy* copy = nullptr, bool pin = true) {
  EvictParams ep;
  memset(&ep, 0, sizeof(ep));
  ep.L = s.L;
  ep.Hkv = s.Hkv;
  ep.sinks = sinks;
  ep.ld = s.N;
  int64_t off = 0;
  for (int l = 0; l < s.L; ++l) {
    ep.n[l] = s.N;
    ep.k[l] = k_per_layer[l];
    ep.out_off[l] = off;
    ep.active[l] = 1;
    off += static_cast<int64_t>(s.Hkv) * k_per_layer[l];
  }
  return cuda_status(launch_evict(score, ep, kept, gmax, pin, copy, st));
}

kvc_status run_compact(const kvc_shape& s, const void* K, const void* V, const int32_t* kept,
                       const int32_t* k_per_layer, void* Kc, void* Vc, cudaStream_t st) {
  CompactParams cp;
  memset(&cp, 0, sizeof(cp));
  cp.L = s.L;
  cp.Hkv = s.Hkv;
  cp.src_ld = s.N;
  cp.dst_ld = -1;
  int64_t off = 0;
  for (int l = 0; l < s.L; ++l) {
    cp.n_src[l] = s.N;
    cp.k[l] = k_per_layer[l];
    cp.idx_off[l] = off;
    cp.dst_off[l] = off;
    cp.active[l] = 1;
    off += static_cast<int64_t>(s.Hkv) * k_per_layer[l];
  }
  return cuda_status(launch_compact(K, V, kept, nullptr, nullptr, Kc, Vc, cp, st));
}

kvc_status check_budgets(const kvc_shape& s, int32_t sinks, const int32_t* k_per_layer) {
  if (!k_per_layer) return KVC_ERR_INVALID;
  for (int l = 0; l < s.L; ++l)
    if (k_per_layer[l] < sinks || k_per_layer[l] > s.N) return KVC_ERR_INVALID;
  return KVC_OK;
}

}  // namespace

extern "C" {

const char* kvc_status_string(kvc_status s) {
  switch (s) {
    case KVC_OK: return "KVC_OK";
    case KVC_ERR_INVALID: return "KVC_ERR_INVALID: invalid argument";
    case KVC_ERR_CUDA: return "KVC_ERR_CUDA: CUDA call or launch failed";
    case KVC_ERR_TIMEOUT: return "KVC_ERR_TIMEOUT: a device-side wait expired";
    case KVC_ERR_BOUNDS: return "KVC_ERR_BOUNDS: a device-side index check failed";
    case KVC_ERR_WORKSPACE: return "KVC_ERR_WORKSPACE: workspace missing, misaligned or too small";
    case KVC_ERR_UNSUPPORTED: return "KVC_ERR_UNSUPPORTED: device is not sm_103";
  }
  return "KVC_ERR_UNKNOWN";
}

kvc_status kvc_device_check(void) { return device_ok(); }

kvc_status kvc_stream_status(kvc_stream stream) {
  if (cudaStreamSynchronize(cs(stream)) != cudaSuccess) return KVC_ERR_CUDA;
  int* w = status_word();
  if (!w) return KVC_ERR_CUDA;
  int v = 0;
  if (cudaMemcpy(&v, w, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess) return KVC_ERR_CUDA;
  if (v != 0) {
    const int zero = 0;
    if (cudaMemcpy(w, &zero, sizeof(int), cudaMemcpyHostToDevice) != cudaSuccess) return KVC_ERR_CUDA;
  }
  if (v == DEV_TIMEOUT) return KVC_ERR_TIMEOUT;
  if (v == DEV_BOUNDS) return KVC_ERR_BOUNDS;
  return v == 0 ? KVC_OK : KVC_ERR_CUDA;
}

kvc_status kvc_profile_begin(void) {
  std::lock_guard<std::mutex> lk(g_mu);
  g_prof.clear();
  g_event_next = 0;
  g_prof_on = true;
  return KVC_OK;
}

kvc_status kvc_profile_end(kvc_kernel_time* out, int32_t max_entries, int32_t* n_entries) {
  if (!n_entries || max_entries < 0 || (max_entries > 0 && !out)) return KVC_ERR_INVALID;
  if (cudaDeviceSynchronize() != cudaSuccess) return KVC_ERR_CUDA;
  std::lock_guard<std::mutex> lk(g_mu);
  g_prof_on = false;
  std::vector<kvc_kernel_time> acc;
  for (const ProfRecord& r : g_prof) {
    float ms = 0.f;
    if (cudaEventElapsedTime(&ms, r.ev0, r.ev1) != cudaSuccess) return KVC_ERR_CUDA;
    size_t i = 0;
    for (; i < acc.size(); ++i)
      if (strncmp(acc[i].name, r.name, sizeof(acc[i].name)) == 0) break;
    if (i == acc.size()) {
      kvc_kernel_time t;
      memset(&t, 0, sizeof(t));
      strncpy(t.name, r.name, sizeof(t.name) - 1);
      acc.push_back(t);
    }
    acc[i].launches += 1;
    acc[i].total_ms += ms;
  }
  g_prof.clear();
  g_event_next = 0;
  *n_entries = static_cast<int32_t>(acc.size());
  for (int32_t i = 0; i < max_entries && i < static_cast<int32_t>(acc.size()); ++i) out[i] = acc[i];
  return KVC_OK;
}

kvc_status kvc_set_wait_limit_ns(uint64_t limit_ns) {
  g_limit_ns = limit_ns ? limit_ns : 1000000000ull;
  return KVC_OK;
}

kvc_status kvc_debug_expire_wait(uint64_t limit_ns, kvc_stream stream) {
  if (limit_ns == 0 || limit_ns > 10000000000ull) return KVC_ERR_INVALID;
  kvc_status d = device_ok();
  if (d != KVC_OK) return d;
  int* w = status_word();
  if (!w) return KVC_ERR_CUDA;
  expire_kernel<<<1, 32, 0, cs(stream)>>>(limit_ns, w);
  return cuda_status(cudaGetLastError());
}

kvc_status kvc_chunk_plan(int32_t N, int32_t sinks, int32_t m, double rho, int32_t* n_chunks, int32_t* chunk_off) {
  ChunkPlan p;
  if (!n_chunks || !make_plan(N, sinks, m, rho, &p)) return KVC_ERR_INVALID;
  *n_chunks = p.n_chunks;
  if (chunk_off) {
    for (int r = 0; r <= p.n_chunks; ++r) chunk_off[r] = (r < p.n_chunks) ? r * p.nq_full : p.Q;
  }
  return KVC_OK;
}

kvc_status kvc_budget_count(double b, int32_t N, int32_t sinks, int32_t* k) {
  if (!k || N < 1 || !(b > 0.0) || !(b <= 1.0)) return KVC_ERR_INVALID;
  const int64_t v = static_cast<int64_t>(std::floor(b * static_cast<double>(N) + 1e-9));
  if (v < sinks || v > N) return KVC_ERR_INVALID;
  *k = static_cast<int32_t>(v);
  return KVC_OK;
}

size_t kvc_workspace_size(kvc_shape shape, int32_t sinks, int32_t m, double rho) {
  ChunkPlan p;
  if (!shape_ok(shape) || !make_plan(shape.N, sinks, m, rho, &p)) return 0;
  return carve_kv2(shape, p, nullptr, 0).bytes;
}

size_t kvc_proxy_workspace_size(kvc_shape shape, int32_t with_scores) {
  if (!shape_ok(shape)) return 0;
  const int LH = shape.L * shape.Hkv;
  Carver c(nullptr, 0);
  if (with_scores) c.take<float>(static_cast<size_t>(LH) * shape.N);
  c.take<uint8_t>(proxy_scratch_bytes(LH, shape.N));
  return (c.used + 255) & ~size_t(255);
}

kvc_status kvc_proxy_score(kvc_shape shape, const void* K, float* p, float* s_opt, void* ws, size_t ws_bytes,
                           kvc_stream stream) {
  return kvc_proxy_score_kind(shape, KVC_PROXY_KEYDIFF, K, p, s_opt, ws, ws_bytes, stream);
}

kvc_status kvc_proxy_score_kind(kvc_shape shape, kvc_proxy_kind kind, const void* K, float* p, float* s_opt,
                                void* ws, size_t ws_bytes, kvc_stream stream) {
  if (!shape_ok(shape) || !K || !p || !aligned16(K) || (kind != KVC_PROXY_KEYDIFF && kind != KVC_PROXY_KNORM))
    return KVC_ERR_INVALID;
  if (!reachable(K, p, s_opt, ws)) return KVC_ERR_INVALID;
  // workspace: the per-head scores (when s_opt is NULL), then the KeyDiff
  // scratch
  const int LH = shape.L * shape.Hkv;
  Carver c(ws, ws ? ws_bytes : 0);
  float* s = s_opt ? s_opt : c.take<float>(static_cast<size_t>(LH) * shape.N);
  void* scratch = kind == KVC_PROXY_KEYDIFF ? c.take<uint8_t>(proxy_scratch_bytes(LH, shape.N)) : nullptr;
  const bool need_ws = !s_opt || (kind == KVC_PROXY_KEYDIFF && proxy_scratch_bytes(LH, shape.N) > 0);
  if (need_ws && (!ws || (reinterpret_cast<uintptr_t>(ws) & 255u) != 0 || !c.ok)) return KVC_ERR_WORKSPACE;
  kvc_status d = device_ok();
  if (d != KVC_OK) return d;
  return cuda_status(kind == KVC_PROXY_KNORM ? launch_knorm(K, LH, shape.N, s, p, cs(stream))
                                             : launch_proxy(K, LH, shape.N, s, p, scratch, cs(stream)));
}

kvc_status kvc_proxy_partial(kvc_shape shape, kvc_proxy_kind kind, const void* K, float* psum, float* s_opt,
                             void* ws, size_t ws_bytes, kvc_stream stream) {
  if (!shape_ok(shape) || !K || !psum || !aligned16(K) || (kind != KVC_PROXY_KEYDIFF && kind != KVC_PROXY_KNORM))
    return KVC_ERR_INVALID;
  if (!reachable(K, psum, s_opt, ws)) return KVC_ERR_INVALID;
  const int LH = shape.L * shape.Hkv;
  float* s = s_opt;
  if (!s) {
    const size_t need = static_cast<size_t>(LH) * shape.N * sizeof(float);
    if (!ws || (reinterpret_cast<uintptr_t>(ws) & 255u) != 0 || ws_bytes < need) return KVC_ERR_WORKSPACE;
    s = static_cast<float*>(ws);
  }
  kvc_status d = device_ok();
  if (d != KVC_OK) return d;
  const cudaError_t e = launch_proxy_scores(kind == KVC_PROXY_KNORM ? 1 : 0, K, LH, shape.N, s, cs(stream));
  if (e != cudaSuccess) return KVC_ERR_CUDA;
  return cuda_status(launch_sum_heads(s, LH, shape.N, shape.N, 0, psum, cs(stream)));
}

kvc_status kvc_refine_partial(kvc_shape shape, const float* score, int32_t sinks, float* psum, kvc_stream stream) {
  if (!shape_ok(shape) || !score || !psum || sinks < 0 || sinks >= shape.N || !reachable(score, psum))
    return KVC_ERR_INVALID;
  kvc_status d = device_ok();
  if (d != KVC_OK) return d;
  return cuda_status(launch_sum_heads(score, shape.L * shape.Hkv, shape.N, shape.N, sinks, psum, cs(stream)));
}

kvc_status kvc_proxy_from_sums(int32_t N, int32_t total_heads, const float* psum, float* p, kvc_stream stream) {
  if (N < 1 || total_heads < 1 || !psum || !p || !reachable(psum, p)) return KVC_ERR_INVALID;
  kvc_status d = device_ok();
  if (d != KVC_OK) return d;
  return cuda_status(launch_sums_to_mean(psum, N, total_heads, p, cs(stream)));
}

kvc_status kvc_score_max(kvc_shape shape, const float* score, int32_t sinks, float* max_out, void* ws, size_t ws_bytes,
                         kvc_stream stream) {
  if (!shape_ok(shape) || !score || !max_out || sinks < 0 || sinks >= shape.N || !reachable(score, max_out, ws))
    return KVC_ERR_INVALID;
  if (!ws || (reinterpret_cast<uintptr_t>(ws) & 255u) != 0 || ws_bytes < 256) return KVC_ERR_WORKSPACE;
  kvc_status d = device_ok();
  if (d != KVC_OK) return d;
  return cuda_status(launch_score_max(score, shape.L * shape.Hkv, shape.N, sinks, static_cast<uint32_t*>(ws), max_out,
                                      cs(stream)));
}

kvc_status kvc_pin_sinks(kvc_shape shape, float* score, int32_t sinks, const float* value, kvc_stream stream) {
  if (!shape_ok(shape) || !score || !value || sinks < 0 || sinks >= shape.N || !reachable(score, value))
    return KVC_ERR_INVALID;
  kvc_status d = device_ok();
  if (d != KVC_OK) return d;
  return cuda_status(launch_pin_value(score, shape.L * shape.Hkv, shape.N, sinks, value, cs(stream)));
}

kvc_status kvc_select_queries(int32_t N, int32_t sinks, int32_t m, double rho, const float* p, int32_t* sel,
                              kvc_stream stream) {
  ChunkPlan plan;
  if (!p || !sel || !make_plan(N, sinks, m, rho, &plan) || !reachable(p, sel)) return KVC_ERR_INVALID;
  kvc_status d = device_ok();
  if (d != KVC_OK) return d;
  return cuda_status(launch_select(p, N, sinks, plan, rho, sel, cs(stream)));
}

kvc_status kvc_recon_score(kvc_shape shape, const void* K, const void* Qpool, const int32_t* sel, int32_t sinks,
                           int32_t m, double rho, const void* Kapp_opt, float* score, float* lse_opt, void* ws,
                           size_t ws_bytes, kvc_stream stream) {
  ChunkPlan plan;
  if (!shape_ok(shape) || !K || !Qpool || !sel || !score || !aligned16(K) || !aligned16(Qpool) ||
      !is_device_memory(K) || !device_can_read(Qpool) || !kapp_ok(Kapp_opt) ||
      !make_plan(shape.N, sinks, m, rho, &plan) || !reachable(sel, score, lse_opt, ws))
    return KVC_ERR_INVALID;
  KV2Workspace w = carve_kv2(shape, plan, ws, ws_bytes);
  kvc_status e = check_ws(ws, ws_bytes, w.bytes);
  if (e != KVC_OK || !w.ok) return KVC_ERR_WORKSPACE;
  kvc_status d = device_ok();
  if (d != KVC_OK) return d;
  return run_recon(shape, plan, sinks, K, Qpool, sel, Kapp_opt, score, lse_opt, w, cs(stream));
}

kvc_status kvc_recon_gather(kvc_shape shape, const void* K, const void* Qpool, const int32_t* sel, int32_t sinks,
                            int32_t m, double rho, const void* Kapp_opt, void* ws, size_t ws_bytes,
                            kvc_stream stream) {
  ChunkPlan plan;
  if (!shape_ok(shape) || !K || !Qpool || !sel || !aligned16(K) || !aligned16(Qpool) || !is_device_memory(K) ||
      !device_can_read(Qpool) || !kapp_ok(Kapp_opt) || !make_plan(shape.N, sinks, m, rho, &plan) ||
      !reachable(sel, ws))
    return KVC_ERR_INVALID;
  KV2Workspace w = carve_kv2(shape, plan, ws, ws_bytes);
  kvc_status e = check_ws(ws, ws_bytes, w.bytes);
  if (e != KVC_OK || !w.ok) return KVC_ERR_WORKSPACE;
  kvc_status d = device_ok();
  if (d != KVC_OK) return d;
  return run_recon(shape, plan, sinks, K, Qpool, sel, Kapp_opt, nullptr, nullptr, w, cs(stream), nullptr,
                   RECON_GATHER);
}

kvc_status kvc_recon_rows(kvc_shape shape, const void* K, int32_t sinks, int32_t m, double rho, const void* Kapp_opt,
                          float* lse_opt, void* ws, size_t ws_bytes, kvc_stream stream) {
  ChunkPlan plan;
  if (!shape_ok(shape) || !K || !aligned16(K) || !is_device_memory(K) || !kapp_ok(Kapp_opt) ||
      !make_plan(shape.N, sinks, m, rho, &plan) || !reachable(lse_opt, ws))
    return KVC_ERR_INVALID;
  KV2Workspace w = carve_kv2(shape, plan, ws, ws_bytes);
  kvc_status e = check_ws(ws, ws_bytes, w.bytes);
  if (e != KVC_OK || !w.ok) return KVC_ERR_WORKSPACE;
  kvc_status d = device_ok();
  if (d != KVC_OK) return d;
  return run_recon(shape, plan, sinks, K, nullptr, nullptr, Kapp_opt, nullptr, lse_opt, w, cs(stream), nullptr,
                   RECON_ROWS);
}

kvc_status kvc_recon_cols(kvc_shape shape, const void* K, int32_t sinks, int32_t m, double rho, float* score,
                          void* ws, size_t ws_bytes, kvc_stream stream) {
  ChunkPlan plan;
  if (!shape_ok(shape) || !K || !score || !aligned16(K) || !is_device_memory(K) ||
      !make_plan(shape.N, sinks, m, rho, &plan) || !reachable(score, ws))
    return KVC_ERR_INVALID;
  KV2Workspace w = carve_kv2(shape, plan, ws, ws_bytes);
  kvc_status e = check_ws(ws, ws_bytes, w.bytes);
  if (e != KVC_OK || !w.ok) return KVC_ERR_WORKSPACE;
  kvc_status d = device_ok();
  if (d != KVC_OK) return d;
  return run_recon(shape, plan, sinks, K, nullptr, nullptr, nullptr, score, nullptr, w, cs(stream), nullptr,
                   RECON_COLS);
}

kvc_status kvc_refine_proxy(kvc_shape shape, const float* score, int32_t sinks, float* p, kvc_stream stream) {
  if (!shape_ok(shape) || !score || !p || sinks < 0 || sinks >= shape.N || !reachable(score, p))
    return KVC_ERR_INVALID;
  kvc_status d = device_ok();
  if (d != KVC_OK) return d;
  return cuda_status(launch_mean_heads(score, shape.L * shape.Hkv, shape.N, shape.N, sinks, p, cs(stream)));
}

kvc_status kvc_evict_topk(kvc_shape shape, float* score, int32_t sinks, const int32_t* k_per_layer, int32_t* kept,
                          void* ws, size_t ws_bytes, kvc_stream stream) {
  if (!shape_ok(shape) || !score || !kept || sinks < 0 || sinks >= shape.N || !reachable(score, kept, ws))
    return KVC_ERR_INVALID;
  if (check_budgets(shape, sinks, k_per_layer) != KVC_OK) return KVC_ERR_INVALID;
  if (!ws || (reinterpret_cast<uintptr_t>(ws) & 255u) != 0 || ws_bytes < 256) return KVC_ERR_WORKSPACE;
  kvc_status d = device_ok();
  if (d != KVC_OK) return d;
  return run_evict(shape, score, sinks, k_per_layer, kept, static_cast<uint32_t*>(ws), cs(stream));
}

kvc_status kvc_evict_compact(kvc_shape shape, float* score, int32_t sinks, const int32_t* k_per_layer, int32_t* kept,
                             const void* K, const void* V, void* Kc, void* Vc, void* ws, size_t ws_bytes,
                             kvc_stream stream) {
  if (!shape_ok(shape) || !score || !kept || !K || !Kc || sinks < 0 || sinks >= shape.N ||
      (V == nullptr) != (Vc == nullptr) || !aligned16(K) || !aligned16(Kc) || (V && (!aligned16(V) || !aligned16(Vc))))
    return KVC_ERR_INVALID;
  if (!device_can_read(K) || (V && !device_can_read(V)) || !reachable(score, kept, Kc, Vc, ws)) return KVC_ERR_INVALID;
  if (check_budgets(shape, sinks, k_per_layer) != KVC_OK) return KVC_ERR_INVALID;
  if (!ws || (reinterpret_cast<uintptr_t>(ws) & 255u) != 0 || ws_bytes < 256) return KVC_ERR_WORKSPACE;
  kvc_status d = device_ok();
  if (d != KVC_OK) return d;
  EvictCopy cp;
  memset(&cp, 0, sizeof(cp));
  cp.K[0] = K;
  cp.V[0] = V;
  cp.Kd[0] = Kc;
  cp.Vd[0] = Vc;
  cp.src_ld = shape.N;
  cp.dst_ld = -1;
  return run_evict(shape, score, sinks, k_per_layer, kept, static_cast<uint32_t*>(ws), cs(stream), &cp);
}

kvc_status kvc_compact(kvc_shape shape, const void* K, const void* V, const int32_t* kept,
                       const int32_t* k_per_layer, void* Kc, void* Vc, kvc_stream stream) {
  if (!shape_ok(shape) || !K || !kept || !Kc || (V == nullptr) != (Vc == nullptr) || !aligned16(K) ||
      !aligned16(Kc) || (V && (!aligned16(V) || !aligned16(Vc))))
    return KVC_ERR_INVALID;
  if (!device_can_read(K) || (V && !device_can_read(V)) || !reachable(kept, Kc, Vc)) return KVC_ERR_INVALID;
  if (check_budgets(shape, 0, k_per_layer) != KVC_OK) return KVC_ERR_INVALID;
  kvc_status d = device_ok();
  if (d != KVC_OK) return d;
  return run_compact(shape, K, V, kept, k_per_layer, Kc, Vc, cs(stream));
}

kvc_status kvc_compress(kvc_shape shape, const void* K, const void* V, const void* Qpool, int32_t sinks, int32_t m,
                        double rho, int32_t passes, const int32_t* k_per_layer, int32_t* kept, void* Kc, void* Vc,
                        float* p_opt, int32_t* sel_opt, float* score_opt, void* ws, size_t ws_bytes,
                        kvc_stream stream) {
  return kvc_compress_ex(shape, KVC_PROXY_KEYDIFF, K, V, Qpool, sinks, m, rho, passes, k_per_layer, kept, Kc, Vc,
                         p_opt, sel_opt, score_opt, ws, ws_bytes, stream, nullptr);
}

kvc_status kvc_compress_ex(kvc_shape shape, kvc_proxy_kind proxy, const void* K, const void* V, const void* Qpool,
                           int32_t sinks, int32_t m, double rho, int32_t passes, const int32_t* k_per_layer,
                           int32_t* kept, void* Kc, void* Vc, float* p_opt, int32_t* sel_opt, float* score_opt,
                           void* ws, size_t ws_bytes, kvc_stream stream, kvc_event gather_done) {
  ChunkPlan plan;
  if (proxy != KVC_PROXY_KEYDIFF && proxy != KVC_PROXY_KNORM) return KVC_ERR_INVALID;
  if (!shape_ok(shape) || !K || !Qpool || !kept || !Kc || passes < 1 || (V == nullptr) != (Vc == nullptr) ||
      !aligned16(K) || !aligned16(Qpool) || !aligned16(Kc) || (V && (!aligned16(V) || !aligned16(Vc))) ||
      !make_plan(shape.N, sinks, m, rho, &plan))
    return KVC_ERR_INVALID;
  if (!is_device_memory(K) || !device_can_read(Qpool) || (V && !device_can_read(V)) ||
      !reachable(kept, Kc, Vc, p_opt, sel_opt, score_opt, ws))
    return KVC_ERR_INVALID;
  if (check_budgets(shape, sinks, k_per_layer) != KVC_OK) return KVC_ERR_INVALID;
  KV2Workspace w = carve_kv2(shape, plan, ws, ws_bytes);
  kvc_status e = check_ws(ws, ws_bytes, w.bytes);
  if (e != KVC_OK || !w.ok) return KVC_ERR_WORKSPACE;
  kvc_status d = device_ok();
  if (d != KVC_OK) return d;
  cudaStream_t st = cs(stream);
  float* p = p_opt ? p_opt : w.p;
  int32_t* sel = sel_opt ? sel_opt : w.sel;
  float* score = score_opt ? score_opt : w.score;
  const int LH = shape.L * shape.Hkv;
  // stage 1: proxy (per-head scratch in the score buffer)
  const cudaError_t pe = (proxy == KVC_PROXY_KNORM) ? launch_knorm(K, LH, shape.N, score, p, st)
                                                    : launch_proxy(K, LH, shape.N, score, p, w.pscratch, st);
  if (pe != cudaSuccess) return KVC_ERR_CUDA;
  for (int t = 0; t < passes; ++t) {
    if (launch_select(p, shape.N, sinks, plan, rho, sel, st) != cudaSuccess) return KVC_ERR_CUDA;
    kvc_status r = run_recon(shape, plan, sinks, K, Qpool, sel, nullptr, score, nullptr, w, st,
                             t + 1 == passes ? reinterpret_cast<cudaEvent_t>(gather_done) : nullptr);
    if (r != KVC_OK) return r;
    if (t + 1 < passes && launch_mean_heads(score, LH, shape.N, shape.N, sinks, p, st) != cudaSuccess)
      return KVC_ERR_CUDA;
  }
  // eviction and compaction in one launch: each (layer, KV head) copies its
  // kept K/V rows into the compacted cache as soon as it has chosen them
  EvictCopy cp;
  memset(&cp, 0, sizeof(cp));
  cp.K[0] = K;
  cp.V[0] = V;
  cp.Kd[0] = Kc;
  cp.Vd[0] = Vc;
  cp.src_ld = shape.N;
  cp.dst_ld = -1;
  // the sinks are kept by construction; their pinned score is written only
  // where the caller can read it
  return run_evict(shape, score, sinks, k_per_layer, kept, w.gmax, st, &cp, score_opt != nullptr);
}

kvc_status kvc_layer_budgets(const float* sens, int32_t L, double alpha, int64_t mean_budget, int32_t sinks,
                             int32_t* k_per_layer) {
  if (!sens || !k_per_layer || L < 1 || L > kMaxLayers || !(alpha >= 0.0) || mean_budget < 1 || sinks < 0)
    return KVC_ERR_INVALID;
  std::vector<double> w(L);
  double tot = 0.0;
  for (int l = 0; l < L; ++l) {
    if (!(sens[l] > 0.0f)) return KVC_ERR_INVALID;
    w[l] = std::pow(static_cast<double>(sens[l]), alpha);
    tot += w[l];
  }
  const int64_t total = static_cast<int64_t>(L) * mean_budget;
  if (total > (int64_t(1) << 40)) return KVC_ERR_INVALID;
  std::vector<int64_t> base(L);
  std::vector<double> frac(L);
  int64_t sum = 0;
  for (int l = 0; l < L; ++l) {
    const double q = static_cast<double>(total) * (w[l] / tot);
    base[l] = static_cast<int64_t>(std::floor(q));
    frac[l] = q - static_cast<double>(base[l]);
    sum += base[l];
  }
  int64_t rem = total - sum;
  std::vector<int> order(L);
  for (int l = 0; l < L; ++l) order[l] = l;
  std::stable_sort(order.begin(), order.end(), [&](int a, int b) { return frac[a] > frac[b]; });
  for (int i = 0; i < L && rem > 0; ++i, --rem) base[order[i]] += 1;
  for (int l = 0; l < L; ++l) {
    const int64_t v = std::max<int64_t>(base[l], sinks);
    if (v > INT32_MAX) return KVC_ERR_INVALID;
    k_per_layer[l] = static_cast<int32_t>(v);
  }
  return KVC_OK;
}

kvc_status kvc_block_state_init(kvc_block_state* st, int32_t L, int32_t Hkv, int32_t Hq, int32_t d, int32_t capacity,
                                int32_t sinks, const int32_t* budgets, void* K0, void* V0, int32_t* pos0, void* K1,
                                void* V1, int32_t* pos1) {
  // no second slab: the kept rows stay in place (one slab)
  const bool in_place = !K1 && !V1 && !pos1;
  if (!st || !budgets || L < 1 || L > kMaxLayers || Hkv < 1 || Hq < Hkv || Hq % Hkv != 0 || d != kHeadDim ||
      sinks < 0 || capacity < 1 || !K0 || !V0 || !pos0 || !aligned16(K0) || !aligned16(V0))
    return KVC_ERR_INVALID;
  if (!in_place && (!K1 || !V1 || !pos1 || !aligned16(K1) || !aligned16(V1))) return KVC_ERR_INVALID;
  // key slabs are tensor-map sources; the rest is read and written in place
  if (!is_device_memory(K0) || (K1 && !is_device_memory(K1)) || !reachable(V0, V1, pos0, pos1))
    return KVC_ERR_INVALID;
  if (static_cast<int64_t>(L) * Hq * capacity >= (int64_t(1) << 31)) return KVC_ERR_INVALID;
  if (in_place && (capacity > kEvictInPlaceRows || Hkv > 65535)) return KVC_ERR_INVALID;
  for (int l = 0; l < L; ++l)
    if (budgets[l] < sinks || budgets[l] > capacity) return KVC_ERR_INVALID;
  memset(st, 0, sizeof(*st));
  st->L = L;
  st->Hkv = Hkv;
  st->Hq = Hq;
  st->d = d;
  st->capacity = capacity;
  st->sinks = sinks;
  st->K[0] = K0;
  st->K[1] = K1;
  st->V[0] = V0;
  st->V[1] = V1;
  st->pos[0] = pos0;
  st->pos[1] = pos1;
  for (int l = 0; l < L; ++l) st->budget[l] = budgets[l];
  return KVC_OK;
}

}  // extern "C"

namespace {

struct BlockWorkspace {
  float* score = nullptr;   // [L][Hkv][capacity]
  int32_t* kept = nullptr;  // [L][Hkv][max budget]
  ReconWorkspace rw{};
  size_t bytes = 0;
  bool ok = false;
};

BlockWorkspace carve_block(const kvc_block_state* st, int32_t P, void* base, size_t cap) {
  BlockWorkspace w;
  Carver c(base, base ? cap : 0);
  const int64_t LH = static_cast<int64_t>(st->L) * st->Hkv;
  int32_t kmax = 0;
  for (int l = 0; l < st->L; ++l) kmax = std::max(kmax, st->budget[l]);
  const int G = st->Hq / st->Hkv;
  w.score = c.take<float>(LH * st->capacity);
  // kept indices, or (one slab) the hole and mover lists of each (l, h)
  w.kept = c.take<int32_t>(LH * kmax * (st->K[1] ? 1 : 2));
  w.rw.Rpad = recon_rows(G, 1, P, P);
  w.rw.Qg = c.take<uint16_t>(LH * w.rw.Rpad * kHeadDim);
  w.rw.Kg = nullptr;
  w.rw.lsx = c.take<uint16_t>(LH * w.rw.Rpad * 16);
  w.bytes = ((c.used + 255) & ~size_t(255)) + 256;
  w.ok = c.ok;
  return w;
}

}  // namespace

extern "C" {

size_t kvc_block_workspace_size(const kvc_block_state* st, int32_t max_block, int32_t P) {
  (void)max_block;
  if (!st || P < 1 || st->L < 1) return 0;
  return carve_block(st, P, nullptr, 0).bytes;
}

kvc_status kvc_block_prefill_step(kvc_block_state* st, const void* Kblk, const void* Vblk, int32_t blk_len,
                                  const void* Qprompt, const void* Kprompt, int32_t P, void* ws, size_t ws_bytes,
                                  kvc_stream stream) {
  if (!st || !Kblk || !Vblk || !Qprompt || !Kprompt || blk_len < 1 || P < 1 || !aligned16(Kblk) ||
      !aligned16(Vblk) || !aligned16(Qprompt) || !aligned16(Kprompt))
    return KVC_ERR_INVALID;
  if (!reachable(Kblk, Vblk, Qprompt, Kprompt, ws)) return KVC_ERR_INVALID;
  if (st->consumed + blk_len > INT32_MAX) return KVC_ERR_INVALID;
  for (int l = 0; l < st->L; ++l)
    if (st->len[l] + static_cast<int64_t>(blk_len) > st->capacity) return KVC_ERR_INVALID;
  BlockWorkspace w = carve_block(st, P, ws, ws_bytes);
  kvc_status e = check_ws(ws, ws_bytes, w.bytes);
  if (e != KVC_OK || !w.ok) return KVC_ERR_WORKSPACE;
  kvc_status d = device_ok();
  if (d != KVC_OK) return d;
  cudaStream_t cst = cs(stream);
  const int L = st->L, Hkv = st->Hkv;

  // 1. append the block behind every layer's kept rows
  AppendParams ap;
  memset(&ap, 0, sizeof(ap));
  ap.L = L;
  ap.Hkv = Hkv;
  ap.B = blk_len;
  ap.ld = st->capacity;
  ap.pos0 = st->consumed;
  for (int l = 0; l < L; ++l) {
    ap.len[l] = st->len[l];
    ap.cur[l] = st->cur[l];
    // one slab: a block row landing at or above the budget of a layer that
    // evicts this step keeps its V only if it is kept, and then the eviction
    // takes it from the block; its K is appended for the scoring
    const int64_t n = static_cast<int64_t>(st->len[l]) + blk_len;
    const bool evicts = n > st->budget[l] && n > st->sinks;
    ap.vrows[l] = (!st->K[1] && evicts) ? std::max(0, st->budget[l] - st->len[l]) : blk_len;
  }
  if (launch_append(Kblk, Vblk, st->K[0], st->V[0], st->pos[0], st->K[1], st->V[1], st->pos[1], ap, cst) !=
      cudaSuccess)
    return KVC_ERR_CUDA;

  // 2. layers over budget: score against the prompt, evict, compact
  ReconProblem pr;
  memset(&pr, 0, sizeof(pr));
  pr.L = L;
  pr.Hkv = Hkv;
  pr.Hq = st->Hq;
  pr.G = st->Hq / Hkv;
  pr.sinks = st->sinks;
  int na = 0;
  int32_t n_now[kMaxLayers];
  for (int l = 0; l < L; ++l) {
    n_now[l] = st->len[l] + blk_len;
    if (n_now[l] > st->budget[l] && n_now[l] > st->sinks) {
      ReconLayer& ly = pr.lay[na++];
      ly.layer = l;
      ly.n = n_now[l];
      ly.m = n_now[l] - st->sinks;
      ly.n_chunks = 1;
      ly.last_len = n_now[l] - st->sinks;
      ly.slab = st->cur[l];
    }
  }
  if (na > 0) {
    pr.n_active = na;
    pr.K[0] = st->K[0];
    pr.K[1] = st->K[1];
    pr.ldK = st->capacity;
    pr.Qsrc = Qprompt;
    pr.ldQ = P;
    pr.sel = nullptr;
    pr.Kapp = Kprompt;
    pr.ldApp = P;
    pr.nq_full = P;
    pr.nq_last = P;
    pr.Q = P;
    pr.score = w.score;
    pr.ldS = st->capacity;
    pr.lse_out = nullptr;
    if (launch_recon(pr, w.rw, cst) != cudaSuccess) return KVC_ERR_CUDA;

    int32_t kmax = 0;
    for (int l = 0; l < L; ++l) kmax = std::max(kmax, st->budget[l]);
    EvictParams ep;
    memset(&ep, 0, sizeof(ep));
    ep.L = L;
    ep.Hkv = Hkv;
    ep.sinks = st->sinks;
    ep.ld = st->capacity;
    for (int a = 0; a < na; ++a) {
      const int l = pr.lay[a].layer;
      ep.n[l] = n_now[l];
      ep.k[l] = st->budget[l];
      ep.out_off[l] = static_cast<int64_t>(l) * Hkv * kmax;
      ep.active[l] = 1;
    }
    EvictCopy cp;
    memset(&cp, 0, sizeof(cp));
    if (!st->K[1]) {
      // one slab: kept rows stay where they are; kept block rows move into
      // the rows of evicted ones
      cp.K[0] = st->K[0];
      cp.V[0] = st->V[0];
      cp.pos[0] = st->pos[0];
      cp.Kd[0] = st->K[0];
      cp.Vd[0] = st->V[0];
      cp.posd[0] = st->pos[0];
      cp.src_ld = st->capacity;
      cp.dst_ld = st->capacity;
      cp.Vblk = Vblk;
      cp.blk_len = blk_len;
      for (int l = 0; l < L; ++l) cp.blk_row0[l] = st->len[l];
      if (launch_evict_in_place(w.score, ep, w.kept, kmax, cp, cst) != cudaSuccess) return KVC_ERR_CUDA;
    }
    // two slabs: eviction and compaction in one launch; each active layer's
    // kept rows (with their global positions) move into its other slab
    for (int from = 0; from < 2 && st->K[1]; ++from) {
      cp.K[from] = st->K[from];
      cp.V[from] = st->V[from];
      cp.pos[from] = st->pos[from];
      cp.Kd[from] = st->K[1 - from];
      cp.Vd[from] = st->V[1 - from];
      cp.posd[from] = st->pos[1 - from];
    }
    cp.src_ld = st->capacity;
    cp.dst_ld = st->capacity;
    for (int l = 0; l < L; ++l) cp.slab[l] = st->cur[l];
    if (st->K[1] && launch_evict(w.score, ep, w.kept, nullptr, false, &cp, cst) != cudaSuccess) return KVC_ERR_CUDA;
  }
  // 3. host bookkeeping
  for (int l = 0; l < L; ++l) {
    const bool active = n_now[l] > st->budget[l] && n_now[l] > st->sinks;
    if (active) {
      st->len[l] = st->budget[l];
      if (st->K[1]) st->cur[l] ^= 1;
    } else {
      st->len[l] = n_now[l];
    }
  }
  st->consumed += blk_len;
  return KVC_OK;
}

}  // extern "C"

// ---------------------------------------------------------------- decode attention
namespace {

struct DecodeWorkspace {
  float* part_o = nullptr;
  float* part_ml = nullptr;
  int32_t* counter = nullptr;
  size_t bytes = 0;
  bool ok = false;
};

DecodeWorkspace carve_decode(int32_t n_seg, int32_t G, const DecodePlan& pl, void* base, size_t cap) {
  DecodeWorkspace w;
  Carver c(base, base ? cap : 0);
  const int64_t parts = pl.n_split > 1 ? int64_t(n_seg) * pl.n_split * G : 0;
  w.part_o = c.take<float>(parts * kHeadDim);
  w.part_ml = c.take<float>(parts * 2);
  w.counter = c.take<int32_t>(64);
  w.bytes = ((c.used + 255) & ~size_t(255)) + 256;
  w.ok = c.ok;
  return w;
}

}  // namespace

extern "C" {

size_t kvc_decode_workspace_size(int32_t n_seg, int32_t G, int32_t max_len) {
  if (n_seg < 0 || G < 1 || G > 8 || max_len < 0) return 0;
  return carve_decode(n_seg, G, make_decode_plan(n_seg, G, max_len), nullptr, 0).bytes;
}

kvc_status kvc_decode_attention(int32_t n_seg, int32_t G, const void* Kc, const void* Vc, int64_t kv_rows,
                                const int64_t* seg_off, const int32_t* seg_len, int32_t max_len, const void* q,
                                float scale, float* out, float* lse_opt, void* ws, size_t ws_bytes,
                                kvc_stream stream) {
  if (n_seg < 0 || G < 1 || G > 8 || max_len < 0 || kv_rows < 0) return KVC_ERR_INVALID;
  if (n_seg == 0) return KVC_OK;
  if (!Kc || !Vc || !seg_off || !seg_len || !q || !out || !aligned16(Kc) || !aligned16(Vc) || !aligned16(q) ||
      (reinterpret_cast<uintptr_t>(out) & 3u) != 0 || (lse_opt && (reinterpret_cast<uintptr_t>(lse_opt) & 3u)))
    return KVC_ERR_INVALID;
  // K, V and q are bulk-copy sources; the rest is read or written in place
  if (!is_device_memory(Kc) || !is_device_memory(Vc) || !is_device_memory(q) ||
      !reachable(seg_off, seg_len, out, lse_opt, ws))
    return KVC_ERR_INVALID;
  if (int64_t(n_seg) * G * kHeadDim >= (int64_t(1) << 31)) return KVC_ERR_INVALID;
  const DecodePlan pl = make_decode_plan(n_seg, G, max_len);
  if (int64_t(n_seg) * pl.n_split >= (int64_t(1) << 31)) return KVC_ERR_INVALID;
  DecodeWorkspace w = carve_decode(n_seg, G, pl, ws, ws_bytes);
  if (check_ws(ws, ws_bytes, w.bytes) != KVC_OK || !w.ok) return KVC_ERR_WORKSPACE;
  kvc_status d = device_ok();
  if (d != KVC_OK) return d;
  DecodeParams p{};
  p.K = static_cast<const uint16_t*>(Kc);
  p.V = static_cast<const uint16_t*>(Vc);
  p.seg_off = seg_off;
  p.seg_len = seg_len;
  p.q = static_cast<const uint16_t*>(q);
  p.out = out;
  p.lse = lse_opt;
  p.part_o = w.part_o;
  p.part_ml = w.part_ml;
  p.counter = w.counter;
  p.kv_rows = kv_rows;
  p.n_seg = n_seg;
  p.G = G;
  p.max_len = max_len;
  p.CH = pl.CH;
  p.n_split = pl.n_split;
  const double sc = scale > 0.f ? double(scale) : 1.0 / std::sqrt(double(kHeadDim));
  p.sc2 = static_cast<float>(sc * 1.4426950408889634);
  p.status = status_word();
  p.limit_ns = wait_limit_ns();
  if (!p.status) return KVC_ERR_CUDA;
  return cuda_status(launch_decode(p, cs(stream)));
}

kvc_status kvc_compact_segments(int32_t L, int32_t Hkv, const int32_t* k_per_layer, int64_t* seg_off,
                                int32_t* seg_len) {
  if (L < 1 || Hkv < 1 || !k_per_layer || !seg_off || !seg_len) return KVC_ERR_INVALID;
  int64_t row = 0;
  for (int32_t l = 0; l < L; ++l) {
    if (k_per_layer[l] < 0) return KVC_ERR_INVALID;
    for (int32_t h = 0; h < Hkv; ++h) {
      seg_off[int64_t(l) * Hkv + h] = row;
      seg_len[int64_t(l) * Hkv + h] = k_per_layer[l];
      row += k_per_layer[l];
    }
  }
  return KVC_OK;
}

}  // extern "C"

// ---------------------------------------------------------------- EpiCache per-turn path
namespace {

bool is_pinned_host(const void* p) {
  cudaPointerAttributes a{};
  if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
    cudaGetLastError();
    return false;
  }
  return a.type == cudaMemoryTypeHost;
}

}  // namespace

extern "C" {

kvc_status kvc_episode_match(int32_t B, int32_t E, int32_t De, const float* queries, const float* centroids,
                             float tau, int32_t* episode, float* dist2_opt, kvc_stream stream) {
  if (B < 0 || E < 1 || De < 4 || De % 4 != 0 || !(tau == tau)) return KVC_ERR_INVALID;
  if (B == 0) return KVC_OK;
  if (!queries || !centroids || !episode || !aligned16(queries) || !aligned16(centroids) ||
      (reinterpret_cast<uintptr_t>(episode) & 3u) || (dist2_opt && (reinterpret_cast<uintptr_t>(dist2_opt) & 3u)))
    return KVC_ERR_INVALID;
  if (!reachable(queries, centroids, episode, dist2_opt)) return KVC_ERR_INVALID;
  kvc_status d = device_ok();
  if (d != KVC_OK) return d;
  return cuda_status(launch_match(B, E, De, queries, centroids, tau, episode, dist2_opt, cs(stream)));
}

int64_t kvc_episode_rows(const kvc_block_state* st) {
  if (!st || st->L < 1 || st->L > kMaxLayers || st->Hkv < 1) return -1;
  int64_t rows = 0;
  for (int l = 0; l < st->L; ++l) rows += int64_t(st->Hkv) * st->len[l];
  return rows;
}

kvc_status kvc_episode_pack(const kvc_block_state* st, void* Kp, void* Vp, int32_t* pos_opt, kvc_stream stream) {
  if (kvc_episode_rows(st) < 0 || !Kp || !Vp || !aligned16(Kp) || !aligned16(Vp) || st->d != kHeadDim)
    return KVC_ERR_INVALID;
  if (!reachable(Kp, Vp, pos_opt)) return KVC_ERR_INVALID;
  PackParams pp{};
  pp.L = st->L;
  pp.Hkv = st->Hkv;
  pp.cap = st->capacity;
  pp.ordered = st->K[1] ? 0 : 1;
  pp.npos = st->consumed;
  int64_t row = 0;
  for (int l = 0; l < st->L; ++l) {
    if (st->len[l] < 0 || st->len[l] > st->capacity || (st->cur[l] != 0 && st->cur[l] != 1)) return KVC_ERR_INVALID;
    pp.len[l] = st->len[l];
    pp.cur[l] = st->cur[l];
    pp.dst_off[l] = row;
    row += int64_t(st->Hkv) * st->len[l];
  }
  kvc_status d = device_ok();
  if (d != KVC_OK) return d;
  return cuda_status(launch_pack(st->K[0], st->V[0], st->pos[0], st->K[1], st->V[1], st->pos[1], Kp, Vp, pos_opt,
                                 pp, cs(stream)));
}

kvc_status kvc_episode_swap(const void* dev_out, void* host_out, size_t bytes_out, const void* host_in, void* dev_in,
                            size_t bytes_in, kvc_stream out_stream, kvc_stream in_stream) {
  if (bytes_out > 0 && (!dev_out || !host_out || !is_device_memory(dev_out) || !is_pinned_host(host_out)))
    return KVC_ERR_INVALID;
  if (bytes_in > 0 && (!host_in || !dev_in || !is_pinned_host(host_in) || !is_device_memory(dev_in)))
    return KVC_ERR_INVALID;
  if (bytes_out > 0) {
    cudaError_t e = cudaMemcpyAsync(host_out, dev_out, bytes_out, cudaMemcpyDeviceToHost, cs(out_stream));
    if (e != cudaSuccess) return KVC_ERR_CUDA;
  }
  if (bytes_in > 0) {
    cudaError_t e = cudaMemcpyAsync(dev_in, host_in, bytes_in, cudaMemcpyHostToDevice, cs(in_stream));
    if (e != cudaSuccess) return KVC_ERR_CUDA;
  }
  return KVC_OK;
}

}  // extern "C"

// ---------------------------------------------------------------- Q4 codec
extern "C" {

kvc_status kvc_q4_encode(int64_t rows, const void* X, void* codes, void* params, kvc_stream stream) {
  if (rows < 0) return KVC_ERR_INVALID;
  if (rows == 0) return KVC_OK;
  if (!X || !codes || !params || !aligned16(X) || (reinterpret_cast<uintptr_t>(codes) & 3u) ||
      (reinterpret_cast<uintptr_t>(params) & 3u))
    return KVC_ERR_INVALID;
  if (!reachable(X, codes, params)) return KVC_ERR_INVALID;
  kvc_status d = device_ok();
  if (d != KVC_OK) return d;
  return cuda_status(launch_q4_encode(rows, X, codes, params, cs(stream)));
}

kvc_status kvc_q4_decode(int64_t rows, const void* codes, const void* params, void* X, kvc_stream stream) {
  if (rows < 0) return KVC_ERR_INVALID;
  if (rows == 0) return KVC_OK;
  if (!X || !codes || !params || !aligned16(X) || (reinterpret_cast<uintptr_t>(codes) & 3u) ||
      (reinterpret_cast<uintptr_t>(params) & 3u))
    return KVC_ERR_INVALID;
  if (!device_can_read(codes) || !device_can_read(params) || !reachable(X)) return KVC_ERR_INVALID;
  kvc_status d = device_ok();
  if (d != KVC_OK) return d;
  return cuda_status(launch_q4_decode(rows, codes, params, X, cs(stream)));
}

}  // extern "C"
