// Host-side internals shared by the library's translation units.
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstddef>
#include <cstdint>

#include "../../include/kvc.h"

namespace kvc {

constexpr int kHeadDim = 128;
constexpr int kMaxLayers = KVC_MAX_LAYERS;

// Memory checks made on the host before a launch.  is_device_memory: device
// or managed memory (tensor-map and bulk-copy sources).  device_can_read:
// memory kernels may read or write in place -- device or managed memory,
// page-locked host memory mapped at the same address, or pageable host memory
// on a device that reaches it through the host page tables.
bool is_device_memory(const void* p);
bool device_can_read(const void* p);

// Shape checks shared by every entry point that takes a kvc_shape: sizes
// in range, d = 128, GQA divisibility, row coordinates within int32 and at
// most 65535 (layer, KV head) pairs.
bool shape_ok(const kvc_shape& s);

// Device address of a __device__ symbol in the current device's current
// context, cached per device under the context's unique ID.  A
// cudaDeviceReset replaces the primary context and the module is loaded
// again, possibly at another address; the next call then finds a new
// context ID and looks the symbol up again instead of reusing a stale
// address.  Null on failure.
struct SymbolSlot {
  unsigned long long ctx;
  void* ptr;
};
void* symbol_address(const void* symbol, SymbolSlot* slots);  // slots: one per device (64)

// Per-device status word (device address) and the process-wide wait limit.
int* status_word();
uint64_t wait_limit_ns();
int num_sms();

// Per-kernel event timing (active between kvc_profile_begin/end): brackets
// the launches made during the scope's lifetime with an event pair.
struct ProfScope {
  int slot = -1;
  cudaStream_t stream = nullptr;
  ProfScope(const char* name, cudaStream_t st);
  ~ProfScope();
  ProfScope(const ProfScope&) = delete;
  ProfScope& operator=(const ProfScope&) = delete;
};

// Chunk plan on the host (same rule as kvc_chunk_plan).
struct ChunkPlan {
  int32_t n_chunks = 0;
  int32_t nq_full = 0;   // n_q of every chunk but the last
  int32_t nq_last = 0;   // n_q of the last chunk
  int32_t Q = 0;         // total reconstruction queries
  int32_t m = 0;         // chunk size
  int32_t last_len = 0;  // |C_last|
};
bool make_plan(int32_t N, int32_t sinks, int32_t m, double rho, ChunkPlan* plan);

// Workspace carving: 256-B aligned slices out of one caller buffer.
struct Carver {
  char* base;
  size_t cap;
  size_t used = 0;
  bool ok = true;
  Carver(void* b, size_t c) : base(static_cast<char*>(b)), cap(c) {}
  template <class T>
  T* take(size_t count) {
    size_t off = (used + 255) & ~size_t(255);
    size_t bytes = count * sizeof(T);
    if (off + bytes > cap || (base == nullptr && bytes > 0)) {
      ok = false;
      used = off + bytes;
      return nullptr;
    }
    used = off + bytes;
    return reinterpret_cast<T*>(base + off);
  }
};

// 2-D bf16 tensor map over `rows` rows of 128 elements, box = 64 x box_rows,
// 128-byte swizzle (the K-major tcgen05 operand layout).
bool make_tmap_rows(CUtensorMap* map, const void* base, uint64_t rows, uint32_t box_rows);
// Rows of 16 bf16 (32 B) in boxes of box_rows rows, 32-byte swizzle.
bool make_tmap_rows16(CUtensorMap* map, const void* base, uint64_t rows, uint32_t box_rows);

// ------------------------------------------------------------------ launchers
// Each returns cudaSuccess or the launch error.

// KeyDiff proxy: s[lh][i] for LH = L*Hkv heads of N rows, then p = mean.
// scratch: proxy_scratch_bytes(LH, N) bytes of device memory, 256-B aligned
// (work-list counter, per-head arrivals and ready flags, partial sums, mean
// keys); its control words are cleared on the stream before the launch.
size_t proxy_scratch_bytes(int LH, int N);
cudaError_t launch_proxy(const void* K, int LH, int N, float* s, float* p, void* scratch, cudaStream_t st);

// Knorm proxy: s[lh][i] = -|k_i|, then p = mean.
cudaError_t launch_knorm(const void* K, int LH, int N, float* s, float* p, cudaStream_t st);

// p[i] = mean over LH rows of x[lh][i] (stride ld); p[i] = 0 for i < zero_below.
cudaError_t launch_mean_heads(const float* x, int LH, int N, int64_t ld, int zero_below, float* p,
                              cudaStream_t st);
// The same sum without the division (a shard's partial sum), and the
// division of summed partials by the total head count.
cudaError_t launch_sum_heads(const float* x, int LH, int N, int64_t ld, int zero_below, float* psum,
                             cudaStream_t st);
cudaError_t launch_sums_to_mean(const float* psum, int N, int heads, float* p, cudaStream_t st);
// Per-head proxy scores only: kind 0 KeyDiff, 1 Knorm.
cudaError_t launch_proxy_scores(int kind, const void* K, int LH, int N, float* s, cudaStream_t st);
// Largest non-sink score of every (l, h) row into *max_out (device f32), and
// score[l][h][s] = *value for s < sinks.
cudaError_t launch_score_max(const float* score, int LH, int N, int sinks, uint32_t* key_word, float* max_out,
                             cudaStream_t st);
cudaError_t launch_pin_value(float* score, int LH, int N, int sinks, const float* value, cudaStream_t st);

// Per-chunk selection of reconstruction queries.
cudaError_t launch_select(const float* p, int N, int sinks, const ChunkPlan& plan, double rho, int32_t* sel,
                          cudaStream_t st);

// Row-wise eviction: for every (l, h) keep sinks + top (k_l - sinks) of
// score[l][h][sinks:n_l); kept rows written at out_off[l] + h*k_l.
struct EvictParams {
  int L, Hkv, sinks;
  int64_t ld;                     // row stride of score
  int32_t n[kMaxLayers];          // scored length per layer
  int32_t k[kMaxLayers];          // kept per (l, h)
  int64_t out_off[kMaxLayers];    // output offset of layer l
  int32_t active[kMaxLayers];     // 0: layer skipped
};
// Copy of the kept rows made by the eviction kernel itself (optional): the
// kept K/V rows of layer l (and their global positions, when pos arrays are
// given) move from the source slab src[slab[l]] to dst[slab[l]].  Rows are
// 256-byte bf16 rows; V (and its destination) may be null.
struct EvictCopy {
  const void* K[2];
  const void* V[2];
  const int32_t* pos[2];
  void* Kd[2];
  void* Vd[2];
  int32_t* posd[2];
  int64_t src_ld;                 // rows per (l, h) in a source slab
  int64_t dst_ld;                 // rows per (l, h) in a destination; < 0: ragged at out_off[l] + h*k_l
  int32_t slab[kMaxLayers];
  // in-place eviction: when Vblk is set, a moved row r takes its V row from
  // the block, Vblk[l][h][r - blk_row0[l]] with blk_len rows per (l, h)
  // (the block's V rows at or above the budget were not appended)
  const void* Vblk;
  int32_t blk_len;
  int32_t blk_row0[kMaxLayers];
};
// gmax_word: two zeroed words of device memory when pin is set (the max
// order key, an arrival counter).  copy: null, or the fused compaction.
cudaError_t launch_evict(float* score, const EvictParams& ep, int32_t* kept, uint32_t* gmax_word, bool pin,
                         const EvictCopy* copy, cudaStream_t st);
// The eviction kernel copies the kept rows itself (one launch) when a row
// keeps at most kFusedCopyRows rows; longer kept lists move in one tiled
// compaction launch after it (a row's copy would otherwise fall to a
// single CTA).
constexpr int kFusedCopyRows = 4096;
// Eviction in place (one launch): the kept rows of every active layer end up
// in rows [0, k_l) of slab 0 (copy.K[0] / V[0] / pos[0], written through
// Kd[0] / Vd[0] / posd[0], the same buffers), in no particular order: each
// kept row at or above k_l moves into an evicted row below it.  A tie at the
// threshold goes to the lower global position (copy.pos[0]).  lists holds
// 2 * list_stride int32 per (l, h) (list_stride >= max k_l).  Rows must fit
// the shared-memory parts (at most kEvictInPlaceRows candidates).
cudaError_t launch_evict_in_place(const float* score, const EvictParams& ep, int32_t* lists, int list_stride,
                                  const EvictCopy& copy, cudaStream_t st);
constexpr int kEvictInPlaceRows = 8 * 49152;

// Compaction: dst row (l, h, t) = src row (l, h, idx[l][h][t]).
struct CompactParams {
  int L, Hkv;
  int64_t src_ld;                 // rows per (l, h) in the source
  int64_t dst_ld;                 // rows per (l, h) in the destination; <0: ragged (use dst_off)
  int32_t n_src[kMaxLayers];      // valid source rows per layer (bounds check)
  int32_t k[kMaxLayers];
  int64_t idx_off[kMaxLayers];    // offset of layer l in the index array
  int64_t dst_off[kMaxLayers];    // ragged destination offset (rows) of layer l
  int32_t active[kMaxLayers];
  int32_t unit_off[kMaxLayers + 1];  // filled by launch_compact: first (head, 64-row tile) unit of layer l
};
cudaError_t launch_compact(const void* K, const void* V, const int32_t* idx, const int32_t* pos_src,
                           int32_t* pos_dst, void* Kc, void* Vc, const CompactParams& cp, cudaStream_t st);

// The same with each layer's rows going from copy.K[slab[l]] (and V, pos)
// to copy.Kd[slab[l]] (EpiCache slabs: one launch for both directions).
cudaError_t launch_compact_slabs(const int32_t* idx, const EvictCopy& copy, const CompactParams& cp, cudaStream_t st);

// Block append: state rows [len_l, len_l + B) of each (l, h) <- block rows.
struct AppendParams {
  int L, Hkv, B;
  int64_t ld;                     // rows per (l, h) in the state slab
  int32_t len[kMaxLayers];
  int32_t cur[kMaxLayers];        // which of the two slabs holds layer l
  int32_t vrows[kMaxLayers];      // V of the block's rows t < vrows[l] is appended (K always is)
  int64_t pos0;                   // global position of the block's first token
};
cudaError_t launch_append(const void* Kblk, const void* Vblk, void* K0, void* V0, int32_t* pos0, void* K1, void* V1,
                          int32_t* pos1, const AppendParams& ap, cudaStream_t st);

// Reconstruction scoring on the tensor cores.
struct ReconLayer {
  int32_t layer;     // model layer index
  int32_t n;         // cache rows of this layer
  int32_t m;         // chunk size of this layer
  int32_t n_chunks;  // chunks of this layer
  int32_t last_len;  // size of the last chunk
  int32_t slab;      // which K slab (0/1) holds the layer (block prefill); 0 otherwise
};
struct ReconProblem {
  int L, Hkv, Hq, G, sinks;
  int n_active;
  ReconLayer lay[kMaxLayers];
  // cache keys: base[slab] + ((layer*Hkv + h) * ldK + row) * d
  const void* K[2];
  int64_t ldK;
  // query source rows: Qsrc + ((layer*Hq + g) * ldQ + src) * d, src = sel ? sel[t] : t
  const void* Qsrc;
  int64_t ldQ;
  const int32_t* sel;
  // appended keys: Kapp + ((layer*Hkv + h) * ldApp + t) * d, or gathered from K at sel if Kapp is null
  const void* Kapp;
  int64_t ldApp;
  // chunk query counts (same for every layer)
  int32_t nq_full, nq_last, Q;
  // outputs
  float* score;       // score + (layer*Hkv + h) * ldS + position
  int64_t ldS;
  float* lse_out;     // optional [L][Hq][Q], natural log
  cudaEvent_t gather_done;  // optional: recorded right after the query gather is launched
};
struct ReconWorkspace {
  void* Qg;       // bf16 [L*Hkv][Rpad][d]
  void* Kg;       // bf16 [L*Hkv][Q][d] (gathered appended keys), when Kapp is null
  void* lsx;      // bf16 [L*Hkv][Rpad][16]: -lse2/scale (row LSE, log2 units) as three bf16 terms, then zeros
  int32_t Rpad;   // rows per (l, h) in Qg, multiple of 128
};
// Rows per (layer, KV head) of the query row space (chunks padded to 128 rows).
int32_t recon_rows(int G, int n_chunks, int nq_full, int nq_last);
// Phases of the scoring (bit mask): query gather into the row space, the
// row-LSE pass, the column-max pass.  They run in that order on one
// workspace; a call may run any contiguous subset of them.
enum : int { RECON_GATHER = 1, RECON_ROWS = 2, RECON_COLS = 4, RECON_ALL = 7 };
cudaError_t launch_recon(const ReconProblem& pr, const ReconWorkspace& ws, cudaStream_t st, int phases = RECON_ALL);

// Device-side wait that expires on purpose (status-path test).
cudaError_t launch_expire_wait(uint64_t limit_ns, cudaStream_t st);

// Decode attention over ragged segments of a compacted cache.
struct DecodePlan {
  int32_t CH = 0;        // keys per split (whole tiles)
  int32_t n_split = 0;   // splits per segment (covers max_len)
};
DecodePlan make_decode_plan(int32_t n_seg, int32_t G, int32_t max_len);
struct DecodeParams {
  const uint16_t* K;
  const uint16_t* V;
  const int64_t* seg_off;
  const int32_t* seg_len;
  const uint16_t* q;      // [n_seg][G][128]
  float* out;             // [n_seg][G][128]
  float* lse;             // [n_seg][G] or null
  float* part_o;          // [n_seg][n_split][G][128] (splits of multi-split segments)
  float* part_ml;         // [n_seg][n_split][G][2]: base-2 max, sum
  int32_t* counter;       // work-item counter, zero on entry
  int64_t kv_rows;
  int32_t n_seg, G, max_len, CH, n_split;
  float sc2;              // softmax scale * log2(e)
  int* status;
  uint64_t limit_ns;
};
cudaError_t launch_decode(const DecodeParams& p, cudaStream_t st);

// EpiCache per-turn path: nearest episode centroid per question (tau <= 0: no
// new-topic threshold), and packing of a block state's kept rows.
cudaError_t launch_match(int B, int E, int De, const float* q, const float* c, float tau, int32_t* ep, float* d2,
                         cudaStream_t st);
struct PackParams {
  int L, Hkv;
  int64_t cap;                    // rows per (l, h) in each slab
  int32_t len[kMaxLayers];
  int32_t cur[kMaxLayers];
  int64_t dst_off[kMaxLayers];    // first packed row of layer l
  int ordered;                    // 1: rows in no order (one slab); pack them by ascending position
  int64_t npos;                   // positions lie in [0, npos)
};
// Q4 codec of bf16 rows of 128 values (codes [rows][64] bytes, params
// [rows][2] x (step, offset) bf16).
cudaError_t launch_q4_encode(int64_t rows, const void* X, void* codes, void* params, cudaStream_t st);
cudaError_t launch_q4_decode(int64_t rows, const void* codes, const void* params, void* X, cudaStream_t st);
cudaError_t launch_pack(const void* K0, const void* V0, const int32_t* P0, const void* K1, const void* V1,
                        const int32_t* P1, void* Kp, void* Vp, int32_t* Pp, const PackParams& pp, cudaStream_t st);

}  // namespace kvc
