/*
 * kvc.h -- C ABI of the GB300 (sm_103a) attention-score KV-cache compressor.
 *
 * The method is KV^2 as described on "KV²가 전체 문맥 재계산 없이 KV 캐시를
 * 압축한다" (onedev.kr/papers/598) and the block prefill of "[26'ICML] EpiCache"
 * (juyoungkimmy-kim.github.io).  Each entry point below names the section it
 * implements.
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 * Types      bf16 tensors are passed as `const void*` (IEEE bfloat16 bit
 *            patterns); scores are float32; indices are int32.
 * Layout     row-major, contiguous, head dimension d innermost:
 *              K, V      [L][Hkv][N][d]        cache keys / values (post-RoPE)
 *              Qpool     [L][Hq][N][d]         one query per position and query head
 *              p         [N]                   token-level proxy score
 *              s         [L][Hkv][N]           per-head proxy score
 *              score     [L][Hkv][N]           stage-2 (reconstruction) score
 *              sel       [Q]                   selected positions, chunk-major, ascending inside a chunk
 *              lse       [L][Hq][Q]            natural-log softmax normaliser of each reconstruction query
 *              kept      ragged, layer-major:  layer l starts at Hkv * sum_{l'<l} k_{l'}, then [Hkv][k_l]
 *              Kc, Vc    ragged like kept, d elements per row
 *            Query head g reads KV head g / (Hq / Hkv).  d must be 128.
 * Memory     The caller owns every buffer (device memory unless stated as
 *            host), including the workspace; the library never allocates or
 *            frees memory.  Pointers must be 16-byte aligned; the workspace
 *            must be 256-byte aligned.  Exception: the query pool Qpool
 *            (kvc_recon_score, kvc_compress) and the sources K, V of
 *            kvc_compact and V of kvc_compress may also be page-locked host
 *            memory mapped into the device address space (cudaHostAlloc, or
 *            cudaHostRegister with mapping); the kernels then read only the
 *            selected query rows and the kept K/V rows, each once, across
 *            the host link (NVLink-C2C on Grace-Blackwell).
 * Streams    All device work is enqueued on `stream` (NULL = legacy default
 *            stream) and is asynchronous; host-side outputs are written
 *            before the call returns.
 * Errors     Argument errors are detected on the host before anything is
 *            launched or written and return KVC_ERR_INVALID (or
 *            KVC_ERR_WORKSPACE).  A failed launch or CUDA call returns
 *            KVC_ERR_CUDA.  Device-side conditions (a bounded wait that
 *            expired, an index that failed its check) are recorded in a
 *            per-device status word and reported by kvc_stream_status().
 *            On such an error the outputs are unspecified.
 */
#ifndef KVC_H_
#define KVC_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#if defined(__GNUC__)
#define KVC_API __attribute__((visibility("default")))
#else
#define KVC_API
#endif

typedef struct CUstream_st* kvc_stream; /* identical to cudaStream_t */
typedef struct CUevent_st* kvc_event;   /* identical to cudaEvent_t */

typedef enum {
  KVC_OK = 0,
  KVC_ERR_INVALID = 1,     /* bad argument; nothing was launched or written */
  KVC_ERR_CUDA = 2,        /* a CUDA runtime call or kernel launch failed */
  KVC_ERR_TIMEOUT = 3,     /* a bounded device-side wait expired */
  KVC_ERR_BOUNDS = 4,      /* a device-side index check failed */
  KVC_ERR_WORKSPACE = 5,   /* workspace missing, misaligned or too small */
  KVC_ERR_UNSUPPORTED = 6  /* current device is not an sm_103 GPU */
} kvc_status;

/* Model shape.  d must be 128, Hq a positive multiple of Hkv, N >= 1. */
typedef struct {
  int32_t L, Hkv, Hq, d, N;
} kvc_shape;

/* Human-readable name of a status code (static string). */
KVC_API const char* kvc_status_string(kvc_status s);

/* Checks that the current CUDA device is an sm_103 GPU this library was
 * built for.  Returns KVC_OK, KVC_ERR_UNSUPPORTED or KVC_ERR_CUDA. */
KVC_API kvc_status kvc_device_check(void);

/* Synchronises `stream`, then returns and clears the device status word of
 * the current device: KVC_OK, KVC_ERR_TIMEOUT or KVC_ERR_BOUNDS (or
 * KVC_ERR_CUDA if the synchronisation itself failed). */
KVC_API kvc_status kvc_stream_status(kvc_stream stream);

/* Upper bound (ns) on every device-side wait of this library's kernels on
 * the current process; 0 restores the default (1 s).  Host-only. */
KVC_API kvc_status kvc_set_wait_limit_ns(uint64_t limit_ns);

/* Launches one block whose wait on a barrier that nothing completes must
 * expire after `limit_ns`; the status word then reads KVC_ERR_TIMEOUT.
 * This exercises the timeout path without hanging the GPU. */
KVC_API kvc_status kvc_debug_expire_wait(uint64_t limit_ns, kvc_stream stream);

/* Per-kernel timing.  Between kvc_profile_begin() and kvc_profile_end()
 * every kernel this library launches is bracketed by a pair of CUDA events
 * on its stream (reused from a pool; no device memory is allocated).
 * kvc_profile_end() synchronises the device, fills up to `max_entries`
 * records (one per kernel name, launches and summed milliseconds, in first-
 * launch order) and sets *n_entries.  Profiling is process-wide and meant
 * for one stream at a time. */
typedef struct {
  char name[32];
  int32_t launches;
  double total_ms;
} kvc_kernel_time;
KVC_API kvc_status kvc_profile_begin(void);
KVC_API kvc_status kvc_profile_end(kvc_kernel_time* out, int32_t max_entries, int32_t* n_entries);

/* ------------------------------------------------------------------ plan
 * KV² page, "어떻게 동작하나": the first `sinks` tokens are kept as they are;
 * the rest is split into chunks C_r = [sinks + r*m, min(sinks + (r+1)*m, N))
 * and each chunk reconstructs n_q = max(floor(rho * |C_r|), 1) queries.
 * Host-only.  `*n_chunks` receives M; if `chunk_off` is not NULL it must hold
 * M + 1 host ints and receives the prefix sums of n_q (chunk_off[M] = Q).
 * Invalid: N < 1, sinks < 0, sinks >= N, m < 1, rho outside (0, 1]. */
KVC_API kvc_status kvc_chunk_plan(int32_t N, int32_t sinks, int32_t m, double rho, int32_t* n_chunks,
                          int32_t* chunk_off);

/* Kept tokens per (layer, KV head) for a budget fraction b in (0, 1]:
 * floor(b * N), sinks included.  Host-only.  Invalid if the result is below
 * `sinks` or above N. */
KVC_API kvc_status kvc_budget_count(double b, int32_t N, int32_t sinks, int32_t* k);

/* Bytes of workspace that every KV² entry point below (and kvc_compress)
 * needs for this shape and chunk plan.  0 on invalid arguments. */
KVC_API size_t kvc_workspace_size(kvc_shape shape, int32_t sinks, int32_t m, double rho);

/* ------------------------------------------------------------------ stage 1
 * KV² page, "어떻게 동작하나": KeyDiff proxy averaged over layers and KV heads.
 * For each (layer, KV head): u = mean over all N positions of k_i / |k_i|,
 * s_i = -(k_i . u) / (|k_i| |u|) (0 for a zero key or a zero u); then
 * p_i = mean over the L*Hkv heads of s_i.
 *   K      device bf16 [L][Hkv][N][d]
 *   p      device f32 [N]                          (output)
 *   s_opt  device f32 [L][Hkv][N] or NULL          (output)
 *   ws     device workspace, 256-byte aligned, of at least
 *          kvc_proxy_workspace_size(shape, s_opt == NULL) bytes (or
 *          kvc_workspace_size() bytes, which covers it); it holds the
 *          per-head scores when s_opt is NULL and may be NULL otherwise.
 *          Too small or misaligned: KVC_ERR_WORKSPACE.
 * The result is deterministic: the mean key of a head is summed in a fixed
 * order. */
KVC_API kvc_status kvc_proxy_score(kvc_shape shape, const void* K, float* p, float* s_opt, void* ws, size_t ws_bytes,
                           kvc_stream stream);

/* Bytes of workspace kvc_proxy_score needs for this shape, with room for the
 * per-head scores when with_scores is nonzero (s_opt NULL).  0 on invalid
 * shapes. */
KVC_API size_t kvc_proxy_workspace_size(kvc_shape shape, int32_t with_scores);

/* Stage-1 proxy kinds.  KV² page, "어떻게 동작하나": KeyDiff is the default;
 * "전제와 한계": Knorm is the close alternative.  Knorm here scores
 * s_i = -|k_i| per (layer, KV head) (keys of smaller L2 norm rank higher),
 * averaged over the heads like KeyDiff. */
typedef enum { KVC_PROXY_KEYDIFF = 0, KVC_PROXY_KNORM = 1 } kvc_proxy_kind;

/* kvc_proxy_score with a selectable proxy kind; same arguments, layouts and
 * errors (KVC_ERR_INVALID for an unknown kind). */
KVC_API kvc_status kvc_proxy_score_kind(kvc_shape shape, kvc_proxy_kind kind, const void* K, float* p, float* s_opt,
                                        void* ws, size_t ws_bytes, kvc_stream stream);

/* Layer-sharded compression.  The KV² page's proxy is a mean over all
 * (layer, KV head) pairs and its sink pin uses the max over all scores;
 * everything else is per (layer, KV head).  A cache split by layers over
 * several devices therefore exchanges only N floats per pass (a sum) and
 * one float (a max).  Each shard calls these with the shape of its own
 * layers (L = its layer count) and its slices of K, V, the query pool and
 * the scores, which are contiguous in the [L][...] layouts:
 *   kvc_proxy_partial    psum[i] = sum over the shard's heads of s_i (no
 *                        division); s_opt/ws as in kvc_proxy_score
 *   (caller: all-reduce(sum) of psum over the shards)
 *   kvc_proxy_from_sums  p[i] = psum[i] / total_heads (L*Hkv of the whole
 *                        cache): the proxy p of the unsharded call, up to
 *                        the order of the additions
 *   kvc_select_queries   on every shard (the same p gives the same queries)
 *   kvc_recon_score      shard-local
 *   kvc_refine_partial   (refinement passes) psum[i] = sum over the shard's
 *                        heads of score[i], 0 for i < sinks; then the same
 *                        all-reduce and kvc_proxy_from_sums
 *   kvc_evict_compact    shard-local (pins the sinks to the shard's max,
 *                        which changes no kept position)
 *   kvc_score_max        *max_out (device f32) = the shard's largest
 *                        non-sink score; ws: 256 bytes of device scratch
 *   (caller: all-reduce(max))
 *   kvc_pin_sinks        score[l][h][s] = *value (device f32) for s < sinks
 * Device pointers throughout; psum, p: f32 [N]. */
KVC_API kvc_status kvc_proxy_partial(kvc_shape shape, kvc_proxy_kind kind, const void* K, float* psum, float* s_opt,
                                     void* ws, size_t ws_bytes, kvc_stream stream);
KVC_API kvc_status kvc_refine_partial(kvc_shape shape, const float* score, int32_t sinks, float* psum,
                                      kvc_stream stream);
KVC_API kvc_status kvc_proxy_from_sums(int32_t N, int32_t total_heads, const float* psum, float* p,
                                       kvc_stream stream);
KVC_API kvc_status kvc_score_max(kvc_shape shape, const float* score, int32_t sinks, float* max_out, void* ws,
                                 size_t ws_bytes, kvc_stream stream);
KVC_API kvc_status kvc_pin_sinks(kvc_shape shape, float* score, int32_t sinks, const float* value, kvc_stream stream);

/* The pages have no counterpart to this entry point.  Same result as
 * kvc_proxy_score (p only) for callers that cannot allocate device memory
 * at the point of the call: runtimes that hand all free HBM to their own
 * pool allocator, or hot paths that must not call cudaMalloc because it can
 * synchronise the device.  The scratch (the per-head scores) lives in a
 * 16 MiB array inside the library, reserved on each GPU the first time the
 * library's module is loaded there and held until the process exits; this
 * call allocates nothing.  Limit: kvc_proxy_workspace_size(shape, 1) <=
 * 16 MiB, that is L*Hkv*N <= 4194304 (e.g. 32 layers x 8 KV heads x 16384
 * tokens, exactly at the limit); larger shapes return KVC_ERR_WORKSPACE
 * before any launch.  The first call on a device (and the first after a
 * cudaDeviceReset) looks up the array's device address with that device
 * current; make that first call before any stream capture.  All calls on a
 * device share the array: calls that may overlap on the GPU race and must
 * be ordered by the caller.  No part of the array needs clearing between
 * calls: every call overwrites all the entries it reads.
 *   K  device bf16 [L][Hkv][N][d];  p  device f32 [N] (output) */
KVC_API kvc_status kvc_proxy_score_noalloc(kvc_shape shape, const void* K, float* p, kvc_stream stream);

/* KV² page, "어떻게 동작하나": inside each chunk the n_q positions with the
 * highest p (the lower position wins a tie; NaN ranks lowest), written
 * ascending, chunk after chunk.
 *   p    device f32 [N]
 *   sel  device int32 [Q], Q from kvc_chunk_plan   (output) */
KVC_API kvc_status kvc_select_queries(int32_t N, int32_t sinks, int32_t m, double rho, const float* p, int32_t* sel,
                              kvc_stream stream);

/* ------------------------------------------------------------------ stage 2
 * KV² page, "무엇과 다른가": the selected tokens are appended after the cache
 * and run causally over the whole cache; the score of cache position i in
 * C_r is the max, over the chunk's queries and over the query heads of the
 * KV head, of the softmax attention paid to i.  For query j of chunk r and
 * query head g the logits are q.k_i / sqrt(d) over the N cache keys followed
 * by q.kapp_t / sqrt(d) for the chunk's appended keys t <= j.
 *   K        device bf16 [L][Hkv][N][d]
 *   Qpool    device bf16 [L][Hq][N][d]; query (g, j of chunk r) is row sel[off_r + j]
 *   sel      device int32 [Q] from kvc_select_queries
 *   Kapp_opt device bf16 [L][Hkv][Q][d] appended keys, or NULL to use K at sel
 *   score    device f32 [L][Hkv][N] (output; positions < sinks are not written)
 *   lse_opt  device f32 [L][Hq][Q] or NULL (output, natural log)
 * Runs on the tensor cores (tcgen05, bf16 inputs, fp32 accumulation). */
KVC_API kvc_status kvc_recon_score(kvc_shape shape, const void* K, const void* Qpool, const int32_t* sel, int32_t sinks,
                           int32_t m, double rho, const void* Kapp_opt, float* score, float* lse_opt, void* ws,
                           size_t ws_bytes, kvc_stream stream);

/* The pages have no counterpart to these entry points: kvc_recon_score split
 * into its three phases, for callers that overlap the phases of consecutive
 * compression steps on several streams (for instance the next step's query
 * gather, whose reads may cross the host link, under this step's column-max
 * pass).  On one workspace (kvc_workspace_size) they must run in this order,
 * on one stream or ordered by events, with the same shape, sinks, m, rho and
 * Kapp_opt; together they compute exactly what kvc_recon_score computes.
 *   kvc_recon_gather  fills the workspace's query rows (and, when Kapp_opt is
 *                     NULL, the appended keys K at sel) from Qpool and sel;
 *   kvc_recon_rows    the row log-sum-exp pass: per query row, the values the
 *                     column-max pass subtracts; lse_opt as kvc_recon_score;
 *   kvc_recon_cols    the column-max pass: writes score as kvc_recon_score.
 * Arguments and errors as kvc_recon_score. */
KVC_API kvc_status kvc_recon_gather(kvc_shape shape, const void* K, const void* Qpool, const int32_t* sel,
                                    int32_t sinks, int32_t m, double rho, const void* Kapp_opt, void* ws,
                                    size_t ws_bytes, kvc_stream stream);
KVC_API kvc_status kvc_recon_rows(kvc_shape shape, const void* K, int32_t sinks, int32_t m, double rho,
                                  const void* Kapp_opt, float* lse_opt, void* ws, size_t ws_bytes, kvc_stream stream);
KVC_API kvc_status kvc_recon_cols(kvc_shape shape, const void* K, int32_t sinks, int32_t m, double rho, float* score,
                                  void* ws, size_t ws_bytes, kvc_stream stream);

/* KV² page, "무엇과 다른가" (iterative refinement): the stage-2 output has the
 * proxy's token granularity, so p_i = mean over the L*Hkv heads of score_i
 * replaces the proxy in the next pass.  p[i] = 0 for i < sinks.
 *   score device f32 [L][Hkv][N]; p device f32 [N] (output) */
KVC_API kvc_status kvc_refine_proxy(kvc_shape shape, const float* score, int32_t sinks, float* p, kvc_stream stream);

/* KV² page, "무엇과 다른가": gather scores, pin the sink positions to the max
 * score, remove the lowest-scored entries down to the budget.
 *   score        device f32 [L][Hkv][N] (in/out: entries < sinks are
 *                overwritten with the max over all entries >= sinks; they
 *                are never read)
 *   k_per_layer  HOST int32 [L], sinks <= k_l <= N
 *   kept         device int32, ragged layer-major (output): the k_l kept
 *                positions of each (l, h) in ascending order; the lower
 *                position wins a tie, so the sinks are always kept. */
KVC_API kvc_status kvc_evict_topk(kvc_shape shape, float* score, int32_t sinks, const int32_t* k_per_layer, int32_t* kept,
                          void* ws, size_t ws_bytes, kvc_stream stream);

/* KV² page, "전제와 한계": headwise compaction of the kept rows into a dense
 * cache, Kc[l][h][t] = K[l][h][kept[l][h][t]] and likewise for V (bit copies).
 *   K, V         device bf16 [L][Hkv][N][d]
 *   kept         device int32 ragged (from kvc_evict_topk)
 *   k_per_layer  HOST int32 [L]
 *   Kc, Vc       device bf16 ragged (output); V/Vc may be NULL together */
KVC_API kvc_status kvc_compact(kvc_shape shape, const void* K, const void* V, const int32_t* kept,
                       const int32_t* k_per_layer, void* Kc, void* Vc, kvc_stream stream);

/* kvc_evict_topk followed by kvc_compact, in one launch: each (layer, KV
 * head) copies its kept K/V rows into the compacted cache as soon as it has
 * chosen them (the same results as the two calls; one kernel ramp instead
 * of two).  Arguments, layouts and errors as in those two calls; ws needs
 * at least 256 bytes, 256-byte aligned. */
KVC_API kvc_status kvc_evict_compact(kvc_shape shape, float* score, int32_t sinks, const int32_t* k_per_layer,
                                     int32_t* kept, const void* K, const void* V, void* Kc, void* Vc, void* ws,
                                     size_t ws_bytes, kvc_stream stream);

/* Whole KV² compression: proxy, then `passes` rounds of query selection and
 * reconstruction scoring (each round's mean score replacing the proxy),
 * then eviction and compaction.  Outputs as in the entry points above;
 * p_opt [N], sel_opt [Q] (last pass) and score_opt [L][Hkv][N] may be NULL
 * (the workspace holds them then; without score_opt the sinks' scores are
 * not pinned, as nothing reads them: the sinks are kept either way). */
KVC_API kvc_status kvc_compress(kvc_shape shape, const void* K, const void* V, const void* Qpool, int32_t sinks, int32_t m,
                        double rho, int32_t passes, const int32_t* k_per_layer, int32_t* kept, void* Kc, void* Vc,
                        float* p_opt, int32_t* sel_opt, float* score_opt, void* ws, size_t ws_bytes,
                        kvc_stream stream);

/* kvc_compress with a selectable stage-1 proxy (kvc_compress uses KeyDiff)
 * and an optional event `gather_done` (NULL: none), recorded on `stream`
 * right after the last pass's gather of the reconstruction queries.  When
 * Qpool (and V) are page-locked host memory read in place, that gather is
 * the call's last large read across the host link: a caller streaming the
 * next cache to the device can make its copy wait on this event so that the
 * two do not compete for the link.  The event must have been created by the
 * caller (cudaEventCreate*); the library only records it. */
KVC_API kvc_status kvc_compress_ex(kvc_shape shape, kvc_proxy_kind proxy, const void* K, const void* V,
                                   const void* Qpool, int32_t sinks, int32_t m, double rho, int32_t passes,
                                   const int32_t* k_per_layer, int32_t* kept, void* Kc, void* Vc, float* p_opt,
                                   int32_t* sel_opt, float* score_opt, void* ws, size_t ws_bytes, kvc_stream stream,
                                   kvc_event gather_done);

/* ------------------------------------------------------------------ EpiCache
 * "[26'ICML] EpiCache", "+α: 레이어별 예산 배분": per-layer budgets from a
 * sensitivity vector with sharpness alpha.  w_l = sens_l^alpha / sum_j
 * sens_j^alpha; the L * mean_budget tokens are split by largest remainder
 * (ties to the lower layer), then each budget is raised to at least `sinks`.
 * Host-only.  sens: host f32 [L] (> 0); k_per_layer: host int32 [L]. */
KVC_API kvc_status kvc_layer_budgets(const float* sens, int32_t L, double alpha, int64_t mean_budget, int32_t sinks,
                             int32_t* k_per_layer);

#define KVC_MAX_LAYERS 128

/* State of one episode's block prefill.  Device buffers are caller-owned;
 * the host fields are maintained by the library.  A layer's rows are always
 * at slab cur[l], rows [0, len[l]), in one of two layouts chosen at init:
 *   two slabs  every step moves the kept rows of each over-budget layer into
 *              its other slab in ascending position order (the EpiCache
 *              page's cache after every step, row order = position order);
 *   one slab   (K[1], V[1], pos[1] NULL, cur[l] always 0) kept rows stay
 *              where they are and each kept row of the new block moves into
 *              the row of an evicted one, so a step moves at most one block
 *              of rows and the state needs half the memory; rows are in no
 *              particular order (pos[0] holds each row's position) until
 *              kvc_episode_pack writes them in ascending position order.
 * Both keep the same rows at every step. */
typedef struct {
  int32_t L, Hkv, Hq, d;
  int32_t capacity;               /* rows per (layer, KV head) in each slab: >= max budget + block */
  int32_t sinks;
  void* K[2];                     /* device bf16 [L][Hkv][capacity][d] per slab ([1] NULL: one slab) */
  void* V[2];                     /* device bf16 [L][Hkv][capacity][d] per slab ([1] NULL: one slab) */
  int32_t* pos[2];                /* device int32 [L][Hkv][capacity]: global position of each row */
  int32_t cur[KVC_MAX_LAYERS];    /* host: slab holding layer l */
  int32_t len[KVC_MAX_LAYERS];    /* host: rows held per layer (same for every KV head) */
  int32_t budget[KVC_MAX_LAYERS]; /* host: M_l */
  int64_t consumed;               /* host: history tokens consumed */
} kvc_block_state;

/* Initialises `st` for an empty cache (no device work).  Each slab must hold
 * L*Hkv*capacity rows.  K1, V1 and pos1 all NULL select the one-slab layout
 * (capacity at most 393216 rows then).  Invalid: L > KVC_MAX_LAYERS,
 * d != 128, a budget below `sinks`, capacity below the largest budget, some
 * but not all of K1, V1, pos1 NULL. */
KVC_API kvc_status kvc_block_state_init(kvc_block_state* st, int32_t L, int32_t Hkv, int32_t Hq, int32_t d, int32_t capacity,
                                int32_t sinks, const int32_t* budgets, void* K0, void* V0, int32_t* pos0, void* K1,
                                void* V1, int32_t* pos1);

/* Workspace bytes for kvc_block_prefill_step with blocks of up to
 * `max_block` tokens and P prompt queries.  The workspace begins with the
 * last step's scores, f32 [L][Hkv][capacity]: for every layer that step
 * scored, row i of (l, h) holds the score of cache row i of the appended
 * cache (its kept rows, then the block) for i in [sinks, len + blk_len); the
 * rest of that region is unspecified.  Callers may read it for diagnostics
 * until the next call that uses the workspace. */
KVC_API size_t kvc_block_workspace_size(const kvc_block_state* st, int32_t max_block, int32_t P);

/* "[26'ICML] EpiCache", "방법: 3단계" step ② and Fig. 1(b,c): append one
 * history block behind each layer's kept cache; every layer that then holds
 * more than its budget M_l scores its non-sink rows against the episode's
 * patched prompt (the KV² max rule with the prompt's P queries appended
 * causally, prompt keys as the appended keys), pins the sinks, keeps the M_l
 * best rows per KV head (lower global position wins a tie) and compacts
 * them: into the other slab in position order (two slabs), or by moving the
 * kept block rows into evicted rows (one slab).  Peak cache size stays at
 * M_l + block.
 *   Kblk, Vblk  device bf16 [L][Hkv][blk_len][d]
 *   Qprompt     device bf16 [L][Hq][P][d]
 *   Kprompt     device bf16 [L][Hkv][P][d]
 * Requires len[l] + blk_len <= capacity. */
KVC_API kvc_status kvc_block_prefill_step(kvc_block_state* st, const void* Kblk, const void* Vblk, int32_t blk_len,
                                  const void* Qprompt, const void* Kprompt, int32_t P, void* ws, size_t ws_bytes,
                                  kvc_stream stream);

/* ------------------------------------------------------------------ decode
 * KV² page, "전제와 한계": the savings of compression reach decoding only
 * through a compact serving backend that attends over the physically
 * compacted cache, whose length differs per (layer, KV head).
 *
 * A segment is a run of rows of one KV head: rows [seg_off[s], seg_off[s] +
 * seg_len[s]) of Kc and Vc.  Its G query heads are rows q[s][0..G-1].  For
 * every (s, g), with z_i = scale * (q[s][g] . k_i) over the segment's rows:
 *   out[s][g][:] = sum_i softmax(z)_i * v_i        (float32)
 *   lse_opt[s][g] = log sum_i exp(z_i)             (natural log)
 * A segment of length 0 gets out = 0 and lse = -inf.
 *   Kc, Vc    device bf16 [kv_rows][128], 16-byte aligned
 *   seg_off   device int64 [n_seg]; seg_len device int32 [n_seg]
 *   max_len   host upper bound of every seg_len (plans the split of long
 *             segments; must match the value given to the workspace query)
 *   q         device bf16 [n_seg][G][128]; 1 <= G <= 8
 *   scale     softmax scale; <= 0 selects 1/sqrt(128)
 *   out       device f32 [n_seg][G][128]; lse_opt device f32 [n_seg][G] or NULL
 * Segments are independent, so one call can cover every (layer, KV head) of
 * one or many caches.  A segment with a negative or too long length, or rows
 * outside [0, kv_rows), is skipped and reported as KVC_ERR_BOUNDS by
 * kvc_stream_status (its output is left unwritten).  Calls sharing a
 * workspace must be stream-ordered. */
KVC_API size_t kvc_decode_workspace_size(int32_t n_seg, int32_t G, int32_t max_len);
KVC_API kvc_status kvc_decode_attention(int32_t n_seg, int32_t G, const void* Kc, const void* Vc, int64_t kv_rows,
                                        const int64_t* seg_off, const int32_t* seg_len, int32_t max_len,
                                        const void* q, float scale, float* out, float* lse_opt, void* ws,
                                        size_t ws_bytes, kvc_stream stream);

/* Segment table of a cache laid out as kvc_compact writes it: segment
 * s = l * Hkv + h starts at row Hkv * sum_{l' < l} k_{l'} + h * k_l and holds
 * k_l rows.  Host-only: k_per_layer, seg_off and seg_len are host arrays of
 * L, L*Hkv and L*Hkv entries.  The pages define no such table; it is the
 * addressing of the compacted layout. */
KVC_API kvc_status kvc_compact_segments(int32_t L, int32_t Hkv, const int32_t* k_per_layer, int64_t* seg_off,
                                        int32_t* seg_len);

/* ------------------------------------------------------------------ EpiCache per turn
 * "[26'ICML] EpiCache", "방법: 3단계" step ③ and Fig. 3: each turn the
 * question's embedding is matched to the closest episode and that episode's
 * compressed cache is brought in (a completely new topic gets a new cache);
 * idle episode caches wait in host memory.
 *
 * Closest episode of each question: episode[b] = argmin_e |q_b - c_e|^2
 * (squared Euclidean, fp32 accumulation; equal distances go to the lower e);
 * with tau > 0, a question whose closest centroid is farther than tau gets -1.
 *   queries    device f32 [B][De]; centroids device f32 [E][De]; De a
 *              multiple of 4, both 16-byte aligned
 *   episode    device int32 [B] (output)
 *   dist2_opt  device f32 [B][E] squared distances, or NULL */
KVC_API kvc_status kvc_episode_match(int32_t B, int32_t E, int32_t De, const float* queries, const float* centroids,
                                     float tau, int32_t* episode, float* dist2_opt, kvc_stream stream);

/* Rows of an episode's packed cache: Hkv * sum_l len[l] (host-only; -1 for
 * an invalid state). */
KVC_API int64_t kvc_episode_rows(const kvc_block_state* st);

/* Packs the kept rows of a block-prefill state into one contiguous image in
 * the compacted layout (segment (l, h) holds len[l] rows; kvc_compact_segments
 * with k_l = len[l] addresses it), so one copy moves the whole episode and
 * kvc_decode_attention reads it in place.  Every segment's rows are in
 * ascending position order, in either state layout.
 *   Kp, Vp    device bf16 [kvc_episode_rows][128] (output)
 *   pos_opt   device int32 [kvc_episode_rows] global positions, or NULL */
KVC_API kvc_status kvc_episode_pack(const kvc_block_state* st, void* Kp, void* Vp, int32_t* pos_opt,
                                    kvc_stream stream);

/* Episode swap: writes the active episode image back (device -> page-locked
 * host) on out_stream and brings another one in (page-locked host -> device)
 * on in_stream, so the two directions share the link at the same time.  Each
 * half is skipped when its byte count is 0.  Host buffers must be page-locked
 * and device buffers device memory (KVC_ERR_INVALID otherwise).  The copies
 * are asynchronous; order them against kernels with the streams. */
KVC_API kvc_status kvc_episode_swap(const void* dev_out, void* host_out, size_t bytes_out, const void* host_in,
                                    void* dev_in, size_t bytes_in, kvc_stream out_stream, kvc_stream in_stream);

/* ------------------------------------------------------------------ Q4 codec
 * "Agent Memory Below the Prompt: Persistent Q4 KV Cache for Multi-Agent LLM
 * Inference on Edge Devices", "방법론 및 시스템 설계": each agent's KV cache is
 * kept 4-bit quantized so that it is loaded back into attention instead of
 * being recomputed.  The page fixes no format; this one quantises every row
 * of 128 bf16 values in two groups of 64:
 *   offset = group min rounded down to bf16 (a -0 minimum counts as +0),
 *   step   = (group max - offset) / 15 in fp32 rounded up to bf16 (0 for a
 *            constant group),
 *   code   = clamp(rint((x - offset) / step), 0, 15) in IEEE fp32 (0 when
 *            step = 0), two codes per byte, even element in the low nibble;
 *   decoded value = bf16_rn(fp32(code * step) + offset), no fused multiply-add.
 * 72 bytes per row instead of 256.  Values must be finite and below 1e37 in
 * magnitude (larger ranges overflow the step).
 *   X       device bf16 [rows][128], 16-byte aligned
 *   codes   uint8 [rows][64]; params bf16 [rows][2][2] = (step, offset) per
 *           group; both 4-byte aligned
 * kvc_q4_decode reads codes and params from device memory or page-locked
 * host memory (read in place across the host link: only the 72 bytes per
 * row travel) and writes X in device memory. */
KVC_API kvc_status kvc_q4_encode(int64_t rows, const void* X, void* codes, void* params, kvc_stream stream);
KVC_API kvc_status kvc_q4_decode(int64_t rows, const void* codes, const void* params, void* X, kvc_stream stream);

#ifdef __cplusplus
}
#endif

#endif /* KVC_H_ */
