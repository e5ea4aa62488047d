/*
 * ltk.h -- C ABI of the GB300 fused Indexer-TopK library (libltk.so).
 *
 * The operation (LiteTopK: "Exploiting the Curse of Dimensionality for a Fused
 * Indexer-TopK Kernel in Long-Context Sparse Attention", gist.science technical
 * summary, Problem Statement and Methodology):
 *
 *   for each query t of a prefill chunk and every key s visible to it
 *   (causal: s <= positions[t]) compute the indexer score
 *
 *       I[t,s] = sum_h w[t,h] * ReLU(q[t,h,:] . k[s,:])
 *
 *   (the DeepSeek Sparse Attention indexer score, named I_{t,s} in the
 *   summary's bin map) and return the exact top-k keys of each query, without
 *   writing the T x S score matrix to device memory.  The library runs the
 *   summary's three stages -- Sample (Methodology step 1), Filter (step 2) and
 *   Select (step 3) -- as CUDA kernels for sm_103a.
 *
 * Conventions shared by every entry point
 *   - Pointers named "device" must point to device memory of the current
 *     device; they stay owned by the caller.  Every device pointer must be
 *     16-byte aligned (TMA requirement); misaligned pointers fail with
 *     LTK_ERR_ARG.
 *   - "stream" is a cudaStream_t passed as void* (NULL = legacy default
 *     stream).  Compute calls are asynchronous on that stream and never
 *     synchronise the host, except where stated.
 *   - Arguments are validated on the host before any launch; a bad argument
 *     returns LTK_ERR_ARG and enqueues nothing.
 *   - Output order: each query's k slots hold the selected keys sorted by
 *     (score descending, key index ascending); slots beyond min(k, V_t), V_t
 *     the number of visible keys, hold index -1 and score -inf.
 *   - Errors raised on the device (a bounded wait that timed out) are
 *     recorded in a status word that ltk_get_stats reports.
 *   - A handle is not thread-safe: calls on one handle must be serialised,
 *     and two calls on one handle must not overlap on the GPU (they share the
 *     handle's workspace), i.e. issue them on one stream or synchronise.
 */
#ifndef LTK_H
#define LTK_H

#ifdef __cplusplus
extern "C" {
#endif

#define LTK_ABI_VERSION 2

typedef enum {
  LTK_OK = 0,
  LTK_ERR_ARG = 1,          /* invalid argument; nothing was enqueued         */
  LTK_ERR_CUDA = 2,         /* a CUDA runtime/driver call failed              */
  LTK_ERR_NOMEM = 3,        /* workspace allocation failed                    */
  LTK_ERR_OVERFLOW = 4,     /* informational: candidate list overflowed; the
                               affected queries were recomputed exactly      */
  LTK_ERR_TIMEOUT = 5,      /* a bounded device-side wait expired             */
  LTK_ERR_UNSUPPORTED = 6   /* shape or mode the library does not implement   */
} ltk_status;

typedef enum { LTK_BF16 = 0, LTK_FP8_E4M3 = 1 } ltk_dtype;

/*
 * Handle configuration (fixed at ltk_create).
 *   heads, dim      H and d of q[T,H,d] and k[S,d] (see engine for the shapes
 *                   each kernel serves).
 *   dtype           LTK_BF16, or LTK_FP8_E4M3 with per-token fp32 scales
 *                   (q_scale[T], k_scale[S]; the value is code * scale).
 *   relu, causal    1 for the indexer score (ReLU per head, key s visible iff
 *                   s <= positions[t]).
 *   max_T, max_S    largest chunk and key cache the workspace is sized for.
 *   k               largest k a call may request (<= 8192).
 *   n_bins          equal-width bins of the Filter stage's gate
 *                   (Methodology step 2, "Bin Mapping"); power of two in
 *                   [32, 512] for bf16, [32, 2048] for fp8.
 *   cand_cap        per-query capacity of the candidate list written by the
 *                   Filter stage; 0 derives it from k and max_S.
 *   sample_size     k' = number of sample keys (Methodology step 1 uses
 *                   k' = 3k); 0 means 3k.  At most 16384.
 *   seed            seed of the random sample used when no previous-chunk
 *                   sample is given.
 *   refresh_interval  key tiles (128 keys) between threshold refreshes by the
 *                   refresh warp ("Threshold Refresh"); 0 disables refresh.
 *   enable_decoupled  1 also allocates the max_T x max_S fp32 score matrix of
 *                   the decoupled baseline (ltk_decoupled_topk).
 *   rescue_rows     queries recomputed concurrently when a candidate list
 *                   overflows (each holds a max_S fp32 score row); 0 = 16.
 *   enable_host_io  1 also allocates device staging for ltk_indexer_topk_host.
 *   engine          0 (auto): the tensor-core kernels where the shape allows
 *                   (H = 64 and d = 128 with ReLU; or H = 1, bf16, no mask),
 *                   otherwise the CUDA-core kernel; 1: tensor cores only;
 *                   2: the CUDA-core kernel with the fused affine bin map
 *                   (any 1 <= H <= 128, d a multiple of 8 -- of 16 for
 *                   e4m3 -- up to 4096, H * d * 4 + n_bins * 4 <= 100 KB).
 *   debug_flags     0 in normal use.  Bit 0 (tests of failure handling): the
 *                   Filter kernel's producer issues no key-tile loads, so its
 *                   bounded waits expire (about 2 s), the kernel records
 *                   LTK_ERR_TIMEOUT, releases its resources and returns; the
 *                   outputs are then undefined and ltk_get_stats reports the
 *                   status.
 */
typedef struct {
  int heads;
  int dim;
  int dtype;
  int relu;
  int causal;
  int max_T;
  long long max_S;
  int k;
  int n_bins;
  int cand_cap;
  int sample_size;
  unsigned long long seed;
  int refresh_interval;
  int enable_decoupled;
  int rescue_rows;
  int enable_host_io;
  int engine;
  int debug_flags;
} ltk_config;

typedef struct ltk_handle ltk_handle;

/*
 * Per-call statistics of the last compute call on a handle.  Reading them
 * synchronises the stream of that call.
 *   cand_written   candidates that passed the gate, summed over queries
 *                  (bytes written per query = 8 * cand_written / T + 8 * k).
 *   cand_max       largest per-query candidate count.
 *   n_overflow     queries whose list exceeded cand_cap (recomputed exactly).
 *   device_status  first error code raised on the device, 0 if none.
 *   visible_pairs  query-key pairs the last call scored (sum of V_t).
 *   ms_*           stage times from CUDA events recorded on each call's
 *                  stream while timing is enabled (ltk_set_timing), averaged
 *                  over the last timed_calls calls (at most 64) since timing
 *                  was last enabled; -1 when no call was timed.
 *   launches       kernels this library launched in the process so far.
 */
typedef struct {
  int T;
  long long S;
  int k;
  long long visible_pairs;
  long long cand_written;
  int cand_max;
  int n_overflow;
  int device_status;
  float ms_sample;
  float ms_filter;
  float ms_select;
  float ms_rescue;
  float ms_total;
  int timed_calls;
  long long launches;
} ltk_stats;

/* ABI version of the loaded library (LTK_ABI_VERSION). */
int ltk_abi_version(void);

/* Static text of a status code. */
const char* ltk_status_string(int status);

/* Fills *cfg with defaults for the indexer (bf16, ReLU, causal, n_bins 512,
 * refresh every tile, derived cand_cap, k' = 3k).  Host only. */
ltk_status ltk_config_init(ltk_config* cfg, int heads, int dim, int k, int max_T,
                           long long max_S);

/* Device bytes ltk_create would allocate for *cfg.  Host only (no CUDA
 * call); LTK_ERR_ARG / LTK_ERR_UNSUPPORTED for an invalid configuration. */
ltk_status ltk_workspace_bytes(const ltk_config* cfg, unsigned long long* bytes);

/* Validates *cfg and allocates the handle and its device workspace on the
 * current device.  The workspace is owned by the handle. */
ltk_status ltk_create(const ltk_config* cfg, ltk_handle** out);

/* Frees the handle and its workspace (synchronises the device first).
 * NULL is accepted. */
void ltk_destroy(ltk_handle* h);

/* Enables (1) or disables (0) per-stage CUDA-event timing on later calls;
 * enabling also restarts the averaging window of ltk_get_stats. */
ltk_status ltk_set_timing(ltk_handle* h, int enable);

/*
 * Seeded random sample for a first chunk (Methodology step 1 contrasts the
 * previous-chunk sample with random sampling): n distinct key ids drawn one
 * per stratum of [0, S), written to sample_out[n] (device int32).
 */
ltk_status ltk_random_sample(ltk_handle* h, long long S, int n, int* sample_out,
                             void* stream);

/*
 * Previous-chunk sample (Methodology step 1: reuse the top-k' tokens of the
 * previous chunk's results, k' = 3k).  prev_idx[T_prev, k_prev] (device int32)
 * is the previous chunk's output; entries < 0 or >= S are ignored.  Key ids
 * are ranked by how many of the previous chunk's queries selected them (ties:
 * higher id first); if fewer than n ids were selected at all, the rest is
 * filled with pseudo-random unselected ids.  Writes n distinct ids to
 * sample_out[n] (device).  Requires n <= S and S <= max_S.
 */
ltk_status ltk_make_sample(ltk_handle* h, const int* prev_idx, int T_prev, int k_prev,
                           long long S, int n, int* sample_out, void* stream);

/*
 * Fused Indexer-TopK (Sample -> Filter -> Select).
 *   q          device [T, H, d] bf16 or e4m3, row-major.
 *   q_scale    device [T] fp32 (e4m3 only, > 0), else NULL.
 *   w          device [T, H] fp32 head weights (any sign).
 *   k_cache    device [S, d] bf16 or e4m3, row-major.
 *   k_scale    device [S] fp32 (e4m3 only, > 0), else NULL.
 *   positions  device [T] int32 absolute query positions (causal mask);
 *              ignored when the handle is not causal.
 *   prev_topk  device int32 sample key ids (e.g. from ltk_make_sample), or
 *              NULL for a seeded random sample of sample_size keys.  Ids
 *              outside [0, S) and duplicates are dropped; ids invisible to a
 *              query are skipped for that query.  n_prev <= 16384.
 *   k          1 <= k <= cfg.k.
 *   out_idx    device [T, k] int32; out_score device [T, k] fp32 (the
 *              kernel's fp32 score of each selected key).
 * 0 <= T <= max_T, 1 <= S <= max_S.  T == 0 enqueues nothing.
 * The call neither synchronises nor allocates, so it can be captured in a CUDA
 * graph (stream capture) and replayed: the graph reads the buffers named here
 * at replay time, and a replay overwrites the handle's statistics like a call.
 * Make one call on the handle outside capture first (it sets kernel
 * attributes on the device), and keep timing off while capturing.
 */
ltk_status ltk_indexer_topk(ltk_handle* h, const void* q, const float* q_scale,
                            const float* w, const void* k_cache, const float* k_scale,
                            const int* positions, int T, long long S,
                            const int* prev_topk, int n_prev, int k,
                            int* out_idx, float* out_score, void* stream);

/*
 * Same contract as ltk_indexer_topk, but every pointer is HOST memory
 * (pinned for asynchronous copies).  The library copies the inputs into its
 * own device staging (enable_host_io), runs the fused path and copies the
 * results back; the call returns once the results are in out_idx/out_score.
 */
ltk_status ltk_indexer_topk_host(ltk_handle* h, const void* q, const float* q_scale,
                                 const float* w, const void* k_cache, const float* k_scale,
                                 const int* positions, int T, long long S,
                                 const int* prev_topk, int n_prev, int k,
                                 int* out_idx, float* out_score, void* stream);

/*
 * Decoupled baseline (the DSA-style two-stage design the summary's Problem
 * Statement describes): write the full fp32 score matrix [T, S] to device
 * memory with the same tensor-core scorer, then run a radix select over each
 * row, reading it several times.  Same arguments and output contract as
 * ltk_indexer_topk (no sample).  Needs enable_decoupled.
 */
ltk_status ltk_decoupled_topk(ltk_handle* h, const void* q, const float* q_scale,
                              const float* w, const void* k_cache, const float* k_scale,
                              const int* positions, int T, long long S, int k,
                              int* out_idx, float* out_score, void* stream);

/*
 * Decoupled top-k that allocates nothing (no counterpart in the paper: it is
 * an integration convenience).  For callers that cannot call cudaMalloc -- a
 * plugin inside an engine that owns all device memory through its own pool,
 * or a latency-critical path where cudaMalloc's implicit device
 * synchronisation is not acceptable.  Same computation and output contract as
 * ltk_decoupled_topk for H = 64, d = 128, ReLU scores, without a handle:
 * dtype is LTK_BF16 or LTK_FP8_E4M3, causal selects the s <= positions[t]
 * mask.  Its scratch, the T x S fp32 score matrix, lives in a static device
 * array of 4,194,304 floats (16 MiB) that every GPU loading the library
 * holds until process exit; T * S above that returns LTK_ERR_ARG.  The
 * caller still owns all inputs and outputs.
 *   device_status  device int (4-byte aligned, caller-owned) or NULL.  The
 *                  call zeroes it on the stream; a bounded wait in the scorer
 *                  that expires (about 2 s) stores LTK_ERR_TIMEOUT there, and
 *                  the outputs of that call are then undefined.  Read it after
 *                  the stream has finished the call.  With NULL such an error
 *                  is not reported anywhere.
 * Each call looks up the array's device address with the caller's device
 * current (no allocation); the first call on a device also loads the
 * library's kernels there and sets their attributes, so make it before any
 * stream capture.  All calls share the array, so calls that overlap on the
 * GPU race and corrupt each other's results: serialise them (one stream, or
 * synchronise between calls).
 */
ltk_status ltk_decoupled_topk_noalloc(int dtype, int causal, const void* q, const float* q_scale,
                                      const float* w, const void* k_cache, const float* k_scale,
                                      const int* positions, int T, long long S, int k,
                                      int* out_idx, float* out_score, int* device_status,
                                      void* stream);

/*
 * LiteDSA candidate packing (LiteTopK arXiv abstract: LiteDSA packs the
 * overlapping candidates of neighbouring query tokens into a shared key/value
 * list for joint attention, with per-query masks that keep each token's own
 * top-k membership).  Consecutive queries form groups of `group`; for group g
 * (queries g*group .. g*group+group-1, the last group may be short):
 *   union_idx  device int32 [ceil(T/group), group*k]: the ascending set union
 *              of the group's valid (>= 0) indices, padded with -1;
 *   union_len  device int32 [ceil(T/group)]: number of valid union entries;
 *   masks      device uint32 [T, ceil(group*k/32)]: bit j of query t's row is
 *              set iff union entry j of t's group is one of t's indices.
 * topk_idx is device int32 [T, k] (e.g. ltk_indexer_topk's out_idx; a row
 * holds distinct indices, -1 = empty slot).  No handle, no allocation.
 * group in [1, 256]; group*k <= 16384 and the group's shared-memory footprint
 * (sorted keys + masks) <= 200 KB, else LTK_ERR_UNSUPPORTED.
 */
ltk_status ltk_litedsa_pack(const int* topk_idx, int T, int k, int group, int* union_idx,
                            int* union_len, unsigned int* masks, void* stream);

/* Statistics of the last compute call (synchronises its stream). */
ltk_status ltk_get_stats(ltk_handle* h, ltk_stats* out);

#ifdef __cplusplus
}
#endif

#endif /* LTK_H */
