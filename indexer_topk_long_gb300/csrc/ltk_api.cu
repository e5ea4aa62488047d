// ltk_api.cu -- C ABI of libltk: argument validation, workspace ownership and
// the launch sequence of the fused Indexer-TopK (Sample -> Filter -> Select)
// and of the decoupled baseline.
//
// LiteTopK technical summary (gist.science): Problem Statement (decoupled
// score-then-select design that materialises the score matrix), Methodology
// steps 1-3 (Sample, Filter, Select).
#include <cudaTypedefs.h>

#include <atomic>
#include <cmath>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <new>

#include "ltk_internal.cuh"

using namespace ltk;

struct ltk_handle {
  ltk_config cfg;
  int device = 0;
  int cap = 0;
  int n_pad_max = 0;
  int rescue_rows = 0;
  int num_sms = 148;
  size_t elem = 2;
  // workspace
  float* samp_scores = nullptr;        // [max_T, n_pad_max]
  void* k_samp = nullptr;              // [n_pad_max, d]
  float* k_scale_samp = nullptr;       // [n_pad_max]
  int* key_ids_pad = nullptr;          // [n_pad_max]
  uint32_t* id_bitmap = nullptr;       // [ceil(max_S / 32)] sample-id dedupe bitmap, clear between calls
  int* id_block_sums = nullptr;        // per-CTA bit counts of the bitmap listing
  int* sample_tmp = nullptr;           // [kMaxSample]
  float* s_min = nullptr;              // [max_T]
  float* delta = nullptr;              // [max_T]
  int* theta0 = nullptr;               // [max_T]
  unsigned long long* cand = nullptr;  // [max_T, cap]
  int* cnt = nullptr;                  // [max_T]
  int* ovf = nullptr;                  // [2 + max_T]: count, next, list
  int* ghist = nullptr;                // [max_T, n_bins] per-query histograms shared by CTAs
  int* seg_cnt = nullptr;              // [max_T, num_sms] segment counts (retrieval lists)
  int last_nseg = 0;                   // segments per query list of the last fused call (0: one list)
  float* rescue_scratch = nullptr;     // [rescue_rows, max_S]
  float* dense = nullptr;              // [max_T, max_S] (decoupled baseline)
  int* status = nullptr;               // [1]
  MakeSampleWs ms{};
  // host-io staging
  void* io_q = nullptr;
  float* io_qs = nullptr;
  float* io_w = nullptr;
  void* io_k = nullptr;
  float* io_ks = nullptr;
  int* io_pos = nullptr;
  int* io_prev = nullptr;
  int* io_oidx = nullptr;
  float* io_oscore = nullptr;
  // timing: a ring of per-call stage events (5 per call)
  static constexpr int kRing = 64;
  cudaEvent_t ring[kRing][5] = {};
  int timing = 0;
  int ring_calls = 0;                  // timed calls since timing was enabled
  cudaEvent_t* ev = nullptr;           // events of the current call (or null)
  unsigned long long* pairs = nullptr; // [2] visible pairs of the last call; key tiles scanned so
                                       // far by the filter (its sweep position, see ScoreParams)
  int last_kind = 0;                   // 0 none, 1 fused, 2 decoupled
  // last call
  int last_T = 0;
  long long last_S = 0;
  int last_k = 0;
  cudaStream_t last_stream = nullptr;
};

namespace ltk {
namespace {
std::atomic<long long> g_launches{0};
}
void count_launches(int n) { g_launches.fetch_add(n, std::memory_order_relaxed); }

namespace {
constexpr int kMaxDevices = 256;
std::atomic<unsigned int> g_smem_done[kMaxDevices] = {};   // bit per slot
}

cudaError_t ensure_smem_limit(const void* func, int slot, size_t bytes) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  const unsigned int bit = 1u << slot;
  if (g_smem_done[dev].load(std::memory_order_acquire) & bit) return cudaSuccess;
  e = cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(bytes));
  if (e == cudaSuccess) g_smem_done[dev].fetch_or(bit, std::memory_order_release);
  return e;
}
long long launches_so_far() { return g_launches.load(std::memory_order_relaxed); }
}  // namespace ltk

namespace {

ltk_status cuda_fail(cudaError_t e, const char* what) {
  if (e == cudaSuccess) return LTK_OK;
  if (std::getenv("LTK_DEBUG")) std::fprintf(stderr, "ltk: %s: %s\n", what, cudaGetErrorString(e));
  cudaGetLastError();
  return e == cudaErrorMemoryAllocation ? LTK_ERR_NOMEM : LTK_ERR_CUDA;
}

#define LTK_CUDA(call)                                      \
  do {                                                      \
    cudaError_t e_ = (call);                                \
    if (e_ != cudaSuccess) return cuda_fail(e_, #call);     \
  } while (0)

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool is_pow2(int x) { return x > 0 && (x & (x - 1)) == 0; }
long long round_up(long long x, long long m) { return (x + m - 1) / m * m; }

int derived_cap(int k, long long max_S, int max_T) {
  // Expected candidates of a streaming threshold grow like k * (1 + ln(S / k));
  // the default keeps a 1.5x margin over k * (4 + ln(S / k)) plus 2048 records
  // (small k starts from a loose sample threshold), never above S (rounded).
  const double ratio = static_cast<double>(max_S) / static_cast<double>(k);
  const double est = k * (4.0 + std::log(ratio > 1.0 ? ratio : 1.0)) * 1.5 + 2048.0;
  long long cap = round_up(static_cast<long long>(est), 1024);
  // Small chunks (decode) split a query's keys over many CTAs, where the shared
  // threshold tightens in coarser steps; memory is no constraint there, so the
  // capacity grows to a budget of 2^27 records spread over max_T queries.
  const long long budget = round_up((1ll << 27) / (max_T > 0 ? max_T : 1), 1024);
  if (cap < budget) cap = budget;
  const long long s_cap = round_up(max_S, 1024);
  if (cap > s_cap) cap = s_cap;
  if (cap < k) cap = k;
  if (cap > (1ll << 30)) cap = 1ll << 30;
  return static_cast<int>(cap);
}

// Shapes each kernel serves.
bool tc_shape(const ltk_config* c) {
  return c->heads == kTcHeads && c->dim == kTcDim && c->relu == 1 &&
         c->n_bins <= score_tc_max_bins(c->dtype == LTK_FP8_E4M3);
}
bool retrieval_shape(const ltk_config* c) {
  return c->heads == 1 && c->dtype == LTK_BF16 && !c->causal && c->dim % 64 == 0 &&
         c->dim <= kRetrievalMaxDim && c->n_bins <= kRetrievalMaxBins && (c->relu == 0 || c->relu == 1);
}
bool cc_shape(const ltk_config* c) {
  const int elem = c->dtype == LTK_FP8_E4M3 ? 1 : 2;
  return c->heads >= 1 && c->heads <= 128 && c->dim % 8 == 0 && c->dim <= 4096 &&
         (c->dim * elem) % 16 == 0 && (c->relu == 0 || c->relu == 1) && c->n_bins <= 4096 &&
         score_cc_smem_bytes(c->heads, c->dim, c->n_bins) <= kCcMaxSmem;
}
// The CUDA-core scorer runs when asked for, or when no tensor-core kernel
// serves the shape.
bool use_cc(const ltk_config* c) {
  return c->engine == 2 || (c->engine == 0 && !tc_shape(c) && !retrieval_shape(c));
}
// One head on the tensor-core path: the vector-retrieval kernel.
bool is_retrieval(const ltk_config* c) { return c->heads == 1 && !use_cc(c); }

ltk_status validate_config(const ltk_config* c) {
  if (c == nullptr) return LTK_ERR_ARG;
  if (c->heads <= 0 || c->dim <= 0 || c->max_T < 0 || c->max_S <= 0) return LTK_ERR_ARG;
  if (c->max_S > 0x7FFFFFFFll) return LTK_ERR_ARG;                 // key ids are int32
  if (c->k <= 0 || c->k > kMaxK) return LTK_ERR_ARG;
  if (c->dtype != LTK_BF16 && c->dtype != LTK_FP8_E4M3) return LTK_ERR_ARG;
  if (c->sample_size < 0 || c->sample_size > kMaxSample) return LTK_ERR_ARG;
  if (c->cand_cap < 0 || c->refresh_interval < 0 || c->rescue_rows < 0) return LTK_ERR_ARG;
  if (c->debug_flags & ~1) return LTK_ERR_ARG;
  if (!is_pow2(c->n_bins) || c->n_bins < 32) return LTK_ERR_ARG;
  if (c->engine < 0 || c->engine > 2) return LTK_ERR_ARG;
  if (c->engine == 1 && !tc_shape(c) && !retrieval_shape(c)) return LTK_ERR_UNSUPPORTED;
  if (c->engine == 2 && !cc_shape(c)) return LTK_ERR_UNSUPPORTED;
  if (c->engine == 0 && !tc_shape(c) && !retrieval_shape(c) && !cc_shape(c)) return LTK_ERR_UNSUPPORTED;
  return LTK_OK;
}

struct Sizes {
  int cap, n_pad_max, rescue_rows;
  size_t elem;
  unsigned long long total;
};

Sizes compute_sizes(const ltk_config* c) {
  Sizes s{};
  s.elem = c->dtype == LTK_FP8_E4M3 ? 1 : 2;
  s.cap = c->cand_cap > 0 ? c->cand_cap : derived_cap(c->k, c->max_S, c->max_T);
  const int ss = c->sample_size > 0 ? c->sample_size : (3 * c->k > kMaxSample ? kMaxSample : 3 * c->k);
  s.n_pad_max = static_cast<int>(round_up(kMaxSample > ss ? kMaxSample : ss, kTile));
  s.rescue_rows = c->rescue_rows > 0 ? c->rescue_rows : 16;
  const unsigned long long T = static_cast<unsigned long long>(c->max_T > 0 ? c->max_T : 1);
  const unsigned long long S = static_cast<unsigned long long>(c->max_S);
  unsigned long long b = 0;
  b += T * s.n_pad_max * 4;                           // sample scores
  b += static_cast<unsigned long long>(s.n_pad_max) * c->dim * s.elem;   // gathered keys
  b += static_cast<unsigned long long>(s.n_pad_max) * 4 * 2;            // scales + ids
  b += (S + 31) / 32 * 4 + (S + 32767) / 32768 * 4 + 4;   // sample-id bitmap + per-CTA counts
  b += kMaxSample * 4ull;                             // random sample ids
  b += T * 4 * 4;                                     // s_min, delta, theta0, cnt
  b += T * static_cast<unsigned long long>(c->n_bins) * 4;   // per-query histograms shared by CTAs
  if (is_retrieval(c)) b += T * 256ull * 4;           // segment counts (at most one segment per SM)
  b += T * static_cast<unsigned long long>(s.cap) * 8;  // candidate lists
  b += (T + 2) * 4;                                   // overflow list
  b += static_cast<unsigned long long>(s.rescue_rows) * S * 4;   // rescue rows
  b += S * 4 + S * 8 + 256 * 4 + 4 * 8;               // previous-chunk sample
  b += 4;                                             // status
  if (c->enable_decoupled) b += T * S * 4;
  if (c->enable_host_io) {
    b += T * c->heads * c->dim * s.elem + T * 4 + T * c->heads * 4 + S * c->dim * s.elem + S * 4 +
         T * 4 + kMaxSample * 4 + T * c->k * 8ull;
  }
  s.total = b;
  return s;
}

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (fn == nullptr) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  }
  return fn;
}

// 2-D tiled map over a row-major [rows, dim] matrix of bf16 or e4m3 codes:
// boxes of 128 bytes x box_rows rows, 128-byte swizzle.
bool make_tmap(CUtensorMap* m, const void* base, bool fp8, int dim, unsigned long long rows,
               int box_rows) {
  auto enc = tensor_map_encoder();
  if (enc == nullptr) return false;
  const cuuint32_t elem = fp8 ? 1 : 2;
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(dim), static_cast<cuuint64_t>(rows)};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(dim) * elem};
  const cuuint32_t box[2] = {128 / elem, static_cast<cuuint32_t>(box_rows)};
  const cuuint32_t estr[2] = {1, 1};
  const CUresult r =
      enc(m, fp8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2,
          const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
          CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

template <typename T>
cudaError_t alloc(T** p, unsigned long long bytes) {
  *p = nullptr;
  if (bytes == 0) return cudaSuccess;
  return cudaMalloc(reinterpret_cast<void**>(p), bytes);
}

void free_all(ltk_handle* h) {
  void* ptrs[] = {h->ghist, h->samp_scores, h->k_samp, h->k_scale_samp, h->key_ids_pad, h->id_bitmap,
                  h->id_block_sums, h->seg_cnt,
                  h->sample_tmp,
                  h->s_min,       h->delta,   h->theta0,       h->cand,         h->cnt,
                  h->ovf,         h->rescue_scratch, h->dense, h->status,       h->ms.counts,
                  h->ms.keys,     h->ms.hist, h->ms.state,     h->io_q,         h->io_qs,
                  h->io_w,        h->io_k,    h->io_ks,        h->io_pos,       h->io_prev,
                  h->io_oidx,     h->io_oscore};
  for (void* p : ptrs)
    if (p) cudaFree(p);
  if (h->pairs) cudaFree(h->pairs);
  for (auto& row : h->ring)
    for (auto& e : row)
      if (e) cudaEventDestroy(e);
}

// Events of this call's stages, or null when timing is off.
cudaEvent_t* begin_timed_call(ltk_handle* h) {
  if (!h->timing) return nullptr;
  cudaEvent_t* ev = h->ring[h->ring_calls % ltk_handle::kRing];
  ++h->ring_calls;
  return ev;
}

bool current_device_is(int dev) {
  int cur = -1;
  return cudaGetDevice(&cur) == cudaSuccess && cur == dev;
}

struct CallArgs {
  const void* q;
  const float* q_scale;
  const float* w;
  const void* k_cache;
  const float* k_scale;
  const int* positions;
  int T;
  long long S;
  int k;
  int* out_idx;
  float* out_score;
};

ltk_status validate_call(const ltk_handle* h, const CallArgs& a) {
  if (h == nullptr) return LTK_ERR_ARG;
  const ltk_config& c = h->cfg;
  if (a.T < 0 || a.T > c.max_T) return LTK_ERR_ARG;
  if (a.S < 1 || a.S > c.max_S) return LTK_ERR_ARG;
  if (a.k < 1 || a.k > c.k) return LTK_ERR_ARG;
  if (a.T == 0) return LTK_OK;
  if (!a.q || !a.w || !a.k_cache || !a.out_idx || !a.out_score) return LTK_ERR_ARG;
  if (!aligned16(a.q) || !aligned16(a.w) || !aligned16(a.k_cache) || !aligned16(a.out_idx) ||
      !aligned16(a.out_score))
    return LTK_ERR_ARG;
  if (c.causal && (a.positions == nullptr || !aligned16(a.positions))) return LTK_ERR_ARG;
  if (c.dtype == LTK_FP8_E4M3) {
    if (!a.q_scale || !a.k_scale || !aligned16(a.q_scale) || !aligned16(a.k_scale)) return LTK_ERR_ARG;
  }
  if (!current_device_is(h->device)) return LTK_ERR_ARG;
  return LTK_OK;
}

// The scorer for the handle's shape: the tensor-core indexer kernel (H = 64,
// d = 128), the tensor-core retrieval kernel (one head), or the CUDA-core
// kernel (any other shape, or when asked for).
cudaError_t launch_scorer(const ltk_handle* h, int mode, const CUtensorMap& qm, const CUtensorMap& km,
                          const ScoreParams& p, cudaStream_t st) {
  const ltk_config& c = h->cfg;
  if (use_cc(&c)) {
    CcParams cp{};
    cp.q = p.q_raw;
    cp.q_scale = p.q_scale;
    cp.w = p.w;
    cp.k_cache = p.k_raw;
    cp.k_scale = p.k_scale;
    cp.positions = p.positions;
    cp.key_ids = p.key_ids;
    cp.T = p.T;
    cp.rows = p.rows;
    cp.H = c.heads;
    cp.d = c.dim;
    cp.causal = p.causal;
    cp.relu = c.relu;
    cp.s_min = p.s_min;
    cp.delta = p.delta;
    cp.theta0 = p.theta0;
    cp.cand = p.cand;
    cp.cnt = p.cnt;
    cp.ghist = p.ghist;
    cp.cap = p.cap;
    cp.nb = p.nb;
    cp.k = p.k;
    cp.refresh_interval = p.refresh_interval;
    cp.b_full = p.b_full;
    cp.s_last = p.s_last;
    cp.status = p.status;
    cp.dense = p.dense;
    cp.ld = p.ld;
    return launch_score_cc(mode, c.dtype == LTK_FP8_E4M3, cp, st);
  }
  if (is_retrieval(&c))
    return launch_retrieval_tc(mode, qm, km, p, c.dim, c.relu, h->ghist, h->num_sms, st);
  return launch_score_tc(mode, c.dtype == LTK_FP8_E4M3, qm, km, p, st);
}

// Work split of the indexer scorer over (query block, key range) units.  Whole
// waves of query blocks stay unsplit; the query blocks of a partial last wave
// (or of a chunk smaller than one wave, e.g. decode) are split along the keys
// into s_last ranges, chosen so that the split units fill the SMs best, with
// at least min_tiles key tiles per range (a filter range starts from the
// sample's threshold, so it must not be tiny; dense scoring has no such limit)
// and at most one range per SM.
void plan_split(int T, long long S, int num_sms, int min_tiles, int* b_full, int* s_last) {
  const int t_blocks = (T + kTcQPB - 1) / kTcQPB;
  const long long tiles = (S + kTile - 1) / kTile;
  const long long by_tiles = tiles / min_tiles;
  const int max_s = static_cast<int>(by_tiles > 1 ? (by_tiles < num_sms ? by_tiles : num_sms) : 1);
  *b_full = t_blocks;
  *s_last = 1;
  if (t_blocks == 0 || max_s <= 1) return;
  const int rem = t_blocks % num_sms;
  if (t_blocks < num_sms) {
    *b_full = 0;
    int sl = num_sms / t_blocks;
    *s_last = sl < max_s ? sl : max_s;
    if (*s_last < 1) *s_last = 1;
    return;
  }
  if (rem == 0) return;
  double best = 1.0;
  int best_s = 1;
  for (int sl = 2; sl <= 8 && sl <= max_s; ++sl) {
    const double cost = static_cast<double>((rem * sl + num_sms - 1) / num_sms) / sl;
    if (cost < best - 0.02) {
      best = cost;
      best_s = sl;
    }
  }
  if (best_s > 1) {
    *b_full = t_blocks - rem;
    *s_last = best_s;
  }
}

// Work units of the CUDA-core scorer: one query each; with fewer queries than
// four per SM the key ranges are split (at least 4096 keys per range).
void plan_split_cc(int T, long long S, int num_sms, int* b_full, int* s_last) {
  *b_full = T;
  *s_last = 1;
  if (T <= 0 || T >= 4 * num_sms) return;
  long long sl = (4ll * num_sms) / T;
  const long long by_keys = S / 4096;
  if (sl > by_keys) sl = by_keys;
  if (sl > 1) {
    *b_full = 0;
    *s_last = static_cast<int>(sl);
  }
}

// Work plan for the handle's scorer; *queries_per_unit is how many queries one
// unrolled unit covers (for the rows of split units).
void plan_work(const ltk_handle* h, int T, long long S, bool dense, int* b_full, int* s_last,
               int* queries_per_unit) {
  if (use_cc(&h->cfg)) {
    plan_split_cc(T, S, h->num_sms, b_full, s_last);
    *queries_per_unit = 1;
  } else {
    plan_split(T, S, h->num_sms, dense ? 2 : 32, b_full, s_last);
    *queries_per_unit = kTcQPB;
  }
}

// Rows of q seen by TMA: [T * H, d].
unsigned long long q_rows(const ltk_config& c, int T) {
  return static_cast<unsigned long long>(T) * c.heads;
}

ltk_status run_fused(ltk_handle* h, const CallArgs& a, const int* prev_topk, int n_prev,
                     cudaStream_t st) {
  const ltk_config& c = h->cfg;
  const bool fp8 = c.dtype == LTK_FP8_E4M3;
  h->last_kind = 1;
  h->last_T = a.T;
  h->last_S = a.S;
  h->last_k = a.k;
  h->last_stream = st;
  if (a.T == 0) return LTK_OK;
  h->ev = begin_timed_call(h);
  if (h->ev) LTK_CUDA(cudaEventRecord(h->ev[0], st));
  LTK_CUDA(cudaMemsetAsync(h->status, 0, sizeof(int), st));
  LTK_CUDA(cudaMemsetAsync(h->pairs, 0, 2 * sizeof(unsigned long long), st));
  LTK_CUDA(cudaMemsetAsync(h->ovf, 0, 2 * sizeof(int), st));

  // ---- Sample (Methodology step 1)
  const int ss = c.sample_size > 0 ? c.sample_size : (3 * c.k > kMaxSample ? kMaxSample : 3 * c.k);
  int n_s;
  const int* ids;
  if (prev_topk != nullptr) {
    n_s = n_prev;
    ids = prev_topk;
  } else {
    n_s = static_cast<int>(ss < a.S ? ss : a.S);
    LTK_CUDA(launch_random_sample(a.S, n_s, c.seed, h->sample_tmp, st));
    ids = h->sample_tmp;
  }
  const int n_pad = static_cast<int>(round_up(n_s > 0 ? n_s : 1, kTile));
  LTK_CUDA(launch_prepare_sample(ids, n_s, a.S, n_pad, h->key_ids_pad, h->id_bitmap, h->id_block_sums, st));
  LTK_CUDA(launch_gather_keys(a.k_cache, a.k_scale, static_cast<int>(h->elem), c.dim, h->key_ids_pad,
                              n_pad, h->k_samp, h->k_scale_samp, st));
  CUtensorMap q_map, ks_map, k_map;
  std::memset(&q_map, 0, sizeof(q_map));
  std::memset(&ks_map, 0, sizeof(ks_map));
  std::memset(&k_map, 0, sizeof(k_map));
  if (!use_cc(&c) &&
      (!make_tmap(&q_map, a.q, fp8, c.dim, q_rows(c, a.T), 256) ||
       !make_tmap(&ks_map, h->k_samp, fp8, c.dim, n_pad, kTile) ||
       !make_tmap(&k_map, a.k_cache, fp8, c.dim, static_cast<unsigned long long>(a.S), kTile)))
    return LTK_ERR_CUDA;
  int qpu = kTcQPB;
  ScoreParams sp{};
  sp.q_raw = a.q;
  sp.k_raw = h->k_samp;
  sp.w = a.w;
  sp.q_scale = a.q_scale;
  sp.k_scale = h->k_scale_samp;
  sp.positions = c.causal ? a.positions : nullptr;
  sp.key_ids = h->key_ids_pad;
  sp.T = a.T;
  sp.rows = n_pad;
  sp.causal = c.causal;
  sp.dense = h->samp_scores;
  sp.ld = n_pad;
  sp.status = h->status;
  plan_work(h, a.T, n_pad, true, &sp.b_full, &sp.s_last, &qpu);
  LTK_CUDA(launch_scorer(h, kModeDense, q_map, ks_map, sp, st));
  SampleStatsParams stp{h->samp_scores, n_pad, n_pad, a.T, a.k, c.n_bins, h->s_min, h->delta, h->theta0,
                        use_cc(&c) ? 1 : 0};
  LTK_CUDA(launch_sample_stats(stp, h->num_sms, st));
  if (h->ev) LTK_CUDA(cudaEventRecord(h->ev[1], st));

  // ---- Filter (Methodology step 2)
  ScoreParams fp{};
  fp.q_raw = a.q;
  fp.k_raw = a.k_cache;
  fp.w = a.w;
  fp.q_scale = a.q_scale;
  fp.k_scale = a.k_scale;
  fp.positions = c.causal ? a.positions : nullptr;
  fp.key_ids = nullptr;
  fp.T = a.T;
  fp.rows = a.S;
  fp.causal = c.causal;
  fp.s_min = h->s_min;
  fp.delta = h->delta;
  fp.theta0 = h->theta0;
  fp.cand = h->cand;
  fp.cnt = h->cnt;
  fp.cap = h->cap;
  fp.nb = c.n_bins;
  fp.k = a.k;
  fp.refresh_interval = c.refresh_interval;
  fp.skip_key_loads = (c.debug_flags & 1) ? 1 : 0;
  fp.sweep = h->pairs + 1;
  fp.num_sms = h->num_sms;
  fp.ghist = h->ghist;
  fp.status = h->status;
  plan_work(h, a.T, a.S, false, &fp.b_full, &fp.s_last, &qpu);
  if (!is_retrieval(&c) && fp.s_last > 1) {
    // split query blocks count and build histograms in global memory
    const size_t t_first = static_cast<size_t>(fp.b_full) * qpu;
    const size_t n = static_cast<size_t>(a.T) - t_first;
    LTK_CUDA(cudaMemsetAsync(h->cnt + t_first, 0, n * sizeof(int), st));
    LTK_CUDA(cudaMemsetAsync(h->ghist + t_first * c.n_bins, 0, n * c.n_bins * sizeof(int), st));
  }
  h->last_nseg = 0;
  if (is_retrieval(&c)) {
    // each corpus range appends to its own segment of the query's list
    int n_split = 1, per = 1;
    retrieval_split(a.T, a.S, h->num_sms, &n_split, &per);
    fp.seg_cnt = h->seg_cnt;
    fp.nseg = n_split;
    fp.seg_cap = h->cap / n_split;
    h->last_nseg = n_split;
    LTK_CUDA(cudaMemsetAsync(h->cnt, 0, static_cast<size_t>(a.T) * sizeof(int), st));
    LTK_CUDA(cudaMemsetAsync(h->ghist, 0, static_cast<size_t>(a.T) * c.n_bins * sizeof(int), st));
  }
  LTK_CUDA(launch_scorer(h, kModeFilter, q_map, k_map, fp, st));
  if (h->ev) LTK_CUDA(cudaEventRecord(h->ev[2], st));

  // ---- Select (Methodology step 3)
  SelectParams sel{h->cand, h->cnt, c.causal ? a.positions : nullptr, a.T, a.S, c.causal, h->cap,
                   a.k, a.out_idx, a.out_score, h->ovf, h->ovf + 2, h->pairs,
                   fp.seg_cnt, fp.nseg, fp.seg_cap};
  LTK_CUDA(launch_select(sel, h->num_sms, st));
  if (h->ev) LTK_CUDA(cudaEventRecord(h->ev[3], st));

  // ---- exact rescue of overflowed candidate lists (no-op when none)
  RescueParams rp{};
  rp.q = a.q;
  rp.q_scale = a.q_scale;
  rp.w = a.w;
  rp.k_cache = a.k_cache;
  rp.k_scale = a.k_scale;
  rp.positions = c.causal ? a.positions : nullptr;
  rp.T = a.T;
  rp.S = a.S;
  rp.causal = c.causal;
  rp.relu = c.relu;
  rp.heads = c.heads;
  rp.dim = c.dim;
  rp.fp8 = fp8 ? 1 : 0;
  rp.k = a.k;
  rp.ovf_count = h->ovf;
  rp.ovf_list = h->ovf + 2;
  rp.ovf_next = h->ovf + 1;
  rp.scratch = h->rescue_scratch;
  rp.scratch_ld = c.max_S;
  rp.out_idx = a.out_idx;
  rp.out_score = a.out_score;
  LTK_CUDA(launch_rescue(rp, h->rescue_rows, st));
  if (h->ev) LTK_CUDA(cudaEventRecord(h->ev[4], st));
  return LTK_OK;
}

}  // namespace

extern "C" {

int ltk_abi_version(void) { return LTK_ABI_VERSION; }

const char* ltk_status_string(int s) {
  switch (s) {
    case LTK_OK: return "ok";
    case LTK_ERR_ARG: return "invalid argument";
    case LTK_ERR_CUDA: return "CUDA error";
    case LTK_ERR_NOMEM: return "out of device memory";
    case LTK_ERR_OVERFLOW: return "candidate list overflow (resolved)";
    case LTK_ERR_TIMEOUT: return "device wait timed out";
    case LTK_ERR_UNSUPPORTED: return "unsupported configuration";
    default: return "unknown status";
  }
}

ltk_status ltk_config_init(ltk_config* cfg, int heads, int dim, int k, int max_T, long long max_S) {
  if (cfg == nullptr) return LTK_ERR_ARG;
  std::memset(cfg, 0, sizeof(*cfg));
  cfg->heads = heads;
  cfg->dim = dim;
  cfg->dtype = LTK_BF16;
  cfg->relu = 1;
  cfg->causal = 1;
  cfg->max_T = max_T;
  cfg->max_S = max_S;
  cfg->k = k;
  cfg->n_bins = 512;
  cfg->cand_cap = 0;
  cfg->sample_size = 0;
  cfg->seed = 20260715ull;
  cfg->refresh_interval = 1;
  cfg->enable_decoupled = 0;
  cfg->rescue_rows = 16;
  cfg->enable_host_io = 0;
  if (heads == 1) {   // vector retrieval: plain inner product over the whole corpus
    cfg->relu = 0;
    cfg->causal = 0;
    cfg->n_bins = kRetrievalMaxBins;
  }
  return LTK_OK;
}

ltk_status ltk_workspace_bytes(const ltk_config* cfg, unsigned long long* bytes) {
  if (bytes == nullptr) return LTK_ERR_ARG;
  const ltk_status s = validate_config(cfg);
  if (s != LTK_OK) return s;
  *bytes = compute_sizes(cfg).total;
  return LTK_OK;
}

ltk_status ltk_create(const ltk_config* cfg, ltk_handle** out) {
  if (out == nullptr) return LTK_ERR_ARG;
  *out = nullptr;
  ltk_status s = validate_config(cfg);
  if (s != LTK_OK) return s;
  ltk_handle* h = new (std::nothrow) ltk_handle();
  if (h == nullptr) return LTK_ERR_NOMEM;
  h->cfg = *cfg;
  const Sizes z = compute_sizes(cfg);
  h->cap = z.cap;
  h->n_pad_max = z.n_pad_max;
  h->rescue_rows = z.rescue_rows;
  h->elem = z.elem;
  cudaError_t e = cudaGetDevice(&h->device);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&h->num_sms, cudaDevAttrMultiProcessorCount, h->device);
  const unsigned long long T = static_cast<unsigned long long>(cfg->max_T > 0 ? cfg->max_T : 1);
  const unsigned long long S = static_cast<unsigned long long>(cfg->max_S);
  const unsigned long long np = static_cast<unsigned long long>(h->n_pad_max);
  auto step = [&](cudaError_t r) {
    if (e == cudaSuccess) e = r;
  };
  step(alloc(&h->samp_scores, T * np * 4));
  step(alloc(reinterpret_cast<char**>(&h->k_samp), np * cfg->dim * h->elem));
  step(alloc(&h->k_scale_samp, np * 4));
  step(alloc(&h->key_ids_pad, np * 4));
  step(alloc(&h->id_bitmap, (S + 31) / 32 * 4));
  step(alloc(&h->id_block_sums, static_cast<unsigned long long>(prepare_sample_blocks(cfg->max_S) + 1) * 4));
  step(alloc(&h->sample_tmp, kMaxSample * 4ull));
  step(alloc(&h->s_min, T * 4));
  step(alloc(&h->delta, T * 4));
  step(alloc(&h->theta0, T * 4));
  step(alloc(&h->ghist, T * static_cast<unsigned long long>(cfg->n_bins) * 4));
  if (is_retrieval(cfg)) step(alloc(&h->seg_cnt, T * static_cast<unsigned long long>(h->num_sms) * 4));
  step(alloc(&h->cand, T * static_cast<unsigned long long>(h->cap) * 8));
  step(alloc(&h->cnt, T * 4));
  step(alloc(&h->ovf, (T + 2) * 4));
  step(alloc(&h->rescue_scratch, static_cast<unsigned long long>(h->rescue_rows) * S * 4));
  step(alloc(&h->status, 4));
  step(alloc(&h->ms.counts, S * 4));
  step(alloc(&h->ms.keys, S * 8));
  step(alloc(&h->ms.hist, 256 * 4));
  step(alloc(&h->ms.state, 4 * 8));
  if (cfg->enable_decoupled) step(alloc(&h->dense, T * S * 4));
  if (cfg->enable_host_io) {
    step(alloc(reinterpret_cast<char**>(&h->io_q), T * cfg->heads * cfg->dim * h->elem));
    step(alloc(&h->io_qs, T * 4));
    step(alloc(&h->io_w, T * cfg->heads * 4));
    step(alloc(reinterpret_cast<char**>(&h->io_k), S * cfg->dim * h->elem));
    step(alloc(&h->io_ks, S * 4));
    step(alloc(&h->io_pos, T * 4));
    step(alloc(&h->io_prev, kMaxSample * 4ull));
    step(alloc(&h->io_oidx, T * cfg->k * 4ull));
    step(alloc(&h->io_oscore, T * cfg->k * 4ull));
  }
  step(alloc(&h->pairs, 16));
  for (auto& row : h->ring)
    for (auto& ev : row) step(cudaEventCreate(&ev));
  if (e == cudaSuccess) e = cudaMemset(h->status, 0, 4);
  if (e == cudaSuccess) e = cudaMemset(h->ovf, 0, 8);
  if (e == cudaSuccess) e = cudaMemset(h->cnt, 0, T * 4);
  if (e == cudaSuccess) e = cudaMemset(h->id_bitmap, 0, (S + 31) / 32 * 4);
  if (e != cudaSuccess) {
    free_all(h);
    delete h;
    return cuda_fail(e, "ltk_create");
  }
  *out = h;
  return LTK_OK;
}

void ltk_destroy(ltk_handle* h) {
  if (h == nullptr) return;
  cudaDeviceSynchronize();
  free_all(h);
  delete h;
}

ltk_status ltk_set_timing(ltk_handle* h, int enable) {
  if (h == nullptr) return LTK_ERR_ARG;
  h->timing = enable ? 1 : 0;
  h->ring_calls = 0;
  return LTK_OK;
}

ltk_status ltk_random_sample(ltk_handle* h, long long S, int n, int* sample_out, void* stream) {
  if (h == nullptr || sample_out == nullptr || S < 1 || S > h->cfg.max_S || n < 1 ||
      n > kMaxSample || n > S)
    return LTK_ERR_ARG;
  if (!current_device_is(h->device)) return LTK_ERR_ARG;
  LTK_CUDA(launch_random_sample(S, n, h->cfg.seed, sample_out, static_cast<cudaStream_t>(stream)));
  return LTK_OK;
}

ltk_status ltk_make_sample(ltk_handle* h, const int* prev_idx, int T_prev, int k_prev, long long S,
                           int n, int* sample_out, void* stream) {
  if (h == nullptr || sample_out == nullptr || T_prev < 0 || k_prev < 0 || S < 1 ||
      S > h->cfg.max_S || n < 1 || n > kMaxSample || n > S)
    return LTK_ERR_ARG;
  const long long n_prev = static_cast<long long>(T_prev) * k_prev;
  if (n_prev > 0 && prev_idx == nullptr) return LTK_ERR_ARG;
  if (!current_device_is(h->device)) return LTK_ERR_ARG;
  LTK_CUDA(launch_make_sample(prev_idx, n_prev, S, n, h->cfg.seed, h->ms, sample_out,
                              static_cast<cudaStream_t>(stream)));
  return LTK_OK;
}

ltk_status ltk_indexer_topk(ltk_handle* h, const void* q, const float* q_scale, const float* w,
                            const void* k_cache, const float* k_scale, const int* positions, int T,
                            long long S, const int* prev_topk, int n_prev, int k, int* out_idx,
                            float* out_score, void* stream) {
  const CallArgs a{q, q_scale, w, k_cache, k_scale, positions, T, S, k, out_idx, out_score};
  ltk_status s = validate_call(h, a);
  if (s != LTK_OK) return s;
  if (prev_topk != nullptr && (n_prev < 1 || n_prev > kMaxSample)) return LTK_ERR_ARG;
  if (prev_topk == nullptr && n_prev != 0) return LTK_ERR_ARG;
  return run_fused(h, a, prev_topk, n_prev, static_cast<cudaStream_t>(stream));
}

ltk_status ltk_indexer_topk_host(ltk_handle* h, const void* q, const float* q_scale, const float* w,
                                 const void* k_cache, const float* k_scale, const int* positions,
                                 int T, long long S, const int* prev_topk, int n_prev, int k,
                                 int* out_idx, float* out_score, void* stream) {
  if (h == nullptr || !h->cfg.enable_host_io) return LTK_ERR_ARG;
  const ltk_config& c = h->cfg;
  if (T < 0 || T > c.max_T || S < 1 || S > c.max_S || k < 1 || k > c.k) return LTK_ERR_ARG;
  if (T == 0) return LTK_OK;
  if (!q || !w || !k_cache || !out_idx || !out_score) return LTK_ERR_ARG;
  if (c.causal && !positions) return LTK_ERR_ARG;
  const bool fp8 = c.dtype == LTK_FP8_E4M3;
  if (fp8 && (!q_scale || !k_scale)) return LTK_ERR_ARG;
  if (prev_topk != nullptr && (n_prev < 1 || n_prev > kMaxSample)) return LTK_ERR_ARG;
  if (prev_topk == nullptr && n_prev != 0) return LTK_ERR_ARG;
  if (!current_device_is(h->device)) return LTK_ERR_ARG;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const size_t qb = static_cast<size_t>(T) * c.heads * c.dim * h->elem;
  const size_t kb = static_cast<size_t>(S) * c.dim * h->elem;
  LTK_CUDA(cudaMemcpyAsync(h->io_q, q, qb, cudaMemcpyHostToDevice, st));
  LTK_CUDA(cudaMemcpyAsync(h->io_w, w, static_cast<size_t>(T) * c.heads * 4, cudaMemcpyHostToDevice, st));
  LTK_CUDA(cudaMemcpyAsync(h->io_k, k_cache, kb, cudaMemcpyHostToDevice, st));
  if (c.causal)
    LTK_CUDA(cudaMemcpyAsync(h->io_pos, positions, static_cast<size_t>(T) * 4, cudaMemcpyHostToDevice, st));
  if (fp8) {
    LTK_CUDA(cudaMemcpyAsync(h->io_qs, q_scale, static_cast<size_t>(T) * 4, cudaMemcpyHostToDevice, st));
    LTK_CUDA(cudaMemcpyAsync(h->io_ks, k_scale, static_cast<size_t>(S) * 4, cudaMemcpyHostToDevice, st));
  }
  if (prev_topk)
    LTK_CUDA(cudaMemcpyAsync(h->io_prev, prev_topk, static_cast<size_t>(n_prev) * 4, cudaMemcpyHostToDevice, st));
  const CallArgs a{h->io_q, fp8 ? h->io_qs : nullptr, h->io_w, h->io_k, fp8 ? h->io_ks : nullptr,
                   c.causal ? h->io_pos : nullptr, T, S, k, h->io_oidx, h->io_oscore};
  ltk_status s = run_fused(h, a, prev_topk ? h->io_prev : nullptr, n_prev, st);
  if (s != LTK_OK) return s;
  LTK_CUDA(cudaMemcpyAsync(out_idx, h->io_oidx, static_cast<size_t>(T) * k * 4, cudaMemcpyDeviceToHost, st));
  LTK_CUDA(cudaMemcpyAsync(out_score, h->io_oscore, static_cast<size_t>(T) * k * 4, cudaMemcpyDeviceToHost, st));
  LTK_CUDA(cudaStreamSynchronize(st));
  return LTK_OK;
}

ltk_status ltk_decoupled_topk(ltk_handle* h, const void* q, const float* q_scale, const float* w,
                              const void* k_cache, const float* k_scale, const int* positions, int T,
                              long long S, int k, int* out_idx, float* out_score, void* stream) {
  const CallArgs a{q, q_scale, w, k_cache, k_scale, positions, T, S, k, out_idx, out_score};
  ltk_status s = validate_call(h, a);
  if (s != LTK_OK) return s;
  if (!h->cfg.enable_decoupled) return LTK_ERR_ARG;
  const ltk_config& c = h->cfg;
  const bool fp8 = c.dtype == LTK_FP8_E4M3;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  h->last_kind = 2;
  h->last_T = T;
  h->last_S = S;
  h->last_k = k;
  h->last_stream = st;
  if (T == 0) return LTK_OK;
  h->ev = begin_timed_call(h);
  if (h->ev) LTK_CUDA(cudaEventRecord(h->ev[0], st));
  LTK_CUDA(cudaMemsetAsync(h->status, 0, sizeof(int), st));
  LTK_CUDA(cudaMemsetAsync(h->pairs, 0, sizeof(unsigned long long), st));
  LTK_CUDA(cudaMemsetAsync(h->ovf, 0, 2 * sizeof(int), st));
  CUtensorMap q_map, k_map;
  std::memset(&q_map, 0, sizeof(q_map));
  std::memset(&k_map, 0, sizeof(k_map));
  if (!use_cc(&c) &&
      (!make_tmap(&q_map, q, fp8, c.dim, q_rows(c, T), 256) ||
       !make_tmap(&k_map, k_cache, fp8, c.dim, static_cast<unsigned long long>(S), kTile)))
    return LTK_ERR_CUDA;
  ScoreParams sp{};
  sp.q_raw = q;
  sp.k_raw = k_cache;
  sp.w = w;
  sp.q_scale = q_scale;
  sp.k_scale = k_scale;
  sp.positions = c.causal ? positions : nullptr;
  sp.key_ids = nullptr;
  sp.T = T;
  sp.rows = S;
  sp.causal = c.causal;
  sp.dense = h->dense;
  sp.ld = S;
  sp.status = h->status;
  int qpu_d = kTcQPB;
  plan_work(h, T, S, true, &sp.b_full, &sp.s_last, &qpu_d);
  if (h->ev) LTK_CUDA(cudaEventRecord(h->ev[1], st));
  LTK_CUDA(launch_scorer(h, kModeDense, q_map, k_map, sp, st));
  if (h->ev) LTK_CUDA(cudaEventRecord(h->ev[2], st));
  RowTopkParams rp{h->dense, S, c.causal ? positions : nullptr, T, S, c.causal, k, out_idx, out_score,
                   h->pairs};
  LTK_CUDA(launch_row_topk(rp, st));
  if (h->ev) {
    LTK_CUDA(cudaEventRecord(h->ev[3], st));
    LTK_CUDA(cudaEventRecord(h->ev[4], st));
  }
  return LTK_OK;
}

ltk_status ltk_litedsa_pack(const int* topk_idx, int T, int k, int group, int* union_idx,
                            int* union_len, unsigned int* masks, void* stream) {
  if (T < 0 || k < 1 || group < 1 || group > 256) return LTK_ERR_ARG;
  if (static_cast<long long>(group) * k > litedsa_max_entries()) return LTK_ERR_UNSUPPORTED;
  if (litedsa_smem_bytes(group, k) > kLitedsaMaxSmem) return LTK_ERR_UNSUPPORTED;
  if (T == 0) return LTK_OK;
  if (!topk_idx || !union_idx || !union_len || !masks) return LTK_ERR_ARG;
  LTK_CUDA(launch_litedsa_pack(topk_idx, T, k, group, union_idx, union_len, masks,
                               static_cast<cudaStream_t>(stream)));
  return LTK_OK;
}

ltk_status ltk_get_stats(ltk_handle* h, ltk_stats* out) {
  if (h == nullptr || out == nullptr) return LTK_ERR_ARG;
  std::memset(out, 0, sizeof(*out));
  out->T = h->last_T;
  out->S = h->last_S;
  out->k = h->last_k;
  out->ms_sample = out->ms_filter = out->ms_select = out->ms_rescue = out->ms_total = -1.f;
  if (h->last_kind == 0) return LTK_OK;
  LTK_CUDA(cudaStreamSynchronize(h->last_stream));
  int status = 0;
  LTK_CUDA(cudaMemcpy(&status, h->status, 4, cudaMemcpyDeviceToHost));
  out->device_status = status;
  if (h->last_kind == 1 && h->last_T > 0) {
    int* cnt = static_cast<int*>(std::malloc(static_cast<size_t>(h->last_T) * 4));
    if (cnt == nullptr) return LTK_ERR_NOMEM;
    cudaError_t e = cudaMemcpy(cnt, h->cnt, static_cast<size_t>(h->last_T) * 4, cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) {
      std::free(cnt);
      return cuda_fail(e, "stats");
    }
    if (h->last_nseg > 0) {
      // segmented lists: a query's count is the sum of its segments' counts
      const size_t ns = static_cast<size_t>(h->last_T) * h->last_nseg;
      int* seg = static_cast<int*>(std::malloc(ns * 4));
      if (seg == nullptr) {
        std::free(cnt);
        return LTK_ERR_NOMEM;
      }
      e = cudaMemcpy(seg, h->seg_cnt, ns * 4, cudaMemcpyDeviceToHost);
      if (e != cudaSuccess) {
        std::free(seg);
        std::free(cnt);
        return cuda_fail(e, "stats");
      }
      for (int i = 0; i < h->last_T; ++i) {
        long long c = 0;
        for (int j = 0; j < h->last_nseg; ++j) c += seg[static_cast<size_t>(i) * h->last_nseg + j];
        if (cnt[i] <= h->cap) cnt[i] = static_cast<int>(c);
      }
      std::free(seg);
    }
    long long sum = 0;
    int mx = 0;
    for (int i = 0; i < h->last_T; ++i) {
      sum += cnt[i];
      if (cnt[i] > mx) mx = cnt[i];
    }
    std::free(cnt);
    out->cand_written = sum;
    out->cand_max = mx;
    int ovf = 0;
    LTK_CUDA(cudaMemcpy(&ovf, h->ovf, 4, cudaMemcpyDeviceToHost));
    out->n_overflow = ovf;
  }
  if (h->last_T > 0) {
    unsigned long long pairs = 0;
    LTK_CUDA(cudaMemcpy(&pairs, h->pairs, 8, cudaMemcpyDeviceToHost));
    out->visible_pairs = static_cast<long long>(pairs);
  }
  out->launches = launches_so_far();
  const int n = h->ring_calls < ltk_handle::kRing ? h->ring_calls : ltk_handle::kRing;
  if (n > 0) {
    double acc[5] = {0, 0, 0, 0, 0};
    const int pairs_of[5][2] = {{0, 1}, {1, 2}, {2, 3}, {3, 4}, {0, 4}};
    for (int i = 0; i < n; ++i) {
      for (int j = 0; j < 5; ++j) {
        float ms = 0.f;
        LTK_CUDA(cudaEventElapsedTime(&ms, h->ring[i][pairs_of[j][0]], h->ring[i][pairs_of[j][1]]));
        acc[j] += ms;
      }
    }
    out->ms_sample = static_cast<float>(acc[0] / n);
    out->ms_filter = static_cast<float>(acc[1] / n);
    out->ms_select = static_cast<float>(acc[2] / n);
    out->ms_rescue = static_cast<float>(acc[3] / n);
    out->ms_total = static_cast<float>(acc[4] / n);
    out->timed_calls = n;
  }
  return LTK_OK;
}

}  // extern "C"

// ---------------------------------------------------------------------------
// Decoupled top-k without any allocation
// ---------------------------------------------------------------------------
// Some callers cannot call cudaMalloc: a plugin running inside an engine that
// owns all device memory through its own pool and rejects allocations made
// behind its back, or a latency-critical path where cudaMalloc's implicit
// device synchronisation would stall the caller's other streams.  This entry
// point serves them: it needs no handle, and its only scratch -- the fp32
// score matrix of the decoupled baseline -- lives in the file-scope device
// array below.  Every GPU that loads this library holds that array until the
// process exits.
namespace {

constexpr long long kNoAllocMaxScores = 4ll << 20;   // T * S <= 4,194,304 (16 MiB of fp32)
static __device__ __align__(256) float g_noalloc_scores[kNoAllocMaxScores];

// Host code must not use g_noalloc_scores directly: on the host it is only a
// stand-in for the device symbol.  Its device address is looked up on every
// call, with the caller's device current, so it stays right after a device
// reset reloads the module.
ltk_status noalloc_scores_for_current_device(float** out) {
  *out = nullptr;
  void* p = nullptr;
  const cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scores);
  if (e != cudaSuccess || p == nullptr)
    return cuda_fail(e == cudaSuccess ? cudaErrorInvalidSymbol : e, "cudaGetSymbolAddress");
  *out = static_cast<float*>(p);
  return LTK_OK;
}

}  // namespace

extern "C" ltk_status ltk_decoupled_topk_noalloc(int dtype, int causal, const void* q,
                                                 const float* q_scale, const float* w,
                                                 const void* k_cache, const float* k_scale,
                                                 const int* positions, int T, long long S, int k,
                                                 int* out_idx, float* out_score, int* device_status,
                                                 void* stream) {
  if (dtype != LTK_BF16 && dtype != LTK_FP8_E4M3) return LTK_ERR_ARG;
  if (T < 0 || S < 1 || S > 0x7FFFFFFFll || k < 1 || k > kMaxK) return LTK_ERR_ARG;
  if (static_cast<long long>(T) * S > kNoAllocMaxScores) return LTK_ERR_ARG;
  if (T == 0) return LTK_OK;
  if (!q || !w || !k_cache || !out_idx || !out_score) return LTK_ERR_ARG;
  if (!aligned16(q) || !aligned16(w) || !aligned16(k_cache) || !aligned16(out_idx) ||
      !aligned16(out_score))
    return LTK_ERR_ARG;
  if (device_status != nullptr && (reinterpret_cast<uintptr_t>(device_status) & 3u) != 0)
    return LTK_ERR_ARG;
  if (causal && (positions == nullptr || !aligned16(positions))) return LTK_ERR_ARG;
  const bool fp8 = dtype == LTK_FP8_E4M3;
  if (fp8 && (!q_scale || !k_scale || !aligned16(q_scale) || !aligned16(k_scale))) return LTK_ERR_ARG;
  float* scores = nullptr;
  const ltk_status st0 = noalloc_scores_for_current_device(&scores);
  if (st0 != LTK_OK) return st0;
  int dev = 0, num_sms = 0;
  LTK_CUDA(cudaGetDevice(&dev));
  LTK_CUDA(cudaDeviceGetAttribute(&num_sms, cudaDevAttrMultiProcessorCount, dev));
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  CUtensorMap q_map, k_map;
  if (!make_tmap(&q_map, q, fp8, kTcDim, static_cast<unsigned long long>(T) * kTcHeads, 256) ||
      !make_tmap(&k_map, k_cache, fp8, kTcDim, static_cast<unsigned long long>(S), kTile))
    return LTK_ERR_CUDA;
  // the caller's status word starts at zero; a bounded wait that expires in
  // the scorer records LTK_ERR_TIMEOUT there
  if (device_status != nullptr) LTK_CUDA(cudaMemsetAsync(device_status, 0, sizeof(int), st));
  ScoreParams sp{};
  sp.w = w;
  sp.q_scale = q_scale;
  sp.k_scale = k_scale;
  sp.positions = causal ? positions : nullptr;
  sp.key_ids = nullptr;
  sp.T = T;
  sp.rows = S;
  sp.causal = causal ? 1 : 0;
  sp.dense = scores;
  sp.ld = S;
  sp.status = device_status;
  // the same (query block, key range) work split as the handle's dense scorer
  plan_split(T, S, num_sms, 2, &sp.b_full, &sp.s_last);
  LTK_CUDA(launch_score_tc(kModeDense, fp8, q_map, k_map, sp, st));
  RowTopkParams rp{scores, S, causal ? positions : nullptr, T, S, causal ? 1 : 0, k, out_idx,
                   out_score, nullptr};
  LTK_CUDA(launch_row_topk(rp, st));
  return LTK_OK;
}
