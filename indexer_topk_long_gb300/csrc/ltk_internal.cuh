// ltk_internal.cuh -- internal declarations and device helpers of libltk.
//
// Hand-written PTX wrappers for sm_103a (mbarrier, TMA, tcgen05/TMEM), the bin
// map of the Filter stage, order-preserving composite keys used by every
// selection, and the launch functions each kernel file exports to the host
// orchestration in ltk_api.cu.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/ltk.h"

namespace ltk {

// ---------------------------------------------------------------------------
// Limits and fixed shapes
// ---------------------------------------------------------------------------
constexpr int kMaxK = 8192;             // largest k a handle may request
constexpr int kMaxSample = 16384;       // largest sample (k') a call may use
constexpr int kTile = 128;              // keys per tensor-core tile (MMA M)
constexpr int kTcHeads = 64;            // H of the tensor-core indexer path
constexpr int kTcDim = 128;             // d of the tensor-core indexer path
constexpr int kTcQPB = 8;               // queries per CTA of the scorer
constexpr int kSelBins = 2048;          // bins of the Select stage's re-binning
constexpr int kRetrievalMaxBins = 64;   // gate bins of the retrieval scorer (shared-memory bound)
constexpr int kRetrievalMaxDim = 1024;
constexpr unsigned long long kWaitLimitNs = 2000000000ull;   // 2 s per wait

// Device status word values (same numbering as ltk_status).
constexpr int kDevOk = 0;
constexpr int kDevTimeout = 5;

// ---------------------------------------------------------------------------
// Small device helpers
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint64_t globaltimer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// Record the first device error (later ones are dropped).
__device__ __forceinline__ void raise_status(int* status, int code) {
  if (status) atomicCAS(status, 0, code);
}

// Gate bin of a score (LiteTopK Methodology step 2, "Bin Mapping": the
// affine map B = (I - s_min) * delta, delta = bins per unit score).
// Rounded to nearest in fp32 and floored, then clamped to [0, nb-1]; NaN maps
// to 0.  The map is monotone non-decreasing in I, and this one function is
// used by the Sample, Filter and Select stages alike.
__device__ __forceinline__ int bin_of(float I, float s_min, float delta, int nb) {
  const float f = __fmul_rn(__fsub_rn(I, s_min), delta);
  // fmaxf returns 0 for a NaN f; truncation of the clamped value is the floor
  return __float2int_rz(fminf(fmaxf(f, 0.f), static_cast<float>(nb - 1)));
}

// Order-preserving map fp32 -> uint32 (larger float -> larger integer).
__device__ __forceinline__ uint32_t ord_f32(float f) {
  if (f == 0.f) f = 0.f;   // -0 and +0 compare equal; give them one code
  const uint32_t b = __float_as_uint(f);
  return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}
__device__ __forceinline__ float unord_f32(uint32_t o) {
  const uint32_t b = (o & 0x80000000u) ? (o & 0x7FFFFFFFu) : ~o;
  return __uint_as_float(b);
}

// Composite key of the exact order: larger key = higher score, then lower
// index.  Keys of distinct indices are distinct.
__device__ __forceinline__ uint64_t ckey(float score, int idx) {
  return (static_cast<uint64_t>(ord_f32(score)) << 32) |
         static_cast<uint64_t>(0xFFFFFFFFu - static_cast<uint32_t>(idx));
}
__device__ __forceinline__ int ckey_idx(uint64_t key) {
  return static_cast<int>(0xFFFFFFFFu - static_cast<uint32_t>(key & 0xFFFFFFFFull));
}
__device__ __forceinline__ float ckey_score(uint64_t key) {
  return unord_f32(static_cast<uint32_t>(key >> 32));
}

// Candidate record written by the Filter stage: raw fp32 score and key index.
__device__ __forceinline__ uint64_t cand_pack(float score, int idx) {
  return (static_cast<uint64_t>(__float_as_uint(score)) << 32) | static_cast<uint32_t>(idx);
}
__device__ __forceinline__ float cand_score(uint64_t c) {
  return __uint_as_float(static_cast<uint32_t>(c >> 32));
}
__device__ __forceinline__ int cand_idx(uint64_t c) {
  return static_cast<int>(static_cast<uint32_t>(c & 0xFFFFFFFFull));
}

// ---------------------------------------------------------------------------
// mbarrier (shared::cta)
// ---------------------------------------------------------------------------
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_fence_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred P;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 P, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, P;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// try_wait with a suspend-time hint: the thread sleeps until the phase
// completes or the hint (ns) expires.  Used only after a short spin, for
// waits that are already long.
constexpr uint32_t kSuspendHintNs = 200000;
__device__ __forceinline__ bool mbar_try_wait_sleep(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred P;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 P, [%1], %2, %3;\n\t"
      "selp.u32 %0, 1, 0, P;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity), "r"(kSuspendHintNs)
      : "memory");
  return ok != 0;
}

// Bounded wait for the completion of phase `parity`.  Returns false when the
// CTA's abort flag is set by another role or when the wait exceeds
// kWaitLimitNs (then it sets the abort flag and the device status itself).
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                          int* status) {
  for (int i = 0; i < 32; ++i)
    if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  while (true) {
    if (mbar_try_wait_sleep(bar, parity)) return true;
    if (abort_flag != nullptr && *abort_flag) return false;
    if (globaltimer_ns() - t0 > kWaitLimitNs) {
      if (abort_flag != nullptr) *abort_flag = 1;
      raise_status(status, kDevTimeout);
      return false;
    }
  }
}

// Bounded wait that ignores the abort flag (used to drain in-flight copies).
__device__ __forceinline__ bool mbar_drain(uint32_t bar, uint32_t parity) {
  const uint64_t t0 = globaltimer_ns();
  while (!mbar_try_wait(bar, parity))
    if (globaltimer_ns() - t0 > kWaitLimitNs) return false;
  return true;
}

// ---------------------------------------------------------------------------
// TMA (cp.async.bulk.tensor), tiled 2-D loads completing on an mbarrier
// ---------------------------------------------------------------------------
__device__ __forceinline__ void tma_prefetch_desc(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, int x, int y,
                                            uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar)
      : "memory");
}

// ---------------------------------------------------------------------------
// tcgen05 / TMEM
// ---------------------------------------------------------------------------
__device__ __forceinline__ void tmem_alloc(uint32_t dst_slot, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_slot),
               "r"(ncols)
               : "memory");
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// D[tmem] (+)= A[smem desc] * B[smem desc]^T, one instruction, issued by one
// thread.  kind::f16 covers bf16 operands; kind::f8f6f4 covers e4m3.
template <bool FP8>
__device__ __forceinline__ void tc_mma(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                       uint32_t idesc, uint32_t accumulate) {
  if constexpr (FP8) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
  } else {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
  }
}

// Arrive on an mbarrier once every tcgen05 operation this thread issued so far
// has completed.
__device__ __forceinline__ void tc_commit(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                   bar)
               : "memory");
}

// 16 consecutive fp32 columns of this thread's TMEM lane (shape 32x32b, 16
// repetitions).  Undefined until tmem_wait_ld_tied on the same array.
__device__ __forceinline__ void tmem_ld32x16(uint32_t taddr, float (&v)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,"
      "%15}, [%16];"
      : "=f"(v[0]), "=f"(v[1]), "=f"(v[2]), "=f"(v[3]), "=f"(v[4]), "=f"(v[5]), "=f"(v[6]),
        "=f"(v[7]), "=f"(v[8]), "=f"(v[9]), "=f"(v[10]), "=f"(v[11]), "=f"(v[12]), "=f"(v[13]),
        "=f"(v[14]), "=f"(v[15])
      : "r"(taddr));
}

// tcgen05.wait::ld that also names the loaded registers as operands, so the
// compiler cannot move a use of them above the wait.
__device__ __forceinline__ void tmem_wait_ld_tied(float (&v)[16]) {
  asm volatile("tcgen05.wait::ld.sync.aligned;"
               : "+f"(v[0]), "+f"(v[1]), "+f"(v[2]), "+f"(v[3]), "+f"(v[4]), "+f"(v[5]),
                 "+f"(v[6]), "+f"(v[7]), "+f"(v[8]), "+f"(v[9]), "+f"(v[10]), "+f"(v[11]),
                 "+f"(v[12]), "+f"(v[13]), "+f"(v[14]), "+f"(v[15])
               :
               : "memory");
}

// Shared-memory matrix descriptor of a K-major operand stored in the
// 128-byte-swizzled layout that a TMA load with CU_TENSOR_MAP_SWIZZLE_128B
// produces: rows of 128 bytes, 8-row atoms of 1024 bytes (stride-dimension
// byte offset 1024), atom base 1024-byte aligned.  Fields (PTX ISA, tcgen05
// shared memory descriptor): start address >> 4 in bits 0-13, leading-dim
// byte offset >> 4 in 16-29 (unused for swizzled K-major), stride-dim byte
// offset >> 4 in 32-45, fixed 0b001 in 46-48, base offset 0, swizzle mode in
// 61-63 (2 = 128-byte swizzle).
__device__ __forceinline__ uint64_t smem_desc_sw128(uint32_t saddr) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);
  d |= static_cast<uint64_t>(1) << 16;
  d |= static_cast<uint64_t>(1024 >> 4) << 32;
  d |= static_cast<uint64_t>(1) << 46;
  d |= static_cast<uint64_t>(2) << 61;
  return d;
}

// Instruction descriptor (PTX ISA, tcgen05 instruction descriptor for
// kind::f16 / kind::f8f6f4): D format f32 (bits 4-5 = 1), A/B format in bits
// 7-9 / 10-12 (bf16 = 1 under kind::f16, e4m3 = 0 under kind::f8f6f4), both
// operands K-major (bits 15, 16 = 0), N >> 3 in bits 17-22, M >> 4 in 24-28.
__host__ __device__ constexpr uint32_t make_idesc(bool fp8, int M, int N) {
  return (1u << 4) | ((fp8 ? 0u : 1u) << 7) | ((fp8 ? 0u : 1u) << 10) |
         (static_cast<uint32_t>(N >> 3) << 17) | (static_cast<uint32_t>(M >> 4) << 24);
}

// ---------------------------------------------------------------------------
// Kernel parameter blocks and launch functions (defined in the kernel files)
// ---------------------------------------------------------------------------
// Raise a kernel's dynamic shared-memory limit to `bytes` on the current
// device (the attribute is per device; set once per device and kernel).
// `slot` identifies the kernel (a small distinct integer per call site).
cudaError_t ensure_smem_limit(const void* func, int slot, size_t bytes);
enum SmemSlot {
  kSlotScoreTc = 0,          // 8 instantiations: + mode * 4 + fp8 * 2 + alternating form
  kSlotRetrieval = 8,        // 4 instantiations: + mode * 2 + relu
  kSlotScoreCc = 12,         // 4 instantiations: + mode * 2 + fp8
  kSlotStats = 16,
  kSlotStatsWide = 17,
  kSlotSelect = 18,
  kSlotSelectWide = 19,
  kSlotRowTopk = 20,
  kSlotRescue = 21,
  kSlotSelectSeg = 22,
  kSlotSelectSegWide = 23,
  kSlotLitedsa = 24,         // 5 instantiations: keys per thread 1, 2, 4, 8, 16
  kSlotCount = 29
};

// Process-wide count of kernels launched by this library (ltk_api.cu).
void count_launches(int n);
long long launches_so_far();

enum ScoreMode { kModeDense = 0, kModeFilter = 1 };

struct ScoreParams {
  const float* w;          // [T, H]
  const float* q_scale;    // [T] (fp8) or null
  const float* k_scale;    // [rows] (fp8) or null
  const int* positions;    // [T] or null (no mask)
  const int* key_ids;      // [rows] key id of each row (gathered sample), or null
  int T;
  long long rows;          // rows of the key source
  int causal;
  // Filter stage
  const float* s_min;      // [T]
  const float* delta;      // [T]
  const int* theta0;       // [T]
  unsigned long long* cand;  // [T, cap]
  int* cnt;                // [T]
  int cap;
  int nb;
  int k;
  int refresh_interval;
  int skip_key_loads;      // failure-handling tests: the producer issues no key tiles
  // Work split (indexer scorer): CTAs [0, b_full) each own one query block and
  // all of its keys; the remaining query blocks are each split into s_last key
  // ranges scanned by s_last CTAs, which append with global atomics to cnt and
  // drain their histograms into ghist [T, nb] (both zeroed before the launch).
  int b_full;
  int s_last;
  int* ghist;
  // Filter sweep (indexer scorer, general form; null: every CTA scans its key
  // range from the first tile): key tiles scanned so far by all CTAs, zeroed
  // before the launch.  A CTA starts its range at tile (sweep / num_sms) mod
  // its block's tiles and wraps around, so CTAs that start in later waves
  // read the tiles the running ones are reading, while L2 still holds them.
  unsigned long long* sweep;
  int num_sms;
  // Segmented lists (retrieval scorer): query t's list holds nseg segments of
  // seg_cap entries, segment s written only by the CTA scanning range s with
  // a CTA-local count; seg_cnt [T, nseg] receives the counts, and cnt[t] is
  // set to cap + 1 when a segment overflowed.  Null: one list per query.
  int* seg_cnt;
  int nseg;
  int seg_cap;
  // raw operand pointers (the CUDA-core scorer reads q and keys directly)
  const void* q_raw;
  const void* k_raw;
  // Dense output
  float* dense;            // [T, ld]
  long long ld;
  int* status;
};

// Tensor-core scorer (k_score_tc.cu).  q_map/k_map are tiled TMA maps built by
// make_q_map/make_k_map.
cudaError_t launch_score_tc(int mode, bool fp8, const CUtensorMap& q_map, const CUtensorMap& k_map,
                            const ScoreParams& p, cudaStream_t stream);
size_t score_tc_smem_bytes(int mode, bool fp8, int nb);
int score_tc_max_bins(bool fp8);

// Retrieval scorer (k_retrieval_tc.cu): one head, d a multiple of 64 up to
// kRetrievalMaxDim, bf16, no causal mask.  The filter mode accumulates p.cnt
// with global atomics and the per-query histogram ghist [T, nb] (zero both
// first) shared by all CTAs that scan a query.
cudaError_t launch_retrieval_tc(int mode, const CUtensorMap& q_map, const CUtensorMap& c_map,
                                const ScoreParams& p, int dim, int relu, int* ghist,
                                int num_sms, cudaStream_t stream);
size_t retrieval_tc_smem_bytes(int mode, int nb);
// Corpus ranges per query block of the retrieval scorer (its CTAs per block)
// and tiles per range.
void retrieval_split(int T, long long rows, int num_sms, int* n_split, int* per);

struct SampleStatsParams {
  const float* scores;     // [T, ld] sample scores (-inf = invisible)
  long long ld;
  int n;                   // valid sample columns
  int T;
  int k;
  int nb;
  float* s_min;
  float* delta;
  int* theta0;
  // 1: delta is rounded down to a power of two (the CUDA-core scorer scales
  // its weights by delta, which is then exact, so its scores come back from
  // bin space without rounding); 0: delta as computed.
  int pow2_delta;
};

// Largest power of two <= x for a positive normal fp32 x (the exponent of x
// with the mantissa cleared).
__host__ __device__ __forceinline__ float pow2_floor(float x) {
#ifdef __CUDA_ARCH__
  return __uint_as_float(__float_as_uint(x) & 0xFF800000u);
#else
  uint32_t b;
  __builtin_memcpy(&b, &x, 4);
  b &= 0xFF800000u;
  float r;
  __builtin_memcpy(&r, &b, 4);
  return r;
#endif
}

// Sample stage (k_sample.cu).
cudaError_t launch_random_sample(long long S, int n, unsigned long long seed, int* out,
                                 cudaStream_t stream);
cudaError_t launch_prepare_sample(const int* ids, int n, long long S, int n_pad, int* key_ids_pad,
                                  uint32_t* bitmap, int* block_sums, cudaStream_t stream);
int prepare_sample_blocks(long long S);   // block_sums entries launch_prepare_sample needs
cudaError_t launch_gather_keys(const void* k_cache, const float* k_scale, int elem_bytes, int dim,
                               const int* key_ids_pad, int n_pad, void* k_samp, float* k_scale_samp,
                               cudaStream_t stream);
cudaError_t launch_sample_stats(const SampleStatsParams& p, int num_sms, cudaStream_t stream);

struct MakeSampleWs {
  int* counts;                  // [max_S]
  unsigned long long* keys;     // [max_S]
  unsigned int* hist;           // [256]
  unsigned long long* state;    // [4]: prefix, mask, remaining, slot
};
cudaError_t launch_make_sample(const int* prev_idx, long long n_prev, long long S, int n,
                               unsigned long long seed, const MakeSampleWs& ws, int* out,
                               cudaStream_t stream);

struct SelectParams {
  const unsigned long long* cand;  // [T, cap]
  const int* cnt;                  // [T] (segmented lists: 0, or cap + 1 on overflow)
  const int* positions;            // [T] or null
  int T;
  long long S;
  int causal;
  int cap;
  int k;
  int* out_idx;                    // [T, k]
  float* out_score;                // [T, k]
  int* ovf_count;
  int* ovf_list;                   // [T]
  unsigned long long* pairs;       // visible pairs of the call (accumulated)
  const int* seg_cnt;              // [T, nseg] segment counts, or null (one list per query)
  int nseg;
  int seg_cap;
};

struct RowTopkParams {
  const float* rows;               // [T, ld] scores (decoupled) or scratch rows
  long long ld;
  const int* positions;
  int T;
  long long S;
  int causal;
  int k;
  int* out_idx;
  float* out_score;
  unsigned long long* pairs;       // visible pairs of the call (accumulated)
};

struct RescueParams {
  const void* q;
  const float* q_scale;
  const float* w;
  const void* k_cache;
  const float* k_scale;
  const int* positions;
  int T;
  long long S;
  int causal;
  int relu;
  int heads;
  int dim;
  int fp8;
  int k;
  const int* ovf_count;
  const int* ovf_list;
  int* ovf_next;
  float* scratch;                  // [rescue_rows, S]
  long long scratch_ld;
  int* out_idx;
  float* out_score;
};

// CUDA-core scorer with the fused affine bin map (k_score_cc.cu): any H <= 128,
// d a multiple of 8 (16 for e4m3) up to 4096 (shared memory permitting).  Work units: query t, or one key
// range of a split query (units [0, b_full) whole, then s_last ranges each).
constexpr size_t kCcMaxSmem = 100 * 1024;
struct CcParams {
  const void* q;            // [T, H, d]
  const float* q_scale;     // [T] (fp8)
  const float* w;           // [T, H]
  const void* k_cache;      // [rows, d]
  const float* k_scale;     // [rows] (fp8)
  const int* positions;     // [T] or null
  const int* key_ids;       // dense mode over gathered rows, or null
  int T;
  long long rows;
  int H;
  int d;
  int causal;
  int relu;
  const float* s_min;
  const float* delta;
  const int* theta0;
  unsigned long long* cand;
  int* cnt;
  int* ghist;
  int cap;
  int nb;
  int k;
  int refresh_interval;
  int b_full;
  int s_last;
  int* status;
  float* dense;
  long long ld;
};
size_t score_cc_smem_bytes(int H, int d, int nb);
cudaError_t launch_score_cc(int mode, bool fp8, const CcParams& p, cudaStream_t stream);

// LiteDSA packing (k_litedsa.cu): per group of G queries, the ascending union
// of their selected indices and per-query membership masks.  Needs
// G * k <= litedsa_max_entries() and litedsa_smem_bytes(G, k) <= kLitedsaMaxSmem.
constexpr size_t kLitedsaMaxSmem = 200 * 1024;
int litedsa_max_entries();
size_t litedsa_smem_bytes(int G, int k);
cudaError_t launch_litedsa_pack(const int* topk, int T, int k, int G, int* union_idx, int* union_len,
                                uint32_t* masks, cudaStream_t stream);

// Select stage, decoupled baseline selection and overflow rescue (k_select.cu).
cudaError_t launch_select(const SelectParams& p, int num_sms, cudaStream_t stream);
cudaError_t launch_row_topk(const RowTopkParams& p, cudaStream_t stream);
cudaError_t launch_rescue(const RescueParams& p, int rescue_rows, cudaStream_t stream);

}  // namespace ltk
