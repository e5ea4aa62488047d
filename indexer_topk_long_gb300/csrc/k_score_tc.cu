// k_score_tc.cu -- tensor-core indexer scorer with the fused Filter epilogue.
//
// LiteTopK (gist.science technical summary), Methodology step 2 "Filtering":
// scores are computed by tensor-core matrix multiplication while CUDA cores map
// each score to a bin, keep it only if its bin is at or above the current
// threshold bin ("Gatekeeping"), append kept candidates to warp-local batches
// that are flushed with one atomic per batch ("Write-Back Optimization"), and
// an otherwise idle warp recomputes the threshold bin from the top of the
// histogram with a plain overwrite ("Threshold Refresh").
//
// GB300 design (one CTA per work unit = 8 queries x a key range, 19 warps):
//   * Q tile: 8 queries x 64 heads x d=128 stays resident in shared memory
//     (bf16 128 KB, e4m3 64 KB), loaded once by TMA with 128-byte swizzle.
//   * K tiles of 128 keys stream through a TMA ring (bf16 2 x 32 KB, e4m3
//     4 x 16 KB).
//   * tcgen05.mma, cta_group::1, M = 128 keys, N = 256 = 4 queries x 64 heads
//     (one query group, half of the block): keys sit on TMEM lanes.  TMEM (512
//     columns) holds two accumulators, one per group; the epilogue drains one
//     while the tensor core fills the other.
//   * Epilogue (16 warps in two groups of 8, group g draining accumulator g
//     only, so the two groups run apart and one group's gate / append tail
//     overlaps the other's head sums): one thread per key row, each warp one
//     TMEM lane quarter and two of the group's queries.  A query's 64 head
//     columns of the thread's row come in four tcgen05.ld 32x32b.x16 pieces
//     (the TMEM read shape with the highest bandwidth), the warp's eight pieces
//     each in flight while the previous one is summed, and the accumulator
//     goes back once the last piece has landed; ReLU (x + |x| as a packed
//     fp32x2 add) and the w-weighted head sum (packed fp32x2 FMAs, weights as
//     shared-memory broadcasts) run two heads per instruction, and each thread
//     ends with its key's whole score -> mask -> [dense: store I] or [filter:
//     bin, gate, warp ballot append, shared-memory histogram].
//   * Warp 0 = TMA producer, warp 1 = TMEM allocator + MMA issuer, warp 2 =
//     threshold refresh.
//   * Work units: whole query blocks, or key ranges of a query block split
//     over several CTAs (they share the query's count and a global histogram).
//   * Scan order (general form, filter mode): a CTA starts at the filter's
//     current sweep position (tiles scanned by all CTAs / SMs, mod its range)
//     and wraps around, so CTAs that start in later waves read the key tiles
//     the running CTAs read, while L2 still holds them (1M bf16: 3.3-5.5
//     instead of 9.0 GB of DRAM reads per launch).  The result does not depend on the
//     order: every visible key is scored once and the threshold only rises.
//   * ALT form (T <= 4): one query group with a narrower MMA (N = 64 per
//     query), the two accumulators alternating between tiles, and the unused
//     query rows used as two more key stages.
// Every wait is bounded (2 s); on expiry the kernel records LTK_ERR_TIMEOUT,
// drains its in-flight copies and MMAs, frees TMEM and exits.
#include <climits>
#include <cmath>

#include "ltk_internal.cuh"

namespace ltk {
namespace {

template <bool FP8>
struct Shape {
  static constexpr int kChunks = FP8 ? 1 : 2;                 // 128-byte chunks along d
  static constexpr int kKSteps = kChunks * 4;                 // MMA K steps (32 bytes each)
  static constexpr int kQChunkBytes = kTcQPB * kTcHeads * 128;
  static constexpr int kQBytes = kChunks * kQChunkBytes;      // 128 KB bf16 / 64 KB e4m3
  static constexpr int kKChunkBytes = kTile * 128;
  static constexpr int kKStage = kChunks * kKChunkBytes;      // 32 KB bf16 / 16 KB e4m3
  static constexpr int kStages = FP8 ? 4 : 2;
  // stages that fit in the query rows of group 1 when it is unused (small T)
  static constexpr int kExtraStages = 2;
  static constexpr int kMaxStages = kStages + kExtraStages;
  static constexpr int kMaxBins = FP8 ? 2048 : 512;
  static constexpr int kBoxCols = FP8 ? 128 : 64;             // elements per 128-byte box row
};

constexpr int kEpiWarp0 = 3;
constexpr int kEpiWarps = 16;           // 2 groups x 4 TMEM lane quarters x 2 query pairs
constexpr int kThreads = 32 * (kEpiWarp0 + kEpiWarps);
constexpr int kRefreshWarp = 2;
constexpr int kN = 256;                 // MMA N: 4 queries x 64 heads
constexpr uint32_t kTmemCols = 512;

struct __align__(8) Ctrl {
  uint64_t q_full;
  uint64_t k_full[6];
  uint64_t k_empty[6];
  uint64_t acc_full[2];
  uint64_t acc_empty[2];
  uint64_t mma_done;
  uint32_t tmem_base;
  int abort_flag;
  int tiles_done;                        // epilogue warp-tiles finished
  int rot;                               // first tile of the scan, relative to tile_lo
  float s_min[kTcQPB];
  float delta[kTcQPB];
  int theta[kTcQPB];
  int pos[kTcQPB];
  int cnt[kTcQPB];
};

template <bool FP8>
constexpr size_t smem_bytes(int nb) {
  return 1024 /* alignment slack */ + Shape<FP8>::kQBytes +
         static_cast<size_t>(Shape<FP8>::kStages) * Shape<FP8>::kKStage +
         kTcQPB * kTcHeads * sizeof(float) + sizeof(Ctrl) +
         static_cast<size_t>(kTcQPB) * nb * sizeof(int);
}

// ReLU of a head pair, doubled: one packed add forms (x0 + |x0|, x1 + |x1|) =
// 2 (max(0, x0), max(0, x1)) exactly (|x| is an operand of the add); a packed
// FMA then accumulates it with the pair's weights, and the two halves of the
// accumulator are added and halved at the end (fold_pair, exact), so the sums
// equal sum_h w[h] * max(0, x[h]) up to fp32 rounding.
__device__ __forceinline__ unsigned long long relu2_pair(float x0, float x1) {
  unsigned long long x, ax, s;
  asm("mov.b64 %0, {%1, %2};" : "=l"(x) : "f"(x0), "f"(x1));
  asm("mov.b64 %0, {%1, %2};" : "=l"(ax) : "f"(fabsf(x0)), "f"(fabsf(x1)));
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(s) : "l"(x), "l"(ax));
  return s;
}

__device__ __forceinline__ float fold_pair(unsigned long long acc) {
  const float lo = __uint_as_float(static_cast<uint32_t>(acc));
  const float hi = __uint_as_float(static_cast<uint32_t>(acc >> 32));
  return __fmul_rn(__fadd_rn(lo, hi), 0.5f);
}

// Weighted ReLU sum over 16 consecutive heads of this thread's key (one
// 32x32b x16 load): head pairs (4r, 4r+1) into a0 and (4r+2, 4r+3) into a1,
// two heads per packed add and packed FMA; w points at the 16 weights.
__device__ __forceinline__ void head_sum16(unsigned long long& a0, unsigned long long& a1,
                                           const float (&x)[16], const float4* w) {
#pragma unroll
  for (int r = 0; r < 4; ++r) {
    const float4 wv = w[r];
    unsigned long long w01, w23;
    asm("mov.b64 %0, {%1, %2};" : "=l"(w01) : "f"(wv.x), "f"(wv.y));
    asm("mov.b64 %0, {%1, %2};" : "=l"(w23) : "f"(wv.z), "f"(wv.w));
    asm("fma.rn.f32x2 %0, %1, %2, %0;" : "+l"(a0) : "l"(relu2_pair(x[4 * r + 0], x[4 * r + 1])), "l"(w01));
    asm("fma.rn.f32x2 %0, %1, %2, %0;" : "+l"(a1) : "l"(relu2_pair(x[4 * r + 2], x[4 * r + 3])), "l"(w23));
  }
}

// Threshold refresh by one warp (Methodology step 2, "Threshold Refresh"):
// accumulate the histogram from the top bin down and publish the highest bin b
// whose cumulative count reaches k.  Counts only grow and each counted key is
// distinct, so any b found is a valid lower bound on the bin of the true k-th
// score; the store is a plain overwrite, never below the current value.
// The scan walks 32-bin segments from the top (lane l reads bin top-1-l, so a
// segment is one conflict-free shared-memory access) and stops at the segment
// holding the current threshold: bins below it cannot raise it.
__device__ __forceinline__ void refresh_threshold(const int* hist, int nb, int k,
                                                  volatile int* theta, int lane) {
  const volatile int* hv = hist;
  const int cur = *theta;
  int run = 0;
  for (int top = nb; top > cur; top -= 32) {
    int cum = hv[top - 1 - lane];
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int n = __shfl_up_sync(0xFFFFFFFFu, cum, o);
      if (lane >= o) cum += n;
    }
    const unsigned m = __ballot_sync(0xFFFFFFFFu, run + cum >= k);
    if (m != 0) {
      const int th = top - 1 - (__ffs(m) - 1);
      if (lane == 0 && th > cur) *theta = th;
      return;
    }
    run += __shfl_sync(0xFFFFFFFFu, cum, 31);
  }
}

// Same result as refresh_threshold, for a histogram row in global memory
// (shared by the CTAs that split a query's keys): the warp fetches 16 segments
// at a time with independent loads, so one L2 round trip covers 512 bins.
__device__ __forceinline__ void refresh_threshold_global(const int* grow, int nb, int k,
                                                         volatile int* theta, int lane) {
  const int cur = *theta;
  int run = 0;
  for (int top0 = nb; top0 > cur; top0 -= 32 * 16) {
    int v[16];
#pragma unroll
    for (int j = 0; j < 16; ++j) {
      const int b = top0 - 1 - lane - 32 * j;
      v[j] = b >= 0 ? __ldcg(grow + b) : 0;
    }
#pragma unroll
    for (int j = 0; j < 16; ++j) {
      const int top = top0 - 32 * j;
      if (top <= cur || top <= 0) return;
      int cum = v[j];
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int n = __shfl_up_sync(0xFFFFFFFFu, cum, o);
        if (lane >= o) cum += n;
      }
      const unsigned m = __ballot_sync(0xFFFFFFFFu, run + cum >= k);
      if (m != 0) {
        const int th = top - 1 - (__ffs(m) - 1);
        if (lane == 0 && th > cur) *theta = th;
        return;
      }
      run += __shfl_sync(0xFFFFFFFFu, cum, 31);
    }
  }
}

// ALT (launched only when every query block has at most 4 queries, i.e.
// T <= 4): one query group whose tiles alternate between the two accumulators,
// and a deeper key ring.  The general form computes up to two groups per tile.
template <int MODE, bool FP8, bool ALT>
__global__ void __launch_bounds__(kThreads, 1)
    score_tc_kernel(const __grid_constant__ CUtensorMap q_map,
                    const __grid_constant__ CUtensorMap k_map, const ScoreParams p) {
  using Sh = Shape<FP8>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t pad = ((raw + 1023u) & ~1023u) - raw;
  uint8_t* smem = smem_raw + pad;
  const uint32_t s_q = raw + pad;
  const uint32_t s_k = s_q + Sh::kQBytes;
  float* w_s = reinterpret_cast<float*>(smem + Sh::kQBytes + Sh::kStages * Sh::kKStage);
  Ctrl* ctrl = reinterpret_cast<Ctrl*>(w_s + kTcQPB * kTcHeads);
  int* hist = reinterpret_cast<int*>(ctrl + 1);
  volatile int* abort_flag = &ctrl->abort_flag;

  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  // work unit: a whole query block, or one key range of a split query block
  int qb = blockIdx.x, split = 0, nsplit = 1;
  if (static_cast<int>(blockIdx.x) >= p.b_full && p.s_last > 1) {
    const int u = blockIdx.x - p.b_full;
    qb = p.b_full + u / p.s_last;
    split = u % p.s_last;
    nsplit = p.s_last;
  }
  const bool shared_query = nsplit > 1;   // other CTAs scan other keys of these queries
  const int t0 = qb * kTcQPB;
  const int nq = min(kTcQPB, p.T - t0);
  // Query groups (halves of the block) and queries per group.  General form:
  // both groups, 4 queries each (missing queries of a partial block are
  // computed and masked).  ALT form (T <= 4): one group of nq queries, a
  // narrower MMA (N = 64 per query), the second group neither loaded nor
  // computed, and the two TMEM accumulators alternating between tiles, so the
  // tensor core fills one while the epilogue drains the other.
  constexpr bool alt = ALT;
  const int hq0 = ALT ? nq : 4;
  constexpr int hq1 = ALT ? 0 : 4;
  constexpr int n_halves = ALT ? 1 : 2;
  const int q_acc = hq0;                                  // queries in one accumulator
  const int warps_per_acc = 4 * (q_acc > 2 ? 2 : 1);      // epilogue warps draining one
  const int n_act = (ALT ? 1 : 2) * warps_per_acc;        // epilogue warp-tiles per key tile
  // The key ring: kStages stages after the query rows, plus, when query group 1
  // is unused, kExtraStages more in its rows (a deeper ring for the
  // cache-streaming small-T case).
  constexpr int ns = Sh::kStages + (alt ? Sh::kExtraStages : 0);
  auto k_stage = [&](int st) -> uint32_t {
    if (st < Sh::kStages) return s_k + st * Sh::kKStage;
    const int e = st - Sh::kStages;
    return FP8 ? s_q + kN * 128 + e * Sh::kKStage : s_q + e * Sh::kQChunkBytes + kN * 128;
  };

  // Keys to scan: up to the largest position in the block when causal.
  long long last_row = p.rows;
  if (p.causal && p.positions != nullptr && p.key_ids == nullptr) {
    int mp = -1;
    for (int i = 0; i < nq; ++i) mp = max(mp, p.positions[t0 + i]);
    last_row = min(static_cast<long long>(mp) + 1, p.rows);
    if (last_row < 0) last_row = 0;
  }
  const int block_tiles = static_cast<int>((last_row + kTile - 1) / kTile);
  const int per_split = (block_tiles + nsplit - 1) / nsplit;
  const int tile_lo = split * per_split;
  const int n_tiles = max(0, min(per_split, block_tiles - tile_lo));

  // ---- setup: weights, per-query state, histogram, barriers, TMEM
  // Weights [ql][h] in head order (the epilogue reads 4 heads per float4
  // broadcast).
  for (int i = tid; i < kTcQPB * kTcHeads; i += kThreads) {
    const int ql = i / kTcHeads;
    const int h = i % kTcHeads;
    float wv = 0.f;
    if (ql < nq) {
      wv = p.w[static_cast<size_t>(t0 + ql) * kTcHeads + h];
      if constexpr (FP8) wv = __fmul_rn(wv, p.q_scale[t0 + ql]);
    }
    w_s[i] = wv;
  }
  if (tid < kTcQPB) {
    const bool ok = tid < nq;
    ctrl->pos[tid] = (ok && p.positions != nullptr) ? p.positions[t0 + tid] : INT_MAX;
    ctrl->cnt[tid] = 0;
    if constexpr (MODE == kModeFilter) {
      ctrl->s_min[tid] = ok ? p.s_min[t0 + tid] : 0.f;
      ctrl->delta[tid] = ok ? p.delta[t0 + tid] : 0.f;
      ctrl->theta[tid] = ok ? p.theta0[t0 + tid] : 0;
    }
  }
  if constexpr (MODE == kModeFilter) {
    for (int i = tid; i < kTcQPB * p.nb; i += kThreads) hist[i] = 0;
  }
  if (tid == 0) {
    ctrl->abort_flag = 0;
    ctrl->tiles_done = 0;
    // the scan starts at the filter's current sweep position (when it falls in
    // this unit's range) and wraps around; any order gives the same result
    int rot = 0;
    if (MODE == kModeFilter && !ALT && p.sweep != nullptr && n_tiles > 1) {
      const unsigned long long done = *reinterpret_cast<volatile unsigned long long*>(p.sweep);
      const long long pos = static_cast<long long>(done / static_cast<unsigned long long>(p.num_sms)) %
                            block_tiles;
      const long long rel = pos - tile_lo;
      if (rel > 0 && rel < n_tiles) rot = static_cast<int>(rel);
    }
    ctrl->rot = rot;
    mbar_init(smem_u32(&ctrl->q_full), 1);
    for (int s = 0; s < Sh::kMaxStages; ++s) {
      mbar_init(smem_u32(&ctrl->k_full[s]), 1);
      mbar_init(smem_u32(&ctrl->k_empty[s]), 1);
    }
    for (int j = 0; j < 2; ++j) {
      mbar_init(smem_u32(&ctrl->acc_full[j]), 1);
      mbar_init(smem_u32(&ctrl->acc_empty[j]), warps_per_acc);
    }
    mbar_init(smem_u32(&ctrl->mma_done), 1);
    mbar_fence_init();
  }
  if (warp == 1) tmem_alloc(smem_u32(&ctrl->tmem_base), kTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = ctrl->tmem_base;
  const int rot = ctrl->rot;

  if (n_tiles > 0) {
    if (warp == 0) {
      // ---------------- TMA producer ----------------
      if (lane == 0) {
        tma_prefetch_desc(&q_map);
        tma_prefetch_desc(&k_map);
        const uint32_t qbar = smem_u32(&ctrl->q_full);
        // the query rows of the groups in use (a group without queries is skipped)
        mbar_arrive_expect_tx(qbar, Sh::kQBytes / 2 * n_halves);
        for (int j = 0; j < n_halves; ++j)
          for (int c = 0; c < Sh::kChunks; ++c)
            tma_load_2d(s_q + c * Sh::kQChunkBytes + j * (kN * 128), &q_map, c * Sh::kBoxCols,
                        (t0 + 4 * j) * kTcHeads, qbar);
        int issued[Sh::kMaxStages];
        for (int s = 0; s < Sh::kMaxStages; ++s) issued[s] = -1;
        for (int i = 0; i < (p.skip_key_loads ? 0 : n_tiles); ++i) {
          const int s = i % ns;
          if (i >= ns &&
              !mbar_wait(smem_u32(&ctrl->k_empty[s]), ((i / ns) - 1) & 1, abort_flag, p.status))
            break;
          const uint32_t fb = smem_u32(&ctrl->k_full[s]);
          mbar_arrive_expect_tx(fb, Sh::kKStage);
          const uint32_t dst = k_stage(s);
          const int ti = i + rot < n_tiles ? i + rot : i + rot - n_tiles;   // rotated scan
          for (int c = 0; c < Sh::kChunks; ++c)
            tma_load_2d(dst + c * Sh::kKChunkBytes, &k_map, c * Sh::kBoxCols, (tile_lo + ti) * kTile, fb);
          issued[s] = i;
        }
        if (*abort_flag) {
          // drain copies still in flight before the CTA may exit
          mbar_drain(qbar, 0);
          for (int s = 0; s < ns; ++s)
            if (issued[s] >= 0) mbar_drain(smem_u32(&ctrl->k_full[s]), (issued[s] / ns) & 1);
        }
      }
    } else if (warp == 1) {
      // ---------------- MMA issuer ----------------
      if (lane == 0) {
        const uint32_t idesc0 = make_idesc(FP8, kTile, kTcHeads * hq0);
        const uint32_t idesc1 = make_idesc(FP8, kTile, kTcHeads * (hq1 > 0 ? hq1 : 1));
        bool ok = mbar_wait(smem_u32(&ctrl->q_full), 0, abort_flag, p.status);
        for (int i = 0; ok && i < n_tiles; ++i) {
          const int s = i % ns;
          if (!mbar_wait(smem_u32(&ctrl->k_full[s]), (i / ns) & 1, abort_flag, p.status))
            break;
          const uint32_t ks_base = k_stage(s);
          tc_fence_after();
#pragma unroll
          for (int g = 0; g < 2; ++g) {   // query group (half of the query block)
            if (g >= n_halves) break;   // unrolled: the MMA issue loop must stay straight-line
            const uint32_t idesc = g == 0 ? idesc0 : idesc1;
            const int j = alt ? (i & 1) : g;      // accumulator
            const int use = alt ? (i >> 1) : i;   // earlier tiles that used accumulator j
            if (use > 0) {
              if (!mbar_wait(smem_u32(&ctrl->acc_empty[j]), (use - 1) & 1, abort_flag, p.status)) {
                ok = false;
                break;
              }
              tc_fence_after();
            }
            const uint32_t d_tmem = tmem + j * kN;
#pragma unroll
            for (int ks = 0; ks < Sh::kKSteps; ++ks) {
              const int c = ks >> 2;
              const int kk = ks & 3;
              const uint64_t a = smem_desc_sw128(ks_base + c * Sh::kKChunkBytes + kk * 32);
              const uint64_t b = smem_desc_sw128(s_q + c * Sh::kQChunkBytes + g * (kN * 128) + kk * 32);
              tc_mma<FP8>(d_tmem, a, b, idesc, ks > 0 ? 1u : 0u);
            }
            tc_commit(smem_u32(&ctrl->acc_full[j]));
          }
          if (!ok) break;
          tc_commit(smem_u32(&ctrl->k_empty[s]));
        }
        // every MMA issued so far must finish before TMEM is freed
        tc_commit(smem_u32(&ctrl->mma_done));
        mbar_drain(smem_u32(&ctrl->mma_done), 0);
      }
    } else if (warp == kRefreshWarp) {
      // ---------------- threshold refresh ----------------
      if constexpr (MODE == kModeFilter) {
        if (p.refresh_interval > 0) {
          int last = 0;
          int prev_done = -1;
          uint64_t t_prog = globaltimer_ns();
          while (true) {
            int done = *reinterpret_cast<volatile int*>(&ctrl->tiles_done) / n_act;
            done = __shfl_sync(0xFFFFFFFFu, done, 0);
            const int ab = __shfl_sync(0xFFFFFFFFu, *abort_flag, 0);
            if (done >= n_tiles || ab) break;
            if (done != prev_done) {
              // advance the filter's sweep counter in steps of 16 tiles (the
              // start of a later CTA's scan; off the MMA and copy paths)
              if (lane == 0 && p.sweep != nullptr && prev_done >= 0 && (done >> 4) > (prev_done >> 4))
                atomicAdd(p.sweep, static_cast<unsigned long long>(16 * ((done >> 4) - (prev_done >> 4))));
              prev_done = done;
              t_prog = globaltimer_ns();
            }
            if (done - last >= p.refresh_interval) {
              last = done;
              for (int ql = 0; ql < nq; ++ql) {
                if (shared_query) {
                  // move this CTA's new counts into the query's histogram over all
                  // CTAs, then take the threshold from those counts
                  int* grow = p.ghist + static_cast<size_t>(t0 + ql) * p.nb;
                  for (int b = lane; b < p.nb; b += 32) {
                    const int cnt_b = atomicExch(&hist[ql * p.nb + b], 0);
                    if (cnt_b != 0) atomicAdd(&grow[b], cnt_b);
                  }
                  __syncwarp();
                  refresh_threshold_global(grow, p.nb, p.k,
                                           reinterpret_cast<volatile int*>(&ctrl->theta[ql]), lane);
                } else {
                  refresh_threshold(hist + ql * p.nb, p.nb, p.k,
                                    reinterpret_cast<volatile int*>(&ctrl->theta[ql]), lane);
                }
              }
            } else {
              __nanosleep(1000);
              bool expired = globaltimer_ns() - t_prog > kWaitLimitNs;
              expired = __shfl_sync(0xFFFFFFFFu, expired, 0);
              if (expired) {
                if (lane == 0) {
                  *abort_flag = 1;
                  raise_status(p.status, kDevTimeout);
                }
                break;
              }
            }
          }
        }
      }
    } else if (warp >= kEpiWarp0) {
      // ---------------- epilogue ----------------
      // Two groups of 8 warps, group g draining accumulator g (so the groups
      // run half a tile apart and one group's bin / gate / append tail
      // overlaps the other's head sums on every scheduler); each warp covers
      // one TMEM lane quarter and a pair of the accumulator's queries, drained
      // back to back.
      const int e = warp - kEpiWarp0;
      const int lq = warp & 3;               // TMEM lane quarter this warp may access
      const int g = e >> 3;                  // accumulator this warp drains
      const int m = (e >> 2) & 1;            // query pair within the accumulator
      const int nu = max(0, min(2, q_acc - 2 * m));   // queries this warp drains per tile
      if (nu > 0) {
        const int row = lq * 32 + lane;        // key row of this thread (32x32b loads)
        const uint32_t lane_base = static_cast<uint32_t>(lq * 32) << 16;
        const int qbase = (alt ? 0 : 4 * g) + 2 * m;   // first of the pair, within the CTA
        const int rows_i = static_cast<int>(p.rows < 0x7FFFFFFF ? p.rows : 0x7FFFFFFF);
        int last_key[2];
        float qs_min[2], qdelta[2];
        int* qhist[2];
        unsigned long long* qcand[2];
#pragma unroll
        for (int u = 0; u < 2; ++u) {
          const int ql = qbase + u;
          const bool valid = u < nu && ql < nq;
          // a key is visible iff key <= last_key (causal position and cache end)
          last_key[u] = valid ? min(p.causal ? ctrl->pos[ql] : 0x7FFFFFFF, rows_i - 1) : -1;
          if constexpr (MODE == kModeFilter) {
            qs_min[u] = ctrl->s_min[ql];
            qdelta[u] = ctrl->delta[ql];
            qhist[u] = hist + ql * p.nb;
            qcand[u] = p.cand + static_cast<size_t>(valid ? t0 + ql : 0) * p.cap;
          }
        }
        const uint32_t acc_full_g = smem_u32(&ctrl->acc_full[g]);
        const uint32_t acc_empty_g = smem_u32(&ctrl->acc_empty[g]);
        // columns of the pair in accumulator g (query 2m of the group at 64 * 2m)
        const uint32_t ta = tmem + lane_base + static_cast<uint32_t>(g * kN + 2 * m * kTcHeads);
        const float4* w0 = reinterpret_cast<const float4*>(w_s + qbase * kTcHeads);
        const float4* w1 = w0 + kTcHeads / 4;
        // ALT form: the accumulators alternate between tiles, so group g takes
        // the tiles of parity g
        for (int i = alt ? g : 0; i < n_tiles; i += alt ? 2 : 1) {
          const int use = alt ? (i >> 1) : i;   // earlier tiles that used accumulator g
          const int ti = i + rot < n_tiles ? i + rot : i + rot - n_tiles;   // rotated scan
          const int key = (tile_lo + ti) * kTile + row;
          const bool key_ok = key < rows_i;
          float kscale = 1.f;
          if constexpr (FP8) kscale = key_ok ? p.k_scale[key] : 0.f;
          int kid = key;
          if (MODE == kModeDense && p.key_ids != nullptr) kid = key_ok ? p.key_ids[key] : INT_MAX;
          bool ok = mbar_wait(acc_full_g, use & 1, abort_flag, p.status);
          ok = __all_sync(0xFFFFFFFFu, ok);
          if (!ok) break;
          tc_fence_after();
          // the thresholds are read before the scores (any value read is a
          // valid lower bound), so the loads' latency overlaps the TMEM loads
          int th_pre[2] = {0, 0};
          if constexpr (MODE == kModeFilter) {
            th_pre[0] = *reinterpret_cast<volatile int*>(&ctrl->theta[qbase]);
            th_pre[1] = *reinterpret_cast<volatile int*>(&ctrl->theta[qbase + 1]);
          }
          // each query's 64 head columns of this thread's key row in four
          // 32x32b x16 loads, one in flight while the previous is summed; the
          // accumulator goes back once the last load has landed
          float xa[16], xb[16];
          unsigned long long a0 = 0ull, a1 = 0ull, b0 = 0ull, b1 = 0ull;   // (+0.f, +0.f)
          tmem_ld32x16(ta, xa);
          tmem_wait_ld_tied(xa);
          tmem_ld32x16(ta + 16u, xb);
          head_sum16(a0, a1, xa, w0);
          tmem_wait_ld_tied(xb);
          tmem_ld32x16(ta + 32u, xa);
          head_sum16(a0, a1, xb, w0 + 4);
          tmem_wait_ld_tied(xa);
          tmem_ld32x16(ta + 48u, xb);
          head_sum16(a0, a1, xa, w0 + 8);
          tmem_wait_ld_tied(xb);
          if (nu == 2) {
            tmem_ld32x16(ta + 64u, xa);
            head_sum16(a0, a1, xb, w0 + 12);
            tmem_wait_ld_tied(xa);
            tmem_ld32x16(ta + 80u, xb);
            head_sum16(b0, b1, xa, w1);
            tmem_wait_ld_tied(xb);
            tmem_ld32x16(ta + 96u, xa);
            head_sum16(b0, b1, xb, w1 + 4);
            tmem_wait_ld_tied(xa);
            tmem_ld32x16(ta + 112u, xb);
            head_sum16(b0, b1, xa, w1 + 8);
            tmem_wait_ld_tied(xb);
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(acc_empty_g);
            head_sum16(b0, b1, xb, w1 + 12);
          } else {
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(acc_empty_g);
            head_sum16(a0, a1, xb, w0 + 12);
          }
          const float I_pair[2] = {__fadd_rn(fold_pair(a0), fold_pair(a1)),
                                   __fadd_rn(fold_pair(b0), fold_pair(b1))};
#pragma unroll
          for (int u = 0; u < 2; ++u) {
            if (u >= nu) break;
            const int ql = qbase + u;   // query within the CTA
            float I = I_pair[u];
            if constexpr (FP8) I = __fmul_rn(I, kscale);
            if constexpr (MODE == kModeDense) {
              if (ql < nq && key_ok) {
                bool vis = kid != INT_MAX;
                if (p.causal && p.positions != nullptr) vis = vis && kid <= ctrl->pos[ql];
                p.dense[static_cast<size_t>(t0 + ql) * p.ld + key] = vis ? I : -INFINITY;
              }
            } else {
              const int b = bin_of(I, qs_min[u], qdelta[u], p.nb);
              const bool pass = key <= last_key[u] && b >= th_pre[u];
              const unsigned msk = __ballot_sync(0xFFFFFFFFu, pass);
              if (msk != 0) {
                const int leader = __ffs(msk) - 1;
                int base = 0;
                if (lane == leader)
                  base = shared_query ? atomicAdd(&p.cnt[t0 + ql], __popc(msk))
                                      : atomicAdd(&ctrl->cnt[ql], __popc(msk));
                base = __shfl_sync(0xFFFFFFFFu, base, leader);
                if (pass) {
                  const int slot = base + __popc(msk & ((1u << lane) - 1u));
                  if (slot < p.cap) qcand[u][slot] = cand_pack(I, key);
                  atomicAdd(&qhist[u][b], 1);
                }
              }
            }
          }
          if (lane == 0) atomicAdd(&ctrl->tiles_done, 1);
        }
      }
    }
  }

  // ---- teardown
  __syncwarp();
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
  if constexpr (MODE == kModeFilter) {
    if (tid < nq && !shared_query) p.cnt[t0 + tid] = ctrl->cnt[tid];
  }
}

template <int MODE, bool FP8, bool ALT>
cudaError_t launch_one(const CUtensorMap& qm, const CUtensorMap& km, const ScoreParams& p,
                       cudaStream_t stream) {
  const int t_blocks = (p.T + kTcQPB - 1) / kTcQPB;
  if (t_blocks == 0) return cudaSuccess;
  const int grid = p.b_full + (t_blocks - p.b_full) * (p.s_last > 1 ? p.s_last : 1);
  const size_t smem = smem_bytes<FP8>(MODE == kModeFilter ? p.nb : 0);
  cudaError_t e = ensure_smem_limit(reinterpret_cast<const void*>(score_tc_kernel<MODE, FP8, ALT>),
                                    kSlotScoreTc + MODE * 4 + (FP8 ? 2 : 0) + (ALT ? 1 : 0),
                                    smem_bytes<FP8>(Shape<FP8>::kMaxBins));
  if (e != cudaSuccess) return e;
  score_tc_kernel<MODE, FP8, ALT><<<grid, kThreads, smem, stream>>>(qm, km, p);
  count_launches(1);
  return cudaGetLastError();
}

}  // namespace

size_t score_tc_smem_bytes(int mode, bool fp8, int nb) {
  const int b = mode == kModeFilter ? nb : 0;
  return fp8 ? smem_bytes<true>(b) : smem_bytes<false>(b);
}

int score_tc_max_bins(bool fp8) { return fp8 ? Shape<true>::kMaxBins : Shape<false>::kMaxBins; }

cudaError_t launch_score_tc(int mode, bool fp8, const CUtensorMap& q_map, const CUtensorMap& k_map,
                            const ScoreParams& p, cudaStream_t stream) {
  const bool alt = p.T <= 4;   // every query block has at most one group of queries
  if (mode == kModeDense) {
    if (fp8) return alt ? launch_one<kModeDense, true, true>(q_map, k_map, p, stream)
                        : launch_one<kModeDense, true, false>(q_map, k_map, p, stream);
    return alt ? launch_one<kModeDense, false, true>(q_map, k_map, p, stream)
               : launch_one<kModeDense, false, false>(q_map, k_map, p, stream);
  }
  if (fp8) return alt ? launch_one<kModeFilter, true, true>(q_map, k_map, p, stream)
                      : launch_one<kModeFilter, true, false>(q_map, k_map, p, stream);
  return alt ? launch_one<kModeFilter, false, true>(q_map, k_map, p, stream)
             : launch_one<kModeFilter, false, false>(q_map, k_map, p, stream);
}

}  // namespace ltk
