// k_retrieval_tc.cu -- tensor-core scorer for the vector-retrieval variant of
// Indexer-TopK (LiteTopK arXiv abstract and the summary's Experimental
// Results: "vector retrieval" with k from 1024 to 8192): one head, a plain
// inner product I[t,s] = w[t] * (q[t,:] . c[s,:]) (optionally ReLU'd), no
// causal mask, d up to 1024.
//
// The Sample / Filter / Select method is the same as for the indexer
// (Methodology steps 1-3); this file supplies the score kernel and its fused
// filter epilogue for this shape.  With d = 768 a query block cannot stay in
// shared memory, so both operands stream:
//   * CTA = (query block of 256 queries) x (a contiguous range of corpus tiles);
//     the grid puts the query blocks of one corpus range next to each other so
//     that they read the same corpus tiles from L2 at about the same time.
//   * tcgen05.mma, cta_group::1, M = 128 corpus rows, N = 256 queries, the K
//     loop runs over d in 64-column chunks staged by TMA (128-byte swizzle) in a
//     3-deep ring of (16 KB corpus chunk + 32 KB query chunk).
//   * TMEM holds two 256-column accumulators: the epilogue drains one corpus
//     tile while the tensor core computes the next.
//   * Epilogue (16 warps, four per scheduler, so that the latency of one warp's
//     global append is covered by the others): each thread owns one corpus row
//     and 64 query columns, read from TMEM 16 columns at a time, each load in
//     flight while the previous 16 columns are gated.
//     The gate "bin >= theta" is evaluated as one compare against a per-query
//     score threshold tau = the smallest float whose bin is >= theta (found by
//     binary search over float order, so the two tests agree exactly).
//   * Several CTAs scan different corpus ranges of the same query.  Each
//     appends to its own segment of the query's candidate list with a
//     CTA-local count (no global atomic on the append path), and the threshold must
//     come from all of the query's kept keys: epilogue threads count kept keys
//     in a shared-memory histogram; at each refresh the refresh warp moves
//     those counts (atomicExch) into a global per-query histogram and derives
//     the threshold bin from the global counts, which cover every CTA's
//     distinct kept keys.
//   * The refresh warp handles 32 queries at a time, one lane per query (shared
//     rows padded to an odd stride, so the lanes hit distinct banks; the global
//     row is read with 16-byte loads).
#include <climits>
#include <cmath>

#include "ltk_internal.cuh"

namespace ltk {
namespace {

constexpr int kRThreads = 640;
constexpr int kREpiWarp0 = 4;
constexpr int kREpiWarps = 16;
constexpr int kRRefreshWarp = 2;
constexpr int kRN = 256;                 // queries per CTA (MMA N)
constexpr int kRStages = 3;
constexpr int kRAChunk = kTile * 128;    // 128 rows x 64 bf16
constexpr int kRBChunk = kRN * 128;      // 256 rows x 64 bf16
constexpr int kRStage = kRAChunk + kRBChunk;
constexpr uint32_t kRTmemCols = 512;

struct QState {
  float s_min;
  float delta;
  int theta;
  int pad;
};

struct __align__(8) RCtrl {
  uint64_t full[kRStages];
  uint64_t empty[kRStages];
  uint64_t acc_full[2];
  uint64_t acc_empty[2];
  uint64_t mma_done;
  uint32_t tmem_base;
  int abort_flag;
  int tiles_done;
  int pad0;
};

// Histogram row stride: nb + 1 words (odd), so 32 lanes reading 32 rows at the
// same bin hit 32 different banks.
__host__ __device__ constexpr int r_hist_stride(int nb) { return nb + 1; }

constexpr size_t r_smem_bytes(int nb) {
  return 1024 + static_cast<size_t>(kRStages) * kRStage + kRN * sizeof(QState) + kRN * sizeof(float2) +
         sizeof(RCtrl) + static_cast<size_t>(kRN) * (nb > 0 ? r_hist_stride(nb) : 0) * sizeof(int);
}

// Smallest float v with bin_of(v, s_min, delta, nb) >= theta (bin_of is
// monotone in v), by binary search over the order-preserving codes between
// -inf and +inf; -inf when theta <= 0.
__device__ float gate_tau(int theta, float s_min, float delta, int nb) {
  if (theta <= 0) return -INFINITY;
  uint32_t lo = ord_f32(-INFINITY), hi = ord_f32(INFINITY);   // pred(lo) false, pred(hi) true
  while (hi - lo > 1u) {
    const uint32_t mid = lo + (hi - lo) / 2u;
    if (bin_of(unord_f32(mid), s_min, delta, nb) >= theta)
      hi = mid;
    else
      lo = mid;
  }
  return unord_f32(hi);
}

// Append the passing rows of one query (whole warp; m = the warp's pass mask,
// nonzero) to this CTA's segment of the query's list: the leader reserves the
// slots on the CTA-local count (shared memory), every passing lane writes its
// (score, row) record and counts it in the query's shared histogram.  Entries
// past the segment are dropped (the count still grows, which marks the
// overflow).  Kept out of line so that the epilogue's per-query loop stays
// small in the instruction cache; it runs only for (query, 32-row) blocks
// with a pass.
__device__ __noinline__ void append_passes(unsigned long long* seg, int seg_cap, int* local_cnt, unsigned m,
                                           bool pass, float I, int key, int* hrow, float s_min, float delta,
                                           int nb) {
  const int lane = threadIdx.x & 31;
  const int leader = __ffs(m) - 1;
  int base = 0;
  if (lane == leader) base = atomicAdd(local_cnt, __popc(m));
  base = __shfl_sync(0xFFFFFFFFu, base, leader);
  if (pass) {
    const int slot = base + __popc(m & ((1u << lane) - 1u));
    if (slot < seg_cap) seg[slot] = cand_pack(I, key);
    atomicAdd(&hrow[bin_of(I, s_min, delta, nb)], 1);
  }
}

template <int MODE, bool RELU>
__global__ void __launch_bounds__(kRThreads, 1)
    retrieval_tc_kernel(const __grid_constant__ CUtensorMap q_map,
                        const __grid_constant__ CUtensorMap c_map, const ScoreParams p,
                        int n_chunks, int t_blocks, int tiles_per_split,
                        int* ghist) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t pad = ((raw + 1023u) & ~1023u) - raw;
  uint8_t* smem = smem_raw + pad;
  const uint32_t s_stage = raw + pad;
  QState* qs = reinterpret_cast<QState*>(smem + kRStages * kRStage);
  float2* tw = reinterpret_cast<float2*>(qs + kRN);   // per query {gate threshold tau, weight}
  RCtrl* ctrl = reinterpret_cast<RCtrl*>(tw + kRN);
  int* hist = reinterpret_cast<int*>(ctrl + 1);
  const int hstride = r_hist_stride(p.nb);
  volatile int* abort_flag = &ctrl->abort_flag;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int qb = blockIdx.x % t_blocks;
  const int split = blockIdx.x / t_blocks;
  const int t0 = qb * kRN;
  const int nq = min(kRN, p.T - t0);
  const int total_tiles = static_cast<int>((p.rows + kTile - 1) / kTile);
  const int tile_lo = split * tiles_per_split;
  const int n_tiles = max(0, min(tiles_per_split, total_tiles - tile_lo));

  for (int q = tid; q < kRN; q += kRThreads) {
    const bool ok = q < nq;
    float tau = INFINITY;
    if constexpr (MODE == kModeFilter) {
      QState st;
      st.s_min = ok ? p.s_min[t0 + q] : 0.f;
      st.delta = ok ? p.delta[t0 + q] : 0.f;
      const int th = ok ? p.theta0[t0 + q] : 0;
      st.theta = th;
      st.pad = 0;
      if (ok) tau = gate_tau(th, st.s_min, st.delta, p.nb);
      qs[q] = st;
    }
    tw[q] = make_float2(tau, ok ? p.w[t0 + q] : 0.f);
  }
  if constexpr (MODE == kModeFilter) {
    for (int i = tid; i < kRN * hstride; i += kRThreads) hist[i] = 0;
  }
  if (tid == 0) {
    ctrl->abort_flag = 0;
    ctrl->tiles_done = 0;
    for (int s = 0; s < kRStages; ++s) {
      mbar_init(smem_u32(&ctrl->full[s]), 1);
      mbar_init(smem_u32(&ctrl->empty[s]), 1);
    }
    for (int j = 0; j < 2; ++j) {
      mbar_init(smem_u32(&ctrl->acc_full[j]), 1);
      mbar_init(smem_u32(&ctrl->acc_empty[j]), kREpiWarps);
    }
    mbar_init(smem_u32(&ctrl->mma_done), 1);
    mbar_fence_init();
  }
  if (warp == 1) tmem_alloc(smem_u32(&ctrl->tmem_base), kRTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = ctrl->tmem_base;

  if (n_tiles > 0) {
    if (warp == 0) {
      // ---------------- TMA producer ----------------
      if (lane == 0) {
        tma_prefetch_desc(&q_map);
        tma_prefetch_desc(&c_map);
        int it = 0;
        int issued[kRStages] = {-1, -1, -1};
        bool ok = true;
        for (int i = 0; i < n_tiles && ok; ++i) {
          const int row0 = (tile_lo + i) * kTile;
          for (int c = 0; c < n_chunks; ++c, ++it) {
            const int s = it % kRStages;
            if (it >= kRStages &&
                !mbar_wait(smem_u32(&ctrl->empty[s]), ((it / kRStages) - 1) & 1, abort_flag,
                           p.status)) {
              ok = false;
              break;
            }
            const uint32_t fb = smem_u32(&ctrl->full[s]);
            mbar_arrive_expect_tx(fb, kRStage);
            tma_load_2d(s_stage + s * kRStage, &c_map, c * 64, row0, fb);
            tma_load_2d(s_stage + s * kRStage + kRAChunk, &q_map, c * 64, t0, fb);
            issued[s] = it;
          }
        }
        if (*abort_flag) {
          for (int s = 0; s < kRStages; ++s)
            if (issued[s] >= 0) mbar_drain(smem_u32(&ctrl->full[s]), (issued[s] / kRStages) & 1);
        }
      }
    } else if (warp == 1) {
      // ---------------- MMA issuer ----------------
      if (lane == 0) {
        const uint32_t idesc = make_idesc(false, kTile, kRN);
        int it = 0;
        bool ok = true;
        for (int i = 0; i < n_tiles && ok; ++i) {
          const int buf = i & 1;
          if (i >= 2) {
            if (!mbar_wait(smem_u32(&ctrl->acc_empty[buf]), ((i >> 1) - 1) & 1, abort_flag,
                           p.status))
              break;
            tc_fence_after();
          }
          const uint32_t d_tmem = tmem + buf * kRN;
          for (int c = 0; c < n_chunks; ++c, ++it) {
            const int s = it % kRStages;
            if (!mbar_wait(smem_u32(&ctrl->full[s]), (it / kRStages) & 1, abort_flag, p.status)) {
              ok = false;
              break;
            }
            tc_fence_after();
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
              const uint64_t a = smem_desc_sw128(s_stage + s * kRStage + kk * 32);
              const uint64_t b = smem_desc_sw128(s_stage + s * kRStage + kRAChunk + kk * 32);
              tc_mma<false>(d_tmem, a, b, idesc, (c > 0 || kk > 0) ? 1u : 0u);
            }
            tc_commit(smem_u32(&ctrl->empty[s]));
          }
          if (!ok) break;
          tc_commit(smem_u32(&ctrl->acc_full[buf]));
        }
        tc_commit(smem_u32(&ctrl->mma_done));
        mbar_drain(smem_u32(&ctrl->mma_done), 0);
      }
    } else if (warp == kRRefreshWarp) {
      // ---------------- threshold refresh ----------------
      if constexpr (MODE == kModeFilter) {
        if (p.refresh_interval > 0) {
          int last = 0, prev_done = -1;
          uint64_t t_prog = globaltimer_ns();
          while (true) {
            int done = *reinterpret_cast<volatile int*>(&ctrl->tiles_done) / kREpiWarps;
            done = __shfl_sync(0xFFFFFFFFu, done, 0);
            const int ab = __shfl_sync(0xFFFFFFFFu, *abort_flag, 0);
            if (done >= n_tiles || ab) break;
            if (done != prev_done) {
              prev_done = done;
              t_prog = globaltimer_ns();
            }
            if (done - last >= p.refresh_interval) {
              last = done;
              for (int q0 = 0; q0 < nq; q0 += 32) {
                const int q = q0 + lane;
                if (q < nq) {
                  int* row = hist + q * hstride;
                  int* grow = ghist + static_cast<size_t>(t0 + q) * p.nb;
                  // move this CTA's new counts into the query's global histogram
                  for (int b = 0; b < p.nb; ++b) {
                    const int c = atomicExch(&row[b], 0);
                    if (c != 0) atomicAdd(&grow[b], c);
                  }
                  __threadfence_block();
                  const int cur = *reinterpret_cast<volatile int*>(&qs[q].theta);
                  int run = 0, found = -1;
                  for (int b4 = p.nb / 4 - 1; b4 >= 0 && found < 0; --b4) {
                    const int4 g = __ldcg(reinterpret_cast<const int4*>(grow) + b4);
                    const int vals[4] = {g.w, g.z, g.y, g.x};
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                      const int b = 4 * b4 + 3 - j;
                      run += vals[j];
                      if (found < 0 && run >= p.k && b > cur) found = b;
                    }
                    if (4 * b4 <= cur) break;
                  }
                  if (found > cur) {
                    const QState st = qs[q];
                    *reinterpret_cast<volatile float*>(&tw[q].x) = gate_tau(found, st.s_min, st.delta, p.nb);
                    *reinterpret_cast<volatile int*>(&qs[q].theta) = found;
                  }
                }
              }
            } else {
              __nanosleep(2000);
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
    } else if (warp >= kREpiWarp0) {
      // ---------------- epilogue ----------------
      const int lq = warp & 3;
      const int ch = (warp - kREpiWarp0) >> 2;      // which 64 of the 256 query columns
      const int row = lq * 32 + lane;
      const uint32_t lane_base = static_cast<uint32_t>(lq * 32) << 16;
      const int rows_i = static_cast<int>(p.rows < 0x7FFFFFFF ? p.rows : 0x7FFFFFFF);
      for (int i = 0; i < n_tiles; ++i) {
        const int buf = i & 1;
        bool ok = mbar_wait(smem_u32(&ctrl->acc_full[buf]), (i >> 1) & 1, abort_flag, p.status);
        ok = __all_sync(0xFFFFFFFFu, ok);
        if (!ok) break;
        tc_fence_after();
        const int key = (tile_lo + i) * kTile + row;
        const bool key_ok = key < rows_i;
        int kid = key;
        if (MODE == kModeDense && p.key_ids != nullptr) kid = key_ok ? p.key_ids[key] : INT_MAX;
        // gate (or store) 16 query columns of this thread's corpus row
        auto columns = [&](const float (&v)[16], const int col0) {
#pragma unroll
          for (int jj = 0; jj < 16; ++jj) {
            const int q = col0 + jj;
            if constexpr (MODE == kModeDense) {
              const float I = __fmul_rn(RELU ? fmaxf(v[jj], 0.f) : v[jj], tw[q].y);
              if (q < nq && key_ok)
                p.dense[static_cast<size_t>(t0 + q) * p.ld + key] = (kid != INT_MAX) ? I : -INFINITY;
            } else {
              // {tau, w} in one load; tau is rewritten by the refresh warp
              const unsigned long long g = *reinterpret_cast<volatile unsigned long long*>(&tw[q]);
              const float I = __fmul_rn(RELU ? fmaxf(v[jj], 0.f) : v[jj],
                                        __uint_as_float(static_cast<uint32_t>(g >> 32)));
              const bool pass = key_ok && q < nq && I >= __uint_as_float(static_cast<uint32_t>(g));
              const unsigned m = __ballot_sync(0xFFFFFFFFu, pass);
              if (m != 0u) {
                const QState st = qs[q];
                int* hrow = hist + q * hstride;
                append_passes(p.cand + static_cast<size_t>(t0 + q) * p.cap + static_cast<size_t>(split) * p.seg_cap,
                              p.seg_cap, hrow + p.nb, m, pass, I, key, hrow, st.s_min, st.delta, p.nb);
              }
            }
          }
        };
        const uint32_t tbase = tmem + lane_base + buf * kRN + ch * 64;
        float va[16], vb[16];
        tmem_ld32x16(tbase, va);
        tmem_wait_ld_tied(va);
#pragma unroll 1
        for (int c2 = 0; c2 < 64; c2 += 32) {
          // piece c2 + 16 loads while piece c2 is gated, and so on
          tmem_ld32x16(tbase + c2 + 16u, vb);
          columns(va, ch * 64 + c2);
          tmem_wait_ld_tied(vb);
          if (c2 == 0) {
            tmem_ld32x16(tbase + 32u, va);
          } else {
            // every column of this tile is in registers: hand the accumulator back
            tc_fence_before();
            __syncwarp();
            if (lane == 0) {
              mbar_arrive(smem_u32(&ctrl->acc_empty[buf]));
              atomicAdd(&ctrl->tiles_done, 1);
            }
          }
          columns(vb, ch * 64 + c2 + 16);
          if (c2 == 0) tmem_wait_ld_tied(va);
        }
      }
    }
  }

  __syncwarp();
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kRTmemCols);
  }
  if constexpr (MODE == kModeFilter) {
    // this CTA's segment counts (the count sits in the pad word of the query's
    // histogram row); an overflowed segment marks the whole query for rescue
    for (int q = tid; q < nq; q += kRThreads) {
      const int c = hist[q * hstride + p.nb];
      p.seg_cnt[static_cast<size_t>(t0 + q) * p.nseg + split] = min(c, p.seg_cap);
      if (c > p.seg_cap) p.cnt[t0 + q] = p.cap + 1;
    }
  }
}

template <int MODE, bool RELU>
cudaError_t launch_r(const CUtensorMap& qm, const CUtensorMap& cm, const ScoreParams& p, int dim,
                     int* ghist, int num_sms, cudaStream_t stream) {
  const int t_blocks = (p.T + kRN - 1) / kRN;
  if (t_blocks == 0) return cudaSuccess;
  int n_split = 1, per = 1;
  retrieval_split(p.T, p.rows, num_sms, &n_split, &per);
  const size_t smem = r_smem_bytes(MODE == kModeFilter ? p.nb : 0);
  cudaError_t e = ensure_smem_limit(reinterpret_cast<const void*>(retrieval_tc_kernel<MODE, RELU>),
                                    kSlotRetrieval + MODE * 2 + (RELU ? 1 : 0),
                                    r_smem_bytes(MODE == kModeFilter ? kRetrievalMaxBins : 0));
  if (e != cudaSuccess) return e;
  retrieval_tc_kernel<MODE, RELU><<<t_blocks * n_split, kRThreads, smem, stream>>>(
      qm, cm, p, dim / 64, t_blocks, per, ghist);
  count_launches(1);
  return cudaGetLastError();
}

}  // namespace

// Fill the GPU, but give every CTA at least kMinTilesPerCta corpus tiles: the
// threshold can only rise while a scan streams, so ranges must not be tiny.
void retrieval_split(int T, long long rows, int num_sms, int* n_split, int* per) {
  constexpr int kMinTilesPerCta = 64;
  const int t_blocks = (T + kRN - 1) / kRN;
  const int total_tiles = static_cast<int>((rows + kTile - 1) / kTile);
  int ns = t_blocks > 0 ? max(1, num_sms / t_blocks) : 1;
  ns = min(ns, max(1, total_tiles / kMinTilesPerCta));
  const int pr = max(1, (total_tiles + ns - 1) / ns);
  *per = pr;
  *n_split = max(1, (total_tiles + pr - 1) / pr);
}

size_t retrieval_tc_smem_bytes(int mode, int nb) { return r_smem_bytes(mode == kModeFilter ? nb : 0); }

cudaError_t launch_retrieval_tc(int mode, const CUtensorMap& q_map, const CUtensorMap& c_map,
                                const ScoreParams& p, int dim, int relu, int* ghist,
                                int num_sms, cudaStream_t stream) {
  if (mode == kModeDense)
    return relu ? launch_r<kModeDense, true>(q_map, c_map, p, dim, ghist, num_sms, stream)
                : launch_r<kModeDense, false>(q_map, c_map, p, dim, ghist, num_sms, stream);
  return relu ? launch_r<kModeFilter, true>(q_map, c_map, p, dim, ghist, num_sms, stream)
              : launch_r<kModeFilter, false>(q_map, c_map, p, dim, ghist, num_sms, stream);
}

}  // namespace ltk
