// k_select.cu -- the Select stage, the decoupled baseline's selection and the
// overflow rescue.
//
// LiteTopK technical summary, Methodology step 3 "Selection (Finalization)":
// once the scan is over, candidates in bins strictly above the final
// threshold bin go straight to the output, and a standard exact top-k runs
// only over the candidates inside the final threshold bin.
//
// The Filter stage stores the raw fp32 score of every kept candidate, so no
// inverse affine map is needed to recover scores: the output score is the
// kernel's own fp32 score.  Select re-bins the candidate list over its own
// [min, max] range with finer bins; any monotone bin map gives the same exact
// result because the list holds every key whose score reaches the k-th one.
//
// Ordering everywhere is the composite key (score desc, index asc), so ties at
// the k-th score go to the lower key index and the result is unique.
//
// Also here: the decoupled baseline's row radix select (the DSA-style design
// of the summary's Problem Statement: select over a fully materialised score
// row, reading it several times), and the rescue of queries whose candidate
// list overflowed: their full row is recomputed on CUDA cores into a scratch
// row and selected with the same row radix select.
#include <climits>
#include <cmath>

#include "block_sort.cuh"
#include "ltk_internal.cuh"

namespace ltk {
namespace {

constexpr int kSelThreads = 512;
constexpr int kSelThreadsWide = 1024;   // few queries: one wide CTA each
constexpr int kBndCap = 4096;        // boundary-bin entries held in shared memory
constexpr int kRankSelect = 1024;    // boundary bins up to this size: select by rank counting

// Bytes of the output-key buffer for k: the next power of two of k keys, at
// least 1024 (the wide form's register sort holds 1024 keys at least).
__host__ __device__ inline size_t outbuf_bytes(int k) {
  int P = 1;
  while (P < k) P <<= 1;
  if (P < kSelThreadsWide) P = kSelThreadsWide;
  return static_cast<size_t>(P) * sizeof(unsigned long long);
}

// ---------------------------------------------------------------------------
// Block helpers
// ---------------------------------------------------------------------------
__device__ __forceinline__ float block_min(float v, float* red) {
  for (int o = 16; o > 0; o >>= 1) v = fminf(v, __shfl_xor_sync(0xFFFFFFFFu, v, o));
  const int w = threadIdx.x >> 5;
  __syncthreads();
  if ((threadIdx.x & 31) == 0) red[w] = v;
  __syncthreads();
  float r = red[0];
  for (int i = 1; i < (blockDim.x >> 5); ++i) r = fminf(r, red[i]);
  return r;
}
__device__ __forceinline__ float block_max(float v, float* red) {
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xFFFFFFFFu, v, o));
  const int w = threadIdx.x >> 5;
  __syncthreads();
  if ((threadIdx.x & 31) == 0) red[w] = v;
  __syncthreads();
  float r = red[0];
  for (int i = 1; i < (blockDim.x >> 5); ++i) r = fmaxf(r, red[i]);
  return r;
}

// Block-wide exclusive prefix sum of one int per thread (thread order);
// *total gets the sum.  ws: 32 ints of shared scratch.
__device__ __forceinline__ int block_excl_scan(int v, int* ws, int* total) {
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5, nw = blockDim.x >> 5;
  int incl = v;
  for (int o = 1; o < 32; o <<= 1) {
    const int u = __shfl_up_sync(0xFFFFFFFFu, incl, o);
    if (lane >= o) incl += u;
  }
  __syncthreads();
  if (lane == 31) ws[w] = incl;
  __syncthreads();
  if (w == 0) {
    const int x = lane < nw ? ws[lane] : 0;
    int sc = x;
    for (int o = 1; o < 32; o <<= 1) {
      const int u = __shfl_up_sync(0xFFFFFFFFu, sc, o);
      if (lane >= o) sc += u;
    }
    if (lane < nw) ws[lane] = sc - x;
    if (lane == 31) ws[32] = sc;
  }
  __syncthreads();
  *total = ws[32];
  return ws[w] + incl - v;
}

// Descending bitonic sort of P (power of two) 64-bit keys in shared memory.
__device__ void bitonic_desc_u64(unsigned long long* a, int P) {
  for (int size = 2; size <= P; size <<= 1) {
    for (int stride = size >> 1; stride > 0; stride >>= 1) {
      for (int i = threadIdx.x; i < (P >> 1); i += blockDim.x) {
        const int lo = 2 * i - (i & (stride - 1));
        const int hi = lo + stride;
        const bool desc = (lo & size) == 0;
        const unsigned long long x = a[lo], y = a[hi];
        if ((x < y) == desc) {
          a[lo] = y;
          a[hi] = x;
        }
      }
      __syncthreads();
    }
  }
}

// Pick the digit holding the r-th largest: 256-bin histogram, scanned top
// down by warp 0.  Writes (digit, count strictly above it) to sh[0..1].
__device__ __forceinline__ void pick_digit(const unsigned* hist256, long long remaining,
                                           long long* sh) {
  if (threadIdx.x < 32) {
    const int lane = threadIdx.x;
    // lane l owns digits [255 - 8l - 7, 255 - 8l]
    long long seg = 0;
    for (int j = 0; j < 8; ++j) seg += hist256[255 - 8 * lane - j];
    long long cum = seg;
    for (int o = 1; o < 32; o <<= 1) {
      const long long n = __shfl_up_sync(0xFFFFFFFFu, cum, o);
      if (lane >= o) cum += n;
    }
    const unsigned m = __ballot_sync(0xFFFFFFFFu, cum >= remaining);
    const int L = m ? __ffs(m) - 1 : 31;
    if (lane == L) {
      long long above = cum - seg;
      int digit = 255 - 8 * L - 7;
      for (int j = 0; j < 8; ++j) {
        const int d = 255 - 8 * L - j;
        const long long c = hist256[d];
        if (above + c >= remaining) {
          digit = d;
          break;
        }
        above += c;
      }
      sh[0] = digit;
      sh[1] = above;
    }
  }
  __syncthreads();
}

// r-th largest (1-based) of m distinct 64-bit keys in shared memory.
__device__ unsigned long long select_u64_smem(const unsigned long long* keys, int m, int r,
                                              unsigned* hist256, long long* sh) {
  unsigned long long prefix = 0, mask = 0;
  long long remaining = r;
  for (int shift = 56; shift >= 0; shift -= 8) {
    for (int i = threadIdx.x; i < 256; i += blockDim.x) hist256[i] = 0;
    __syncthreads();
    for (int i = threadIdx.x; i < m; i += blockDim.x) {
      const unsigned long long k = keys[i];
      if ((k & mask) == prefix) atomicAdd(&hist256[(k >> shift) & 255u], 1u);
    }
    __syncthreads();
    pick_digit(hist256, remaining, sh);
    prefix |= static_cast<unsigned long long>(sh[0]) << shift;
    mask |= 0xFFull << shift;
    remaining -= sh[1];
    __syncthreads();
  }
  return prefix;
}

// r-th largest composite key among the list entries whose select-bin is `bin`
// (global-memory variant for a boundary bin too large for shared memory).
// A query's retained candidates: one contiguous list of n entries, or (SEG)
// nseg segments of seg_cap entries, each with its own count (cnts, shared
// memory), walked one segment per warp.  Callers only need every entry once,
// in any order.
template <bool SEG>
struct CandList {
  const unsigned long long* base;
  int n;
  const int* cnts;
  int nseg;
  int seg_cap;
  template <typename F>
  __device__ __forceinline__ void for_each(F f) const {
    if constexpr (!SEG) {
      for (int i = threadIdx.x; i < n; i += blockDim.x) f(base[i]);
    } else {
      const int lane = threadIdx.x & 31, w = threadIdx.x >> 5, nw = blockDim.x >> 5;
      for (int sg = w; sg < nseg; sg += nw) {
        const unsigned long long* b = base + static_cast<size_t>(sg) * seg_cap;
        const int c = cnts[sg];
        for (int i = lane; i < c; i += 32) f(b[i]);
      }
    }
  }
};

template <bool SEG>
__device__ unsigned long long select_u64_list(const CandList<SEG>& L, float lo, float delta, int bin, int r,
                                              unsigned* hist256, long long* sh) {
  unsigned long long prefix = 0, mask = 0;
  long long remaining = r;
  for (int shift = 56; shift >= 0; shift -= 8) {
    for (int i = threadIdx.x; i < 256; i += blockDim.x) hist256[i] = 0;
    __syncthreads();
    L.for_each([&](unsigned long long c) {
      const float s = cand_score(c);
      if (bin_of(s, lo, delta, kSelBins) != bin) return;
      const unsigned long long k = ckey(s, cand_idx(c));
      if ((k & mask) == prefix) atomicAdd(&hist256[(k >> shift) & 255u], 1u);
    });
    __syncthreads();
    pick_digit(hist256, remaining, sh);
    prefix |= static_cast<unsigned long long>(sh[0]) << shift;
    mask |= 0xFFull << shift;
    remaining -= sh[1];
    __syncthreads();
  }
  return prefix;
}

__device__ __forceinline__ int visible_of(const int* positions, int t, long long S, int causal) {
  if (!causal || positions == nullptr) return static_cast<int>(S);
  const long long v = static_cast<long long>(positions[t]) + 1;
  return static_cast<int>(v < 0 ? 0 : (v > S ? S : v));
}

// Sort the kk selected keys (buffer padded to P with 0) and write the row.
__device__ void write_sorted(unsigned long long* buf, int kk, int k, int t, int* out_idx,
                             float* out_score) {
  int P = 1;
  while (P < kk) P <<= 1;
  for (int i = kk + threadIdx.x; i < P; i += blockDim.x) buf[i] = 0ull;
  __syncthreads();
  bitonic_desc_u64(buf, P);
  int* oi = out_idx + static_cast<size_t>(t) * k;
  float* os = out_score + static_cast<size_t>(t) * k;
  for (int i = threadIdx.x; i < k; i += blockDim.x) {
    if (i < kk) {
      oi[i] = ckey_idx(buf[i]);
      os[i] = ckey_score(buf[i]);
    } else {
      oi[i] = -1;
      os[i] = -INFINITY;
    }
  }
}

// write_sorted for a 1024-thread CTA: the keys go into registers (slot-major
// loads from buf, conflict-free), a register bitonic sort orders them
// descending, and thread t writes output slots [t E, t E + E).  buf must hold
// at least max(next power of two of kk, 1024) keys.  Larger sorts fall back to
// write_sorted.
template <int E>
__device__ void write_sorted_regs(unsigned long long* buf, int kk, int k, int t, int* out_idx,
                                  float* out_score) {
  const int nt = blockDim.x, tid = threadIdx.x;
  const int P = E * nt;
  for (int i = kk + tid; i < P; i += nt) buf[i] = 0ull;
  __syncthreads();
  unsigned long long v[E];
#pragma unroll
  for (int e = 0; e < E; ++e) v[e] = buf[e * nt + tid];   // any order: the sort follows
  __syncthreads();
  block_sort_regs<E, true>(v, buf);
  int* oi = out_idx + static_cast<size_t>(t) * k;
  float* os = out_score + static_cast<size_t>(t) * k;
#pragma unroll
  for (int e = 0; e < E; ++e) {
    const int i = tid * E + e;
    if (i < k) {
      oi[i] = i < kk ? ckey_idx(v[e]) : -1;
      os[i] = i < kk ? ckey_score(v[e]) : -INFINITY;
    }
  }
  for (int i = P + tid; i < k; i += nt) {
    oi[i] = -1;
    os[i] = -INFINITY;
  }
}

__device__ void write_sorted_wide(unsigned long long* buf, int kk, int k, int t, int* out_idx,
                                  float* out_score) {
  int P = 1;
  while (P < kk) P <<= 1;
  const int nt = blockDim.x;
  const int E = P <= nt ? 1 : P / nt;
  switch (E) {
    case 1: write_sorted_regs<1>(buf, kk, k, t, out_idx, out_score); break;
    case 2: write_sorted_regs<2>(buf, kk, k, t, out_idx, out_score); break;
    case 4: write_sorted_regs<4>(buf, kk, k, t, out_idx, out_score); break;
    case 8: write_sorted_regs<8>(buf, kk, k, t, out_idx, out_score); break;
    default: write_sorted(buf, kk, k, t, out_idx, out_score); break;
  }
}

// Final threshold bin of the select histogram: the highest b with
// count(>= b) >= kk (sh[0]; sh[1] = count strictly above it; sh[0] = 0 with
// everything but bin 0 above when no bin reaches kk), then the output slot
// offsets of the bins above it, highest bin first: hist[b] becomes bin b's
// start offset and cur[b] its cursor.  Bins are split into equal segments,
// segment 0 the highest.
//  * warp-0 form (narrow CTAs, many queries per SM): 32 segments.
//  * block form (wide CTA, few queries): one segment per thread and block scans.
__device__ void theta_and_offsets_warp0(int* hist, int* cur, int kk, int* sh) {
  if (threadIdx.x < 32) {
    const int lane = threadIdx.x;
    const int per = kSelBins / 32;
    const int top = kSelBins - lane * per;
    int seg = 0;
    for (int b = top - per; b < top; ++b) seg += hist[b];
    int cum = seg;
    for (int o = 1; o < 32; o <<= 1) {
      const int v = __shfl_up_sync(0xFFFFFFFFu, cum, o);
      if (lane >= o) cum += v;
    }
    const unsigned m = __ballot_sync(0xFFFFFFFFu, cum >= kk);
    if (m == 0u) {
      if (lane == 31) {
        sh[0] = 0;
        sh[1] = cum - hist[0];
      }
    } else if (lane == __ffs(m) - 1) {
      int above = cum - seg;
      int th = top - per;
      for (int b = top - 1; b >= top - per; --b) {
        if (above + hist[b] >= kk) {
          th = b;
          break;
        }
        above += hist[b];
      }
      sh[0] = th;
      sh[1] = above;
    }
    if (lane == 0) {
      sh[2] = 0;
      sh[3] = 0;
    }
    __syncwarp();
    const int theta_f = sh[0];
    seg = 0;
    for (int b = top - 1; b >= top - per; --b) seg += (b > theta_f) ? hist[b] : 0;
    int incl = seg;
    for (int o = 1; o < 32; o <<= 1) {
      const int v = __shfl_up_sync(0xFFFFFFFFu, incl, o);
      if (lane >= o) incl += v;
    }
    int run = incl - seg;
    for (int b = top - 1; b >= top - per; --b) {
      const int h = (b > theta_f) ? hist[b] : 0;
      hist[b] = run;
      cur[b] = run;
      run += h;
    }
  }
  __syncthreads();
}

__device__ void theta_and_offsets_block(int* hist, int* cur, int kk, int* scan_ws, int* sh) {
  const int per = kSelBins / static_cast<int>(blockDim.x);
  const int top = kSelBins - static_cast<int>(threadIdx.x) * per;
  int seg = 0;
  for (int b = top - per; b < top; ++b) seg += hist[b];
  int total = 0;
  const int above0 = block_excl_scan(seg, scan_ws, &total);
  if (threadIdx.x == 0) {
    sh[0] = 0;
    sh[1] = total - hist[0];
    sh[2] = 0;
    sh[3] = 0;
  }
  __syncthreads();
  if (above0 < kk && above0 + seg >= kk) {
    int above = above0;
    int th = top - per;
    for (int b = top - 1; b >= top - per; --b) {
      if (above + hist[b] >= kk) {
        th = b;
        break;
      }
      above += hist[b];
    }
    sh[0] = th;
    sh[1] = above;
  }
  __syncthreads();
  const int theta_f = sh[0];
  seg = 0;
  for (int b = top - 1; b >= top - per; --b) seg += (b > theta_f) ? hist[b] : 0;
  int run = block_excl_scan(seg, scan_ws, &total);
  for (int b = top - 1; b >= top - per; --b) {
    const int h = (b > theta_f) ? hist[b] : 0;
    hist[b] = run;
    cur[b] = run;
    run += h;
  }
  __syncthreads();
}

// ---------------------------------------------------------------------------
// Select stage (fused path), one CTA per query
// ---------------------------------------------------------------------------
constexpr int kMaxSegs = 256;   // segments per query of a segmented list

template <int THREADS, bool SEG>
__global__ void __launch_bounds__(THREADS) select_kernel(const SelectParams p) {
  extern __shared__ unsigned long long sel_smem[];
  __shared__ int hist[kSelBins];
  __shared__ int cur[kSelBins];
  __shared__ unsigned hist256[256];
  __shared__ long long sh[2];
  __shared__ float red[32];
  __shared__ int scan_ws[33];
  __shared__ int sh_int[4];   // theta_f, c_above, n_out, n_bnd
  __shared__ int seg_s[SEG ? kMaxSegs : 1];

  const int t = blockIdx.x;
  const int V = visible_of(p.positions, t, p.S, p.causal);
  const int kk = min(p.k, V);
  if (threadIdx.x == 0 && p.pairs != nullptr) atomicAdd(p.pairs, static_cast<unsigned long long>(V));
  const int n_raw = p.cnt[t];
  if (n_raw > p.cap) {
    if (threadIdx.x == 0) {
      const int slot = atomicAdd(p.ovf_count, 1);
      p.ovf_list[slot] = t;
    }
    return;
  }
  int P = 1;
  while (P < max(kk, 1)) P <<= 1;
  unsigned long long* outbuf = sel_smem;          // [P]
  unsigned long long* bnd = sel_smem + P;         // [kBndCap]
  const unsigned long long* list = p.cand + static_cast<size_t>(t) * p.cap;
  int n = n_raw;
  if constexpr (SEG) {
    int c = 0;
    for (int i = threadIdx.x; i < p.nseg; i += blockDim.x) {
      seg_s[i] = p.seg_cnt[static_cast<size_t>(t) * p.nseg + i];
      c += seg_s[i];
    }
    int total = 0;
    block_excl_scan(c, scan_ws, &total);
    n = total;
  }
  const CandList<SEG> L{list, n, seg_s, p.nseg, p.seg_cap};
  if (kk == 0 || n == 0) {
    write_sorted(outbuf, 0, p.k, t, p.out_idx, p.out_score);
    return;
  }

  // pass A: range of the retained scores
  float mn = INFINITY, mx = -INFINITY;
  L.for_each([&](unsigned long long c) {
    const float s = cand_score(c);
    mn = fminf(mn, s);
    mx = fmaxf(mx, s);
  });
  const float lo = block_min(mn, red);
  const float hi = block_max(mx, red);
  float delta = 0.f;
  if (hi > lo) {
    delta = __fdiv_rn(static_cast<float>(kSelBins), __fsub_rn(hi, lo));
    if (!(delta <= 1e30f)) delta = 1e30f;
  }

  // pass B: histogram of the retained list
  for (int i = threadIdx.x; i < kSelBins; i += blockDim.x) hist[i] = 0;
  __syncthreads();
  L.for_each([&](unsigned long long c) { atomicAdd(&hist[bin_of(cand_score(c), lo, delta, kSelBins)], 1); });
  __syncthreads();

  // final threshold bin (highest b with count(>= b) >= kk), then the slot
  // offsets of the bins above it (descending prefix sum: bins above theta_f
  // go straight to the output, already ordered by bin; hist becomes the start
  // offsets, cur the cursors)
  if constexpr (THREADS >= kSelThreadsWide)
    theta_and_offsets_block(hist, cur, kk, scan_ws, sh_int);
  else
    theta_and_offsets_warp0(hist, cur, kk, sh_int);
  const int theta_f = sh_int[0];
  const int c_above = min(sh_int[1], kk);
  const int r = kk - c_above;
  L.for_each([&](unsigned long long c) {
    const float s = cand_score(c);
    const int b = bin_of(s, lo, delta, kSelBins);
    if (b > theta_f) {
      const int slot = atomicAdd(&cur[b], 1);
      if (slot < kk) outbuf[slot] = ckey(s, cand_idx(c));
    } else if (b == theta_f) {
      const int slot = atomicAdd(&sh_int[3], 1);
      if (slot < kBndCap) bnd[slot] = ckey(s, cand_idx(c));
    }
  });
  __syncthreads();
  const int m_bnd = sh_int[3];

  // Order inside each bin above theta_f: a bin holds few entries, so one
  // thread insertion-sorts its bins' ranges; if some bin is crowded (heavy
  // ties), the whole output is sorted at the end instead.
  bool crowded = false;
  for (int b = threadIdx.x; b < kSelBins; b += blockDim.x) {
    if (b <= theta_f) continue;
    const int a0 = hist[b], a1 = min(cur[b], kk);
    if (a1 - a0 > 32) {
      crowded = true;
      continue;
    }
    for (int i = a0 + 1; i < a1; ++i) {
      const unsigned long long x = outbuf[i];
      int j = i - 1;
      while (j >= a0 && outbuf[j] < x) {
        outbuf[j + 1] = outbuf[j];
        --j;
      }
      outbuf[j + 1] = x;
    }
  }
  const bool need_full_sort = __syncthreads_or(crowded ? 1 : 0) != 0;

  // exact top-r inside the boundary bin, placed after the c_above entries
  if (r > 0) {
    if (m_bnd <= kRankSelect) {
      // the rank of each boundary key among the boundary keys is its output slot
      for (int i = threadIdx.x; i < m_bnd; i += blockDim.x) {
        const unsigned long long x = bnd[i];
        int rank = 0;
        for (int j = 0; j < m_bnd; ++j) rank += bnd[j] > x ? 1 : 0;
        if (rank < r) outbuf[c_above + rank] = x;
      }
    } else {
      if (threadIdx.x == 0) sh_int[2] = c_above;
      __syncthreads();
      unsigned long long kth;
      if (m_bnd <= kBndCap) {
        kth = select_u64_smem(bnd, m_bnd, r, hist256, sh);
        for (int i = threadIdx.x; i < m_bnd; i += blockDim.x)
          if (bnd[i] >= kth) {
            const int slot = atomicAdd(&sh_int[2], 1);
            if (slot < kk) outbuf[slot] = bnd[i];
          }
      } else {
        kth = select_u64_list(L, lo, delta, theta_f, r, hist256, sh);
        L.for_each([&](unsigned long long c) {
          const float s = cand_score(c);
          if (bin_of(s, lo, delta, kSelBins) != theta_f) return;
          const unsigned long long key = ckey(s, cand_idx(c));
          if (key >= kth) {
            const int slot = atomicAdd(&sh_int[2], 1);
            if (slot < kk) outbuf[slot] = key;
          }
        });
      }
    }
  }
  __syncthreads();
  // a large boundary bin was selected unordered: sort the whole output
  if (need_full_sort || (r > 0 && m_bnd > kRankSelect)) {
    if constexpr (THREADS >= kSelThreadsWide)
      write_sorted_wide(outbuf, kk, p.k, t, p.out_idx, p.out_score);
    else
      write_sorted(outbuf, kk, p.k, t, p.out_idx, p.out_score);
  } else {
    int* oi = p.out_idx + static_cast<size_t>(t) * p.k;
    float* os = p.out_score + static_cast<size_t>(t) * p.k;
    for (int i = threadIdx.x; i < p.k; i += blockDim.x) {
      if (i < kk) {
        oi[i] = ckey_idx(outbuf[i]);
        os[i] = ckey_score(outbuf[i]);
      } else {
        oi[i] = -1;
        os[i] = -INFINITY;
      }
    }
  }
}

// ---------------------------------------------------------------------------
// Row top-k over a materialised score row (decoupled baseline and rescue)
// ---------------------------------------------------------------------------
// Bucket select over the value range, three reads of the row: (1) the row's
// minimum and maximum; (2) a histogram of kRowBins equal-width bins over
// [min, max] (the same monotone bin map as the Filter stage), which spreads
// even concentrated scores over many bins, so plain shared-memory atomics
// rarely collide; the bin holding the k-th score follows from a top-down scan;
// (3) every score in a higher bin goes straight to the output, and the entries
// of that bin are gathered, as (score, index) keys, into shared memory, where
// the exact top of the bin is selected (ties to the lower index: the keys
// order by score, then index).  A bin too crowded for shared memory (many
// equal scores, or no spread) falls back to an 8-bit radix select over the
// scores' order-preserving codes and an ordered collection of the ties.
constexpr int kRowBins = 2048;
constexpr int kRowCandCap = 4096;      // boundary-bin entries gathered in shared memory

__device__ void row_topk_radix(const float* row, int V, int kk, int k, int t, int* out_idx,
                               float* out_score, unsigned long long* outbuf, unsigned* hist256,
                               long long* sh, int* sh_int) {
  if (kk <= 0) {
    write_sorted(outbuf, 0, k, t, out_idx, out_score);
    return;
  }
  uint32_t prefix = 0, mask = 0;
  long long remaining = kk;
  const bool vec = (reinterpret_cast<uintptr_t>(row) & 15u) == 0;
  for (int shift = 24; shift >= 0; shift -= 8) {
    for (int i = threadIdx.x; i < 256; i += blockDim.x) hist256[i] = 0;
    __syncthreads();
    if (vec) {
      const int nv = V >> 2;
      const float4* r4 = reinterpret_cast<const float4*>(row);
      for (int i = threadIdx.x; i < nv; i += blockDim.x) {
        const float4 x = r4[i];
        const float xs[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const uint32_t o = ord_f32(xs[j]);
          if ((o & mask) == prefix) atomicAdd(&hist256[(o >> shift) & 255u], 1u);
        }
      }
      for (int i = (nv << 2) + threadIdx.x; i < V; i += blockDim.x) {
        const uint32_t o = ord_f32(row[i]);
        if ((o & mask) == prefix) atomicAdd(&hist256[(o >> shift) & 255u], 1u);
      }
    } else {
      for (int i = threadIdx.x; i < V; i += blockDim.x) {
        const uint32_t o = ord_f32(row[i]);
        if ((o & mask) == prefix) atomicAdd(&hist256[(o >> shift) & 255u], 1u);
      }
    }
    __syncthreads();
    pick_digit(hist256, remaining, sh);
    prefix |= static_cast<uint32_t>(sh[0]) << shift;
    mask |= 0xFFu << shift;
    remaining -= sh[1];
    __syncthreads();
  }
  const uint32_t kth = prefix;
  const int need_ties = static_cast<int>(remaining);   // entries equal to kth to keep
  if (threadIdx.x == 0) {
    sh_int[0] = 0;   // output slot
    sh_int[1] = 0;   // ties taken so far
  }
  __syncthreads();
  // scores strictly above the k-th: anywhere in the row
  for (int i = threadIdx.x; i < V; i += blockDim.x) {
    const float s = row[i];
    if (ord_f32(s) > kth) {
      const int slot = atomicAdd(&sh_int[0], 1);
      if (slot < kk) outbuf[slot] = ckey(s, i);
    }
  }
  __syncthreads();
  // ties at the k-th score: lowest indices first (ordered chunks)
  __shared__ int warp_cnt[kSelThreads / 32];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
  for (int base = 0; base < V; base += blockDim.x) {
    if (sh_int[1] >= need_ties) break;
    const int i = base + threadIdx.x;
    const bool tie = i < V && ord_f32(row[i]) == kth;
    const unsigned m = __ballot_sync(0xFFFFFFFFu, tie);
    if (lane == 0) warp_cnt[warp] = __popc(m);
    __syncthreads();
    int before = 0, total = 0;
    for (int w = 0; w < nw; ++w) {
      if (w < warp) before += warp_cnt[w];
      total += warp_cnt[w];
    }
    const int rank = sh_int[1] + before + __popc(m & ((1u << lane) - 1u));
    if (tie && rank < need_ties) {
      const int slot = atomicAdd(&sh_int[0], 1);
      if (slot < kk) outbuf[slot] = ckey(row[i], i);
    }
    __syncthreads();
    if (threadIdx.x == 0) sh_int[1] += total;
    __syncthreads();
  }
  __syncthreads();
  write_sorted(outbuf, min(sh_int[0], kk), k, t, out_idx, out_score);
}

// Digit d of an nb-bin histogram (nb a multiple of the block size) with
// count(bins > d) < remaining <= count(bins >= d): sh[0] = d,
// sh[1] = count(bins > d).  Top-down block scan.
__device__ void pick_digit_block(const unsigned* hist, int nb, long long remaining, long long* sh,
                                 long long* warp_sums) {
  const int per = nb / static_cast<int>(blockDim.x);
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  // thread i owns bins nb-1-(per*i) .. nb-per*(i+1), counted from the top
  long long own = 0;
  for (int r = 0; r < per; ++r) own += hist[nb - 1 - per * threadIdx.x - r];
  long long cum = own;
  for (int o = 1; o < 32; o <<= 1) {
    const long long n = __shfl_up_sync(0xFFFFFFFFu, cum, o);
    if (lane >= o) cum += n;
  }
  if (lane == 31) warp_sums[warp] = cum;
  __syncthreads();
  long long before = 0;
  for (int w = 0; w < warp; ++w) before += warp_sums[w];
  cum += before;
  const long long excl = cum - own;
  if (excl < remaining && cum >= remaining) {
    long long above = excl;
    int digit = nb - per * (static_cast<int>(threadIdx.x) + 1);
    for (int r = 0; r < per; ++r) {
      const int d = nb - 1 - per * threadIdx.x - r;
      const long long c = hist[d];
      if (above + c >= remaining) {
        digit = d;
        break;
      }
      above += c;
    }
    sh[0] = digit;
    sh[1] = above;
  }
  __syncthreads();
}

// Warp-aggregated slot reservation: every lane calls it; returns the slot of
// a lane with take (-1 otherwise) from the shared counter ctr.
__device__ __forceinline__ int reserve_slot(int* ctr, bool take) {
  const unsigned m = __ballot_sync(0xFFFFFFFFu, take);
  if (m == 0) return -1;
  const int lane = threadIdx.x & 31;
  const int leader = __ffs(m) - 1;
  int base = 0;
  if (lane == leader) base = atomicAdd(ctr, __popc(m));
  base = __shfl_sync(0xFFFFFFFFu, base, leader);
  return take ? base + __popc(m & ((1u << lane) - 1u)) : -1;
}

__device__ void row_topk_block(const float* row, int V, int kk, int k, int t, int* out_idx,
                               float* out_score, unsigned long long* outbuf,
                               unsigned long long* cand, unsigned* hist, unsigned* hist256,
                               long long* sh, long long* warp_sums, int* sh_int, float* red) {
  if (kk <= 0) {
    write_sorted(outbuf, 0, k, t, out_idx, out_score);
    return;
  }
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
  const bool vec = (reinterpret_cast<uintptr_t>(row) & 15u) == 0;
  const int nv = vec ? (V >> 2) : 0;   // float4 part; the rest one by one
  const float4* r4 = reinterpret_cast<const float4*>(row);
  // (1) range of the row (four float4 loads in flight per thread)
  float lo = INFINITY, hi = -INFINITY;
  {
    const int step = blockDim.x;
    int i = threadIdx.x;
    for (; i + 3 * step < nv; i += 4 * step) {
      const float4 x0 = __ldcs(r4 + i), x1 = __ldcs(r4 + i + step);
      const float4 x2 = __ldcs(r4 + i + 2 * step), x3 = __ldcs(r4 + i + 3 * step);
      lo = fminf(lo, fminf(fminf(fminf(x0.x, x0.y), fminf(x0.z, x0.w)), fminf(fminf(x1.x, x1.y), fminf(x1.z, x1.w))));
      lo = fminf(lo, fminf(fminf(fminf(x2.x, x2.y), fminf(x2.z, x2.w)), fminf(fminf(x3.x, x3.y), fminf(x3.z, x3.w))));
      hi = fmaxf(hi, fmaxf(fmaxf(fmaxf(x0.x, x0.y), fmaxf(x0.z, x0.w)), fmaxf(fmaxf(x1.x, x1.y), fmaxf(x1.z, x1.w))));
      hi = fmaxf(hi, fmaxf(fmaxf(fmaxf(x2.x, x2.y), fmaxf(x2.z, x2.w)), fmaxf(fmaxf(x3.x, x3.y), fmaxf(x3.z, x3.w))));
    }
    for (; i < nv; i += step) {
      const float4 x = __ldcs(r4 + i);
      lo = fminf(fminf(lo, x.x), fminf(x.y, fminf(x.z, x.w)));
      hi = fmaxf(fmaxf(hi, x.x), fmaxf(x.y, fmaxf(x.z, x.w)));
    }
  }
  for (int i = (nv << 2) + threadIdx.x; i < V; i += blockDim.x) {
    const float x = row[i];
    lo = fminf(lo, x);
    hi = fmaxf(hi, x);
  }
  lo = block_min(lo, red);
  hi = block_max(hi, red);
  const float span = __fsub_rn(hi, lo);
  float scale = span > 0.f ? __fdiv_rn(static_cast<float>(kRowBins), span) : 0.f;
  if (!(scale <= 1e30f)) scale = 1e30f;
  // (2) histogram of the equal-width bins (two float4 loads in flight per thread)
  for (int i = threadIdx.x; i < kRowBins; i += blockDim.x) hist[i] = 0;
  __syncthreads();
  {
    const int step = blockDim.x;
    int i = threadIdx.x;
    for (; i + step < nv; i += 2 * step) {
      const float4 x0 = __ldcs(r4 + i), x1 = __ldcs(r4 + i + step);
      atomicAdd(&hist[bin_of(x0.x, lo, scale, kRowBins)], 1u);
      atomicAdd(&hist[bin_of(x0.y, lo, scale, kRowBins)], 1u);
      atomicAdd(&hist[bin_of(x0.z, lo, scale, kRowBins)], 1u);
      atomicAdd(&hist[bin_of(x0.w, lo, scale, kRowBins)], 1u);
      atomicAdd(&hist[bin_of(x1.x, lo, scale, kRowBins)], 1u);
      atomicAdd(&hist[bin_of(x1.y, lo, scale, kRowBins)], 1u);
      atomicAdd(&hist[bin_of(x1.z, lo, scale, kRowBins)], 1u);
      atomicAdd(&hist[bin_of(x1.w, lo, scale, kRowBins)], 1u);
    }
    for (; i < nv; i += step) {
      const float4 x = __ldcs(r4 + i);
      atomicAdd(&hist[bin_of(x.x, lo, scale, kRowBins)], 1u);
      atomicAdd(&hist[bin_of(x.y, lo, scale, kRowBins)], 1u);
      atomicAdd(&hist[bin_of(x.z, lo, scale, kRowBins)], 1u);
      atomicAdd(&hist[bin_of(x.w, lo, scale, kRowBins)], 1u);
    }
  }
  for (int i = (nv << 2) + threadIdx.x; i < V; i += blockDim.x)
    atomicAdd(&hist[bin_of(row[i], lo, scale, kRowBins)], 1u);
  __syncthreads();
  pick_digit_block(hist, kRowBins, kk, sh, warp_sums);
  const int bstar = static_cast<int>(sh[0]);
  const int need = kk - static_cast<int>(sh[1]);   // entries taken from bin bstar (>= 1)
  const unsigned in_bin = hist[bstar];
  __syncthreads();
  if (in_bin > static_cast<unsigned>(kRowCandCap)) {
    row_topk_radix(row, V, kk, k, t, out_idx, out_score, outbuf, hist256, sh, sh_int);
    return;
  }
  if (threadIdx.x == 0) {
    sh_int[0] = 0;   // output slots
    sh_int[1] = 0;   // gathered bin entries
  }
  __syncthreads();
  // (3) higher bins -> output; bin bstar -> shared memory.  A float4 whose
  // largest score is below tau (the smallest score whose bin reaches bstar,
  // found by bisection over the fp32 order: the same decision as the bin
  // test) needs no further work, and a warp skips on one vote.
  if (threadIdx.x == 0) {
    // over the row's own range [lo, hi] (finite, and bin_of(hi) is the top bin)
    uint32_t a = ord_f32(lo), b = ord_f32(hi);   // invariant: bin_of(unord(b)) >= bstar
    while (a < b) {
      const uint32_t mid = a + (b - a) / 2;
      if (bin_of(unord_f32(mid), lo, scale, kRowBins) >= bstar) b = mid; else a = mid + 1;
    }
    sh_int[2] = static_cast<int>(a);
  }
  __syncthreads();
  const uint32_t tau_ord = static_cast<uint32_t>(sh_int[2]);
  auto take_one = [&](float sv, int i, bool ok) {
    const int b = bin_of(sv, lo, scale, kRowBins);
    const int so = reserve_slot(&sh_int[0], ok && b > bstar);
    if (so >= 0 && so < kk) outbuf[so] = ckey(sv, i);
    const int sc = reserve_slot(&sh_int[1], ok && b == bstar);
    if (sc >= 0 && sc < kRowCandCap) cand[sc] = ckey(sv, i);
  };
  for (int base = warp * 32; base < nv; base += nw * 32) {
    const int i4 = base + lane;
    const bool ok = i4 < nv;
    const float4 x = ok ? __ldcs(r4 + i4) : make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
    const float mx = fmaxf(fmaxf(x.x, x.y), fmaxf(x.z, x.w));
    if (!__any_sync(0xFFFFFFFFu, ok && ord_f32(mx) >= tau_ord)) continue;
    take_one(x.x, 4 * i4 + 0, ok);
    take_one(x.y, 4 * i4 + 1, ok);
    take_one(x.z, 4 * i4 + 2, ok);
    take_one(x.w, 4 * i4 + 3, ok);
  }
  for (int base = (nv << 2) + warp * 32; base < V; base += nw * 32) {   // the rest, one by one
    const int i = base + lane;
    const bool ok = i < V;
    take_one(ok ? row[i] : 0.f, i, ok);
  }
  __syncthreads();
  const int m = min(sh_int[1], kRowCandCap);
  unsigned long long kth_key = 0ull;
  if (need < m) kth_key = select_u64_smem(cand, m, need, hist256, sh);
  __syncthreads();
  for (int base = 0; base < m; base += blockDim.x) {
    const int j = base + threadIdx.x;
    const bool take = j < m && (need >= m || cand[j] >= kth_key);
    const int so = reserve_slot(&sh_int[0], take);
    if (so >= 0 && so < kk) outbuf[so] = cand[j];
  }
  __syncthreads();
  write_sorted(outbuf, min(sh_int[0], kk), k, t, out_idx, out_score);
}

__global__ void __launch_bounds__(kSelThreads, 2) row_topk_kernel(const RowTopkParams p) {
  extern __shared__ unsigned long long rt_smem[];   // [outbuf keys][kRowCandCap bin entries]
  __shared__ unsigned hist[kRowBins];
  __shared__ unsigned hist256[256];
  __shared__ long long sh[2];
  __shared__ long long warp_sums[kSelThreads / 32];
  __shared__ int sh_int[3];
  __shared__ float red[kSelThreads / 32];
  const int t = blockIdx.x;
  const int V = visible_of(p.positions, t, p.S, p.causal);
  const int kk = min(p.k, V);
  if (threadIdx.x == 0 && p.pairs != nullptr) atomicAdd(p.pairs, static_cast<unsigned long long>(V));
  unsigned long long* cand = rt_smem + outbuf_bytes(p.k) / sizeof(unsigned long long);
  row_topk_block(p.rows + static_cast<size_t>(t) * p.ld, V, kk, p.k, t, p.out_idx, p.out_score,
                 rt_smem, cand, hist, hist256, sh, warp_sums, sh_int, red);
}

// ---------------------------------------------------------------------------
// Overflow rescue: CUDA-core recompute of a full score row, then row top-k
// ---------------------------------------------------------------------------
__device__ __forceinline__ float e4m3_value(uint32_t c) {
  // OCP fp8 E4M3: sign, 4-bit exponent (bias 7), 3-bit mantissa; exponent 0
  // is subnormal (m * 2^-9).  NaN codes do not occur in valid inputs.
  const uint32_t sgn = (c & 0x80u) << 24;
  const uint32_t e = (c >> 3) & 0xFu;
  const uint32_t m = c & 0x7u;
  float v;
  if (e == 0) {
    v = static_cast<float>(m) * 0.001953125f;   // exact: m * 2^-9
  } else {
    v = __uint_as_float(((e + 120u) << 23) | (m << 20));
  }
  return __uint_as_float(__float_as_uint(v) | sgn);
}

constexpr int kRescueThreads = 256;

// One head (vector retrieval): I[s] = w[t] * f(q[t] . c[s]), f = ReLU or identity.
__device__ void rescue_row_scores_one_head(const RescueParams& p, int t, int V, float* row,
                                           float* qf) {
  const int d = p.dim;
  const uint16_t* q = static_cast<const uint16_t*>(p.q) + static_cast<size_t>(t) * d;
  for (int i = threadIdx.x; i < d; i += blockDim.x) qf[i] = __uint_as_float(static_cast<uint32_t>(q[i]) << 16);
  const float wt = p.w[t];
  __syncthreads();
  for (int s = threadIdx.x; s < V; s += blockDim.x) {
    const uint4* src = reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(p.k_cache) +
                                                      static_cast<size_t>(s) * d);
    float acc = 0.f;
    for (int v8 = 0; v8 < d / 8; ++v8) {
      const uint4 r = src[v8];
      const uint32_t w4[4] = {r.x, r.y, r.z, r.w};
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        acc = __fmaf_rn(qf[8 * v8 + 2 * j], __uint_as_float(w4[j] << 16), acc);
        acc = __fmaf_rn(qf[8 * v8 + 2 * j + 1], __uint_as_float(w4[j] & 0xFFFF0000u), acc);
      }
    }
    row[s] = __fmul_rn(p.relu ? fmaxf(acc, 0.f) : acc, wt);
  }
  __syncthreads();
}

// Any head count and dimension (the CUDA-core engine's shapes): one thread per
// key, heads one after another, the key row re-read from cache per head.
__device__ void rescue_row_scores_generic(const RescueParams& p, int t, int V, float* row,
                                          float* qf, float* wf) {
  const int H = p.heads, d = p.dim;
  const size_t qoff = static_cast<size_t>(t) * H * d;
  for (int i = threadIdx.x; i < H * d; i += blockDim.x) {
    qf[i] = p.fp8 ? e4m3_value(static_cast<const uint8_t*>(p.q)[qoff + i])
                  : __uint_as_float(static_cast<uint32_t>(static_cast<const uint16_t*>(p.q)[qoff + i]) << 16);
  }
  for (int h = threadIdx.x; h < H; h += blockDim.x) {
    float wv = p.w[static_cast<size_t>(t) * H + h];
    if (p.fp8) wv = __fmul_rn(wv, p.q_scale[t]);
    wf[h] = wv;
  }
  __syncthreads();
  for (int s = threadIdx.x; s < V; s += blockDim.x) {
    float I = 0.f;
    for (int h = 0; h < H; ++h) {
      const float* qh = qf + h * d;
      float acc = 0.f;
      for (int i = 0; i < d; ++i) {
        const float kv = p.fp8 ? e4m3_value(static_cast<const uint8_t*>(p.k_cache)[static_cast<size_t>(s) * d + i])
                               : __uint_as_float(static_cast<uint32_t>(static_cast<const uint16_t*>(
                                     p.k_cache)[static_cast<size_t>(s) * d + i]) << 16);
        acc = __fmaf_rn(qh[i], kv, acc);
      }
      I = __fmaf_rn(p.relu ? fmaxf(acc, 0.f) : acc, wf[h], I);
    }
    if (p.fp8) I = __fmul_rn(I, p.k_scale[s]);
    row[s] = I;
  }
  __syncthreads();
}

__device__ void rescue_row_scores(const RescueParams& p, int t, int V, float* row, float* qf,
                                  float* wf) {
  if (p.heads == 1 && !p.fp8) {
    rescue_row_scores_one_head(p, t, V, row, qf);
    return;
  }
  if (p.heads != kTcHeads || p.dim != kTcDim) {
    rescue_row_scores_generic(p, t, V, row, qf, wf);
    return;
  }
  const int H = kTcHeads, d = kTcDim;
  const size_t qoff = static_cast<size_t>(t) * H * d;
  for (int i = threadIdx.x; i < H * d; i += blockDim.x) {
    float v;
    if (p.fp8) {
      v = e4m3_value(static_cast<const uint8_t*>(p.q)[qoff + i]);
    } else {
      const uint16_t b = static_cast<const uint16_t*>(p.q)[qoff + i];
      v = __uint_as_float(static_cast<uint32_t>(b) << 16);
    }
    qf[i] = v;
  }
  for (int h = threadIdx.x; h < H; h += blockDim.x) {
    float wv = p.w[static_cast<size_t>(t) * H + h];
    if (p.fp8) wv = __fmul_rn(wv, p.q_scale[t]);
    wf[h] = wv;
  }
  __syncthreads();
  for (int s = threadIdx.x; s < V; s += blockDim.x) {
    float acc[kTcHeads];
#pragma unroll
    for (int h = 0; h < kTcHeads; ++h) acc[h] = 0.f;
    for (int dc = 0; dc < d; dc += 16) {
      float kv[16];
      if (p.fp8) {
        const uint4 raw = *reinterpret_cast<const uint4*>(static_cast<const uint8_t*>(p.k_cache) +
                                                           static_cast<size_t>(s) * d + dc);
        const uint32_t w4[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
        for (int j = 0; j < 16; ++j) kv[j] = e4m3_value((w4[j >> 2] >> (8 * (j & 3))) & 0xFFu);
      } else {
        const uint4* src = reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(p.k_cache) +
                                                          static_cast<size_t>(s) * d + dc);
        const uint4 r0 = src[0], r1 = src[1];
        const uint32_t w8[8] = {r0.x, r0.y, r0.z, r0.w, r1.x, r1.y, r1.z, r1.w};
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          kv[2 * j] = __uint_as_float(w8[j] << 16);
          kv[2 * j + 1] = __uint_as_float(w8[j] & 0xFFFF0000u);
        }
      }
#pragma unroll
      for (int h = 0; h < kTcHeads; ++h) {
        const float* qh = qf + h * d + dc;
        float a = acc[h];
#pragma unroll
        for (int j = 0; j < 16; ++j) a = __fmaf_rn(qh[j], kv[j], a);
        acc[h] = a;
      }
    }
    float I = 0.f;
#pragma unroll
    for (int h = 0; h < kTcHeads; ++h) I = __fmaf_rn(p.relu ? fmaxf(acc[h], 0.f) : acc[h], wf[h], I);
    if (p.fp8) I = __fmul_rn(I, p.k_scale[s]);
    row[s] = I;
  }
  __syncthreads();
}

__global__ void __launch_bounds__(kRescueThreads) rescue_kernel(const RescueParams p) {
  extern __shared__ unsigned long long rs_smem[];
  __shared__ unsigned hist[kRowBins];
  __shared__ unsigned hist256[256];
  __shared__ long long sh[2];
  __shared__ long long warp_sums[kRescueThreads / 32];
  __shared__ int sh_int[3];
  __shared__ float red[kRescueThreads / 32];
  __shared__ int s_slot;
  __shared__ float wf[128];
  float* qf = reinterpret_cast<float*>(rs_smem);   // [H*d] fp32, reused as output buffer later
  float* row = p.scratch + static_cast<size_t>(blockIdx.x) * p.scratch_ld;
  while (true) {
    if (threadIdx.x == 0) s_slot = atomicAdd(p.ovf_next, 1);
    __syncthreads();
    const int slot = s_slot;
    __syncthreads();
    if (slot >= *p.ovf_count) break;
    const int t = p.ovf_list[slot];
    const int V = visible_of(p.positions, t, p.S, p.causal);
    const int kk = min(p.k, V);
    rescue_row_scores(p, t, V, row, qf, wf);
    row_topk_block(row, V, kk, p.k, t, p.out_idx, p.out_score, rs_smem,
                   rs_smem + outbuf_bytes(p.k) / sizeof(unsigned long long), hist, hist256, sh,
                   warp_sums, sh_int, red);
    __syncthreads();
  }
}


}  // namespace

template <int THREADS, bool SEG>
cudaError_t launch_select_as(const SelectParams& p, int slot, cudaStream_t stream) {
  const size_t smem = outbuf_bytes(p.k) + kBndCap * sizeof(unsigned long long);
  const size_t smem_max = outbuf_bytes(kMaxK) + kBndCap * sizeof(unsigned long long);
  cudaError_t e = ensure_smem_limit(reinterpret_cast<const void*>(select_kernel<THREADS, SEG>), slot, smem_max);
  if (e != cudaSuccess) return e;
  select_kernel<THREADS, SEG><<<p.T, THREADS, smem, stream>>>(p);
  count_launches(1);
  return cudaGetLastError();
}

cudaError_t launch_select(const SelectParams& p, int num_sms, cudaStream_t stream) {
  if (p.T <= 0) return cudaSuccess;
  if (p.seg_cnt != nullptr && (p.nseg < 1 || p.nseg > kMaxSegs)) return cudaErrorInvalidValue;
  // one wide CTA per query when there are few queries (the per-query work is
  // latency-bound) or when k is large (the output buffer then allows one CTA
  // per SM anyway, and the wide form sorts in registers)
  const bool wide = p.T < num_sms || p.k > 2048;
  if (p.seg_cnt != nullptr)
    return wide ? launch_select_as<kSelThreadsWide, true>(p, kSlotSelectSegWide, stream)
                : launch_select_as<kSelThreads, true>(p, kSlotSelectSeg, stream);
  return wide ? launch_select_as<kSelThreadsWide, false>(p, kSlotSelectWide, stream)
              : launch_select_as<kSelThreads, false>(p, kSlotSelect, stream);
}

cudaError_t launch_row_topk(const RowTopkParams& p, cudaStream_t stream) {
  if (p.T <= 0) return cudaSuccess;
  const size_t cand_bytes = kRowCandCap * sizeof(unsigned long long);
  const size_t smem = outbuf_bytes(p.k) + cand_bytes;
  cudaError_t e = ensure_smem_limit(reinterpret_cast<const void*>(row_topk_kernel), kSlotRowTopk,
                                    outbuf_bytes(kMaxK) + cand_bytes);
  if (e != cudaSuccess) return e;
  row_topk_kernel<<<p.T, kSelThreads, smem, stream>>>(p);
  count_launches(1);
  return cudaGetLastError();
}

cudaError_t launch_rescue(const RescueParams& p, int rescue_rows, cudaStream_t stream) {
  if (p.T <= 0 || rescue_rows <= 0) return cudaSuccess;
  const size_t qbytes = static_cast<size_t>(p.heads) * p.dim * sizeof(float);
  const size_t cand_bytes = kRowCandCap * sizeof(unsigned long long);
  const size_t sel = outbuf_bytes(p.k) + cand_bytes;
  const size_t smem = qbytes > sel ? qbytes : sel;
  const size_t sel_max = outbuf_bytes(kMaxK) + cand_bytes;
  const size_t mx = kCcMaxSmem > sel_max ? kCcMaxSmem : sel_max;
  cudaError_t e = ensure_smem_limit(reinterpret_cast<const void*>(rescue_kernel), kSlotRescue, mx);
  if (e != cudaSuccess) return e;
  rescue_kernel<<<rescue_rows, kRescueThreads, smem, stream>>>(p);
  count_launches(1);
  return cudaGetLastError();
}

}  // namespace ltk
