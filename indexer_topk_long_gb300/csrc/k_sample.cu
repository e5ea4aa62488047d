// k_sample.cu -- the Sample stage (LiteTopK technical summary, Methodology
// step 1 "Sampling (Initialization)").
//
// The summary's Sample stage scores a small set of keys -- the top-k' tokens of
// the previous chunk's results, k' = 3k, instead of a random sample -- to
// estimate each query's score range [s_min, s_max], splits that range into
// equal-width bins, and starts the threshold at the bin holding the sample's
// k-th largest score.  This file provides:
//   * random_sample    -- seeded stratified sample for a first chunk;
//   * make_sample      -- previous-chunk sample: key ids ranked by how many of
//                         the previous chunk's queries selected them;
//   * prepare_sample   -- drops out-of-range and duplicate ids (a duplicate
//                         would count one key twice in the sample's k-th score
//                         and could lift the threshold above the true one):
//                         the ids mark a bitmap of the key range, whose set
//                         bits are listed in ascending order;
//   * gather_keys      -- copies the sample's key rows into a dense tile;
//   * sample_stats     -- per query: s_min, s_max, delta and the initial
//                         threshold bin from the scored sample.
// The sample's scores themselves come from the tensor-core scorer in dense
// mode over the gathered rows, i.e. the same arithmetic as the Filter scan.
#include <climits>
#include <cmath>

#include "ltk_internal.cuh"

namespace ltk {
namespace {

// SplitMix64 finaliser (Steele, Lea, Flood, "Fast splittable pseudorandom
// number generators", OOPSLA 2014): a counter-based 64-bit mixer.
__device__ __forceinline__ uint64_t splitmix64(uint64_t x) {
  x += 0x9E3779B97F4A7C15ull;
  x = (x ^ (x >> 30)) * 0xBF58476D1CE4E5B9ull;
  x = (x ^ (x >> 27)) * 0x94D049BB133111EBull;
  return x ^ (x >> 31);
}

// Bijection of [0, 2^31): xor with a seed, odd multiply mod 2^31, xorshift.
__device__ __forceinline__ uint32_t perm31(uint32_t x, uint64_t seed) {
  x ^= static_cast<uint32_t>(seed) & 0x7FFFFFFFu;
  x = (x * 0x2545F491u) & 0x7FFFFFFFu;
  x ^= x >> 15;
  x = (x * 0x6C8E9CF5u) & 0x7FFFFFFFu;
  x ^= x >> 13;
  return x;
}

// One id per stratum [floor(i*S/n), floor((i+1)*S/n)): distinct by
// construction and spread over the whole cache.
__global__ void random_sample_kernel(long long S, int n, unsigned long long seed, int* out) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= n) return;
  const long long lo = static_cast<long long>(i) * S / n;
  const long long hi = static_cast<long long>(i + 1) * S / n;
  const long long span = hi - lo;
  const uint64_t r = splitmix64(seed ^ (0xD1B54A32D192ED03ull * static_cast<uint64_t>(i + 1)));
  out[i] = static_cast<int>(lo + (span > 0 ? static_cast<long long>(r % static_cast<uint64_t>(span)) : 0));
}

// Set the bit of every valid id (the bitmap is all clear on entry).
__global__ void mark_ids_kernel(const int* __restrict__ ids, int n, long long S, uint32_t* bitmap) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= n) return;
  const int x = ids[i];
  if (x >= 0 && static_cast<long long>(x) < S) atomicOr(&bitmap[x >> 5], 1u << (x & 31));
}

// The set bits, in ascending order, become the sample's distinct key ids; the
// tail up to n_pad gets INT_MAX ("no key"); every word read is cleared for the
// next call.  CTA g owns words [g * 1024, (g + 1) * 1024), four per thread:
// count_bits sums each CTA's bits, list_bits offsets each CTA by the sums of
// the CTAs before it and each thread by a block scan.
constexpr int kCompactThreads = 256;
constexpr int kWordsPerCta = 4 * kCompactThreads;

__device__ __forceinline__ int block_sum(int v, int* ws) {
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, o);
  __syncthreads();
  if ((threadIdx.x & 31) == 0) ws[threadIdx.x >> 5] = v;
  __syncthreads();
  int r = 0;
  for (int i = 0; i < static_cast<int>(blockDim.x >> 5); ++i) r += ws[i];
  return r;
}

__global__ void fill_ids_kernel(int* key_ids_pad, int n_pad) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i < n_pad) key_ids_pad[i] = INT_MAX;
}

__global__ void __launch_bounds__(kCompactThreads) count_bits_kernel(const uint32_t* __restrict__ bitmap,
                                                                     long long words, int* block_sums) {
  __shared__ int ws[kCompactThreads / 32];
  const long long w0 = static_cast<long long>(blockIdx.x) * kWordsPerCta + 4 * threadIdx.x;
  int c = 0;
#pragma unroll
  for (int u = 0; u < 4; ++u)
    if (w0 + u < words) c += __popc(bitmap[w0 + u]);
  const int total = block_sum(c, ws);
  if (threadIdx.x == 0) block_sums[blockIdx.x] = total;
}

__global__ void __launch_bounds__(kCompactThreads) list_bits_kernel(uint32_t* bitmap, long long words,
                                                                    const int* __restrict__ block_sums,
                                                                    int n_pad, int* key_ids_pad) {
  __shared__ int ws[kCompactThreads / 32];
  __shared__ int wsc[kCompactThreads / 32];
  int pre = 0, all = 0;
  for (int i = threadIdx.x; i < static_cast<int>(gridDim.x); i += blockDim.x) {
    const int v = block_sums[i];
    all += v;
    if (i < static_cast<int>(blockIdx.x)) pre += v;
  }
  pre = block_sum(pre, ws);
  all = block_sum(all, ws);
  const long long w0 = static_cast<long long>(blockIdx.x) * kWordsPerCta + 4 * threadIdx.x;
  uint32_t b[4];
  int c = 0;
#pragma unroll
  for (int u = 0; u < 4; ++u) {
    b[u] = w0 + u < words ? bitmap[w0 + u] : 0u;
    c += __popc(b[u]);
  }
  // exclusive scan of the per-thread counts
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int incl = c;
  for (int o = 1; o < 32; o <<= 1) {
    const int x = __shfl_up_sync(0xFFFFFFFFu, incl, o);
    if (lane >= o) incl += x;
  }
  if (lane == 31) wsc[warp] = incl;
  __syncthreads();
  int wbase = 0;
  for (int i = 0; i < warp; ++i) wbase += wsc[i];
  int q = pre + wbase + incl - c;
#pragma unroll
  for (int u = 0; u < 4; ++u) {
    uint32_t bb = b[u];
    if (bb == 0u) continue;
    bitmap[w0 + u] = 0u;
    while (bb != 0u) {
      const int bit = __ffs(bb) - 1;
      bb &= bb - 1u;
      if (q < n_pad) key_ids_pad[q] = static_cast<int>((w0 + u) * 32 + bit);
      ++q;
    }
  }
  for (long long r = all + static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; r < n_pad;
       r += static_cast<long long>(gridDim.x) * blockDim.x)
    key_ids_pad[r] = INT_MAX;
}

// Copy sample rows (16-byte vectors); missing ids give zero rows.
__global__ void gather_keys_kernel(const uint4* __restrict__ k_cache, const float* __restrict__ k_scale,
                                   int vec_per_row, const int* __restrict__ key_ids_pad, int n_pad,
                                   uint4* __restrict__ k_samp, float* __restrict__ k_scale_samp) {
  const long long gid = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
  const long long total = static_cast<long long>(n_pad) * vec_per_row;
  if (gid >= total) return;
  const int r = static_cast<int>(gid / vec_per_row);
  const int v = static_cast<int>(gid % vec_per_row);
  const int id = key_ids_pad[r];
  uint4 x = make_uint4(0, 0, 0, 0);
  if (id != INT_MAX) x = k_cache[static_cast<long long>(id) * vec_per_row + v];
  k_samp[gid] = x;
  if (k_scale != nullptr && v == 0) k_scale_samp[r] = (id != INT_MAX) ? k_scale[id] : 0.f;
}

constexpr int kStatsThreads = 256;

// Block-wide radix select of the r-th largest (1-based) of m uint32 values in
// shared memory (blockDim.x a multiple of 32, at least 256).  Returns the
// value.  Per 8-bit digit: a histogram of shared atomics (one per warp when
// all its lanes share the digit), then the first
// 256 threads scan the digits from the top in parallel and the one whose digit
// holds the r-th value publishes it.
__device__ uint32_t block_select_u32(const uint32_t* vals, int m, int r, unsigned* hist256,
                                     uint32_t* sh_state, unsigned* warp_tot) {
  uint32_t prefix = 0, mask = 0;
  int remaining = r;
  const int tid = threadIdx.x, lane = tid & 31;
  for (int shift = 24; shift >= 0; shift -= 8) {
    for (int i = tid; i < 256; i += blockDim.x) hist256[i] = 0;
    __syncthreads();
    for (int i0 = 0; i0 < m; i0 += blockDim.x) {
      const int i = i0 + tid;
      const uint32_t v = i < m ? vals[i] : 0u;
      const bool in = i < m && (v & mask) == prefix;
      const unsigned act = __ballot_sync(0xFFFFFFFFu, in);
      if (in) {
        // one atomic when every active lane has the same digit (the common case
        // for the high digits of a narrow score range), else one per lane
        const unsigned dig = (v >> shift) & 255u;
        const int leader = __ffs(act) - 1;
        const unsigned d0 = __shfl_sync(act, dig, leader);
        if (__all_sync(act, dig == d0)) {
          if (lane == leader) atomicAdd(&hist256[dig], static_cast<unsigned>(__popc(act)));
        } else {
          atomicAdd(&hist256[dig], 1u);
        }
      }
    }
    __syncthreads();
    unsigned c = 0, incl = 0;
    if (tid < 256) {
      c = hist256[255 - tid];             // thread t looks at digit 255 - t
      incl = c;
      for (int o = 1; o < 32; o <<= 1) {
        const unsigned u = __shfl_up_sync(0xFFFFFFFFu, incl, o);
        if (lane >= o) incl += u;
      }
      if (lane == 31) warp_tot[tid >> 5] = incl;
    }
    __syncthreads();
    if (tid < 256) {
      for (int w = 0; w < (tid >> 5); ++w) incl += warp_tot[w];
      const unsigned above = incl - c;    // values with a larger digit
      if (above < static_cast<unsigned>(remaining) && incl >= static_cast<unsigned>(remaining)) {
        sh_state[0] = static_cast<uint32_t>(255 - tid);
        sh_state[1] = above;
      }
    }
    __syncthreads();
    prefix |= sh_state[0] << shift;
    mask |= 0xFFu << shift;
    remaining -= static_cast<int>(sh_state[1]);
    __syncthreads();
  }
  return prefix;
}

constexpr int kStatBins = 1024;

// The r-th largest of m order codes in shared memory (0 = invisible score),
// the visible scores spanning [lo, hi]: a histogram of kStatBins equal-width
// bins over [lo, hi] (monotone in the score) finds the bin holding it and the
// count above that bin; that bin's codes are gathered into hb (the histogram
// is no longer needed) and ranked by counting, one code per thread (a radix
// select when the bin holds more codes than the block has threads).  Two
// passes over the m codes instead of four; a crowded bin (more than kStatBins
// codes) falls back to the radix select over all m.
__device__ uint32_t block_select_binned(const uint32_t* vals, int m, int r, float lo, float hi, unsigned* hb,
                                        unsigned* hist256, uint32_t* sh_state, unsigned* warp_tot,
                                        int* sh_int) {
  const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
  const int bd = static_cast<int>(blockDim.x);
  float delta = 0.f;
  if (hi > lo) {
    delta = __fdiv_rn(static_cast<float>(kStatBins), __fsub_rn(hi, lo));
    if (!(delta <= 1e30f)) delta = 1e30f;
  }
  for (int i = tid; i < kStatBins; i += bd) hb[i] = 0u;
  __syncthreads();
  for (int i = tid; i < m; i += bd) {
    const uint32_t v = vals[i];
    if (v != 0u) atomicAdd(&hb[bin_of(unord_f32(v), lo, delta, kStatBins)], 1u);
  }
  __syncthreads();
  // thread t owns bins [top - per, top), top = kStatBins - t * per
  const int per = kStatBins / bd;
  const int top = kStatBins - tid * per;
  int seg = 0;
  for (int b = top - per; b < top; ++b) seg += static_cast<int>(hb[b]);
  int incl = seg;
  for (int o = 1; o < 32; o <<= 1) {
    const int u = __shfl_up_sync(0xFFFFFFFFu, incl, o);
    if (lane >= o) incl += u;
  }
  if (lane == 31) warp_tot[w] = static_cast<unsigned>(incl);
  __syncthreads();
  for (int i = 0; i < w; ++i) incl += static_cast<int>(warp_tot[i]);
  int above = incl - seg;
  if (above < r && incl >= r) {
    int b = top - 1;
    for (; b > top - per; --b) {
      if (above + static_cast<int>(hb[b]) >= r) break;
      above += static_cast<int>(hb[b]);
    }
    sh_int[0] = b;
    sh_int[1] = above;
    sh_int[2] = static_cast<int>(hb[b]);
  }
  if (tid == 0) sh_int[3] = 0;
  __syncthreads();
  const int bstar = sh_int[0], cb = sh_int[2];
  const int r_in = r - sh_int[1];
  if (cb > kStatBins) return block_select_u32(vals, m, r, hist256, sh_state, warp_tot);
  for (int i = tid; i < m; i += bd) {
    const uint32_t v = vals[i];
    if (v != 0u && bin_of(unord_f32(v), lo, delta, kStatBins) == bstar) hb[atomicAdd(&sh_int[3], 1)] = v;
  }
  __syncthreads();
  if (cb > bd) return block_select_u32(hb, cb, r_in, hist256, sh_state, warp_tot);
  // rank by counting (one code per thread): code i has rank #{j : c_j > c_i}
  // + #{j < i : c_j == c_i}, a permutation of 0..cb-1, so exactly one thread
  // holds rank r_in - 1, and its code is the r_in-th largest
  if (tid < cb) {
    const uint32_t v = hb[tid];
    int rank = 0;
    for (int j = 0; j < cb; ++j) {
      const uint32_t u = hb[j];
      rank += (u > v || (u == v && j < tid)) ? 1 : 0;
    }
    if (rank == r_in - 1) sh_state[0] = v;
  }
  __syncthreads();
  return sh_state[0];
}

// Per query, from the visible sample scores: the equal-width bins and the
// start threshold bin.  Bins below the start threshold are never used (the
// threshold only rises), so the bins span from just below the sample's k-th
// largest score s_k up to s_max + (s_max - s_k): the span above s_k, doubled
// as headroom for top-k scores beyond the sample's maximum (a small sample of a
// large cache rarely contains the true top scores).  s_k sits three bins above
// the lower end; the start threshold is bin(s_k) - 1, one bin of slack below
// it, and everything under the range clamps into bin 0 and is rejected.  With
// fewer than k visible sample keys (or no spread above s_k) the bins cover
// [s_min, s_max + (s_max - s_min)] and the threshold starts at 0.
template <int THREADS>
__global__ void __launch_bounds__(THREADS) sample_stats_kernel(const SampleStatsParams p) {
  extern __shared__ uint32_t s_ord[];
  __shared__ unsigned hist256[256];
  __shared__ uint32_t sh_state[2];
  __shared__ unsigned warp_tot[32];
  __shared__ unsigned hbins[kStatBins];
  __shared__ int sh_int[4];
  __shared__ float red_min[32], red_max[32];
  __shared__ int red_cnt[32];
  const int t = blockIdx.x;
  const float* row = p.scores + static_cast<size_t>(t) * p.ld;
  float mn = INFINITY, mx = -INFINITY;
  int cnt = 0;
#pragma unroll 4
  for (int i = threadIdx.x; i < p.n; i += blockDim.x) {
    const float v = row[i];
    const bool vis = v != -INFINITY;
    s_ord[i] = vis ? ord_f32(v) : 0u;
    if (vis) {
      mn = fminf(mn, v);
      mx = fmaxf(mx, v);
      ++cnt;
    }
  }
  for (int o = 16; o > 0; o >>= 1) {
    mn = fminf(mn, __shfl_xor_sync(0xFFFFFFFFu, mn, o));
    mx = fmaxf(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, o));
    cnt += __shfl_xor_sync(0xFFFFFFFFu, cnt, o);
  }
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (lane == 0) {
    red_min[warp] = mn;
    red_max[warp] = mx;
    red_cnt[warp] = cnt;
  }
  __syncthreads();
  if (warp == 0) {
    const bool have = lane < static_cast<int>(blockDim.x / 32);
    mn = have ? red_min[lane] : INFINITY;
    mx = have ? red_max[lane] : -INFINITY;
    cnt = have ? red_cnt[lane] : 0;
    for (int o = 16; o > 0; o >>= 1) {
      mn = fminf(mn, __shfl_xor_sync(0xFFFFFFFFu, mn, o));
      mx = fmaxf(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, o));
      cnt += __shfl_xor_sync(0xFFFFFFFFu, cnt, o);
    }
    __syncwarp();
    if (lane == 0) {
      red_min[0] = mn;
      red_max[0] = mx;
      red_cnt[0] = cnt;
    }
  }
  __syncthreads();
  mn = red_min[0];
  mx = red_max[0];
  cnt = red_cnt[0];
  float smin = 0.f, delta = 0.f;
  int theta = 0;
  bool ranged = false;
  if (cnt >= p.k && p.k > 0) {
    const float sk =
        unord_f32(block_select_binned(s_ord, p.n, p.k, mn, mx, hbins, hist256, sh_state, warp_tot, sh_int));
    const float span = __fsub_rn(mx, sk);
    if (span > 0.f) {
      const float hi = __fadd_rn(mx, span);
      delta = __fdiv_rn(static_cast<float>(p.nb - 3), __fsub_rn(hi, sk));
      if (!(delta <= 1e30f)) delta = 1e30f;
      if (p.pow2_delta) delta = pow2_floor(delta);   // wider bins: the span still fits
      smin = __fsub_rn(sk, __fdiv_rn(3.f, delta));
      theta = max(0, bin_of(sk, smin, delta, p.nb) - 1);
      ranged = true;
    }
  }
  if (!ranged && cnt > 0) {
    smin = mn;
    theta = 0;
    if (mx > mn) {
      delta = __fdiv_rn(static_cast<float>(p.nb), __fmul_rn(2.f, __fsub_rn(mx, mn)));
      if (!(delta <= 1e30f)) delta = 1e30f;
      if (p.pow2_delta) delta = pow2_floor(delta);
    }
  }
  if (threadIdx.x == 0) {
    p.s_min[t] = smin;
    p.delta[t] = delta;
    p.theta0[t] = theta;
  }
}

// ---- previous-chunk sample: rank key ids by selection count ----
__global__ void count_kernel(const int* __restrict__ prev, long long n_prev, long long S,
                             int* __restrict__ counts) {
  for (long long i = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; i < n_prev;
       i += static_cast<long long>(gridDim.x) * blockDim.x) {
    const int id = prev[i];
    if (id >= 0 && id < S) atomicAdd(&counts[id], 1);
  }
}

// Ranking key: count in the high word; ties broken by the higher id among
// selected keys, pseudo-randomly (a bijection of the id) among unselected ones.
__global__ void rank_keys_kernel(const int* __restrict__ counts, long long S, unsigned long long seed,
                                 unsigned long long* __restrict__ keys) {
  for (long long s = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; s < S;
       s += static_cast<long long>(gridDim.x) * blockDim.x) {
    const uint32_t c = static_cast<uint32_t>(counts[s]);
    const uint32_t lo = c > 0 ? static_cast<uint32_t>(s) : perm31(static_cast<uint32_t>(s), seed);
    keys[s] = (static_cast<uint64_t>(c) << 32) | lo;
  }
}

// state: [0] prefix, [1] mask, [2] remaining, [3] output slot
__global__ void digit_hist_kernel(const unsigned long long* __restrict__ keys, long long S, int shift,
                                  const unsigned long long* __restrict__ state,
                                  unsigned int* __restrict__ hist) {
  __shared__ unsigned int h[256];
  for (int i = threadIdx.x; i < 256; i += blockDim.x) h[i] = 0;
  __syncthreads();
  const uint64_t prefix = state[0], mask = state[1];
  for (long long s = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; s < S;
       s += static_cast<long long>(gridDim.x) * blockDim.x) {
    const uint64_t k = keys[s];
    if ((k & mask) == prefix) atomicAdd(&h[(k >> shift) & 255u], 1u);
  }
  __syncthreads();
  for (int i = threadIdx.x; i < 256; i += blockDim.x)
    if (h[i]) atomicAdd(&hist[i], h[i]);
}

// One CTA of 256 threads: thread t looks at digit 255 - t; a block scan of the
// counts from the top finds the digit holding the remaining rank, and every
// thread clears its bin for the next pass.
__global__ void __launch_bounds__(256) digit_pick_kernel(unsigned int* hist, int shift,
                                                         unsigned long long* state) {
  __shared__ long long warp_tot[8];
  const int t = threadIdx.x, lane = t & 31, w = t >> 5;
  const long long remaining = static_cast<long long>(state[2]);
  const int d = 255 - t;
  const long long c = hist[d];
  long long incl = c;
  for (int o = 1; o < 32; o <<= 1) {
    const long long u = __shfl_up_sync(0xFFFFFFFFu, incl, o);
    if (lane >= o) incl += u;
  }
  if (lane == 31) warp_tot[w] = incl;
  __syncthreads();
  for (int i = 0; i < w; ++i) incl += warp_tot[i];
  const long long above = incl - c;   // keys with a larger digit
  hist[d] = 0;
  // (the last digit takes the rank when the counts fall short, as the
  // sequential scan would)
  if ((above < remaining && incl >= remaining) || (d == 0 && incl < remaining)) {
    state[0] |= static_cast<uint64_t>(d) << shift;
    state[1] |= static_cast<uint64_t>(0xFF) << shift;
    state[2] = static_cast<uint64_t>(remaining - above);
  }
}

__global__ void collect_top_kernel(const unsigned long long* __restrict__ keys, long long S,
                                   unsigned long long* state, int n, int* __restrict__ out) {
  const uint64_t kth = state[0];
  for (long long s = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; s < S;
       s += static_cast<long long>(gridDim.x) * blockDim.x) {
    if (keys[s] >= kth) {
      const unsigned long long slot = atomicAdd(&state[3], 1ull);
      if (slot < static_cast<unsigned long long>(n)) out[slot] = static_cast<int>(s);
    }
  }
}

__global__ void init_select_state_kernel(unsigned long long* state, unsigned int* hist, int n) {
  if (threadIdx.x == 0) {
    state[0] = 0;
    state[1] = 0;
    state[2] = static_cast<unsigned long long>(n);
    state[3] = 0;
  }
  for (int d = threadIdx.x; d < 256; d += blockDim.x) hist[d] = 0;
}

int grid_for(long long n, int threads, int cap_blocks) {
  long long b = (n + threads - 1) / threads;
  if (b < 1) b = 1;
  if (b > cap_blocks) b = cap_blocks;
  return static_cast<int>(b);
}

}  // namespace

cudaError_t launch_random_sample(long long S, int n, unsigned long long seed, int* out,
                                 cudaStream_t stream) {
  if (n <= 0) return cudaSuccess;
  random_sample_kernel<<<(n + 255) / 256, 256, 0, stream>>>(S, n, seed, out);
  count_launches(1);
  return cudaGetLastError();
}

cudaError_t launch_prepare_sample(const int* ids, int n, long long S, int n_pad, int* key_ids_pad,
                                  uint32_t* bitmap, int* block_sums, cudaStream_t stream) {
  if (n > 0) {
    mark_ids_kernel<<<(n + 255) / 256, 256, 0, stream>>>(ids, n, S, bitmap);
    count_launches(1);
  }
  const long long words = (S + 31) / 32;
  const int blocks = static_cast<int>((words + kWordsPerCta - 1) / kWordsPerCta);
  if (blocks == 0) {
    fill_ids_kernel<<<(n_pad + 255) / 256, 256, 0, stream>>>(key_ids_pad, n_pad);
    count_launches(1);
    return cudaGetLastError();
  }
  count_bits_kernel<<<blocks, kCompactThreads, 0, stream>>>(bitmap, words, block_sums);
  list_bits_kernel<<<blocks, kCompactThreads, 0, stream>>>(bitmap, words, block_sums, n_pad, key_ids_pad);
  count_launches(2);
  return cudaGetLastError();
}

int prepare_sample_blocks(long long S) {
  return static_cast<int>(((S + 31) / 32 + kWordsPerCta - 1) / kWordsPerCta);
}

cudaError_t launch_gather_keys(const void* k_cache, const float* k_scale, int elem_bytes, int dim,
                               const int* key_ids_pad, int n_pad, void* k_samp, float* k_scale_samp,
                               cudaStream_t stream) {
  const int vec = dim * elem_bytes / 16;
  const long long total = static_cast<long long>(n_pad) * vec;
  const int blocks = static_cast<int>((total + 255) / 256);
  if (blocks == 0) return cudaSuccess;
  gather_keys_kernel<<<blocks, 256, 0, stream>>>(static_cast<const uint4*>(k_cache), k_scale, vec,
                                                 key_ids_pad, n_pad, static_cast<uint4*>(k_samp),
                                                 k_scale_samp);
  count_launches(1);
  return cudaGetLastError();
}

cudaError_t launch_sample_stats(const SampleStatsParams& p, int num_sms, cudaStream_t stream) {
  if (p.T <= 0) return cudaSuccess;
  const size_t smem = static_cast<size_t>(p.n) * sizeof(uint32_t);
  cudaError_t e;
  if (p.T < num_sms) {
    // few queries: one wide CTA each (the per-query work is latency-bound)
    e = ensure_smem_limit(reinterpret_cast<const void*>(sample_stats_kernel<1024>), kSlotStatsWide,
                          kMaxSample * sizeof(uint32_t));
    if (e != cudaSuccess) return e;
    sample_stats_kernel<1024><<<p.T, 1024, smem, stream>>>(p);
  } else {
    e = ensure_smem_limit(reinterpret_cast<const void*>(sample_stats_kernel<kStatsThreads>), kSlotStats,
                          kMaxSample * sizeof(uint32_t));
    if (e != cudaSuccess) return e;
    sample_stats_kernel<kStatsThreads><<<p.T, kStatsThreads, smem, stream>>>(p);
  }
  count_launches(1);
  return cudaGetLastError();
}

cudaError_t launch_make_sample(const int* prev_idx, long long n_prev, long long S, int n,
                               unsigned long long seed, const MakeSampleWs& ws, int* out,
                               cudaStream_t stream) {
  cudaError_t e = cudaMemsetAsync(ws.counts, 0, static_cast<size_t>(S) * sizeof(int), stream);
  if (e != cudaSuccess) return e;
  if (n_prev > 0) {
    count_kernel<<<grid_for(n_prev, 256, 4096), 256, 0, stream>>>(prev_idx, n_prev, S, ws.counts);
  }
  rank_keys_kernel<<<grid_for(S, 256, 4096), 256, 0, stream>>>(ws.counts, S, seed, ws.keys);
  init_select_state_kernel<<<1, 256, 0, stream>>>(ws.state, ws.hist, n);
  for (int shift = 56; shift >= 0; shift -= 8) {
    digit_hist_kernel<<<grid_for(S, 256, 1024), 256, 0, stream>>>(ws.keys, S, shift, ws.state, ws.hist);
    digit_pick_kernel<<<1, 256, 0, stream>>>(ws.hist, shift, ws.state);
  }
  collect_top_kernel<<<grid_for(S, 256, 4096), 256, 0, stream>>>(ws.keys, S, ws.state, n, out);
  count_launches((n_prev > 0 ? 1 : 0) + 3 + 2 * 8);
  return cudaGetLastError();
}

}  // namespace ltk
