// k_litedsa.cu -- LiteDSA candidate packing (LiteTopK arXiv abstract: pack the
// overlapping candidates of neighbouring query tokens into a shared key/value
// list for joint attention, with per-query masks that keep each token's own
// top-k membership).
//
// One CTA per group of G consecutive queries:
//   1. the group's G * k selected indices become 64-bit keys
//      (index << 8 | query-within-group); invalid slots (-1) sort last;
//   2. a bitonic sort in shared memory orders them by index;
//   3. one block-wide scan over "first occurrence of an index" flags gives
//      every key its position j in the ascending union; the first occurrence
//      writes union[j], and every occurrence sets bit j of its query's mask
//      (shared-memory atomicOr);
//   4. lengths, the -1 padding of the union and the masks go to device memory.
// G * k <= 16384 keeps the sort in shared memory (128 KB of keys).
#include "ltk_internal.cuh"

namespace ltk {
namespace {

constexpr int kLdThreads = 1024;
constexpr int kLdMaxEntries = 16384;

__global__ void __launch_bounds__(kLdThreads)
    litedsa_pack_kernel(const int* __restrict__ topk, int T, int k, int G, int W, int* union_idx,
                        int* union_len, uint32_t* masks) {
  extern __shared__ unsigned long long ld_keys[];
  __shared__ int warp_sum[kLdThreads / 32];
  __shared__ int total_starts;
  const int g = blockIdx.x;
  const int t0 = g * G;
  const int ng = min(G, T - t0);
  const int n = ng * k;
  int P = 1;
  while (P < n) P <<= 1;
  uint32_t* smask = reinterpret_cast<uint32_t*>(ld_keys + P);   // [G][W]
  const unsigned long long kNone = ~0ull;

  for (int e = threadIdx.x; e < P; e += blockDim.x) {
    unsigned long long key = kNone;
    if (e < n) {
      const int idx = topk[static_cast<size_t>(t0) * k + e];
      if (idx >= 0) key = (static_cast<unsigned long long>(idx) << 8) | static_cast<unsigned>(e / k);
    }
    ld_keys[e] = key;
  }
  for (int i = threadIdx.x; i < G * W; i += blockDim.x) smask[i] = 0u;
  __syncthreads();

  // bitonic sort, ascending
  for (int size = 2; size <= P; size <<= 1) {
    for (int stride = size >> 1; stride > 0; stride >>= 1) {
      for (int i = threadIdx.x; i < (P >> 1); i += blockDim.x) {
        const int lo = 2 * i - (i & (stride - 1));
        const int hi = lo + stride;
        const bool up = (lo & size) == 0;
        const unsigned long long a = ld_keys[lo], b = ld_keys[hi];
        if ((a > b) == up) {
          ld_keys[lo] = b;
          ld_keys[hi] = a;
        }
      }
      __syncthreads();
    }
  }

  // each thread owns a contiguous segment of the sorted keys
  const int per = (P + blockDim.x - 1) / blockDim.x;
  const int lo = threadIdx.x * per;
  const int hi = min(P, lo + per);
  auto is_start = [&](int i) {
    const unsigned long long key = ld_keys[i];
    if (key == kNone) return false;
    return i == 0 || (ld_keys[i - 1] >> 8) != (key >> 8);
  };
  int cnt = 0;
  for (int i = lo; i < hi; ++i) cnt += is_start(i) ? 1 : 0;
  // exclusive scan of the per-thread counts
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int incl = cnt;
  for (int o = 1; o < 32; o <<= 1) {
    const int v = __shfl_up_sync(0xFFFFFFFFu, incl, o);
    if (lane >= o) incl += v;
  }
  if (lane == 31) warp_sum[warp] = incl;
  __syncthreads();
  if (threadIdx.x == 0) {
    int run = 0;
    for (int w = 0; w < static_cast<int>(blockDim.x >> 5); ++w) {
      const int v = warp_sum[w];
      warp_sum[w] = run;
      run += v;
    }
    total_starts = run;
  }
  __syncthreads();
  int j = warp_sum[warp] + incl - cnt - 1;   // position of the run before this segment
  int* urow = union_idx + static_cast<size_t>(g) * G * k;
  for (int i = lo; i < hi; ++i) {
    const unsigned long long key = ld_keys[i];
    if (key == kNone) break;
    if (is_start(i)) {
      ++j;
      urow[j] = static_cast<int>(key >> 8);
    }
    const int r = static_cast<int>(key & 0xFFu);
    atomicOr(&smask[r * W + (j >> 5)], 1u << (j & 31));
  }
  __syncthreads();
  const int len = total_starts;
  if (threadIdx.x == 0) union_len[g] = len;
  for (int i = len + threadIdx.x; i < G * k; i += blockDim.x) urow[i] = -1;
  for (int i = threadIdx.x; i < ng * W; i += blockDim.x)
    masks[static_cast<size_t>(t0) * W + i] = smask[i];
}

}  // namespace

int litedsa_max_entries() { return kLdMaxEntries; }

// Shared memory of one group: the sorted keys (next power of two of G * k) and
// the G masks of ceil(G * k / 32) words.
size_t litedsa_smem_bytes(int G, int k) {
  int P = 1;
  while (P < G * k) P <<= 1;
  return static_cast<size_t>(P) * 8 + static_cast<size_t>(G) * ((G * k + 31) / 32) * 4;
}

cudaError_t launch_litedsa_pack(const int* topk, int T, int k, int G, int* union_idx, int* union_len,
                                uint32_t* masks, cudaStream_t stream) {
  const int n_groups = (T + G - 1) / G;
  if (n_groups == 0) return cudaSuccess;
  const int W = (G * k + 31) / 32;
  const size_t smem = litedsa_smem_bytes(G, k);
  cudaError_t e = ensure_smem_limit(reinterpret_cast<const void*>(litedsa_pack_kernel), kSlotLitedsa,
                                    kLitedsaMaxSmem);
  if (e != cudaSuccess) return e;
  litedsa_pack_kernel<<<n_groups, kLdThreads, smem, stream>>>(topk, T, k, G, W, union_idx, union_len,
                                                              masks);
  count_launches(1);
  return cudaGetLastError();
}

}  // namespace ltk
