// k_litedsa.cu -- LiteDSA candidate packing (LiteTopK arXiv abstract: pack the
// overlapping candidates of neighbouring query tokens into a shared key/value
// list for joint attention, with per-query masks that keep each token's own
// top-k membership).
//
// One CTA of 1024 threads per group of G consecutive queries:
//   1. the group's G * k selected indices become 64-bit keys
//      (index << 8 | query-within-group); invalid slots (-1) and the padding
//      up to P = E * 1024 keys (E a power of two, 1..16) sort last;
//   2. a bitonic sort with the keys in registers (block_sort.cuh): thread t
//      holds keys [t E, t E + E); only strides of 32 E and more go through
//      shared memory;
//   3. a key starts a run when its index differs from the previous key's; a
//      block scan of the per-thread run counts gives every key its position j
//      in the ascending union; the first key of a run writes union[j], and
//      every key sets bit j of its query's mask (shared-memory atomicOr);
//   4. lengths, the -1 padding of the union and the masks go to device memory.
// G * k <= 16384.
#include "block_sort.cuh"
#include "ltk_internal.cuh"

namespace ltk {
namespace {

constexpr int kLdThreads = 1024;
constexpr int kLdMaxEntries = 16384;
// Pack one group with keys of type K: index << 8 | query-within-group, none =
// all ones (sorts last).
template <int E, typename K>
__device__ void ld_pack_group(const int* __restrict__ topk, int k, int G, int W, int t0, int ng, int g,
                              K* xs, uint32_t* smask, int* warp_sum, K* warp_last, int* total_starts,
                              int* union_idx, int* union_len, uint32_t* masks) {
  constexpr K kNone = static_cast<K>(~static_cast<K>(0));
  const int n = ng * k;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int nw = static_cast<int>(blockDim.x >> 5);
  const int base = tid * E;
  K v[E];
#pragma unroll
  for (int e = 0; e < E; ++e) {
    const int i = base + e;
    K key = kNone;
    if (i < n) {
      const int idx = topk[static_cast<size_t>(t0) * k + i];
      if (idx >= 0) key = (static_cast<K>(idx) << 8) | static_cast<K>(i / k);
    }
    v[e] = key;
  }
  block_sort_regs<E, false>(v, xs);

  // the key before this thread's first key: the previous lane's last, or for
  // lane 0 the previous warp's last
  K prev = shfl_up_key(v[E - 1]);
  if (lane == 31) warp_last[warp] = v[E - 1];
  __syncthreads();
  if (lane == 0) prev = warp > 0 ? warp_last[warp - 1] : kNone;
  int cnt = 0;
#pragma unroll
  for (int e = 0; e < E; ++e) {
    const K before = e == 0 ? prev : v[e - 1];
    cnt += (v[e] != kNone && (base + e == 0 || (before >> 8) != (v[e] >> 8))) ? 1 : 0;
  }
  int incl = cnt;
  for (int o = 1; o < 32; o <<= 1) {
    const int u = __shfl_up_sync(0xFFFFFFFFu, incl, o);
    if (lane >= o) incl += u;
  }
  if (lane == 31) warp_sum[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    const int x = lane < nw ? warp_sum[lane] : 0;
    int sc = x;
    for (int o = 1; o < 32; o <<= 1) {
      const int u = __shfl_up_sync(0xFFFFFFFFu, sc, o);
      if (lane >= o) sc += u;
    }
    if (lane < nw) warp_sum[lane] = sc - x;
    if (lane == 31) *total_starts = sc;
  }
  __syncthreads();
  int cur = warp_sum[warp] + incl - cnt - 1;   // the run before this thread's first key
  int* urow = union_idx + static_cast<size_t>(g) * G * k;
#pragma unroll
  for (int e = 0; e < E; ++e) {
    const K key = v[e];
    if (key == kNone) break;
    const K before = e == 0 ? prev : v[e - 1];
    if (base + e == 0 || (before >> 8) != (key >> 8)) {
      ++cur;
      urow[cur] = static_cast<int>(key >> 8);
    }
    const int r = static_cast<int>(key & static_cast<K>(0xFF));
    atomicOr(&smask[r * W + (cur >> 5)], 1u << (cur & 31));
  }
  __syncthreads();
  const int len = *total_starts;
  if (tid == 0) union_len[g] = len;
  for (int i = len + tid; i < G * k; i += blockDim.x) urow[i] = -1;
  for (int i = tid; i < ng * W; i += blockDim.x) masks[static_cast<size_t>(t0) * W + i] = smask[i];
}

template <int E>
__global__ void __launch_bounds__(kLdThreads)
    litedsa_pack_kernel(const int* __restrict__ topk, int T, int k, int G, int W, int* union_idx,
                        int* union_len, uint32_t* masks) {
  extern __shared__ unsigned long long ld_xs[];                  // [E * 1024] exchange
  uint32_t* smask = reinterpret_cast<uint32_t*>(ld_xs + E * kLdThreads);   // [G][W]
  __shared__ int warp_sum[kLdThreads / 32];
  __shared__ unsigned long long warp_last[kLdThreads / 32];
  __shared__ int total_starts;
  const int g = blockIdx.x;
  const int t0 = g * G;
  const int ng = min(G, T - t0);
  for (int i = threadIdx.x; i < G * W; i += blockDim.x) smask[i] = 0u;
  // 32-bit keys when every index of the group is below 2^24 (the common case:
  // half the exchange work of 64-bit keys, single-instruction min and max)
  bool big = false;
  for (int i = threadIdx.x; i < ng * k; i += blockDim.x) big |= topk[static_cast<size_t>(t0) * k + i] >= (1 << 24);
  if (__syncthreads_or(big ? 1 : 0))
    ld_pack_group<E, unsigned long long>(topk, k, G, W, t0, ng, g, ld_xs, smask, warp_sum, warp_last,
                                         &total_starts, union_idx, union_len, masks);
  else
    ld_pack_group<E, uint32_t>(topk, k, G, W, t0, ng, g, reinterpret_cast<uint32_t*>(ld_xs), smask,
                               warp_sum, reinterpret_cast<uint32_t*>(warp_last), &total_starts, union_idx,
                               union_len, masks);
}

int ld_elems(int G, int k) {
  int E = 1;
  while (E * kLdThreads < G * k) E <<= 1;
  return E;
}

}  // namespace

int litedsa_max_entries() { return kLdMaxEntries; }

// Shared memory of one group: the exchange buffer of the sort (E * 1024 keys)
// and the G masks of ceil(G * k / 32) words.
size_t litedsa_smem_bytes(int G, int k) {
  return static_cast<size_t>(ld_elems(G, k)) * kLdThreads * 8 + static_cast<size_t>(G) * ((G * k + 31) / 32) * 4;
}

template <int E>
cudaError_t launch_ld(const int* topk, int T, int k, int G, int W, int* union_idx, int* union_len,
                      uint32_t* masks, int n_groups, size_t smem, cudaStream_t stream) {
  cudaError_t e = ensure_smem_limit(reinterpret_cast<const void*>(litedsa_pack_kernel<E>),
                                    kSlotLitedsa + (E == 1 ? 0 : E == 2 ? 1 : E == 4 ? 2 : E == 8 ? 3 : 4),
                                    kLitedsaMaxSmem);
  if (e != cudaSuccess) return e;
  litedsa_pack_kernel<E><<<n_groups, kLdThreads, smem, stream>>>(topk, T, k, G, W, union_idx, union_len, masks);
  count_launches(1);
  return cudaGetLastError();
}

cudaError_t launch_litedsa_pack(const int* topk, int T, int k, int G, int* union_idx, int* union_len,
                                uint32_t* masks, cudaStream_t stream) {
  const int n_groups = (T + G - 1) / G;
  if (n_groups == 0) return cudaSuccess;
  const int W = (G * k + 31) / 32;
  const size_t smem = litedsa_smem_bytes(G, k);
  switch (ld_elems(G, k)) {
    case 1: return launch_ld<1>(topk, T, k, G, W, union_idx, union_len, masks, n_groups, smem, stream);
    case 2: return launch_ld<2>(topk, T, k, G, W, union_idx, union_len, masks, n_groups, smem, stream);
    case 4: return launch_ld<4>(topk, T, k, G, W, union_idx, union_len, masks, n_groups, smem, stream);
    case 8: return launch_ld<8>(topk, T, k, G, W, union_idx, union_len, masks, n_groups, smem, stream);
    case 16: return launch_ld<16>(topk, T, k, G, W, union_idx, union_len, masks, n_groups, smem, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace ltk
