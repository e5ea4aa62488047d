// block_sort.cuh -- block-wide bitonic sort with the keys held in registers.
//
// E keys per thread (E a power of two, 1..16), thread t holding keys
// [t E, t E + E) of the E * blockDim keys.  Every merge of blocks of `size`
// keys starts with the mirrored step (key i against key i ^ (size - 1)) and
// continues with halving strides, so every exchange has the same direction and
// needs no direction flag: the lower index keeps the minimum (ascending) or
// the maximum (DESC).  Strides below E stay inside the thread, strides below
// 32 E go through warp shuffles, longer ones through the shared-memory buffer
// xs (E * blockDim keys), stored slot-major (xs[e * blockDim + t]) so that
// every access is conflict-free.  Used by the LiteDSA packing (32- or 64-bit
// keys, ascending) and by Select's final ordering (64-bit keys, descending).
#ifndef LTK_BLOCK_SORT_CUH
#define LTK_BLOCK_SORT_CUH

#include <cstdint>

namespace ltk {

template <typename K>
__device__ __forceinline__ K shfl_xor_key(K v, int m) {
  if constexpr (sizeof(K) == 4) {
    return __shfl_xor_sync(0xFFFFFFFFu, v, m);
  } else {
    const uint32_t lo = __shfl_xor_sync(0xFFFFFFFFu, static_cast<uint32_t>(v), m);
    const uint32_t hi = __shfl_xor_sync(0xFFFFFFFFu, static_cast<uint32_t>(v >> 32), m);
    return (static_cast<K>(hi) << 32) | lo;
  }
}

template <typename K>
__device__ __forceinline__ K shfl_up_key(K v) {
  if constexpr (sizeof(K) == 4) {
    return __shfl_up_sync(0xFFFFFFFFu, v, 1);
  } else {
    const uint32_t lo = __shfl_up_sync(0xFFFFFFFFu, static_cast<uint32_t>(v), 1);
    const uint32_t hi = __shfl_up_sync(0xFFFFFFFFu, static_cast<uint32_t>(v >> 32), 1);
    return (static_cast<K>(hi) << 32) | lo;
  }
}

template <typename K>
__device__ __forceinline__ K kmin(K a, K b) { return a < b ? a : b; }
template <typename K>
__device__ __forceinline__ K kmax(K a, K b) { return a < b ? b : a; }

// The value the lower index of a pair keeps (first) and the upper one (second).
template <bool DESC, typename K>
__device__ __forceinline__ K keep_lower(K a, K b) { return DESC ? kmax(a, b) : kmin(a, b); }
template <bool DESC, typename K>
__device__ __forceinline__ K keep_upper(K a, K b) { return DESC ? kmin(a, b) : kmax(a, b); }

// In-thread steps: pairs (e, e ^ (2S - 1)) (mirrored first step) or (e, e + S).
template <int E, int S, bool MIRROR, bool DESC, typename K>
__device__ __forceinline__ void sort_in_thread(K (&v)[E]) {
#pragma unroll
  for (int e = 0; e < E; ++e) {
    if ((e & S) == 0) {
      const int f = MIRROR ? (e ^ (2 * S - 1)) : (e + S);
      const K a = v[e], b = v[f];
      v[e] = keep_lower<DESC>(a, b);
      v[f] = keep_upper<DESC>(a, b);
    }
  }
}

template <int E, bool MIRROR, bool DESC, typename K>
__device__ __forceinline__ void sort_in_thread_at(K (&v)[E], int half) {
  switch (half) {
    case 1: sort_in_thread<E, 1, MIRROR, DESC>(v); break;
    case 2: if constexpr (E > 2) sort_in_thread<E, 2, MIRROR, DESC>(v); break;
    case 4: if constexpr (E > 4) sort_in_thread<E, 4, MIRROR, DESC>(v); break;
    case 8: if constexpr (E > 8) sort_in_thread<E, 8, MIRROR, DESC>(v); break;
    default: break;
  }
}

template <int E, bool DESC, typename K>
__device__ void block_sort_regs(K (&v)[E], K* xs) {
  const int tid = threadIdx.x, lane = tid & 31;
  const int nt = blockDim.x;
  const int P = E * nt;
#pragma unroll 1
  for (int size = 2; size <= P; size <<= 1) {
#pragma unroll 1
    for (int half = size >> 1; half > 0; half >>= 1) {
      const bool mirror = half == (size >> 1);
      if (half < E) {
        if constexpr (E > 1) {
          if (mirror) sort_in_thread_at<E, true, DESC>(v, half);
          else sort_in_thread_at<E, false, DESC>(v, half);
        }
      } else if (half < 32 * E) {
        const int lm = mirror ? (size / E - 1) : (half / E);   // partner lane: lane ^ lm
        const bool lower = (lane & (half / E)) == 0;
        if (mirror) {
          K o[E];
#pragma unroll
          for (int e = 0; e < E; ++e) o[e] = shfl_xor_key(v[E - 1 - e], lm);   // partner slot E-1-e
#pragma unroll
          for (int e = 0; e < E; ++e)
            v[e] = lower ? keep_lower<DESC>(v[e], o[e]) : keep_upper<DESC>(v[e], o[e]);
        } else {
#pragma unroll
          for (int e = 0; e < E; ++e) {
            const K o = shfl_xor_key(v[e], lm);
            v[e] = lower ? keep_lower<DESC>(v[e], o) : keep_upper<DESC>(v[e], o);
          }
        }
      } else {
        const int tm = mirror ? (size / E - 1) : (half / E);   // partner thread: tid ^ tm
        const bool lower = (tid & (half / E)) == 0;
#pragma unroll
        for (int e = 0; e < E; ++e) xs[e * nt + tid] = v[e];
        __syncthreads();
#pragma unroll
        for (int e = 0; e < E; ++e) {
          const K o = xs[(mirror ? E - 1 - e : e) * nt + (tid ^ tm)];
          v[e] = lower ? keep_lower<DESC>(v[e], o) : keep_upper<DESC>(v[e], o);
        }
        __syncthreads();
      }
    }
  }
}

}  // namespace ltk

#endif  // LTK_BLOCK_SORT_CUH
