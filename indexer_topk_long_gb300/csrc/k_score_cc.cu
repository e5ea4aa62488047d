// k_score_cc.cu -- CUDA-core indexer scorer with the bin map fused into the
// score (LiteTopK technical summary, Methodology step 2 "Bin Mapping": for
// CUDA-core kernels such as DSA's, the affine map B = (I - s_min) * delta is
// folded into the score computation, so the bin id costs no extra
// instruction on the critical path; Methodology step 3: scores come back from
// bin space through the inverse affine map).
//
// With w'[h] = w[h] * delta (and, for e4m3, times q_scale) the kernel forms
//     V = sum_h w'[h] * f(q[h] . k) * k_scale   (f = ReLU or id),
//     B = V - s_min * delta
// directly; bin = clamp(floor(B), 0, nb - 1), the gate is bin >= theta, and a
// kept candidate stores I = V / delta.  The sample stage rounds delta down to
// a power of two for this kernel, so w * delta, s_min * delta and V / delta
// are exact: V is exactly delta times the score the same sum forms with the
// unscaled weights, the inverse map returns that score bit for bit (integer
// inputs: the exact score), and B is the same fp32 value as the shared bin
// map's (I - s_min) * delta.  Dense mode (sample scoring, decoupled baseline)
// forms I itself with the unscaled weights.
//
// It serves any head count H <= 128 and head dim d (multiple of 8, <= 4096):
// shapes the tensor-core kernels do not cover, and small decode batches.
// Work unit: one query x one key range (the ranges of a query share its
// candidate count and a global histogram, as in the tensor-core kernels).
// 8 compute warps process two keys per thread per step (head groups of 16,
// query rows broadcast from shared memory as fp32); a ninth warp refreshes the
// threshold bin from the histogram with plain overwrites.
#include <climits>
#include <cmath>

#include "ltk_internal.cuh"

namespace ltk {
namespace {

constexpr int kCcComputeWarps = 8;
constexpr int kCcThreads = 32 * (kCcComputeWarps + 1);
constexpr int kCcRefreshWarp = kCcComputeWarps;

struct __align__(8) CcCtrl {
  float c0;          // s_min * delta (filter) or 0 (dense)
  float s_min;
  float delta;
  int theta;
  int cnt;
  int steps_done;    // compute-warp steps finished
  int abort_flag;
  int pos;
};

__device__ __forceinline__ float cc_bf16(uint32_t bits16) { return __uint_as_float(bits16 << 16); }

// fp8 E4M3 code -> float, from the format's definition (sign, 4-bit exponent
// with bias 7, 3-bit mantissa; exponent 0 is subnormal m * 2^-9).
__device__ __forceinline__ float cc_e4m3(uint32_t c) {
  const uint32_t sgn = (c & 0x80u) << 24;
  const uint32_t e = (c >> 3) & 0xFu;
  const uint32_t m = c & 0x7u;
  const float v = e == 0 ? static_cast<float>(m) * 0.001953125f : __uint_as_float(((e + 120u) << 23) | (m << 20));
  return __uint_as_float(__float_as_uint(v) | sgn);
}

// 8 consecutive key elements starting at column c as fp32.
template <bool FP8>
__device__ __forceinline__ void load8(const void* kc, size_t row, int d, int c, float* out) {
  if constexpr (FP8) {
    const uint2 r = *reinterpret_cast<const uint2*>(static_cast<const uint8_t*>(kc) + row * d + c);
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      out[j] = cc_e4m3((r.x >> (8 * j)) & 0xFFu);
      out[4 + j] = cc_e4m3((r.y >> (8 * j)) & 0xFFu);
    }
  } else {
    const uint4 r = *reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(kc) + row * d + c);
    const uint32_t w4[4] = {r.x, r.y, r.z, r.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      out[2 * j] = cc_bf16(w4[j] & 0xFFFFu);
      out[2 * j + 1] = __uint_as_float(w4[j] & 0xFFFF0000u);
    }
  }
}

// sum_h wf[h] * f(qf[h] . key_r) for two keys at once (row0, row1; row1 may
// equal row0 when there is no second key).  qf: [H][d] fp32 in shared memory.
template <bool FP8>
__device__ __forceinline__ void score_two(const float* qf, const float* wf, int H, int d, int relu,
                                          const void* kc, size_t row0, size_t row1, float& out0,
                                          float& out1) {
  float s0 = 0.f, s1 = 0.f;
  for (int hg = 0; hg < H; hg += 16) {
    float a0[16], a1[16];
#pragma unroll
    for (int h = 0; h < 16; ++h) {
      a0[h] = 0.f;
      a1[h] = 0.f;
    }
    for (int c = 0; c < d; c += 8) {
      float k0[8], k1[8];
      load8<FP8>(kc, row0, d, c, k0);
      load8<FP8>(kc, row1, d, c, k1);
#pragma unroll
      for (int h = 0; h < 16; ++h) {
        if (hg + h < H) {
          const float4* qr = reinterpret_cast<const float4*>(qf + (hg + h) * d + c);
          const float4 qa = qr[0], qb = qr[1];
          const float qv[8] = {qa.x, qa.y, qa.z, qa.w, qb.x, qb.y, qb.z, qb.w};
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            a0[h] = __fmaf_rn(qv[j], k0[j], a0[h]);
            a1[h] = __fmaf_rn(qv[j], k1[j], a1[h]);
          }
        }
      }
    }
#pragma unroll
    for (int h = 0; h < 16; ++h) {
      if (hg + h < H) {
        const float w = wf[hg + h];
        s0 = __fmaf_rn(relu ? fmaxf(a0[h], 0.f) : a0[h], w, s0);
        s1 = __fmaf_rn(relu ? fmaxf(a1[h], 0.f) : a1[h], w, s1);
      }
    }
  }
  out0 = s0;
  out1 = s1;
}

template <int MODE, bool FP8>
__global__ void __launch_bounds__(kCcThreads)
    score_cc_kernel(const CcParams p) {
  extern __shared__ float cc_smem[];
  float* qf = cc_smem;                          // [H][d]
  float* wf = qf + p.H * p.d;                   // [H]
  int* hist = reinterpret_cast<int*>(wf + p.H);  // [nb] (filter)
  __shared__ CcCtrl ctrl;

  // work unit: a whole query, or one key range of a split query
  int t = blockIdx.x, split = 0, nsplit = 1;
  if (static_cast<int>(blockIdx.x) >= p.b_full && p.s_last > 1) {
    const int u = blockIdx.x - p.b_full;
    t = p.b_full + u / p.s_last;
    split = u % p.s_last;
    nsplit = p.s_last;
  }
  const bool shared_query = nsplit > 1;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int pos = (p.causal && p.positions != nullptr) ? p.positions[t] : INT_MAX;
  long long last = p.rows;
  if (p.causal && p.positions != nullptr && p.key_ids == nullptr)
    last = min(static_cast<long long>(pos) + 1, p.rows);
  if (last < 0) last = 0;
  const long long per = (last + nsplit - 1) / nsplit;
  const long long k_lo = split * per;
  const long long k_hi = min(last, k_lo + per);

  // setup: query rows (fp32), weights, state
  const size_t qoff = static_cast<size_t>(t) * p.H * p.d;
  for (int i = tid; i < p.H * p.d; i += kCcThreads) {
    qf[i] = FP8 ? cc_e4m3(static_cast<const uint8_t*>(p.q)[qoff + i])
                : cc_bf16(static_cast<const uint16_t*>(p.q)[qoff + i]);
  }
  float delta = 1.f, s_min = 0.f;
  if constexpr (MODE == kModeFilter) {
    delta = p.delta[t];
    s_min = p.s_min[t];
    if (!(delta > 0.f)) {   // no spread in the sample: any monotone map will do
      delta = 1.f;
    }
    delta = pow2_floor(delta);   // already a power of two from the sample stage
  }
  for (int h = tid; h < p.H; h += kCcThreads) {
    float w = p.w[static_cast<size_t>(t) * p.H + h];
    if constexpr (FP8) w = __fmul_rn(w, p.q_scale[t]);
    if constexpr (MODE == kModeFilter) w = __fmul_rn(w, delta);
    wf[h] = w;
  }
  if constexpr (MODE == kModeFilter) {
    for (int b = tid; b < p.nb; b += kCcThreads) hist[b] = 0;
  }
  if (tid == 0) {
    ctrl.c0 = MODE == kModeFilter ? __fmul_rn(s_min, delta) : 0.f;
    ctrl.s_min = s_min;
    ctrl.delta = delta;
    ctrl.theta = MODE == kModeFilter ? p.theta0[t] : 0;
    ctrl.cnt = 0;
    ctrl.steps_done = 0;
    ctrl.abort_flag = 0;
    ctrl.pos = pos;
  }
  __syncthreads();

  const long long span = k_hi - k_lo;
  const long long keys_per_step = 2ll * 32 * kCcComputeWarps;
  const int n_steps = static_cast<int>((span + keys_per_step - 1) / keys_per_step);

  if (warp < kCcComputeWarps) {
    const float c0 = ctrl.c0;
    const float inv_delta = __fdiv_rn(1.f, delta);
    for (int it = 0; it < n_steps; ++it) {
      const long long base = k_lo + it * keys_per_step + 2ll * tid;
      const bool ok0 = base < k_hi, ok1 = base + 1 < k_hi;
      const long long r0 = ok0 ? base : k_lo, r1 = ok1 ? base + 1 : (ok0 ? base : k_lo);
      float v0 = 0.f, v1 = 0.f;
      if (ok0 || ok1) score_two<FP8>(qf, wf, p.H, p.d, p.relu, p.k_cache, r0, r1, v0, v1);
      if constexpr (FP8) {
        v0 = __fmul_rn(v0, ok0 ? p.k_scale[r0] : 0.f);
        v1 = __fmul_rn(v1, ok1 ? p.k_scale[r1] : 0.f);
      }
#pragma unroll
      for (int r = 0; r < 2; ++r) {
        const long long key = base + r;
        const bool kok = r == 0 ? ok0 : ok1;
        const float v = r == 0 ? v0 : v1;
        if constexpr (MODE == kModeDense) {
          if (kok) {
            int kid = static_cast<int>(key);
            if (p.key_ids != nullptr) kid = p.key_ids[key];
            bool vis = kid != INT_MAX;
            if (p.causal && p.positions != nullptr) vis = vis && kid <= pos;
            p.dense[static_cast<size_t>(t) * p.ld + key] = vis ? v : -INFINITY;
          }
        } else {
          const float B = __fsub_rn(v, c0);                       // fused affine map
          const int b = __float2int_rz(fminf(fmaxf(B, 0.f), static_cast<float>(p.nb - 1)));
          const int th = *reinterpret_cast<volatile int*>(&ctrl.theta);
          const bool pass = kok && b >= th;
          const unsigned m = __ballot_sync(0xFFFFFFFFu, pass);
          if (m != 0) {
            const int leader = __ffs(m) - 1;
            int slot0 = 0;
            if (lane == leader) slot0 = shared_query ? atomicAdd(&p.cnt[t], __popc(m)) : atomicAdd(&ctrl.cnt, __popc(m));
            slot0 = __shfl_sync(0xFFFFFFFFu, slot0, leader);
            if (pass) {
              const int slot = slot0 + __popc(m & ((1u << lane) - 1u));
              // inverse affine map back to the score (exact: delta is a power of two)
              const float I = __fmul_rn(v, inv_delta);
              if (slot < p.cap) p.cand[static_cast<size_t>(t) * p.cap + slot] = cand_pack(I, static_cast<int>(key));
              atomicAdd(&hist[b], 1);
            }
          }
        }
      }
      if (lane == 0) atomicAdd(&ctrl.steps_done, 1);
    }
  } else if (MODE == kModeFilter && warp == kCcRefreshWarp && p.refresh_interval > 0) {
    // threshold refresh: plain overwrite of the bin, never lowered
    int last_done = 0, prev = -1;
    uint64_t t_prog = globaltimer_ns();
    while (true) {
      int done = *reinterpret_cast<volatile int*>(&ctrl.steps_done) / kCcComputeWarps;
      done = __shfl_sync(0xFFFFFFFFu, done, 0);
      if (done >= n_steps) break;
      if (done != prev) {
        prev = done;
        t_prog = globaltimer_ns();
      }
      if (done - last_done >= p.refresh_interval) {
        last_done = done;
        const int* src = hist;
        if (shared_query) {
          int* grow = p.ghist + static_cast<size_t>(t) * p.nb;
          for (int b = lane; b < p.nb; b += 32) {
            const int c = atomicExch(&hist[b], 0);
            if (c != 0) atomicAdd(&grow[b], c);
          }
          __syncwarp();
          src = grow;
        }
        const volatile int* hv = src;
        const int cur = *reinterpret_cast<volatile int*>(&ctrl.theta);
        int run = 0;
        for (int top = p.nb; top > cur; top -= 32) {
          int cum = top - 1 - lane >= 0 ? hv[top - 1 - lane] : 0;
#pragma unroll
          for (int o = 1; o < 32; o <<= 1) {
            const int n = __shfl_up_sync(0xFFFFFFFFu, cum, o);
            if (lane >= o) cum += n;
          }
          const unsigned m = __ballot_sync(0xFFFFFFFFu, run + cum >= p.k);
          if (m != 0) {
            const int th = top - 1 - (__ffs(m) - 1);
            if (lane == 0 && th > cur) *reinterpret_cast<volatile int*>(&ctrl.theta) = th;
            break;
          }
          run += __shfl_sync(0xFFFFFFFFu, cum, 31);
        }
      } else {
        __nanosleep(1000);
        bool expired = globaltimer_ns() - t_prog > kWaitLimitNs;
        expired = __shfl_sync(0xFFFFFFFFu, expired, 0);
        if (expired) {
          if (lane == 0) raise_status(p.status, kDevTimeout);
          break;
        }
      }
    }
  }
  __syncthreads();
  if constexpr (MODE == kModeFilter) {
    if (tid == 0 && !shared_query) p.cnt[t] = ctrl.cnt;
  }
}

template <int MODE, bool FP8>
cudaError_t launch_cc(const CcParams& p, cudaStream_t stream) {
  if (p.T <= 0) return cudaSuccess;
  const int grid = p.b_full + (p.T - p.b_full) * (p.s_last > 1 ? p.s_last : 1);
  const size_t smem = score_cc_smem_bytes(p.H, p.d, MODE == kModeFilter ? p.nb : 0);
  cudaError_t e = ensure_smem_limit(reinterpret_cast<const void*>(score_cc_kernel<MODE, FP8>),
                                    kSlotScoreCc + MODE * 2 + (FP8 ? 1 : 0), kCcMaxSmem);
  if (e != cudaSuccess) return e;
  score_cc_kernel<MODE, FP8><<<grid, kCcThreads, smem, stream>>>(p);
  count_launches(1);
  return cudaGetLastError();
}

}  // namespace

size_t score_cc_smem_bytes(int H, int d, int nb) {
  return static_cast<size_t>(H) * d * 4 + static_cast<size_t>(H) * 4 + static_cast<size_t>(nb) * 4;
}

cudaError_t launch_score_cc(int mode, bool fp8, const CcParams& p, cudaStream_t stream) {
  if (mode == kModeDense)
    return fp8 ? launch_cc<kModeDense, true>(p, stream) : launch_cc<kModeDense, false>(p, stream);
  return fp8 ? launch_cc<kModeFilter, true>(p, stream) : launch_cc<kModeFilter, false>(p, stream);
}

}  // namespace ltk
