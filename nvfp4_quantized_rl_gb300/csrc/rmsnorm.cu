// AQN-noised RMSNorm (sm_103a).
//
// QeRL explainer, section "ゼロオーバーヘッド：レイヤー正規化への統合": the noise vector
// is folded into the RMSNorm weight, X_noise = (Z_noise + w) * X / sqrt(sum(X^2) + delta),
// so channel-wise additive noise becomes row-wise multiplicative noise with no extra
// parameters; the mean of squares is used, as in standard RMSNorm. The noise is
// z = sigma * eps with eps standard-normal draws passed in and sigma from the
// exponential schedule (section "AQNの仕組み").
//
// Rows are spread over a grid of resident CTAs of 256 threads (row = cta, cta + G, ...). Each
// thread owns the columns 8j .. 8j + 7 for j = thread, thread + 256, ... in every row, so it forms
// w + sigma*eps of those columns once, in fp32 registers, for all its rows: late in the schedule
// sigma is far below a bf16 ulp of w, so a 16-bit weight would lose the noise, and re-reading the
// fp32 weight for every row would move four times the bytes of x through L2. A row (H bf16) is read
// with 128-bit loads into registers, the next row's load is issued before this row's reduction,
// the sum of squares is reduced with warp shuffles and then over the eight warps in order, and
// (w + sigma*eps) * x * r is written as bf16. With `amax_bits` the kernel also accumulates max |y| over
// the bf16 values it writes (fp32 bit pattern, one atomicMax per CTA): the amax pass that the NVFP4
// encoding of y would otherwise make.
#include <algorithm>
#include <map>
#include <mutex>

#include "common.cuh"

namespace nvfp4rl {
namespace {

constexpr int kThreads = 256;
constexpr int kMaxVecPerThread = 4;  // H <= 4 * 8 * 256 = 8192 keeps the row in registers

template <bool kNoise, int kVec>
__global__ void __launch_bounds__(kThreads) rmsnorm_aqn_kernel(const uint16_t* __restrict__ x, int64_t M, int64_t H,
                                                               const float* __restrict__ w,
                                                               const float* __restrict__ eps, float sigma,
                                                               float delta, uint16_t* __restrict__ y,
                                                               uint32_t* __restrict__ amax_bits) {
  __shared__ float red[2][kThreads / 32];  // per-warp sums of squares, by row parity
  __shared__ uint32_t mred[kThreads / 32];
  uint32_t m2 = 0;  // max |y| of this thread, both bf16 halves
  griddep_wait();  // the preceding kernel's writes (x, or even w or eps) are visible from here on
  griddep_launch_dependents();
  const int nvec = static_cast<int>(H / 8);
  float wt[kVec][8];
#pragma unroll
  for (int i = 0; i < kVec; ++i) {
    const int j = threadIdx.x + i * kThreads;
#pragma unroll
    for (int t = 0; t < 8; ++t) wt[i][t] = 0.0f;
    if (j < nvec) {
      const float4 w0 = __ldg(reinterpret_cast<const float4*>(w) + 2 * j);
      const float4 w1 = __ldg(reinterpret_cast<const float4*>(w) + 2 * j + 1);
      wt[i][0] = w0.x; wt[i][1] = w0.y; wt[i][2] = w0.z; wt[i][3] = w0.w;
      wt[i][4] = w1.x; wt[i][5] = w1.y; wt[i][6] = w1.z; wt[i][7] = w1.w;
      if (kNoise) {
        const float4 e0 = __ldg(reinterpret_cast<const float4*>(eps) + 2 * j);
        const float4 e1 = __ldg(reinterpret_cast<const float4*>(eps) + 2 * j + 1);
        const float et[8] = {e0.x, e0.y, e0.z, e0.w, e1.x, e1.y, e1.z, e1.w};
#pragma unroll
        for (int t = 0; t < 8; ++t) wt[i][t] = fmaf(sigma, et[t], wt[i][t]);
      }
    }
  }
  const int64_t G = gridDim.x;
  int64_t row = blockIdx.x;
  uint4 v[kVec];
#pragma unroll
  for (int i = 0; i < kVec; ++i) {
    const int j = threadIdx.x + i * kThreads;
    v[i] = row < M && j < nvec ? ld_nc_v4(reinterpret_cast<const uint4*>(x + row * H) + j) : make_uint4(0, 0, 0, 0);
  }
  for (int par = 0; row < M; row += G, par ^= 1) {
    const int64_t next = row + G;
    uint4 nx[kVec];
#pragma unroll
    for (int i = 0; i < kVec; ++i) {
      const int j = threadIdx.x + i * kThreads;
      nx[i] = next < M && j < nvec ? ld_nc_v4(reinterpret_cast<const uint4*>(x + next * H) + j)
                                   : make_uint4(0, 0, 0, 0);
    }
    float ss = 0.0f;
#pragma unroll
    for (int i = 0; i < kVec; ++i) {
      const int j = threadIdx.x + i * kThreads;
      if (j < nvec) {
        const uint32_t q[4] = {v[i].x, v[i].y, v[i].z, v[i].w};
#pragma unroll
        for (int t = 0; t < 4; ++t) {
          const float a = __uint_as_float(bf16_lo_bits(q[t])), b = __uint_as_float(bf16_hi_bits(q[t]));
          ss = fmaf(a, a, ss);
          ss = fmaf(b, b, ss);
        }
      }
    }
    ss = warp_sum(ss);
    if ((threadIdx.x & 31) == 0) red[par][threadIdx.x >> 5] = ss;
    __syncthreads();  // red[par] is rewritten two rows later, after the next row's barrier
    float tot = 0.0f;
#pragma unroll
    for (int i = 0; i < kThreads / 32; ++i) tot += red[par][i];
    const float r = rsqrtf(tot / static_cast<float>(H) + delta);
    uint4* yr = reinterpret_cast<uint4*>(y + row * H);
#pragma unroll
    for (int i = 0; i < kVec; ++i) {
      const int j = threadIdx.x + i * kThreads;
      if (j < nvec) {
        const uint32_t q[4] = {v[i].x, v[i].y, v[i].z, v[i].w};
        uint32_t o[4];
#pragma unroll
        for (int t = 0; t < 4; ++t) {
          const float a = __uint_as_float(bf16_lo_bits(q[t])) * r * wt[i][2 * t];
          const float b = __uint_as_float(bf16_hi_bits(q[t])) * r * wt[i][2 * t + 1];
          o[t] = f32_to_bf16_bits(a) | (f32_to_bf16_bits(b) << 16);
          m2 = __vmaxu2(m2, o[t] & 0x7FFF7FFFu);
        }
        yr[j] = make_uint4(o[0], o[1], o[2], o[3]);
      }
      v[i] = nx[i];
    }
  }
  if (amax_bits) {
    uint32_t m = max(m2 & 0xFFFFu, m2 >> 16) << 16;
    m = __reduce_max_sync(0xFFFFFFFFu, m);
    if ((threadIdx.x & 31) == 0) mred[threadIdx.x >> 5] = m;
    __syncthreads();
    if (threadIdx.x == 0) {
      uint32_t r = 0;
      for (int i = 0; i < kThreads / 32; ++i) r = max(r, mred[i]);
      atomicMax(amax_bits, r);
    }
  }
}

// Resident CTAs per SM of one instance (occupancy query, once per device and instance).
template <bool kNoise, int kVec>
int resident_ctas(const DeviceInfo& dev) {
  static std::mutex mu;
  static std::map<int, int> per_dev;
  std::lock_guard<std::mutex> lock(mu);
  auto it = per_dev.find(dev.device);
  if (it != per_dev.end()) return it->second;
  int n = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, rmsnorm_aqn_kernel<kNoise, kVec>, kThreads, 0) != cudaSuccess)
    n = 0;
  cudaGetLastError();
  n = std::max(n, 1);
  per_dev[dev.device] = n;
  return n;
}

template <bool kNoise, int kVec>
cudaError_t launch_rows(const uint16_t* x, int64_t M, int64_t H, const float* w, const float* eps, float sigma,
                        float delta, uint16_t* y, uint32_t* amax, const DeviceInfo& dev, cudaStream_t st) {
  const int64_t G = std::min<int64_t>(M, static_cast<int64_t>(dev.sm_count) * resident_ctas<kNoise, kVec>(dev));
  return launch_pdl(rmsnorm_aqn_kernel<kNoise, kVec>, dim3(static_cast<unsigned>(G)), dim3(kThreads), 0, st, x, M, H,
                    w, eps, sigma, delta, y, amax);
}

template <bool kNoise>
cudaError_t launch_vec(const uint16_t* x, int64_t M, int64_t H, const float* w, const float* eps, float sigma,
                       float delta, uint16_t* y, uint32_t* amax, const DeviceInfo& dev, cudaStream_t st) {
  const int64_t vec = (H / 8 + kThreads - 1) / kThreads;
  if (vec <= 1) return launch_rows<kNoise, 1>(x, M, H, w, eps, sigma, delta, y, amax, dev, st);
  if (vec == 2) return launch_rows<kNoise, 2>(x, M, H, w, eps, sigma, delta, y, amax, dev, st);
  if (vec == 3) return launch_rows<kNoise, 3>(x, M, H, w, eps, sigma, delta, y, amax, dev, st);
  return launch_rows<kNoise, 4>(x, M, H, w, eps, sigma, delta, y, amax, dev, st);
}

}  // namespace

nvfp4rl_status launch_rmsnorm_aqn(const uint16_t* x, int64_t M, int64_t H, const float* w, const float* eps,
                                  float sigma, float delta, uint16_t* y, const DeviceInfo& dev, cudaStream_t st,
                                  uint32_t* amax) {
  if (M == 0) return NVFP4RL_OK;
  const cudaError_t e = eps ? launch_vec<true>(x, M, H, w, eps, sigma, delta, y, amax, dev, st)
                            : launch_vec<false>(x, M, H, w, eps, sigma, delta, y, amax, dev, st);
  if (e != cudaSuccess) return NVFP4RL_ERR_CUDA;
  return launch_status();
}

// Largest H the kernel keeps in registers.
int64_t rmsnorm_max_h() { return static_cast<int64_t>(kMaxVecPerThread) * 8 * kThreads; }

}  // namespace nvfp4rl
