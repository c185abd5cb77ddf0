// AQN-noised RMSNorm (sm_103a).
//
// QeRL explainer, section "ゼロオーバーヘッド：レイヤー正規化への統合": the noise vector
// is folded into the RMSNorm weight, X_noise = (Z_noise + w) * X / sqrt(sum(X^2) + delta),
// so channel-wise additive noise becomes row-wise multiplicative noise with no extra
// parameters; the mean of squares is used, as in standard RMSNorm. The noise is
// z = sigma * eps with eps standard-normal draws passed in and sigma from the
// exponential schedule (section "AQNの仕組み").
//
// One CTA per row: the row (H bf16) is read once with 128-bit loads into registers,
// the sum of squares is reduced with warp shuffles, and (w + sigma*eps) * x * r is
// written as bf16. w + sigma*eps is formed in fp32: late in the schedule sigma is far
// below a bf16 ulp of w, so a 16-bit weight would lose the noise.
#include "common.cuh"

namespace nvfp4rl {
namespace {

constexpr int kThreads = 256;
constexpr int kMaxVecPerThread = 4;  // H <= 4 * 8 * 256 = 8192 keeps the row in registers

template <bool kNoise>
__global__ void __launch_bounds__(kThreads) rmsnorm_aqn_kernel(const uint16_t* __restrict__ x, int64_t H,
                                                               const float* __restrict__ w,
                                                               const float* __restrict__ eps, float sigma,
                                                               float delta, uint16_t* __restrict__ y) {
  griddep_wait();
  griddep_launch_dependents();
  const int64_t row = blockIdx.x;
  const int nvec = static_cast<int>(H / 8);
  const uint4* xr = reinterpret_cast<const uint4*>(x + row * H);
  uint4 v[kMaxVecPerThread];
  float ss = 0.0f;
#pragma unroll
  for (int i = 0; i < kMaxVecPerThread; ++i) {
    const int j = threadIdx.x + i * kThreads;
    if (j < nvec) {
      v[i] = ld_nc_v4(xr + j);
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
  __shared__ float red[kThreads / 32];
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = ss;
  __syncthreads();
  float tot = 0.0f;
#pragma unroll
  for (int i = 0; i < kThreads / 32; ++i) tot += red[i];
  const float r = rsqrtf(tot / static_cast<float>(H) + delta);

  uint4* yr = reinterpret_cast<uint4*>(y + row * H);
#pragma unroll
  for (int i = 0; i < kMaxVecPerThread; ++i) {
    const int j = threadIdx.x + i * kThreads;
    if (j < nvec) {
      const float4 w0 = __ldg(reinterpret_cast<const float4*>(w) + 2 * j);
      const float4 w1 = __ldg(reinterpret_cast<const float4*>(w) + 2 * j + 1);
      float wt[8] = {w0.x, w0.y, w0.z, w0.w, w1.x, w1.y, w1.z, w1.w};
      if (kNoise) {
        const float4 e0 = __ldg(reinterpret_cast<const float4*>(eps) + 2 * j);
        const float4 e1 = __ldg(reinterpret_cast<const float4*>(eps) + 2 * j + 1);
        const float et[8] = {e0.x, e0.y, e0.z, e0.w, e1.x, e1.y, e1.z, e1.w};
#pragma unroll
        for (int t = 0; t < 8; ++t) wt[t] = fmaf(sigma, et[t], wt[t]);
      }
      const uint32_t q[4] = {v[i].x, v[i].y, v[i].z, v[i].w};
      uint32_t o[4];
#pragma unroll
      for (int t = 0; t < 4; ++t) {
        const float a = __uint_as_float(bf16_lo_bits(q[t])) * r * wt[2 * t];
        const float b = __uint_as_float(bf16_hi_bits(q[t])) * r * wt[2 * t + 1];
        o[t] = f32_to_bf16_bits(a) | (f32_to_bf16_bits(b) << 16);
      }
      yr[j] = make_uint4(o[0], o[1], o[2], o[3]);
    }
  }
}

}  // namespace

nvfp4rl_status launch_rmsnorm_aqn(const uint16_t* x, int64_t M, int64_t H, const float* w, const float* eps,
                                  float sigma, float delta, uint16_t* y, const DeviceInfo&, cudaStream_t st) {
  if (M == 0) return NVFP4RL_OK;
  const cudaError_t e =
      eps ? launch_pdl(rmsnorm_aqn_kernel<true>, dim3(static_cast<unsigned>(M)), dim3(kThreads), 0, st, x, H, w, eps,
                       sigma, delta, y)
          : launch_pdl(rmsnorm_aqn_kernel<false>, dim3(static_cast<unsigned>(M)), dim3(kThreads), 0, st, x, H, w, eps,
                       sigma, delta, y);
  if (e != cudaSuccess) return NVFP4RL_ERR_CUDA;
  return launch_status();
}

// Largest H the kernel keeps in registers.
int64_t rmsnorm_max_h() { return static_cast<int64_t>(kMaxVecPerThread) * 8 * kThreads; }

}  // namespace nvfp4rl
