// AIS mixing coefficient over a batch of tokens (sm_103a).
//
// AIS summary, section 2.1 "混合係数": from statistics the policy update already has, the
// correction strength is alpha = clip(alpha_ess - beta alpha_var, 0, 1) alpha_mis, with
//   alpha_ess = (1 + CV^2(w))^-1/2           (reliability of the truncated weights w),
//   alpha_mis = min(1, dbar / delta)          (mean absolute log-prob mismatch, saturating),
//   alpha_var = max(0, (dsigma - gamma) / gamma) (variance amplification beyond a tolerance);
// section 2.2: each token's weight in the GRPO objective becomes w~ = 1 + alpha (min(rho, C) - 1).
// Per token rho = exp(logp_train - logp_rollout), w = min(rho, C); statistics over the n tokens
// with weight 1/n; dsigma = std(w A) / std(A) - 1 (0 when std(A) = 0).
//
// Three kernels, chained by programmatic dependent launch (no grid-wide wait anywhere): a
// one-thread clear of the ticket word, then two that do the work. ais_reduce_kernel: each thread streams its tokens (128-bit loads) and sums seven quantities --
// w', w'^2, |d|, A', A'^2, (wA)', (wA)'^2, each ' marking a shift by token 0's value, so that every
// variance keeps its digits and constant data gives exactly zero -- in plain fp32 over chunks of 16
// tokens, each chunk added to compensated (Kahan) fp32 sums; the warp and block
// trees add (hi, lo) fp32 pairs with TwoSum (about 44 bits), and each CTA writes its pairs to its
// slot of the workspace and takes a ticket. The CTA that takes the last ticket adds the slots in
// slot order (one warp per quantity, again in pairs) and computes alpha and the statistics: the
// means and the variances (differences of means) in fp64 multiplications, the rest in fp32
// (fp64 division and square root are slow on this GPU and the results need no more). The
// result does not depend on which CTA finishes last. ais_weights_kernel then rewrites every
// token's weight with that alpha (the log-probs are read again, from L2 at the sizes of a
// training batch).
#include "common.cuh"

namespace nvfp4rl {
namespace {

constexpr int kAisThreads = 1024;
constexpr int kAisSums = 7;

struct AisParams {
  float C, delta, gamma, beta;
};

// An unevaluated sum hi + lo of two floats (|lo| <= ulp(hi) / 2 after df_add).
struct DF {
  float hi, lo;
};

// (a.hi + a.lo) + (b.hi + b.lo): TwoSum of the heads (exact error term), tails added to the error.
__device__ __forceinline__ DF df_add(DF a, DF b) {
  const float s = __fadd_rn(a.hi, b.hi);
  const float v = __fsub_rn(s, a.hi);
  float e = __fadd_rn(__fsub_rn(a.hi, __fsub_rn(s, v)), __fsub_rn(b.hi, v));
  e = __fadd_rn(e, __fadd_rn(a.lo, b.lo));
  const float hi = __fadd_rn(s, e);
  return {hi, __fsub_rn(e, __fsub_rn(hi, s))};
}

__device__ __forceinline__ DF warp_sum_df(DF v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1)
    v = df_add(v, DF{__shfl_xor_sync(0xFFFFFFFFu, v.hi, o), __shfl_xor_sync(0xFFFFFFFFu, v.lo, o)});
  return v;
}

// Compensated running sum (Kahan): sum - c is the exact running total to within a few ulp.
struct Kahan {
  float sum = 0.0f, c = 0.0f;
  __device__ __forceinline__ void add(float x) {
    const float y = __fsub_rn(x, c);
    const float t = __fadd_rn(sum, y);
    c = __fsub_rn(__fsub_rn(t, sum), y);
    sum = t;
  }
};

// Token 0's values, by which every term is shifted (the same in every thread): the variance of
// shifted data keeps its digits, and constant data gives exactly zero.
struct Shift {
  float w, a, wa;
};

// One token's terms, added in plain fp32 to a chunk sum c (at most 16 tokens per chunk).
__device__ __forceinline__ void accumulate(float lr, float lt, float a, float C, const Shift& k,
                                           float (&c)[kAisSums]) {
  const float d = lt - lr;
  const float w = fminf(expf(d), C);
  const float ws = w - k.w, as = a - k.a, was = w * a - k.wa;
  c[0] += ws;
  c[1] = fmaf(ws, ws, c[1]);
  c[2] += fabsf(d);
  c[3] += as;
  c[4] = fmaf(as, as, c[4]);
  c[5] += was;
  c[6] = fmaf(was, was, c[6]);
}

// A chunk's sums into the compensated running sums, the chunk restarted.
__device__ __forceinline__ void fold(float (&c)[kAisSums], Kahan (&s)[kAisSums]) {
#pragma unroll
  for (int q = 0; q < kAisSums; ++q) {
    s[q].add(c[q]);
    c[q] = 0.0f;
  }
}

__global__ void __launch_bounds__(kAisThreads, 1)
    ais_reduce_kernel(const float* __restrict__ lr, const float* __restrict__ lt, const float* __restrict__ adv,
                      int64_t n, AisParams p, double* __restrict__ stats, float2* __restrict__ slots,
                      unsigned int* __restrict__ ticket, float* __restrict__ alpha_out) {
  __shared__ DF part[kAisSums][32];
  __shared__ DF tot[kAisSums];
  __shared__ int last;
  griddep_wait();  // the ticket was cleared by the preceding kernel
  griddep_launch_dependents();
  const int64_t G = gridDim.x;
  const int64_t tid = static_cast<int64_t>(blockIdx.x) * kAisThreads + threadIdx.x;
  const int64_t nthreads = G * kAisThreads;
  const int64_t n4 = n / 4;
  Shift k0;
  k0.w = fminf(expf(__ldg(lt) - __ldg(lr)), p.C);
  k0.a = __ldg(adv);
  k0.wa = k0.w * k0.a;
  Kahan s[kAisSums];
  float c[kAisSums] = {0, 0, 0, 0, 0, 0, 0};
  int in_chunk = 0;
#pragma unroll 2
  for (int64_t j = tid; j < n4; j += nthreads) {
    const float4 r = __ldg(reinterpret_cast<const float4*>(lr) + j);
    const float4 t = __ldg(reinterpret_cast<const float4*>(lt) + j);
    const float4 a = __ldg(reinterpret_cast<const float4*>(adv) + j);
    accumulate(r.x, t.x, a.x, p.C, k0, c);
    accumulate(r.y, t.y, a.y, p.C, k0, c);
    accumulate(r.z, t.z, a.z, p.C, k0, c);
    accumulate(r.w, t.w, a.w, p.C, k0, c);
    if (++in_chunk == 4) {  // 16 tokens
      fold(c, s);
      in_chunk = 0;
    }
  }
  // the last n % 4 tokens: one per thread of the first threads of the grid
  if (4 * n4 + tid < n) accumulate(lr[4 * n4 + tid], lt[4 * n4 + tid], adv[4 * n4 + tid], p.C, k0, c);
  fold(c, s);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
#pragma unroll
  for (int k = 0; k < kAisSums; ++k) {
    const DF v = warp_sum_df(DF{s[k].sum, -s[k].c});
    if (lane == 0) part[k][warp] = v;
  }
  __syncthreads();
  if (warp < kAisSums) {  // warp k: quantity k over the 32 warps, in a fixed tree
    const DF v = warp_sum_df(part[warp][lane]);
    if (lane == 0) {
      slots[blockIdx.x * 8 + warp] = make_float2(v.hi, v.lo);
      __threadfence();  // visible to the last CTA before this CTA's ticket
    }
  }
  __syncthreads();
  if (threadIdx.x == 0) last = atomicAdd(ticket, 1u) == static_cast<unsigned int>(G - 1);
  __syncthreads();
  if (!last) return;
  __threadfence();  // every other CTA's slots are visible from here on
  if (warp < kAisSums) {  // quantity `warp` over all slots: lane-strided pairs, then a fixed tree
    DF v{0.0f, 0.0f};
    for (int64_t c = lane; c < G; c += 32) {
      const float2 q = __ldcg(slots + c * 8 + warp);
      v = df_add(v, DF{q.x, q.y});
    }
    v = warp_sum_df(v);
    if (lane == 0) tot[warp] = v;
  }
  __syncthreads();
  if (threadIdx.x != 0) return;
  const auto val = [&](int k) { return static_cast<double>(tot[k].hi) + static_cast<double>(tot[k].lo); };
  const double inv_n = 1.0 / static_cast<double>(n);
  const double m1 = val(0) * inv_n;                          // mean(w) - w_0
  const double vw = fmax(0.0, val(1) * inv_n - m1 * m1);     // population variance of w
  const double mw = static_cast<double>(k0.w) + m1;
  const double dbar = val(2) * inv_n;
  const double ma = val(3) * inv_n, va = fmax(0.0, val(4) * inv_n - ma * ma);
  const double mwa = val(5) * inv_n, vwa = fmax(0.0, val(6) * inv_n - mwa * mwa);
  const float cv2 = static_cast<float>(vw) / static_cast<float>(mw * mw);
  const float a_ess = 1.0f / sqrtf(1.0f + cv2);
  const float a_mis = fminf(1.0f, static_cast<float>(dbar) / p.delta);
  const float amp = va > 0.0 ? sqrtf(static_cast<float>(vwa) / static_cast<float>(va)) - 1.0f : 0.0f;
  const float a_var = fmaxf(0.0f, (amp - p.gamma) / p.gamma);
  const float alpha = fminf(1.0f, fmaxf(0.0f, a_ess - p.beta * a_var)) * a_mis;
  stats[0] = alpha;
  stats[1] = a_ess;
  stats[2] = a_mis;
  stats[3] = a_var;
  stats[4] = dbar;
  stats[5] = cv2;
  stats[6] = amp;
  stats[7] = mw;
  *alpha_out = alpha;
}

// w~ = 1 + alpha (min(exp(logp_train - logp_rollout), C) - 1) for every token.
__global__ void __launch_bounds__(512) ais_weights_kernel(const float* __restrict__ lr, const float* __restrict__ lt,
                                                          int64_t n, float C, const float* __restrict__ alpha_in,
                                                          float* __restrict__ w_out) {
  griddep_wait();  // alpha is written by the preceding kernel
  griddep_launch_dependents();
  const float alpha = __ldcg(alpha_in);
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  const int64_t tid = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  const int64_t n4 = n / 4;
  for (int64_t j = tid; j < n4; j += stride) {
    const float4 r = __ldcg(reinterpret_cast<const float4*>(lr) + j);
    const float4 t = __ldcg(reinterpret_cast<const float4*>(lt) + j);
    float4 o;
    o.x = fmaf(alpha, fminf(expf(t.x - r.x), C) - 1.0f, 1.0f);
    o.y = fmaf(alpha, fminf(expf(t.y - r.y), C) - 1.0f, 1.0f);
    o.z = fmaf(alpha, fminf(expf(t.z - r.z), C) - 1.0f, 1.0f);
    o.w = fmaf(alpha, fminf(expf(t.w - r.w), C) - 1.0f, 1.0f);
    __stcs(reinterpret_cast<float4*>(w_out) + j, o);
  }
  if (4 * n4 + tid < n) {
    const int64_t i = 4 * n4 + tid;
    w_out[i] = fmaf(alpha, fminf(expf(lt[i] - lr[i]), C) - 1.0f, 1.0f);
  }
}

// Clears the ticket counter (a kernel rather than a memset, so that it chains by programmatic
// dependent launch).
__global__ void ais_clear_kernel(unsigned int* __restrict__ ticket) {
  griddep_wait();
  griddep_launch_dependents();
  if (threadIdx.x == 0) *ticket = 0u;
}

}  // namespace

size_t ais_workspace_bytes() { return 256 + static_cast<size_t>(kAisMaxCtas) * 8 * sizeof(float2); }

nvfp4rl_status launch_ais(const float* lr, const float* lt, const float* adv, int64_t n, float C, float delta,
                          float gamma, float beta, float* w_out, double* stats, void* workspace,
                          const DeviceInfo& dev, cudaStream_t st) {
  if (n == 0) return NVFP4RL_OK;
  // workspace: the ticket (bytes 0-3), alpha as fp32 (bytes 16-19), then one slot of 8 (hi, lo)
  // pairs per CTA from byte 256
  auto* ticket = static_cast<unsigned int*>(workspace);
  auto* alpha = reinterpret_cast<float*>(static_cast<uint8_t*>(workspace) + 16);
  auto* slots = reinterpret_cast<float2*>(static_cast<uint8_t*>(workspace) + 256);
  if (launch_pdl(ais_clear_kernel, dim3(1), dim3(32), 0, st, ticket) != cudaSuccess) return NVFP4RL_ERR_CUDA;
  if (launch_status() != NVFP4RL_OK) return NVFP4RL_ERR_CUDA;
  const int64_t want = (n / 4 + kAisThreads - 1) / kAisThreads;
  const int64_t G = std::max<int64_t>(1, std::min<int64_t>({want, static_cast<int64_t>(dev.sm_count),
                                                              static_cast<int64_t>(kAisMaxCtas)}));
  const AisParams p{C, delta, gamma, beta};
  if (launch_pdl(ais_reduce_kernel, dim3(static_cast<unsigned>(G)), dim3(kAisThreads), 0, st, lr, lt, adv, n, p, stats,
                 slots, ticket, alpha) != cudaSuccess)
    return NVFP4RL_ERR_CUDA;
  if (launch_status() != NVFP4RL_OK) return NVFP4RL_ERR_CUDA;
  if (!w_out) return NVFP4RL_OK;
  const int64_t want2 = (n / 4 + 511) / 512;
  const int64_t G2 = std::max<int64_t>(1, std::min<int64_t>(want2, static_cast<int64_t>(dev.sm_count) * 4));
  if (launch_pdl(ais_weights_kernel, dim3(static_cast<unsigned>(G2)), dim3(512), 0, st, lr, lt, n, C,
                 static_cast<const float*>(alpha), w_out) != cudaSuccess)
    return NVFP4RL_ERR_CUDA;
  return launch_status();
}

}  // namespace nvfp4rl
