// NVFP4-weight linear layer with the LoRA branch fused (W4A16 and W4A4), sm_103a.
//
// QeRL explainer, section "NVFP4量子化とLoRA": frozen NVFP4 base weights plus trainable
// low-rank factors; Y = x deq(W)^T + s (x A^T) B^T. TRACE summary, sections "論文が取り組む
// 課題" / "実験結果と性能": the rollout also runs with FP4 activations (W4A4): x is
// quantized on the fly with the same recipe (one per-tensor g_x) and the LoRA branch
// keeps the bf16 x. Grouped W4A4 runs one weight matrix per MoE expert over that
// expert's contiguous rows.
//
// This file holds the portable tensor-core path: the weight tile is dequantized from
// its 4-bit codes into bf16 in shared memory (code * E4M3(s) is exact in bf16: at most
// 6 significant bits), the bf16 activation tile is staged beside it, and warps run
// mma.sync m16n8k16 with fp32 accumulation. The per-tensor factors (w_g, and g_x for
// W4A4) and the LoRA up-projection are applied in the epilogue kernel. K is split
// across CTAs; partial sums meet in an fp32 workspace through atomic adds.
#include <algorithm>

#include "common.cuh"

namespace nvfp4rl {
namespace {

constexpr int kBN = 128;  // weight rows per CTA
constexpr int kBM = 64;   // activation rows (tokens) per CTA
constexpr int kBK = 64;   // K per main-loop step
constexpr int kPad = 8;   // bf16 elements of row padding (conflict-free ldmatrix)
constexpr int kThreads = 256;

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void ldmatrix_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

__device__ __forceinline__ void mma_bf16_16816(float c[4], const uint32_t a[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// bf16 bits of e2m1(code) * dec: exact, sign kept.
__device__ __forceinline__ uint32_t dequant_bf16(uint32_t code, float dec) {
  const uint32_t mag = code & 7u;
  const uint32_t gbits = mag >= 2u ? (0x3F00u + (mag << 6)) : (mag ? 0x3F00u : 0u);  // bf16 of the grid value
  const float v = __uint_as_float(gbits << 16) * dec;
  return (__float_as_uint(v) >> 16) | ((code & 8u) << 12);
}

// Expert of a routed row (or of a tile) by binary search over non-decreasing starts.
__device__ __forceinline__ int find_group(const int32_t* starts, int groups, int64_t v) {
  int lo = 0, hi = groups - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (starts[mid] <= v) lo = mid;
    else hi = mid - 1;
  }
  return lo;
}

// U[m][j] = sum_k x[m][k] A[j][k] in fp32 (LoRA down-projection). One CTA per row, one warp per j.
__global__ void __launch_bounds__(kThreads) lora_down_kernel(const uint16_t* __restrict__ x, int64_t K,
                                                             const uint16_t* __restrict__ A, int r,
                                                             float* __restrict__ U) {
  const int64_t m = blockIdx.x;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint4* xr = reinterpret_cast<const uint4*>(x + m * K);
  for (int j = warp; j < r; j += kThreads / 32) {
    const uint4* ar = reinterpret_cast<const uint4*>(A + static_cast<int64_t>(j) * K);
    float acc = 0.0f;
    for (int64_t v = lane; v < K / 8; v += 32) {
      const uint4 xv = xr[v], av = __ldg(ar + v);
      const uint32_t xq[4] = {xv.x, xv.y, xv.z, xv.w}, aq[4] = {av.x, av.y, av.z, av.w};
#pragma unroll
      for (int t = 0; t < 4; ++t) {
        acc = fmaf(__uint_as_float(bf16_lo_bits(xq[t])), __uint_as_float(bf16_lo_bits(aq[t])), acc);
        acc = fmaf(__uint_as_float(bf16_hi_bits(xq[t])), __uint_as_float(bf16_hi_bits(aq[t])), acc);
      }
    }
    acc = warp_sum(acc);
    if (lane == 0) U[m * r + j] = acc;
  }
}

// W4A4 operand: xb[m][k] = bf16(e2m1(code) * E4M3(s)), the quantized activation without g_x.
__global__ void __launch_bounds__(kThreads) dequant_rows_kernel(const uint8_t* __restrict__ codes,
                                                                const uint8_t* __restrict__ scales, int64_t n8,
                                                                uint16_t* __restrict__ out) {
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n8; i += stride) {
    const uint32_t cw = reinterpret_cast<const uint32_t*>(codes)[i];  // 8 codes
    const float dec = e4m3_decode_pos(scales[i >> 1]);
    uint32_t o[4];
#pragma unroll
    for (int t = 0; t < 4; ++t)
      o[t] = dequant_bf16((cw >> (8 * t)) & 15u, dec) | (dequant_bf16((cw >> (8 * t + 4)) & 15u, dec) << 16);
    reinterpret_cast<uint4*>(out)[i] = make_uint4(o[0], o[1], o[2], o[3]);
  }
}

// tile_start[e] = sum over e' < e of ceil(rows(e') / kBM); tile_start[groups] = total tiles.
__global__ void __launch_bounds__(1024) tile_map_kernel(const int32_t* __restrict__ offsets, int groups,
                                                        int32_t* __restrict__ tile_start) {
  __shared__ int32_t s[1024];
  const int e = threadIdx.x;
  const int32_t t = e < groups ? (offsets[e + 1] - offsets[e] + kBM - 1) / kBM : 0;
  s[e] = t;
  __syncthreads();
  for (int o = 1; o < 1024; o <<= 1) {
    const int32_t add = e >= o ? s[e - o] : 0;
    __syncthreads();
    s[e] += add;
    __syncthreads();
  }
  // s[e] is the inclusive prefix sum
  if (e < groups) tile_start[e + 1] = s[e];
  if (e == 0) tile_start[0] = 0;
}

__global__ void __launch_bounds__(kThreads) gemm_dequant_mma_kernel(
    const uint16_t* __restrict__ xb, int64_t M, int64_t K, int64_t N, const uint8_t* __restrict__ wc,
    const uint8_t* __restrict__ wsc, float* __restrict__ acc, int64_t k_split,
    const int32_t* __restrict__ offsets, const int32_t* __restrict__ tile_start, int groups) {
  __shared__ __align__(16) uint16_t Ws[kBN][kBK + kPad];
  __shared__ __align__(16) uint16_t Xs[kBM][kBK + kPad];

  int64_t m0, m_end;
  int e = 0;
  if (offsets) {
    const int t = blockIdx.y;
    if (t >= tile_start[groups]) return;
    e = find_group(tile_start, groups, t);
    m0 = offsets[e] + static_cast<int64_t>(t - tile_start[e]) * kBM;
    m_end = offsets[e + 1];
  } else {
    m0 = static_cast<int64_t>(blockIdx.y) * kBM;
    m_end = M;
  }
  const int64_t n0 = static_cast<int64_t>(blockIdx.x) * kBN;
  const int64_t kb = static_cast<int64_t>(blockIdx.z) * k_split;
  const int64_t ke = min(K, kb + k_split);
  const uint8_t* wce = wc + static_cast<int64_t>(e) * N * (K / 2);
  const uint8_t* wse = wsc + static_cast<int64_t>(e) * N * (K / 16);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int wn = warp & 3, wm = warp >> 2;
  float c[2][4][4];
#pragma unroll
  for (int i = 0; i < 2; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j)
#pragma unroll
      for (int q = 0; q < 4; ++q) c[i][j][q] = 0.0f;

  for (int64_t k0 = kb; k0 < ke; k0 += kBK) {
    {  // dequantize 128 x 64 weights: thread -> (row, 32-code half)
      const int row = tid >> 1, half = tid & 1;
      const uint4 cw = *reinterpret_cast<const uint4*>(wce + (n0 + row) * (K / 2) + k0 / 2 + half * 16);
      const uint8_t* sp = wse + (n0 + row) * (K / 16) + k0 / 16 + half * 2;
      const float d0 = e4m3_decode_pos(sp[0]), d1 = e4m3_decode_pos(sp[1]);
      const uint32_t words[4] = {cw.x, cw.y, cw.z, cw.w};
      uint32_t o[16];
#pragma unroll
      for (int wi = 0; wi < 4; ++wi)
#pragma unroll
        for (int t = 0; t < 4; ++t) {
          const float d = wi < 2 ? d0 : d1;
          o[wi * 4 + t] = dequant_bf16((words[wi] >> (8 * t)) & 15u, d) |
                          (dequant_bf16((words[wi] >> (8 * t + 4)) & 15u, d) << 16);
        }
      uint4* dst = reinterpret_cast<uint4*>(&Ws[row][half * 32]);
#pragma unroll
      for (int q = 0; q < 4; ++q) dst[q] = make_uint4(o[4 * q], o[4 * q + 1], o[4 * q + 2], o[4 * q + 3]);
    }
#pragma unroll
    for (int cc = 0; cc < 2; ++cc) {  // activation tile: 64 rows x 8 chunks of 16 B
      const int chunk = tid + cc * kThreads;
      const int tr = chunk >> 3, kc = chunk & 7;
      const int64_t m = m0 + tr;
      uint4 v = make_uint4(0, 0, 0, 0);
      if (m < m_end) v = *reinterpret_cast<const uint4*>(xb + m * K + k0 + kc * 8);
      *reinterpret_cast<uint4*>(&Xs[tr][kc * 8]) = v;
    }
    __syncthreads();
#pragma unroll
    for (int kk = 0; kk < kBK / 16; ++kk) {
      uint32_t a[2][4];
#pragma unroll
      for (int i = 0; i < 2; ++i)
        ldmatrix_x4(smem_u32(&Ws[wn * 32 + i * 16 + (lane & 15)][kk * 16 + (lane >> 4) * 8]), a[i][0], a[i][1],
                    a[i][2], a[i][3]);
      uint32_t b[4][2];
#pragma unroll
      for (int j2 = 0; j2 < 2; ++j2) {
        const int q = lane >> 3;
        const int tok = wm * 32 + j2 * 16 + (q >> 1) * 8 + (lane & 7);
        ldmatrix_x4(smem_u32(&Xs[tok][kk * 16 + (q & 1) * 8]), b[2 * j2][0], b[2 * j2][1], b[2 * j2 + 1][0],
                    b[2 * j2 + 1][1]);
      }
#pragma unroll
      for (int i = 0; i < 2; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) mma_bf16_16816(c[i][j], a[i], b[j][0], b[j][1]);
    }
    __syncthreads();
  }
  // C fragment: c0,c1 at (weight row lane/4, tokens 2(lane%4), +1); c2,c3 at weight row +8
#pragma unroll
  for (int i = 0; i < 2; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j)
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const int64_t n = n0 + wn * 32 + i * 16 + (lane >> 2) + (q >> 1) * 8;
        const int64_t m = m0 + wm * 32 + j * 8 + 2 * (lane & 3) + (q & 1);
        if (m < m_end) atomicAdd(acc + m * N + n, c[i][j][q]);
      }
}

// y[m][n] = bf16(scale * acc[m][n] + s * sum_j U[m][j] B[n][j]); scale = w_g[e] (* g_x).
__global__ void __launch_bounds__(kThreads) epilogue_kernel(const float* __restrict__ acc, int64_t N,
                                                            const float* __restrict__ w_g,
                                                            const float* __restrict__ g_x,
                                                            const float* __restrict__ U,
                                                            const uint16_t* __restrict__ B, int r, float s,
                                                            const int32_t* __restrict__ offsets, int groups,
                                                            uint16_t* __restrict__ y) {
  __shared__ float u[256];
  const int64_t m = blockIdx.y;
  for (int j = threadIdx.x; j < r; j += blockDim.x) u[j] = U[m * r + j];
  __syncthreads();
  const int e = offsets ? find_group(offsets, groups, m) : 0;
  float scale = w_g[e];
  if (g_x) scale *= *g_x;
  const int64_t n = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (n >= N) return;
  float v = scale * acc[m * N + n];
  if (r) {
    float l = 0.0f;
    const uint16_t* br = B + n * r;
    for (int j = 0; j < r; ++j) l = fmaf(u[j], __uint_as_float(static_cast<uint32_t>(br[j]) << 16), l);
    v = fmaf(s, l, v);
  }
  y[m * N + n] = static_cast<uint16_t>(f32_to_bf16_bits(v));
}

struct WsLayout {
  size_t acc, U, tiles, xcodes, xscales, amax, gx, xb, total;
};

WsLayout layout(bool w4a4, int64_t M, int64_t N, int64_t K, int r, int groups) {
  WsLayout L{};
  size_t o = 0;
  auto take = [&](size_t bytes) {
    const size_t at = o;
    o = align_up(o + bytes, 256);
    return at;
  };
  L.acc = take(static_cast<size_t>(M) * N * 4);
  L.U = take(static_cast<size_t>(M) * std::max(r, 1) * 4);
  L.tiles = take(static_cast<size_t>(groups + 2) * 4);
  if (w4a4) {
    L.xcodes = take(static_cast<size_t>(M) * K / 2);
    L.xscales = take(static_cast<size_t>(M) * K / 16);
    L.amax = take(kQuantizeWorkspace);
    L.gx = take(16);
    L.xb = take(static_cast<size_t>(M) * K * 2);
  }
  L.total = o;
  return L;
}

}  // namespace

size_t linear_workspace_bytes(bool w4a4, int64_t M, int64_t N, int64_t K, int r, int groups) {
  if (!w4a4 && w4a16_tc_supported(M, N, K, r)) return w4a16_tc_workspace_bytes(M, N, K, r, kPlanSMs);
  if (w4a4 && w4a4_tc_supported(M, N, K, r)) return w4a4_tc_workspace_bytes(M, N, K, r, groups);
  return layout(w4a4, M, N, K, r, groups).total;
}

nvfp4rl_status launch_linear(const LinearArgs& a, void* ws, size_t ws_bytes, const DeviceInfo& dev, cudaStream_t st) {
  if (a.M == 0) return NVFP4RL_OK;
  if (!a.w4a4 && w4a16_tc_supported(a.M, a.N, a.K, a.r)) return launch_w4a16_tc(a, ws, ws_bytes, dev, st);
  if (a.w4a4 && w4a4_tc_supported(a.M, a.N, a.K, a.r)) return launch_w4a4_tc(a, ws, ws_bytes, dev, st);
  const int groups = a.offsets ? a.groups : 1;
  const WsLayout L = layout(a.w4a4, a.M, a.N, a.K, a.r, groups);
  if (ws_bytes < L.total) return NVFP4RL_ERR_WORKSPACE;
  char* base = static_cast<char*>(ws);
  float* acc = reinterpret_cast<float*>(base + L.acc);
  float* U = reinterpret_cast<float*>(base + L.U);
  int32_t* tiles = reinterpret_cast<int32_t*>(base + L.tiles);

  if (cudaMemsetAsync(acc, 0, static_cast<size_t>(a.M) * a.N * 4, st) != cudaSuccess) return NVFP4RL_ERR_CUDA;
  if (a.r > 0) {
    lora_down_kernel<<<static_cast<unsigned>(a.M), kThreads, 0, st>>>(a.x, a.K, a.A, a.r, U);
    if (launch_status() != NVFP4RL_OK) return NVFP4RL_ERR_CUDA;
  }
  const uint16_t* xb = a.x;
  const float* gx = nullptr;
  if (a.w4a4) {
    uint8_t* xc = reinterpret_cast<uint8_t*>(base + L.xcodes);
    uint8_t* xs = reinterpret_cast<uint8_t*>(base + L.xscales);
    float* gxp = reinterpret_cast<float*>(base + L.gx);
    uint16_t* xbp = reinterpret_cast<uint16_t*>(base + L.xb);
    nvfp4rl_status stq = launch_quantize(a.x, NVFP4RL_BF16, a.M, a.K, nullptr, xc, xs, gxp, nullptr,
                                         reinterpret_cast<uint32_t*>(base + L.amax), dev, st);
    if (stq != NVFP4RL_OK) return stq;
    const int64_t n8 = a.M * a.K / 8;
    const int grid = static_cast<int>(std::min<int64_t>((n8 + kThreads - 1) / kThreads, dev.sm_count * 8));
    dequant_rows_kernel<<<grid, kThreads, 0, st>>>(xc, xs, n8, xbp);
    if (launch_status() != NVFP4RL_OK) return NVFP4RL_ERR_CUDA;
    xb = xbp;
    gx = gxp;
  }
  int64_t m_tiles;
  if (a.offsets) {
    tile_map_kernel<<<1, 1024, 0, st>>>(a.offsets, groups, tiles);
    if (launch_status() != NVFP4RL_OK) return NVFP4RL_ERR_CUDA;
    m_tiles = (a.M + kBM - 1) / kBM + groups;  // upper bound on sum_e ceil(rows_e / kBM)
  } else {
    m_tiles = (a.M + kBM - 1) / kBM;
  }
  const int64_t n_tiles = a.N / kBN;
  const int64_t ksteps = a.K / kBK;
  const int64_t target = static_cast<int64_t>(dev.sm_count) * 4;
  int64_t splits = std::max<int64_t>(1, std::min<int64_t>(ksteps, target / std::max<int64_t>(1, n_tiles * m_tiles)));
  const int64_t steps_per = (ksteps + splits - 1) / splits;
  splits = (ksteps + steps_per - 1) / steps_per;
  dim3 grid(static_cast<unsigned>(n_tiles), static_cast<unsigned>(m_tiles), static_cast<unsigned>(splits));
  gemm_dequant_mma_kernel<<<grid, kThreads, 0, st>>>(xb, a.M, a.K, a.N, a.w_codes, a.w_scales, acc,
                                                     steps_per * kBK, a.offsets, tiles, groups);
  if (launch_status() != NVFP4RL_OK) return NVFP4RL_ERR_CUDA;
  dim3 eg(static_cast<unsigned>((a.N + kThreads - 1) / kThreads), static_cast<unsigned>(a.M));
  epilogue_kernel<<<eg, kThreads, 0, st>>>(acc, a.N, a.w_g, gx, U, a.B, a.r, a.s, a.offsets, groups, a.y);
  return launch_status();
}

}  // namespace nvfp4rl
