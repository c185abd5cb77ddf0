// LoRA down-projection U = bf16(x A^T) on tcgen05 for prefill-sized M (QeRL explainer, section
// "NVFP4量子化とLoRA": the low-rank branch runs on the unquantized bf16 activations; its first
// factor, x A^T, is what the up-projection consumes).
//
// A plain streaming GEMM: x is M x K bf16 (read once), A is r x K bf16 (r <= 128, read from L2),
// U is M x r. One CTA per 128 rows and K range; a cluster of `ks` CTAs (blockIdx.x) covers all of
// K for one row tile (blockIdx.y). Per stage a TMA loads 128 rows x 64 K of x and r rows x 64 K of
// A (128-byte rows, 128-byte swizzle) and one thread issues four kind::f16 MMAs (M = 128, N = r,
// K = 16) into a TMEM accumulator. After the K loop each CTA stores its fp32 partial tile in
// shared memory (the ring's space); after a cluster barrier CTA q sums rows [q 128 / ks, (q + 1)
// 128 / ks) over all partials in rank order (distributed shared memory) and writes U, or, for the
// W4A4 path, hi and lo of c U (LoraDownScale). The sums run through the same K ranges and rank
// order on every call, so U is deterministic.
// With `amax` the kernel also accumulates max |x| over every element it loads (fp32 bit pattern, an
// atomicMax per warp): the tensor amax that the NVFP4 encoding of x needs, without a pass of its own.
//   warp 0   TMA producer (one thread)
//   warp 1   TMEM allocation; one thread issues the MMAs
//   warps 2-3 with `amax`: each scans half of every landed x tile
//   warps 0-3 after the K loop: TMEM -> shared-memory partials, then the cluster reduction

#include <cuda.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <map>
#include <mutex>
#include <utility>

#include "common.cuh"
#include "sm100.cuh"

namespace nvfp4rl {
namespace {

using namespace sm100;

constexpr int kRows = 128;                 // rows of x per CTA (MMA M)
constexpr int kChunk = 64;                 // K per stage (128 bytes of bf16)
constexpr int kXBytes = kRows * kChunk * 2;  // 16 KB
constexpr int kMaxRank = 128;
constexpr int kStages = 6;
constexpr int kThreadsDown = 128;
constexpr int kPartStride = kMaxRank + 4;  // fp32 words per partial row (+4: fewer bank conflicts)

struct DownParams {
  int64_t M, K;
  int r;
  int chunks_per_cta;  // K chunks of a CTA (the last CTA of a cluster takes what is left)
  int nchunks;
  uint16_t* U;
  LoraDownScale ls;
  uint32_t* amax;  // or null
  uint32_t* status;
};

__device__ __forceinline__ uint32_t tmem_cols_for(int r) { return r <= 32 ? 32u : r <= 64 ? 64u : 128u; }

__global__ void __launch_bounds__(kThreadsDown, 1)
    lora_down_tc_kernel(const __grid_constant__ CUtensorMap map_x, const __grid_constant__ CUtensorMap map_a,
                        const DownParams p) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int abytes = p.r * kChunk * 2;          // A rows of one stage
  const int stage_bytes = kXBytes + abytes;      // multiple of 1024 (r a multiple of 16 -> 2 KB steps)
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + kStages * stage_bytes);
  uint64_t* empty = full + kStages;
  uint64_t* done = empty + kStages;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(done + 1);
  float* part = reinterpret_cast<float*>(smem);  // [kRows][kPartStride] after the K loop

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int q = static_cast<int>(cluster_ctarank());
  const int ks = static_cast<int>(gridDim.x);
  const int64_t m0 = static_cast<int64_t>(blockIdx.y) * kRows;
  const int c0 = q * p.chunks_per_cta;
  const int n = max(0, min(p.nchunks, c0 + p.chunks_per_cta) - c0);
  const uint32_t ncols = tmem_cols_for(p.r);

  // x (and g_x) are written by earlier kernels on the stream: wait for them before any load
  griddep_wait();
  griddep_launch_dependents();
  if (threadIdx.x == 0) {
    for (int i = 0; i < kStages; ++i) {
      mbar_init(smem_addr(&full[i]), 1);
      mbar_init(smem_addr(&empty[i]), p.amax ? 3 : 1);  // the MMAs' commit (+ the two scanning warps)
    }
    mbar_init(smem_addr(done), 1);
    fence_barrier_init();
  }
  if (warp == 1) tmem_alloc(smem_addr(tmem_slot), ncols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  bool ok = true;

  if (warp == 0 && lane == 0) {
    // ---------------------------------------------------------------- TMA producer
    prefetch_tensormap(&map_x);
    prefetch_tensormap(&map_a);
    int issued = 0;
    for (int i = 0; i < n && ok; ++i) {
      const int s = i % kStages;
      if (i >= kStages && !mbar_wait(smem_addr(&empty[s]), ((i / kStages) - 1) & 1, p.status, kStatusTimeoutProducer)) {
        ok = false;
        break;
      }
      const uint32_t bar = smem_addr(&full[s]);
      mbar_arrive_expect_tx(bar, static_cast<uint32_t>(stage_bytes));
      const int k = (c0 + i) * kChunk;
      tma_load_2d(smem_addr(smem + s * stage_bytes), &map_x, k, static_cast<int32_t>(m0), bar);
      tma_load_2d(smem_addr(smem + s * stage_bytes + kXBytes), &map_a, k, 0, bar);
      ++issued;
    }
    // do not leave with copies in flight
    for (int i = max(0, issued - kStages); i < issued; ++i)
      mbar_wait(smem_addr(&full[i % kStages]), (i / kStages) & 1, p.status, kStatusTimeoutDrain);
  } else if (warp == 1) {
    // ---------------------------------------------------------------- MMA issuer
    // The whole warp walks the chunks and waits; one elected lane issues the MMAs and commits.
    const uint32_t idesc = idesc_bf16_f32(kRows, static_cast<uint32_t>(p.r));
    for (int i = 0; i < n && ok; ++i) {
      const int s = i % kStages;
      ok = __all_sync(0xFFFFFFFFu, mbar_wait(smem_addr(&full[s]), (i / kStages) & 1, p.status, kStatusTimeoutMma));
      if (!ok) break;
      tc_fence_after();
      const uint64_t xd = smem_desc(smem_addr(smem + s * stage_bytes), 16, 1024, 2);
      const uint64_t ad = smem_desc(smem_addr(smem + s * stage_bytes + kXBytes), 16, 1024, 2);
      if (elect_one()) {
#pragma unroll
        for (int kk = 0; kk < kChunk / 16; ++kk) mma_f16_ss(tmem, xd + 2 * kk, ad + 2 * kk, idesc, (i | kk) ? 1u : 0u);
        mma_commit(smem_addr(&empty[s]));
      }
      __syncwarp();
    }
    if (elect_one()) mma_commit(smem_addr(done));  // every MMA above has completed (also when there were none)
    __syncwarp();
  } else if (p.amax && (warp == 2 || warp == 3)) {
    // ---------------------------------------------------------------- max |x| of the landed tiles
    uint32_t m2 = 0;
    const int half = warp - 2;  // bytes [half 8 KB, half 8 KB + 8 KB) of the x tile
    for (int i = 0; i < n && ok; ++i) {
      const int s = i % kStages;
      ok = __all_sync(0xFFFFFFFFu, mbar_wait(smem_addr(&full[s]), (i / kStages) & 1, p.status, kStatusTimeoutMma));
      if (!ok) break;
      const uint4* t = reinterpret_cast<const uint4*>(smem + s * stage_bytes + half * (kXBytes / 2));
#pragma unroll 4
      for (int e = lane; e < kXBytes / 2 / 16; e += 32) {
        const uint4 v = t[e];
        m2 = __vmaxu2(m2, __vmaxu2(__vmaxu2(v.x & 0x7FFF7FFFu, v.y & 0x7FFF7FFFu),
                                   __vmaxu2(v.z & 0x7FFF7FFFu, v.w & 0x7FFF7FFFu)));
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_addr(&empty[s]));
    }
    uint32_t m = max(m2 & 0xFFFFu, m2 >> 16) << 16;
    m = __reduce_max_sync(0xFFFFFFFFu, m);
    if (lane == 0) atomicMax(p.amax, m);
  }
  __syncwarp();
  // ---------------------------------------------------------------- partial tile -> shared memory
  const bool done_ok = __all_sync(0xFFFFFFFFu, mbar_wait(smem_addr(done), 0, p.status, kStatusTimeoutEpilogue));
  __syncthreads();  // the ring is free: every stage's MMAs have completed and every copy has landed
  tc_fence_after();
  {
    const int row = warp * 32 + lane;
    float* prow = part + row * kPartStride;
    for (int c = 0; c < p.r; c += 16) {
      uint32_t d[16];
      if (n > 0 && done_ok) {
        tmem_ld16(tmem + (static_cast<uint32_t>(warp * 32) << 16) + c, d);
        tmem_ld_wait();
      } else {
#pragma unroll
        for (int e = 0; e < 16; ++e) d[e] = 0u;  // an empty K range adds zeros
      }
#pragma unroll
      for (int e = 0; e < 16; e += 4)
        *reinterpret_cast<float4*>(prow + c + e) = make_float4(__uint_as_float(d[e]), __uint_as_float(d[e + 1]),
                                                               __uint_as_float(d[e + 2]), __uint_as_float(d[e + 3]));
    }
  }
  tc_fence_before();
  cluster_sync_all();  // every CTA's partial is in its shared memory
  // ---------------------------------------------------------------- reduction over the cluster, U
  float cu = 1.f;  // c of the W4A4 form
  if (p.ls.folded()) {
    const float alpha = p.ls.gx() * *p.ls.w_g;
    cu = alpha == 0.f ? p.ls.s : p.ls.s / alpha;
    if (blockIdx.x == 0 && blockIdx.y == 0 && threadIdx.x == 0 && !(fabsf(cu) <= 0x1p100f))
      atomicOr(p.ls.status, kStatusRange);
  }
  const int rb = q * kRows / ks, re = (q + 1) * kRows / ks;
  const int r4 = p.r / 4;
  for (int idx = threadIdx.x; idx < (re - rb) * r4; idx += kThreadsDown) {
    const int row = rb + idx / r4, j4 = (idx % r4) * 4;
    const int64_t m = m0 + row;
    const uint32_t local = smem_addr(part + row * kPartStride + j4);
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int sp = 0; sp < ks; ++sp) {
      const float4 v = dsmem_ld_v4(dsmem_map(local, static_cast<uint32_t>(sp)));
      acc.x += v.x;
      acc.y += v.y;
      acc.z += v.z;
      acc.w += v.w;
    }
    if (m >= p.M) continue;
    const float av[4] = {acc.x, acc.y, acc.z, acc.w};
    uint32_t o[4], lo[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const uint32_t u = f32_to_bf16_bits(av[e]);
      if (p.ls.folded()) {
        // c U = hi + lo: hi = bf16(c U), lo = bf16(c U - hi) (c U - hi is exact in fp32). U is
        // bf16(x A^T) when g_x comes from memory (W4A4: the same U as the calls that learn g_x
        // after the LoRA-down), x A^T as accumulated in fp32 when it is given by value (W4A16).
        const float cuv = (p.ls.g_x ? __uint_as_float(u << 16) : av[e]) * cu;
        o[e] = f32_to_bf16_bits(cuv);
        lo[e] = f32_to_bf16_bits(cuv - __uint_as_float(o[e] << 16));
      } else {
        o[e] = u;
      }
    }
    const int64_t at = m * p.r + j4;  // 8-byte aligned: r and j4 are multiples of 4
    *reinterpret_cast<uint2*>(p.U + at) = make_uint2(o[0] | (o[1] << 16), o[2] | (o[3] << 16));
    if (p.ls.folded())
      *reinterpret_cast<uint2*>(p.ls.lo + at) = make_uint2(lo[0] | (lo[1] << 16), lo[2] | (lo[3] << 16));
  }
  cluster_sync_all();  // partials read by every peer before any CTA leaves
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, ncols);
  }
}

}  // namespace

namespace {

// U (bf16) -> hi and lo of c U in place (hi over U, lo into `lo`), c = s / (g_x w_g) (s when that
// is 0): the form the W4A4 GEMM consumes, for a LoRA-down that ran before g_x was known.
__global__ void __launch_bounds__(256) lora_scale_kernel(uint16_t* __restrict__ U, uint16_t* __restrict__ lo,
                                                         int64_t n8, LoraDownScale ls) {
  const float alpha = ls.gx() * *ls.w_g;
  const float cu = alpha == 0.f ? ls.s : ls.s / alpha;
  if (blockIdx.x == 0 && threadIdx.x == 0 && !(fabsf(cu) <= 0x1p100f)) atomicOr(ls.status, kStatusRange);
  for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < n8;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const uint4 v = reinterpret_cast<const uint4*>(U)[i];
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
    uint32_t h[4], l[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      uint32_t hh[2], ll[2];
#pragma unroll
      for (int k = 0; k < 2; ++k) {
        const float cuv = __uint_as_float(k ? (w[e] & 0xFFFF0000u) : (w[e] << 16)) * cu;
        hh[k] = f32_to_bf16_bits(cuv);
        ll[k] = f32_to_bf16_bits(cuv - __uint_as_float(hh[k] << 16));
      }
      h[e] = hh[0] | (hh[1] << 16);
      l[e] = ll[0] | (ll[1] << 16);
    }
    reinterpret_cast<uint4*>(U)[i] = make_uint4(h[0], h[1], h[2], h[3]);
    reinterpret_cast<uint4*>(lo)[i] = make_uint4(l[0], l[1], l[2], l[3]);
  }
}

size_t down_smem_bytes(int r) {
  return 1024 + static_cast<size_t>(kStages) * (kXBytes + static_cast<size_t>(r) * kChunk * 2) + 256;
}

// Largest cluster size (<= 8) whose clusters of this kernel fit on the device at once, per device
// and rank (the shared-memory size depends on r).
int down_tc_max_cluster(int device, int r) {
  static std::mutex mu;
  static std::map<std::pair<int, int>, int> cache;
  std::lock_guard<std::mutex> lock(mu);
  const auto key = std::make_pair(device, r);
  auto it = cache.find(key);
  if (it != cache.end()) return it->second;
  const int smem = static_cast<int>(down_smem_bytes(r));
  int best = 0;
  if (cudaFuncSetAttribute(lora_down_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) == cudaSuccess) {
    for (int c = 8; c >= 1 && !best; c >>= 1) {
      cudaLaunchConfig_t cfg = {};
      cfg.gridDim = dim3(c, 1, 1);
      cfg.blockDim = dim3(kThreadsDown, 1, 1);
      cfg.dynamicSmemBytes = static_cast<size_t>(smem);
      cudaLaunchAttribute attr[1];
      attr[0].id = cudaLaunchAttributeClusterDimension;
      attr[0].val.clusterDim.x = c;
      attr[0].val.clusterDim.y = 1;
      attr[0].val.clusterDim.z = 1;
      cfg.attrs = attr;
      cfg.numAttrs = 1;
      int n = 0;
      if (cudaOccupancyMaxActiveClusters(&n, reinterpret_cast<const void*>(lora_down_tc_kernel), &cfg) == cudaSuccess &&
          n > 0)
        best = c;
    }
  }
  cudaGetLastError();
  cache[key] = best;
  return best;
}

}  // namespace

bool lora_down_tc_supported(int64_t M, int64_t K, int r) {
  return M >= kLoraDownTcMinRows && K % kChunk == 0 && r % 16 == 0 && r >= 16 && r <= kMaxRank;
}

nvfp4rl_status launch_lora_down_tc(const uint16_t* x, int64_t M, int64_t K, const uint16_t* A, int r, uint16_t* U,
                                   const DeviceInfo& dev, cudaStream_t st, const LoraDownScale& scale, uint32_t* amax) {
  const int maxc = down_tc_max_cluster(dev.device, r);
  if (maxc == 0) return NVFP4RL_ERR_CUDA;
  const int nchunks = static_cast<int>(K / kChunk);
  const int64_t row_tiles = (M + kRows - 1) / kRows;
  // split K over a cluster only as far as the row tiles alone leave SMs idle (one CTA per SM)
  int ks = static_cast<int>(std::max<int64_t>(1, std::min<int64_t>(std::min(dev.sm_count, kPlanSMs) / row_tiles, nchunks)));
  int c = 1;
  while (c * 2 <= std::min(ks, maxc)) c *= 2;
  ks = c;
  CUtensorMap mx, ma;
  if (!make_tensor_map_2d(&mx, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, x, K, M, 2, kChunk, kRows, CU_TENSOR_MAP_SWIZZLE_128B) ||
      !make_tensor_map_2d(&ma, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, A, K, r, 2, kChunk, r, CU_TENSOR_MAP_SWIZZLE_128B))
    return NVFP4RL_ERR_CUDA;
  DownParams p{};
  p.M = M;
  p.K = K;
  p.r = r;
  p.nchunks = nchunks;
  p.chunks_per_cta = (nchunks + ks - 1) / ks;
  p.U = U;
  p.ls = scale;
  p.amax = amax;
  p.status = dev.status;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(ks), static_cast<unsigned>(row_tiles), 1);
  cfg.blockDim = dim3(kThreadsDown, 1, 1);
  cfg.dynamicSmemBytes = down_smem_bytes(r);
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = ks;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;  // overlaps the previous kernel's tail
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  if (cudaLaunchKernelEx(&cfg, lora_down_tc_kernel, mx, ma, p) != cudaSuccess) return NVFP4RL_ERR_CUDA;
  return launch_status();
}

nvfp4rl_status launch_lora_scale(uint16_t* U, int64_t M, int r, const LoraDownScale& scale, const DeviceInfo& dev,
                                 cudaStream_t st) {
  const int64_t n8 = M * r / 8;
  if (n8 == 0) return NVFP4RL_OK;
  const int grid = static_cast<int>(std::min<int64_t>((n8 + 255) / 256, static_cast<int64_t>(dev.sm_count) * 4));
  lora_scale_kernel<<<grid, 256, 0, st>>>(U, scale.lo, n8, scale);
  return launch_status();
}

}  // namespace nvfp4rl
