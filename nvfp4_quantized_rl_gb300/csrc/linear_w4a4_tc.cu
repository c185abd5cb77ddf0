// W4A4 NVFP4 LoRA linear on tcgen05 block-scaled FP4 MMA (kind::mxf4nvf4), sm_103a.
//
// TRACE summary, sections "論文が取り組む課題" and "実験結果と性能": the rollout runs with
// FP4 weights and FP4 activations. The activations are quantized on the fly with the
// NVFP4 recipe (one per-tensor g_x, 16-element E4M3 block scales); the tensor cores then
// take both operands as packed E2M1 with their block scales, and the epilogue applies
// g_x * g_w and adds the LoRA branch s (x A^T) B^T computed from the bf16 activations
// (QeRL explainer, section "NVFP4量子化とLoRA"). Grouped mode runs one weight matrix per
// MoE expert over that expert's contiguous block of routed rows. U = bf16(x A^T) comes from the
// cluster LoRA-down kernel that the W4A16 path uses (linear_tc.cu), launched before this one.
//
// Two persistent kernels (one CTA per SM, 256-K stages): w4a4_wide_kernel (tiles of 128 activation
// rows x 256 weight rows; LoRA rank up to 64, i.e. every shape of the workloads) and w4a4_tc_kernel
// (128 x 128 tiles, any rank up to 128), described here; the wide kernel is described at its
// definition. The MMAs of a stage take ~0.13 us while one trip through a shared-memory ring (TMA,
// scale factors to TMEM, MMA issue, MMA completion back to the producer) takes well over
// 1 us, so the operand codes have a deep ring of their own and the small scale tiles a
// separate one that runs ahead:
//   warps 0, 11 code producers (TMA): per stage the activation (warp 0) and the weight (warp 11)
//               code tile, 128 x 128 bytes each with 128-byte swizzle, into the code ring; warp 0
//               also loads the LoRA tiles. One issuing thread completes only about three
//               copies per microsecond (wait, expect_tx, copy), so each stream has its own.
//   warp 1      allocates TMEM; one thread issues four tcgen05.mma
//               kind::mxf4nvf4.block_scale.scale_vec::4X (K = 64 each) per stage; at the end of
//               a tile the LoRA up-projection (U tile x B_lora tile^T, kind::f16) goes to a
//               separate accumulator.
//   warps 2-5   epilogue: TMEM -> registers, Y = g_x g_w D + s D_lora, bf16 stores; the
//               accumulator is double buffered so it overlaps the next tile's main loop.
//   warps 6-9, 13-16  scale factors (two groups, alternate stages): each warp writes the
//               stage's scale bytes of both operands into
//               its own TMEM lane quarter with tcgen05.st (lane i, column 4t + w holds the four
//               bytes of row 32w + i for K step t: the four lane quarters hold the same copy),
//               into one of four TMEM slots that the MMAs release. This keeps the scale traffic
//               off the tensor pipe, where a shared-memory -> TMEM copy per K step and operand
//               would cost about as much as the MMAs.
//   warps 10,12 scale producers (TMA): the activation (warp 10) and weight (warp 12) 128 x 16-byte
//               scale tiles per stage into the scale ring, which the scale warps release once the
//               scales are in TMEM.

#include <cuda.h>
#include <cudaTypedefs.h>

#include <algorithm>

#include "common.cuh"
#include "sm100.cuh"

namespace nvfp4rl {
namespace {

using namespace sm100;

constexpr int kTile = 128;
constexpr int kKStage = 256;
constexpr int kCodeBytes = kTile * kKStage / 2;   // 16 KB per operand
constexpr int kSfBytes = kTile * kKStage / 16;    // 2 KB per operand
constexpr int kCodeStageBytes = 2 * kCodeBytes;  // code ring stage: activation + weight codes
constexpr int kSfStageBytes = 2 * kSfBytes;      // scale ring stage: activation + weight scales
constexpr int kSfRing = 4;                       // scale ring stages
constexpr int kSfSlots = 4;                      // TMEM scale-factor slots (32 columns each)
constexpr int kMaxCodeStages = 6;
constexpr int kDoneRing = 8;                     // "stage's MMAs done" barriers, > kMaxCodeStages, kSfSlots
constexpr int kThreads = 544;
constexpr int kFirstSfWarp = 6;        // scale warps 6-9 take the even stages, 13-16 the odd ones
constexpr int kSecondSfWarp = 13;
constexpr int kSfProducerWarp = 10;   // activation scales; weight scales: warp 12
constexpr int kWCodeWarp = 11;
constexpr uint32_t kD0 = 0, kD1 = 128, kDL = 256, kSF = 384;  // TMEM columns

struct W4a4Params {
  int64_t M, N, K;
  int tiles_n;
  int tiles_m;             // dense row tiles
  int total_tiles;         // dense: tiles_m * tiles_n; grouped: read from tile_start[groups] * tiles_n
  int r, lora_box_bytes;
  float s;
  const float* g_x;
  const float* w_g;        // [groups]
  const int32_t* offsets;  // grouped row offsets or null
  const int32_t* tile_start;
  int groups;
  uint16_t* y;
  uint32_t* status;
  int stages;
};

__device__ __forceinline__ int find_group(const int32_t* starts, int groups, int64_t v) {
  int lo = 0, hi = groups - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (starts[mid] <= v) lo = mid;
    else hi = mid - 1;
  }
  return lo;
}

struct TileInfo {
  int e;          // expert (0 when dense)
  int64_t m0;     // first activation row
  int64_t m_end;  // one past the last row this tile may write
  int n0;         // first weight row within the expert
};

// Dense tiles are visited in groups of kGroupRows row tiles; within a group consecutive tiles step
// through the row tiles first. A wave of CTAs then covers a block of a few weight tiles times those
// row tiles, whose operands stay in L2 while the wave runs (visiting all weight tiles of one row tile
// first would stream the whole weight matrix through L2 once per wave). Grouped (MoE) tiles keep the
// row-major order: their row tiles belong to different experts.
constexpr int kGroupRows = 32;

__device__ __forceinline__ void tile_coords(const W4a4Params& p, int t, int& tm, int& tn) {
  if (p.offsets) {
    tm = t / p.tiles_n;
    tn = t % p.tiles_n;
  } else {
    const int per_group = kGroupRows * p.tiles_n;
    const int first = (t / per_group) * kGroupRows, rem = t % per_group;
    const int rows = min(kGroupRows, p.tiles_m - first);
    tm = first + rem % rows;
    tn = rem / rows;
  }
}

__device__ __forceinline__ TileInfo tile_info(const W4a4Params& p, int t) {
  TileInfo ti;
  int tm, tn;
  tile_coords(p, t, tm, tn);
  ti.n0 = tn * kTile;
  if (p.offsets) {
    ti.e = find_group(p.tile_start, p.groups, tm);
    ti.m0 = p.offsets[ti.e] + static_cast<int64_t>(tm - p.tile_start[ti.e]) * kTile;
    ti.m_end = p.offsets[ti.e + 1];
  } else {
    ti.e = 0;
    ti.m0 = static_cast<int64_t>(tm) * kTile;
    ti.m_end = p.M;
  }
  return ti;
}

// Tile t of a kernel whose tiles cover `tile_n` weight rows (tiles_n tiles per row tile).
__device__ __forceinline__ TileInfo tile_info_n(const W4a4Params& p, int t, int tile_n) {
  TileInfo ti = tile_info(p, t);
  ti.n0 = ti.n0 / kTile * tile_n;
  return ti;
}

__device__ __forceinline__ int total_tiles(const W4a4Params& p) {
  return p.offsets ? p.tile_start[p.groups] * p.tiles_n : p.total_tiles;
}

__device__ __forceinline__ uint32_t lora_swizzle(int box_bytes) {
  return box_bytes == 128 ? 2u : box_bytes == 64 ? 4u : 6u;
}

// Four block-scaled MMAs over one 256-K stage from one instruction sequence: K step t reads the
// operand tiles 32 bytes further along the swizzled rows (descriptor start address + 2) and
// scale-factor columns 4t further on.
__device__ __forceinline__ void mma_stage_nvf4(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                               uint32_t sfa_tmem, uint32_t sfb_tmem, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p, t;\n\t.reg .b64 a1, b1;\n\t.reg .b32 s1, s2;\n\t"
      "setp.ne.b32 p, %6, 0;\n\tsetp.eq.u32 t, 0, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::mxf4nvf4.block_scale.scale_vec::4X [%0], %1, %2, %3, [%4], [%5], p;\n\t"
      "add.u64 a1, %1, 2;\n\tadd.u64 b1, %2, 2;\n\tadd.u32 s1, %4, 4;\n\tadd.u32 s2, %5, 4;\n\t"
      "tcgen05.mma.cta_group::1.kind::mxf4nvf4.block_scale.scale_vec::4X [%0], a1, b1, %3, [s1], [s2], t;\n\t"
      "add.u64 a1, %1, 4;\n\tadd.u64 b1, %2, 4;\n\tadd.u32 s1, %4, 8;\n\tadd.u32 s2, %5, 8;\n\t"
      "tcgen05.mma.cta_group::1.kind::mxf4nvf4.block_scale.scale_vec::4X [%0], a1, b1, %3, [s1], [s2], t;\n\t"
      "add.u64 a1, %1, 6;\n\tadd.u64 b1, %2, 6;\n\tadd.u32 s1, %4, 12;\n\tadd.u32 s2, %5, 12;\n\t"
      "tcgen05.mma.cta_group::1.kind::mxf4nvf4.block_scale.scale_vec::4X [%0], a1, b1, %3, [s1], [s2], t;\n\t}" ::"r"(
          d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(sfa_tmem), "r"(sfb_tmem), "r"(accumulate)
      : "memory");
}

__global__ void __launch_bounds__(kThreads, 1)
    w4a4_tc_kernel(const __grid_constant__ CUtensorMap map_xc, const __grid_constant__ CUtensorMap map_xs,
                   const __grid_constant__ CUtensorMap map_wc, const __grid_constant__ CUtensorMap map_ws,
                   const __grid_constant__ CUtensorMap map_u, const __grid_constant__ CUtensorMap map_bl,
                   const W4a4Params p) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int S = p.stages;                           // code ring stages
  uint8_t* sfring = smem + S * kCodeStageBytes;     // kSfRing x kSfStageBytes
  uint8_t* lora_u = sfring + kSfRing * kSfStageBytes;  // 128 x 2r
  const int lbytes = p.r ? kTile * 2 * p.r : 0;
  uint8_t* lora_b = lora_u + lbytes;                // 128 x 2r
  // mdone[i % kDoneRing]: one tcgen05.commit per stage i. The code producer waits for stage
  // i - S before refilling its code slot, the scale warps for stage i - kSfSlots before
  // rewriting its TMEM scale slot. Neither can fall kDoneRing stages behind the MMAs (those
  // stages would need operands that the waiter has not provided yet), so the parity of the
  // phase a waiter looks for is never ambiguous.
  uint64_t* cfull = reinterpret_cast<uint64_t*>(lora_b + lbytes);
  uint64_t* mdone = cfull + kMaxCodeStages;         // [kDoneRing]
  uint64_t* ffull = mdone + kDoneRing;              // scale tiles landed
  uint64_t* fempty = ffull + kSfRing;               // scale tiles read by the 4 scale warps
  uint64_t* sfready = fempty + kSfRing;             // TMEM scale slot written by the 4 scale warps
  uint64_t* dfull = sfready + kSfSlots;             // [2]
  uint64_t* dempty = dfull + 2;                     // [2]
  uint64_t* lfull = dempty + 2;                     // LoRA operands landed
  uint64_t* lempty = lfull + 1;                     // LoRA operand smem + D_lora free
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(lempty + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int ksteps = static_cast<int>(p.K / kKStage);
  const int ntiles = total_tiles(p);

  if (threadIdx.x == 0) {
    for (int i = 0; i < S; ++i) mbar_init(smem_addr(&cfull[i]), 2);  // activation + weight producer
    for (int i = 0; i < kDoneRing; ++i) mbar_init(smem_addr(&mdone[i]), 1);
    for (int i = 0; i < kSfRing; ++i) {
      mbar_init(smem_addr(&ffull[i]), 2);
      mbar_init(smem_addr(&fempty[i]), 4);
    }
    for (int i = 0; i < kSfSlots; ++i) mbar_init(smem_addr(&sfready[i]), 4);
    for (int i = 0; i < 2; ++i) {
      mbar_init(smem_addr(&dfull[i]), 1);
      mbar_init(smem_addr(&dempty[i]), 4);
    }
    mbar_init(smem_addr(lfull), 1);
    mbar_init(smem_addr(lempty), 4);
    fence_barrier_init();
  }
  if (warp == 1) tmem_alloc(smem_addr(tmem_slot), 512);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  bool ok = true;

  if (warp == 0 || warp == kWCodeWarp) {
    // ---------------------------------------------------------------- code producers
    if (lane == 0) {
      const bool wside = warp == kWCodeWarp;
      const CUtensorMap* map = wside ? &map_wc : &map_xc;
      prefetch_tensormap(map);
      int c = 0, li = 0, issued = 0, lora_issued = 0;
      for (int t = blockIdx.x; t < ntiles && ok; t += gridDim.x, ++li) {
        const TileInfo ti = tile_info(p, t);
        const int wrow = ti.e * static_cast<int>(p.N) + ti.n0;
        for (int k = 0; k < ksteps; ++k) {
          const int prev = issued - S;  // the stage that last used code slot c
          if (prev >= 0 && !mbar_wait(smem_addr(&mdone[prev % kDoneRing]), (prev / kDoneRing) & 1, p.status,
                                      kStatusTimeoutProducer)) {
            ok = false;
            break;
          }
          const uint32_t bar = smem_addr(&cfull[c]);
          mbar_arrive_expect_tx(bar, kCodeBytes);
          tma_load_2d(smem_addr(smem + c * kCodeStageBytes + (wside ? kCodeBytes : 0)), map, k * (kKStage / 2),
                      wside ? wrow : static_cast<int32_t>(ti.m0), bar);
          ++issued;
          if (++c == S) c = 0;
        }
        if (ok && p.r && !wside) {
          // LoRA operands of this tile (U rows m0.., B_lora rows n0..), needed after its main loop,
          // once the epilogue of the previous tile has read the LoRA accumulator
          if (!mbar_wait(smem_addr(lempty), (li & 1) ^ 1, p.status, kStatusTimeoutProducer)) {
            ok = false;
            break;
          }
          const uint32_t bar = smem_addr(lfull);
          mbar_arrive_expect_tx(bar, 2 * lbytes);
          const int nbox = 2 * p.r / p.lora_box_bytes, box_el = p.lora_box_bytes / 2;
          for (int b = 0; b < nbox; ++b) {
            tma_load_2d(smem_addr(lora_u + b * kTile * p.lora_box_bytes), &map_u, b * box_el,
                        static_cast<int32_t>(ti.m0), bar);
            tma_load_2d(smem_addr(lora_b + b * kTile * p.lora_box_bytes), &map_bl, b * box_el, ti.n0, bar);
          }
          lora_issued = li + 1;
        }
      }
      // do not exit with copies in flight: wait for the last S stages to land
      for (int j = max(0, issued - S); j < issued; ++j)
        mbar_wait(smem_addr(&cfull[j % S]), (j / S) & 1, p.status, kStatusTimeoutDrain);
      if (lora_issued) mbar_wait(smem_addr(lfull), (lora_issued - 1) & 1, p.status, kStatusTimeoutDrain);
    }
  } else if (warp == kSfProducerWarp || warp == kSfProducerWarp + 2) {
    // ---------------------------------------------------------------- scale producers
    if (lane == 0) {
      const bool wside = warp != kSfProducerWarp;
      const CUtensorMap* map = wside ? &map_ws : &map_xs;
      prefetch_tensormap(map);
      int f = 0, issued = 0;
      uint32_t ph = 0;
      for (int t = blockIdx.x; t < ntiles && ok; t += gridDim.x) {
        const TileInfo ti = tile_info(p, t);
        const int wrow = ti.e * static_cast<int>(p.N) + ti.n0;
        for (int k = 0; k < ksteps; ++k) {
          if (!mbar_wait(smem_addr(&fempty[f]), ph ^ 1u, p.status, kStatusTimeoutProducer)) {
            ok = false;
            break;
          }
          const uint32_t bar = smem_addr(&ffull[f]);
          mbar_arrive_expect_tx(bar, kSfBytes);
          tma_load_2d(smem_addr(sfring + f * kSfStageBytes + (wside ? kSfBytes : 0)), map, k * (kKStage / 16),
                      wside ? wrow : static_cast<int32_t>(ti.m0), bar);
          ++issued;
          if (++f == kSfRing) {
            f = 0;
            ph ^= 1u;
          }
        }
      }
      for (int j = max(0, issued - kSfRing); j < issued; ++j)
        mbar_wait(smem_addr(&ffull[j % kSfRing]), (j / kSfRing) & 1, p.status, kStatusTimeoutDrain);
    }
  } else if (warp == 1) {
    // ---------------------------------------------------------------- MMA issuer (one thread)
    if (lane == 0) {
      const uint32_t idesc = idesc_nvf4_f32(kTile, kTile);
      const uint32_t idesc_l = idesc_bf16_f32(kTile, kTile);
      // code stage 0's operand descriptors; stage c adds c * kCodeStageBytes to the start address field
      const uint64_t xdesc0 = smem_desc(smem_addr(smem), 16, 1024, 2);
      const uint64_t wdesc0 = smem_desc(smem_addr(smem + kCodeBytes), 16, 1024, 2);
      int c = 0, j = 0, li = 0, it = 0;
      uint32_t jph = 0;
      for (int t = blockIdx.x; t < ntiles && ok; t += gridDim.x, ++li) {
        const int buf = li & 1;
        const uint32_t dcol = buf ? kD1 : kD0;
        if (!mbar_wait(smem_addr(&dempty[buf]), ((li >> 1) & 1) ^ 1, p.status, kStatusTimeoutMma)) {
          ok = false;
          break;
        }
        tc_fence_after();
        for (int k = 0; k < ksteps; ++k) {
          // scale slot j written (tcgen05.st + fence by the scale warps), which the scale warps
          // signal only after they have seen code stage c land: one wait per stage here
          if (!mbar_wait(smem_addr(&sfready[j]), jph, p.status, kStatusTimeoutMma)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t sfcol = kSF + j * 32;
          const uint64_t soff = static_cast<uint64_t>(c * (kCodeStageBytes >> 4));
          mma_stage_nvf4(tmem + dcol, xdesc0 + soff, wdesc0 + soff, idesc, tmem + sfcol, tmem + sfcol + 16,
                         k ? 1u : 0u);
          mma_commit(smem_addr(&mdone[it % kDoneRing]));
          ++it;
          if (++c == S) c = 0;
          if (++j == kSfSlots) {
            j = 0;
            jph ^= 1u;
          }
        }
        if (!ok) break;
        if (p.r) {
          if (!mbar_wait(smem_addr(lfull), li & 1, p.status, kStatusTimeoutMma)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t sw = lora_swizzle(p.lora_box_bytes), sbo = 8 * p.lora_box_bytes;
          const uint32_t ua = smem_addr(lora_u), ba = smem_addr(lora_b);
          for (int kk = 0; kk < p.r / 16; ++kk) {
            const int off = kk * 32, box = off / p.lora_box_bytes, in = off % p.lora_box_bytes;
            mma_f16_ss(tmem + kDL, smem_desc(ua + box * kTile * p.lora_box_bytes + in, 16, sbo, sw),
                       smem_desc(ba + box * kTile * p.lora_box_bytes + in, 16, sbo, sw), idesc_l, kk ? 1u : 0u);
          }
        }
        mma_commit(smem_addr(&dfull[buf]));
      }
    }
    __syncwarp();
  } else if ((warp >= kFirstSfWarp && warp < kFirstSfWarp + 4) || (warp >= kSecondSfWarp && warp < kSecondSfWarp + 4)) {
    // ---------------------------------------------------------------- scale factors -> TMEM
    // Scale tile in shared memory: [128 rows][16 bytes], word t = the four block scales of K
    // step t. Lane i gathers rows i, 32 + i, 64 + i, 96 + i and writes, per operand, 16 columns:
    // column 4t + w = row 32w + i, K step t (the layout the MMA reads for M = 128). Two groups of
    // four warps (one per lane quarter) take alternate stages; ring slots and TMEM slots are
    // stage mod 4, so each group keeps its own slots.
    const uint32_t lane_base = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const int grp = warp >= kSecondSfWarp ? 1 : 0;
    const int my_tiles = blockIdx.x < ntiles ? (ntiles - 1 - static_cast<int>(blockIdx.x)) / gridDim.x + 1 : 0;
    const int total = my_tiles * ksteps;
    for (int it = grp; it < total && ok; it += 2) {
      const int f = it % kSfRing, j = it % kSfSlots;
      const uint32_t fph = static_cast<uint32_t>((it / kSfRing) & 1);
      {
        ok = __all_sync(0xFFFFFFFFu, mbar_wait(smem_addr(&ffull[f]), fph, p.status, kStatusTimeoutMma));
        if (!ok) break;
        const uint8_t* st = sfring + f * kSfStageBytes;
        uint32_t v[2][16];
#pragma unroll
        for (int op = 0; op < 2; ++op) {
          const uint4* sf = reinterpret_cast<const uint4*>(st + op * kSfBytes);
          const uint4 r0 = sf[lane], r1 = sf[32 + lane], r2 = sf[64 + lane], r3 = sf[96 + lane];
          const uint32_t w[16] = {r0.x, r1.x, r2.x, r3.x, r0.y, r1.y, r2.y, r3.y,
                                  r0.z, r1.z, r2.z, r3.z, r0.w, r1.w, r2.w, r3.w};
#pragma unroll
          for (int q = 0; q < 16; ++q) v[op][q] = w[q];
        }
        // TMEM slot j is free once the MMAs of the stage that last used it have completed
        const int prev = it - kSfSlots;
        if (prev >= 0) {
          ok = __all_sync(0xFFFFFFFFu, mbar_wait(smem_addr(&mdone[prev % kDoneRing]), (prev / kDoneRing) & 1,
                                                 p.status, kStatusTimeoutMma));
          if (!ok) break;
        }
        tc_fence_after();
        const uint32_t sfcol = kSF + j * 32;
        tmem_st16(tmem + lane_base + sfcol, v[0]);
        tmem_st16(tmem + lane_base + sfcol + 16, v[1]);
        tmem_st_wait();
        tc_fence_before();
        // the stage's code tiles have landed too (the MMA issuer then waits on sfready alone)
        ok = __all_sync(0xFFFFFFFFu, mbar_wait(smem_addr(&cfull[it % S]), static_cast<uint32_t>((it / S) & 1),
                                               p.status, kStatusTimeoutMma));
        if (!ok) break;
        __syncwarp();
        if (lane == 0) {
          mbar_arrive(smem_addr(&sfready[j]));
          mbar_arrive(smem_addr(&fempty[f]));  // the shared-memory scale tiles may be refilled
        }
      }
    }
  } else if (warp >= 2 && warp < 6) {
    // ---------------------------------------------------------------- epilogue (warps 2..5)
    const int quarter = warp & 3;
    const uint32_t lane_base = static_cast<uint32_t>(quarter * 32) << 16;
    const float gx = *p.g_x;
    int li = 0;
    for (int t = blockIdx.x; t < ntiles && ok; t += gridDim.x, ++li) {
      const int buf = li & 1;
      const uint32_t dcol = buf ? kD1 : kD0;
      ok = __all_sync(0xFFFFFFFFu, mbar_wait(smem_addr(&dfull[buf]), (li >> 1) & 1, p.status, kStatusTimeoutEpilogue));
      if (!ok) break;
      tc_fence_after();
      const TileInfo ti = tile_info(p, t);
      const float alpha = gx * p.w_g[ti.e];
      const int64_t m = ti.m0 + quarter * 32 + lane;
      const bool live = m < ti.m_end;
      uint16_t* yrow = p.y + m * p.N + ti.n0;
#pragma unroll 1
      for (int c = 0; c < kTile; c += 16) {
        uint32_t d[16], l[16];
        tmem_ld16(tmem + lane_base + dcol + c, d);
        if (p.r) tmem_ld16(tmem + lane_base + kDL + c, l);
        tmem_ld_wait();
        uint32_t o[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          float a = __uint_as_float(d[2 * i]) * alpha, b = __uint_as_float(d[2 * i + 1]) * alpha;
          if (p.r) {
            a = fmaf(p.s, __uint_as_float(l[2 * i]), a);
            b = fmaf(p.s, __uint_as_float(l[2 * i + 1]), b);
          }
          o[i] = f32_to_bf16_bits(a) | (f32_to_bf16_bits(b) << 16);
        }
        if (live) {
          uint4* dst = reinterpret_cast<uint4*>(yrow + c);
          dst[0] = make_uint4(o[0], o[1], o[2], o[3]);
          dst[1] = make_uint4(o[4], o[5], o[6], o[7]);
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(smem_addr(&dempty[buf]));
        if (p.r) mbar_arrive(smem_addr(lempty));
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// ---------------------------------------------------------------------------------------------
// Wide tiles: 128 activation rows x 256 weight rows per tile, one MMA of N = 256 per K step.
//
// Every 256-K stage carries twice the work of a 128 x 128 stage for the same handoffs (one
// code-ring slot, one scale slot, one commit), and reads a quarter fewer operand bytes from L2 per
// flop. TMEM: the accumulator D (256 columns, single buffer), the LoRA accumulator DL (128
// columns, used twice per tile: first for weight rows 0..127 of the tile, then for 128..255), and
// two scale slots of 64 columns (activation scales: 4 columns per K step, of which the MMA reads
// column w in lane quarter w, so each quarter writes its own rows there; weight scales: 8 columns
// per K step, column w = rows 32w .. 32w + 31, the same in every lane quarter). The epilogue
// (16 warps, 64 columns each, one 32-byte store per 16 outputs of a row) releases D once it has
// read it all; the next tile's MMAs wait for that.
//   warp 0      activation code producer (TMA, 128 x 128 B per stage) and the LoRA tiles
//   warp 1      TMEM allocation; one thread issues the MMAs (4 per stage) and the LoRA MMAs
//   warp 2      weight code producer (TMA, 256 x 128 B per stage)
//   warps 3, 4  activation (128 x 16 B) and weight (256 x 16 B) scale producers
//   warps 5-12  scale warps, two groups of four (one per lane quarter), alternate stages, each
//               group owning one TMEM scale slot
//   warps 13-28 epilogue: quarter = warp % 4, columns 64 ((warp - 13) / 4) .. + 64
constexpr int kWN = 256;
constexpr int kWCode = kWN * kKStage / 2;             // 32 KB of weight codes per stage
constexpr int kWStage = kCodeBytes + kWCode;          // 48 KB code-ring stage
constexpr int kWSfA = kTile * kKStage / 16;           // 2 KB activation scales per stage
constexpr int kWSfB = kWN * kKStage / 16;             // 4 KB weight scales per stage
constexpr int kWSfStage = kWSfA + kWSfB;
constexpr int kWSfRing = 4;
constexpr int kWMaxStages = 4;
constexpr int kWDone = 16;                            // commit ring, > code stages and scale slots
constexpr int kWThreads = 29 * 32;
constexpr int kWFirstSf = 5, kWFirstEpi = 13;
constexpr uint32_t kWD = 0, kWDL = 256, kWSF = 384;   // TMEM columns; scale slot j at kWSF + 64 j

// Four block-scaled MMAs (M = 128, N = 256, K = 64 each) over one stage: K step t reads the code
// tiles 32 bytes further along the swizzled rows, activation scales at column 4t and weight scales
// at column 8t of the slot.
__device__ __forceinline__ void mma_stage_wide(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                               uint32_t sfa_tmem, uint32_t sfb_tmem, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p, t;\n\t.reg .b64 a1, b1;\n\t.reg .b32 s1, s2;\n\t"
      "setp.ne.b32 p, %6, 0;\n\tsetp.eq.u32 t, 0, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::mxf4nvf4.block_scale.scale_vec::4X [%0], %1, %2, %3, [%4], [%5], p;\n\t"
      "add.u64 a1, %1, 2;\n\tadd.u64 b1, %2, 2;\n\tadd.u32 s1, %4, 4;\n\tadd.u32 s2, %5, 8;\n\t"
      "tcgen05.mma.cta_group::1.kind::mxf4nvf4.block_scale.scale_vec::4X [%0], a1, b1, %3, [s1], [s2], t;\n\t"
      "add.u64 a1, %1, 4;\n\tadd.u64 b1, %2, 4;\n\tadd.u32 s1, %4, 8;\n\tadd.u32 s2, %5, 16;\n\t"
      "tcgen05.mma.cta_group::1.kind::mxf4nvf4.block_scale.scale_vec::4X [%0], a1, b1, %3, [s1], [s2], t;\n\t"
      "add.u64 a1, %1, 6;\n\tadd.u64 b1, %2, 6;\n\tadd.u32 s1, %4, 12;\n\tadd.u32 s2, %5, 24;\n\t"
      "tcgen05.mma.cta_group::1.kind::mxf4nvf4.block_scale.scale_vec::4X [%0], a1, b1, %3, [s1], [s2], t;\n\t}" ::"r"(
          d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(sfa_tmem), "r"(sfb_tmem), "r"(accumulate)
      : "memory");
}

// One 32-byte store (16 bf16 outputs of a row; the address is 32-byte aligned).
__device__ __forceinline__ void st_global_v8(void* p, const uint32_t (&o)[8]) {
  asm volatile("st.global.v8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"l"(p), "r"(o[0]), "r"(o[1]), "r"(o[2]),
               "r"(o[3]), "r"(o[4]), "r"(o[5]), "r"(o[6]), "r"(o[7])
               : "memory");
}

// 16 columns from four words: column 4t + w holds word t, for every w (the MMA reads only column
// 4t + quarter of this lane quarter).
__device__ __forceinline__ void tmem_st16_rep4(uint32_t taddr, uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%1,%1,%1,%2,%2,%2,%2,%3,%3,%3,%3,%4,%4,%4,%4};" ::"r"(taddr),
      "r"(a0), "r"(a1), "r"(a2), "r"(a3)
      : "memory");
}

__global__ void __launch_bounds__(kWThreads, 1)
    w4a4_wide_kernel(const __grid_constant__ CUtensorMap map_xc, const __grid_constant__ CUtensorMap map_xs,
                     const __grid_constant__ CUtensorMap map_wc, const __grid_constant__ CUtensorMap map_ws,
                     const __grid_constant__ CUtensorMap map_u, const __grid_constant__ CUtensorMap map_bl,
                     const W4a4Params p) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int S = p.stages;                                  // code ring stages
  uint8_t* sfring = smem + S * kWStage;                    // kWSfRing x kWSfStage
  uint8_t* lora_u = sfring + kWSfRing * kWSfStage;         // 128 rows x 2r bytes
  const int ubytes = p.r ? kTile * 2 * p.r : 0;
  uint8_t* lora_b = lora_u + ubytes;                       // 256 rows x 2r bytes
  const int bbytes = p.r ? kWN * 2 * p.r : 0;
  uint64_t* cfull = reinterpret_cast<uint64_t*>(lora_b + bbytes);  // [kWMaxStages] codes landed
  uint64_t* mdone = cfull + kWMaxStages;                  // [kWDone] one commit per stage
  uint64_t* ffull = mdone + kWDone;                       // [kWSfRing] scale tiles landed
  uint64_t* fempty = ffull + kWSfRing;                    // [kWSfRing] scale tiles read
  uint64_t* sfready = fempty + kWSfRing;                  // [2] TMEM scale slot written
  uint64_t* dfull = sfready + 2;                          // D complete (and DL = LoRA of rows 0..127)
  uint64_t* dlfree = dfull + 1;                           // DL read by the first-half epilogue warps
  uint64_t* dfull2 = dlfree + 1;                          // DL = LoRA of rows 128..255
  uint64_t* dfree = dfull2 + 1;                           // D (and DL) read by every epilogue warp
  uint64_t* lfull = dfree + 1;                            // LoRA tiles landed
  uint64_t* lempty = lfull + 1;                           // LoRA tiles read by the LoRA MMAs
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(lempty + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int ksteps = static_cast<int>(p.K / kKStage);
  const int ntiles = total_tiles(p);
  const bool lora = p.r > 0;

  if (threadIdx.x == 0) {
    for (int i = 0; i < S; ++i) mbar_init(smem_addr(&cfull[i]), 2);  // activation + weight producer
    for (int i = 0; i < kWDone; ++i) mbar_init(smem_addr(&mdone[i]), 1);
    for (int i = 0; i < kWSfRing; ++i) {
      mbar_init(smem_addr(&ffull[i]), 2);
      mbar_init(smem_addr(&fempty[i]), 4);
    }
    for (int i = 0; i < 2; ++i) mbar_init(smem_addr(&sfready[i]), 4);
    mbar_init(smem_addr(dfull), 1);
    mbar_init(smem_addr(dlfree), 8);
    mbar_init(smem_addr(dfull2), 1);
    mbar_init(smem_addr(dfree), 16);
    mbar_init(smem_addr(lfull), 1);
    mbar_init(smem_addr(lempty), 1);
    fence_barrier_init();
  }
  if (warp == 1) tmem_alloc(smem_addr(tmem_slot), 512);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  bool ok = true;

  if (warp == 0 || warp == 2) {
    // ---------------------------------------------------------------- code producers
    if (lane == 0) {
      const bool wside = warp == 2;
      const CUtensorMap* map = wside ? &map_wc : &map_xc;
      prefetch_tensormap(map);
      const uint32_t bytes = wside ? kWCode : kCodeBytes;
      int c = 0, li = 0, issued = 0, lora_issued = 0;
      for (int t = blockIdx.x; t < ntiles && ok; t += gridDim.x, ++li) {
        const TileInfo ti = tile_info_n(p, t, kWN);
        const int wrow = ti.e * static_cast<int>(p.N) + ti.n0;
        for (int k = 0; k < ksteps; ++k) {
          const int prev = issued - S;  // the stage that last used code slot c
          if (prev >= 0 && !mbar_wait(smem_addr(&mdone[prev % kWDone]), (prev / kWDone) & 1, p.status,
                                      kStatusTimeoutProducer)) {
            ok = false;
            break;
          }
          const uint32_t bar = smem_addr(&cfull[c]);
          mbar_arrive_expect_tx(bar, bytes);
          tma_load_2d(smem_addr(smem + c * kWStage + (wside ? kCodeBytes : 0)), map, k * (kKStage / 2),
                      wside ? wrow : static_cast<int32_t>(ti.m0), bar);
          ++issued;
          if (++c == S) c = 0;
        }
        if (ok && lora && !wside) {
          // LoRA operands of this tile (U rows m0.., B_lora rows n0.., both r wide), needed after its
          // main loop, once the LoRA MMAs of the previous tile have read the previous ones
          if (!mbar_wait(smem_addr(lempty), (li & 1) ^ 1, p.status, kStatusTimeoutProducer)) {
            ok = false;
            break;
          }
          const uint32_t bar = smem_addr(lfull);
          mbar_arrive_expect_tx(bar, ubytes + bbytes);
          const int nbox = 2 * p.r / p.lora_box_bytes, box_el = p.lora_box_bytes / 2;
          for (int b = 0; b < nbox; ++b) {
            tma_load_2d(smem_addr(lora_u + b * kTile * p.lora_box_bytes), &map_u, b * box_el,
                        static_cast<int32_t>(ti.m0), bar);
            tma_load_2d(smem_addr(lora_b + b * kWN * p.lora_box_bytes), &map_bl, b * box_el, ti.n0, bar);
          }
          lora_issued = li + 1;
        }
      }
      // do not exit with copies in flight: wait for the last S stages to land
      for (int j = max(0, issued - S); j < issued; ++j)
        mbar_wait(smem_addr(&cfull[j % S]), (j / S) & 1, p.status, kStatusTimeoutDrain);
      if (lora_issued) {
        mbar_wait(smem_addr(lfull), (lora_issued - 1) & 1, p.status, kStatusTimeoutDrain);
        // and the last LoRA MMAs' commit has landed before the CTA (and its barriers) go away
        mbar_wait(smem_addr(lempty), (lora_issued - 1) & 1, p.status, kStatusTimeoutDrain);
      }
    }
  } else if (warp == 3 || warp == 4) {
    // ---------------------------------------------------------------- scale producers
    if (lane == 0) {
      const bool wside = warp == 4;
      const CUtensorMap* map = wside ? &map_ws : &map_xs;
      prefetch_tensormap(map);
      int f = 0, issued = 0;
      uint32_t ph = 0;
      for (int t = blockIdx.x; t < ntiles && ok; t += gridDim.x) {
        const TileInfo ti = tile_info_n(p, t, kWN);
        const int wrow = ti.e * static_cast<int>(p.N) + ti.n0;
        for (int k = 0; k < ksteps; ++k) {
          if (!mbar_wait(smem_addr(&fempty[f]), ph ^ 1u, p.status, kStatusTimeoutProducer)) {
            ok = false;
            break;
          }
          const uint32_t bar = smem_addr(&ffull[f]);
          mbar_arrive_expect_tx(bar, wside ? kWSfB : kWSfA);
          tma_load_2d(smem_addr(sfring + f * kWSfStage + (wside ? kWSfA : 0)), map, k * (kKStage / 16),
                      wside ? wrow : static_cast<int32_t>(ti.m0), bar);
          ++issued;
          if (++f == kWSfRing) {
            f = 0;
            ph ^= 1u;
          }
        }
      }
      for (int j = max(0, issued - kWSfRing); j < issued; ++j)
        mbar_wait(smem_addr(&ffull[j % kWSfRing]), (j / kWSfRing) & 1, p.status, kStatusTimeoutDrain);
    }
  } else if (warp == 1) {
    // ---------------------------------------------------------------- MMA issuer (one thread)
    if (lane == 0) {
      const uint32_t idesc = idesc_nvf4_f32(kTile, kWN);
      const uint32_t idesc_l = idesc_bf16_f32(kTile, kTile);
      // stage c's operand descriptors add c * kWStage to the start address field
      const uint64_t xdesc0 = smem_desc(smem_addr(smem), 16, 1024, 2);
      const uint64_t wdesc0 = smem_desc(smem_addr(smem + kCodeBytes), 16, 1024, 2);
      const uint32_t sw = lora_swizzle(p.lora_box_bytes), sbo = 8 * p.lora_box_bytes;
      int c = 0, li = 0, it = 0;
      for (int t = blockIdx.x; t < ntiles && ok; t += gridDim.x, ++li) {
        // the previous tile's epilogue has read D and DL
        if (!mbar_wait(smem_addr(dfree), (li & 1) ^ 1, p.status, kStatusTimeoutMma)) {
          ok = false;
          break;
        }
        tc_fence_after();
        for (int k = 0; k < ksteps; ++k) {
          const int j = it & 1;  // TMEM scale slot (one per scale-warp group)
          if (!mbar_wait(smem_addr(&sfready[j]), (it >> 1) & 1, p.status, kStatusTimeoutMma)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t sf = tmem + kWSF + 64 * j;
          const uint64_t soff = static_cast<uint64_t>(c * (kWStage >> 4));
          mma_stage_wide(tmem + kWD, xdesc0 + soff, wdesc0 + soff, idesc, sf, sf + 16, k ? 1u : 0u);
          mma_commit(smem_addr(&mdone[it % kWDone]));
          ++it;
          if (++c == S) c = 0;
        }
        if (!ok) break;
        if (lora) {
          if (!mbar_wait(smem_addr(lfull), li & 1, p.status, kStatusTimeoutMma)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t ua = smem_addr(lora_u), ba = smem_addr(lora_b);
          for (int h = 0; h < 2; ++h) {
            if (h == 1) {
              // the first-half epilogue warps have read DL
              if (!mbar_wait(smem_addr(dlfree), li & 1, p.status, kStatusTimeoutMma)) {
                ok = false;
                break;
              }
              tc_fence_after();
            }
            for (int kk = 0; kk < p.r / 16; ++kk) {
              const int off = kk * 32, box = off / p.lora_box_bytes, in = off % p.lora_box_bytes;
              mma_f16_ss(tmem + kWDL, smem_desc(ua + box * kTile * p.lora_box_bytes + in, 16, sbo, sw),
                         smem_desc(ba + box * kWN * p.lora_box_bytes + h * kTile * p.lora_box_bytes + in, 16, sbo,
                                   sw),
                         idesc_l, kk ? 1u : 0u);
            }
            mma_commit(smem_addr(h ? dfull2 : dfull));
          }
          if (!ok) break;
          mma_commit(smem_addr(lempty));  // the LoRA tiles may be refilled
        } else {
          mma_commit(smem_addr(dfull));
        }
      }
    }
    __syncwarp();
  } else if (warp >= kWFirstSf && warp < kWFirstEpi) {
    // ---------------------------------------------------------------- scale factors -> TMEM
    // Group g (warps 5-8: g = 0, 9-12: g = 1) takes the stages it with it % 2 == g and owns TMEM scale
    // slot g. Activation scales: lane i of quarter q reads row 32q + i (its four K-step words) and
    // writes them to columns 4t + w (for every w; the MMA reads 4t + q). Weight scales: lane i reads
    // rows 32w + i, w = 0..7, and writes column 8t + w = row 32w + i, K step t.
    const int q = warp & 3;
    const uint32_t lane_base = static_cast<uint32_t>(q * 32) << 16;
    const int g = (warp - kWFirstSf) >> 2;
    const uint32_t slot = tmem + lane_base + kWSF + 64 * g;
    const int my_tiles = blockIdx.x < ntiles ? (ntiles - 1 - static_cast<int>(blockIdx.x)) / gridDim.x + 1 : 0;
    const int total = my_tiles * ksteps;
    for (int it = g; it < total && ok; it += 2) {
      const int f = it % kWSfRing;
      ok = __all_sync(0xFFFFFFFFu, mbar_wait(smem_addr(&ffull[f]), static_cast<uint32_t>((it / kWSfRing) & 1),
                                             p.status, kStatusTimeoutMma));
      if (!ok) break;
      // TMEM slot g is free once the MMAs of the stage that last used it (it - 2) have completed
      const int prev = it - 2;
      if (prev >= 0) {
        ok = __all_sync(0xFFFFFFFFu, mbar_wait(smem_addr(&mdone[prev % kWDone]), (prev / kWDone) & 1, p.status,
                                               kStatusTimeoutMma));
        if (!ok) break;
      }
      tc_fence_after();
      const uint8_t* st = sfring + f * kWSfStage;
      const uint4 a = reinterpret_cast<const uint4*>(st)[q * 32 + lane];
      tmem_st16_rep4(slot, a.x, a.y, a.z, a.w);
      // weight scales in two halves of 16 columns: K steps 0-1, then 2-3
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {
        uint32_t b[16];
#pragma unroll
        for (int w = 0; w < 8; ++w) {
          const uint2 r = reinterpret_cast<const uint2*>(st + kWSfA)[(w * 32 + lane) * 2 + hh];
          b[w] = r.x;
          b[8 + w] = r.y;
        }
        tmem_st16(slot + 16 + 16 * hh, b);
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_addr(&fempty[f]));  // the scale tiles have been read
      tmem_st_wait();
      tc_fence_before();
      // the stage's code tiles have landed too (the MMA issuer then waits on sfready alone)
      ok = __all_sync(0xFFFFFFFFu, mbar_wait(smem_addr(&cfull[it % S]), static_cast<uint32_t>((it / S) & 1),
                                             p.status, kStatusTimeoutMma));
      if (!ok) break;
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_addr(&sfready[g]));
    }
  } else if (warp >= kWFirstEpi) {
    // ---------------------------------------------------------------- epilogue (16 warps)
    const int q = warp & 3;
    const int part = (warp - kWFirstEpi) >> 2;  // columns 64 part .. 64 part + 63
    const int half = part >> 1;                 // LoRA half: weight rows 0..127 or 128..255 of the tile
    const uint32_t lane_base = static_cast<uint32_t>(q * 32) << 16;
    const float gx = *p.g_x;
    int li = 0;
    for (int t = blockIdx.x; t < ntiles && ok; t += gridDim.x, ++li) {
      const uint32_t ph = static_cast<uint32_t>(li & 1);
      ok = __all_sync(0xFFFFFFFFu, mbar_wait(smem_addr(lora && half ? dfull2 : dfull), ph, p.status,
                                             kStatusTimeoutEpilogue));
      if (!ok) break;
      tc_fence_after();
      const TileInfo ti = tile_info_n(p, t, kWN);
      const float alpha = gx * p.w_g[ti.e];
      const int64_t m = ti.m0 + q * 32 + lane;
      const bool live = m < ti.m_end;
      uint16_t* yrow = p.y + m * p.N + ti.n0;
#pragma unroll 1
      for (int c = part * 64; c < part * 64 + 64; c += 16) {
        uint32_t d[16], l[16];
        tmem_ld16(tmem + lane_base + kWD + c, d);
        if (lora) tmem_ld16(tmem + lane_base + kWDL + (c & 127), l);
        tmem_ld_wait();
        uint32_t o[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          float x0 = __uint_as_float(d[2 * i]) * alpha, x1 = __uint_as_float(d[2 * i + 1]) * alpha;
          if (lora) {
            x0 = fmaf(p.s, __uint_as_float(l[2 * i]), x0);
            x1 = fmaf(p.s, __uint_as_float(l[2 * i + 1]), x1);
          }
          o[i] = f32_to_bf16_bits(x0) | (f32_to_bf16_bits(x1) << 16);
        }
        if (live && ti.n0 + c < p.N) st_global_v8(yrow + c, o);
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        if (lora && half == 0) mbar_arrive(smem_addr(dlfree));
        mbar_arrive(smem_addr(dfree));
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// tile_start[e] = sum over e' < e of ceil(rows(e') / 128); tile_start[groups] = total row tiles.
__global__ void __launch_bounds__(1024) tile_map128_kernel(const int32_t* __restrict__ offsets, int groups,
                                                           int32_t* __restrict__ tile_start) {
  __shared__ int32_t s[1024];
  const int e = threadIdx.x;
  s[e] = e < groups ? (offsets[e + 1] - offsets[e] + kTile - 1) / kTile : 0;
  __syncthreads();
  for (int o = 1; o < 1024; o <<= 1) {
    const int32_t add = e >= o ? s[e - o] : 0;
    __syncthreads();
    s[e] += add;
    __syncthreads();
  }
  if (e < groups) tile_start[e + 1] = s[e];
  if (e == 0) tile_start[0] = 0;
}

struct W4a4Plan {
  bool wide;   // 128 x 256 tiles (w4a4_wide_kernel), else 128 x 128 (w4a4_tc_kernel)
  int stages;
  size_t smem, ws_codes, ws_scales, ws_amax, ws_gx, ws_u, ws_tiles, ws_total;
};

// Wide tiles when three 48 KB code stages still fit beside the LoRA tiles (r <= 64), otherwise
// 128 x 128 tiles.
W4a4Plan w4a4_plan(int64_t M, int64_t K, int r, int groups, bool prequantized = false) {
  W4a4Plan t{};
  const size_t wlora = r ? static_cast<size_t>(kTile + kWN) * 2 * r : 0;
  const size_t wfixed = 1024 + wlora + kWSfRing * kWSfStage + 512;
  const int wstages = static_cast<int>(std::min<size_t>(kWMaxStages, (227 * 1024 - wfixed) / kWStage));
  if (wstages >= 3) {
    t.wide = true;
    t.stages = wstages;
    t.smem = wfixed + wstages * kWStage;
  } else {
    const size_t lora = r ? 2 * static_cast<size_t>(kTile) * 2 * r : 0;
    const size_t fixed = 1024 + lora + kSfRing * kSfStageBytes + 512;
    t.stages = static_cast<int>(std::min<size_t>(kMaxCodeStages, (227 * 1024 - fixed) / kCodeStageBytes));
    t.smem = fixed + t.stages * kCodeStageBytes;
  }
  size_t o = 0;
  auto take = [&](size_t b) { size_t at = o; o = align_up(o + b, 256); return at; };
  // activation codes, scales, amax word and g_x, unless the caller passes them in NVFP4
  t.ws_codes = take(prequantized ? 0 : static_cast<size_t>(M) * K / 2);
  t.ws_scales = take(prequantized ? 0 : static_cast<size_t>(M) * K / 16);
  t.ws_amax = take(prequantized ? 0 : kQuantizeWorkspace);
  t.ws_gx = take(prequantized ? 0 : 16);
  t.ws_u = take(static_cast<size_t>(M) * std::max(r, 1) * 2);
  t.ws_tiles = take(static_cast<size_t>(groups + 2) * 4);
  t.ws_total = o;
  return t;
}

CUtensorMapSwizzle lora_map_swizzle(int box_bytes) {
  return box_bytes == 128 ? CU_TENSOR_MAP_SWIZZLE_128B
         : box_bytes == 64 ? CU_TENSOR_MAP_SWIZZLE_64B
                           : CU_TENSOR_MAP_SWIZZLE_32B;
}

}  // namespace

bool w4a4_tc_supported(int64_t M, int64_t N, int64_t K, int r) {
  return M > 0 && N % kTile == 0 && K % kKStage == 0 && (r == 0 || (r % 16 == 0 && r <= kMaxLoraRank)) &&
         w4a4_plan(M, K, r, 1).stages >= 2;
}

size_t w4a4_tc_workspace_bytes(int64_t M, int64_t N, int64_t K, int r, int groups, bool prequantized) {
  (void)N;
  return w4a4_plan(M, K, r, groups, prequantized).ws_total;
}

nvfp4rl_status launch_w4a4_tc(const LinearArgs& a, void* ws, size_t ws_bytes, const DeviceInfo& dev,
                              cudaStream_t st) {
  const int groups = a.offsets ? a.groups : 1;
  const bool pre = a.xq_codes != nullptr;
  const W4a4Plan t = w4a4_plan(a.M, a.K, a.r, groups, pre);
  if (ws_bytes < t.ws_total) return NVFP4RL_ERR_WORKSPACE;
  char* base = static_cast<char*>(ws);
  const uint8_t* xc = pre ? a.xq_codes : reinterpret_cast<uint8_t*>(base + t.ws_codes);
  const uint8_t* xs = pre ? a.xq_scales : reinterpret_cast<uint8_t*>(base + t.ws_scales);
  const float* gx = pre ? a.xq_g : reinterpret_cast<float*>(base + t.ws_gx);
  uint16_t* U = reinterpret_cast<uint16_t*>(base + t.ws_u);
  int32_t* tiles = reinterpret_cast<int32_t*>(base + t.ws_tiles);

  if (!pre) {
    nvfp4rl_status sq = launch_quantize(a.x, NVFP4RL_BF16, a.M, a.K, nullptr, reinterpret_cast<uint8_t*>(base + t.ws_codes),
                                        reinterpret_cast<uint8_t*>(base + t.ws_scales),
                                        reinterpret_cast<float*>(base + t.ws_gx), nullptr,
                                        reinterpret_cast<uint32_t*>(base + t.ws_amax), dev, st);
    if (sq != NVFP4RL_OK) return sq;
  }
  if (a.r) {
    const nvfp4rl_status sd = launch_lora_down(a.x, a.M, a.K, a.A, a.r, U, dev, st);
    if (sd != NVFP4RL_OK) return sd;
  }
  if (a.offsets) {
    tile_map128_kernel<<<1, 1024, 0, st>>>(a.offsets, groups, tiles);
    if (launch_status() != NVFP4RL_OK) return NVFP4RL_ERR_CUDA;
  }
  CUtensorMap mxc, mxs, mwc, mws, mu, mb;
  const int lbox = a.r ? std::min(2 * a.r, 128) : 128;
  const uint64_t wrows = static_cast<uint64_t>(groups) * a.N;
  const uint32_t wbox = t.wide ? kWN : kTile;  // weight rows per tile
  if (!make_tensor_map_2d(&mxc, CU_TENSOR_MAP_DATA_TYPE_UINT8, xc, a.K / 2, a.M, 1, 128, kTile, CU_TENSOR_MAP_SWIZZLE_128B) ||
      !make_tensor_map_2d(&mxs, CU_TENSOR_MAP_DATA_TYPE_UINT8, xs, a.K / 16, a.M, 1, 16, kTile, CU_TENSOR_MAP_SWIZZLE_NONE) ||
      !make_tensor_map_2d(&mwc, CU_TENSOR_MAP_DATA_TYPE_UINT8, a.w_codes, a.K / 2, wrows, 1, 128, wbox,
                          CU_TENSOR_MAP_SWIZZLE_128B) ||
      !make_tensor_map_2d(&mws, CU_TENSOR_MAP_DATA_TYPE_UINT8, a.w_scales, a.K / 16, wrows, 1, 16, wbox,
                          CU_TENSOR_MAP_SWIZZLE_NONE))
    return NVFP4RL_ERR_CUDA;
  if (a.r) {
    if (!make_tensor_map_2d(&mu, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, U, a.r, a.M, 2, lbox / 2, kTile,
                            lora_map_swizzle(lbox)) ||
        !make_tensor_map_2d(&mb, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, a.B, a.r, a.N, 2, lbox / 2, wbox,
                            lora_map_swizzle(lbox)))
      return NVFP4RL_ERR_CUDA;
  } else {
    mu = mxc;
    mb = mxc;
  }
  W4a4Params p{};
  p.M = a.M;
  p.N = a.N;
  p.K = a.K;
  p.tiles_n = static_cast<int>((a.N + wbox - 1) / wbox);
  const int64_t tiles_m_bound = a.offsets ? (a.M + kTile - 1) / kTile + groups : (a.M + kTile - 1) / kTile;
  p.tiles_m = static_cast<int>((a.M + kTile - 1) / kTile);
  p.total_tiles = p.tiles_m * p.tiles_n;
  p.r = a.r;
  p.lora_box_bytes = lbox;
  p.s = a.s;
  p.g_x = gx;
  p.w_g = a.w_g;
  p.offsets = a.offsets;
  p.tile_start = tiles;
  p.groups = groups;
  p.y = a.y;
  p.status = dev.status;
  p.stages = t.stages;
  const int64_t max_tiles = tiles_m_bound * p.tiles_n;
  const int grid = static_cast<int>(std::min<int64_t>(max_tiles, dev.sm_count));
  if (t.wide) {
    if (cudaFuncSetAttribute(w4a4_wide_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(t.smem)) != cudaSuccess)
      return NVFP4RL_ERR_CUDA;
    w4a4_wide_kernel<<<grid, kWThreads, t.smem, st>>>(mxc, mxs, mwc, mws, mu, mb, p);
  } else {
    if (cudaFuncSetAttribute(w4a4_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(t.smem)) != cudaSuccess)
      return NVFP4RL_ERR_CUDA;
    w4a4_tc_kernel<<<grid, kThreads, t.smem, st>>>(mxc, mxs, mwc, mws, mu, mb, p);
  }
  return launch_status();
}

}  // namespace nvfp4rl
