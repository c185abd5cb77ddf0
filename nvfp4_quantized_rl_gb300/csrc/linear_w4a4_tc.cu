// W4A4 NVFP4 LoRA linear on tcgen05 block-scaled FP4 MMA (kind::mxf4nvf4), sm_103a.
//
// TRACE summary, sections "論文が取り組む課題" and "実験結果と性能": the rollout runs with
// FP4 weights and FP4 activations. The activations are quantized on the fly with the
// NVFP4 recipe (one per-tensor g_x, 16-element E4M3 block scales); the tensor cores then
// take both operands as packed E2M1 with their block scales, the product is scaled by
// alpha = g_x g_w, and the LoRA branch s (x A^T) B^T computed from the bf16 activations is
// added (QeRL explainer, section "NVFP4量子化とLoRA"). Grouped mode runs one weight matrix per
// MoE expert over that expert's contiguous block of routed rows. U = bf16(x A^T) comes from the
// cluster LoRA-down kernel that the W4A16 path uses (linear_tc.cu), launched before this one.
//
// One persistent kernel, one CTA per SM, in two forms. Dense calls with more than 128 rows run on
// CTA pairs (a cluster of two, tcgen05 cta_group::2): a pair tile is 256 activation rows x 256
// weight rows; each CTA loads its own 128 activation rows and half of the weight rows (so a ring
// stage is 32 KB and six fit), keeps the scales of its rows and of all 256 weight rows in its own
// TMEM, and holds its 128 rows of the accumulator; the even CTA issues the MMAs, its commits
// arrive in both CTAs, and the odd CTA's scale and epilogue warps arrive on the even CTA's
// barriers. Grouped (MoE) calls, whose row tiles may belong to different experts, and calls of
// at most 128 rows run one CTA per tile of 128 x 256 (48 KB stages, four of them). A pair's
// tensor cores move the same FP4 work per SM as a lone CTA (measured: 65 ns per 128 x 256 x 64
// MMA either way, resident operands) but it reads two thirds of the operand bytes per flop from
// L2, which bounds the lone CTA's ring.
//
// The LoRA branch shares the FP4 product's fp32 accumulator. With c = s / alpha,
//   y = alpha * (x_q W_q^T + c U B^T),
// and c U is not a bf16 value, so the LoRA-down kernel writes it as two bf16 matrices, hi =
// bf16(c U) and lo = bf16(c U - hi), and each tile runs the up-projection (kind::f16 MMAs, hi
// slice x B_lora slice^T, then lo slice x B_lora slice^T) as the last stages of its K loop,
// through the same operand ring as the codes: 64 ranks of U (128 rows x 128 bytes) and of B_lora
// (256 rows x 128 bytes) fill a ring stage exactly as 256 K of activation and weight codes do. The
// accumulator receives c U B^T to ~2^-17 relative, as if U = bf16(x A^T) were scaled
// in fp32. There is then no second accumulator, no LoRA buffer of its own in shared memory, and no
// hand-over between the epilogue and a late LoRA MMA. When alpha = 0 (an all-zero weight or
// activation tensor) the FP4 MMAs are skipped and the tile computes s U B^T with an output scale
// of 1. c above 2^100 (s / alpha so large that c U or c U B^T could leave the fp32 range: the
// product of the two tensors' amax below about 1e-23 for s = 2) sets a range bit in the device
// status word.
//
// A stage's four FP4 MMAs take ~0.26 us, while a trip through the operand ring (MMA completion ->
// TMA refill of the slot -> data landed -> scales in TMEM -> MMA issue) takes over 1 us, so
// several stages are in flight. Roles (28 warps: the 72 registers a thread
// gets at that size hold every role without spilling; 29 warps would leave 64):
//   warp 0      activation code producer (TMA, 128 x 128 B per stage; a U slice on LoRA stages)
//   warp 1      TMEM allocation; one thread issues the MMAs
//   warp 2      weight code producer (TMA, 256 x 128 B per stage, 128 x 128 B in a pair; a B_lora
//               slice on LoRA stages)
//   warp 3      scale producers, FP4 stages only: lane 0 the activation (128 x 16 B), lane 1 the
//               weight (256 x 16 B) scale tiles
//   warps 4-11  two groups of four scale warps (one per TMEM lane quarter) taking alternate
//               stages: an FP4 stage's scale bytes go to one of four TMEM scale slots with
//               tcgen05.st; on a LoRA stage the group only passes the landed slices on
//   warps 12-27 epilogue (quarter = warp % 4, 64 columns each): TMEM -> registers, scaled by
//               alpha and packed to bf16 (cvt.rn.bf16x2); D is released to the next tile's MMAs
//               as soon as it has been read, then the rows are stored, 128-byte pieces at a time
//               after a shuffle transpose within groups of 8 lanes
// TMEM: the accumulator D in columns 0..255; five scale slots: slot j's activation scales in
// columns 256 + 16 j .. + 15 (4 per K step: the MMA reads column 4t + w in lane quarter w, so each
// quarter writes its own rows there), its weight scales in 352 + 32 j .. + 31 (8 per K step:
// column 8t + w holds rows 32w .. 32w + 31, the same in every lane quarter). A slot is rewritten
// only after the MMAs of the stage five earlier have completed, so four stages of MMAs stay
// queued while the scale warps refill it.

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

constexpr int kTile = 128;                        // activation rows per tile (MMA M)
constexpr int kWN = 256;                          // weight rows per tile (MMA N)
constexpr int kKStage = 256;                      // K per FP4 stage
constexpr int kLoraK = 64;                        // ranks per LoRA slice (128 bytes of bf16), two stages each
constexpr int kACode = kTile * kKStage / 2;       // 16 KB: activation codes or a U slice
constexpr int kSfA = kTile * kKStage / 16;        // 2 KB activation scales per stage
constexpr int kSfB = kWN * kKStage / 16;          // 4 KB weight scales per stage
constexpr int kSfStage = kSfA + kSfB;
constexpr int kSfRing = 4;                        // scale ring stages
constexpr int kSlots = 5;                         // TMEM scale slots
constexpr int kDone = 16;                         // commit ring, > operand stages and scale slots
constexpr int kThreads = 28 * 32;
constexpr int kFirstSf = 4, kFirstEpi = 12;
// TMEM columns of scale slot j: activation scales at kSfACol + 16 j (16 columns), weight scales at
// kSfBCol + 32 j (32 columns); five slots fill columns 256..511 with D in 0..255.
constexpr uint32_t kSfACol = 256, kSfBCol = 352;
static_assert(kSfACol + 16 * kSlots <= kSfBCol && kSfBCol + 32 * kSlots <= 512, "scale slots fit TMEM");

struct W4a4Params {
  int64_t M, N, K;
  int tiles_n;
  int tiles_m;             // dense row tiles
  int total_tiles;         // dense: tiles_m * tiles_n; grouped: read from tile_start[groups] * tiles_n
  int r;
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

__device__ __forceinline__ TileInfo tile_info(const W4a4Params& p, int t) {
  int tm, tn;
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
  TileInfo ti;
  ti.n0 = tn * kWN;
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

__device__ __forceinline__ int total_tiles(const W4a4Params& p) {
  return p.offsets ? p.tile_start[p.groups] * p.tiles_n : p.total_tiles;
}

// Four block-scaled MMAs (M = 128, N = 256, K = 64 each) over one stage: K step t reads the code
// tiles 32 bytes further along the swizzled rows, activation scales at column 4t and weight scales
// at column 8t of the slot.
__device__ __forceinline__ void mma_stage_nvf4(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
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

// 16 columns from four words: column 4t + w holds word t, for every w (the MMA reads only column
// 4t + quarter of this lane quarter).
__device__ __forceinline__ void tmem_st16_rep4(uint32_t taddr, uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%1,%1,%1,%2,%2,%2,%2,%3,%3,%3,%3,%4,%4,%4,%4};" ::"r"(taddr),
      "r"(a0), "r"(a1), "r"(a2), "r"(a3)
      : "memory");
}

// ---- CTA pairs (tcgen05 cta_group::2) --------------------------------------------------------

__device__ __forceinline__ void tmem_alloc_pair(uint32_t dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem), "r"(ncols)
               : "memory");
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc_pair(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
// Arrives once on `bar` in both CTAs of the pair when every tcgen05 operation this thread issued
// before has completed.
__device__ __forceinline__ void mma_commit_pair(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::"r"(
                   bar),
               "h"(static_cast<uint16_t>(3))
               : "memory");
}
// Arrival on a barrier of another CTA of the cluster (address from dsmem_map). Relaxed: what the
// arrival announces (TMEM stores waited for with tcgen05.wait::st, operand tiles whose TMA
// completion this thread observed) is complete before it, and a release at cluster scope measured
// ~1 us of extra latency per arrival on the critical path.
__device__ __forceinline__ void mbar_arrive_remote(uint32_t cluster_bar) {
  asm volatile("mbarrier.arrive.relaxed.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_bar) : "memory");
}
__device__ __forceinline__ void mma_f16_pair(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                             uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// mma_stage_nvf4 for a CTA pair: M = 256 (128 rows in each CTA's shared memory and TMEM), each
// CTA holding half of the 256 weight rows and the full weight scales.
__device__ __forceinline__ void mma_stage_nvf4_pair(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                                    uint32_t idesc, uint32_t sfa_tmem, uint32_t sfb_tmem,
                                                    uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p, t;\n\t.reg .b64 a1, b1;\n\t.reg .b32 s1, s2;\n\t"
      "setp.ne.b32 p, %6, 0;\n\tsetp.eq.u32 t, 0, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::mxf4nvf4.block_scale.scale_vec::4X [%0], %1, %2, %3, [%4], [%5], p;\n\t"
      "add.u64 a1, %1, 2;\n\tadd.u64 b1, %2, 2;\n\tadd.u32 s1, %4, 4;\n\tadd.u32 s2, %5, 8;\n\t"
      "tcgen05.mma.cta_group::2.kind::mxf4nvf4.block_scale.scale_vec::4X [%0], a1, b1, %3, [s1], [s2], t;\n\t"
      "add.u64 a1, %1, 4;\n\tadd.u64 b1, %2, 4;\n\tadd.u32 s1, %4, 8;\n\tadd.u32 s2, %5, 16;\n\t"
      "tcgen05.mma.cta_group::2.kind::mxf4nvf4.block_scale.scale_vec::4X [%0], a1, b1, %3, [s1], [s2], t;\n\t"
      "add.u64 a1, %1, 6;\n\tadd.u64 b1, %2, 6;\n\tadd.u32 s1, %4, 12;\n\tadd.u32 s2, %5, 24;\n\t"
      "tcgen05.mma.cta_group::2.kind::mxf4nvf4.block_scale.scale_vec::4X [%0], a1, b1, %3, [s1], [s2], t;\n\t}" ::"r"(
          d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(sfa_tmem), "r"(sfb_tmem), "r"(accumulate)
      : "memory");
}

// Operand ring geometry: a CTA of a pair holds half of the tile's 256 weight rows.
template <bool kPair>
struct Ring {
  static constexpr int kBRows = kPair ? kWN / 2 : kWN;     // weight rows in this CTA's shared memory
  static constexpr int kBBytes = kBRows * kKStage / 2;    // 16 or 32 KB per stage
  static constexpr int kStageBytes = kACode + kBBytes;    // 32 or 48 KB
  static constexpr int kMaxStages = kPair ? 6 : 4;
};
constexpr int kRingBarriers = 6;  // cfull barriers, >= either ring's stages

// The tile a CTA works on in round t of its persistent loop: a CTA alone takes tile t (128 x 256);
// a CTA pair takes pair tile t (256 x 256), rank r of the pair its row tile 2 pm + r.
template <bool kPair>
__device__ __forceinline__ TileInfo tile_of(const W4a4Params& p, int t, uint32_t rank) {
  if constexpr (!kPair) {
    return tile_info(p, t);
  } else {
    const int rows2 = (p.tiles_m + 1) >> 1;  // pair rows
    const int per_group = (kGroupRows / 2) * p.tiles_n;
    const int first = (t / per_group) * (kGroupRows / 2), rem = t % per_group;
    const int rows = min(kGroupRows / 2, rows2 - first);
    TileInfo ti;
    ti.e = 0;
    ti.m0 = static_cast<int64_t>(2 * (first + rem % rows) + static_cast<int>(rank)) * kTile;
    ti.m_end = p.M;
    ti.n0 = (rem / rows) * kWN;
    return ti;
  }
}

template <bool kPair>
__global__ void __launch_bounds__(kThreads, 1)
    w4a4_wide_kernel(const __grid_constant__ CUtensorMap map_xc, const __grid_constant__ CUtensorMap map_xs,
                     const __grid_constant__ CUtensorMap map_wc, const __grid_constant__ CUtensorMap map_ws,
                     const __grid_constant__ CUtensorMap map_uh, const __grid_constant__ CUtensorMap map_ul,
                     const __grid_constant__ CUtensorMap map_bl, const W4a4Params p) {
  using R = Ring<kPair>;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int S = p.stages;                                  // operand ring stages
  uint8_t* sfring = smem + S * R::kStageBytes;             // kSfRing x kSfStage
  // mdone[i % kDone]: one tcgen05.commit per stage i (of every tile, LoRA stages included). The
  // operand producers wait for stage i - S before refilling a ring slot, the scale warps for stage
  // i - kSlots before rewriting a TMEM scale slot. Neither can fall kDone stages behind the MMAs
  // (those would need operands the waiter has not provided yet), so the parity a waiter looks for
  // is never ambiguous. In a pair the leader's commits arrive in both CTAs.
  uint64_t* cfull = reinterpret_cast<uint64_t*>(sfring + kSfRing * kSfStage);  // operands landed
  uint64_t* mdone = cfull + kRingBarriers;                // [kDone]
  uint64_t* ffull = mdone + kDone;                        // [kSfRing] scale tiles landed
  uint64_t* fempty = ffull + kSfRing;                     // [kSfRing] scale tiles read
  uint64_t* sfready = fempty + kSfRing;                   // [kSlots] stage ready for its MMAs (leader's)
  uint64_t* dfull = sfready + kSlots;                     // the tile's accumulator is complete
  uint64_t* dfree = dfull + 1;                            // ... and has been read by every epilogue warp
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(dfree + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int ksteps = static_cast<int>(p.K / kKStage);     // FP4 stages per tile
  const int nl = 2 * ((p.r + kLoraK - 1) / kLoraK);        // LoRA stages per tile (hi, lo per slice), last
  const int ns = nl + ksteps;
  const int ntiles = total_tiles(p);
  const uint32_t rank = kPair ? cluster_ctarank() : 0u;
  const int unit = kPair ? static_cast<int>(blockIdx.x >> 1) : static_cast<int>(blockIdx.x);  // CTA or pair
  const int units = kPair ? static_cast<int>(gridDim.x >> 1) : static_cast<int>(gridDim.x);
  constexpr int kPeers = kPair ? 2 : 1;

  if (threadIdx.x == 0) {
    for (int i = 0; i < S; ++i) mbar_init(smem_addr(&cfull[i]), 2);  // activation + weight producer
    for (int i = 0; i < kDone; ++i) mbar_init(smem_addr(&mdone[i]), 1);
    for (int i = 0; i < kSfRing; ++i) {
      mbar_init(smem_addr(&ffull[i]), 2);
      mbar_init(smem_addr(&fempty[i]), 4);
    }
    for (int i = 0; i < kSlots; ++i) mbar_init(smem_addr(&sfready[i]), 4 * kPeers);
    mbar_init(smem_addr(dfull), 1);
    mbar_init(smem_addr(dfree), 16 * kPeers);
    fence_barrier_init();
  }
  if (warp == 1) {
    if constexpr (kPair) tmem_alloc_pair(smem_addr(tmem_slot), 512);
    else tmem_alloc(smem_addr(tmem_slot), 512);
  }
  tc_fence_before();
  __syncthreads();
  if constexpr (kPair) cluster_sync_all();  // the peer's barriers exist before anything signals them
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  bool ok = true;

  if (warp == 0 || warp == 2) {
    // ---------------------------------------------------------------- operand producers
    if (lane == 0) {
      const bool wside = warp == 2;
      const CUtensorMap* map = wside ? &map_wc : &map_xc;
      prefetch_tensormap(map);
      if (nl) {
        prefetch_tensormap(wside ? &map_bl : &map_uh);
        if (!wside) prefetch_tensormap(&map_ul);
      }
      const uint32_t off = wside ? kACode : 0;
      const uint32_t bytes = wside ? R::kBBytes : kACode;
      const int half = static_cast<int>(rank) * R::kBRows;  // this CTA's weight rows of the tile
      int c = 0, issued = 0;
      bool u_ready = wside;  // B_lora is an input of the call; U is the LoRA-down kernel's output
      for (int t = unit; t < ntiles && ok; t += units) {
        const TileInfo ti = tile_of<kPair>(p, t, rank);
        const int row = wside ? ti.e * static_cast<int>(p.N) + ti.n0 + half : static_cast<int>(ti.m0);
        const int lrow = wside ? ti.n0 + half : static_cast<int>(ti.m0);  // B_lora is shared by the experts
        for (int k = 0; k < ns; ++k) {
          const int prev = issued - S;  // the stage that last used ring slot c
          if (prev >= 0 && !mbar_wait(smem_addr(&mdone[prev % kDone]), (prev / kDone) & 1, p.status,
                                      kStatusTimeoutProducer)) {
            ok = false;
            break;
          }
          const uint32_t bar = smem_addr(&cfull[c]);
          const uint32_t dst = smem_addr(smem + c * R::kStageBytes + off);
          if (k >= ksteps && !u_ready) {
            griddep_wait();  // the LoRA-down kernel has completed and its hi and lo are visible
            u_ready = true;
          }
          mbar_arrive_expect_tx(bar, bytes);
          const int kl = k - ksteps;
          if (kl >= 0)  // slice kl / 2 of hi (kl even) or lo (kl odd), and of B_lora
            tma_load_2d(dst, wside ? &map_bl : (kl & 1) ? &map_ul : &map_uh, (kl >> 1) * kLoraK, lrow, bar);
          else tma_load_2d(dst, map, k * (kKStage / 2), row, bar);
          ++issued;
          if (++c == S) c = 0;
        }
      }
      // do not exit with copies in flight (the last S stages to land), nor before the last S
      // stages' commits have arrived here
      for (int j = max(0, issued - S); j < issued; ++j) {
        mbar_wait(smem_addr(&cfull[j % S]), (j / S) & 1, p.status, kStatusTimeoutDrain);
        if (wside) mbar_wait(smem_addr(&mdone[j % kDone]), (j / kDone) & 1, p.status, kStatusTimeoutDrain);
      }
    }
  } else if (warp == 3) {
    // ---------------------------------------------------------------- scale producers (FP4 stages)
    if (lane < 2) {
      const bool wside = lane == 1;
      const CUtensorMap* map = wside ? &map_ws : &map_xs;
      prefetch_tensormap(map);
      int f = 0, issued = 0;
      uint32_t ph = 0;
      for (int t = unit; t < ntiles && ok; t += units) {
        const TileInfo ti = tile_of<kPair>(p, t, rank);
        // the weight scales of all 256 rows of the tile, in both CTAs of a pair
        const int row = wside ? ti.e * static_cast<int>(p.N) + ti.n0 : static_cast<int>(ti.m0);
        for (int k = 0; k < ksteps; ++k) {
          if (!mbar_wait(smem_addr(&fempty[f]), ph ^ 1u, p.status, kStatusTimeoutProducer)) {
            ok = false;
            break;
          }
          const uint32_t bar = smem_addr(&ffull[f]);
          mbar_arrive_expect_tx(bar, wside ? kSfB : kSfA);
          tma_load_2d(smem_addr(sfring + f * kSfStage + (wside ? kSfA : 0)), map, k * (kKStage / 16), row, bar);
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
    // ---------------------------------------------------------------- MMA issuer (a pair's leader)
    // The whole warp walks the tiles and stages and waits; one elected lane issues the MMAs and
    // commits (the same lane every time).
    if (rank == 0) {
      const uint32_t idesc = idesc_nvf4_f32(kTile * kPeers, kWN);
      const uint32_t idesc_l = idesc_bf16_f32(kTile * kPeers, kWN);
      // ring slot c's operand descriptors add c * stage bytes to the start address field; a K step
      // (64 E2M1 codes or 16 bf16 values: 32 bytes of a swizzled row) adds 2
      const uint64_t adesc0 = smem_desc(smem_addr(smem), 16, 1024, 2);
      const uint64_t bdesc0 = smem_desc(smem_addr(smem + kACode), 16, 1024, 2);
      const float gx = *p.g_x;
      int c = 0, li = 0, it = 0;
      for (int t = unit; t < ntiles && ok; t += units, ++li) {
        // the previous tile's epilogue has read D (in both CTAs of a pair)
        ok = __all_sync(0xFFFFFFFFu, mbar_wait(smem_addr(dfree), (li & 1) ^ 1, p.status, kStatusTimeoutMma));
        if (!ok) break;
        tc_fence_after();
        const TileInfo ti = tile_of<kPair>(p, t, 0);
        // alpha = 0 with a LoRA branch: D = s U B^T alone (the FP4 product would be scaled by 0)
        const bool fp4 = !(nl && gx * p.w_g[ti.e] == 0.f);
        for (int k = 0; k < ns; ++k) {
          const int j = it % kSlots;
          ok = __all_sync(0xFFFFFFFFu, mbar_wait(smem_addr(&sfready[j]), (it / kSlots) & 1, p.status, kStatusTimeoutMma));
          if (!ok) break;
          tc_fence_after();
          const uint64_t soff = static_cast<uint64_t>(c * (R::kStageBytes >> 4));
          const uint32_t sfa = tmem + kSfACol + 16 * j, sfb = tmem + kSfBCol + 32 * j;
          const int kl = k - ksteps;  // LoRA stages come last
          if (elect_one()) {
            if constexpr (kPair) {
              if (kl >= 0) {
#pragma unroll
                for (int kk = 0; kk < kLoraK / 16; ++kk)
                  mma_f16_pair(tmem, adesc0 + soff + 2 * kk, bdesc0 + soff + 2 * kk, idesc_l,
                               (fp4 || kl || kk) ? 1u : 0u);
              } else if (fp4) {
                mma_stage_nvf4_pair(tmem, adesc0 + soff, bdesc0 + soff, idesc, sfa, sfb, k ? 1u : 0u);
              }
              mma_commit_pair(smem_addr(&mdone[it % kDone]));
            } else {
              if (kl >= 0) {
#pragma unroll
                for (int kk = 0; kk < kLoraK / 16; ++kk)
                  mma_f16_ss(tmem, adesc0 + soff + 2 * kk, bdesc0 + soff + 2 * kk, idesc_l, (fp4 || kl || kk) ? 1u : 0u);
              } else if (fp4) {
                mma_stage_nvf4(tmem, adesc0 + soff, bdesc0 + soff, idesc, sfa, sfb, k ? 1u : 0u);
              }
              mma_commit(smem_addr(&mdone[it % kDone]));
            }
          }
          __syncwarp();
          ++it;
          if (++c == S) c = 0;
        }
        if (!ok) break;
        if (elect_one()) {
          if constexpr (kPair) mma_commit_pair(smem_addr(dfull));
          else mma_commit(smem_addr(dfull));
        }
        __syncwarp();
      }
    }
    __syncwarp();
  } else if (warp >= kFirstSf && warp < kFirstEpi) {
    // ---------------------------------------------------------------- scale warps
    // Group g (warps 4-7: g = 0, 8-11: g = 1) takes the stages it with it % 2 == g; stage it uses
    // TMEM scale slot it % kSlots. FP4 stage: lane i of quarter q reads activation row 32q + i (its
    // four K-step words) and writes them to columns 4t + w of the slot's activation part (for every
    // w; the MMA reads 4t + q), and reads weight rows 32w + i, w = 0..7, writing column 8t + w of the
    // slot's weight part = row 32w + i, K step t (all 256 rows, in each CTA of a pair). LoRA stage: the slices have landed. Either way the group
    // then arrives on sfready (a pair's leader's), which the MMA issuer waits on alone.
    const int q = warp & 3;
    const uint32_t lane_base = static_cast<uint32_t>(q * 32) << 16;
    const int g = (warp - kFirstSf) >> 2;
    const int my_tiles = unit < ntiles ? (ntiles - 1 - unit) / units + 1 : 0;
    const int total = my_tiles * ns;
    for (int it = g; it < total && ok; it += 2) {
      const int li = it / ns, k = it - li * ns;
      const int j = it % kSlots;
      // slot j (and, for its barrier, stage it - kSlots's hand-over) is free once the MMAs of
      // that stage have completed
      const int prev = it - kSlots;
      if (prev >= 0) {
        ok = __all_sync(0xFFFFFFFFu, mbar_wait(smem_addr(&mdone[prev % kDone]), (prev / kDone) & 1, p.status,
                                               kStatusTimeoutMma));
        if (!ok) break;
      }
      if (k < ksteps) {
        const int fi = li * ksteps + k;  // FP4 stage count: the scale ring's index
        const int f = fi % kSfRing;
        ok = __all_sync(0xFFFFFFFFu, mbar_wait(smem_addr(&ffull[f]), static_cast<uint32_t>((fi / kSfRing) & 1),
                                               p.status, kStatusTimeoutMma));
        if (!ok) break;
        tc_fence_after();
        const uint32_t slot_a = tmem + lane_base + kSfACol + 16 * j, slot_b = tmem + lane_base + kSfBCol + 32 * j;
        const uint8_t* st = sfring + f * kSfStage;
        const uint4 a = reinterpret_cast<const uint4*>(st)[q * 32 + lane];
        tmem_st16_rep4(slot_a, a.x, a.y, a.z, a.w);
        // weight scales: row 32w + lane whole (16 bytes, one conflict-free load per row), then two
        // stores of 16 columns: K steps 0-1 (words x, y), then 2-3 (words z, w)
        uint4 r[8];
#pragma unroll
        for (int w = 0; w < 8; ++w) r[w] = reinterpret_cast<const uint4*>(st + kSfA)[w * 32 + lane];
        {
          uint32_t b[16];
#pragma unroll
          for (int w = 0; w < 8; ++w) {
            b[w] = r[w].x;
            b[8 + w] = r[w].y;
          }
          tmem_st16(slot_b, b);
        }
        {
          uint32_t b[16];
#pragma unroll
          for (int w = 0; w < 8; ++w) {
            b[w] = r[w].z;
            b[8 + w] = r[w].w;
          }
          tmem_st16(slot_b + 16, b);
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_addr(&fempty[f]));  // the scale tiles have been read
        tmem_st_wait();
        tc_fence_before();
      }
      // the stage's operand tiles have landed too
      ok = __all_sync(0xFFFFFFFFu, mbar_wait(smem_addr(&cfull[it % S]), static_cast<uint32_t>((it / S) & 1),
                                             p.status, kStatusTimeoutMma));
      if (!ok) break;
      __syncwarp();
      if (lane == 0) {
        if (rank == 0) mbar_arrive(smem_addr(&sfready[j]));
        else mbar_arrive_remote(dsmem_map(smem_addr(&sfready[j]), 0));
      }
    }
  } else if (warp >= kFirstEpi) {
    // ---------------------------------------------------------------- epilogue (16 warps)
    const int q = warp & 3;
    const int part = (warp - kFirstEpi) >> 2;  // columns 64 part .. 64 part + 63
    const uint32_t lane_base = static_cast<uint32_t>(q * 32) << 16;
    const float gx = *p.g_x;
    int li = 0;
    for (int t = unit; t < ntiles && ok; t += units, ++li) {
      ok = __all_sync(0xFFFFFFFFu, mbar_wait(smem_addr(dfull), static_cast<uint32_t>(li & 1), p.status,
                                             kStatusTimeoutEpilogue));
      if (!ok) break;
      tc_fence_after();
      const TileInfo ti = tile_of<kPair>(p, t, rank);
      const float alpha = gx * p.w_g[ti.e];
      const float out = nl && alpha == 0.f ? 1.f : alpha;
      // this thread's row (TMEM lane 32q + lane), columns 64 part .. + 63, scaled and packed: unit u
      // (16 bytes) = o[4u .. 4u + 3] = columns 8u .. 8u + 7
      // 32 columns per load, each waited and packed: two waits instead of four
      uint32_t o[32];
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {
        uint32_t d[32];
        tmem_ld32(tmem + lane_base + part * 64 + hh * 32, d);
        tmem_ld_wait();
#pragma unroll
        for (int i = 0; i < 16; ++i)
          o[hh * 16 + i] = pack_bf16x2(__uint_as_float(d[2 * i]) * out, __uint_as_float(d[2 * i + 1]) * out);
      }
      // D has been read: the next tile's MMAs may start while this warp stores
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        if (rank == 0) mbar_arrive(smem_addr(dfree));
        else mbar_arrive_remote(dsmem_map(smem_addr(dfree), 0));
      }
      // 8 x 8 transpose of 16-byte units within each group of 8 lanes: afterwards lane 8G + k holds
      // unit k of rows 8G .. 8G + 7 of the warp's 32 (in o[4j .. 4j + 3] for row 8G + j), so that
      // each store instruction writes four whole 128-byte row pieces instead of 32 scattered 32-byte
      // ones
#pragma unroll
      for (int dd = 1; dd < 8; dd <<= 1) {
        const bool hi = (lane & dd) != 0;
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          if (u & dd) continue;
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const uint32_t send = hi ? o[4 * u + e] : o[4 * (u ^ dd) + e];
            const uint32_t recv = __shfl_xor_sync(0xFFFFFFFFu, send, dd);
            if (hi) o[4 * u + e] = recv;
            else o[4 * (u ^ dd) + e] = recv;
          }
        }
      }
      const int kk = lane & 7, grp = lane >> 3;
      if (ti.n0 + part * 64 < p.N) {
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const int64_t m = ti.m0 + q * 32 + grp * 8 + j;
          if (m < ti.m_end)
            *reinterpret_cast<uint4*>(p.y + m * p.N + ti.n0 + part * 64 + kk * 8) =
                make_uint4(o[4 * j], o[4 * j + 1], o[4 * j + 2], o[4 * j + 3]);
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if constexpr (kPair) cluster_sync_all();  // neither CTA leaves while the other may still signal it
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    if constexpr (kPair) tmem_dealloc_pair(tmem, 512);
    else tmem_dealloc(tmem, 512);
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
  bool pair;   // CTA pairs (dense calls with at least two row tiles)
  int stages;
  size_t smem, ws_codes, ws_scales, ws_amax, ws_gx, ws_uh, ws_ul, ws_tiles, ws_total;
};

W4a4Plan w4a4_plan(int64_t M, int64_t K, int r, int groups, bool prequantized = false, bool grouped = false) {
  W4a4Plan t{};
  t.pair = !grouped && M > kTile;
  const size_t fixed = 1024 + kSfRing * kSfStage + 512;
  const size_t stage = t.pair ? Ring<true>::kStageBytes : Ring<false>::kStageBytes;
  const size_t max_stages = t.pair ? Ring<true>::kMaxStages : Ring<false>::kMaxStages;
  t.stages = static_cast<int>(std::min<size_t>(max_stages, (227 * 1024 - fixed) / stage));
  t.smem = fixed + t.stages * stage;
  size_t o = 0;
  auto take = [&](size_t b) { size_t at = o; o = align_up(o + b, 256); return at; };
  // activation codes, scales, amax word and g_x, unless the caller passes them in NVFP4
  t.ws_codes = take(prequantized ? 0 : static_cast<size_t>(M) * K / 2);
  t.ws_scales = take(prequantized ? 0 : static_cast<size_t>(M) * K / 16);
  t.ws_amax = take(prequantized ? 0 : kQuantizeWorkspace);
  t.ws_gx = take(prequantized ? 0 : 16);
  // hi and lo of c U
  t.ws_uh = take(static_cast<size_t>(M) * std::max(r, 1) * 2);
  t.ws_ul = take(static_cast<size_t>(M) * std::max(r, 1) * 2);
  t.ws_tiles = take(static_cast<size_t>(groups + 2) * 4);
  t.ws_total = o;
  return t;
}

// CTA pairs of the pair kernel that fit on the device at once (cached per device and shared-memory size).
int pair_clusters(int device, int smem) {
  static std::mutex mu;
  static std::map<std::pair<int, int>, int> cache;
  std::lock_guard<std::mutex> lock(mu);
  const auto key = std::make_pair(device, smem);
  auto it = cache.find(key);
  if (it != cache.end()) return it->second;
  int n = 0;
  if (cudaFuncSetAttribute(w4a4_wide_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) == cudaSuccess &&
      cudaFuncSetAttribute(w4a4_wide_kernel<true>, cudaFuncAttributeNonPortableClusterSizeAllowed, 0) == cudaSuccess) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2, 1, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = static_cast<size_t>(smem);
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (cudaOccupancyMaxActiveClusters(&n, reinterpret_cast<const void*>(w4a4_wide_kernel<true>), &cfg) != cudaSuccess)
      n = 0;
  }
  if (n <= 0) cudaGetLastError();
  cache[key] = n;
  return n;
}

}  // namespace

bool w4a4_tc_supported(int64_t M, int64_t N, int64_t K, int r) {
  return M > 0 && N % kTile == 0 && K % kKStage == 0 && (r == 0 || (r % 16 == 0 && r <= kMaxLoraRank)) &&
         w4a4_plan(M, K, r, 1).stages >= 3;
}

size_t w4a4_tc_workspace_bytes(int64_t M, int64_t N, int64_t K, int r, int groups, bool prequantized) {
  (void)N;
  return w4a4_plan(M, K, r, groups, prequantized).ws_total;
}

nvfp4rl_status launch_w4a4_tc(const LinearArgs& a, void* ws, size_t ws_bytes, const DeviceInfo& dev,
                              cudaStream_t st) {
  const int groups = a.offsets ? a.groups : 1;
  const bool pre = a.xq_codes != nullptr;
  const W4a4Plan t = w4a4_plan(a.M, a.K, a.r, groups, pre, a.offsets != nullptr);
  if (ws_bytes < t.ws_total) return NVFP4RL_ERR_WORKSPACE;
  const uint32_t brows = t.pair ? Ring<true>::kBRows : Ring<false>::kBRows;  // weight rows per CTA
  char* base = static_cast<char*>(ws);
  const uint8_t* xc = pre ? a.xq_codes : reinterpret_cast<uint8_t*>(base + t.ws_codes);
  const uint8_t* xs = pre ? a.xq_scales : reinterpret_cast<uint8_t*>(base + t.ws_scales);
  const float* gx = pre ? a.xq_g : reinterpret_cast<float*>(base + t.ws_gx);
  uint16_t* Uh = reinterpret_cast<uint16_t*>(base + t.ws_uh);
  uint16_t* Ul = reinterpret_cast<uint16_t*>(base + t.ws_ul);
  int32_t* tiles = reinterpret_cast<int32_t*>(base + t.ws_tiles);

  LoraDownScale ls;  // hi and lo of c U
  ls.g_x = gx;
  ls.w_g = a.w_g;
  ls.s = a.s;
  ls.lo = Ul;
  ls.status = dev.status;
  uint8_t* qcodes = reinterpret_cast<uint8_t*>(base + t.ws_codes);
  uint8_t* qscales = reinterpret_cast<uint8_t*>(base + t.ws_scales);
  float* qg = reinterpret_cast<float*>(base + t.ws_gx);
  uint32_t* amax = reinterpret_cast<uint32_t*>(base + t.ws_amax);
  if (!pre && a.r && lora_down_tc_supported(a.M, a.K, a.r)) {
    // x is read twice instead of three times: the tensor-core LoRA-down takes max |x| from the tiles it
    // streams, the encoding then needs no amax pass; U is scaled to hi/lo once g_x is known
    nvfp4rl_status e = launch_zero_word(amax, st);
    if (e == NVFP4RL_OK) e = launch_lora_down_tc(a.x, a.M, a.K, a.A, a.r, Uh, dev, st, LoraDownScale{}, amax);
    if (e == NVFP4RL_OK)
      e = launch_quantize(a.x, NVFP4RL_BF16, a.M, a.K, nullptr, qcodes, qscales, qg, nullptr, amax, dev, st, true);
    if (e == NVFP4RL_OK) e = launch_lora_scale(Uh, a.M, a.r, ls, dev, st);
    if (e != NVFP4RL_OK) return e;
  } else {
    if (!pre) {
      const nvfp4rl_status sq = launch_quantize(a.x, NVFP4RL_BF16, a.M, a.K, nullptr, qcodes, qscales, qg, nullptr,
                                                amax, dev, st);
      if (sq != NVFP4RL_OK) return sq;
    }
    if (a.r) {
      const nvfp4rl_status sd = launch_lora_down(a.x, a.M, a.K, a.A, a.r, Uh, dev, st, ls);
      if (sd != NVFP4RL_OK) return sd;
    }
  }
  if (a.offsets) {
    tile_map128_kernel<<<1, 1024, 0, st>>>(a.offsets, groups, tiles);
    if (launch_status() != NVFP4RL_OK) return NVFP4RL_ERR_CUDA;
  }
  CUtensorMap mxc, mxs, mwc, mws, muh, mul, mb;
  const uint64_t wrows = static_cast<uint64_t>(groups) * a.N;
  if (!make_tensor_map_2d(&mxc, CU_TENSOR_MAP_DATA_TYPE_UINT8, xc, a.K / 2, a.M, 1, 128, kTile, CU_TENSOR_MAP_SWIZZLE_128B) ||
      !make_tensor_map_2d(&mxs, CU_TENSOR_MAP_DATA_TYPE_UINT8, xs, a.K / 16, a.M, 1, 16, kTile, CU_TENSOR_MAP_SWIZZLE_NONE) ||
      !make_tensor_map_2d(&mwc, CU_TENSOR_MAP_DATA_TYPE_UINT8, a.w_codes, a.K / 2, wrows, 1, 128, brows,
                          CU_TENSOR_MAP_SWIZZLE_128B) ||
      !make_tensor_map_2d(&mws, CU_TENSOR_MAP_DATA_TYPE_UINT8, a.w_scales, a.K / 16, wrows, 1, 16, kWN,
                          CU_TENSOR_MAP_SWIZZLE_NONE))
    return NVFP4RL_ERR_CUDA;
  if (a.r) {
    // 64-rank slices (128-byte rows, 128-byte swizzle, like the code tiles); ranks past r (r not a
    // multiple of 64) read as zeros
    if (!make_tensor_map_2d(&muh, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, Uh, a.r, a.M, 2, kLoraK, kTile,
                            CU_TENSOR_MAP_SWIZZLE_128B) ||
        !make_tensor_map_2d(&mul, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, Ul, a.r, a.M, 2, kLoraK, kTile,
                            CU_TENSOR_MAP_SWIZZLE_128B) ||
        !make_tensor_map_2d(&mb, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, a.B, a.r, a.N, 2, kLoraK, brows,
                            CU_TENSOR_MAP_SWIZZLE_128B))
      return NVFP4RL_ERR_CUDA;
  } else {
    muh = mul = mb = mxc;
  }
  W4a4Params p{};
  p.M = a.M;
  p.N = a.N;
  p.K = a.K;
  p.tiles_n = static_cast<int>((a.N + kWN - 1) / kWN);
  const int64_t tiles_m_bound = a.offsets ? (a.M + kTile - 1) / kTile + groups : (a.M + kTile - 1) / kTile;
  p.tiles_m = static_cast<int>((a.M + kTile - 1) / kTile);
  p.total_tiles = (t.pair ? (p.tiles_m + 1) / 2 : p.tiles_m) * p.tiles_n;  // pair tiles for a pair
  p.r = a.r;
  p.s = a.s;
  p.g_x = gx;
  p.w_g = a.w_g;
  p.offsets = a.offsets;
  p.tile_start = tiles;
  p.groups = groups;
  p.y = a.y;
  p.status = dev.status;
  p.stages = t.stages;
  // With LoRA, the GEMM is a programmatic dependent of the kernel before it (the LoRA-down, or the
  // hi/lo split): it runs its FP4 stages while that kernel finishes and waits for it
  // (griddepcontrol.wait) only before loading U, for the LoRA stages at the end of a tile. What it
  // reads before that (activation codes, scales and g_x, the weights, B_lora) was complete before
  // that kernel's own wait returned. Without LoRA the kernel before it may be the activation encode,
  // so the launch is an ordinary one.
  cudaLaunchAttribute pdl;
  pdl.id = cudaLaunchAttributeProgrammaticStreamSerialization;
  pdl.val.programmaticStreamSerializationAllowed = 1;
  if (!t.pair) {
    const int64_t max_tiles = tiles_m_bound * p.tiles_n;
    const int grid = static_cast<int>(std::min<int64_t>(max_tiles, dev.sm_count));
    if (cudaFuncSetAttribute(w4a4_wide_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(t.smem)) != cudaSuccess)
      return NVFP4RL_ERR_CUDA;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(grid), 1, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = t.smem;
    cfg.stream = st;
    cfg.attrs = &pdl;
    cfg.numAttrs = a.r ? 1 : 0;
    if (cudaLaunchKernelEx(&cfg, w4a4_wide_kernel<false>, mxc, mxs, mwc, mws, muh, mul, mb, p) != cudaSuccess)
      return NVFP4RL_ERR_CUDA;
    return launch_status();
  }
  const int clusters = pair_clusters(dev.device, static_cast<int>(t.smem));
  if (clusters <= 0) return NVFP4RL_ERR_CUDA;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(2 * std::min<int64_t>(p.total_tiles, clusters)), 1, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = t.smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1] = pdl;
  cfg.attrs = attr;
  cfg.numAttrs = a.r ? 2 : 1;
  if (cudaLaunchKernelEx(&cfg, w4a4_wide_kernel<true>, mxc, mxs, mwc, mws, muh, mul, mb, p) != cudaSuccess)
    return NVFP4RL_ERR_CUDA;
  return launch_status();
}

}  // namespace nvfp4rl
