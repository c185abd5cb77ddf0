// W4A16 NVFP4 LoRA linear on the 5th-generation tensor cores (tcgen05), sm_103a.
//
// QeRL explainer, section "NVFP4量子化とLoRA": the rollout runs frozen NVFP4 base weights
// plus trainable LoRA factors, Y = x deq(W)^T + s (x A^T) B^T. In decode the layer is bound
// by the HBM stream of 4-bit weights (0.5625 bytes per weight with the block scales).
//
// One call = two kernels on the caller's stream:
//   w4a16_lora_down_kernel  U = bf16(x A^T) for the LoRA up-projection: a cluster of CTAs
//                           splits K, each streams its chunks through a cp.async ring into
//                           mma.sync, and the partial sums meet in distributed shared memory
//                           (fixed order, no atomics).
//   w4a16_tc_kernel         launched as a programmatic dependent of the first: it starts while
//                           the LoRA-down runs and waits for it (griddepcontrol.wait) only
//                           before loading U, after its whole weight stream has been issued.
//
// w4a16_tc_kernel (one CTA = 128 weight rows x one K range x up to 128 tokens):
//   warp 0      weight producer (TMA): per 256-K stage the 128 x 128-byte code tile (128-byte
//               swizzle) and the 128 x 16-byte scale tile, into a deep weight ring.
//   warp 1      allocates TMEM; one thread issues tcgen05.mma kind::f16 with A (the
//               dequantized weights) in TMEM and B (activations) in shared memory, then the
//               LoRA up-projection (B_lora tile x U^T) into a second accumulator.
//   warp 2      activation producer (TMA): per 128-K sub-stage two boxes of 64 bf16 x tokens
//               (128-byte swizzle, read straight from x) into a separate, shallower ring;
//               plus the LoRA tiles.
//   warps 3-18  dequantize: thread = one weight row and a quarter of the stage's K; each code
//               byte is converted to f16x2 by the hardware, moved to a bf16 pattern (one shift
//               and mask) and scaled by one bf16x2 FMA by E4M3(s) * 2^80, written to TMEM with
//               tcgen05.st; then the epilogue: TMEM -> registers, g and s applied, bf16 stores.
// The weight ring is released by the dequant warps and the activation ring by the MMAs, so
// the HBM weight stream runs ahead independently of the L2-resident activation tiles. Each
// output tile starts its K range at a different stage (the CTAs then read different
// activation tiles at any one time).
// When K is split across CTAs, the CTAs of one output tile form a cluster; each CTA owns a slice
// of the tile's tokens. After a cluster barrier every CTA pushes its fp32 partial of each token
// into the owner's shared memory (remote stores into the free activation ring); after a second
// barrier each owner sums its slice over the partials in split order and writes it.
// The thread that initializes the barriers also requests the first ring stages, before the
// block's set-up (TMEM allocation, the block barrier) completes.
//
// Dequant: each code byte becomes an f16x2 by the hardware conversion (cvt.rn.f16x2.e2m1x2); the
// f16 pattern shifted right by 3 (sign kept) is the bf16 pattern of the value times 2^-112, and
// one bf16x2 FMA by E4M3(s) * 2^80 gives grid(m) * E4M3(s) * 2^-32 exactly (at most 6 significant
// bits); the epilogue multiplies the fp32 accumulator by 2^32 and then by g. Byte c of a code
// word holds the K pair (2c, 2c+1) of TMEM column c.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <map>
#include <mutex>
#include <tuple>

#include "common.cuh"
#include "sm100.cuh"

namespace nvfp4rl {
namespace {

using namespace sm100;

constexpr int kRows = 128;        // weight rows per CTA (MMA M)
constexpr int kKStage = 256;      // K per pipeline stage
constexpr int kCodeBytes = kRows * kKStage / 2;   // 16 KB
constexpr int kScaleBytes = kRows * kKStage / 16;  // 2 KB
constexpr int kWStageBytes = kCodeBytes + kScaleBytes;  // one weight stage: codes + scales
constexpr int kFirstDeqWarp = 3;  // warps 0-2: weight producer, MMA issuer, activation producer
constexpr int kMaxSplits = 8;     // split-K factor cap = the portable cluster size

constexpr int kDownK = 64;        // K per LoRA-down chunk
constexpr int kDownM = 64;        // activation rows per LoRA-down cluster
constexpr int kDownPad = 8;       // bf16 row padding (conflict-free ldmatrix)
constexpr int kDownStages = 3;    // chunks in flight (cp.async ring)
constexpr int kDownCluster = 16;  // CTAs per LoRA-down cluster (K split); 8 where 16 is not available
// One pass of the kernel covers RP ranks (32, or 64 so that r = 64 reads x once).
template <int RP>
struct DownShape {
  static constexpr int kStageElems = (kDownM + RP) * (kDownK + kDownPad);
  static constexpr int kSmem = kDownStages * kStageElems * 2 + kDownM * RP * 4;
};
constexpr int kDownSmem = DownShape<32>::kSmem;  // the decode instance, which shares an SM with the main kernel

struct TcParams {
  int64_t M, N, K;
  int stages_per_split;  // 256-K stages per CTA
  int splits;            // CTAs per cluster along K (1: no split)
  int r;                 // LoRA rank (0 or a multiple of 16)
  int lora_box_bytes;    // lora_box_bytes_for(r)
  float s;
  const float* w_g;
  uint16_t* y;
  uint32_t* status;
  int w_stages;          // weight ring depth (256-K stages)
};

// activation stage: 256 K (four boxes of 64 bf16) x tokens
__host__ __device__ constexpr int x_stage_bytes(int mbox) { return 4 * mbox * 128; }
// depth of the A-buffer / activation / stage-ready rings
__host__ __device__ constexpr int ring_depth(int mbox) { return mbox <= 64 ? 3 : 2; }
__host__ __device__ constexpr int threads_for(int deq_warps) { return 32 * (kFirstDeqWarp + deq_warps); }

// LoRA operand tiles (B_lora rows, U rows) are loaded in boxes of 2r bytes for r <= 32 and of 128
// bytes (64 ranks) otherwise; a rank that is not a multiple of 64 then leaves the last box partly
// beyond r, which the copy fills with zeros. Shared memory holds lora_padded_rank(r) ranks per row.
__host__ __device__ constexpr int lora_box_bytes_for(int r) { return r <= 32 ? 2 * r : 128; }
__host__ __device__ constexpr int lora_padded_rank(int r) { return r <= 32 ? r : (r + 63) / 64 * 64; }

__device__ __forceinline__ uint32_t swizzle_mode_for(int box_bytes) {
  return box_bytes == 128 ? 2u : box_bytes == 64 ? 4u : 6u;
}

// bf16x2 fma with -0 addend: an exact product where the product is representable.
__device__ __forceinline__ uint32_t bf16x2_mul(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("fma.rn.bf16x2 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(0x80008000u));
  return d;
}

// Four code bytes (two E2M1 elements each, low nibble first) -> four f16x2 (low half = low nibble).
__device__ __forceinline__ void e2m1x8_f16x2(uint32_t w, uint32_t (&d)[4]) {
  asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\t"
      "mov.b32 {b0, b1, b2, b3}, %4;\n\t"
      "cvt.rn.f16x2.e2m1x2 %0, b0;\n\t"
      "cvt.rn.f16x2.e2m1x2 %1, b1;\n\t"
      "cvt.rn.f16x2.e2m1x2 %2, b2;\n\t"
      "cvt.rn.f16x2.e2m1x2 %3, b3;\n\t}"
      : "=r"(d[0]), "=r"(d[1]), "=r"(d[2]), "=r"(d[3])
      : "r"(w));
}

// Four TMEM columns from one word of 8 codes (K order e0..e7): column c = (e_2c, e_2c+1), each a
// bf16 of grid(m) * E4M3(s) * 2^-32 with the code's sign (scale2 = E4M3(s) * 2^80). Byte c of the
// word is converted to f16x2 by the hardware; an E2M1 value as f16 has its mantissa in the top
// bit, so the f16 pattern shifted right by 3 (sign kept in place) is the bf16 pattern of the same
// value times 2^-112; the bf16x2 FMA by E4M3(s) * 2^80 is then exact (at most 6 significant bits).
__device__ __forceinline__ void expand_word(uint32_t w, uint32_t scale2, uint32_t* out) {
  uint32_t h[4];
  e2m1x8_f16x2(w, h);
#pragma unroll
  for (int c = 0; c < 4; ++c) out[c] = bf16x2_mul(((h[c] >> 3) & 0x0FFF0FFFu) | (h[c] & 0x80008000u), scale2);
}

// bf16x2 of E4M3(s) * 2^80 for a normal scale byte s (8 <= s <= 0x7E): the bf16 bits are
// (s << 4) + (200 << 7), i.e. exponent e + 200 and mantissa m << 4; one multiply-add writes
// both halves.
__device__ __forceinline__ uint32_t scale_bf16x2_normal(uint32_t s) { return (s & 0x7Fu) * 0x00100010u + 0x64006400u; }

// bf16x2 of E4M3(s) * 2^80 for any scale byte (exact: at most 4 significant bits).
__device__ __forceinline__ uint32_t scale_bf16x2(uint32_t s) {
  const uint32_t b = __float_as_uint(e4m3_decode_pos(s & 0x7Fu) * 0x1p80f) >> 16;
  return b | (b << 16);
}

// True when any of the eight scale bytes is below 8 (zero or subnormal E4M3).
__device__ __forceinline__ bool has_small_scale(uint2 sc) {
  const uint32_t y0 = sc.x & 0x78787878u, y1 = sc.y & 0x78787878u;
  return (((y0 - 0x01010101u) & ~y0) | ((y1 - 0x01010101u) & ~y1)) & 0x80808080u;
}

// The 16 MMAs of one 256-K stage (M = 128 weight rows, N = MBOX tokens, K = 16 each), issued
// from one instruction sequence: K-step kk reads A from TMEM columns a_tmem + 8 kk and B from the
// activation stage at desc0 advanced by ((kk / 4) MBOX 128 + (kk % 4) 32) bytes (128-byte
// swizzled boxes of 64 bf16 K). The first MMA accumulates only if `accumulate`; the other 15
// always do. Two integer adds per MMA keep the issuing thread's instruction count low.
template <int MBOX>
__device__ __forceinline__ void mma_stage16(uint32_t d_tmem, uint32_t a_tmem, uint64_t desc0, uint32_t idesc,
                                            uint32_t accumulate) {
#define NVFP4RL_BOFF(kk) ((((kk) >> 2) * MBOX * 128 + ((kk)&3) * 32) >> 4)
  asm volatile(
      "{\n\t.reg .pred p, t;\n\t.reg .b32 ta;\n\t.reg .b64 bd;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "setp.eq.b32 t, 0, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t"
      "add.u32 ta, %1, 8;\n\tadd.u64 bd, %2, %5;\n\ttcgen05.mma.cta_group::1.kind::f16 [%0], [ta], bd, %3, t;\n\t"
      "add.u32 ta, %1, 16;\n\tadd.u64 bd, %2, %6;\n\ttcgen05.mma.cta_group::1.kind::f16 [%0], [ta], bd, %3, t;\n\t"
      "add.u32 ta, %1, 24;\n\tadd.u64 bd, %2, %7;\n\ttcgen05.mma.cta_group::1.kind::f16 [%0], [ta], bd, %3, t;\n\t"
      "add.u32 ta, %1, 32;\n\tadd.u64 bd, %2, %8;\n\ttcgen05.mma.cta_group::1.kind::f16 [%0], [ta], bd, %3, t;\n\t"
      "add.u32 ta, %1, 40;\n\tadd.u64 bd, %2, %9;\n\ttcgen05.mma.cta_group::1.kind::f16 [%0], [ta], bd, %3, t;\n\t"
      "add.u32 ta, %1, 48;\n\tadd.u64 bd, %2, %10;\n\ttcgen05.mma.cta_group::1.kind::f16 [%0], [ta], bd, %3, t;\n\t"
      "add.u32 ta, %1, 56;\n\tadd.u64 bd, %2, %11;\n\ttcgen05.mma.cta_group::1.kind::f16 [%0], [ta], bd, %3, t;\n\t"
      "add.u32 ta, %1, 64;\n\tadd.u64 bd, %2, %12;\n\ttcgen05.mma.cta_group::1.kind::f16 [%0], [ta], bd, %3, t;\n\t"
      "add.u32 ta, %1, 72;\n\tadd.u64 bd, %2, %13;\n\ttcgen05.mma.cta_group::1.kind::f16 [%0], [ta], bd, %3, t;\n\t"
      "add.u32 ta, %1, 80;\n\tadd.u64 bd, %2, %14;\n\ttcgen05.mma.cta_group::1.kind::f16 [%0], [ta], bd, %3, t;\n\t"
      "add.u32 ta, %1, 88;\n\tadd.u64 bd, %2, %15;\n\ttcgen05.mma.cta_group::1.kind::f16 [%0], [ta], bd, %3, t;\n\t"
      "add.u32 ta, %1, 96;\n\tadd.u64 bd, %2, %16;\n\ttcgen05.mma.cta_group::1.kind::f16 [%0], [ta], bd, %3, t;\n\t"
      "add.u32 ta, %1, 104;\n\tadd.u64 bd, %2, %17;\n\ttcgen05.mma.cta_group::1.kind::f16 [%0], [ta], bd, %3, t;\n\t"
      "add.u32 ta, %1, 112;\n\tadd.u64 bd, %2, %18;\n\ttcgen05.mma.cta_group::1.kind::f16 [%0], [ta], bd, %3, t;\n\t"
      "add.u32 ta, %1, 120;\n\tadd.u64 bd, %2, %19;\n\ttcgen05.mma.cta_group::1.kind::f16 [%0], [ta], bd, %3, t;\n\t"
      "}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(desc0), "r"(idesc), "r"(accumulate), "n"(NVFP4RL_BOFF(1)), "n"(NVFP4RL_BOFF(2)),
      "n"(NVFP4RL_BOFF(3)), "n"(NVFP4RL_BOFF(4)), "n"(NVFP4RL_BOFF(5)), "n"(NVFP4RL_BOFF(6)), "n"(NVFP4RL_BOFF(7)),
      "n"(NVFP4RL_BOFF(8)), "n"(NVFP4RL_BOFF(9)), "n"(NVFP4RL_BOFF(10)), "n"(NVFP4RL_BOFF(11)),
      "n"(NVFP4RL_BOFF(12)), "n"(NVFP4RL_BOFF(13)), "n"(NVFP4RL_BOFF(14)), "n"(NVFP4RL_BOFF(15))
      : "memory");
#undef NVFP4RL_BOFF
}

// Dequantizes one thread's share of a stage (row `row`, chunks c0 .. c0 + NCH - 1 of 32 codes)
// into TMEM columns starting at taddr + 16 * chunk. sc holds the chunks' scale bytes, two per
// chunk, in order.
template <bool kAnyScale, int NCH>
__device__ __forceinline__ void dequant_chunks(const uint8_t* crow, int row, int c0, uint2 sc, uint32_t taddr) {
  const uint32_t sbytes[2] = {sc.x, sc.y};
#pragma unroll
  for (int c = 0; c < NCH; ++c) {  // 16-byte chunk = 32 codes = two MMA K-steps
    const int chunk = c0 + c;
    const uint4 cw = *reinterpret_cast<const uint4*>(crow + ((chunk ^ (row & 7)) << 4));
    const uint32_t b0 = (sbytes[c >> 1] >> (16 * (c & 1))) & 0xFFu;
    const uint32_t b1 = (sbytes[c >> 1] >> (16 * (c & 1) + 8)) & 0xFFu;
    const uint32_t s0 = kAnyScale ? scale_bf16x2(b0) : scale_bf16x2_normal(b0);
    const uint32_t s1 = kAnyScale ? scale_bf16x2(b1) : scale_bf16x2_normal(b1);
    uint32_t col[8];
    expand_word(cw.x, s0, col);
    expand_word(cw.y, s0, col + 4);
    tmem_st8(taddr + chunk * 16, col);
    expand_word(cw.z, s1, col);
    expand_word(cw.w, s1, col + 4);
    tmem_st8(taddr + chunk * 16 + 8, col);
  }
}

// Split-K reduction over distributed shared memory, for a cluster of C CTAs that computed the same
// output tile over C ranges of K. CTA q owns the tile's tokens [q slice, (q + 1) slice), slice =
// ceil(MBOX / C). After a cluster barrier (every CTA's MMAs done: `red` is free in every CTA) each
// CTA writes its fp32 partial of every token into the owner's buffer, red[q][token - slice owner]
// [row] (remote stores, rows in lanes); after a second barrier each owner sums its tokens over the
// splits in split order from its own shared memory and writes them, 8 rows (16 bytes) per store.
// No CTA reads another's memory, so none has to wait for its peers before leaving. load16(col, v):
// this thread's 16 partial values of its row (TMEM lane) from token col on.
template <int MBOX, int DW, class Load16>
__device__ __forceinline__ void splitk_push_reduce(float* red, const TcParams& p, bool have, int warp, int lane,
                                                   int64_t m0, int n0, Load16 load16) {
  constexpr int kEpiTok = MBOX / (DW / 4);  // tokens per epilogue warp
  const int C = p.splits;
  const int q = static_cast<int>(cluster_ctarank());
  const int slice = (MBOX + C - 1) / C;
  __syncwarp();
  cluster_sync_all();
  if (warp >= kFirstDeqWarp && have) {
    tc_fence_after();
    const int row = (warp & 3) * 32 + lane;
    const int t0 = ((warp - kFirstDeqWarp) >> 2) * kEpiTok;
#pragma unroll 1
    for (int c = 0; c < kEpiTok; c += 16) {
      float v[16];
      load16(t0 + c, v);
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        const int t = t0 + c + i;
        const int owner = t / slice;
        const uint32_t local = smem_addr(red + (q * slice + (t - owner * slice)) * kRows + row);
        dsmem_st_f32(dsmem_map(local, static_cast<uint32_t>(owner)), v[i]);
      }
    }
  }
  __syncwarp();
  cluster_sync_all();
  if (warp >= kFirstDeqWarp) {
    const int tb = q * slice, te = min(MBOX, tb + slice);
    constexpr int kPerTok = kRows / 8;  // 8 rows (two float4) per item
    for (int idx = (warp - kFirstDeqWarp) * 32 + lane; idx < (te - tb) * kPerTok; idx += DW * 32) {
      const int lt = idx / kPerTok, r8 = (idx % kPerTok) * 8;
      const int64_t m = m0 + tb + lt;
      if (m >= p.M) continue;
      float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
      for (int sp = 0; sp < C; ++sp) {
        const float4* src = reinterpret_cast<const float4*>(red + (sp * slice + lt) * kRows + r8);
        const float4 va = src[0], vb = src[1];
        acc[0] += va.x; acc[1] += va.y; acc[2] += va.z; acc[3] += va.w;
        acc[4] += vb.x; acc[5] += vb.y; acc[6] += vb.z; acc[7] += vb.w;
      }
      uint32_t o[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) o[i] = f32_to_bf16_bits(acc[2 * i]) | (f32_to_bf16_bits(acc[2 * i + 1]) << 16);
      *reinterpret_cast<uint4*>(p.y + m * p.N + n0 + r8) = make_uint4(o[0], o[1], o[2], o[3]);
    }
  }
}

// 88 registers per thread: 608 threads of this kernel and a 128-thread LoRA-down CTA (72 registers)
// fit the 64K-register file of one SM together.
template <int MBOX, int DW>
__global__ void __maxnreg__(88)
    w4a16_tc_kernel(const __grid_constant__ CUtensorMap map_codes, const __grid_constant__ CUtensorMap map_scales,
                    const __grid_constant__ CUtensorMap map_x, const __grid_constant__ CUtensorMap map_blora,
                    const __grid_constant__ CUtensorMap map_u, const TcParams p) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int SW = p.w_stages;
  constexpr int R = ring_depth(MBOX);                // A buffers = activation stages = ready slots
  constexpr int kWarpsPerQuarter = DW / 4;           // dequant warps sharing one TMEM lane quarter
  constexpr int kChunks = 8 / kWarpsPerQuarter;      // 16-byte code chunks per thread and stage
  constexpr uint32_t kDcol = 0, kLcol = MBOX, kAcol0 = 2 * MBOX;
  constexpr int kXBytes = x_stage_bytes(MBOX);
  constexpr int kEpiTok = MBOX / kWarpsPerQuarter;  // tokens per epilogue warp (multiple of 16)
  static_assert((MBOX + kMaxSplits - 1) * kRows * 4 <= R * kXBytes, "split-K partials fit the activation ring");

  // layout: activation ring (reused as the fp32 partial tile after the K loop) | weight ring |
  //         lora A tile | lora U tile | barriers
  uint8_t* xring = smem;
  uint8_t* wring = xring + R * kXBytes;
  uint8_t* lora_a = wring + SW * kWStageBytes;
  const int lora_a_bytes = p.r ? kRows * 2 * lora_padded_rank(p.r) : 0;
  uint8_t* lora_u = lora_a + lora_a_bytes;
  const int lora_u_bytes = p.r ? MBOX * 2 * lora_padded_rank(p.r) : 0;
  uint64_t* bars = reinterpret_cast<uint64_t*>(lora_u + lora_u_bytes);
  uint64_t* wfull = bars;             // [SW] weight stage landed
  uint64_t* wempty = wfull + SW;      // [SW] weight stage dequantized (DW arrivals)
  // Stage j of the MMAs needs its A buffer written and its activation tile landed: one barrier
  // per slot collects both (DW dequant arrivals + the activation producer's arrival and bytes),
  // so the MMA issuer waits once per stage. One commit per stage releases both again.
  uint64_t* ready = wempty + SW;      // [R]
  uint64_t* consumed = ready + R;     // [R] the stage's MMAs have completed (commit)
  uint64_t* dfull = consumed + R;
  uint64_t* lfull = dfull + 1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(lfull + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int tile_n = blockIdx.x, split = blockIdx.y, tile_m = blockIdx.z;
  const int n0 = tile_n * kRows;
  const int m0 = tile_m * MBOX;
  const int st0 = split * p.stages_per_split;
  const int nst = min(p.stages_per_split, static_cast<int>(p.K / kKStage) - st0);
  const bool do_lora = p.r > 0 && split == 0;

  if (threadIdx.x == 0) {
    for (int i = 0; i < SW; ++i) {
      mbar_init(smem_addr(&wfull[i]), 1);
      mbar_init(smem_addr(&wempty[i]), DW);
    }
    for (int i = 0; i < R; ++i) {
      mbar_init(smem_addr(&ready[i]), DW + 1);
      mbar_init(smem_addr(&consumed[i]), 1);
    }
    mbar_init(smem_addr(dfull), 1);
    mbar_init(smem_addr(lfull), 1);
    fence_barrier_init();
  }
  // Each output tile starts its K range at a different stage, so that the CTAs do not all read
  // the same activation tile from L2 at the same time. Producers and consumers all walk the
  // stages in this order.
  auto kstage = [&](int j) { return st0 + (j + tile_n) % nst; };
  // The first weight and activation stages (as many as the rings hold) are requested by the
  // thread that initialized their barriers, before TMEM is allocated and the block meets; the
  // producers continue from there. (x and the weights are complete when this kernel starts: it
  // is launched after, or as the programmatic dependent of a kernel that waited for, their
  // producers.)
  const int w_pre = min(SW, nst), x_pre = min(R, nst);
  if (threadIdx.x == 0) {
    for (int j = 0; j < w_pre; ++j) {
      uint8_t* st = wring + j * kWStageBytes;
      const uint32_t bar = smem_addr(&wfull[j]);
      mbar_arrive_expect_tx(bar, kWStageBytes);
      tma_load_2d(smem_addr(st), &map_codes, kstage(j) * (kKStage / 2), n0, bar);
      tma_load_2d(smem_addr(st + kCodeBytes), &map_scales, kstage(j) * (kKStage / 16), n0, bar);
    }
    for (int j = 0; j < x_pre; ++j) {
      uint8_t* st = xring + j * kXBytes;
      const uint32_t bar = smem_addr(&ready[j]);
      mbar_arrive_expect_tx(bar, kXBytes);
#pragma unroll
      for (int q = 0; q < 4; ++q)
        tma_load_2d(smem_addr(st + q * MBOX * 128), &map_x, kstage(j) * kKStage + q * 64, m0, bar);
    }
  }
  if (warp == 1) tmem_alloc(smem_addr(tmem_slot), 512);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  // Sixteen tokens of this thread's weight row (TMEM lane) from the accumulators, starting at
  // token col: the base product times 2^32 g, plus s times the LoRA accumulator.
  auto epilogue16 = [&](uint32_t tlane, int col, bool lora, float g, float s_lora, float(&v)[16]) {
    uint32_t d[16], l[16];
    tmem_ld16(tlane + kDcol + col, d);
    if (lora) tmem_ld16(tlane + kLcol + col, l);
    tmem_ld_wait();
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      v[i] = (__uint_as_float(d[i]) * 0x1p32f) * g;
      if (lora) v[i] = fmaf(s_lora, __uint_as_float(l[i]), v[i]);
    }
  };

  bool ok = true;
  if (warp == 0) {
    // ------------------------------------------------------------------ weight producer
    if (lane == 0) {
      int issued = w_pre;
      for (int j = w_pre; j < nst && ok; ++j) {
        const int s = j % SW;
        if (!mbar_wait(smem_addr(&wempty[s]), ((j / SW) & 1) ^ 1, p.status, kStatusTimeoutProducer)) {
          ok = false;
          break;
        }
        uint8_t* st = wring + s * kWStageBytes;
        const uint32_t bar = smem_addr(&wfull[s]);
        mbar_arrive_expect_tx(bar, kWStageBytes);
        const int kst = kstage(j);
        tma_load_2d(smem_addr(st), &map_codes, kst * (kKStage / 2), n0, bar);
        tma_load_2d(smem_addr(st + kCodeBytes), &map_scales, kst * (kKStage / 16), n0, bar);
        issued = j + 1;
      }
      // drain: every issued copy has landed before the CTA exits
      for (int j = max(0, issued - SW); j < issued; ++j)
        mbar_wait(smem_addr(&wfull[j % SW]), (j / SW) & 1, p.status, kStatusTimeoutDrain);
    }
  } else if (warp == 2) {
    // ------------------------------------------------------------------ activation + LoRA producer
    if (lane == 0) {
      const int nbox = do_lora ? 2 * lora_padded_rank(p.r) / p.lora_box_bytes : 0;
      const int box_el = p.lora_box_bytes / 2;
      if (do_lora) {
        // B_lora is an input of the call; U comes from the LoRA-down kernel (loaded at the end)
        prefetch_tensormap(&map_blora);
        prefetch_tensormap(&map_u);
        mbar_arrive_expect_tx(smem_addr(lfull), lora_a_bytes + lora_u_bytes);
        for (int b = 0; b < nbox; ++b)
          tma_load_2d(smem_addr(lora_a + b * kRows * p.lora_box_bytes), &map_blora, b * box_el, n0, smem_addr(lfull));
      }
      int issued = x_pre;
      for (int j = x_pre; j < nst && ok; ++j) {
        const int s = j % R;
        if (!mbar_wait(smem_addr(&consumed[s]), ((j / R) & 1) ^ 1, p.status, kStatusTimeoutProducer)) {
          ok = false;
          break;
        }
        uint8_t* st = xring + s * kXBytes;
        const uint32_t bar = smem_addr(&ready[s]);
        mbar_arrive_expect_tx(bar, kXBytes);
        const int k0 = kstage(j) * kKStage;
#pragma unroll
        for (int q = 0; q < 4; ++q) tma_load_2d(smem_addr(st + q * MBOX * 128), &map_x, k0 + q * 64, m0, bar);
        issued = j + 1;
      }
      if (do_lora) {
        griddep_wait();  // the LoRA-down kernel has completed and its U is visible
        for (int b = 0; b < nbox; ++b)
          tma_load_2d(smem_addr(lora_u + b * MBOX * p.lora_box_bytes), &map_u, b * box_el, m0, smem_addr(lfull));
      }
      // drain: the last stages' activation copies have landed (their ready phases completed)
      // before the shared memory is reused or the CTA exits
      for (int j = max(0, issued - R); j < issued; ++j)
        mbar_wait(smem_addr(&ready[j % R]), (j / R) & 1, p.status, kStatusTimeoutDrain);
      if (do_lora) mbar_wait(smem_addr(lfull), 0, p.status, kStatusTimeoutDrain);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------------ MMA issuer
    // The whole warp walks the stages and waits; one elected lane issues each stage's MMAs
    // and commit (the same lane every time).
    const uint32_t idesc = idesc_bf16_f32(kRows, MBOX);
    for (int j = 0; j < nst && ok; ++j) {
      const int a = j % R;
      ok = __all_sync(0xFFFFFFFFu, mbar_wait(smem_addr(&ready[a]), (j / R) & 1, p.status, kStatusTimeoutMma));
      if (!ok) break;
      tc_fence_after();
      if (elect_one()) {
        mma_stage16<MBOX>(tmem + kDcol, tmem + kAcol0 + a * 128, smem_desc(smem_addr(xring + a * kXBytes), 16, 1024, 2),
                          idesc, j ? 1u : 0u);
        mma_commit(smem_addr(&consumed[a]));
      }
      __syncwarp();
    }
    if (ok && do_lora) {
      ok = __all_sync(0xFFFFFFFFu, mbar_wait(smem_addr(lfull), 0, p.status, kStatusTimeoutMma));
      if (ok) {
        tc_fence_after();
        const uint32_t sw = swizzle_mode_for(p.lora_box_bytes);
        const uint32_t sbo = 8 * p.lora_box_bytes;
        const uint32_t la = smem_addr(lora_a), lu = smem_addr(lora_u);
        if (elect_one()) {
          for (int kk = 0; kk < p.r / 16; ++kk) {
            const int off = kk * 32;
            const int box = off / p.lora_box_bytes, in = off % p.lora_box_bytes;
            const uint64_t ad = smem_desc(la + box * kRows * p.lora_box_bytes + in, 16, sbo, sw);
            const uint64_t bd = smem_desc(lu + box * MBOX * p.lora_box_bytes + in, 16, sbo, sw);
            mma_f16_ss(tmem + kLcol, ad, bd, idesc, kk ? 1u : 0u);
          }
        }
        __syncwarp();
      }
    }
    if (elect_one()) mma_commit(smem_addr(dfull));  // also the completion point of every MMA issued above
    __syncwarp();
  } else {
    // ------------------------------------------------------------------ dequant + epilogue
    const int dw = warp - kFirstDeqWarp;  // 0..DW-1
    const int quarter = warp & 3;         // TMEM lane quarter this warp may access
    const int part_k = dw >> 2;           // which share of the stage's K (and of the tile's tokens)
    const int row = quarter * 32 + lane;  // weight row within the tile
    const uint32_t lane_base = static_cast<uint32_t>(quarter * 32) << 16;
    for (int j = 0; j < nst && ok; ++j) {
      const int s = j % SW, a = j % R;
      // every lane waits; the warp leaves together if any lane ran out of time
      ok = __all_sync(0xFFFFFFFFu, mbar_wait(smem_addr(&wfull[s]), (j / SW) & 1, p.status, kStatusTimeoutDequant) &&
                                       mbar_wait(smem_addr(&consumed[a]), ((j / R) & 1) ^ 1, p.status,
                                                 kStatusTimeoutDequant));
      if (!ok) break;
      const uint8_t* st = wring + s * kWStageBytes;
      const uint8_t* crow = st + row * 128;
      const uint32_t* srow = reinterpret_cast<const uint32_t*>(st + kCodeBytes + row * 16);
      const uint32_t taddr = tmem + lane_base + kAcol0 + a * 128;
      // this thread's scale bytes: two per chunk
      const uint2 sc = kChunks == 4 ? *reinterpret_cast<const uint2*>(srow + part_k * 2)
                                    : make_uint2(srow[part_k], 0x08080808u);
      // scale bytes below 8 (zero or subnormal E4M3) take the general decode (warp-uniform branch)
      if (__any_sync(0xFFFFFFFFu, has_small_scale(sc)))
        dequant_chunks<true, kChunks>(crow, row, part_k * kChunks, sc, taddr);
      else
        dequant_chunks<false, kChunks>(crow, row, part_k * kChunks, sc, taddr);
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(smem_addr(&ready[a]));
        mbar_arrive(smem_addr(&wempty[s]));
      }
    }
    // ---------------------------------------------------------------- epilogue
    ok = __all_sync(0xFFFFFFFFu, ok && mbar_wait(smem_addr(dfull), 0, p.status, kStatusTimeoutEpilogue));
    tc_fence_after();
    if (ok && p.splits == 1) {
      const float g = *p.w_g;
      const int64_t n = n0 + row;
      const int t0 = part_k * kEpiTok;
#pragma unroll
      for (int c = 0; c < kEpiTok; c += 16) {
        float v[16];
        epilogue16(tmem + lane_base, t0 + c, do_lora, g, p.s, v);
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const int64_t m = m0 + t0 + c + i;
          if (m < p.M) p.y[m * p.N + n] = static_cast<uint16_t>(f32_to_bf16_bits(v[i]));
        }
      }
    }
  }
  if (p.splits > 1) {
    // ---------------------------------------------------------------- split-K reduction
    const uint32_t lane_base = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const float g = *p.w_g;
    splitk_push_reduce<MBOX, DW>(reinterpret_cast<float*>(xring), p, ok, warp, lane, m0, n0,
                                 [&](int col, float(&v)[16]) { epilogue16(tmem + lane_base, col, do_lora, g, p.s, v); });
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// ---- 256-token tiles ---------------------------------------------------------------------------
//
// w4a16_tc256_kernel: one CTA = 128 weight rows x one K range x 256 tokens, for calls with more
// than 128 tokens and a LoRA rank of at most 64. The fp32 accumulator D (128 x 256) takes TMEM
// columns 0..255 and two A buffers (one 256-K stage each) the other 256, so there is no room for a
// LoRA accumulator of its own: the LoRA branch is folded into D. The LoRA-down kernel writes c U as
// two bf16 matrices hi = bf16(c U) and lo = bf16(c U - hi) with c = s / (2^32 g) (c = s when
// g = 0); after its K loop the tile adds B_lora hi^T + B_lora lo^T to D, and the epilogue's scale
// 2^32 g (1 when g = 0) turns D into x deq(W)^T + s U B^T, the LoRA term to ~2^-17 relative of
// c U (the hi + lo sum). Each weight tile is dequantized once for all 256 tokens and every MMA is
// 128 x 256 x 16. A stage's activations (256 K x 256 tokens, 128 KB) stream in 64-K slots of 32 KB
// (one 128-byte swizzled box of 256 rows), five slots in flight; after the K loop the slots hold
// the LoRA tiles (B_lora, hi, lo), and with split K the partials.
constexpr int kQ = 64;              // K per activation slot
constexpr int kQBytes = 256 * 128;  // one slot: 64 bf16 K x 256 tokens
constexpr int kQPerStage = 4;       // slots per 256-K stage
constexpr int kQSlots = 5;          // slots in flight
constexpr int kMaxFoldRank = 64;    // the B_lora, hi and lo tiles are one 128-byte box each
static_assert(kKStage == kQPerStage * kQ, "a stage is four activation slots");
static_assert((256 + kMaxSplits - 1) * kRows * 4 <= kQSlots * kQBytes + 2 * kWStageBytes,
              "split-K partials fit the activation slots and two weight stages");

__host__ __device__ constexpr size_t smem256_fixed() { return 1024 + static_cast<size_t>(kQSlots) * kQBytes + 512; }

template <int DW>
__global__ void __maxnreg__(88)
    w4a16_tc256_kernel(const __grid_constant__ CUtensorMap map_codes, const __grid_constant__ CUtensorMap map_scales,
                       const __grid_constant__ CUtensorMap map_x, const __grid_constant__ CUtensorMap map_blora,
                       const __grid_constant__ CUtensorMap map_uhi, const __grid_constant__ CUtensorMap map_ulo,
                       const TcParams p) {
  constexpr int MBOX = 256;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int SW = p.w_stages;
  constexpr int kWarpsPerQuarter = DW / 4;       // dequant warps sharing one TMEM lane quarter
  constexpr int kChunks = 8 / kWarpsPerQuarter;  // 16-byte code chunks per thread and stage
  constexpr uint32_t kAcol0 = 256;               // A buffer a: TMEM columns 256 + 128 a
  constexpr int kEpiTok = MBOX / kWarpsPerQuarter;

  // layout: activation slots (then the LoRA tiles, then split-K partials) | weight ring | barriers
  uint8_t* xring = smem;
  uint8_t* wring = xring + kQSlots * kQBytes;
  uint64_t* bars = reinterpret_cast<uint64_t*>(wring + SW * kWStageBytes);
  uint64_t* wfull = bars;             // [SW] weight stage landed
  uint64_t* wempty = wfull + SW;      // [SW] weight stage dequantized (DW arrivals)
  uint64_t* xfull = wempty + SW;      // [kQSlots] activation slot landed
  uint64_t* xempty = xfull + kQSlots; // [kQSlots] its MMAs have completed (commit)
  uint64_t* aready = xempty + kQSlots;  // [2] A buffer written (DW arrivals)
  uint64_t* afree = aready + 2;       // [2] the stage's MMAs have completed (commit)
  uint64_t* lfull = afree + 2;        // LoRA tiles landed
  uint64_t* dfull = lfull + 1;        // every MMA has completed
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(dfull + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int tile_n = blockIdx.x, split = blockIdx.y, tile_m = blockIdx.z;
  const int n0 = tile_n * kRows;
  const int m0 = tile_m * MBOX;
  const int st0 = split * p.stages_per_split;
  const int nst = min(p.stages_per_split, static_cast<int>(p.K / kKStage) - st0);
  const int nq = kQPerStage * nst;  // activation slot loads of the K loop
  const bool do_lora = p.r > 0 && split == 0;

  if (threadIdx.x == 0) {
    for (int i = 0; i < SW; ++i) {
      mbar_init(smem_addr(&wfull[i]), 1);
      mbar_init(smem_addr(&wempty[i]), DW);
    }
    for (int i = 0; i < kQSlots; ++i) {
      mbar_init(smem_addr(&xfull[i]), 1);
      mbar_init(smem_addr(&xempty[i]), 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(smem_addr(&aready[i]), DW);
      mbar_init(smem_addr(&afree[i]), 1);
    }
    mbar_init(smem_addr(lfull), 1);
    mbar_init(smem_addr(dfull), 1);
    fence_barrier_init();
  }
  // stage order: each output tile starts its K range at a different stage (see w4a16_tc_kernel)
  auto kstage = [&](int j) { return st0 + (j + tile_n) % nst; };
  auto load_x = [&](int i) {  // activation slot load i (slot i % kQSlots): stage i / 4, K quarter i % 4
    const int sl = i % kQSlots;
    const uint32_t bar = smem_addr(&xfull[sl]);
    mbar_arrive_expect_tx(bar, kQBytes);
    tma_load_2d(smem_addr(xring + sl * kQBytes), &map_x, kstage(i / kQPerStage) * kKStage + (i % kQPerStage) * kQ, m0,
                bar);
  };
  // the first weight stages and activation slots are requested before the block's set-up completes
  const int w_pre = min(SW, nst), x_pre = min(kQSlots, nq);
  if (threadIdx.x == 0) {
    for (int j = 0; j < w_pre; ++j) {
      uint8_t* st = wring + j * kWStageBytes;
      const uint32_t bar = smem_addr(&wfull[j]);
      mbar_arrive_expect_tx(bar, kWStageBytes);
      tma_load_2d(smem_addr(st), &map_codes, kstage(j) * (kKStage / 2), n0, bar);
      tma_load_2d(smem_addr(st + kCodeBytes), &map_scales, kstage(j) * (kKStage / 16), n0, bar);
    }
    for (int i = 0; i < x_pre; ++i) load_x(i);
  }
  if (warp == 1) tmem_alloc(smem_addr(tmem_slot), 512);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  bool ok = true;
  if (warp == 0) {
    // ------------------------------------------------------------------ weight producer
    if (lane == 0) {
      int issued = w_pre;
      for (int j = w_pre; j < nst && ok; ++j) {
        const int s = j % SW;
        if (!mbar_wait(smem_addr(&wempty[s]), ((j / SW) & 1) ^ 1, p.status, kStatusTimeoutProducer)) {
          ok = false;
          break;
        }
        uint8_t* st = wring + s * kWStageBytes;
        const uint32_t bar = smem_addr(&wfull[s]);
        mbar_arrive_expect_tx(bar, kWStageBytes);
        const int kst = kstage(j);
        tma_load_2d(smem_addr(st), &map_codes, kst * (kKStage / 2), n0, bar);
        tma_load_2d(smem_addr(st + kCodeBytes), &map_scales, kst * (kKStage / 16), n0, bar);
        issued = j + 1;
      }
      for (int j = max(0, issued - SW); j < issued; ++j)
        mbar_wait(smem_addr(&wfull[j % SW]), (j / SW) & 1, p.status, kStatusTimeoutDrain);
    }
  } else if (warp == 2) {
    // ------------------------------------------------------------------ activation + LoRA producer
    if (lane == 0) {
      int issued = x_pre;
      for (int i = x_pre; i < nq && ok; ++i) {
        const int sl = i % kQSlots;
        if (!mbar_wait(smem_addr(&xempty[sl]), ((i / kQSlots) & 1) ^ 1, p.status, kStatusTimeoutProducer)) {
          ok = false;
          break;
        }
        load_x(i);
        issued = i + 1;
      }
      if (do_lora && ok) {
        // slots 0..2 take the LoRA tiles once the K loop's MMAs have read them
        for (int sl = 0; sl < 3 && ok; ++sl) {
          const int uses = sl < nq ? (nq - sl + kQSlots - 1) / kQSlots : 0;
          if (uses > 0)
            ok = mbar_wait(smem_addr(&xempty[sl]), (uses - 1) & 1, p.status, kStatusTimeoutProducer);
        }
        if (ok) {
          griddep_wait();  // the LoRA-down kernel has completed and its hi and lo are visible
          const int lb = p.lora_box_bytes;
          mbar_arrive_expect_tx(smem_addr(lfull), static_cast<uint32_t>(kRows * lb + 2 * MBOX * lb));
          tma_load_2d(smem_addr(xring), &map_blora, 0, n0, smem_addr(lfull));
          tma_load_2d(smem_addr(xring + kQBytes), &map_uhi, 0, m0, smem_addr(lfull));
          tma_load_2d(smem_addr(xring + 2 * kQBytes), &map_ulo, 0, m0, smem_addr(lfull));
          mbar_wait(smem_addr(lfull), 0, p.status, kStatusTimeoutDrain);
        }
      }
      // drain: the last activation copies have landed before the CTA exits
      for (int i = max(0, issued - kQSlots); i < issued; ++i)
        mbar_wait(smem_addr(&xfull[i % kQSlots]), (i / kQSlots) & 1, p.status, kStatusTimeoutDrain);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------------ MMA issuer
    // The whole warp walks the stages and waits; one elected lane issues the MMAs and commits.
    const uint32_t idesc = idesc_bf16_f32(kRows, MBOX);
    for (int j = 0; j < nst && ok; ++j) {
      const int a = j & 1;
      ok = __all_sync(0xFFFFFFFFu, mbar_wait(smem_addr(&aready[a]), (j >> 1) & 1, p.status, kStatusTimeoutMma));
      if (!ok) break;
      tc_fence_after();
      for (int q = 0; q < kQPerStage && ok; ++q) {
        const int i = j * kQPerStage + q, sl = i % kQSlots;
        ok = __all_sync(0xFFFFFFFFu, mbar_wait(smem_addr(&xfull[sl]), (i / kQSlots) & 1, p.status, kStatusTimeoutMma));
        if (!ok) break;
        tc_fence_after();
        if (elect_one()) {
          const uint64_t bd = smem_desc(smem_addr(xring + sl * kQBytes), 16, 1024, 2);
          const uint32_t at = tmem + kAcol0 + a * 128 + q * 32;
#pragma unroll
          for (int kk = 0; kk < kQ / 16; ++kk)
            mma_f16_ts(tmem, at + 8 * kk, bd + 2 * kk, idesc, (j | q | kk) ? 1u : 0u);
          mma_commit(smem_addr(&xempty[sl]));
        }
        __syncwarp();
      }
      if (!ok) break;
      if (elect_one()) mma_commit(smem_addr(&afree[a]));
      __syncwarp();
    }
    if (ok && do_lora) {
      ok = __all_sync(0xFFFFFFFFu, mbar_wait(smem_addr(lfull), 0, p.status, kStatusTimeoutMma));
      if (ok) {
        tc_fence_after();
        const int lb = p.lora_box_bytes;
        const uint32_t sw = swizzle_mode_for(lb), sbo = 8 * lb;
        if (elect_one()) {
          for (int part = 0; part < 2; ++part)
            for (int kk = 0; kk < p.r / 16; ++kk) {
              const uint64_t ad = smem_desc(smem_addr(xring) + kk * 32, 16, sbo, sw);
              const uint64_t bd = smem_desc(smem_addr(xring + (1 + part) * kQBytes) + kk * 32, 16, sbo, sw);
              mma_f16_ss(tmem, ad, bd, idesc, 1u);
            }
        }
        __syncwarp();
      }
    }
    if (elect_one()) mma_commit(smem_addr(dfull));  // also the completion point of every MMA issued above
    __syncwarp();
  } else {
    // ------------------------------------------------------------------ dequant + epilogue
    const int dw = warp - kFirstDeqWarp;
    const int quarter = warp & 3;
    const int part_k = dw >> 2;
    const int row = quarter * 32 + lane;
    const uint32_t lane_base = static_cast<uint32_t>(quarter * 32) << 16;
    for (int j = 0; j < nst && ok; ++j) {
      const int s = j % SW, a = j & 1;
      ok = __all_sync(0xFFFFFFFFu, mbar_wait(smem_addr(&wfull[s]), (j / SW) & 1, p.status, kStatusTimeoutDequant) &&
                                       mbar_wait(smem_addr(&afree[a]), ((j >> 1) & 1) ^ 1, p.status,
                                                 kStatusTimeoutDequant));
      if (!ok) break;
      const uint8_t* st = wring + s * kWStageBytes;
      const uint8_t* crow = st + row * 128;
      const uint32_t* srow = reinterpret_cast<const uint32_t*>(st + kCodeBytes + row * 16);
      const uint32_t taddr = tmem + lane_base + kAcol0 + a * 128;
      const uint2 sc = kChunks == 4 ? *reinterpret_cast<const uint2*>(srow + part_k * 2)
                                    : make_uint2(srow[part_k], 0x08080808u);
      if (__any_sync(0xFFFFFFFFu, has_small_scale(sc)))
        dequant_chunks<true, kChunks>(crow, row, part_k * kChunks, sc, taddr);
      else
        dequant_chunks<false, kChunks>(crow, row, part_k * kChunks, sc, taddr);
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(smem_addr(&aready[a]));
        mbar_arrive(smem_addr(&wempty[s]));
      }
    }
    // ---------------------------------------------------------------- epilogue
    ok = __all_sync(0xFFFFFFFFu, ok && mbar_wait(smem_addr(dfull), 0, p.status, kStatusTimeoutEpilogue));
    tc_fence_after();
    if (ok && p.splits == 1) {
      const float g = *p.w_g;
      const float out = p.r > 0 && g == 0.f ? 1.f : 0x1p32f * g;
      const int64_t n = n0 + row;
      const int t0 = part_k * kEpiTok;
#pragma unroll 1
      for (int c = 0; c < kEpiTok; c += 16) {
        uint32_t d[16];
        tmem_ld16(tmem + lane_base + t0 + c, d);
        tmem_ld_wait();
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const int64_t m = m0 + t0 + c + i;
          if (m < p.M) p.y[m * p.N + n] = static_cast<uint16_t>(f32_to_bf16_bits(__uint_as_float(d[i]) * out));
        }
      }
    }
  }
  if (p.splits > 1) {
    // ---------------------------------------------------------------- split-K reduction
    // (the partials take the activation slots, and the weight ring behind them where needed)
    const uint32_t lane_base = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const float g = *p.w_g;
    const float out = p.r > 0 && g == 0.f ? 1.f : 0x1p32f * g;
    splitk_push_reduce<MBOX, DW>(reinterpret_cast<float*>(xring), p, ok, warp, lane, m0, n0, [&](int col, float(&v)[16]) {
      uint32_t d[16];
      tmem_ld16(tmem + lane_base + col, d);
      tmem_ld_wait();
#pragma unroll
      for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(d[i]) * out;
    });
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

__device__ __forceinline__ void mma16816(float c[4], const uint32_t a[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ void cp_async16(void* smem_dst, const void* gmem_src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(static_cast<uint32_t>(__cvta_generic_to_shared(smem_dst))),
               "l"(gmem_src)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }

// LoRA down-projection U = bf16(x A^T), [M][r]. A cluster of CTAs (blockIdx.x, 16 or 8) covers 64
// rows of x (blockIdx.y); CTA q takes a contiguous range of the 64-K chunks. A ring of three
// chunk buffers is filled with cp.async (x: 64 x 64, A: RP x 64 bf16) while mma.sync m16n8k16
// runs on the oldest (warp w: rows 16w..16w+15, RP ranks per pass over x), accumulating in
// registers. The fp32 partial [64][RP] goes to shared memory; after a cluster barrier, CTA q sums
// its share of the rows over all CTAs' partials in rank order (distributed shared memory) and
// writes U. Rows past M read as zero and are not written. Each rank's sum runs through the same
// chunks and instructions whatever RP is, so U does not depend on it. With a LoraDownScale (the
// W4A4 path) the kernel writes hi and lo of c U instead.
template <int RP>
__global__ void __launch_bounds__(128) w4a16_lora_down_kernel(const uint16_t* __restrict__ x, int64_t M, int64_t K,
                                                              const uint16_t* __restrict__ A, int r,
                                                              uint16_t* __restrict__ U, const LoraDownScale ls) {
  // Earlier kernels on the stream (which may have written x, or g_x) have completed once
  // griddep_wait returns; only then may the main kernel start: it reads x and the weights
  // without waiting, and waits (griddepcontrol.wait) for this kernel before reading U.
  griddep_wait();
  griddep_launch_dependents();
  float cu = 1.f;  // c of the W4A4 form
  if (ls.folded()) {
    const float alpha = ls.gx() * *ls.w_g;
    cu = alpha == 0.f ? ls.s : ls.s / alpha;
    if (blockIdx.x == 0 && blockIdx.y == 0 && threadIdx.x == 0 && !(fabsf(cu) <= 0x1p100f))
      atomicOr(ls.status, kStatusRange);
  }
  extern __shared__ __align__(16) uint8_t down_smem[];
  constexpr int kDownStageElems = DownShape<RP>::kStageElems;
  uint16_t* ring = reinterpret_cast<uint16_t*>(down_smem);  // [kDownStages][64 + RP][kDownK + kDownPad]
  float(*part)[RP] = reinterpret_cast<float(*)[RP]>(down_smem + kDownStages * kDownStageElems * 2);
  constexpr int kRow = kDownK + kDownPad;
  const int64_t m0 = static_cast<int64_t>(blockIdx.y) * kDownM;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int C = static_cast<int>(gridDim.x);
  const int q = static_cast<int>(cluster_ctarank());
  const int nchunks = static_cast<int>(K / kDownK);
  const int cb = q * nchunks / C, n = (q + 1) * nchunks / C - cb;
  for (int j0 = 0; j0 < r; j0 += RP) {
    // one chunk: rows 0..63 of the buffer hold x, rows 64..63+RP hold A (ranks j0..j0+RP-1)
    auto load = [&](int i, int buf) {
      uint16_t* b = ring + buf * kDownStageElems;
      const int64_t k0 = static_cast<int64_t>(cb + i) * kDownK;
#pragma unroll
      for (int u = 0; u < ((kDownM + RP) * kDownK / 8) / 128; ++u) {  // 64 + RP rows x 8 vectors of 8 bf16
        const int idx = tid + u * 128, row = idx >> 3, vec = idx & 7;
        uint16_t* dst = b + row * kRow + vec * 8;
        const uint16_t* src = nullptr;
        if (row < kDownM) {
          if (m0 + row < M) src = x + (m0 + row) * K + k0 + vec * 8;
        } else if (j0 + row - kDownM < r) {
          src = A + static_cast<int64_t>(j0 + row - kDownM) * K + k0 + vec * 8;
        }
        if (src) cp_async16(dst, src);
        else *reinterpret_cast<uint4*>(dst) = make_uint4(0, 0, 0, 0);
      }
    };
    float c[RP / 8][4] = {};
#pragma unroll
    for (int st = 0; st < kDownStages - 1; ++st) {
      if (st < n) load(st, st);
      cp_async_commit();
    }
    for (int i = 0; i < n; ++i) {
      cp_async_wait<kDownStages - 2>();
      __syncthreads();  // chunk i is visible to all threads; buffer (i - 1) % kDownStages is free
      if (i + kDownStages - 1 < n) load(i + kDownStages - 1, (i + kDownStages - 1) % kDownStages);
      cp_async_commit();
      const uint16_t* xs = ring + (i % kDownStages) * kDownStageElems;
      const uint16_t* as = xs + kDownM * kRow;
#pragma unroll
      for (int ks = 0; ks < kDownK / 16; ++ks) {
        uint32_t a[4];
        ldsm_x4(static_cast<uint32_t>(__cvta_generic_to_shared(xs + (warp * 16 + (lane & 15)) * kRow + ks * 16 + (lane >> 4) * 8)),
                a[0], a[1], a[2], a[3]);
#pragma unroll
        for (int jp = 0; jp < RP / 16; ++jp) {
          const int g8 = lane >> 3;
          uint32_t b0, b1, b2, b3;
          ldsm_x4(static_cast<uint32_t>(__cvta_generic_to_shared(as + (jp * 16 + (g8 >> 1) * 8 + (lane & 7)) * kRow + ks * 16 + (g8 & 1) * 8)),
                  b0, b1, b2, b3);
          mma16816(c[2 * jp], a, b0, b1);
          mma16816(c[2 * jp + 1], a, b2, b3);
        }
      }
    }
    cp_async_wait<0>();
    // C fragment: c0,c1 at (row lane/4, cols 2(lane%4), +1); c2,c3 at row + 8
#pragma unroll
    for (int nt = 0; nt < RP / 8; ++nt)
#pragma unroll
      for (int e = 0; e < 4; ++e)
        part[warp * 16 + (lane >> 2) + (e >> 1) * 8][nt * 8 + 2 * (lane & 3) + (e & 1)] = c[nt][e];
    cluster_sync_all();
    // CTA q: rows [q*64/C, (q+1)*64/C), four ranks per thread and step
    const int rb = q * kDownM / C, re = (q + 1) * kDownM / C;
    for (int idx = tid; idx < (re - rb) * (RP / 4); idx += 128) {
      const int row = rb + idx / (RP / 4), j4 = (idx % (RP / 4)) * 4;
      const int64_t m = m0 + row;
      const uint32_t local = static_cast<uint32_t>(__cvta_generic_to_shared(&part[row][j4]));
      float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
      for (int sp = 0; sp < C; ++sp) {
        const float4 v = dsmem_ld_v4(dsmem_map(local, static_cast<uint32_t>(sp)));
        acc.x += v.x; acc.y += v.y; acc.z += v.z; acc.w += v.w;
      }
      if (m < M) {
        const float av[4] = {acc.x, acc.y, acc.z, acc.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          if (j0 + j4 + e >= r) continue;
          const uint32_t u = f32_to_bf16_bits(av[e]);
          const int64_t at = m * r + j0 + j4 + e;
          if (ls.folded()) {
            // c U = hi + lo: hi = bf16(c U), lo = bf16(c U - hi) (c U - hi is exact in fp32). U
            // is bf16(x A^T) when g_x comes from memory (W4A4: the same U as the calls that learn
            // g_x after the LoRA-down), x A^T as accumulated in fp32 when it is given by value
            // (W4A16 on 256-token tiles).
            const float cuv = (ls.g_x ? __uint_as_float(u << 16) : av[e]) * cu;
            const uint32_t hi = f32_to_bf16_bits(cuv);
            U[at] = static_cast<uint16_t>(hi);
            ls.lo[at] = static_cast<uint16_t>(f32_to_bf16_bits(cuv - __uint_as_float(hi << 16)));
          } else {
            U[at] = static_cast<uint16_t>(u);
          }
        }
      }
    }
    cluster_sync_all();  // partials read by every peer before the next pass overwrites them
  }
}

// ---- host ---------------------------------------------------------------------------------

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static std::once_flag once;
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
  });
  return fn;
}

bool make_map(CUtensorMap* m, CUtensorMapDataType dt, const void* base, uint64_t cols, uint64_t rows, int esize,
              uint32_t box_cols, uint32_t box_rows, CUtensorMapSwizzle sw);

CUtensorMapSwizzle swizzle_for(int box_bytes) {
  return box_bytes == 128 ? CU_TENSOR_MAP_SWIZZLE_128B
         : box_bytes == 64 ? CU_TENSOR_MAP_SWIZZLE_64B
                           : CU_TENSOR_MAP_SWIZZLE_32B;
}

constexpr int kDW = 16;  // dequant warps of the tcgen05 kernel (4 per TMEM lane quarter)

struct TcPlan {
  int mbox, tiles_m, tiles_n, w_stages;
  size_t smem_bytes, ws_u, ws_lo, ws_total;  // ws_lo: the lo part of c U (256-token tiles with LoRA)
};

// Tile shape, shared-memory rings and workspace (U only), for `mbox`-token tiles. With
// reserve_down the rings leave room for one LoRA-down CTA on the same SM, so that kernel never
// delays a CTA of this one. The activation ring has ring_depth stages; the weight ring takes the
// rest (at most 8 stages).
TcPlan plan_for(int64_t M, int64_t N, int r, int mbox, bool reserve_down) {
  TcPlan t{};
  t.mbox = mbox;
  t.tiles_m = static_cast<int>((M + t.mbox - 1) / t.mbox);
  t.tiles_n = static_cast<int>(N / kRows);
  const size_t lora = r ? static_cast<size_t>(kRows + t.mbox) * 2 * lora_padded_rank(r) : 0;
  const size_t fixed = 1024 + lora + 512;
  const size_t xring = static_cast<size_t>(ring_depth(t.mbox)) * x_stage_bytes(t.mbox);
  const size_t budget = 227 * 1024 - (reserve_down ? kDownSmem + 1024 : 0);
  t.w_stages = budget > fixed + xring ? static_cast<int>(std::min<size_t>(8, (budget - fixed - xring) / kWStageBytes)) : 0;
  t.smem_bytes = fixed + xring + t.w_stages * kWStageBytes;
  size_t o = 0;
  auto take = [&](size_t b) { size_t at = o; o = align_up(o + b, 256); return at; };
  t.ws_u = take(static_cast<size_t>(M) * std::max(r, 1) * 2);
  t.ws_total = o;
  return t;
}

// 256-token tiles (w4a16_tc256_kernel): four activation slots, the rest of shared memory for the
// weight ring; the workspace holds hi and lo of c U.
TcPlan plan256(int64_t M, int64_t N, int r) {
  TcPlan t{};
  t.mbox = 256;
  t.tiles_m = static_cast<int>((M + 255) / 256);
  t.tiles_n = static_cast<int>(N / kRows);
  const size_t fixed = smem256_fixed();
  const size_t budget = 227 * 1024;
  t.w_stages = static_cast<int>(std::min<size_t>(8, (budget - fixed) / kWStageBytes));
  t.smem_bytes = fixed + t.w_stages * kWStageBytes;
  size_t o = 0;
  auto take = [&](size_t b) { size_t at = o; o = align_up(o + b, 256); return at; };
  t.ws_u = take(static_cast<size_t>(M) * std::max(r, 1) * 2);
  t.ws_lo = r ? take(static_cast<size_t>(M) * r * 2) : 0;
  t.ws_total = o;
  return t;
}

// 256-token tiles for more than 128 tokens at LoRA ranks up to 64 when they fill at least half the
// SMs or K has 64 stages or more (measured on the 32B-shaped layer at 256 tokens: gate 79 -> 66 us
// and down 104 -> 72 us per call, while q and k, 40 and 8 such tiles over 20 stages, are faster on
// twice as many 128-token CTAs); else 128-token tiles when M exceeds one 64-token tile and two
// weight stages still fit beside the 128-token activation ring and the LoRA tiles; otherwise
// 64-token tiles (always the case for r = 128 at M > 64), leaving room for a LoRA-down CTA where
// that still leaves two weight stages.
TcPlan plan(int64_t M, int64_t N, int64_t K, int r) {
  if (M > 128 && r <= kMaxFoldRank) {
    const int64_t tiles256 = (N / kRows) * ((M + 255) / 256);
    if (2 * tiles256 >= kPlanSMs || K / kKStage >= 64) return plan256(M, N, r);
  }
  if (M > 64) {
    const TcPlan t = plan_for(M, N, r, 128, false);
    if (t.w_stages >= 2) return t;
  }
  const TcPlan t = plan_for(M, N, r, 64, r > 0);
  if (t.w_stages >= 2) return t;
  return plan_for(M, N, r, 64, false);
}

void* tc_kernel_ptr(int mbox) {
  return mbox == 256 ? reinterpret_cast<void*>(w4a16_tc256_kernel<kDW>)
         : mbox == 128 ? reinterpret_cast<void*>(w4a16_tc_kernel<128, kDW>)
                       : reinterpret_cast<void*>(w4a16_tc_kernel<64, kDW>);
}

// Clusters of `c` CTAs of the tcgen05 kernel that can be resident at once on this device.
int cluster_capacity(int device, int mbox, size_t smem, int c) {
  static std::mutex mu;
  static std::map<std::tuple<int, int, size_t, int>, int> cache;
  std::lock_guard<std::mutex> lock(mu);
  const auto key = std::make_tuple(device, mbox, smem, c);
  auto it = cache.find(key);
  if (it != cache.end()) return it->second;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(1, c, 1);
  cfg.blockDim = dim3(threads_for(kDW));
  cfg.dynamicSmemBytes = smem;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 1;
  attr[0].val.clusterDim.y = c;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int n = 0;
  const void* fn = tc_kernel_ptr(mbox);
  if (cudaOccupancyMaxActiveClusters(&n, fn, &cfg) != cudaSuccess) {
    cudaGetLastError();
    n = 0;
  }
  cache[key] = n;
  return n;
}

// Split-K factor: the cluster size c (<= 8, <= the number of 256-K stages, the stages dividing
// into exactly c splits) that minimises waves(c) x (stages per CTA + 1 + 4 [c > 1]), where waves(c)
// is the number of rounds of resident clusters that tiles x c CTAs take, the + 1 stands for a CTA's
// fixed cost (set-up, pipeline fill, epilogue) and the + 4 for the split-K reduction through
// distributed shared memory (measured: ~4 stages' time).
int choose_splits_waves(int device, const TcPlan& t, int64_t K) {
  const int tiles = t.tiles_n * t.tiles_m;
  const int kst = static_cast<int>(K / kKStage);
  int best = 1;
  int64_t best_cost = INT64_MAX;
  for (int c = 1; c <= std::min(kMaxSplits, kst); ++c) {
    const int sps = (kst + c - 1) / c;
    if ((kst + sps - 1) / sps != c) continue;
    const int cap = cluster_capacity(device, t.mbox, t.smem_bytes, c);
    if (cap <= 0) continue;
    const int64_t cost = static_cast<int64_t>((tiles + cap - 1) / cap) * (sps + 1 + (c > 1 ? 4 : 0));
    if (cost < best_cost) {
      best_cost = cost;
      best = c;
    }
  }
  return best;
}

bool make_map(CUtensorMap* m, CUtensorMapDataType dt, const void* base, uint64_t cols, uint64_t rows, int esize,
              uint32_t box_cols, uint32_t box_rows, CUtensorMapSwizzle sw) {
  return make_tensor_map_2d(m, dt, base, cols, rows, esize, box_cols, box_rows, sw);
}

template <int RP>
int down_cluster_size_for(int device) {
  static std::mutex mu;
  static std::map<int, int> cache;
  std::lock_guard<std::mutex> lock(mu);
  auto it = cache.find(device);
  if (it != cache.end()) return it->second;
  int c = 8;
  const int smem = DownShape<RP>::kSmem;
  auto* kern = w4a16_lora_down_kernel<RP>;
  const bool attrs =
      cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) == cudaSuccess &&
      cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout,
                           static_cast<int>(cudaSharedmemCarveoutMaxShared)) == cudaSuccess;
  if (attrs && cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) == cudaSuccess) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(kDownCluster, 1, 1);
    cfg.blockDim = dim3(128);
    cfg.dynamicSmemBytes = smem;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = kDownCluster;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, reinterpret_cast<const void*>(kern), &cfg) == cudaSuccess && n > 0)
      c = kDownCluster;
  }
  cudaGetLastError();
  if (!attrs) c = 0;  // the kernel cannot be launched with its shared memory
  cache[device] = c;
  return c;
}

// Cluster size of the LoRA-down kernel (ranks-per-pass instance RP) on this device: 16
// (non-portable) where a 16-CTA cluster of it can be resident, else 8; 0 when it cannot be
// launched. Also sets the kernel's attributes (once per device).
int down_cluster_size(int device, int rp) {
  return rp == 64 ? down_cluster_size_for<64>(device) : down_cluster_size_for<32>(device);
}

}  // namespace

// 2-D tensor map over a row-major [rows][cols] array of `esize`-byte elements; zero fill outside.
bool make_tensor_map_2d(CUtensorMap* m, CUtensorMapDataType dt, const void* base, uint64_t cols, uint64_t rows,
                        int esize, uint32_t box_cols, uint32_t box_rows, CUtensorMapSwizzle sw) {
  auto fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[2] = {cols, rows};
  const cuuint64_t strides[1] = {cols * static_cast<uint64_t>(esize)};
  const cuuint32_t box[2] = {box_cols, box_rows};
  const cuuint32_t estr[2] = {1, 1};
  return fn(m, dt, 2, const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, sw,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// LoRA down-projection: one cluster per 64 rows of x, K (a multiple of 64) split over the cluster.
// Ranks per pass over x: 64 when r > 32 and M exceeds one decode tile (x is then read once for
// r = 64); 32 otherwise, the instance whose shared memory leaves room beside a decode CTA of the
// main kernel.
nvfp4rl_status launch_lora_down(const uint16_t* x, int64_t M, int64_t K, const uint16_t* A, int r, uint16_t* U,
                                const DeviceInfo& dev, cudaStream_t st, const LoraDownScale& scale) {
  if (lora_down_tc_supported(M, K, r)) return launch_lora_down_tc(x, M, K, A, r, U, dev, st, scale);
  const int nchunks = static_cast<int>(K / kDownK);
  const int rp = r > 32 && M > 64 ? 64 : 32;
  const int dc = down_cluster_size(dev.device, rp);
  if (dc == 0) return NVFP4RL_ERR_CUDA;
  // split K over a cluster only as far as the row blocks alone leave SMs idle (about three CTAs
  // per SM in all)
  const int64_t row_blocks = (M + kDownM - 1) / kDownM;
  const int64_t want = std::max<int64_t>(1, (3 * static_cast<int64_t>(std::min(dev.sm_count, kPlanSMs)) + row_blocks - 1) /
                                                row_blocks);
  const int cd = static_cast<int>(std::min<int64_t>({static_cast<int64_t>(dc), static_cast<int64_t>(nchunks), want}));
  cudaLaunchConfig_t dcfg = {};
  dcfg.gridDim = dim3(cd, static_cast<unsigned>((M + kDownM - 1) / kDownM), 1);
  dcfg.blockDim = dim3(128);
  dcfg.dynamicSmemBytes = rp == 64 ? DownShape<64>::kSmem : DownShape<32>::kSmem;
  dcfg.stream = st;
  cudaLaunchAttribute dattr[2];
  dattr[0].id = cudaLaunchAttributeClusterDimension;
  dattr[0].val.clusterDim.x = cd;
  dattr[0].val.clusterDim.y = 1;
  dattr[0].val.clusterDim.z = 1;
  dattr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;  // overlaps the previous kernel's tail
  dattr[1].val.programmaticStreamSerializationAllowed = 1;
  dcfg.attrs = dattr;
  dcfg.numAttrs = 2;
  const cudaError_t e = rp == 64 ? cudaLaunchKernelEx(&dcfg, w4a16_lora_down_kernel<64>, x, M, K, A, r, U, scale)
                                 : cudaLaunchKernelEx(&dcfg, w4a16_lora_down_kernel<32>, x, M, K, A, r, U, scale);
  if (e != cudaSuccess) return NVFP4RL_ERR_CUDA;
  return launch_status();
}

// True when the tcgen05 W4A16 path takes this shape.
bool w4a16_tc_supported(int64_t M, int64_t N, int64_t K, int r) {
  if (!(M > 0 && N % kRows == 0 && K % kKStage == 0 && (r == 0 || (r % 16 == 0 && r <= kMaxLoraRank)))) return false;
  const TcPlan t = plan(M, N, K, r);
  return t.w_stages >= 2;
}

size_t w4a16_tc_workspace_bytes(int64_t M, int64_t N, int64_t K, int r, int) {
  return plan(M, N, K, r).ws_total;
}

// 256-token tiles: the LoRA-down writes hi and lo of c U, c = s / (2^32 g), and the main kernel
// folds them into its accumulator.
nvfp4rl_status launch_w4a16_tc256(const LinearArgs& a, const TcPlan& t, void* ws, const DeviceInfo& dev,
                                  cudaStream_t st) {
  uint16_t* U = reinterpret_cast<uint16_t*>(static_cast<char*>(ws) + t.ws_u);
  uint16_t* Ulo = a.r ? reinterpret_cast<uint16_t*>(static_cast<char*>(ws) + t.ws_lo) : nullptr;
  if (cudaFuncSetAttribute(w4a16_tc256_kernel<kDW>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(t.smem_bytes)) != cudaSuccess)
    return NVFP4RL_ERR_CUDA;
  const int splits = choose_splits_waves(dev.device, t, a.K);
  const int kst = static_cast<int>(a.K / kKStage);
  if (a.r) {
    LoraDownScale ls;
    ls.g_x_value = 0x1p32f;  // the dequantized weights carry 2^-32 of their value
    ls.w_g = a.w_g;
    ls.s = a.s;
    ls.lo = Ulo;
    ls.status = dev.status;
    const nvfp4rl_status sd = launch_lora_down(a.x, a.M, a.K, a.A, a.r, U, dev, st, ls);
    if (sd != NVFP4RL_OK) return sd;
  }
  CUtensorMap mc, ms, mx, mb, mh, ml;
  const int lbox = a.r ? lora_box_bytes_for(a.r) : 128;
  if (!make_map(&mc, CU_TENSOR_MAP_DATA_TYPE_UINT8, a.w_codes, a.K / 2, a.N, 1, 128, kRows, CU_TENSOR_MAP_SWIZZLE_128B) ||
      !make_map(&ms, CU_TENSOR_MAP_DATA_TYPE_UINT8, a.w_scales, a.K / 16, a.N, 1, 16, kRows, CU_TENSOR_MAP_SWIZZLE_NONE) ||
      !make_map(&mx, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, a.x, a.K, a.M, 2, kQ, 256, CU_TENSOR_MAP_SWIZZLE_128B))
    return NVFP4RL_ERR_CUDA;
  if (a.r) {
    if (!make_map(&mb, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, a.B, a.r, a.N, 2, lbox / 2, kRows, swizzle_for(lbox)) ||
        !make_map(&mh, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, U, a.r, a.M, 2, lbox / 2, 256, swizzle_for(lbox)) ||
        !make_map(&ml, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, Ulo, a.r, a.M, 2, lbox / 2, 256, swizzle_for(lbox)))
      return NVFP4RL_ERR_CUDA;
  } else {
    mb = mh = ml = mc;
  }
  TcParams p{};
  p.M = a.M;
  p.N = a.N;
  p.K = a.K;
  p.stages_per_split = (kst + splits - 1) / splits;
  p.splits = splits;
  p.r = a.r;
  p.lora_box_bytes = lbox;
  p.s = a.s;
  p.w_g = a.w_g;
  p.y = a.y;
  p.status = dev.status;
  p.w_stages = t.w_stages;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(t.tiles_n, splits, t.tiles_m);
  cfg.blockDim = dim3(threads_for(kDW));
  cfg.dynamicSmemBytes = t.smem_bytes;
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 1;
  attr[0].val.clusterDim.y = splits;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;  // as in launch_w4a16_tc
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = a.r ? 2 : 1;
  if (cudaLaunchKernelEx(&cfg, w4a16_tc256_kernel<kDW>, mc, ms, mx, mb, mh, ml, p) != cudaSuccess)
    return NVFP4RL_ERR_CUDA;
  return launch_status();
}

nvfp4rl_status launch_w4a16_tc(const LinearArgs& a, void* ws, size_t ws_bytes, const DeviceInfo& dev,
                               cudaStream_t st) {
  const TcPlan t = plan(a.M, a.N, a.K, a.r);
  if (ws_bytes < t.ws_total) return NVFP4RL_ERR_WORKSPACE;
  if (t.w_stages < 2) return NVFP4RL_ERR_UNSUPPORTED_SHAPE;
  if (t.mbox == 256) return launch_w4a16_tc256(a, t, ws, dev, st);
  uint16_t* U = reinterpret_cast<uint16_t*>(static_cast<char*>(ws) + t.ws_u);
  const int smem = static_cast<int>(t.smem_bytes);
  cudaError_t e =
      t.mbox == 64 ? cudaFuncSetAttribute(w4a16_tc_kernel<64, kDW>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem)
                   : cudaFuncSetAttribute(w4a16_tc_kernel<128, kDW>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return NVFP4RL_ERR_CUDA;
  const int splits = choose_splits_waves(dev.device, t, a.K);
  const int kst = static_cast<int>(a.K / kKStage);

  if (a.r) {
    const nvfp4rl_status sd = launch_lora_down(a.x, a.M, a.K, a.A, a.r, U, dev, st);
    if (sd != NVFP4RL_OK) return sd;
  }

  CUtensorMap mc, ms, mx, mb, mu;
  const int lbox = a.r ? lora_box_bytes_for(a.r) : 128;
  if (!make_map(&mc, CU_TENSOR_MAP_DATA_TYPE_UINT8, a.w_codes, a.K / 2, a.N, 1, 128, kRows, CU_TENSOR_MAP_SWIZZLE_128B) ||
      !make_map(&ms, CU_TENSOR_MAP_DATA_TYPE_UINT8, a.w_scales, a.K / 16, a.N, 1, 16, kRows, CU_TENSOR_MAP_SWIZZLE_NONE) ||
      !make_map(&mx, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, a.x, a.K, a.M, 2, 64, t.mbox, CU_TENSOR_MAP_SWIZZLE_128B))
    return NVFP4RL_ERR_CUDA;
  if (a.r) {
    if (!make_map(&mb, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, a.B, a.r, a.N, 2, lbox / 2, kRows, swizzle_for(lbox)) ||
        !make_map(&mu, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, U, a.r, a.M, 2, lbox / 2, t.mbox, swizzle_for(lbox)))
      return NVFP4RL_ERR_CUDA;
  } else {
    mb = mc;
    mu = mc;
  }
  TcParams p{};
  p.M = a.M;
  p.N = a.N;
  p.K = a.K;
  p.stages_per_split = (kst + splits - 1) / splits;
  p.splits = splits;
  p.r = a.r;
  p.lora_box_bytes = lbox;
  p.s = a.s;
  p.w_g = a.w_g;
  p.y = a.y;
  p.status = dev.status;
  p.w_stages = t.w_stages;
  // Split K runs as clusters of `splits` CTAs along y. With LoRA, the launch is a programmatic
  // dependent of the LoRA-down kernel: it runs alongside it and waits for it only before loading
  // U. Everything else it reads (x, weights, B_lora, g) was complete before the LoRA-down kernel
  // started. Without LoRA the launch is an ordinary one (nothing would order it after the
  // caller's previous kernel).
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(t.tiles_n, splits, t.tiles_m);
  cfg.blockDim = dim3(threads_for(kDW));
  cfg.dynamicSmemBytes = t.smem_bytes;
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 1;
  attr[0].val.clusterDim.y = splits;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = a.r ? 2 : 1;
  e = t.mbox == 64 ? cudaLaunchKernelEx(&cfg, w4a16_tc_kernel<64, kDW>, mc, ms, mx, mb, mu, p)
                   : cudaLaunchKernelEx(&cfg, w4a16_tc_kernel<128, kDW>, mc, ms, mx, mb, mu, p);
  if (e != cudaSuccess) return NVFP4RL_ERR_CUDA;
  return launch_status();
}

}  // namespace nvfp4rl
