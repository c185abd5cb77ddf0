// W4A16 NVFP4 LoRA linear on the 5th-generation tensor cores (tcgen05), sm_103a.
//
// QeRL explainer, section "NVFP4量子化とLoRA": the rollout runs frozen NVFP4 base weights
// plus trainable LoRA factors, Y = x deq(W)^T + s (x A^T) B^T. In decode the layer is bound
// by the HBM stream of 4-bit weights (0.5625 bytes per weight with the block scales).
//
// Structure (one CTA = 128 weight rows x one K range x up to 128 tokens):
//   warp 0      TMA producer: per 256-K stage, the 128 x 128-byte code tile (128-byte
//               swizzle), the 128 x 16-byte scale tile and the activation tile (4 boxes of
//               64 bf16 x tokens, 128-byte swizzle) into a ring of shared-memory stages.
//   warp 1      allocates TMEM; one thread issues tcgen05.mma kind::f16 with A (the
//               dequantized weights) in TMEM and B (activations) in shared memory, then the
//               LoRA up-projection (B_lora tile x U^T) into a second accumulator.
//   warps 2-9   dequantize: thread = one weight row and half of the stage's K; 4-bit codes
//               are expanded to bf16 with integer ops (sign and magnitude bits moved into a
//               bf16 bit pattern, then one bf16x2 FMA by E4M3(s) * 2^94), written to TMEM
//               with tcgen05.st; then the epilogue: TMEM -> registers, g and s applied,
//               bf16 stores (or fp32 split-K partial slabs, reduced by the last CTA).
//
// The bf16 pattern of a code magnitude m = (e1 e0 m0) placed in bits 8..6 is the value
// grid(m) * 2^-126 (a subnormal when e = 0), so multiplying by E4M3(s) * 2^94 gives
// grid(m) * E4M3(s) * 2^-32 exactly (at most 6 significant bits); the epilogue multiplies
// the fp32 accumulator by 2^32 and then by g. A code word's nibbles j and j+4 (16 bits
// apart) share their shifts, so each 32-bit TMEM column holds elements (8q+j, 8q+j+4);
// the activations are stored with the same permutation of K inside each group of 8
// (the product over K is unchanged), written by the prep kernel next to the LoRA
// down-projection U = x A^T.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <mutex>

#include "common.cuh"
#include "sm100.cuh"

namespace nvfp4rl {
namespace {

using namespace sm100;

constexpr int kRows = 128;        // weight rows per CTA (MMA M)
constexpr int kKStage = 256;      // K per pipeline stage
constexpr int kCodeBytes = kRows * kKStage / 2;   // 16 KB
constexpr int kScaleBytes = kRows * kKStage / 16;  // 2 KB
constexpr int kThreads = 320;     // 10 warps
constexpr int kDeqWarps = 8;
constexpr int kMaxSplits = 8;     // split-K factor cap (the last CTA keeps one load per split in flight)

struct TcParams {
  int64_t M, N, K;
  int stages_per_split;  // 256-K stages per CTA
  int splits;
  int r;                 // LoRA rank (0 or a multiple of 16)
  int lora_box_bytes;    // min(2r, 128)
  float s;
  const float* w_g;
  uint16_t* y;
  float* slabs;          // [splits][M][N] fp32 when splits > 1
  uint32_t* counters;    // [tiles_m * tiles_n]
  uint32_t* status;
  int smem_stages;
};

__host__ __device__ constexpr int x_stage_bytes(int mbox) { return 4 * mbox * 128; }
__host__ __device__ constexpr int stage_bytes(int mbox) { return kCodeBytes + x_stage_bytes(mbox) + kScaleBytes; }

__device__ __forceinline__ uint32_t swizzle_mode_for(int box_bytes) {
  return box_bytes == 128 ? 2u : box_bytes == 64 ? 4u : 6u;
}

// bf16x2 fma with -0 addend: an exact product where the product is representable.
__device__ __forceinline__ uint32_t bf16x2_mul(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("fma.rn.bf16x2 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(0x80008000u));
  return d;
}

// Four TMEM columns from one word of 8 codes: column j = (code j, code j+4), each a bf16
// pattern of grid(m) * 2^-126 with the code's sign, times the bf16x2 scale.
__device__ __forceinline__ void expand_word(uint32_t w, uint32_t scale2, uint32_t* out) {
  const uint32_t kMag = 0x01C001C0u, kSign = 0x80008000u;
  const uint32_t p0 = ((w << 6) & kMag) | ((w << 12) & kSign);
  const uint32_t p1 = ((w << 2) & kMag) | ((w << 8) & kSign);
  const uint32_t p2 = ((w >> 2) & kMag) | ((w << 4) & kSign);
  const uint32_t p3 = ((w >> 6) & kMag) | (w & kSign);
  out[0] = bf16x2_mul(p0, scale2);
  out[1] = bf16x2_mul(p1, scale2);
  out[2] = bf16x2_mul(p2, scale2);
  out[3] = bf16x2_mul(p3, scale2);
}

// bf16x2 of E4M3(s) * 2^94 (exact: at most 4 significant bits).
__device__ __forceinline__ uint32_t scale_bf16x2(uint32_t s) {
  const uint32_t b = __float_as_uint(e4m3_decode_pos(s & 0x7Fu) * 0x1p94f) >> 16;
  return b | (b << 16);
}

template <int MBOX>
__global__ void __launch_bounds__(kThreads, 1)
    w4a16_tc_kernel(const __grid_constant__ CUtensorMap map_codes, const __grid_constant__ CUtensorMap map_scales,
                    const __grid_constant__ CUtensorMap map_x, const __grid_constant__ CUtensorMap map_blora,
                    const __grid_constant__ CUtensorMap map_u, const TcParams p) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int S = p.smem_stages;
  constexpr int kAbuf = MBOX <= 64 ? 3 : 2;
  constexpr uint32_t kDcol = 0, kLcol = MBOX, kAcol0 = 2 * MBOX;

  // layout: stages | lora A tile | lora U tile | barriers
  const int sb = stage_bytes(MBOX);
  uint8_t* lora_a = smem + S * sb;
  const int lora_a_bytes = p.r ? kRows * 2 * p.r : 0;
  uint8_t* lora_u = lora_a + lora_a_bytes;
  const int lora_u_bytes = p.r ? MBOX * 2 * p.r : 0;
  uint64_t* bars = reinterpret_cast<uint64_t*>(lora_u + lora_u_bytes);
  // full[S], empty[S], afull[kAbuf], aempty[kAbuf], dfull, lfull, drain
  uint64_t* full = bars;
  uint64_t* empty = full + S;
  uint64_t* afull = empty + S;
  uint64_t* aempty = afull + kAbuf;
  uint64_t* dfull = aempty + kAbuf;
  uint64_t* lfull = dfull + 1;
  uint64_t* drain = lfull + 1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  volatile uint32_t* last_flag = tmem_slot + 1;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int tile_n = blockIdx.x, split = blockIdx.y, tile_m = blockIdx.z;
  const int n0 = tile_n * kRows;
  const int m0 = tile_m * MBOX;
  const int st0 = split * p.stages_per_split;
  const int nst = min(p.stages_per_split, static_cast<int>(p.K / kKStage) - st0);
  const bool do_lora = p.r > 0 && split == 0;

  if (threadIdx.x == 0) {
    for (int i = 0; i < S; ++i) {
      mbar_init(smem_addr(&full[i]), 1);
      mbar_init(smem_addr(&empty[i]), kDeqWarps + 1);
    }
    for (int i = 0; i < kAbuf; ++i) {
      mbar_init(smem_addr(&afull[i]), kDeqWarps);
      mbar_init(smem_addr(&aempty[i]), 1);
    }
    mbar_init(smem_addr(dfull), 1);
    mbar_init(smem_addr(lfull), 1);
    mbar_init(smem_addr(drain), 1);
    *last_flag = 0;
    fence_barrier_init();
  }
  if (warp == 1) tmem_alloc(smem_addr(tmem_slot), 512);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  bool ok = true;
  if (warp == 0) {
    // ------------------------------------------------------------------ producer
    if (lane == 0) {
      prefetch_tensormap(&map_codes);
      prefetch_tensormap(&map_scales);
      prefetch_tensormap(&map_x);
      if (do_lora) {
        prefetch_tensormap(&map_blora);
        prefetch_tensormap(&map_u);
        const uint32_t bar = smem_addr(lfull);
        mbar_arrive_expect_tx(bar, lora_a_bytes + lora_u_bytes);
        const int nbox = 2 * p.r / p.lora_box_bytes;
        const int box_el = p.lora_box_bytes / 2;
        for (int b = 0; b < nbox; ++b) {
          tma_load_2d(smem_addr(lora_a + b * kRows * p.lora_box_bytes), &map_blora, b * box_el, n0, bar);
          tma_load_2d(smem_addr(lora_u + b * MBOX * p.lora_box_bytes), &map_u, b * box_el, m0, bar);
        }
      }
      int issued = 0;
      for (int j = 0; j < nst && ok; ++j) {
        const int s = j % S;
        const uint32_t ph = (j / S) & 1;
        if (!mbar_wait(smem_addr(&empty[s]), ph ^ 1, p.status, kStatusTimeoutProducer)) {
          ok = false;
          break;
        }
        uint8_t* st = smem + s * sb;
        const uint32_t bar = smem_addr(&full[s]);
        mbar_arrive_expect_tx(bar, sb);
        const int kst = st0 + j;
        tma_load_2d(smem_addr(st), &map_codes, kst * (kKStage / 2), n0, bar);
        tma_load_2d(smem_addr(st + kCodeBytes + x_stage_bytes(MBOX)), &map_scales, kst * (kKStage / 16), n0, bar);
#pragma unroll
        for (int q = 0; q < 4; ++q)
          tma_load_2d(smem_addr(st + kCodeBytes + q * MBOX * 128), &map_x, kst * kKStage + q * 64, m0, bar);
        issued = j + 1;
      }
      // drain: every issued stage has landed before the CTA can exit
      for (int j = max(0, issued - S); j < issued; ++j)
        mbar_wait(smem_addr(&full[j % S]), (j / S) & 1, p.status, kStatusTimeoutDrain);
      if (do_lora) mbar_wait(smem_addr(lfull), 0, p.status, kStatusTimeoutDrain);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      const uint32_t idesc = idesc_bf16_f32(kRows, MBOX);
      for (int j = 0; j < nst && ok; ++j) {
        const int s = j % S, a = j % kAbuf;
        // the dequant warps arrive on afull only after waiting for this stage's full barrier, so
        // afull also orders the activation tile the MMAs read
        if (!mbar_wait(smem_addr(&afull[a]), (j / kAbuf) & 1, p.status, kStatusTimeoutMma)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t xs = smem_addr(smem + s * sb + kCodeBytes);
#pragma unroll
        for (int kk = 0; kk < kKStage / 16; ++kk) {
          const uint64_t bdesc = smem_desc(xs + (kk >> 2) * MBOX * 128 + (kk & 3) * 32, 16, 1024, 2);
          mma_f16_ts(tmem + kDcol, tmem + kAcol0 + a * 128 + kk * 8, bdesc, idesc, (j | kk) ? 1u : 0u);
        }
        mma_commit(smem_addr(&aempty[a]));
        mma_commit(smem_addr(&empty[s]));
      }
      if (ok && do_lora) {
        if (mbar_wait(smem_addr(lfull), 0, p.status, kStatusTimeoutMma)) {
          tc_fence_after();
          const uint32_t sw = swizzle_mode_for(p.lora_box_bytes);
          const uint32_t sbo = 8 * p.lora_box_bytes;
          const uint32_t la = smem_addr(lora_a), lu = smem_addr(lora_u);
          for (int kk = 0; kk < p.r / 16; ++kk) {
            const int off = kk * 32;
            const int box = off / p.lora_box_bytes, in = off % p.lora_box_bytes;
            const uint64_t ad = smem_desc(la + box * kRows * p.lora_box_bytes + in, 16, sbo, sw);
            const uint64_t bd = smem_desc(lu + box * MBOX * p.lora_box_bytes + in, 16, sbo, sw);
            mma_f16_ss(tmem + kLcol, ad, bd, idesc, kk ? 1u : 0u);
          }
        } else {
          ok = false;
        }
      }
      mma_commit(smem_addr(dfull));  // also the completion point of every MMA issued above
    }
  } else {
    // ------------------------------------------------------------------ dequant + epilogue
    const int dw = warp - 2;             // 0..7
    const int quarter = warp & 3;        // TMEM lane quarter this warp may access
    const int half = dw >> 2;            // which 128-K half of the stage
    const int row = quarter * 32 + lane;  // weight row within the tile
    const uint32_t lane_base = static_cast<uint32_t>(quarter * 32) << 16;
    for (int j = 0; j < nst && ok; ++j) {
      const int s = j % S, a = j % kAbuf;
      // every lane waits; the warp leaves together if any lane ran out of time
      ok = __all_sync(0xFFFFFFFFu, mbar_wait(smem_addr(&full[s]), (j / S) & 1, p.status, kStatusTimeoutDequant) &&
                                       mbar_wait(smem_addr(&aempty[a]), ((j / kAbuf) & 1) ^ 1, p.status,
                                                 kStatusTimeoutDequant));
      if (!ok) break;
      const uint8_t* st = smem + s * sb;
      const uint8_t* crow = st + row * 128;
      const uint2 sc = *reinterpret_cast<const uint2*>(st + kCodeBytes + x_stage_bytes(MBOX) + row * 16 + half * 8);
      const uint32_t sbytes[2] = {sc.x, sc.y};
#pragma unroll
      for (int c = 0; c < 4; ++c) {  // 16-byte chunk = 32 codes = two MMA K-steps
        const int chunk = half * 4 + c;
        const uint4 cw = *reinterpret_cast<const uint4*>(crow + ((chunk ^ (row & 7)) << 4));
        const uint32_t s0 = scale_bf16x2((sbytes[c >> 1] >> (16 * (c & 1))) & 0xFFu);
        const uint32_t s1 = scale_bf16x2((sbytes[c >> 1] >> (16 * (c & 1) + 8)) & 0xFFu);
        uint32_t col[8];
        expand_word(cw.x, s0, col);
        expand_word(cw.y, s0, col + 4);
        tmem_st8(tmem + lane_base + kAcol0 + a * 128 + chunk * 16, col);
        expand_word(cw.z, s1, col);
        expand_word(cw.w, s1, col + 4);
        tmem_st8(tmem + lane_base + kAcol0 + a * 128 + chunk * 16 + 8, col);
      }
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(smem_addr(&afull[a]));
        mbar_arrive(smem_addr(&empty[s]));
      }
    }
    // ---------------------------------------------------------------- epilogue
    ok = __all_sync(0xFFFFFFFFu, ok && mbar_wait(smem_addr(dfull), 0, p.status, kStatusTimeoutEpilogue));
    tc_fence_after();
    if (ok) {
      const float g = *p.w_g;
      const int64_t n = n0 + row;
      constexpr int kTokHalf = MBOX / 2;
      const int t0 = half * kTokHalf;
      float* slab = p.splits > 1 ? p.slabs + static_cast<int64_t>(split) * p.M * p.N : nullptr;
#pragma unroll
      for (int c = 0; c < kTokHalf; c += 16) {
        uint32_t d[16], l[16];
        tmem_ld16(tmem + lane_base + kDcol + t0 + c, d);
        if (do_lora) tmem_ld16(tmem + lane_base + kLcol + t0 + c, l);
        tmem_ld_wait();
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const int64_t m = m0 + t0 + c + i;
          if (m >= p.M) break;
          float v = (__uint_as_float(d[i]) * 0x1p32f) * g;
          if (do_lora) v = fmaf(p.s, __uint_as_float(l[i]), v);
          if (slab) slab[m * p.N + n] = v;
          else p.y[m * p.N + n] = static_cast<uint16_t>(f32_to_bf16_bits(v));
        }
      }
    }
    if (p.splits > 1) {
      // last CTA of this output tile sums the fp32 partials in split order
      __threadfence();
      asm volatile("bar.sync 1, 256;" ::: "memory");
      if (dw == 0 && lane == 0) {
        const uint32_t cidx = tile_m * gridDim.x + tile_n;
        const uint32_t old = atomicAdd(&p.counters[cidx], 1u);
        *last_flag = (old == static_cast<uint32_t>(p.splits - 1)) ? 1u : 0u;
        if (old == static_cast<uint32_t>(p.splits - 1)) p.counters[cidx] = 0;
      }
      asm volatile("bar.sync 1, 256;" ::: "memory");
      if (*last_flag) {
        __threadfence();
        // 256 threads over the MBOX x 128 output tile: thread -> one row, a run of kCols columns
        constexpr int kThreadsPerRow = 256 / MBOX, kCols = kRows / kThreadsPerRow;
        const int t = dw * 32 + lane;
        const int64_t m = m0 + t / kThreadsPerRow;
        const int64_t nb = n0 + (t % kThreadsPerRow) * kCols;
        if (m < p.M) {
          uint4* dst = reinterpret_cast<uint4*>(p.y + m * p.N + nb);
#pragma unroll 1
          for (int c8 = 0; c8 < kCols; c8 += 8) {
            // all splits' loads of these 8 columns are issued before any is summed
            float4 va[kMaxSplits], vb[kMaxSplits];
#pragma unroll
            for (int sp = 0; sp < kMaxSplits; ++sp) {
              if (sp < p.splits) {
                const float4* src =
                    reinterpret_cast<const float4*>(p.slabs + (static_cast<int64_t>(sp) * p.M + m) * p.N + nb + c8);
                va[sp] = __ldcg(src);
                vb[sp] = __ldcg(src + 1);
              }
            }
            float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int sp = 0; sp < kMaxSplits; ++sp) {
              if (sp < p.splits) {
                acc[0] += va[sp].x; acc[1] += va[sp].y; acc[2] += va[sp].z; acc[3] += va[sp].w;
                acc[4] += vb[sp].x; acc[5] += vb[sp].y; acc[6] += vb[sp].z; acc[7] += vb[sp].w;
              }
            }
            uint32_t o[4];
#pragma unroll
            for (int q = 0; q < 4; ++q) o[q] = f32_to_bf16_bits(acc[2 * q]) | (f32_to_bf16_bits(acc[2 * q + 1]) << 16);
            dst[c8 / 8] = make_uint4(o[0], o[1], o[2], o[3]);
          }
        }
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

constexpr int kPrepK = 128;   // K per prep CTA
constexpr int kPrepM = 64;    // activation rows per prep CTA
constexpr int kPrepPad = 8;   // bf16 row padding (conflict-free ldmatrix)

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

// Prep: x_perm (K permuted inside groups of 8 as 0,4,1,5,2,6,3,7) and the LoRA down-projection
// U = bf16(x A^T). CTA (k chunk, row tile) stages a 64 x 128 slice of x and a 32 x 128 slice of A
// in shared memory, writes its slice of x_perm, and runs the small GEMM on mma.sync (warp w:
// rows 16w..16w+15, 32 ranks per pass); partial sums go to the fp32 accumulator U32 (zeroed by
// the caller); the last chunk of a row tile (arrival counter) converts its rows of U to bf16.
__global__ void __launch_bounds__(128) w4a16_prep_kernel(const uint16_t* __restrict__ x, int64_t M, int64_t K,
                                                         const uint16_t* __restrict__ A, int r,
                                                         uint16_t* __restrict__ xp, float* __restrict__ U32,
                                                         uint16_t* __restrict__ U, uint32_t* __restrict__ tilecnt) {
  __shared__ __align__(16) uint16_t xs[kPrepM][kPrepK + kPrepPad];
  __shared__ __align__(16) uint16_t as[32][kPrepK + kPrepPad];
  const int64_t m0 = static_cast<int64_t>(blockIdx.y) * kPrepM;
  const int64_t k0 = static_cast<int64_t>(blockIdx.x) * kPrepK;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  // 64 rows x 16 vectors of 8 bf16: 8 per thread
#pragma unroll
  for (int i = 0; i < (kPrepM * kPrepK / 8) / 128; ++i) {
    const int idx = tid + i * 128, row = idx >> 4, vec = idx & 15;
    const int64_t m = m0 + row;
    uint4 a = make_uint4(0, 0, 0, 0);
    if (m < M) {
      a = *reinterpret_cast<const uint4*>(x + m * K + k0 + vec * 8);
      uint4 o;  // elements e0..e7 (two per word) -> e0 e4 | e1 e5 | e2 e6 | e3 e7
      o.x = __byte_perm(a.x, a.z, 0x5410);
      o.y = __byte_perm(a.x, a.z, 0x7632);
      o.z = __byte_perm(a.y, a.w, 0x5410);
      o.w = __byte_perm(a.y, a.w, 0x7632);
      *reinterpret_cast<uint4*>(xp + m * K + k0 + vec * 8) = o;
    }
    *reinterpret_cast<uint4*>(&xs[row][vec * 8]) = a;
  }
  if (r == 0) return;
  for (int j0 = 0; j0 < r; j0 += 32) {
    __syncthreads();
#pragma unroll
    for (int i = 0; i < (32 * kPrepK / 8) / 128; ++i) {
      const int idx = tid + i * 128, jr = idx >> 4, vec = idx & 15;
      uint4 v = make_uint4(0, 0, 0, 0);
      if (j0 + jr < r) v = __ldg(reinterpret_cast<const uint4*>(A + static_cast<int64_t>(j0 + jr) * K + k0 + vec * 8));
      *reinterpret_cast<uint4*>(&as[jr][vec * 8]) = v;
    }
    __syncthreads();
    float c[4][4] = {};
#pragma unroll
    for (int ks = 0; ks < kPrepK / 16; ++ks) {
      uint32_t a[4];
      ldsm_x4(static_cast<uint32_t>(__cvta_generic_to_shared(&xs[warp * 16 + (lane & 15)][ks * 16 + (lane >> 4) * 8])),
              a[0], a[1], a[2], a[3]);
#pragma unroll
      for (int jp = 0; jp < 2; ++jp) {
        const int q = lane >> 3;
        uint32_t b0, b1, b2, b3;
        ldsm_x4(static_cast<uint32_t>(__cvta_generic_to_shared(&as[jp * 16 + (q >> 1) * 8 + (lane & 7)][ks * 16 + (q & 1) * 8])),
                b0, b1, b2, b3);
        mma16816(c[2 * jp], a, b0, b1);
        mma16816(c[2 * jp + 1], a, b2, b3);
      }
    }
    // C fragment: c0,c1 at (row lane/4, cols 2(lane%4), +1); c2,c3 at row + 8
#pragma unroll
    for (int nt = 0; nt < 4; ++nt)
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const int64_t m = m0 + warp * 16 + (lane >> 2) + (q >> 1) * 8;
        const int j = j0 + nt * 8 + 2 * (lane & 3) + (q & 1);
        if (m < M && j < r) atomicAdd(U32 + m * r + j, c[nt][q]);
      }
  }
  __threadfence();
  __syncthreads();
  __shared__ uint32_t last;
  if (tid == 0) last = (atomicAdd(tilecnt + blockIdx.y, 1u) == gridDim.x - 1) ? 1u : 0u;
  __syncthreads();
  if (last) {
    __threadfence();
    for (int i = tid; i < kPrepM * r; i += blockDim.x) {
      const int64_t m = m0 + i / r;
      if (m < M) U[m * r + i % r] = static_cast<uint16_t>(f32_to_bf16_bits(__ldcg(U32 + m * r + i % r)));
    }
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

struct TcPlan {
  int mbox, tiles_m, tiles_n, splits, stages_per_split, smem_stages;
  // ws_zero .. ws_zero + zero_bytes is cleared every call: U32, per-row and per-tile counters
  size_t smem_bytes, ws_xperm, ws_u, ws_zero, zero_bytes, ws_u32, ws_rowcnt, ws_counters, ws_slabs, ws_total;
};

TcPlan plan(int64_t M, int64_t N, int64_t K, int r, int sm_count) {
  TcPlan t{};
  t.mbox = M <= 64 ? 64 : 128;
  t.tiles_m = static_cast<int>((M + t.mbox - 1) / t.mbox);
  t.tiles_n = static_cast<int>(N / kRows);
  const int kst = static_cast<int>(K / kKStage);
  const int ctas = t.tiles_n * t.tiles_m;
  int splits = std::max(1, std::min({kst, sm_count / std::max(1, ctas), kMaxSplits}));
  t.stages_per_split = (kst + splits - 1) / splits;
  t.splits = (kst + t.stages_per_split - 1) / t.stages_per_split;
  const size_t lora = r ? static_cast<size_t>(kRows + t.mbox) * 2 * r : 0;
  const size_t fixed = 1024 + lora + 256;
  const size_t sb = stage_bytes(t.mbox);
  t.smem_stages = static_cast<int>(std::min<size_t>(4, (227 * 1024 - fixed) / sb));
  t.smem_bytes = fixed + t.smem_stages * sb;
  size_t o = 0;
  auto take = [&](size_t b) { size_t at = o; o = align_up(o + b, 256); return at; };
  t.ws_xperm = take(static_cast<size_t>(M) * K * 2);
  t.ws_u = take(static_cast<size_t>(M) * std::max(r, 1) * 2);
  t.ws_u32 = take(static_cast<size_t>(M) * std::max(r, 1) * 4);
  t.ws_rowcnt = take(static_cast<size_t>(M) * 4);
  t.ws_counters = take(static_cast<size_t>(t.tiles_m) * t.tiles_n * 4);
  t.ws_zero = t.ws_u32;
  t.zero_bytes = o - t.ws_u32;
  t.ws_slabs = take(t.splits > 1 ? static_cast<size_t>(t.splits) * M * N * 4 : 0);
  t.ws_total = o;
  return t;
}

bool make_map(CUtensorMap* m, CUtensorMapDataType dt, const void* base, uint64_t cols, uint64_t rows, int esize,
              uint32_t box_cols, uint32_t box_rows, CUtensorMapSwizzle sw) {
  return make_tensor_map_2d(m, dt, base, cols, rows, esize, box_cols, box_rows, sw);
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

// True when the tcgen05 W4A16 path takes this shape.
bool w4a16_tc_supported(int64_t M, int64_t N, int64_t K, int r) {
  if (!(M > 0 && N % kRows == 0 && K % kKStage == 0 && (r == 0 || (r % 16 == 0 && r <= 128)))) return false;
  return plan(M, N, K, r, kPlanSMs).smem_stages >= 2;
}

size_t w4a16_tc_workspace_bytes(int64_t M, int64_t N, int64_t K, int r, int sm_count) {
  return plan(M, N, K, r, sm_count).ws_total;
}

nvfp4rl_status launch_w4a16_tc(const LinearArgs& a, void* ws, size_t ws_bytes, const DeviceInfo& dev,
                               cudaStream_t st) {
  const TcPlan t = plan(a.M, a.N, a.K, a.r, std::min(dev.sm_count, kPlanSMs));
  if (ws_bytes < t.ws_total) return NVFP4RL_ERR_WORKSPACE;
  if (t.smem_stages < 2) return NVFP4RL_ERR_UNSUPPORTED_SHAPE;
  char* base = static_cast<char*>(ws);
  uint16_t* xp = reinterpret_cast<uint16_t*>(base + t.ws_xperm);
  uint16_t* U = reinterpret_cast<uint16_t*>(base + t.ws_u);
  uint32_t* counters = reinterpret_cast<uint32_t*>(base + t.ws_counters);
  float* slabs = reinterpret_cast<float*>(base + t.ws_slabs);

  if (cudaMemsetAsync(base + t.ws_zero, 0, t.zero_bytes, st) != cudaSuccess) return NVFP4RL_ERR_CUDA;
  dim3 pgrid(static_cast<unsigned>(a.K / kPrepK), static_cast<unsigned>((a.M + kPrepM - 1) / kPrepM));
  w4a16_prep_kernel<<<pgrid, 128, 0, st>>>(a.x, a.M, a.K, a.A, a.r, xp, reinterpret_cast<float*>(base + t.ws_u32), U,
                                           reinterpret_cast<uint32_t*>(base + t.ws_rowcnt));
  if (launch_status() != NVFP4RL_OK) return NVFP4RL_ERR_CUDA;

  CUtensorMap mc, ms, mx, mb, mu;
  const int lbox = a.r ? std::min(2 * a.r, 128) : 128;
  if (!make_map(&mc, CU_TENSOR_MAP_DATA_TYPE_UINT8, a.w_codes, a.K / 2, a.N, 1, 128, kRows, CU_TENSOR_MAP_SWIZZLE_128B) ||
      !make_map(&ms, CU_TENSOR_MAP_DATA_TYPE_UINT8, a.w_scales, a.K / 16, a.N, 1, 16, kRows, CU_TENSOR_MAP_SWIZZLE_NONE) ||
      !make_map(&mx, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, xp, a.K, a.M, 2, 64, t.mbox, CU_TENSOR_MAP_SWIZZLE_128B))
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
  p.stages_per_split = t.stages_per_split;
  p.splits = t.splits;
  p.r = a.r;
  p.lora_box_bytes = lbox;
  p.s = a.s;
  p.w_g = a.w_g;
  p.y = a.y;
  p.slabs = slabs;
  p.counters = counters;
  p.status = dev.status;
  p.smem_stages = t.smem_stages;
  dim3 grid(t.tiles_n, t.splits, t.tiles_m);
  cudaError_t e;
  if (t.mbox == 64) {
    e = cudaFuncSetAttribute(w4a16_tc_kernel<64>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(t.smem_bytes));
    if (e == cudaSuccess) w4a16_tc_kernel<64><<<grid, kThreads, t.smem_bytes, st>>>(mc, ms, mx, mb, mu, p);
  } else {
    e = cudaFuncSetAttribute(w4a16_tc_kernel<128>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(t.smem_bytes));
    if (e == cudaSuccess) w4a16_tc_kernel<128><<<grid, kThreads, t.smem_bytes, st>>>(mc, ms, mx, mb, mu, p);
  }
  if (e != cudaSuccess) return NVFP4RL_ERR_CUDA;
  return launch_status();
}

}  // namespace nvfp4rl
