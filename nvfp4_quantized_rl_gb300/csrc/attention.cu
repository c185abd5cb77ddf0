// Decode attention over an NVFP4 KV cache (sm_103a).
//
// TRACE summary, section "実験結果と性能": rollouts run with FP4 weights, activations and KV
// cache. Each cached K/V row of a head is NVFP4-encoded (16-element blocks along the head
// dimension, E4M3 block scales, a per-tensor fp32 g given by the caller); decode attention reads
// the dequantized rows: out[b][h] = softmax(scale q[b][h] K^T) V over the first lens[b] cached
// tokens of KV head h / (Hq / Hkv).
//
// Split-KV ("flash decoding"): one CTA of four warps per (sequence, KV head, token span); warp w
// takes the 64-token groups w, w + 4, ... of the span and works alone: its own ring of two
// shared-memory slots, filled by two TMA tensor copies (the K and V code rows of the group, 64-byte
// swizzle) and 8-byte cp.async copies of the scale rows (zeros past the sequence's length), all
// completing on the slot's mbarrier. Per 16-token step of a group the warp
//   - computes S^T = K Q^T with mma.sync m16n8k16 in f16: K is the A operand, its fragments built
//     in registers straight from the code bytes (one cvt e2m1x2 -> f16x2 per byte, one f16x2
//     multiply by the E4M3 block scale: both exact), the group's query heads the N columns (one
//     8-column tile, two for more than 8 heads). Q enters as f16 scaled by a power of two that puts
//     max |q| of the group in [2^14, 2^15): exact for every bf16 element down to 2^-31 of the max;
//   - keeps an online softmax in exp2 (ex2.approx) per query head (column), rescaling O only when
//     a maximum grows;
//   - transposes P (f16) with movmatrix and adds O^T += V^T P^T, V^T the A operand: a nibble
//     interleave of two tokens' code words gives bytes holding one dimension of both tokens, so
//     the same cvt yields the (token, token) pairs the fragment wants.
// The dot products run over a permutation of the head dimension (the same for Q and K) and the
// tokens of a step over a permutation chosen with the swizzle so that every shared-memory load
// of the step is free of bank conflicts. The four warps' (max, sum, O) are merged in shared
// memory; with several spans per sequence a second kernel merges the spans' partials.
#include <climits>
#include <map>
#include <mutex>

#include "common.cuh"
#include "sm100.cuh"

namespace nvfp4rl {
namespace {

using namespace sm100;

constexpr int kHeadDim = 128;
constexpr int kTok = 64;  // tokens per ring slot: one iteration of a warp
constexpr int kWarps = 4;
constexpr int kAttnThreads = 32 * kWarps;
constexpr int kStages = 2;                                      // ring slots per warp
constexpr int kCodeBytes = kTok * kHeadDim / 2;                 // one head's code rows of a group
constexpr int kScaleBytes = kTok * kHeadDim / 16;               // one head's scale rows of a group
constexpr int kSlotBytes = 2 * kCodeBytes + 2 * kScaleBytes;    // K codes | V codes | K scales | V scales
constexpr int kRingBytes = kWarps * kStages * kSlotBytes;
constexpr int kAttnSmem = kRingBytes + 1024;                    // + room to align the ring to 1024 B
constexpr int kPartFloats = 132;                                // per (span, head): max, sum, O[128], padding
constexpr float kLog2e = 1.4426950408889634f;
static_assert(kSlotBytes % 1024 == 0 && kCodeBytes % 1024 == 0, "boxes start on 1024-byte boundaries");
static_assert(kRingBytes >= kWarps * 16 * kHeadDim * 4, "the ring doubles as the merge area");

// Token (0..15) of row / k index i of a 16-token step: bits (i0, i1, i2, i3) -> (i0 ^ i1, i0, i2, i3).
// With the swizzle below, the two K rows of a quarter-warp's 16-byte loads differ in bit 0 (other
// bank halves) and the four V rows of a half-warp's 8-byte loads differ in bits 0 and 2 (four
// different 32-byte bank windows): no load of a step has a bank conflict.
__host__ __device__ constexpr int step_token(int i) {
  return ((i & 1) ^ ((i >> 1) & 1)) | ((i & 1) << 1) | (i & 4) | (i & 8);
}

// Byte offset of byte c of 64-byte row r in a TMA box stored with the 64-byte swizzle (16-byte
// unit bits 4..5 XOR bits 7..8 of the offset), from a 1024-byte aligned base.
__host__ __device__ constexpr uint32_t swz(int r, int c) {
  return (64u * r + c) ^ ((((64u * r + c) >> 7) & 3u) << 4);
}

__device__ __forceinline__ uint4 lds128(uint32_t a) {
  uint4 v;
  asm volatile("ld.shared.v4.b32 {%0,%1,%2,%3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(a));
  return v;
}
__device__ __forceinline__ uint2 lds64(uint32_t a) {
  uint2 v;
  asm volatile("ld.shared.v2.b32 {%0,%1}, [%2];" : "=r"(v.x), "=r"(v.y) : "r"(a));
  return v;
}
__device__ __forceinline__ uint32_t lds_u16(uint32_t a) {
  uint16_t v;
  asm volatile("ld.shared.u16 %0, [%1];" : "=h"(v) : "r"(a));
  return v;
}
__device__ __forceinline__ uint32_t lds_u8(uint32_t a) {
  uint32_t v;
  asm volatile("ld.shared.u8 %0, [%1];" : "=r"(v) : "r"(a));
  return v;
}

// Four code bytes (two E2M1 elements each, low nibble first) -> four f16x2 (low half = low nibble).
__device__ __forceinline__ void e2m1x8_f16(uint32_t w, uint32_t (&d)[4]) {
  asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\t"
      "mov.b32 {b0, b1, b2, b3}, %4;\n\t"
      "cvt.rn.f16x2.e2m1x2 %0, b0;\n\t"
      "cvt.rn.f16x2.e2m1x2 %1, b1;\n\t"
      "cvt.rn.f16x2.e2m1x2 %2, b2;\n\t"
      "cvt.rn.f16x2.e2m1x2 %3, b3;\n\t}"
      : "=r"(d[0]), "=r"(d[1]), "=r"(d[2]), "=r"(d[3])
      : "r"(w));
}

// Two E4M3 bytes (low byte first) -> f16x2, exact: every E4M3 value is an f16 normal.
__device__ __forceinline__ uint32_t e4m3x2_f16(uint32_t two_bytes) {
  uint32_t d;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(d) : "h"(static_cast<uint16_t>(two_bytes)));
  return d;
}

// Exact here: an E2M1 value times an E4M3 value has at most 6 significant bits and lies within
// [2^-10, 2688] or is zero.
__device__ __forceinline__ uint32_t hmul2(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}

__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
  uint32_t d;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
  return d;
}

__device__ __forceinline__ uint32_t pack_f16(float lo, float hi) {
  uint32_t d;
  asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(d) : "f"(hi), "f"(lo));
  return d;
}

// Transposes the warp's 8x8 b16 fragment (lane l: row l / 4, columns 2 (l % 4), +1).
__device__ __forceinline__ uint32_t movm_t(uint32_t a) {
  uint32_t d;
  asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(d) : "r"(a));
  return d;
}

__device__ __forceinline__ void mma_f16(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                        uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// 2^x (approximate, about 2 ulp; results below 2^-126 flush to zero, 2^-inf = 0).
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ void cp_async8(uint32_t dst, const void* src, uint32_t src_bytes) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 8, %2;" ::"r"(dst), "l"(src), "r"(src_bytes) : "memory");
}
// The mbarrier receives one arrival once every cp.async this thread issued before has landed
// (the barrier's expected count includes it).
__device__ __forceinline__ void cp_async_arrive_noinc(uint32_t bar) {
  asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }
__device__ __forceinline__ void fence_proxy_async() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

struct AttnArgs {
  const uint16_t* q;
  const uint8_t *ks, *vs;
  const float *gk, *gv;
  const int32_t* lens;
  int64_t Hq, Hkv, Lmax;
  int nsplit, span;  // token spans per sequence and their length (a multiple of kTok)
  float scale;
  uint16_t* out;     // used when nsplit == 1
  float* part;       // [B*Hkv][nsplit][16][kPartFloats] when nsplit > 1
  uint32_t* status;  // the library's error word: a wait that gave up sets a timeout bit
};

// kNH: 8-column tiles of query heads (1: up to 8 heads per KV head, 2: up to 16).
template <int kNH>
__global__ void __launch_bounds__(kAttnThreads, kNH == 1 ? 3 : 2)
    kv_attention_kernel(const __grid_constant__ CUtensorMap map_k, const __grid_constant__ CUtensorMap map_v,
                        const AttnArgs a) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ __align__(8) uint64_t bars[kWarps][kStages];
  __shared__ float msm[kWarps][16], lsm[kWarps][16];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, g = lane >> 2, q = lane & 3;
  const uint32_t raw = smem_addr(smem_raw);
  const uint32_t ring0 = (raw + 1023u) & ~1023u;
  const uint32_t ring = ring0 + warp * (kStages * kSlotBytes);
  const uint32_t bar0 = smem_addr(&bars[warp][0]);
  if (lane == 0) {
#pragma unroll
    for (int s = 0; s < kStages; ++s) mbar_init(bar0 + 8 * s, 33);  // lane 0's expect_tx + 32 cp.async arrivals
    fence_barrier_init();
  }
  __syncwarp();
  const int64_t bh = blockIdx.y, b = bh / a.Hkv, kvh = bh % a.Hkv;
  const int group = static_cast<int>(a.Hq / a.Hkv);
  griddep_wait();
  griddep_launch_dependents();
  const int64_t len = min(max(static_cast<int64_t>(a.lens[b]), int64_t(0)), a.Lmax);
  const int64_t t_begin = static_cast<int64_t>(blockIdx.x) * a.span;
  const int64_t t_end = min(t_begin + a.span, len);
  const int ngroups = t_end > t_begin ? static_cast<int>((t_end - t_begin + kTok - 1) / kTok) : 0;
  const int mine = ngroups > warp ? (ngroups - warp + kWarps - 1) / kWarps : 0;  // groups warp, warp + 4, ...
  const int64_t row0 = b * a.Lmax;  // cache row of the sequence's token 0
  // scale rows: lane l copies rows l and l + 32 of each group; sr = the row offset of its first
  // row of group 0, advanced by one stride per group
  const int64_t srow_step = static_cast<int64_t>(kWarps) * kTok * a.Hkv * (kHeadDim / 16);
  const int64_t sr0 = ((row0 + t_begin + static_cast<int64_t>(warp) * kTok + lane) * a.Hkv + kvh) * (kHeadDim / 16);
  const int64_t t_lane = t_begin + static_cast<int64_t>(warp) * kTok + lane;  // token of that row

  // group n of this warp (tokens t_begin + 64 (warp + 4 n) ..) into slot n % kStages
  const auto issue = [&](int n) {
    const int slot = n % kStages;
    const int64_t t0 = t_begin + static_cast<int64_t>(warp + n * kWarps) * kTok;
    const uint32_t sb = ring + slot * kSlotBytes, bar = bar0 + 8 * slot;
    if (lane == 0) {
      fence_proxy_async();  // this warp's reads of the slot's previous bytes come before the copies
      mbar_arrive_expect_tx(bar, 2 * kCodeBytes);
      tma_load_2d(sb, &map_k, static_cast<int32_t>(kvh * 64), static_cast<int32_t>(row0 + t0), bar);
      tma_load_2d(sb + kCodeBytes, &map_v, static_cast<int32_t>(kvh * 64), static_cast<int32_t>(row0 + t0), bar);
    }
    // rows at or past t_end read nothing and land as zeros, which zeroes those tokens' K and V
    // whatever their code bytes
    const int64_t t = t_lane + static_cast<int64_t>(n) * kWarps * kTok;
    const int64_t off = sr0 + n * srow_step;
    const int64_t off32 = off + 32 * a.Hkv * (kHeadDim / 16);
    const bool live0 = t < t_end, live1 = t + 32 < t_end;
    cp_async8(sb + 2 * kCodeBytes + 8 * lane, a.ks + (live0 ? off : 0), live0 ? 8u : 0u);
    cp_async8(sb + 2 * kCodeBytes + kScaleBytes + 8 * lane, a.vs + (live0 ? off : 0), live0 ? 8u : 0u);
    cp_async8(sb + 2 * kCodeBytes + 8 * (lane + 32), a.ks + (live1 ? off32 : 0), live1 ? 8u : 0u);
    cp_async8(sb + 2 * kCodeBytes + kScaleBytes + 8 * (lane + 32), a.vs + (live1 ? off32 : 0), live1 ? 8u : 0u);
    cp_async_arrive_noinc(bar);
  };
  const int pre = min(mine, kStages);
  for (int n = 0; n < pre; ++n) issue(n);

  // Q^T fragments: head 8 h + g (zero past the group), dims 32 q .. 32 q + 31 as f16 times 2^e,
  // 2^e putting max |q| over the group's heads in [2^14, 2^15); k-step s takes words 2 s, 2 s + 1
  uint32_t qb[kNH][16];
  uint32_t amax16 = 0;
#pragma unroll
  for (int h = 0; h < kNH; ++h) {
    const int hh = 8 * h + g;
    if (hh < group) {
      const uint4* src = reinterpret_cast<const uint4*>(a.q + ((b * a.Hq + kvh * group + hh) * kHeadDim + 32 * q));
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const uint4 v = src[i];
        qb[h][4 * i] = v.x;
        qb[h][4 * i + 1] = v.y;
        qb[h][4 * i + 2] = v.z;
        qb[h][4 * i + 3] = v.w;
      }
    } else {
#pragma unroll
      for (int i = 0; i < 16; ++i) qb[h][i] = 0u;
    }
#pragma unroll
    for (int i = 0; i < 16; ++i) amax16 = __vmaxu2(amax16, qb[h][i] & 0x7FFF7FFFu);
  }
  amax16 = __reduce_max_sync(0xFFFFFFFFu, max(amax16 & 0xFFFFu, amax16 >> 16));
  const int qexp = static_cast<int>((amax16 >> 7) & 0xFFu);  // biased exponent of max |q|
  const float qscale = __uint_as_float(static_cast<uint32_t>(min(max(268 - qexp, 1), 254)) << 23);
#pragma unroll
  for (int h = 0; h < kNH; ++h)
#pragma unroll
    for (int i = 0; i < 16; ++i)
      qb[h][i] = pack_f16(__uint_as_float(qb[h][i] << 16) * qscale, __uint_as_float(qb[h][i] & 0xFFFF0000u) * qscale);
  const float sl2 = a.scale * __ldg(a.gk) * kLog2e / qscale;  // scores in log2 units

  // per-thread constant offsets: K rows step_token(g), step_token(g + 8) (16-byte unit q); V rows
  // step_token(2 q + {0, 1, 8, 9}) (bytes 8 g .. 8 g + 7); their scale bytes
  const int tk0 = step_token(g), tk1 = step_token(g + 8);
  const int tv[4] = {step_token(2 * q), step_token(2 * q + 1), step_token(2 * q + 8), step_token(2 * q + 9)};
  const uint32_t koff0 = swz(tk0, 16 * q), koff1 = swz(tk1, 16 * q);
  uint32_t voff[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) voff[i] = swz(tv[i], 8 * g);

  float m_run[kNH][2], l_run[kNH][2];
  float oacc[8][kNH][4];  // O^T tile m: rows dims 16 g + 2 m (c0, c1) and + 1 (c2, c3), columns heads 8 h + 2 q + e
#pragma unroll
  for (int h = 0; h < kNH; ++h)
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      m_run[h][e] = -INFINITY;
      l_run[h][e] = 0.0f;
    }
#pragma unroll
  for (int m = 0; m < 8; ++m)
#pragma unroll
    for (int h = 0; h < kNH; ++h) oacc[m][h][0] = oacc[m][h][1] = oacc[m][h][2] = oacc[m][h][3] = 0.0f;

  int done = 0;
  bool ok = true;
  for (; done < mine; ++done) {
    const int slot = done % kStages;
    const bool landed = mbar_wait(bar0 + 8 * slot, static_cast<uint32_t>((done / kStages) & 1), a.status,
                                  kStatusTimeoutProducer);
    if (!__all_sync(0xFFFFFFFFu, landed)) {
      ok = false;
      break;
    }
    const uint32_t kb = ring + slot * kSlotBytes, vb = kb + kCodeBytes, ksb = kb + 2 * kCodeBytes,
                   vsb = ksb + kScaleBytes;
    const int64_t t0 = t_begin + static_cast<int64_t>(warp + done * kWarps) * kTok;

    // S^T = K Q^T, one 16-token step (rows step_token(g), step_token(g + 8)) at a time
    float sacc[4][kNH][4];
#pragma unroll
    for (int kk = 0; kk < 4; ++kk) {
#pragma unroll
      for (int h = 0; h < kNH; ++h) sacc[kk][h][0] = sacc[kk][h][1] = sacc[kk][h][2] = sacc[kk][h][3] = 0.0f;
      const uint4 c0 = lds128(kb + 1024 * kk + koff0), c1 = lds128(kb + 1024 * kk + koff1);
      const uint32_t f0 = e4m3x2_f16(lds_u16(ksb + 128 * kk + 8 * tk0 + 2 * q));
      const uint32_t f1 = e4m3x2_f16(lds_u16(ksb + 128 * kk + 8 * tk1 + 2 * q));
      const uint32_t s0[2] = {prmt(f0, f0, 0x1010u), prmt(f0, f0, 0x3232u)};  // blocks 2 q, 2 q + 1 of row tk0
      const uint32_t s1[2] = {prmt(f1, f1, 0x1010u), prmt(f1, f1, 0x3232u)};
      const uint32_t w0[4] = {c0.x, c0.y, c0.z, c0.w}, w1[4] = {c1.x, c1.y, c1.z, c1.w};
#pragma unroll
      for (int w = 0; w < 4; ++w) {
        uint32_t k0[4], k1[4];
        e2m1x8_f16(w0[w], k0);
        e2m1x8_f16(w1[w], k1);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          k0[i] = hmul2(k0[i], s0[w >> 1]);
          k1[i] = hmul2(k1[i], s1[w >> 1]);
        }
        // k-steps 2 w and 2 w + 1 take bytes (4 w, 4 w + 1) and (4 w + 2, 4 w + 3)
#pragma unroll
        for (int j = 0; j < 2; ++j)
#pragma unroll
          for (int h = 0; h < kNH; ++h)
            mma_f16(sacc[kk][h], k0[2 * j], k1[2 * j], k0[2 * j + 1], k1[2 * j + 1], qb[h][4 * w + 2 * j],
                    qb[h][4 * w + 2 * j + 1]);
      }
    }

    // online softmax per query head (column 8 h + 2 q + e); rows: tokens t0 + 16 kk + tk0 / tk1
    float mx[kNH][2];
#pragma unroll
    for (int h = 0; h < kNH; ++h) mx[h][0] = mx[h][1] = -INFINITY;
#pragma unroll
    for (int kk = 0; kk < 4; ++kk)
#pragma unroll
      for (int h = 0; h < kNH; ++h)
#pragma unroll
        for (int i = 0; i < 4; ++i) sacc[kk][h][i] *= sl2;
    if (t0 + kTok > t_end) {  // the span's last group: tokens at or past t_end do not count
#pragma unroll
      for (int kk = 0; kk < 4; ++kk) {
        const bool dead0 = t0 + 16 * kk + tk0 >= t_end, dead1 = t0 + 16 * kk + tk1 >= t_end;
#pragma unroll
        for (int h = 0; h < kNH; ++h)
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            if (dead0) sacc[kk][h][e] = -INFINITY;
            if (dead1) sacc[kk][h][2 + e] = -INFINITY;
          }
      }
    }
#pragma unroll
    for (int kk = 0; kk < 4; ++kk)
#pragma unroll
      for (int h = 0; h < kNH; ++h)
#pragma unroll
        for (int e = 0; e < 2; ++e) mx[h][e] = fmaxf(mx[h][e], fmaxf(sacc[kk][h][e], sacc[kk][h][2 + e]));
    bool grew = false;
#pragma unroll
    for (int h = 0; h < kNH; ++h)
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        mx[h][e] = fmaxf(mx[h][e], __shfl_xor_sync(0xFFFFFFFFu, mx[h][e], 4));
        mx[h][e] = fmaxf(mx[h][e], __shfl_xor_sync(0xFFFFFFFFu, mx[h][e], 8));
        mx[h][e] = fmaxf(mx[h][e], __shfl_xor_sync(0xFFFFFFFFu, mx[h][e], 16));
        grew |= mx[h][e] > m_run[h][e];
      }
    if (__any_sync(0xFFFFFFFFu, grew)) {
#pragma unroll
      for (int h = 0; h < kNH; ++h)
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const float m_new = fmaxf(m_run[h][e], mx[h][e]);
          const float corr = m_new == -INFINITY ? 1.0f : ex2(m_run[h][e] - m_new);
          m_run[h][e] = m_new;
          l_run[h][e] *= corr;
#pragma unroll
          for (int m = 0; m < 8; ++m) {
            oacc[m][h][e] *= corr;
            oacc[m][h][2 + e] *= corr;
          }
        }
    }
    // P (f16) transposed into the B fragments of O^T += V^T P^T: k index i <-> token step_token(i)
    uint32_t pb[4][kNH][2];
#pragma unroll
    for (int kk = 0; kk < 4; ++kk)
#pragma unroll
      for (int h = 0; h < kNH; ++h) {
        float p[4];
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const float base = m_run[h][e] == -INFINITY ? 0.0f : m_run[h][e];  // nothing seen yet: every p is 0
          p[e] = ex2(sacc[kk][h][e] - base);
          p[2 + e] = ex2(sacc[kk][h][2 + e] - base);
          l_run[h][e] += p[e] + p[2 + e];
        }
        pb[kk][h][0] = movm_t(pack_f16(p[0], p[1]));
        pb[kk][h][1] = movm_t(pack_f16(p[2], p[3]));
      }

    // O^T += V^T P^T: tile m = 4 u + k takes byte 8 g + m of the V rows (dims 16 g + 2 m, + 1)
#pragma unroll
    for (int kk = 0; kk < 4; ++kk) {
      const uint2 X0 = lds64(vb + 1024 * kk + voff[0]), X1 = lds64(vb + 1024 * kk + voff[1]);
      const uint2 X2 = lds64(vb + 1024 * kk + voff[2]), X3 = lds64(vb + 1024 * kk + voff[3]);
      const uint32_t sv01 = e4m3x2_f16(lds_u8(vsb + 128 * kk + 8 * tv[0] + g) |
                                       (lds_u8(vsb + 128 * kk + 8 * tv[1] + g) << 8));
      const uint32_t sv23 = e4m3x2_f16(lds_u8(vsb + 128 * kk + 8 * tv[2] + g) |
                                       (lds_u8(vsb + 128 * kk + 8 * tv[3] + g) << 8));
#pragma unroll
      for (int u = 0; u < 2; ++u) {
        const uint32_t x0 = u ? X0.y : X0.x, x1 = u ? X1.y : X1.x, x2 = u ? X2.y : X2.x, x3 = u ? X3.y : X3.x;
        // bytes (token A nibble | token B nibble << 4) of the even and of the odd dimensions
        uint32_t e01[4], o01[4], e23[4], o23[4];
        e2m1x8_f16((x0 & 0x0F0F0F0Fu) | ((x1 << 4) & 0xF0F0F0F0u), e01);
        e2m1x8_f16(((x0 >> 4) & 0x0F0F0F0Fu) | (x1 & 0xF0F0F0F0u), o01);
        e2m1x8_f16((x2 & 0x0F0F0F0Fu) | ((x3 << 4) & 0xF0F0F0F0u), e23);
        e2m1x8_f16(((x2 >> 4) & 0x0F0F0F0Fu) | (x3 & 0xF0F0F0F0u), o23);
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const uint32_t a0 = hmul2(e01[k], sv01), a1 = hmul2(o01[k], sv01);
          const uint32_t a2 = hmul2(e23[k], sv23), a3 = hmul2(o23[k], sv23);
#pragma unroll
          for (int h = 0; h < kNH; ++h) mma_f16(oacc[4 * u + k][h], a0, a1, a2, a3, pb[kk][h][0], pb[kk][h][1]);
        }
      }
    }
    __syncwarp();  // the slot is read; refill it
    if (done + kStages < mine) issue(done + kStages);
  }
  if (!ok) {
    // a copy never landed: wait (bounded) for what this warp still has in flight before the ring
    // is reused and the CTA exits; the result is unspecified, the status word says why
    for (int n = done; n < min(mine, done + kStages); ++n)
      mbar_wait(bar0 + 8 * (n % kStages), static_cast<uint32_t>((n / kStages) & 1), a.status, kStatusTimeoutDrain);
  }
  cp_async_wait_all();

  // merge the four warps: row sums over the rows (g), then (max, sum, O) per warp in shared memory
#pragma unroll
  for (int h = 0; h < kNH; ++h)
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      l_run[h][e] += __shfl_xor_sync(0xFFFFFFFFu, l_run[h][e], 4);
      l_run[h][e] += __shfl_xor_sync(0xFFFFFFFFu, l_run[h][e], 8);
      l_run[h][e] += __shfl_xor_sync(0xFFFFFFFFu, l_run[h][e], 16);
    }
  __syncthreads();  // every warp is done with its ring: it becomes the merge area
  float* Osm = reinterpret_cast<float*>(smem_raw + (ring0 - raw));  // [warp][16 heads][128 dims]
  if (g == 0) {
#pragma unroll
    for (int h = 0; h < kNH; ++h)
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        msm[warp][8 * h + 2 * q + e] = m_run[h][e];
        lsm[warp][8 * h + 2 * q + e] = l_run[h][e];
      }
  }
#pragma unroll
  for (int m = 0; m < 8; ++m)
#pragma unroll
    for (int h = 0; h < kNH; ++h)
#pragma unroll
      for (int e = 0; e < 2; ++e)
        *reinterpret_cast<float2*>(Osm + (warp * 16 + 8 * h + 2 * q + e) * kHeadDim + 16 * g + 2 * m) =
            make_float2(oacc[m][h][e], oacc[m][h][2 + e]);
  __syncthreads();
  const float gv = __ldg(a.gv);
  for (int i = threadIdx.x; i < group * kHeadDim; i += kAttnThreads) {
    const int r = i / kHeadDim, d = i % kHeadDim;
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) M = fmaxf(M, msm[w][r]);
    float L = 0.0f, O = 0.0f;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) {
      const float f = msm[w][r] == -INFINITY ? 0.0f : exp2f(msm[w][r] - M);
      L += f * lsm[w][r];
      O += f * Osm[(w * 16 + r) * kHeadDim + d];
    }
    if (a.nsplit == 1) {
      const float y = L > 0.0f ? O / L * gv : 0.0f;
      a.out[(b * a.Hq + kvh * group + r) * kHeadDim + d] = static_cast<uint16_t>(f32_to_bf16_bits(y));
    } else {
      float* pr = a.part + ((bh * a.nsplit + blockIdx.x) * 16 + r) * kPartFloats;
      if (d == 0) {
        pr[0] = M;
        pr[1] = L;
      }
      pr[4 + d] = O;
    }
  }
}

// Merges the spans of every (sequence, query head): out = sum_s f_s O_s / sum_s f_s L_s * gv,
// f_s = exp2(M_s - max_s M_s); one warp per (sequence, query head), four dims per lane.
__global__ void __launch_bounds__(128) kv_attention_merge_kernel(const float* __restrict__ part, int64_t B,
                                                                 int64_t Hq, int64_t Hkv, int nsplit,
                                                                 const float* __restrict__ gvp,
                                                                 uint16_t* __restrict__ out) {
  griddep_wait();
  griddep_launch_dependents();
  const int64_t row = static_cast<int64_t>(blockIdx.x) * 4 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (row >= B * Hq) return;
  const int64_t b = row / Hq, h = row % Hq, group = Hq / Hkv, kvh = h / group, r = h % group;
  const float* base = part + ((b * Hkv + kvh) * nsplit * 16 + r) * kPartFloats;
  float M = -INFINITY;
  for (int s = 0; s < nsplit; ++s) M = fmaxf(M, base[s * 16 * kPartFloats]);
  float L = 0.0f, O[4] = {0.0f, 0.0f, 0.0f, 0.0f};
  for (int s = 0; s < nsplit; ++s) {
    const float* pr = base + s * 16 * kPartFloats;
    const float f = pr[0] == -INFINITY ? 0.0f : exp2f(pr[0] - M);
    L += f * pr[1];
    const float4 v = *reinterpret_cast<const float4*>(pr + 4 + 4 * lane);
    O[0] += f * v.x;
    O[1] += f * v.y;
    O[2] += f * v.z;
    O[3] += f * v.w;
  }
  const float gv = __ldg(gvp);
  const float inv = L > 0.0f ? gv / L : 0.0f;
  uint2 packed;
  packed.x = f32_to_bf16_bits(O[0] * inv) | (f32_to_bf16_bits(O[1] * inv) << 16);
  packed.y = f32_to_bf16_bits(O[2] * inv) | (f32_to_bf16_bits(O[3] * inv) << 16);
  *reinterpret_cast<uint2*>(out + row * kHeadDim + 4 * lane) = packed;
}

}  // namespace

int attention_splits(int64_t B, int64_t Hkv, int64_t Lmax) {
  const int64_t chunks = std::max<int64_t>(1, (Lmax + kTok - 1) / kTok);
  const int64_t want = (2 * kNumSMsHint + B * Hkv - 1) / (B * Hkv);  // few spans: a CTA's start-up is costly
  return static_cast<int>(std::max<int64_t>(1, std::min<int64_t>({chunks, want, 256})));
}

size_t attention_workspace_bytes(int64_t B, int64_t Hkv, int64_t Lmax) {
  const int ns = attention_splits(B, Hkv, Lmax);
  return ns == 1 ? 0 : static_cast<size_t>(B * Hkv) * ns * 16 * kPartFloats * sizeof(float);
}

nvfp4rl_status launch_kv_attention(const uint16_t* q, const uint8_t* kc, const uint8_t* ks, const float* gk,
                                   const uint8_t* vc, const uint8_t* vs, const float* gv, const int32_t* lens,
                                   int64_t B, int64_t Hq, int64_t Hkv, int64_t Lmax, float scale, uint16_t* out,
                                   void* workspace, const DeviceInfo& dev, cudaStream_t st) {
  if (B == 0) return NVFP4RL_OK;
  // TMA row coordinates are 32-bit: every cache row of a box, b Lmax + t + 63, must fit
  if (B * Lmax > static_cast<int64_t>(INT32_MAX) - kTok) return NVFP4RL_ERR_UNSUPPORTED_SHAPE;
  const int ns = attention_splits(B, Hkv, Lmax);
  const int64_t chunks = (Lmax + kTok - 1) / kTok;
  const int span = static_cast<int>((chunks + ns - 1) / ns) * kTok;
  // code rows as a [B Lmax][Hkv 64] byte array; a box is one head's 64-byte rows of 64 tokens
  CUtensorMap mk, mv;
  if (!make_tensor_map_2d(&mk, CU_TENSOR_MAP_DATA_TYPE_UINT8, kc, static_cast<uint64_t>(Hkv) * 64,
                          static_cast<uint64_t>(B * Lmax), 1, 64, kTok, CU_TENSOR_MAP_SWIZZLE_64B) ||
      !make_tensor_map_2d(&mv, CU_TENSOR_MAP_DATA_TYPE_UINT8, vc, static_cast<uint64_t>(Hkv) * 64,
                          static_cast<uint64_t>(B * Lmax), 1, 64, kTok, CU_TENSOR_MAP_SWIZZLE_64B))
    return NVFP4RL_ERR_CUDA;
  AttnArgs a{q, ks, vs, gk, gv, lens, Hq, Hkv, Lmax, ns, span, scale, out, static_cast<float*>(workspace),
             dev.status};
  const bool wide = Hq / Hkv > 8;
  {
    static std::mutex mu;
    static std::map<int, bool> set;
    std::lock_guard<std::mutex> lock(mu);
    if (!set[dev.device]) {
      if (cudaFuncSetAttribute(kv_attention_kernel<1>, cudaFuncAttributeMaxDynamicSharedMemorySize, kAttnSmem) !=
              cudaSuccess ||
          cudaFuncSetAttribute(kv_attention_kernel<2>, cudaFuncAttributeMaxDynamicSharedMemorySize, kAttnSmem) !=
              cudaSuccess)
        return NVFP4RL_ERR_CUDA;
      set[dev.device] = true;
    }
  }
  const dim3 grid(static_cast<unsigned>(ns), static_cast<unsigned>(B * Hkv));
  const cudaError_t e = wide ? launch_pdl(kv_attention_kernel<2>, grid, dim3(kAttnThreads), kAttnSmem, st, mk, mv, a)
                             : launch_pdl(kv_attention_kernel<1>, grid, dim3(kAttnThreads), kAttnSmem, st, mk, mv, a);
  if (e != cudaSuccess) return NVFP4RL_ERR_CUDA;
  if (launch_status() != NVFP4RL_OK) return NVFP4RL_ERR_CUDA;
  if (ns == 1) return NVFP4RL_OK;
  if (launch_pdl(kv_attention_merge_kernel, dim3(static_cast<unsigned>((B * Hq + 3) / 4)), dim3(128), 0, st,
                 static_cast<const float*>(workspace), B, Hq, Hkv, ns, gv, out) != cudaSuccess)
    return NVFP4RL_ERR_CUDA;
  return launch_status();
}

}  // namespace nvfp4rl
