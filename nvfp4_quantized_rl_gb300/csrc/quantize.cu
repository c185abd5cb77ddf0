// NVFP4 block quantization: plain, rollout-guided, recorded and cached (sm_103a).
//
// Format: QeRL explainer, section "NVFP4量子化とLoRA" (4-bit weights with hardware
// support); TRACE summary, section "仕組みの工学的な理解" (a few values share one
// scale, each value is 4 bits; the rounding direction is a per-value choice between
// the two neighbouring grid points). Recipe: g = fl32(amax / 2688); the 16-element
// block scale is the E4M3 byte nearest to bamax / (6 g); each element's code is the
// E2M1 grid index nearest to |x| / (E4M3(s) g) with its sign in bit 3; both roundings
// apply to the exact real quotient, ties to the even encoding, saturating.
//
// Kernels:
//   amax_kernel, amax_bulk_kernel  the tensor amax (grid-stride 128-bit loads, or for large
//                    tensors a cp.async.bulk ring per SM), one atomicMax per CTA.
//   Four modes: plain, guided (a mask picks the rounding direction), record (plain, plus one
//   rounding-direction bit per element: TRACE's rollout side), cached (guided against given scale
//   bytes and g, one pass: TRACE's training side).
//   encode_ring_kernel  bf16 input, every mode: a cp.async.bulk ring per CTA feeds encode warps
//                    that take the codes from the hardware E2M1 conversion of x times a reciprocal
//                    of the scale, chosen per scale byte so that the result is exact (else the
//                    compare form below for that byte's blocks).
//   quantize_kernel  fp32 input: one thread per 16-element block (two blocks in flight per
//                    thread), per-block thresholds and integer compares.
//   encode_amax_ring_kernel  the weight refresh: one tensor's encoding while the next tensor's
//                    amax streams through a shared-memory ring.
//   rmsnorm_quant_kernel  RMSNorm-AQN and the quantization of its output in one cooperative
//                    kernel, the normalized rows kept in shared memory across a grid barrier.
//   kv_append_kernel one decode step's K/V rows encoded at a given g into an NVFP4 KV cache.
//
// Exactness without division per element: for an fp32 value a and a real P,
//   a > P  <=>  a > RD(P)      a >= P  <=>  a >= RU(P)
// where RD/RU are P rounded down/up to fp32. Every P used here is T * dec(s) * g
// with T * dec(s) exact in fp32 (at most 7 significant bits), so RD/RU are single
// directed-rounding multiplies (__fmul_rd / __fmul_ru). Non-negative fp32 values
// order like their bit patterns, so the compares run on integers.
#include <map>
#include <type_traits>
#include <mutex>
#include <vector>

#include "common.cuh"
#include "sm100.cuh"

namespace nvfp4rl {
namespace {

using namespace sm100;

// Approximate E4M3 byte of v (round to nearest, saturating): a starting point that is
// within one byte of the exact answer; the caller corrects it exactly.
__device__ __forceinline__ uint32_t e4m3_estimate(float v) {
  uint16_t pair;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %1;" : "=h"(pair) : "f"(v));
  return pair & 0x7Fu;
}

// Exact E4M3 byte nearest to bamax / (6 g), ties to the even byte, saturating at 0x7E.
// g > 0. `est` is a fp32 approximation of the quotient.
__device__ __forceinline__ uint32_t scale_byte(float bamax, float g, float est) {
  uint32_t b = e4m3_estimate(est);
  uint32_t dec = 0, inc = 0;
  if (b > 0) {
    // 6 * midpoint(b-1, b) = 3 * (E4M3(b-1) + E4M3(b)), exact in fp32
    const float t = 3.0f * (e4m3_decode_pos(b - 1) + e4m3_decode_pos(b));
    const float ru = __fmul_ru(t, g), rd = __fmul_rd(t, g);
    if (bamax < ru) dec = 1;
    else if (rd == ru && bamax == ru && (b & 1u)) dec = 1;  // exact tie: to the even byte b-1
  }
  if (b < 0x7Eu) {
    const float t = 3.0f * (e4m3_decode_pos(b) + e4m3_decode_pos(b + 1));
    const float ru = __fmul_ru(t, g), rd = __fmul_rd(t, g);
    if (bamax > rd) inc = 1;
    else if (rd == ru && bamax == rd && (b & 1u)) inc = 1;  // exact tie: to the even byte b+1
  }
  return b - dec + inc;
}

// Strict-compare thresholds (fp32 bit patterns) of the seven E2M1 midpoints for the real
// scale S = dec * g: |x| bits > th[i] exactly when |x| rounds above midpoint i.
// Midpoints 0.25, 1.25, 2.5 and 5 round down on a tie (to the even code below),
// 0.75, 1.75 and 3.5 round up on a tie (to the even code above).
__device__ __forceinline__ void plain_thresholds(float dec, float g, uint32_t th[7]) {
  th[0] = __float_as_uint(__fmul_rd(0.25f * dec, g));
  th[1] = __float_as_uint(__fmul_ru(0.75f * dec, g)) - 1u;
  th[2] = __float_as_uint(__fmul_rd(1.25f * dec, g));
  th[3] = __float_as_uint(__fmul_ru(1.75f * dec, g)) - 1u;
  th[4] = __float_as_uint(__fmul_rd(2.5f * dec, g));
  th[5] = __float_as_uint(__fmul_ru(3.5f * dec, g)) - 1u;
  th[6] = __float_as_uint(__fmul_rd(5.0f * dec, g));
}

// Guided thresholds at the grid points 0.5 .. 6 (k = 1..7):
//   ge[k-1]: |x| bits > ge  <=>  |x| >= grid[k] S      gt[k-1]: |x| bits > gt  <=>  |x| > grid[k] S
__device__ __forceinline__ void guided_thresholds(float dec, float g, uint32_t ge[7], uint32_t gt[7]) {
  const float grid[7] = {0.5f, 1.0f, 1.5f, 2.0f, 3.0f, 4.0f, 6.0f};
#pragma unroll
  for (int k = 0; k < 7; ++k) {
    ge[k] = __float_as_uint(__fmul_ru(grid[k] * dec, g)) - 1u;
    gt[k] = __float_as_uint(__fmul_rd(grid[k] * dec, g));
  }
}

// Encoding modes.
enum : int {
  kModePlain = 0,   // nvfp4_quantize
  kModeGuided = 1,  // nvfp4_quantize_guided: rounding directions from a mask
  kModeRecord = 2,  // nvfp4_quantize_record: plain, and the record of its rounding directions
  kModeCached = 3,  // nvfp4_quantize_cached: guided, against given scale bytes and g
};

// Two 16-bit maxima of |bf16| bit patterns over the eight values of a 128-bit word (the sign
// bits are cleared before the unsigned compares).
__device__ __forceinline__ uint32_t max4_abs_bf16(uint4 v) {
  return __vmaxu2(__vmaxu2(v.x & 0x7FFF7FFFu, v.y & 0x7FFF7FFFu), __vmaxu2(v.z & 0x7FFF7FFFu, v.w & 0x7FFF7FFFu));
}

template <int kDtype>
__global__ void __launch_bounds__(256) amax_kernel(const void* __restrict__ x, int64_t nvec,
                                                   uint32_t* __restrict__ amax_bits) {
  griddep_wait();
  griddep_launch_dependents();
  uint32_t m = 0;
  const uint4* p = static_cast<const uint4*>(x);
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  const int64_t first = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  // main loop: four 128-bit loads in flight per thread, no bounds test per load; then the tail
  int64_t i = first;
  if (kDtype == NVFP4RL_BF16) {
    uint32_t m2 = 0;  // two running 16-bit maxima of |bf16| bit patterns
    for (; i + 3 * stride < nvec; i += 4 * stride) {
      const uint4 v0 = ld_nc_v4(p + i), v1 = ld_nc_v4(p + i + stride);
      const uint4 v2 = ld_nc_v4(p + i + 2 * stride), v3 = ld_nc_v4(p + i + 3 * stride);
      m2 = __vmaxu2(m2, max4_abs_bf16(v0));
      m2 = __vmaxu2(m2, max4_abs_bf16(v1));
      m2 = __vmaxu2(m2, max4_abs_bf16(v2));
      m2 = __vmaxu2(m2, max4_abs_bf16(v3));
    }
    for (; i < nvec; i += stride) {
      const uint4 v = ld_nc_v4(p + i);
      m2 = __vmaxu2(m2, max4_abs_bf16(v));
    }
    m = max(m2 & 0xFFFFu, m2 >> 16) << 16;
  } else {
    for (; i + 3 * stride < nvec; i += 4 * stride) {
      const uint4 v0 = ld_nc_v4(p + i), v1 = ld_nc_v4(p + i + stride);
      const uint4 v2 = ld_nc_v4(p + i + 2 * stride), v3 = ld_nc_v4(p + i + 3 * stride);
      m = max(m, max(max(v0.x & 0x7FFFFFFFu, v0.y & 0x7FFFFFFFu), max(v0.z & 0x7FFFFFFFu, v0.w & 0x7FFFFFFFu)));
      m = max(m, max(max(v1.x & 0x7FFFFFFFu, v1.y & 0x7FFFFFFFu), max(v1.z & 0x7FFFFFFFu, v1.w & 0x7FFFFFFFu)));
      m = max(m, max(max(v2.x & 0x7FFFFFFFu, v2.y & 0x7FFFFFFFu), max(v2.z & 0x7FFFFFFFu, v2.w & 0x7FFFFFFFu)));
      m = max(m, max(max(v3.x & 0x7FFFFFFFu, v3.y & 0x7FFFFFFFu), max(v3.z & 0x7FFFFFFFu, v3.w & 0x7FFFFFFFu)));
    }
    for (; i < nvec; i += stride) {
      const uint4 v = ld_nc_v4(p + i);
      m = max(m, max(max(v.x & 0x7FFFFFFFu, v.y & 0x7FFFFFFFu), max(v.z & 0x7FFFFFFFu, v.w & 0x7FFFFFFFu)));
    }
  }
  m = __reduce_max_sync(0xFFFFFFFFu, m);
  __shared__ uint32_t red[8];
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = m;
  __syncthreads();
  if (threadIdx.x < 32) {
    m = threadIdx.x < (blockDim.x >> 5) ? red[threadIdx.x] : 0u;
    m = __reduce_max_sync(0xFFFFFFFFu, m);
    if (threadIdx.x == 0) atomicMax(amax_bits, m);
  }
}

// amax through the bulk-copy engine: one CTA per SM; lane 0 of warp 0 streams 16 KB chunks
// (chunk blockIdx.x, then every gridDim.x-th) into a ring of shared-memory stages with
// cp.async.bulk; four warps reduce each chunk from shared memory. Twelve stages keep 192 KB
// in flight per SM with a single issuing thread.
constexpr int kAmaxChunk = 16384;
constexpr int kAmaxStages = 12;
constexpr int kAmaxWarps = 4;
constexpr int kAmaxSmem = kAmaxChunk * kAmaxStages;

template <int kDtype>
__global__ void __launch_bounds__(32 * (kAmaxWarps + 1), 1)
    amax_bulk_kernel(const uint8_t* __restrict__ x, int64_t bytes, uint32_t* __restrict__ amax_bits,
                     uint32_t* __restrict__ status) {
  griddep_wait();
  griddep_launch_dependents();
  extern __shared__ __align__(128) uint8_t ring[];
  __shared__ uint64_t full[kAmaxStages], empty[kAmaxStages];
  __shared__ uint32_t red[kAmaxWarps];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t nchunks = (bytes + kAmaxChunk - 1) / kAmaxChunk;
  const int64_t mine = blockIdx.x < nchunks ? (nchunks - 1 - blockIdx.x) / gridDim.x + 1 : 0;
  if (threadIdx.x == 0) {
    for (int i = 0; i < kAmaxStages; ++i) {
      mbar_init(smem_addr(&full[i]), 1);
      mbar_init(smem_addr(&empty[i]), kAmaxWarps);
    }
    fence_barrier_init();
  }
  __syncthreads();
  uint32_t m = 0;
  if (warp == 0) {
    if (lane == 0) {
      int64_t issued = 0;
      for (int64_t j = 0; j < mine; ++j) {
        const int s = static_cast<int>(j % kAmaxStages);
        if (!mbar_wait(smem_addr(&empty[s]), static_cast<uint32_t>((j / kAmaxStages) & 1) ^ 1u, status,
                       kStatusTimeoutProducer))
          break;
        const int64_t off = (blockIdx.x + j * gridDim.x) * static_cast<int64_t>(kAmaxChunk);
        const uint32_t size = static_cast<uint32_t>(min(static_cast<int64_t>(kAmaxChunk), bytes - off));
        mbar_arrive_expect_tx(smem_addr(&full[s]), size);
        bulk_load(smem_addr(ring + s * kAmaxChunk), x + off, size, smem_addr(&full[s]));
        issued = j + 1;
      }
      // every issued copy has landed before the CTA exits
      for (int64_t j = max(int64_t(0), issued - kAmaxStages); j < issued; ++j)
        mbar_wait(smem_addr(&full[j % kAmaxStages]), static_cast<uint32_t>((j / kAmaxStages) & 1), status,
                  kStatusTimeoutDrain);
    }
  } else {
    const int t = threadIdx.x - 32;
    uint32_t m2 = 0;
    for (int64_t j = 0; j < mine; ++j) {
      const int s = static_cast<int>(j % kAmaxStages);
      if (!__all_sync(0xFFFFFFFFu, mbar_wait(smem_addr(&full[s]), static_cast<uint32_t>((j / kAmaxStages) & 1), status,
                                             kStatusTimeoutDequant)))
        break;
      const int64_t off = (blockIdx.x + j * gridDim.x) * static_cast<int64_t>(kAmaxChunk);
      const int nvec = static_cast<int>(min(static_cast<int64_t>(kAmaxChunk), bytes - off) / 16);
      const uint4* v = reinterpret_cast<const uint4*>(ring + s * kAmaxChunk);
#pragma unroll 8
      for (int i = t; i < nvec; i += 32 * kAmaxWarps) {
        const uint4 w = v[i];
        if (kDtype == NVFP4RL_BF16) {
          m2 = __vmaxu2(m2, max4_abs_bf16(w));
        } else {
          m = max(m, max(max(w.x & 0x7FFFFFFFu, w.y & 0x7FFFFFFFu), max(w.z & 0x7FFFFFFFu, w.w & 0x7FFFFFFFu)));
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_addr(&empty[s]));
    }
    if (kDtype == NVFP4RL_BF16) m = max(m2 & 0xFFFFu, m2 >> 16) << 16;
    m = __reduce_max_sync(0xFFFFFFFFu, m);
    if (lane == 0) red[warp - 1] = m;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    uint32_t r = 0;
    for (int i = 0; i < kAmaxWarps; ++i) r = max(r, red[i]);
    atomicMax(amax_bits, r);
  }
}

// Raw 128-bit words of one 16-element block: 2 (bf16) or 4 (fp32).
template <int kDtype>
struct BlockWords {
  uint4 v[kDtype == NVFP4RL_BF16 ? 2 : 4];
};

template <int kDtype>
__device__ __forceinline__ void load_block(const void* __restrict__ x, int64_t blk, BlockWords<kDtype>& w) {
  const uint4* p = reinterpret_cast<const uint4*>(static_cast<const uint8_t*>(x) +
                                                  blk * 16 * (kDtype == NVFP4RL_BF16 ? 2 : 4));
#pragma unroll
  for (int q = 0; q < (kDtype == NVFP4RL_BF16 ? 2 : 4); ++q) w.v[q] = ld_nc_v4(p + q);
}

__device__ __forceinline__ uint32_t bf16x2_gt(uint32_t a, uint32_t b) {  // per half: 1.0 if a > b else 0.0
  uint32_t d;
  asm("set.gt.bf16x2.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}

// Four code bytes from eight fp32 values (y[2i] the low nibble of byte i): E2M1 codes by the
// hardware conversion (round to nearest, ties to even, saturating; the sign of zero kept).
__device__ __forceinline__ uint32_t e2m1_word(const float (&y)[8]) {
  uint32_t d;
  asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b0, %2, %1;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b1, %4, %3;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b2, %6, %5;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b3, %8, %7;\n\t"
      "mov.b32 %0, {b0, b1, b2, b3};\n\t}"
      : "=r"(d)
      : "f"(y[0]), "f"(y[1]), "f"(y[2]), "f"(y[3]), "f"(y[4]), "f"(y[5]), "f"(y[6]), "f"(y[7]));
  return d;
}

__device__ __forceinline__ uint32_t bf16x2_add(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("add.rn.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}

// bf16 pattern of the largest bf16 <= v (v >= 0 finite fp32): truncation.
__device__ __forceinline__ uint32_t bf16_rd(float v) { return __float_as_uint(v) >> 16; }
// bf16 pattern of the smallest bf16 >= v (v >= 0 finite fp32).
__device__ __forceinline__ uint32_t bf16_ru(float v) { return (__float_as_uint(v) + 0xFFFFu) >> 16; }

// bar.sync on a named barrier among `threads` threads (whole warps) of the CTA.
__device__ __forceinline__ void named_barrier_sync(int id, int threads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(threads) : "memory");
}

// Per-tensor lookup tables for the bf16 plain encoding, built in shared memory by every CTA
// (they depend only on g):
//   mid[i]  = (RD, RU) of 3 g (E4M3(i) + E4M3(i + 1)): six times the midpoint between scale
//             bytes i and i + 1, rounded down and up (i = 0 .. 0x7D), for the exact scale byte;
//   thr[b]  = for scale byte b, the seven element thresholds as bf16 patterns in both halves of a
//             word, ready for the two-element compares (b = 0: +inf);
//   rcp[b]  = a reciprocal of E4M3(b) g with which the hardware conversion of fl32(x) * rcp[b] to
//             E2M1 gives every element's exact code (cvt_reciprocal), else -1; 0 for a zero scale.
struct EncodeTables {
  float2 mid[0x7E];
  uint4 thr[0x7F][2];
  float rcp[0x7F];
};

// A reciprocal r of d = E4M3(b) g for the conversion forms of the encodings, or -1.
// cvt.rn.satfinite.e2m1x2 rounds y = fl32(x r) to E2M1 (nearest, ties to the even code,
// saturating at 6), which is the exact rounding of |x|/d unless y and x/d fall on different sides
// of a midpoint m (or y lands on m while x/d does not). With r within 3.5 fp32 ulps of 1/d, y is
// within 2^-21.2 of x/d (relative), so only a bf16 x within 2^-20 of m d can be misrounded, and
// there is at most one such bf16 value B per midpoint (their spacing is 2^-8 relative). All in
// fp32: m d = ph + pl exactly (an FMA gives the product's rounding error), so for each such B the
// exact side of m d it lies on (above, below, or on it: then the even code) is known, and
// fl32(B r) is one multiply; r is taken as RN(1/fl32(d)) or one of its four nearest fp32
// neighbours, the first for which every such B goes to its exact side. With `grid` the seven grid
// points G (0.5 .. 6) are checked the same way, strictly: y must lie on the side of G that x/d lies
// on and never on G itself, and a bf16 value exactly on G d rejects the byte; then y is on the
// grid only for x = 0. `mids` false skips the midpoints (the guided encodings need only the grid
// points). Zero scale (b = 0, or g not positive): 0, so x 0 = +-0 and every code is sign|0, as the
// compares give.
__device__ float cvt_reciprocal(int b, float g, bool mids = true, bool grid = false) {
  if (b == 0 || !(g > 0.0f)) return 0.0f;
  const float dec = e4m3_decode_pos(b);
  const float dh = __fmul_rn(dec, g);
  if (!(dh > 0x1p-120f) || !(dh <= 0x1.fffffep127f)) return -1.0f;  // 1/d near the fp32 range: the compare form
  const float r0 = __frcp_rn(dh);
  // points 0-6: the midpoints (a tie goes to the even code: up at odd k); 7-13: the grid points
  const float pts[14] = {0.25f, 0.75f, 1.25f, 1.75f, 2.5f, 3.5f, 5.0f, 0.5f, 1.0f, 1.5f, 2.0f, 3.0f, 4.0f, 6.0f};
  float B[14];
  bool near[14], up[14];
#pragma unroll
  for (int k = 0; k < 14; ++k) {
    near[k] = false;
    B[k] = 0.0f;
    up[k] = false;
    if (k < 7 ? !mids : !grid) continue;
    const float md = pts[k] * dec;  // exact: at most 7 significant bits
    const float ph = __fmul_rn(md, g), pl = __fmaf_rn(md, g, -ph);
    const uint32_t t = __float_as_uint(ph) & 0xFFFF0000u;  // the bf16 grid points around m d
    const float lo = __uint_as_float(t), hi = __uint_as_float(t + 0x10000u);
    const float dlo = (lo - ph) - pl, dhi = (hi - ph) - pl;  // B - m d, with its exact sign
    const float tol = 0x1p-20f * ph;
    near[k] = fabsf(dlo) <= tol || fabsf(dhi) <= tol;
    B[k] = fabsf(dlo) <= tol ? lo : hi;
    const float dB = fabsf(dlo) <= tol ? dlo : dhi;
    if (k >= 7 && near[k] && dB == 0.0f) return -1.0f;  // a bf16 value on a grid point
    up[k] = dB > 0.0f || (dB == 0.0f && (k & 1));  // exact side; a midpoint tie at odd k goes up to the even code
  }
  const int step[5] = {0, -1, 1, -2, 2};
#pragma unroll 1
  for (int i = 0; i < 5; ++i) {
    const float r = __uint_as_float(__float_as_uint(r0) + step[i]);
    bool ok = true;
#pragma unroll
    for (int k = 0; k < 14; ++k) {
      const float y = __fmul_rn(B[k], r);
      const bool side = k < 7 ? (y > pts[k] || (y == pts[k] && (k & 1))) : y > pts[k];
      ok = ok && (!near[k] || (side == up[k] && (k < 7 || y != pts[k])));
    }
    if (ok) return r;
  }
  return -1.0f;
}

__device__ void build_encode_tables(EncodeTables& t, float g, bool with_rcp, int tid, int nthreads) {
  for (int i = tid; i < 0x7E; i += nthreads) {
    const float m3 = 3.0f * (e4m3_decode_pos(i) + e4m3_decode_pos(i + 1));  // exact in fp32
    t.mid[i] = make_float2(__fmul_rd(m3, g), __fmul_ru(m3, g));
  }
  for (int b = tid; b < 0x7F; b += nthreads) {
    uint32_t tk[8];
    if (b == 0 || !(g > 0.0f)) {
#pragma unroll
      for (int k = 0; k < 8; ++k) tk[k] = 0x7F807F80u;  // zero scale: every code is sign|0
    } else {
      const float dec = e4m3_decode_pos(b);
      const uint32_t t[7] = {bf16_rd(__fmul_rd(0.25f * dec, g)), bf16_ru(__fmul_ru(0.75f * dec, g)) - 1u,
                             bf16_rd(__fmul_rd(1.25f * dec, g)), bf16_ru(__fmul_ru(1.75f * dec, g)) - 1u,
                             bf16_rd(__fmul_rd(2.5f * dec, g)),  bf16_ru(__fmul_ru(3.5f * dec, g)) - 1u,
                             bf16_rd(__fmul_rd(5.0f * dec, g))};
#pragma unroll
      for (int k = 0; k < 7; ++k) tk[k] = t[k] | (t[k] << 16);
      tk[7] = 0u;
    }
    t.thr[b][0] = make_uint4(tk[0], tk[1], tk[2], tk[3]);
    t.thr[b][1] = make_uint4(tk[4], tk[5], tk[6], tk[7]);
    t.rcp[b] = with_rcp ? cvt_reciprocal(b, g) : -1.0f;
  }
}

// Per-tensor tables of the guided, record and cached bf16 encodings, built in shared memory by
// every CTA: mid as in EncodeTables (the scale byte; not built for cached), and rcp[b] a reciprocal
// of E4M3(b) g checked against the grid points (and for the record against the midpoints too)
// by cvt_reciprocal, else -1 (those scale bytes take the compare form).
struct ModeTables {
  float2 mid[0x7E];
  float rcp[0x7F];
};

__device__ void build_mode_tables(ModeTables& t, float g, bool with_mid, bool mids, int tid, int nthreads) {
  if (with_mid) {
    for (int i = tid; i < 0x7E; i += nthreads) {
      const float m3 = 3.0f * (e4m3_decode_pos(i) + e4m3_decode_pos(i + 1));  // exact in fp32
      t.mid[i] = make_float2(__fmul_rd(m3, g), __fmul_ru(m3, g));
    }
  }
  for (int b = tid; b < 0x7F; b += nthreads) t.rcp[b] = cvt_reciprocal(b, g, mids, true);
}

// Exact E4M3 scale byte of bamax / (6 g) from the estimate `est` and the midpoint table: the
// same decision as scale_byte, with the midpoint products looked up instead of computed.
template <class Tables>
__device__ __forceinline__ uint32_t scale_byte_tab(float bamax, float est, const Tables& t) {
  const uint32_t b = min(e4m3_estimate(est), 0x7Eu);
  uint32_t dec = 0, inc = 0;
  if (b > 0) {
    const float2 m = t.mid[b - 1];
    if (bamax < m.y) dec = 1;
    else if (m.x == m.y && bamax == m.y && (b & 1u)) dec = 1;  // exact tie: to the even byte b-1
  }
  if (b < 0x7Eu) {
    const float2 m = t.mid[b];
    if (bamax > m.x) inc = 1;
    else if (m.x == m.y && bamax == m.x && (b & 1u)) inc = 1;  // exact tie: to the even byte b+1
  }
  return b - dec + inc;
}

// The compare form of the plain bf16 encoding (scale byte b already chosen): for bf16 x and a real
// P, x > P <=> x > RD_bf16(P) and x >= P <=> x > pred(RU_bf16(P)), with RD_bf16(P) =
// RD_bf16(RD_fp32(P)) and RU_bf16(P) = RU_bf16(RU_fp32(P)); so the seven midpoint thresholds
// become bf16 values compared with set.gt.bf16x2, and the magnitude code is the number of
// thresholds exceeded, accumulated with add.bf16x2 on 128.0 (128 + c is exact and its low
// three bits are c). Taken for the blocks the conversion form cannot round exactly (rare);
// not inlined, so the common form's warps branch around it.
__device__ __noinline__ void encode_block_bf16_compare(uint4 v0, uint4 v1, int64_t blk, uint32_t b,
                                                       const EncodeTables& tab, uint8_t* __restrict__ codes,
                                                       uint8_t* __restrict__ scales) {
  const uint32_t w[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
  const uint4 ta = tab.thr[b][0], tb = tab.thr[b][1];
  const uint32_t T2[7] = {ta.x, ta.y, ta.z, ta.w, tb.x, tb.y, tb.z};
  uint32_t byte[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const uint32_t aw = w[i] & 0x7FFF7FFFu;
    uint32_t acc = 0x43004300u;  // bf16x2 (128, 128)
#pragma unroll
    for (int k = 0; k < 7; ++k) acc = bf16x2_add(acc, bf16x2_gt(aw, T2[k]));
    const uint32_t m = acc & 0x00070007u;
    const uint32_t s = w[i] & 0x80008000u;
    // low byte: magnitude of element 2i in bits 0-2, its sign in bit 3, element 2i+1 in bits 4-7
    byte[i] = m | (m >> 12) | (s >> 12) | (s >> 24);
  }
  const uint32_t lo = __byte_perm(__byte_perm(byte[0], byte[1], 0x0040), __byte_perm(byte[2], byte[3], 0x0040), 0x5410);
  const uint32_t hi = __byte_perm(__byte_perm(byte[4], byte[5], 0x0040), __byte_perm(byte[6], byte[7], 0x0040), 0x5410);
  *reinterpret_cast<uint2*>(codes + blk * 8) = make_uint2(lo, hi);
  scales[blk] = static_cast<uint8_t>(b);
}

// Plain encoding of one block of bf16 values: the exact scale byte from the block amax, then the
// codes by the hardware conversion of fl32(x) / (E4M3(s) g) where cvt_reciprocal shows that
// exact, else by the compare form. The scale byte's midpoint products come from the per-tensor
// tables in shared memory.
__device__ __forceinline__ void encode_block_bf16(const uint4 (&v)[2], int64_t blk, float g, float inv_g6,
                                                  float est_scale, const EncodeTables& tab,
                                                  uint8_t* __restrict__ codes, uint8_t* __restrict__ scales) {
  const uint32_t w[8] = {v[0].x, v[0].y, v[0].z, v[0].w, v[1].x, v[1].y, v[1].z, v[1].w};
  uint32_t m2 = 0;
#pragma unroll
  for (int i = 0; i < 8; ++i) m2 = __vmaxu2(m2, w[i] & 0x7FFF7FFFu);
  const uint32_t bamax_bits = max(m2 & 0xFFFFu, m2 >> 16);
  const float bamax = __uint_as_float(bamax_bits << 16);
  uint32_t b = 0;
  if (g > 0.0f) b = scale_byte_tab(bamax, (bamax * est_scale) * inv_g6, tab);
  const float rcp = tab.rcp[b];
  if (!(rcp >= 0.0f && bamax_bits < 0x7F80u)) {
    encode_block_bf16_compare(v[0], v[1], blk, b, tab, codes, scales);
    return;
  }
  uint32_t out[2];
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    float y[8];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      y[2 * i] = __fmul_rn(__uint_as_float(w[4 * h + i] << 16), rcp);
      y[2 * i + 1] = __fmul_rn(__uint_as_float(w[4 * h + i] & 0xFFFF0000u), rcp);
    }
    out[h] = e2m1_word(y);
  }
  *reinterpret_cast<uint2*>(codes + blk * 8) = make_uint2(out[0], out[1]);
  scales[blk] = static_cast<uint8_t>(b);
}

// Scale byte and codes of one block, written to scales[blk] and codes[8 blk .. 8 blk + 7], with
// exact integer compares of fp32 bit patterns against per-block thresholds. kModeRecord also writes
// the block's 16 rounding-direction bits to record16[blk]; kModeCached takes the scale byte from
// scales_in[blk] (above 0x7E read as 0x7E; 0 when g is not positive) and writes none.
template <int kDtype, int kMode>
__device__ __forceinline__ void encode_block(const BlockWords<kDtype>& w, int64_t blk, float g, float est_scale,
                                             float g6, const uint32_t* __restrict__ mask,
                                             uint8_t* __restrict__ codes, uint8_t* __restrict__ scales,
                                             uint16_t* __restrict__ record16, const uint8_t* __restrict__ scales_in) {
  constexpr bool kGuided = kMode == kModeGuided || kMode == kModeCached;
  uint32_t ax[16];
  uint32_t sgn = 0;
  if (kDtype == NVFP4RL_BF16) {
    const uint32_t words[8] = {w.v[0].x, w.v[0].y, w.v[0].z, w.v[0].w, w.v[1].x, w.v[1].y, w.v[1].z, w.v[1].w};
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const uint32_t lo = words[i] << 16, hi = words[i] & 0xFFFF0000u;
      ax[2 * i] = lo & 0x7FFFFFFFu;
      ax[2 * i + 1] = hi & 0x7FFFFFFFu;
      sgn |= ((lo >> 31) << (2 * i)) | ((hi >> 31) << (2 * i + 1));
    }
  } else {
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const uint32_t words[4] = {w.v[q].x, w.v[q].y, w.v[q].z, w.v[q].w};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        ax[4 * q + i] = words[i] & 0x7FFFFFFFu;
        sgn |= (words[i] >> 31) << (4 * q + i);
      }
    }
  }
  uint32_t mx = 0;
#pragma unroll
  for (int i = 0; i < 16; ++i) mx = max(mx, ax[i]);
  const float bamax = __uint_as_float(mx);

  uint32_t b = 0;
  if (kMode == kModeCached) {
    if (g > 0.0f) b = min(static_cast<uint32_t>(scales_in[blk]), 0x7Eu);
  } else if (g > 0.0f) {
    b = scale_byte(bamax, g, __fdiv_rn(bamax * est_scale, g6));
  }
  const float dec = e4m3_decode_pos(b);

  uint32_t lo32 = 0, hi32 = 0;
  if (!kGuided) {
    uint32_t th[7], ge[7], gt[7];
    plain_thresholds(dec, g, th);
    if (kMode == kModeRecord) guided_thresholds(dec, g, ge, gt);
    if (b == 0) {
#pragma unroll
      for (int k = 0; k < 7; ++k) th[k] = ge[k] = 0x7F800000u;  // zero scale: every code is sign|0
    }
    uint32_t bits = 0;
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      uint32_t mag = 0;
#pragma unroll
      for (int k = 0; k < 7; ++k) mag += ax[i] > th[k] ? 1u : 0u;
      if (kMode == kModeRecord) {
        uint32_t c_ge = 0;  // grid points at or below |x|: the plain magnitude is c_ge or c_ge + 1
#pragma unroll
        for (int k = 0; k < 7; ++k) c_ge += ax[i] > ge[k] ? 1u : 0u;
        bits |= (mag - c_ge) << i;
      }
      const uint32_t code = mag | (((sgn >> i) & 1u) << 3);
      if (i < 8) lo32 |= code << (4 * i);
      else hi32 |= code << (4 * (i - 8));
    }
    if (kMode == kModeRecord) record16[blk] = static_cast<uint16_t>(bits);
  } else {
    uint32_t ge[7], gt[7];
    guided_thresholds(dec, g, ge, gt);
    const uint32_t up_bits = (mask[blk >> 1] >> ((blk & 1) * 16)) & (b ? 0xFFFFu : 0u);
    if (b == 0) {
#pragma unroll
      for (int k = 0; k < 7; ++k) ge[k] = gt[k] = 0x7F800000u;
    }
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      uint32_t c_ge = 0, c_gt = 0;
#pragma unroll
      for (int k = 0; k < 7; ++k) {
        c_ge += ax[i] > ge[k] ? 1u : 0u;
        c_gt += ax[i] > gt[k] ? 1u : 0u;
      }
      const bool on_grid = (c_ge != c_gt) || ax[i] == 0u;
      const uint32_t up = (up_bits >> i) & 1u;
      const uint32_t mag = (c_ge == 7u) ? 7u : c_ge + ((up && !on_grid) ? 1u : 0u);
      const uint32_t code = mag | (((sgn >> i) & 1u) << 3);
      if (i < 8) lo32 |= code << (4 * i);
      else hi32 |= code << (4 * (i - 8));
    }
  }
  *reinterpret_cast<uint2*>(codes + blk * 8) = make_uint2(lo32, hi32);
  if (kMode != kModeCached) scales[blk] = static_cast<uint8_t>(b);
}

// Four code bytes (two E2M1 codes each, low nibble first) -> four f16x2 grid values (low half =
// low nibble).
__device__ __forceinline__ void e2m1x8_to_f16x2(uint32_t w, uint32_t (&d)[4]) {
  asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\t"
      "mov.b32 {b0, b1, b2, b3}, %4;\n\t"
      "cvt.rn.f16x2.e2m1x2 %0, b0;\n\t"
      "cvt.rn.f16x2.e2m1x2 %1, b1;\n\t"
      "cvt.rn.f16x2.e2m1x2 %2, b2;\n\t"
      "cvt.rn.f16x2.e2m1x2 %3, b3;\n\t}"
      : "=r"(d[0]), "=r"(d[1]), "=r"(d[2]), "=r"(d[3])
      : "r"(w));
}

// f16x2 of (hi, lo), each rounded toward zero.
__device__ __forceinline__ uint32_t f16x2_rz(float hi, float lo) {
  uint32_t d;
  asm("cvt.rz.f16x2.f32 %0, %1, %2;" : "=r"(d) : "f"(hi), "f"(lo));
  return d;
}

// Per 16-bit half: 0xFFFF where a < b (f16), else 0.
__device__ __forceinline__ uint32_t f16x2_lt_mask(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("set.lt.u32.f16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}

// Per 16-bit half: 0xFFFF where a == b (f16), else 0.
__device__ __forceinline__ uint32_t f16x2_eq_mask(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("set.eq.u32.f16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}

// Per 16-bit half: 0xFFFF where the bf16 value is not +-0 (finite input), else 0.
__device__ __forceinline__ uint32_t bf16x2_nonzero_mask(uint32_t a) {
  uint32_t d;
  asm("set.ne.u32.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(0u));
  return d;
}

// a b + c (low 32 bits) and the high 32 bits of the signed 64-bit product a b, plus c.
__device__ __forceinline__ uint32_t mad_lo_u32(uint32_t a, uint32_t b, uint32_t c) {
  uint32_t d;
  asm("mad.lo.u32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
  return d;
}
__device__ __forceinline__ uint32_t mad_hi_s32(uint32_t a, int32_t b, uint32_t c) {
  uint32_t d;
  asm("mad.hi.s32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
  return d;
}

// Per bf16 half: max(|a|, |b|) (sign bits: the XOR of the inputs'; the canonical NaN 0x7FFF if
// either input is NaN).
__device__ __forceinline__ uint32_t bf16x2_max_abs(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("max.NaN.xorsign.abs.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}

// Guided, cached or record encoding of one bf16 block (kMode != kModePlain) in the conversion
// form. The scale byte is the plain one (scale_byte_tab), or for kModeCached the given byte
// (above 0x7E read as 0x7E; 0 when g is not positive). With r = tab.rcp[b] (cvt_reciprocal with
// the grid points) and y = fl32(x r): c, the nearest code of y (cvt.rn.satfinite.e2m1x2), is the
// floor or the ceiling of |x| / d on the E2M1 grid, and lt = (|y| < G_c) decides which, exactly
// (y is on the side of every grid point that |x| / d is on; the compare runs on f16 values
// rounded toward zero, G_c being a short f16 value). So, per element:
//   plain code c, rounding-direction bit lt (kModeRecord);
//   floor c - lt, ceiling c + 1 - lt for x != 0, capped at code 7 (guided: the ceiling where the
//   mask bit is set, the scale byte nonzero and x off the grid, which is every x != 0 here: no
//   bf16 value lies on a grid point for the bytes the table accepts).
// Non-finite blocks and bytes the table rejects take encode_block's compare form, which writes
// the same bytes. `mask_word` is mask[blk >> 1] (guided and cached).
template <int kMode, class Tables>
__device__ __forceinline__ void encode_block_bf16_conv(const uint4 (&v)[2], int64_t blk, float g, float inv_g6,
                                                       float est_scale, float g6, const Tables& tab,
                                                       uint32_t mask_word, uint32_t given_scale,
                                                       const uint32_t* __restrict__ mask, uint8_t* __restrict__ codes,
                                                       uint8_t* __restrict__ scales, uint16_t* __restrict__ record16,
                                                       const uint8_t* __restrict__ scales_in) {
  constexpr bool kGuided = kMode == kModeGuided || kMode == kModeCached;
  const uint32_t w[8] = {v[0].x, v[0].y, v[0].z, v[0].w, v[1].x, v[1].y, v[1].z, v[1].w};
  uint32_t m2 = w[0];
#pragma unroll
  for (int i = 1; i < 8; ++i) m2 = bf16x2_max_abs(m2, w[i]);
  const uint32_t bamax_bits = max(m2 & 0x7FFFu, (m2 >> 16) & 0x7FFFu);  // 0x7FFF if any x is NaN
  uint32_t b = 0;
  if constexpr (kMode == kModeCached) {
    if (g > 0.0f) b = min(given_scale, 0x7Eu);
  } else {
    const float bamax = __uint_as_float(bamax_bits << 16);
    if (g > 0.0f) b = scale_byte_tab(bamax, (bamax * est_scale) * inv_g6, tab);
  }
  const float r = tab.rcp[b];
  if (!(r >= 0.0f && bamax_bits < 0x7F80u)) {
    BlockWords<NVFP4RL_BF16> bw;
    bw.v[0] = v[0];
    bw.v[1] = v[1];
    encode_block<NVFP4RL_BF16, kMode>(bw, blk, g, est_scale, g6, mask, codes, scales, record16, scales_in);
    return;
  }
  // up bits of elements 8h .. 8h + 7 at bits 0, 4, .., 28 of upn[h]: the nibble layout of the codes
  uint32_t upn[2] = {0u, 0u};
  if constexpr (kGuided) {
    const uint32_t up16 = b ? (mask_word >> ((blk & 1) * 16)) & 0xFFFFu : 0u;
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      uint32_t x = (up16 >> (8 * h)) & 0xFFu;  // pair j's two bits to nibble j, then a byte lookup:
      x = (x | (x << 4)) & 0x0F0Fu;            // 0 -> 0x00, 1 -> 0x01, 2 -> 0x10, 3 -> 0x11
      x = (x | (x << 2)) & 0x3333u;
      upn[h] = __byte_perm(0x11100100u, 0u, x);
    }
  }
  uint32_t out[2], rec = 0;
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    float y[8];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      y[2 * j] = __fmul_rn(__uint_as_float(w[4 * h + j] << 16), r);
      y[2 * j + 1] = __fmul_rn(__uint_as_float(w[4 * h + j] & 0xFFFF0000u), r);
    }
    uint32_t q = e2m1_word(y);  // nearest codes, signed
    uint32_t G[4];
    e2m1x8_to_f16x2(q & 0x77777777u, G);  // |G_c|
    uint32_t ltn = 0, xn = 0;  // per element, in the nibble layout: |y| < G_c; x != 0 and c < 7
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const uint32_t z = f16x2_rz(fabsf(y[2 * j + 1]), fabsf(y[2 * j]));
      const uint32_t lt = f16x2_lt_mask(z, G[j]);  // |y| < G_c: c is the ceiling
      if constexpr (kMode == kModeRecord) {
        rec |= lt & (0x00010001u << (4 * h + j));
      } else {
        const uint32_t c7 = f16x2_eq_mask(G[j], 0x46004600u);
        const uint32_t nz = bf16x2_nonzero_mask(w[4 * h + j]);
        // bit 12 (low half) and bit 16 (high half) of each mask, moved to this pair's two nibbles
        // (bits 8j and 8j + 4) by integer multiply-adds, which run beside the logic ops
        const uint32_t lt_b = lt & 0x00011000u, x_b = nz & ~c7 & 0x00011000u;
        if (j < 2) {
          ltn = mad_hi_s32(lt_b, 1 << (20 + 8 * j), ltn);  // (lt_b << (20 + 8j)) >> 32 = lt_b >> (12 - 8j)
          xn = mad_hi_s32(x_b, 1 << (20 + 8 * j), xn);
        } else {
          ltn = mad_lo_u32(lt_b, 1u << (8 * j - 12), ltn);
          xn = mad_lo_u32(x_b, 1u << (8 * j - 12), xn);
        }
      }
    }
    // floor = c - lt; the ceiling adds one where c is the ceiling already (lt) or x != 0 lies above
    // G_c below the top of the grid: code = c - lt + (up & (lt | (x != 0 & c < 7)))
    if constexpr (kGuided) q = q + (upn[h] & (ltn | xn)) - ltn;
    out[h] = q;
  }
  *reinterpret_cast<uint2*>(codes + blk * 8) = make_uint2(out[0], out[1]);
  if constexpr (kMode != kModeCached) scales[blk] = static_cast<uint8_t>(b);
  if constexpr (kMode == kModeRecord) {
    // element 2p's bit at p, element 2p + 1's at 16 + p -> bits 2p and 2p + 1
    uint32_t x = rec;
    x = (x | (x << 4)) & 0x0F0F0F0Fu;
    x = (x | (x << 2)) & 0x33333333u;
    x = (x | (x << 1)) & 0x55555555u;
    record16[blk] = static_cast<uint16_t>((x & 0xFFFFu) | ((x >> 16) << 1));
  }
}

// kModeCached reads g from g_in and the scale bytes from scales_in, and writes the codes only;
// the other modes take g = amax / 2688 (amax from amax_in, else the accumulated amax_bits) and
// write g, the scale bytes and the codes (kModeRecord also the rounding-direction bits).
template <int kDtype, int kMode>
__global__ void __launch_bounds__(256) quantize_kernel(const void* __restrict__ x, int64_t nblocks,
                                                       const uint32_t* __restrict__ amax_bits,
                                                       const float* __restrict__ amax_in,
                                                       const uint32_t* __restrict__ mask,
                                                       uint8_t* __restrict__ codes, uint8_t* __restrict__ scales,
                                                       float* __restrict__ g_out, uint16_t* __restrict__ record16,
                                                       const uint8_t* __restrict__ scales_in,
                                                       const float* __restrict__ g_in) {
  griddep_wait();
  griddep_launch_dependents();
  float g;
  if (kMode == kModeCached) {
    g = *g_in;
  } else {
    const float amax = amax_in ? *amax_in : __uint_as_float(*amax_bits);
    g = __fdiv_rn(amax, 2688.0f);
    if (blockIdx.x == 0 && threadIdx.x == 0) *g_out = g;
  }
  // The estimate of bamax / (6 g) is taken on operands scaled by 2^64 when g is tiny,
  // so that 6 g keeps full precision; the exact correction uses the unscaled values.
  const bool tiny = g < 0x1p-60f;
  const float est_scale = tiny ? 0x1p64f : 1.0f;
  const float g6 = 6.0f * (g * est_scale);
  // Two blocks per iteration, both loaded before either is encoded, and the next iteration's
  // two loaded before this one's are encoded (software pipelining: more bytes in flight).
  // The blocks are visited from the end of the tensor to its start: the amax pass that
  // precedes this kernel reads from start to end, so the tensor's tail is still in L2.
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  BlockWords<kDtype> na, nb;
  const int64_t j0 = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (j0 < nblocks) load_block<kDtype>(x, nblocks - 1 - j0, na);
  if (j0 + stride < nblocks) load_block<kDtype>(x, nblocks - 1 - j0 - stride, nb);
  for (int64_t j = j0; j < nblocks; j += 2 * stride) {
    const int64_t blk = nblocks - 1 - j;
    const bool two = j + stride < nblocks;
    const int64_t blk2 = blk - stride;
    const BlockWords<kDtype> a = na, b = nb;
    if (j + 2 * stride < nblocks) load_block<kDtype>(x, blk - 2 * stride, na);
    if (j + 3 * stride < nblocks) load_block<kDtype>(x, blk - 3 * stride, nb);
    encode_block<kDtype, kMode>(a, blk, g, est_scale, g6, mask, codes, scales, record16, scales_in);
    if (two) encode_block<kDtype, kMode>(b, blk2, g, est_scale, g6, mask, codes, scales, record16, scales_in);
  }
}

// Encoding of one bf16 tensor fed through shared memory: warp 0 streams the tensor in 16 KB chunks
// with cp.async.bulk into a ring of kEncRingStages stages (bulk copies keep far more bytes in
// flight than per-thread loads), and warps 1-8 encode the chunk's 512 blocks from shared memory,
// two per thread. Plain: EncodeTables and encode_block_bf16; guided, record and cached:
// ModeTables and encode_block_bf16_conv (each thread loads its blocks' mask words and given
// scale bytes one chunk ahead). Chunks are visited from the end of the tensor to its
// start (the amax pass before it reads from start to end, so the tail is still in L2). kModeCached
// takes g from g_in and writes codes only; the other modes take g = amax / 2688 and write g, the
// scale bytes and the codes (kModeRecord also the rounding-direction bits).
constexpr int kEncRingWarps = 8;
constexpr int kEncRingThreads = 32 * (kEncRingWarps + 1);
constexpr int kEncRingStages = 4;
constexpr int kEncRingSmem = kAmaxChunk * kEncRingStages;
constexpr int kChunkBlocks = kAmaxChunk / 32;  // bf16 blocks of 16 elements per chunk

template <int kMode>
__global__ void __launch_bounds__(kEncRingThreads, 3)
    encode_ring_kernel(const uint8_t* __restrict__ x, int64_t nblocks, const uint32_t* __restrict__ amax_bits,
                       const float* __restrict__ amax_in, const uint32_t* __restrict__ mask,
                       uint8_t* __restrict__ codes, uint8_t* __restrict__ scales, float* __restrict__ g_out,
                       uint16_t* __restrict__ record16, const uint8_t* __restrict__ scales_in,
                       const float* __restrict__ g_in, uint32_t* __restrict__ status) {
  constexpr bool kPlain = kMode == kModePlain;
  extern __shared__ __align__(128) uint8_t ring[];
  __shared__ uint64_t full[kEncRingStages], empty[kEncRingStages];
  __shared__ std::conditional_t<kPlain, EncodeTables, ModeTables> tab;
  griddep_wait();
  griddep_launch_dependents();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  float g;
  if constexpr (kMode == kModeCached) {
    g = *g_in;
  } else {
    const float amax = amax_in ? *amax_in : __uint_as_float(*amax_bits);
    g = __fdiv_rn(amax, 2688.0f);
    if (blockIdx.x == 0 && threadIdx.x == 0) *g_out = g;
  }
  const bool tiny = g < 0x1p-60f;  // as in quantize_kernel
  const float est_scale = tiny ? 0x1p64f : 1.0f;
  const float g6 = 6.0f * (g * est_scale);
  const float inv_g6 = 1.0f / g6;
  if (threadIdx.x == 0) {
    for (int i = 0; i < kEncRingStages; ++i) {
      mbar_init(smem_addr(&full[i]), 1);
      mbar_init(smem_addr(&empty[i]), kEncRingWarps);
    }
    fence_barrier_init();
  }
  __syncthreads();
  // the encode warps build the tables (named barrier 1) while warp 0 starts the stream
  if (warp > 0) {
    if constexpr (kPlain) build_encode_tables(tab, g, true, threadIdx.x - 32, 32 * kEncRingWarps);
    else build_mode_tables(tab, g, kMode != kModeCached, kMode == kModeRecord, threadIdx.x - 32, 32 * kEncRingWarps);
    named_barrier_sync(1, 32 * kEncRingWarps);
  }
  const int64_t bytes = nblocks * 32;
  const int64_t nchunks = (bytes + kAmaxChunk - 1) / kAmaxChunk;
  const int64_t mine = blockIdx.x < nchunks ? (nchunks - 1 - blockIdx.x) / gridDim.x + 1 : 0;
  if (warp == 0) {
    if (lane == 0) {
      int64_t issued = 0;
      for (int64_t j = 0; j < mine; ++j) {
        const int s = static_cast<int>(j % kEncRingStages);
        if (!mbar_wait(smem_addr(&empty[s]), static_cast<uint32_t>((j / kEncRingStages) & 1) ^ 1u, status,
                       kStatusTimeoutProducer))
          break;
        const int64_t c = nchunks - 1 - (blockIdx.x + j * gridDim.x);
        const int64_t off = c * kAmaxChunk;
        const uint32_t size = static_cast<uint32_t>(min(static_cast<int64_t>(kAmaxChunk), bytes - off));
        mbar_arrive_expect_tx(smem_addr(&full[s]), size);
        bulk_load(smem_addr(ring + s * kAmaxChunk), x + off, size, smem_addr(&full[s]));
        issued = j + 1;
      }
      // every issued copy has landed before the CTA exits
      for (int64_t j = max(int64_t(0), issued - kEncRingStages); j < issued; ++j)
        mbar_wait(smem_addr(&full[j % kEncRingStages]), static_cast<uint32_t>((j / kEncRingStages) & 1), status,
                  kStatusTimeoutDrain);
    }
  } else {
    const int t = threadIdx.x - 32;
    // this thread's blocks of chunk j: the mask words and given scale bytes are loaded one chunk
    // ahead, while the previous chunk is encoded
    const auto side = [&](int64_t jj, uint32_t (&sv)[4]) {
      const int64_t cc = nchunks - 1 - (blockIdx.x + jj * gridDim.x);
      const int nb = static_cast<int>(min(static_cast<int64_t>(kChunkBlocks), nblocks - cc * kChunkBlocks));
      const int64_t ba = cc * kChunkBlocks + t, bb = ba + 32 * kEncRingWarps;
      sv[0] = sv[1] = sv[2] = sv[3] = 0u;
      if constexpr (kMode == kModeGuided || kMode == kModeCached) {
        if (t < nb) sv[0] = __ldg(mask + (ba >> 1));
        if (t + 32 * kEncRingWarps < nb) sv[1] = __ldg(mask + (bb >> 1));
      }
      if constexpr (kMode == kModeCached) {
        if (t < nb) sv[2] = __ldg(scales_in + ba);
        if (t + 32 * kEncRingWarps < nb) sv[3] = __ldg(scales_in + bb);
      }
    };
    uint32_t cur[4] = {0u, 0u, 0u, 0u}, nxt[4] = {0u, 0u, 0u, 0u};
    if constexpr (!kPlain) {
      if (mine > 0) side(0, cur);
    }
    for (int64_t j = 0; j < mine; ++j) {
      const int s = static_cast<int>(j % kEncRingStages);
      const int64_t c = nchunks - 1 - (blockIdx.x + j * gridDim.x);
      const int nblk = static_cast<int>(min(static_cast<int64_t>(kChunkBlocks), nblocks - c * kChunkBlocks));
      const bool one = t < nblk, two = t + 32 * kEncRingWarps < nblk;
      const int64_t blk_a = c * kChunkBlocks + t, blk_b = blk_a + 32 * kEncRingWarps;
      if constexpr (!kPlain) {
        if (j + 1 < mine) side(j + 1, nxt);
      }
      const uint32_t mw_a = cur[0], mw_b = cur[1], sb_a = cur[2], sb_b = cur[3];
      if (!__all_sync(0xFFFFFFFFu, mbar_wait(smem_addr(&full[s]), static_cast<uint32_t>((j / kEncRingStages) & 1),
                                             status, kStatusTimeoutDequant)))
        break;
      const uint4* v = reinterpret_cast<const uint4*>(ring + s * kAmaxChunk);
      uint4 a[2], b[2];
      if (one) {
        a[0] = v[2 * t];
        a[1] = v[2 * t + 1];
      }
      if (two) {
        b[0] = v[2 * (t + 32 * kEncRingWarps)];
        b[1] = v[2 * (t + 32 * kEncRingWarps) + 1];
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_addr(&empty[s]));  // this warp has read the stage
      if constexpr (kPlain) {
        if (one) encode_block_bf16(a, blk_a, g, inv_g6, est_scale, tab, codes, scales);
        if (two) encode_block_bf16(b, blk_b, g, inv_g6, est_scale, tab, codes, scales);
      } else {
        if (one)
          encode_block_bf16_conv<kMode>(a, blk_a, g, inv_g6, est_scale, g6, tab, mw_a, sb_a, mask, codes, scales,
                                        record16, scales_in);
        if (two)
          encode_block_bf16_conv<kMode>(b, blk_b, g, inv_g6, est_scale, g6, tab, mw_b, sb_b, mask, codes, scales,
                                        record16, scales_in);
#pragma unroll
        for (int i = 0; i < 4; ++i) cur[i] = nxt[i];
      }
    }
  }
}

// Encoding of one bf16 tensor (plain rounding) fused with the amax pass over the next tensor of
// a batch: the encoding is bound by arithmetic and the amax pass by memory. Two CTAs per SM:
// warp 0 streams the next tensor through a ring of 16 KB shared-memory stages with
// cp.async.bulk (the amax_bulk_kernel scheme), warps 1-2 reduce it from shared memory, and
// warps 3-19 encode this tensor exactly as quantize_kernel does (same blocks, tables and
// order). The amax stream costs the encoding warps neither registers nor load slots.
constexpr int kFusedThreads = 640;   // two CTAs per SM
constexpr int kFusedEncodeWarps = 17;
constexpr int kFusedStages = 4;
constexpr int kFusedSmem = kAmaxChunk * kFusedStages;

__global__ void __launch_bounds__(kFusedThreads, 2)
    encode_amax_ring_kernel(const void* __restrict__ x, int64_t nblocks, const uint32_t* __restrict__ amax_bits,
                            uint8_t* __restrict__ codes, uint8_t* __restrict__ scales, float* __restrict__ g_out,
                            const uint8_t* __restrict__ xn, int64_t bytes_n, uint32_t* __restrict__ amax_next,
                            uint32_t* __restrict__ status) {
  griddep_wait();
  griddep_launch_dependents();
  extern __shared__ __align__(128) uint8_t ring[];
  __shared__ uint64_t full[kFusedStages], empty[kFusedStages];
  __shared__ uint32_t red[2];
  __shared__ EncodeTables tab;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const float amax = __uint_as_float(*amax_bits);
  const float g = __fdiv_rn(amax, 2688.0f);
  if (blockIdx.x == 0 && threadIdx.x == 0) *g_out = g;
  const bool tiny = g < 0x1p-60f;
  const float est_scale = tiny ? 0x1p64f : 1.0f;
  const float inv_g6 = 1.0f / (6.0f * (g * est_scale));
  if (threadIdx.x == 0) {
    for (int i = 0; i < kFusedStages; ++i) {
      mbar_init(smem_addr(&full[i]), 1);
      mbar_init(smem_addr(&empty[i]), 2);
    }
    fence_barrier_init();
  }
  __syncthreads();
  // the encode warps build the tables (named barrier 1) while warps 0-2 start the amax stream
  if (warp >= 3) {
    build_encode_tables(tab, g, true, threadIdx.x - 96, 32 * kFusedEncodeWarps);
    named_barrier_sync(1, 32 * kFusedEncodeWarps);
  }
  const int64_t nchunks = (bytes_n + kAmaxChunk - 1) / kAmaxChunk;
  const int64_t mine = blockIdx.x < nchunks ? (nchunks - 1 - blockIdx.x) / gridDim.x + 1 : 0;
  if (warp == 0) {
    // ---------------------------------------------------------------- next tensor -> ring
    if (lane == 0) {
      int64_t issued = 0;
      for (int64_t j = 0; j < mine; ++j) {
        const int s = static_cast<int>(j % kFusedStages);
        if (!mbar_wait(smem_addr(&empty[s]), static_cast<uint32_t>((j / kFusedStages) & 1) ^ 1u, status,
                       kStatusTimeoutProducer))
          break;
        const int64_t off = (blockIdx.x + j * gridDim.x) * static_cast<int64_t>(kAmaxChunk);
        const uint32_t size = static_cast<uint32_t>(min(static_cast<int64_t>(kAmaxChunk), bytes_n - off));
        mbar_arrive_expect_tx(smem_addr(&full[s]), size);
        bulk_load(smem_addr(ring + s * kAmaxChunk), xn + off, size, smem_addr(&full[s]));
        issued = j + 1;
      }
      for (int64_t j = max(int64_t(0), issued - kFusedStages); j < issued; ++j)
        mbar_wait(smem_addr(&full[j % kFusedStages]), static_cast<uint32_t>((j / kFusedStages) & 1), status,
                  kStatusTimeoutDrain);
    }
  } else if (warp <= 2) {
    // ---------------------------------------------------------------- amax of the next tensor
    const int t = threadIdx.x - 32;
    uint32_t m2 = 0;
    for (int64_t j = 0; j < mine; ++j) {
      const int s = static_cast<int>(j % kFusedStages);
      if (!__all_sync(0xFFFFFFFFu, mbar_wait(smem_addr(&full[s]), static_cast<uint32_t>((j / kFusedStages) & 1),
                                             status, kStatusTimeoutDequant)))
        break;
      const int64_t off = (blockIdx.x + j * gridDim.x) * static_cast<int64_t>(kAmaxChunk);
      const int nvec = static_cast<int>(min(static_cast<int64_t>(kAmaxChunk), bytes_n - off) / 16);
      const uint4* v = reinterpret_cast<const uint4*>(ring + s * kAmaxChunk);
#pragma unroll 8
      for (int i = t; i < nvec; i += 64) m2 = __vmaxu2(m2, max4_abs_bf16(v[i]));
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_addr(&empty[s]));
    }
    uint32_t m = max(m2 & 0xFFFFu, m2 >> 16) << 16;
    m = __reduce_max_sync(0xFFFFFFFFu, m);
    if (lane == 0) red[warp - 1] = m;
  } else {
    // ---------------------------------------------------------------- encode this tensor
    const int64_t stride = static_cast<int64_t>(gridDim.x) * (kFusedEncodeWarps * 32);
    for (int64_t j = static_cast<int64_t>(blockIdx.x) * (kFusedEncodeWarps * 32) + (threadIdx.x - 96); j < nblocks;
         j += 2 * stride) {
      const int64_t blk = nblocks - 1 - j;
      const bool two = j + stride < nblocks;
      const int64_t blk2 = blk - stride;
      BlockWords<NVFP4RL_BF16> a, b;
      load_block<NVFP4RL_BF16>(x, blk, a);
      if (two) load_block<NVFP4RL_BF16>(x, blk2, b);
      encode_block_bf16(a.v, blk, g, inv_g6, est_scale, tab, codes, scales);
      if (two) encode_block_bf16(b.v, blk2, g, inv_g6, est_scale, tab, codes, scales);
    }
  }
  __syncthreads();
  if (threadIdx.x == 0) atomicMax(amax_next, max(red[0], red[1]));
}

// RMSNorm-AQN fused with the NVFP4 quantization of its output, for outputs that fit in shared
// memory across the grid (one CTA per SM, launched cooperatively so that all CTAs are resident):
//   phase 1  every row of the CTA is requested at once (one bulk copy per row into its slot),
//            then eight warps per row, four rows at a time (each thread keeps the noised
//            weight of its own columns in registers for all its rows): y = bf16((w + sigma eps) x /
//            sqrt(mean x^2 + delta)) as in
//            rmsnorm_aqn_kernel, written to y and over the row's slot; the running
//            max of |y| (bf16 patterns) is reduced per CTA and folded into sync[0];
//   barrier  every CTA arrives on the counter sync[4] and waits (bounded) for all the others:
//            then sync[0] holds amax over all of y, so g = amax / 2688 is known;
//   phase 2  this CTA's rows are encoded from shared memory with the plain bf16 block encoder
//            (same blocks, tables and results as nvfp4_quantize of y).
// y is read from HBM never: x in, y and the codes out. sync[0] and sync[4] start at zero.
constexpr int kFuseThreads = 1024;
constexpr int kFuseGroup = 256;  // threads per row (eight warps)
constexpr int kFuseVec = 2;      // 128-bit words of a row per thread: H <= 256 * 2 * 8 = 4096

__global__ void __launch_bounds__(kFuseThreads, 1)
    rmsnorm_quant_kernel(const uint16_t* __restrict__ x, int64_t M, int64_t H, const float* __restrict__ w,
                         const float* __restrict__ eps, float sigma, float delta, uint16_t* __restrict__ y,
                         uint8_t* __restrict__ codes, uint8_t* __restrict__ scales, float* __restrict__ g_out,
                         uint32_t* __restrict__ sync, uint32_t* __restrict__ status) {
  extern __shared__ __align__(16) uint8_t ysm[];  // row slot i: H bf16 values; then one mbarrier per slot
  __shared__ EncodeTables tab;
  __shared__ float part[2][kFuseThreads / 32];    // per-warp sums of squares, by iteration parity
  __shared__ uint32_t red[kFuseThreads / 32];
  __shared__ int good;
  constexpr int kGroups = kFuseThreads / kFuseGroup;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int grp = threadIdx.x / kFuseGroup, t = threadIdx.x % kFuseGroup;
  const int64_t G = gridDim.x, cta = blockIdx.x;
  const int nrows = cta < M ? static_cast<int>((M - 1 - cta) / G + 1) : 0;
  const int rmax = static_cast<int>((M + G - 1) / G);
  const int nvec = static_cast<int>(H / 8);
  const uint32_t row_bytes = static_cast<uint32_t>(H * 2);
  uint64_t* bars = reinterpret_cast<uint64_t*>(ysm + static_cast<size_t>(rmax) * row_bytes);
  for (int i = threadIdx.x; i < nrows; i += kFuseThreads) mbar_init(smem_addr(&bars[i]), 1);
  fence_barrier_init();
  __syncthreads();
  // every row of this CTA is requested at once (one bulk copy per row, lane 0 of each warp
  // issuing rows warp, warp + 32, ...), so the loads of all rows are in flight together
  if (lane == 0) {
    for (int i = warp; i < nrows; i += kFuseThreads / 32) {
      mbar_arrive_expect_tx(smem_addr(&bars[i]), row_bytes);
      bulk_load(smem_addr(ysm + static_cast<size_t>(i) * row_bytes), x + (cta + static_cast<int64_t>(i) * G) * H,
                row_bytes, smem_addr(&bars[i]));
    }
  }
  // the noised weight w + sigma eps of this thread's columns (the same in every row), as rmsnorm_aqn forms it
  float wt[kFuseVec][8];
#pragma unroll
  for (int k = 0; k < kFuseVec; ++k) {
    const int j = t + kFuseGroup * k;
    if (j < nvec) {
      const float4 w0 = __ldg(reinterpret_cast<const float4*>(w) + 2 * j);
      const float4 w1 = __ldg(reinterpret_cast<const float4*>(w) + 2 * j + 1);
      wt[k][0] = w0.x; wt[k][1] = w0.y; wt[k][2] = w0.z; wt[k][3] = w0.w;
      wt[k][4] = w1.x; wt[k][5] = w1.y; wt[k][6] = w1.z; wt[k][7] = w1.w;
      if (eps) {
        const float4 e0 = __ldg(reinterpret_cast<const float4*>(eps) + 2 * j);
        const float4 e1 = __ldg(reinterpret_cast<const float4*>(eps) + 2 * j + 1);
        const float et[8] = {e0.x, e0.y, e0.z, e0.w, e1.x, e1.y, e1.z, e1.w};
#pragma unroll
        for (int u = 0; u < 8; ++u) wt[k][u] = fmaf(sigma, et[u], wt[k][u]);
      }
    } else {
#pragma unroll
      for (int u = 0; u < 8; ++u) wt[k][u] = 0.0f;
    }
  }
  uint32_t am2 = 0;
  // rows i = grp + kGroups * it of this CTA, each group of eight warps on its own (named barrier 1 + grp)
  for (int it = 0; grp + kGroups * it < nrows; ++it) {
    const int i = grp + kGroups * it;
    const int64_t row = cta + static_cast<int64_t>(i) * G;
    uint4* ys = reinterpret_cast<uint4*>(ysm + static_cast<size_t>(i) * row_bytes);
    // a timeout is recorded in the status word; the row is then processed as it stands, so that
    // the grid barrier below is still reached by every CTA
    mbar_wait(smem_addr(&bars[i]), 0u, status, kStatusTimeoutDequant);
    uint4 v[kFuseVec];
    float ss = 0.0f;
#pragma unroll
    for (int k = 0; k < kFuseVec; ++k) {
      const int j = t + kFuseGroup * k;
      v[k] = j < nvec ? ys[j] : make_uint4(0, 0, 0, 0);
    }
#pragma unroll
    for (int k = 0; k < kFuseVec; ++k) {
      const uint32_t q[4] = {v[k].x, v[k].y, v[k].z, v[k].w};
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const float a = __uint_as_float(bf16_lo_bits(q[u])), b = __uint_as_float(bf16_hi_bits(q[u]));
        ss = fmaf(a, a, ss);
        ss = fmaf(b, b, ss);
      }
    }
    ss = warp_sum(ss);
    if (lane == 0) part[it & 1][warp] = ss;
    asm volatile("bar.sync %0, %1;" ::"r"(1 + grp), "r"(kFuseGroup) : "memory");
    const float* pg = &part[it & 1][grp * (kFuseGroup / 32)];
    float sum = 0.0f;
#pragma unroll
    for (int u = 0; u < kFuseGroup / 32; ++u) sum += pg[u];
    const float r = rsqrtf(sum / static_cast<float>(H) + delta);
    uint4* yr = reinterpret_cast<uint4*>(y + row * H);
#pragma unroll
    for (int k = 0; k < kFuseVec; ++k) {
      const int j = t + kFuseGroup * k;
      if (j < nvec) {
        const uint32_t q[4] = {v[k].x, v[k].y, v[k].z, v[k].w};
        uint32_t o[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const float a = __uint_as_float(bf16_lo_bits(q[u])) * r * wt[k][2 * u];
          const float b = __uint_as_float(bf16_hi_bits(q[u])) * r * wt[k][2 * u + 1];
          o[u] = f32_to_bf16_bits(a) | (f32_to_bf16_bits(b) << 16);
          am2 = __vmaxu2(am2, o[u] & 0x7FFF7FFFu);
        }
        const uint4 ov = make_uint4(o[0], o[1], o[2], o[3]);
        yr[j] = ov;
        ys[j] = ov;
      }
    }
  }
  uint32_t m = max(am2 & 0xFFFFu, am2 >> 16) << 16;
  m = __reduce_max_sync(0xFFFFFFFFu, m);
  if (lane == 0) red[warp] = m;
  __syncthreads();
  if (threadIdx.x == 0) {
    uint32_t cm = 0;
    for (int i = 0; i < kFuseThreads / 32; ++i) cm = max(cm, red[i]);
    atomicMax(sync, cm);
    __threadfence();
    atomicAdd(sync + 4, 1u);
    // grid barrier: all CTAs are resident (cooperative launch); the wait is bounded all the same
    const uint64_t t0 = globaltimer();
    int ok = 1;
    while (*reinterpret_cast<volatile uint32_t*>(sync + 4) < static_cast<uint32_t>(G)) {
      if (globaltimer() - t0 > kWaitLimitNs) {
        atomicOr(status, kStatusTimeoutProducer);
        ok = 0;
        break;
      }
      __nanosleep(64);
    }
    __threadfence();
    good = ok;
  }
  __syncthreads();
  if (!good) return;
  const float amax = __uint_as_float(*reinterpret_cast<volatile uint32_t*>(sync));
  const float g = __fdiv_rn(amax, 2688.0f);
  if (cta == 0 && threadIdx.x == 0) *g_out = g;
  const bool tiny = g < 0x1p-60f;
  const float est_scale = tiny ? 0x1p64f : 1.0f;
  const float inv_g6 = 1.0f / (6.0f * (g * est_scale));
  // no reciprocals here: built after the grid barrier they cost more than the conversion saves at
  // the sizes that fit on chip
  build_encode_tables(tab, g, false, threadIdx.x, blockDim.x);
  __syncthreads();
  const int nb_row = static_cast<int>(H / 16);
  const int total = nrows * nb_row;
  for (int b = threadIdx.x; b < total; b += kFuseThreads) {
    const int i = b / nb_row, cb = b - i * nb_row;
    const uint4* src = reinterpret_cast<const uint4*>(ysm + static_cast<size_t>(i) * H * 2 + static_cast<size_t>(cb) * 32);
    const uint4 vv[2] = {src[0], src[1]};
    encode_block_bf16(vv, (cta + i * G) * nb_row + cb, g, inv_g6, est_scale, tab, codes, scales);
  }
}

// Appends one token's K and V rows per sequence to an NVFP4 KV cache: block i of the 2 B Hkv D/16
// blocks (K first, then V) of the new rows [B][Hkv][D] is encoded with the given per-tensor g and
// written to row (b, pos[b], h) of the cache ([B][Lmax][Hkv][D/2] codes, [B][Lmax][Hkv][D/16]
// scales). Sequences whose pos is outside [0, Lmax) are skipped.
__global__ void __launch_bounds__(256) kv_append_kernel(const uint16_t* __restrict__ k, const uint16_t* __restrict__ v,
                                                        int64_t B, int64_t Hkv, int64_t D,
                                                        const int32_t* __restrict__ pos, const float* __restrict__ gk,
                                                        const float* __restrict__ gv, uint8_t* __restrict__ kc,
                                                        uint8_t* __restrict__ ks, uint8_t* __restrict__ vc,
                                                        uint8_t* __restrict__ vs, int64_t Lmax) {
  griddep_wait();
  griddep_launch_dependents();
  const int64_t nb = D / 16, per = B * Hkv * nb;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < 2 * per; i += stride) {
    const bool is_v = i >= per;
    const int64_t j = is_v ? i - per : i;
    const int64_t blk = j % nb, bh = j / nb, b = bh / Hkv, h = bh % Hkv;
    const int64_t p = pos[b];
    if (p < 0 || p >= Lmax) continue;
    const float g = is_v ? *gv : *gk;
    const float est_scale = g < 0x1p-60f ? 0x1p64f : 1.0f;  // as in quantize_kernel
    const float g6 = 6.0f * (g * est_scale);
    BlockWords<NVFP4RL_BF16> w;
    load_block<NVFP4RL_BF16>((is_v ? v : k) + bh * D, blk, w);
    const int64_t row = (b * Lmax + p) * Hkv + h;
    encode_block<NVFP4RL_BF16, kModePlain>(w, blk, g, est_scale, g6, nullptr, (is_v ? vc : kc) + row * (D / 2),
                                           (is_v ? vs : ks) + row * nb, nullptr, nullptr);
  }
}

// Clears the amax accumulator word (a kernel rather than a memset, so that it chains with the
// neighbouring kernels by programmatic dependent launch).
__global__ void zero_word_kernel(uint32_t* __restrict__ p) {
  griddep_wait();
  griddep_launch_dependents();
  if (threadIdx.x == 0) *p = 0u;
}

// Clears n amax accumulator words, 4 words (16 bytes) apart.
__global__ void zero_words_kernel(uint32_t* __restrict__ p, int n) {
  griddep_wait();
  griddep_launch_dependents();
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < n; i += gridDim.x * blockDim.x) p[4 * i] = 0u;
}

}  // namespace

namespace {

// amax of n elements accumulated (atomicMax of the bit pattern) into *amax_bits, which the
// caller has zeroed.
nvfp4rl_status launch_amax_accumulate(const void* x, int dtype, int64_t n, uint32_t* amax_bits, const DeviceInfo& dev,
                                      cudaStream_t st) {
  if (n == 0) return NVFP4RL_OK;
  const int64_t bytes = n * (dtype == NVFP4RL_BF16 ? 2 : 4);
  const int64_t nchunks = (bytes + kAmaxChunk - 1) / kAmaxChunk;
  if (nchunks >= dev.sm_count) {
    // large tensors: bulk-copy pipeline, one CTA per SM
    const int grid = dev.sm_count;
    const uint8_t* xb = static_cast<const uint8_t*>(x);
    cudaError_t e;
    if (dtype == NVFP4RL_BF16) {
      e = cudaFuncSetAttribute(amax_bulk_kernel<NVFP4RL_BF16>, cudaFuncAttributeMaxDynamicSharedMemorySize, kAmaxSmem);
      if (e == cudaSuccess)
        amax_bulk_kernel<NVFP4RL_BF16><<<grid, 32 * (kAmaxWarps + 1), kAmaxSmem, st>>>(xb, bytes, amax_bits, dev.status);
    } else {
      e = cudaFuncSetAttribute(amax_bulk_kernel<NVFP4RL_F32>, cudaFuncAttributeMaxDynamicSharedMemorySize, kAmaxSmem);
      if (e == cudaSuccess)
        amax_bulk_kernel<NVFP4RL_F32><<<grid, 32 * (kAmaxWarps + 1), kAmaxSmem, st>>>(xb, bytes, amax_bits, dev.status);
    }
    if (e != cudaSuccess) return NVFP4RL_ERR_CUDA;
    return launch_status();
  }
  const int threads = 256;
  const int64_t nvec = bytes / 16;
  const int64_t want = (nvec + threads - 1) / threads;
  const int grid = static_cast<int>(want < dev.sm_count * 4 ? want : dev.sm_count * 4);
  if (dtype == NVFP4RL_BF16) amax_kernel<NVFP4RL_BF16><<<grid, threads, 0, st>>>(x, nvec, amax_bits);
  else amax_kernel<NVFP4RL_F32><<<grid, threads, 0, st>>>(x, nvec, amax_bits);
  return launch_status();
}

}  // namespace

nvfp4rl_status launch_zero_word(uint32_t* p, cudaStream_t st) {
  if (launch_pdl(zero_word_kernel, dim3(1), dim3(32), 0, st, p) != cudaSuccess) return NVFP4RL_ERR_CUDA;
  return launch_status();
}

nvfp4rl_status launch_amax(const void* x, int dtype, int64_t n, uint32_t* amax_bits, const DeviceInfo& dev,
                           cudaStream_t st) {
  if (launch_pdl(zero_word_kernel, dim3(1), dim3(32), 0, st, amax_bits) != cudaSuccess) return NVFP4RL_ERR_CUDA;
  if (launch_status() != NVFP4RL_OK) return NVFP4RL_ERR_CUDA;
  return launch_amax_accumulate(x, dtype, n, amax_bits, dev, st);
}

namespace {

// CTAs of quantize_kernel resident per SM (once per device and variant).
template <int kDtype, int kMode>
int quantize_ctas_per_sm(int device) {
  static std::mutex mu;
  static std::map<int, int> cache;
  std::lock_guard<std::mutex> lock(mu);
  auto it = cache.find(device);
  if (it != cache.end()) return it->second;
  int n = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, quantize_kernel<kDtype, kMode>, 256, 0) != cudaSuccess ||
      n < 1) {
    cudaGetLastError();
    n = 8;
  }
  cache[device] = n;
  return n;
}

}  // namespace

namespace {

// CTAs of encode_ring_kernel<kMode> resident per SM (once per device; sets its shared-memory size).
template <int kMode>
int encode_ring_ctas_per_sm(int device) {
  static std::mutex mu;
  static std::map<int, int> cache;
  std::lock_guard<std::mutex> lock(mu);
  auto it = cache.find(device);
  if (it != cache.end()) return it->second;
  int n = 0;
  if (cudaFuncSetAttribute(encode_ring_kernel<kMode>, cudaFuncAttributeMaxDynamicSharedMemorySize, kEncRingSmem) !=
          cudaSuccess ||
      cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, encode_ring_kernel<kMode>, kEncRingThreads, kEncRingSmem) !=
          cudaSuccess ||
      n < 1) {
    cudaGetLastError();
    n = 0;
  }
  cache[device] = n;
  return n;
}

// bf16 input: every mode through encode_ring_kernel; fp32 input: quantize_kernel.
template <int kDtype, int kMode>
cudaError_t launch_encode(int64_t nblocks, const DeviceInfo& dev, cudaStream_t st, const void* x,
                          const uint32_t* amax_bits, const float* amax_in, const uint32_t* mask, uint8_t* codes,
                          uint8_t* scales, float* g, uint16_t* record16, const uint8_t* scales_in, const float* g_in) {
  if constexpr (kDtype == NVFP4RL_BF16) {
    const int per_sm = encode_ring_ctas_per_sm<kMode>(dev.device);
    if (per_sm == 0) return cudaErrorLaunchFailure;
    const int64_t nchunks = (nblocks * 32 + kAmaxChunk - 1) / kAmaxChunk;
    const int grid = static_cast<int>(std::min<int64_t>(nchunks, static_cast<int64_t>(dev.sm_count) * per_sm));
    return launch_pdl(encode_ring_kernel<kMode>, dim3(grid), dim3(kEncRingThreads), kEncRingSmem, st,
                      static_cast<const uint8_t*>(x), nblocks, amax_bits, amax_in, mask, codes, scales, g, record16,
                      scales_in, g_in, dev.status);
  } else {
    // one wave: as many CTAs as can be resident at once (each loops over its share of the blocks)
    const int threads = 256;
    const int64_t want = (nblocks + threads - 1) / threads;
    const int per_sm = quantize_ctas_per_sm<kDtype, kMode>(dev.device);
    const int grid = static_cast<int>(std::min<int64_t>(want, static_cast<int64_t>(dev.sm_count) * per_sm));
    return launch_pdl(quantize_kernel<kDtype, kMode>, dim3(grid), dim3(threads), 0, st, x, nblocks, amax_bits,
                      amax_in, mask, codes, scales, g, record16, scales_in, g_in);
  }
}

template <int kMode>
cudaError_t launch_encode_dtype(int dtype, int64_t nblocks, const DeviceInfo& dev, cudaStream_t st, const void* x,
                                const uint32_t* amax_bits, const float* amax_in, const uint32_t* mask,
                                uint8_t* codes, uint8_t* scales, float* g, uint16_t* record16,
                                const uint8_t* scales_in, const float* g_in) {
  return dtype == NVFP4RL_BF16
             ? launch_encode<NVFP4RL_BF16, kMode>(nblocks, dev, st, x, amax_bits, amax_in, mask, codes, scales, g,
                                                  record16, scales_in, g_in)
             : launch_encode<NVFP4RL_F32, kMode>(nblocks, dev, st, x, amax_bits, amax_in, mask, codes, scales, g,
                                                 record16, scales_in, g_in);
}

}  // namespace

nvfp4rl_status launch_quantize(const void* x, int dtype, int64_t rows, int64_t cols, const uint32_t* mask,
                               uint8_t* codes, uint8_t* scales, float* g, const float* amax_in,
                               uint32_t* amax_scratch, const DeviceInfo& dev, cudaStream_t st, bool amax_done,
                               uint32_t* record) {
  const int64_t n = rows * cols;
  const int64_t nblocks = n / 16;
  if (nblocks == 0) return NVFP4RL_OK;
  if (amax_in == nullptr && !amax_done) {
    const nvfp4rl_status sa = launch_amax(x, dtype, n, amax_scratch, dev, st);
    if (sa != NVFP4RL_OK) return sa;
  }
  uint16_t* record16 = reinterpret_cast<uint16_t*>(record);
  const cudaError_t e =
      record ? launch_encode_dtype<kModeRecord>(dtype, nblocks, dev, st, x, amax_scratch, amax_in, nullptr, codes,
                                                scales, g, record16, nullptr, nullptr)
      : mask ? launch_encode_dtype<kModeGuided>(dtype, nblocks, dev, st, x, amax_scratch, amax_in, mask, codes,
                                                scales, g, nullptr, nullptr, nullptr)
             : launch_encode_dtype<kModePlain>(dtype, nblocks, dev, st, x, amax_scratch, amax_in, nullptr, codes,
                                               scales, g, nullptr, nullptr, nullptr);
  if (e != cudaSuccess) return NVFP4RL_ERR_CUDA;
  return launch_status();
}

nvfp4rl_status launch_kv_append(const uint16_t* k, const uint16_t* v, int64_t B, int64_t Hkv, int64_t D,
                                const int32_t* pos, const float* gk, const float* gv, uint8_t* kc, uint8_t* ks,
                                uint8_t* vc, uint8_t* vs, int64_t Lmax, const DeviceInfo& dev, cudaStream_t st) {
  const int64_t n = 2 * B * Hkv * (D / 16);
  if (n == 0) return NVFP4RL_OK;
  const int grid = static_cast<int>(std::min<int64_t>((n + 255) / 256, static_cast<int64_t>(dev.sm_count) * 8));
  if (launch_pdl(kv_append_kernel, dim3(grid), dim3(256), 0, st, k, v, B, Hkv, D, pos, gk, gv, kc, ks, vc, vs, Lmax) !=
      cudaSuccess)
    return NVFP4RL_ERR_CUDA;
  return launch_status();
}

nvfp4rl_status launch_quantize_cached(const void* x, int dtype, int64_t rows, int64_t cols, const uint32_t* mask,
                                      const uint8_t* scales, const float* g, uint8_t* codes, const DeviceInfo& dev,
                                      cudaStream_t st) {
  const int64_t nblocks = rows * cols / 16;
  if (nblocks == 0) return NVFP4RL_OK;
  if (launch_encode_dtype<kModeCached>(dtype, nblocks, dev, st, x, nullptr, nullptr, mask, codes, nullptr, nullptr,
                                       nullptr, scales, g) != cudaSuccess)
    return NVFP4RL_ERR_CUDA;
  return launch_status();
}

nvfp4rl_status launch_quantize_batch(int count, const void* const* x, const int64_t* rows, const int64_t* cols,
                                     int dtype, uint8_t* const* codes, uint8_t* const* scales, float* const* g,
                                     uint32_t* amax_words, const DeviceInfo& dev, cudaStream_t st) {
  // Non-empty tensors: the smallest first (its amax pass is the one that runs alone), then the
  // rest largest first (the fused kernels then pair tensors of similar size, and the encoding
  // that runs alone at the end is that of the smallest remaining tensor).
  std::vector<int> order;
  for (int i = 0; i < count; ++i)
    if (rows[i] > 0) order.push_back(i);
  if (order.empty()) return NVFP4RL_OK;
  const auto numel = [&](int i) { return rows[i] * cols[i]; };
  std::stable_sort(order.begin(), order.end(), [&](int a, int b) { return numel(a) > numel(b); });
  std::rotate(order.begin(), order.end() - 1, order.end());
  uint32_t* word = amax_words;  // tensor i: word[4 i]
  if (launch_pdl(zero_words_kernel, dim3(static_cast<unsigned>((count + 255) / 256)), dim3(256), 0, st, amax_words,
                 count) != cudaSuccess)
    return NVFP4RL_ERR_CUDA;
  if (launch_status() != NVFP4RL_OK) return NVFP4RL_ERR_CUDA;
  if (dtype != NVFP4RL_BF16) {
    for (int i : order) {
      const nvfp4rl_status s1 = launch_amax_accumulate(x[i], dtype, numel(i), word + 4 * i, dev, st);
      if (s1 != NVFP4RL_OK) return s1;
      const nvfp4rl_status s2 = launch_quantize(x[i], dtype, rows[i], cols[i], nullptr, codes[i], scales[i], g[i],
                                                nullptr, word + 4 * i, dev, st, /*amax_done=*/true);
      if (s2 != NVFP4RL_OK) return s2;
    }
    return NVFP4RL_OK;
  }
  const int first = order[0];
  nvfp4rl_status sa = launch_amax_accumulate(x[first], dtype, numel(first), word + 4 * first, dev, st);
  if (sa != NVFP4RL_OK) return sa;
  static std::mutex attr_mu;
  {
    std::lock_guard<std::mutex> lock(attr_mu);
    if (cudaFuncSetAttribute(encode_amax_ring_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kFusedSmem) !=
        cudaSuccess)
      return NVFP4RL_ERR_CUDA;
  }
  for (size_t k = 0; k + 1 < order.size(); ++k) {
    const int i = order[k], n = order[k + 1];
    const int64_t nblocks = numel(i) / 16, bytes_n = numel(n) * 2;
    if (launch_pdl(encode_amax_ring_kernel, dim3(static_cast<unsigned>(2 * dev.sm_count)), dim3(kFusedThreads),
                   static_cast<size_t>(kFusedSmem), st, x[i], nblocks, static_cast<const uint32_t*>(word + 4 * i),
                   codes[i], scales[i], g[i], static_cast<const uint8_t*>(x[n]), bytes_n, word + 4 * n,
                   dev.status) != cudaSuccess)
      return NVFP4RL_ERR_CUDA;
    if (launch_status() != NVFP4RL_OK) return NVFP4RL_ERR_CUDA;
  }
  const int last = order.back();
  return launch_quantize(x[last], dtype, rows[last], cols[last], nullptr, codes[last], scales[last], g[last], nullptr,
                         word + 4 * last, dev, st, /*amax_done=*/true);
}

nvfp4rl_status launch_rmsnorm_quantize(const uint16_t* x, int64_t M, int64_t H, const float* w, const float* eps,
                                      float sigma, float delta, uint16_t* y, uint8_t* codes, uint8_t* scales,
                                      float* g, uint32_t* sync, const DeviceInfo& dev, cudaStream_t st) {
  if (M == 0) return NVFP4RL_OK;
  if (launch_pdl(zero_words_kernel, dim3(1), dim3(32), 0, st, sync, 2) != cudaSuccess) return NVFP4RL_ERR_CUDA;
  if (launch_status() != NVFP4RL_OK) return NVFP4RL_ERR_CUDA;
  // fused path: every CTA's rows of y fit in its shared memory, one CTA per SM
  const int64_t G = std::min<int64_t>(M, dev.sm_count);
  const int64_t rows_per_cta = (M + G - 1) / G;
  const size_t smem = static_cast<size_t>(rows_per_cta) * (H * 2 + 8);
  if (H / 8 <= kFuseGroup * kFuseVec && smem + 8 * 1024 <= dev.smem_optin) {
    // per device: the largest dynamic shared-memory size set so far, and whether one CTA of that
    // size is resident per SM
    struct FuseState {
      size_t smem_set = 0;
      bool resident = false;
    };
    static std::mutex mu;
    static std::map<int, FuseState> states;
    std::lock_guard<std::mutex> lock(mu);
    FuseState& fs = states[dev.device];
    if (smem > fs.smem_set) {
      int per_sm = 0;
      fs.resident = false;
      if (cudaFuncSetAttribute(rmsnorm_quant_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               static_cast<int>(smem)) == cudaSuccess &&
          cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, rmsnorm_quant_kernel, kFuseThreads, smem) ==
              cudaSuccess &&
          per_sm >= 1) {
        fs.smem_set = smem;
        fs.resident = true;
      }
      cudaGetLastError();
    }
    if (fs.resident) {
      void* args[] = {const_cast<uint16_t**>(&x), &M, &H, const_cast<float**>(&w), const_cast<float**>(&eps), &sigma,
                      &delta, &y, &codes, &scales, &g, &sync, const_cast<uint32_t**>(&dev.status)};
      if (cudaLaunchCooperativeKernel(reinterpret_cast<const void*>(rmsnorm_quant_kernel), dim3(static_cast<unsigned>(G)),
                                      dim3(kFuseThreads), args, smem, st) == cudaSuccess)
        return launch_status();
      cudaGetLastError();  // fall back below
    }
  }
  // otherwise: RMSNorm-AQN accumulating max |y| into the amax word (cleared above), then the
  // encoding of y
  const nvfp4rl_status s1 = launch_rmsnorm_aqn(x, M, H, w, eps, sigma, delta, y, dev, st, sync);
  if (s1 != NVFP4RL_OK) return s1;
  return launch_quantize(y, NVFP4RL_BF16, M, H, nullptr, codes, scales, g, nullptr, sync, dev, st, true);
}

}  // namespace nvfp4rl
