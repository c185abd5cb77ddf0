// Decode attention over an NVFP4 KV cache (sm_103a).
//
// TRACE summary, section "実験結果と性能": rollouts run with FP4 weights, activations and KV
// cache. Each cached K/V row of a head is NVFP4-encoded (16-element blocks along the head
// dimension, E4M3 block scales, a per-tensor fp32 g given by the caller); decode attention reads
// the dequantized rows: out[b][h] = softmax(scale q[b][h] K^T) V over the first lens[b] cached
// tokens of KV head h / (Hq / Hkv).
//
// Split-KV ("flash decoding"): one CTA of four warps per (sequence, KV head, token span); warp w
// takes tokens 16 w .. 16 w + 15 of every 64-token chunk of the span and works alone (its own
// shared-memory region, __syncwarp only). Per 16-token group the warp
//   - streams the code and scale bytes of its tokens into a two-stage ring with cp.async;
//   - dequantizes the K and V rows into bf16 tiles: the sign and magnitude bits of an E2M1 code
//     placed as bf16 bits are grid * 2^-126 exactly, and one bf16x2 FMA by E4M3(s) 2^119 makes
//     grid E4M3(s) 2^-7, exact (at most 6 significant bits); 2^7 g is applied as a scalar later;
//   - computes S = Q K^T with mma.sync m16n8k16 (the group's query heads are the rows, padded to
//     16), keeps an online softmax in exp2, and adds P V with the V fragments read transposed by
//     ldmatrix.
// The contraction is skinny (Hq / Hkv rows), so warp-level MMAs leave the tensor pipe mostly
// idle and tcgen05 would add nothing; the dequantization's instructions, not the HBM read, bound
// the kernel as it stands. The four warps' states are merged in shared memory; with several spans
// per sequence a second kernel merges the spans' (max, sum, O) partials.
#include <map>
#include <mutex>

#include "common.cuh"

namespace nvfp4rl {
namespace {

constexpr int kHeadDim = 128;
constexpr int kChunk = 64;       // tokens per CTA iteration (16 per warp)
constexpr int kAttnThreads = 128;
constexpr int kRow = kHeadDim + 8;  // bf16 row stride of the K/V tiles (conflict-free ldmatrix)
constexpr int kPartFloats = 132;    // per (span, row): max, sum, O[128], padding
constexpr float kLog2e = 1.4426950408889634f;
constexpr int kWarpTok = 16;  // tokens per warp and group
constexpr int kStageBytes = 2 * kWarpTok * (kHeadDim / 2) + 2 * kWarpTok * (kHeadDim / 16);  // K, V codes + scales
constexpr int kTileBytes = 2 * kWarpTok * kRow * 2;                                         // K and V bf16 tiles
constexpr int kWarpBytes = kTileBytes + 2 * kStageBytes;
constexpr int kAttnSmem = 4 * kWarpBytes;

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

__device__ __forceinline__ void mma16816(float (&c)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// a * b per bf16 half, exact for the E2M1 x E4M3 products used here (fma with -0 keeps signed zeros).
__device__ __forceinline__ uint32_t bf16x2_mul(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("fma.rn.bf16x2 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(0x80008000u));
  return d;
}

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  return f32_to_bf16_bits(lo) | (f32_to_bf16_bits(hi) << 16);
}

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, uint32_t src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(src_bytes) : "memory");
}
__device__ __forceinline__ void cp_async8(uint32_t dst, const void* src, uint32_t src_bytes) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 8, %2;" ::"r"(dst), "l"(src), "r"(src_bytes) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait1() { asm volatile("cp.async.wait_group 1;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait0() { asm volatile("cp.async.wait_group 0;" ::: "memory"); }

// bf16 bits of E4M3(byte) 2^119 (at most 448 2^119 < the largest bf16), byte 0x00 .. 0x7E.
__device__ __forceinline__ uint32_t scale_bf16_2p119(uint32_t byte) {
  return __float_as_uint(e4m3_decode_pos(byte) * 0x1p119f) >> 16;
}

// One code byte's two elements (low nibble first) as a bf16x2 pattern grid * 2^-126 with signs: with
// u = byte + byte * 2^12 the high nibble also sits at bits 16..19, so one mask-and-shift pair places
// both magnitudes (bits 6..8 of each half) and one places both signs (bit 15 of each half).
// byte must be 0 .. 255.
__device__ __forceinline__ uint32_t code_pair_bits(uint32_t byte) {
  const uint32_t u = byte * 4097u;
  return ((u & 0x00070007u) << 6) | ((u & 0x00080008u) << 12);
}

// 16 code bytes (32 elements = two blocks) and their two scale bytes, dequantized to grid E4M3(s)
// 2^-7 into 32 bf16 values at dst.
__device__ __forceinline__ void dequant32(uint4 codes, uint32_t s0, uint32_t s1, uint16_t* dst) {
  const uint32_t a = scale_bf16_2p119(s0), c = scale_bf16_2p119(s1);
  const uint32_t S0 = a | (a << 16), S1 = c | (c << 16);
  const uint32_t w[4] = {codes.x, codes.y, codes.z, codes.w};
  uint32_t o[16];
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j) o[4 * i + j] = bf16x2_mul(code_pair_bits((w[i] >> (8 * j)) & 0xFFu), i < 2 ? S0 : S1);
  uint4* d = reinterpret_cast<uint4*>(dst);
#pragma unroll
  for (int i = 0; i < 4; ++i) d[i] = make_uint4(o[4 * i], o[4 * i + 1], o[4 * i + 2], o[4 * i + 3]);
}

struct AttnArgs {
  const uint16_t* q;
  const uint8_t *kc, *ks, *vc, *vs;
  const float *gk, *gv;
  const int32_t* lens;
  int64_t Hq, Hkv, Lmax;
  int nsplit, span;  // token spans per sequence and their length (a multiple of kChunk)
  float scale;
  uint16_t* out;     // used when nsplit == 1
  float* part;       // [B*Hkv][nsplit][16][kPartFloats] when nsplit > 1
};

__global__ void __launch_bounds__(kAttnThreads) kv_attention_kernel(AttnArgs a) {
  extern __shared__ __align__(16) uint8_t smem[];
  __shared__ float msm[4][16], lsm[4][16];
  griddep_wait();
  griddep_launch_dependents();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  uint8_t* wbase = smem + warp * kWarpBytes;
  uint16_t* Ks = reinterpret_cast<uint16_t*>(wbase);  // [16][kRow]
  uint16_t* Vs = Ks + kWarpTok * kRow;
  uint8_t* stage = wbase + kTileBytes;  // [2][K codes 1 KB | V codes 1 KB | K scales 128 B | V scales 128 B]
  const int64_t bh = blockIdx.y, b = bh / a.Hkv, kvh = bh % a.Hkv;
  const int group = static_cast<int>(a.Hq / a.Hkv);
  const int split = blockIdx.x;
  const int64_t len = min(max(static_cast<int64_t>(a.lens[b]), int64_t(0)), a.Lmax);
  const int64_t t_begin = static_cast<int64_t>(split) * a.span;
  const int64_t t_end = min(t_begin + a.span, len);
  // Q fragments of the group's heads (rows >= group are zero), 8 k-steps of 16 dims
  uint32_t qa[8][4];
  {
    const int r0 = lane >> 2, c0 = (lane & 3) * 2;
    const uint32_t* q32 = reinterpret_cast<const uint32_t*>(a.q + (b * a.Hq + kvh * group) * kHeadDim);
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      const int c = k * 16 + c0;
      qa[k][0] = r0 < group ? q32[(r0 * kHeadDim + c) >> 1] : 0u;
      qa[k][1] = r0 + 8 < group ? q32[((r0 + 8) * kHeadDim + c) >> 1] : 0u;
      qa[k][2] = r0 < group ? q32[(r0 * kHeadDim + c + 8) >> 1] : 0u;
      qa[k][3] = r0 + 8 < group ? q32[((r0 + 8) * kHeadDim + c + 8) >> 1] : 0u;
    }
  }
  const float sl2 = a.scale * __ldg(a.gk) * 128.0f * kLog2e;  // scores in log2 units (K tiles carry 2^-7)
  float m_run[2] = {-INFINITY, -INFINITY}, l_run[2] = {0.0f, 0.0f};
  float o[16][4];
#pragma unroll
  for (int j = 0; j < 16; ++j) o[j][0] = o[j][1] = o[j][2] = o[j][3] = 0.0f;

  // group i of this warp = tokens t_begin + 64 i + 16 warp .. + 15, into stage i % 2: lane l copies the
  // 16-byte units u = l + 32 j (j < 4) of the K then V code rows (row (u % 64) / 4, bytes 16 (u % 4) ..)
  // and the 8 scale bytes of row l % 16 (K for l < 16, V otherwise); rows at or beyond t_end are
  // zero-filled (source bytes 0)
  const auto issue = [&](int64_t g0, int st) {
    uint8_t* sb = stage + st * kStageBytes;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int u = lane + 32 * j, is_v = u >> 6, r = (u & 63) >> 2, c = u & 3;
      const int64_t t = g0 + r;
      const bool live = t < t_end;
      const int64_t row = (b * a.Lmax + (live ? t : 0)) * a.Hkv + kvh;
      cp_async16(smem_u32(sb + is_v * kWarpTok * (kHeadDim / 2) + r * (kHeadDim / 2) + 16 * c),
                 (is_v ? a.vc : a.kc) + row * (kHeadDim / 2) + 16 * c, live ? 16u : 0u);
    }
    {
      const int is_v = lane >> 4, r = lane & 15;
      const int64_t t = g0 + r;
      const bool live = t < t_end;
      const int64_t row = (b * a.Lmax + (live ? t : 0)) * a.Hkv + kvh;
      cp_async8(smem_u32(sb + 2 * kWarpTok * (kHeadDim / 2) + is_v * kWarpTok * (kHeadDim / 16) + r * (kHeadDim / 16)),
                (is_v ? a.vs : a.ks) + row * (kHeadDim / 16), live ? 8u : 0u);
    }
  };
  const int64_t first = t_begin + kWarpTok * warp;
  if (first < t_end) issue(first, 0);
  cp_async_commit();
  if (first + kChunk < t_end) issue(first + kChunk, 1);
  cp_async_commit();
  int st = 0;
  for (int64_t t0 = first; t0 < t_end; t0 += kChunk, st ^= 1) {
    cp_async_wait1();  // this group's bytes (the older of the two groups in flight) have landed
    __syncwarp();
    {
      const uint8_t* sb = stage + st * kStageBytes;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int u = lane + 32 * j, is_v = u >> 6, r = (u & 63) >> 2, c = u & 3;
        const uint4 codes =
            *reinterpret_cast<const uint4*>(sb + is_v * kWarpTok * (kHeadDim / 2) + r * (kHeadDim / 2) + 16 * c);
        const uint8_t* sc = sb + 2 * kWarpTok * (kHeadDim / 2) + is_v * kWarpTok * (kHeadDim / 16) + r * (kHeadDim / 16);
        dequant32(codes, sc[2 * c], sc[2 * c + 1], (is_v ? Vs : Ks) + r * kRow + 32 * c);
      }
    }
    __syncwarp();  // tiles complete; this stage may be refilled
    if (t0 + 2 * kChunk < t_end) issue(t0 + 2 * kChunk, st);
    cp_async_commit();
    // S = Q K^T for this warp's 16 tokens: two n-tiles of 8 tokens
    float s[2][4] = {{0, 0, 0, 0}, {0, 0, 0, 0}};
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      uint32_t b0, b1, b2, b3;
      const int tok = (lane & 7) + ((lane >> 4) << 3), dim = k * 16 + ((lane >> 3) & 1) * 8;
      ldsm_x4(smem_u32(Ks + tok * kRow + dim), b0, b1, b2, b3);
      mma16816(s[0], qa[k], b0, b1);
      mma16816(s[1], qa[k], b2, b3);
    }
    // online softmax over the two rows this thread holds (r0: s[.][0..1], r0 + 8: s[.][2..3])
    float p[2][4];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      float mx = -INFINITY;
#pragma unroll
      for (int j = 0; j < 2; ++j)
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const int64_t t = t0 + j * 8 + (lane & 3) * 2 + e;
          float& v = s[j][2 * h + e];
          v = t < t_end ? v * sl2 : -INFINITY;
          mx = fmaxf(mx, v);
        }
      mx = fmaxf(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, 1));
      mx = fmaxf(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, 2));
      const float m_new = fmaxf(m_run[h], mx);
      const float base = m_new == -INFINITY ? 0.0f : m_new;  // no token seen yet: nothing to rescale
      const float corr = exp2f(m_run[h] - base);
      m_run[h] = m_new;
      float sum = 0.0f;
#pragma unroll
      for (int j = 0; j < 2; ++j)
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          p[j][2 * h + e] = exp2f(s[j][2 * h + e] - base);
          sum += p[j][2 * h + e];
        }
      l_run[h] = l_run[h] * corr + sum;
#pragma unroll
      for (int j = 0; j < 16; ++j) {
        o[j][2 * h] *= corr;
        o[j][2 * h + 1] *= corr;
      }
    }
    // O += P V: P as the A fragment (16 rows x 16 tokens), V fragments transposed from the tile
    const uint32_t pa[4] = {pack_bf16(p[0][0], p[0][1]), pack_bf16(p[0][2], p[0][3]), pack_bf16(p[1][0], p[1][1]),
                            pack_bf16(p[1][2], p[1][3])};
#pragma unroll
    for (int j = 0; j < 16; j += 2) {
      uint32_t b0, b1, b2, b3;
      const int tok = (lane & 7) + ((lane >> 3) & 1) * 8, dim = j * 8 + (lane >> 4) * 8;
      ldsm_x4_t(smem_u32(Vs + tok * kRow + dim), b0, b1, b2, b3);
      mma16816(o[j], pa, b0, b1);
      mma16816(o[j + 1], pa, b2, b3);
    }
  }
  // merge the four warps: row sums over the quad, then (max, sum, O) per warp in shared memory
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    l_run[h] += __shfl_xor_sync(0xFFFFFFFFu, l_run[h], 1);
    l_run[h] += __shfl_xor_sync(0xFFFFFFFFu, l_run[h], 2);
  }
  cp_async_wait0();  // no copy may still land in the region reused below
  __syncthreads();   // every warp's tiles are reused below for the warps' O
  float* Osm = reinterpret_cast<float*>(smem);  // [4][16][128] fp32 = 32 KB <= the four warp regions
  {
    const int r0 = lane >> 2, c0 = (lane & 3) * 2;
    if ((lane & 3) == 0) {
      msm[warp][r0] = m_run[0];
      msm[warp][r0 + 8] = m_run[1];
      lsm[warp][r0] = l_run[0];
      lsm[warp][r0 + 8] = l_run[1];
    }
#pragma unroll
    for (int j = 0; j < 16; ++j) {
      float* row0 = Osm + (warp * 16 + r0) * kHeadDim + j * 8 + c0;
      float* row8 = Osm + (warp * 16 + r0 + 8) * kHeadDim + j * 8 + c0;
      row0[0] = o[j][0];
      row0[1] = o[j][1];
      row8[0] = o[j][2];
      row8[1] = o[j][3];
    }
  }
  __syncthreads();
  const float gv = __ldg(a.gv) * 128.0f;  // the V tiles carry 2^-7
  for (int i = threadIdx.x; i < group * kHeadDim; i += kAttnThreads) {
    const int r = i / kHeadDim, d = i % kHeadDim;
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < 4; ++w) M = fmaxf(M, msm[w][r]);
    float L = 0.0f, O = 0.0f;
#pragma unroll
    for (int w = 0; w < 4; ++w) {
      const float f = msm[w][r] == -INFINITY ? 0.0f : exp2f(msm[w][r] - M);
      L += f * lsm[w][r];
      O += f * Osm[(w * 16 + r) * kHeadDim + d];
    }
    if (a.nsplit == 1) {
      const float y = L > 0.0f ? O / L * gv : 0.0f;
      a.out[(b * a.Hq + kvh * group + r) * kHeadDim + d] = static_cast<uint16_t>(f32_to_bf16_bits(y));
    } else {
      float* pr = a.part + ((bh * a.nsplit + split) * 16 + r) * kPartFloats;
      if (d == 0) {
        pr[0] = M;
        pr[1] = L;
      }
      pr[4 + d] = O * 128.0f;  // the V tiles carry 2^-7
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
  const int64_t chunks = std::max<int64_t>(1, (Lmax + kChunk - 1) / kChunk);
  const int64_t want = (12 * kNumSMsHint + B * Hkv - 1) / (B * Hkv);  // several waves: a short tail
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
  const int ns = attention_splits(B, Hkv, Lmax);
  const int64_t chunks = (Lmax + kChunk - 1) / kChunk;
  const int span = static_cast<int>((chunks + ns - 1) / ns) * kChunk;
  AttnArgs a{q, kc, ks, vc, vs, gk, gv, lens, Hq, Hkv, Lmax, ns, span, scale, out, static_cast<float*>(workspace)};
  const size_t smem = kAttnSmem;
  static_assert(kAttnSmem >= 4 * 16 * kHeadDim * sizeof(float), "merge area");
  {
    static std::mutex mu;
    static std::map<int, bool> set;
    std::lock_guard<std::mutex> lock(mu);
    if (!set[dev.device]) {
      if (cudaFuncSetAttribute(kv_attention_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kAttnSmem) !=
          cudaSuccess)
        return NVFP4RL_ERR_CUDA;
      set[dev.device] = true;
    }
  }
  if (launch_pdl(kv_attention_kernel, dim3(static_cast<unsigned>(ns), static_cast<unsigned>(B * Hkv)),
                 dim3(kAttnThreads), smem, st, a) != cudaSuccess)
    return NVFP4RL_ERR_CUDA;
  if (launch_status() != NVFP4RL_OK) return NVFP4RL_ERR_CUDA;
  if (ns == 1) return NVFP4RL_OK;
  if (launch_pdl(kv_attention_merge_kernel, dim3(static_cast<unsigned>((B * Hq + 3) / 4)), dim3(128), 0, st,
                 static_cast<const float*>(workspace), B, Hq, Hkv, ns, gv, out) != cudaSuccess)
    return NVFP4RL_ERR_CUDA;
  return launch_status();
}

}  // namespace nvfp4rl
