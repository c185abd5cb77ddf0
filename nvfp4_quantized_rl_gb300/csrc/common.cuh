// Shared device helpers of the NVFP4 rollout-linear library (sm_103a).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <utility>
#include <stdint.h>

#include "../../include/nvfp4rl.h"

namespace nvfp4rl {

constexpr int kNumSMsHint = 152;  // GB300: 2 dies x 76 SMs; the real count is queried at run time

// ---- bf16 / fp32 bit helpers ------------------------------------------------------------

__device__ __forceinline__ uint32_t bf16_lo_bits(uint32_t pair) { return pair << 16; }
__device__ __forceinline__ uint32_t bf16_hi_bits(uint32_t pair) { return pair & 0xFFFF0000u; }

// fp32 -> bf16 bits, round to nearest even (finite inputs; one cvt instruction)
__device__ __forceinline__ uint32_t f32_to_bf16_bits(float f) {
  uint16_t h;
  asm("cvt.rn.bf16.f32 %0, %1;" : "=h"(h) : "f"(f));
  return h;
}

// Two fp32 values -> a bf16 pair (lo in bits 0-15, hi in bits 16-31), round to nearest even.
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

// E4M3 (OCP FP8 E4M3FN) value of a non-negative byte 0x00..0x7E, built from its bits.
__device__ __forceinline__ float e4m3_decode_pos(uint32_t b) {
  const uint32_t e = b >> 3, m = b & 7u;
  // normal: (1 + m/8) 2^(e-7) -> fp32 exponent field e + 120, mantissa m << 20
  const float normal = __uint_as_float(((e + 120u) << 23) | (m << 20));
  const float sub = static_cast<float>(m) * 0.001953125f;  // m * 2^-9
  return e ? normal : sub;
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xFFFFFFFFu, v, o));
  return v;
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, o);
  return v;
}

__device__ __forceinline__ uint4 ld_nc_v4(const void* p) {
  uint4 r;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "l"(p));
  return r;
}

// ---- host side ---------------------------------------------------------------------------

struct DeviceInfo {
  int device = -1;
  int sm_count = 0;
  int cc_major = 0, cc_minor = 0;
  size_t smem_optin = 0;
  uint32_t* status = nullptr;  // device address of the library's error word on this device
};

// Cached attributes of the current device; NVFP4RL_ERR_DEVICE unless compute capability 10.3.
nvfp4rl_status current_device(DeviceInfo* out);

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

inline bool overlap(const void* a, size_t na, const void* b, size_t nb) {
  const uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
  return na && nb && x < y + nb && y < x + na;
}

inline size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

// Programmatic dependent launch. A kernel launched with launch_pdl may start once every CTA of
// the preceding kernel on the stream has called griddep_launch_dependents (or exited).
// griddep_wait blocks until that preceding kernel has completed and its memory is visible (a
// no-op for a kernel launched without the attribute). The library's kernels on the decode path
// call griddep_wait before touching global memory and only then griddep_launch_dependents, so
// every kernel still observes all earlier kernels complete, while the next launch overlaps the
// current kernel's tail.
#ifdef __CUDACC__
__device__ __forceinline__ void griddep_launch_dependents() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
__device__ __forceinline__ void griddep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
#endif

template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                       Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// Counts one kernel launch (diagnostic, see nvfp4rl_kernel_launches) and reports its status.
void count_launch();
inline nvfp4rl_status launch_status() {
  count_launch();
  return cudaGetLastError() == cudaSuccess ? NVFP4RL_OK : NVFP4RL_ERR_CUDA;
}

// ---- internal launchers (quantize.cu, rmsnorm.cu, linear_tc.cu, linear_w4a4_tc.cu, ...) -----------

// Quantization scratch: one 32-bit word holding the running amax bits.
constexpr size_t kQuantizeWorkspace = 256;

nvfp4rl_status launch_amax(const void* x, int dtype, int64_t n, uint32_t* amax_bits, const DeviceInfo& dev,
                           cudaStream_t st);

// Batched quantization: at most this many tensors per call; one amax word (16 bytes) each.
constexpr int64_t kQuantizeBatchMax = 4096;
inline size_t quantize_batch_workspace_bytes(int64_t count) {
  return static_cast<size_t>(((std::max<int64_t>(count, 1) * 16 + 255) / 256) * 256);
}
nvfp4rl_status launch_quantize_batch(int count, const void* const* x, const int64_t* rows, const int64_t* cols,
                                     int dtype, uint8_t* const* codes, uint8_t* const* scales, float* const* g,
                                     uint32_t* amax_words, const DeviceInfo& dev, cudaStream_t st);

// amax_done: *amax_scratch already holds the tensor's amax bits (no amax pass is launched).
// record (non-NULL only without mask): the plain encoding also writes its rounding directions,
// 16 bits per 16-element block.
// Clears one word (the amax accumulator) with a one-thread kernel chained by programmatic dependent launch.
nvfp4rl_status launch_zero_word(uint32_t* p, cudaStream_t st);
nvfp4rl_status launch_quantize(const void* x, int dtype, int64_t rows, int64_t cols, const uint32_t* mask,
                               uint8_t* codes, uint8_t* scales, float* g, const float* amax_in,
                               uint32_t* amax_scratch, const DeviceInfo& dev, cudaStream_t st, bool amax_done = false,
                               uint32_t* record = nullptr);

// NVFP4 KV cache: append one token's rows per sequence (quantize.cu) and decode attention over the
// cache (attention.cu, head dimension 128).
nvfp4rl_status launch_kv_append(const uint16_t* k, const uint16_t* v, int64_t B, int64_t Hkv, int64_t D,
                                const int32_t* pos, const float* gk, const float* gv, uint8_t* kc, uint8_t* ks,
                                uint8_t* vc, uint8_t* vs, int64_t Lmax, const DeviceInfo& dev, cudaStream_t st);
int attention_splits(int64_t B, int64_t Hkv, int64_t Lmax);
size_t attention_workspace_bytes(int64_t B, int64_t Hkv, int64_t Lmax);
nvfp4rl_status launch_kv_attention(const uint16_t* q, const uint8_t* kc, const uint8_t* ks, const float* gk,
                                   const uint8_t* vc, const uint8_t* vs, const float* gv, const int32_t* lens,
                                   int64_t B, int64_t Hq, int64_t Hkv, int64_t Lmax, float scale, uint16_t* out,
                                   void* workspace, const DeviceInfo& dev, cudaStream_t st);

// AIS mixing coefficient and rectified weights of n tokens (ais.cu); workspace: a barrier counter
// and one slot of partial sums per CTA (at most kAisMaxCtas CTAs).
constexpr int kAisMaxCtas = 1024;
size_t ais_workspace_bytes();
nvfp4rl_status launch_ais(const float* lr, const float* lt, const float* adv, int64_t n, float C, float delta,
                          float gamma, float beta, float* w_out, double* stats, void* workspace,
                          const DeviceInfo& dev, cudaStream_t st);

// Guided codes of x against the given scale bytes and g (device), in one pass (quantize.cu).
nvfp4rl_status launch_quantize_cached(const void* x, int dtype, int64_t rows, int64_t cols, const uint32_t* mask,
                                      const uint8_t* scales, const float* g, uint8_t* codes, const DeviceInfo& dev,
                                      cudaStream_t st);

nvfp4rl_status launch_rmsnorm_aqn(const uint16_t* x, int64_t M, int64_t H, const float* w, const float* eps,
                                  float sigma, float delta, uint16_t* y, const DeviceInfo& dev, cudaStream_t st,
                                  uint32_t* amax = nullptr);

// RMSNorm-AQN of x into y and the NVFP4 quantization of y (quantize.cu); sync: two zeroable
// words 16 bytes apart (kQuantizeWorkspace bytes).
nvfp4rl_status launch_rmsnorm_quantize(const uint16_t* x, int64_t M, int64_t H, const float* w, const float* eps,
                                      float sigma, float delta, uint16_t* y, uint8_t* codes, uint8_t* scales,
                                      float* g, uint32_t* sync, const DeviceInfo& dev, cudaStream_t st);

struct LinearArgs {
  const uint16_t* x;
  int64_t M, K, N;
  const uint8_t* w_codes;
  const uint8_t* w_scales;
  const float* w_g;
  const uint16_t* A;
  const uint16_t* B;
  int r;
  float s;
  const int32_t* offsets;
  int groups;
  uint16_t* y;
  bool w4a4;
  // W4A4 with activations already in NVFP4 (codes, scales, g as the quantizer wrote them for x);
  // null: the call quantizes x itself
  const uint8_t* xq_codes = nullptr;
  const uint8_t* xq_scales = nullptr;
  const float* xq_g = nullptr;
};

// LoRA ranks the linears take: 0 (no LoRA) or a multiple of 16 up to this bound (the rank is the K
// of the up-projection MMA, 16 per instruction; both LoRA tiles stay resident in shared memory).
constexpr int kMaxLoraRank = 128;

// Workspace bytes of a linear call (0 when the shape is not supported); prequantized: W4A4 on
// activations given in NVFP4 (the workspace then holds no activation codes).
size_t linear_workspace_bytes(bool w4a4, int64_t M, int64_t N, int64_t K, int r, int groups, bool prequantized = false);

// Split-K planning uses at most this many SMs, so workspace sizes do not depend on the device.
constexpr int kPlanSMs = 152;

// 2-D TMA tensor map over a row-major [rows][cols] array of `esize`-byte elements (linear_tc.cu).
bool make_tensor_map_2d(CUtensorMap* m, CUtensorMapDataType dt, const void* base, uint64_t cols, uint64_t rows,
                        int esize, uint32_t box_cols, uint32_t box_rows, CUtensorMapSwizzle sw);

// Folded form of the LoRA down-projection's output (the W4A4 path, and W4A16 with 256-token
// tiles): instead of U = bf16(x A^T), the two bf16 parts of c U with c = s / (g_x w_g) (c = s
// when g_x w_g = 0): hi = bf16(c U) into U, lo = bf16(c U - hi) into `lo`. g_x comes from device
// memory (W4A4: the activations' g; U is then bf16(x A^T)) or by value (W4A16: 2^32, the
// dequantized weights' offset; U is then x A^T as accumulated in fp32). |c| above 2^100 sets the
// range bit of `status`.
struct LoraDownScale {
  const float* g_x = nullptr;  // null: g_x_value, or plain U when that is 0 too
  const float* w_g = nullptr;
  float s = 0.f;
  uint16_t* lo = nullptr;  // [M][r]
  uint32_t* status = nullptr;
  float g_x_value = 0.f;
  __host__ __device__ bool folded() const { return g_x != nullptr || g_x_value != 0.f; }
  __device__ float gx() const { return g_x ? *g_x : g_x_value; }
};

// LoRA down-projection U = bf16(x A^T), [M][r] row-major, K a multiple of 64 (linear_tc.cu):
// clusters of CTAs split K and reduce in distributed shared memory. Launched as a programmatic
// dependent of the previous kernel on the stream; it waits for that kernel before reading x
// (and g_x).
nvfp4rl_status launch_lora_down(const uint16_t* x, int64_t M, int64_t K, const uint16_t* A, int r, uint16_t* U,
                                const DeviceInfo& dev, cudaStream_t st, const LoraDownScale& scale = {});

// The same on tcgen05 for prefill-sized M (lora_down_tc.cu); launch_lora_down takes it for
// M >= kLoraDownTcMinRows.
constexpr int64_t kLoraDownTcMinRows = 1024;
bool lora_down_tc_supported(int64_t M, int64_t K, int r);
// amax (or null): accumulates max |x| into that word (atomicMax of the fp32 bit pattern; the caller
// clears it first), the amax the NVFP4 encoding of x needs.
nvfp4rl_status launch_lora_down_tc(const uint16_t* x, int64_t M, int64_t K, const uint16_t* A, int r, uint16_t* U,
                                   const DeviceInfo& dev, cudaStream_t st, const LoraDownScale& scale,
                                   uint32_t* amax = nullptr);
// U (plain, [M][r] bf16) -> hi and lo of c U in place (hi over U, lo into scale.lo).
nvfp4rl_status launch_lora_scale(uint16_t* U, int64_t M, int r, const LoraDownScale& scale, const DeviceInfo& dev,
                                 cudaStream_t st);

// tcgen05 W4A4 block-scaled path (linear_w4a4_tc.cu).
bool w4a4_tc_supported(int64_t M, int64_t N, int64_t K, int r);
size_t w4a4_tc_workspace_bytes(int64_t M, int64_t N, int64_t K, int r, int groups, bool prequantized);
nvfp4rl_status launch_w4a4_tc(const LinearArgs& a, void* ws, size_t ws_bytes, const DeviceInfo& dev,
                              cudaStream_t st);

// tcgen05 W4A16 path (linear_tc.cu).
bool w4a16_tc_supported(int64_t M, int64_t N, int64_t K, int r);
size_t w4a16_tc_workspace_bytes(int64_t M, int64_t N, int64_t K, int r, int sm_count);
nvfp4rl_status launch_w4a16_tc(const LinearArgs& a, void* ws, size_t ws_bytes, const DeviceInfo& dev,
                               cudaStream_t st);
nvfp4rl_status launch_linear(const LinearArgs& a, void* ws, size_t ws_bytes, const DeviceInfo& dev, cudaStream_t st);

}  // namespace nvfp4rl
