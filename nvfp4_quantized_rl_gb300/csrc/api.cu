// C ABI of the NVFP4 rollout-linear library: argument validation and dispatch.
// Every check runs on the host before any launch; see include/nvfp4rl.h for the contract.
#include <algorithm>
#include <atomic>
#include <cmath>
#include <mutex>
#include <vector>

#include "common.cuh"
#include "sm100.cuh"

namespace nvfp4rl {

// Device-side error word (bounded waits set bits here instead of hanging).
__device__ uint32_t g_device_status;

namespace {
std::mutex g_dev_mutex;
DeviceInfo g_dev_cache[64];
std::atomic<uint64_t> g_launches{0};
}  // namespace

void count_launch() { g_launches.fetch_add(1, std::memory_order_relaxed); }

size_t linear_workspace_bytes(bool w4a4, int64_t M, int64_t N, int64_t K, int r, int groups, bool prequantized) {
  if (w4a4) return w4a4_tc_supported(M, N, K, r) ? w4a4_tc_workspace_bytes(M, N, K, r, groups, prequantized) : 0;
  return w4a16_tc_supported(M, N, K, r) ? w4a16_tc_workspace_bytes(M, N, K, r, kPlanSMs) : 0;
}

// Both linears run on the tcgen05 kernels; the host checks admit only the shapes they take.
nvfp4rl_status launch_linear(const LinearArgs& a, void* ws, size_t ws_bytes, const DeviceInfo& dev, cudaStream_t st) {
  if (a.M == 0) return NVFP4RL_OK;
  if (a.w4a4) {
    if (!w4a4_tc_supported(a.M, a.N, a.K, a.r)) return NVFP4RL_ERR_UNSUPPORTED_SHAPE;
    return launch_w4a4_tc(a, ws, ws_bytes, dev, st);
  }
  if (!w4a16_tc_supported(a.M, a.N, a.K, a.r)) return NVFP4RL_ERR_UNSUPPORTED_SHAPE;
  return launch_w4a16_tc(a, ws, ws_bytes, dev, st);
}

nvfp4rl_status current_device(DeviceInfo* out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return NVFP4RL_ERR_CUDA;
  if (dev < 0 || dev >= 64) return NVFP4RL_ERR_DEVICE;
  std::lock_guard<std::mutex> lock(g_dev_mutex);
  DeviceInfo& d = g_dev_cache[dev];
  if (d.device != dev) {
    DeviceInfo n;
    n.device = dev;
    int v = 0;
    if (cudaDeviceGetAttribute(&n.cc_major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&n.cc_minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&n.sm_count, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&v, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess)
      return NVFP4RL_ERR_CUDA;
    n.smem_optin = static_cast<size_t>(v);
    void* sp = nullptr;
    if (cudaGetSymbolAddress(&sp, g_device_status) != cudaSuccess) return NVFP4RL_ERR_CUDA;
    n.status = static_cast<uint32_t*>(sp);
    d = n;
  }
  if (d.cc_major != 10 || d.cc_minor != 3) return NVFP4RL_ERR_DEVICE;
  *out = d;
  return NVFP4RL_OK;
}

int64_t rmsnorm_max_h();

// One thread waits, through the kernels' bounded wait, on a fresh mbarrier that nothing ever
// arrives on; after 1 ms the wait gives up, sets kStatusTimeoutProducer and the kernel returns.
__global__ void wait_timeout_probe_kernel(uint32_t* status) {
  __shared__ uint64_t bar;
  if (threadIdx.x == 0) {
    sm100::mbar_init(sm100::smem_addr(&bar), 1);
    sm100::fence_barrier_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) sm100::mbar_wait<1000000ull>(sm100::smem_addr(&bar), 0, status, sm100::kStatusTimeoutProducer);
  __syncthreads();
}

}  // namespace nvfp4rl

using namespace nvfp4rl;

namespace {

// record (nvfp4_quantize_record only): the rounding-direction bits, one per element.
nvfp4rl_status quantize_common(const void* x, int32_t dtype, int64_t rows, int64_t cols, const uint32_t* mask,
                               bool guided, uint8_t* codes, uint8_t* scales, float* g, const float* amax_in,
                               void* ws, size_t ws_bytes, void* stream, uint32_t* record = nullptr,
                               bool recording = false) {
  if (dtype != NVFP4RL_BF16 && dtype != NVFP4RL_F32) return NVFP4RL_ERR_INVALID_ARG;
  if (rows < 0 || cols <= 0) return NVFP4RL_ERR_INVALID_ARG;
  if (cols % 16 != 0) return NVFP4RL_ERR_UNSUPPORTED_SHAPE;
  if (rows == 0) return NVFP4RL_OK;  // empty tensor: nothing to read or write (g is left as is)
  if (!x || !codes || !scales || !g || (guided && !mask) || (recording && !record)) return NVFP4RL_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(codes) || !aligned16(scales) || (mask && !aligned16(mask)) ||
      (record && !aligned16(record)) || (reinterpret_cast<uintptr_t>(g) & 3u) ||
      (amax_in && (reinterpret_cast<uintptr_t>(amax_in) & 3u)))
    return NVFP4RL_ERR_MISALIGNED;
  if (!amax_in) {
    if (!ws || ws_bytes < kQuantizeWorkspace) return NVFP4RL_ERR_WORKSPACE;
    if (!aligned16(ws)) return NVFP4RL_ERR_MISALIGNED;
  }
  const size_t n = static_cast<size_t>(rows) * static_cast<size_t>(cols);
  const size_t xbytes = n * (dtype == NVFP4RL_BF16 ? 2 : 4);
  const size_t mbytes = guided ? (n + 31) / 32 * 4 : 0;
  const int nouts = recording ? 4 : 3;
  const void* outs[4] = {codes, scales, g, record};
  const size_t osz[4] = {n / 2, n / 16, 4, n / 8};  // the record: 16 bits per block
  for (int i = 0; i < nouts; ++i) {
    if (overlap(outs[i], osz[i], x, xbytes) || (guided && overlap(outs[i], osz[i], mask, mbytes)) ||
        (amax_in && overlap(outs[i], osz[i], amax_in, 4)) || (!amax_in && overlap(outs[i], osz[i], ws, kQuantizeWorkspace)))
      return NVFP4RL_ERR_ALIAS;
    for (int j = i + 1; j < nouts; ++j)
      if (overlap(outs[i], osz[i], outs[j], osz[j])) return NVFP4RL_ERR_ALIAS;
  }
  DeviceInfo dev;
  nvfp4rl_status st = current_device(&dev);
  if (st != NVFP4RL_OK) return st;
  return launch_quantize(x, dtype, rows, cols, guided ? mask : nullptr, codes, scales, g, amax_in,
                         static_cast<uint32_t*>(ws), dev, static_cast<cudaStream_t>(stream), false,
                         recording ? record : nullptr);
}

// True when any two of the [begin, end) ranges overlap (n log n).
bool any_overlap(std::vector<std::pair<uintptr_t, uintptr_t>>& r) {
  std::sort(r.begin(), r.end());
  for (size_t i = 1; i < r.size(); ++i)
    if (r[i].first < r[i - 1].second) return true;
  return false;
}

// True when [a, b) overlaps one of the sorted, disjoint ranges r.
bool hits(const std::vector<std::pair<uintptr_t, uintptr_t>>& r, uintptr_t a, uintptr_t b) {
  auto it = std::lower_bound(r.begin(), r.end(), std::make_pair(b, uintptr_t(0)));
  return it != r.begin() && std::prev(it)->second > a;
}

// xq_codes / xq_scales / xq_g: W4A4 on activations given in NVFP4 (x is then read by the LoRA
// branch only and may be NULL without LoRA); all NULL: x is quantized by the call.
nvfp4rl_status linear_common(bool w4a4, const uint16_t* x, int64_t M, int64_t K, const uint8_t* w_codes,
                             const uint8_t* w_scales, const float* w_g, int64_t N, const uint16_t* A,
                             const uint16_t* B, int32_t r, float s, const int32_t* offsets, int32_t groups,
                             uint16_t* y, void* ws, size_t ws_bytes, void* stream, const uint8_t* xq_codes = nullptr,
                             const uint8_t* xq_scales = nullptr, const float* xq_g = nullptr) {
  const bool pre = xq_codes || xq_scales || xq_g;
  if (M < 0 || K <= 0 || N <= 0 || r < 0 || r > 256) return NVFP4RL_ERR_INVALID_ARG;
  if (r % 16 != 0 || r > kMaxLoraRank) return NVFP4RL_ERR_UNSUPPORTED_SHAPE;
  if (M == 0) return NVFP4RL_OK;  // no activation rows: nothing to read or write
  if (pre && (!xq_codes || !xq_scales || !xq_g)) return NVFP4RL_ERR_INVALID_ARG;
  if ((!x && !(pre && r == 0)) || !w_codes || !w_scales || !w_g || !y) return NVFP4RL_ERR_INVALID_ARG;
  if (r > 0 && (!A || !B)) return NVFP4RL_ERR_INVALID_ARG;
  if (!std::isfinite(s)) return NVFP4RL_ERR_INVALID_ARG;
  if (offsets) {
    if (!w4a4) return NVFP4RL_ERR_UNSUPPORTED_SHAPE;
    if (groups < 1 || groups > 1024 || r != 0) return NVFP4RL_ERR_INVALID_ARG;
  } else if (groups != 0 && groups != 1) {
    return NVFP4RL_ERR_INVALID_ARG;
  }
  if (K % 256 != 0 || N % 128 != 0 || M > 65535) return NVFP4RL_ERR_UNSUPPORTED_SHAPE;
  const void* arrays[] = {x, w_codes, w_scales, A, B, offsets, y, ws, xq_codes, xq_scales};
  for (const void* p : arrays)
    if (p && !aligned16(p)) return NVFP4RL_ERR_MISALIGNED;
  if ((reinterpret_cast<uintptr_t>(w_g) & 3u) || (reinterpret_cast<uintptr_t>(xq_g) & 3u))
    return NVFP4RL_ERR_MISALIGNED;
  const int G = offsets ? groups : 1;
  const size_t need = linear_workspace_bytes(w4a4, M, N, K, r, G, pre);
  if (need == 0) return NVFP4RL_ERR_UNSUPPORTED_SHAPE;
  if (!ws || ws_bytes < need) return NVFP4RL_ERR_WORKSPACE;
  const size_t ybytes = static_cast<size_t>(M) * N * 2;
  const void* ins[] = {x, w_codes, w_scales, w_g, A, B, offsets, ws, xq_codes, xq_scales, xq_g};
  const size_t isz[] = {static_cast<size_t>(M) * K * 2, static_cast<size_t>(G) * N * K / 2,
                        static_cast<size_t>(G) * N * K / 16, static_cast<size_t>(G) * 4,
                        A ? static_cast<size_t>(r) * K * 2 : 0, B ? static_cast<size_t>(N) * r * 2 : 0,
                        offsets ? static_cast<size_t>(groups + 1) * 4 : 0, ws ? need : 0,
                        static_cast<size_t>(M) * K / 2, static_cast<size_t>(M) * K / 16, 4};
  for (int i = 0; i < 11; ++i)
    if (ins[i] && overlap(y, ybytes, ins[i], isz[i])) return NVFP4RL_ERR_ALIAS;
  // the workspace (U, tile map) is written by the call: it may not overlap an input either
  for (int i = 0; i < 11; ++i)
    if (i != 7 && ins[i] && ws && overlap(ws, need, ins[i], isz[i])) return NVFP4RL_ERR_ALIAS;
  DeviceInfo dev;
  nvfp4rl_status st = current_device(&dev);
  if (st != NVFP4RL_OK) return st;
  LinearArgs a{x, M, K, N, w_codes, w_scales, w_g, A, B, r, s, offsets, G, y, w4a4};
  a.xq_codes = xq_codes;
  a.xq_scales = xq_scales;
  a.xq_g = xq_g;
  return launch_linear(a, ws, ws_bytes, dev, static_cast<cudaStream_t>(stream));
}

}  // namespace

extern "C" {

nvfp4rl_status nvfp4_amax(const void* x, int32_t dtype, int64_t n, float* amax, void* stream) {
  if (!amax) return NVFP4RL_ERR_INVALID_ARG;
  if (dtype != NVFP4RL_BF16 && dtype != NVFP4RL_F32) return NVFP4RL_ERR_INVALID_ARG;
  if (n < 0 || (n > 0 && !x)) return NVFP4RL_ERR_INVALID_ARG;
  if (n % 16 != 0) return NVFP4RL_ERR_UNSUPPORTED_SHAPE;
  if (!aligned16(x) || (reinterpret_cast<uintptr_t>(amax) & 3u)) return NVFP4RL_ERR_MISALIGNED;
  if (overlap(amax, 4, x, static_cast<size_t>(n) * (dtype == NVFP4RL_BF16 ? 2 : 4))) return NVFP4RL_ERR_ALIAS;
  DeviceInfo dev;
  nvfp4rl_status st = current_device(&dev);
  if (st != NVFP4RL_OK) return st;
  return launch_amax(x, dtype, n, reinterpret_cast<uint32_t*>(amax), dev, static_cast<cudaStream_t>(stream));
}

nvfp4rl_status nvfp4_quantize(const void* x, int32_t dtype, int64_t rows, int64_t cols, uint8_t* codes,
                              uint8_t* scales, float* g, const float* amax_in, void* workspace,
                              size_t workspace_bytes, void* stream) {
  return quantize_common(x, dtype, rows, cols, nullptr, false, codes, scales, g, amax_in, workspace,
                         workspace_bytes, stream);
}

nvfp4rl_status nvfp4_quantize_guided(const void* x, int32_t dtype, int64_t rows, int64_t cols,
                                     const uint32_t* mask, uint8_t* codes, uint8_t* scales, float* g,
                                     const float* amax_in, void* workspace, size_t workspace_bytes,
                                     void* stream) {
  return quantize_common(x, dtype, rows, cols, mask, true, codes, scales, g, amax_in, workspace, workspace_bytes,
                         stream);
}

nvfp4rl_status nvfp4_quantize_record(const void* x, int32_t dtype, int64_t rows, int64_t cols, uint8_t* codes,
                                     uint8_t* scales, float* g, uint32_t* record, const float* amax_in,
                                     void* workspace, size_t workspace_bytes, void* stream) {
  return quantize_common(x, dtype, rows, cols, nullptr, false, codes, scales, g, amax_in, workspace, workspace_bytes,
                         stream, record, true);
}

nvfp4rl_status nvfp4_quantize_cached(const void* x, int32_t dtype, int64_t rows, int64_t cols, const uint32_t* mask,
                                     const uint8_t* scales, const float* g, uint8_t* codes, void* stream) {
  if (dtype != NVFP4RL_BF16 && dtype != NVFP4RL_F32) return NVFP4RL_ERR_INVALID_ARG;
  if (rows < 0 || cols <= 0) return NVFP4RL_ERR_INVALID_ARG;
  if (cols % 16 != 0) return NVFP4RL_ERR_UNSUPPORTED_SHAPE;
  if (rows == 0) return NVFP4RL_OK;
  if (!x || !mask || !scales || !g || !codes) return NVFP4RL_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(mask) || !aligned16(scales) || !aligned16(codes) ||
      (reinterpret_cast<uintptr_t>(g) & 3u))
    return NVFP4RL_ERR_MISALIGNED;
  const size_t n = static_cast<size_t>(rows) * static_cast<size_t>(cols);
  if (overlap(codes, n / 2, x, n * (dtype == NVFP4RL_BF16 ? 2 : 4)) || overlap(codes, n / 2, mask, (n + 31) / 32 * 4) ||
      overlap(codes, n / 2, scales, n / 16) || overlap(codes, n / 2, g, 4))
    return NVFP4RL_ERR_ALIAS;
  DeviceInfo dev;
  nvfp4rl_status st = current_device(&dev);
  if (st != NVFP4RL_OK) return st;
  return launch_quantize_cached(x, dtype, rows, cols, mask, scales, g, codes, dev, static_cast<cudaStream_t>(stream));
}

nvfp4rl_status ais_mixing(const float* lr, const float* lt, const float* adv, int64_t n, float C, float delta,
                          float gamma, float beta, float* w_out, double* stats, void* workspace,
                          size_t workspace_bytes, void* stream) {
  if (n < 0) return NVFP4RL_ERR_INVALID_ARG;
  if (!(C > 0.0f) || !(delta > 0.0f) || !(gamma > 0.0f) || !(beta >= 0.0f) || !std::isfinite(C) ||
      !std::isfinite(delta) || !std::isfinite(gamma) || !std::isfinite(beta))
    return NVFP4RL_ERR_INVALID_ARG;
  if (n == 0) return NVFP4RL_OK;
  if (!lr || !lt || !adv || !stats) return NVFP4RL_ERR_INVALID_ARG;
  if (!aligned16(lr) || !aligned16(lt) || !aligned16(adv) || (w_out && !aligned16(w_out)) ||
      (reinterpret_cast<uintptr_t>(stats) & 7u))
    return NVFP4RL_ERR_MISALIGNED;
  const size_t need = ais_workspace_bytes();
  if (!workspace || workspace_bytes < need) return NVFP4RL_ERR_WORKSPACE;
  if (!aligned16(workspace)) return NVFP4RL_ERR_MISALIGNED;
  const size_t nb = static_cast<size_t>(n) * 4;
  const void* ins[3] = {lr, lt, adv};
  for (const void* in : ins)
    if ((w_out && overlap(w_out, nb, in, nb)) || overlap(stats, 64, in, nb) || overlap(workspace, need, in, nb))
      return NVFP4RL_ERR_ALIAS;
  if ((w_out && (overlap(w_out, nb, stats, 64) || overlap(w_out, nb, workspace, need))) ||
      overlap(stats, 64, workspace, need))
    return NVFP4RL_ERR_ALIAS;
  DeviceInfo dev;
  nvfp4rl_status st = current_device(&dev);
  if (st != NVFP4RL_OK) return st;
  return launch_ais(lr, lt, adv, n, C, delta, gamma, beta, w_out, stats, workspace, dev,
                    static_cast<cudaStream_t>(stream));
}

nvfp4rl_status nvfp4_kv_append(const uint16_t* k, const uint16_t* v, int64_t B, int64_t Hkv, int64_t D,
                               const int32_t* pos, const float* gk, const float* gv, uint8_t* kc, uint8_t* ks,
                               uint8_t* vc, uint8_t* vs, int64_t Lmax, void* stream) {
  if (B < 0 || Hkv <= 0 || D <= 0 || Lmax <= 0) return NVFP4RL_ERR_INVALID_ARG;
  if (D % 16 != 0) return NVFP4RL_ERR_UNSUPPORTED_SHAPE;
  if (B == 0) return NVFP4RL_OK;
  if (!k || !v || !pos || !gk || !gv || !kc || !ks || !vc || !vs) return NVFP4RL_ERR_INVALID_ARG;
  if (!aligned16(k) || !aligned16(v) || !aligned16(kc) || !aligned16(ks) || !aligned16(vc) || !aligned16(vs) ||
      (reinterpret_cast<uintptr_t>(pos) & 3u) || (reinterpret_cast<uintptr_t>(gk) & 3u) ||
      (reinterpret_cast<uintptr_t>(gv) & 3u))
    return NVFP4RL_ERR_MISALIGNED;
  const size_t rows = static_cast<size_t>(B) * static_cast<size_t>(Lmax) * static_cast<size_t>(Hkv);
  const size_t in_b = static_cast<size_t>(B) * Hkv * D * 2;
  std::vector<std::pair<uintptr_t, uintptr_t>> outs, ins;
  const auto rng = [](const void* p, size_t n) {
    return std::make_pair(reinterpret_cast<uintptr_t>(p), reinterpret_cast<uintptr_t>(p) + n);
  };
  outs = {rng(kc, rows * (D / 2)), rng(ks, rows * (D / 16)), rng(vc, rows * (D / 2)), rng(vs, rows * (D / 16))};
  ins = {rng(k, in_b), rng(v, in_b), rng(pos, static_cast<size_t>(B) * 4), rng(gk, 4), rng(gv, 4)};
  if (any_overlap(outs)) return NVFP4RL_ERR_ALIAS;
  std::sort(outs.begin(), outs.end());
  for (const auto& r : ins)
    if (hits(outs, r.first, r.second)) return NVFP4RL_ERR_ALIAS;
  DeviceInfo dev;
  nvfp4rl_status st = current_device(&dev);
  if (st != NVFP4RL_OK) return st;
  return launch_kv_append(k, v, B, Hkv, D, pos, gk, gv, kc, ks, vc, vs, Lmax, dev, static_cast<cudaStream_t>(stream));
}

nvfp4rl_status nvfp4_kv_decode_attention(const uint16_t* q, const uint8_t* kc, const uint8_t* ks, const float* gk,
                                         const uint8_t* vc, const uint8_t* vs, const float* gv, const int32_t* lens,
                                         int64_t B, int64_t Hq, int64_t Hkv, int64_t D, int64_t Lmax, float scale,
                                         uint16_t* out, void* workspace, size_t workspace_bytes, void* stream) {
  if (B < 0 || Hq <= 0 || Hkv <= 0 || D <= 0 || Lmax <= 0 || !std::isfinite(scale)) return NVFP4RL_ERR_INVALID_ARG;
  if (D != 128 || Hq % Hkv != 0 || Hq / Hkv > 16 || B * Hkv > 65535) return NVFP4RL_ERR_UNSUPPORTED_SHAPE;
  if (B == 0) return NVFP4RL_OK;
  if (!q || !kc || !ks || !gk || !vc || !vs || !gv || !lens || !out) return NVFP4RL_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(kc) || !aligned16(ks) || !aligned16(vc) || !aligned16(vs) || !aligned16(out) ||
      (reinterpret_cast<uintptr_t>(gk) & 3u) || (reinterpret_cast<uintptr_t>(gv) & 3u) ||
      (reinterpret_cast<uintptr_t>(lens) & 3u))
    return NVFP4RL_ERR_MISALIGNED;
  const size_t need = attention_workspace_bytes(B, Hkv, Lmax);
  if (need > 0) {
    if (!workspace || workspace_bytes < need) return NVFP4RL_ERR_WORKSPACE;
    if (!aligned16(workspace)) return NVFP4RL_ERR_MISALIGNED;
  }
  const size_t rows = static_cast<size_t>(B) * static_cast<size_t>(Lmax) * static_cast<size_t>(Hkv);
  const size_t ob = static_cast<size_t>(B) * Hq * D * 2;
  const void* ins[9] = {q, kc, ks, vc, vs, gk, gv, lens, workspace};
  const size_t isz[9] = {ob, rows * (D / 2), rows * (D / 16), rows * (D / 2), rows * (D / 16), 4, 4,
                         static_cast<size_t>(B) * 4, need};
  for (int i = 0; i < 9; ++i)
    if (ins[i] && isz[i] && overlap(out, ob, ins[i], isz[i])) return NVFP4RL_ERR_ALIAS;
  DeviceInfo dev;
  nvfp4rl_status st = current_device(&dev);
  if (st != NVFP4RL_OK) return st;
  return launch_kv_attention(q, kc, ks, gk, vc, vs, gv, lens, B, Hq, Hkv, Lmax, scale, out, workspace, dev,
                             static_cast<cudaStream_t>(stream));
}

nvfp4rl_status nvfp4_quantize_batch(int32_t count, const void* const* x, const int64_t* rows, const int64_t* cols,
                                    int32_t dtype, uint8_t* const* codes, uint8_t* const* scales, float* const* g,
                                    void* workspace, size_t workspace_bytes, void* stream) {
  if (count < 0 || count > kQuantizeBatchMax) return NVFP4RL_ERR_INVALID_ARG;
  if (dtype != NVFP4RL_BF16 && dtype != NVFP4RL_F32) return NVFP4RL_ERR_INVALID_ARG;
  if (count == 0) return NVFP4RL_OK;
  if (!x || !rows || !cols || !codes || !scales || !g) return NVFP4RL_ERR_INVALID_ARG;
  const size_t esz = dtype == NVFP4RL_BF16 ? 2 : 4;
  std::vector<std::pair<uintptr_t, uintptr_t>> outs, ins;
  int live = 0;
  for (int32_t i = 0; i < count; ++i) {
    if (rows[i] < 0 || cols[i] <= 0) return NVFP4RL_ERR_INVALID_ARG;
    if (cols[i] % 16 != 0) return NVFP4RL_ERR_UNSUPPORTED_SHAPE;
    if (rows[i] == 0) continue;
    if (!x[i] || !codes[i] || !scales[i] || !g[i]) return NVFP4RL_ERR_INVALID_ARG;
    if (!aligned16(x[i]) || !aligned16(codes[i]) || !aligned16(scales[i]) || (reinterpret_cast<uintptr_t>(g[i]) & 3u))
      return NVFP4RL_ERR_MISALIGNED;
    const size_t n = static_cast<size_t>(rows[i]) * static_cast<size_t>(cols[i]);
    const auto rng = [](const void* p, size_t b) {
      return std::make_pair(reinterpret_cast<uintptr_t>(p), reinterpret_cast<uintptr_t>(p) + b);
    };
    ins.push_back(rng(x[i], n * esz));
    outs.push_back(rng(codes[i], n / 2));
    outs.push_back(rng(scales[i], n / 16));
    outs.push_back(rng(g[i], 4));
    ++live;
  }
  if (live == 0) return NVFP4RL_OK;
  const size_t need = quantize_batch_workspace_bytes(count);
  if (!workspace || workspace_bytes < need) return NVFP4RL_ERR_WORKSPACE;
  if (!aligned16(workspace)) return NVFP4RL_ERR_MISALIGNED;
  if (any_overlap(outs)) return NVFP4RL_ERR_ALIAS;
  ins.push_back(std::make_pair(reinterpret_cast<uintptr_t>(workspace), reinterpret_cast<uintptr_t>(workspace) + need));
  for (const auto& r : ins)
    if (hits(outs, r.first, r.second)) return NVFP4RL_ERR_ALIAS;
  DeviceInfo dev;
  nvfp4rl_status st = current_device(&dev);
  if (st != NVFP4RL_OK) return st;
  return launch_quantize_batch(count, x, rows, cols, dtype, codes, scales, g, static_cast<uint32_t*>(workspace), dev,
                               static_cast<cudaStream_t>(stream));
}

double aqn_sigma(double sigma0, double sigmaK, int64_t k, int64_t K) {
  if (K <= 0 || !(sigma0 > 0.0) || !(sigmaK > 0.0)) return NAN;
  return sigma0 * std::pow(sigmaK / sigma0, static_cast<double>(k) / static_cast<double>(K));
}

nvfp4rl_status rmsnorm_aqn(const uint16_t* x, int64_t M, int64_t H, const float* w, const float* eps, float sigma,
                           float delta, uint16_t* y, void* stream) {
  if (M < 0 || H <= 0 || !std::isfinite(sigma) || !(delta >= 0.0f) || !std::isfinite(delta))
    return NVFP4RL_ERR_INVALID_ARG;
  if (M == 0) return NVFP4RL_OK;
  if (!x || !w || !y) return NVFP4RL_ERR_INVALID_ARG;
  if (H % 8 != 0 || H > rmsnorm_max_h() || M > 2147483647LL) return NVFP4RL_ERR_UNSUPPORTED_SHAPE;
  if (!aligned16(x) || !aligned16(w) || !aligned16(y) || (eps && !aligned16(eps))) return NVFP4RL_ERR_MISALIGNED;
  const size_t yb = static_cast<size_t>(M) * H * 2;
  if (overlap(y, yb, x, yb) || overlap(y, yb, w, H * 4) || (eps && overlap(y, yb, eps, H * 4)))
    return NVFP4RL_ERR_ALIAS;
  DeviceInfo dev;
  nvfp4rl_status st = current_device(&dev);
  if (st != NVFP4RL_OK) return st;
  return launch_rmsnorm_aqn(x, M, H, w, eps, sigma, delta, y, dev, static_cast<cudaStream_t>(stream));
}

nvfp4rl_status rmsnorm_aqn_quantize(const uint16_t* x, int64_t M, int64_t H, const float* w, const float* eps,
                                    float sigma, float delta, uint16_t* y, uint8_t* codes, uint8_t* scales, float* g,
                                    void* workspace, size_t workspace_bytes, void* stream) {
  if (M < 0 || H <= 0 || !std::isfinite(sigma) || !(delta >= 0.0f) || !std::isfinite(delta))
    return NVFP4RL_ERR_INVALID_ARG;
  if (M == 0) return NVFP4RL_OK;
  if (!x || !w || !y || !codes || !scales || !g) return NVFP4RL_ERR_INVALID_ARG;
  if (H % 16 != 0 || H > rmsnorm_max_h() || M > 2147483647LL) return NVFP4RL_ERR_UNSUPPORTED_SHAPE;
  if (!aligned16(x) || !aligned16(w) || !aligned16(y) || (eps && !aligned16(eps)) || !aligned16(codes) ||
      !aligned16(scales) || (reinterpret_cast<uintptr_t>(g) & 3u))
    return NVFP4RL_ERR_MISALIGNED;
  if (!workspace || workspace_bytes < kQuantizeWorkspace) return NVFP4RL_ERR_WORKSPACE;
  if (!aligned16(workspace)) return NVFP4RL_ERR_MISALIGNED;
  const size_t n = static_cast<size_t>(M) * H;
  const void* outs[4] = {y, codes, scales, g};
  const size_t osz[4] = {n * 2, n / 2, n / 16, 4};
  for (int i = 0; i < 4; ++i) {
    if (overlap(outs[i], osz[i], x, n * 2) || overlap(outs[i], osz[i], w, H * 4) ||
        (eps && overlap(outs[i], osz[i], eps, H * 4)) || overlap(outs[i], osz[i], workspace, kQuantizeWorkspace))
      return NVFP4RL_ERR_ALIAS;
    for (int j = i + 1; j < 4; ++j)
      if (overlap(outs[i], osz[i], outs[j], osz[j])) return NVFP4RL_ERR_ALIAS;
  }
  DeviceInfo dev;
  nvfp4rl_status st = current_device(&dev);
  if (st != NVFP4RL_OK) return st;
  return launch_rmsnorm_quantize(x, M, H, w, eps, sigma, delta, y, codes, scales, g, static_cast<uint32_t*>(workspace),
                                 dev, static_cast<cudaStream_t>(stream));
}

nvfp4rl_status nvfp4_lora_linear(const uint16_t* x, int64_t M, int64_t K, const uint8_t* w_codes,
                                 const uint8_t* w_scales, const float* w_g, int64_t N, const uint16_t* lora_A,
                                 const uint16_t* lora_B, int32_t r, float s, const int32_t* group_offsets,
                                 int32_t num_groups, uint16_t* y, void* workspace, size_t workspace_bytes,
                                 void* stream) {
  return linear_common(false, x, M, K, w_codes, w_scales, w_g, N, lora_A, lora_B, r, s, group_offsets, num_groups,
                       y, workspace, workspace_bytes, stream);
}

nvfp4rl_status nvfp4_lora_linear_w4a4(const uint16_t* x, int64_t M, int64_t K, const uint8_t* w_codes,
                                      const uint8_t* w_scales, const float* w_g, int64_t N,
                                      const uint16_t* lora_A, const uint16_t* lora_B, int32_t r, float s,
                                      const int32_t* group_offsets, int32_t num_groups, uint16_t* y,
                                      void* workspace, size_t workspace_bytes, void* stream) {
  return linear_common(true, x, M, K, w_codes, w_scales, w_g, N, lora_A, lora_B, r, s, group_offsets, num_groups,
                       y, workspace, workspace_bytes, stream);
}

nvfp4rl_status nvfp4_lora_linear_w4a4_quantized(const uint16_t* x, const uint8_t* x_codes, const uint8_t* x_scales,
                                                const float* x_g, int64_t M, int64_t K, const uint8_t* w_codes,
                                                const uint8_t* w_scales, const float* w_g, int64_t N,
                                                const uint16_t* lora_A, const uint16_t* lora_B, int32_t r, float s,
                                                const int32_t* group_offsets, int32_t num_groups, uint16_t* y,
                                                void* workspace, size_t workspace_bytes, void* stream) {
  if (!x_codes || !x_scales || !x_g) return NVFP4RL_ERR_INVALID_ARG;
  return linear_common(true, x, M, K, w_codes, w_scales, w_g, N, lora_A, lora_B, r, s, group_offsets, num_groups, y,
                       workspace, workspace_bytes, stream, x_codes, x_scales, x_g);
}

size_t nvfp4rl_workspace_bytes(int32_t op, int64_t M, int64_t N, int64_t K, int32_t r, int32_t num_groups) {
  if (M < 0 || N < 0 || K < 0 || r < 0 || r > 256 || num_groups < 0 || num_groups > 1024) return 0;
  switch (op) {
    case NVFP4RL_OP_QUANTIZE: return kQuantizeWorkspace;
    case NVFP4RL_OP_QUANTIZE_BATCH: return M <= kQuantizeBatchMax ? quantize_batch_workspace_bytes(M) : 0;
    case NVFP4RL_OP_RMSNORM_QUANTIZE: return kQuantizeWorkspace;
    case NVFP4RL_OP_AIS: return ais_workspace_bytes();
    case NVFP4RL_OP_KV_ATTENTION: return N > 0 && K > 0 ? attention_workspace_bytes(M, N, K) : 0;
    case NVFP4RL_OP_LINEAR_W4A16: return linear_workspace_bytes(false, M, N, K, r, 1);
    case NVFP4RL_OP_LINEAR_W4A4: return linear_workspace_bytes(true, M, N, K, r, num_groups > 0 ? num_groups : 1);
    case NVFP4RL_OP_LINEAR_W4A4_QUANTIZED:
      return linear_workspace_bytes(true, M, N, K, r, num_groups > 0 ? num_groups : 1, true);
    default: return 0;
  }
}

const char* nvfp4rl_status_string(nvfp4rl_status status) {
  switch (status) {
    case NVFP4RL_OK: return "ok";
    case NVFP4RL_ERR_INVALID_ARG: return "invalid argument";
    case NVFP4RL_ERR_MISALIGNED: return "pointer not 16-byte aligned";
    case NVFP4RL_ERR_UNSUPPORTED_SHAPE: return "unsupported shape";
    case NVFP4RL_ERR_WORKSPACE: return "workspace missing or too small";
    case NVFP4RL_ERR_CUDA: return "CUDA error";
    case NVFP4RL_ERR_TIMEOUT: return "device-side wait timed out";
    case NVFP4RL_ERR_ALIAS: return "output overlaps an input";
    case NVFP4RL_ERR_DEVICE: return "device is not compute capability 10.3";
    case NVFP4RL_ERR_RANGE: return "folded LoRA scale (s / (g_x g_w), or s / (2^32 g_w)) out of range";
  }
  return "unknown status";
}

uint64_t nvfp4rl_kernel_launches(void) { return g_launches.load(std::memory_order_relaxed); }

nvfp4rl_status nvfp4rl_selftest_wait_timeout(void* stream) {
  DeviceInfo dev;
  nvfp4rl_status st = current_device(&dev);
  if (st != NVFP4RL_OK) return st;
  wait_timeout_probe_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(dev.status);
  return launch_status();
}

nvfp4rl_status nvfp4rl_device_status(uint32_t* word_out, int32_t clear) {
  if (cudaDeviceSynchronize() != cudaSuccess) return NVFP4RL_ERR_CUDA;
  uint32_t w = 0;
  if (cudaMemcpyFromSymbol(&w, g_device_status, sizeof(w)) != cudaSuccess) return NVFP4RL_ERR_CUDA;
  if (word_out) *word_out = w;
  if (clear) {
    const uint32_t z = 0;
    if (cudaMemcpyToSymbol(g_device_status, &z, sizeof(z)) != cudaSuccess) return NVFP4RL_ERR_CUDA;
  }
  if (w & sm100::kStatusTimeoutMask) return NVFP4RL_ERR_TIMEOUT;
  return w ? NVFP4RL_ERR_RANGE : NVFP4RL_OK;
}

}  // extern "C"
