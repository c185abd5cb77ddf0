// Allocation-free W4A16 LoRA linear: the same computation as nvfp4_lora_linear, with its
// scratch memory in a fixed array of device memory that this library owns, for callers that
// cannot allocate device memory themselves (code running inside another framework's memory
// planner or a restricted runtime that forbids cudaMalloc, code that must not grow the device
// footprint after start-up).
//
// The array below is a file-scope __device__ variable: every GPU that loads this library holds
// it (kNoallocScratchBytes) until the process exits. Host code cannot use its name as a device
// address, so the entry point looks the address up with cudaGetSymbolAddress once per device
// (on the first call on that device, with that device current) and passes it on as the
// workspace. Every call on a device shares the one array; calls that overlap on the GPU (on
// different streams without ordering) race on it.
//
// The W4A16 workspace holds only U = bf16(x A^T), M * max(r, 1) * 2 bytes rounded up to 256 (for
// more than 128 tokens at rank <= 64, the two bf16 parts of the scaled U: twice that): 4 MiB covers
// M * r up to 2^21, or 2^20 in the two-part case (e.g. 16384 tokens at rank 128, 16384 tokens at
// rank 64); larger problems are rejected with NVFP4RL_ERR_WORKSPACE.
#include <mutex>

#include "common.cuh"

namespace {

constexpr size_t kNoallocScratchBytes = size_t(4) << 20;  // 4 MiB

__device__ __align__(256) unsigned char g_noalloc_scratch[kNoallocScratchBytes];

std::mutex g_noalloc_mutex;
void* g_noalloc_ptr[64] = {};

}  // namespace

extern "C" nvfp4rl_status nvfp4_lora_linear_noalloc(const uint16_t* x, int64_t M, int64_t K, const uint8_t* w_codes,
                                                    const uint8_t* w_scales, const float* w_g, int64_t N,
                                                    const uint16_t* lora_A, const uint16_t* lora_B, int32_t r,
                                                    float s, uint16_t* y, void* stream) {
  if (M < 0 || K <= 0 || N <= 0 || r < 0 || r > 256) return NVFP4RL_ERR_INVALID_ARG;
  if (M == 0) return NVFP4RL_OK;
  const size_t need = nvfp4rl_workspace_bytes(NVFP4RL_OP_LINEAR_W4A16, M, N, K, r, 0);
  // A shape the linear does not take: nvfp4_lora_linear reports which argument is wrong, and
  // launches nothing.
  if (need == 0)
    return nvfp4_lora_linear(x, M, K, w_codes, w_scales, w_g, N, lora_A, lora_B, r, s, nullptr, 0, y, nullptr, 0,
                             stream);
  if (need > kNoallocScratchBytes) return NVFP4RL_ERR_WORKSPACE;  // the problem needs more than the fixed array
  // The current device must be one this library's kernels run on before its module is touched.
  nvfp4rl::DeviceInfo dev;
  const nvfp4rl_status ds = nvfp4rl::current_device(&dev);
  if (ds != NVFP4RL_OK) return ds;
  if (dev.device < 0 || dev.device >= 64) return NVFP4RL_ERR_DEVICE;
  void* scratch = nullptr;
  {
    std::lock_guard<std::mutex> lock(g_noalloc_mutex);
    if (!g_noalloc_ptr[dev.device]) {
      void* p = nullptr;
      if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) {
        cudaGetLastError();  // leave no error pending for the next call's launch check
        return NVFP4RL_ERR_CUDA;
      }
      g_noalloc_ptr[dev.device] = p;
    }
    scratch = g_noalloc_ptr[dev.device];
  }
  // Nothing in the workspace has to start at zero: every call writes what it later reads.
  return nvfp4_lora_linear(x, M, K, w_codes, w_scales, w_g, N, lora_A, lora_B, r, s, nullptr, 0, y, scratch,
                           kNoallocScratchBytes, stream);
}

extern "C" size_t nvfp4rl_noalloc_scratch_bytes(void) { return kNoallocScratchBytes; }
