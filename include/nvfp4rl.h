/*
 * nvfp4rl.h -- C ABI of the NVFP4 rollout-linear library (one GB300 GPU, sm_103a).
 *
 * The library implements the quantized rollout linear layer of QeRL-style
 * low-precision RL: NVFP4 block quantization (plain and rollout-guided),
 * AQN-noised RMSNorm, and the NVFP4-weight linear layer with a fused LoRA
 * branch, with 16-bit activations (W4A16) or activations quantized on the fly
 * (W4A4, optionally grouped per MoE expert).
 *
 * Sources of the operations (the pages describe them in prose; the concrete
 * recipe is stated with each entry point):
 *   - "QeRL: Beyond Efficiency -- Quantization-enhanced Reinforcement Learning
 *     for LLMs" explainer (lifetechia.com), sections "NVFP4量子化とLoRA",
 *     "AQNの仕組み" and "ゼロオーバーヘッド：レイヤー正規化への統合";
 *   - "TRACE: rollout-guided quantization-aware training" summary (sns.style),
 *     sections "TRACE の中心的なアイデア" and "仕組みの工学的な理解".
 *
 * Conventions shared by every entry point:
 *   - Memory: every pointer argument is DEVICE memory, allocated and owned by
 *     the caller, and must be 16-byte aligned. The library allocates nothing;
 *     it keeps only per-device cached attributes and kernel resources.
 *   - Streams: `stream` is a cudaStream_t passed as void* (NULL = legacy default
 *     stream). Calls are asynchronous on that stream; outputs are complete when
 *     the stream reaches the call. Inputs are never written.
 *   - bf16 tensors are passed as uint16_t bit patterns, row-major.
 *   - Errors: arguments are validated on the host before any launch; a failed
 *     check returns its status and launches nothing. A launch failure returns
 *     NVFP4RL_ERR_CUDA. Inputs must be finite (not checked on the device).
 *   - Outputs must not overlap inputs (NVFP4RL_ERR_ALIAS).
 *   - Zero-sized problems (rows == 0, M == 0) are valid no-ops.
 *   - Device state: on its first call on a device the library caches that device's attributes,
 *     kernel attributes and the device addresses of its own __device__ variables (the status word,
 *     the allocation-free scratch array). cudaDeviceReset() discards all of them on the GPU side:
 *     after a reset of a device it has been used on, the library must not be called again in that
 *     process.
 *   - Device status: bounded device-side waits report through one status word per device, shared
 *     by every stream and call on that device; nvfp4rl_device_status() synchronizes the device,
 *     reads it and optionally clears it. A timeout is therefore attributed to the device, not to
 *     one call or workspace.
 */
#ifndef NVFP4RL_H_
#define NVFP4RL_H_

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define NVFP4RL_API __attribute__((visibility("default")))
#else
#define NVFP4RL_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum nvfp4rl_status {
  NVFP4RL_OK = 0,
  NVFP4RL_ERR_INVALID_ARG = 1,       /* null pointer, negative size, bad dtype, r or groups out of range */
  NVFP4RL_ERR_MISALIGNED = 2,        /* a pointer is not 16-byte aligned */
  NVFP4RL_ERR_UNSUPPORTED_SHAPE = 3, /* a dimension is not a multiple of what the kernel needs */
  NVFP4RL_ERR_WORKSPACE = 4,         /* workspace missing or smaller than nvfp4rl_workspace_bytes() */
  NVFP4RL_ERR_CUDA = 5,              /* a CUDA runtime call or a kernel launch failed */
  NVFP4RL_ERR_TIMEOUT = 6,           /* a bounded device-side wait ran out (reported by nvfp4rl_device_status) */
  NVFP4RL_ERR_ALIAS = 7,             /* an output buffer overlaps an input buffer */
  NVFP4RL_ERR_DEVICE = 8,            /* the current device is not a compute-capability 10.3 GPU */
  NVFP4RL_ERR_RANGE = 9              /* a folded LoRA scale (W4A4: s / (g_x g_w); W4A16 at
                                        M > 128, r <= 64: s / (2^32 g_w)) exceeded 2^100
                                        (reported by nvfp4rl_device_status) */
} nvfp4rl_status;

/* Element types of quantizer inputs. */
enum { NVFP4RL_BF16 = 0, NVFP4RL_F32 = 1 };

/* Operations for nvfp4rl_workspace_bytes(). */
enum {
  NVFP4RL_OP_QUANTIZE = 0,
  NVFP4RL_OP_LINEAR_W4A16 = 1,
  NVFP4RL_OP_LINEAR_W4A4 = 2,
  NVFP4RL_OP_QUANTIZE_BATCH = 3, /* M = number of tensors */
  NVFP4RL_OP_RMSNORM_QUANTIZE = 4,
  NVFP4RL_OP_AIS = 5,
  NVFP4RL_OP_KV_ATTENTION = 6, /* M = B, N = Hkv, K = Lmax */
  NVFP4RL_OP_LINEAR_W4A4_QUANTIZED = 7
};

/*
 * nvfp4_amax -- per-tensor absolute maximum, the input of the NVFP4 per-tensor
 *   scale g = amax / (6 * 448) (QeRL explainer, "NVFP4量子化とLoRA"; TRACE summary,
 *   "仕組みの工学的な理解": block scaling under one tensor-level scale).
 *   x      [n] bf16 bits or fp32 (dtype), n multiple of 16.
 *   amax   out, one fp32 = max |x_i| (0 for n == 0). Its result can be passed as
 *          amax_in to nvfp4_quantize / nvfp4_quantize_guided.
 */
NVFP4RL_API nvfp4rl_status nvfp4_amax(const void* x, int32_t dtype, int64_t n, float* amax, void* stream);

/*
 * nvfp4_quantize -- NVFP4 block quantization of a rows x cols tensor.
 *   QeRL explainer, "NVFP4量子化とLoRA" (4-bit weights with hardware support);
 *   TRACE summary, "仕組みの工学的な理解" (a few values share one scale, each
 *   value is 4 bits).
 * Recipe: g = fl32(amax / 2688) with amax = max |x| over the tensor (or *amax_in);
 *   for each 16-element block b along a row, s_b = the E4M3 byte nearest to
 *   bamax_b / (6 g) (ties to the even byte, saturating at 448, 0 when g == 0);
 *   each element's 4-bit code = sign bit (bit 3) | the index of the E2M1 grid
 *   point {0,.5,1,1.5,2,3,4,6} nearest to |x| / (E4M3(s_b) g) (ties to the even
 *   index, saturating at 6; code sign|0 when the scale is 0). Both roundings
 *   apply to the exact real quotient.
 * Arguments:
 *   x        [rows][cols] bf16 bits (dtype NVFP4RL_BF16) or fp32 (NVFP4RL_F32).
 *   cols     multiple of 16.
 *   codes    out, [rows][cols/2] bytes; element 2j in the low nibble of byte j.
 *   scales   out, [rows][cols/16] E4M3 bytes.
 *   g        out, one fp32.
 *   amax_in  optional device fp32; when non-NULL it replaces the computed
 *            amax and the tensor is read once (workspace may then be NULL).
 *   workspace >= nvfp4rl_workspace_bytes(NVFP4RL_OP_QUANTIZE, ...) bytes when
 *            amax_in is NULL; scratch, contents undefined between calls.
 */
NVFP4RL_API nvfp4rl_status nvfp4_quantize(const void* x, int32_t dtype, int64_t rows, int64_t cols,
                              uint8_t* codes, uint8_t* scales, float* g, const float* amax_in,
                              void* workspace, size_t workspace_bytes, void* stream);

/*
 * nvfp4_quantize_batch -- nvfp4_quantize of `count` independent tensors in one call: the
 *   re-quantization of a model's linear weights after a training step, before the next
 *   rollout (QeRL explainer, "NVFP4量子化とLoRA": the rollout reads the base weights in
 *   NVFP4). Each tensor has its own amax and g; tensor i's codes, scales and g are exactly
 *   what nvfp4_quantize(x[i], ..., amax_in = NULL) writes for it.
 * Arguments:
 *   count    number of tensors, in [0, 4096].
 *   x, rows, cols, codes, scales, g
 *            HOST arrays of `count` entries (owned by the caller, read during the call only);
 *            entry i describes tensor i with nvfp4_quantize's layout, alignment and shape
 *            rules; the pointers in them are device pointers. rows[i] == 0: tensor i is
 *            skipped (g[i] is left as is).
 *   dtype    NVFP4RL_BF16 or NVFP4RL_F32, for every tensor.
 *   workspace >= nvfp4rl_workspace_bytes(NVFP4RL_OP_QUANTIZE_BATCH, count, 0, 0, 0, 0) bytes,
 *            device, 16-byte aligned; scratch.
 * No output may overlap an input, another output or the workspace (NVFP4RL_ERR_ALIAS).
 * For bf16 one kernel encodes a tensor while it reduces the amax of the next one (the
 * encoding is bound by arithmetic, the amax pass by memory): the smallest tensor first, then
 * the others largest first; the order changes no result.
 */
NVFP4RL_API nvfp4rl_status nvfp4_quantize_batch(int32_t count, const void* const* x, const int64_t* rows,
                                                const int64_t* cols, int32_t dtype, uint8_t* const* codes,
                                                uint8_t* const* scales, float* const* g, void* workspace,
                                                size_t workspace_bytes, void* stream);

/*
 * nvfp4_quantize_guided -- NVFP4 quantization whose rounding direction comes
 *   from a cached 1-bit-per-element mask (TRACE summary, "TRACE の中心的なアイデア":
 *   the trainer reproduces the rollout's rounding decisions from cached mantissa
 *   and scale information; "仕組みの工学的な理解": the rounding direction is a
 *   per-value choice between the two neighbouring grid points).
 * Same as nvfp4_quantize, except for each element's magnitude code: with
 *   a = |x| / (E4M3(s_b) g): a >= 6 gives 6; a grid point a is kept; otherwise
 *   mask bit 1 takes the larger-magnitude neighbour, bit 0 the smaller one.
 *   Scale bytes and g are those of nvfp4_quantize.
 *   mask     [ceil(rows*cols/32)] uint32 words; element i (flat row-major index)
 *            uses bit (i % 32) of word i / 32.
 */
NVFP4RL_API nvfp4rl_status nvfp4_quantize_guided(const void* x, int32_t dtype, int64_t rows, int64_t cols,
                                     const uint32_t* mask, uint8_t* codes, uint8_t* scales, float* g,
                                     const float* amax_in, void* workspace, size_t workspace_bytes,
                                     void* stream);

/*
 * nvfp4_quantize_record -- nvfp4_quantize that also records the direction of every
 *   rounding: the rollout side of TRACE (TRACE summary, "仕組みの工学的な理解": the rollout
 *   engine quantizes and keeps a record of the result, which the training side consults to
 *   round the same way).
 * Codes, scales and g are exactly those of nvfp4_quantize. In addition:
 *   record   out, [ceil(rows*cols/32)] uint32 words, 16-byte aligned; element i (flat row-major
 *            index) sets bit (i % 32) of word i / 32 to 1 when its plain code's magnitude exceeds
 *            |x| / (E4M3(s_b) g) (rounded up in magnitude), else 0 (rounded down, on the grid,
 *            saturated at 6, or a zero scale). The call writes the first rows*cols/8 bytes: when
 *            rows*cols/16 is odd the upper 16 bits of the last word are left as they were.
 *   nvfp4_quantize_guided(x, mask = record) then gives these codes again, and so does
 *   nvfp4_quantize_cached(x, record, scales, g).
 * Other arguments, workspace and errors as nvfp4_quantize; record may overlap nothing else.
 */
NVFP4RL_API nvfp4rl_status nvfp4_quantize_record(const void* x, int32_t dtype, int64_t rows, int64_t cols,
                                                 uint8_t* codes, uint8_t* scales, float* g, uint32_t* record,
                                                 const float* amax_in, void* workspace, size_t workspace_bytes,
                                                 void* stream);

/*
 * nvfp4_quantize_cached -- the training side of TRACE: codes of x rounded as a cache says
 *   (TRACE summary, "TRACE の中心的なアイデア": rounding decisions guided by the rollout's cached
 *   mantissa and scale information), in one pass over x: no amax, no scale search.
 *   codes[i] = guided code of x[i] (nvfp4_quantize_guided's rule) for the real scale
 *   E4M3(s_b) g with s_b = scales[block of i] and g = *g as given; a byte above 0x7E (never
 *   written by the quantizer) is read as 0x7E, and g <= 0 or NaN gives sign|0 everywhere.
 *   x        [rows][cols] bf16 bits or fp32 (dtype), 16-byte aligned; cols multiple of 16.
 *   mask     [ceil(rows*cols/32)] uint32 words (record layout), 16-byte aligned.
 *   scales   [rows][cols/16] E4M3 bytes, 16-byte aligned (e.g. from nvfp4_quantize_record).
 *   g        device fp32 (e.g. from nvfp4_quantize_record), 4-byte aligned.
 *   codes    out, [rows][cols/2] bytes, 16-byte aligned; may overlap no input.
 * No workspace. Errors: NVFP4RL_ERR_INVALID_ARG (bad dtype, negative rows, NULL pointer),
 *   NVFP4RL_ERR_UNSUPPORTED_SHAPE (cols % 16), NVFP4RL_ERR_MISALIGNED, NVFP4RL_ERR_ALIAS.
 */
NVFP4RL_API nvfp4rl_status nvfp4_quantize_cached(const void* x, int32_t dtype, int64_t rows, int64_t cols,
                                                 const uint32_t* mask, const uint8_t* scales, const float* g,
                                                 uint8_t* codes, void* stream);

/*
 * ais_mixing -- the adaptive importance-sampling correction of a batch of n tokens (AIS summary,
 *   section 2.1 "混合係数" and section 2.2 "GRPO への統合"):
 *     rho_i = exp(logp_train[i] - logp_rollout[i]),  w_i = min(rho_i, C),
 *     alpha_ess = (1 + CV^2(w))^-1/2,  alpha_mis = min(1, mean|logp_train - logp_rollout| / delta),
 *     dsigma = std(w A) / std(A) - 1 (0 when std(A) = 0),  alpha_var = max(0, (dsigma - gamma) / gamma),
 *     alpha = clip(alpha_ess - beta alpha_var, 0, 1) alpha_mis,  w~_i = 1 + alpha (w_i - 1),
 *   means and standard deviations over the n tokens with weight 1/n.
 * Arguments:
 *   logp_rollout, logp_train, adv  device fp32 [n], 16-byte aligned: the sampled tokens' log-probs
 *            under the rollout and the training policy, and their advantages.
 *   n        tokens (>= 0; 0: nothing is written).
 *   C, delta, gamma  > 0 and finite; beta >= 0 and finite (else NVFP4RL_ERR_INVALID_ARG).
 *   w_out    out, device fp32 [n], 16-byte aligned, or NULL (statistics only).
 *   stats    out, device fp64 [8], 8-byte aligned: alpha, alpha_ess, alpha_mis, alpha_var,
 *            mean |logp_train - logp_rollout|, CV^2(w), dsigma, mean(w).
 *   workspace >= nvfp4rl_workspace_bytes(NVFP4RL_OP_AIS, 0, 0, 0, 0, 0) bytes, device, 16-byte
 *            aligned; scratch.
 * Outputs may overlap no input, each other or the workspace (NVFP4RL_ERR_ALIAS). The sums are
 * fp32 over 16-token chunks folded into compensated fp32 sums per thread, and (hi, lo) fp32 pairs
 * across threads and CTAs, added in a fixed
 * order: the result does not depend on timing. alpha and the ratios are formed in fp32 from
 * fp64 means. Three kernels chained by programmatic dependent launch; no device-side waits.
 */
NVFP4RL_API nvfp4rl_status ais_mixing(const float* logp_rollout, const float* logp_train, const float* adv,
                                      int64_t n, float C, float delta, float gamma, float beta, float* w_out,
                                      double* stats, void* workspace, size_t workspace_bytes, void* stream);

/*
 * nvfp4_kv_append -- writes one token's keys and values per sequence into an NVFP4 KV cache (TRACE
 *   summary, "実験結果と性能": rollouts with FP4 weights, activations and KV cache). Each new row of
 *   a head is encoded like nvfp4_quantize with the per-tensor scale *gk (keys) or *gv (values) as
 *   given (a calibrated constant: a growing cache cannot re-derive g from its amax):
 *   cache row (b, pos[b], h) = NVFP4(k[b][h][:]) and likewise for v.
 * Arguments:
 *   k, v     device bf16 [B][Hkv][D], 16-byte aligned; D a multiple of 16.
 *   pos      device int32 [B]: the cache row of each sequence's new token; a sequence whose pos is
 *            outside [0, Lmax) is skipped (nothing written for it).
 *   gk, gv   device fp32 scalars (g <= 0 or NaN: every code is sign|0, every scale byte 0).
 *   k_codes, v_codes   device [B][Lmax][Hkv][D/2] bytes; k_scales, v_scales [B][Lmax][Hkv][D/16]
 *            E4M3 bytes; all 16-byte aligned. Only the rows (b, pos[b], *) are written.
 * Errors: NVFP4RL_ERR_INVALID_ARG (negative sizes, NULL pointers), NVFP4RL_ERR_UNSUPPORTED_SHAPE
 *   (D % 16), NVFP4RL_ERR_MISALIGNED, NVFP4RL_ERR_ALIAS (a cache overlapping an input or another
 *   cache array).
 */
NVFP4RL_API nvfp4rl_status nvfp4_kv_append(const uint16_t* k, const uint16_t* v, int64_t B, int64_t Hkv, int64_t D,
                                           const int32_t* pos, const float* gk, const float* gv, uint8_t* k_codes,
                                           uint8_t* k_scales, uint8_t* v_codes, uint8_t* v_scales, int64_t Lmax,
                                           void* stream);

/*
 * nvfp4_kv_decode_attention -- one decode step of attention over an NVFP4 KV cache:
 *   out[b][h] = softmax(scale * q[b][h] . K^[b, t, h / (Hq/Hkv)]) . V^[b, t, h / (Hq/Hkv)] over
 *   t < lens[b], K^ and V^ the dequantized cache rows (E2M1 x E4M3(s) x g).
 * Arguments:
 *   q        device bf16 [B][Hq][D], 16-byte aligned; D must be 128; Hq a multiple of Hkv with
 *            Hq / Hkv <= 16; B * Hkv <= 65535.
 *   k_codes, k_scales, v_codes, v_scales  the cache as nvfp4_kv_append writes it; gk, gv its scales.
 *            Scale bytes are 0x00 .. 0x7E as the encoder writes them; other bytes give unspecified
 *            (finite or not) results but no fault.
 *   lens     device int32 [B]: tokens attended per sequence, clamped to [0, Lmax]; 0 gives zeros.
 *   scale    softmax scale (typically 1/sqrt(D)), finite.
 *   out      device bf16 [B][Hq][D], 16-byte aligned; may overlap no input.
 *   workspace >= nvfp4rl_workspace_bytes(NVFP4RL_OP_KV_ATTENTION, B, Hkv, Lmax, 0, 0) bytes (may be 0
 *            and NULL), device, 16-byte aligned; scratch.
 * Scores and the softmax are fp32 (exp2 on scores prescaled by log2 e); the products P V take P
 *   rounded to f16; K and V are dequantized exactly (f16), q enters as f16 scaled by a power of two
 *   (exact for every element above 2^-31 of the group's max |q|). Long caches are split into spans
 *   merged by a second kernel. B * Lmax must stay below 2^31 - 64 (32-bit copy coordinates).
 * Errors: NVFP4RL_ERR_INVALID_ARG, NVFP4RL_ERR_UNSUPPORTED_SHAPE, NVFP4RL_ERR_MISALIGNED,
 *   NVFP4RL_ERR_WORKSPACE, NVFP4RL_ERR_ALIAS.
 */
NVFP4RL_API nvfp4rl_status nvfp4_kv_decode_attention(const uint16_t* q, const uint8_t* k_codes,
                                                     const uint8_t* k_scales, const float* gk,
                                                     const uint8_t* v_codes, const uint8_t* v_scales,
                                                     const float* gv, const int32_t* lens, int64_t B, int64_t Hq,
                                                     int64_t Hkv, int64_t D, int64_t Lmax, float scale,
                                                     uint16_t* out, void* workspace, size_t workspace_bytes,
                                                     void* stream);

/*
 * aqn_sigma -- AQN exponential noise schedule (QeRL explainer, "AQNの仕組み":
 *   large noise early, small noise late): sigma_k = sigma0 * (sigmaK/sigma0)^(k/K),
 *   k = 0..K. Host function, no device work. Returns NaN for K <= 0 or
 *   non-positive sigmas.
 */
NVFP4RL_API double aqn_sigma(double sigma0, double sigmaK, int64_t k, int64_t K);

/*
 * rmsnorm_aqn -- RMSNorm with adaptive quantization noise folded into its
 *   weight (QeRL explainer, "ゼロオーバーヘッド：レイヤー正規化への統合":
 *   X_noise = (Z_noise + w) * X / sqrt(sum(X^2) + delta); the mean of squares is
 *   used, as in standard RMSNorm).
 *   y[m][j] = bf16( (w[j] + sigma * eps[j]) * x[m][j] / sqrt(mean_j x[m][j]^2 + delta) )
 *   x    [M][H] bf16 bits; H multiple of 8.
 *   w    [H] fp32 norm weight.  eps [H] fp32 standard-normal draws, or NULL (no noise).
 *   y    out, [M][H] bf16 bits.
 *   w + sigma*eps and the statistics are formed in fp32.
 */
NVFP4RL_API nvfp4rl_status rmsnorm_aqn(const uint16_t* x, int64_t M, int64_t H, const float* w, const float* eps,
                           float sigma, float delta, uint16_t* y, void* stream);

/*
 * rmsnorm_aqn_quantize -- rmsnorm_aqn followed by nvfp4_quantize of its output, the activation
 *   operand of a W4A4 linear (TRACE summary, "論文が取り組む課題": FP4 activations; QeRL
 *   explainer, "ゼロオーバーヘッド：レイヤー正規化への統合": the noise lives in the norm).
 *   y is exactly what rmsnorm_aqn writes; codes, scales and g are exactly what
 *   nvfp4_quantize(y, ...) writes (amax over all of y).
 *   Arguments as rmsnorm_aqn and nvfp4_quantize; H a multiple of 16, at most 8192.
 *   workspace >= nvfp4rl_workspace_bytes(NVFP4RL_OP_RMSNORM_QUANTIZE, 0, 0, 0, 0, 0) bytes.
 *   When every SM's share of y fits in its shared memory (e.g. 4096 x 3584), one cooperative
 *   kernel keeps y on chip between the norm and the encoding (x read once, y and the codes
 *   written once); otherwise RMSNorm-AQN, the amax and the encoding run one after another.
 */
NVFP4RL_API nvfp4rl_status rmsnorm_aqn_quantize(const uint16_t* x, int64_t M, int64_t H, const float* w,
                                                const float* eps, float sigma, float delta, uint16_t* y,
                                                uint8_t* codes, uint8_t* scales, float* g, void* workspace,
                                                size_t workspace_bytes, void* stream);

/*
 * nvfp4_lora_linear -- W4A16 linear layer with the LoRA branch fused
 *   (QeRL explainer, "NVFP4量子化とLoRA": frozen NVFP4 base weights plus
 *   trainable low-rank factors):
 *   Y = x deq(W)^T + s (x A^T) B^T,  deq(W)[n][k] = e2m1(code) * E4M3(s_b) * w_g.
 *   x        [M][K] bf16 bits; K multiple of 256 (one 256-K pipeline stage); M <= 65535.
 *   w_codes  [N][K/2], w_scales [N][K/16]: as written by nvfp4_quantize; N multiple of 128.
 *   w_g      one fp32 (device), the tensor's g.
 *   lora_A   [r][K] bf16 bits, lora_B [N][r] bf16 bits; r = 0 (no LoRA, A and B may then be
 *            NULL) or a multiple of 16 up to 128 (other ranks in [0, 256]:
 *            NVFP4RL_ERR_UNSUPPORTED_SHAPE; outside it: NVFP4RL_ERR_INVALID_ARG).
 *   y        out, [M][N] bf16 bits.
 *   group_offsets, num_groups: must be NULL / 0 (grouped W4A16 is not provided).
 *   workspace >= nvfp4rl_workspace_bytes(NVFP4RL_OP_LINEAR_W4A16, M, N, K, r, 0): U = bf16(x A^T),
 *            or on 256-token tiles (below) the two bf16 parts of c U, scratch, contents undefined
 *            between calls.
 * For M > 128 with r <= 64, where 256-token tiles fill half the SMs or K / 256 >= 64, the call
 *   works on 256-token tiles and folds the LoRA branch into the base product's accumulator: U
 *   (x A^T as accumulated in fp32, not rounded to bf16) enters as the two bf16 parts
 *   hi = bf16(c U), lo = bf16(c U - hi) of c U, c = s / (2^32 w_g) (c = s when w_g = 0), i.e. to
 *   ~2^-17 relative of c U, as the W4A4 call does. |c| above 2^100 (weights with amax below ~1e-36) sets the range bit of the device
 *   status word (NVFP4RL_ERR_RANGE from nvfp4rl_device_status).
 * Deterministic: split-K partial tiles are summed in a fixed order, so equal inputs give equal bits.
 */
NVFP4RL_API nvfp4rl_status nvfp4_lora_linear(const uint16_t* x, int64_t M, int64_t K, const uint8_t* w_codes,
                                 const uint8_t* w_scales, const float* w_g, int64_t N,
                                 const uint16_t* lora_A, const uint16_t* lora_B, int32_t r, float s,
                                 const int32_t* group_offsets, int32_t num_groups, uint16_t* y,
                                 void* workspace, size_t workspace_bytes, void* stream);

/*
 * nvfp4_lora_linear_w4a4 -- the W4A4 variant: x is quantized on the fly with
 *   the nvfp4_quantize recipe (one per-tensor g_x over all M rows), the base
 *   GEMM runs on FP4 x FP4 with the block scales, and the LoRA branch uses the
 *   unquantized bf16 x (TRACE summary, "論文が取り組む課題" and "実験結果と性能":
 *   FP4 weights and activations in the rollout):
 *   Y = deq(quant(x)) deq(W)^T + s (x A^T) B^T.
 *   Arguments, shape rules and determinism as nvfp4_lora_linear, plus grouping:
 *   group_offsets  NULL (dense) or device int32 [num_groups + 1], non-decreasing,
 *                  offsets[0] == 0, offsets[num_groups] == M: rows
 *                  [offsets[e], offsets[e+1]) use expert e's weights
 *                  w_codes + e*N*K/2, w_scales + e*N*K/16, w_g[e].
 *                  Grouped calls take r == 0 (no LoRA). num_groups in [1, 1024].
 *   workspace >= nvfp4rl_workspace_bytes(NVFP4RL_OP_LINEAR_W4A4, M, N, K, r, num_groups).
 *   The LoRA branch is added inside the FP4 product's fp32 accumulator: with alpha = g_x w_g,
 *   c = s / alpha and P the product of the E2M1 codes times their E4M3 block scales (deq without
 *   the two g's), Y = alpha (P + (c U) B^T), where c U (U = bf16(x A^T)) enters as the sum of two
 *   bf16 parts (~2^-17 relative). alpha == 0 (an all-zero x or weight) gives Y = s U B^T. If |c| > 2^100
 *   (the product of the two tensors' amax below ~1e-23 times |s|) the result may overflow and the
 *   call sets the range bit of the device status word (nvfp4rl_device_status ->
 *   NVFP4RL_ERR_RANGE).
 */
NVFP4RL_API nvfp4rl_status nvfp4_lora_linear_w4a4(const uint16_t* x, int64_t M, int64_t K, const uint8_t* w_codes,
                                      const uint8_t* w_scales, const float* w_g, int64_t N,
                                      const uint16_t* lora_A, const uint16_t* lora_B, int32_t r, float s,
                                      const int32_t* group_offsets, int32_t num_groups, uint16_t* y,
                                      void* workspace, size_t workspace_bytes, void* stream);

/*
 * nvfp4_lora_linear_w4a4_quantized -- nvfp4_lora_linear_w4a4 on activations that are already in
 *   NVFP4: the rollout's normalized activations quantized once (e.g. by rmsnorm_aqn_quantize) and
 *   shared by every linear that reads them (TRACE summary, "論文が取り組む課題" and "実験結果と性能":
 *   FP4 activations in the rollout; QeRL explainer, "NVFP4量子化とLoRA": the LoRA branch).
 *   Y = deq(x_codes, x_scales, x_g) deq(W)^T + s (x A^T) B^T.
 *   x_codes  [M][K/2], x_scales [M][K/16] (16-byte aligned), x_g one fp32 (4-byte aligned): the
 *            NVFP4 encoding of the activations as nvfp4_quantize / rmsnorm_aqn_quantize write it.
 *   x        [M][K] bf16 bits, the unquantized activations, read by the LoRA branch only; may be NULL
 *            when r == 0.
 *   Other arguments, shape rules, grouping and determinism as nvfp4_lora_linear_w4a4; given the codes
 *   that nvfp4_lora_linear_w4a4 would compute from x, the result is the same bits.
 *   workspace >= nvfp4rl_workspace_bytes(NVFP4RL_OP_LINEAR_W4A4_QUANTIZED, M, N, K, r, num_groups)
 *            (the two bf16 parts of c U and the grouped tile map; no activation codes); it may overlap no input.
 */
NVFP4RL_API nvfp4rl_status nvfp4_lora_linear_w4a4_quantized(
    const uint16_t* x, const uint8_t* x_codes, const uint8_t* x_scales, const float* x_g, int64_t M, int64_t K,
    const uint8_t* w_codes, const uint8_t* w_scales, const float* w_g, int64_t N, const uint16_t* lora_A,
    const uint16_t* lora_B, int32_t r, float s, const int32_t* group_offsets, int32_t num_groups, uint16_t* y,
    void* workspace, size_t workspace_bytes, void* stream);

/* Workspace bytes an operation needs for these sizes (0 on invalid sizes). */
NVFP4RL_API size_t nvfp4rl_workspace_bytes(int32_t op, int64_t M, int64_t N, int64_t K, int32_t r, int32_t num_groups);

/*
 * nvfp4rl_selftest_wait_timeout -- failure-path self-test (the pages have no counterpart):
 *   launches one small kernel on `stream` in which a thread waits, through the same bounded
 *   wait every pipeline kernel uses, on a barrier that nothing ever completes. After 1 ms
 *   the wait gives up, sets its bit in the device status word and the kernel returns, so
 *   the next nvfp4rl_device_status() reports NVFP4RL_ERR_TIMEOUT and the context stays
 *   usable. Returns the launch status.
 */
NVFP4RL_API nvfp4rl_status nvfp4rl_selftest_wait_timeout(void* stream);

/* Static, human-readable name of a status code. */
NVFP4RL_API const char* nvfp4rl_status_string(nvfp4rl_status status);

/*
 * nvfp4rl_device_status -- synchronizes the current device and reports the
 *   library's device-side error word: NVFP4RL_ERR_TIMEOUT if a bounded wait in
 *   a kernel ran out since the last clear, else NVFP4RL_ERR_RANGE if a folded LoRA
 *   scale was out of range, else NVFP4RL_OK. *word_out (may be NULL) receives
 *   the raw word (bits 0-4: timeouts, bit 5: range); clear != 0 resets it.
 */
NVFP4RL_API nvfp4rl_status nvfp4rl_device_status(uint32_t* word_out, int32_t clear);

/*
 * nvfp4_lora_linear_noalloc -- nvfp4_lora_linear without a caller-supplied workspace, for
 *   callers that cannot allocate device memory (code inside another framework's memory
 *   planner, restricted runtimes that forbid cudaMalloc, code that must not grow its device
 *   footprint after start-up). The pages have no counterpart: this is a deployment entry
 *   point of this library, not part of the method.
 *   Same arguments and result as nvfp4_lora_linear (dense only), bit for bit. The scratch lives
 *   in a fixed array of nvfp4rl_noalloc_scratch_bytes() (4 MiB) that every GPU loading this
 *   library holds until the process exits. Nothing is allocated by the call.
 *   - Returns NVFP4RL_ERR_WORKSPACE when the problem needs more scratch than the array
 *     (nvfp4rl_workspace_bytes(NVFP4RL_OP_LINEAR_W4A16, ...) > 4 MiB, i.e. M * r > 2^21, or
 *     M * r > 2^20 on 256-token tiles, where the workspace holds two parts of U).
 *   - The first call on a device checks that it is a compute-capability 10.3 GPU
 *     (NVFP4RL_ERR_DEVICE otherwise) and looks up the array's device address
 *     (cudaGetSymbolAddress); make that first call before any stream capture. The address is
 *     kept for the process: do not use this entry point after cudaDeviceReset() of that device.
 *   - All calls on a device share the array and each overwrites it: calls that may overlap
 *     on the GPU (unordered streams) race and must not be issued.
 */
NVFP4RL_API nvfp4rl_status nvfp4_lora_linear_noalloc(const uint16_t* x, int64_t M, int64_t K, const uint8_t* w_codes,
                                                     const uint8_t* w_scales, const float* w_g, int64_t N,
                                                     const uint16_t* lora_A, const uint16_t* lora_B, int32_t r,
                                                     float s, uint16_t* y, void* stream);

/* Bytes of the fixed scratch array nvfp4_lora_linear_noalloc uses (4 MiB). Host only. */
NVFP4RL_API size_t nvfp4rl_noalloc_scratch_bytes(void);

/*
 * nvfp4rl_kernel_launches -- diagnostic: number of kernels this library has
 *   launched in this process (all devices, all streams). Host only.
 */
NVFP4RL_API uint64_t nvfp4rl_kernel_launches(void);

#ifdef __cplusplus
}
#endif

#endif /* NVFP4RL_H_ */
