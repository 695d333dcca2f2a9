/*
 * qerl.h -- C ABI of libqerl: the NVFP4 weight-only linear layer with a LoRA
 * branch and Adaptive Quantization Noise, for NVIDIA GB300 (sm_103a).
 *
 * The operation (QeRL, "QeRL: Beyond Efficiency -- Quantization-enhanced
 * Reinforcement Learning for LLMs", paper-graph-ui digest, section 3.4):
 *
 *   y = x~ . dequant(Wq)^T + (alpha / r) . (x~ . A^T) . B^T,   x~ = bf16(x (.) (1 + z))
 *
 *   dequant: "NVFP4 Quantization", Eq. 6: W_hat = S_FP32 * (S_E4M3 (.) W~),
 *            E2M1 codes, one E4M3 scale per 16 contiguous elements along K,
 *            one FP32 tensor scale.
 *   LoRA:    "Low-Rank Adaptation (LoRA) Within Quantized Layers", Eq. 2:
 *            W + BA with B in R^{d x r} and A in R^{r x k} (d = N output,
 *            k = K input features), so the forward of an input row x is
 *            x W^T + x A^T B^T; both branches see the same noisy activations.
 *            A is r x K and B is N x r, row-major (the layout of a PEFT
 *            lora_A / lora_B weight).
 *   noise:   "Adaptive Quantization Noise (AQN)", Eq. 7 (one Gaussian value
 *            per input channel), Eq. 8 (exponential decay of sigma), and
 *            "Noise Merging", Eq. 10-12 (the noise merged into the RMSNorm
 *            scale acts as the per-input-channel factor (1 + z)).
 *
 * Conventions for every call:
 *   - The caller owns every buffer; the library never allocates or frees
 *     memory and keeps no global state.  Pointers marked "device" must be
 *     CUDA device (or managed) memory of the current device.
 *   - All device work is asynchronous and ordered on `stream` (a
 *     cudaStream_t passed as void*; NULL = the legacy default stream).
 *   - Argument errors are detected on the host and returned immediately; no
 *     work is enqueued then.  Errors found by a kernel (a non-finite weight,
 *     a wait that timed out) are recorded in a status word inside the
 *     caller's workspace and read back with qerl_read_status().
 *   - Matrices are row-major.  bf16 values are IEEE bfloat16 bit patterns.
 */
#ifndef QERL_H
#define QERL_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define QERL_API __attribute__((visibility("default")))
#else
#define QERL_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    QERL_OK = 0,
    QERL_ERR_INVALID_ARGUMENT = 1, /* null pointer, negative size, bad dtype, ld too small */
    QERL_ERR_UNSUPPORTED_SHAPE = 2, /* K not a multiple of the required block, r too large */
    QERL_ERR_MISALIGNED = 3,        /* a pointer or leading dimension breaks the stated alignment */
    QERL_ERR_CUDA = 4,              /* a CUDA runtime call failed (the CUDA error is not cleared) */
    QERL_ERR_TIMEOUT = 5,           /* a kernel's bounded wait expired (recorded in the status word) */
    QERL_ERR_NONFINITE = 6,         /* NaN or Inf in the weights (recorded in the status word) */
    QERL_ERR_WORKSPACE = 7,         /* workspace missing or smaller than the *_workspace_size() */
    QERL_ERR_RANGE = 8              /* a weight the packed layout cannot hold (MXFP4 scale span; status word) */
} qerl_status;

typedef enum { QERL_F32 = 0, QERL_BF16 = 1 } qerl_dtype;
/* Element code of a packed weight (qerl_linear_desc.w_format): E2M1
 * (NVFP4, and MXFP4 after qerl_mxfp4_pack) or the NF4 level table. */
typedef enum { QERL_W_NVFP4 = 0, QERL_W_NF4 = 1 } qerl_w_format;

/* Human-readable name of a status code (static string, never NULL). */
QERL_API const char* qerl_status_string(int status);

/* ABI version of this header (major * 100 + minor). */
QERL_API int qerl_version(void);

/* ========================================================================
 * NVFP4 quantization ("NVFP4 Quantization", Eq. 6; the encoder is the
 * library's reading, since the digest gives only the decoder):
 *   S     = amax(|W|) / (6 * 448)           (E2M1 q_max 6 times E4M3 max 448;
 *                                            S = 1 if that is 0)
 *   r_b   = (amax_b / 6) / S                 per 16-element block b along K
 *   s_b   = E4M3(r_b)  round-to-nearest-even, saturating at 448
 *   c     = E2M1(w / (S * dec(s_b)))  nearest level, ties to the even code,
 *           saturating at 6; a value rounding to zero is code 0x0 (never -0)
 * All arithmetic is IEEE fp32 in exactly that order, so results are
 * bit-reproducible.
 *
 * W       device, n x k, dtype w_dtype (QERL_F32 or QERL_BF16), row stride
 *         ld_w elements; 16-byte aligned, ld_w * sizeof(elem) % 16 == 0.
 * codes   device, n x k/2 bytes, row-major; element 2j in the low nibble of
 *         byte j, element 2j+1 in the high nibble.  E2M1 nibble: sign bit 3,
 *         exponent bits 2..1, mantissa bit 0.  16-byte aligned.
 * scales  device, n x k/16 bytes (E4M3 bit patterns), row-major.
 * tensor_scale  device, one float (S).  Written by qerl_nvfp4_quantize;
 *         read by qerl_nvfp4_quantize_with_scale.
 * workspace device, >= qerl_nvfp4_quantize_workspace_size() bytes,
 *         256-byte aligned, zero-filled before its first use.
 * Requires k % 32 == 0, n >= 0, ld_w >= k.  A non-finite weight sets
 * QERL_ERR_NONFINITE in the workspace status word; tensor_scale is then NaN
 * and codes/scales are unspecified.
 * ======================================================================== */
QERL_API size_t qerl_nvfp4_quantize_workspace_size(void);

QERL_API qerl_status qerl_nvfp4_quantize(const void* W, int w_dtype, int64_t n, int64_t k, int64_t ld_w,
                                uint8_t* codes, uint8_t* scales, float* tensor_scale,
                                void* workspace, size_t ws_bytes, void* stream);

/* Same encoding with a caller-provided tensor scale (e.g. the S of a larger
 * tensor this W is a shard of).  *tensor_scale must be finite and > 0. */
QERL_API qerl_status qerl_nvfp4_quantize_with_scale(const void* W, int w_dtype, int64_t n, int64_t k, int64_t ld_w,
                                           const float* tensor_scale, uint8_t* codes, uint8_t* scales,
                                           void* workspace, size_t ws_bytes, void* stream);

/* amax(|W|) into *amax (device float), e.g. to combine shards before
 * computing S = amax / 2688.  NaN/Inf give a non-finite *amax. */
QERL_API qerl_status qerl_nvfp4_amax(const void* W, int w_dtype, int64_t n, int64_t k, int64_t ld_w, float* amax,
                            void* workspace, size_t ws_bytes, void* stream);

/* The tensor scale of a weight from its amax: S = amax / 2688 in fp32 (S = 1
 * if that is 0), the rule qerl_nvfp4_quantize applies.  amax and tensor_scale
 * are device floats.  For a weight sharded across devices (a column- or
 * row-parallel linear): each shard's qerl_nvfp4_amax, an all-reduce(max) of
 * those, this call, then qerl_nvfp4_quantize_with_scale on every shard gives
 * codes and scales bit-identical to quantizing the whole tensor.  A negative
 * or non-finite amax gives S = NaN (which _with_scale then rejects). */
QERL_API qerl_status qerl_nvfp4_tensor_scale(const float* amax, float* tensor_scale, void* stream);

/* ========================================================================
 * Packed weights for the linear (a layout of the same codes and scales; no
 * counterpart in the paper, which fixes the format, not its byte order).
 *
 * One contiguous 18432-byte block per (128-row tile t, 256-wide K stage g),
 * blocks in row-tile-major order: block (t, g) at (t * ceil(k/256) + g) * 18432.
 *   bytes [0, 16384): for row r (0..127) of the tile, the 128 code bytes of
 *       K range [256 g, 256 g + 256) (two codes per byte, even k in the low
 *       nibble, as qerl_nvfp4_quantize writes them) at r * 128, with 16-byte
 *       chunk c stored at chunk position c XOR (r mod 8);
 *   bytes [16384, 18432): the E4M3 scales of the stage as pairs: pair p
 *       (16-element blocks 2p and 2p+1) of row r at 16384 + p * 256 + 2 r.
 * Rows past n and columns past k are zero.  Each block is the exact image the
 * linear's kernel stages in shared memory, so one bulk copy moves it.
 *
 * qerl_nvfp4_packed_size: bytes of the packed form of an n x k weight
 * (ceil(n/128) * ceil(k/256) * 18432).
 * qerl_nvfp4_pack: codes [n][k/2] (16-byte aligned) and scales [n][k/16]
 * (4-byte aligned) as written by qerl_nvfp4_quantize -> packed (16-byte
 * aligned, qerl_nvfp4_packed_size bytes, caller-allocated device memory).
 * Requires k % 64 == 0 and k <= 65536.  Asynchronous on `stream`.
 * ======================================================================== */
QERL_API size_t qerl_nvfp4_packed_size(int64_t n, int64_t k);
QERL_API qerl_status qerl_nvfp4_pack(const uint8_t* codes, const uint8_t* scales, int64_t n, int64_t k,
                                     uint8_t* packed, void* stream);

/* The transposed packed layout, for the input gradient of the linear
 * (qerl_lora_linear_backward): the n x k weight's k x n transpose, its
 * contraction running along n.  Same block size and code bytes as
 * qerl_nvfp4_pack's layout with the roles of n and k exchanged (blocks per
 * 128-row tile over k and 256-wide stage over n; row kk of a tile holds the
 * codes of W[n][k] for the stage's n, two per byte, n even in the low
 * nibble); the 2048 scale bytes of a block hold the E4M3 scale of (n, k),
 * scales[n][k/16], for each of the tile's eight 16-row groups and the
 * stage's 256 n, at 16384 + (kk / 16) * 256 + (n mod 256).  Size:
 * qerl_nvfp4_packed_size(k, n) bytes.  Requires n % 64 == 0, n <= 65536,
 * k % 32 == 0; codes and packed_t 16-byte aligned.  Weights are frozen in
 * LoRA training, so this runs once per weight, beside qerl_nvfp4_pack. */
QERL_API qerl_status qerl_nvfp4_pack_transposed(const uint8_t* codes, const uint8_t* scales, int64_t n, int64_t k,
                                                uint8_t* packed_t, void* stream);

/* ========================================================================
 * NF4, the QLoRA format the digest sets against NVFP4 ("QLoRA's 4-bit
 * Quantization Addresses Memory but Degrades Speed", and "NVFP4
 * Quantization", comparison to other 4-bit formats: its levels sit at
 * quantiles of the Gaussian and are recovered through a lookup table, the
 * unpacking cost the digest ascribes to QLoRA).  Levels (the QLoRA
 * construction; the digest gives none): standard-normal quantiles at evenly
 * spaced probabilities with an exact zero -- Phi^-1(1/2 + (i/8)(p - 1/2)),
 * i = 1..8, their 7-point negative counterpart and 0, p = (1 - 1/32 + 1 -
 * 1/30) / 2 -- divided by the largest (range [-1, 1]); code c is the c-th
 * level in ascending order (code 7 = 0).  Scaling: NVFP4's dual scaling with a
 * level range of 1: S = amax / 448 (1 if 0), block scale E4M3(amax_b / S) per
 * 16, element code = the level nearest to w / (S dec(s)) (fp32 quotient
 * compared with the fp32 midpoints of adjacent levels; on a midpoint, the
 * upper level).  Codes and scales have qerl_nvfp4_quantize's layout, so
 * qerl_nvfp4_pack packs them; the linear takes them with w_format =
 * QERL_W_NF4 (its dequantization looks each code byte up in a table; the
 * product with the block scale is rounded once to fp16).  Arguments, errors
 * and workspace as qerl_nvfp4_quantize.
 * ======================================================================== */
QERL_API qerl_status qerl_nf4_quantize(const void* W, int w_dtype, int64_t n, int64_t k, int64_t ld_w,
                                       uint8_t* codes, uint8_t* scales, float* tensor_scale, void* workspace,
                                       size_t ws_bytes, void* stream);

/* ========================================================================
 * MXFP4, the 4-bit format the digest's "NVFP4 Quantization" section compares
 * NVFP4 with: E2M1 elements with one shared E8M0 (power-of-two) scale per 32
 * contiguous elements along K, no tensor scale.  The same linear kernels run
 * it: qerl_mxfp4_pack writes the linear's packed layout plus a tensor scale,
 * and qerl_lora_linear / _group take those exactly as for NVFP4.
 *
 * qerl_mxfp4_quantize: W [n][ld_w] f32 or bf16 (device, 16-byte aligned rows)
 *   -> codes [n][k/2] (two per byte, even k in the low nibble; device,
 *   16-byte aligned) and scales [n][k/32] (E8M0 codes, 127 = 2^0).  The
 *   scale rule (the digest does not give one; the OCP MX rule):
 *   e = floor(log2(amax_b)) - 2 clamped to [-127, 127], code e + 127, so the
 *   block max lands in [4, 8) * 2^e and values above 6 * 2^e saturate; an
 *   all-zero block gets code 0.  Elements: E2M1 of w / 2^e, round to nearest,
 *   ties to the even code, saturating at 6, -0 written as 0.  workspace:
 *   qerl_nvfp4_quantize_workspace_size() bytes, 256-byte aligned, zero-filled
 *   before first use.  Requires k % 32 == 0, ld_w >= k.  A non-finite weight
 *   records QERL_ERR_NONFINITE in the workspace status word (that block's
 *   codes and scale are then not written).
 *
 * qerl_mxfp4_pack: codes and scales as above -> packed (the layout described
 *   for qerl_nvfp4_pack, qerl_nvfp4_packed_size(n, k) bytes) and
 *   *tensor_scale (device float).  The layout holds E4M3 block scales times
 *   an fp32 tensor scale; an E8M0 scale 2^(e-127) is stored as
 *   S = 2^(e_max - 135) (e_max: the largest code over blocks with a non-zero
 *   element) times the E4M3 code of 2^(e - e_max + 8), exact for every block
 *   scale down to 2^-17 of the largest (E4M3 holds 2^-9 .. 2^8 exactly).  A
 *   non-zero block further below is packed as zeros and records
 *   QERL_ERR_RANGE in the workspace status word.  An all-zero weight gives
 *   S = 1.  Same shape rules and alignment as qerl_nvfp4_pack; scales need
 *   no alignment.  workspace as for qerl_mxfp4_quantize.
 * ======================================================================== */
QERL_API qerl_status qerl_mxfp4_quantize(const void* W, int w_dtype, int64_t n, int64_t k, int64_t ld_w,
                                         uint8_t* codes, uint8_t* scales, void* workspace, size_t ws_bytes,
                                         void* stream);
QERL_API qerl_status qerl_mxfp4_pack(const uint8_t* codes, const uint8_t* scales, int64_t n, int64_t k,
                                     uint8_t* packed, float* tensor_scale, void* workspace, size_t ws_bytes,
                                     void* stream);

/* ========================================================================
 * AQN schedule ("Adaptive Quantization Noise", Eq. 8 and Algorithm 1).
 * Host functions, pure, no CUDA.
 *
 * qerl_aqn_sigma: Eq. 8, sigma(k) = sigma_start * (sigma_end/sigma_start)^((k-1)/(K-1))
 * for k = 1..K, indexed by stage = k - 1 in [0, K).  stage < 0 returns 0
 * (Algorithm 1's warm-up stage: quantization noise only); stage >= K clamps
 * to K-1; num_stages <= 1 returns sigma_start.
 *
 * qerl_aqn_stage: Algorithm 1's stage of a training step: total_steps split
 * into num_stages stages of floor(total_steps / num_stages) steps (at least
 * 1); stage = min(step / that, num_stages - 1); step < 0 gives -1.
 * ======================================================================== */
QERL_API double qerl_aqn_sigma(int stage, int num_stages, double sigma_start, double sigma_end);
QERL_API int qerl_aqn_stage(int64_t step, int64_t total_steps, int num_stages);

/* The decay schedules the digest's AQN section compares ("Why exponential
 * decay"; the ablation's Figures 9 and 15), over the same stages as
 * qerl_aqn_sigma: with k = stage + 1 and u = (k-1)/(K-1),
 *   QERL_SCHEDULE_EXPONENTIAL  sigma_start * (sigma_end/sigma_start)^u  (Eq. 8,
 *                              identical to qerl_aqn_sigma)
 *   QERL_SCHEDULE_LINEAR       sigma_start - (sigma_start - sigma_end) * u
 *   QERL_SCHEDULE_COSINE       sigma_end + (sigma_start - sigma_end) * (1 + cos(pi u)) / 2
 *   QERL_SCHEDULE_LOGARITHMIC  sigma_start - (sigma_start - sigma_end) * ln(k) / ln(K)
 * stage < 0 returns 0, stage >= K clamps to K-1, num_stages <= 1 returns
 * sigma_start.  An unknown schedule returns NaN.  Host, pure, no CUDA. */
typedef enum {
  QERL_SCHEDULE_EXPONENTIAL = 0,
  QERL_SCHEDULE_LINEAR = 1,
  QERL_SCHEDULE_COSINE = 2,
  QERL_SCHEDULE_LOGARITHMIC = 3
} qerl_schedule;
QERL_API double qerl_aqn_sigma_schedule(int schedule, int stage, int num_stages, double sigma_start,
                                        double sigma_end);

/* AQN noise vector ("Adaptive Quantization Noise", Eq. 7: Z ~ N(0, sigma^2 I),
 * one value per input channel, resampled per forward pass).  Generator (the
 * digest only says Gaussian): channels 4i..4i+3 come from Philox4x32-10
 * (Salmon et al., SC'11) with counter (i, stream_id, counter_lo, counter_hi)
 * and key (seed_lo, seed_hi); u = (bits + 0.5) * 2^-32; Box-Muller in fp64,
 * (u0,u1) -> channels 4i, 4i+1 and (u2,u3) -> 4i+2, 4i+3; z = (float)(sigma * n).
 * z: device float[k].  Requires k >= 0 (k == 0 is a no-op). */
QERL_API qerl_status qerl_aqn_sample(float* z, int64_t k, float sigma, uint64_t seed, uint32_t stream_id,
                            uint64_t counter, void* stream);

/* ========================================================================
 * The linear layer.
 *
 *   x~[m][k] = bf16_RN( float(x[m][k]) * (1.0f + z[k]) )       (z == NULL: x~ = x)
 *   y[m][n]  = out_RN( S * sum_k x~[m][k] * dec(scale[n][k/16]) * e2m1(code[n][k])
 *                     + (alpha / r) * sum_j (sum_k x~[m][k] * A[j][k]) * B[n][j] )
 *
 * x       device bf16, m x k, row stride ldx elements (ldx >= k, ldx % 8 == 0,
 *         16-byte aligned).
 * wpacked the n x k weight's codes and scales (n = output features, k = input
 *         features) as packed by qerl_nvfp4_pack, 16-byte aligned.
 * tensor_scale device float, the S written by qerl_nvfp4_quantize (finite
 *         and > 0).  With a LoRA branch, a non-positive or non-finite S drops
 *         the LoRA term and records QERL_ERR_NONFINITE in the status word (the
 *         up-projection is accumulated pre-divided by S).
 * z       device float[k] or NULL (no noise).
 * A       device bf16 r x k, B device bf16 n x r (row-major), or both NULL /
 *         r == 0 (no LoRA branch).  r % 8 == 0 and r <= 128; A and B
 *         16-byte aligned.  Ranks above 64 with 33..128 tokens (m) can need
 *         more shared memory than a CTA has: the call then returns
 *         QERL_ERR_UNSUPPORTED_SHAPE before launching anything.  Every
 *         r <= 64 is supported at every m.
 * y       device, m x n (row stride n), y_dtype QERL_BF16 (round to nearest
 *         even) or QERL_F32.
 * workspace device, >= qerl_lora_linear_workspace_size(m, n, k, r) bytes,
 *         256-byte aligned, zero-filled before its first use; holds the
 *         staged noisy activations, the LoRA down-projection x~.A and the
 *         status word.  Calls sharing a workspace must be stream-ordered.
 * Requires k % 64 == 0, 0 < k <= 65536, m >= 0, n >= 0 (m == 0 or n == 0: no-op).
 * Accumulation is fp32; x~ and the dequantized weights enter the tensor
 * cores exactly (see the design notes for the power-of-two row staging).
 * ======================================================================== */
QERL_API size_t qerl_lora_linear_workspace_size(int64_t m, int64_t n, int64_t k, int r);

QERL_API qerl_status qerl_lora_linear(const void* x, int64_t m, int64_t k, int64_t ldx, const uint8_t* wpacked,
                                      const float* tensor_scale, int64_t n, const float* z, const void* A,
                                      const void* B, int r, float alpha, void* y, int y_dtype, void* workspace,
                                      size_t ws_bytes, void* stream);

/* ========================================================================
 * Several linears of one input in one launch (q/k/v of an attention block,
 * gate/up of an MLP; no counterpart in the pages, which describe one layer at
 * a time).  Up to 4 linears share x, z and k; each has its own packed
 * weights, tensor scale, LoRA adapters (A, B, r, alpha; A/B NULL or r == 0:
 * none) and output y [m][n] of its y_dtype.  Every output equals what
 * qerl_lora_linear gives for that linear alone (up to fp32 summation order).
 * One noise/staging pass serves all of them and their weight tiles run in one
 * grid, so small linears (k/v) do not pay a launch of their own.
 * `linears` is a host array of `count` descriptors (1 <= count <= 4), read
 * during the call.  Argument rules as for qerl_lora_linear, per linear; a
 * linear with n == 0 is skipped.  workspace: at least
 * qerl_lora_linear_group_workspace_size(m, k, linears, count) bytes.
 * ======================================================================== */
typedef struct qerl_linear_desc {
  const uint8_t* wpacked;     /* qerl_nvfp4_pack output for this n x k weight */
  const float* tensor_scale;  /* device float S */
  int64_t n;                  /* output features */
  const void* A;              /* bf16 [r][k] or NULL */
  const void* B;              /* bf16 [n][r] or NULL */
  int r;
  float alpha;
  void* y;                    /* device [m][n] */
  int y_dtype;                /* QERL_BF16 or QERL_F32 */
  int w_format;               /* QERL_W_NVFP4 (also MXFP4 packed by qerl_mxfp4_pack; 0) or QERL_W_NF4 */
} qerl_linear_desc;

QERL_API size_t qerl_lora_linear_group_workspace_size(int64_t m, int64_t k, const qerl_linear_desc* linears,
                                                      int count);
QERL_API qerl_status qerl_lora_linear_group(const void* x, int64_t m, int64_t k, int64_t ldx, const float* z,
                                            const qerl_linear_desc* linears, int count, void* workspace,
                                            size_t ws_bytes, void* stream);

/* ========================================================================
 * Per-rollout noise ("Adaptive Quantization Noise", noise injection: each
 * rollout sees its own noise sample).  As qerl_lora_linear_group, with a row
 * stride for z: z == NULL: no noise; ldz == 0: one vector z[k] for every row
 * (the batch broadcast of Eq. 9); ldz >= k: row i of x uses z + i * ldz (one
 * vector per rollout / token row).  ldz % 4 == 0 (16-byte aligned rows).
 * Workspace: qerl_lora_linear_group_workspace_size(m, k, linears, count).
 * ======================================================================== */
QERL_API qerl_status qerl_lora_linear_group_rowz(const void* x, int64_t m, int64_t k, int64_t ldx, const float* z,
                                                 int64_t ldz, const qerl_linear_desc* linears, int count,
                                                 void* workspace, size_t ws_bytes, void* stream);

/* ========================================================================
 * RMSNorm with the noise merged into its scale, feeding the linears
 * ("Noise Merging", Eq. 10-11: the noise Z is added to the RMSNorm weight w,
 * which is equivalent to the per-input-channel factor (1 + Z/w) on the
 * normalised activation):
 *
 *   x~[i][j] = bf16_RN( (w[j] + Z[j]) * (h[i][j] / sqrt((1/k) sum_l h[i][l]^2 + delta)) )
 *
 * computed in fp64 in that order with one rounding, then the grouped linear of
 * qerl_lora_linear_group on x~ (no further noise; both branches see x~).
 * h       device bf16 [m][ldh] (the pre-norm hidden state), 16-byte aligned,
 *         ldh % 8 == 0.
 * w_norm  device bf16 [k] (the RMSNorm weight), 16-byte aligned.
 * Z       device fp32 [k] (the AQN noise of this norm's consumers) or NULL
 *         (plain RMSNorm), 16-byte aligned.
 * delta   the RMSNorm epsilon, finite and >= 0 (delta == 0 on an all-zero row
 *         gives NaN, as the definition does).
 * Requires k % 64 == 0, m <= 65535.  workspace: at least
 * qerl_rmsnorm_lora_linear_group_workspace_size(m, k, linears, count) bytes
 * (it also holds x~ when a linear has a LoRA branch).
 * ======================================================================== */
QERL_API size_t qerl_rmsnorm_lora_linear_group_workspace_size(int64_t m, int64_t k, const qerl_linear_desc* linears,
                                                              int count);
QERL_API qerl_status qerl_rmsnorm_lora_linear_group(const void* h, int64_t m, int64_t k, int64_t ldh,
                                                    const void* w_norm, const float* Z, double delta,
                                                    const qerl_linear_desc* linears, int count, void* workspace,
                                                    size_t ws_bytes, void* stream);

/* The normalisation step above on its own: out device bf16 [m][ldo] receives
 * x~ (16-byte aligned, ldo % 8 == 0).  k % 8 == 0, m <= 65535.  No workspace. */
QERL_API qerl_status qerl_rmsnorm_noise(const void* h, int64_t m, int64_t k, int64_t ldh, const void* w_norm,
                                        const float* Z, double delta, void* out, int64_t ldo, void* stream);

/* ========================================================================
 * The backward pass of the linear ("Low-Rank Adaptation (LoRA) Within
 * Quantized Layers", gradient flow: the quantized base weight is frozen and
 * only carries the input gradient; A and B are trained).  For the forward
 * y = x~ W_hat^T + s (x~ A^T) B^T, s = alpha / r:
 *
 *   dx~ = dy W_hat + s (dy B) A        [m][k]  (bf16 or fp32, row stride k)
 *   dA  = s (dy B)^T x~                [r][k]  fp32
 *   dB  = s dy^T (x~ A^T)              [n][r]  fp32
 *
 * xt      device bf16 [m][ldxt]: the forward's input to both branches, x~
 *         (needed for dA and dB; may be NULL when both are NULL or r == 0).
 * dy      device bf16 [m][lddy].
 * wpacked_t  the weight in the transposed packed layout
 *         (qerl_nvfp4_pack_transposed), tensor_scale its S (device float).
 * A, B    the adapters as in the forward (bf16 [r][k], [n][r]), or both NULL
 *         (r ignored: no LoRA terms; dA, dB untouched).
 * dxt     device [m][k], dxt_dtype QERL_BF16 or QERL_F32; dA, dB device fp32
 *         or NULL to skip.
 * workspace  >= qerl_lora_linear_backward_workspace_size(m, n, k, r) bytes,
 *         256-byte aligned, zero-filled before first use; its status word
 *         (qerl_read_status) records kernel-detected errors as for the linear.
 * Requires n % 64 == 0 (n <= 65536), k % 64 == 0 (as the forward does),
 * r % 8 == 0 (r <= 128),
 * 16-byte aligned xt, dy, A, B and packed weights, ldxt and lddy multiples
 * of 8.  m == 0 zero-fills dA and dB.  dx~ runs on the forward's
 * tensor-core kernel (the transposed problem: dy contracts with W_hat along
 * n; u = dy B is its LoRA down-projection and A its up-projection); dA and
 * dB are rank-r reductions over the m tokens on CUDA cores, deterministic.
 * ======================================================================== */
QERL_API size_t qerl_lora_linear_backward_workspace_size(int64_t m, int64_t n, int64_t k, int r);
QERL_API qerl_status qerl_lora_linear_backward(const void* xt, int64_t m, int64_t k, int64_t ldxt, const void* dy,
                                               int64_t n, int64_t lddy, const uint8_t* wpacked_t,
                                               const float* tensor_scale, const void* A, const void* B, int r,
                                               float alpha, void* dxt, int dxt_dtype, float* dA, float* dB,
                                               void* workspace, size_t ws_bytes, void* stream);

/* The same linear for callers that cannot allocate device memory where they
 * run it (a runtime with a fixed memory pool, a latency-critical loop that must
 * not enter the CUDA allocator, a hard memory budget).  No counterpart in the
 * paper: this is a library convenience.  Arguments as for qerl_lora_linear,
 * without the workspace: the scratch lives in one library-owned device array
 * of 8 MiB, held by every GPU that loads the library until exit.
 *   - A problem fits exactly when qerl_lora_linear_workspace_size(m, n, k, r)
 *     <= 8 MiB (e.g. m = 128 with k up to ~28000 at r = 32); a larger one returns
 *     QERL_ERR_WORKSPACE; nothing is allocated, ever.
 *   - All calls share the array: calls that may overlap on the GPU race, so
 *     keep them ordered (e.g. on one stream).
 *   - The first call on a device looks up the array's address on that device;
 *     make it before any stream capture.
 *   - Argument errors are returned as by qerl_lora_linear (same checks, same
 *     order).  Kernel-detected errors are not reported: the status word is
 *     private and cleared per call.  An expired bounded wait leaves zeros in
 *     the output tile it hit; a non-positive or non-finite tensor scale gives
 *     non-finite outputs. */
QERL_API qerl_status qerl_lora_linear_noalloc(const void* x, int64_t m, int64_t k, int64_t ldx,
                                              const uint8_t* wpacked, const float* tensor_scale, int64_t n,
                                              const float* z, const void* A, const void* B, int r, float alpha,
                                              void* y, int y_dtype, void* stream);

/* Synchronizes `stream`, returns the status word recorded in `workspace` by
 * the kernels of earlier calls (QERL_OK if none failed) and resets it to
 * QERL_OK.  A failing CUDA call returns QERL_ERR_CUDA. */
QERL_API qerl_status qerl_read_status(void* workspace, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* QERL_H */
