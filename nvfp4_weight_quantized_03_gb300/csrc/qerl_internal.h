// qerl_internal.h -- host-side declarations shared by the library's .cu files.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>

#include "../../include/qerl.h"

namespace qerl {

constexpr size_t kWsHeaderBytes = 256;

inline size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

inline qerl_status cuda_status(cudaError_t e) { return e == cudaSuccess ? QERL_OK : QERL_ERR_CUDA; }

// quantize.cu
qerl_status launch_amax(const void* W, bool bf16, int64_t n, int64_t k, int64_t ld_w, unsigned* amax_bits,
                        cudaStream_t s);
qerl_status launch_encode(const void* W, bool bf16, int64_t n, int64_t k, int64_t ld_w,
                          const unsigned* amax_bits, const float* s_in, float* s_out, uint8_t* codes,
                          uint8_t* scales, int* status, cudaStream_t s, bool nf4 = false);
// NF4 (quantize.cu): the 16 levels (fp64, ascending, code c = level c) and
// the fp32 midpoints of adjacent levels.
struct Nf4Tables {
  double level[16];
  float mid[15];
};
const Nf4Tables& nf4_tables();
qerl_status launch_amax_to_float(const unsigned* amax_bits, float* amax, cudaStream_t s);
qerl_status launch_tensor_scale(const float* amax, float* S, cudaStream_t s);

// Packed weights for the linear (quantize.cu): 128 rows x 256 K per block.
constexpr size_t kPackedBlockBytes = 16384 + 2048;
size_t packed_weight_bytes(int64_t n, int64_t k);
qerl_status launch_pack(const uint8_t* codes, const uint8_t* scales, int64_t n, int64_t k, uint8_t* packed,
                        cudaStream_t s);
// The transposed packed layout of an n x k weight (its k x n transpose, the
// contraction along n), for the input gradient (quantize.cu).
qerl_status launch_pack_t(const uint8_t* codes, const uint8_t* scales, int64_t n, int64_t k, uint8_t* packed,
                          cudaStream_t s);
// MXFP4 (quantize.cu): the encoder, and the pack into the same layout with a
// power-of-two tensor scale (emax1: a zeroed device word of the workspace).
qerl_status launch_mx_encode(const void* W, bool bf16, int64_t n, int64_t k, int64_t ld_w, uint8_t* codes,
                             uint8_t* scales, int* status, cudaStream_t s);
qerl_status launch_mx_pack(const uint8_t* codes, const uint8_t* scales, int64_t n, int64_t k, uint8_t* packed,
                           float* tensor_scale, unsigned* emax1, int* status, cudaStream_t s);

// aqn.cu
qerl_status launch_aqn_sample(float* z, int64_t k, float sigma, uint64_t seed, uint32_t stream_id,
                              uint64_t counter, cudaStream_t s);

// linear.cu
struct LinearDesc {
  const uint8_t* wpacked;
  const float* tensor_scale;
  int64_t n;
  const void* A;
  const void* B;
  int r;
  float alpha;
  void* y;
  bool y_f32;
  bool nf4;  // NF4 element codes (the level table) instead of E2M1
};
struct LinearArgs {  // up to 4 linears sharing x, z and k
  const void* x;
  int64_t m, k, ldx;
  const float* z;
  int64_t ldz;  // noise row stride: 0 = one vector for every row
  // RMSNorm with merged noise in front of the linears (x holds h): x~ =
  // bf16((w_norm + Zn) * h / sqrt(mean(h^2) + delta)); z is then unused.
  bool rmsnorm;
  const void* w_norm;
  const float* Zn;
  double delta;
  LinearDesc lin[4];
  int nlin;
  // The weights are packed transposed (qerl_nvfp4_pack_transposed): the
  // linear then multiplies by W_hat instead of W_hat^T (k is W's n).
  bool wt;
  void* workspace;
  size_t ws_bytes;
};
size_t linear_workspace_bytes(int64_t m, int64_t k, const int* ranks, int nlin, bool rmsnorm = false);
// The normalisation step alone: out [m][ldo] bf16 (linear.cu).
qerl_status launch_rmsnorm_noise(const void* h, int64_t m, int64_t k, int64_t ldh, const void* w_norm, const float* Zn,
                                 double delta, void* out, int64_t ldo, cudaStream_t s);

// The LoRA down-projection t = x~ . A^T of a linear ([m][r] fp32), as the
// sum of `parts` partial arrays part_stride floats apart (linear.cu).
struct LoraDown {
  const float* t;
  int parts;
  int64_t part_stride;
};
// Where linear i's down-projection lies in the workspace after launch_lora_linear(a).
LoraDown linear_lora_down(const LinearArgs& a, int i);
// The down-projection alone, of x (bf16 [m][ldx], no noise) with A [r][k].
size_t lora_down_workspace_bytes(int64_t m, int64_t k, int r);
qerl_status launch_lora_down(const void* x, int64_t m, int64_t k, int64_t ldx, const void* A, int r, void* workspace,
                             LoraDown* out, int* status, cudaStream_t s);

// The backward pass (backward.cu): dx~, dA, dB of the LoRA linear.
struct BackwardArgs {
  const void* xt;  // bf16 [m][ldxt]: the forward's x~
  int64_t m, k, ldxt;
  const void* dy;  // bf16 [m][lddy]
  int64_t n, lddy;
  const uint8_t* wpacked_t;  // the weight in the transposed packed layout
  const float* tensor_scale;
  const void* A;  // bf16 [r][k]
  const void* B;  // bf16 [n][r]
  int r;
  float alpha;
  void* dxt;  // [m][k]
  bool dxt_f32;
  float* dA;  // [r][k] or null
  float* dB;  // [n][r] or null
  void* workspace;
};
size_t backward_workspace_bytes(int64_t m, int64_t n, int64_t k, int r);
qerl_status launch_lora_linear_backward(const BackwardArgs& b, cudaStream_t s);

// api.cu: the argument checks shared by every linear entry point.
qerl_status prepare_linear_group(const void* x, int64_t m, int64_t k, int64_t ldx, const float* z,
                                 const qerl_linear_desc* linears, int count, LinearArgs* out, bool* empty);
qerl_status launch_lora_linear(const LinearArgs& a, cudaStream_t s);

}  // namespace qerl
