// api.cu -- the extern "C" entry points declared in include/qerl.h: argument
// validation on the host, workspace layout, and the kernel launches.
#include <cmath>
#include <cstdint>

#include "qerl_internal.h"
#include "qerl_ptx.cuh"

namespace {

using qerl::kWsHeaderBytes;

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

cudaStream_t as_stream(void* s) { return static_cast<cudaStream_t>(s); }

qerl_status check_weight_args(const void* W, int w_dtype, int64_t n, int64_t k, int64_t ld_w) {
  if (w_dtype != QERL_F32 && w_dtype != QERL_BF16) return QERL_ERR_INVALID_ARGUMENT;
  if (n < 0 || k < 0 || ld_w < k) return QERL_ERR_INVALID_ARGUMENT;
  if (k % 32 != 0) return QERL_ERR_UNSUPPORTED_SHAPE;
  if (n > 0 && k > 0 && W == nullptr) return QERL_ERR_INVALID_ARGUMENT;
  const int64_t esz = w_dtype == QERL_BF16 ? 2 : 4;
  if (!aligned(W, 16) || (ld_w * esz) % 16 != 0) return QERL_ERR_MISALIGNED;
  if (n > INT32_MAX || k > INT32_MAX) return QERL_ERR_UNSUPPORTED_SHAPE;
  return QERL_OK;
}

qerl_status check_ws(void* workspace, size_t ws_bytes, size_t need) {
  if (workspace == nullptr || ws_bytes < need) return QERL_ERR_WORKSPACE;
  if (!aligned(workspace, 256)) return QERL_ERR_MISALIGNED;
  return QERL_OK;
}

}  // namespace

namespace qerl {

// Argument checks of a grouped linear call (the order every linear entry point
// uses), filling `a` with the linears that have output features.  *empty is
// set when there is nothing to compute (m == 0 or every n == 0): the call is
// then a no-op and needs no workspace.
qerl_status prepare_linear_group(const void* x, int64_t m, int64_t k, int64_t ldx, const float* z,
                                 const qerl_linear_desc* linears, int count, LinearArgs* out, bool* empty) {
  *empty = false;
  if (linears == nullptr || count < 1 || count > 4) return QERL_ERR_INVALID_ARGUMENT;
  if (m < 0 || k <= 0 || ldx < k) return QERL_ERR_INVALID_ARGUMENT;
  if (k % 64 != 0) return QERL_ERR_UNSUPPORTED_SHAPE;
  if (k > 65536 || m > INT32_MAX || m * k > (int64_t{1} << 40)) return QERL_ERR_UNSUPPORTED_SHAPE;
  LinearArgs a{};
  int64_t total_n = 0;
  for (int i = 0; i < count; ++i) {
    const qerl_linear_desc& d = linears[i];
    int r = d.r;
    if (d.n < 0 || r < 0) return QERL_ERR_INVALID_ARGUMENT;
    if (d.y_dtype != QERL_BF16 && d.y_dtype != QERL_F32) return QERL_ERR_INVALID_ARGUMENT;
    if (d.w_format != QERL_W_NVFP4 && d.w_format != QERL_W_NF4) return QERL_ERR_INVALID_ARGUMENT;
    if ((d.A == nullptr) != (d.B == nullptr)) return QERL_ERR_INVALID_ARGUMENT;
    if (r > 0 && d.A == nullptr) r = 0;
    if (d.A != nullptr && r == 0) return QERL_ERR_INVALID_ARGUMENT;
    if (r > 128 || r % 8 != 0) return QERL_ERR_UNSUPPORTED_SHAPE;
    if (d.n > INT32_MAX) return QERL_ERR_UNSUPPORTED_SHAPE;
    total_n += d.n;
    a.lin[i].wpacked = d.wpacked;
    a.lin[i].tensor_scale = d.tensor_scale;
    a.lin[i].n = d.n;
    a.lin[i].A = r > 0 ? d.A : nullptr;
    a.lin[i].B = r > 0 ? d.B : nullptr;
    a.lin[i].r = r;
    a.lin[i].alpha = d.alpha;
    a.lin[i].y = d.y;
    a.lin[i].y_f32 = d.y_dtype == QERL_F32;
    a.lin[i].nf4 = d.w_format == QERL_W_NF4;
  }
  if (m == 0 || total_n == 0) {
    *empty = true;
    return QERL_OK;
  }
  if (x == nullptr) return QERL_ERR_INVALID_ARGUMENT;
  if (!aligned(x, 16) || ldx % 8 != 0) return QERL_ERR_MISALIGNED;
  if (z != nullptr && !aligned(z, 16)) return QERL_ERR_MISALIGNED;
  // Linears with no output features are dropped from the launch.
  int nl = 0;
  for (int i = 0; i < count; ++i) {
    const qerl_linear_desc& d = linears[i];
    if (d.n == 0) continue;
    if (d.wpacked == nullptr || d.tensor_scale == nullptr || d.y == nullptr) return QERL_ERR_INVALID_ARGUMENT;
    if (!aligned(d.wpacked, 16)) return QERL_ERR_MISALIGNED;
    if (d.y_dtype == QERL_F32 ? !aligned(d.y, 4) : !aligned(d.y, 2)) return QERL_ERR_MISALIGNED;
    if (a.lin[i].r > 0 && (!aligned(d.A, 16) || !aligned(d.B, 16))) return QERL_ERR_MISALIGNED;
    a.lin[nl] = a.lin[i];
    ++nl;
  }
  a.nlin = nl;
  a.x = x;
  a.m = m;
  a.k = k;
  a.ldx = ldx;
  a.z = z;
  *out = a;
  return QERL_OK;
}

}  // namespace qerl

extern "C" {

const char* qerl_status_string(int status) {
  switch (status) {
    case QERL_OK: return "QERL_OK";
    case QERL_ERR_INVALID_ARGUMENT: return "QERL_ERR_INVALID_ARGUMENT";
    case QERL_ERR_UNSUPPORTED_SHAPE: return "QERL_ERR_UNSUPPORTED_SHAPE";
    case QERL_ERR_MISALIGNED: return "QERL_ERR_MISALIGNED";
    case QERL_ERR_CUDA: return "QERL_ERR_CUDA";
    case QERL_ERR_TIMEOUT: return "QERL_ERR_TIMEOUT";
    case QERL_ERR_NONFINITE: return "QERL_ERR_NONFINITE";
    case QERL_ERR_WORKSPACE: return "QERL_ERR_WORKSPACE";
    case QERL_ERR_RANGE: return "QERL_ERR_RANGE";
    default: return "QERL_ERR_UNKNOWN";
  }
}

int qerl_version(void) { return 100; }

size_t qerl_nvfp4_quantize_workspace_size(void) { return kWsHeaderBytes; }

qerl_status qerl_nvfp4_amax(const void* W, int w_dtype, int64_t n, int64_t k, int64_t ld_w, float* amax,
                            void* workspace, size_t ws_bytes, void* stream) {
  qerl_status st = check_weight_args(W, w_dtype, n, k, ld_w);
  if (st != QERL_OK) return st;
  if (amax == nullptr) return QERL_ERR_INVALID_ARGUMENT;
  if ((st = check_ws(workspace, ws_bytes, kWsHeaderBytes)) != QERL_OK) return st;
  auto* hdr = static_cast<qerl::WsHeader*>(workspace);
  cudaStream_t s = as_stream(stream);
  if (cudaMemsetAsync(&hdr->amax_bits, 0, sizeof(unsigned), s) != cudaSuccess) return QERL_ERR_CUDA;
  if ((st = qerl::launch_amax(W, w_dtype == QERL_BF16, n, k, ld_w, &hdr->amax_bits, s)) != QERL_OK) return st;
  return qerl::launch_amax_to_float(&hdr->amax_bits, amax, s);
}

qerl_status qerl_nvfp4_quantize(const void* W, int w_dtype, int64_t n, int64_t k, int64_t ld_w, uint8_t* codes,
                                uint8_t* scales, float* tensor_scale, void* workspace, size_t ws_bytes,
                                void* stream) {
  qerl_status st = check_weight_args(W, w_dtype, n, k, ld_w);
  if (st != QERL_OK) return st;
  if (tensor_scale == nullptr) return QERL_ERR_INVALID_ARGUMENT;
  if (n > 0 && k > 0 && (codes == nullptr || scales == nullptr)) return QERL_ERR_INVALID_ARGUMENT;
  if (!aligned(codes, 16)) return QERL_ERR_MISALIGNED;
  if ((st = check_ws(workspace, ws_bytes, kWsHeaderBytes)) != QERL_OK) return st;
  auto* hdr = static_cast<qerl::WsHeader*>(workspace);
  cudaStream_t s = as_stream(stream);
  if (cudaMemsetAsync(&hdr->amax_bits, 0, sizeof(unsigned), s) != cudaSuccess) return QERL_ERR_CUDA;
  const bool bf16 = w_dtype == QERL_BF16;
  if ((st = qerl::launch_amax(W, bf16, n, k, ld_w, &hdr->amax_bits, s)) != QERL_OK) return st;
  return qerl::launch_encode(W, bf16, n, k, ld_w, &hdr->amax_bits, nullptr, tensor_scale, codes, scales,
                             &hdr->status, s);
}

qerl_status qerl_nf4_quantize(const void* W, int w_dtype, int64_t n, int64_t k, int64_t ld_w, uint8_t* codes,
                              uint8_t* scales, float* tensor_scale, void* workspace, size_t ws_bytes, void* stream) {
  qerl_status st = check_weight_args(W, w_dtype, n, k, ld_w);
  if (st != QERL_OK) return st;
  if (tensor_scale == nullptr) return QERL_ERR_INVALID_ARGUMENT;
  if (n > 0 && k > 0 && (codes == nullptr || scales == nullptr)) return QERL_ERR_INVALID_ARGUMENT;
  if (!aligned(codes, 16)) return QERL_ERR_MISALIGNED;
  if ((st = check_ws(workspace, ws_bytes, kWsHeaderBytes)) != QERL_OK) return st;
  auto* hdr = static_cast<qerl::WsHeader*>(workspace);
  cudaStream_t s = as_stream(stream);
  if (cudaMemsetAsync(&hdr->amax_bits, 0, sizeof(unsigned), s) != cudaSuccess) return QERL_ERR_CUDA;
  const bool bf16 = w_dtype == QERL_BF16;
  if ((st = qerl::launch_amax(W, bf16, n, k, ld_w, &hdr->amax_bits, s)) != QERL_OK) return st;
  return qerl::launch_encode(W, bf16, n, k, ld_w, &hdr->amax_bits, nullptr, tensor_scale, codes, scales,
                             &hdr->status, s, true);
}

qerl_status qerl_nvfp4_quantize_with_scale(const void* W, int w_dtype, int64_t n, int64_t k, int64_t ld_w,
                                           const float* tensor_scale, uint8_t* codes, uint8_t* scales,
                                           void* workspace, size_t ws_bytes, void* stream) {
  qerl_status st = check_weight_args(W, w_dtype, n, k, ld_w);
  if (st != QERL_OK) return st;
  if (tensor_scale == nullptr) return QERL_ERR_INVALID_ARGUMENT;
  if (n > 0 && k > 0 && (codes == nullptr || scales == nullptr)) return QERL_ERR_INVALID_ARGUMENT;
  if (!aligned(codes, 16)) return QERL_ERR_MISALIGNED;
  if ((st = check_ws(workspace, ws_bytes, kWsHeaderBytes)) != QERL_OK) return st;
  auto* hdr = static_cast<qerl::WsHeader*>(workspace);
  if (n == 0 || k == 0) return QERL_OK;
  return qerl::launch_encode(W, w_dtype == QERL_BF16, n, k, ld_w, nullptr, tensor_scale, nullptr, codes, scales,
                             &hdr->status, as_stream(stream));
}

qerl_status qerl_nvfp4_tensor_scale(const float* amax, float* tensor_scale, void* stream) {
  if (amax == nullptr || tensor_scale == nullptr) return QERL_ERR_INVALID_ARGUMENT;
  return qerl::launch_tensor_scale(amax, tensor_scale, as_stream(stream));
}

qerl_status qerl_aqn_sample(float* z, int64_t k, float sigma, uint64_t seed, uint32_t stream_id, uint64_t counter,
                            void* stream) {
  if (k < 0) return QERL_ERR_INVALID_ARGUMENT;
  if (k == 0) return QERL_OK;
  if (z == nullptr) return QERL_ERR_INVALID_ARGUMENT;
  if (k > (int64_t{1} << 34)) return QERL_ERR_UNSUPPORTED_SHAPE;
  return qerl::launch_aqn_sample(z, k, sigma, seed, stream_id, counter, as_stream(stream));
}

size_t qerl_nvfp4_packed_size(int64_t n, int64_t k) {
  if (n < 0 || k < 0) return 0;
  return qerl::packed_weight_bytes(n, k);
}

qerl_status qerl_nvfp4_pack(const uint8_t* codes, const uint8_t* scales, int64_t n, int64_t k, uint8_t* packed,
                            void* stream) {
  if (n < 0 || k < 0) return QERL_ERR_INVALID_ARGUMENT;
  if (k % 64 != 0) return QERL_ERR_UNSUPPORTED_SHAPE;
  if (n > INT32_MAX || k > 65536) return QERL_ERR_UNSUPPORTED_SHAPE;
  if (n == 0 || k == 0) return QERL_OK;
  if (codes == nullptr || scales == nullptr || packed == nullptr) return QERL_ERR_INVALID_ARGUMENT;
  if (!aligned(codes, 16) || !aligned(scales, 4) || !aligned(packed, 16)) return QERL_ERR_MISALIGNED;
  return qerl::launch_pack(codes, scales, n, k, packed, as_stream(stream));
}

qerl_status qerl_mxfp4_quantize(const void* W, int w_dtype, int64_t n, int64_t k, int64_t ld_w, uint8_t* codes,
                                uint8_t* scales, void* workspace, size_t ws_bytes, void* stream) {
  qerl_status st = check_weight_args(W, w_dtype, n, k, ld_w);
  if (st != QERL_OK) return st;
  if (n > 0 && k > 0 && (codes == nullptr || scales == nullptr)) return QERL_ERR_INVALID_ARGUMENT;
  if (!aligned(codes, 16)) return QERL_ERR_MISALIGNED;
  if ((st = check_ws(workspace, ws_bytes, kWsHeaderBytes)) != QERL_OK) return st;
  auto* hdr = static_cast<qerl::WsHeader*>(workspace);
  return qerl::launch_mx_encode(W, w_dtype == QERL_BF16, n, k, ld_w, codes, scales, &hdr->status,
                                as_stream(stream));
}

qerl_status qerl_mxfp4_pack(const uint8_t* codes, const uint8_t* scales, int64_t n, int64_t k, uint8_t* packed,
                            float* tensor_scale, void* workspace, size_t ws_bytes, void* stream) {
  if (n < 0 || k < 0) return QERL_ERR_INVALID_ARGUMENT;
  if (k % 64 != 0) return QERL_ERR_UNSUPPORTED_SHAPE;
  if (n > INT32_MAX || k > 65536) return QERL_ERR_UNSUPPORTED_SHAPE;
  if (tensor_scale == nullptr) return QERL_ERR_INVALID_ARGUMENT;
  if (n > 0 && k > 0 && (codes == nullptr || scales == nullptr || packed == nullptr))
    return QERL_ERR_INVALID_ARGUMENT;
  if (!aligned(codes, 16) || !aligned(packed, 16)) return QERL_ERR_MISALIGNED;
  qerl_status st = check_ws(workspace, ws_bytes, kWsHeaderBytes);
  if (st != QERL_OK) return st;
  auto* hdr = static_cast<qerl::WsHeader*>(workspace);
  cudaStream_t s = as_stream(stream);
  if (cudaMemsetAsync(&hdr->amax_bits, 0, sizeof(unsigned), s) != cudaSuccess) return QERL_ERR_CUDA;
  return qerl::launch_mx_pack(codes, scales, n, k, packed, tensor_scale, &hdr->amax_bits, &hdr->status, s);
}

qerl_status qerl_nvfp4_pack_transposed(const uint8_t* codes, const uint8_t* scales, int64_t n, int64_t k,
                                       uint8_t* packed_t, void* stream) {
  if (n < 0 || k < 0) return QERL_ERR_INVALID_ARGUMENT;
  if (n % 64 != 0 || k % 32 != 0) return QERL_ERR_UNSUPPORTED_SHAPE;
  if (n > 65536 || k > INT32_MAX) return QERL_ERR_UNSUPPORTED_SHAPE;
  if (n == 0 || k == 0) return QERL_OK;
  if (codes == nullptr || scales == nullptr || packed_t == nullptr) return QERL_ERR_INVALID_ARGUMENT;
  if (!aligned(codes, 16) || !aligned(packed_t, 16)) return QERL_ERR_MISALIGNED;
  return qerl::launch_pack_t(codes, scales, n, k, packed_t, as_stream(stream));
}

size_t qerl_lora_linear_backward_workspace_size(int64_t m, int64_t n, int64_t k, int r) {
  if (m < 0 || n < 0 || k < 0 || r < 0) return 0;
  return qerl::backward_workspace_bytes(m, n, k, r);
}

qerl_status qerl_lora_linear_backward(const void* xt, int64_t m, int64_t k, int64_t ldxt, const void* dy, int64_t n,
                                      int64_t lddy, const uint8_t* wpacked_t, const float* tensor_scale,
                                      const void* A, const void* B, int r, float alpha, void* dxt, int dxt_dtype,
                                      float* dA, float* dB, void* workspace, size_t ws_bytes, void* stream) {
  if (m < 0 || n <= 0 || k <= 0 || r < 0) return QERL_ERR_INVALID_ARGUMENT;
  if (ldxt < k || lddy < n) return QERL_ERR_INVALID_ARGUMENT;
  if (dxt_dtype != QERL_BF16 && dxt_dtype != QERL_F32) return QERL_ERR_INVALID_ARGUMENT;
  if ((A == nullptr) != (B == nullptr)) return QERL_ERR_INVALID_ARGUMENT;
  if (A == nullptr) r = 0;
  if (A != nullptr && r == 0) return QERL_ERR_INVALID_ARGUMENT;
  if (r > 128 || r % 8 != 0) return QERL_ERR_UNSUPPORTED_SHAPE;
  // The input gradient is a linear contracting over n (the transposed layout's
  // K); t = x~ A^T contracts over k as the forward does (k % 64 == 0 there too).
  if (n % 64 != 0 || k % 64 != 0) return QERL_ERR_UNSUPPORTED_SHAPE;
  if (n > 65536 || k > INT32_MAX || m > INT32_MAX || m * n > (int64_t{1} << 40)) return QERL_ERR_UNSUPPORTED_SHAPE;
  if (!std::isfinite(alpha)) return QERL_ERR_INVALID_ARGUMENT;
  cudaStream_t s = as_stream(stream);
  if (m == 0) {  // empty sums: zero gradients for the adapters
    if (r > 0 && dA != nullptr && cudaMemsetAsync(dA, 0, static_cast<size_t>(r) * k * 4, s) != cudaSuccess)
      return QERL_ERR_CUDA;
    if (r > 0 && dB != nullptr && cudaMemsetAsync(dB, 0, static_cast<size_t>(n) * r * 4, s) != cudaSuccess)
      return QERL_ERR_CUDA;
    return QERL_OK;
  }
  if (dy == nullptr || wpacked_t == nullptr || tensor_scale == nullptr || dxt == nullptr)
    return QERL_ERR_INVALID_ARGUMENT;
  if (r > 0 && (dA != nullptr || dB != nullptr) && xt == nullptr) return QERL_ERR_INVALID_ARGUMENT;
  if (!aligned(dy, 16) || lddy % 8 != 0 || !aligned(wpacked_t, 16)) return QERL_ERR_MISALIGNED;
  if (xt != nullptr && (!aligned(xt, 16) || ldxt % 8 != 0)) return QERL_ERR_MISALIGNED;
  if (dxt_dtype == QERL_F32 ? !aligned(dxt, 4) : !aligned(dxt, 2)) return QERL_ERR_MISALIGNED;
  if (r > 0 && (!aligned(A, 16) || !aligned(B, 16) || !aligned(dA, 4) || !aligned(dB, 4)))
    return QERL_ERR_MISALIGNED;
  qerl_status st = check_ws(workspace, ws_bytes, qerl::backward_workspace_bytes(m, n, k, r));
  if (st != QERL_OK) return st;
  qerl::BackwardArgs b{};
  b.xt = xt;
  b.m = m;
  b.k = k;
  b.ldxt = ldxt;
  b.dy = dy;
  b.n = n;
  b.lddy = lddy;
  b.wpacked_t = wpacked_t;
  b.tensor_scale = tensor_scale;
  b.A = r > 0 ? A : nullptr;
  b.B = r > 0 ? B : nullptr;
  b.r = r;
  b.alpha = alpha;
  b.dxt = dxt;
  b.dxt_f32 = dxt_dtype == QERL_F32;
  b.dA = r > 0 ? dA : nullptr;
  b.dB = r > 0 ? dB : nullptr;
  b.workspace = workspace;
  return qerl::launch_lora_linear_backward(b, s);
}

size_t qerl_lora_linear_workspace_size(int64_t m, int64_t n, int64_t k, int r) {
  (void)n;
  if (m < 0 || k < 0 || r < 0) return 0;
  return qerl::linear_workspace_bytes(m, k, &r, 1);
}

size_t qerl_lora_linear_group_workspace_size(int64_t m, int64_t k, const qerl_linear_desc* linears, int count) {
  if (m < 0 || k < 0 || count < 1 || count > 4 || linears == nullptr) return 0;
  int ranks[4] = {0, 0, 0, 0};
  for (int i = 0; i < count; ++i) ranks[i] = linears[i].r > 0 ? linears[i].r : 0;
  return qerl::linear_workspace_bytes(m, k, ranks, count);
}

qerl_status qerl_lora_linear_group(const void* x, int64_t m, int64_t k, int64_t ldx, const float* z,
                                   const qerl_linear_desc* linears, int count, void* workspace, size_t ws_bytes,
                                   void* stream) {
  qerl::LinearArgs a{};
  bool empty = false;
  qerl_status st = qerl::prepare_linear_group(x, m, k, ldx, z, linears, count, &a, &empty);
  if (st != QERL_OK || empty) return st;
  int ranks[4] = {0, 0, 0, 0};
  for (int i = 0; i < a.nlin; ++i) ranks[i] = a.lin[i].r;
  st = check_ws(workspace, ws_bytes, qerl::linear_workspace_bytes(m, k, ranks, a.nlin));
  if (st != QERL_OK) return st;
  a.workspace = workspace;
  a.ws_bytes = ws_bytes;
  return qerl::launch_lora_linear(a, as_stream(stream));
}

qerl_status qerl_lora_linear_group_rowz(const void* x, int64_t m, int64_t k, int64_t ldx, const float* z, int64_t ldz,
                                        const qerl_linear_desc* linears, int count, void* workspace, size_t ws_bytes,
                                        void* stream) {
  qerl::LinearArgs a{};
  bool empty = false;
  qerl_status st = qerl::prepare_linear_group(x, m, k, ldx, z, linears, count, &a, &empty);
  if (st != QERL_OK || empty) return st;
  if (z != nullptr && ldz != 0) {
    if (ldz < k) return QERL_ERR_INVALID_ARGUMENT;
    if (ldz % 4 != 0) return QERL_ERR_MISALIGNED;  // every row 16-byte aligned
  }
  int ranks[4] = {0, 0, 0, 0};
  for (int i = 0; i < a.nlin; ++i) ranks[i] = a.lin[i].r;
  st = check_ws(workspace, ws_bytes, qerl::linear_workspace_bytes(m, k, ranks, a.nlin));
  if (st != QERL_OK) return st;
  a.ldz = z != nullptr ? ldz : 0;
  a.workspace = workspace;
  a.ws_bytes = ws_bytes;
  return qerl::launch_lora_linear(a, as_stream(stream));
}

size_t qerl_rmsnorm_lora_linear_group_workspace_size(int64_t m, int64_t k, const qerl_linear_desc* linears,
                                                     int count) {
  if (m < 0 || k < 0 || count < 1 || count > 4 || linears == nullptr) return 0;
  int ranks[4] = {0, 0, 0, 0};
  for (int i = 0; i < count; ++i) ranks[i] = linears[i].r > 0 && linears[i].A != nullptr ? linears[i].r : 0;
  return qerl::linear_workspace_bytes(m, k, ranks, count, true);
}

namespace {
qerl_status check_rmsnorm_args(int64_t m, int64_t k, const void* w_norm, const float* Z, double delta) {
  if (!(delta >= 0.0) || !std::isfinite(delta)) return QERL_ERR_INVALID_ARGUMENT;
  if (m > 65535) return QERL_ERR_UNSUPPORTED_SHAPE;  // one CTA per row on the grid's y axis
  if (k % 8 != 0) return QERL_ERR_UNSUPPORTED_SHAPE;
  if (m > 0 && k > 0 && w_norm == nullptr) return QERL_ERR_INVALID_ARGUMENT;
  if (!aligned(w_norm, 16) || (Z != nullptr && !aligned(Z, 16))) return QERL_ERR_MISALIGNED;
  return QERL_OK;
}
}  // namespace

qerl_status qerl_rmsnorm_lora_linear_group(const void* h, int64_t m, int64_t k, int64_t ldh, const void* w_norm,
                                           const float* Z, double delta, const qerl_linear_desc* linears, int count,
                                           void* workspace, size_t ws_bytes, void* stream) {
  qerl::LinearArgs a{};
  bool empty = false;
  qerl_status st = qerl::prepare_linear_group(h, m, k, ldh, nullptr, linears, count, &a, &empty);
  if (st != QERL_OK || empty) return st;
  if ((st = check_rmsnorm_args(m, k, w_norm, Z, delta)) != QERL_OK) return st;
  int ranks[4] = {0, 0, 0, 0};
  for (int i = 0; i < a.nlin; ++i) ranks[i] = a.lin[i].r;
  st = check_ws(workspace, ws_bytes, qerl::linear_workspace_bytes(m, k, ranks, a.nlin, true));
  if (st != QERL_OK) return st;
  a.rmsnorm = true;
  a.w_norm = w_norm;
  a.Zn = Z;
  a.delta = delta;
  a.workspace = workspace;
  a.ws_bytes = ws_bytes;
  return qerl::launch_lora_linear(a, as_stream(stream));
}

qerl_status qerl_rmsnorm_noise(const void* h, int64_t m, int64_t k, int64_t ldh, const void* w_norm, const float* Z,
                               double delta, void* out, int64_t ldo, void* stream) {
  if (m < 0 || k < 0 || ldh < k || ldo < k) return QERL_ERR_INVALID_ARGUMENT;
  qerl_status st = check_rmsnorm_args(m, k, w_norm, Z, delta);
  if (st != QERL_OK) return st;
  if (m == 0 || k == 0) return QERL_OK;
  if (h == nullptr || out == nullptr) return QERL_ERR_INVALID_ARGUMENT;
  if (!aligned(h, 16) || !aligned(out, 16) || ldh % 8 != 0 || ldo % 8 != 0) return QERL_ERR_MISALIGNED;
  if (k > INT32_MAX) return QERL_ERR_UNSUPPORTED_SHAPE;
  return qerl::launch_rmsnorm_noise(h, m, k, ldh, w_norm, Z, delta, out, ldo, as_stream(stream));
}

qerl_status qerl_lora_linear(const void* x, int64_t m, int64_t k, int64_t ldx, const uint8_t* wpacked,
                             const float* tensor_scale, int64_t n, const float* z, const void* A, const void* B,
                             int r, float alpha, void* y, int y_dtype, void* workspace, size_t ws_bytes,
                             void* stream) {
  if (n < 0 || r < 0) return QERL_ERR_INVALID_ARGUMENT;
  qerl_linear_desc d{};
  d.wpacked = wpacked;
  d.tensor_scale = tensor_scale;
  d.n = n;
  d.A = A;
  d.B = B;
  d.r = r;
  d.alpha = alpha;
  d.y = y;
  d.y_dtype = y_dtype;
  return qerl_lora_linear_group(x, m, k, ldx, z, &d, 1, workspace, ws_bytes, stream);
}

qerl_status qerl_read_status(void* workspace, void* stream) {
  if (workspace == nullptr) return QERL_ERR_INVALID_ARGUMENT;
  cudaStream_t s = as_stream(stream);
  int host = 0;
  if (cudaMemcpyAsync(&host, workspace, sizeof(int), cudaMemcpyDeviceToHost, s) != cudaSuccess) return QERL_ERR_CUDA;
  if (cudaMemsetAsync(workspace, 0, sizeof(int), s) != cudaSuccess) return QERL_ERR_CUDA;
  if (cudaStreamSynchronize(s) != cudaSuccess) return QERL_ERR_CUDA;
  return static_cast<qerl_status>(host);
}

}  // extern "C"
