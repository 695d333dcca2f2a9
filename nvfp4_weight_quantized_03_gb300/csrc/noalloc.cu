// noalloc.cu -- qerl_lora_linear_noalloc: the LoRA linear for callers that
// cannot hand the library a workspace.
//
// Some callers are not allowed to allocate device memory where they run the
// layer: an embedding runtime that owns a fixed memory pool and forbids new
// allocations after start-up, a latency-critical host loop that must not
// enter the CUDA allocator (cudaMalloc may synchronize the device and take
// unbounded time), or a tool running under a hard memory budget.  For them
// this entry point keeps its scratch (the staged noisy activations, the row
// scales, the LoRA down-projection and the status word) in one file-scope
// device array instead of a caller-provided workspace.  Inputs and outputs
// are still the caller's buffers.
//
// Rules of use:
//   - The array is kNoallocScratchBytes (8 MiB).  Every GPU that loads the
//     library holds it until the process exits.  A problem fits exactly when
//     qerl_lora_linear_workspace_size(m, n, k, r) <= 8 MiB (decode-sized
//     batches do, e.g. m = 128 with k up to ~28000 at r = 32); a larger one is
//     rejected with QERL_ERR_WORKSPACE -- use qerl_lora_linear with a
//     workspace for it.
//   - All calls share the array, which keeps the last call's contents.  Calls
//     that may overlap on the GPU (different streams, or unordered host
//     threads) race on it; keep the calls ordered, e.g. on one stream.
//   - The first call on each device looks up the array's device address
//     (cudaGetSymbolAddress, with that device current) and caches it.  Make
//     that first call on a device before any stream capture.
//   - The status word is cleared at the start of every call.  Errors that the
//     kernels detect are not reported through this entry point (argument
//     errors are returned as usual): an expired bounded wait leaves zeros in
//     the output tile it hit, and a non-positive or non-finite tensor scale
//     gives non-finite outputs.
#include <mutex>

#include "qerl_internal.h"

namespace {

constexpr size_t kNoallocScratchBytes = size_t{8} << 20;
constexpr int kMaxDevices = 64;

// The scratch.  In host code this name is only a stand-in for the device
// symbol, not a device address; the address comes from cudaGetSymbolAddress.
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoallocScratchBytes];

std::mutex g_setup_mutex;
void* g_scratch_ptr[kMaxDevices] = {};

// Device address of g_noalloc_scratch on the current device, looked up once per device.
qerl_status scratch_for_current_device(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return QERL_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return QERL_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_setup_mutex);
  if (g_scratch_ptr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr) return QERL_ERR_CUDA;
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return QERL_OK;
}

}  // namespace

extern "C" qerl_status qerl_lora_linear_noalloc(const void* x, int64_t m, int64_t k, int64_t ldx,
                                                const uint8_t* wpacked, const float* tensor_scale, int64_t n,
                                                const float* z, const void* A, const void* B, int r, float alpha,
                                                void* y, int y_dtype, void* stream) {
  // The same argument checks, in the same order, as qerl_lora_linear: a call
  // that the workspace entry point rejects is rejected here with the same
  // code, before anything is enqueued.
  if (n < 0 || r < 0) return QERL_ERR_INVALID_ARGUMENT;
  const qerl_linear_desc d{wpacked, tensor_scale, n, A, B, r, alpha, y, y_dtype, QERL_W_NVFP4};
  qerl::LinearArgs a{};
  bool empty = false;
  qerl_status st = qerl::prepare_linear_group(x, m, k, ldx, z, &d, 1, &a, &empty);
  if (st != QERL_OK || empty) return st;
  // The scratch this problem needs is exactly qerl_lora_linear_workspace_size(m, n, k, r).
  if (qerl::linear_workspace_bytes(m, k, &a.lin[0].r, 1) > kNoallocScratchBytes) return QERL_ERR_WORKSPACE;
  void* scratch = nullptr;
  if ((st = scratch_for_current_device(&scratch)) != QERL_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  // The status word must start at zero for this call.
  if (cudaMemsetAsync(scratch, 0, sizeof(int), s) != cudaSuccess) return QERL_ERR_CUDA;
  a.workspace = scratch;
  a.ws_bytes = kNoallocScratchBytes;
  return qerl::launch_lora_linear(a, s);
}
