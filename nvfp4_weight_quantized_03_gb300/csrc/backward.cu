// backward.cu -- the LoRA linear's backward pass through the frozen NVFP4
// weight (QeRL digest, section 3.4, "Low-Rank Adaptation (LoRA) Within
// Quantized Layers", gradient flow: only A and B are trained; the quantized
// base weight is frozen and only carries the input gradient).
//
// Forward: y = x~ W_hat^T + s (x~ A^T) B^T with s = alpha / r, t = x~ A^T.
//   dx~ = dy W_hat + s (dy B) A        [m][k]
//   dA  = s (dy B)^T x~                [r][k]
//   dB  = s dy^T t                     [n][r]
//
// dx~ is the forward linear of the transposed problem: x <- dy (contraction
// over n), W <- W_hat^T (the weight packed transposed, so the dequantizing
// MMA kernel multiplies by W_hat), LoRA down <- B^T [r][n] (its output u =
// dy B lands in the linear's workspace) and LoRA up <- A^T [k][r].  So the
// tensor-core kernel, its pipelines and its epilogue are the forward's; only
// the weight layout's scale addressing differs.
// dA and dB are rank-r products summed over the m tokens: t = x~ A^T comes
// from the prep kernel's LoRA tiles, and `skinny_kernel` forms
// out[p][j] = sum_m X[m][p] T[m][j] (X = dy or x~, T = t or u) on CUDA cores,
// split over m into fixed partial sums that `skinny_reduce_kernel` adds in
// order (deterministic).
#include <cuda_bf16.h>

#include <algorithm>
#include <mutex>

#include "qerl_internal.h"
#include "qerl_ptx.cuh"

namespace qerl {
namespace {

constexpr int kThreads = 256;
constexpr int kSkM = 32;  // tokens per shared-memory chunk

// out[c][r] = in[r][c] for a bf16 rows x cols matrix (row stride ld_in); 32x32 tiles.
__global__ void __launch_bounds__(kThreads) transpose_bf16_kernel(const __nv_bfloat16* __restrict__ in, int64_t ld_in,
                                                                  int rows, int cols,
                                                                  __nv_bfloat16* __restrict__ out) {
  __shared__ __nv_bfloat16 tile[32][33];
  const int r0 = blockIdx.y * 32, c0 = blockIdx.x * 32;
  const int tx = threadIdx.x & 31, ty = threadIdx.x >> 5;  // 8 rows of threads
  for (int i = ty; i < 32; i += 8) {
    const int r = r0 + i, c = c0 + tx;
    if (r < rows && c < cols) tile[i][tx] = in[static_cast<int64_t>(r) * ld_in + c];
  }
  __syncthreads();
  for (int i = ty; i < 32; i += 8) {
    const int c = c0 + i, r = r0 + tx;
    if (c < cols && r < rows) out[static_cast<int64_t>(c) * rows + r] = tile[tx][i];
  }
}

// Partial sums over the token range of split blockIdx.y:
//   partial[split][p][j] = sum_{m in range} X[m][p] * T[m][j],
// T[m][j] = sum over `parts` arrays (part_stride apart) of [m][r] fp32.
// A thread owns 4 consecutive p and 8 consecutive j; the block's p tile is
// 4 * (256 / jg) wide, jg = the power of two >= ceil(r / 8).  kSkM-token
// chunks go through shared memory (X as fp32, T summed over its parts); the
// next chunk's loads are issued into registers before the current chunk's
// FMAs, so their latency overlaps the arithmetic.
template <int JG>
__global__ void __launch_bounds__(kThreads) skinny_kernel(const __nv_bfloat16* __restrict__ X, int64_t ldx, int M,
                                                          int P, const float* __restrict__ T, int parts,
                                                          int64_t part_stride, int r, int m_per_split,
                                                          float* __restrict__ partial) {
  extern __shared__ __align__(16) float sk_smem[];
  constexpr int ptile = 4 * (kThreads / JG);
  constexpr int tw = 8 * JG;
  constexpr int nxv = kSkM * ptile / 8 / kThreads;  // X loads (8 bf16 each) per thread per chunk
  constexpr int ntv = kSkM * tw / kThreads;          // T values per thread per chunk
  static_assert(nxv >= 1 && ntv >= 1, "chunk covers every thread");
  constexpr int kSkMaxXv = nxv, kSkMaxTv = ntv;
  float* Xs = sk_smem;                 // [kSkM][ptile]
  float* Ts = sk_smem + kSkM * ptile;  // [kSkM][tw]
  const int p0 = blockIdx.x * ptile;
  const int m_begin = blockIdx.y * m_per_split, m_end = min(M, m_begin + m_per_split);
  const int tj = threadIdx.x % JG, tp = threadIdx.x / JG;
  float acc[4][8];
#pragma unroll
  for (int a = 0; a < 4; ++a)
#pragma unroll
    for (int b = 0; b < 8; ++b) acc[a][b] = 0.0f;
  uint4 xv[kSkMaxXv];
  float tv[kSkMaxTv];
  auto load = [&](int m0) {
#pragma unroll
    for (int u = 0; u < kSkMaxXv; ++u) {
      const int idx = threadIdx.x + u * kThreads;
      const int row = idx / (ptile / 8), c8 = (idx % (ptile / 8)) * 8;
      const int m = m0 + row, p = p0 + c8;
      xv[u] = (m < m_end && p < P) ? __ldg(reinterpret_cast<const uint4*>(X + static_cast<int64_t>(m) * ldx + p))
                                   : make_uint4(0u, 0u, 0u, 0u);
    }
#pragma unroll
    for (int u = 0; u < kSkMaxTv; ++u) {
      const int idx = threadIdx.x + u * kThreads;
      const int row = idx / tw, j = idx % tw;
      const int m = m0 + row;
      float v = 0.0f;
      if (m < m_end && j < r)
        for (int g = 0; g < parts; ++g) v += __ldg(T + g * part_stride + static_cast<int64_t>(m) * r + j);
      tv[u] = v;
    }
  };
  auto store = [&]() {
#pragma unroll
    for (int u = 0; u < kSkMaxXv; ++u) {
      const int idx = threadIdx.x + u * kThreads;
      const int row = idx / (ptile / 8), c8 = (idx % (ptile / 8)) * 8;
      const uint32_t w[4] = {xv[u].x, xv[u].y, xv[u].z, xv[u].w};
      float4* d = reinterpret_cast<float4*>(Xs + row * ptile + c8);
      d[0] = make_float4(__uint_as_float(w[0] << 16), __uint_as_float(w[0] & 0xFFFF0000u),
                         __uint_as_float(w[1] << 16), __uint_as_float(w[1] & 0xFFFF0000u));
      d[1] = make_float4(__uint_as_float(w[2] << 16), __uint_as_float(w[2] & 0xFFFF0000u),
                         __uint_as_float(w[3] << 16), __uint_as_float(w[3] & 0xFFFF0000u));
    }
#pragma unroll
    for (int u = 0; u < kSkMaxTv; ++u) Ts[threadIdx.x + u * kThreads] = tv[u];
  };
  if (m_begin < m_end) load(m_begin);
  for (int m0 = m_begin; m0 < m_end; m0 += kSkM) {
    store();
    __syncthreads();
    if (m0 + kSkM < m_end) load(m0 + kSkM);  // in flight during the FMAs below
#pragma unroll 4
    for (int mm = 0; mm < kSkM; ++mm) {
      const float4 xq = *reinterpret_cast<const float4*>(Xs + mm * ptile + 4 * tp);
      const float4 t0 = *reinterpret_cast<const float4*>(Ts + mm * tw + 8 * tj);
      const float4 t1 = *reinterpret_cast<const float4*>(Ts + mm * tw + 8 * tj + 4);
      const float xa[4] = {xq.x, xq.y, xq.z, xq.w};
      const float ta[8] = {t0.x, t0.y, t0.z, t0.w, t1.x, t1.y, t1.z, t1.w};
#pragma unroll
      for (int a = 0; a < 4; ++a)
#pragma unroll
        for (int b = 0; b < 8; ++b) acc[a][b] = fmaf(xa[a], ta[b], acc[a][b]);
    }
    __syncthreads();
  }
  float* out = partial + static_cast<int64_t>(blockIdx.y) * P * r;
#pragma unroll
  for (int a = 0; a < 4; ++a) {
    const int p = p0 + 4 * tp + a;
    if (p >= P) continue;
#pragma unroll
    for (int b = 0; b < 8; ++b) {
      const int j = 8 * tj + b;
      if (j < r) out[static_cast<int64_t>(p) * r + j] = acc[a][b];
    }
  }
}

// out = scale * sum over the splits, in split order: [P][r] (transposed = 0)
// or [r][P] (transposed = 1), fp32.
__global__ void __launch_bounds__(kThreads) skinny_reduce_kernel(const float* __restrict__ partial, int splits, int P,
                                                                 int r, float scale, int transposed,
                                                                 float* __restrict__ out) {
  const int64_t total = static_cast<int64_t>(P) * r;
  for (int64_t idx = blockIdx.x * static_cast<int64_t>(kThreads) + threadIdx.x; idx < total;
       idx += static_cast<int64_t>(gridDim.x) * kThreads) {
    // transposed: idx walks [j][p] (p fastest, coalesced stores); else [p][j]
    const int64_t p = transposed ? idx % P : idx / r;
    const int64_t j = transposed ? idx / P : idx % r;
    // Eight partials' loads in flight before their adds (in split order).
    const float* src = partial + p * r + j;
    float v = 0.0f;
    int sp = 0;
    for (; sp + 8 <= splits; sp += 8) {
      float w[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) w[u] = __ldg(src + (sp + u) * total);
#pragma unroll
      for (int u = 0; u < 8; ++u) v += w[u];
    }
    for (; sp < splits; ++sp) v += __ldg(src + sp * total);
    out[idx] = scale * v;
  }
}

int sms() {
  int dev = 0, n = 148;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
  return n;
}

struct SkinnyPlan {
  int jg, ptile, ptiles, splits, m_per_split;
  size_t smem;
};

SkinnyPlan skinny_plan(int64_t M, int64_t P, int r) {
  SkinnyPlan s;
  s.jg = 1;
  while (8 * s.jg < r) s.jg *= 2;
  s.ptile = 4 * (kThreads / s.jg);
  s.ptiles = static_cast<int>((P + s.ptile - 1) / s.ptile);
  // Two blocks per SM at most (one wave; a few blocks over that would form a
  // second wave of their own), at least 64 tokens per split.
  const int64_t max_splits = std::max<int64_t>(1, (M + 63) / 64);
  int64_t splits = std::max<int64_t>(1, (2 * sms()) / s.ptiles);
  splits = std::min(splits, max_splits);
  const int64_t mps = ((M + splits - 1) / splits + kSkM - 1) / kSkM * kSkM;
  s.m_per_split = static_cast<int>(std::max<int64_t>(mps, kSkM));
  s.splits = static_cast<int>((M + s.m_per_split - 1) / s.m_per_split);
  if (s.splits < 1) s.splits = 1;
  s.smem = static_cast<size_t>(kSkM) * (s.ptile + 8 * s.jg) * sizeof(float);
  return s;
}

struct BwdLayout {
  size_t lin, at, bt, down, partial, total;
};

BwdLayout bwd_layout(int64_t m, int64_t n, int64_t k, int r) {
  BwdLayout L;
  L.lin = 0;
  const int ranks[1] = {r};
  size_t off = align_up(linear_workspace_bytes(m, n, ranks, 1), 256);
  L.at = off;  // A^T [k][r] bf16
  off = align_up(off + static_cast<size_t>(k) * r * 2, 256);
  L.bt = off;  // B^T [r][n] bf16
  off = align_up(off + static_cast<size_t>(r) * n * 2, 256);
  L.down = off;  // t = x~ A^T (the prep kernel's LoRA tiles, own counters)
  off = align_up(off + lora_down_workspace_bytes(m, k, r), 256);
  L.partial = off;  // skinny partial sums, reused by dB then dA
  size_t part = 0;
  if (r > 0) {
    const SkinnyPlan pb = skinny_plan(m, n, r), pa = skinny_plan(m, k, r);
    part = std::max(static_cast<size_t>(pb.splits) * n * r, static_cast<size_t>(pa.splits) * k * r) * 4;
  }
  off = align_up(off + part, 256);
  L.total = off;
  return L;
}

qerl_status launch_skinny(const void* X, int64_t ldx, int64_t M, int64_t P, const LoraDown& T, int r, float scale,
                          bool transposed, float* partial, float* out, cudaStream_t s) {
  const SkinnyPlan sp = skinny_plan(M, P, r);
  static std::once_flag once;
  static cudaError_t err = cudaSuccess;
  std::call_once(once, [] {
    const int lim = 160 * 1024;  // the r <= 8 tile: 32 x (1024 + 8) floats
    err = cudaFuncSetAttribute(skinny_kernel<1>, cudaFuncAttributeMaxDynamicSharedMemorySize, lim);
    if (err == cudaSuccess) err = cudaFuncSetAttribute(skinny_kernel<2>, cudaFuncAttributeMaxDynamicSharedMemorySize, lim);
    if (err == cudaSuccess) err = cudaFuncSetAttribute(skinny_kernel<4>, cudaFuncAttributeMaxDynamicSharedMemorySize, lim);
    if (err == cudaSuccess) err = cudaFuncSetAttribute(skinny_kernel<8>, cudaFuncAttributeMaxDynamicSharedMemorySize, lim);
    if (err == cudaSuccess) err = cudaFuncSetAttribute(skinny_kernel<16>, cudaFuncAttributeMaxDynamicSharedMemorySize, lim);
  });
  if (err != cudaSuccess) return QERL_ERR_CUDA;
  const dim3 grid(static_cast<unsigned>(sp.ptiles), static_cast<unsigned>(sp.splits));
  const auto* xb = static_cast<const __nv_bfloat16*>(X);
  const int Mi = static_cast<int>(M), Pi = static_cast<int>(P);
  switch (sp.jg) {
    case 1: skinny_kernel<1><<<grid, kThreads, sp.smem, s>>>(xb, ldx, Mi, Pi, T.t, T.parts, T.part_stride, r, sp.m_per_split, partial); break;
    case 2: skinny_kernel<2><<<grid, kThreads, sp.smem, s>>>(xb, ldx, Mi, Pi, T.t, T.parts, T.part_stride, r, sp.m_per_split, partial); break;
    case 4: skinny_kernel<4><<<grid, kThreads, sp.smem, s>>>(xb, ldx, Mi, Pi, T.t, T.parts, T.part_stride, r, sp.m_per_split, partial); break;
    case 8: skinny_kernel<8><<<grid, kThreads, sp.smem, s>>>(xb, ldx, Mi, Pi, T.t, T.parts, T.part_stride, r, sp.m_per_split, partial); break;
    default: skinny_kernel<16><<<grid, kThreads, sp.smem, s>>>(xb, ldx, Mi, Pi, T.t, T.parts, T.part_stride, r, sp.m_per_split, partial); break;
  }
  if (cudaGetLastError() != cudaSuccess) return QERL_ERR_CUDA;
  const int64_t total = P * r;
  const int blocks = static_cast<int>(std::min<int64_t>((total + kThreads - 1) / kThreads, 4 * sms()));
  skinny_reduce_kernel<<<std::max(blocks, 1), kThreads, 0, s>>>(partial, sp.splits, static_cast<int>(P), r, scale,
                                                                transposed ? 1 : 0, out);
  return cuda_status(cudaGetLastError());
}

}  // namespace

size_t backward_workspace_bytes(int64_t m, int64_t n, int64_t k, int r) { return bwd_layout(m, n, k, r).total; }

qerl_status launch_lora_linear_backward(const BackwardArgs& b, cudaStream_t s) {
  const int64_t m = b.m, n = b.n, k = b.k;
  const int r = b.r;
  const BwdLayout L = bwd_layout(m, n, k, r);
  uint8_t* ws = static_cast<uint8_t*>(b.workspace);
  __nv_bfloat16* At = reinterpret_cast<__nv_bfloat16*>(ws + L.at);
  __nv_bfloat16* Bt = reinterpret_cast<__nv_bfloat16*>(ws + L.bt);
  if (r > 0) {
    transpose_bf16_kernel<<<dim3(static_cast<unsigned>((k + 31) / 32), static_cast<unsigned>((r + 31) / 32)), kThreads,
                            0, s>>>(static_cast<const __nv_bfloat16*>(b.A), k, r, static_cast<int>(k), At);
    if (cudaGetLastError() != cudaSuccess) return QERL_ERR_CUDA;
    transpose_bf16_kernel<<<dim3(static_cast<unsigned>((r + 31) / 32), static_cast<unsigned>((n + 31) / 32)), kThreads,
                            0, s>>>(static_cast<const __nv_bfloat16*>(b.B), r, static_cast<int>(n), r, Bt);
    if (cudaGetLastError() != cudaSuccess) return QERL_ERR_CUDA;
  }
  // dx~ = dy W_hat + s (dy B) A: the forward kernels on the transposed problem.
  LinearArgs a{};
  a.x = b.dy;
  a.m = m;
  a.k = n;
  a.ldx = b.lddy;
  a.z = nullptr;
  a.nlin = 1;
  a.wt = true;
  a.lin[0].wpacked = b.wpacked_t;
  a.lin[0].tensor_scale = b.tensor_scale;
  a.lin[0].n = k;
  a.lin[0].A = r > 0 ? Bt : nullptr;
  a.lin[0].B = r > 0 ? At : nullptr;
  a.lin[0].r = r;
  a.lin[0].alpha = b.alpha;
  a.lin[0].y = b.dxt;
  a.lin[0].y_f32 = b.dxt_f32;
  a.workspace = ws + L.lin;
  a.ws_bytes = L.at - L.lin;
  qerl_status st = launch_lora_linear(a, s);
  if (st != QERL_OK || r == 0 || (b.dA == nullptr && b.dB == nullptr)) return st;
  const float scale = b.alpha / static_cast<float>(r);
  float* partial = reinterpret_cast<float*>(ws + L.partial);
  if (b.dB != nullptr) {
    // dB = s dy^T t with t = x~ A^T.
    LoraDown t;
    if ((st = launch_lora_down(b.xt, m, k, b.ldxt, b.A, r, ws + L.down, &t, reinterpret_cast<int*>(ws), s)) !=
        QERL_OK)
      return st;
    if ((st = launch_skinny(b.dy, b.lddy, m, n, t, r, scale, false, partial, b.dB, s)) != QERL_OK) return st;
  }
  if (b.dA != nullptr) {
    // dA = s u^T x~ with u = dy B, the down-projection of the dx~ launch.
    const LoraDown u = linear_lora_down(a, 0);
    if ((st = launch_skinny(b.xt, b.ldxt, m, k, u, r, scale, true, partial, b.dA, s)) != QERL_OK) return st;
  }
  return QERL_OK;
}

}  // namespace qerl
