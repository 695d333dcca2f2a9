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
// from the LoRA down-projection kernels, and `skinny_tc_kernel` forms
// out[p][j] = sum_m X[m][p] T[m][j] (X = dy or x~, T = t or u) on the tensor
// cores, split over m into fixed partial sums that `skinny_reduce_kernel`
// adds in order (deterministic).
#include <cuda_bf16.h>

#include <algorithm>
#include <mutex>

#include "qerl_internal.h"
#include "qerl_ptx.cuh"

namespace qerl {
namespace {

constexpr int kThreads = 256;

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

// ---------------------------------------------------------------------------
// Partial sums over the token range of split blockIdx.y, on the tensor cores:
//   partial[split][p][j] = sum_{m in range} X[m][p] * T[m][j]
// (T[m][j] = sum over `parts` arrays, part_stride apart, of [m][r] fp32), as
//   D[p][j] += sum_m A[p][m] B[j][m],  A = X^T (128 p rows per CTA), B = T^T.
// Each 64-token chunk of X (bf16) is transposed through registers into the
// K-major 128-byte-swizzled layout of A (128 rows x 64 tokens), and T (fp32)
// into three bf16 terms t1 = bf16(T), t2 = bf16(T - t1), t3 = bf16(T - t1 -
// t2) (together T to ~24 significant bits), each laid out likewise as a B
// tile (rn = round16(r) rows x 64 tokens).  Per chunk 4 K-steps of MMAs
// (M = 128, K = 16, bf16 products exact, fp32 accumulation in tensor
// memory); two A/B buffers, each released by the MMAs' commit.
constexpr int kTcThreads = 256;
constexpr int kTcM = 64;   // tokens per chunk (the MMAs' K)
constexpr int kTcP = 128;  // p rows per CTA (the MMAs' M)
__host__ __device__ inline int tc_rn(int r) { return (r + 15) / 16 * 16; }
// Up to r = 64 the three terms' B tiles form one B operand of 3 rn rows (one
// MMA per K-step; the accumulator's three column blocks are added at the
// end); above, one MMA per term into the same accumulator.
__host__ __device__ inline bool tc_fused(int r) { return 3 * tc_rn(r) <= 256; }
__host__ __device__ inline int tc_tmem_cols(int r) {
  const int need = tc_fused(r) ? 3 * tc_rn(r) : tc_rn(r);
  int c = 32;
  while (c < need) c *= 2;
  return c;
}
__host__ __device__ inline uint32_t tc_buf_bytes(int r) { return 16384u + 3u * static_cast<uint32_t>(tc_rn(r)) * 128u; }
// Staging of one chunk as it arrives (cp.async): X [64][128] bf16, T [64][rn] fp32.
constexpr int kTcStages = 2;
__host__ __device__ inline uint32_t tc_stage_bytes(int r) { return 16384u + 64u * static_cast<uint32_t>(tc_rn(r)) * 4u; }
__host__ __device__ inline size_t tc_smem_bytes(int r) {
  return 1024 + 2 * static_cast<size_t>(tc_buf_bytes(r)) + kTcStages * static_cast<size_t>(tc_stage_bytes(r)) + 64;
}

__device__ __forceinline__ uint32_t bf16_bits(float v) {
  return static_cast<uint32_t>(__bfloat16_as_ushort(__float2bfloat16_rn(v)));
}

// RMAX: the rank class (32, 64 or 128).
template <int RMAX>
__global__ void __launch_bounds__(kTcThreads, 1) skinny_tc_kernel(const __nv_bfloat16* __restrict__ X, int64_t ldx,
                                                                 int M, int P, const float* __restrict__ T,
                                                                 int parts, int64_t part_stride, int r,
                                                                 int m_per_split, float* __restrict__ partial,
                                                                 int* status) {
  extern __shared__ __align__(1024) uint8_t tc_smem_raw[];
  const uint32_t raw = static_cast<uint32_t>(__cvta_generic_to_shared(tc_smem_raw));
  const uint32_t sbase = (raw + 1023u) & ~1023u;
  uint8_t* sgen = tc_smem_raw + (sbase - raw);
  const int rn = tc_rn(r);
  const uint32_t bufb = tc_buf_bytes(r);
  const uint32_t bars = sbase + 2 * bufb + kTcStages * tc_stage_bytes(r);
  auto mma_done = [&](int b) { return bars + 8u * b; };
  const uint32_t acc_done = bars + 16u;
  const uint32_t holder = bars + 24u;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(sgen + (bars - sbase) + 28);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int p0 = blockIdx.x * kTcP;
  const int m_begin = blockIdx.y * m_per_split, m_end = min(M, m_begin + m_per_split);
  const uint32_t ncols = static_cast<uint32_t>(tc_tmem_cols(r));
  if (tid == 0) {
    mbar_init_a(mma_done(0), 1);
    mbar_init_a(mma_done(1), 1);
    mbar_init_a(acc_done, 1);
    *abort_flag = 0;
    fence_mbarrier_init();
  }
  if (warp == 0) {
    tmem_alloc(holder, ncols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(sgen + (bars - sbase) + 24);
  const bool fused = tc_fused(r);
  const uint32_t idesc = idesc_bf16_f32(kTcP, static_cast<uint32_t>(fused ? 3 * rn : rn));
  const int nchunks = m_end > m_begin ? (m_end - m_begin + kTcM - 1) / kTcM : 0;
  // Chunks arrive by cp.async into a kTcStages-deep staging ring (X rows as
  // they are, T part 0; rows past the split and p past P zero-filled), so
  // that the loads of the next chunks are in flight while the current one
  // is transposed into its A/B buffer and multiplied.  Other T parts (small
  // token counts) are added from global memory during the transpose.
  const uint32_t stage0 = sbase + 2 * bufb;
  const uint32_t sstride = tc_stage_bytes(r);
  auto issue_chunk = [&](int c) {
    if (c < nchunks) {
      const uint32_t st = stage0 + static_cast<uint32_t>(c % kTcStages) * sstride;
      const int m0 = m_begin + c * kTcM;
      for (int v = tid; v < kTcM * (kTcP / 8); v += kTcThreads) {  // X: 64 rows x 16 pieces of 16 B
        const int ml = v >> 4, pc = (v & 15) * 8;
        const bool in = m0 + ml < m_end && p0 + pc < P;
        cp_async_16(st + static_cast<uint32_t>(v) * 16u,
                    in ? static_cast<const void*>(X + static_cast<int64_t>(m0 + ml) * ldx + p0 + pc) : X, in ? 16u : 0u);
      }
      const int tq = rn / 4;  // T: 64 rows x rn / 4 pieces of 16 B (r % 8 == 0: a piece is all in or all out)
      for (int v = tid; v < kTcM * tq; v += kTcThreads) {
        const int ml = v / tq, jc = (v % tq) * 4;
        const bool in = m0 + ml < m_end && jc < r;
        cp_async_16(st + 16384u + static_cast<uint32_t>(v) * 16u,
                    in ? static_cast<const void*>(T + static_cast<int64_t>(m0 + ml) * r + jc) : T, in ? 16u : 0u);
      }
    }
    cp_async_commit();  // one group per chunk slot (empty past the end)
  };
  bool ok = true;
  for (int c = 0; c < kTcStages; ++c) issue_chunk(c);
  for (int c = 0; c < nchunks; ++c) {
    const int b = c & 1;
    const uint32_t abuf = sbase + static_cast<uint32_t>(b) * bufb, bbuf = abuf + 16384u;
    const uint32_t st = stage0 + static_cast<uint32_t>(c % kTcStages) * sstride;
    cp_async_wait_group<kTcStages - 1>();  // this thread's copies of chunk c have landed
    // The buffer's previous MMAs (chunk c - 2) are done reading it.
    if (c >= 2 && !mbar_wait_a(mma_done(b), static_cast<uint32_t>(((c - 2) >> 1) & 1), abort_flag, status)) {
      ok = false;
      break;
    }
    __syncthreads();  // every thread's copies of chunk c are visible
    {
      // X: work item (token octet mo, p pair pp): eight 32-bit words (tokens
      // 8 mo .. 8 mo + 7, p pair) give A rows 2 pp and 2 pp + 1 one 16-byte
      // piece each (tokens of a row are contiguous in the K-major layout).
      // Lanes take consecutive p pairs: conflict-free reads, and the
      // swizzle spreads the 16-byte stores.
#pragma unroll
      for (int u = 0; u < (kTcM / 8) * (kTcP / 2) / kTcThreads; ++u) {
        const int item = tid + u * kTcThreads;
        const int pp = item & (kTcP / 2 - 1), mo = item / (kTcP / 2);
        uint32_t w[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) w[e] = lds32(st + static_cast<uint32_t>((8 * mo + e) * (kTcP * 2) + 4 * pp));
        uint4 lo, hi;
        lo.x = __byte_perm(w[0], w[1], 0x5410);
        lo.y = __byte_perm(w[2], w[3], 0x5410);
        lo.z = __byte_perm(w[4], w[5], 0x5410);
        lo.w = __byte_perm(w[6], w[7], 0x5410);
        hi.x = __byte_perm(w[0], w[1], 0x7632);
        hi.y = __byte_perm(w[2], w[3], 0x7632);
        hi.z = __byte_perm(w[4], w[5], 0x7632);
        hi.w = __byte_perm(w[6], w[7], 0x7632);
        const int R = 2 * pp;
        sts128(abuf + static_cast<uint32_t>((R >> 3) * 1024 + (R & 7) * 128 + ((mo ^ (R & 7)) << 4)), lo);
        sts128(abuf + static_cast<uint32_t>(((R + 1) >> 3) * 1024 + ((R + 1) & 7) * 128 + ((mo ^ ((R + 1) & 7)) << 4)),
               hi);
      }
      // T: work item (token octet mo, j): eight values -> three bf16 terms,
      // one 16-byte piece of row j in each of the B tiles.
      const int m0 = m_begin + c * kTcM;
      for (int item = tid; item < (kTcM / 8) * rn; item += kTcThreads) {
        const int j = item % rn, mo = item / rn;
        float v[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) v[e] = ldsf(st + 16384u + static_cast<uint32_t>(((8 * mo + e) * rn + j) * 4));
        if (parts > 1 && j < r)
          for (int g = 1; g < parts; ++g)
#pragma unroll
            for (int e = 0; e < 8; ++e)
              if (m0 + 8 * mo + e < m_end) v[e] += __ldg(T + g * part_stride + static_cast<int64_t>(m0 + 8 * mo + e) * r + j);
        const uint32_t off = static_cast<uint32_t>((j >> 3) * 1024 + (j & 7) * 128 + ((mo ^ (j & 7)) << 4));
#pragma unroll
        for (int k3 = 0; k3 < 3; ++k3) {
          uint32_t hb[8];
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            hb[e] = bf16_bits(v[e]);
            v[e] -= __uint_as_float(hb[e] << 16);  // exact: the remainder of a rounding
          }
          sts128(bbuf + static_cast<uint32_t>(k3 * rn * 128) + off,
                 make_uint4(hb[0] | (hb[1] << 16), hb[2] | (hb[3] << 16), hb[4] | (hb[5] << 16), hb[6] | (hb[7] << 16)));
        }
      }
    }
    fence_proxy_async_smem();  // the tiles are read by the MMAs (async proxy)
    __syncthreads();           // A/B ready; the staging slot of chunk c is free
    issue_chunk(c + kTcStages);
    if (tid == 0) {
      tc_fence_after();
#pragma unroll
      for (int ks = 0; ks < kTcM / 16; ++ks) {
        const uint64_t ad = sw128_kmajor_desc(abuf + 32u * ks);
        if (fused) {
          tc_mma_f16(tmem, ad, sw128_kmajor_desc(bbuf + 32u * ks), idesc, (c > 0 || ks > 0) ? 1u : 0u);
        } else {
#pragma unroll
          for (int k3 = 0; k3 < 3; ++k3)
            tc_mma_f16(tmem, ad, sw128_kmajor_desc(bbuf + static_cast<uint32_t>(k3 * rn * 128) + 32u * ks), idesc,
                       (c > 0 || ks > 0 || k3 > 0) ? 1u : 0u);
        }
      }
      tc_commit(mma_done(b));
    }
  }
  cp_async_wait_group<0>();  // no copy outlives the block
  if (tid == 0) tc_commit(acc_done);  // once every MMA issued above is done (at once without any)
  ok = mbar_wait_a(acc_done, 0, abort_flag, status) && ok;
  tc_fence_after();
  // Warp w reads lanes 32 (w % 4) .. + 31 (its TMEM quadrant), columns of half w / 4.
  {
    const int q = warp & 3, half = warp >> 2;
    const int p = p0 + 32 * q + lane;
    float* out = partial + static_cast<int64_t>(blockIdx.y) * P * r + static_cast<int64_t>(p) * r;
    const int cb = half * (rn / 2), ce = cb + rn / 2;
    const uint32_t lane_addr = tmem + (static_cast<uint32_t>(32 * q) << 16);
    for (int c8 = cb; c8 < ce; c8 += 8) {
      float v[8];
      tmem_ld_x8(lane_addr + static_cast<uint32_t>(c8), v);
      if (fused) {  // the three terms' column blocks, added in term order
        float v2[8], v3[8];
        tmem_ld_x8(lane_addr + static_cast<uint32_t>(rn + c8), v2);
        tmem_ld_x8(lane_addr + static_cast<uint32_t>(2 * rn + c8), v3);
        tmem_ld_wait();
#pragma unroll
        for (int e = 0; e < 8; ++e) v[e] = (v[e] + v2[e]) + v3[e];
      }
      tmem_ld_wait();
      if (p < P) {
#pragma unroll
        for (int e = 0; e < 8; ++e)
          if (c8 + e < r) out[c8 + e] = (ok && nchunks > 0) ? v[e] : 0.0f;
      }
    }
  }
  if (*abort_flag) {
    // Let the MMAs already issued finish before shared and tensor memory go.
    const long long t0 = clock64();
    while (clock64() - t0 < 200000ll) {
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tmem, ncols);
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

// The tensor-core reduction's grid: 128 p rows per block, the tokens split
// so that the blocks fit one wave at two per SM, 64-token chunks.
struct TcPlan {
  int ptiles, splits, m_per_split;
  size_t smem;
};
TcPlan skinny_tc_plan(int64_t M, int64_t P, int r) {
  TcPlan t;
  t.ptiles = static_cast<int>((P + kTcP - 1) / kTcP);
  const int64_t max_splits = std::max<int64_t>(1, (M + kTcM - 1) / kTcM);
  int64_t splits = std::max<int64_t>(1, (2 * sms()) / t.ptiles);
  splits = std::min(splits, max_splits);
  const int64_t mps = ((M + splits - 1) / splits + kTcM - 1) / kTcM * kTcM;
  t.m_per_split = static_cast<int>(std::max<int64_t>(mps, kTcM));
  t.splits = std::max(1, static_cast<int>((M + t.m_per_split - 1) / t.m_per_split));
  t.smem = tc_smem_bytes(r);
  return t;
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
    const TcPlan pb = skinny_tc_plan(m, n, r), pa = skinny_tc_plan(m, k, r);
    part = std::max(static_cast<size_t>(pb.splits) * n * r, static_cast<size_t>(pa.splits) * k * r) * 4;
  }
  off = align_up(off + part, 256);
  L.total = off;
  return L;
}

qerl_status launch_skinny(const void* X, int64_t ldx, int64_t M, int64_t P, const LoraDown& T, int r, float scale,
                          bool transposed, float* partial, float* out, int* status, cudaStream_t s) {
  const TcPlan tp = skinny_tc_plan(M, P, r);
  static std::once_flag once;
  static cudaError_t err = cudaSuccess;
  std::call_once(once, [] {
    const int lim = static_cast<int>(tc_smem_bytes(128));
    err = cudaFuncSetAttribute(skinny_tc_kernel<32>, cudaFuncAttributeMaxDynamicSharedMemorySize, lim);
    if (err == cudaSuccess) err = cudaFuncSetAttribute(skinny_tc_kernel<64>, cudaFuncAttributeMaxDynamicSharedMemorySize, lim);
    if (err == cudaSuccess) err = cudaFuncSetAttribute(skinny_tc_kernel<128>, cudaFuncAttributeMaxDynamicSharedMemorySize, lim);
  });
  if (err != cudaSuccess) return QERL_ERR_CUDA;
  const dim3 grid(static_cast<unsigned>(tp.ptiles), static_cast<unsigned>(tp.splits));
  const auto* xb = static_cast<const __nv_bfloat16*>(X);
  const int Mi = static_cast<int>(M), Pi = static_cast<int>(P);
  if (r <= 32)
    skinny_tc_kernel<32><<<grid, kTcThreads, tp.smem, s>>>(xb, ldx, Mi, Pi, T.t, T.parts, T.part_stride, r, tp.m_per_split, partial, status);
  else if (r <= 64)
    skinny_tc_kernel<64><<<grid, kTcThreads, tp.smem, s>>>(xb, ldx, Mi, Pi, T.t, T.parts, T.part_stride, r, tp.m_per_split, partial, status);
  else
    skinny_tc_kernel<128><<<grid, kTcThreads, tp.smem, s>>>(xb, ldx, Mi, Pi, T.t, T.parts, T.part_stride, r, tp.m_per_split, partial, status);
  if (cudaGetLastError() != cudaSuccess) return QERL_ERR_CUDA;
  const int64_t total = P * r;
  const int blocks = static_cast<int>(std::min<int64_t>((total + kThreads - 1) / kThreads, 4 * sms()));
  skinny_reduce_kernel<<<std::max(blocks, 1), kThreads, 0, s>>>(partial, tp.splits, static_cast<int>(P), r, scale,
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
    if ((st = launch_skinny(b.dy, b.lddy, m, n, t, r, scale, false, partial, b.dB, reinterpret_cast<int*>(ws), s)) !=
        QERL_OK)
      return st;
  }
  if (b.dA != nullptr) {
    // dA = s u^T x~ with u = dy B, the down-projection of the dx~ launch.
    const LoraDown u = linear_lora_down(a, 0);
    if ((st = launch_skinny(b.xt, b.ldxt, m, k, u, r, scale, true, partial, b.dA, reinterpret_cast<int*>(ws), s)) !=
        QERL_OK)
      return st;
  }
  return QERL_OK;
}

}  // namespace qerl
