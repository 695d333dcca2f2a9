// linear.cu -- the NVFP4 weight-only linear with the LoRA branch and AQN noise.
//
//   x~ = bf16(x (.) (1 + z))                               ("Noise Merging", Eq. 10-12)
//   y  = S * x~ . (dec(S_E4M3) (.) e2m1(W~))^T             ("NVFP4 Quantization", Eq. 6)
//      + (alpha / r) * (x~ . A) . B                         ("Low-Rank Adaptation", Eq. 2)
//   (QeRL digest, section 3.4)
//
// Two kernels per call:
//
// prep_kernel  (CUDA cores, tiny): the noise step and the LoRA down-projection.
//   - row tasks: x~ for one token row, staged as fp16 times 2^e_m with e_m
//     chosen so the row's largest |x~| lies in [2^14, 2^15).  bf16 values
//     (8 significant bits) are exact in fp16 (11 bits) over that window, so
//     the tensor cores see x~ exactly (up to entries below 2^-28 of the row
//     maximum); 2^-e_m is undone in the epilogue.
//   - LoRA tasks: t = x~ . A over a K-slice, fp32, reduced with atomics.
//
// mma_kernel  (tcgen05 + TMA, the hot loop): a 128-output-feature tile of W
//   is the MMA's M side, tokens are the MMA's N side (16..256), K streams in
//   64-element stages.
//     warp 8      producer: TMA of the packed codes (128 rows x 32 B, 32-byte
//                 swizzle), cp.async of the E4M3 scales (128 x 4 B), TMA of the
//                 staged x~ tile (n_tok x 64 fp16, 128-byte swizzle).
//     warps 0..7  dequant: E2M1 pairs -> fp16 pairs (cvt.f16x2.e2m1x2), times
//                 the block scale (cvt.f16x2.e4m3x2) -- exact products -- written
//                 in the 128-byte-swizzled K-major layout the MMA reads.
//     warp 9      MMA issuer: 4 x tcgen05.mma kind::f16 (M=128, N=n_tok, K=16)
//                 per stage into an fp32 TMEM accumulator; tcgen05.commit frees
//                 the stage.
//   Epilogue (warps 0..7): TMEM -> registers, y = acc * S * 2^-e_m
//   + (alpha/r) t.B, rounded to bf16.  Small-N decode shapes split K across a
//   thread-block cluster; partner CTAs reduce their fp32 partial tiles
//   through distributed shared memory, with no global scratch and no atomics.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <atomic>
#include <cstring>
#include <mutex>

#include "qerl_internal.h"
#include "qerl_ptx.cuh"

namespace qerl {
namespace {

// ------------------------------------------------------------------ prep

constexpr int kPrepThreads = 256;
constexpr int kLoraMaxRows = 64;  // token rows per LoRA task (fewer for large r)
constexpr int kLoraOutPerThread = 8;

struct PrepParams {
  const __nv_bfloat16* x;
  const float* z;
  const __nv_bfloat16* A;
  __half* xs;   // [M][K] staged x~ * 2^e_m
  float* rinv;  // [M] 2^-e_m
  float* t;     // [M][r]
  int64_t ldx;
  int M, K, r;
  int row_tasks;       // = M
  int lora_rows;       // token rows per LoRA task: rows * r <= 256 * kLoraOutPerThread
  int lora_row_tiles;  // ceil(M / lora_rows)
  int lora_k_chunks;   // number of K slices
  int k64_per_chunk;   // 64-wide K blocks per slice
};

__device__ __forceinline__ float noisy(float xv, float zv) {
  // bf16_RN( x * (1 + z) ): one fp32 add, one fp32 multiply, one rounding.
  return __bfloat162float(__float2bfloat16_rn(__fmul_rn(xv, __fadd_rn(1.0f, zv))));
}

__global__ void __launch_bounds__(kPrepThreads) prep_kernel(PrepParams p) {
  extern __shared__ __align__(16) uint8_t sm[];
  const int tid = threadIdx.x;
  if (blockIdx.x < p.row_tasks) {
    // ---- row task: x~ row -> smem (bf16), amax, then fp16 * 2^e
    const int m = blockIdx.x;
    __nv_bfloat16* xt = reinterpret_cast<__nv_bfloat16*>(sm);
    const uint4* xrow = reinterpret_cast<const uint4*>(p.x + static_cast<int64_t>(m) * p.ldx);
    unsigned amax = 0;
    for (int v = tid; v < p.K / 8; v += kPrepThreads) {
      uint4 raw = __ldg(xrow + v);
      __nv_bfloat16* e = reinterpret_cast<__nv_bfloat16*>(&raw);
      if (p.z != nullptr) {
        const float4 z0 = __ldg(reinterpret_cast<const float4*>(p.z) + 2 * v);
        const float4 z1 = __ldg(reinterpret_cast<const float4*>(p.z) + 2 * v + 1);
        const float zz[8] = {z0.x, z0.y, z0.z, z0.w, z1.x, z1.y, z1.z, z1.w};
#pragma unroll
        for (int j = 0; j < 8; ++j) e[j] = __float2bfloat16_rn(__fmul_rn(__bfloat162float(e[j]), __fadd_rn(1.0f, zz[j])));
      }
#pragma unroll
      for (int j = 0; j < 8; ++j) amax = max(amax, static_cast<unsigned>(__bfloat16_as_ushort(e[j]) & 0x7FFFu));
      reinterpret_cast<uint4*>(xt)[v] = raw;
    }
    amax = __reduce_max_sync(0xFFFFFFFFu, amax);
    __shared__ unsigned red[kPrepThreads / 32];
    if ((tid & 31) == 0) red[tid >> 5] = amax;
    __syncthreads();
    unsigned a = 0;
#pragma unroll
    for (int i = 0; i < kPrepThreads / 32; ++i) a = max(a, red[i]);
    const float af = __uint_as_float(a << 16);
    int e = 0;
    if (af > 0.0f && af < INFINITY) {
      int ex;
      frexpf(af, &ex);  // af in [2^(ex-1), 2^ex)
      e = 15 - ex;      // af * 2^e in [2^14, 2^15)
      e = max(-126, min(126, e));
    }
    const float scale = __uint_as_float(static_cast<uint32_t>(127 + e) << 23);
    if (tid == 0) p.rinv[m] = __uint_as_float(static_cast<uint32_t>(127 - e) << 23);
    uint4* dst = reinterpret_cast<uint4*>(p.xs + static_cast<int64_t>(m) * p.K);
    for (int v = tid; v < p.K / 8; v += kPrepThreads) {
      uint4 raw = reinterpret_cast<const uint4*>(xt)[v];
      const __nv_bfloat16* e8 = reinterpret_cast<const __nv_bfloat16*>(&raw);
      uint4 out;
      __half2* o = reinterpret_cast<__half2*>(&out);
#pragma unroll
      for (int j = 0; j < 4; ++j)
        o[j] = __floats2half2_rn(__bfloat162float(e8[2 * j]) * scale, __bfloat162float(e8[2 * j + 1]) * scale);
      dst[v] = out;
    }
    return;
  }
  // ---- LoRA task: t[rows][:] += x~[rows][kslice] . A[kslice][:]
  const int task = blockIdx.x - p.row_tasks;
  const int rt = task % p.lora_row_tiles;
  const int kc = task / p.lora_row_tiles;
  const int row0 = rt * p.lora_rows;
  const int rows = min(p.lora_rows, p.M - row0);
  const int r = p.r;
  float* xsm = reinterpret_cast<float*>(sm);  // [lora_rows][64]
  float* asm_ = xsm + p.lora_rows * 64;       // [64][r]
  const int nout = rows * r;
  float acc[kLoraOutPerThread];
#pragma unroll
  for (int i = 0; i < kLoraOutPerThread; ++i) acc[i] = 0.0f;
  const int kb_begin = kc * p.k64_per_chunk;
  const int kb_end = min(p.K / 64, kb_begin + p.k64_per_chunk);
  for (int kb = kb_begin; kb < kb_end; ++kb) {
    __syncthreads();
    const int k0 = kb * 64;
    for (int i = tid; i < rows * 64; i += kPrepThreads) {
      const int rr = i / 64, kk = i % 64;
      const float xv = __bfloat162float(p.x[static_cast<int64_t>(row0 + rr) * p.ldx + k0 + kk]);
      xsm[rr * 64 + kk] = p.z != nullptr ? noisy(xv, __ldg(p.z + k0 + kk)) : xv;
    }
    for (int i = tid; i < 64 * r; i += kPrepThreads)
      asm_[i] = __bfloat162float(p.A[static_cast<int64_t>(k0) * r + i]);
    __syncthreads();
#pragma unroll
    for (int q = 0; q < kLoraOutPerThread; ++q) {
      const int o = tid + q * kPrepThreads;
      if (o < nout) {
        const int rr = o / r, j = o % r;
        float s = acc[q];
#pragma unroll 8
        for (int kk = 0; kk < 64; ++kk) s = fmaf(xsm[rr * 64 + kk], asm_[kk * r + j], s);
        acc[q] = s;
      }
    }
  }
#pragma unroll
  for (int q = 0; q < kLoraOutPerThread; ++q) {
    const int o = tid + q * kPrepThreads;
    if (o < nout) atomicAdd(p.t + static_cast<int64_t>(row0 + o / r) * r + (o % r), acc[q]);
  }
}

// ------------------------------------------------------------------ MMA kernel

constexpr int kMmaThreads = 320;  // warps 0-7 dequant+epilogue, 8 producer, 9 MMA
constexpr int kTileN = 128;       // output features per CTA (MMA M)
constexpr int kStageK = 64;       // K per pipeline stage
constexpr int kCodesStageBytes = kTileN * kStageK / 2;   // 4096
constexpr int kScalesStageBytes = kTileN * kStageK / 16; // 512
constexpr int kAStageBytes = kTileN * kStageK * 2;       // 16384 (fp16)
constexpr int kMaxStages = 8;
constexpr int kSmemLimit = 232448;  // 227 KB opt-in per CTA

struct MmaParams {
  const uint8_t* scales;
  const float* tensor_scale;
  const float* rinv;
  const float* t;
  const __nv_bfloat16* B;
  void* y;
  int* status;
  int M, N, K, r;
  int n_tok;   // tokens per tile (MMA N), multiple of 16, <= 256
  int split;   // K split across the cluster (gridDim.x)
  int stages;  // pipeline depth
  int tmem_cols;
  uint32_t bars_off;  // barrier block offset: after both the ring and the epilogue staging
  float lora_scale;
  int y_f32;
};

struct SmemLayout {
  uint32_t a, b, codes, scales, ring_bytes;
};

__host__ __device__ inline SmemLayout smem_layout(int n_tok, int stages) {
  SmemLayout L;
  const uint32_t b_stage = static_cast<uint32_t>(n_tok) * 128u;
  L.a = 0;
  L.b = L.a + stages * kAStageBytes;
  L.codes = L.b + stages * b_stage;
  L.scales = L.codes + stages * kCodesStageBytes;
  L.ring_bytes = L.scales + stages * kScalesStageBytes;
  return L;
}

__host__ __device__ inline uint32_t epilogue_bytes(int n_tok, int r, int split) {
  uint32_t part = split > 1 ? static_cast<uint32_t>(n_tok) * kTileN * 4u : 0u;
  return part + static_cast<uint32_t>(n_tok) * r * 4u + static_cast<uint32_t>(r) * kTileN * 4u +
         static_cast<uint32_t>(n_tok) * 4u;
}

__device__ __forceinline__ void named_bar_sync(int id, int nthreads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

__device__ __forceinline__ void store_out(const MmaParams& p, int m, int n, float v) {
  const int64_t idx = static_cast<int64_t>(m) * p.N + n;
  if (p.y_f32)
    reinterpret_cast<float*>(p.y)[idx] = v;
  else
    reinterpret_cast<__nv_bfloat16*>(p.y)[idx] = __float2bfloat16_rn(v);
}

__global__ void __launch_bounds__(kMmaThreads, 1)
    mma_kernel(const __grid_constant__ CUtensorMap tm_codes, const __grid_constant__ CUtensorMap tm_xs,
               const MmaParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const SmemLayout L = smem_layout(p.n_tok, p.stages);
  uint64_t* raw_full = reinterpret_cast<uint64_t*>(smem + p.bars_off);
  uint64_t* op_full = raw_full + kMaxStages;
  uint64_t* empty = op_full + kMaxStages;
  uint64_t* acc_full = empty + kMaxStages;
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(acc_full + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_holder + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int split_idx = blockIdx.x;
  const int n0 = blockIdx.y * kTileN;
  const int m0 = blockIdx.z * p.n_tok;
  const int ks_total = p.K / kStageK;
  const int ks_begin = static_cast<int>(static_cast<int64_t>(split_idx) * ks_total / p.split);
  const int ks_end = static_cast<int>(static_cast<int64_t>(split_idx + 1) * ks_total / p.split);
  const int nks = ks_end - ks_begin;
  const int stages = p.stages;

  if (threadIdx.x == 0) {
    for (int s = 0; s < stages; ++s) {
      mbar_init(&raw_full[s], 33);  // producer expect_tx + 32 cp.async arrivals
      mbar_init(&op_full[s], 9);    // 8 dequant warps + producer expect_tx (x~ tile)
      mbar_init(&empty[s], 1);      // tcgen05.commit
    }
    mbar_init(acc_full, 1);
    *abort_flag = 0;
    fence_mbarrier_init();
  }
  if (warp == 9) {
    tmem_alloc(tmem_holder, p.tmem_cols);
    tmem_relinquish();
  }
  if (warp == 8 && lane == 0) {
    tma_prefetch_desc(&tm_codes);
    tma_prefetch_desc(&tm_xs);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_holder;

  if (warp == 8) {
    // ------------------------------------------------------------ producer
    const int kq = p.K / 16;  // scale bytes per row
    for (int i = 0; i < nks; ++i) {
      const int s = i % stages;
      const uint32_t ph = (i / stages) & 1;
      int ok = 1;
      if (lane == 0) ok = mbar_wait(&empty[s], ph ^ 1, abort_flag, p.status);
      ok = __shfl_sync(0xFFFFFFFFu, ok, 0);
      if (!ok) break;
      const int kidx = ks_begin + i;
      if (lane == 0) {
        mbar_arrive_expect_tx(&raw_full[s], kCodesStageBytes);
        tma_load_2d(smem + L.codes + s * kCodesStageBytes, &tm_codes, kidx * (kStageK / 2), n0, &raw_full[s]);
      }
      uint8_t* sdst = smem + L.scales + s * kScalesStageBytes;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int row = lane * 4 + j;
        const int n = n0 + row;
        const bool in = n < p.N;
        const uint8_t* src = p.scales + static_cast<int64_t>(in ? n : 0) * kq + kidx * 4;
        cp_async_4(sdst + row * 4, src, in ? 4u : 0u);
      }
      cp_async_mbar_arrive_noinc(&raw_full[s]);
      if (lane == 0) {
        mbar_arrive_expect_tx(&op_full[s], static_cast<uint32_t>(p.n_tok) * 128u);
        tma_load_2d(smem + L.b + s * (p.n_tok * 128), &tm_xs, kidx * kStageK, m0, &op_full[s]);
      }
    }
  } else if (warp == 9) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      const uint32_t idesc = idesc_f16_f32(kTileN, static_cast<uint32_t>(p.n_tok));
      for (int i = 0; i < nks; ++i) {
        const int s = i % stages;
        const uint32_t ph = (i / stages) & 1;
        if (!mbar_wait(&op_full[s], ph, abort_flag, p.status)) break;
        tc_fence_after();
        const uint32_t a_addr = smem_u32(smem + L.a + s * kAStageBytes);
        const uint32_t b_addr = smem_u32(smem + L.b + s * (p.n_tok * 128));
#pragma unroll
        for (int kk = 0; kk < kStageK / 16; ++kk)
          tc_mma_f16(tmem_base, sw128_kmajor_desc(a_addr + kk * 32), sw128_kmajor_desc(b_addr + kk * 32), idesc,
                     (i > 0 || kk > 0) ? 1u : 0u);
        tc_commit(&empty[s]);
      }
      tc_commit(acc_full);  // always, so the epilogue's wait completes even after an abort
    }
  } else {
    // ------------------------------------------------------------ dequant (warps 0-7)
    const int row = 16 * warp + (lane & 15);
    const int half = lane >> 4;
    for (int i = 0; i < nks; ++i) {
      const int s = i % stages;
      const uint32_t ph = (i / stages) & 1;
      if (!mbar_wait(&raw_full[s], ph, abort_flag, p.status)) break;
      uint32_t coff = static_cast<uint32_t>(row * 32 + half * 16);
      coff ^= ((coff >> 7) & 1u) << 4;  // 32-byte TMA swizzle: bit 4 ^= bit 7
      const uint4 cw = *reinterpret_cast<const uint4*>(smem + L.codes + s * kCodesStageBytes + coff);
      const uint32_t sc2 =
          *reinterpret_cast<const uint16_t*>(smem + L.scales + s * kScalesStageBytes + row * 4 + half * 2);
      const __half2 s01 = e4m3x2_to_half2(sc2);
      const __half2 sa = __low2half2(s01), sb = __high2half2(s01);
      const uint32_t words[4] = {cw.x, cw.y, cw.z, cw.w};
      uint8_t* arow = smem + L.a + s * kAStageBytes + row * 128;
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const __half2 sq = q < 2 ? sa : sb;
        uint4 o;
        __half2* oh = reinterpret_cast<__half2*>(&o);
#pragma unroll
        for (int b = 0; b < 4; ++b) oh[b] = __hmul2(e2m1x2_to_half2((words[q] >> (8 * b)) & 0xFFu), sq);
        const int chunk = half * 4 + q;
        *reinterpret_cast<uint4*>(arow + ((chunk ^ (row & 7)) << 4)) = o;
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(&op_full[s]);
    }
  }

  // ---------------------------------------------------------------- epilogue
  float* part = reinterpret_cast<float*>(smem);  // [n_tok][128] fp32 partial (split > 1)
  float* ts = part + (p.split > 1 ? p.n_tok * kTileN : 0);  // [n_tok][r]
  float* bs = ts + p.n_tok * p.r;                            // [r][128]
  float* sm = bs + p.r * kTileN;                             // [n_tok] S * 2^-e_m
  if (warp < 8) {
    const bool ok = mbar_wait(acc_full, 0, abort_flag, p.status);
    tc_fence_after();
    // The ring is idle once the accumulator is complete: stage the epilogue operands there.
    const float S = *p.tensor_scale;
    for (int i = threadIdx.x; i < p.n_tok * p.r; i += 256) {
      const int m = m0 + i / p.r;
      ts[i] = (m < p.M) ? p.t[static_cast<int64_t>(m) * p.r + (i % p.r)] : 0.0f;
    }
    for (int i = threadIdx.x; i < p.r * kTileN; i += 256) {
      const int n = n0 + (i % kTileN);
      bs[i] = (n < p.N) ? __bfloat162float(p.B[static_cast<int64_t>(i / kTileN) * p.N + n]) : 0.0f;
    }
    for (int i = threadIdx.x; i < p.n_tok; i += 256) sm[i] = (m0 + i < p.M) ? S * p.rinv[m0 + i] : 0.0f;
    named_bar_sync(1, 256);

    const int q = warp & 3;
    const int nl = q * 32 + lane;
    const int n = n0 + nl;
    const int cols = p.n_tok / 2;
    const int c0 = (warp >> 2) * cols;
    const uint32_t taddr = tmem_base + (static_cast<uint32_t>(q * 32) << 16);
    for (int c = c0; c < c0 + cols; c += 8) {
      float v[8];
      tmem_ld_x8(taddr + c, v);
      tmem_ld_wait();
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const int ml = c + j;
        const float acc = ok ? v[j] : 0.0f;
        if (p.split > 1) {
          part[ml * kTileN + nl] = acc;
        } else if (m0 + ml < p.M && n < p.N) {
          float l = 0.0f;
          for (int jj = 0; jj < p.r; ++jj) l = fmaf(ts[ml * p.r + jj], bs[jj * kTileN + nl], l);
          store_out(p, m0 + ml, n, fmaf(p.lora_scale, l, acc * sm[ml]));
        }
      }
    }
  }
  if (*abort_flag) {
    // Let copies that were already issued land before shared memory is released.
    const uint64_t t0 = globaltimer_ns();
    while (globaltimer_ns() - t0 < 50000ull) {
    }
  }
  tc_fence_before();
  __syncthreads();

  if (p.split > 1) {
    cluster_sync_all();  // every partner's partial tile is in its shared memory
    if (warp < 8) {
      const int rank = static_cast<int>(cluster_ctarank());
      const int per = (p.n_tok + p.split - 1) / p.split;
      const int mb = rank * per;
      const int me = min(p.n_tok, mb + per);
      const uint32_t part_addr = smem_u32(part);
      for (int i = threadIdx.x; i < (me - mb) * kTileN; i += 256) {
        const int ml = mb + i / kTileN, nl = i % kTileN;
        const int n = n0 + nl;
        if (m0 + ml >= p.M || n >= p.N) continue;
        const uint32_t off = static_cast<uint32_t>(ml * kTileN + nl) * 4u;
        float acc = 0.0f;
        for (int qq = 0; qq < p.split; ++qq) acc += ld_shared_cluster_f32(mapa_shared(part_addr + off, qq));
        float l = 0.0f;
        for (int jj = 0; jj < p.r; ++jj) l = fmaf(ts[ml * p.r + jj], bs[jj * kTileN + nl], l);
        store_out(p, m0 + ml, n, fmaf(p.lora_scale, l, acc * sm[ml]));
      }
    }
    cluster_sync_all();  // partners are done reading this CTA's partial tile
  }
  if (warp == 9) tmem_dealloc(tmem_base, p.tmem_cols);
}

// ------------------------------------------------------------------ host side

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  static std::atomic<PFN_cuTensorMapEncodeTiled_v12000> fn{nullptr};
  PFN_cuTensorMapEncodeTiled_v12000 f = fn.load();
  if (f == nullptr) {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) !=
            cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      return nullptr;
    f = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
    fn.store(f);
  }
  return f;
}

bool make_map_2d(CUtensorMap* map, CUtensorMapDataType dt, const void* base, uint64_t inner, uint64_t outer,
                 uint64_t row_bytes, uint32_t box_inner, uint32_t box_outer, CUtensorMapSwizzle swz) {
  auto enc = tensor_map_encoder();
  if (enc == nullptr) return false;
  const cuuint64_t dims[2] = {inner, outer};
  const cuuint64_t strides[1] = {row_bytes};
  const cuuint32_t box[2] = {box_inner, box_outer};
  const cuuint32_t estr[2] = {1, 1};
  return enc(map, dt, 2, const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, swz,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

struct DeviceInfo {
  int sms = 148;
};

DeviceInfo device_info() {
  DeviceInfo d;
  int dev = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev);
  return d;
}

struct LinearLayout {
  size_t xs, rinv, t, total;
};

LinearLayout linear_layout(int64_t m, int64_t k, int r) {
  LinearLayout L;
  L.xs = kWsHeaderBytes;
  L.rinv = align_up(L.xs + static_cast<size_t>(m) * k * 2, 256);
  L.t = align_up(L.rinv + static_cast<size_t>(m) * 4, 256);
  L.total = align_up(L.t + static_cast<size_t>(m) * (r > 0 ? r : 0) * 4, 256);
  return L;
}

}  // namespace

size_t linear_workspace_bytes(int64_t m, int64_t k, int r) { return linear_layout(m, k, r).total; }

qerl_status launch_lora_linear(const LinearArgs& a, cudaStream_t s) {
  const int M = static_cast<int>(a.m), N = static_cast<int>(a.n), K = static_cast<int>(a.k);
  const bool lora = a.r > 0 && a.A != nullptr && a.B != nullptr;
  const int r = lora ? a.r : 0;
  const LinearLayout WL = linear_layout(a.m, a.k, r);
  uint8_t* ws = static_cast<uint8_t*>(a.workspace);
  int* status = reinterpret_cast<int*>(ws);
  __half* xs = reinterpret_cast<__half*>(ws + WL.xs);
  float* rinv = reinterpret_cast<float*>(ws + WL.rinv);
  float* t = reinterpret_cast<float*>(ws + WL.t);
  const DeviceInfo dev = device_info();

  // ---- prep: noise + fp16 staging (+ LoRA down-projection)
  PrepParams pp{};
  pp.x = static_cast<const __nv_bfloat16*>(a.x);
  pp.z = a.z;
  pp.A = static_cast<const __nv_bfloat16*>(a.A);
  pp.xs = xs;
  pp.rinv = rinv;
  pp.t = t;
  pp.ldx = a.ldx;
  pp.M = M;
  pp.K = K;
  pp.r = r;
  pp.row_tasks = M;
  int lora_blocks = 0;
  if (lora) {
    if (cudaMemsetAsync(t, 0, static_cast<size_t>(M) * r * 4, s) != cudaSuccess) return QERL_ERR_CUDA;
    pp.lora_rows = std::min(kLoraMaxRows, kPrepThreads * kLoraOutPerThread / r);
    pp.lora_row_tiles = (M + pp.lora_rows - 1) / pp.lora_rows;
    const int k64 = K / 64;
    const int target = 2 * dev.sms;
    int per = (k64 * pp.lora_row_tiles + target - 1) / target;
    per = std::max(per, 1);
    pp.k64_per_chunk = per;
    pp.lora_k_chunks = (k64 + per - 1) / per;
    lora_blocks = pp.lora_row_tiles * pp.lora_k_chunks;
  }
  size_t prep_smem = static_cast<size_t>(K) * 2;
  if (lora) prep_smem = std::max(prep_smem, static_cast<size_t>(pp.lora_rows * 64 + 64 * r) * 4);
  if (prep_smem > 48 * 1024) {
    if (cudaFuncSetAttribute(prep_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(prep_smem)) != cudaSuccess)
      return QERL_ERR_CUDA;
  }
  prep_kernel<<<M + lora_blocks, kPrepThreads, prep_smem, s>>>(pp);
  if (cudaGetLastError() != cudaSuccess) return QERL_ERR_CUDA;

  // ---- tile shape
  int n_tok, m_tiles;
  if (M <= 256) {
    n_tok = (M + 15) / 16 * 16;
    m_tiles = 1;
  } else {
    n_tok = 256;
    m_tiles = (M + 255) / 256;
  }
  const int n_tiles = (N + kTileN - 1) / kTileN;
  const int ks_total = K / kStageK;
  int split = 1;
  if (n_tok <= 128) {
    // K split across a cluster when the tiles alone leave SMs idle: minimise
    // waves x stages per CTA, with a small per-CTA fixed cost.
    double best = 1e30;
    for (int sp = 1; sp <= 8 && sp <= ks_total; ++sp) {
      const int ctas = n_tiles * m_tiles * sp;
      const int waves = (ctas + dev.sms - 1) / dev.sms;
      const double cost = waves * (static_cast<double>((ks_total + sp - 1) / sp) + 3.0);
      if (cost < best - 1e-9) {
        best = cost;
        split = sp;
      }
    }
  }
  const uint32_t epi = epilogue_bytes(n_tok, r, split);
  int stages = kMaxStages;
  while (stages > 2 && std::max(smem_layout(n_tok, stages).ring_bytes, epi) + 256 + 1024 > kSmemLimit) --stages;
  const SmemLayout SL = smem_layout(n_tok, stages);
  const uint32_t bars_off = static_cast<uint32_t>(align_up(std::max(SL.ring_bytes, epi), 16));
  const uint32_t smem_bytes = bars_off + 256 + 1024;  // + barrier block + 1024-byte alignment slack
  if (smem_bytes > kSmemLimit) return QERL_ERR_UNSUPPORTED_SHAPE;
  int tmem_cols = 32;
  while (tmem_cols < n_tok) tmem_cols *= 2;

  CUtensorMap tm_codes, tm_xs;
  if (!make_map_2d(&tm_codes, CU_TENSOR_MAP_DATA_TYPE_UINT8, a.codes, static_cast<uint64_t>(K) / 2,
                   static_cast<uint64_t>(N), static_cast<uint64_t>(K) / 2, kStageK / 2, kTileN,
                   CU_TENSOR_MAP_SWIZZLE_32B))
    return QERL_ERR_CUDA;
  if (!make_map_2d(&tm_xs, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, xs, static_cast<uint64_t>(K), static_cast<uint64_t>(M),
                   static_cast<uint64_t>(K) * 2, kStageK, static_cast<uint32_t>(n_tok), CU_TENSOR_MAP_SWIZZLE_128B))
    return QERL_ERR_CUDA;

  MmaParams mp{};
  mp.scales = a.scales;
  mp.tensor_scale = a.tensor_scale;
  mp.rinv = rinv;
  mp.t = t;
  mp.B = static_cast<const __nv_bfloat16*>(a.B);
  mp.y = a.y;
  mp.status = status;
  mp.M = M;
  mp.N = N;
  mp.K = K;
  mp.r = r;
  mp.n_tok = n_tok;
  mp.split = split;
  mp.stages = stages;
  mp.tmem_cols = tmem_cols;
  mp.bars_off = bars_off;
  mp.lora_scale = lora ? a.alpha / static_cast<float>(r) : 0.0f;
  mp.y_f32 = a.y_f32 ? 1 : 0;

  static std::once_flag attr_once;
  static cudaError_t attr_err = cudaSuccess;
  std::call_once(attr_once, [] {
    attr_err = cudaFuncSetAttribute(mma_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemLimit);
  });
  if (attr_err != cudaSuccess) return QERL_ERR_CUDA;

  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(static_cast<unsigned>(split), static_cast<unsigned>(n_tiles), static_cast<unsigned>(m_tiles));
  cfg.blockDim = dim3(kMmaThreads, 1, 1);
  cfg.dynamicSmemBytes = smem_bytes;
  cfg.stream = s;
  cudaLaunchAttribute attrs[1];
  attrs[0].id = cudaLaunchAttributeClusterDimension;
  attrs[0].val.clusterDim.x = static_cast<unsigned>(split);
  attrs[0].val.clusterDim.y = 1;
  attrs[0].val.clusterDim.z = 1;
  cfg.attrs = attrs;
  cfg.numAttrs = 1;
  if (cudaLaunchKernelEx(&cfg, mma_kernel, tm_codes, tm_xs, mp) != cudaSuccess) return QERL_ERR_CUDA;
  return QERL_OK;
}

}  // namespace qerl
