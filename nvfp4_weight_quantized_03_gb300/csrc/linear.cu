// linear.cu -- the NVFP4 weight-only linear with the LoRA branch and AQN noise.
//
//   x~ = bf16(x (.) (1 + z))                               ("Noise Merging", Eq. 10-12)
//   y  = S * x~ . (dec(S_E4M3) (.) e2m1(W~))^T             ("NVFP4 Quantization", Eq. 6)
//      + (alpha / r) * (x~ . A) . B                         ("Low-Rank Adaptation", Eq. 2)
//   (QeRL digest, section 3.4)
//
// Two kernels per launch; one launch serves up to four linears that share x,
// z and K (q/k/v, gate/up), their 128-row weight tiles concatenated on the
// grid's y axis.
//
// prep_kernel  (CUDA cores, latency-bound, tiny): the noise step and the LoRA
//   down-projection.
//   - row tasks: x~ for one token row, staged as fp16 times 2^e_m with e_m
//     chosen so the row's largest |x~| lies in [2^14, 2^15).  bf16 values
//     (8 significant bits) are exact in fp16 (11 bits) over that window, so
//     the tensor cores see x~ exactly (up to entries below 2^-28 of the row
//     maximum); 2^-e_m is undone in the epilogue.  For decode (<= 128
//     tokens) the rows are written as swizzled 64-wide K slabs that one bulk
//     copy moves per weight stage.
//   - LoRA tasks: t = x~ . A^T for a 16-row x 32-rank tile over one K group;
//     the CTAs of a thread-block cluster split the group and reduce through
//     distributed shared memory.  Groups are summed in order by the consumer:
//     no atomics, bit-reproducible.
//
// mma_kernel  (tcgen05, the hot loop): a 128-output-feature tile of W is the
//   MMA's M side, tokens are its N side (16..256).  Weights arrive in the
//   packed layout (one 18432-byte block per 128 rows x 256 K: swizzled E2M1
//   codes + interleaved E4M3 scale pairs), one 1-D bulk copy per block.
//   Nineteen warps; the light roles take the low (older) warp numbers so the
//   scheduler does not starve them behind the ALU-bound dequant warps:
//     warp 0       weight producer: L2 prefetch a few stages ahead, bulk copy
//                  of each block (the first ring of blocks is requested
//                  before waiting for the preceding kernel).
//     warp 1       activation producer: x~ per stage, bulk-copied slabs up to
//                  128 tokens, 2-D TMA tiles beyond.  Up to 64 tokens a weight
//                  stage's slabs share its tensor-memory A slot's index and
//                  empty barrier (one commit per issuer frees both).
//     warp 2       LoRA operands: sums the down-projection groups, scales each
//                  token row and splits t into bf16 hi + lo.
//     warps 3..10  MMA issuers (2, 4 or 8 of them; lane 0 issues):
//                  tcgen05.mma kind::f16, K=16, each into its own fp32 TMEM
//                  accumulator, so that the ~150-cycle issue cost of an MMA
//                  overlaps across threads; the epilogue adds them.  Up to 64
//                  tokens they form two groups on alternate weight stages.
//                  Issuer 0 also adds the LoRA up-projection
//                  B . (t_hi + t_lo)^T into its accumulator.
//     warps 11..18 dequant: E2M1 pairs -> fp16 pairs, times the block scale
//                  (exact products).  Decode writes them to tensor memory as
//                  the MMA's A operand (tcgen05.st), a weight stage per
//                  hand-over; prefill writes them to shared memory in the
//                  128-byte-swizzled K-major layout.
//   Epilogue (dequant warps): y = S * 2^-e_m * (sum of accumulators), rounded
//   to bf16 or kept fp32.  When the weight tiles leave SMs idle, K is split
//   across a cluster; each CTA writes its scaled partial tile to shared
//   memory and the partners sum them through distributed shared memory.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <atomic>
#include <cstring>
#include <mutex>
#include <type_traits>

#include "qerl_internal.h"
#include "qerl_ptx.cuh"

namespace qerl {
namespace {

// ------------------------------------------------------------------ prep

constexpr int kMaxLinears = 4;  // linears sharing one launch (x, z and K)
constexpr int kPrepThreads = 256;
constexpr uint32_t kSmemPerSm = 233472;  // 228 KB per SM, 1 KB of it reserved per resident CTA
constexpr int kLoraTileM = 16;   // token rows per LoRA tile
constexpr int kLoraTileR = 32;   // ranks per LoRA tile
constexpr int kLoraKc = 64;      // K per shared-memory chunk
constexpr int kLoraPad = 68;     // padded row length (floats): conflict-free float4 reads
constexpr int kLoraStages = 3;   // chunks in flight (cp.async ring)
// One ring stage: x [16][64] bf16, A [32][64] bf16, z [16][64] fp32 (one
// row of it when the noise is shared by all rows).
constexpr int kLoraStageBytes = (kLoraTileM + kLoraTileR) * kLoraKc * 2 + kLoraTileM * kLoraKc * 4;
constexpr int kLoraTileSmemBytes = kLoraStages * kLoraStageBytes + (kLoraTileM + kLoraTileR) * kLoraPad * 4;
constexpr int kPrepMaxCluster = 8;
// + the receive buffer of the partial-tile push (each CTA of a cluster owns
// ceil(512 / cluster) entries and receives them from every partner: at most
// 519 fp32) and its mbarrier.
constexpr int kLoraRecvBytes = 2080;
constexpr bool lora_recv_fits(int c) {
  return c > kPrepMaxCluster ||
         (4 * c * ((kLoraTileM * kLoraTileR + c - 1) / c) <= kLoraRecvBytes && lora_recv_fits(c + 1));
}
static_assert(lora_recv_fits(1), "LoRA receive buffer");
constexpr int kLoraSmemBytes = kLoraTileSmemBytes + kLoraRecvBytes + 16;

struct PrepParams {
  const __nv_bfloat16* x;
  const float* z;
  int64_t ldz;  // noise row stride: 0 = one vector z[K] for every row, else row m uses z + m * ldz
  // RMSNorm with merged noise (row tasks; "Noise Merging", Eq. 10-11): x holds
  // h, and x~ = bf16((w_norm + Zn) * (h / sqrt(mean(h^2) + delta))) in fp64
  // with one rounding.  xt_out (row stride ldo) receives x~ when not null;
  // the staged copy (xs) is skipped when xs is null.
  const __nv_bfloat16* w_norm;
  const float* Zn;
  double delta;
  __nv_bfloat16* xt_out;
  int64_t ldo;
  int rmsnorm;
  const __nv_bfloat16* A[kMaxLinears];  // [r][K] per linear (LoRA down-projections)
  int r[kMaxLinears];
  float* t[kMaxLinears];   // [groups][M][r] partial sums of x~ . A^T over K group g, per linear
  float* tf[kMaxLinears];  // [M][r] their sum (written by the last cluster to finish a LoRA tile)
  unsigned* tile_count;    // per LoRA tile (lora_tiles of them): clusters done; reset by the last one
  int* status;             // error record (a partial-tile push that never completed)
  int sum_groups;          // 1: sum the groups into tf (the consumer reads one sum); 0: the consumer adds them
  int tile_begin[kMaxLinears + 1];  // LoRA tiles of linear l: [tile_begin[l], tile_begin[l+1])
  __half* xs;   // staged x~ * 2^e_m: [M][K], or tiled (see xs_tile_offset)
  float* rinv;  // [M] 2^-e_m
  int64_t ldx;
  int M, K;
  int row_groups;    // blockIdx.y < row_groups: token rows blockIdx.y * cluster + blockIdx.x
  int lora_m_tiles;  // ceil(M / kLoraTileM)
  int lora_tiles;    // all linears' tiles: sum of lora_m_tiles * ceil(r / kLoraTileR)
  int cluster;       // CTAs per cluster (gridDim.x)
  int groups;        // K groups; the cluster's CTAs split a group's K range
  int tiled_rows;    // > 0: x~ in the tiled layout for this many rows (>= M; rows past M are zero)
};

// Tiled x~ (token tiles of up to 128 rows, one tile): for each 256-wide K
// stage g, four 64-wide slabs of tiled_rows rows x 128 bytes, each row's
// 16-byte chunk c at position c ^ (row % 8) -- the shared-memory image of
// the MMA's 128-byte-swizzled K-major operand, so one bulk copy per stage
// moves it.  Byte offset of elements k .. k + 7 (k % 8 == 0) of row m:
__host__ __device__ inline size_t xs_tile_offset(int m, int k, int rows) {
  const int g = k >> 8, sl = (k >> 6) & 3, c = (k >> 3) & 7;
  return static_cast<size_t>(g) * (4u * rows * 128u) + static_cast<size_t>(sl) * rows * 128u + m * 128u +
         ((c ^ (m & 7)) << 4);
}

// K is cut into groups * cluster slices of 64-wide chunks, about two chunks
// per CTA.  Each group's partial t is reduced inside its cluster; the MMA
// kernel adds the groups.  Fewer groups for larger token tiles keep that last
// sum small.
struct LoraSplit {
  int cluster, groups;
};
// The last cluster to finish a tile sums the groups (see prep_kernel), so the
// group count only trades prep parallelism against that final sum.  Tiles
// count their finished clusters in a fixed region of the workspace
// (kMaxLoraCounters); a call with more LoRA tiles uses one group per tile.
constexpr int kMaxLoraCounters = 4096;
__host__ inline int lora_tile_count(int64_t m, const int* ranks, int nlin) {
  int64_t tiles = 0;
  for (int i = 0; i < nlin; ++i)
    if (ranks[i] > 0) tiles += ((m + kLoraTileM - 1) / kLoraTileM) * ((ranks[i] + kLoraTileR - 1) / kLoraTileR);
  return static_cast<int>(std::min<int64_t>(tiles, INT32_MAX));
}
// Above 64 tokens (pair-mode-sized tiles, prefill) the prep kernel sums the
// groups; smaller tiles stage every group's partial sums and add them, so
// their group count is bounded by that staging buffer (256 / n_tok groups).
__host__ inline bool lora_sum_in_prep(int64_t m) { return m > 64; }
// `chunks`: the 64-wide chunks a prep CTA takes up to 64 tokens (2 by
// default; the workspace is sized for that, the largest group count).
__host__ inline LoraSplit lora_split(int64_t m, int64_t k, const int* ranks, int nlin, int chunks = 2) {
  const int kc_total = static_cast<int>(k / kLoraKc);
  LoraSplit L;
  L.cluster = std::max(1, std::min(kPrepMaxCluster, kc_total));
  int g = (kc_total + 2 * L.cluster - 1) / (2 * L.cluster);
  if (lora_sum_in_prep(m)) {
    if (lora_tile_count(m, ranks, nlin) > kMaxLoraCounters) g = 1;
  } else {
    g = (kc_total + chunks * L.cluster - 1) / (chunks * L.cluster);
    const int64_t n_tok = std::min<int64_t>(256, (m + 15) / 16 * 16);
    g = std::min<int>(g, static_cast<int>(std::max<int64_t>(1, 256 / std::max<int64_t>(n_tok, 1))));
  }
  L.groups = std::max(1, std::min(16, g));
  return L;
}

// fp64 -> bf16, round to nearest even, one rounding: the value is first
// rounded to fp32 toward zero with the inexact bit kept in the last place
// (round to odd; fp32 carries 16 more bits than bf16, so the final rounding
// sees the exact tie/half-way situation), then rounded to bf16.
__device__ __forceinline__ __nv_bfloat16 f64_to_bf16_rn(double v) {
  float f = __double2float_rz(v);
  if (static_cast<double>(f) != v && isfinite(f)) f = __uint_as_float(__float_as_uint(f) | 1u);
  return __float2bfloat16_rn(f);
}

__device__ __forceinline__ float noisy(float xv, float zv) {
  // bf16_RN( x * (1 + z) ): one fp32 add, one fp32 multiply, one rounding.
  return __bfloat162float(__float2bfloat16_rn(__fmul_rn(xv, __fadd_rn(1.0f, zv))));
}

// Grid (cluster, row_groups + LoRA tiles), clusters of `cluster` CTAs along x.
//   Row tasks: x~ for one token row, staged as fp16 * 2^e_m.
//   LoRA tiles: t[16 rows][32 ranks] = x~ . A^T; the cluster's CTAs each sum
//   one K slice and the partial tiles are added over distributed shared
//   memory in a fixed order, so t is written once, deterministically.
// At most 64 registers (four CTAs' worth per SM): two of its warps fit beside
// four 96-register MMA warps in an SM sub-partition.
__global__ void __launch_bounds__(kPrepThreads, 4) prep_kernel(PrepParams p) {
  extern __shared__ __align__(16) uint8_t sm[];
  const int tid = threadIdx.x;
  // The MMA kernel may start its prologue (barriers, TMEM, weight loads) now;
  // it waits for this grid's results before it reads them.
  griddep_launch_dependents();
  if (static_cast<int>(blockIdx.y) < p.row_groups) {
    // ---- row task: x~ row -> smem (bf16), amax, then fp16 * 2^e
    const int m = blockIdx.y * p.cluster + blockIdx.x;
    if (m >= p.M) {
      if (m < p.tiled_rows)  // padding row of the token tile: zeros
        for (int v = tid; v < p.K / 8; v += kPrepThreads)
          *reinterpret_cast<uint4*>(reinterpret_cast<uint8_t*>(p.xs) + xs_tile_offset(m, 8 * v, p.tiled_rows)) =
              make_uint4(0u, 0u, 0u, 0u);
      return;
    }
    __nv_bfloat16* xt = reinterpret_cast<__nv_bfloat16*>(sm);
    const uint4* xrow = reinterpret_cast<const uint4*>(p.x + static_cast<int64_t>(m) * p.ldx);
    unsigned amax = 0;
    const int nv = p.K / 8;
    if (p.rmsnorm) {
      // x~ = (w + Z) * (h / sqrt(mean(h^2) + delta)), fp64, one rounding to
      // bf16 (the op order of the definition; the mean's summation order is
      // the only difference from a sequential sum: ~1e-16 relative).
      __shared__ double red_d[kPrepThreads / 32];
      double ss = 0.0;
      for (int v = tid; v < nv; v += kPrepThreads) {
        const uint4 raw = __ldg(xrow + v);
        reinterpret_cast<uint4*>(xt)[v] = raw;
        const __nv_bfloat16* e = reinterpret_cast<const __nv_bfloat16*>(&raw);
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const double hv = static_cast<double>(__bfloat162float(e[j]));
          ss = fma(hv, hv, ss);
        }
      }
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) ss += __shfl_xor_sync(0xFFFFFFFFu, ss, off);
      if ((tid & 31) == 0) red_d[tid >> 5] = ss;
      __syncthreads();
      double tot = 0.0;
#pragma unroll
      for (int i = 0; i < kPrepThreads / 32; ++i) tot += red_d[i];
      const double denom = sqrt(tot / static_cast<double>(p.K) + p.delta);
      const uint4* w4 = reinterpret_cast<const uint4*>(p.w_norm);
      const float4* Z4 = reinterpret_cast<const float4*>(p.Zn);
      __nv_bfloat16* orow = p.xt_out != nullptr ? p.xt_out + static_cast<int64_t>(m) * p.ldo : nullptr;
      for (int v = tid; v < nv; v += kPrepThreads) {
        uint4 raw = reinterpret_cast<const uint4*>(xt)[v];
        const uint4 wr = __ldg(w4 + v);
        float zz[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
        if (p.Zn != nullptr) {
          const float4 za = __ldg(Z4 + 2 * v), zb = __ldg(Z4 + 2 * v + 1);
          zz[0] = za.x; zz[1] = za.y; zz[2] = za.z; zz[3] = za.w;
          zz[4] = zb.x; zz[5] = zb.y; zz[6] = zb.z; zz[7] = zb.w;
        }
        __nv_bfloat16* e = reinterpret_cast<__nv_bfloat16*>(&raw);
        const __nv_bfloat16* we = reinterpret_cast<const __nv_bfloat16*>(&wr);
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const double wn = static_cast<double>(__bfloat162float(we[j])) + static_cast<double>(zz[j]);
          e[j] = f64_to_bf16_rn(wn * (static_cast<double>(__bfloat162float(e[j])) / denom));
          amax = max(amax, static_cast<unsigned>(__bfloat16_as_ushort(e[j]) & 0x7FFFu));
        }
        reinterpret_cast<uint4*>(xt)[v] = raw;
        if (orow != nullptr) reinterpret_cast<uint4*>(orow)[v] = raw;
      }
      if (p.xs == nullptr) return;  // the normalisation step alone
    } else {
    // kRowVec vectors per thread per round: their loads are all in flight
    // before the first is used.
    const float4* z4 = reinterpret_cast<const float4*>(p.z != nullptr ? p.z + m * p.ldz : nullptr);
    uint4* xo = p.xt_out != nullptr ? reinterpret_cast<uint4*>(p.xt_out + static_cast<int64_t>(m) * p.ldo) : nullptr;
    constexpr int kRowVec = 4;
    for (int v0 = tid; v0 < nv; v0 += kRowVec * kPrepThreads) {
      uint4 raw[kRowVec];
      float4 za[kRowVec], zb[kRowVec];
#pragma unroll
      for (int u = 0; u < kRowVec; ++u) {
        const int v = v0 + u * kPrepThreads;
        if (v < nv) {
          raw[u] = __ldg(xrow + v);
          if (p.z != nullptr) {
            za[u] = __ldg(z4 + 2 * v);
            zb[u] = __ldg(z4 + 2 * v + 1);
          }
        }
      }
#pragma unroll
      for (int u = 0; u < kRowVec; ++u) {
        const int v = v0 + u * kPrepThreads;
        if (v >= nv) break;
        __nv_bfloat16* e = reinterpret_cast<__nv_bfloat16*>(&raw[u]);
        if (p.z != nullptr) {
          const float zz[8] = {za[u].x, za[u].y, za[u].z, za[u].w, zb[u].x, zb[u].y, zb[u].z, zb[u].w};
#pragma unroll
          for (int j = 0; j < 8; ++j)
            e[j] = __float2bfloat16_rn(__fmul_rn(__bfloat162float(e[j]), __fadd_rn(1.0f, zz[j])));
        }
#pragma unroll
        for (int j = 0; j < 8; ++j) amax = max(amax, static_cast<unsigned>(__bfloat16_as_ushort(e[j]) & 0x7FFFu));
        reinterpret_cast<uint4*>(xt)[v] = raw[u];
        if (xo != nullptr) xo[v] = raw[u];
      }
    }
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
    uint8_t* dst_t = reinterpret_cast<uint8_t*>(p.xs);
    for (int v = tid; v < p.K / 8; v += kPrepThreads) {
      uint4 raw = reinterpret_cast<const uint4*>(xt)[v];
      const __nv_bfloat16* e8 = reinterpret_cast<const __nv_bfloat16*>(&raw);
      uint4 out;
      __half2* o = reinterpret_cast<__half2*>(&out);
#pragma unroll
      for (int j = 0; j < 4; ++j)
        o[j] = __floats2half2_rn(__bfloat162float(e8[2 * j]) * scale, __bfloat162float(e8[2 * j + 1]) * scale);
      if (p.tiled_rows > 0)
        *reinterpret_cast<uint4*>(dst_t + xs_tile_offset(m, 8 * v, p.tiled_rows)) = out;
      else
        dst[v] = out;
    }
    return;
  }
  // ---- LoRA tile: thread (rank = tid % 32, row pair = tid / 32): 2 accumulators.
  const int lt = blockIdx.y - p.row_groups;
  const int g = lt / p.lora_tiles;
  int tile = lt - g * p.lora_tiles;
  const int tile_lin = tile;  // this LoRA tile over all linears (its counter)
  int li = 0;
  while (tile >= p.tile_begin[li + 1]) ++li;
  tile -= p.tile_begin[li];
  const __nv_bfloat16* Am = p.A[li];
  const int rr_ = p.r[li];
  float* tout = p.t[li];
  const int mt = tile % p.lora_m_tiles;
  const int rt = tile / p.lora_m_tiles;
  const int ks = blockIdx.x;  // this CTA's rank in the cluster
  const int row0 = mt * kLoraTileM, rank0 = rt * kLoraTileR;
  // The slice's 64-wide chunks stream through a kLoraStages-deep cp.async
  // ring (raw bf16 x, A and fp32 z; rows past M and ranks past r zero-filled)
  // so that their loads overlap; each chunk is then converted once into the
  // fp32 tiles below (x~ with the noise applied, A) that the FMA loop reads.
  float* xsm = reinterpret_cast<float*>(sm + kLoraStages * kLoraStageBytes);  // [kLoraTileM][kLoraPad]
  float* asm_ = xsm + kLoraTileM * kLoraPad;                                   // [kLoraTileR][kLoraPad]
  const uint32_t ring = smem_u32(sm);
  constexpr int kRowsPerThread = kLoraTileM * kLoraTileR / kPrepThreads;
  static_assert(kRowsPerThread * (kPrepThreads / 32) == kLoraTileM, "LoRA tile map");
  const int lr = tid & 31, rq = tid >> 5;
  float acc[kRowsPerThread];
#pragma unroll
  for (int i = 0; i < kRowsPerThread; ++i) acc[i] = 0.0f;
  const int kc_total = p.K / kLoraKc;
  const int slices = p.cluster * p.groups;
  const int sl = g * p.cluster + ks;
  const int kc_begin = static_cast<int>(static_cast<int64_t>(sl) * kc_total / slices);
  const int kc_end = static_cast<int>(static_cast<int64_t>(sl + 1) * kc_total / slices);
  auto issue_chunk = [&](int kc, int st) {
    const uint32_t base = ring + st * kLoraStageBytes;
    const int k0 = kc * kLoraKc;
    constexpr int kXv = kLoraTileM * kLoraKc / 8, kAv = kLoraTileR * kLoraKc / 8;
    const int kZv = (p.ldz > 0 ? kLoraTileM : 1) * kLoraKc / 4;  // z rows staged
    for (int v = tid; v < kXv + kAv + kZv; v += kPrepThreads) {
      if (v < kXv) {
        const int rr = v >> 3, c = v & 7;
        const bool in = row0 + rr < p.M;
        cp_async_16(base + v * 16, in ? p.x + static_cast<int64_t>(row0 + rr) * p.ldx + k0 + c * 8 : p.x, in ? 16u : 0u);
      } else if (v < kXv + kAv) {
        const int jj = (v - kXv) >> 3, c = (v - kXv) & 7;
        const bool in = rank0 + jj < rr_;
        cp_async_16(base + v * 16, in ? Am + static_cast<int64_t>(rank0 + jj) * p.K + k0 + c * 8 : Am,
                    in ? 16u : 0u);
      } else {
        const int c = v - kXv - kAv;                          // 16 per z row
        const int zr = c >> 4, zc = c & 15;
        const bool in = p.z != nullptr && (p.ldz == 0 || row0 + zr < p.M);
        cp_async_16(base + v * 16, in ? p.z + (row0 + zr) * p.ldz + k0 + zc * 4 : reinterpret_cast<const float*>(p.x),
                    in ? 16u : 0u);
      }
    }
  };
  // Without a group sum, the cluster's partial tiles are pushed to their
  // owners -- CTA q owns entries [q * E, (q + 1) * E) of the 512, E =
  // ceil(512 / cluster) -- into a receive buffer [cluster][E], each 4-byte
  // store counted on the owner's mbarrier; the owner adds the partners in
  // rank order.  The barriers are initialised before any CTA of the cluster
  // pushes (one cluster barrier here, none at the end).
  constexpr int kTileEntries = kLoraTileM * kLoraTileR;
  const bool group_sum = p.sum_groups && p.groups > 1;
  const bool push = !group_sum && p.cluster > 1;
  const int E = (kTileEntries + p.cluster - 1) / p.cluster;
  const int own = max(0, min(E, kTileEntries - ks * E));  // entries this CTA owns
  const uint32_t recv = smem_u32(sm) + static_cast<uint32_t>(kLoraTileSmemBytes);
  const uint32_t recv_bar = recv + static_cast<uint32_t>(kLoraRecvBytes);
  if (push) {
    if (tid == 0) {
      mbar_init_a(recv_bar, 1);
      mbar_arrive_expect_tx_a(recv_bar, static_cast<uint32_t>(p.cluster * own * 4));
      fence_mbarrier_init();
    }
    cluster_sync_all();
  }
  for (int st = 0; st < kLoraStages; ++st) {
    if (kc_begin + st < kc_end) issue_chunk(kc_begin + st, st);
    cp_async_commit();  // one group per chunk slot, empty past the slice
  }
  for (int kc = kc_begin, st = 0; kc < kc_end; ++kc) {
    cp_async_wait_group<kLoraStages - 1>();  // this chunk's group has landed
    __syncthreads();                          // ... for every thread; the FMA loop above is done
    {
      const uint8_t* stg = sm + st * kLoraStageBytes;
      const __nv_bfloat16* xr = reinterpret_cast<const __nv_bfloat16*>(stg);
      const __nv_bfloat16* ar = xr + kLoraTileM * kLoraKc;
      const float* zr = reinterpret_cast<const float*>(ar + kLoraTileR * kLoraKc);
      for (int i = tid; i < kLoraTileM * kLoraKc / 4; i += kPrepThreads) {
        const int rr = i >> 4, k4 = (i & 15) * 4;  // 16 rows x 64 k, four per item
        float4 f;
        const float* zrow = zr + (p.ldz > 0 ? rr * kLoraKc : 0);
        f.x = noisy(__bfloat162float(xr[rr * kLoraKc + k4]), zrow[k4]);
        f.y = noisy(__bfloat162float(xr[rr * kLoraKc + k4 + 1]), zrow[k4 + 1]);
        f.z = noisy(__bfloat162float(xr[rr * kLoraKc + k4 + 2]), zrow[k4 + 2]);
        f.w = noisy(__bfloat162float(xr[rr * kLoraKc + k4 + 3]), zrow[k4 + 3]);
        *reinterpret_cast<float4*>(xsm + rr * kLoraPad + k4) = f;
      }
      for (int i = tid; i < kLoraTileR * kLoraKc / 8; i += kPrepThreads) {
        const int jj = i >> 3, k8 = (i & 7) * 8;  // 32 ranks x 64 k, eight per item
        const uint4 raw = *reinterpret_cast<const uint4*>(ar + jj * kLoraKc + k8);
        const __nv_bfloat16* e = reinterpret_cast<const __nv_bfloat16*>(&raw);
        float4* d = reinterpret_cast<float4*>(asm_ + jj * kLoraPad + k8);
        d[0] = make_float4(__bfloat162float(e[0]), __bfloat162float(e[1]), __bfloat162float(e[2]), __bfloat162float(e[3]));
        d[1] = make_float4(__bfloat162float(e[4]), __bfloat162float(e[5]), __bfloat162float(e[6]), __bfloat162float(e[7]));
      }
    }
    __syncthreads();  // fp32 tiles ready; the raw stage is free
    if (kc + kLoraStages < kc_end) issue_chunk(kc + kLoraStages, st);
    cp_async_commit();
    if (++st == kLoraStages) st = 0;
#pragma unroll 4
    for (int kk = 0; kk < kLoraKc; kk += 4) {
      const float4 av = *reinterpret_cast<const float4*>(asm_ + lr * kLoraPad + kk);
#pragma unroll
      for (int i = 0; i < kRowsPerThread; ++i) {
        const float4 xv = *reinterpret_cast<const float4*>(xsm + (kRowsPerThread * rq + i) * kLoraPad + kk);
        acc[i] = fmaf(xv.x, av.x, acc[i]);
        acc[i] = fmaf(xv.y, av.y, acc[i]);
        acc[i] = fmaf(xv.z, av.z, acc[i]);
        acc[i] = fmaf(xv.w, av.w, acc[i]);
      }
    }
  }
  cp_async_wait_group<0>();
  auto write_t = [&](int idx, float v) {
    const int row = row0 + idx / kLoraTileR, rank = rank0 + idx % kLoraTileR;
    if (row < p.M && rank < rr_) {
      if (p.sum_groups && p.groups == 1)
        p.tf[li][static_cast<int64_t>(row) * rr_ + rank] = v;  // one group: already the sum
      else
        tout[(static_cast<int64_t>(g) * p.M + row) * rr_ + rank] = v;
    }
  };
  if (!group_sum) {
    if (!push) {  // one CTA: its partial tile is the sum
#pragma unroll
      for (int i = 0; i < kRowsPerThread; ++i) write_t((kRowsPerThread * rq + i) * kLoraTileR + lr, acc[i]);
      return;
    }
#pragma unroll
    for (int i = 0; i < kRowsPerThread; ++i) {
      const int idx = (kRowsPerThread * rq + i) * kLoraTileR + lr;
      const int owner = idx / E;
      const uint32_t slot = static_cast<uint32_t>(ks * E + (idx - owner * E));
      st_async_f32(mapa_shared(recv + 4u * slot, static_cast<uint32_t>(owner)), acc[i],
                   mapa_shared(recv_bar, static_cast<uint32_t>(owner)));
    }
    if (own == 0) return;
    // Bounded wait for every partner's entries (parity 0: the first phase).
    const long long t0 = clock64();
    while (!mbar_try_wait_a(recv_bar, 0)) {
      if (clock64() - t0 > QERL_WAIT_LIMIT) {
        if (tid == 0) record_error(p.status, 5);
        return;
      }
    }
    if (tid < own) {
      float v = 0.0f;
      for (int q = 0; q < p.cluster; ++q) v += ldsf(recv + 4u * static_cast<uint32_t>(q * E + tid));
      write_t(ks * E + tid, v);
    }
    return;
  }
  // Group sum: partial tile [kLoraTileM][kLoraTileR] of this K slice -> shared
  // memory, then CTA q of the cluster sums entries q, q + cluster, ... over
  // all slices, and the last cluster of the tile adds the groups.
  __syncthreads();
  float* part = reinterpret_cast<float*>(sm);
#pragma unroll
  for (int i = 0; i < kRowsPerThread; ++i) part[(kRowsPerThread * rq + i) * kLoraTileR + lr] = acc[i];
  cluster_sync_all();
  const uint32_t part_s = smem_u32(part);
  // Every partner's value is loaded before the first add (the remote-load
  // latency is paid once, not once per partner), then added in rank order.
  // A thread sums at most two entries (512 per tile, 256 threads).
  constexpr int kPerThread = (kLoraTileM * kLoraTileR + kPrepThreads - 1) / kPrepThreads;
  // Entry u of this thread: idx0 + u * stride (fixed trip count, so the
  // sums stay in registers).
  const int idx0 = ks * kPrepThreads + tid, stride = p.cluster * kPrepThreads;
  float vsum[kPerThread];
#pragma unroll
  for (int u = 0; u < kPerThread; ++u) {
    const int idx = idx0 + u * stride;
    float v = 0.0f;
    if (idx < kLoraTileM * kLoraTileR) {
      float vq[kPrepMaxCluster];
#pragma unroll
      for (int q = 0; q < kPrepMaxCluster; ++q)
        vq[q] = q < p.cluster ? ld_shared_cluster_f32(mapa_shared(part_s + 4u * idx, q)) : 0.0f;
#pragma unroll
      for (int q = 0; q < kPrepMaxCluster; ++q)
        if (q < p.cluster) v += vq[q];
    }
    vsum[u] = v;
  }
#pragma unroll
  for (int u = 0; u < kPerThread; ++u) {
    const int idx = idx0 + u * stride;
    if (idx >= kLoraTileM * kLoraTileR) break;
    write_t(idx, vsum[u]);
  }
  // The group's writes are done before the arrival (release): the counter
  // below sees them.
  cluster_arrive();
  cluster_wait();  // partners are done reading this CTA's partial tile
  // The last cluster to finish this LoRA tile (one per K group) adds the
  // groups' partial sums in group order -- deterministic -- into tf, so the
  // MMA kernel reads one sum per element.  It resets the counter for the next
  // call.  (Release: the cluster barrier above orders the group's writes
  // before this CTA's fence and atomic; acquire: the fence after it.)
  if (ks != 0) return;
  __shared__ unsigned last;
  if (tid == 0) {
    __threadfence();
    const unsigned done = atomicAdd(p.tile_count + tile_lin, 1u);
    last = done == static_cast<unsigned>(p.groups - 1) ? 1u : 0u;
    if (last) {
      __threadfence();
      p.tile_count[tile_lin] = 0u;
    }
  }
  __syncthreads();
  if (!last) return;
  float* tfin = p.tf[li];
  for (int idx = tid; idx < kLoraTileM * kLoraTileR; idx += kPrepThreads) {
    const int row = row0 + idx / kLoraTileR, rank = rank0 + idx % kLoraTileR;
    if (row >= p.M || rank >= rr_) continue;
    float v = 0.0f;
    for (int gg = 0; gg < p.groups; ++gg) v += __ldcg(tout + (static_cast<int64_t>(gg) * p.M + row) * rr_ + rank);
    tfin[static_cast<int64_t>(row) * rr_ + rank] = v;
  }
}

// ------------------------------------------------------------------ MMA kernel

// Warp roles.  The issue scheduler favours older (lower-numbered) warps, so
// the light, latency-critical roles come first and the eight ALU-bound
// dequant warps last: otherwise the MMA issuers starve behind them.  Each
// group of four consecutive dequant warps covers the four tensor-memory lane
// quadrants (warp % 4).
constexpr int kMmaThreads = 608;  // 19 warps (15 when coupled: four issuer warps)
constexpr int kWeightWarp = 0, kActWarp = 1, kLoraWarp = 2;
constexpr int kIssuerWarp0 = 3, kMaxIssuers = 8;
constexpr int kDeqWarp0 = kIssuerWarp0 + kMaxIssuers;  // dequant + epilogue: warps 11..18
static_assert(kDeqWarp0 + 8 == kMmaThreads / 32, "warp roles");
// Coupled launches (up to 64 tokens) run 15 warps: issuers 3..6, dequant
// 7..14.  With 96 registers a thread, four warps per SM sub-partition leave
// room for two warps of a 256-thread, 64-register prep CTA beside them (a
// sub-partition holds 16384 registers), so the prep grid does not keep MMA
// CTAs off its SMs.
constexpr int kCoupledWarps = 15;
constexpr int kTileN = 128;       // output features per CTA (MMA M)
constexpr int kStageK = 64;       // K per MMA stage (4 x K=16 instructions)
constexpr int kRawK = 256;        // K per weight-load stage: 128 contiguous bytes of codes per row
constexpr int kSub = kRawK / kStageK;                  // MMA stages per weight stage
constexpr int kCodesRawBytes = kTileN * kRawK / 2;     // 16384
constexpr int kRawSlotBytes = kCodesRawBytes + kTileN * kRawK / 16;  // + 2048 scale bytes: one packed block
constexpr int kAStageCols = kStageK / 2;               // 32 TMEM columns (fp16 pairs, tensor-memory A operand)
constexpr int kLoraChunkK = 64;                        // r is processed in 64-wide chunks (one 128-B swizzle atom)
constexpr int kBtChunkBytes = kTileN * 128;            // B^T chunk: 128 rows x 64 bf16
constexpr int kMaxRaw = 8, kMaxAB = 8, kMaxB = 16;
constexpr int kMaxSplit = 8;  // CTAs of a K-split cluster (portable cluster size)
// Weight blocks prefetched into L2 ahead of the ring: the ring's copies are
// held for a stage's whole dequant + MMA time, so the ring alone cannot cover
// HBM latency at full rate; the ring refills from L2.
constexpr int kPrefetchStages = 4;  // (8 and 12 measured 0.8% and 1.2% slower per decode layer)
// Pair mode uses two issuer warps; the other six build the LoRA operand's t
// tiles while the weights stream.
constexpr int kPairLoraWarps = kMaxIssuers - 2;
constexpr int kSmemLimit = 232448;  // 227 KB opt-in per CTA
constexpr int kBarBytes = 1024;
constexpr int kTmemCols = 512;

// One linear of a launch: several linears sharing x (and K) run in one grid,
// their 128-row tiles concatenated along gridDim.y.
struct LinearSlot {
  const uint8_t* wpacked;     // packed weight blocks (see qerl_nvfp4_pack)
  const float* tensor_scale;  // S
  const float* t;             // LoRA partial sums [t_groups][M][r]
  void* y;                    // [M][N]
  int N, r, y_f32;
  int tile_begin;             // first tile index (gridDim.y) of this linear
  float lora_scale;           // alpha / r
  int nf4;                    // NF4 element codes: dequantized through the level table
};

struct MmaParams {
  const __half* xs;        // staged x~ (fp16 * 2^e_m): tiled up to 128 tokens, else [M][K]
  const float* rinv;
  LinearSlot lin[kMaxLinears];
  int nlin;
  int* status;
  int M, K;
  int n_tok;       // tokens per tile (MMA N), multiple of 16, <= 256
  int split;       // K split across the cluster (gridDim.x), in weight stages
  int raw_stages;  // weight-stage ring depth
  int ab_stages;   // tensor-memory A ring depth, in MMA stages
  int b_stages;    // !coupled: activation ring depth in 64-wide slabs (one barrier pair each; a multiple of kSub)
  int coupled;     // a weight stage's activation slabs sit in the slot of its A stage (same index and empty barrier)
  int issuers;     // MMA-issuing threads, each with its own accumulator
  int t_groups;    // t holds this many partial sums [t_groups][M][r], added in order
  uint32_t off_raw, off_b, off_lora, off_tstage, off_sm, off_bars;
  uint32_t raw_b_bytes;  // coupled: activation slot bytes per weight stage (kSub slabs)
  uint32_t col_a;  // TMEM column of the A stages (accumulators: issuer i at i * n_tok)
  int lora_early;  // LoRA operand tiles built at kernel start (dedicated region) or after the mainloop (in the ring)
  int wave;        // CTAs per wave (one per SM) when split == 1, else 0
  int n_warps;     // 19, or kCoupledWarps (dequant warps: the last eight)
  // 1: the staged x~ and row scales come from a kernel that finished before
  // the preceding one (the tensor-core LoRA down-projection) started, so they
  // are read without waiting for that kernel; only t waits for it.
  int acts_ready;
  int w_evict_first;  // one token tile: each weight block is read once, so it leaves L2 first
  int stage_out;   // the widest output tile (fp32) fits in the idle ring: staged stores
  // More than 64 tokens: a CTA takes a pair of adjacent 128-row tiles
  // of one linear (grid y counts pairs), so every activation slab it receives
  // serves 256 weight rows.  Dequant group g and issuer g own tile g; the
  // tensor-memory A slots are handed over per MMA stage (one per tile and
  // stage of the weight stage), the LoRA operands are built in the idle ring.
  int pair;
  int xs_rowmajor;  // x~ staged as [M][K] (more than 128 tokens: several token tiles), read by 2-D TMA
  int wt;           // the weights are in the transposed packed layout (input gradient of the linear)
  // NF4 (a linear with nf4 set): the 16 levels as fp16 bits; the dequant
  // warps expand them into a 256-entry table of fp16 pairs (one per code
  // byte) at off_lut.
  unsigned short nf4_half[16];
  uint32_t off_lut;
};

// The LoRA up-projection's B matrices, one TMA map per linear of the launch.
struct BtMaps {
  CUtensorMap m[kMaxLinears];
};

__host__ __device__ inline int lora_chunks(int r) { return (r + kLoraChunkK - 1) / kLoraChunkK; }
// LoRA operand region: `nbt` sets of B^T chunks (one per weight tile of the
// CTA), then the t_hi and t_lo chunks shared by them.
__host__ __device__ inline uint32_t lora_bytes(int r, int n_tok, int nbt = 1) {
  return r > 0 ? static_cast<uint32_t>(lora_chunks(r)) * (nbt * kBtChunkBytes + 2u * n_tok * 128u) : 0u;
}

__device__ __forceinline__ void store_out(const LinearSlot& L, int m, int n, float v) {
  const int64_t idx = static_cast<int64_t>(m) * L.N + n;
  if (L.y_f32)
    reinterpret_cast<float*>(L.y)[idx] = v;
  else
    reinterpret_cast<__nv_bfloat16*>(L.y)[idx] = __float2bfloat16_rn(v);
}

// (a, b) -> bf16 pairs hi = (trunc(a), trunc(b)) and lo = (trunc(a - hi_a),
// trunc(b - hi_b)), element a in the low half.  hi + lo carries each value to
// ~15 significant bits (relative error < 2^-14); a - hi is exact in fp32.
// Integer ops only: the conversion pipe is kept busy by the dequant warps.
__device__ __forceinline__ void split_bf16x2(float a, float b, uint32_t& hi, uint32_t& lo) {
  const uint32_t ua = __float_as_uint(a), ub = __float_as_uint(b);
  const float ra = a - __uint_as_float(ua & 0xFFFF0000u), rb = b - __uint_as_float(ub & 0xFFFF0000u);
  hi = __byte_perm(ua, ub, 0x7632);
  lo = __byte_perm(__float_as_uint(ra), __float_as_uint(rb), 0x7632);
}

// LoRA up-projection operands, in the 128-byte-swizzled K-major layout (the
// rank index j is the MMA's K):
//   B^T chunk c:  128 rows n  x 64 j   bf16  = B[n0 + n][c*64 + j]   (TMA from B [N][r])
//   t_hi chunk c: n_tok rows m x 64 j  bf16  = t[m0 + m][c*64 + j] truncated
//   t_lo chunk c: n_tok rows m x 64 j  bf16  = (t - t_hi) truncated
// so B^T . t_hi + B^T . t_lo carries t to ~15 significant bits.  The t tiles
// are built by `nthr` threads (tid < nthr); zero past M and r.
// The up-projection accumulates into the main accumulator, which the epilogue
// scales by S * 2^-e_m per token row m; so row m of t enters pre-scaled by
// (alpha / r) / (S * 2^-e_m) (fp32, before the hi/lo split: a relative change
// of a few fp32 ulps).  S must be positive and finite; otherwise the row
// factor is 0 and the call records QERL_ERR_NONFINITE.
// Row factors for tokens m0 .. m0 + n_tok - 1 into shared memory `fac`
// (n_tok floats), computed by `nthr` threads with their loads issued together.
__device__ __forceinline__ void fill_lora_factors(const MmaParams& p, const LinearSlot& L, uint32_t fac, int m0,
                                                  int tid, int nthr) {
  float rv[4];
#pragma unroll
  for (int u = 0; u < 4; ++u) {
    const int i = tid + u * nthr;
    rv[u] = (i < p.n_tok && m0 + i < p.M) ? __ldg(p.rinv + m0 + i) : 0.0f;
  }
  const float S = *L.tensor_scale;
#pragma unroll
  for (int u = 0; u < 4; ++u) {
    const int i = tid + u * nthr;
    if (i >= p.n_tok) break;
    float f = 0.0f;
    if (m0 + i < p.M) {
      const float sr = S * rv[u];
      if (!(sr > 0.0f) || sr > 3.0e38f)
        record_error(p.status, 6);
      else
        f = L.lora_scale / sr;
    }
    stsf(fac + 4u * i, f);
  }
}
__device__ void build_t_tiles(const MmaParams& p, const LinearSlot& L, uint32_t base, uint32_t fac, int m0, int tid,
                              int nthr, int nbt = 1) {
  const int rc = lora_chunks(L.r);
  const uint32_t thi = base + nbt * rc * kBtChunkBytes;
  const uint32_t tlo = thi + rc * p.n_tok * 128;
  for (int idx = tid; idx < rc * p.n_tok * 8; idx += nthr) {
    const int c = idx / (p.n_tok * 8), rem = idx - c * (p.n_tok * 8);
    const int ml = rem >> 3, g = rem & 7;
    const int m = m0 + ml;
    const float f = ldsf(fac + 4u * ml);
    float tv[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      const int j = c * kLoraChunkK + g * 8 + e;
      float v = 0.0f;
      if (m < p.M && j < L.r)
        for (int g = 0; g < p.t_groups; ++g) v += __ldg(L.t + (static_cast<int64_t>(g) * p.M + m) * L.r + j);
      tv[e] = v * f;
    }
    uint32_t hw[4], lw[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) split_bf16x2(tv[2 * e], tv[2 * e + 1], hw[e], lw[e]);
    const uint32_t off = c * p.n_tok * 128 + ml * 128 + ((g ^ (ml & 7)) << 4);
    sts128(thi + off, make_uint4(hw[0], hw[1], hw[2], hw[3]));
    sts128(tlo + off, make_uint4(lw[0], lw[1], lw[2], lw[3]));
  }
}

// Same tiles from the partial sums staged in shared memory by bulk copies:
// tstage[g][ml][j] = t_part[g][m0 + ml][j] for ml < rows.
__device__ void build_t_tiles_staged(const MmaParams& p, const LinearSlot& L, uint32_t base, uint32_t tstage,
                                     uint32_t fac, int rows, int tid, int nthr) {
  const int rc = lora_chunks(L.r);
  const uint32_t thi = base + rc * kBtChunkBytes;
  const uint32_t tlo = thi + rc * p.n_tok * 128;
  const uint32_t gstride = static_cast<uint32_t>(p.n_tok * L.r * 4);
  for (int idx = tid; idx < rc * p.n_tok * 8; idx += nthr) {
    const int c = idx / (p.n_tok * 8), rem = idx - c * (p.n_tok * 8);
    const int ml = rem >> 3, g8 = rem & 7;
    const int j0 = c * kLoraChunkK + g8 * 8;
    float tv[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) tv[e] = 0.0f;
    if (ml < rows && j0 < L.r) {  // r is a multiple of 8: all eight ranks valid
      const uint32_t src = tstage + static_cast<uint32_t>((ml * L.r + j0) * 4);
      for (int g = 0; g < p.t_groups; ++g) {
        const float4 a = lds128f(src + g * gstride), b = lds128f(src + g * gstride + 16);
        tv[0] += a.x;
        tv[1] += a.y;
        tv[2] += a.z;
        tv[3] += a.w;
        tv[4] += b.x;
        tv[5] += b.y;
        tv[6] += b.z;
        tv[7] += b.w;
      }
      const float f = ldsf(fac + 4u * ml);
#pragma unroll
      for (int e = 0; e < 8; ++e) tv[e] *= f;
    }
    uint32_t hw[4], lw[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) split_bf16x2(tv[2 * e], tv[2 * e + 1], hw[e], lw[e]);
    const uint32_t off = c * p.n_tok * 128 + ml * 128 + ((g8 ^ (ml & 7)) << 4);
    sts128(thi + off, make_uint4(hw[0], hw[1], hw[2], hw[3]));
    sts128(tlo + off, make_uint4(lw[0], lw[1], lw[2], lw[3]));
  }
}

// TMA of the B^T chunks (rows n0..n0+127 of B [N][r], 64 ranks per chunk,
// zero-filled past N and r) into `base`, completing on `bar`; for `ntl` tiles
// (rows n0 + 128 i, chunk set i at base + i * rc * kBtChunkBytes), one arrival.
__device__ __forceinline__ void load_bt_tiles(const LinearSlot& L, const CUtensorMap* tm_bl, uint32_t base, int n0,
                                              uint32_t bar, int ntl = 1) {
  const int rc = lora_chunks(L.r);
  mbar_arrive_expect_tx_a(bar, static_cast<uint32_t>(rc * ntl) * kBtChunkBytes);
  for (int i = 0; i < ntl; ++i)
    for (int c = 0; c < rc; ++c)
      tma_load_2d(base + (i * rc + c) * kBtChunkBytes, tm_bl, c * kLoraChunkK, n0 + i * kTileN, bar);
}

// Warp-cooperative bounded wait.  Every lane polls: one convergent try_wait
// by the whole warp costs less than a single lane's poll inside a divergent
// branch, and each lane then holds its own acquire.  The vote keeps the warp's
// answer uniform when a bounded wait gives up.
__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, volatile int* abort_flag, int* status) {
  bool ok = mbar_probe_a(bar, parity);
  if (__all_sync(0xFFFFFFFFu, ok)) return true;
  if (!ok) ok = mbar_wait_a(bar, parity, abort_flag, status);
  return __all_sync(0xFFFFFFFFu, ok);
}

// D += B^T . t_hi^T + B^T . t_lo^T over the rank dimension (bf16 x bf16 ->
// fp32), into an accumulator that already holds this thread's main-loop sum.
// `bt` is this tile's B^T chunk set, `thi` the t_hi chunks (t_lo follows).
__device__ __forceinline__ void issue_lora_mmas(const MmaParams& p, const LinearSlot& L, uint32_t bt, uint32_t thi,
                                                uint32_t d2) {
  const int rc = lora_chunks(L.r);
  const uint32_t idesc = idesc_bf16_f32(kTileN, static_cast<uint32_t>(p.n_tok));
  const uint32_t tlo = thi + rc * p.n_tok * 128;
  for (int c = 0; c < rc; ++c)
    for (int kk = 0; kk < kLoraChunkK / 16 && c * kLoraChunkK + kk * 16 < L.r; ++kk) {
      const uint64_t ad = sw128_kmajor_desc(bt + c * kBtChunkBytes + kk * 32);
      tc_mma_f16(d2, ad, sw128_kmajor_desc(thi + c * p.n_tok * 128 + kk * 32), idesc, 1u);
      tc_mma_f16(d2, ad, sw128_kmajor_desc(tlo + c * p.n_tok * 128 + kk * 32), idesc, 1u);
    }
}

// The dequantized weight operand goes to tensor memory (tcgen05.st), each MMA
// reads it from there, and `issuers` threads issue MMAs for disjoint K steps
// into their own accumulators (an MMA occupies its issuing thread for
// far longer than the tensor pipe needs for a 128 x n_tok x 16 product, so
// one issuer cannot keep the pipe busy at decode token counts).
// One MMA stage (64 K) of weight row `row` of a staged packed block at
// `slot` -> 32 fp16 pairs o[] (element pairs along K), exact: an E2M1 value
// times an E4M3 scale fits fp16.  Forward layout: one scale per 16 K, as
// pairs at kCodesRawBytes + p * 256 + 2 * row.  Transposed layout (wt; the
// weight's transpose for the input gradient, K being the original output
// dimension): a scale per element along K, shared by the 16 rows of a row
// group, at kCodesRawBytes + (row / 16) * 256 + k.
// Element pairs of 8 codes (a 32-bit word): E2M1 by conversion, or (kLut)
// NF4 by the byte-indexed table of fp16 pairs at `lut`.
template <bool kLut>
__device__ __forceinline__ void codes8_to_f16x2x4(uint32_t w, uint32_t lut, uint32_t (&u)[4]) {
  if constexpr (!kLut) {
    e2m1x8_to_f16x2x4(w, u);
  } else {
#pragma unroll
    for (int b = 0; b < 4; ++b) u[b] = lds32(lut + 4u * ((w >> (8 * b)) & 0xFFu));
  }
}

template <bool kLut, bool kWt>
__device__ __forceinline__ void dequant_mma_stage(uint32_t slot, int row, int q, uint32_t lut,
                                                  uint32_t (&o)[32]) {
  const uint32_t crow = slot + row * 128;
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const uint4 cw = lds128(crow + (((2 * q + h) ^ (row & 7)) << 4));
    const uint32_t words[4] = {cw.x, cw.y, cw.z, cw.w};
    if constexpr (!kWt) {
      const __half2 s01 = e4m3x2_to_half2(lds16(slot + kCodesRawBytes + row * 2 + (2 * q + h) * 256));
      const __half2 sa2 = __low2half2(s01), sb2 = __high2half2(s01);
      const uint32_t sa = *reinterpret_cast<const uint32_t*>(&sa2);
      const uint32_t sb = *reinterpret_cast<const uint32_t*>(&sb2);
#pragma unroll
      for (int qq = 0; qq < 4; ++qq) {
        uint32_t u[4];
        codes8_to_f16x2x4<kLut>(words[qq], lut, u);
#pragma unroll
        for (int b = 0; b < 4; ++b) o[16 * h + 4 * qq + b] = hmul2_bits(u[b], qq < 2 ? sa : sb);
      }
    } else {
      const uint32_t sbase = slot + kCodesRawBytes + (row >> 4) * 256 + (2 * q + h) * 32;
      const uint4 s0 = lds128(sbase), s1 = lds128(sbase + 16);
      const uint32_t sw[8] = {s0.x, s0.y, s0.z, s0.w, s1.x, s1.y, s1.z, s1.w};
#pragma unroll
      for (int qq = 0; qq < 4; ++qq) {
        uint32_t u[4];
        codes8_to_f16x2x4<kLut>(words[qq], lut, u);
#pragma unroll
        for (int b = 0; b < 4; ++b) {
          const __half2 sc = e4m3x2_to_half2((sw[2 * qq + (b >> 1)] >> (16 * (b & 1))) & 0xFFFFu);
          o[16 * h + 4 * qq + b] = hmul2_bits(u[b], *reinterpret_cast<const uint32_t*>(&sc));
        }
      }
    }
  }
}

// kCoupledT: the coupled layout (up to 64 tokens, single tiles, 15 warps) or
// the general one (pair mode and the rest); kWtT: the transposed weight
// layout (the input gradient).  Each instantiation carries only its own
// paths, so the code a CTA runs once is more compact.
template <int kCoupledT, int kWtT>
__global__ void __launch_bounds__(kMmaThreads, 1)
    mma_kernel(const __grid_constant__ CUtensorMap tm_xs, const __grid_constant__ BtMaps tm_bls,
               const MmaParams p) {
  constexpr bool kCpl = kCoupledT != 0;
  constexpr bool kWt = kWtT != 0;
  const bool pairm = !kCpl && p.pair != 0;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  const uint32_t raw_addr = smem_u32(smem_raw);
  const uint32_t sbase = (raw_addr + 1023u) & ~1023u;
  uint8_t* smem_gen = smem_raw + (sbase - raw_addr);  // generic view (abort flag, TMEM holder)
  const uint32_t bars = sbase + p.off_bars;
  auto raw_full = [&](int s) { return bars + 8u * s; };
  auto raw_empty = [&](int s) { return bars + 8u * (kMaxRaw + s); };
  auto ab_full = [&](int s) { return bars + 8u * (2 * kMaxRaw + s); };
  auto ab_empty = [&](int s) { return bars + 8u * (2 * kMaxRaw + kMaxAB + s); };
  constexpr int kB2 = 2 * kMaxRaw + 2 * kMaxAB;
  const uint32_t ring_free = bars + 8u * kB2;
  const uint32_t lora_full = bars + 8u * (kB2 + 1);
  const uint32_t acc_full = bars + 8u * (kB2 + 2);
  const uint32_t tmem_holder = bars + 8u * (kB2 + 3);
  const uint32_t t_full = bars + 8u * (kB2 + 4);
  // The activation ring has its own depth and barriers.
  auto b_full = [&](int s) { return bars + 8u * (kB2 + 8 + s); };
  auto b_empty = [&](int s) { return bars + 8u * (kB2 + 8 + kMaxB + s); };

  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem_gen + p.off_bars + 8 * (kB2 + 3) + 4);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int deq0 = p.n_warps - 8;  // first dequant warp
  const int split_idx = blockIdx.x;
  // This CTA's linear: the one whose tile range holds blockIdx.y.
  int gi = 0;
  while (gi + 1 < p.nlin && static_cast<int>(blockIdx.y) >= p.lin[gi + 1].tile_begin) ++gi;
  const LinearSlot& L = p.lin[gi];
  const CUtensorMap* tm_bl = &tm_bls.m[gi];
  const int n0 = (static_cast<int>(blockIdx.y) - L.tile_begin) * kTileN * (pairm ? 2 : 1);
  // Weight tiles this CTA streams: 1, or 2 in pair mode (1 for an odd last tile).
  const int ntl = pairm ? min(2, (L.N - n0 + kTileN - 1) / kTileN) : 1;
  const uint32_t rslot = static_cast<uint32_t>(pairm ? 2 : 1) * kRawSlotBytes;  // raw-ring slot size
  const int m0 = blockIdx.z * p.n_tok;
  const int raw_total = (p.K + kRawK - 1) / kRawK;
  const int rb = static_cast<int>(static_cast<int64_t>(split_idx) * raw_total / p.split);
  const int re = static_cast<int>(static_cast<int64_t>(split_idx + 1) * raw_total / p.split);
  const int nraw = re - rb;
  const int kb_total = p.K / kStageK;
  const int mma_begin = kSub * rb;
  const int nmma = min(kSub * re, kb_total) - mma_begin;
  const int RS = p.raw_stages, AS = p.ab_stages, NI = p.issuers, BS = p.b_stages;
  const bool do_lora = L.r > 0 && split_idx == 0;  // one CTA of a K-split cluster adds the LoRA term
  const int n_iss = pairm ? ntl : NI;              // issuers with work (each commits once to the barriers below)

  if (threadIdx.x == 0) {
    for (int s = 0; s < RS; ++s) {
      mbar_init_a(raw_full(s), 1);  // producer expect_tx
      // The four dequant warps of the stage's group; pair mode: the groups
      // of both tiles.
      mbar_init_a(raw_empty(s), pairm ? 4 * ntl : 4);
    }
    if (pairm) {
      // One barrier pair per (tile, MMA stage) slot of tensor memory: the
      // tile's four dequant warps arrive, its issuer commits.
      for (int w = 0; w < 2 * kSub; ++w) {
        mbar_init_a(ab_full(w), 4);
        mbar_init_a(ab_empty(w), 1);
      }
    } else {
      // A ring of 2 x (tensor-memory A slots) barrier pairs: weight stage i
      // uses pair i mod 2AW and A slot i mod AW, so every pair serves stages
      // of one parity -- one dequant group and, coupled, one issuer group --
      // and each waiter visits its pairs' phases in order.  Full: the four
      // warps of the dequant group that wrote the stage (+ coupled, the
      // activation producer's expect_tx for the stage's slabs); empty: every
      // issuer of the stage once.
      for (int b = 0; b < 2 * (AS / kSub); ++b) {
        mbar_init_a(ab_full(b), 4 + (kCpl ? 1 : 0));
        mbar_init_a(ab_empty(b), kCpl ? NI / 2 : NI);
      }
    }
    for (int s = 0; s < BS; ++s) {
        mbar_init_a(b_full(s), 1);                  // producer expect_tx
        mbar_init_a(b_empty(s), pairm ? ntl : 1);  // tcgen05.commit of each issuer reading the slab
      }
    mbar_init_a(ring_free, n_iss);
    // B^T TMA (expect_tx) + the warps that build the t tiles: the eight
    // dequant warps, or in pair mode the six issuer warps without a tile.
    mbar_init_a(lora_full, pairm ? 1 + kPairLoraWarps : 9);
#ifdef QERL_TEST_HOOKS
    mbar_init_a(acc_full, n_iss + (g_test_extra_arrival ? 1 : 0));
#else
    mbar_init_a(acc_full, n_iss);
#endif
    mbar_init_a(t_full, 1);
    *abort_flag = 0;
    fence_mbarrier_init();
  }
  if (warp == kIssuerWarp0) {
    tmem_alloc(tmem_holder, kTmemCols);
    tmem_relinquish();
  }
  if (warp == kWeightWarp && lane == 0) {
    if (p.xs_rowmajor) tma_prefetch_desc(&tm_xs);
    if (L.r > 0) tma_prefetch_desc(tm_bl);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *reinterpret_cast<volatile uint32_t*>(smem_gen + p.off_bars + 8 * (kB2 + 3));
  const uint32_t lora_base = p.lora_early ? sbase + p.off_lora : sbase;  // late: inside the idle ring
  const uint32_t smv = sbase + p.off_sm;

  if (warp == kWeightWarp) {
    // ------------------------------------------------------------ weight producer
    // One bulk copy per weight stage: the packed block (codes in their
    // swizzled image, then the scale pairs) is contiguous in memory.
    const uint8_t* wtile = L.wpacked + static_cast<int64_t>(n0 / kTileN) * raw_total * kRawSlotBytes;
    const int64_t tile_stride = static_cast<int64_t>(raw_total) * kRawSlotBytes;  // next tile's blocks (pair mode)
    // The copies into the ring are held for a stage's whole dequant time,
    // so the ring alone cannot cover HBM latency at full rate: the
    // blocks kPrefetch stages ahead are prefetched into L2 (bounded by L2
    // capacity, not shared memory) and the ring refills from L2.
    constexpr int kPrefetch = kPrefetchStages;
    // The first ring of weight blocks (and L2 prefetches further
    // ahead) is requested at once: the weights were written before the
    // preceding kernel of this call started, so the dequant of those stages
    // runs while that kernel is still at work.
    const int early = min(RS, nraw);
    // Coupled, the prep grid runs beside this one and its loads (x, z, the
    // LoRA A) gate the first MMAs: the L2 prefetches beyond the ring wait
    // until it has finished, so they do not queue ahead of its loads.
    auto prefetch_first = [&](int from) {
      for (int i = from; i < min(kPrefetch, nraw); ++i)
        for (int t = 0; t < ntl; ++t)
          bulk_prefetch_l2(wtile + t * tile_stride + static_cast<int64_t>(rb + i) * kRawSlotBytes, kRawSlotBytes);
    };
    // One token tile reads each weight block once: after its copy into the
    // ring it is marked first to leave L2, so the stream does not evict the
    // activations, the outputs and this kernel's code.
    const uint64_t wpol = p.w_evict_first ? l2_policy_evict_first() : 0ull;
    auto load_w = [&](uint32_t dst, const uint8_t* src, uint32_t bar) {
      if (p.w_evict_first)
        bulk_load_hint(dst, src, kRawSlotBytes, bar, wpol);
      else
        bulk_load(dst, src, kRawSlotBytes, bar);
    };
    if (lane == 0) {
      if (!kCpl) prefetch_first(0);
      for (int i = 0; i < early; ++i) {
        mbar_arrive_expect_tx_a(raw_full(i), ntl * kRawSlotBytes);
        for (int t = 0; t < ntl; ++t)
          load_w(sbase + p.off_raw + i * rslot + t * kRawSlotBytes,
                 wtile + t * tile_stride + static_cast<int64_t>(rb + i) * kRawSlotBytes, raw_full(i));
      }
    }
    if (kCpl) {
      griddep_wait();
      if (lane == 0) prefetch_first(early);  // the ring's blocks are being loaded
    }
    if (lane == 0) {
      uint32_t ph = 0;
      for (int i = 0, s = 0; i < nraw; ++i) {
        if (i + kPrefetch < nraw)
          for (int t = 0; t < ntl; ++t)
            bulk_prefetch_l2(wtile + t * tile_stride + static_cast<int64_t>(rb + i + kPrefetch) * kRawSlotBytes,
                             kRawSlotBytes);
        const int rst = rb + i;
        if (i >= early) {
          if (!mbar_wait_a(raw_empty(s), ph ^ 1, abort_flag, p.status)) break;
          mbar_arrive_expect_tx_a(raw_full(s), ntl * kRawSlotBytes);
          for (int t = 0; t < ntl; ++t)
            load_w(sbase + p.off_raw + s * rslot + t * kRawSlotBytes,
                   wtile + t * tile_stride + static_cast<int64_t>(rst) * kRawSlotBytes, raw_full(s));
        }
        if (++s == RS) {
          s = 0;
          ph ^= 1;
        }
      }
      // The tile the next wave runs (one CTA per SM: `wave` CTAs later) gets
      // its first blocks prefetched into L2 now, so that CTA does not start
      // on a cold stream.
      if (p.split == 1 && p.wave > 0) {
        const int ty = static_cast<int>(blockIdx.y) + p.wave;
        int gj = 0;
        while (gj + 1 < p.nlin && ty >= p.lin[gj + 1].tile_begin) ++gj;
        if (ty < p.lin[p.nlin - 1].tile_begin + (p.lin[p.nlin - 1].N + kTileN - 1) / kTileN) {
          const uint8_t* nt = p.lin[gj].wpacked + static_cast<int64_t>(ty - p.lin[gj].tile_begin) * raw_total *
                                                      kRawSlotBytes;
          for (int i = 0; i < min(kPrefetch, raw_total); ++i)
            bulk_prefetch_l2(nt + static_cast<int64_t>(i) * kRawSlotBytes, kRawSlotBytes);
        }
      }
    }
  } else if (warp == kActWarp) {
    // ------------------------------------------------------------ activation producer
    if (!p.acts_ready) griddep_wait();  // the staged activations are written by the preceding kernel
    {
      if (kCpl && lane == 0) {
        // Up to 64 tokens: one bulk copy of a weight stage's kSub slabs (the
        // tiled layout keeps them contiguous) into the activation slot of its
        // tensor-memory A slot, completing on the stage's full barrier.  The
        // stage AW earlier (same slots) must have finished its MMAs: its
        // empty barrier releases A and the slabs together, so a weight slot
        // is refilled as soon as it is dequantized, whatever the MMAs still
        // read.  (That stage's completion also orders the previous phase of
        // this full barrier before the arrival below.)  For the first AW
        // stages the wait is on a fresh barrier's parity 1 and passes.
        const int AW = AS / kSub, BW = 2 * AW;
        const int kslabs = p.K / kStageK;
        int w = 0, b = 0, e = AW;  // A slot, barrier pair of stage i; barrier pair of stage i - AW
        uint32_t eph = 1;          // phase parity of stage i - AW on its pair (use -1 at first)
        for (int i = 0; i < nraw; ++i) {
          if (!mbar_wait_a(ab_empty(e), eph, abort_flag, p.status)) break;
          const int rst = rb + i;
          const uint32_t xbytes = static_cast<uint32_t>(min(kSub, kslabs - rst * kSub) * p.n_tok * 128);
          mbar_arrive_expect_tx_a(ab_full(b), xbytes);
          bulk_load(sbase + p.off_b + w * p.raw_b_bytes,
                    reinterpret_cast<const uint8_t*>(p.xs) + static_cast<int64_t>(rst) * p.raw_b_bytes, xbytes,
                    ab_full(b));
          if (++w == AW) w = 0;
          if (++b == BW) b = 0;
          if (++e == BW) {
            e = 0;
            eph ^= 1;
          }
        }
      } else if (pairm && lane == 0) {
        // Pair mode: the ring's BS slabs form two halves of G = BS / 2 slabs
        // (a weight stage's kSub slabs, or half of them), each half one
        // barrier pair filled at once, so each issuer waits and commits once
        // per G MMA stages.  One token tile: the tiled layout keeps the slabs
        // contiguous (one bulk copy); several token tiles: one 2-D TMA tile
        // per slab from [M][K] (rows past M are zero-filled).
        const uint32_t slab = static_cast<uint32_t>(p.n_tok) * 128u;
        const uint8_t* src = reinterpret_cast<const uint8_t*>(p.xs) + static_cast<int64_t>(mma_begin) * slab;
        const bool rowmajor = p.xs_rowmajor != 0;
        const int G = BS / 2;
        int sj = 0;
        uint32_t sph = 0;
        for (int g0 = 0; g0 < nmma; g0 += G) {
          const int nq = min(G, nmma - g0);
          if (!mbar_wait_a(b_empty(sj), sph ^ 1, abort_flag, p.status)) break;
          mbar_arrive_expect_tx_a(b_full(sj), static_cast<uint32_t>(nq) * slab);
          const uint32_t dst = sbase + p.off_b + static_cast<uint32_t>(sj * G) * slab;
          if (rowmajor) {
            for (int q = 0; q < nq; ++q)
              tma_load_2d(dst + static_cast<uint32_t>(q) * slab, &tm_xs, (mma_begin + g0 + q) * kStageK, m0,
                          b_full(sj));
          } else {
            bulk_load(dst, src + static_cast<int64_t>(g0) * slab, static_cast<uint32_t>(nq) * slab, b_full(sj));
          }
          sj ^= 1;
          if (sj == 0) sph ^= 1;
        }
      } else if (!kCpl && lane == 0) {
        // One bulk copy per 64-wide K slab (tiled layout: the slabs of
        // consecutive MMA stages are contiguous), each slot with its own full
        // and empty barrier, so a slot is refilled as soon as the MMAs that
        // read it are done -- the copy of the next slabs overlaps the MMAs of
        // the current ones.
        // One token tile (up to 128 tokens): the slabs are contiguous in the
        // tiled layout (one bulk copy each); several token tiles read [M][K]
        // through the 2-D tensor map (rows past M are zero-filled).
        const uint32_t slab = static_cast<uint32_t>(p.n_tok) * 128u;
        const uint8_t* src = reinterpret_cast<const uint8_t*>(p.xs) + static_cast<int64_t>(mma_begin) * slab;
        const bool rowmajor = p.xs_rowmajor != 0;
        int sb = 0;
        uint32_t bph = 0;
        for (int j = 0; j < nmma; ++j) {
          if (!mbar_wait_a(b_empty(sb), bph ^ 1, abort_flag, p.status)) break;
          mbar_arrive_expect_tx_a(b_full(sb), slab);
          if (rowmajor)
            tma_load_2d(sbase + p.off_b + sb * slab, &tm_xs, (mma_begin + j) * kStageK, m0, b_full(sb));
          else
            bulk_load(sbase + p.off_b + sb * slab, src + static_cast<int64_t>(j) * slab, slab, b_full(sb));
          if (++sb == BS) {
            sb = 0;
            bph ^= 1;
          }
        }
      }
    }
  } else if (warp >= kIssuerWarp0 && warp < deq0) {
    // ------------------------------------------------------------ MMA issuers
    const int ii = warp - kIssuerWarp0;
    if (ii < n_iss) {
      const uint32_t idesc = idesc_f16_f32(kTileN, static_cast<uint32_t>(p.n_tok));
      const uint32_t d_acc = tmem_base + static_cast<uint32_t>(ii * p.n_tok);
      uint32_t acc = 0;
      if (pairm) {
        // Pair mode: this issuer owns tile ii of the pair (its accumulator,
        // its tensor-memory A slot per MMA stage q: ab_*(ii * kSub + q)) and
        // reads the activation slabs half a ring (G = BS / 2 MMA stages) at a
        // time: one wait before a half's first MMA stage, one commit after its
        // last.
        const uint32_t b_slab = static_cast<uint32_t>(p.n_tok * 128);
        const int G = BS / 2;
        int sj = 0, jj = 0, j = 0;  // slab half, MMA stage within it, MMA stage of the CTA
        uint32_t sph = 0;
        bool ok = true;
        for (int wi = 0; ok && wi < nraw; ++wi) {
          const int nq = min(kSub, nmma - wi * kSub);
          for (int q = 0; q < nq; ++q, ++j) {
            const int sl = ii * kSub + q;
            if ((jj == 0 && !warp_wait(b_full(sj), sph, abort_flag, p.status)) ||
                !warp_wait(ab_full(sl), wi & 1, abort_flag, p.status)) {
              ok = false;
              break;
            }
            tc_fence_after();
            const uint32_t a_st = tmem_base + p.col_a + static_cast<uint32_t>(sl * kAStageCols);
            const uint32_t b_addr = sbase + p.off_b + static_cast<uint32_t>(sj * G + jj) * b_slab;
            const bool last = ++jj == G || j + 1 == nmma;
            if (lane == 0) {
#pragma unroll
              for (int kk = 0; kk < 4; ++kk)
                tc_mma_f16_ts(d_acc, a_st + kk * 8, sw128_kmajor_desc(b_addr + kk * 32), idesc,
                              (wi > 0 || q > 0 || kk > 0) ? 1u : 0u);
              tc_commit(ab_empty(sl));
              if (last) tc_commit(b_empty(sj));
            }
            if (last) {
              jj = 0;
              sj ^= 1;
              if (sj == 0) sph ^= 1;
            }
          }
          __syncwarp();
        }
      } else {
        // The whole warp runs the loop (waits, addresses and descriptors are
        // warp-uniform); lane 0 issues the MMAs and their commits.  A weight
        // stage holds kSub x 4 MMAs (u = 4 q + kk: MMA stage q, K step kk).
        // Coupled, the issuers form two groups that take alternate weight
        // stages (the stages of one barrier pair), so one group's waits,
        // fences and commits overlap the other's MMAs; otherwise one group
        // takes every stage.  Within a group, issuer j takes the contiguous
        // block of `per` MMAs starting at j * per, into its own accumulator.
        // Every issuer of the group waits for the stage's full barrier and
        // commits once to its empty barrier, so the slots cannot be refilled
        // before all of them are done.  Coupled, the stage's activation slabs
        // sit in the activation slot of its A slot's index and land on the
        // same full barrier.
        const int AW = AS / kSub, BW = 2 * AW;
        const int NG = kCpl ? 2 : 1;
        const int gsz = NI / NG;
        const int g = ii / gsz;
        const int per = kSub * 4 / gsz;
        const int u0 = (ii - g * gsz) * per;
        const uint32_t b_slab = static_cast<uint32_t>(p.n_tok * 128);
        int w = g, b = g;  // A slot and barrier pair of stage wi
        uint32_t bph = 0;
        int js = 0, jsb = 0;  // separate activation ring: slab 0 is in slot 0, phase 0
        uint32_t jph = 0;
        for (int wi = g; wi < nraw; wi += NG) {
          if (!warp_wait(ab_full(b), bph, abort_flag, p.status)) break;
          const int nq = min(kSub, nmma - wi * kSub);
          const int u1 = min(u0 + per, 4 * nq);  // this issuer's MMAs in this weight stage: [u0, u1)
          const uint32_t a_st = tmem_base + p.col_a + static_cast<uint32_t>(w * kSub * kAStageCols);
          tc_fence_after();
          if (kCpl) {
            const uint32_t b_st = sbase + p.off_b + static_cast<uint32_t>(w) * p.raw_b_bytes;
            if (lane == 0) {
              for (int u = u0; u < u1; ++u)
                tc_mma_f16_ts(d_acc, a_st + (u >> 2) * kAStageCols + (u & 3) * 8,
                              sw128_kmajor_desc(b_st + (u >> 2) * b_slab + (u & 3) * 32), idesc,
                              u > u0 ? 1u : acc);
              tc_commit(ab_empty(b));
            }
            if (u1 > u0) acc = 1;
          } else {
            // Separate activation ring: each MMA stage's slab has its own
            // full and empty barrier; with <= kSub issuers an MMA stage has a
            // single issuer.  (js, jsb, jph) track this issuer's slab index,
            // its ring slot and phase incrementally (no division in the loop).
            bool ok = true;
            for (int q = u0 >> 2; q < (u1 + 3) >> 2; ++q) {
              const int j = wi * kSub + q;
              while (js < j) {
                ++js;
                if (++jsb == BS) {
                  jsb = 0;
                  jph ^= 1;
                }
              }
              const int sb = jsb;
              if (!warp_wait(b_full(sb), jph, abort_flag, p.status)) {
                ok = false;
                break;
              }
              tc_fence_after();
              const uint32_t b_addr = sbase + p.off_b + sb * b_slab;
              if (lane == 0) {
#pragma unroll
                for (int kk = 0; kk < 4; ++kk)
                  tc_mma_f16_ts(d_acc, a_st + q * kAStageCols + kk * 8, sw128_kmajor_desc(b_addr + kk * 32), idesc,
                                kk > 0 ? 1u : acc);
                tc_commit(b_empty(sb));
              }
              acc = 1;
            }
            if (!ok) break;
            if (lane == 0) tc_commit(ab_empty(b));
          }
          __syncwarp();
          w += NG;
          if (w >= AW) w -= AW;
          b += NG;
          if (b >= BW) {
            b -= BW;
            bph ^= 1;
          }
        }
      }
      if (lane == 0) {
        // The LoRA up-projection goes last, so a slow producer of t never
        // holds up the weight stream.
        if ((pairm || ii == 0) && do_lora && p.lora_early) {
          // Pair mode: each issuer adds its own tile's up-projection (its B^T
          // chunk set; the t tiles are shared).  Otherwise issuer 0 does.
          if (mbar_wait_a(lora_full, 0, abort_flag, p.status)) {
            tc_fence_after();
            const int rc = lora_chunks(L.r);
            const int nbt = pairm ? 2 : 1;
            issue_lora_mmas(p, L, lora_base + static_cast<uint32_t>((pairm ? ii : 0) * rc * kBtChunkBytes),
                            lora_base + static_cast<uint32_t>(nbt * rc * kBtChunkBytes), d_acc);
          }
        }
        if (do_lora && !p.lora_early) {
          tc_commit(ring_free);  // the ring is idle once every mainloop MMA is done
          // Pair mode: each issuer adds its own tile's up-projection (its B^T
          // chunk set; the t tiles are shared).  Otherwise issuer 0 does.
          if ((pairm || ii == 0) && mbar_wait_a(lora_full, 0, abort_flag, p.status)) {
            tc_fence_after();
            const int rc = lora_chunks(L.r);
            const int nbt = pairm ? 2 : 1;
            issue_lora_mmas(p, L, lora_base + static_cast<uint32_t>((pairm ? ii : 0) * rc * kBtChunkBytes),
                            lora_base + static_cast<uint32_t>(nbt * rc * kBtChunkBytes), d_acc);
          }
        }
        tc_commit(acc_full);  // always, so the epilogue's wait completes even after an abort
      }
    } else if (pairm && do_lora && ii >= 2) {
      // Pair mode: the issuer warps without a tile build the LoRA operand's
      // t tiles (shared by both tiles) from the partial sums in global
      // memory while the weights stream, into the dedicated LoRA region.
      const int ltid = static_cast<int>(threadIdx.x) - 32 * (kIssuerWarp0 + 2);
      const int lthr = 32 * kPairLoraWarps;
      griddep_wait();  // t and the row exponents come from the preceding kernel
      fill_lora_factors(p, L, smv + 4u * p.n_tok, m0, ltid, lthr);
      named_barrier_sync(2, lthr);
      // Without room for a dedicated region (large ranks) the operand is
      // built in the ring once the mainloop has left it.
      if (p.lora_early || warp_wait(ring_free, 0, abort_flag, p.status))
        build_t_tiles(p, L, lora_base, smv + 4u * p.n_tok, m0, ltid, lthr, 2);
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive_a(lora_full);
    }
  } else if (warp >= deq0) {
    // ------------------------------------------------------------ dequant warps
    const int dw = warp - deq0;
    uint32_t lut = 0u;
    if (L.nf4) {
      // The NF4 table: entry e (a code byte) = the fp16 pair (level[e & 15],
      // level[e >> 4]), low element in the low half as the E2M1 conversion.
      lut = sbase + p.off_lut;
      const int e = static_cast<int>(threadIdx.x) - 32 * deq0;  // 0..255
      sts32(lut + 4u * e, static_cast<uint32_t>(p.nf4_half[e & 15]) | (static_cast<uint32_t>(p.nf4_half[e >> 4]) << 16));
      named_barrier_sync(3, 256);
    }
    // The loops are instantiated with and without the NF4 table, so the E2M1
    // path carries no per-word branch.
    auto dequant_loops = [&](auto lut_on) {
      constexpr bool kLut = decltype(lut_on)::value;
      if (pairm) {
        // Pair mode: group g = dw / 4 dequantizes tile g of the pair (a thread
        // is one weight row of it), every weight stage, and hands each MMA
        // stage's 32 TMEM columns over as soon as they are stored, so the next
        // stage's conversion overlaps the current stage's remaining MMAs.
        const int g = dw >> 2;
        if (g < ntl) {
          const int row = 32 * (warp & 3) + lane;
          const uint32_t lane_base = static_cast<uint32_t>(32 * (warp & 3)) << 16;
          int s = 0;
          uint32_t ph = 0;
          for (int i = 0; i < nraw; ++i) {
            if (!warp_wait(raw_full(s), ph, abort_flag, p.status)) break;
            const uint32_t slot = sbase + p.off_raw + s * rslot + g * kRawSlotBytes;
            const int nq = min(kSub, nmma - i * kSub);
            bool ok = true;
#pragma unroll
            for (int q = 0; q < kSub; ++q) {
              if (q >= nq) break;
              uint32_t o[32];
              dequant_mma_stage<kLut, kWt>(slot, row, q, lut, o);
              const int sl = g * kSub + q;
              if (!warp_wait(ab_empty(sl), (i & 1) ^ 1, abort_flag, p.status)) {
                ok = false;
                break;
              }
              tmem_st_x32(tmem_base + lane_base + p.col_a + static_cast<uint32_t>(sl * kAStageCols), o);
              tmem_st_wait();
              tc_fence_before();
              __syncwarp();
              if (lane == 0) mbar_arrive_a(ab_full(sl));
            }
            if (!ok) break;
            __syncwarp();
            if (lane == 0) mbar_arrive_a(raw_empty(s));
            if (++s == RS) {
              s = 0;
              ph ^= 1;
            }
          }
        }
      } else {
        // Two groups of four warps (one per TMEM lane quadrant, warp % 4) take
        // alternate weight stages: group g = dw / 4 dequantizes stages g, g + 2,
        // ...  A thread is one weight row (its lane of the quadrant) and covers
        // the stage's whole 256-wide K range, one MMA stage (64 K = 32 TMEM
        // columns of fp16 pairs) at a time: convert, store to tensor memory,
        // next.  While one group stores and hands a stage over, the other
        // converts the next one, so the conversion units stay busy.
        const int grp = dw >> 2;
        const int row = 32 * (warp & 3) + lane;
        const uint32_t lane_base = static_cast<uint32_t>(32 * (warp & 3)) << 16;
        const int AW = AS / kSub, BW = 2 * AW;  // tensor-memory slots (one weight stage each, >= 2); barrier pairs
        // Stage i: raw slot i mod RS, A slot i mod AW, barrier pair i mod BW;
        // before its first store, stage i - AW (same A slot) must have
        // finished its MMAs: pair (i - AW) mod BW, whose phase parity for
        // that stage starts at 1 (a fresh barrier: the first AW stages pass).
        int s = grp, w = grp, b = grp, e = grp + AW;
        uint32_t ph = 0, eph = 1;
        for (int i = grp; i < nraw; i += 2) {
          if (!warp_wait(raw_full(s), ph, abort_flag, p.status)) break;
          const uint32_t slot = sbase + p.off_raw + s * kRawSlotBytes;
          const int nq = min(kSub, nmma - i * kSub);
          const uint32_t a_slot = tmem_base + lane_base + p.col_a + static_cast<uint32_t>(w * kSub * kAStageCols);
          bool ok = true;
          // Unrolled by two, not four: the smaller loop body measured 3-5% faster
          // on short launches (instruction fetch), equal on long ones.
#pragma unroll 2
          for (int q = 0; q < kSub; ++q) {
            if (q >= nq) break;
            // MMA stage q: 16-byte code chunks 2q, 2q + 1 of the row (128-byte
            // swizzle) and the scales of the same K range.
            uint32_t o[32];
            dequant_mma_stage<kLut, kWt>(slot, row, q, lut, o);
            // The slot's previous MMAs must be done before the first store
            // (the first conversion overlaps that wait).
            if (q == 0 && !warp_wait(ab_empty(e), eph, abort_flag, p.status)) {
              ok = false;
              break;
            }
            tmem_st_x32(a_slot + q * kAStageCols, o);
          }
          if (!ok) break;
          tmem_st_wait();
          tc_fence_before();
          __syncwarp();
          if (lane == 0) {
            mbar_arrive_a(ab_full(b));
            mbar_arrive_a(raw_empty(s));
          }
          s += 2;
          if (s >= RS) {
            s -= RS;
            ph ^= 1;
          }
          w += 2;
          if (w >= AW) w -= AW;
          b += 2;
          if (b >= BW) b -= BW;
          e += 2;
          if (e >= BW) {
            e -= BW;
            eph ^= 1;
          }
        }
      }
    };
    if (lut != 0u)
      dequant_loops(std::true_type{});
    else
      dequant_loops(std::false_type{});
    if (do_lora && !pairm) {
      // The LoRA operand's t tiles, by all 256 dequant threads once their
      // stream is done: from the rows the LoRA warp staged (early), or from
      // global memory into the idle ring (late).
      const int dtid = static_cast<int>(threadIdx.x) - 32 * deq0;
      griddep_wait();  // the row exponents come from the preceding kernel
      fill_lora_factors(p, L, smv + 4u * p.n_tok, m0, dtid, 256);
      named_barrier_sync(1, 256);
      if (p.lora_early) {
        if (warp_wait(t_full, 0, abort_flag, p.status))
          build_t_tiles_staged(p, L, lora_base, sbase + p.off_tstage, smv + 4u * p.n_tok, min(p.n_tok, p.M - m0),
                               dtid, 256);
      } else if (warp_wait(ring_free, 0, abort_flag, p.status)) {
        build_t_tiles(p, L, lora_base, smv + 4u * p.n_tok, m0, dtid, 256, pairm ? 2 : 1);
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive_a(lora_full);
    }
  } else if (warp == kLoraWarp) {
    // ------------------------------------------------------------ LoRA operands
    if (do_lora) {
      if (p.lora_early && pairm) {
        // Both tiles' B^T chunk sets (a missing second tile: zeros); the
        // idle issuer warps build the t tiles.
        if (lane == 0) load_bt_tiles(L, tm_bl, lora_base, n0, lora_full, 2);
      } else if (p.lora_early) {
        if (lane == 0) load_bt_tiles(L, tm_bl, lora_base, n0, lora_full);
        griddep_wait();  // t comes from the preceding kernel
        // Bulk-copy this tile's rows of every partial sum, then convert from
        // shared memory (scalar loads from L2 would serialize on latency).
        const int rows = min(p.n_tok, p.M - m0);
        const uint32_t bytes = static_cast<uint32_t>(rows * L.r * 4);
        const uint32_t tstage = sbase + p.off_tstage;
        if (lane == 0) {
          mbar_arrive_expect_tx_a(t_full, bytes * static_cast<uint32_t>(p.t_groups));
          for (int g = 0; g < p.t_groups; ++g)
            bulk_load(tstage + static_cast<uint32_t>(g * p.n_tok * L.r * 4),
                      L.t + (static_cast<int64_t>(g) * p.M + m0) * L.r, bytes, t_full);
        }
        // The dequant warps build the t tiles from these rows after their main loop.
      } else if (warp_wait(ring_free, 0, abort_flag, p.status)) {
        // Pair mode: both tiles' B^T chunk sets (the second one's rows past N
        // read as zeros); otherwise this tile's.
        if (lane == 0) load_bt_tiles(L, tm_bl, lora_base, n0, lora_full, pairm ? ntl : 1);
      } else if (lane == 0) {
        mbar_arrive_expect_tx_a(lora_full, 0);  // after an abort: keep the barrier count consistent
      }
    }
  }

  // ---------------------------------------------------------------- epilogue
  const uint32_t part = sbase;  // [tile][n_tok][128] fp32 scaled partial tiles (split > 1), ring reused
  const int dt = static_cast<int>(threadIdx.x) - 32 * deq0;  // dequant-warp thread index
  const int ntl_e = pairm ? ntl : 1;                              // weight tiles of this CTA
  if (warp >= deq0) {
    // Row scales S * 2^-e_m come from the preceding kernel (or, acts_ready,
    // the one before it); the dequant above did not need them.
    if (!p.acts_ready) griddep_wait();
    {
      const float S = *L.tensor_scale;
      for (int i = dt; i < p.n_tok; i += 256)
        stsf(smv + 4u * i, (m0 + i < p.M) ? S * __ldg(p.rinv + m0 + i) : 0.0f);
    }
    named_barrier_sync(1, 256);
    const bool ok = warp_wait(acc_full, 0, abort_flag, p.status);
    tc_fence_after();
    const int q = warp & 3;
    const int nl = q * 32 + lane;
    // Pair mode: warp group eg reads tile eg's accumulator, all token columns;
    // otherwise the two groups split the token columns of the one tile.
    const int eg = pairm ? (warp - deq0) >> 2 : 0;
    const bool live = eg < ntl_e;
    const int n = n0 + eg * kTileN + nl;
    const int cols = pairm ? p.n_tok : p.n_tok / 2;
    const int c0 = pairm ? 0 : ((warp - deq0) >> 2) * cols;
    const uint32_t lane_off = static_cast<uint32_t>(q * 32) << 16;
    const uint32_t acc0 = static_cast<uint32_t>(eg * p.n_tok);       // first accumulator column
    const uint32_t tile_out = static_cast<uint32_t>(eg * p.n_tok * kTileN);  // element offset of its staged tile
    // Issuer a holds a sum iff it issued an MMA, i.e. iff its block of MMAs
    // starts inside the first weight stage of its group (only the last stage
    // can be short).  One group: a prefix of the issuers.  Two groups
    // (coupled): group g's first stage is stage g.  Pair mode: one
    // accumulator per tile.
    uint32_t accs = 1u;
    if (!pairm) {
      const int NG = kCpl ? 2 : 1, gsz = NI / NG, per = kSub * 4 / gsz;
      accs = 0u;
      for (int g = 0; g < NG && g < nraw; ++g) {
        const int nq = min(kSub, nmma - g * kSub);
        for (int j = 0; j < gsz && j * per < 4 * nq; ++j) accs |= 1u << (g * gsz + j);
      }
    }
    const int nacc = 32 - __clz(static_cast<int>(accs));  // accumulator slots to scan
    if (pairm && live) {
      // One accumulator per tile: 32 token columns per TMEM load and wait
      // (columns past n_tok are read -- they lie inside tensor memory -- but
      // not stored).  The row scales come in as vectors; an unsplit tile is
      // stored straight from registers (a warp writes 32 consecutive outputs
      // of one token row per store), a split one goes to its partial tile.
      const int rows = min(p.n_tok, p.M - m0);
      for (int c = 0; c < p.n_tok; c += 32) {
        float w[32], sc[32];
        tmem_ld_x32(tmem_base + acc0 + lane_off + c, w);
#pragma unroll
        for (int e = 0; e < 32; e += 4) {
          const float4 s4 = lds128f(smv + 4u * (c + e));
          sc[e] = s4.x;
          sc[e + 1] = s4.y;
          sc[e + 2] = s4.z;
          sc[e + 3] = s4.w;
        }
        tmem_ld_wait();
        if (p.split > 1) {
#pragma unroll
          for (int e = 0; e < 32; ++e)
            if (c + e < p.n_tok)
              stsf(part + 4u * (tile_out + static_cast<uint32_t>((c + e) * kTileN + nl)), ok ? w[e] * sc[e] : 0.0f);
        } else if (p.stage_out) {
          // staged [tile][token][128 rows], stored below as 16-byte vectors
          const uint32_t el0 = tile_out + static_cast<uint32_t>(c * kTileN + nl);
          if (L.y_f32) {
#pragma unroll
            for (int e = 0; e < 32; ++e)
              if (c + e < p.n_tok) stsf(sbase + 4u * (el0 + e * kTileN), ok ? w[e] * sc[e] : 0.0f);
          } else {
#pragma unroll
            for (int e = 0; e < 32; ++e)
              if (c + e < p.n_tok)
                sts16(sbase + 2u * (el0 + e * kTileN), __bfloat16_as_ushort(__float2bfloat16_rn(ok ? w[e] * sc[e] : 0.0f)));
          }
        } else if (n < L.N) {
#pragma unroll
          for (int e = 0; e < 32; ++e)
            if (c + e < rows) store_out(L, m0 + c + e, n, ok ? w[e] * sc[e] : 0.0f);
        }
      }
    }
    // Up to two accumulators (65-128 tokens): 32 token columns of each per
    // TMEM wait.  More (up to 64 tokens): 8 columns of up to four of them per
    // wait.  The row scales arrive as vectors (one shared-memory load per
    // four values, not one per value).  (This runs once per CTA, its
    // instructions fetched cold: kept compact -- rolled loops, one store loop
    // per output kind.)
    auto emit8 = [&](int c, const float (&val)[8]) {
      const uint32_t el0 = tile_out + static_cast<uint32_t>(c * kTileN + nl);
      if (p.split > 1) {
#pragma unroll
        for (int e = 0; e < 8; ++e) stsf(part + 4u * (el0 + e * kTileN), val[e]);
      } else if (!p.stage_out) {
        for (int e = 0; e < 8; ++e)
          if (m0 + c + e < p.M && n < L.N) store_out(L, m0 + c + e, n, val[e]);
      } else if (L.y_f32) {
#pragma unroll
        for (int e = 0; e < 8; ++e) stsf(sbase + 4u * (el0 + e * kTileN), val[e]);  // staged: [tile][token][128 rows]
      } else {
#pragma unroll
        for (int e = 0; e < 8; ++e)
          sts16(sbase + 2u * (el0 + e * kTileN), __bfloat16_as_ushort(__float2bfloat16_rn(val[e])));
      }
    };
    if (!pairm && (accs == 1u || accs == 3u) && cols % 32 == 0) {
      for (int c = c0; c < c0 + cols; c += 32) {
        float w[32], w2[32];
        tmem_ld_x32(tmem_base + acc0 + lane_off + c, w);
        if (nacc == 2) tmem_ld_x32(tmem_base + acc0 + static_cast<uint32_t>(p.n_tok) + lane_off + c, w2);
        tmem_ld_wait();
#pragma unroll
        for (int e8 = 0; e8 < 32; e8 += 8) {
          const float4 s0 = lds128f(smv + 4u * (c + e8)), s1 = lds128f(smv + 4u * (c + e8 + 4));
          const float sc[8] = {s0.x, s0.y, s0.z, s0.w, s1.x, s1.y, s1.z, s1.w};
          float o8[8];
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            const float a = nacc == 2 ? w[e8 + e] + w2[e8 + e] : w[e8 + e];
            o8[e] = ok ? a * sc[e] : 0.0f;
          }
          emit8(c + e8, o8);
        }
      }
    } else {
    for (int c = c0; !pairm && c < c0 + cols; c += 8) {
      float v[8];
      // Four accumulators' columns per wait (issuer 0's holds the LoRA term).
#pragma unroll 1
      for (int a0 = 0; a0 < nacc; a0 += 4) {
        float w[4][8];
#pragma unroll
        for (int a = 0; a < 4; ++a)
          if ((accs >> (a0 + a)) & 1u)
            tmem_ld_x8(tmem_base + acc0 + static_cast<uint32_t>((a0 + a) * p.n_tok) + lane_off + c, w[a]);
        tmem_ld_wait();
        // (Accumulator 0 always holds a sum.)
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          float t = a0 == 0 ? w[0][e] : v[e];
          if (a0 > 0 && ((accs >> a0) & 1u)) t += w[0][e];
#pragma unroll
          for (int a = 1; a < 4; ++a)
            if ((accs >> (a0 + a)) & 1u) t += w[a][e];
          v[e] = t;
        }
      }
      const float4 s0 = lds128f(smv + 4u * c), s1 = lds128f(smv + 4u * (c + 4));
      const float sc[8] = {s0.x, s0.y, s0.z, s0.w, s1.x, s1.y, s1.z, s1.w};
      float o8[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) o8[e] = ok ? v[e] * sc[e] : 0.0f;
      emit8(c, o8);
    }
    }
    if (p.split == 1 && p.stage_out) {
      // The output tile leaves shared memory (the idle ring) a token row at a
      // time: one bulk copy per row when rows are 16-byte aligned (the writes
      // drain after the CTA has moved on), else 16-byte vectors.
      fence_proxy_async_smem();  // the staged tile is read by bulk copies below
      named_barrier_sync(1, 256);
      const int rows = min(p.n_tok, p.M - m0);
      const int es = L.y_f32 ? 4 : 2;
      uint8_t* ybase = reinterpret_cast<uint8_t*>(L.y);
      const bool vec = (reinterpret_cast<uintptr_t>(ybase) & 15u) == 0 && (static_cast<int64_t>(L.N) * es) % 16 == 0;
      for (int t = 0; t < ntl_e; ++t) {
      const int n0t = n0 + t * kTileN;
      const int nvalid = min(kTileN, L.N - n0t);
      const uint32_t stile = sbase + static_cast<uint32_t>(t * p.n_tok * kTileN * es);
      // (Bulk copies are processed one after another: many token rows go out
      // as coalesced vector stores instead.)
      if (vec && (nvalid * es) % 16 == 0 && p.n_tok <= 64) {
        if (dt < rows) {
          bulk_store(ybase + (static_cast<int64_t>(m0 + dt) * L.N + n0t) * es,
                     stile + static_cast<uint32_t>(dt * kTileN * es), static_cast<uint32_t>(nvalid * es));
          bulk_commit_group();
          bulk_wait_group_read0();
        }
      } else {
        const int chunks = vec ? nvalid * es / 16 : 0;  // whole 16-byte chunks per token row
        for (int it = dt; it < rows * chunks; it += 256) {
          const int ml = it / chunks, ch = it - ml * chunks;
          const uint4 val = lds128(stile + static_cast<uint32_t>(ml * kTileN * es + ch * 16));
          *reinterpret_cast<uint4*>(ybase + (static_cast<int64_t>(m0 + ml) * L.N + n0t) * es + ch * 16) = val;
        }
        const int e0 = chunks * 16 / es;  // the rest element by element
        const int rest = nvalid - e0;
        for (int it = dt; it < rows * rest; it += 256) {
          const int ml = it / rest, nn = e0 + (it - ml * rest);
          const int64_t gi = static_cast<int64_t>(m0 + ml) * L.N + n0t + nn;
          if (L.y_f32)
            reinterpret_cast<float*>(ybase)[gi] = ldsf(stile + 4u * (ml * kTileN + nn));
          else
            reinterpret_cast<uint16_t*>(ybase)[gi] = lds16(stile + 2u * (ml * kTileN + nn));
        }
      }
      }
    }
  }
  if (*abort_flag) {
    // Let copies that were already issued land before shared memory is released.
    const long long t0 = clock64();
    while (clock64() - t0 < 200000ll) {
    }
  }
  tc_fence_before();
  __syncthreads();

  if (p.split > 1) {
    cluster_sync_all();  // every partner's scaled partial tile is in its shared memory
    if (warp >= deq0) {
      const int rank = static_cast<int>(cluster_ctarank());
      const int per = (p.n_tok + p.split - 1) / p.split;
      const int mb = rank * per;
      const int me = min(min(p.n_tok, mb + per), p.M - m0);
      // Four consecutive outputs per thread: one 8- (bf16) or 16-byte (f32)
      // store when the row pitch and base allow it.
      const bool vec4 = (reinterpret_cast<uintptr_t>(L.y) & 15u) == 0 && L.N % 4 == 0;
      const int per_tile = max(0, me - mb) * (kTileN / 4);
      // Every partner's partial tile, mapped once.  Each thread sums one
      // 4-column group per step and issues all its partners' remote loads (up
      // to 8) before the first add, so the distributed-shared-memory latency
      // is paid once per group, not once per partner.  (One group per step,
      // not two: this code runs once per CTA and its instructions are fetched
      // cold, so it is kept small.)
      uint32_t rpart[kMaxSplit];
#pragma unroll
      for (int qq = 0; qq < kMaxSplit; ++qq) rpart[qq] = qq < p.split ? mapa_shared(part, qq) : 0u;
      for (int it = dt; it < ntl_e * per_tile; it += 256) {
        const int t = it / per_tile, rem = it - t * per_tile;
        const int ml = mb + rem / (kTileN / 4);
        const int nl4 = 4 * (rem % (kTileN / 4)) + t * kTileN;  // column within this CTA's tiles
        const uint32_t off = 4u * static_cast<uint32_t>(t * p.n_tok * kTileN + ml * kTileN + 4 * (rem % (kTileN / 4)));
        float4 v[kMaxSplit];
#pragma unroll
        for (int qq = 0; qq < kMaxSplit; ++qq)
          if (qq < p.split) v[qq] = ld_shared_cluster_f32x4(rpart[qq] + off);
        float4 acc = v[0];
#pragma unroll
        for (int qq = 1; qq < kMaxSplit; ++qq)
          if (qq < p.split) {
            acc.x += v[qq].x;
            acc.y += v[qq].y;
            acc.z += v[qq].z;
            acc.w += v[qq].w;
          }
        const int64_t gi = static_cast<int64_t>(m0 + ml) * L.N + n0 + nl4;
        if (vec4 && n0 + nl4 + 3 < L.N) {
          if (L.y_f32) {
            *reinterpret_cast<float4*>(reinterpret_cast<float*>(L.y) + gi) = acc;
          } else {
            uint2 pk;
            pk.x = static_cast<uint32_t>(__bfloat16_as_ushort(__float2bfloat16_rn(acc.x))) |
                   (static_cast<uint32_t>(__bfloat16_as_ushort(__float2bfloat16_rn(acc.y))) << 16);
            pk.y = static_cast<uint32_t>(__bfloat16_as_ushort(__float2bfloat16_rn(acc.z))) |
                   (static_cast<uint32_t>(__bfloat16_as_ushort(__float2bfloat16_rn(acc.w))) << 16);
            *reinterpret_cast<uint2*>(reinterpret_cast<__nv_bfloat16*>(L.y) + gi) = pk;
          }
        } else {
          const float out[4] = {acc.x, acc.y, acc.z, acc.w};
#pragma unroll
          for (int e = 0; e < 4; ++e)
            if (n0 + nl4 + e < L.N) store_out(L, m0 + ml, n0 + nl4 + e, out[e]);
        }
      }
    }
    // Partners are done reading this CTA's partial tile.  (Relaxed: this
    // CTA's own remote loads have all been consumed, and its output stores
    // need not be ordered for the partners.)
    cluster_arrive_relaxed();
    cluster_wait();
  }
  if (warp == kIssuerWarp0) tmem_dealloc(tmem_base, kTmemCols);
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

// ---------------------------------------------------------------------------
// The LoRA down-projection on the tensor cores, for more than 128 tokens
// ("Low-Rank Adaptation (LoRA) Within Quantized Layers", Eq. 2: the branch's
// first factor, t = x~ A^T, which the up-projection in the linear's epilogue
// consumes):  t_i[m][j] = sum_k X[m][k] A_i[j][k],  X bf16 [M][K] (x~),
// A_i bf16 [r_i][K], t_i fp32 [M][r_i].
// A CTA: 128 token rows x round16(r_i) ranks over a K range; grid (split,
// token tiles, linears), clusters of `split` CTAs along K whose fp32
// accumulators are added over distributed shared memory in rank order
// (deterministic).  Warp 0 lane 0 streams (X, A) 64-wide K stages by TMA
// (128-byte swizzle; rows past M and ranks past r read as zeros); warp 1
// lane 0 issues kind::f16 MMAs with bf16 operands (products exact, fp32
// accumulation) into tensor memory; all four warps read the accumulator back.
constexpr int kLdThreads = 128;
constexpr int kLdStages = 4;
constexpr int kLdMaxSplit = 8;

struct LdMaps {
  CUtensorMap x;
  CUtensorMap a[kMaxLinears];
};
struct LdParams {
  int M, K;
  int r[kMaxLinears];
  float* t[kMaxLinears];
  int lin_of[kMaxLinears];  // blockIdx.z -> linear
  int split;
  // groups > 1: K is cut into groups * split slices; each cluster (one
  // group) writes its partial sum to tpart[i] + g * M * r, and the last
  // cluster of a token tile to finish (counted in counters[], reset by it)
  // adds the groups in group order into t[i].
  int groups, m_tiles;
  float* tpart[kMaxLinears];
  unsigned* counters;
  int* status;
};

__host__ __device__ constexpr uint32_t ld_stage_bytes(int r16) { return 16384u + static_cast<uint32_t>(r16) * 128u; }
__host__ __device__ constexpr uint32_t ld_smem_bytes(int r16) {
  return 1024u + kLdStages * ld_stage_bytes(r16) + 8u * (2 * kLdStages + 2) + 8u;
}

__global__ void __launch_bounds__(kLdThreads, 1)
    lora_down_tc_kernel(const __grid_constant__ LdMaps maps, const LdParams p) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  const uint32_t raw_addr = smem_u32(smem_raw);
  const uint32_t sbase = (raw_addr + 1023u) & ~1023u;
  uint8_t* smem_gen = smem_raw + (sbase - raw_addr);
  const int li = p.lin_of[blockIdx.z];
  const int r = p.r[li];
  const int r16 = (r + 15) & ~15;
  const uint32_t stage_bytes = ld_stage_bytes(r16);  // a multiple of 2048: stages stay 1024-byte aligned
  const uint32_t ring_bytes = kLdStages * stage_bytes;
  const uint32_t bars = sbase + ring_bytes;
  auto full = [&](int s) { return bars + 8u * s; };
  auto empty = [&](int s) { return bars + 8u * (kLdStages + s); };
  const uint32_t acc_full = bars + 8u * (2 * kLdStages);
  const uint32_t tmem_holder = bars + 8u * (2 * kLdStages + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem_gen + ring_bytes + 8 * (2 * kLdStages + 1) + 4);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int split = p.split, sidx = static_cast<int>(blockIdx.x);
  const int mt = static_cast<int>(blockIdx.y) / p.groups, g = static_cast<int>(blockIdx.y) % p.groups;
  const int m0 = mt * 128;
  const int nk = p.K / 64;
  const int pieces = p.groups * split, piece = g * split + sidx;
  const int kc0 = piece * nk / pieces, kc1 = (piece + 1) * nk / pieces;  // >= 1 chunk each (pieces <= nk)
  const uint32_t tcols = r16 <= 32 ? 32u : (r16 <= 64 ? 64u : 128u);

  if (threadIdx.x == 0) {
    for (int s = 0; s < kLdStages; ++s) {
      mbar_init_a(full(s), 1);
      mbar_init_a(empty(s), 1);
    }
    mbar_init_a(acc_full, 1);
    *abort_flag = 0;
    fence_mbarrier_init();
  }
  if (warp == 1) {
    tmem_alloc(tmem_holder, tcols);
    tmem_relinquish();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&maps.x);
    tma_prefetch_desc(&maps.a[li]);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(smem_gen + ring_bytes + 8 * (2 * kLdStages + 1));
  // Every CTA of this grid is resident and holds its tensor memory: the
  // linear's MMA kernel may start its prologue (it waits for this grid's
  // completion before it reads t).
  griddep_launch_dependents();

  if (warp == 0 && lane == 0) {
    int issued = 0;
    for (int kc = kc0; kc < kc1; ++kc) {
      const int i = kc - kc0, s = i % kLdStages;
      if (i >= kLdStages && !mbar_wait_a(empty(s), ((i / kLdStages) & 1) ^ 1, abort_flag, p.status)) break;
      mbar_arrive_expect_tx_a(full(s), stage_bytes);
      const uint32_t st = sbase + s * stage_bytes;
      tma_load_2d(st, &maps.x, kc * 64, m0, full(s));
      tma_load_2d(st + 16384u, &maps.a[li], kc * 64, 0, full(s));
      issued = i + 1;
    }
    // Every issued copy lands before the ring is reused or the CTA exits
    // (after an expired wait too): wait for each slot's last copy, bounded.
    volatile int no_abort = 0;
    for (int s = 0; s < min(issued, kLdStages); ++s) {
      const int last = issued - 1 - ((issued - 1 - s) % kLdStages);
      mbar_wait_a(full(s), (last / kLdStages) & 1, &no_abort, p.status);
    }
  } else if (warp == 1 && lane == 0) {
    const uint32_t idesc = idesc_bf16_f32(128, static_cast<uint32_t>(r16));
    for (int kc = kc0; kc < kc1; ++kc) {
      const int i = kc - kc0, s = i % kLdStages;
      if (!mbar_wait_a(full(s), (i / kLdStages) & 1, abort_flag, p.status)) break;
      tc_fence_after();
      const uint32_t st = sbase + s * stage_bytes;
#pragma unroll
      for (int kk = 0; kk < 4; ++kk)
        tc_mma_f16(tmem, sw128_kmajor_desc(st + kk * 32), sw128_kmajor_desc(st + 16384u + kk * 32), idesc,
                   (i > 0 || kk > 0) ? 1u : 0u);
      tc_commit(empty(s));
    }
    tc_commit(acc_full);  // also after an expired wait: arrives once the issued MMAs are done
  }
  __syncwarp();
  const bool ok = mbar_wait_a(acc_full, 0, abort_flag, p.status);
  tc_fence_after();
  __syncthreads();  // the producer's copies have landed: the ring is free
  const int row = 32 * warp + lane;
  const int m = m0 + row;
  const uint32_t lane_addr = tmem + (static_cast<uint32_t>(32 * warp) << 16);
  float* tout = p.groups > 1 ? p.tpart[li] + static_cast<int64_t>(g) * p.M * r : p.t[li];
  if (split == 1) {
    for (int c = 0; c < r16; c += 8) {
      float v[8];
      tmem_ld_x8(lane_addr + c, v);
      tmem_ld_wait();
      if (ok && m < p.M)
#pragma unroll
        for (int e = 0; e < 8; ++e)
          if (c + e < r) tout[static_cast<int64_t>(m) * r + c + e] = v[e];
    }
  } else {
    // Partial tile -> this CTA's shared memory ([128][r16] fp32 in the idle
    // ring), then rank c of the cluster adds rows c, c + split, ... over all
    // partners in rank order.
    const uint32_t red = sbase;
    for (int c = 0; c < r16; c += 8) {
      float v[8];
      tmem_ld_x8(lane_addr + c, v);
      tmem_ld_wait();
#pragma unroll
      for (int e = 0; e < 8; ++e) stsf(red + static_cast<uint32_t>((row * r16 + c + e) * 4), v[e]);
    }
    cluster_sync_all();
    const int q4 = r16 / 4;
    const int my_rows = (128 - sidx + split - 1) / split;
    for (int it = threadIdx.x; it < my_rows * q4; it += kLdThreads) {
      const int rr = sidx + split * (it / q4), c4 = (it % q4) * 4;
      const uint32_t off = red + static_cast<uint32_t>((rr * r16 + c4) * 4);
      float4 v[kLdMaxSplit];
#pragma unroll
      for (int q = 0; q < kLdMaxSplit; ++q)
        if (q < split) v[q] = ld_shared_cluster_f32x4(mapa_shared(off, static_cast<uint32_t>(q)));
      float4 acc = v[0];
#pragma unroll
      for (int q = 1; q < kLdMaxSplit; ++q)
        if (q < split) {
          acc.x += v[q].x;
          acc.y += v[q].y;
          acc.z += v[q].z;
          acc.w += v[q].w;
        }
      const int mm = m0 + rr;
      if (ok && mm < p.M) {
        const float a4[4] = {acc.x, acc.y, acc.z, acc.w};
#pragma unroll
        for (int e = 0; e < 4; ++e)
          if (c4 + e < r) tout[static_cast<int64_t>(mm) * r + c4 + e] = a4[e];
      }
    }
    cluster_sync_all();  // partners are done reading this CTA's partial tile
  }
  if (p.groups > 1) {
    // Rank sidx of every group's cluster wrote rows sidx, sidx + split, ...:
    // the last of them to finish adds those rows over the groups in group
    // order (release: this CTA's barrier orders its writes before the fence
    // and atomic of thread 0; acquire: the fence after it).
    __shared__ unsigned last;
    __syncthreads();
    if (threadIdx.x == 0) {
      unsigned* cnt = p.counters + (static_cast<int>(blockIdx.z) * p.m_tiles + mt) * split + sidx;
      __threadfence();
      const unsigned done = atomicAdd(cnt, 1u);
      last = done == static_cast<unsigned>(p.groups - 1) ? 1u : 0u;
      if (last) {
        __threadfence();
        *cnt = 0u;
      }
    }
    __syncthreads();
    if (last && ok) {
      const float* tp = p.tpart[li];
      const int r4 = r / 4;
      const int my_rows = (128 - sidx + split - 1) / split;
      const int64_t gstride = static_cast<int64_t>(p.M) * r;
      for (int it = threadIdx.x; it < my_rows * r4; it += kLdThreads) {
        const int mm = m0 + sidx + split * (it / r4), c4 = (it % r4) * 4;
        if (mm >= p.M) break;
        const float* src = tp + static_cast<int64_t>(mm) * r + c4;
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
        for (int g0 = 0; g0 < p.groups; g0 += 4) {
          float4 v[4];
#pragma unroll
          for (int u = 0; u < 4; ++u)
            if (g0 + u < p.groups) v[u] = __ldcg(reinterpret_cast<const float4*>(src + (g0 + u) * gstride));
#pragma unroll
          for (int u = 0; u < 4; ++u)
            if (g0 + u < p.groups) {
              acc.x += v[u].x;
              acc.y += v[u].y;
              acc.z += v[u].z;
              acc.w += v[u].w;
            }
        }
        *reinterpret_cast<float4*>(p.t[li] + static_cast<int64_t>(mm) * r + c4) = acc;
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) tmem_dealloc(tmem, tcols);
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

// SM count of the current device, queried once per device.
int sm_count() {
  constexpr int kMaxDevices = 64;
  static std::atomic<int> cached[kMaxDevices] = {};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev >= 0 && dev < kMaxDevices) {
    const int c = cached[dev].load(std::memory_order_relaxed);
    if (c > 0) return c;
  }
  int sms = 148;
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (dev >= 0 && dev < kMaxDevices && sms > 0) cached[dev].store(sms, std::memory_order_relaxed);
  return sms;
}

// How many clusters of `sp` decode-kernel CTAs (maximal shared memory, one
// per SM) can be resident on the current device at once; queried once per
// device and cluster size.  sp == 1: the SM count.
int resident_clusters(int sp) {
  constexpr int kMaxDevices = 64;
  static std::atomic<int> cached[kMaxDevices][kMaxSplit + 1] = {};
  int dev = 0;
  cudaGetDevice(&dev);
  const bool cacheable = dev >= 0 && dev < kMaxDevices && sp >= 1 && sp <= kMaxSplit;
  if (cacheable) {
    const int c = cached[dev][sp].load(std::memory_order_relaxed);
    if (c > 0) return c;
  }
  int n = 0;
  if (sp == 1) {
    n = sm_count();
  } else {
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(static_cast<unsigned>(sp), 1, 1);
    cfg.blockDim = dim3(kMmaThreads, 1, 1);
    cfg.dynamicSmemBytes = kSmemLimit;
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeClusterDimension;
    at[0].val.clusterDim.x = static_cast<unsigned>(sp);
    at[0].val.clusterDim.y = 1;
    at[0].val.clusterDim.z = 1;
    cfg.attrs = at;
    cfg.numAttrs = 1;
    if (cudaOccupancyMaxActiveClusters(&n, mma_kernel<0, 0>, &cfg) != cudaSuccess) {
      cudaGetLastError();  // the query failed: fall back to whole SMs
      n = sm_count() / sp;
    }
  }
  if (cacheable && n > 0) cached[dev][sp].store(n, std::memory_order_relaxed);
  return n;
}

// The tensor-core LoRA down-projection (lora_down_tc_kernel) of up to four
// linears sharing X (bf16 [M][ldx]): t[i] fp32 [M][r[i]] (r[i] == 0: skipped).
qerl_status lora_down_tc(const void* x, int64_t ldx, int64_t M, int64_t K, const void* const* A, const int* r,
                         float* const* t, float* const* tpart, int max_groups, unsigned* counters, int nlin,
                         int* status, cudaStream_t s) {
  static std::once_flag once;
  static cudaError_t err = cudaSuccess;
  std::call_once(once, [] {
    err = cudaFuncSetAttribute(lora_down_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               static_cast<int>(ld_smem_bytes(128)));
  });
  if (err != cudaSuccess) return QERL_ERR_CUDA;
  LdMaps maps;
  std::memset(&maps, 0, sizeof(maps));
  if (!make_map_2d(&maps.x, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, x, static_cast<uint64_t>(K), static_cast<uint64_t>(M),
                   static_cast<uint64_t>(ldx) * 2, 64, 128, CU_TENSOR_MAP_SWIZZLE_128B))
    return QERL_ERR_CUDA;
  LdParams lp{};
  lp.M = static_cast<int>(M);
  lp.K = static_cast<int>(K);
  lp.status = status;
  int nz = 0, r16max = 0;
  for (int i = 0; i < nlin; ++i) {
    if (r[i] <= 0) continue;
    const int r16 = (r[i] + 15) & ~15;
    if (!make_map_2d(&maps.a[i], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, A[i], static_cast<uint64_t>(K),
                     static_cast<uint64_t>(r[i]), static_cast<uint64_t>(K) * 2, 64, static_cast<uint32_t>(r16),
                     CU_TENSOR_MAP_SWIZZLE_128B))
      return QERL_ERR_CUDA;
    lp.r[i] = r[i];
    lp.t[i] = t[i];
    lp.lin_of[nz++] = i;
    r16max = std::max(r16max, r16);
  }
  if (nz == 0 || M == 0) return QERL_OK;
  const int m_tiles = static_cast<int>((M + 127) / 128);
  const int nk = static_cast<int>(K / 64);
  // Split K over a cluster, then over groups of clusters, until the grid
  // covers the SMs once (a CTA streams 20 KB per K chunk into one SM, so few
  // CTAs over a long K are bound by that SM's ingress).
  // One token tile (decode, up to 128 tokens): a quarter of the SMs.  The
  // MMA grid that follows reads t only after its main loop, and the SMs this
  // grid leaves free take MMA CTAs at once.
  const int cover = m_tiles == 1 ? std::max(1, sm_count() / 4) : sm_count();
  const int want = (cover + m_tiles * nz - 1) / (m_tiles * nz);
  int split = std::max(1, std::min(want, std::min(kLdMaxSplit, nk)));
  int groups = (want + split - 1) / split;
  groups = std::max(1, std::min({groups, max_groups, nk / split}));
  if (m_tiles * nz * split > kMaxLoraCounters) groups = 1;  // one completion counter per (tile, cluster rank)
  lp.split = split;
  lp.groups = groups;
  lp.m_tiles = m_tiles;
  lp.counters = counters;
  for (int i = 0; i < nlin; ++i) lp.tpart[i] = tpart != nullptr ? tpart[i] : nullptr;
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(static_cast<unsigned>(split), static_cast<unsigned>(m_tiles * groups), static_cast<unsigned>(nz));
  cfg.blockDim = dim3(kLdThreads, 1, 1);
  cfg.dynamicSmemBytes = ld_smem_bytes(r16max);
  cfg.stream = s;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeClusterDimension;
  at[0].val.clusterDim.x = static_cast<unsigned>(split);
  at[0].val.clusterDim.y = 1;
  at[0].val.clusterDim.z = 1;
  cfg.attrs = at;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, lora_down_tc_kernel, maps, lp) == cudaSuccess ? QERL_OK : QERL_ERR_CUDA;
}

// Above 64 tokens (where the consumers read one summed t) the LoRA
// down-projection runs on the tensor cores: on CUDA cores its cost grows with
// M * K and dominated the 65-128-token launches.
__host__ inline bool lora_down_on_tc(int64_t m) { return lora_sum_in_prep(m); }

struct LinearLayout {
  size_t xs, rinv, t[kMaxLinears], tf[kMaxLinears], count, xt, total;
};

// Token tiles of up to 128 rows stage x~ in the tiled layout (one tile of
// round_up(m, 16) rows); larger m keeps the row-major [m][k] layout.
inline int tiled_rows_for(int64_t m) { return m <= 128 ? static_cast<int>((m + 15) / 16 * 16) : 0; }

LinearLayout linear_layout(int64_t m, int64_t k, const int* ranks, int nlin, bool rmsnorm) {
  LinearLayout L;
  // Fixed offset, whatever the shape: the LoRA tiles' completion counters,
  // zero between calls (each is reset by the cluster that finishes its tile).
  L.count = kWsHeaderBytes;
  L.xs = align_up(L.count + kMaxLoraCounters * sizeof(unsigned), 256);
  const int tr = tiled_rows_for(m);
  const size_t xs_bytes =
      tr > 0 ? static_cast<size_t>((k + kRawK - 1) / kRawK) * 4u * tr * 128u : static_cast<size_t>(m) * k * 2;
  L.rinv = align_up(L.xs + xs_bytes, 256);
  size_t off = align_up(L.rinv + static_cast<size_t>(m) * 4, 256);
  const size_t groups = static_cast<size_t>(lora_split(m, k, ranks, nlin).groups);
  for (int i = 0; i < kMaxLinears; ++i) {
    L.t[i] = off;
    const int r = i < nlin && ranks[i] > 0 ? ranks[i] : 0;
    off = align_up(off + groups * static_cast<size_t>(m) * r * 4, 256);
    L.tf[i] = off;
    off = align_up(off + static_cast<size_t>(m) * r * 4, 256);
  }
  // x~ in bf16 [m][k] for the LoRA down-projection when it does not read x
  // itself: RMSNorm mode, and (with noise) the tensor-core down-projection.
  L.xt = off;
  bool lora = false;
  for (int i = 0; i < nlin; ++i) lora = lora || ranks[i] > 0;
  if ((rmsnorm || lora_down_on_tc(m)) && lora) off = align_up(off + static_cast<size_t>(m) * k * 2, 256);
  L.total = off;
  return L;
}

constexpr int kPrepSmemLimit = kSmemLimit - 1024;  // leaves room for the kernel's static shared memory

// Kernel attributes are set once per process (not per call), so calls can be
// captured into CUDA graphs.
// One attribute on every instantiation of the MMA kernel.
cudaError_t mma_kernel_attrs(cudaFuncAttribute attr, int value) {
  cudaError_t e = cudaFuncSetAttribute(mma_kernel<0, 0>, attr, value);
  if (e == cudaSuccess) e = cudaFuncSetAttribute(mma_kernel<0, 1>, attr, value);
  if (e == cudaSuccess) e = cudaFuncSetAttribute(mma_kernel<1, 0>, attr, value);
  if (e == cudaSuccess) e = cudaFuncSetAttribute(mma_kernel<1, 1>, attr, value);
  return e;
}

bool kernel_attrs_ok() {
  static std::once_flag attr_once;
  static cudaError_t attr_err = cudaSuccess;
  std::call_once(attr_once, [] {
    attr_err = cudaFuncSetAttribute(prep_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kPrepSmemLimit);
    // The prep grid runs beside the MMA kernel's CTAs (which start early and
    // hold most of shared memory): the same carveout lets them share an SM.
    if (attr_err == cudaSuccess)
      attr_err = cudaFuncSetAttribute(prep_kernel, cudaFuncAttributePreferredSharedMemoryCarveout,
                                      cudaSharedmemCarveoutMaxShared);
    if (attr_err == cudaSuccess)
      attr_err = mma_kernel_attrs(cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemLimit);
    if (attr_err == cudaSuccess)
      attr_err = mma_kernel_attrs(cudaFuncAttributePreferredSharedMemoryCarveout, cudaSharedmemCarveoutMaxShared);
  });
  return attr_err == cudaSuccess;
}

// The prep kernel's LoRA tiles for one linear (rank r, down-projection A
// [r][k]) over x (bf16 [m][ldx], no noise): fills the fields of `pp` they use.
void lora_prep_params(PrepParams& pp, int64_t m, int64_t k, int r, const void* A, uint8_t* ws,
                      const LinearLayout& WL) {
  const int ranks[1] = {r};
  const LoraSplit ls = lora_split(m, k, ranks, 1);
  pp.M = static_cast<int>(m);
  pp.K = static_cast<int>(k);
  pp.cluster = ls.cluster;
  pp.groups = ls.groups;
  pp.lora_m_tiles = static_cast<int>((m + kLoraTileM - 1) / kLoraTileM);
  pp.tile_begin[0] = 0;
  for (int i = 0; i < kMaxLinears; ++i) {
    const bool on = i == 0;
    pp.A[i] = on ? static_cast<const __nv_bfloat16*>(A) : nullptr;
    pp.r[i] = on ? r : 0;
    pp.t[i] = reinterpret_cast<float*>(ws + WL.t[i]);
    pp.tf[i] = reinterpret_cast<float*>(ws + WL.tf[i]);
    pp.tile_begin[i + 1] = pp.tile_begin[i] + (on ? pp.lora_m_tiles * ((r + kLoraTileR - 1) / kLoraTileR) : 0);
  }
  pp.lora_tiles = pp.tile_begin[kMaxLinears];
  pp.tile_count = reinterpret_cast<unsigned*>(ws + WL.count);
  pp.sum_groups = lora_sum_in_prep(m) ? 1 : 0;
}

}  // namespace

// The LoRA split of a launch.  When the launch streams many weight stages
// per SM (a long main loop, e.g. gate + up or down), a prep CTA takes three
// chunks (four from 32 tokens) instead of two: fewer CTAs and fewer K groups
// (whose partial sums the MMA kernel stages in shared memory), later t, which
// the long main loop hides.  (Measured on the 7B launches: gate + up at 64
// tokens 50.9 -> 44.9 us, at 32 tokens 42.0 -> 40.7 us; with the prep grid
// sharing SMs, two chunks everywhere was 2% slower -- down then needs 16
// groups, whose staging shortens the MMA kernel's ring.  q, k, v and o keep
// two.)
LoraSplit launch_lora_split(const LinearArgs& a, const int* ranks) {
  int64_t stage_tiles = 0;
  for (int i = 0; i < a.nlin; ++i)
    stage_tiles += ((a.lin[i].n + kTileN - 1) / kTileN) * ((a.k + kRawK - 1) / kRawK);
  int chunks = stage_tiles < 8 * static_cast<int64_t>(sm_count()) ? 2 : (a.m >= 32 ? 4 : 3);
  LoraSplit L = lora_split(a.m, a.k, ranks, a.nlin, chunks);
  // Up to 32 tokens each SM holds one prep CTA beside its MMA CTA: more
  // chunks per LoRA CTA until the prep grid (row tasks + LoRA tiles) fits
  // one CTA per SM.
  if (a.m <= 32) {
    int ltiles = 0;
    for (int i = 0; i < a.nlin; ++i)
      if (ranks[i] > 0)
        ltiles += static_cast<int>((a.m + kLoraTileM - 1) / kLoraTileM) * ((ranks[i] + kLoraTileR - 1) / kLoraTileR);
    const int n_tok = static_cast<int>((a.m + 15) / 16 * 16);
    const int sms = sm_count();
    for (;;) {
      const int rows = (std::max(static_cast<int>(a.m), n_tok) + L.cluster - 1) / L.cluster * L.cluster;
      if (rows + ltiles * L.groups * L.cluster <= sms || L.groups == 1 || chunks >= 64) break;
      L = lora_split(a.m, a.k, ranks, a.nlin, ++chunks);
    }
  }
  return L;
}

LoraDown linear_lora_down(const LinearArgs& a, int i) {
  int ranks[kMaxLinears] = {0, 0, 0, 0};
  for (int j = 0; j < a.nlin; ++j)
    ranks[j] = (a.lin[j].r > 0 && a.lin[j].A != nullptr && a.lin[j].B != nullptr) ? a.lin[j].r : 0;
  const LinearLayout WL = linear_layout(a.m, a.k, ranks, a.nlin, a.rmsnorm);
  const uint8_t* ws = static_cast<const uint8_t*>(a.workspace);
  LoraDown d;
  if (lora_sum_in_prep(a.m)) {
    d.t = reinterpret_cast<const float*>(ws + WL.tf[i]);
    d.parts = 1;
  } else {
    d.t = reinterpret_cast<const float*>(ws + WL.t[i]);
    d.parts = launch_lora_split(a, ranks).groups;
  }
  d.part_stride = a.m * ranks[i];
  return d;
}

size_t lora_down_workspace_bytes(int64_t m, int64_t k, int r) {
  const LinearLayout WL = linear_layout(m, k, &r, 1, false);
  // Only the counters and t / tf of the layout are used; xs and rinv are not.
  return WL.total - (WL.t[0] - WL.xs);
}

qerl_status launch_lora_down(const void* x, int64_t m, int64_t k, int64_t ldx, const void* A, int r, void* workspace,
                             LoraDown* out, int* status, cudaStream_t s) {
  if (!kernel_attrs_ok()) return QERL_ERR_CUDA;
  LinearLayout WL = linear_layout(m, k, &r, 1, false);
  // Drop the unused staging regions: t / tf follow the counters directly.
  const size_t shift = WL.t[0] - WL.xs;
  for (int i = 0; i < kMaxLinears; ++i) {
    WL.t[i] -= shift;
    WL.tf[i] -= shift;
  }
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  PrepParams pp{};
  pp.x = static_cast<const __nv_bfloat16*>(x);
  pp.ldx = ldx;
  lora_prep_params(pp, m, k, r, A, ws, WL);
  pp.row_groups = 0;
  pp.status = status;
  out->t = pp.sum_groups ? pp.tf[0] : pp.t[0];
  out->parts = pp.sum_groups ? 1 : pp.groups;
  out->part_stride = m * r;
  if (m == 0 || r == 0) return QERL_OK;
  if (lora_down_on_tc(m)) {  // the sum lands in tf (sum_groups holds for these m)
    const void* As[1] = {A};
    const int rs[1] = {r};
    float* ts[1] = {pp.tf[0]};
    float* tps[1] = {pp.t[0]};
    return lora_down_tc(x, ldx, m, k, As, rs, ts, tps, pp.groups, pp.tile_count, 1, status, s);
  }
  cudaLaunchConfig_t pc{};
  pc.gridDim = dim3(static_cast<unsigned>(pp.cluster), static_cast<unsigned>(pp.lora_tiles * pp.groups), 1);
  pc.blockDim = dim3(kPrepThreads, 1, 1);
  pc.dynamicSmemBytes = kLoraSmemBytes;
  pc.stream = s;
  cudaLaunchAttribute pa[1];
  pa[0].id = cudaLaunchAttributeClusterDimension;
  pa[0].val.clusterDim.x = static_cast<unsigned>(pp.cluster);
  pa[0].val.clusterDim.y = 1;
  pa[0].val.clusterDim.z = 1;
  pc.attrs = pa;
  pc.numAttrs = 1;
  return cudaLaunchKernelEx(&pc, prep_kernel, pp) == cudaSuccess ? QERL_OK : QERL_ERR_CUDA;
}

size_t linear_workspace_bytes(int64_t m, int64_t k, const int* ranks, int nlin, bool rmsnorm) {
  return linear_layout(m, k, ranks, nlin, rmsnorm).total;
}

qerl_status launch_rmsnorm_noise(const void* h, int64_t m, int64_t k, int64_t ldh, const void* w_norm, const float* Zn,
                                 double delta, void* out, int64_t ldo, cudaStream_t s) {
  if (m == 0 || k == 0) return QERL_OK;
  static std::once_flag once;
  static cudaError_t err = cudaSuccess;
  std::call_once(once, [] {
    err = cudaFuncSetAttribute(prep_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemLimit - 1024);
  });
  if (err != cudaSuccess) return QERL_ERR_CUDA;
  if (k * 2 > kSmemLimit - 1024) return QERL_ERR_UNSUPPORTED_SHAPE;
  PrepParams q{};
  q.x = static_cast<const __nv_bfloat16*>(h);
  q.ldx = ldh;
  q.M = static_cast<int>(m);
  q.K = static_cast<int>(k);
  q.rmsnorm = 1;
  q.w_norm = static_cast<const __nv_bfloat16*>(w_norm);
  q.Zn = Zn;
  q.delta = delta;
  q.xt_out = static_cast<__nv_bfloat16*>(out);
  q.ldo = ldo;
  q.cluster = 1;
  q.row_groups = static_cast<int>(m);
  cudaLaunchConfig_t pc{};
  pc.gridDim = dim3(1, static_cast<unsigned>(m), 1);
  pc.blockDim = dim3(kPrepThreads, 1, 1);
  pc.dynamicSmemBytes = static_cast<size_t>(k) * 2;
  pc.stream = s;
  return cudaLaunchKernelEx(&pc, prep_kernel, q) == cudaSuccess ? QERL_OK : QERL_ERR_CUDA;
}

qerl_status launch_lora_linear(const LinearArgs& a, cudaStream_t s) {
  const int M = static_cast<int>(a.m), K = static_cast<int>(a.k);
  const int nlin = a.nlin;
  if (nlin < 1 || nlin > kMaxLinears) return QERL_ERR_INVALID_ARGUMENT;
  // Token tiles: one of round_up(M, 16) rows up to 128 tokens, else 128-row
  // tiles (prefill: in pair mode each CTA's activation slab then serves 256
  // weight rows; a 256-token tile of one weight tile would need 1.5x the
  // activation bytes per MAC, and activation ingress into an SM is what
  // bounds these tiles).
  const int n_tok = M <= 128 ? (M + 15) / 16 * 16 : 128;
  const int m_tiles = M <= 128 ? 1 : (M + 127) / 128;
  const bool xs_rowmajor = M > 128;
  const int raw_total = (K + kRawK - 1) / kRawK;
  int ranks[kMaxLinears] = {0, 0, 0, 0};
  int tiles[kMaxLinears] = {0, 0, 0, 0};
  int r = 0;  // the largest rank: sizes the LoRA operand region
  int all_pairs = 0;
  for (int i = 0; i < nlin; ++i) {
    const LinearDesc& d = a.lin[i];
    ranks[i] = (d.r > 0 && d.A != nullptr && d.B != nullptr) ? d.r : 0;
    r = std::max(r, ranks[i]);
    tiles[i] = static_cast<int>((d.n + kTileN - 1) / kTileN);
    all_pairs += (tiles[i] + 1) / 2;
  }
  // K split across a cluster when the CTAs alone leave SMs idle: minimise
  // waves x weight stages per CTA, with a small per-CTA fixed cost.  A wave is
  // as many clusters as can be resident at once (clusters live inside one
  // GPC, so e.g. 7-CTA clusters leave SMs unused).
  // Coupled launches (up to 64 tokens, single tiles) share each SM with a
  // prep CTA.  Pair-mode launches (33-64 tokens) cannot: the prep grid holds
  // SMs until its LoRA tiles finish, so MMA CTAs beyond the free SMs start
  // only then.  When the chosen split does not fit the free SMs but a smaller one
  // does, at most twice the weight stages per CTA, the smaller one is taken:
  // every CTA then dequantizes ahead while prep runs (measured: the 7B o
  // launch at <= 16 tokens, 13.1 -> 12.2 us with 3-way instead of 5-way
  // splits).
  int prep_busy = 0;
  if (M > 32 && M <= 64 && r > 0) {  // up to 32 tokens the launch is coupled: prep runs beside it
    const LoraSplit ls0 = launch_lora_split(a, ranks);
    int ltiles = 0;
    for (int i = 0; i < nlin; ++i)
      if (ranks[i] > 0) ltiles += ((M + kLoraTileM - 1) / kLoraTileM) * ((ranks[i] + kLoraTileR - 1) / kLoraTileR);
    const int rows = (std::max(M, n_tok) + ls0.cluster - 1) / ls0.cluster * ls0.cluster;
    prep_busy = rows + ltiles * ls0.groups * ls0.cluster;
  }
  const int sms_all = sm_count();
  auto fits_beside_prep = [&](int units, int sp) {
    const int resident = resident_clusters(sp);
    return resident > 0 &&
           units * m_tiles <= static_cast<int64_t>(resident) * std::max(0, sms_all - prep_busy) / std::max(1, sms_all);
  };
  auto best_split = [&](int units) {
    if (m_tiles > 1) return 1;  // several token tiles fill the GPU without a K split
    int sp_best = 1;
    double best = 1e30;
    for (int sp = 1; sp <= kMaxSplit && sp <= raw_total; ++sp) {
      const int resident = resident_clusters(sp);
      if (resident <= 0) continue;
      const int waves = (units * m_tiles + resident - 1) / resident;
      const double cost = waves * (static_cast<double>((raw_total + sp - 1) / sp) + 1.5);
      if (cost < best - 1e-9) {
        best = cost;
        sp_best = sp;
      }
    }
    if (prep_busy > 0 && !fits_beside_prep(units, sp_best)) {
      const int stages_best = (raw_total + sp_best - 1) / sp_best;
      for (int sp = sp_best - 1; sp >= 1; --sp)
        if (fits_beside_prep(units, sp)) {
          if ((raw_total + sp - 1) / sp <= 2 * stages_best) sp_best = sp;
          break;
        }
    }
    return sp_best;
  };
  // Tiles above 32 tokens run in pair mode -- one CTA per two adjacent 128-row
  // weight tiles of a linear, sharing the activation slabs, with the
  // activation ring separate from the weights -- when each CTA then streams at
  // least 12 weight stages: half as many CTAs (one wave instead of two for the
  // 7B gate + up launch) and half the activation bytes per weight byte; its
  // fixed costs (two tiles' epilogue) are higher, and it cannot share SMs with
  // the prep grid.  (Measured: 6 stages made the 7B down launch 2-6 us slower
  // at 48-128 tokens, as 9-10-stage pair CTAs; gate + up keeps 14.)
  const int split_pair = n_tok > 32 && n_tok <= 128 ? best_split(all_pairs) : 1;
  const bool pair = n_tok > 32 && n_tok <= 128 && (raw_total + split_pair - 1) / split_pair >= 12;
  int tile_begin[kMaxLinears + 1] = {0, 0, 0, 0, 0};  // in grid-y units: tiles, or pairs of tiles
  for (int i = 0; i < nlin; ++i) tile_begin[i + 1] = tile_begin[i] + (pair ? (tiles[i] + 1) / 2 : tiles[i]);
  const bool lora = r > 0;
  const int n_tiles = tile_begin[nlin];  // grid-y units
  const LinearLayout WL = linear_layout(a.m, a.k, ranks, nlin, a.rmsnorm);
  uint8_t* ws = static_cast<uint8_t*>(a.workspace);
  int* status = reinterpret_cast<int*>(ws);
  __half* xs = reinterpret_cast<__half*>(ws + WL.xs);
  float* rinv = reinterpret_cast<float*>(ws + WL.rinv);
  const int sms = sm_count();

  if (!kernel_attrs_ok()) return QERL_ERR_CUDA;

  // ---- tile shape and pipeline depth (host-side checks before any launch)
  const int split = best_split(n_tiles);
  const int tpc = pair ? 2 : 1;  // weight tiles per CTA
  const uint32_t lb = lora_bytes(r, n_tok, tpc);
  // The LoRA operand is built early (its own region) up to 128 tokens: from
  // partial sums staged in shared memory, or in pair mode straight from
  // global memory by the idle issuer warps.
  const int t_groups = lora_sum_in_prep(M) ? 1 : launch_lora_split(a, ranks).groups;  // partial sums the MMA kernel adds
  const uint32_t tstage_bytes = (r > 0 && !pair) ? static_cast<uint32_t>(t_groups * n_tok * r * 4) : 0u;
  int lora_early = (r > 0 && n_tok <= 128) ? 1 : 0;
  const uint32_t part_bytes = split > 1 ? static_cast<uint32_t>(tpc * n_tok) * kTileN * 4u : 0u;
  const uint32_t b_stage = static_cast<uint32_t>(n_tok) * 128u;
  // The dequantized weights go to tensor memory as the MMA's A operand.
  // Each MMA occupies its issuing thread for ~150 cycles whatever the token
  // count, and each weight stage costs an issuer ~600 more cycles of waits,
  // fences and commits; so small tiles take more issuers, each with its own
  // accumulator (which tensor memory must hold next to the A ring, and which
  // the epilogue reads and adds).  Up to 64 tokens two groups of two issuers
  // take alternate weight stages (the 15-warp layout has four issuer warps).
  // Pair mode: one issuer per tile.
  const int issuers = pair ? 2 : (n_tok <= 64 ? 4 : 2);
  const uint32_t col_a = static_cast<uint32_t>(align_up(issuers * n_tok, 32));
  if (col_a > static_cast<uint32_t>(kTmemCols)) return QERL_ERR_UNSUPPORTED_SHAPE;
  // (Up to four weight stages; the barrier pairs are per weight stage, or
  // per (tile, MMA stage) in pair mode.)
  int ab_cap = std::min(pair ? kMaxAB : 4 * kSub, static_cast<int>((kTmemCols - col_a) / kAStageCols));
  // The ring is handed over a weight stage (kSub consecutive MMA stages) at
  // a time: a multiple of kSub.
  ab_cap -= ab_cap % kSub;
  if (pair) ab_cap = std::min(ab_cap, 2 * kSub);  // one slot per (tile, MMA stage)
  if (ab_cap < kSub) return QERL_ERR_UNSUPPORTED_SHAPE;
  struct Plan {
    uint32_t raw, b, lora, tstage, sm, bars, lut, total;
  };
  bool any_nf4 = false;
  for (int i = 0; i < nlin; ++i) any_nf4 = any_nf4 || a.lin[i].nf4;
  const uint32_t lut_bytes = any_nf4 ? 1024u : 0u;  // 256 fp16 pairs
  // Up to 64 tokens a weight stage's activation slabs (one bulk copy) sit in
  // the activation slot of its tensor-memory A stage and are released with it;
  // above, a separate activation ring holds one slab per slot.
  const int coupled = (n_tok <= 64 && !pair) ? 1 : 0;
  const uint32_t raw_b = coupled ? static_cast<uint32_t>(kSub) * b_stage : 0u;
  auto plan_for = [&](int rs, int bs) {
    Plan P;
    P.raw = 0;  // packed weight blocks (codes + scale pairs); 18 KB slots keep 1024-byte alignment
    P.b = P.raw + rs * tpc * kRawSlotBytes;
    uint32_t ring = P.b + (coupled ? static_cast<uint32_t>(ab_cap / kSub) * raw_b : bs * b_stage);
    if (!lora_early) ring = std::max(ring, lb);  // late LoRA tiles are built inside the ring
    ring = std::max(ring, part_bytes);
    P.lora = static_cast<uint32_t>(align_up(ring, 1024));
    P.tstage = P.lora + (lora_early ? lb : 0u);
    P.sm = static_cast<uint32_t>(align_up(P.tstage + (lora_early ? tstage_bytes : 0u), 16));
    P.bars = static_cast<uint32_t>(align_up(P.sm + static_cast<uint32_t>(n_tok) * 8u, 16));  // row scales, LoRA factors
    // + 1024-byte alignment slack; at least 116 KB so that two CTAs never share
    // an SM (each allocates all of tensor memory, and partners in a cluster
    // wait for one another).
    P.lut = P.bars + kBarBytes;
    P.total = std::max(P.lut + lut_bytes + 1024u, 118784u);
    return P;
  };
  const int ab_stages = ab_cap;
  int raw_stages = 0, b_stages = 0;
  // Coupled (up to 64 tokens) a prep CTA runs beside each MMA CTA: the ring
  // leaves room for its shared memory (dynamic + static) and both CTAs'
  // reserved kilobyte.
  size_t prep_smem_est = static_cast<size_t>(K) * 2;
  if (r > 0) prep_smem_est = std::max(prep_smem_est, static_cast<size_t>(kLoraSmemBytes));
  const uint32_t smem_cap = (coupled && prep_smem_est + 3072 < kSmemPerSm)
                                ? std::min<uint32_t>(kSmemLimit, kSmemPerSm - 3072u - static_cast<uint32_t>(prep_smem_est))
                                : static_cast<uint32_t>(kSmemLimit);
  {
    // A lives in tensor memory: keep its depth.  Mbarrier waits test a phase
    // parity, so every ring slot must always be waited on by the same thread
    // group in phase order (a waiter that is two phases ahead would pass
    // early): the weight ring has an even number of slots (the two dequant
    // groups take alternate stages, so each group owns the slots of its
    // parity) and the activation ring a multiple of kSub slabs (each issuer
    // owns fixed MMA stages of every weight stage).  Coupled: the deepest
    // weight ring.  Separate activation ring: at least four weight stages if
    // possible (blocks further ahead are prefetched into L2), then the
    // deepest activation ring.
    // (Pair mode: both dequant groups visit every weight slot in order, so
    // any depth >= 2 works.)
    auto max_rs = [&](int bs) {
      int rs = kMaxRaw;
      while (rs >= 2 && plan_for(rs, bs).total > smem_cap) --rs;
      return pair ? rs : rs & ~1;
    };
    int best_rs = 0, best_bs = 0;
    if (coupled) {
      best_bs = kSub;
      best_rs = max_rs(kSub);
    } else {
      // Pair mode: each slab waits for both tiles' MMAs before it is
      // refilled, so two weight stages of activations come first.  The ring
      // holds multiples of kSub slabs (each issuer owns fixed MMA stages).
      const int rs_pref = pair ? 2 : 4;
      for (int bs = 2 * kSub; bs >= kSub; bs -= kSub) {
        const int rs = max_rs(bs);
        if (rs >= 2 && (best_rs == 0 || std::min(rs, rs_pref) > std::min(best_rs, rs_pref))) {
          best_rs = rs;
          best_bs = bs;
        }
      }
    }
    raw_stages = best_rs;
    b_stages = best_bs;
  }
  if (lora_early && raw_stages < 2) {
    // Large rank: no room for a dedicated LoRA region; build the operand in
    // the idle ring after the mainloop instead.
    lora_early = 0;
    for (int bs = coupled ? kSub : 2 * kSub; bs >= kSub && raw_stages < 2; bs -= kSub) {
      int rs = kMaxRaw;
      while (rs >= 2 && plan_for(rs, bs).total > static_cast<uint32_t>(kSmemLimit)) --rs;
      if (!pair) rs &= ~1;
      if (rs >= 2) {
        raw_stages = rs;
        b_stages = bs;
      }
    }
  }
  if (raw_stages < 2) return QERL_ERR_UNSUPPORTED_SHAPE;
  // A weight stage is handed over (and its activations loaded) at once.
  if (ab_stages < 2 * kSub || ab_stages % kSub != 0 || b_stages < kSub || b_stages % kSub != 0 ||
      (!pair && raw_stages % 2 != 0) || (kSub * 4) % issuers != 0 || (!coupled && issuers > kSub) ||
      (pair && (issuers != 2 || ab_stages != 2 * kSub)) || (coupled && issuers > kCoupledWarps - 8 - kIssuerWarp0))
    return QERL_ERR_UNSUPPORTED_SHAPE;
  const Plan P = plan_for(raw_stages, b_stages);

  // x~: tiled layout moved by bulk copies; several 128-token tiles
  // read [M][K] through a 2D tensor map.
  CUtensorMap tm_xs;
  if (!xs_rowmajor) {
    std::memset(&tm_xs, 0, sizeof(tm_xs));
  } else if (!make_map_2d(&tm_xs, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, xs, static_cast<uint64_t>(K),
                          static_cast<uint64_t>(M), static_cast<uint64_t>(K) * 2, kStageK,
                          static_cast<uint32_t>(n_tok), CU_TENSOR_MAP_SWIZZLE_128B)) {
    return QERL_ERR_CUDA;
  }

  BtMaps tm_bls;
  std::memset(&tm_bls, 0, sizeof(tm_bls));
  for (int i = 0; i < nlin; ++i)
    if (ranks[i] > 0 &&
        !make_map_2d(&tm_bls.m[i], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, a.lin[i].B, static_cast<uint64_t>(ranks[i]),
                     static_cast<uint64_t>(a.lin[i].n), static_cast<uint64_t>(ranks[i]) * 2, kLoraChunkK, kTileN,
                     CU_TENSOR_MAP_SWIZZLE_128B))
      return QERL_ERR_CUDA;

  // ---- prep: noise + fp16 staging (+ LoRA down-projection)
  PrepParams pp{};
  pp.x = static_cast<const __nv_bfloat16*>(a.x);
  pp.z = a.z;
  pp.ldz = a.z != nullptr ? a.ldz : 0;
  pp.xs = xs;
  pp.rinv = rinv;
  pp.ldx = a.ldx;
  pp.M = M;
  pp.K = K;
  const LoraSplit ls = launch_lora_split(a, ranks);
  pp.cluster = lora ? ls.cluster : 1;
  pp.groups = lora ? ls.groups : 0;
  pp.tiled_rows = xs_rowmajor ? 0 : n_tok;
  pp.row_groups = (std::max(M, pp.tiled_rows) + pp.cluster - 1) / pp.cluster;
  pp.lora_m_tiles = (M + kLoraTileM - 1) / kLoraTileM;
  pp.tile_begin[0] = 0;
  for (int i = 0; i < kMaxLinears; ++i) {
    const bool on = i < nlin && ranks[i] > 0;
    pp.A[i] = on ? static_cast<const __nv_bfloat16*>(a.lin[i].A) : nullptr;
    pp.r[i] = on ? ranks[i] : 0;
    pp.t[i] = reinterpret_cast<float*>(ws + WL.t[i]);
    pp.tf[i] = reinterpret_cast<float*>(ws + WL.tf[i]);
    pp.tile_begin[i + 1] = pp.tile_begin[i] + (on ? pp.lora_m_tiles * ((ranks[i] + kLoraTileR - 1) / kLoraTileR) : 0);
  }
  pp.lora_tiles = pp.tile_begin[kMaxLinears];
  pp.tile_count = reinterpret_cast<unsigned*>(ws + WL.count);
  pp.status = status;
  pp.sum_groups = lora_sum_in_prep(M) ? 1 : 0;
  size_t prep_smem = static_cast<size_t>(K) * 2;  // row tasks stage the row
  if (lora) prep_smem = std::max(prep_smem, static_cast<size_t>(kLoraSmemBytes));
  if (prep_smem > static_cast<size_t>(kPrepSmemLimit)) return QERL_ERR_UNSUPPORTED_SHAPE;
  auto launch_prep = [&](const PrepParams& q, int row_groups, int lora_ctas_y, int cluster) {
    cudaLaunchConfig_t pc{};
    pc.gridDim = dim3(static_cast<unsigned>(cluster), static_cast<unsigned>(row_groups + lora_ctas_y), 1);
    pc.blockDim = dim3(kPrepThreads, 1, 1);
    pc.dynamicSmemBytes = prep_smem;
    pc.stream = s;
    cudaLaunchAttribute pa[1];
    pa[0].id = cudaLaunchAttributeClusterDimension;
    pa[0].val.clusterDim.x = static_cast<unsigned>(cluster);
    pa[0].val.clusterDim.y = 1;
    pa[0].val.clusterDim.z = 1;
    pc.attrs = pa;
    pc.numAttrs = 1;
    return cudaLaunchKernelEx(&pc, prep_kernel, q) == cudaSuccess;
  };
  const bool tc_lora = lora && lora_down_on_tc(M);
  auto down_tc = [&](const void* xsrc, int64_t ld) {
    const void* As[kMaxLinears] = {nullptr, nullptr, nullptr, nullptr};
    for (int i = 0; i < nlin; ++i) As[i] = a.lin[i].A;
    return lora_down_tc(xsrc, ld, M, K, As, ranks, pp.tf, pp.t, pp.groups, pp.tile_count, nlin, status, s);
  };
  if (tc_lora) {
    // Row tasks (noise or RMSNorm, fp16 staging; x~ in bf16 when it differs
    // from x), then the down-projection on the tensor cores; its sums go
    // where the consumers of summed partials read them (tf).
    PrepParams rq = pp;
    rq.lora_tiles = 0;
    if (a.rmsnorm) {
      rq.rmsnorm = 1;
      rq.w_norm = static_cast<const __nv_bfloat16*>(a.w_norm);
      rq.Zn = a.Zn;
      rq.delta = a.delta;
      rq.z = nullptr;
      rq.ldz = 0;
      rq.cluster = 1;
      rq.row_groups = std::max(M, pp.tiled_rows);
    }
    const bool own_xt = a.rmsnorm || a.z != nullptr;
    rq.xt_out = own_xt ? reinterpret_cast<__nv_bfloat16*>(ws + WL.xt) : nullptr;
    rq.ldo = K;
    if (!launch_prep(rq, rq.row_groups, 0, rq.cluster)) return QERL_ERR_CUDA;
    const qerl_status st = own_xt ? down_tc(ws + WL.xt, K) : down_tc(a.x, a.ldx);
    if (st != QERL_OK) return st;
  } else if (a.rmsnorm) {
    // RMSNorm with merged noise: the row tasks normalise h into x~ (staged for
    // the MMA kernel, and written out for the LoRA down-projection), then a
    // second launch runs the LoRA tiles on that x~ with no further noise.
    PrepParams rq = pp;
    rq.rmsnorm = 1;
    rq.w_norm = static_cast<const __nv_bfloat16*>(a.w_norm);
    rq.Zn = a.Zn;
    rq.delta = a.delta;
    rq.xt_out = lora ? reinterpret_cast<__nv_bfloat16*>(ws + WL.xt) : nullptr;
    rq.ldo = K;
    rq.z = nullptr;
    rq.ldz = 0;
    rq.cluster = 1;
    rq.row_groups = std::max(M, pp.tiled_rows);
    rq.lora_tiles = 0;
    if (!launch_prep(rq, rq.row_groups, 0, 1)) return QERL_ERR_CUDA;
    if (lora) {
      PrepParams lq = pp;
      lq.x = rq.xt_out;
      lq.ldx = K;
      lq.z = nullptr;
      lq.ldz = 0;
      lq.row_groups = 0;
      if (!launch_prep(lq, 0, pp.lora_tiles * pp.groups, pp.cluster)) return QERL_ERR_CUDA;
    }
  } else if (!launch_prep(pp, pp.row_groups, pp.lora_tiles * pp.groups, pp.cluster)) {
    return QERL_ERR_CUDA;
  }

  MmaParams mp{};
  mp.xs = xs;
  mp.rinv = rinv;
  mp.nlin = nlin;
  for (int i = 0; i < nlin; ++i) {
    LinearSlot& L = mp.lin[i];
    L.wpacked = a.lin[i].wpacked;
    L.tensor_scale = a.lin[i].tensor_scale;
    L.t = pp.sum_groups ? pp.tf[i] : pp.t[i];  // the summed down-projection, or its group partials
    L.y = a.lin[i].y;
    L.N = static_cast<int>(a.lin[i].n);
    L.r = ranks[i];
    L.y_f32 = a.lin[i].y_f32 ? 1 : 0;
    L.tile_begin = tile_begin[i];
    L.lora_scale = ranks[i] > 0 ? a.lin[i].alpha / static_cast<float>(ranks[i]) : 0.0f;
    L.nf4 = a.lin[i].nf4 ? 1 : 0;
  }
  if (any_nf4) {
    const Nf4Tables& nt = nf4_tables();
    for (int j = 0; j < 16; ++j)
      mp.nf4_half[j] = __half_as_ushort(__float2half_rn(static_cast<float>(nt.level[j])));
    mp.off_lut = P.lut;
  }
  mp.status = status;
  mp.M = M;
  mp.K = K;
  mp.n_tok = n_tok;
  mp.split = split;
  mp.raw_stages = raw_stages;
  mp.ab_stages = ab_stages;
  mp.b_stages = b_stages;
  mp.coupled = coupled;
  mp.raw_b_bytes = raw_b;
  mp.issuers = issuers;
  mp.n_warps = coupled ? kCoupledWarps : kMmaThreads / 32;
  mp.acts_ready = tc_lora ? 1 : 0;  // prep, then the down-projection, then this kernel
  mp.w_evict_first = m_tiles == 1 ? 1 : 0;
  mp.t_groups = pp.sum_groups ? 1 : pp.groups;  // == t_groups
  mp.col_a = col_a;
  mp.off_raw = P.raw;
  mp.off_b = P.b;
  mp.off_lora = P.lora;
  mp.off_tstage = P.tstage;
  mp.off_sm = P.sm;
  mp.off_bars = P.bars;
  mp.lora_early = lora_early;
  mp.wave = (split == 1 && !pair) ? sms : 0;
  mp.stage_out = static_cast<uint32_t>(tpc * n_tok) * kTileN * 4u <= P.lora ? 1 : 0;
  mp.pair = pair ? 1 : 0;
  mp.xs_rowmajor = xs_rowmajor ? 1 : 0;
  mp.wt = a.wt ? 1 : 0;

  const uint32_t smem_bytes = P.total;

  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(static_cast<unsigned>(split), static_cast<unsigned>(n_tiles), static_cast<unsigned>(m_tiles));
  cfg.blockDim = dim3(static_cast<unsigned>(32 * mp.n_warps), 1, 1);
  cfg.dynamicSmemBytes = smem_bytes;
  cfg.stream = s;
  cudaLaunchAttribute attrs[2];
  attrs[0].id = cudaLaunchAttributeClusterDimension;
  attrs[0].val.clusterDim.x = static_cast<unsigned>(split);
  attrs[0].val.clusterDim.y = 1;
  attrs[0].val.clusterDim.z = 1;
  attrs[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attrs[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attrs;
  cfg.numAttrs = 2;
  const cudaError_t le =
      coupled ? (a.wt ? cudaLaunchKernelEx(&cfg, mma_kernel<1, 1>, tm_xs, tm_bls, mp)
                      : cudaLaunchKernelEx(&cfg, mma_kernel<1, 0>, tm_xs, tm_bls, mp))
              : (a.wt ? cudaLaunchKernelEx(&cfg, mma_kernel<0, 1>, tm_xs, tm_bls, mp)
                      : cudaLaunchKernelEx(&cfg, mma_kernel<0, 0>, tm_xs, tm_bls, mp));
  if (le != cudaSuccess) return QERL_ERR_CUDA;
  return QERL_OK;
}

}  // namespace qerl

#ifdef QERL_TEST_HOOKS
// Test-only entry point of the hooks build: the bounded waits' limit in clock
// cycles, and whether the accumulator barrier gets an arrival that never comes
// (the epilogue's wait then runs out after every MMA and copy has completed).
extern "C" __attribute__((visibility("default"))) int qerl_test_set_hooks(long long wait_limit_cycles,
                                                                         int extra_arrival) {
  if (cudaMemcpyToSymbol(qerl::g_test_wait_limit, &wait_limit_cycles, sizeof(wait_limit_cycles)) != cudaSuccess)
    return 1;
  if (cudaMemcpyToSymbol(qerl::g_test_extra_arrival, &extra_arrival, sizeof(extra_arrival)) != cudaSuccess) return 1;
  return 0;
}
#endif
