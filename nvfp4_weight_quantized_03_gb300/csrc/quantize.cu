// quantize.cu -- NVFP4 quantizer kernels (QeRL digest, section 3.4 "NVFP4
// Quantization": E2M1 elements, one E4M3 scale per 16 contiguous elements,
// one FP32 tensor scale; Eq. 6 is the decoder this encoder inverts).
//
// Two streaming passes over W (HBM-bound):
//   1. amax_kernel  : max |w| over the tensor as fp32 bit patterns.  For
//      non-negative floats the unsigned order equals the float order and
//      NaN/Inf sort above every finite value, so one atomicMax per CTA both
//      reduces and flags non-finite input.
//   2. encode_kernel: per 16-element block: amax_b, E4M3 block scale, the
//      decoded scale times S, 16 E2M1 codes packed two per byte.  Every fp32
//      operation is a single IEEE RN operation (__fdiv_rn / __fmul_rn) in the
//      documented order, so codes and scales are bit-reproducible.
#include <cuda_bf16.h>

#include <cmath>

#include "qerl_internal.h"
#include "qerl_ptx.cuh"

namespace qerl {
namespace {

constexpr int kThreads = 256;

__device__ __forceinline__ unsigned abs_bits_f32(uint32_t w) { return w & 0x7FFFFFFFu; }
__device__ __forceinline__ unsigned abs_bits_bf16(uint32_t h) { return (h & 0x7FFFu) << 16; }

__device__ __forceinline__ unsigned max_bits_of_vec(uint4 v, bool bf16) {
  uint32_t w[4] = {v.x, v.y, v.z, v.w};
  unsigned m = 0;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    if (bf16) {
      m = max(m, abs_bits_bf16(w[i] & 0xFFFFu));
      m = max(m, abs_bits_bf16(w[i] >> 16));
    } else {
      m = max(m, abs_bits_f32(w[i]));
    }
  }
  return m;
}

// Rows are strided over CTAs, 16-byte vectors over threads.
__global__ void __launch_bounds__(kThreads) amax_kernel(const uint8_t* __restrict__ W, int64_t n,
                                                        int64_t row_vecs, int64_t ld_bytes, bool bf16,
                                                        unsigned* __restrict__ amax_bits) {
  unsigned m = 0;
  for (int64_t row = blockIdx.x; row < n; row += gridDim.x) {
    const uint4* p = reinterpret_cast<const uint4*>(W + row * ld_bytes);
    for (int64_t v = threadIdx.x; v < row_vecs; v += kThreads) m = max(m, max_bits_of_vec(__ldg(p + v), bf16));
  }
  m = __reduce_max_sync(0xFFFFFFFFu, m);
  __shared__ unsigned red[kThreads / 32];
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = m;
  __syncthreads();
  if (threadIdx.x < 32) {
    unsigned v = threadIdx.x < kThreads / 32 ? red[threadIdx.x] : 0u;
    v = __reduce_max_sync(0xFFFFFFFFu, v);
    if (threadIdx.x == 0 && v != 0u) atomicMax(amax_bits, v);
  }
}

// One thread per 16-element block; threads of a warp cover consecutive blocks
// of a row, so loads (64 B or 32 B per thread) and the 8-byte code stores are
// contiguous across the warp.
// NF4 mode (nf4.on): the level range is 1 instead of 6 -- S = amax / 448,
// block scale E4M3(amax_b / S) -- and an element's code is the number of
// level midpoints (fp32, ascending) at or below w / (S dec(s)).
struct Nf4Mids {
  float mid[15];
  int on;
};

__global__ void __launch_bounds__(kThreads) encode_kernel(const uint8_t* __restrict__ W, int64_t n, int64_t k,
                                                          int64_t ld_bytes, bool bf16,
                                                          const unsigned* __restrict__ amax_bits,
                                                          const float* __restrict__ s_in, float* __restrict__ s_out,
                                                          uint8_t* __restrict__ codes, uint8_t* __restrict__ scales,
                                                          int* __restrict__ status, const Nf4Mids nf4) {
  float S;
  if (s_in != nullptr) {
    S = *s_in;
    if (!(S > 0.0f) || !isfinite(S)) {
      if (blockIdx.x == 0 && threadIdx.x == 0) record_error(status, isfinite(S) ? 1 : 6);
      return;
    }
  } else {
    const unsigned ab = *amax_bits;
    if (ab >= 0x7F800000u) {  // NaN or Inf somewhere in W
      if (blockIdx.x == 0 && threadIdx.x == 0) {
        record_error(status, 6);
        *s_out = __uint_as_float(0x7FC00000u);
      }
      return;
    }
    S = __fdiv_rn(__uint_as_float(ab), nf4.on ? 448.0f : 2688.0f);  // amax / (level range * 448)
    if (S == 0.0f) S = 1.0f;
    if (blockIdx.x == 0 && threadIdx.x == 0 && s_out != nullptr) *s_out = S;
  }

  const int64_t nb = k / 16;
  for (int64_t row = blockIdx.x; row < n; row += gridDim.x) {
    const uint8_t* rowp = W + row * ld_bytes;
    for (int64_t b = threadIdx.x; b < nb; b += kThreads) {
      float w[16];
      if (bf16) {
        const uint4* p = reinterpret_cast<const uint4*>(rowp) + 2 * b;
        uint4 v0 = __ldg(p), v1 = __ldg(p + 1);
        uint32_t u[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          w[2 * i] = __uint_as_float(u[i] << 16);
          w[2 * i + 1] = __uint_as_float(u[i] & 0xFFFF0000u);
        }
      } else {
        const float4* p = reinterpret_cast<const float4*>(rowp) + 4 * b;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          float4 v = __ldg(p + i);
          w[4 * i] = v.x;
          w[4 * i + 1] = v.y;
          w[4 * i + 2] = v.z;
          w[4 * i + 3] = v.w;
        }
      }
      unsigned mb = 0;
#pragma unroll
      for (int i = 0; i < 16; ++i) mb = max(mb, __float_as_uint(w[i]) & 0x7FFFFFFFu);
      if (mb >= 0x7F800000u) {  // only reachable with a caller-given scale
        record_error(status, 6);
        continue;
      }
      const float rb = nf4.on ? __fdiv_rn(__uint_as_float(mb), S) : __fdiv_rn(__fdiv_rn(__uint_as_float(mb), 6.0f), S);
      const uint32_t sb = f32_to_e4m3_satfinite(rb);
      const float dec = __half2float(__low2half(e4m3x2_to_half2(sb)));
      const float sc = __fmul_rn(S, dec);
      uint32_t packed[2] = {0u, 0u};
      if (nf4.on) {
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          uint32_t c = 7u;  // zero
          if (sc != 0.0f) {
            const float q = __fdiv_rn(w[i], sc);
            c = 0u;
#pragma unroll
            for (int j = 0; j < 15; ++j) c += nf4.mid[j] <= q ? 1u : 0u;
          }
          packed[i >> 3] |= c << (4 * (i & 7));
        }
      } else if (sc != 0.0f) {
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          uint32_t byte = f32x2_to_e2m1x2_satfinite(__fdiv_rn(w[2 * i], sc), __fdiv_rn(w[2 * i + 1], sc));
          if ((byte & 0x07u) == 0u) byte &= 0xF0u;  // a zero magnitude is +0 (code 0x0)
          if ((byte & 0x70u) == 0u) byte &= 0x0Fu;
          packed[i >> 2] |= byte << (8 * (i & 3));
        }
      }
      *reinterpret_cast<uint2*>(codes + row * (k / 2) + b * 8) = make_uint2(packed[0], packed[1]);
      scales[row * nb + b] = static_cast<uint8_t>(sb);
    }
  }
}

__global__ void amax_to_float_kernel(const unsigned* amax_bits, float* amax) { *amax = __uint_as_float(*amax_bits); }

// S from an amax the caller combined (e.g. the max over the shards of a
// tensor): the rule of the quantizer's own prologue, bit for bit.
__global__ void tensor_scale_kernel(const float* amax, float* S) {
  const float a = *amax;
  if (!(a >= 0.0f) || !isfinite(a)) {
    *S = __uint_as_float(0x7FC00000u);
    return;
  }
  float s = __fdiv_rn(a, 2688.0f);  // amax / (6 * 448)
  if (s == 0.0f) s = 1.0f;
  *S = s;
}

int grid_for_rows(int64_t n) {
  int dev = 0, sms = 148;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  int64_t g = sms * 8;
  if (g > n) g = n;
  return g < 1 ? 1 : static_cast<int>(g);
}

// Packed (kernel-native) weight layout for the linear: one contiguous
// 18432-byte block per (128-row tile t, 256-wide K stage g), blocks in
// (t, g) order.  Block bytes [0, 16384): row r's 128 code bytes (K range
// g*256 .. +255, two codes per byte, even k in the low nibble) at r * 128,
// 16-byte chunk c stored at chunk position c ^ (r % 8).  Bytes [16384, 18432):
// E4M3 scale pair p (16-blocks 2p, 2p+1 of the stage) of row r at
// 16384 + p * 256 + r * 2.  Rows >= n and K past k are zero.
__global__ void __launch_bounds__(kThreads) pack_kernel(const uint8_t* __restrict__ codes,
                                                         const uint8_t* __restrict__ scales, int n, int k,
                                                         uint8_t* __restrict__ packed) {
  const int g = blockIdx.x, t = blockIdx.y;
  const int kg = gridDim.x;
  uint8_t* blk = packed + (static_cast<int64_t>(t) * kg + g) * kPackedBlockBytes;
  const int row_bytes = k / 2, srow_bytes = k / 16;
  for (int idx = threadIdx.x; idx < 128 * 8; idx += kThreads) {
    const int r = idx >> 3, c = idx & 7;
    const int nrow = t * 128 + r;
    const int off = g * 128 + c * 16;
    uint4 v = make_uint4(0u, 0u, 0u, 0u);
    if (nrow < n && off < row_bytes) v = __ldg(reinterpret_cast<const uint4*>(codes + static_cast<int64_t>(nrow) * row_bytes + off));
    *reinterpret_cast<uint4*>(blk + r * 128 + ((c ^ (r & 7)) << 4)) = v;
  }
  for (int idx = threadIdx.x; idx < 8 * 128; idx += kThreads) {
    const int pr = idx >> 7, r = idx & 127;
    const int nrow = t * 128 + r;
    const int off = g * 16 + 2 * pr;
    unsigned short v = 0;
    if (nrow < n && off < srow_bytes)
      v = __ldg(reinterpret_cast<const unsigned short*>(scales + static_cast<int64_t>(nrow) * srow_bytes + off));
    *reinterpret_cast<unsigned short*>(blk + 16384 + pr * 256 + r * 2) = v;
  }
}

// ---------------------------------------------------------------------------
// MXFP4 (the 4-bit format the digest's "NVFP4 Quantization" section compares
// with): E2M1 elements and one E8M0 scale X = 2^e per 32 contiguous elements,
// no tensor scale.  The digest does not fix the scale rule; this follows the
// OCP MX one, e = floor(log2(amax_b)) - 2 clamped to [-127, 127] (2 is the
// largest E2M1 exponent, so the block max lands in [4, 8) X and values above
// 6 X saturate), code e + 127, an all-zero block code 0.  w / X is exact
// (a power-of-two scaling; a result below 2^-126 encodes to 0 either way).
// One thread per 32-element block; a warp covers consecutive blocks of a row.
__global__ void __launch_bounds__(kThreads) mx_encode_kernel(const uint8_t* __restrict__ W, int64_t n, int64_t k,
                                                             int64_t ld_bytes, bool bf16,
                                                             uint8_t* __restrict__ codes,
                                                             uint8_t* __restrict__ scales, int* __restrict__ status) {
  const int64_t nb = k / 32;
  for (int64_t row = blockIdx.x; row < n; row += gridDim.x) {
    const uint8_t* rowp = W + row * ld_bytes;
    for (int64_t b = threadIdx.x; b < nb; b += kThreads) {
      float w[32];
      if (bf16) {
        const uint4* p = reinterpret_cast<const uint4*>(rowp) + 4 * b;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const uint4 v = __ldg(p + q);
          const uint32_t u[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            w[8 * q + 2 * i] = __uint_as_float(u[i] << 16);
            w[8 * q + 2 * i + 1] = __uint_as_float(u[i] & 0xFFFF0000u);
          }
        }
      } else {
        const float4* p = reinterpret_cast<const float4*>(rowp) + 8 * b;
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          const float4 v = __ldg(p + q);
          w[4 * q] = v.x;
          w[4 * q + 1] = v.y;
          w[4 * q + 2] = v.z;
          w[4 * q + 3] = v.w;
        }
      }
      unsigned mb = 0;
#pragma unroll
      for (int i = 0; i < 32; ++i) mb = max(mb, __float_as_uint(w[i]) & 0x7FFFFFFFu);
      if (mb >= 0x7F800000u) {
        record_error(status, 6);
        continue;
      }
      int e = -127;
      if (mb != 0u) {
        const int bexp = static_cast<int>(mb >> 23);
        const int fl = bexp > 0 ? bexp - 127 : (31 - __clz(static_cast<int>(mb))) - 149;  // floor(log2(amax))
        e = min(max(fl - 2, -127), 127);
      }
      // 2^-e for e in [-127, 125] is a normal float.
      const float inv = __uint_as_float(static_cast<uint32_t>(127 - e) << 23);
      uint32_t packed[4] = {0u, 0u, 0u, 0u};
      if (mb != 0u) {
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          uint32_t byte = f32x2_to_e2m1x2_satfinite(__fmul_rn(w[2 * i], inv), __fmul_rn(w[2 * i + 1], inv));
          if ((byte & 0x07u) == 0u) byte &= 0xF0u;  // a zero magnitude is +0 (code 0x0)
          if ((byte & 0x70u) == 0u) byte &= 0x0Fu;
          packed[i >> 2] |= byte << (8 * (i & 3));
        }
      }
      *reinterpret_cast<uint4*>(codes + row * (k / 2) + b * 16) = make_uint4(packed[0], packed[1], packed[2], packed[3]);
      scales[row * nb + b] = static_cast<uint8_t>(e + 127);
    }
  }
}

__device__ __forceinline__ bool any_magnitude(uint4 v) { return ((v.x | v.y | v.z | v.w) & 0x77777777u) != 0u; }

// Largest E8M0 code over the 32-blocks holding a non-zero code, plus one (0:
// no such block), into *emax1 (zeroed by the caller).
__global__ void __launch_bounds__(kThreads) mx_emax_kernel(const uint8_t* __restrict__ codes,
                                                           const uint8_t* __restrict__ scales, int64_t n, int64_t k,
                                                           unsigned* __restrict__ emax1) {
  const int64_t nb = k / 32;
  unsigned m = 0;
  for (int64_t row = blockIdx.x; row < n; row += gridDim.x)
    for (int64_t b = threadIdx.x; b < nb; b += kThreads)
      if (any_magnitude(__ldg(reinterpret_cast<const uint4*>(codes + row * (k / 2) + b * 16))))
        m = max(m, static_cast<unsigned>(scales[row * nb + b]) + 1u);
  m = __reduce_max_sync(0xFFFFFFFFu, m);
  if ((threadIdx.x & 31) == 0 && m != 0u) atomicMax(emax1, m);
}

// MXFP4 -> the linear's packed layout.  The kernel decodes E4M3 block scales
// times one fp32 tensor scale, so a power-of-two block scale 2^(e-127) is
// written as S * 2^d with S = 2^(e_ref - 127), e_ref = e_max - 8, and the E4M3
// code of 2^d (d = e - e_ref in [-9, 8]: E4M3 holds those powers exactly,
// 2^-9 .. 2^-7 as subnormals), the same code in both 16-element slots of the
// 32-block.  The product is the MXFP4 value exactly.  A non-zero block with
// d < -9 (a block scale more than 2^17 below the weight's largest) does not
// fit: it is written as zero and the call records QERL_ERR_RANGE.
__global__ void __launch_bounds__(kThreads) mx_pack_kernel(const uint8_t* __restrict__ codes,
                                                           const uint8_t* __restrict__ scales, int n, int k,
                                                           const unsigned* __restrict__ emax1,
                                                           uint8_t* __restrict__ packed, float* __restrict__ S_out,
                                                           int* __restrict__ status) {
  const int g = blockIdx.x, t = blockIdx.y;
  const int kg = gridDim.x;
  const unsigned em1 = *emax1;
  const int e_ref = em1 == 0u ? 127 : static_cast<int>(em1) - 1 - 8;
  if (g == 0 && t == 0 && threadIdx.x == 0) {
    const int se = e_ref - 127;  // in [-135, 119]
    *S_out = em1 == 0u ? 1.0f
                       : __uint_as_float(se >= -126 ? static_cast<uint32_t>(se + 127) << 23 : 1u << (se + 149));
  }
  if (n == 0 || k == 0) return;  // an empty weight: only S
  uint8_t* blk = packed + (static_cast<int64_t>(t) * kg + g) * kPackedBlockBytes;
  const int row_bytes = k / 2, srow = k / 32;
  for (int idx = threadIdx.x; idx < 128 * 8; idx += kThreads) {
    const int r = idx >> 3, c = idx & 7;
    const int nrow = t * 128 + r;
    const int off = g * 128 + c * 16;  // chunk c is 32-block g * 8 + c
    uint4 v = make_uint4(0u, 0u, 0u, 0u);
    unsigned short sv = 0;
    if (nrow < n && off < row_bytes) {
      v = __ldg(reinterpret_cast<const uint4*>(codes + static_cast<int64_t>(nrow) * row_bytes + off));
      if (any_magnitude(v)) {
        const int d = static_cast<int>(scales[static_cast<int64_t>(nrow) * srow + g * 8 + c]) - e_ref;
        if (d < -9) {
          record_error(status, QERL_ERR_RANGE);
          v = make_uint4(0u, 0u, 0u, 0u);
        } else {
          const unsigned c4 = d >= -6 ? static_cast<unsigned>(d + 7) << 3 : 1u << (d + 9);
          sv = static_cast<unsigned short>(c4 | (c4 << 8));
        }
      }
    }
    *reinterpret_cast<uint4*>(blk + r * 128 + ((c ^ (r & 7)) << 4)) = v;
    *reinterpret_cast<unsigned short*>(blk + 16384 + c * 256 + r * 2) = sv;
  }
}

// The transposed packed layout (the weight's transpose, for the input
// gradient dx~ = dy . W_hat, whose contraction runs along W's n): one
// 18432-byte block per (128-row tile t over k, 256-wide stage g over n),
// blocks in (t, g) order.  Bytes [0, 16384): for row kk of the tile (k =
// 128 t + kk), the 128 code bytes of n in [256 g, 256 g + 256), n even in the
// low nibble, 16-byte chunk c at position c ^ (kk % 8).  Bytes [16384,
// 18432): the E4M3 scale of (n, k) -- scales[n][k / 16], shared by the 16
// rows of a row group -- at 16384 + (kk / 16) * 256 + (n - 256 g).  Rows
// past k and n past the weight are zero.  The codes of the stage are first
// gathered into shared memory (256 n x 64 bytes), then re-paired along n.
__global__ void __launch_bounds__(kThreads) pack_t_kernel(const uint8_t* __restrict__ codes,
                                                           const uint8_t* __restrict__ scales, int n, int k,
                                                           uint8_t* __restrict__ packed) {
  __shared__ __align__(16) uint8_t sm[256 * 64];
  const int g = blockIdx.x, t = blockIdx.y;
  const int kg = gridDim.x;
  uint8_t* blk = packed + (static_cast<int64_t>(t) * kg + g) * kPackedBlockBytes;
  const int row_bytes = k / 2, srow = k / 16;
  for (int idx = threadIdx.x; idx < 256 * 4; idx += kThreads) {
    const int nl = idx >> 2, c = idx & 3;
    const int nn = g * 256 + nl;
    const int off = t * 64 + c * 16;
    uint4 v = make_uint4(0u, 0u, 0u, 0u);
    if (nn < n && off < row_bytes)
      v = __ldg(reinterpret_cast<const uint4*>(codes + static_cast<int64_t>(nn) * row_bytes + off));
    *reinterpret_cast<uint4*>(sm + nl * 64 + c * 16) = v;
  }
  __syncthreads();
  for (int idx = threadIdx.x; idx < 128 * 8; idx += kThreads) {
    const int kk = idx >> 3, c = idx & 7;
    const int shift = 4 * (kk & 1);
    uint32_t w[4] = {0u, 0u, 0u, 0u};
#pragma unroll
    for (int j = 0; j < 16; ++j) {  // output byte j of the chunk: n = 32 c + 2 j, 2 j + 1
      const uint32_t lo = (sm[(32 * c + 2 * j) * 64 + (kk >> 1)] >> shift) & 0xFu;
      const uint32_t hi = (sm[(32 * c + 2 * j + 1) * 64 + (kk >> 1)] >> shift) & 0xFu;
      w[j >> 2] |= (lo | (hi << 4)) << (8 * (j & 3));
    }
    *reinterpret_cast<uint4*>(blk + kk * 128 + ((c ^ (kk & 7)) << 4)) = make_uint4(w[0], w[1], w[2], w[3]);
  }
  for (int idx = threadIdx.x; idx < 8 * 256; idx += kThreads) {
    const int rg = idx >> 8, nl = idx & 255;
    const int nn = g * 256 + nl, sc = t * 8 + rg;
    blk[16384 + rg * 256 + nl] = (nn < n && sc < srow) ? scales[static_cast<int64_t>(nn) * srow + sc] : 0;
  }
}

}  // namespace

qerl_status launch_pack_t(const uint8_t* codes, const uint8_t* scales, int64_t n, int64_t k, uint8_t* packed,
                          cudaStream_t s) {
  const dim3 grid(static_cast<unsigned>((n + 255) / 256), static_cast<unsigned>((k + 127) / 128));
  pack_t_kernel<<<grid, kThreads, 0, s>>>(codes, scales, static_cast<int>(n), static_cast<int>(k), packed);
  return cuda_status(cudaGetLastError());
}

qerl_status launch_mx_encode(const void* W, bool bf16, int64_t n, int64_t k, int64_t ld_w, uint8_t* codes,
                             uint8_t* scales, int* status, cudaStream_t s) {
  if (n == 0 || k == 0) return QERL_OK;
  const int64_t esz = bf16 ? 2 : 4;
  mx_encode_kernel<<<grid_for_rows(n), kThreads, 0, s>>>(static_cast<const uint8_t*>(W), n, k, ld_w * esz, bf16,
                                                          codes, scales, status);
  return cuda_status(cudaGetLastError());
}

qerl_status launch_mx_pack(const uint8_t* codes, const uint8_t* scales, int64_t n, int64_t k, uint8_t* packed,
                           float* tensor_scale, unsigned* emax1, int* status, cudaStream_t s) {
  mx_emax_kernel<<<grid_for_rows(n), kThreads, 0, s>>>(codes, scales, n, k, emax1);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return QERL_ERR_CUDA;
  const dim3 grid(static_cast<unsigned>(n > 0 && k > 0 ? (k + 255) / 256 : 1),
                  static_cast<unsigned>(n > 0 && k > 0 ? (n + 127) / 128 : 1));
  mx_pack_kernel<<<grid, kThreads, 0, s>>>(codes, scales, static_cast<int>(n), static_cast<int>(k), emax1, packed,
                                           tensor_scale, status);
  return cuda_status(cudaGetLastError());
}

size_t packed_weight_bytes(int64_t n, int64_t k) {
  return static_cast<size_t>((n + 127) / 128) * static_cast<size_t>((k + 255) / 256) * kPackedBlockBytes;
}

qerl_status launch_pack(const uint8_t* codes, const uint8_t* scales, int64_t n, int64_t k, uint8_t* packed,
                        cudaStream_t s) {
  const dim3 grid(static_cast<unsigned>((k + 255) / 256), static_cast<unsigned>((n + 127) / 128));
  pack_kernel<<<grid, kThreads, 0, s>>>(codes, scales, static_cast<int>(n), static_cast<int>(k), packed);
  return cuda_status(cudaGetLastError());
}

qerl_status launch_amax(const void* W, bool bf16, int64_t n, int64_t k, int64_t ld_w, unsigned* amax_bits,
                        cudaStream_t s) {
  if (n == 0 || k == 0) return QERL_OK;
  const int64_t esz = bf16 ? 2 : 4;
  amax_kernel<<<grid_for_rows(n), kThreads, 0, s>>>(static_cast<const uint8_t*>(W), n, k * esz / 16, ld_w * esz,
                                                     bf16, amax_bits);
  return cuda_status(cudaGetLastError());
}

qerl_status launch_encode(const void* W, bool bf16, int64_t n, int64_t k, int64_t ld_w,
                          const unsigned* amax_bits, const float* s_in, float* s_out, uint8_t* codes,
                          uint8_t* scales, int* status, cudaStream_t s, bool nf4) {
  const int64_t esz = bf16 ? 2 : 4;
  Nf4Mids mids{};
  if (nf4) {
    const Nf4Tables& t = nf4_tables();
    for (int i = 0; i < 15; ++i) mids.mid[i] = t.mid[i];
    mids.on = 1;
  }
  encode_kernel<<<grid_for_rows(n > 0 ? n : 1), kThreads, 0, s>>>(static_cast<const uint8_t*>(W), n, k,
                                                                   ld_w * esz, bf16, amax_bits, s_in, s_out,
                                                                   codes, scales, status, mids);
  return cuda_status(cudaGetLastError());
}

// The NF4 levels (QLoRA's construction: normalised standard-normal quantiles
// at evenly spaced probabilities with an exact zero; see qerl.h), computed
// once in fp64 by Newton's method on Phi(x) = erfc(-x / sqrt 2) / 2, then the
// fp32 midpoints the encoder compares against and the fp16 levels the linear
// looks up.
const Nf4Tables& nf4_tables() {
  static Nf4Tables t = [] {
    auto ppf = [](double prob) {
      double x = 0.0;
      for (int it = 0; it < 100; ++it) {
        const double f = 0.5 * std::erfc(-x / std::sqrt(2.0)) - prob;
        const double d = std::exp(-0.5 * x * x) / std::sqrt(2.0 * 3.14159265358979323846);
        const double nx = x - f / d;
        if (nx == x) break;
        x = nx;
      }
      return x;
    };
    Nf4Tables r{};
    const double p = ((1.0 - 1.0 / 32.0) + (1.0 - 1.0 / 30.0)) / 2.0;
    const double top = ppf(p);
    double lv[16];
    for (int i = 1; i <= 7; ++i) lv[7 - i] = -ppf(0.5 + (i / 7.0) * (p - 0.5)) / top;
    lv[7] = 0.0;
    for (int i = 1; i <= 8; ++i) lv[7 + i] = ppf(0.5 + (i / 8.0) * (p - 0.5)) / top;
    lv[0] = -1.0;
    lv[15] = 1.0;
    for (int i = 0; i < 15; ++i) r.mid[i] = static_cast<float>((lv[i] + lv[i + 1]) / 2.0);
    for (int i = 0; i < 16; ++i) r.level[i] = lv[i];
    return r;
  }();
  return t;
}

qerl_status launch_tensor_scale(const float* amax, float* S, cudaStream_t s) {
  tensor_scale_kernel<<<1, 1, 0, s>>>(amax, S);
  return cuda_status(cudaGetLastError());
}

qerl_status launch_amax_to_float(const unsigned* amax_bits, float* amax, cudaStream_t s) {
  amax_to_float_kernel<<<1, 1, 0, s>>>(amax_bits, amax);
  return cuda_status(cudaGetLastError());
}

}  // namespace qerl
