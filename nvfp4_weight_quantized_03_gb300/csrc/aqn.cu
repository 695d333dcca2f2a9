// aqn.cu -- Adaptive Quantization Noise: the sigma schedule (host) and the
// channel-wise Gaussian sampler (device).
//
// QeRL digest, section 3.4 "Adaptive Quantization Noise (AQN)": Eq. 7
// (Z ~ N(0, sigma^2 I), one value per input channel of the layer, resampled
// per forward pass), Eq. 8 (sigma(k) = sigma_start (sigma_end/sigma_start)^((k-1)/(K-1)),
// k = 1..K) and "Algorithm 1" (K stages of floor(M/K) steps, a warm-up
// stage with sigma = 0).  The digest does not name a generator; this library
// uses Philox4x32-10 (Salmon, Moraes, Dror, Shaw, SC'11) with Box-Muller.
#include <cmath>

#include "qerl_internal.h"

namespace qerl {
namespace {

// Philox4x32 with 10 rounds: per round two 32x32->64 products of the even
// counter words with the round multipliers, the high halves XORed with the
// odd words and the key; the key advances by the Weyl increments.
__device__ __forceinline__ uint4 philox4x32_10(uint4 c, uint2 key) {
  constexpr uint32_t kMul0 = 0xD2511F53u, kMul1 = 0xCD9E8D57u;
  constexpr uint32_t kWeyl0 = 0x9E3779B9u, kWeyl1 = 0xBB67AE85u;
#pragma unroll
  for (int round = 0; round < 10; ++round) {
    const uint32_t hi0 = __umulhi(kMul0, c.x), lo0 = kMul0 * c.x;
    const uint32_t hi1 = __umulhi(kMul1, c.z), lo1 = kMul1 * c.z;
    c = make_uint4(hi1 ^ c.y ^ key.x, lo1, hi0 ^ c.w ^ key.y, lo0);
    key.x += kWeyl0;
    key.y += kWeyl1;
  }
  return c;
}

// One thread per Box-Muller pair: pair p covers channels 2p, 2p+1 and uses
// words (x, y) or (z, w) of the Philox block of counter index p / 2.  fp64
// transcendental throughput per SM is low, so blocks are small and spread the
// pairs over many SMs.
__global__ void aqn_sample_kernel(float* __restrict__ z, int64_t k, float sigma, uint64_t seed, uint32_t stream_id,
                                  uint64_t counter) {
  const int64_t pair = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (2 * pair >= k) return;
  const int64_t i = pair >> 1;
  const uint4 bits = philox4x32_10(
      make_uint4(static_cast<uint32_t>(i), stream_id, static_cast<uint32_t>(counter),
                 static_cast<uint32_t>(counter >> 32)),
      make_uint2(static_cast<uint32_t>(seed), static_cast<uint32_t>(seed >> 32)));
  constexpr double kInv32 = 1.0 / 4294967296.0;
  constexpr double kTwoPi = 6.283185307179586476925286766559;
  const uint32_t w0 = (pair & 1) ? bits.z : bits.x;
  const uint32_t w1 = (pair & 1) ? bits.w : bits.y;
  const double ua = (static_cast<double>(w0) + 0.5) * kInv32;
  const double ub = (static_cast<double>(w1) + 0.5) * kInv32;
  const double rho = sqrt(-2.0 * log(ua));
  const double sd = static_cast<double>(sigma);
  z[2 * pair] = static_cast<float>(sd * (rho * cos(kTwoPi * ub)));
  if (2 * pair + 1 < k) z[2 * pair + 1] = static_cast<float>(sd * (rho * sin(kTwoPi * ub)));
}

}  // namespace

qerl_status launch_aqn_sample(float* z, int64_t k, float sigma, uint64_t seed, uint32_t stream_id,
                              uint64_t counter, cudaStream_t s) {
  if (k == 0) return QERL_OK;
  const int64_t pairs = (k + 1) / 2;
  const int threads = 32;
  const int64_t blocks = (pairs + threads - 1) / threads;
  aqn_sample_kernel<<<static_cast<unsigned>(blocks), threads, 0, s>>>(z, k, sigma, seed, stream_id, counter);
  return cuda_status(cudaGetLastError());
}

}  // namespace qerl

extern "C" double qerl_aqn_sigma(int stage, int num_stages, double sigma_start, double sigma_end) {
  if (stage < 0) return 0.0;  // Algorithm 1 warm-up: quantization noise only
  if (num_stages <= 1) return sigma_start;
  if (stage >= num_stages) stage = num_stages - 1;
  const double expo = static_cast<double>(stage) / static_cast<double>(num_stages - 1);  // (k-1)/(K-1)
  return sigma_start * std::pow(sigma_end / sigma_start, expo);
}

// The four decay schedules the digest compares in section 3.4 ("Why
// exponential decay") and in its ablation (Figures 9 and 15), over the same
// stages: with k = stage + 1 and u = (k-1)/(K-1),
//   exponential  sigma_start * (sigma_end / sigma_start)^u           (Eq. 8)
//   linear       sigma_start - (sigma_start - sigma_end) * u
//   cosine       sigma_end + (sigma_start - sigma_end) * (1 + cos(pi u)) / 2
//   logarithmic  sigma_start - (sigma_start - sigma_end) * log(k) / log(K)
extern "C" double qerl_aqn_sigma_schedule(int schedule, int stage, int num_stages, double sigma_start,
                                          double sigma_end) {
  if (schedule < QERL_SCHEDULE_EXPONENTIAL || schedule > QERL_SCHEDULE_LOGARITHMIC) return std::nan("");
  if (stage < 0) return 0.0;
  if (num_stages <= 1) return sigma_start;
  if (stage >= num_stages) stage = num_stages - 1;
  const double span = sigma_start - sigma_end;
  const double u = static_cast<double>(stage) / static_cast<double>(num_stages - 1);
  switch (schedule) {
    case QERL_SCHEDULE_LINEAR:
      return sigma_start - span * u;
    case QERL_SCHEDULE_COSINE:
      return sigma_end + span * (1.0 + std::cos(M_PI * u)) / 2.0;
    case QERL_SCHEDULE_LOGARITHMIC:
      return sigma_start - span * std::log(static_cast<double>(stage + 1)) / std::log(static_cast<double>(num_stages));
    default:
      return qerl_aqn_sigma(stage, num_stages, sigma_start, sigma_end);
  }
}

extern "C" int qerl_aqn_stage(int64_t step, int64_t total_steps, int num_stages) {
  if (num_stages <= 0 || step < 0) return -1;
  int64_t steps_per_stage = total_steps / num_stages;
  if (steps_per_stage < 1) steps_per_stage = 1;
  const int64_t st = step / steps_per_stage;
  return st >= num_stages ? num_stages - 1 : static_cast<int>(st);
}
