// rz_math.cuh -- small device helpers shared by the loss kernels: the
// importance weight, the per-token D3 term and fixed-order reductions.
#pragma once

#include <cstdint>

namespace rz {

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

// w = pi/mu = exp(log pi - log mu), never clipped.
__device__ __forceinline__ float is_weight(float logpi, float logmu) {
  return expf(logpi - logmu);
}

// Per-token D3 term  w - 1 - log w  with w = e^x (so log w = x exactly):
// e^x - 1 - x.  For |x| <= 1/2 the Taylor series
//   e^x - 1 - x = x^2 (1/2! + x/3! + x^2/4! + ... + x^7/9!)
// avoids the cancellation of e^x - 1 against x (truncation error below
// 3e-9 relative); beyond that expm1(x) - x loses no significant digits.
__device__ __forceinline__ float d3_term(float x) {
  if (fabsf(x) <= 0.5f) {
    float p = 1.0f / 362880.0f;
    p = fmaf(p, x, 1.0f / 40320.0f);
    p = fmaf(p, x, 1.0f / 5040.0f);
    p = fmaf(p, x, 1.0f / 720.0f);
    p = fmaf(p, x, 1.0f / 120.0f);
    p = fmaf(p, x, 1.0f / 24.0f);
    p = fmaf(p, x, 1.0f / 6.0f);
    p = fmaf(p, x, 0.5f);
    return x * x * p;
  }
  return expm1f(x) - x;
}

// Deterministic block sum: butterfly within each warp, then the warp totals
// in warp order by thread 0.  Result valid in thread 0 only.
template <typename Tv, int kThreadsPerBlock>
__device__ __forceinline__ Tv block_sum(Tv v, Tv* scratch /* >= kThreadsPerBlock/32 */) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  const int warp = threadIdx.x >> 5;
  if ((threadIdx.x & 31) == 0) scratch[warp] = v;
  __syncthreads();
  Tv tot = Tv(0);
  if (threadIdx.x == 0) {
#pragma unroll 1
    for (int w = 0; w < kThreadsPerBlock / 32; ++w) tot += scratch[w];
  }
  __syncthreads();
  return tot;
}

// Block max / min (thread 0 holds the result).
template <int kThreadsPerBlock, bool kMax>
__device__ __forceinline__ float block_extreme(float v, float* scratch) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float u = __shfl_xor_sync(0xffffffffu, v, o);
    v = kMax ? fmaxf(v, u) : fminf(v, u);
  }
  const int warp = threadIdx.x >> 5;
  if ((threadIdx.x & 31) == 0) scratch[warp] = v;
  __syncthreads();
  float r = scratch[0];
  if (threadIdx.x == 0) {
    for (int w = 1; w < kThreadsPerBlock / 32; ++w)
      r = kMax ? fmaxf(r, scratch[w]) : fminf(r, scratch[w]);
  }
  __syncthreads();
  return r;
}

// Merge two (max in log2 units, sum of 2^(x - max)) pairs.
__device__ __forceinline__ void lse2_merge(float& m, float& s, float m_o, float s_o) {
  if (m_o > m) {
    s = s * exp2f(m - m_o) + s_o;
    m = m_o;
  } else if (m_o > -INFINITY) {
    s = s + s_o * exp2f(m_o - m);
  }
}

}  // namespace rz
