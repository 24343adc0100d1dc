// rz_lse.cuh -- the per-row log-sum-exp arithmetic shared by every kernel
// that produces a logprob (the rollout logprob, the learner's forward pass
// and the fused sampler).  Written once, with explicit rounding intrinsics
// (no compiler-chosen FMA contraction), so that all of them produce the same
// float for the same row: the "diff 0" property between rollout and learner
// ("Zero Mismatch" post, s.5).
#pragma once

#include <cmath>
#include <cstdint>

#include "rz_math.cuh"
#include "rz_ptx.cuh"

namespace rz {

// Fold 32 logits (natural units; -inf marks a column past V) into the running
// base-2 state (m2 = max z*log2(e), s = sum 2^(z*log2(e) - m2)).  The caller
// guarantees at least one finite logit.
__device__ __forceinline__ void lse_fold32(float& m2, float& s, const float (&v)[32]) {
  float mx[4] = {v[0], v[1], v[2], v[3]};
#pragma unroll
  for (int j = 4; j < 32; j += 4) {
    mx[0] = fmaxf(mx[0], v[j]);
    mx[1] = fmaxf(mx[1], v[j + 1]);
    mx[2] = fmaxf(mx[2], v[j + 2]);
    mx[3] = fmaxf(mx[3], v[j + 3]);
  }
  const float cm2 = __fmul_rn(fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3])), kLog2e);
  if (cm2 > m2) {
    s = __fmul_rn(s, ex2_approx(__fsub_rn(m2, cm2)));
    m2 = cm2;
  }
  const float nm = -m2;
  float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
  for (int j = 0; j < 32; ++j) acc[j & 3] = __fadd_rn(acc[j & 3], ex2_approx(fmaf(v[j], kLog2e, nm)));
  s = __fadd_rn(s, __fadd_rn(__fadd_rn(acc[0], acc[1]), __fadd_rn(acc[2], acc[3])));
}

// Merge the S split states of a row in split order -> log2-sum-exp.
// P is any struct with .x = m2 and .y = s (float2, float4).
template <class P>
__device__ __forceinline__ float lse2_of_splits(const P* pp, int S) {
  float M = -INFINITY;
  for (int g = 0; g < S; ++g) M = fmaxf(M, pp[g].x);
  float sum = 0.f;
  for (int g = 0; g < S; ++g) sum = fmaf(pp[g].y, exp2f(__fsub_rn(pp[g].x, M)), sum);
  return __fadd_rn(M, log2f(sum));
}

// log pi = z_a - lse, lse = lse2 * ln 2.
__device__ __forceinline__ float logprob_from(float za, float lse2) {
  return __fsub_rn(za, __fmul_rn(lse2, kLn2));
}

}  // namespace rz
