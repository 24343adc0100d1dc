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
// state (m = max z so far, s = sum 2^((z - m) log2 e)).  z - m is exact for
// the maximum itself, whose term is exactly 1.  The caller guarantees at
// least one finite logit.  With kKeep the 32 terms 2^((z - m) log2 e), taken
// against the updated m, are also returned in e (0 past V); the state is
// computed by the very same operations either way.  The steps are also
// used one by one, over many chunks at once, by the decode-mode fold: the
// chunk's maximum, the factor that rescales s when the maximum grows, and
// the chunk's sum against the updated maximum.
__device__ __forceinline__ float fold32_max(const float (&v)[32]) {
  float mx[4] = {v[0], v[1], v[2], v[3]};
#pragma unroll
  for (int j = 4; j < 32; j += 4) {
    mx[0] = fmaxf(mx[0], v[j]);
    mx[1] = fmaxf(mx[1], v[j + 1]);
    mx[2] = fmaxf(mx[2], v[j + 2]);
    mx[3] = fmaxf(mx[3], v[j + 3]);
  }
  return fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3]));
}

// The factor s is multiplied by when the maximum grows from m to cm.
__device__ __forceinline__ float fold32_scale(float m, float cm) {
  return ex2_approx(__fmul_rn(__fsub_rn(m, cm), kLog2e));
}

__device__ __forceinline__ void fold32_rescale(float& m, float& s, float cm) {
  if (cm > m) {
    s = __fmul_rn(s, fold32_scale(m, cm));
    m = cm;
  }
}

template <bool kKeep>
__device__ __forceinline__ float fold32_sum(const float (&v)[32], float m, float (&e)[32],
                                            float (&acc)[4]) {
#pragma unroll
  for (int q = 0; q < 4; ++q) acc[q] = 0.f;
#pragma unroll
  for (int j = 0; j < 32; ++j) {
    const float t = ex2_approx(__fmul_rn(__fsub_rn(v[j], m), kLog2e));
    if (kKeep) e[j] = t;
    acc[j & 3] = __fadd_rn(acc[j & 3], t);
  }
  return __fadd_rn(__fadd_rn(acc[0], acc[1]), __fadd_rn(acc[2], acc[3]));
}

template <bool kKeep>
__device__ __forceinline__ void lse_fold32_impl(float& m, float& s, const float (&v)[32],
                                                float (&e)[32], float (&acc)[4], float& w) {
  fold32_rescale(m, s, fold32_max(v));
  w = fold32_sum<kKeep>(v, m, e, acc);
  s = __fadd_rn(s, w);
}

__device__ __forceinline__ void lse_fold32(float& m, float& s, const float (&v)[32]) {
  float unused[32], acc[4], w;
  lse_fold32_impl<false>(m, s, v, unused, acc, w);
}

__device__ __forceinline__ void lse_fold32_keep(float& m, float& s, const float (&v)[32],
                                                float (&e)[32]) {
  float acc[4], w;
  lse_fold32_impl<true>(m, s, v, e, acc, w);
}

// The same fold, also returning the terms e, their sums over the four
// classes of columns j mod 4 (acc) and the chunk's total w (the amount added
// to s): what the fused sampler draws from.
__device__ __forceinline__ void lse_fold32_terms(float& m, float& s, const float (&v)[32],
                                                 float (&e)[32], float (&acc)[4], float& w) {
  lse_fold32_impl<true>(m, s, v, e, acc, w);
}

// Merge the partial states of a row in a fixed order.  P is any struct with
// .x = m and .y = s (float2, float4).  Returns M = max m and sets *sum to the
// row's sum 2^((z - M) log2 e) over the whole vocabulary.
// The merge's two steps are also taken apart by the decode-mode kernels,
// which evaluate the splits' factors on the lanes of a warp at once: the
// maximum over the states in order, and the factor of a state against it.
template <class P>
__device__ __forceinline__ float lse_merge_max(const P* pp, int S) {
  float M = -INFINITY;
  for (int g = 0; g < S; ++g) M = fmaxf(M, pp[g].x);
  return M;
}
__device__ __forceinline__ float lse_merge_factor(float m, float M) {
  return exp2f(__fmul_rn(__fsub_rn(m, M), kLog2e));
}
template <class P>
__device__ __forceinline__ float lse_merge_parts(const P* pp, int S, float* sum) {
  const float M = lse_merge_max(pp, S);
  float acc = 0.f;
  for (int g = 0; g < S; ++g) acc = fmaf(pp[g].y, lse_merge_factor(pp[g].x, M), acc);
  *sum = acc;
  return M;
}

// log pi = (z_a - M) - ln(sum): exactly 0 when a is the only token, and
// logsumexp = M + ln(sum).
__device__ __forceinline__ float logprob_from(float za, float M, float sum) {
  return __fsub_rn(__fsub_rn(za, M), __fmul_rn(log2f(sum), kLn2));
}
__device__ __forceinline__ float lse_from(float M, float sum) {
  return __fadd_rn(M, __fmul_rn(log2f(sum), kLn2));
}

}  // namespace rz
