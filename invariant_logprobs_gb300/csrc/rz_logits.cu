// rz_logits.cu -- the given-logits variant: per row of bf16 logits, the
// log-softmax normaliser, the sampled token's logprob, the unclipped ratio
// and the dlogits c_t (softmax - onehot), written back over the logits.
//
// Purely bandwidth-bound (no contraction): one CTA streams one row with
// 16-byte loads, four in flight per thread.  Pass 1 computes (max, sum exp)
// online and keeps the first 96 KB of the row in shared memory; pass 2
// re-reads the rest (mostly from L2) and overwrites the row with dz.  Two
// CTAs of 768 threads per SM keep ~304 rows in flight, their re-read parts
// inside the L2.
// The loss and D3 over all rows are then reduced by the same fixed-order
// kernels as the hidden-state path.
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>

#include "rz_check.cuh"
#include "rz_internal.h"
#include "rz_math.cuh"
#include "rz_ptx.cuh"

namespace rz {

namespace {

constexpr int kRowThreads = 768;
constexpr int kRowsPerSm = 2;
// 96 KB of each row kept in shared memory: two rows per SM in flight, and
// the rest of their rows (re-read in pass 2, ~208 KB each at V = 151936,
// ~63 MB over 304 rows) stays in the L2.  Measured per 262,144-row step at
// V = 151936: 512 threads, 64 KB stash, three rows per SM: 27.5 ms; 768
// threads, 96 KB, two rows: 26.2 ms.  With 768 threads the time is touchy
// in the stash size: 80 KB 30.0 ms, 88 KB 27.5 ms, 104 KB 30.2 ms; forcing
// the shared-memory carveout to its maximum makes 96 KB take 30.5 ms, and
// predicating the last four-wide round instead of finishing with single
// loads 30.4 ms.
constexpr int kStashVec = 6144;
constexpr size_t kRowSmem = kStashVec * sizeof(uint4);

// L2 eviction priorities: the part of a row that pass 2 will read again from
// L2 is loaded evict-last; everything read for the last time, and the dz
// written back, is evict-first, so the rows in flight keep their second
// halves resident in the 129 MB L2.
__device__ __forceinline__ float bf_lo(uint32_t x) { return __uint_as_float(x << 16); }
__device__ __forceinline__ float bf_hi(uint32_t x) { return __uint_as_float(x & 0xffff0000u); }

// Online (m, s): m = the largest logit so far (natural units, an exact
// logit value), s = sum 2^((z - m) log2 e).  z - m is taken first, so the
// maximum's own term is exactly 1 and a peaked row keeps its precision.
__device__ __forceinline__ void fold8(const uint4& q, float& m, float& s) {
  const float v[8] = {bf_lo(q.x), bf_hi(q.x), bf_lo(q.y), bf_hi(q.y),
                      bf_lo(q.z), bf_hi(q.z), bf_lo(q.w), bf_hi(q.w)};
  const float cm = fmaxf(fmaxf(fmaxf(v[0], v[1]), fmaxf(v[2], v[3])),
                         fmaxf(fmaxf(v[4], v[5]), fmaxf(v[6], v[7])));
  if (cm > m) {
    s *= ex2_approx((m - cm) * kLog2e);
    m = cm;
  }
  float a0 = 0.f, a1 = 0.f;
#pragma unroll
  for (int j = 0; j < 8; j += 2) {
    a0 += ex2_approx((v[j] - m) * kLog2e);
    a1 += ex2_approx((v[j + 1] - m) * kLog2e);
  }
  s += a0 + a1;
}

// Merge two (m, s) states of fold8.
__device__ __forceinline__ void lse_merge_nat(float& m, float& s, float m_o, float s_o) {
  if (m_o > m) {
    s = s * ex2_approx((m - m_o) * kLog2e) + s_o;
    m = m_o;
  } else if (m_o > -INFINITY) {
    s = s + s_o * ex2_approx((m_o - m) * kLog2e);
  }
}

// dz of 8 columns: c p_v = c 2^((z_v - M) log2 e - log2 S), and at the
// sampled column c expm1(log pi) (no cancellation of p - 1 as p -> 1).
__device__ __forceinline__ uint4 dz8(const uint4& q, float M, float nl2s, float c,
                                     float c_onehot, int rel) {
  const float v[8] = {bf_lo(q.x), bf_hi(q.x), bf_lo(q.y), bf_hi(q.y),
                      bf_lo(q.z), bf_hi(q.z), bf_lo(q.w), bf_hi(q.w)};
  float g[8];
#pragma unroll
  for (int j = 0; j < 8; ++j) g[j] = c * ex2_approx(fmaf(v[j] - M, kLog2e, nl2s));
  if (static_cast<unsigned>(rel) < 8u) {
#pragma unroll
    for (int j = 0; j < 8; ++j)
      if (rel == j) g[j] = c_onehot;
  }
  uint4 o;
  o.x = pack_bf16x2(g[0], g[1]);
  o.y = pack_bf16x2(g[2], g[3]);
  o.z = pack_bf16x2(g[4], g[5]);
  o.w = pack_bf16x2(g[6], g[7]);
  return o;
}

__global__ void __launch_bounds__(kRowThreads, kRowsPerSm)  // <= 42 registers
    logits_row_kernel(uint16_t* __restrict__ logits, long long T, int V,
                      const int32_t* __restrict__ tokens, const float* __restrict__ logmu,
                      const int64_t* __restrict__ cu, const float2* __restrict__ fac,
                      const uint8_t* __restrict__ mask, int B, float* __restrict__ logprob,
                      int* err) {
  extern __shared__ uint4 stash[];
  __shared__ float red_m[kRowThreads / 32], red_s[kRowThreads / 32];
  __shared__ float bc[4];
  __shared__ int bci;
  const long long row = blockIdx.x;
  uint4* rowp = reinterpret_cast<uint4*>(logits + row * static_cast<long long>(V));
  const int nvec = V >> 3;
  const int nstash = nvec < kStashVec ? nvec : kStashVec;

  const uint64_t keep = l2_policy_last();
  const uint64_t drop = l2_policy_first();

  // ---- pass 1: online (max, sum exp)
  float m2 = -INFINITY, s = 0.f;
  int i = threadIdx.x;
  // four independent 16-byte loads in flight per thread
  for (; i + 3 * kRowThreads < nvec; i += 4 * kRowThreads) {
    uint4 q[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int ii = i + u * kRowThreads;
      q[u] = ld_l2hint(rowp + ii, ii < nstash ? drop : keep);
    }
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      if (i + u * kRowThreads < nstash) stash[i + u * kRowThreads] = q[u];
      fold8(q[u], m2, s);
    }
  }
  for (; i < nvec; i += kRowThreads) {
    const uint4 q0 = ld_l2hint(rowp + i, i < nstash ? drop : keep);
    if (i < nstash) stash[i] = q0;
    fold8(q0, m2, s);
  }
  // warp butterfly merge, then warps in order
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float mo = __shfl_xor_sync(0xffffffffu, m2, o);
    const float so = __shfl_xor_sync(0xffffffffu, s, o);
    lse_merge_nat(m2, s, mo, so);
  }
  const int warp = threadIdx.x >> 5;
  if ((threadIdx.x & 31) == 0) {
    red_m[warp] = m2;
    red_s[warp] = s;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    float M = red_m[0], S = red_s[0];
    for (int w = 1; w < kRowThreads / 32; ++w) lse_merge_nat(M, S, red_m[w], red_s[w]);
    const float log2s = log2f(S);
    const int a = tokens[row];
    float lp, c = 0.f;
    if (a < 0 || a >= V) {
      lp = __int_as_float(0x7fc00000);
      if (err) atomicOr(err, 1);
    } else {
      const uint16_t zb = logits[row * static_cast<long long>(V) + a];
      // log pi = (z_a - M) - ln S: z_a - M is exact, so a peaked row's
      // log pi near 0 keeps its relative precision
      lp = (__uint_as_float(static_cast<uint32_t>(zb) << 16) - M) - log2s * kLn2;
      // response of this row: the last i with cu[i] <= row
      int lo = 0, hi = B;  // invariant cu[lo] <= row < cu[hi]
      while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (cu[mid] <= row) lo = mid;
        else hi = mid;
      }
      // c_t = A_i w_t / (B T_i); 0 for a masked (non-action) token
      const bool act = !mask || mask[row] != 0;
      // same factors and rounding as the hidden-state learner:
      // fac[i] = (A_i, 1/(B T_i)), c = A_i w_t (1/(B T_i))
      c = act ? fac[lo].x * is_weight(lp, logmu[row]) * fac[lo].y : 0.f;
    }
    logprob[row] = lp;
    bc[0] = M;
    bc[1] = -log2s;
    bc[2] = c;
    bc[3] = c * expm1f(lp);  // 0 for a masked token; unused for a bad one
    bci = a;
  }
  __syncthreads();
  const float M = bc[0];
  const float nl2s = bc[1];
  const float c = bc[2];
  const float c1 = bc[3];
  const int a = bci;

  // ---- pass 2: dz = c (softmax - onehot), in place.  The part re-read from
  // L2 goes first and backwards (most recently loaded lines first); the
  // stashed head comes from shared memory.
  const int R = nvec - nstash;
  int k = threadIdx.x;
  for (; k + 3 * kRowThreads < R; k += 4 * kRowThreads) {
    uint4 q[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) q[u] = ld_l2hint(rowp + (nvec - 1 - (k + u * kRowThreads)), drop);
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int jj = nvec - 1 - (k + u * kRowThreads);
      if (!RZ_DCHECK(jj >= nstash && jj < nvec, 20)) continue;
      st_l2hint(rowp + jj, dz8(q[u], M, nl2s, c, c1, a - 8 * jj), drop);
    }
  }
  for (; k < R; k += kRowThreads) {
    const int jj = nvec - 1 - k;
    st_l2hint(rowp + jj, dz8(ld_l2hint(rowp + jj, drop), M, nl2s, c, c1, a - 8 * jj), drop);
  }
  for (int j = threadIdx.x; j < nstash; j += kRowThreads)
    if (RZ_DCHECK(j < kStashVec && j < nvec, 21))
      st_l2hint(rowp + j, dz8(stash[j], M, nl2s, c, c1, a - 8 * j), drop);
}

}  // namespace

cudaError_t check_read_logits(unsigned int* count, int* site) {
#ifdef RZ_CHECKS
  return check_read_and_clear(count, site);
#else
  *count = 0;
  *site = 0;
  return cudaSuccess;
#endif
}

cudaError_t launch_logits_rows(uint16_t* logits, int64_t T, int V, const int32_t* tokens,
                               const float* logmu, const int64_t* cu, const float2* fac,
                               const uint8_t* mask, int B, float* logprob, int* err,
                               cudaStream_t st) {
  if (T <= 0) return cudaSuccess;
  cudaError_t e = cudaFuncSetAttribute(logits_row_kernel,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(kRowSmem));
  if (e != cudaSuccess) return e;
  logits_row_kernel<<<static_cast<unsigned>(T), kRowThreads, kRowSmem, st>>>(
      logits, T, V, tokens, logmu, cu, fac, mask, B, logprob, err);
  return cudaGetLastError();
}

}  // namespace rz
