// rz_loss.cu -- group advantages, the importance-sampled REINFORCE Zero loss
// with its per-token gradient coefficient, and the D3 diagnostic.
//
//   A_i  = r_i - mean of the rewards of i's group          (vLLM post s.4 item 3)
//   w_t  = exp(log pi_t - log mu_t), never clipped          (vLLM post s.4 item 2)
//   L    = -(1/B) sum_i (A_i/T_i) sum_{t in i} w_t          (project page s.02)
//   D3   = (1/T) sum_t (w_t - 1 - log w_t)                   (vLLM post s.3)
//   c_t  = A_i w_t / (B T_i) = -dL/dlog pi_t
//
// An optional action mask removes tokens from every sum ("T_i counts valid
// action tokens", project page s.02): T_i is the number of valid tokens of
// response i, D3 averages over valid tokens, and c_t = 0 for masked tokens.
//
// Numerics: w = 1 + expm1(log pi - log mu), so the loss is evaluated as
//   L = -(1/B) [ sum_i A_i  +  sum_i A_i (1/T_i) sum_t expm1(d_t) ]
// over responses with T_i > 0; the first sum is exact for centred rewards
// and the second keeps full relative precision of the (small) lag term.
// All reductions run in a fixed order: results are bitwise reproducible.
#include <cooperative_groups.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>

#include "rz_internal.h"
#include "rz_math.cuh"

namespace cg = cooperative_groups;

namespace rz {

namespace {

constexpr int kRespThreads = 256;
constexpr int kFinalThreads = 1024;
constexpr int kD3Threads = 1024;
// The whole-call reductions of rz_d3 and rz_is_stats run as one cluster of
// kStatBlocks CTAs: CTA r reduces tokens r*1024 + k*8192 + lane, then CTA 0
// adds the CTAs' partial sums in rank order through distributed shared
// memory.  The split depends on nothing but the token index, so the result
// is the same on every run.
constexpr int kStatBlocks = 8;

struct RespPart {
  double lag;   // A_i (1/T_i) sum_t expm1(d_t)
  double base;  // A_i if T_i > 0 else 0
  double d3;    // sum_t (w_t - 1 - log w_t)
  double cnt;   // T_i (valid tokens of the response)
};

// Valid tokens of response [s, e): all of them, or those with mask != 0.
__device__ __forceinline__ long long valid_count(const uint8_t* mask, long long s, long long e,
                                                 int* red) {
  if (!mask) return e - s;
  int c = 0;
  for (long long t = s + threadIdx.x; t < e; t += kRespThreads) c += mask[t] != 0;
  return block_sum<int, kRespThreads>(c, red);  // valid in thread 0
}

__global__ void __launch_bounds__(kRespThreads)
    is_loss_resp_kernel(const float* __restrict__ logpi, const float* __restrict__ logmu,
                        const int64_t* __restrict__ cu, const float* __restrict__ adv,
                        const uint8_t* __restrict__ mask, int B, int Bn, long long T,
                        float* __restrict__ coef, RespPart* __restrict__ part, int* err) {
  __shared__ float red[kRespThreads / 32];
  __shared__ int redi[kRespThreads / 32];
  __shared__ long long nvalid;
  const int i = blockIdx.x;
  long long s = cu[i];
  long long e = cu[i + 1];
  const bool bad = s < 0 || e < s || e > T || (i == 0 && s != 0) || (i == B - 1 && e != T);
  if (bad) {
    if (threadIdx.x == 0 && err) atomicOr(err, 2);
    if (s < 0 || s > T) s = 0;
    if (e < s || e > T) e = s;
  }
  const long long v = valid_count(mask, s, e, redi);
  if (threadIdx.x == 0) nvalid = v;
  __syncthreads();
  const long long Ti = nvalid;
  const float A = adv[i];
  const float inv_bt = Ti > 0 ? static_cast<float>(1.0 / (static_cast<double>(Bn) * Ti)) : 0.f;
  float em1 = 0.f, d3s = 0.f;
  for (long long t = s + threadIdx.x; t < e; t += kRespThreads) {
    const bool ok = !mask || mask[t] != 0;
    const float dl = logpi[t] - logmu[t];
    const float w = expf(dl);
    if (coef) coef[t] = ok ? A * w * inv_bt : 0.f;
    if (ok) {
      em1 += expm1f(dl);
      d3s += d3_term(dl);
    }
  }
  const float em1_tot = block_sum<float, kRespThreads>(em1, red);
  const float d3_tot = block_sum<float, kRespThreads>(d3s, red);
  if (threadIdx.x == 0) {
    RespPart r;
    r.lag = Ti > 0 ? static_cast<double>(A) * static_cast<double>(em1_tot) / static_cast<double>(Ti)
                   : 0.0;
    r.base = Ti > 0 ? static_cast<double>(A) : 0.0;
    r.d3 = static_cast<double>(d3_tot);
    r.cnt = static_cast<double>(Ti);
    part[i] = r;
  }
}

// Per-response factors (A_i, 1/(Bn T_i)) (second 0 for an empty response),
// from which the learner and the given-logits kernel form
// c_t = A_i w_t (1/(Bn T_i)) with the same rounding as is_loss_resp_kernel's
// coefficient.  Bn is the number of responses the loss averages over: B, or
// the whole batch's count when this call holds one shard of it.
__global__ void resp_factors_kernel(const int64_t* __restrict__ cu, const float* __restrict__ adv,
                                    const uint8_t* __restrict__ mask, int Bn, long long T,
                                    float2* __restrict__ fac) {
  __shared__ int redi[kRespThreads / 32];
  const int i = blockIdx.x;
  long long s = cu[i];
  long long e = cu[i + 1];
  if (s < 0 || s > T) s = 0;
  if (e < s || e > T) e = s;
  const long long Ti = valid_count(mask, s, e, redi);
  if (threadIdx.x == 0)
    fac[i] = make_float2(adv[i],
                         Ti > 0 ? static_cast<float>(1.0 / (static_cast<double>(Bn) * Ti)) : 0.f);
}

// Score Centering: Abar = mean of A_i over the responses with valid tokens
// (fac[i].y > 0), then fac[i].x = A_i - Abar; fixed-order fp64 sum.
__global__ void __launch_bounds__(kFinalThreads) sc_centre_kernel(float2* __restrict__ fac, int B) {
  __shared__ double red[kFinalThreads / 32];
  __shared__ double abar;
  double sum = 0.0, cnt = 0.0;
  for (int i = threadIdx.x; i < B; i += kFinalThreads) {
    if (fac[i].y > 0.f) {
      sum += static_cast<double>(fac[i].x);
      cnt += 1.0;
    }
  }
  const double tot = block_sum<double, kFinalThreads>(sum, red);
  const double n = block_sum<double, kFinalThreads>(cnt, red);
  if (threadIdx.x == 0) abar = n > 0.0 ? tot / n : 0.0;
  __syncthreads();
  for (int i = threadIdx.x; i < B; i += kFinalThreads)
    fac[i].x = static_cast<float>(static_cast<double>(fac[i].x) - abar);
}

// Score Centering loss, per response: (sum of log pi over valid tokens, T_i)
// in fp64.  Same cu_seqlens checks as is_loss_resp_kernel.
__global__ void __launch_bounds__(kRespThreads)
    sc_loss_resp_kernel(const float* __restrict__ logpi, const int64_t* __restrict__ cu,
                        const uint8_t* __restrict__ mask, int B, long long T,
                        double2* __restrict__ part, int* err) {
  __shared__ double red[kRespThreads / 32];
  __shared__ int redi[kRespThreads / 32];
  const int i = blockIdx.x;
  long long s = cu[i];
  long long e = cu[i + 1];
  const bool bad = s < 0 || e < s || e > T || (i == 0 && s != 0) || (i == B - 1 && e != T);
  if (bad) {
    if (threadIdx.x == 0 && err) atomicOr(err, 2);
    if (s < 0 || s > T) s = 0;
    if (e < s || e > T) e = s;
  }
  const long long Ti = valid_count(mask, s, e, redi);
  double acc = 0.0;
  for (long long t = s + threadIdx.x; t < e; t += kRespThreads)
    if (!mask || mask[t] != 0) acc += static_cast<double>(logpi[t]);
  const double tot = block_sum<double, kRespThreads>(acc, red);
  if (threadIdx.x == 0) part[i] = make_double2(tot, static_cast<double>(Ti));
}

// L_SC = -(1/B) sum_i (A_i - Abar) (1/T_i) sum_t log pi_t, fixed order.
__global__ void __launch_bounds__(kFinalThreads)
    sc_loss_final_kernel(const double2* __restrict__ part, const float2* __restrict__ fac, int B,
                         float* loss) {
  __shared__ double red[kFinalThreads / 32];
  double acc = 0.0;
  for (int i = threadIdx.x; i < B; i += kFinalThreads)
    if (part[i].y > 0.0) acc += static_cast<double>(fac[i].x) * (part[i].x / part[i].y);
  const double tot = block_sum<double, kFinalThreads>(acc, red);
  if (threadIdx.x == 0) *loss = B > 0 ? static_cast<float>(-tot / B) : 0.f;
}

__global__ void __launch_bounds__(kFinalThreads)
    is_loss_final_kernel(const RespPart* __restrict__ part, int B, int Bn, float* loss,
                         float* d3) {
  __shared__ double red[kFinalThreads / 32];
  double lag = 0.0, base = 0.0, dd = 0.0, cnt = 0.0;
  for (int i = threadIdx.x; i < B; i += kFinalThreads) {
    lag += part[i].lag;
    base += part[i].base;
    dd += part[i].d3;
    cnt += part[i].cnt;
  }
  const double lag_t = block_sum<double, kFinalThreads>(lag, red);
  const double base_t = block_sum<double, kFinalThreads>(base, red);
  const double d3_t = block_sum<double, kFinalThreads>(dd, red);
  const double cnt_t = block_sum<double, kFinalThreads>(cnt, red);
  if (threadIdx.x == 0) {
    if (loss) *loss = Bn > 0 ? static_cast<float>(-(base_t + lag_t) / Bn) : 0.f;
    if (d3) *d3 = cnt_t > 0 ? static_cast<float>(d3_t / cnt_t) : 0.f;
  }
}

__global__ void __cluster_dims__(kStatBlocks, 1, 1) __launch_bounds__(kD3Threads)
    d3_kernel(const float* __restrict__ logpi, const float* __restrict__ logmu, long long T,
              float* d3) {
  __shared__ double red[kD3Threads / 32];
  __shared__ double part;
  cg::cluster_group cluster = cg::this_cluster();
  const unsigned rank = cluster.block_rank();
  float acc = 0.f;
  for (long long t = static_cast<long long>(rank) * kD3Threads + threadIdx.x; t < T;
       t += kStatBlocks * kD3Threads)
    acc += d3_term(logpi[t] - logmu[t]);
  const double tot = block_sum<double, kD3Threads>(static_cast<double>(acc), red);
  if (threadIdx.x == 0) part = tot;
  cluster.sync();
  if (rank == 0 && threadIdx.x == 0) {
    double sum = 0.0;
    for (int r = 0; r < kStatBlocks; ++r) sum += *cluster.map_shared_rank(&part, r);
    *d3 = T > 0 ? static_cast<float>(sum / static_cast<double>(T)) : 0.f;
  }
  cluster.sync();  // keep every CTA's partial alive until CTA 0 has read it
}

// Per-update diagnostics over all T tokens, one cluster, fixed order:
// out = {D3 (= k3), k1 = mean(-d), k2 = mean(d^2/2), mean w, max w, min w,
// max |d|}.
struct StatPart {
  double s3, s1, s2, sw;
  float wmax, wmin, dmax;
};

__global__ void __cluster_dims__(kStatBlocks, 1, 1) __launch_bounds__(kD3Threads)
    is_stats_kernel(const float* __restrict__ logpi, const float* __restrict__ logmu,
                    long long T, float* out) {
  __shared__ double red[kD3Threads / 32];
  __shared__ float redf[kD3Threads / 32];
  __shared__ StatPart part;
  cg::cluster_group cluster = cg::this_cluster();
  const unsigned rank = cluster.block_rank();
  float s3 = 0.f, s1 = 0.f, s2 = 0.f, sw = 0.f;
  float wmax = 0.f, wmin = INFINITY, dmax = 0.f;
  for (long long t = static_cast<long long>(rank) * kD3Threads + threadIdx.x; t < T;
       t += kStatBlocks * kD3Threads) {
    const float d = logpi[t] - logmu[t];
    const float w = expf(d);
    s3 += d3_term(d);
    s1 -= d;
    s2 += 0.5f * d * d;
    sw += w;
    wmax = fmaxf(wmax, w);
    wmin = fminf(wmin, w);
    dmax = fmaxf(dmax, fabsf(d));
  }
  const double t3 = block_sum<double, kD3Threads>(static_cast<double>(s3), red);
  const double t1 = block_sum<double, kD3Threads>(static_cast<double>(s1), red);
  const double t2 = block_sum<double, kD3Threads>(static_cast<double>(s2), red);
  const double tw = block_sum<double, kD3Threads>(static_cast<double>(sw), red);
  const float mx = block_extreme<kD3Threads, true>(wmax, redf);
  const float mn = block_extreme<kD3Threads, false>(wmin, redf);
  const float dm = block_extreme<kD3Threads, true>(dmax, redf);
  if (threadIdx.x == 0) part = StatPart{t3, t1, t2, tw, mx, mn, dm};
  cluster.sync();
  if (rank == 0 && threadIdx.x == 0) {
    StatPart a = part;
    for (int r = 1; r < kStatBlocks; ++r) {
      const StatPart b = *cluster.map_shared_rank(&part, r);
      a.s3 += b.s3;
      a.s1 += b.s1;
      a.s2 += b.s2;
      a.sw += b.sw;
      a.wmax = fmaxf(a.wmax, b.wmax);
      a.wmin = fminf(a.wmin, b.wmin);
      a.dmax = fmaxf(a.dmax, b.dmax);
    }
    const double inv = T > 0 ? 1.0 / static_cast<double>(T) : 0.0;
    out[0] = static_cast<float>(a.s3 * inv);
    out[1] = static_cast<float>(a.s1 * inv);
    out[2] = static_cast<float>(a.s2 * inv);
    out[3] = static_cast<float>(a.sw * inv);
    out[4] = T > 0 ? a.wmax : 0.f;
    out[5] = T > 0 ? a.wmin : 0.f;
    out[6] = T > 0 ? a.dmax : 0.f;
  }
  cluster.sync();  // keep every CTA's partial alive until CTA 0 has read it
}

__global__ void group_advantage_kernel(const float* __restrict__ r, int B, int G,
                                       float* __restrict__ adv) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= B) return;
  const int g0 = (i / G) * G;
  double sum = 0.0;
  for (int j = 0; j < G; ++j) sum += static_cast<double>(r[g0 + j]);
  adv[i] = static_cast<float>(static_cast<double>(r[i]) - sum / G);
}

}  // namespace

size_t is_loss_ws_bytes(int32_t B) {
  const size_t b = B > 0 ? static_cast<size_t>(B) : 0;
  return (b * sizeof(RespPart) + 255) / 256 * 256;
}

cudaError_t launch_group_advantage(const float* r, int B, int G, float* adv, cudaStream_t st) {
  if (B <= 0) return cudaSuccess;
  const int threads = 256;
  group_advantage_kernel<<<(B + threads - 1) / threads, threads, 0, st>>>(r, B, G, adv);
  return cudaGetLastError();
}

cudaError_t launch_is_loss(const float* logpi, const float* logmu, const int64_t* cu,
                           const float* adv, const uint8_t* mask, int B, int Bn, int64_t T,
                           float* loss, float* d3, float* coef, void* ws, int* err,
                           cudaStream_t st) {
  RespPart* part = static_cast<RespPart*>(ws);
  if (B > 0) {
    is_loss_resp_kernel<<<B, kRespThreads, 0, st>>>(logpi, logmu, cu, adv, mask, B, Bn, T, coef,
                                                    part, err);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  is_loss_final_kernel<<<1, kFinalThreads, 0, st>>>(part, B, Bn, loss, d3);
  return cudaGetLastError();
}

size_t resp_factors_ws_bytes(int32_t B) {
  const size_t b = B > 0 ? static_cast<size_t>(B) : 0;
  return (b * sizeof(float2) + 255) / 256 * 256;
}

cudaError_t launch_resp_factors(const int64_t* cu, const float* adv, const uint8_t* mask, int B,
                                int Bn, int64_t T, float2* fac, cudaStream_t st) {
  if (B <= 0) return cudaSuccess;
  resp_factors_kernel<<<B, kRespThreads, 0, st>>>(cu, adv, mask, Bn, T, fac);
  return cudaGetLastError();
}

cudaError_t launch_sc_centre(float2* fac, int B, cudaStream_t st) {
  if (B <= 0) return cudaSuccess;
  sc_centre_kernel<<<1, kFinalThreads, 0, st>>>(fac, B);
  return cudaGetLastError();
}

cudaError_t launch_sc_loss(const float* logpi, const int64_t* cu, const uint8_t* mask,
                           const float2* fac, int B, int64_t T, float* loss, void* ws, int* err,
                           cudaStream_t st) {
  double2* part = static_cast<double2*>(ws);
  if (B > 0) {
    sc_loss_resp_kernel<<<B, kRespThreads, 0, st>>>(logpi, cu, mask, B, T, part, err);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  sc_loss_final_kernel<<<1, kFinalThreads, 0, st>>>(part, fac, B, loss);
  return cudaGetLastError();
}

namespace {
// The fixed-order sum of the data-parallel exchange: element i of the output
// is parts[0][i] + parts[1][i] + ... + parts[n-1][i], added left to right in
// fp32, so every rank that runs it on the same gathered partials gets the
// same bits.  Four elements per thread when the rows allow 16-byte access.
__global__ void sum_partials_kernel(const float* __restrict__ parts, int n, long long count,
                                    float* __restrict__ out) {
  const long long stride = static_cast<long long>(gridDim.x) * blockDim.x;
  const long long i0 = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
  if ((count & 3) == 0 && (reinterpret_cast<uintptr_t>(parts) & 15u) == 0 &&
      (reinterpret_cast<uintptr_t>(out) & 15u) == 0) {
    const long long n4 = count >> 2;
    const float4* p4 = reinterpret_cast<const float4*>(parts);
    float4* o4 = reinterpret_cast<float4*>(out);
    for (long long i = i0; i < n4; i += stride) {
      float4 a = __ldcs(p4 + i);
      for (int r = 1; r < n; ++r) {
        const float4 b = __ldcs(p4 + static_cast<long long>(r) * n4 + i);
        a.x = __fadd_rn(a.x, b.x);
        a.y = __fadd_rn(a.y, b.y);
        a.z = __fadd_rn(a.z, b.z);
        a.w = __fadd_rn(a.w, b.w);
      }
      __stcs(o4 + i, a);
    }
  } else {
    for (long long i = i0; i < count; i += stride) {
      float a = parts[i];
      for (int r = 1; r < n; ++r) a = __fadd_rn(a, parts[static_cast<long long>(r) * count + i]);
      out[i] = a;
    }
  }
}
}  // namespace

cudaError_t launch_sum_partials(const float* parts, int n_parts, int64_t count, float* out,
                                cudaStream_t st) {
  if (count <= 0) return cudaSuccess;
  const int threads = 256;
  long long blocks = (count / 4 + threads - 1) / threads;
  const long long cap = static_cast<long long>(num_sms()) * 8;
  if (blocks > cap) blocks = cap;
  if (blocks < 1) blocks = 1;
  sum_partials_kernel<<<static_cast<unsigned>(blocks), threads, 0, st>>>(parts, n_parts, count,
                                                                        out);
  return cudaGetLastError();
}

cudaError_t launch_is_stats(const float* logpi, const float* logmu, int64_t T, float* out,
                            cudaStream_t st) {
  is_stats_kernel<<<kStatBlocks, kD3Threads, 0, st>>>(logpi, logmu, T, out);
  return cudaGetLastError();
}

cudaError_t launch_d3(const float* logpi, const float* logmu, int64_t T, float* d3,
                      cudaStream_t st) {
  d3_kernel<<<kStatBlocks, kD3Threads, 0, st>>>(logpi, logmu, T, d3);
  return cudaGetLastError();
}

}  // namespace rz
