// rz_lmhead.cu -- the LM-head contractions and their fused epilogues.
//
//   lse_partial  (rollout) z = H W^T per 128x256 tile in TMEM; the epilogue
//                folds each row's logits into a running (max, sum of exp)
//                over the tiles of its vocab split, in ascending vocab
//                order, and picks out z[t, a_t].
//   lse_merge    fixed-order merge of the splits -> logsumexp, log pi.
//   lse_keep     (learner, one token chunk) the lse_partial fold on the
//                same tiles, bitwise, keeping its terms 2^((z - m) log2 e)
//                as fp16 and the running max m per 32 columns.
//   merge_coef   the fixed-order merge, then c_t = A_i w_t / (B T_i).
//   dz_rows      HBM pass: dz = c_t (softmax - onehot) as bf16, in place
//                over the kept terms (the logits are never recomputed).
//   dH, dW       dz W and dz^T H on the same tensor-core pipeline.
//   logits_f32   plain z = H W^T (same tiles) for callers that want logits.
//
// Formulas: log pi(a|h) = z_a - logsumexp_v z_v (the sampled token's
// logprob, "REINFORCE Zero" project page s.02 and the vLLM post s.4 item 1);
// dz from differentiating the loss through the numerator pi only (project
// page s.02, "A minimal REINFORCE objective").
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>

#include "rz_check.cuh"
#include "rz_gemm.cuh"
#include "rz_internal.h"
#include "rz_lse.cuh"
#include "rz_math.cuh"
#include "rz_ptx.cuh"

namespace rz {

// ============================================================== epilogues
// Online log-sum-exp: state (m, s) with m = max z so far and
// s = sum 2^((z - m) log2 e); the row's logsumexp is m + ln s.
struct EpiLsePartial {
  struct Params {
    const int32_t* tokens;
    float2* part;    // [T, S]
    float* zgather;  // [T]
    long long T;
    int V;
    int S;
  };
  struct State {
    float m, s, za;
    int a;
    bool found;
  };

  static __device__ __forceinline__ void task_begin(const Params& p, State& st, int m_blk, int,
                                                    int row) {
    const long long g = static_cast<long long>(m_blk) * kBM + row;
    st.m = -INFINITY;
    st.s = 0.f;
    st.za = 0.f;
    st.found = false;
    st.a = g < p.T ? __ldg(p.tokens + g) : -1;
  }

  static __device__ __forceinline__ void chunk(const Params& p, State& st, const uint32_t (&r)[32],
                                               int cbase) {
    float v[32];
#pragma unroll
    for (int j = 0; j < 32; ++j) v[j] = __uint_as_float(r[j]);
    if (cbase + 32 > p.V) {
#pragma unroll
      for (int j = 0; j < 32; ++j)
        if (cbase + j >= p.V) v[j] = -INFINITY;
    }
    lse_fold32(st.m, st.s, v);
    const unsigned rel = static_cast<unsigned>(st.a - cbase);
    if (rel < 32u) {
#pragma unroll
      for (int j = 0; j < 32; ++j)
        if (rel == static_cast<unsigned>(j)) st.za = v[j];
      st.found = true;
    }
  }

  static __device__ __forceinline__ void tile(const Params& p, State& st, int, int n_tile,
                                              uint32_t taddr, int, uint8_t*) {
    const int col0 = n_tile * kBN;
#pragma unroll 1
    for (int c = 0; c < kBN; c += 64) {
      if (col0 + c >= p.V) break;  // warp-uniform
      uint32_t r0[32], r1[32];
      tmem_ld32(taddr + c, r0);
      tmem_ld32(taddr + c + 32, r1);
      tmem_ld_wait();
      chunk(p, st, r0, col0 + c);
      if (col0 + c + 32 < p.V) chunk(p, st, r1, col0 + c + 32);
    }
  }

  static __device__ __forceinline__ void task_end(const Params& p, State& st, int m_blk, int grp,
                                                  int row) {
    const long long g = static_cast<long long>(m_blk) * kBM + row;
    if (g >= p.T) return;
    if (!RZ_DCHECK(g >= 0 && grp >= 0 && grp < p.S, 10)) return;
    p.part[g * p.S + grp] = make_float2(st.m, st.s);
    if (st.found) p.zgather[g] = st.za;
  }
};

// Learner pass 1 for one chunk of rows: exactly the EpiLsePartial fold (so
// log pi is the rollout's, bit for bit), keeping what the backward pass needs
// to form the softmax without recomputing the logits: the fold's own terms
// e_tv = 2^((z_tv - m) log2 e) in (0, 1] as fp16, and m, the running maximum
// they were taken against, once per 32 columns.  p_tv = e_tv 2^((m - lse_t)
// log2 e) then needs only the row's final log-sum-exp.
struct EpiLseKeep {
  struct Params {
    CUtensorMap tm_e16;         // the terms [rows, V] fp16, box 64 x 32, 128-byte swizzle
    EpiLsePartial::Params lse;  // chunk-local rows: T = rows of the chunk
    float* emax;                // [rows, ldm] m per 32-column slice
    long long ldm;              // >= ceil(V / 32), even
  };
  using State = EpiLsePartial::State;

  static __device__ __forceinline__ void task_begin(const Params& p, State& st, int m_blk,
                                                    int grp, int row) {
    EpiLsePartial::task_begin(p.lse, st, m_blk, grp, row);
  }
  static __device__ __forceinline__ void task_end(const Params& p, State& st, int m_blk, int grp,
                                                  int row) {
    EpiLsePartial::task_end(p.lse, st, m_blk, grp, row);
  }

  // EpiLsePartial::chunk with the terms kept, packed to 16 fp16 pairs.
  static __device__ __forceinline__ void chunk(const Params& p, State& st, const uint32_t (&r)[32],
                                               int cbase, uint32_t* w) {
    float v[32];
#pragma unroll
    for (int j = 0; j < 32; ++j) v[j] = __uint_as_float(r[j]);
    if (cbase + 32 > p.lse.V) {
#pragma unroll
      for (int j = 0; j < 32; ++j)
        if (cbase + j >= p.lse.V) v[j] = -INFINITY;
    }
    float e[32];
    lse_fold32_keep(st.m, st.s, v, e);
    const unsigned rel = static_cast<unsigned>(st.a - cbase);
    if (rel < 32u) {
#pragma unroll
      for (int j = 0; j < 32; ++j)
        if (rel == static_cast<unsigned>(j)) st.za = v[j];
      st.found = true;
    }
#pragma unroll
    for (int j = 0; j < 16; ++j) w[j] = pack_f16x2(e[2 * j], e[2 * j + 1]);
  }

  // A 64-column slab of the warp's 32 rows goes through the warp's stage
  // (row r at r*128, 16-byte piece j at j ^ (r & 7): the 128-byte swizzle)
  // and out with one TMA store (evict-first: the terms are read back only
  // after the whole chunk and would otherwise push the H and W tiles the
  // CTAs share out of L2).  Rows past the chunk and columns past V are
  // clipped by the tensor map.
  static __device__ __forceinline__ void tile(const Params& p, State& st, int m_blk, int n_tile,
                                              uint32_t taddr, int row, uint8_t* stage) {
    const int col0 = n_tile * kBN;
    const int V = p.lse.V;
    const int lane = row & 31;
    const long long grow = static_cast<long long>(m_blk) * kBM + row;
    const int rbase = m_blk * kBM + (row & ~31);
    const uint64_t pol = l2_policy_first();
    uint4* mine = reinterpret_cast<uint4*>(stage + lane * 128);
#pragma unroll 1
    for (int c = 0; c < kBN; c += 64) {
      if (col0 + c >= V) break;  // warp-uniform
      uint32_t r0[32], r1[32];
      tmem_ld32(taddr + c, r0);
      tmem_ld32(taddr + c + 32, r1);
      tmem_ld_wait();
      uint32_t w[32];
      chunk(p, st, r0, col0 + c, w);
      const float m0 = st.m;
      float m1 = m0;
      if (col0 + c + 32 < V) {
        chunk(p, st, r1, col0 + c + 32, w + 16);
        m1 = st.m;
      }
      if (grow < p.lse.T &&
          RZ_DCHECK(grow >= 0 && ((col0 + c) >> 5) + (col0 + c + 32 < V ? 2 : 1) <= p.ldm, 11)) {
        float* em = p.emax + grow * p.ldm + ((col0 + c) >> 5);
        if (col0 + c + 32 < V) {
          *reinterpret_cast<float2*>(em) = make_float2(m0, m1);
        } else {
          em[0] = m0;
        }
      }
      if (lane == 0) bulk_wait_read();  // the previous slab's store has read the stage
      __syncwarp();
#pragma unroll
      for (int j = 0; j < 8; ++j)
        mine[j ^ (lane & 7)] = make_uint4(w[4 * j], w[4 * j + 1], w[4 * j + 2], w[4 * j + 3]);
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0 && rbase < p.lse.T &&
          RZ_DCHECK(rbase >= 0 && col0 + c >= 0 && col0 + c < V && ((col0 + c) & 7) == 0, 12)) {
        tma_store_2d_hint(&p.tm_e16, stage, col0 + c, rbase, pol);
        bulk_commit();
      }
    }
  }
};

// Philox4x32 with 10 rounds (Salmon et al., "Parallel Random Numbers: As
// Easy as 1, 2, 3", SC 2011): each round multiplies c0 and c2 by fixed odd
// constants, mixes the 64-bit products' halves with c1, c3 and the key, and
// the key is bumped by two fixed increments between rounds.
__device__ __forceinline__ void philox4x32_10(uint32_t c0, uint32_t c1, uint32_t c2, uint32_t c3,
                                              uint32_t k0, uint32_t k1, uint32_t (&out)[4]) {
#pragma unroll
  for (int r = 0; r < 10; ++r) {
    const uint32_t lo0 = 0xD2511F53u * c0;
    const uint32_t hi0 = __umulhi(0xD2511F53u, c0);
    const uint32_t lo1 = 0xCD9E8D57u * c2;
    const uint32_t hi1 = __umulhi(0xCD9E8D57u, c2);
    c0 = hi1 ^ c1 ^ k0;
    c1 = lo1;
    c2 = hi0 ^ c3 ^ k1;
    c3 = lo0;
    k0 += 0x9E3779B9u;
    k1 += 0xBB67AE85u;
  }
  out[0] = c0;
  out[1] = c1;
  out[2] = c2;
  out[3] = c3;
}

// The same Philox4x32-10 for a fixed row: counter (x, row lo, row hi, 0)
// and a fixed key.  Everything that does not depend on x -- the round keys,
// the c2-product of round 1 and the c0-product of round 2 -- is computed once
// per row, so each word costs about two thirds of the plain evaluation.
struct PhiloxRow {
  uint32_t rk0[10], rk1[10];
  uint32_t r1_c0, r1_c1;  // round-1 outputs c0, c1 (x-independent)
  uint32_t r2_lo0, r2_hi0;  // round-2 product of those c0

  __device__ __forceinline__ void init(uint32_t row_lo, uint32_t row_hi, uint32_t k0,
                                       uint32_t k1) {
#pragma unroll
    for (int r = 0; r < 10; ++r) {
      rk0[r] = k0 + static_cast<uint32_t>(r) * 0x9E3779B9u;
      rk1[r] = k1 + static_cast<uint32_t>(r) * 0xBB67AE85u;
    }
    r1_c0 = __umulhi(0xCD9E8D57u, row_hi) ^ row_lo ^ rk0[0];
    r1_c1 = 0xCD9E8D57u * row_hi;
    r2_lo0 = 0xD2511F53u * r1_c0;
    r2_hi0 = __umulhi(0xD2511F53u, r1_c0);
  }

  __device__ __forceinline__ void words(uint32_t x, uint32_t (&out)[4]) const {
    // round 1 (c3 = 0)
    uint32_t c0 = r1_c0, c1 = r1_c1;
    uint32_t c2 = __umulhi(0xD2511F53u, x) ^ rk1[0];
    uint32_t c3 = 0xD2511F53u * x;
    // round 2 (the c0 product is precomputed)
    {
      const uint32_t lo1 = 0xCD9E8D57u * c2;
      const uint32_t hi1 = __umulhi(0xCD9E8D57u, c2);
      const uint32_t n0 = hi1 ^ c1 ^ rk0[1];
      const uint32_t n2 = r2_hi0 ^ c3 ^ rk1[1];
      c0 = n0;
      c1 = lo1;
      c2 = n2;
      c3 = r2_lo0;
    }
#pragma unroll
    for (int r = 2; r < 10; ++r) {
      const uint32_t lo0 = 0xD2511F53u * c0;
      const uint32_t hi0 = __umulhi(0xD2511F53u, c0);
      const uint32_t lo1 = 0xCD9E8D57u * c2;
      const uint32_t hi1 = __umulhi(0xCD9E8D57u, c2);
      c0 = hi1 ^ c1 ^ rk0[r];
      c1 = lo1;
      c2 = hi0 ^ c3 ^ rk1[r];
      c3 = lo0;
    }
    out[0] = c0;
    out[1] = c1;
    out[2] = c2;
    out[3] = c3;
  }
};

__device__ __forceinline__ float lg2_approx(float x) {
  float y;
  asm("lg2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Fused sampling in the rollout's logprob GEMM: besides the log-sum-exp state
// (the very same arithmetic as EpiLsePartial) each row keeps the running
// Gumbel-max winner over its split: key = z log2(e) - log2(-log2 U), which
// orders tokens exactly as z + Gumbel noise does (the two differ by the
// constant log2(ln 2) and the factor log2(e)).  U for (row, v) is word
// v mod 4 of Philox4x32-10 at counter (v / 4, row id lo, row id hi, 0) under
// the caller's 64-bit seed, mapped to ((x >> 9) + 1/2) 2^-23 in (0, 1).  Ties
// go to the smaller vocabulary index.
struct EpiSample {
  struct Params {
    const int64_t* row_ids;  // nullable: row index (row0 + local row)
    float4* part;            // [T, S]: m, s, best key, z at best
    int* part_idx;           // [T, S]: best vocabulary index
    long long row0;          // first row of this launch (row ids only)
    long long T;
    int V;
    int S;
    uint32_t k0, k1;
  };
  struct State {
    float m, s, bk, bz;
    int bi;
    PhiloxRow rng;
  };

  static __device__ __forceinline__ void task_begin(const Params& p, State& st, int m_blk, int,
                                                    int row) {
    const long long g = static_cast<long long>(m_blk) * kBM + row;
    st.m = -INFINITY;
    st.s = 0.f;
    st.bk = -INFINITY;
    st.bz = 0.f;
    st.bi = -1;
    const long long rid = g < p.T ? (p.row_ids ? __ldg(p.row_ids + g) : p.row0 + g) : 0;
    st.rng.init(static_cast<uint32_t>(static_cast<unsigned long long>(rid) & 0xffffffffull),
                static_cast<uint32_t>(static_cast<unsigned long long>(rid) >> 32), p.k0, p.k1);
  }

  // -log2(U) to full relative precision for U = (m + 1/2) 2^-23.  Next to 1
  // (1 - U < 2^-6), where -log2 U is tiny and the largest Gumbel draws come
  // from, the fast hardware log2 has only absolute accuracy, so the Taylor
  // series -ln(1 - v) = v (1 + v/2 + v^2/3 + v^3/4 + v^4/5 + ...) is used
  // (truncation < 2^-26 relative); elsewhere the hardware log2 is accurate
  // to ~1e-5 relative or better.
  static __device__ __forceinline__ float neg_log2_uniform(uint32_t bits) {
    const uint32_t m = bits >> 9;
    const float u = __fmul_rn(__fadd_rn(__uint2float_rn(m), 0.5f), 1.1920928955078125e-7f);
    const float v = __fmul_rn(__fsub_rn(__uint2float_rn(8388608u - m), 0.5f),
                              1.1920928955078125e-7f);  // 1 - u, exact
    float ser = fmaf(v, 0.2f, 0.25f);
    ser = fmaf(v, ser, 0.33333334f);
    ser = fmaf(v, ser, 0.5f);
    ser = fmaf(v, ser, 1.0f);
    const float near1 = __fmul_rn(__fmul_rn(v, kLog2e), ser);
    return v < 0.015625f ? near1 : -lg2_approx(u);
  }

  // 32 columns of this thread's row; `words` holds the row's 32 Philox
  // words (8 pieces of 16 B, piece q at position q ^ (lane & 7)).
  static __device__ __forceinline__ void chunk(const Params& p, State& st, const uint32_t (&r)[32],
                                               int cbase, const uint4* words, int sw) {
    float v[32];
#pragma unroll
    for (int j = 0; j < 32; ++j) v[j] = __uint_as_float(r[j]);
    if (cbase + 32 > p.V) {
#pragma unroll
      for (int j = 0; j < 32; ++j)
        if (cbase + j >= p.V) v[j] = -INFINITY;
    }
    lse_fold32(st.m, st.s, v);
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      const uint4 x4 = words[q ^ sw];
      const uint32_t x[4] = {x4.x, x4.y, x4.z, x4.w};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int j = 4 * q + e;
        const float key = fmaf(v[j], kLog2e, -lg2_approx(neg_log2_uniform(x[e])));
        if (key > st.bk) {  // -inf (masked) never wins; ties keep the smaller index
          st.bk = key;
          st.bz = v[j];
          st.bi = cbase + j;
        }
      }
    }
  }

  static __device__ __forceinline__ void tile(const Params& p, State& st, int, int n_tile,
                                              uint32_t taddr, int row, uint8_t* stage) {
    const int col0 = n_tile * kBN;
    const int lane = row & 31;
    const int sw = lane & 7;
    uint4* words = reinterpret_cast<uint4*>(stage + lane * 128);  // this row only
#pragma unroll 1
    for (int c = 0; c < kBN; c += 32) {
      if (col0 + c >= p.V) break;  // warp-uniform
      uint32_t r0[32];
      tmem_ld32(taddr + c, r0);
#pragma unroll 2  // two independent Philox blocks in flight: the chain is latency-bound
      for (int q = 0; q < 8; ++q) {
        uint32_t x[4];
        st.rng.words(static_cast<uint32_t>((col0 + c) >> 2) + q, x);
        words[q ^ sw] = make_uint4(x[0], x[1], x[2], x[3]);
      }
      tmem_ld_wait();
      chunk(p, st, r0, col0 + c, words, sw);
    }
  }

  static __device__ __forceinline__ void task_end(const Params& p, State& st, int m_blk, int grp,
                                                  int row) {
    const long long g = static_cast<long long>(m_blk) * kBM + row;
    if (g >= p.T) return;
    if (!RZ_DCHECK(g >= 0 && grp >= 0 && grp < p.S, 13)) return;
    p.part[g * p.S + grp] = make_float4(st.m, st.s, st.bk, st.bz);
    p.part_idx[g * p.S + grp] = st.bi;
  }
};

// Plain stores of the accumulator: bf16 (dH) or fp32 (logits), optionally
// fp32 accumulate (dW over token chunks, in chunk order).
template <int kMode>  // 0: bf16 store, 1: fp32 store, 2: fp32 accumulate-or-store
struct EpiStore {
  struct Params {
    void* out;
    long long ld;    // row stride in elements
    long long row0;  // row offset into out
    long long rows;  // valid rows (block-local numbering)
    int cols;        // valid columns
    int accumulate;  // mode 2 only
  };
  struct State {};

  static __device__ __forceinline__ void task_begin(const Params&, State&, int, int, int) {}
  static __device__ __forceinline__ void task_end(const Params&, State&, int, int, int) {}

  static __device__ __forceinline__ void chunk(const Params& p, const uint32_t (&r)[32], long long rr,
                                               int cbase) {
    if (!RZ_DCHECK(rr >= 0 && rr < p.rows && cbase >= 0 && cbase < p.cols && p.cols <= p.ld, 14))
      return;
    if (kMode == 0) {
      uint16_t* dst = static_cast<uint16_t*>(p.out) + (p.row0 + rr) * p.ld + cbase;
      if (cbase + 32 <= p.cols) {
        uint32_t w[16];
#pragma unroll
        for (int j = 0; j < 16; ++j)
          w[j] = pack_bf16x2(__uint_as_float(r[2 * j]), __uint_as_float(r[2 * j + 1]));
#pragma unroll
        for (int q = 0; q < 4; ++q)
          st_global_v4(dst + 8 * q, w[4 * q], w[4 * q + 1], w[4 * q + 2], w[4 * q + 3]);
      } else {
        for (int j = 0; j < 32; ++j)
          if (cbase + j < p.cols)
            dst[j] = static_cast<uint16_t>(pack_bf16x2(__uint_as_float(r[j]), 0.f) & 0xffffu);
      }
    } else {
      float* dst = static_cast<float*>(p.out) + (p.row0 + rr) * p.ld + cbase;
      const bool acc = (kMode == 2) && p.accumulate;
      const bool vec = (cbase + 32 <= p.cols) && ((p.ld & 3) == 0);
      if (vec) {
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          float4 v = make_float4(__uint_as_float(r[4 * q]), __uint_as_float(r[4 * q + 1]),
                                 __uint_as_float(r[4 * q + 2]), __uint_as_float(r[4 * q + 3]));
          float4* d4 = reinterpret_cast<float4*>(dst) + q;
          if (acc) {
            const float4 o = *d4;
            v.x += o.x;
            v.y += o.y;
            v.z += o.z;
            v.w += o.w;
          }
          *d4 = v;
        }
      } else {
        for (int j = 0; j < 32; ++j)
          if (cbase + j < p.cols) dst[j] = __uint_as_float(r[j]) + (acc ? dst[j] : 0.f);
      }
    }
  }

  static __device__ __forceinline__ void tile(const Params& p, State&, int m_blk, int n_tile,
                                              uint32_t taddr, int row, uint8_t*) {
    const int col0 = n_tile * kBN;
    const long long rr = static_cast<long long>(m_blk) * kBM + row;
    const bool valid = rr < p.rows;
#pragma unroll 1
    for (int c = 0; c < kBN; c += 64) {
      if (col0 + c >= p.cols) break;
      uint32_t r0[32], r1[32];
      tmem_ld32(taddr + c, r0);
      tmem_ld32(taddr + c + 32, r1);
      tmem_ld_wait();
      if (valid) {
        chunk(p, r0, rr, col0 + c);
        if (col0 + c + 32 < p.cols) chunk(p, r1, rr, col0 + c + 32);
      }
    }
  }
};

// ============================================================== merge kernels
// Merge one row's S split states in split order; log pi = z[t, a_t] - lse.
// An out-of-range token gives NaN for both and raises RZ_DEVERR_TOKEN_RANGE.
__device__ __forceinline__ float merge_row(const float2* pp, int S, int V, int a,
                                           const float* zg, float* l_out, int* err) {
  float sum;
  const float M = lse_merge_parts(pp, S, &sum);
  if (a < 0 || a >= V) {
    if (err) atomicOr(err, 1);
    *l_out = __int_as_float(0x7fc00000);
    return *l_out;
  }
  *l_out = lse_from(M, sum);
  return logprob_from(*zg, M, sum);
}

// One thread per row.
__global__ void lse_merge_kernel(long long T, int V, int S, const int32_t* __restrict__ tokens,
                                 const float2* __restrict__ part,
                                 const float* __restrict__ zgather, float* __restrict__ logprob,
                                 float* __restrict__ lse, float* __restrict__ lse_ws, int* err) {
  const long long t = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (t >= T) return;
  float l;
  const float lp = merge_row(part + t * S, S, V, tokens[t], zgather + t, &l, err);
  logprob[t] = lp;
  if (lse) lse[t] = l;
  if (lse_ws) lse_ws[t] = l;
}

// Learner, one chunk of rows (row0 = the chunk's first global row; every
// other pointer is chunk-local except cu and fac): the merge above, then the
// per-token coefficient c_t = A_i w_t / (B T_i), w_t = exp(log pi - log mu)
// (w_t = 1 when logmu is null: the Score Centering estimator, whose fac
// holds the centred advantages), 0 for a masked token.
// fac[i] = (A_i, 1/(B T_i)).  Response of a row: the last i with
// cu[i] <= row (empty responses own no row).
__global__ void lse_merge_coef_kernel(long long rows, int V, int S, long long row0,
                                      const int32_t* __restrict__ tokens,
                                      const float2* __restrict__ part,
                                      const float* __restrict__ zgather,
                                      float* __restrict__ logprob, float* __restrict__ lse_ws,
                                      const float* __restrict__ logmu,
                                      const int64_t* __restrict__ cu,
                                      const float2* __restrict__ fac,
                                      const uint8_t* __restrict__ mask, int B,
                                      float* __restrict__ coef, int* err) {
  const long long t = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (t >= rows) return;
  float l;
  const float lp = merge_row(part + t * S, S, V, tokens[t], zgather + t, &l, err);
  logprob[t] = lp;
  lse_ws[t] = l;
  const long long g = row0 + t;
  int lo = 0, hi = B;  // cu[lo] <= g < cu[hi] for a valid cu
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (cu[mid] <= g) lo = mid;
    else hi = mid;
  }
  const bool act = !mask || mask[t] != 0;
  const float2 f = fac[lo];
  const float w = logmu ? is_weight(lp, logmu[t]) : 1.f;
  coef[t] = act ? f.x * w * f.y : 0.f;
}

// ============================================================== dz pass
// dz_tv = c_t (p_tv - [v = a_t]) in bf16, written in place over the chunk's
// kept fp16 terms: p_tv = e_tv 2^((m - lse_t) log2 e) with m the running
// maximum of the term's 32-column slice; at v = a_t the exact
// c_t expm1(log pi_t) (no cancellation of p - 1 as p -> 1).  One CTA per row,
// 8 columns per 16-byte step (never straddling a slice), four steps in
// flight per thread.  Columns >= V are not touched.
constexpr int kDzThreads = 256;

__device__ __forceinline__ uint4 dz8(const uint4& q, float scale, float c_onehot, int rel) {
  const uint32_t w[4] = {q.x, q.y, q.z, q.w};
  float g[8];
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const __half2 h = *reinterpret_cast<const __half2*>(&w[j]);
    const float2 f = __half22float2(h);
    g[2 * j] = __fmul_rn(scale, f.x);
    g[2 * j + 1] = __fmul_rn(scale, f.y);
  }
  if (static_cast<unsigned>(rel) < 8u) {
#pragma unroll
    for (int j = 0; j < 8; ++j)
      if (rel == j) g[j] = c_onehot;
  }
  return make_uint4(pack_bf16x2(g[0], g[1]), pack_bf16x2(g[2], g[3]), pack_bf16x2(g[4], g[5]),
                    pack_bf16x2(g[6], g[7]));
}

__global__ void __launch_bounds__(kDzThreads)
    dz_rows_kernel(uint16_t* __restrict__ ez, long long lde, const float* __restrict__ emax,
                   long long ldm, int V, const int32_t* __restrict__ tokens,
                   const float* __restrict__ lse, const float* __restrict__ coef,
                   const float* __restrict__ logpi) {
  const long long row = blockIdx.x;
  uint4* er = reinterpret_cast<uint4*>(ez + row * lde);
  const float* mr = emax + row * ldm;
  const float l = lse[row];
  const float c = coef[row];
  const int a = tokens[row];
  const float c_onehot = __fmul_rn(c, expm1f(logpi[row]));
  const int n8 = V >> 3;
  int i = threadIdx.x;
  for (; i + 3 * kDzThreads < n8; i += 4 * kDzThreads) {
    uint4 q[4];
    float sc[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int k = i + u * kDzThreads;
      if (!RZ_DCHECK(8ll * k + 8 <= lde && (k >> 2) < ldm, 16)) return;
      q[u] = __ldcs(er + k);
      sc[u] = __fmul_rn(c, ex2_approx(__fmul_rn(__fsub_rn(__ldg(mr + (k >> 2)), l), kLog2e)));
    }
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int k = i + u * kDzThreads;
      __stcs(er + k, dz8(q[u], sc[u], c_onehot, a - 8 * k));
    }
  }
  for (; i < n8; i += kDzThreads) {
    const float sc = __fmul_rn(c, ex2_approx(__fmul_rn(__fsub_rn(__ldg(mr + (i >> 2)), l), kLog2e)));
    __stcs(er + i, dz8(__ldcs(er + i), sc, c_onehot, a - 8 * i));
  }
  // ragged tail: V % 8 columns
  const int v = 8 * n8 + static_cast<int>(threadIdx.x);
  if (v < V) {
    uint16_t* p = ez + row * lde + v;
    float g;
    if (v == a) {
      g = c_onehot;
    } else {
      const float sc = __fmul_rn(c, ex2_approx(__fmul_rn(__fsub_rn(mr[v >> 5], l), kLog2e)));
      g = __fmul_rn(sc, __half2float(__ushort_as_half(*p)));
    }
    *p = static_cast<uint16_t>(pack_bf16x2(g, 0.f) & 0xffffu);
  }
}

// One thread per row: log-sum-exp exactly as lse_merge_kernel, and the
// Gumbel-max winner over the splits in split order (ties: earlier split,
// i.e. smaller vocabulary index).
__global__ void sample_merge_kernel(long long T, int S, const float4* __restrict__ part,
                                    const int* __restrict__ part_idx, int32_t* __restrict__ tokens,
                                    float* __restrict__ logprob, float* __restrict__ lse) {
  const long long t = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (t >= T) return;
  const float4* pp = part + t * S;
  float sum;
  const float M = lse_merge_parts(pp, S, &sum);
  float bk = -INFINITY, bz = 0.f;
  int bi = 0;
  for (int g = 0; g < S; ++g) {
    if (pp[g].z > bk) {
      bk = pp[g].z;
      bz = pp[g].w;
      bi = part_idx[t * S + g];
    }
  }
  tokens[t] = bi;
  logprob[t] = logprob_from(bz, M, sum);
  if (lse) lse[t] = lse_from(M, sum);
}

// ============================================================== launchers
namespace {

// Launch a GEMM: one persistent CTA per SM (or per task, if fewer).
template <class Epi, bool kAMN, bool kBMN>
cudaError_t run_gemm(const CUtensorMap& a, const CUtensorMap& b, const GemmSched& s,
                     const typename Epi::Params& p, cudaStream_t st) {
  if (s.num_tasks <= 0) return cudaSuccess;
  auto kern = gemm_kernel<Epi, kAMN, kBMN>;
  cudaError_t e =
      cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
  if (e != cudaSuccess) return e;
  const int grid = s.num_tasks < num_sms() ? s.num_tasks : num_sms();
  kern<<<grid, kThreads, kSmemBytes, st>>>(a, b, s, p);
  return cudaGetLastError();
}

// m-blocks per raster group of the vocab-split GEMMs: half the SMs, so at
// any time about two vocab splits are in flight, each shared by ~76 CTAs.
int vocab_raster_group() {
  const int g = num_sms() / 2;
  return g > 0 ? g : 1;
}

GemmSched sched_of(long long m_rows, int n_cols, int n_groups, long long k_depth, int* err) {
  GemmSched s{};
  s.m_blocks = static_cast<int>((m_rows + kBM - 1) / kBM);
  s.n_tiles = (n_cols + kBN - 1) / kBN;
  s.n_groups = n_groups;
  s.tiles_per_group = (s.n_tiles + n_groups - 1) / n_groups;
  s.k_blocks = static_cast<int>((k_depth + kBK - 1) / kBK);
  s.num_tasks = s.m_blocks * n_groups;
  s.m_group = 1;
  s.err = err;
  return s;
}

}  // namespace

// The vocab-split GEMMs over many rows are launched in row blocks of
// kChunkRowsMax (120 tasks per CTA at V = 151936): with fixed round-robin
// task order, CTAs of one long launch drift apart by many vocab splits and
// lose the L2 sharing of W (several times the DRAM traffic, and under the
// power cap a lower clock).  A row's result does not depend on the block.
cudaError_t launch_lse_partial(const CUtensorMap& tmH, const CUtensorMap& tmW, int64_t T, int d,
                               int V, const int32_t* tokens, float2* part, float* zgather,
                               int* err, cudaStream_t st) {
  const int S = vocab_splits(V);
  for (int64_t r0 = 0; r0 < T; r0 += kChunkRowsMax) {
    const int64_t rows = (T - r0) < kChunkRowsMax ? (T - r0) : kChunkRowsMax;
    GemmSched s = sched_of(rows, V, S, d, err);
    s.tiles_per_group = vocab_tiles_per_split(V);
    s.m_group = vocab_raster_group();
    s.a_m_off = static_cast<int>(r0);
    EpiLsePartial::Params p{tokens + r0, part + r0 * S, zgather + r0,
                            static_cast<long long>(rows), V, S};
    cudaError_t e = run_gemm<EpiLsePartial, false, false>(tmH, tmW, s, p, st);
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

cudaError_t launch_lse_merge(int64_t T, int V, const int32_t* tokens, const float2* part,
                             const float* zgather, float* logprob, float* lse, float* lse_ws,
                             int* err, cudaStream_t st) {
  if (T <= 0) return cudaSuccess;
  const int threads = 256;
  const long long blocks = (T + threads - 1) / threads;
  lse_merge_kernel<<<static_cast<unsigned>(blocks), threads, 0, st>>>(
      T, V, vocab_splits(V), tokens, part, zgather, logprob, lse, lse_ws, err);
  return cudaGetLastError();
}

cudaError_t launch_sample(const CUtensorMap& tmH, const CUtensorMap& tmW, int64_t T, int d, int V,
                          const int64_t* row_ids, uint64_t seed, float4* part, int* part_idx,
                          int32_t* tokens, float* logprob, float* lse, int* err, cudaStream_t st) {
  const int S = vocab_splits(V);
  for (int64_t r0 = 0; r0 < T; r0 += kChunkRowsMax) {  // row blocks as in launch_lse_partial
    const int64_t rows = (T - r0) < kChunkRowsMax ? (T - r0) : kChunkRowsMax;
    GemmSched s = sched_of(rows, V, S, d, err);
    s.tiles_per_group = vocab_tiles_per_split(V);
    s.m_group = vocab_raster_group();
    s.a_m_off = static_cast<int>(r0);
    EpiSample::Params p{row_ids ? row_ids + r0 : nullptr,
                        part + r0 * S,
                        part_idx + r0 * S,
                        static_cast<long long>(r0),
                        static_cast<long long>(rows),
                        V,
                        S,
                        static_cast<uint32_t>(seed & 0xffffffffull),
                        static_cast<uint32_t>(seed >> 32)};
    cudaError_t e = run_gemm<EpiSample, false, false>(tmH, tmW, s, p, st);
    if (e != cudaSuccess) return e;
  }
  const int threads = 256;
  const long long blocks = (T + threads - 1) / threads;
  sample_merge_kernel<<<static_cast<unsigned>(blocks), threads, 0, st>>>(T, S, part, part_idx,
                                                                         tokens, logprob, lse);
  return cudaGetLastError();
}

cudaError_t launch_lse_keep(const CUtensorMap& tmH, const CUtensorMap& tmW, int64_t row0,
                            int64_t rows, int d, int V, const int32_t* tokens, float2* part,
                            float* zgather, const CUtensorMap& tmE16, float* emax, int64_t ldm,
                            int* err, cudaStream_t st) {
  const int S = vocab_splits(V);
  GemmSched s = sched_of(rows, V, S, d, err);
  s.tiles_per_group = vocab_tiles_per_split(V);
  s.m_group = vocab_raster_group();
  s.a_m_off = static_cast<int>(row0);
  EpiLseKeep::Params p{tmE16, {tokens, part, zgather, static_cast<long long>(rows), V, S}, emax,
                       ldm};
  return run_gemm<EpiLseKeep, false, false>(tmH, tmW, s, p, st);
}

cudaError_t launch_lse_merge_coef(int64_t row0, int64_t rows, int V, const int32_t* tokens,
                                  const float2* part, const float* zgather, float* logprob,
                                  float* lse_ws, const float* logmu, const int64_t* cu,
                                  const float2* fac, const uint8_t* mask, int B, float* coef,
                                  int* err, cudaStream_t st) {
  if (rows <= 0) return cudaSuccess;
  const int threads = 256;
  const long long blocks = (rows + threads - 1) / threads;
  lse_merge_coef_kernel<<<static_cast<unsigned>(blocks), threads, 0, st>>>(
      rows, V, vocab_splits(V), row0, tokens, part, zgather, logprob, lse_ws, logmu, cu, fac,
      mask, B, coef, err);
  return cudaGetLastError();
}

cudaError_t launch_dz_rows(uint16_t* ez, int64_t lde, const float* emax, int64_t ldm,
                           int64_t rows, int V, const int32_t* tokens, const float* lse,
                           const float* coef, const float* logpi, cudaStream_t st) {
  if (rows <= 0) return cudaSuccess;
  dz_rows_kernel<<<static_cast<unsigned>(rows), kDzThreads, 0, st>>>(ez, lde, emax, ldm, V,
                                                                     tokens, lse, coef, logpi);
  return cudaGetLastError();
}

cudaError_t launch_logits_f32(const CUtensorMap& tmH, const CUtensorMap& tmW, int64_t T, int d,
                              int V, float* out, int* err, cudaStream_t st) {
  const int S = vocab_splits(V);
  for (int64_t r0 = 0; r0 < T; r0 += kChunkRowsMax) {  // row blocks as in launch_lse_partial
    const int64_t rows = (T - r0) < kChunkRowsMax ? (T - r0) : kChunkRowsMax;
    GemmSched s = sched_of(rows, V, S, d, err);
    s.tiles_per_group = vocab_tiles_per_split(V);
    s.m_group = vocab_raster_group();
    s.a_m_off = static_cast<int>(r0);
    EpiStore<1>::Params p{out, V, r0, rows, V, 0};
    cudaError_t e = run_gemm<EpiStore<1>, false, false>(tmH, tmW, s, p, st);
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

cudaError_t launch_dH(const CUtensorMap& tmDz, const CUtensorMap& tmWmn, int64_t row0,
                      int64_t rows, int d, int V, uint16_t* dH, int* err, cudaStream_t st) {
  const int nt = (d + kBN - 1) / kBN;
  GemmSched s = sched_of(rows, d, nt, V, err);
  EpiStore<0>::Params p{dH, d, row0, rows, d, 0};
  return run_gemm<EpiStore<0>, false, true>(tmDz, tmWmn, s, p, st);
}

cudaError_t check_read_lmhead(unsigned int* count, int* site) {
#ifdef RZ_CHECKS
  return check_read_and_clear(count, site);
#else
  *count = 0;
  *site = 0;
  return cudaSuccess;
#endif
}

cudaError_t launch_dW(const CUtensorMap& tmDzMn, const CUtensorMap& tmHmn, int64_t row0,
                      int64_t rows, int d, int V, float* dW, bool accumulate, int* err,
                      cudaStream_t st) {
  const int nt = (d + kBN - 1) / kBN;
  GemmSched s = sched_of(V, d, nt, rows, err);
  s.b_k_off = static_cast<int>(row0);
  EpiStore<2>::Params p{dW, d, 0, V, d, accumulate ? 1 : 0};
  return run_gemm<EpiStore<2>, true, true>(tmDzMn, tmHmn, s, p, st);
}

}  // namespace rz
