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
#include <cooperative_groups.h>
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

namespace cg = cooperative_groups;

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
// to form the softmax without recomputing the logits.
//   kRef = false: the fold's own terms e_tv = 2^((z_tv - m) log2 e) in (0, 1]
//     as fp16, and m, the running maximum they were taken against, once per
//     32 columns; p_tv = e_tv 2^((m - lse_t) log2 e) then needs only the
//     row's final log-sum-exp (the dz pass forms it).
//   kRef = true: the same terms taken against one reference R_t per row
//     (the caller's, e.g. the rollout's log-sum-exp of the row), e'_tv =
//     2^((z_tv - R_t) log2 e) = e_tv 2^((m - R_t) log2 e), as bf16 (whose
//     range is fp32's); p_tv = e'_tv e^(R_t - lse_t), one factor per row, so
//     the backward GEMMs take e' as it is.  m - R_t above kRefRange (e'
//     would overflow) raises RZ_DEVERR_RANGE and is clamped.
constexpr float kRefRange = 80.f;  // nats
constexpr int kErrRange = 8;       // RZ_DEVERR_RANGE

template <bool kRef>
struct EpiLseKeepT {
  struct Params {
    CUtensorMap tm_e16;         // the terms [rows, V], box 64 x 32, 128-byte swizzle
    EpiLsePartial::Params lse;  // chunk-local rows: T = rows of the chunk
    float* emax;                // [rows, ldm] m per 32-column slice (kRef: unused)
    long long ldm;              // >= ceil(V / 32), even
    const float* ref;           // [rows] R_t (kRef only; chunk-local)
    int* err;
  };
  struct State : EpiLsePartial::State {
    float R;
  };

  static __device__ __forceinline__ void task_begin(const Params& p, State& st, int m_blk,
                                                    int grp, int row) {
    EpiLsePartial::task_begin(p.lse, st, m_blk, grp, row);
    if (kRef) {
      const long long g = static_cast<long long>(m_blk) * kBM + row;
      st.R = g < p.lse.T ? __ldg(p.ref + g) : 0.f;
    }
  }
  static __device__ __forceinline__ void task_end(const Params& p, State& st, int m_blk, int grp,
                                                  int row) {
    EpiLsePartial::task_end(p.lse, st, m_blk, grp, row);
  }

  // EpiLsePartial::chunk with the terms kept, packed to 16 pairs (fp16, or
  // bf16 against the row's reference).
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
    if constexpr (kRef) {
      float gap = __fsub_rn(st.m, st.R);
      if (!(gap <= kRefRange)) {  // also NaN
        if (p.err) atomicOr(p.err, kErrRange);
        gap = gap > kRefRange ? kRefRange : 0.f;
      }
      const float f = ex2_approx(__fmul_rn(gap, kLog2e));
#pragma unroll
      for (int j = 0; j < 16; ++j)
        w[j] = pack_bf16x2(__fmul_rn(e[2 * j], f), __fmul_rn(e[2 * j + 1], f));
    } else {
#pragma unroll
      for (int j = 0; j < 16; ++j) w[j] = pack_f16x2(e[2 * j], e[2 * j + 1]);
    }
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
    float mt[8];
#pragma unroll
    for (int q = 0; q < 8; ++q) mt[q] = 0.f;
#pragma unroll
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
      if (!kRef) {
        mt[(c >> 5)] = m0;
        mt[(c >> 5) + 1] = m1;
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
    // the tile's running maxima, one per 32-column slice, written together
    // (two 16-byte stores per row: ldm is a multiple of 4 and col0 / 32 of 8)
    const int nsl = (V - col0 + 31) >> 5;  // valid 32-column slices of this tile
    if (!kRef && grow < p.lse.T &&
        RZ_DCHECK(grow >= 0 && (col0 >> 5) + (nsl < 8 ? nsl : 8) <= p.ldm, 11)) {
      float* em = p.emax + grow * p.ldm + (col0 >> 5);
      if (nsl >= 8) {
        reinterpret_cast<float4*>(em)[0] = make_float4(mt[0], mt[1], mt[2], mt[3]);
        reinterpret_cast<float4*>(em)[1] = make_float4(mt[4], mt[5], mt[6], mt[7]);
      } else {
#pragma unroll
        for (int q = 0; q < 8; ++q)
          if (q < nsl) em[q] = mt[q];
      }
    }
  }
};

using EpiLseKeep = EpiLseKeepT<false>;
using EpiLseKeepRef = EpiLseKeepT<true>;

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

// U in (0, 1) from a 32-bit word: ((x >> 9) + 1/2) 2^-23, exact in fp32.
__device__ __forceinline__ float uniform_of(uint32_t x) {
  return __fmul_rn(__fadd_rn(__uint2float_rn(x >> 9), 0.5f), 1.1920928955078125e-7f);
}

// Fused sampling in the rollout's logprob GEMM: a_t ~ softmax(z_t) drawn in
// the same pass that folds the row's log-sum-exp, by a two-level weighted
// reservoir over the vocabulary in ascending order.
//   * Within a vocabulary split, the row's 32-column chunks come in order.
//     With R the running sum of the fold's terms over the chunks seen so far
//     (this one included) and W this chunk's sum, the split's candidate is
//     replaced by a draw from this chunk when U1 R < W; the draw picks the
//     first token, in the order (column mod 4, then column), at which the
//     running sum of terms passes U2 W.  The terms are the fold's own
//     2^((z - m) log2 e), so the (m, s) state is bitwise the rollout's.
//   * The splits are merged the same way, in split order (sample_merge_kernel).
// Each token is then drawn with probability exactly its softmax weight.  U1,
// U2 are words 0 and 1 of Philox4x32-10 at counter (column / 32, row id lo,
// row id hi, 0) under the caller's 64-bit seed, the split's U3 word 0 at
// counter (split, row id lo, row id hi, 1), each mapped by uniform_of: a
// row's sample depends on its own id, hidden state and W only.
struct EpiSample {
  struct Params {
    const int64_t* row_ids;  // nullable: row index (row0 + local row)
    float4* part;            // [T, S]: m, s, z at the split's candidate, -
    int* part_idx;           // [T, S]: the split's candidate (-1: none)
    long long row0;          // first row of this launch (row ids only)
    long long T;
    int V;
    int S;
    uint32_t k0, k1;
  };
  struct State {
    float m, s, bz;
    int bi;
    PhiloxRow rng;
  };

  static __device__ __forceinline__ void task_begin(const Params& p, State& st, int m_blk, int,
                                                    int row) {
    const long long g = static_cast<long long>(m_blk) * kBM + row;
    st.m = -INFINITY;
    st.s = 0.f;
    st.bz = 0.f;
    st.bi = -1;
    const long long rid = g < p.T ? (p.row_ids ? __ldg(p.row_ids + g) : p.row0 + g) : 0;
    st.rng.init(static_cast<uint32_t>(static_cast<unsigned long long>(rid) & 0xffffffffull),
                static_cast<uint32_t>(static_cast<unsigned long long>(rid) >> 32), p.k0, p.k1);
  }

  // 32 columns of this thread's row.
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
    float e[32], acc[4], W;
    lse_fold32_terms(st.m, st.s, v, e, acc, W);
    uint32_t x[4];
    st.rng.words(static_cast<uint32_t>(cbase) >> 5, x);
    const bool rep = __fmul_rn(uniform_of(x[0]), st.s) < W;
    if (!__any_sync(0xffffffffu, rep)) return;  // the warp stays converged
    float zsel;
    const int off = draw_in_chunk(v, e, acc, W, x[1], zsel);
    if (rep && off >= 0) {
      st.bi = cbase + off;
      st.bz = zsel;
    }
  }

  // The draw inside a chunk that replaces the split's candidate: the class
  // (column mod 4) by the class sums, then the member inside it; on
  // rounding past the end, the last positive one.  Returns the column inside
  // the chunk (-1: none) and its logit in zsel_out.
  static __device__ __forceinline__ int draw_in_chunk(const float (&v)[32], const float (&e)[32],
                                                      const float (&acc)[4], float W, uint32_t x1,
                                                      float& zsel_out) {
    const float tgt = __fmul_rn(uniform_of(x1), W);
    int k = -1, lastk = 0;
    float cum = 0.f, base = 0.f, lastbase = 0.f;
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const float prev = cum;
      cum = __fadd_rn(cum, acc[q]);
      if (acc[q] > 0.f) {
        lastk = q;
        lastbase = prev;
      }
      if (k < 0 && cum > tgt) {
        k = q;
        base = prev;
      }
    }
    if (k < 0) {
      k = lastk;
      base = lastbase;
    }
    const float t2 = __fsub_rn(tgt, base);
    float ev[8], zv[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      ev[i] = k == 0 ? e[4 * i] : (k == 1 ? e[4 * i + 1] : (k == 2 ? e[4 * i + 2] : e[4 * i + 3]));
      zv[i] = k == 0 ? v[4 * i] : (k == 1 ? v[4 * i + 1] : (k == 2 ? v[4 * i + 2] : v[4 * i + 3]));
    }
    int sel = -1, last = -1;
    float zsel = 0.f, zlast = 0.f;
    cum = 0.f;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      cum = __fadd_rn(cum, ev[i]);
      if (ev[i] > 0.f) {
        last = i;
        zlast = zv[i];
      }
      if (sel < 0 && cum > t2) {
        sel = i;
        zsel = zv[i];
      }
    }
    if (sel < 0) {
      sel = last;
      zsel = zlast;
    }
    zsel_out = zsel;
    return sel >= 0 ? 4 * sel + k : -1;
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
    if (!RZ_DCHECK(g >= 0 && grp >= 0 && grp < p.S, 13)) return;
    p.part[g * p.S + grp] = make_float4(st.m, st.s, st.bz, 0.f);
    p.part_idx[g * p.S + grp] = st.bi;
  }
};

// Plain stores of the accumulator: bf16 (dH) or fp32 (logits), optionally
// fp32 accumulate (dW over token chunks, in chunk order).
template <int kMode>  // 0: bf16 store, 1: fp32 store, 2: fp32 accumulate-or-store,
                     // 3: bf16 store of the row times rowscale[row]
struct EpiStore {
  struct Params {
    void* out;
    long long ld;    // row stride in elements
    long long row0;  // row offset into out
    long long rows;  // valid rows (block-local numbering)
    int cols;        // valid columns
    int accumulate;  // mode 2 only
    const float* rowscale;  // mode 3 only: [rows] (block-local)
  };
  struct State {};

  static __device__ __forceinline__ void task_begin(const Params&, State&, int, int, int) {}
  static __device__ __forceinline__ void task_end(const Params&, State&, int, int, int) {}

  static __device__ __forceinline__ void chunk(const Params& p, const uint32_t (&r)[32], long long rr,
                                               int cbase) {
    if (!RZ_DCHECK(rr >= 0 && rr < p.rows && cbase >= 0 && cbase < p.cols && p.cols <= p.ld, 14))
      return;
    if (kMode == 0 || kMode == 3) {
      const float sc = kMode == 3 ? p.rowscale[rr] : 1.f;
      uint16_t* dst = static_cast<uint16_t*>(p.out) + (p.row0 + rr) * p.ld + cbase;
      if (cbase + 32 <= p.cols) {
        uint32_t w[16];
#pragma unroll
        for (int j = 0; j < 16; ++j)
          w[j] = kMode == 3 ? pack_bf16x2(__fmul_rn(sc, __uint_as_float(r[2 * j])),
                                          __fmul_rn(sc, __uint_as_float(r[2 * j + 1])))
                            : pack_bf16x2(__uint_as_float(r[2 * j]), __uint_as_float(r[2 * j + 1]));
#pragma unroll
        for (int q = 0; q < 4; ++q)
          st_global_v4(dst + 8 * q, w[4 * q], w[4 * q + 1], w[4 * q + 2], w[4 * q + 3]);
      } else {
        for (int j = 0; j < 32; ++j)
          if (cbase + j < p.cols)
            dst[j] = static_cast<uint16_t>(
                pack_bf16x2(kMode == 3 ? __fmul_rn(sc, __uint_as_float(r[j])) : __uint_as_float(r[j]),
                            0.f) &
                0xffffu);
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
__device__ __forceinline__ float merge_finish(float M, float sum, int V, int a, const float* zg,
                                              float* l_out, int* err) {
  if (a < 0 || a >= V) {
    if (err) atomicOr(err, 1);
    *l_out = __int_as_float(0x7fc00000);
    return *l_out;
  }
  *l_out = lse_from(M, sum);
  return logprob_from(*zg, M, sum);
}
__device__ __forceinline__ float merge_row(const float2* pp, int S, int V, int a,
                                           const float* zg, float* l_out, int* err) {
  float sum;
  const float M = lse_merge_parts(pp, S, &sum);
  return merge_finish(M, sum, V, a, zg, l_out, err);
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
// With a per-row reference (ref, the kept terms e' = 2^((z - R) log2 e) in
// bf16): coef becomes the row factor sigma_t = c_t e^(R_t - lse_t) of
// dz_tv = sigma_t e'_tv, and the sampled column's term is overwritten with
// expm1(log pi_t) e^(lse_t - R_t), so that sigma_t times it is
// c_t expm1(log pi_t) (no cancellation of p - 1 as p -> 1).  |lse - R|
// above kRefGap raises RZ_DEVERR_RANGE (sigma would lose its digits).
constexpr float kRefGap = 60.f;  // nats

__global__ void lse_merge_coef_kernel(long long rows, int V, int S, long long row0,
                                      const int32_t* __restrict__ tokens,
                                      const float2* __restrict__ part,
                                      const float* __restrict__ zgather,
                                      float* __restrict__ logprob, float* __restrict__ lse_ws,
                                      const float* __restrict__ logmu,
                                      const int64_t* __restrict__ cu,
                                      const float2* __restrict__ fac,
                                      const uint8_t* __restrict__ mask, int B,
                                      float* __restrict__ coef, const float* __restrict__ ref,
                                      uint16_t* __restrict__ ez, long long lde, int* err) {
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
  const float c = act ? f.x * w * f.y : 0.f;
  if (!ref) {
    coef[t] = c;
    return;
  }
  const float R = ref[t];
  const float gap = __fsub_rn(l, R);
  if (!(fabsf(gap) <= kRefGap) && err) atomicOr(err, kErrRange);
  coef[t] = __fmul_rn(c, expf(-gap));
  const int a = tokens[t];
  if (a >= 0 && a < V)
    ez[t * lde + a] = static_cast<uint16_t>(pack_bf16x2(__fmul_rn(expm1f(lp), expf(gap)), 0.f) &
                                            0xffffu);
}

// H'[r, :] = sigma_r H[row0 + r, :] in bf16 for the rows of one chunk: the B
// operand of dW = e'^T H' when the kept terms are taken against a per-row
// reference.  One CTA per row, 16-byte vectors (d % 8 == 0).
__global__ void scale_rows_kernel(const uint16_t* __restrict__ H, long long row0, int d,
                                  const float* __restrict__ sigma, uint16_t* __restrict__ Hs) {
  const long long r = blockIdx.x;
  const float sg = sigma[r];
  const uint4* src = reinterpret_cast<const uint4*>(H + (row0 + r) * d);
  uint4* dst = reinterpret_cast<uint4*>(Hs + r * d);
  for (int i = threadIdx.x; i < (d >> 3); i += blockDim.x) {
    const uint4 q = __ldg(src + i);
    const uint32_t in[4] = {q.x, q.y, q.z, q.w};
    uint32_t o[4];
#pragma unroll
    for (int j = 0; j < 4; ++j)
      o[j] = pack_bf16x2(__fmul_rn(sg, __uint_as_float(in[j] << 16)),
                         __fmul_rn(sg, __uint_as_float(in[j] & 0xffff0000u)));
    dst[i] = make_uint4(o[0], o[1], o[2], o[3]);
  }
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

// The split level of the sampler's reservoir for one row, given the row's
// maximum M and the splits' factors f(g) = e^(m_g - M) (lse_merge_factor):
// splits in order, the running sum R of their totals (scaled to the row's
// maximum as the log-sum-exp scales them), the sample replaced by split g's
// candidate when U3 R < its total (u(g) = U3 of split g).
template <class F, class U>
__device__ __forceinline__ int sample_merge_pick(const float4* pp, const int* pidx, int S,
                                                 const F& f, const U& u, float* bz_out) {
  float R = 0.f, bz = 0.f;
  int bi = 0;
  for (int g = 0; g < S; ++g) {
    const float w = __fmul_rn(pp[g].y, f(g));
    R = __fadd_rn(R, w);
    if (__fmul_rn(u(g), R) < w && pidx[g] >= 0) {
      bi = pidx[g];
      bz = pp[g].z;
    }
  }
  *bz_out = bz;
  return bi;
}

// U3 of split g: word 0 of Philox at counter (split, row id lo, row id hi, 1).
__device__ __forceinline__ float split_uniform(int g, uint32_t rlo, uint32_t rhi, uint32_t k0,
                                               uint32_t k1) {
  uint32_t x[4];
  philox4x32_10(static_cast<uint32_t>(g), rlo, rhi, 1u, k0, k1, x);
  return uniform_of(x[0]);
}

// One thread per row: the log-sum-exp exactly as lse_merge_kernel, then the
// split level of the reservoir (sample_merge_pick).
__global__ void sample_merge_kernel(long long T, int S, const float4* __restrict__ part,
                                    const int* __restrict__ part_idx,
                                    const int64_t* __restrict__ row_ids, uint32_t k0, uint32_t k1,
                                    int32_t* __restrict__ tokens, float* __restrict__ logprob,
                                    float* __restrict__ lse) {
  const long long t = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (t >= T) return;
  const float4* pp = part + t * S;
  float sum;
  const float M = lse_merge_parts(pp, S, &sum);
  const unsigned long long rid =
      static_cast<unsigned long long>(row_ids ? row_ids[t] : static_cast<int64_t>(t));
  const uint32_t rlo = static_cast<uint32_t>(rid & 0xffffffffull);
  const uint32_t rhi = static_cast<uint32_t>(rid >> 32);
  float bz;
  tokens[t] = sample_merge_pick(
      pp, part_idx + t * S, S, [&](int g) { return lse_merge_factor(pp[g].x, M); },
      [&](int g) { return split_uniform(g, rlo, rhi, k0, k1); }, &bz);
  logprob[t] = logprob_from(bz, M, sum);
  if (lse) lse[t] = lse_from(M, sum);
}

// ============================================================== decode mode
// The logprob pass over stored logits z ([T, ldz] fp32, ldz a multiple of 64
// and >= V, so a chunk's 32 loads stay inside its row): one warp per
// (vocabulary split, row), one cluster of kDecCluster CTAs per row.  The
// fused epilogue folds a split's 32-column chunks one after the other; here
// its steps are taken apart, a round of 32 chunks at a time (lane l holding
// chunk l of the round): every lane takes its chunk's maximum, a running
// maximum over the chunks in order gives each chunk the m its terms are
// summed against and the factor that rescales s when the maximum grows,
// every lane sums its chunk against that m, and the rescales and additions
// of s then run in chunk order.  The same operations on the same values
// (fold32_max, fold32_scale, fold32_sum), so the same bits as the fused
// pass.  The split states then go through distributed shared memory to the
// cluster's first CTA, which merges them in split order as the merge
// kernels do (lse_merge_max, lse_merge_factor, the same sums in the same
// order), with the splits' factors evaluated on the lanes of one warp.  The
// logits GEMM and this kernel are launched with programmatic stream
// serialization, so each starts while the kernel ahead of it finishes and
// waits (griddepcontrol) only before touching memory.
constexpr int kDecWarps = 8;    // warps per CTA, one vocabulary split each
constexpr int kDecCluster = 8;  // CTAs per row
static_assert(kDecWarps * kDecCluster >= kMaxVocabSplits, "one warp per split");

// Columns [c0, c0 + 32 C) of split grp (C: its chunks that start below V).
__device__ __forceinline__ int dec_split_chunks(int grp, int tps, int n_tiles, int V, int* c0) {
  *c0 = grp * tps * kBN;
  int c_end = (grp + 1) * tps * kBN;
  if (c_end > n_tiles * kBN) c_end = n_tiles * kBN;
  if (c_end > V) c_end = V;
  return (c_end - *c0 + 31) / 32;
}

// The lane's chunk (columns cs .. cs + 31) of row zr; -inf past V and for a
// lane without a chunk.
__device__ __forceinline__ void dec_load(const float* zr, int cs, bool have, int V,
                                         float (&v)[32]) {
  if (have) {
    const float4* src = reinterpret_cast<const float4*>(zr + cs);
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const float4 q = __ldg(src + i);
      v[4 * i] = q.x;
      v[4 * i + 1] = q.y;
      v[4 * i + 2] = q.z;
      v[4 * i + 3] = q.w;
    }
    if (cs + 32 > V) {
#pragma unroll
      for (int j = 0; j < 32; ++j)
        if (cs + j >= V) v[j] = -INFINITY;
    }
  } else {
#pragma unroll
    for (int j = 0; j < 32; ++j) v[j] = -INFINITY;
  }
}

// One round of nk chunks (lane l: the round's chunk l, loaded in v): the
// fold's state (m_run, s) carried through them in order.  Returns the lane's
// chunk sum w (against the running maximum after its chunk); e and acc get
// its terms and class sums (kKeep); s_mine gets s right after the lane's own
// chunk.
template <bool kKeep>
__device__ __forceinline__ float dec_round(const float (&v)[32], bool have, int nk, int lane,
                                           float& m_run, float& s, float (&e)[32],
                                           float (&acc)[4], float& s_mine) {
  const float cm = have ? fold32_max(v) : -INFINITY;
  // M_k: the running maximum after chunk k (max is exact in any order)
  float incl = cm;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const float t = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl = fmaxf(incl, t);
  }
  incl = fmaxf(incl, m_run);
  float prev = __shfl_up_sync(0xffffffffu, incl, 1);  // M_{k-1}
  if (lane == 0) prev = m_run;
  const float w = have ? fold32_sum<kKeep>(v, incl, e, acc) : 0.f;
  // fold32_rescale(M_{k-1}, s, cm) of every chunk: the factors first, on
  // all lanes at once, then s through the chunks in order
  const bool up = cm > prev;
  const float f = up ? fold32_scale(prev, cm) : 1.f;
  const unsigned upm = __ballot_sync(0xffffffffu, up);
#pragma unroll
  for (int j = 0; j < 32; ++j) {
    if (j < nk) {  // warp-uniform
      const float fj = __shfl_sync(0xffffffffu, f, j);
      const float wj = __shfl_sync(0xffffffffu, w, j);
      if ((upm >> j) & 1u) s = __fmul_rn(s, fj);
      s = __fadd_rn(s, wj);
      if (lane == j) s_mine = s;
    }
  }
  m_run = __shfl_sync(0xffffffffu, incl, 31);
  return w;
}

// The row's maximum over the split states in order (every lane) and the
// splits' factors against it (fs[g], written by lane g % 32).
template <class P>
__device__ __forceinline__ float dec_merge_factors(const P* parts, int S, int lane, float* fs) {
  const float M = lse_merge_max(parts, S);
  for (int g = lane; g < S; g += 32) fs[g] = lse_merge_factor(parts[g].x, M);
  __syncwarp();
  return M;
}

__global__ void __cluster_dims__(kDecCluster, 1, 1) __launch_bounds__(kDecWarps * 32, 1)
    decode_logprob_kernel(const float* __restrict__ z, long long ldz, int V, int S, int tps,
                          int n_tiles, const int32_t* __restrict__ tokens,
                          float* __restrict__ logprob, float* __restrict__ lse,
                          float* __restrict__ lse_ws, int* err) {
  grid_dep_launch();  // a following call's GEMM may start its set-up
  grid_dep_wait();    // the logits GEMM ahead of this kernel has finished
  __shared__ float2 parts[kDecWarps * kDecCluster];
  __shared__ float fs[kDecWarps * kDecCluster];
  __shared__ float za;
  cg::cluster_group cluster = cg::this_cluster();
  const unsigned rank = cluster.block_rank();
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int grp = static_cast<int>(rank) * kDecWarps + warp;
  const long long g = blockIdx.y;
  const int a = __ldg(tokens + g);
  if (grp < S) {
    const float* zr = z + g * ldz;
    int c0;
    const int C = dec_split_chunks(grp, tps, n_tiles, V, &c0);
    float m_run = -INFINITY, s = 0.f;
    for (int base = 0; base < C; base += 32) {
      const int k = base + lane;
      const bool have = k < C;
      const int cs = c0 + 32 * k;
      float v[32], e[32], acc[4], s_mine;
      dec_load(zr, cs, have, V, v);
      const unsigned rel = static_cast<unsigned>(a - cs);
      if (have && rel < 32u) {
        float zv = 0.f;
#pragma unroll
        for (int j = 0; j < 32; ++j)
          if (rel == static_cast<unsigned>(j)) zv = v[j];
        *cluster.map_shared_rank(&za, 0) = zv;
      }
      dec_round<false>(v, have, C - base < 32 ? C - base : 32, lane, m_run, s, e, acc, s_mine);
    }
    if (lane == 0 && RZ_DCHECK(grp < kDecWarps * kDecCluster, 14))
      *cluster.map_shared_rank(&parts[grp], 0) = make_float2(m_run, s);
  }
  cluster.sync();
  if (rank != 0 || warp != 0) return;
  const float M = dec_merge_factors(parts, S, lane, fs);
  if (lane != 0) return;
  float sum = 0.f;
  for (int q = 0; q < S; ++q) sum = fmaf(parts[q].y, fs[q], sum);
  float l;
  const float lp = merge_finish(M, sum, V, a, &za, &l, err);
  logprob[g] = lp;
  if (lse) lse[g] = l;
  if (lse_ws) lse_ws[g] = l;
}

// The fused sampler over stored logits: each warp folds its split as above,
// every chunk's terms kept while its round is in registers, the running sum
// after each chunk recorded by the chunk's lane; then each lane's replace
// decision (the epilogue's test, on the same Philox words) and, for a
// replacing chunk, the same in-chunk draw (EpiSample::draw_in_chunk).  The
// split's sample is the draw of the last chunk that replaced, as in the
// epilogue's walk.  The merge takes the split level of the reservoir as
// sample_merge_kernel does (sample_merge_pick), the Philox words of the
// splits drawn on the lanes of one warp.  The same bits as the fused pass.
__global__ void __cluster_dims__(kDecCluster, 1, 1) __launch_bounds__(kDecWarps * 32, 1)
    decode_sample_kernel(const float* __restrict__ z, long long ldz, int V, int S, int tps,
                         int n_tiles, const int64_t* __restrict__ row_ids, uint32_t k0,
                         uint32_t k1, int32_t* __restrict__ tokens, float* __restrict__ logprob,
                         float* __restrict__ lse) {
  grid_dep_launch();  // a following call's GEMM may start its set-up
  grid_dep_wait();    // the logits GEMM ahead of this kernel has finished
  __shared__ float4 parts[kDecWarps * kDecCluster];
  __shared__ int pidx[kDecWarps * kDecCluster];
  __shared__ float fs[kDecWarps * kDecCluster];
  __shared__ float us[kDecWarps * kDecCluster];
  cg::cluster_group cluster = cg::this_cluster();
  const unsigned rank = cluster.block_rank();
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int grp = static_cast<int>(rank) * kDecWarps + warp;
  const long long g = blockIdx.y;
  const unsigned long long rid =
      static_cast<unsigned long long>(row_ids ? __ldg(row_ids + g) : static_cast<int64_t>(g));
  const uint32_t rlo = static_cast<uint32_t>(rid & 0xffffffffull);
  const uint32_t rhi = static_cast<uint32_t>(rid >> 32);
  if (grp < S) {
    const float* zr = z + g * ldz;
    int c0;
    const int C = dec_split_chunks(grp, tps, n_tiles, V, &c0);
    PhiloxRow rng;
    rng.init(rlo, rhi, k0, k1);
    float m_run = -INFINITY, s = 0.f;
    int bi = -1;
    float bz = 0.f;
    for (int base = 0; base < C; base += 32) {
      const int k = base + lane;
      const bool have = k < C;
      const int cs = c0 + 32 * k;
      float v[32], e[32], acc[4];
      float s_mine = 0.f;
      dec_load(zr, cs, have, V, v);
      const float w =
          dec_round<true>(v, have, C - base < 32 ? C - base : 32, lane, m_run, s, e, acc, s_mine);
      bool rep = false;
      int off = -1;
      float zs = 0.f;
      if (have) {
        uint32_t x[4];
        rng.words(static_cast<uint32_t>(cs) >> 5, x);
        rep = __fmul_rn(uniform_of(x[0]), s_mine) < w;
        if (rep) off = EpiSample::draw_in_chunk(v, e, acc, w, x[1], zs);
      }
      const unsigned take = __ballot_sync(0xffffffffu, rep && off >= 0);
      if (take) {
        const int src_lane = 31 - __clz(static_cast<int>(take));
        const int off_l = __shfl_sync(0xffffffffu, off, src_lane);
        const float zs_l = __shfl_sync(0xffffffffu, zs, src_lane);
        bi = c0 + 32 * (base + src_lane) + off_l;
        bz = zs_l;
      }
    }
    if (lane == 0 && RZ_DCHECK(grp < kDecWarps * kDecCluster, 15)) {
      *cluster.map_shared_rank(&parts[grp], 0) = make_float4(m_run, s, bz, 0.f);
      *cluster.map_shared_rank(&pidx[grp], 0) = bi;
    }
  }
  cluster.sync();
  if (rank != 0 || warp != 0) return;
  for (int q = lane; q < S; q += 32) us[q] = split_uniform(q, rlo, rhi, k0, k1);
  const float M = dec_merge_factors(parts, S, lane, fs);  // ends with __syncwarp
  if (lane != 0) return;
  float sum = 0.f;
  for (int q = 0; q < S; ++q) sum = fmaf(parts[q].y, fs[q], sum);
  float bz;
  tokens[g] = sample_merge_pick(
      parts, pidx, S, [&](int q) { return fs[q]; }, [&](int q) { return us[q]; }, &bz);
  logprob[g] = logprob_from(bz, M, sum);
  if (lse) lse[g] = lse_from(M, sum);
}

// ============================================================== launchers
namespace {

// Launch a GEMM: one persistent CTA per SM (or per task, if fewer).
template <class Epi, bool kAMN, bool kBMN>
cudaError_t run_gemm(const CUtensorMap& a, const CUtensorMap& b, const GemmSched& s,
                     const typename Epi::Params& p, cudaStream_t st, bool overlap = false) {
  if (s.num_tasks <= 0) return cudaSuccess;
  auto kern = gemm_kernel<Epi, kAMN, kBMN>;
  cudaError_t e =
      cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
  if (e != cudaSuccess) return e;
  const int grid = s.num_tasks < num_sms() ? s.num_tasks : num_sms();
  if (!overlap) {
    kern<<<grid, kThreads, kSmemBytes, st>>>(a, b, s, p);
    return cudaGetLastError();
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(grid));
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = kSmemBytes;
  cfg.stream = st;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = at;
  cfg.numAttrs = 1;
  e = cudaLaunchKernelEx(&cfg, kern, a, b, s, p);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

// A small kernel launched to overlap the tail of the kernel ahead of it
// (it starts with grid_dep_wait).
template <class K, class... Args>
cudaError_t launch_overlapped(K kern, dim3 grid, dim3 block, cudaStream_t st, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.stream = st;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = at;
  cfg.numAttrs = 1;
  cudaError_t e = cudaLaunchKernelEx(&cfg, kern, args...);
  if (e != cudaSuccess) return e;
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
                               int* err, cudaStream_t st, uint32_t a_rows) {
  const int S = vocab_splits(V);
  for (int64_t r0 = 0; r0 < T; r0 += kChunkRowsMax) {
    const int64_t rows = (T - r0) < kChunkRowsMax ? (T - r0) : kChunkRowsMax;
    GemmSched s = sched_of(rows, V, S, d, err);
    s.tiles_per_group = vocab_tiles_per_split(V);
    s.m_group = vocab_raster_group();
    s.a_m_off = static_cast<int>(r0);
    s.a_bytes = a_rows * kBK * 2u;
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
                          int32_t* tokens, float* logprob, float* lse, int* err, cudaStream_t st,
                          uint32_t a_rows) {
  const int S = vocab_splits(V);
  for (int64_t r0 = 0; r0 < T; r0 += kChunkRowsMax) {  // row blocks as in launch_lse_partial
    const int64_t rows = (T - r0) < kChunkRowsMax ? (T - r0) : kChunkRowsMax;
    GemmSched s = sched_of(rows, V, S, d, err);
    s.tiles_per_group = vocab_tiles_per_split(V);
    s.m_group = vocab_raster_group();
    s.a_m_off = static_cast<int>(r0);
    s.a_bytes = a_rows * kBK * 2u;
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
  sample_merge_kernel<<<static_cast<unsigned>(blocks), threads, 0, st>>>(
      T, S, part, part_idx, row_ids, static_cast<uint32_t>(seed & 0xffffffffull),
      static_cast<uint32_t>(seed >> 32), tokens, logprob, lse);
  return cudaGetLastError();
}

cudaError_t launch_lse_keep(const CUtensorMap& tmH, const CUtensorMap& tmW, int64_t row0,
                            int64_t rows, int d, int V, const int32_t* tokens, float2* part,
                            float* zgather, const CUtensorMap& tmE16, float* emax, int64_t ldm,
                            const float* ref, int* err, cudaStream_t st, uint32_t a_rows) {
  const int S = vocab_splits(V);
  GemmSched s = sched_of(rows, V, S, d, err);
  s.tiles_per_group = vocab_tiles_per_split(V);
  s.m_group = vocab_raster_group();
  s.a_m_off = static_cast<int>(row0);
  s.a_bytes = a_rows * kBK * 2u;
  const EpiLsePartial::Params lp{tokens, part, zgather, static_cast<long long>(rows), V, S};
  if (ref) {
    EpiLseKeepRef::Params p{tmE16, lp, nullptr, ldm, ref, err};
    return run_gemm<EpiLseKeepRef, false, false>(tmH, tmW, s, p, st);
  }
  EpiLseKeep::Params p{tmE16, lp, emax, ldm, nullptr, err};
  return run_gemm<EpiLseKeep, false, false>(tmH, tmW, s, p, st);
}

cudaError_t launch_scale_rows(const uint16_t* H, int64_t row0, int64_t rows, int d,
                              const float* sigma, uint16_t* Hs, cudaStream_t st) {
  if (rows <= 0) return cudaSuccess;
  scale_rows_kernel<<<static_cast<unsigned>(rows), 256, 0, st>>>(H, row0, d, sigma, Hs);
  return cudaGetLastError();
}

cudaError_t launch_lse_merge_coef(int64_t row0, int64_t rows, int V, const int32_t* tokens,
                                  const float2* part, const float* zgather, float* logprob,
                                  float* lse_ws, const float* logmu, const int64_t* cu,
                                  const float2* fac, const uint8_t* mask, int B, float* coef,
                                  const float* ref, uint16_t* ez, int64_t lde, int* err,
                                  cudaStream_t st) {
  if (rows <= 0) return cudaSuccess;
  const int threads = 256;
  const long long blocks = (rows + threads - 1) / threads;
  lse_merge_coef_kernel<<<static_cast<unsigned>(blocks), threads, 0, st>>>(
      rows, V, vocab_splits(V), row0, tokens, part, zgather, logprob, lse_ws, logmu, cu, fac,
      mask, B, coef, ref, ez, lde, err);
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
                              int V, float* out, int* err, cudaStream_t st, uint32_t a_rows) {
  const int S = vocab_splits(V);
  for (int64_t r0 = 0; r0 < T; r0 += kChunkRowsMax) {  // row blocks as in launch_lse_partial
    const int64_t rows = (T - r0) < kChunkRowsMax ? (T - r0) : kChunkRowsMax;
    GemmSched s = sched_of(rows, V, S, d, err);
    s.tiles_per_group = vocab_tiles_per_split(V);
    s.m_group = vocab_raster_group();
    s.a_m_off = static_cast<int>(r0);
    s.a_bytes = a_rows * kBK * 2u;
    EpiStore<1>::Params p{out, V, r0, rows, V, 0};
    cudaError_t e = run_gemm<EpiStore<1>, false, false>(tmH, tmW, s, p, st);
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

cudaError_t launch_dH(const CUtensorMap& tmDz, const CUtensorMap& tmWmn, int64_t row0,
                      int64_t rows, int d, int V, uint16_t* dH, const float* rowscale, int* err,
                      cudaStream_t st) {
  const int nt = (d + kBN - 1) / kBN;
  GemmSched s = sched_of(rows, d, nt, V, err);
  if (rowscale) {
    EpiStore<3>::Params p{dH, d, row0, rows, d, 0, rowscale};
    return run_gemm<EpiStore<3>, false, true>(tmDz, tmWmn, s, p, st);
  }
  EpiStore<0>::Params p{dH, d, row0, rows, d, 0, nullptr};
  return run_gemm<EpiStore<0>, false, true>(tmDz, tmWmn, s, p, st);
}

cudaError_t launch_decode_logits(const CUtensorMap& tmH, const CUtensorMap& tmW, int64_t T, int d,
                                 int V, float* z, int* err, cudaStream_t st, uint32_t a_rows) {
  const int nt = vocab_tiles(V);
  GemmSched s = sched_of(T, V, nt, d, err);  // one 256-column tile per task
  s.m_group = s.m_blocks;                    // a tile's row blocks run together
  s.a_bytes = a_rows * kBK * 2u;
  EpiStore<1>::Params p{z, decode_ld(V), 0, static_cast<long long>(T), V, 0};
  return run_gemm<EpiStore<1>, false, false>(tmH, tmW, s, p, st, true);
}

cudaError_t launch_decode_logprob(const float* z, int64_t T, int V, const int32_t* tokens,
                                  float* logprob, float* lse, float* lse_ws, int* err,
                                  cudaStream_t st) {
  if (T <= 0) return cudaSuccess;
  const dim3 grid(kDecCluster, static_cast<unsigned>(T));
  return launch_overlapped(decode_logprob_kernel, grid, dim3(kDecWarps * 32), st,
                           z, static_cast<long long>(decode_ld(V)), V, vocab_splits(V),
                           vocab_tiles_per_split(V), vocab_tiles(V), tokens, logprob, lse,
                           lse_ws, err);
}

cudaError_t launch_decode_sample(const float* z, int64_t T, int V, const int64_t* row_ids,
                                 uint64_t seed, int32_t* tokens, float* logprob, float* lse,
                                 cudaStream_t st) {
  if (T <= 0) return cudaSuccess;
  const uint32_t k0 = static_cast<uint32_t>(seed & 0xffffffffull);
  const uint32_t k1 = static_cast<uint32_t>(seed >> 32);
  const dim3 grid(kDecCluster, static_cast<unsigned>(T));
  return launch_overlapped(decode_sample_kernel, grid, dim3(kDecWarps * 32), st,
                           z, static_cast<long long>(decode_ld(V)), V, vocab_splits(V),
                           vocab_tiles_per_split(V), vocab_tiles(V), row_ids, k0, k1, tokens,
                           logprob, lse);
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

cudaError_t launch_dW(const CUtensorMap& tmDzMn, const CUtensorMap& tmHmn, int64_t b_row0,
                      int64_t rows, int d, int V, float* dW, bool accumulate, int* err,
                      cudaStream_t st) {
  const int nt = (d + kBN - 1) / kBN;
  GemmSched s = sched_of(V, d, nt, rows, err);
  s.b_k_off = static_cast<int>(b_row0);
  EpiStore<2>::Params p{dW, d, 0, V, d, accumulate ? 1 : 0};
  return run_gemm<EpiStore<2>, true, true>(tmDzMn, tmHmn, s, p, st);
}

}  // namespace rz
