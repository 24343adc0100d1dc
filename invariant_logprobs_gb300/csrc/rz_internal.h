// rz_internal.h -- host-side declarations shared by the library's
// translation units (not part of the public ABI).
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

#include "rz_gemm.cuh"

namespace rz {

// Vocabulary split of the logprob pass: a function of V only (never of the
// number of rows), so the per-row reduction order is batch-invariant.  Up to
// 64 splits (~9 tiles each at V = 151936) let a decode-sized batch of one
// 128-row block still occupy 64 SMs.
constexpr int kMaxVocabSplits = 64;
inline int vocab_tiles(int V) { return (V + kBN - 1) / kBN; }
inline int vocab_tiles_per_split(int V) {
  const int nt = vocab_tiles(V);
  const int s = nt < kMaxVocabSplits ? nt : kMaxVocabSplits;
  return (nt + s - 1) / s;
}
inline int vocab_splits(int V) {
  const int nt = vocab_tiles(V);
  const int tps = vocab_tiles_per_split(V);
  return (nt + tps - 1) / tps;
}

// Rows per backward chunk: the chunk's kept terms (fp16, overwritten in place
// by bf16 dz, with one fp32 running max per 32 columns; or bf16 against the
// reference) live in the workspace.
constexpr int64_t kChunkRowsMax = 38912;  // 256 * 152
int64_t chunk_rows(int32_t V);
inline int64_t dz_ld(int32_t V) { return (static_cast<int64_t>(V) + 7) / 8 * 8; }
inline int64_t emax_ld(int32_t V) { return (static_cast<int64_t>(V) + 127) / 128 * 4; }

// ---- argument checks and the logprob pass's scratch layout, shared by
// every entry point that runs that pass (rz_api.cu, rz_noalloc.cu)
inline size_t al256(size_t x) { return (x + 255) / 256 * 256; }
inline bool a16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
inline bool a256(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 255u) == 0; }
inline bool sizes_ok(int64_t T, int32_t d, int32_t V) {
  return T >= 0 && T < (int64_t(1) << 31) && V >= 1 && V <= (1 << 24) && d >= 8 && d <= 65536;
}
struct FwdLayout {  // logprob pass scratch: split states [T, S], gathered logit [T]
  size_t part, zg, total;
};
inline FwdLayout fwd_layout(int64_t T, int32_t V) {
  FwdLayout L{};
  const size_t t = T > 0 ? static_cast<size_t>(T) : 0;
  L.part = 0;
  L.zg = al256(t * vocab_splits(V) * sizeof(float2));
  L.total = L.zg + al256(t * sizeof(float));
  return L;
}

// Decode-sized batches (at most kDecodeRows rows, with a logits scratch of
// at most kDecodeBytes): the logprob pass first computes the fp32 logits
// with one 256-column tile per task -- every SM streams W, where one task
// per (row block, vocab split) keeps only 60 SMs busy -- into the
// workspace, then a fold kernel takes the fused epilogue's per-row fold over
// them with the same operations in the same order: the same bits.
// (1-7 rows: 0.175 -> 0.150 ms at d = 2560; 64 rows about even; 128 rows
// slower, as the fold grows with the rows while the GEMM does not)
constexpr int64_t kDecodeRows = 64;
constexpr size_t kDecodeBytes = size_t(256) << 20;
inline int64_t decode_ld(int32_t V) { return (static_cast<int64_t>(V) + 63) / 64 * 64; }
inline bool decode_mode(int64_t T, int32_t V) {
  return T > 0 && T <= kDecodeRows &&
         static_cast<size_t>(T) * static_cast<size_t>(decode_ld(V)) * 4 <= kDecodeBytes;
}
// the logits scratch, appended to the pass's workspace (0 outside decode mode)
inline size_t decode_bytes(int64_t T, int32_t V) {
  return decode_mode(T, V) ? al256(static_cast<size_t>(T) * static_cast<size_t>(decode_ld(V)) * 4)
                           : 0;
}

int num_sms();
bool device_ok();  // current device is sm_103 (or newer family member we compiled for)

bool make_tmap_bf16(CUtensorMap* tm, const void* base, uint64_t inner, uint64_t outer,
                    uint64_t row_stride_bytes, uint32_t box_inner, uint32_t box_outer);

// ---- launch-class timing (rz_profile.cu): while rz_profile_begin() is in
// effect, brackets the launches made in its lifetime with CUDA events on
// `st` (classes RZ_PROF_*, `launches` kernels); otherwise does nothing.
class ProfScope {
 public:
  ProfScope(int cls, int launches, cudaStream_t st);
  ~ProfScope();
  ProfScope(const ProfScope&) = delete;
  ProfScope& operator=(const ProfScope&) = delete;

 private:
  int cls_, launches_;
  cudaStream_t st_;
  void* e0_;
};

// ---- debug build (-DRZ_CHECKS): each unit's count of failed device bounds
// checks and the site of the first one, read and cleared (0 and 0 in the
// normal build)
cudaError_t check_read_lmhead(unsigned int* count, int* site);
cudaError_t check_read_logits(unsigned int* count, int* site);

// ---- lm-head kernels (rz_lmhead.cu)
// Rows of the K-major A box (the hidden states) of a call over T rows: a
// batch of fewer than 128 rows loads exactly its own rows (a box lying past
// the last row is slow to fill: 0.23-0.26 vs 0.15-0.18 ms for one row), the
// GEMM keeps the rest of its A stages zero.  The tensor map of H and the
// launch take the same value.
inline uint32_t a_box_rows(int64_t T) {
  return T < 1 ? 1u : (T < kBM ? static_cast<uint32_t>(T) : static_cast<uint32_t>(kBM));
}
cudaError_t launch_lse_partial(const CUtensorMap& tmH, const CUtensorMap& tmW, int64_t T, int d,
                               int V, const int32_t* tokens, float2* part, float* zgather,
                               int* err, cudaStream_t st, uint32_t a_rows);
cudaError_t launch_lse_merge(int64_t T, int V, const int32_t* tokens, const float2* part,
                             const float* zgather, float* logprob, float* lse, float* lse_ws,
                             int* err, cudaStream_t st);
cudaError_t launch_sample(const CUtensorMap& tmH, const CUtensorMap& tmW, int64_t T, int d, int V,
                          const int64_t* row_ids, uint64_t seed, float4* part, int* part_idx,
                          int32_t* tokens, float* logprob, float* lse, int* err, cudaStream_t st,
                          uint32_t a_rows);
// tmE16: the chunk's kept terms [rows, V] (row stride dz_ld(V)), box 64 x 32:
// fp16 with running maxima in emax, or (ref != null) bf16 against the
// per-row reference ref [rows] (chunk-local), no maxima.
cudaError_t launch_lse_keep(const CUtensorMap& tmH, const CUtensorMap& tmW, int64_t row0,
                            int64_t rows, int d, int V, const int32_t* tokens, float2* part,
                            float* zgather, const CUtensorMap& tmE16, float* emax, int64_t ldm,
                            const float* ref, int* err, cudaStream_t st, uint32_t a_rows);
// Hs[r, :] = sigma[r] H[row0 + r, :] (bf16) for one chunk's rows.
cudaError_t launch_scale_rows(const uint16_t* H, int64_t row0, int64_t rows, int d,
                              const float* sigma, uint16_t* Hs, cudaStream_t st);
cudaError_t launch_lse_merge_coef(int64_t row0, int64_t rows, int V, const int32_t* tokens,
                                  const float2* part, const float* zgather, float* logprob,
                                  float* lse_ws, const float* logmu, const int64_t* cu,
                                  const float2* fac, const uint8_t* mask, int B, float* coef,
                                  const float* ref, uint16_t* ez, int64_t lde, int* err,
                                  cudaStream_t st);
cudaError_t launch_dz_rows(uint16_t* ez, int64_t lde, const float* emax, int64_t ldm,
                           int64_t rows, int V, const int32_t* tokens, const float* lse,
                           const float* coef, const float* logpi, cudaStream_t st);
cudaError_t launch_logits_f32(const CUtensorMap& tmH, const CUtensorMap& tmW, int64_t T, int d,
                              int V, float* out, int* err, cudaStream_t st, uint32_t a_rows);
// Decode mode (decode_mode(T, V)): z [T, decode_ld(V)] fp32 with one tile per
// task, then the fused epilogue's fold over it and the merge of the split
// states in one launch: log pi, lse (nullable) and lse_ws (nullable) as
// launch_lse_merge gives them ...
cudaError_t launch_decode_logits(const CUtensorMap& tmH, const CUtensorMap& tmW, int64_t T, int d,
                                 int V, float* z, int* err, cudaStream_t st, uint32_t a_rows);
cudaError_t launch_decode_logprob(const float* z, int64_t T, int V, const int32_t* tokens,
                                  float* logprob, float* lse, float* lse_ws, int* err,
                                  cudaStream_t st);
// ... or the fused sampler's fold and merge (sampled tokens, log mu, lse)
cudaError_t launch_decode_sample(const float* z, int64_t T, int V, const int64_t* row_ids,
                                 uint64_t seed, int32_t* tokens, float* logprob, float* lse,
                                 cudaStream_t st);
// rowscale (nullable, [rows]): dH rows multiplied by it before rounding.
cudaError_t launch_dH(const CUtensorMap& tmDz, const CUtensorMap& tmWmn, int64_t row0,
                      int64_t rows, int d, int V, uint16_t* dH, const float* rowscale, int* err,
                      cudaStream_t st);
// b_row0: the chunk's first row in the B operand (0 when it holds the chunk only).
cudaError_t launch_dW(const CUtensorMap& tmDzMn, const CUtensorMap& tmHmn, int64_t b_row0,
                      int64_t rows, int d, int V, float* dW, bool accumulate, int* err,
                      cudaStream_t st);

// ---- loss kernels (rz_loss.cu)
size_t is_loss_ws_bytes(int32_t B);
cudaError_t launch_group_advantage(const float* r, int B, int G, float* adv, cudaStream_t st);
// Bn: the number of responses the loss averages over (B, or the whole
// batch's count when the call holds one shard of it).
cudaError_t launch_is_loss(const float* logpi, const float* logmu, const int64_t* cu,
                           const float* adv, const uint8_t* mask, int B, int Bn, int64_t T,
                           float* loss, float* d3, float* coef, void* ws, int* err,
                           cudaStream_t st);
// Per-response factors (A_i, 1/(Bn T_i)) of the coefficient c_t = A_i w_t/(Bn T_i).
size_t resp_factors_ws_bytes(int32_t B);
cudaError_t launch_resp_factors(const int64_t* cu, const float* adv, const uint8_t* mask, int B,
                                int Bn, int64_t T, float2* fac, cudaStream_t st);
// out[i] = parts[0][i] + parts[1][i] + ... in that order (n_parts >= 1).
cudaError_t launch_sum_partials(const float* parts, int n_parts, int64_t count, float* out,
                                cudaStream_t st);
// Score Centering: fac[i].x -= mean of A over responses with fac[i].y > 0;
// the loss from log pi (ws: is_loss_ws_bytes(B)).
cudaError_t launch_sc_centre(float2* fac, int B, cudaStream_t st);
cudaError_t launch_sc_loss(const float* logpi, const int64_t* cu, const uint8_t* mask,
                           const float2* fac, int B, int64_t T, float* loss, void* ws, int* err,
                           cudaStream_t st);
cudaError_t launch_d3(const float* logpi, const float* logmu, int64_t T, float* d3,
                      cudaStream_t st);
cudaError_t launch_is_stats(const float* logpi, const float* logmu, int64_t T, float* out,
                            cudaStream_t st);

// ---- given-logits kernel (rz_logits.cu)
cudaError_t launch_logits_rows(uint16_t* logits, int64_t T, int V, const int32_t* tokens,
                               const float* logmu, const int64_t* cu, const float2* fac,
                               const uint8_t* mask, int B, float* logprob, int* err,
                               cudaStream_t st);

}  // namespace rz
