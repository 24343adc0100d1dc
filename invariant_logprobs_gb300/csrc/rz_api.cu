// rz_api.cu -- the C ABI declared in include/rz.h: argument checks,
// workspace carving, tensor-map construction and the launch sequence of
// each operation.  Every step of every operation runs in this library's own
// kernels; there is no host or library fallback.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <cstdint>
#include <cstring>
#include <mutex>
#include <vector>

#include "rz.h"
#include "rz_internal.h"

namespace rz {

// ------------------------------------------------------------------ device facts
int num_sms() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 1;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 1;
  return n > 0 ? n : 1;
}

bool device_ok() {
  int dev = 0, major = 0, minor = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return false;
  if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess)
    return false;
  if (cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
    return false;
  return major == 10 && minor == 3;  // the library is built for sm_103a only
}

int64_t chunk_rows(int32_t V) {
  // one chunk keeps rows x round_up(V, 8) terms (fp16 then bf16 dz on the
  // plain route, bf16 on the reference route) and, on the plain route, a
  // running max per 32 columns: at most 40 GiB together.  Both routes use
  // the plain route's (larger) bytes per row, so they chunk alike.
  const int64_t per_row = dz_ld(V) * 2 + emax_ld(V) * 4;
  int64_t rows = kChunkRowsMax;
  const int64_t cap = (int64_t(40) << 30) / (per_row > 0 ? per_row : 1);
  if (rows > cap) rows = cap / kBM * kBM;
  if (rows < kBM) rows = kBM;
  return rows;
}

// ------------------------------------------------------------------ tensor maps
namespace {
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;
}  // namespace

bool make_tmap_bf16(CUtensorMap* tm, const void* base, uint64_t inner, uint64_t outer,
                    uint64_t row_stride_bytes, uint32_t box_inner, uint32_t box_outer) {
  std::call_once(g_encode_once, [] {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q{};
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  });
  if (!g_encode) return false;
  if ((reinterpret_cast<uintptr_t>(base) & 15u) || (row_stride_bytes & 15u)) return false;
  cuuint64_t dims[2] = {inner, outer};
  cuuint64_t strides[1] = {row_stride_bytes};
  cuuint32_t box[2] = {box_inner, box_outer};
  cuuint32_t estr[2] = {1, 1};
  const CUresult r =
      g_encode(tm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides,
               box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

namespace {

// ------------------------------------------------------------------ workspace
struct SampleLayout {
  size_t part, idx, total;
};
SampleLayout sample_layout(int64_t T, int32_t V) {
  SampleLayout L{};
  const size_t t = T > 0 ? static_cast<size_t>(T) : 0;
  L.part = 0;
  L.idx = al256(t * vocab_splits(V) * sizeof(float4));
  L.total = L.idx + al256(t * vocab_splits(V) * sizeof(int));
  return L;
}

struct LearnLayout {
  int64_t rows;  // rows per chunk
  FwdLayout fwd;  // split states of one chunk
  size_t logpi, lse_ws, coef, resp, fac, emax, ez, hs, total;
};
// ref: the kept terms are taken against a per-row reference (no running
// maxima; the chunk's rows of H scaled by sigma, bf16, for the dW GEMM).
LearnLayout learn_layout(int64_t T, int32_t V, int32_t B, bool ref = false, int32_t d = 0) {
  LearnLayout L{};
  const size_t t = T > 0 ? static_cast<size_t>(T) : 0;
  int64_t rows = chunk_rows(V);
  if (T < rows) rows = (T + kBM - 1) / kBM * kBM;
  L.rows = rows;
  const size_t r = static_cast<size_t>(rows);
  L.fwd = fwd_layout(rows, V);
  L.logpi = L.fwd.total;
  L.lse_ws = L.logpi + al256(t * 4);
  L.coef = L.lse_ws + al256(r * 4);
  L.resp = L.coef + al256(r * 4);
  L.fac = L.resp + is_loss_ws_bytes(B);
  L.emax = L.fac + resp_factors_ws_bytes(B);
  L.ez = L.emax + (ref ? 0 : al256(r * static_cast<size_t>(emax_ld(V)) * 4));
  L.hs = L.ez + al256(r * static_cast<size_t>(dz_ld(V)) * 2);
  L.total = L.hs + (ref ? al256(r * static_cast<size_t>(d > 0 ? d : 0) * 2) : 0);
  return L;
}

inline int cuda_status(cudaError_t e) { return e == cudaSuccess ? RZ_OK : RZ_ERR_CUDA; }

#define RZ_TRY(expr)                                  \
  do {                                                \
    cudaError_t _e = (expr);                          \
    if (_e != cudaSuccess) return RZ_ERR_CUDA;        \
  } while (0)

// log pi for all T rows: identical launch sequence for rollout and learner.
// A decode-sized batch (decode_mode) given the scratch after the pass's own
// workspace takes the logits through it and folds them there (the same
// bits as the fused pass, which runs otherwise).
int logprob_pass(const rz_bf16* H, const rz_bf16* W, const int32_t* tokens, int64_t T, int32_t d,
                 int32_t V, float* logprob, float* lse, float* lse_ws, uint8_t* ws, int* err,
                 cudaStream_t st, bool scratch) {
  if (T == 0) return RZ_OK;
  CUtensorMap tmH, tmW;
  if (!make_tmap_bf16(&tmH, H, d, T, uint64_t(d) * 2, kBK, a_box_rows(T))) return RZ_ERR_UNSUPPORTED;
  if (!make_tmap_bf16(&tmW, W, d, V, uint64_t(d) * 2, kBK, kBN)) return RZ_ERR_UNSUPPORTED;
  const FwdLayout L = fwd_layout(T, V);
  float2* part = reinterpret_cast<float2*>(ws + L.part);
  float* zg = reinterpret_cast<float*>(ws + L.zg);
  if (scratch && decode_mode(T, V)) {
    float* z = reinterpret_cast<float*>(ws + L.total);
    {
      ProfScope ps(RZ_PROF_LOGPROB_GEMM, 1, st);
      RZ_TRY(launch_decode_logits(tmH, tmW, T, d, V, z, err, st, a_box_rows(T)));
    }
    ProfScope ps(RZ_PROF_MERGE, 1, st);
    RZ_TRY(launch_decode_logprob(z, T, V, tokens, logprob, lse, lse_ws, err, st));
    return RZ_OK;
  }
  {
    ProfScope ps(RZ_PROF_LOGPROB_GEMM, static_cast<int>((T + kChunkRowsMax - 1) / kChunkRowsMax),
                 st);
    RZ_TRY(launch_lse_partial(tmH, tmW, T, d, V, tokens, part, zg, err, st, a_box_rows(T)));
  }
  ProfScope ps(RZ_PROF_MERGE, 1, st);
  RZ_TRY(launch_lse_merge(T, V, tokens, part, zg, logprob, lse, lse_ws, err, st));
  return RZ_OK;
}

// The learner step shared by the IS loss and, with sc set, the Score
// Centering loss (no weight, advantages centred, no log mu, no D3).
// Bn is the response count the loss averages over: B, or the whole batch's
// count when this call holds one shard of it (rz_loss_fwd_bwd_shard).
// ref_lse (nullable, [T]): a per-row reference for the kept terms (the
// rollout's log-sum-exp of the row); with it the backward pass takes the
// terms as they are (no dz pass).
int learner_step(bool sc, const rz_bf16* H, const rz_bf16* W, const int32_t* tokens,
                 const float* logmu, const float* ref_lse, const int64_t* cu_seqlens,
                 const float* adv,
                 const uint8_t* action_mask, int32_t B, int32_t Bn, int64_t T, int32_t d,
                 int32_t V,
                 float* loss_out, float* d3_out, float* logprob_out, rz_bf16* dH, float* dW,
                 void* ws, size_t ws_bytes, int32_t* err_flag, cudaStream_t st) {
  if (!sizes_ok(T, d, V) || B < 0 || (B == 0 && T > 0) || Bn < B) return RZ_ERR_INVALID_ARG;
  if (!W || !dW || !loss_out || !cu_seqlens) return RZ_ERR_INVALID_ARG;
  if (T > 0 && (!H || !tokens || !dH)) return RZ_ERR_INVALID_ARG;
  if (B > 0 && !adv) return RZ_ERR_INVALID_ARG;
  if (d % 8 != 0) return RZ_ERR_UNSUPPORTED;
  if (!a16(W) || !a16(dW) || (T > 0 && (!a16(H) || !a16(dH)))) return RZ_ERR_UNSUPPORTED;
  const bool ref = ref_lse != nullptr;
  const LearnLayout L = learn_layout(T, V, B, ref, d);
  if (!ws || ws_bytes < L.total || !a256(ws)) return RZ_ERR_WORKSPACE;
  if (!device_ok()) return RZ_ERR_UNSUPPORTED;
  uint8_t* w8 = static_cast<uint8_t*>(ws);
  float2* fac = reinterpret_cast<float2*>(w8 + L.fac);

  if (T == 0) {
    ProfScope ps(RZ_PROF_SMALL, sc ? 3 : 2, st);
    RZ_TRY(cudaMemsetAsync(dW, 0, size_t(V) * size_t(d) * sizeof(float), st));
    if (sc) {
      RZ_TRY(launch_resp_factors(cu_seqlens, adv, nullptr, B, Bn, 0, fac, st));
      RZ_TRY(launch_sc_loss(nullptr, cu_seqlens, nullptr, fac, B, 0, loss_out, w8 + L.resp,
                            err_flag, st));
    } else {
      RZ_TRY(launch_is_loss(nullptr, nullptr, cu_seqlens, adv, nullptr, B, Bn, 0, loss_out, d3_out,
                            nullptr, w8 + L.resp, err_flag, st));
    }
    return RZ_OK;
  }

  float* logpi = logprob_out ? logprob_out : reinterpret_cast<float*>(w8 + L.logpi);
  float* lse_c = reinterpret_cast<float*>(w8 + L.lse_ws);
  float* coef_c = reinterpret_cast<float*>(w8 + L.coef);
  float2* part = reinterpret_cast<float2*>(w8 + L.fwd.part);
  float* zg = reinterpret_cast<float*>(w8 + L.fwd.zg);
  float* emax = reinterpret_cast<float*>(w8 + L.emax);
  uint16_t* dz = reinterpret_cast<uint16_t*>(w8 + L.ez);  // kept terms, then dz in place
  uint16_t* hs = ref ? reinterpret_cast<uint16_t*>(w8 + L.hs) : nullptr;
  const int64_t ldz = dz_ld(V);
  const int64_t ldm = emax_ld(V);
  CUtensorMap tmH, tmW, tmWmn, tmHmn;
  if (!make_tmap_bf16(&tmH, H, d, T, uint64_t(d) * 2, kBK, a_box_rows(T))) return RZ_ERR_UNSUPPORTED;
  if (!make_tmap_bf16(&tmW, W, d, V, uint64_t(d) * 2, kBK, kBN)) return RZ_ERR_UNSUPPORTED;
  if (!make_tmap_bf16(&tmWmn, W, d, V, uint64_t(d) * 2, 64, 64)) return RZ_ERR_UNSUPPORTED;
  if (!make_tmap_bf16(&tmHmn, H, d, T, uint64_t(d) * 2, 64, 64)) return RZ_ERR_UNSUPPORTED;

  // (A_i, 1/(B T_i)) per response: all the coefficient needs besides w_t
  // (Score Centering: A_i - Abar).
  {
    ProfScope ps(RZ_PROF_SMALL, sc ? 2 : 1, st);
    RZ_TRY(launch_resp_factors(cu_seqlens, adv, action_mask, B, Bn, T, fac, st));
    if (sc) RZ_TRY(launch_sc_centre(fac, B, st));
  }

  // Chunk by chunk in row order: logits once, folded exactly as the rollout
  // folds them, keeping the fold's terms; merge + c_t; dz in place; dH, dW.
  // With a reference: the terms against it; merge + sigma_t and the sampled
  // column's term; H scaled by sigma; dH (scaled rows) and dW on the terms.
  for (int64_t r0 = 0; r0 < T; r0 += L.rows) {
    const int64_t rows = (T - r0) < L.rows ? (T - r0) : L.rows;
    CUtensorMap tmDz, tmDzMn, tmHsMn;
    if (ref && !make_tmap_bf16(&tmHsMn, hs, d, rows, uint64_t(d) * 2, 64, 64))
      return RZ_ERR_UNSUPPORTED;
    if (!make_tmap_bf16(&tmDz, dz, V, rows, uint64_t(ldz) * 2, kBK, kBM))
      return RZ_ERR_UNSUPPORTED;
    if (!make_tmap_bf16(&tmDzMn, dz, V, rows, uint64_t(ldz) * 2, 64, 64))
      return RZ_ERR_UNSUPPORTED;
    CUtensorMap tmE16;
    if (!make_tmap_bf16(&tmE16, dz, V, rows, uint64_t(ldz) * 2, 64, 32))
      return RZ_ERR_UNSUPPORTED;
    {
      ProfScope ps(RZ_PROF_KEEP_GEMM, 1, st);
      RZ_TRY(launch_lse_keep(tmH, tmW, r0, rows, d, V, tokens + r0, part, zg, tmE16, emax, ldm,
                             ref ? ref_lse + r0 : nullptr, err_flag, st, a_box_rows(T)));
    }
    {
      ProfScope ps(RZ_PROF_MERGE, 1, st);
      RZ_TRY(launch_lse_merge_coef(r0, rows, V, tokens + r0, part, zg, logpi + r0, lse_c,
                                   sc ? nullptr : logmu + r0, cu_seqlens, fac,
                                   action_mask ? action_mask + r0 : nullptr, B, coef_c,
                                   ref ? ref_lse + r0 : nullptr, dz, ldz, err_flag, st));
    }
    if (ref) {
      ProfScope ps(RZ_PROF_DZ, 1, st);
      RZ_TRY(launch_scale_rows(H, r0, rows, d, coef_c, hs, st));
    } else {
      ProfScope ps(RZ_PROF_DZ, 1, st);
      RZ_TRY(launch_dz_rows(dz, ldz, emax, ldm, rows, V, tokens + r0, lse_c, coef_c, logpi + r0,
                            st));
    }
    {
      ProfScope ps(RZ_PROF_DH_GEMM, 1, st);
      RZ_TRY(launch_dH(tmDz, tmWmn, r0, rows, d, V, dH, ref ? coef_c : nullptr, err_flag, st));
    }
    ProfScope ps(RZ_PROF_DW_GEMM, 1, st);
    if (ref) {
      RZ_TRY(launch_dW(tmDzMn, tmHsMn, 0, rows, d, V, dW, r0 > 0, err_flag, st));
    } else {
      RZ_TRY(launch_dW(tmDzMn, tmHmn, r0, rows, d, V, dW, r0 > 0, err_flag, st));
    }
  }

  // Loss (and D3) over all rows (fixed-order reductions).
  ProfScope ps(RZ_PROF_SMALL, 2, st);
  if (sc) {
    RZ_TRY(launch_sc_loss(logpi, cu_seqlens, action_mask, fac, B, T, loss_out, w8 + L.resp,
                          err_flag, st));
  } else {
    RZ_TRY(launch_is_loss(logpi, logmu, cu_seqlens, adv, action_mask, B, Bn, T, loss_out, d3_out,
                          nullptr, w8 + L.resp, err_flag, st));
  }
  return RZ_OK;
}

}  // namespace
}  // namespace rz

using namespace rz;

extern "C" {

const char* rz_status_string(int status) {
  switch (status) {
    case RZ_OK: return "ok";
    case RZ_ERR_INVALID_ARG: return "invalid argument";
    case RZ_ERR_UNSUPPORTED: return "unsupported (alignment, d % 8, or device is not sm_103)";
    case RZ_ERR_WORKSPACE: return "workspace missing or too small";
    case RZ_ERR_CUDA: return "CUDA error";
    case RZ_ERR_TOO_LARGE: return "problem exceeds the built-in scratch of the no-alloc entry point";
    default: return "unknown status";
  }
}

size_t rz_workspace_size(int op, int64_t T, int32_t d, int32_t V, int32_t B) {
  if (T < 0) T = 0;
  switch (op) {
    case RZ_OP_TOKEN_LOGPROB:
      return fwd_layout(T, V > 0 ? V : 1).total + decode_bytes(T, V > 0 ? V : 1);
    case RZ_OP_LOSS_FWD_BWD:
    case RZ_OP_SC_LOSS_FWD_BWD: return learn_layout(T, V > 0 ? V : 1, B).total;
    case RZ_OP_LOSS_FWD_BWD_REF: return learn_layout(T, V > 0 ? V : 1, B, true, d).total;
    case RZ_OP_LOGITS_LOSS: return is_loss_ws_bytes(B) + resp_factors_ws_bytes(B);
    case RZ_OP_IS_LOSS: return is_loss_ws_bytes(B);
    case RZ_OP_SAMPLE:
      return sample_layout(T, V > 0 ? V : 1).total + decode_bytes(T, V > 0 ? V : 1);
    default: return 0;
  }
}

int rz_token_logprob(const rz_bf16* H, const rz_bf16* W, const int32_t* tokens, int64_t T,
                     int32_t d, int32_t V, float* logprob_out, float* lse_out, void* ws,
                     size_t ws_bytes, int32_t* err_flag, rz_stream_t stream) {
  if (!sizes_ok(T, d, V)) return RZ_ERR_INVALID_ARG;
  if (T > 0 && (!H || !W || !tokens || !logprob_out)) return RZ_ERR_INVALID_ARG;
  if (d % 8 != 0) return RZ_ERR_UNSUPPORTED;
  if (T == 0) return RZ_OK;
  if (!a16(H) || !a16(W)) return RZ_ERR_UNSUPPORTED;
  const size_t need = fwd_layout(T, V).total;
  if (!ws || ws_bytes < need || !a256(ws)) return RZ_ERR_WORKSPACE;
  if (!device_ok()) return RZ_ERR_UNSUPPORTED;
  return logprob_pass(H, W, tokens, T, d, V, logprob_out, lse_out, nullptr,
                      static_cast<uint8_t*>(ws), err_flag, reinterpret_cast<cudaStream_t>(stream),
                      ws_bytes >= need + decode_bytes(T, V));
}

int rz_sample_logprob(const rz_bf16* H, const rz_bf16* W, const int64_t* row_ids, int64_t T,
                      int32_t d, int32_t V, uint64_t seed, int32_t* tokens_out,
                      float* logprob_out, float* lse_out, void* ws, size_t ws_bytes,
                      int32_t* err_flag, rz_stream_t stream) {
  if (!sizes_ok(T, d, V)) return RZ_ERR_INVALID_ARG;
  if (T > 0 && (!H || !W || !tokens_out || !logprob_out)) return RZ_ERR_INVALID_ARG;
  if (d % 8 != 0) return RZ_ERR_UNSUPPORTED;
  if (T == 0) return RZ_OK;
  if (!a16(H) || !a16(W)) return RZ_ERR_UNSUPPORTED;
  const SampleLayout L = sample_layout(T, V);
  if (!ws || ws_bytes < L.total || !a256(ws)) return RZ_ERR_WORKSPACE;
  if (!device_ok()) return RZ_ERR_UNSUPPORTED;
  CUtensorMap tmH, tmW;
  if (!make_tmap_bf16(&tmH, H, d, T, uint64_t(d) * 2, kBK, a_box_rows(T))) return RZ_ERR_UNSUPPORTED;
  if (!make_tmap_bf16(&tmW, W, d, V, uint64_t(d) * 2, kBK, kBN)) return RZ_ERR_UNSUPPORTED;
  uint8_t* w8 = static_cast<uint8_t*>(ws);
  if (decode_mode(T, V) && ws_bytes >= L.total + decode_bytes(T, V)) {
    // decode-sized batch: logits through the workspace, then the sampler's
    // fold and merge over them (the same bits)
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    float* z = reinterpret_cast<float*>(w8 + L.total);
    {
      ProfScope ps(RZ_PROF_LOGPROB_GEMM, 1, st);
      RZ_TRY(launch_decode_logits(tmH, tmW, T, d, V, z, err_flag, st, a_box_rows(T)));
    }
    ProfScope ps(RZ_PROF_MERGE, 1, st);
    return cuda_status(
        launch_decode_sample(z, T, V, row_ids, seed, tokens_out, logprob_out, lse_out, st));
  }
  ProfScope ps(RZ_PROF_LOGPROB_GEMM, static_cast<int>((T + kChunkRowsMax - 1) / kChunkRowsMax) + 1,
               reinterpret_cast<cudaStream_t>(stream));
  return cuda_status(launch_sample(tmH, tmW, T, d, V, row_ids, seed,
                                   reinterpret_cast<float4*>(w8 + L.part),
                                   reinterpret_cast<int*>(w8 + L.idx), tokens_out, logprob_out,
                                   lse_out, err_flag, reinterpret_cast<cudaStream_t>(stream),
                                   a_box_rows(T)));
}

int rz_group_advantage(const float* rewards, int32_t B, int32_t G, float* adv_out,
                       rz_stream_t stream) {
  if (B < 0 || G <= 0 || (B % G) != 0) return RZ_ERR_INVALID_ARG;
  if (B == 0) return RZ_OK;
  if (!rewards || !adv_out) return RZ_ERR_INVALID_ARG;
  if (!device_ok()) return RZ_ERR_UNSUPPORTED;
  ProfScope ps(RZ_PROF_SMALL, 1, reinterpret_cast<cudaStream_t>(stream));
  return cuda_status(
      launch_group_advantage(rewards, B, G, adv_out, reinterpret_cast<cudaStream_t>(stream)));
}

int rz_is_loss(const float* logpi, const float* logmu, const int64_t* cu_seqlens,
               const float* adv, const uint8_t* action_mask, int32_t B, int64_t T,
               float* loss_out, float* d3_out, float* coef_out, void* ws, size_t ws_bytes,
               int32_t* err_flag, rz_stream_t stream) {
  if (B < 0 || T < 0 || (B == 0 && T > 0)) return RZ_ERR_INVALID_ARG;
  if (!loss_out || !d3_out || !cu_seqlens) return RZ_ERR_INVALID_ARG;
  if (T > 0 && (!logpi || !logmu)) return RZ_ERR_INVALID_ARG;
  if (B > 0 && !adv) return RZ_ERR_INVALID_ARG;
  const size_t need = rz_workspace_size(RZ_OP_IS_LOSS, T, 0, 0, B);
  if (need > 0 && (!ws || ws_bytes < need || !a256(ws))) return RZ_ERR_WORKSPACE;
  if (!device_ok()) return RZ_ERR_UNSUPPORTED;
  ProfScope ps(RZ_PROF_SMALL, 2, reinterpret_cast<cudaStream_t>(stream));
  return cuda_status(launch_is_loss(logpi, logmu, cu_seqlens, adv, action_mask, B, B, T, loss_out,
                                    d3_out, coef_out, ws, err_flag,
                                    reinterpret_cast<cudaStream_t>(stream)));
}

int rz_d3(const float* logpi, const float* logmu, int64_t T, float* d3_out, rz_stream_t stream) {
  if (T < 0 || !d3_out) return RZ_ERR_INVALID_ARG;
  if (T > 0 && (!logpi || !logmu)) return RZ_ERR_INVALID_ARG;
  if (!device_ok()) return RZ_ERR_UNSUPPORTED;
  ProfScope ps(RZ_PROF_SMALL, 1, reinterpret_cast<cudaStream_t>(stream));
  return cuda_status(launch_d3(logpi, logmu, T, d3_out, reinterpret_cast<cudaStream_t>(stream)));
}

int rz_is_stats(const float* logpi, const float* logmu, int64_t T, float* stats_out,
                rz_stream_t stream) {
  if (T < 0 || !stats_out) return RZ_ERR_INVALID_ARG;
  if (T > 0 && (!logpi || !logmu)) return RZ_ERR_INVALID_ARG;
  if (!device_ok()) return RZ_ERR_UNSUPPORTED;
  ProfScope ps(RZ_PROF_SMALL, 1, reinterpret_cast<cudaStream_t>(stream));
  return cuda_status(
      launch_is_stats(logpi, logmu, T, stats_out, reinterpret_cast<cudaStream_t>(stream)));
}

int rz_peak_to_median(const float* series, int64_t n, double* ratio_out) {
  if (!series || !ratio_out || n <= 0) return RZ_ERR_INVALID_ARG;
  std::vector<double> v(series, series + n);
  std::sort(v.begin(), v.end());
  const double med = (n % 2) ? v[n / 2] : 0.5 * (v[n / 2 - 1] + v[n / 2]);
  *ratio_out = v.back() / med;
  return RZ_OK;
}

int rz_loss_fwd_bwd(const rz_bf16* H, const rz_bf16* W, const int32_t* tokens, const float* logmu,
                    const int64_t* cu_seqlens, const float* adv, const uint8_t* action_mask,
                    int32_t B, int64_t T, int32_t d, int32_t V, float* loss_out, float* d3_out,
                    float* logprob_out, rz_bf16* dH, float* dW, void* ws, size_t ws_bytes,
                    int32_t* err_flag, rz_stream_t stream) {
  if (!d3_out || (T > 0 && !logmu)) return RZ_ERR_INVALID_ARG;
  return learner_step(false, H, W, tokens, logmu, nullptr, cu_seqlens, adv, action_mask, B, B, T,
                      d, V, loss_out, d3_out, logprob_out, dH, dW, ws, ws_bytes, err_flag,
                      reinterpret_cast<cudaStream_t>(stream));
}

int rz_loss_fwd_bwd_ref(const rz_bf16* H, const rz_bf16* W, const int32_t* tokens,
                        const float* logmu, const float* ref_lse, const int64_t* cu_seqlens,
                        const float* adv, const uint8_t* action_mask, int32_t B, int64_t T,
                        int32_t d, int32_t V, float* loss_out, float* d3_out, float* logprob_out,
                        rz_bf16* dH, float* dW, void* ws, size_t ws_bytes, int32_t* err_flag,
                        rz_stream_t stream) {
  if (!d3_out || (T > 0 && (!logmu || !ref_lse))) return RZ_ERR_INVALID_ARG;
  return learner_step(false, H, W, tokens, logmu, T > 0 ? ref_lse : nullptr, cu_seqlens, adv,
                      action_mask, B, B, T, d, V, loss_out, d3_out, logprob_out, dH, dW, ws,
                      ws_bytes, err_flag, reinterpret_cast<cudaStream_t>(stream));
}

int rz_loss_fwd_bwd_shard(const rz_bf16* H, const rz_bf16* W, const int32_t* tokens,
                          const float* logmu, const float* ref_lse, const int64_t* cu_seqlens,
                          const float* adv,
                          const uint8_t* action_mask, int32_t B, int32_t B_total, int64_t T,
                          int32_t d, int32_t V, float* loss_out, float* d3_out,
                          float* logprob_out, rz_bf16* dH, float* dW, void* ws,
                          size_t ws_bytes, int32_t* err_flag, rz_stream_t stream) {
  if (!d3_out || (T > 0 && !logmu) || B_total < B || (B_total == 0 && B > 0))
    return RZ_ERR_INVALID_ARG;
  return learner_step(false, H, W, tokens, logmu, T > 0 ? ref_lse : nullptr, cu_seqlens, adv,
                      action_mask, B, B_total, T, d, V, loss_out, d3_out, logprob_out, dH, dW, ws,
                      ws_bytes, err_flag, reinterpret_cast<cudaStream_t>(stream));
}

int rz_sum_partials(const float* parts, int32_t n_parts, int64_t count, float* out,
                    rz_stream_t stream) {
  if (n_parts < 1 || count < 0) return RZ_ERR_INVALID_ARG;
  if (count == 0) return RZ_OK;
  if (!parts || !out) return RZ_ERR_INVALID_ARG;
  if (!device_ok()) return RZ_ERR_UNSUPPORTED;
  ProfScope ps(RZ_PROF_SMALL, 1, reinterpret_cast<cudaStream_t>(stream));
  return cuda_status(
      launch_sum_partials(parts, n_parts, count, out, reinterpret_cast<cudaStream_t>(stream)));
}

int rz_sc_loss_fwd_bwd(const rz_bf16* H, const rz_bf16* W, const int32_t* tokens,
                       const int64_t* cu_seqlens, const float* adv, const uint8_t* action_mask,
                       int32_t B, int64_t T, int32_t d, int32_t V, float* loss_out,
                       float* logprob_out, rz_bf16* dH, float* dW, void* ws, size_t ws_bytes,
                       int32_t* err_flag, rz_stream_t stream) {
  return learner_step(true, H, W, tokens, nullptr, nullptr, cu_seqlens, adv, action_mask, B, B, T,
                      d, V,
                      loss_out, nullptr, logprob_out, dH, dW, ws, ws_bytes, err_flag,
                      reinterpret_cast<cudaStream_t>(stream));
}

int rz_logits_loss_fwd_bwd(rz_bf16* logits_inout, const int32_t* tokens, const float* logmu,
                           const int64_t* cu_seqlens, const float* adv,
                           const uint8_t* action_mask, int32_t B, int64_t T, int32_t V,
                           float* loss_out, float* d3_out, float* logprob_out, void* ws,
                           size_t ws_bytes, int32_t* err_flag, rz_stream_t stream) {
  if (T < 0 || T >= (int64_t(1) << 31) || V < 1 || V > (1 << 24) || B < 0 || (B == 0 && T > 0))
    return RZ_ERR_INVALID_ARG;
  if (!loss_out || !d3_out || !cu_seqlens) return RZ_ERR_INVALID_ARG;
  if (T > 0 && (!logits_inout || !tokens || !logmu || !logprob_out)) return RZ_ERR_INVALID_ARG;
  if (B > 0 && !adv) return RZ_ERR_INVALID_ARG;
  if (V % 8 != 0 || (T > 0 && !a16(logits_inout))) return RZ_ERR_UNSUPPORTED;
  const size_t need = rz_workspace_size(RZ_OP_LOGITS_LOSS, T, 0, V, B);
  if (need > 0 && (!ws || ws_bytes < need || !a256(ws))) return RZ_ERR_WORKSPACE;
  if (!device_ok()) return RZ_ERR_UNSUPPORTED;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  uint8_t* w8 = static_cast<uint8_t*>(ws);
  float2* fac = reinterpret_cast<float2*>(w8 + is_loss_ws_bytes(B));
  {
    ProfScope ps(RZ_PROF_SMALL, 1, st);
    RZ_TRY(launch_resp_factors(cu_seqlens, adv, action_mask, B, B, T, fac, st));
  }
  {
    ProfScope ps(RZ_PROF_LOGITS_ROWS, 1, st);
    RZ_TRY(launch_logits_rows(logits_inout, T, V, tokens, logmu, cu_seqlens, fac, action_mask, B,
                              logprob_out, err_flag, st));
  }
  ProfScope ps(RZ_PROF_SMALL, 2, st);
  RZ_TRY(launch_is_loss(logprob_out, logmu, cu_seqlens, adv, action_mask, B, B, T, loss_out, d3_out,
                        nullptr, ws, err_flag, st));
  return RZ_OK;
}

int rz_debug_check_failures(uint32_t* count_out, int32_t* first_site_out) {
  if (!count_out || !first_site_out) return RZ_ERR_INVALID_ARG;
#ifndef RZ_CHECKS
  return RZ_ERR_UNSUPPORTED;
#else
  unsigned int c1 = 0, c2 = 0;
  int s1 = 0, s2 = 0;
  if (check_read_lmhead(&c1, &s1) != cudaSuccess || check_read_logits(&c2, &s2) != cudaSuccess)
    return RZ_ERR_CUDA;
  *count_out = c1 + c2;
  *first_site_out = c1 ? s1 : s2;
  return RZ_OK;
#endif
}

int rz_lmhead_logits(const rz_bf16* H, const rz_bf16* W, int64_t T, int32_t d, int32_t V,
                     float* logits_out, int32_t* err_flag, rz_stream_t stream) {
  if (!sizes_ok(T, d, V)) return RZ_ERR_INVALID_ARG;
  if (T > 0 && (!H || !W || !logits_out)) return RZ_ERR_INVALID_ARG;
  if (d % 8 != 0) return RZ_ERR_UNSUPPORTED;
  if (T == 0) return RZ_OK;
  if (!a16(H) || !a16(W)) return RZ_ERR_UNSUPPORTED;
  if (!device_ok()) return RZ_ERR_UNSUPPORTED;
  CUtensorMap tmH, tmW;
  if (!make_tmap_bf16(&tmH, H, d, T, uint64_t(d) * 2, kBK, a_box_rows(T))) return RZ_ERR_UNSUPPORTED;
  if (!make_tmap_bf16(&tmW, W, d, V, uint64_t(d) * 2, kBK, kBN)) return RZ_ERR_UNSUPPORTED;
  return cuda_status(launch_logits_f32(tmH, tmW, T, d, V, logits_out, err_flag,
                                       reinterpret_cast<cudaStream_t>(stream), a_box_rows(T)));
}

}  // extern "C"
