// rz_noalloc.cu -- rz_token_logprob_noalloc: the rollout logprob path for
// callers that cannot allocate device memory.
//
// Some callers hold only a stream and the tensors they were handed: a
// sampler hook running inside an inference engine whose memory pool was
// reserved up front (a fresh cudaMalloc there can fail or fragment the pool,
// and it synchronises the device), a plug-in invoked by a host that owns all
// allocation, or code that runs between captured graph segments where an
// allocation would break the capture.  For them this entry point uses a
// fixed scratch array compiled into the library instead of a caller
// workspace.  It launches the same two kernels with the same launch shape
// as rz_token_logprob, so its results are bitwise the same.
//
// The scratch is a file-scope __device__ array: every GPU that loads the
// library holds kNoAllocScratchBytes of it until the process exits.  Host
// code cannot use the array's name as a device address (on the host it is
// only a stand-in symbol), so the device address is looked up once per
// device with cudaGetSymbolAddress on the first call made with that device
// current.  Make that first call before any stream capture starts.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>

#include "rz.h"
#include "rz_internal.h"

namespace rz {
namespace {

constexpr size_t kNoAllocScratchBytes = size_t(32) << 20;  // 32 MiB per device
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

std::mutex g_mu;
void* g_scratch_ptr[kMaxDevices] = {};

// Device address of the scratch array on the current device (looked up once
// per device).  Returns nullptr if the lookup fails.
void* scratch_on_current_device() {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_scratch_ptr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess) return nullptr;
    g_scratch_ptr[dev] = p;
  }
  return g_scratch_ptr[dev];
}

}  // namespace
}  // namespace rz

using namespace rz;

extern "C" {

size_t rz_noalloc_scratch_bytes(void) { return kNoAllocScratchBytes; }

int rz_token_logprob_noalloc(const rz_bf16* H, const rz_bf16* W, const int32_t* tokens, int64_t T,
                             int32_t d, int32_t V, float* logprob_out, float* lse_out,
                             int32_t* err_flag, rz_stream_t stream) {
  if (!sizes_ok(T, d, V)) return RZ_ERR_INVALID_ARG;
  if (T > 0 && (!H || !W || !tokens || !logprob_out)) return RZ_ERR_INVALID_ARG;
  if (d % 8 != 0) return RZ_ERR_UNSUPPORTED;
  if (T == 0) return RZ_OK;
  if (!a16(H) || !a16(W)) return RZ_ERR_UNSUPPORTED;
  // The workspace layout of rz_token_logprob: per-row split states, then the
  // gathered logit of each row.  Nothing in it needs zeroing: every entry
  // the merge reads is written by the GEMM earlier in the same call.
  const FwdLayout L = fwd_layout(T, V);
  if (L.total > kNoAllocScratchBytes) return RZ_ERR_TOO_LARGE;
  if (!device_ok()) return RZ_ERR_UNSUPPORTED;
  uint8_t* scratch = static_cast<uint8_t*>(scratch_on_current_device());
  if (!scratch) return RZ_ERR_CUDA;

  CUtensorMap tmH, tmW;
  if (!make_tmap_bf16(&tmH, H, d, T, uint64_t(d) * 2, kBK, a_box_rows(T))) return RZ_ERR_UNSUPPORTED;
  if (!make_tmap_bf16(&tmW, W, d, V, uint64_t(d) * 2, kBK, kBN)) return RZ_ERR_UNSUPPORTED;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  if (decode_mode(T, V) && L.total + decode_bytes(T, V) <= kNoAllocScratchBytes) {
    // a decode-sized batch whose logits fit the scratch (up to 55 rows at
    // V = 151936): as rz_token_logprob does, the same bits
    float* z = reinterpret_cast<float*>(scratch + L.total);
    if (launch_decode_logits(tmH, tmW, T, d, V, z, err_flag, st, a_box_rows(T)) != cudaSuccess ||
        launch_decode_logprob(z, T, V, tokens, logprob_out, lse_out, nullptr, err_flag, st) !=
            cudaSuccess)
      return RZ_ERR_CUDA;
    return RZ_OK;
  }
  float2* part = reinterpret_cast<float2*>(scratch + L.part);
  float* zg = reinterpret_cast<float*>(scratch + L.zg);
  if (launch_lse_partial(tmH, tmW, T, d, V, tokens, part, zg, err_flag, st, a_box_rows(T)) !=
          cudaSuccess ||
      launch_lse_merge(T, V, tokens, part, zg, logprob_out, lse_out, nullptr, err_flag, st) !=
          cudaSuccess)
    return RZ_ERR_CUDA;
  return RZ_OK;
}

}  // extern "C"
