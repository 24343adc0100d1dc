// rz_profile.cu -- launch-class timing: while enabled, each entry point
// brackets every class of launch with a pair of CUDA events recorded on the
// stream it launches on, so a caller can split one call's device time by
// kernel without a profiler.  Off by default; nothing is recorded then.
#include <cuda_runtime.h>

#include <atomic>
#include <mutex>
#include <vector>

#include "rz.h"
#include "rz_internal.h"

namespace rz {
namespace {

struct Rec {
  int cls;
  int launches;
  cudaEvent_t e0, e1;
};

std::atomic<bool> g_on{false};
std::mutex g_mu;
std::vector<Rec> g_recs;

bool capturing(cudaStream_t st) {
  cudaStreamCaptureStatus s = cudaStreamCaptureStatusNone;
  if (cudaStreamIsCapturing(st, &s) != cudaSuccess) return true;  // do not touch the stream
  return s != cudaStreamCaptureStatusNone;
}

}  // namespace

ProfScope::ProfScope(int cls, int launches, cudaStream_t st)
    : cls_(cls), launches_(launches), st_(st), e0_(nullptr) {
  if (!g_on.load(std::memory_order_relaxed) || launches <= 0 || capturing(st)) return;
  cudaEvent_t e = nullptr;
  if (cudaEventCreate(&e) != cudaSuccess) return;
  if (cudaEventRecord(e, st) != cudaSuccess) {
    cudaEventDestroy(e);
    return;
  }
  e0_ = e;
}

ProfScope::~ProfScope() {
  if (!e0_) return;
  cudaEvent_t e0 = static_cast<cudaEvent_t>(e0_);
  cudaEvent_t e1 = nullptr;
  if (cudaEventCreate(&e1) != cudaSuccess || cudaEventRecord(e1, st_) != cudaSuccess) {
    if (e1) cudaEventDestroy(e1);
    cudaEventDestroy(e0);
    return;
  }
  std::lock_guard<std::mutex> lk(g_mu);
  g_recs.push_back({cls_, launches_, e0, e1});
}

}  // namespace rz

using namespace rz;

extern "C" {

int rz_profile_begin(void) {
  std::lock_guard<std::mutex> lk(g_mu);
  for (Rec& r : g_recs) {
    cudaEventDestroy(r.e0);
    cudaEventDestroy(r.e1);
  }
  g_recs.clear();
  g_on.store(true);
  return RZ_OK;
}

int rz_profile_end(float* ms_out, int32_t* launches_out, int32_t n_classes) {
  if (!ms_out || n_classes < RZ_PROF_CLASSES) return RZ_ERR_INVALID_ARG;
  g_on.store(false);
  std::vector<Rec> recs;
  {
    std::lock_guard<std::mutex> lk(g_mu);
    recs.swap(g_recs);
  }
  for (int c = 0; c < n_classes; ++c) {
    ms_out[c] = 0.f;
    if (launches_out) launches_out[c] = 0;
  }
  int status = RZ_OK;
  for (Rec& r : recs) {
    float ms = 0.f;
    if (cudaEventSynchronize(r.e1) != cudaSuccess ||
        cudaEventElapsedTime(&ms, r.e0, r.e1) != cudaSuccess) {
      status = RZ_ERR_CUDA;
    } else if (r.cls >= 0 && r.cls < n_classes) {
      ms_out[r.cls] += ms;
      if (launches_out) launches_out[r.cls] += r.launches;
    }
    cudaEventDestroy(r.e0);
    cudaEventDestroy(r.e1);
  }
  return status;
}

}  // extern "C"
