// rz_check.cuh -- device-side bounds checks of the debug build (-DRZ_CHECKS).
//
// RZ_DCHECK(cond, site) guards one computed index: in the debug build a
// false condition counts a failure, records the site of the first one, and
// evaluates to false so the caller skips the access (no trap, no assert: a
// wrong index never reaches memory).  In the normal build it is the
// constant true and compiles away.  The counters are per translation unit
// (no relocatable device code); each unit that uses checks reports its own
// through rz_check_read_<unit>() and rz_debug_check_failures() adds them up.
#pragma once

#include <cstdint>

#ifdef RZ_CHECKS

namespace rz {
static __device__ unsigned int g_check_fail;
static __device__ int g_check_site;

__device__ __forceinline__ bool dcheck(bool ok, int site) {
  if (!ok) {
    if (atomicAdd(&g_check_fail, 1u) == 0u) atomicExch(&g_check_site, site);
  }
  return ok;
}

// Host side: this unit's count and first site, then clear them.
inline cudaError_t check_read_and_clear(unsigned int* count, int* site) {
  cudaError_t e = cudaMemcpyFromSymbol(count, g_check_fail, sizeof(unsigned int));
  if (e == cudaSuccess) e = cudaMemcpyFromSymbol(site, g_check_site, sizeof(int));
  const unsigned int zero = 0;
  const int none = 0;
  if (e == cudaSuccess) e = cudaMemcpyToSymbol(g_check_fail, &zero, sizeof(zero));
  if (e == cudaSuccess) e = cudaMemcpyToSymbol(g_check_site, &none, sizeof(none));
  return e;
}
}  // namespace rz

#define RZ_DCHECK(cond, site) (::rz::dcheck(static_cast<bool>(cond), (site)))

#else

#define RZ_DCHECK(cond, site) (true)

#endif
