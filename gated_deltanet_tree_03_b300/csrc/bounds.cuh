// Address checks of the debug build. Compiled with -DGDN_DEBUG_BOUNDS (the library's build script
// makes that build on request, beside the release one), every global index the verify, commit
// and attention kernels compute is checked against the extent of its array before the access: an
// index outside the array ORs GDN_STATUS_OUT_OF_BOUNDS into the caller's status word and the
// access is skipped (a skipped load yields zero). Nothing traps. In the release build every check
// is the constant true and compiles away.
#pragma once

#include "common.cuh"

namespace gdn {

#ifdef GDN_DEBUG_BOUNDS
constexpr bool kDebugBounds = true;
#else
constexpr bool kDebugBounds = false;
#endif

// Element i of an array of n elements.
__device__ __forceinline__ bool in_bounds(long long i, long long n, int32_t *status) {
  if constexpr (!kDebugBounds) {
    return true;
  } else {
    if (i >= 0 && i < n) return true;
    report(status, GDN_STATUS_OUT_OF_BOUNDS);
    return false;
  }
}

// Elements [i, i + len) of an array of n elements.
__device__ __forceinline__ bool range_in_bounds(long long i, long long len, long long n, int32_t *status) {
  if constexpr (!kDebugBounds) {
    return true;
  } else {
    if (i >= 0 && len >= 0 && i + len <= n) return true;
    report(status, GDN_STATUS_OUT_OF_BOUNDS);
    return false;
  }
}

// States in ST: the pool's slots under a serving layout, else one per request.
template <bool SV>
__device__ __forceinline__ long long state_count(const Serving &L, int B) {
  if constexpr (SV) return L.slot ? L.n_slots : B;
  else return B;
}

}  // namespace gdn
