// Range checks of data-dependent indices, compiled in by -DMOE_BOUNDS_CHECK.
//
// That debug build stands in for a device memory checker: every index that a
// kernel derives from device data (expert ids, offsets, slot rows, row
// tokens, staged pair numbers) is checked against the size of the buffer it
// addresses before the access.  A failed check records kStatusBounds in the
// status word (when the kernel has one; moe_check_status reports it as
// MOE_ERR_BOUNDS) and the access is skipped; nothing traps.  In normal builds
// every check is the constant `true` and compiles away.
#pragma once
#include <cstdint>

namespace moe {

constexpr int kStatusBounds = -6;  // mirrors MOE_ERR_BOUNDS

#ifdef MOE_BOUNDS_CHECK
constexpr bool kBoundsChecked = true;
__device__ __forceinline__ bool idx_ok(int64_t i, int64_t n, int* status) {
  if (i >= 0 && i < n) return true;
  if (status != nullptr) atomicExch(status, kStatusBounds);
  return false;
}
#else
constexpr bool kBoundsChecked = false;
__device__ __forceinline__ bool idx_ok(int64_t, int64_t, int*) { return true; }
#endif

}  // namespace moe
