// Device-side status flags. Kernels receive a pointer to one 32-bit word (a
// static __device__ variable owned by the library) and OR bits into it; the
// host reads and clears it in mcs_check_status().
#pragma once
#include <cstdint>

namespace mcs {

constexpr uint32_t kStatusBounds = 1u;   // an index outside [0, N) was met and skipped
constexpr uint32_t kStatusTimeout = 2u;  // a bounded wait ran out; the kernel stopped early

__device__ __forceinline__ void raise_status(uint32_t* st, uint32_t bits) { atomicOr(st, bits); }
__device__ __forceinline__ uint32_t peek_status(const uint32_t* st) {
  return *reinterpret_cast<const volatile uint32_t*>(st);
}

}  // namespace mcs
