// Shared-memory operand layout shared by the tcgen05 kernels.
//
// A [rows x 64k] bf16 operand tile is stored as k regions of 128 rows x 128 B
// (64 elements along the contiguous dimension per region), each row's eight
// 16-byte chunks permuted by the 128-byte swizzle (chunk c of row r sits at
// chunk c ^ (r % 8)). This is the layout TMA writes with 128-byte swizzling and
// the layout the tensor core reads through a SWIZZLE_128B matrix descriptor
// with 1024-byte stride between 8-row groups.
#pragma once
#include <cstdint>

#include "ptx.cuh"

namespace mcs {

constexpr int kRegion = 128 * 128;  // bytes of one 128-row x 128-byte region

// Byte offset of 16-byte chunk `ch` (8 bf16 along the contiguous dim) of `row`.
__device__ __forceinline__ uint32_t sw128_off(int row, int ch) {
  return uint32_t((ch >> 3) * kRegion + row * 128 + (((ch & 7) ^ (row & 7)) << 4));
}

// K-major operand (rows = M or N, contiguous dim = K): k-step s covers K elements
// [16s, 16s+16): region s/4, +32 B per step inside the 128-byte swizzle atom.
__device__ __forceinline__ uint64_t desc_kmajor(uint32_t base, int s) {
  return smem_desc_sw128(base + uint32_t((s >> 2) * kRegion + (s & 3) * 32), 16, 1024);
}

// MN-major operand (contiguous dim = N, rows = K): k-step s covers rows
// [16s, 16s+16). Leading byte offset = stride between 64-element N chunks (one
// region); stride byte offset = stride between groups of 8 rows.
__device__ __forceinline__ uint64_t desc_mnmajor(uint32_t base, int s) {
  return smem_desc_sw128(base + uint32_t(s * 16 * 128), kRegion, 1024);
}

__device__ __forceinline__ bool warp_all(bool v) { return __all_sync(0xffffffffu, v); }

}  // namespace mcs
