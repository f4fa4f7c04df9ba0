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

// Descriptor words for MMA issue loops. A step along K (K-major operand) or
// along rows (MN-major operand) only moves the start address, which sits in the
// low word and cannot carry out of its 14-bit field for shared-memory addresses,
// so a loop keeps one base low word per operand and adds compile-time step
// offsets; the high word (stride byte offset 1024, version, 128-byte swizzle) is
// the same constant for every operand here. desc_kmajor(b, s) has the words
// {desc_lo_kmajor(b) + kstep_kmajor(s), kDescHi}; desc_mnmajor likewise.
constexpr uint32_t kDescHi = (1024u >> 4) | (1u << 14) | (2u << 29);
__device__ __forceinline__ uint32_t desc_lo_kmajor(uint32_t base) { return ((base >> 4) & 0x3FFFu) | (1u << 16); }
__device__ __forceinline__ uint32_t desc_lo_mnmajor(uint32_t base) {
  return ((base >> 4) & 0x3FFFu) | (uint32_t(kRegion >> 4) << 16);
}
__host__ __device__ constexpr uint32_t kstep_kmajor(int s) { return uint32_t((s >> 2) * (kRegion >> 4) + (s & 3) * 2); }
__host__ __device__ constexpr uint32_t kstep_mnmajor(int s) { return uint32_t(s * 16 * 128 / 16); }

// D[tmem] (+)= A[smem] * B[smem]^T from descriptor low words (high word kDescHi).
__device__ __forceinline__ void tc_mma_ss_lo(uint32_t d_tmem, uint32_t a_lo, uint32_t b_lo, uint32_t idesc,
                                             uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n .reg .b64 da, db;\n setp.ne.b32 p, %4, 0;\n"
      " mov.b64 da, {%1, %5};\n mov.b64 db, {%2, %5};\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], da, db, %3, p;\n}\n" ::"r"(d_tmem),
      "r"(a_lo), "r"(b_lo), "r"(idesc), "r"(accumulate), "r"(kDescHi)
      : "memory");
}
// D[tmem] (+)= A[tmem] * B[smem] from the B descriptor's low word.
__device__ __forceinline__ void tc_mma_ts_lo(uint32_t d_tmem, uint32_t a_tmem, uint32_t b_lo, uint32_t idesc,
                                             uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n .reg .b64 db;\n setp.ne.b32 p, %4, 0;\n"
      " mov.b64 db, {%2, %5};\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], db, %3, p;\n}\n" ::"r"(d_tmem),
      "r"(a_tmem), "r"(b_lo), "r"(idesc), "r"(accumulate), "r"(kDescHi)
      : "memory");
}

// Warp-wide forms: every lane of the issuing warp executes the statement with
// the same (warp-uniform) operands and only the lane with `issue` set issues the
// MMA or the commit, so the operands can live in uniform registers.
__device__ __forceinline__ void tc_mma_ss_lo_if(bool issue, uint32_t d_tmem, uint32_t a_lo, uint32_t b_lo,
                                                uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p, q;\n .reg .b64 da, db;\n setp.ne.b32 p, %4, 0;\n setp.ne.b32 q, %6, 0;\n"
      " mov.b64 da, {%1, %5};\n mov.b64 db, {%2, %5};\n"
      " @q tcgen05.mma.cta_group::1.kind::f16 [%0], da, db, %3, p;\n}\n" ::"r"(d_tmem),
      "r"(a_lo), "r"(b_lo), "r"(idesc), "r"(accumulate), "r"(kDescHi), "r"(uint32_t(issue))
      : "memory");
}
__device__ __forceinline__ void tc_mma_ts_lo_if(bool issue, uint32_t d_tmem, uint32_t a_tmem, uint32_t b_lo,
                                                uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p, q;\n .reg .b64 db;\n setp.ne.b32 p, %4, 0;\n setp.ne.b32 q, %6, 0;\n"
      " mov.b64 db, {%2, %5};\n"
      " @q tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], db, %3, p;\n}\n" ::"r"(d_tmem),
      "r"(a_tmem), "r"(b_lo), "r"(idesc), "r"(accumulate), "r"(kDescHi), "r"(uint32_t(issue))
      : "memory");
}
__device__ __forceinline__ void tc_commit_if(bool issue, uint64_t* bar) {
  asm volatile(
      "{\n .reg .pred q;\n setp.ne.b32 q, %1, 0;\n"
      " @q tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n}\n" ::"r"(smem_u32(bar)),
      "r"(uint32_t(issue))
      : "memory");
}

__device__ __forceinline__ bool warp_all(bool v) { return __all_sync(0xffffffffu, v); }

}  // namespace mcs
