// Block-wide helpers for 1024-thread CTAs: exclusive scan of a predicate and
// radix-select digit search. Deterministic (no floating-point atomics).
#pragma once
#include <cstdint>

namespace mcs {

// Exclusive prefix count of `flag` over the block in thread order; *total gets
// the block-wide count. `warp_tot` is shared scratch of (blockDim.x/32) ints.
// Contains two __syncthreads(): every thread of the block must call it.
__device__ __forceinline__ int block_excl_count(bool flag, int* warp_tot, int* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
  const unsigned b = __ballot_sync(0xffffffffu, flag);
  const int lane_pre = __popc(b & ((1u << lane) - 1u));
  if (lane == 0) warp_tot[warp] = __popc(b);
  __syncthreads();
  int pre = 0, tot = 0;
  for (int w = 0; w < nw; ++w) {
    const int c = warp_tot[w];
    pre += (w < warp) ? c : 0;
    tot += c;
  }
  __syncthreads();
  *total = tot;
  return pre + lane_pre;
}

// Radix-select digit search over a 256-bin histogram, run by one full warp.
// Finds the bin b such that the number of elements in bins ordered before b is
// < remaining <= that number + hist[b]. `descending` orders bins from 255 down.
// Returns b and writes the count before b to *before.
__device__ __forceinline__ int warp_find_digit(const uint32_t* hist, uint32_t remaining, bool descending,
                                               uint32_t* before) {
  const int lane = threadIdx.x & 31;
  uint32_t c[8];
  uint32_t tot = 0;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int bin = descending ? 255 - (lane * 8 + i) : lane * 8 + i;
    c[i] = hist[bin];
    tot += c[i];
  }
  uint32_t incl = tot;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const uint32_t y = __shfl_up_sync(0xffffffffu, incl, off);
    if (lane >= off) incl += y;
  }
  uint32_t run = incl - tot;  // elements in bins ordered before this lane's bins
  int found = -1;
  uint32_t found_before = 0;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    if (found < 0 && run < remaining && remaining <= run + c[i]) {
      found = descending ? 255 - (lane * 8 + i) : lane * 8 + i;
      found_before = run;
    }
    run += c[i];
  }
  const unsigned who = __ballot_sync(0xffffffffu, found >= 0);
  const int src = who ? (__ffs(who) - 1) : 0;
  *before = __shfl_sync(0xffffffffu, found_before, src);
  return __shfl_sync(0xffffffffu, found, src);
}

}  // namespace mcs
