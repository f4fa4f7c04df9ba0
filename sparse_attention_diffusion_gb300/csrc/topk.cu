// Exact per-group top-K over the pass-2 score rows [MC-Sparse summary: anchor
// two-pass paragraph: keep the K keys with the largest summed attention weight].
// One CTA per row: an 8-bit-digit radix select finds the K-th largest score
// (scores are non-negative fp32, so their bit patterns order like the values),
// then an ordered block-scan compaction writes every key above it plus the
// lowest-index keys equal to it, which gives ascending indices and the
// ties-to-lower-index rule at once. The captured mass is summed in a fixed order.
#include "block_scan.cuh"
#include "common.cuh"
#include "kernels.h"
#include "status.cuh"

namespace mcs {
namespace {

constexpr int kTopkThreads = 1024;

__global__ void __launch_bounds__(kTopkThreads) topk_kernel(const TopkParams p) {
  __shared__ uint32_t hist[256];
  __shared__ int warp_tot[32];
  __shared__ uint32_t sh_prefix, sh_remaining;
  __shared__ float warp_sum[32];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int row = blockIdx.x;
  const int grow = p.row0 + row;
  const float* S = p.scores + size_t(row) * p.N;
  const uint32_t* U = reinterpret_cast<const uint32_t*>(S);

  uint32_t prefix = 0, mask = 0, remaining = uint32_t(p.K);
  for (int pass = 0; pass < 4; ++pass) {
    const int shift = 24 - 8 * pass;
    for (int i = tid; i < 256; i += kTopkThreads) hist[i] = 0;
    __syncthreads();
    for (int j = tid; j < p.N; j += kTopkThreads) {
      const uint32_t u = U[j];
      if ((u & mask) == prefix) atomicAdd(&hist[(u >> shift) & 255u], 1u);
    }
    __syncthreads();
    if (warp == 0) {
      uint32_t before;
      const int b = warp_find_digit(hist, remaining, /*descending=*/true, &before);
      if (lane == 0) {
        sh_prefix = prefix | (uint32_t(b < 0 ? 0 : b) << shift);
        sh_remaining = remaining - before;
      }
    }
    __syncthreads();
    prefix = sh_prefix;
    remaining = sh_remaining;
    mask |= 0xFFu << shift;
  }
  const uint32_t thr = prefix;       // bit pattern of the K-th largest score
  const uint32_t need_eq = remaining; // how many scores equal to it are kept (lowest indices)

  int32_t* out = p.idx + size_t(grow) * p.K;
  int base_out = 0, base_eq = 0;
  float msum = 0.f;
  for (int c0 = 0; c0 < p.N; c0 += kTopkThreads) {
    const int j = c0 + tid;
    const bool valid = j < p.N;
    const uint32_t u = valid ? U[j] : 0u;
    const bool gt = valid && u > thr, eq = valid && u == thr;
    int eq_tot, sel_tot;
    const int eq_pre = block_excl_count(eq, warp_tot, &eq_tot);
    const bool sel = gt || (eq && uint32_t(base_eq + eq_pre) < need_eq);
    const int sel_pre = block_excl_count(sel, warp_tot, &sel_tot);
    if (sel && base_out + sel_pre < p.K) {
      out[base_out + sel_pre] = j;
      msum += __uint_as_float(u);
    }
    base_eq += eq_tot;
    base_out += sel_tot;
  }
  if (p.mass != nullptr) {
    const int bh = grow / p.G, g = grow % p.G;
    int real = 0;
    if (tid < p.C) {
      const int t = p.perm[size_t(bh) * p.N_pad + size_t(g) * p.C + tid];
      real = (t >= 0 && t < p.N) ? 1 : 0;
    }
    const int nreal = __syncthreads_count(real);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) msum += __shfl_xor_sync(0xffffffffu, msum, off);
    if (lane == 0) warp_sum[warp] = msum;
    __syncthreads();
    if (tid == 0) {
      float tsum = 0.f;
      for (int w = 0; w < kTopkThreads / 32; ++w) tsum += warp_sum[w];
      p.mass[grow] = nreal > 0 ? tsum / float(nreal) : 0.f;
    }
  }
  if (tid == 0 && base_out != p.K) raise_status(p.status, kStatusBounds);
}

}  // namespace

cudaError_t topk_rows(const TopkParams& p, int nrows, cudaStream_t stream) {
  if (nrows <= 0) return cudaSuccess;
  topk_kernel<<<nrows, kTopkThreads, 0, stream>>>(p);
  note_launches(1);
  return cudaGetLastError();
}

}  // namespace mcs
