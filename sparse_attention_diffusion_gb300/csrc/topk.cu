// Exact per-group top-K over the pass-2 score rows [MC-Sparse summary: anchor
// two-pass paragraph: keep the K keys with the largest summed attention weight].
// One CTA per row: an 8-bit-digit radix select finds the K-th largest score
// (scores are non-negative fp32, so their bit patterns order like the values),
// then an ordered compaction (contiguous slice per warp, one scan over the
// warps) writes every key above it plus the lowest-index keys equal to it,
// which gives ascending indices and the ties-to-lower-index rule at once. The
// captured mass is summed in a fixed order.
#include "block_scan.cuh"
#include "common.cuh"
#include "kernels.h"
#include "status.cuh"

namespace mcs {
namespace {

constexpr int kTopkThreads = 1024;
constexpr int kTopkWarps = kTopkThreads / 32;
constexpr int kLoads = 8;  // independent row loads in flight per thread

__global__ void __launch_bounds__(kTopkThreads) topk_kernel(const TopkParams p) {
  __shared__ uint32_t hist[256];
  __shared__ uint32_t sh_prefix, sh_remaining;
  __shared__ int wgt[kTopkWarps], weq[kTopkWarps];
  __shared__ float warp_sum[kTopkWarps];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int row = blockIdx.x;
  const int grow = p.row0 + row;
  const float* S = p.scores + size_t(row) * p.N;
  const uint32_t* U = reinterpret_cast<const uint32_t*>(S);
  const uint32_t lanes_below = (1u << lane) - 1u;

  // Radix select, four 8-bit digits from the top. The block walks the row in
  // chunks of 1024 so every warp stays converged; lanes of a warp that hit the
  // same bin add their count with one shared-memory atomic (score exponents
  // cluster, so a per-element atomic would serialise on a few bins).
  uint32_t prefix = 0, mask = 0, remaining = uint32_t(p.K);
  for (int pass = 0; pass < 4; ++pass) {
    const int shift = 24 - 8 * pass;
    for (int i = tid; i < 256; i += kTopkThreads) hist[i] = 0;
    __syncthreads();
    // kLoads chunks per step: their loads are issued together (the row does not
    // fit in L1, so each is an L2 round trip)
    for (int c0 = 0; c0 < p.N; c0 += kLoads * kTopkThreads) {
      uint32_t u4[kLoads];
#pragma unroll
      for (int k = 0; k < kLoads; ++k) {
        const int j = c0 + k * kTopkThreads + tid;
        u4[k] = j < p.N ? __ldg(U + j) : 0u;
      }
#pragma unroll
      for (int k = 0; k < kLoads; ++k) {
        const int j = c0 + k * kTopkThreads + tid;
        const bool cand = j < p.N && (u4[k] & mask) == prefix;
        const unsigned act = __ballot_sync(0xffffffffu, cand);
        if (cand) {
          const uint32_t bin = (u4[k] >> shift) & 255u;
          const unsigned peers = __match_any_sync(act, bin);
          if (lane == __ffs(peers) - 1) atomicAdd(&hist[bin], uint32_t(__popc(peers)));
        }
      }
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
  const uint32_t thr = prefix;                 // bit pattern of the K-th largest score
  const int need_eq = int(remaining);          // how many scores equal to it are kept (lowest indices)

  // Ordered compaction: warp w owns the contiguous slice [lo, hi) of the row.
  // Counting pass, one exclusive scan over the warps' counts, then each warp
  // writes its selected ids in index order with ballots (ties to the lower
  // index: a warp keeps the first equal scores that the warps before it left).
  const int span = ((p.N + kTopkWarps - 1) / kTopkWarps + 31) & ~31;
  const int lo = min(p.N, warp * span), hi = min(p.N, lo + span);
  int cgt = 0, ceq = 0;
  for (int c = lo; c < hi; c += kLoads * 32) {
    uint32_t u4[kLoads];
#pragma unroll
    for (int k = 0; k < kLoads; ++k) {
      const int j = c + k * 32 + lane;
      u4[k] = j < hi ? __ldg(U + j) : 0u;
    }
#pragma unroll
    for (int k = 0; k < kLoads; ++k) {
      const bool v = c + k * 32 + lane < hi;
      cgt += (v && u4[k] > thr) ? 1 : 0;
      ceq += (v && u4[k] == thr) ? 1 : 0;
    }
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    cgt += __shfl_xor_sync(0xffffffffu, cgt, off);
    ceq += __shfl_xor_sync(0xffffffffu, ceq, off);
  }
  if (lane == 0) {
    wgt[warp] = cgt;
    weq[warp] = ceq;
  }
  __syncthreads();
  int gt_before = 0, eq_before = 0, gt_all = 0, eq_all = 0;
  for (int w = 0; w < kTopkWarps; ++w) {
    const int a = wgt[w], b = weq[w];
    gt_before += w < warp ? a : 0;
    eq_before += w < warp ? b : 0;
    gt_all += a;
    eq_all += b;
  }
  const int take_eq = max(0, min(ceq, need_eq - eq_before));
  int out_pos = gt_before + min(eq_before, need_eq);
  int eq_seen = 0;
  float msum = 0.f;
  int32_t* out = p.idx + size_t(grow) * p.K;
  for (int c = lo; c < hi; c += kLoads * 32) {
    uint32_t u4[kLoads];
#pragma unroll
    for (int k = 0; k < kLoads; ++k) {
      const int j = c + k * 32 + lane;
      u4[k] = j < hi ? __ldg(U + j) : 0u;
    }
#pragma unroll
    for (int k = 0; k < kLoads; ++k) {  // chunks in index order
      const int j = c + k * 32 + lane;
      const bool v = j < hi;
      const bool gt = v && u4[k] > thr, eq = v && u4[k] == thr;
      const unsigned beq = __ballot_sync(0xffffffffu, eq);
      const bool sel = gt || (eq && eq_seen + __popc(beq & lanes_below) < take_eq);
      const unsigned bsel = __ballot_sync(0xffffffffu, sel);
      const int pos = out_pos + __popc(bsel & lanes_below);
      if (sel && pos < p.K) {
        out[pos] = j;
        msum += __uint_as_float(u4[k]);
      }
      out_pos += __popc(bsel);
      eq_seen += __popc(beq);
    }
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
      for (int w = 0; w < kTopkWarps; ++w) tsum += warp_sum[w];
      p.mass[grow] = nreal > 0 ? tsum / float(nreal) : 0.f;
    }
  }
  if (tid == 0 && gt_all + min(eq_all, need_eq) != p.K) raise_status(p.status, kStatusBounds);
}

}  // namespace

cudaError_t topk_rows(const TopkParams& p, int nrows, cudaStream_t stream) {
  if (nrows <= 0) return cudaSuccess;
  topk_kernel<<<nrows, kTopkThreads, 0, stream>>>(p);
  note_launches(1);
  return cudaGetLastError();
}

}  // namespace mcs
