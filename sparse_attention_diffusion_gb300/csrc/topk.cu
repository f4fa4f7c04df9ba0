// Exact per-group top-K over the pass-2 score rows [MC-Sparse summary: anchor
// two-pass paragraph: keep the K keys with the largest summed attention weight].
// One CTA per row. The K-th largest score is found by a radix
// select on the scores' bit patterns (scores are non-negative fp32, so their
// bit patterns order like the values), then an ordered compaction (contiguous
// slice per warp, one scan over the warps) writes every key above it plus the
// lowest-index keys equal to it, which gives ascending indices and the
// ties-to-lower-index rule at once. The captured mass is summed in a fixed order.
//
// Three passes over the row in the common case. Pass A histograms the top 12
// bits of every score (4,096 bins in shared memory). Pass B walks each warp's
// contiguous slice of the row: it counts the scores in bins above the K-th
// score's bin (all kept) and keeps that bin's scores (up to kCap of them, with
// their positions) in shared memory, where the remaining 20 bits are resolved
// (12, then 8) and each warp's counts of kept and equal scores are completed
// from the candidates' positions. The compaction pass then writes each warp's
// slice, a lane taking a run of 8 consecutive scores (two 16-byte loads) and
// one warp scan per 256 scores placing the lanes' kept positions. A bin holding
// more than kCap scores is resolved by two more passes over the row, and the
// slices are then counted by one more. Rows whose length is not a multiple of 4
// are read 4 bytes per load.
#include "block_scan.cuh"
#include "common.cuh"
#include "kernels.h"
#include "status.cuh"

namespace mcs {
namespace {

constexpr int kTopkThreads = 1024;
constexpr int kTopkWarps = kTopkThreads / 32;
constexpr int kLoads = 8;       // independent 4-byte row loads in flight per thread (strided passes)
constexpr int kVecLoads = 2;    // independent 16-byte row loads in flight per thread (pass A)
constexpr int kBinsA = 4096;    // pass A digit: bits 31..20
constexpr int kCap = 8192;      // scores of the K-th bin kept in shared memory
constexpr int kSmemBytes = kBinsA * 4 + kCap * 8;  // histogram, candidate scores and positions

// Finds, over kBins bins ordered from the highest down, the bin b with
// (elements in bins above b) < remaining <= that count + hist[b]. kBins is a
// multiple of 1024; every thread of the block calls it. Writes the count above
// b to *before and returns b (-1 if remaining exceeds the total).
template <int kBins>
__device__ __forceinline__ int block_find_digit_desc(const uint32_t* hist, uint32_t remaining, uint32_t* before,
                                                     uint32_t* warp_tot, int* sh_bin, uint32_t* sh_before) {
  constexpr int nbins = kBins, per = kBins / kTopkThreads;  // bins per thread, highest bins to thread 0
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  uint32_t c[per];
  uint32_t tot = 0;
#pragma unroll
  for (int i = 0; i < per; ++i) {
    c[i] = hist[nbins - 1 - (tid * per + i)];
    tot += c[i];
  }
  uint32_t incl = tot;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const uint32_t y = __shfl_up_sync(0xffffffffu, incl, off);
    if (lane >= off) incl += y;
  }
  if (lane == 31) warp_tot[warp] = incl;
  if (tid == 0) *sh_bin = -1;
  __syncthreads();
  uint32_t run = incl - tot;
  for (int w = 0; w < warp; ++w) run += warp_tot[w];
#pragma unroll
  for (int i = 0; i < per; ++i) {
    if (run < remaining && remaining <= run + c[i]) {  // exactly one thread matches (when remaining <= total)
      *sh_bin = nbins - 1 - (tid * per + i);
      *sh_before = run;
    }
    run += c[i];
  }
  __syncthreads();
  *before = *sh_before;
  return *sh_bin;
}

// Loads the V consecutive scores of a row starting at j0 (a multiple of V),
// zeros from hi on: two 16-byte loads (kVec: hi is then a multiple of 4) or V
// independent 4-byte loads.
template <int V, bool kVec>
__device__ __forceinline__ void load_run(const uint32_t* U, int j0, int hi, uint32_t (&u)[V]) {
  if constexpr (kVec) {
    static_assert(V % 4 == 0, "runs of whole 16-byte vectors");
#pragma unroll
    for (int h = 0; h < V / 4; ++h) {
      const int j = j0 + 4 * h;
      const uint4 x = j < hi ? __ldg(reinterpret_cast<const uint4*>(U + j)) : make_uint4(0, 0, 0, 0);
      u[4 * h] = x.x;
      u[4 * h + 1] = x.y;
      u[4 * h + 2] = x.z;
      u[4 * h + 3] = x.w;
    }
  } else {
#pragma unroll
    for (int t = 0; t < V; ++t) u[t] = j0 + t < hi ? __ldg(U + j0 + t) : 0u;
  }
}

// Exclusive prefix sum of v over the warp's lanes; *total gets the warp's sum.
__device__ __forceinline__ int warp_excl_sum(int v, int lane, int* total) {
  int incl = v;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, incl, off);
    if (lane >= off) incl += y;
  }
  *total = __shfl_sync(0xffffffffu, incl, 31);
  return incl - v;
}

template <bool kVec>
__global__ void __launch_bounds__(kTopkThreads) topk_kernel(const TopkParams p) {
  // a lane's run of consecutive scores in the slice passes: 8 (two 16-byte
  // loads) when rows allow 16-byte loads, else 4
  constexpr int V = kVec ? 8 : 4;
  extern __shared__ uint32_t dyn[];
  uint32_t* hist = dyn;                                        // [kBinsA]
  uint32_t* cand = dyn + kBinsA;                               // [kCap] scores of bin bA
  int32_t* cand_idx = reinterpret_cast<int32_t*>(cand + kCap);  // [kCap] their positions
  __shared__ uint32_t warp_tot[kTopkWarps];
  __shared__ int wgt[kTopkWarps], weq[kTopkWarps];
  __shared__ float warp_sum[kTopkWarps];
  __shared__ int sh_bin;
  __shared__ uint32_t sh_before, sh_ncand;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int row = blockIdx.x;
  const int grow = p.row0 + row;
  const float* S = p.scores + size_t(row) * p.N;
  const uint32_t* U = reinterpret_cast<const uint32_t*>(S);
  const uint4* U4 = reinterpret_cast<const uint4*>(S);
  const int N4 = p.N / 4;
  // warp w owns the contiguous slice [lo, hi) of the row in the slice passes
  // (a multiple of 256 scores long, so runs never straddle two warps)
  const int span = ((p.N + kTopkWarps - 1) / kTopkWarps + 255) & ~255;
  const int lo = min(p.N, warp * span), hi = min(p.N, lo + span);

  // ---- pass A: histogram of bits 31..20 over the whole row
  for (int i = tid; i < kBinsA; i += kTopkThreads) hist[i] = 0;
  __syncthreads();
  if (kVec) {
    for (int c0 = 0; c0 < N4; c0 += kVecLoads * kTopkThreads) {
      uint4 v[kVecLoads];
#pragma unroll
      for (int k = 0; k < kVecLoads; ++k) {
        const int j = c0 + k * kTopkThreads + tid;
        v[k] = j < N4 ? __ldg(U4 + j) : make_uint4(0, 0, 0, 0);
      }
#pragma unroll
      for (int k = 0; k < kVecLoads; ++k) {
        if (c0 + k * kTopkThreads + tid < N4) {
          atomicAdd(&hist[v[k].x >> 20], 1u);
          atomicAdd(&hist[v[k].y >> 20], 1u);
          atomicAdd(&hist[v[k].z >> 20], 1u);
          atomicAdd(&hist[v[k].w >> 20], 1u);
        }
      }
    }
  } else {
    for (int c0 = 0; c0 < p.N; c0 += kLoads * kTopkThreads) {
      uint32_t u[kLoads];
#pragma unroll
      for (int k = 0; k < kLoads; ++k) {
        const int j = c0 + k * kTopkThreads + tid;
        u[k] = j < p.N ? __ldg(U + j) : 0u;
      }
#pragma unroll
      for (int k = 0; k < kLoads; ++k)
        if (c0 + k * kTopkThreads + tid < p.N) atomicAdd(&hist[u[k] >> 20], 1u);
    }
  }
  __syncthreads();
  uint32_t before;
  const int bA = block_find_digit_desc<kBinsA>(hist, uint32_t(p.K), &before, warp_tot, &sh_bin, &sh_before);
  uint32_t remaining = uint32_t(p.K) - before;  // how many of bin bA's scores are kept
  const uint32_t nA = bA >= 0 ? hist[bA] : 0u;
  uint32_t prefix = uint32_t(bA < 0 ? 0 : bA) << 20, mask = 0xFFF00000u;
  __syncthreads();

  if (nA <= uint32_t(kCap)) {
    // ---- pass B, over each warp's slice: count the scores in bins above bA
    // (all kept) and keep bin bA's scores with their positions in shared memory
    if (tid == 0) sh_ncand = 0;
    if (tid < kTopkWarps) weq[tid] = 0;
    __syncthreads();
    int above = 0;
    for (int c = lo; c < hi; c += 32 * V) {
      const int j0 = c + lane * V;
      uint32_t u[V];
      load_run<V, kVec>(U, j0, hi, u);
#pragma unroll
      for (int t = 0; t < V; ++t) {
        const int b = int(u[t] >> 20);
        if (j0 + t < hi) {
          above += b > bA ? 1 : 0;
          if (b == bA) {
            const uint32_t slot = atomicAdd(&sh_ncand, 1u);
            if (slot < uint32_t(kCap)) {
              cand[slot] = u[t];
              cand_idx[slot] = j0 + t;
            }
          }
        }
      }
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) above += __shfl_xor_sync(0xffffffffu, above, off);
    if (lane == 0) wgt[warp] = above;
    __syncthreads();
    const int nc = int(min(sh_ncand, uint32_t(kCap)));  // == nA
    if (tid == 0 && sh_ncand != nA) raise_status(p.status, kStatusBounds);
    // bits 19..8 (4,096 bins), then bits 7..0 (256 bins), over the kept scores
    for (int i = tid; i < kBinsA; i += kTopkThreads) hist[i] = 0;
    __syncthreads();
    for (int i = tid; i < nc; i += kTopkThreads) atomicAdd(&hist[(cand[i] >> 8) & 0xFFFu], 1u);
    __syncthreads();
    const int bB = block_find_digit_desc<kBinsA>(hist, remaining, &before, warp_tot, &sh_bin, &sh_before);
    remaining -= before;
    prefix |= uint32_t(bB < 0 ? 0 : bB) << 8;
    mask |= 0xFFF00u;
    __syncthreads();
    for (int i = tid; i < 256; i += kTopkThreads) hist[i] = 0;
    __syncthreads();
    for (int i = tid; i < nc; i += kTopkThreads)
      if ((cand[i] & mask) == prefix) atomicAdd(&hist[cand[i] & 0xFFu], 1u);
    __syncthreads();
    if (warp == 0) {
      uint32_t b4;
      const int b = warp_find_digit(hist, remaining, /*descending=*/true, &b4);
      if (lane == 0) {
        sh_bin = b < 0 ? 0 : b;
        sh_before = b4;
      }
    }
    __syncthreads();
    prefix |= uint32_t(sh_bin);
    remaining -= sh_before;
    // each warp's counts of kept (> threshold) and equal scores: its bin-bA
    // candidates added to the scores above bin bA
    for (int i = tid; i < nc; i += kTopkThreads) {
      const int w = cand_idx[i] / span;
      if (cand[i] > prefix) atomicAdd(&wgt[w], 1);
      else if (cand[i] == prefix) atomicAdd(&weq[w], 1);
    }
    __syncthreads();
  } else {
    // ---- a crowded bin: bits 19..8 and 7..0 by two more passes over the row
    for (int pass = 0; pass < 2; ++pass) {
      const int shift = pass == 0 ? 8 : 0;
      const uint32_t dmask = pass == 0 ? 0xFFFu : 0xFFu;
      const int nbins = pass == 0 ? kBinsA : 256;
      for (int i = tid; i < nbins; i += kTopkThreads) hist[i] = 0;
      __syncthreads();
      for (int c0 = 0; c0 < p.N; c0 += kLoads * kTopkThreads) {
        uint32_t u[kLoads];
#pragma unroll
        for (int k = 0; k < kLoads; ++k) {
          const int j = c0 + k * kTopkThreads + tid;
          u[k] = j < p.N ? __ldg(U + j) : 0u;
        }
#pragma unroll
        for (int k = 0; k < kLoads; ++k)
          if (c0 + k * kTopkThreads + tid < p.N && (u[k] & mask) == prefix)
            atomicAdd(&hist[(u[k] >> shift) & dmask], 1u);
      }
      __syncthreads();
      int b;
      if (pass == 0) {
        b = block_find_digit_desc<kBinsA>(hist, remaining, &before, warp_tot, &sh_bin, &sh_before);
      } else {
        if (warp == 0) {
          uint32_t b4;
          const int bb = warp_find_digit(hist, remaining, /*descending=*/true, &b4);
          if (lane == 0) {
            sh_bin = bb;
            sh_before = b4;
          }
        }
        __syncthreads();
        b = sh_bin;
        before = sh_before;
      }
      remaining -= before;
      prefix |= uint32_t(b < 0 ? 0 : b) << shift;
      mask |= dmask << shift;
      __syncthreads();
    }
    // each warp counts its slice's kept and equal scores
    int cgt = 0, ceq = 0;
    for (int c = lo; c < hi; c += 32 * V) {
      const int j0 = c + lane * V;
      uint32_t u[V];
      load_run<V, kVec>(U, j0, hi, u);
#pragma unroll
      for (int t = 0; t < V; ++t) {
        const bool v = j0 + t < hi;
        cgt += (v && u[t] > prefix) ? 1 : 0;
        ceq += (v && u[t] == prefix) ? 1 : 0;
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
  }
  const uint32_t thr = prefix;            // bit pattern of the K-th largest score
  const int need_eq = int(remaining);     // how many scores equal to it are kept (lowest indices)

  // Ordered compaction over the warps' slices: one scan over the warps' counts
  // gives each warp its first output position; a warp then writes its kept
  // positions in index order, a lane taking a run of V consecutive scores and
  // one warp scan placing the runs (ties to the lower index: a warp keeps the
  // first equal scores that the warps before it left).
  int gt_before = 0, eq_before = 0, gt_all = 0, eq_all = 0;
  for (int w = 0; w < kTopkWarps; ++w) {
    const int a = wgt[w], b = weq[w];
    gt_before += w < warp ? a : 0;
    eq_before += w < warp ? b : 0;
    gt_all += a;
    eq_all += b;
  }
  const int take_eq = max(0, min(weq[warp], need_eq - eq_before));
  int out_pos = gt_before + min(eq_before, need_eq);
  int eq_seen = 0;
  float msum = 0.f;
  int32_t* out = p.idx + size_t(grow) * p.K;
  for (int c = lo; c < hi; c += 32 * V) {
    const int j0 = c + lane * V;
    uint32_t u[V];
    load_run<V, kVec>(U, j0, hi, u);
    bool sel[V];
    int ns = 0, ne = 0;
#pragma unroll
    for (int t = 0; t < V; ++t) {
      const bool v = j0 + t < hi;
      sel[t] = v && u[t] > thr;
      ne += (v && u[t] == thr) ? 1 : 0;
    }
    if (__any_sync(0xffffffffu, ne > 0)) {  // equal scores: the first take_eq of the slice are kept
      int ne_all;
      int e = eq_seen + warp_excl_sum(ne, lane, &ne_all);
#pragma unroll
      for (int t = 0; t < V; ++t) {
        if (j0 + t < hi && u[t] == thr) {
          sel[t] = e < take_eq;
          ++e;
        }
      }
      eq_seen += ne_all;
    }
#pragma unroll
    for (int t = 0; t < V; ++t) ns += sel[t] ? 1 : 0;
    int ns_all;
    int pos = out_pos + warp_excl_sum(ns, lane, &ns_all);
#pragma unroll
    for (int t = 0; t < V; ++t) {
      if (sel[t]) {
        if (pos < p.K) out[pos] = j0 + t;
        msum += __uint_as_float(u[t]);
        ++pos;
      }
    }
    out_pos += ns_all;
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

template <bool kVec>
cudaError_t launch_topk(const TopkParams& p, int nrows, cudaStream_t stream) {
  auto kern = topk_kernel<kVec>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
  if (e != cudaSuccess) return e;
  kern<<<nrows, kTopkThreads, kSmemBytes, stream>>>(p);
  note_launches(1);
  return cudaGetLastError();
}

}  // namespace

cudaError_t topk_rows(const TopkParams& p, int nrows, cudaStream_t stream) {
  if (nrows <= 0) return cudaSuccess;
  // 16-byte loads need every row to start on a 16-byte boundary (N % 4 == 0;
  // the score rows start at a 256-byte-aligned base)
  if (p.N % 4 == 0 && (reinterpret_cast<uintptr_t>(p.scores) & 15u) == 0) return launch_topk<true>(p, nrows, stream);
  return launch_topk<false>(p, nrows, stream);
}

}  // namespace mcs
