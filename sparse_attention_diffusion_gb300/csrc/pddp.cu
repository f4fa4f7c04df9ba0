// PDDP query grouping on the GPU [MC-Sparse summary: PDDP paragraph: project the
// queries onto their principal direction, split at the median, repeat, giving
// groups of exactly C].
//
// Every head is processed at once, one tree level per round of launches. The
// tree shape depends only on G: a node of n groups splits into floor(n/2) and
// n - floor(n/2) groups, so node k of level l is found by walking the bits of
// k from the root. The current ordering `perm` keeps every node's members in a
// contiguous, ascending run; a level
//   1. sums the members of each chunk (<= 8 groups of one node; one group on
//      the fp64 path of a layer with few chunks) -> node mean,
//   2. accumulates each chunk's centred covariance (d x d) -> node covariance,
//   3. runs exactly `iters` power iterations w = Cov v, v = w/|w| from 1/sqrt(d),
//   4. projects every member on v and turns the projection into an
//      order-preserving integer key (pads get the largest key),
//   5. radix-selects the rank floor(n/2)*C key of each node and stably
//      partitions the run: smaller keys (ties: earlier, i.e. lower token id) left.
// All reductions run in a fixed order, so a run is deterministic. fp32 inputs
// accumulate in fp64 end to end; bf16 inputs accumulate in fp32. For bf16 at
// d = 128, steps 1 and 2 are one tensor-core pass (pddp_tc.cu) giving each
// chunk's sum and raw second moment sum x x^T; the node covariance is then
// their fixed-order sum minus n mu mu^T.
#include <cmath>
#include <type_traits>
#include <vector>

#include "block_scan.cuh"
#include "common.cuh"
#include "kernels.h"
#include "status.cuh"

namespace mcs {
namespace {

constexpr int kChunkGroups = 8;  // groups per moment chunk (the usual case)

// Groups per moment chunk. A chunk is one CTA of the moment kernels; on the fp64
// path (fp32 inputs) a layer with few chunks would leave most SMs idle on
// fp64 arithmetic (the tiny 1,024-token head has 2 chunks of 8 groups per
// level), so there every group is its own chunk while the chunks stay few
// enough for the fp64 partial moments to stay small.
inline int chunk_groups(int BH, int G, bool bf16) {
  return (!bf16 && BH * ((G + kChunkGroups - 1) / kChunkGroups) < 256) ? 1 : kChunkGroups;
}

__host__ __device__ inline bool pddp_node(int G, int level, int k, int* start, int* n) {
  int s = 0, m = G;
  for (int b = level - 1; b >= 0; --b) {
    if (m < 2) return false;
    const int nl = m / 2;
    if ((k >> b) & 1) {
      s += nl;
      m -= nl;
    } else {
      m = nl;
    }
  }
  *start = s;
  *n = m;
  return true;
}

int num_levels(int G) {
  int L = 0;
  while ((1 << L) < G) ++L;
  return L;
}

int host_level_chunks(int G, int level, int cg) {
  int total = 0;
  for (int k = 0; k < (1 << level); ++k) {
    int s, n;
    if (pddp_node(G, level, k, &s, &n) && n >= 2) total += (n + cg - 1) / cg;
  }
  return total;
}

struct Tables {
  int* node_start;   // [L][G]
  int* node_n;       // [L][G]: groups in the node, 0 when absent or a leaf
  int* node_chunk0;  // [L][G]
  int* node_nchunks; // [L][G]
  int* chunk_node;   // [L][G]
  int* chunk_g0;     // [L][G]
  int* chunk_ng;     // [L][G]
  int cg;            // groups per chunk
};

__global__ void __launch_bounds__(1024) tables_kernel(Tables t, int G) {
  __shared__ int warp_tot[32];
  __shared__ int s_base;
  const int level = blockIdx.x;
  const int nodes = 1 << level;
  if (threadIdx.x == 0) s_base = 0;
  __syncthreads();
  for (int k0 = 0; k0 < nodes; k0 += 1024) {
    const int k = k0 + threadIdx.x;
    int s = 0, n = 0;
    const bool exists = k < nodes && pddp_node(G, level, k, &s, &n);
    const bool active = exists && n >= 2;
    const int nch = active ? (n + t.cg - 1) / t.cg : 0;
    // exclusive prefix of nch over the block (nch <= G fits easily)
    int pre = 0, tot = 0;
    {
      // scan of small integers via per-bit predicate counts would be wasteful; use warp scan + block sum
      const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
      int incl = nch;
      for (int off = 1; off < 32; off <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, incl, off);
        if (lane >= off) incl += y;
      }
      if (lane == 31) warp_tot[warp] = incl;
      __syncthreads();
      int wpre = 0;
      for (int w = 0; w < 32; ++w) {
        wpre += (w < warp) ? warp_tot[w] : 0;
        tot += warp_tot[w];
      }
      pre = wpre + incl - nch;
      __syncthreads();
    }
    const int c0 = s_base + pre;
    if (k < nodes) {
      const size_t o = size_t(level) * G + k;
      t.node_start[o] = s;
      t.node_n[o] = active ? n : 0;
      t.node_chunk0[o] = c0;
      t.node_nchunks[o] = nch;
      for (int c = 0; c < nch; ++c) {
        const size_t co = size_t(level) * G + c0 + c;
        t.chunk_node[co] = k;
        t.chunk_g0[co] = s + c * t.cg;
        t.chunk_ng[co] = min(t.cg, n - c * t.cg);
      }
    }
    __syncthreads();
    if (threadIdx.x == 0) s_base += tot;
    __syncthreads();
  }
}

__global__ void init_perm_kernel(int32_t* perm, int N_pad, size_t total) {
  for (size_t i = blockIdx.x * size_t(blockDim.x) + threadIdx.x; i < total; i += size_t(gridDim.x) * blockDim.x)
    perm[i] = int32_t(i % N_pad);
}

__global__ void finalize_kernel(const int32_t* perm, int32_t* group_of, int N, int N_pad, int C, size_t total,
                                uint32_t* status) {
  for (size_t i = blockIdx.x * size_t(blockDim.x) + threadIdx.x; i < total; i += size_t(gridDim.x) * blockDim.x) {
    const size_t bh = i / N_pad;
    const int pos = int(i % N_pad);
    const int t = perm[i];
    if (t < 0 || t >= N_pad) {
      raise_status(status, kStatusBounds);
      continue;
    }
    if (t < N) group_of[bh * N + t] = pos / C;
  }
}

template <typename T>
__device__ __forceinline__ float ld_f(const T* p) {
  return to_f32(*p);
}

// 1. per-chunk sums of real members: thread (row lane rl, chunk cc) sums the
// 16-byte chunk cc of rows rl, rl + RL, ..., four rows in flight at a time; the
// row lanes are then added in a fixed order
template <typename T, typename A, int D>
__global__ void __launch_bounds__(256) sum_kernel(const T* __restrict__ x, const int32_t* __restrict__ perm, Tables t,
                                                  int level, int N, int N_pad, int C, int G, A* psum, int* pcnt,
                                                  int max_chunks) {
  constexpr int V = 16 / int(sizeof(T));  // elements per 16-byte chunk
  constexpr int CPR = D / V;              // chunks per row
  constexpr int RL = 256 / CPR;           // row lanes
  constexpr int R = 4;
  __shared__ A part[RL][D];
  __shared__ int cnt_part[RL];
  const int c = blockIdx.x, bh = blockIdx.y;
  const size_t to = size_t(level) * G + c;
  const int g0 = t.chunk_g0[to], ng = t.chunk_ng[to];
  const int cc = threadIdx.x % CPR, rl = threadIdx.x / CPR;
  const int32_t* pr = perm + size_t(bh) * N_pad + size_t(g0) * C;
  const T* xb = x + size_t(bh) * N * D + cc * V;
  A acc[V];
#pragma unroll
  for (int k = 0; k < V; ++k) acc[k] = 0;
  int cnt = 0;
  const int rows = ng * C;
  for (int r0 = rl; r0 < rows; r0 += R * RL) {
    int tok[R];
#pragma unroll
    for (int q = 0; q < R; ++q) tok[q] = r0 + q * RL < rows ? pr[r0 + q * RL] : N;
    uint4 raw[R];
#pragma unroll
    for (int q = 0; q < R; ++q)
      if (tok[q] < N) raw[q] = *reinterpret_cast<const uint4*>(xb + size_t(tok[q]) * D);
#pragma unroll
    for (int q = 0; q < R; ++q) {
      if (tok[q] < N) {
        const T* vals = reinterpret_cast<const T*>(&raw[q]);
#pragma unroll
        for (int k = 0; k < V; ++k) acc[k] += A(to_f32(vals[k]));
        ++cnt;
      }
    }
  }
#pragma unroll
  for (int k = 0; k < V; ++k) part[rl][cc * V + k] = acc[k];
  if (cc == 0) cnt_part[rl] = cnt;
  __syncthreads();
  if (threadIdx.x < D) {
    A s = 0;
    for (int l = 0; l < RL; ++l) s += part[l][threadIdx.x];
    psum[(size_t(bh) * max_chunks + c) * D + threadIdx.x] = s;
  }
  if (threadIdx.x == 0) {
    int s = 0;
    for (int l = 0; l < RL; ++l) s += cnt_part[l];
    pcnt[size_t(bh) * max_chunks + c] = s;
  }
}

// 2. node mean, start vector
template <typename A, int D>
__global__ void mean_kernel(Tables t, int level, int G, const A* psum, const int* pcnt, A* node_mu, A* node_v,
                            int max_chunks, const float* dirs_in, int slots) {
  const int k = blockIdx.x, bh = blockIdx.y;
  const size_t to = size_t(level) * G + k;
  if (t.node_n[to] < 2) return;
  const int c0 = t.node_chunk0[to], nc = t.node_nchunks[to];
  A s = 0;
  int cnt = 0;
  for (int c = 0; c < nc; ++c) {
    s += psum[(size_t(bh) * max_chunks + c0 + c) * D + threadIdx.x];
    cnt += pcnt[size_t(bh) * max_chunks + c0 + c];
  }
  node_mu[(size_t(bh) * G + k) * D + threadIdx.x] = cnt > 0 ? s / A(cnt) : A(0);
  // start vector: the stored direction of this node (warm start; level-by-level
  // slot 2^level - 1 + k) or 1/sqrt(D) * ones
  node_v[(size_t(bh) * G + k) * D + threadIdx.x] =
      dirs_in != nullptr ? A(dirs_in[(size_t(bh) * slots + (size_t(1) << level) - 1 + k) * D + threadIdx.x])
                         : A(1) / sqrt(A(D));
}

// 3a. per-chunk centred covariance; thread (bi, bj) owns a TB x TB block.
template <typename T, typename A, int D>
__global__ void __launch_bounds__(256) cov_kernel(const T* __restrict__ x, const int32_t* __restrict__ perm, Tables t,
                                                  int level, int N, int N_pad, int C, int G, const A* node_mu,
                                                  A* pcov, int max_chunks) {
  constexpr int TB = D / 16;
  constexpr int RB = 32;
  __shared__ A mu[D];
  __shared__ A xs[RB][D];
  const int c = blockIdx.x, bh = blockIdx.y;
  const size_t to = size_t(level) * G + c;
  const int node = t.chunk_node[to], g0 = t.chunk_g0[to], ng = t.chunk_ng[to];
  if (threadIdx.x < D) mu[threadIdx.x] = node_mu[(size_t(bh) * G + node) * D + threadIdx.x];
  const int bi = threadIdx.x / 16, bj = threadIdx.x % 16;
  A acc[TB][TB];
#pragma unroll
  for (int i = 0; i < TB; ++i)
#pragma unroll
    for (int j = 0; j < TB; ++j) acc[i][j] = 0;
  const int32_t* pr = perm + size_t(bh) * N_pad + size_t(g0) * C;
  const T* xb = x + size_t(bh) * N * D;
  const int rows = ng * C;
  __syncthreads();
  // rows are staged 16 bytes at a time (one index lookup per 16-byte chunk of a
  // row), then centred; the products below are the same in the same order
  constexpr int V = 16 / int(sizeof(T));  // elements per 16-byte chunk
  constexpr int CPR = D / V;              // chunks per row
  for (int r0 = 0; r0 < rows; r0 += RB) {
    for (int e = threadIdx.x; e < RB * CPR; e += 256) {
      const int rr = e / CPR, cc = e % CPR;
      const int r = r0 + rr;
      int tok = N;
      if (r < rows) tok = pr[r];
      if (tok < N) {
        const uint4 raw = *reinterpret_cast<const uint4*>(xb + size_t(tok) * D + cc * V);
        const T* vals = reinterpret_cast<const T*>(&raw);
#pragma unroll
        for (int k = 0; k < V; ++k) xs[rr][cc * V + k] = A(to_f32(vals[k])) - mu[cc * V + k];
      } else {
#pragma unroll
        for (int k = 0; k < V; ++k) xs[rr][cc * V + k] = A(0);
      }
    }
    __syncthreads();
#pragma unroll 4
    for (int rr = 0; rr < RB; ++rr) {
      A a[TB], b[TB];
#pragma unroll
      for (int i = 0; i < TB; ++i) {
        a[i] = xs[rr][bi * TB + i];
        b[i] = xs[rr][bj * TB + i];
      }
#pragma unroll
      for (int i = 0; i < TB; ++i)
#pragma unroll
        for (int j = 0; j < TB; ++j) acc[i][j] += a[i] * b[j];
    }
    __syncthreads();
  }
  A* out = pcov + (size_t(bh) * max_chunks + c) * D * D;
#pragma unroll
  for (int i = 0; i < TB; ++i)
#pragma unroll
    for (int j = 0; j < TB; ++j) out[(bi * TB + i) * D + bj * TB + j] = acc[i][j];
}

// 3b. node covariance (fixed-order sum of its chunks) and the power iterations.
// kRaw: the chunks hold raw second moments (tensor-core path), so the node's
// n mu mu^T is subtracted once here. The chunk sum keeps kEb elements of a
// thread in registers so that their loads of one chunk are in flight together
// (the sum over chunks stays in chunk order; a shallow node has dozens of
// chunks, and one load at a time left the sum waiting on memory latency).
template <typename A, int D, bool kRaw>
__global__ void __launch_bounds__(256) power_kernel(Tables t, int level, int G, const A* pcov, A* node_v, int iters,
                                                    int max_chunks, const A* node_mu, const int* pcnt, float* dirs_out,
                                                    int slots) {
  constexpr int kThreads = 256;
  constexpr int kEb = 16;            // covariance elements per thread per round of the chunk sum
  static_assert((D * D) % (kThreads * kEb) == 0, "shape");
  extern __shared__ uint8_t dyn[];
  A* cov = reinterpret_cast<A*>(dyn);  // [D][D]
  A* v = cov + D * D;                  // [D]
  A* w = v + D;                        // [D]
  __shared__ A red[D / 32];
  const int k = blockIdx.x, bh = blockIdx.y;
  const size_t to = size_t(level) * G + k;
  if (t.node_n[to] < 2) return;
  const int c0 = t.node_chunk0[to], nc = t.node_nchunks[to];
  if (kRaw && threadIdx.x < D) w[threadIdx.x] = node_mu[(size_t(bh) * G + k) * D + threadIdx.x];
  int cnt = 0;
  if (kRaw)
    for (int c = 0; c < nc; ++c) cnt += pcnt[size_t(bh) * max_chunks + c0 + c];
  __syncthreads();
  const A* pc = pcov + (size_t(bh) * max_chunks + c0) * D * D;
  for (int e0 = threadIdx.x; e0 < D * D; e0 += kThreads * kEb) {
    A acc[kEb];
#pragma unroll
    for (int i = 0; i < kEb; ++i) acc[i] = 0;
    for (int c = 0; c < nc; ++c) {
      const A* src = pc + size_t(c) * D * D + e0;
#pragma unroll
      for (int i = 0; i < kEb; ++i) acc[i] += src[i * kThreads];
    }
#pragma unroll
    for (int i = 0; i < kEb; ++i) {
      const int e = e0 + i * kThreads;
      A s = acc[i];
      if (kRaw) s -= (A(cnt) * w[e / D]) * w[e % D];
      cov[e] = s;
    }
  }
  __syncthreads();
  if (threadIdx.x < D) v[threadIdx.x] = node_v[(size_t(bh) * G + k) * D + threadIdx.x];
  __syncthreads();
  // fp64 (fp32 inputs): a column's sum is split over the 256 / D threads that
  // share it, each with four partial sums (fp64 FMAs are few per SM and a
  // D-long dependent chain would be pure latency); the parts are added in a
  // fixed order. fp32 accumulation keeps one in-order chain per column.
  constexpr bool kSplit = std::is_same<A, double>::value;
  constexpr int kH = kSplit ? 256 / D : 1, kJL = D / kH;
  __shared__ A part[kH][D];
  for (int it = 0; it < iters; ++it) {
    if constexpr (kSplit) {
      const int col = threadIdx.x % D, hh = threadIdx.x / D;
      A s4[4] = {A(0), A(0), A(0), A(0)};
#pragma unroll
      for (int jj = 0; jj < kJL; jj += 4) {
#pragma unroll
        for (int q = 0; q < 4; ++q) s4[q] += cov[(hh * kJL + jj + q) * D + col] * v[hh * kJL + jj + q];
      }
      part[hh][col] = (s4[0] + s4[1]) + (s4[2] + s4[3]);
      __syncthreads();
    }
    if (threadIdx.x < D) {
      // the covariance is exactly symmetric, so read column i (conflict-free)
      A s = 0;
      if constexpr (kSplit) {
#pragma unroll
        for (int i = 0; i < kH; ++i) s += part[i][threadIdx.x];
      } else {
        for (int j = 0; j < D; ++j) s += cov[j * D + threadIdx.x] * v[j];
      }
      w[threadIdx.x] = s;
      A sq = s * s;
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) sq += __shfl_xor_sync(0xffffffffu, sq, off);
      if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = sq;
    }
    __syncthreads();
    A nrm2 = 0;
    for (int i = 0; i < D / 32; ++i) nrm2 += red[i];
    if (threadIdx.x < D && nrm2 > A(0)) v[threadIdx.x] = w[threadIdx.x] / sqrt(nrm2);
    __syncthreads();
  }
  if (threadIdx.x < D) {
    node_v[(size_t(bh) * G + k) * D + threadIdx.x] = v[threadIdx.x];
    if (dirs_out != nullptr)
      dirs_out[(size_t(bh) * slots + (size_t(1) << level) - 1 + k) * D + threadIdx.x] = float(v[threadIdx.x]);
  }
}

__device__ __forceinline__ uint32_t order_key(float f) {
  uint32_t u = __float_as_uint(f == 0.f ? 0.f : f);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
__device__ __forceinline__ uint64_t order_key(double f) {
  uint64_t u = uint64_t(__double_as_longlong(f == 0.0 ? 0.0 : f));
  return (u >> 63) ? ~u : (u | (uint64_t(1) << 63));
}

// 4. projection keys, one warp per member (four members per warp iteration)
template <typename T, typename A, int D, typename KeyT>
__global__ void __launch_bounds__(256) keys_kernel(const T* __restrict__ x, const int32_t* __restrict__ perm, Tables t,
                                                   int level, int N, int N_pad, int C, int G, const A* node_mu,
                                                   const A* node_v, KeyT* keys) {
  __shared__ A mu[D], vv[D];
  const int c = blockIdx.x, bh = blockIdx.y;
  const size_t to = size_t(level) * G + c;
  const int node = t.chunk_node[to], g0 = t.chunk_g0[to], ng = t.chunk_ng[to];
  if (threadIdx.x < D) {
    mu[threadIdx.x] = node_mu[(size_t(bh) * G + node) * D + threadIdx.x];
    vv[threadIdx.x] = node_v[(size_t(bh) * G + node) * D + threadIdx.x];
  }
  __syncthreads();
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const size_t base = size_t(bh) * N_pad + size_t(g0) * C;
  const T* xb = x + size_t(bh) * N * D;
  // lane l holds elements [l*E, l*E + E) of a row (one vector load); four rows
  // per warp iteration so their loads are in flight together
  constexpr int E = D / 32;
  constexpr int R = 4;
  const int rows = ng * C;
  for (int r0 = warp * R; r0 < rows; r0 += 8 * R) {
    int tok[R];
#pragma unroll
    for (int q = 0; q < R; ++q) tok[q] = r0 + q < rows ? perm[base + r0 + q] : N;
    A vals[R][E];
#pragma unroll
    for (int q = 0; q < R; ++q) {
      T raw[E];
      if (tok[q] < N) {
        const T* src = xb + size_t(tok[q]) * D + lane * E;
        if constexpr (E * sizeof(T) == 16) *reinterpret_cast<uint4*>(raw) = *reinterpret_cast<const uint4*>(src);
        else if constexpr (E * sizeof(T) == 8) *reinterpret_cast<uint2*>(raw) = *reinterpret_cast<const uint2*>(src);
        else *reinterpret_cast<uint32_t*>(raw) = *reinterpret_cast<const uint32_t*>(src);
      } else {
#pragma unroll
        for (int k = 0; k < E; ++k) raw[k] = from_f32<T>(0.f);
      }
#pragma unroll
      for (int k = 0; k < E; ++k) vals[q][k] = A(to_f32(raw[k]));
    }
#pragma unroll
    for (int q = 0; q < R; ++q) {
      A s = 0;
#pragma unroll
      for (int k = 0; k < E; ++k) s += (vals[q][k] - mu[lane * E + k]) * vv[lane * E + k];
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) s += __shfl_xor_sync(0xffffffffu, s, off);
      if (lane == 0 && r0 + q < rows) keys[base + r0 + q] = tok[q] < N ? order_key(s) : ~KeyT(0);
    }
  }
}

// 5. rank split of each node: radix select + stable partition into perm_next
template <typename KeyT>
__global__ void __launch_bounds__(1024) split_kernel(const int32_t* __restrict__ perm_cur, int32_t* perm_next,
                                                     const KeyT* __restrict__ keys, Tables t, int level, int N_pad,
                                                     int C, int G, uint32_t* status) {
  __shared__ uint32_t hist[256];
  __shared__ int warp_tot[32];
  __shared__ KeyT sh_prefix;
  __shared__ uint32_t sh_remaining;
  const int k = blockIdx.x, bh = blockIdx.y;
  const size_t to = size_t(level) * G + k;
  const int n = t.node_n[to];
  if (n < 2) return;
  const int tid = threadIdx.x;
  const int len = n * C, m = (n / 2) * C;
  const size_t base = size_t(bh) * N_pad + size_t(t.node_start[to]) * C;
  constexpr int kBits = int(sizeof(KeyT)) * 8;
  KeyT prefix = 0, mask = 0;
  uint32_t remaining = uint32_t(m);
  for (int shift = kBits - 8; shift >= 0; shift -= 8) {
    for (int i = tid; i < 256; i += blockDim.x) hist[i] = 0;
    __syncthreads();
    for (int i = tid; i < len; i += blockDim.x) {
      const KeyT key = keys[base + i];
      if ((key & mask) == prefix) atomicAdd(&hist[uint32_t(key >> shift) & 255u], 1u);
    }
    __syncthreads();
    if (tid < 32) {
      uint32_t before;
      const int b = warp_find_digit(hist, remaining, /*descending=*/false, &before);
      if (tid == 0) {
        sh_prefix = prefix | (KeyT(b < 0 ? 0 : b) << shift);
        sh_remaining = remaining - before;
      }
    }
    __syncthreads();
    prefix = sh_prefix;
    remaining = sh_remaining;
    mask |= KeyT(0xFF) << shift;
  }
  const KeyT thr = prefix;
  const uint32_t need_eq = remaining;
  int base_left = 0, base_right = 0, base_eq = 0;
  for (int c0 = 0; c0 < len; c0 += blockDim.x) {
    const int i = c0 + tid;
    const bool valid = i < len;
    const KeyT key = valid ? keys[base + i] : KeyT(0);
    const int tok = valid ? perm_cur[base + i] : 0;
    const bool lt = valid && key < thr, eq = valid && key == thr;
    int eq_tot, left_tot, valid_tot;
    const int eq_pre = block_excl_count(eq, warp_tot, &eq_tot);
    const bool left = lt || (eq && uint32_t(base_eq + eq_pre) < need_eq);
    const int left_pre = block_excl_count(left, warp_tot, &left_tot);
    const int valid_pre = block_excl_count(valid, warp_tot, &valid_tot);
    if (valid) {
      // a correct select gives exactly m left members; stay inside the node regardless
      const int dst = left ? base_left + left_pre : m + base_right + (valid_pre - left_pre);
      if (dst < len) perm_next[base + dst] = tok;
      else raise_status(status, kStatusBounds);
    }
    base_left += left_tot;
    base_right += valid_tot - left_tot;
    base_eq += eq_tot;
  }
}

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

struct WsLayout {
  size_t perm_tmp, keys, tables, psum, pcnt, node_mu, node_v, pcov, total;
  int L, max_chunks;
  int cg;  // groups per moment chunk
};

WsLayout layout(int BH, int N_pad, int C, int G, int d, bool bf16) {
  WsLayout w{};
  const size_t asz = bf16 ? sizeof(float) : sizeof(double);
  w.L = num_levels(G);
  w.cg = chunk_groups(BH, G, bf16);
  int mc = 1;
  for (int l = 0; l < w.L; ++l) mc = std::max(mc, host_level_chunks(G, l, w.cg));
  w.max_chunks = mc;
  size_t off = 0;
  w.perm_tmp = off; off = align256(off + size_t(BH) * N_pad * 4);
  w.keys = off; off = align256(off + size_t(BH) * N_pad * 8);
  w.tables = off; off = align256(off + size_t(7) * std::max(w.L, 1) * G * 4);
  w.psum = off; off = align256(off + size_t(BH) * mc * d * asz);
  w.pcnt = off; off = align256(off + size_t(BH) * mc * 4);
  w.node_mu = off; off = align256(off + size_t(BH) * G * d * asz);
  w.node_v = off; off = align256(off + size_t(BH) * G * d * asz);
  w.pcov = off; off = align256(off + size_t(BH) * mc * d * d * asz);
  w.total = off;
  return w;
}

template <typename T, typename A, int D, typename KeyT>
cudaError_t run_typed(const PddpProblem& p, uint8_t* ws, cudaStream_t s) {
  const WsLayout w = layout(p.BH, p.N_pad, p.C, p.G, p.d, p.bf16);
  const int G = p.G;
  const T* x = static_cast<const T*>(p.q);
  int32_t* bufs[2];
  // level l reads bufs[l & 1] and writes bufs[(l + 1) & 1]; the last write lands in p.perm
  bufs[w.L & 1] = p.perm;
  bufs[(w.L & 1) ^ 1] = reinterpret_cast<int32_t*>(ws + w.perm_tmp);
  const size_t total = size_t(p.BH) * p.N_pad;
  const int slots = (1 << w.L) - 1;  // direction-table rows per head
  int nlaunch = 0;
  init_perm_kernel<<<1024, 256, 0, s>>>(bufs[0], p.N_pad, total);
  ++nlaunch;
  Tables t;
  int* tb = reinterpret_cast<int*>(ws + w.tables);
  const size_t TL = size_t(std::max(w.L, 1)) * G;
  t.node_start = tb;
  t.node_n = tb + TL;
  t.node_chunk0 = tb + 2 * TL;
  t.node_nchunks = tb + 3 * TL;
  t.chunk_node = tb + 4 * TL;
  t.chunk_g0 = tb + 5 * TL;
  t.chunk_ng = tb + 6 * TL;
  t.cg = w.cg;
  A* psum = reinterpret_cast<A*>(ws + w.psum);
  int* pcnt = reinterpret_cast<int*>(ws + w.pcnt);
  A* node_mu = reinterpret_cast<A*>(ws + w.node_mu);
  A* node_v = reinterpret_cast<A*>(ws + w.node_v);
  A* pcov = reinterpret_cast<A*>(ws + w.pcov);
  KeyT* keys = reinterpret_cast<KeyT*>(ws + w.keys);
  if (w.L > 0) {
    tables_kernel<<<w.L, 1024, 0, s>>>(t, G);
    ++nlaunch;
  }
  // bf16 at d = 128: chunk moments on the tensor cores (raw second moments)
  constexpr bool kTc = std::is_same<T, __nv_bfloat16>::value && D == 128;
  const int power_smem = int((D * D + 2 * D) * sizeof(A));
  cudaError_t e = cudaFuncSetAttribute(power_kernel<A, D, kTc>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       power_smem);
  if (e != cudaSuccess) return e;
  for (int l = 0; l < w.L; ++l) {
    const int nodes = 1 << l;
    const int nch = host_level_chunks(G, l, w.cg);
    const dim3 gc(nch, p.BH), gn(nodes, p.BH);
    int32_t* cur = bufs[l & 1];
    int32_t* nxt = bufs[(l + 1) & 1];
    if constexpr (kTc) {
      e = pddp_moments_tc(x, cur, t.chunk_g0 + size_t(l) * G, t.chunk_ng + size_t(l) * G, nch, p.BH, p.N, p.N_pad,
                          p.C, psum, pcnt, pcov, w.max_chunks, p.status, p.num_sms, s);
      if (e != cudaSuccess) return e;
      mean_kernel<A, D><<<gn, D, 0, s>>>(t, l, G, psum, pcnt, node_mu, node_v, w.max_chunks, p.dirs_in, slots);
      nlaunch += 1;
    } else {
      sum_kernel<T, A, D><<<gc, 256, 0, s>>>(x, cur, t, l, p.N, p.N_pad, p.C, G, psum, pcnt, w.max_chunks);
      mean_kernel<A, D><<<gn, D, 0, s>>>(t, l, G, psum, pcnt, node_mu, node_v, w.max_chunks, p.dirs_in, slots);
      cov_kernel<T, A, D><<<gc, 256, 0, s>>>(x, cur, t, l, p.N, p.N_pad, p.C, G, node_mu, pcov, w.max_chunks);
      nlaunch += 3;
    }
    power_kernel<A, D, kTc><<<gn, 256, power_smem, s>>>(t, l, G, pcov, node_v, p.iters, w.max_chunks, node_mu, pcnt,
                                                        p.dirs_out, slots);
    keys_kernel<T, A, D, KeyT><<<gc, 256, 0, s>>>(x, cur, t, l, p.N, p.N_pad, p.C, G, node_mu, node_v, keys);
    e = cudaMemcpyAsync(nxt, cur, total * sizeof(int32_t), cudaMemcpyDeviceToDevice, s);
    if (e != cudaSuccess) return e;
    split_kernel<KeyT><<<gn, 1024, 0, s>>>(cur, nxt, keys, t, l, p.N_pad, p.C, G, p.status);
    nlaunch += 3;
  }
  finalize_kernel<<<1024, 256, 0, s>>>(p.perm, p.group_of, p.N, p.N_pad, p.C, total, p.status);
  ++nlaunch;
  note_launches(nlaunch);
  return cudaGetLastError();
}

}  // namespace

int pddp_dir_slots(int G) { return (1 << num_levels(G)) - 1; }

size_t pddp_workspace_bytes(int BH, int N_pad, int C, int G, int d, bool bf16) {
  return layout(BH, N_pad, C, G, d, bf16).total;
}

cudaError_t pddp_run(const PddpProblem& p, void* ws, size_t ws_bytes, cudaStream_t stream) {
  uint8_t* w = static_cast<uint8_t*>(ws);
  if (p.bf16) {
    if (p.d == 128) return run_typed<__nv_bfloat16, float, 128, uint32_t>(p, w, stream);
    if (p.d == 64) return run_typed<__nv_bfloat16, float, 64, uint32_t>(p, w, stream);
  } else {
    if (p.d == 128) return run_typed<float, double, 128, uint64_t>(p, w, stream);
    if (p.d == 64) return run_typed<float, double, 64, uint64_t>(p, w, stream);
  }
  return cudaErrorInvalidValue;
}

}  // namespace mcs
