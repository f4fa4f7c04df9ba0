// fp32 attention path (CUDA-core FFMA, no tensor cores): fp32 inputs must match
// the float64 reference to 1e-5, which tf32 tensor-core products cannot do.
// Same operations as the tcgen05 path: dense attention with the row LSE, the
// token-gather sparse attention with its residual epilogues, and pass 2 of the
// anchor selection [MC-Sparse summary: index-gather/PDDP, anchor two-pass and
// residual paragraphs]. Exponentials use the accurate expf/logf.
#include <cmath>

#include "common.cuh"
#include "kernels.h"
#include "status.cuh"

namespace mcs {
namespace {

constexpr int kRowsPerCta = 64;
constexpr int kKeyTile = 32;

// 256 threads: 64 query rows x 4 threads; thread q4 of a row owns dims i*4 + q4.
template <int D, bool kSparse, int kEpi, bool kPV>
__global__ void __launch_bounds__(256) simt_attn_kernel(const SimtAttnParams p) {
  constexpr int DQ = D / 4;
  __shared__ __align__(16) float ks[kKeyTile][D];
  __shared__ __align__(16) float vs[kKeyTile][D];
  __shared__ int ktok[kKeyTile];
  const int tid = threadIdx.x, r = tid >> 2, q4 = tid & 3;
  const int bh = blockIdx.y;
  const int halves = kSparse ? p.C / kRowsPerCta : 1;
  const int g = kSparse ? blockIdx.x / halves : 0;
  const int half = kSparse ? blockIdx.x % halves : 0;
  int tok = -1;
  if (kSparse) {
    const int t = p.perm[size_t(bh) * p.N_pad + size_t(g) * p.C + half * kRowsPerCta + r];
    if (t < 0 || t >= p.N_pad) {
      if (q4 == 0) raise_status(p.status, kStatusBounds);
    } else if (t < p.N) {
      tok = t;
    }
  } else {
    const int t = blockIdx.x * kRowsPerCta + r;
    if (t < p.N) tok = t;
  }
  const float* qb = p.q + size_t(bh) * p.N * D;
  const float* kb = p.k + size_t(bh) * p.N * D;
  const float* vb = p.v + size_t(bh) * p.N * D;
  float q[DQ], o[DQ];
#pragma unroll
  for (int i = 0; i < DQ; ++i) {
    q[i] = tok >= 0 ? qb[size_t(tok) * D + i * 4 + q4] : 0.f;
    o[i] = 0.f;
  }
  const int nkv = kSparse ? p.K : p.N;
  const int32_t* idxg = kSparse ? p.idx + (size_t(bh) * p.G + g) * size_t(p.K) : nullptr;
  float m = -INFINITY, l = 0.f;
  for (int j0 = 0; j0 < nkv; j0 += kKeyTile) {
    if (tid < kKeyTile) {
      int t = -1;
      if (j0 + tid < nkv) {
        const int c = kSparse ? idxg[j0 + tid] : j0 + tid;
        if (c < 0 || c >= p.N) raise_status(p.status, kStatusBounds);
        else t = c;
      }
      ktok[tid] = t;
    }
    __syncthreads();
    for (int e = tid; e < kKeyTile * D / 4; e += 256) {
      const int jj = e / (D / 4), c4 = e % (D / 4);
      const int t = ktok[jj];
      float4 kv = make_float4(0.f, 0.f, 0.f, 0.f), vv = kv;
      if (t >= 0) {
        kv = reinterpret_cast<const float4*>(kb + size_t(t) * D)[c4];
        if (kPV) vv = reinterpret_cast<const float4*>(vb + size_t(t) * D)[c4];
      }
      reinterpret_cast<float4*>(&ks[jj][0])[c4] = kv;
      reinterpret_cast<float4*>(&vs[jj][0])[c4] = vv;
    }
    __syncthreads();
    const int nv = min(kKeyTile, nkv - j0);
    float s[kKeyTile];
    float tmax = -INFINITY;
#pragma unroll
    for (int jj = 0; jj < kKeyTile; ++jj) {
      float part = 0.f;
#pragma unroll
      for (int i = 0; i < DQ; ++i) part = fmaf(q[i], ks[jj][i * 4 + q4], part);
      part += __shfl_xor_sync(0xffffffffu, part, 1);
      part += __shfl_xor_sync(0xffffffffu, part, 2);
      s[jj] = (jj < nv && ktok[jj] >= 0) ? part * p.scale : -INFINITY;
      tmax = fmaxf(tmax, s[jj]);
    }
    const float m_new = fmaxf(m, tmax);
    const float alpha = (m == -INFINITY) ? 0.f : expf(m - m_new);
    l *= alpha;
#pragma unroll
    for (int i = 0; i < DQ; ++i) o[i] *= alpha;
#pragma unroll
    for (int jj = 0; jj < kKeyTile; ++jj) {
      const float pj = s[jj] == -INFINITY ? 0.f : expf(s[jj] - m_new);
      l += pj;
      if (kPV) {
#pragma unroll
        for (int i = 0; i < DQ; ++i) o[i] = fmaf(pj, vs[jj][i * 4 + q4], o[i]);
      }
    }
    m = m_new;
    __syncthreads();
  }
  if (tok < 0) return;
  if (!kSparse && p.lse != nullptr && q4 == 0) p.lse[size_t(bh) * p.N + tok] = m + logf(l);
  if (!kPV) return;
  const float inv_l = 1.f / l;
  const size_t rowoff = (size_t(bh) * p.N + tok) * D;
#pragma unroll
  for (int i = 0; i < DQ; ++i) {
    const size_t off = rowoff + i * 4 + q4;
    float val = o[i] * inv_l;
    if (kEpi == kEpiAddResidual) val += p.res_in[off];
    if (kEpi == kEpiStoreResidual) {
      p.res_out[off] = p.res_in[off] - val;
    } else if (p.o != nullptr) {
      p.o[off] = val;
    }
  }
}

template <int D>
__global__ void __launch_bounds__(128) simt_colsum_kernel(const SimtColsumParams p) {
  extern __shared__ __align__(16) float dyn[];
  float* qs = dyn;              // [C][D]
  float* lse = dyn + p.C * D;   // [C]
  const int key = blockIdx.x * 128 + threadIdx.x;
  const int grow = p.row0 + blockIdx.y;
  const int bh = grow / p.G, g = grow % p.G;
  for (int e = threadIdx.x; e < p.C * D; e += blockDim.x) {
    const int i = e / D, dd = e % D;
    const int t = p.perm[size_t(bh) * p.N_pad + size_t(g) * p.C + i];
    qs[e] = (t >= 0 && t < p.N) ? p.q[(size_t(bh) * p.N + t) * D + dd] : 0.f;
  }
  for (int i = threadIdx.x; i < p.C; i += blockDim.x) {
    const int t = p.perm[size_t(bh) * p.N_pad + size_t(g) * p.C + i];
    if ((t < 0 || t >= p.N_pad) && blockIdx.x == 0) raise_status(p.status, kStatusBounds);
    lse[i] = (t >= 0 && t < p.N) ? p.lse[size_t(bh) * p.N + t] : INFINITY;
  }
  __syncthreads();
  if (key >= p.N) return;
  float k[D];
  const float* kr = p.k + (size_t(bh) * p.N + key) * D;
#pragma unroll
  for (int i = 0; i < D; ++i) k[i] = kr[i];
  float acc = 0.f;
  for (int i = 0; i < p.C; ++i) {
    float s = 0.f;
#pragma unroll
    for (int dd = 0; dd < D; ++dd) s = fmaf(qs[i * D + dd], k[dd], s);
    if (lse[i] != INFINITY) acc += expf(s * p.scale - lse[i]);
  }
  p.scores[size_t(blockIdx.y) * p.N + key] = acc;
}

template <int D, bool kSparse, int kEpi, bool kPV>
cudaError_t launch_simt(const SimtAttnParams& p, int BH, cudaStream_t s) {
  dim3 grid(kSparse ? p.G * (p.C / kRowsPerCta) : (p.N + kRowsPerCta - 1) / kRowsPerCta, BH);
  simt_attn_kernel<D, kSparse, kEpi, kPV><<<grid, 256, 0, s>>>(p);
  note_launches(1);
  return cudaGetLastError();
}

}  // namespace

cudaError_t simt_dense_attn(const SimtAttnParams& p, int BH, cudaStream_t s) {
  const bool pv = p.o != nullptr;
  if (p.d == 64) return pv ? launch_simt<64, false, kEpiPlain, true>(p, BH, s) : launch_simt<64, false, kEpiPlain, false>(p, BH, s);
  if (p.d == 128) return pv ? launch_simt<128, false, kEpiPlain, true>(p, BH, s) : launch_simt<128, false, kEpiPlain, false>(p, BH, s);
  return cudaErrorInvalidValue;
}

cudaError_t simt_sparse_attn(int epi, const SimtAttnParams& p, int BH, cudaStream_t s) {
#define MCS_SIMT_CASE(DD, EE) \
  if (p.d == DD && epi == EE) return launch_simt<DD, true, EE, true>(p, BH, s);
  MCS_SIMT_CASE(64, kEpiPlain)
  MCS_SIMT_CASE(64, kEpiAddResidual)
  MCS_SIMT_CASE(64, kEpiStoreResidual)
  MCS_SIMT_CASE(128, kEpiPlain)
  MCS_SIMT_CASE(128, kEpiAddResidual)
  MCS_SIMT_CASE(128, kEpiStoreResidual)
#undef MCS_SIMT_CASE
  return cudaErrorInvalidValue;
}

cudaError_t simt_colsum(const SimtColsumParams& p, int nrows, cudaStream_t s) {
  const int smem = (p.C * p.d + p.C) * int(sizeof(float));
  dim3 grid((p.N + 127) / 128, nrows);
  if (p.d == 64) {
    cudaError_t e = cudaFuncSetAttribute(simt_colsum_kernel<64>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    simt_colsum_kernel<64><<<grid, 128, smem, s>>>(p);
  } else if (p.d == 128) {
    cudaError_t e = cudaFuncSetAttribute(simt_colsum_kernel<128>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    simt_colsum_kernel<128><<<grid, 128, smem, s>>>(p);
  } else {
    return cudaErrorInvalidValue;
  }
  note_launches(1);
  return cudaGetLastError();
}

}  // namespace mcs
