// tcgen05 (5th-generation tensor core) attention kernels for bf16 inputs on sm_103a.
//
//  * colsum_tc_kernel: pass 2 of the anchor selection. For one query group it
//    forms the transposed logits S^T = K_tile Q_g^T (the key on the TMEM lane),
//    so each thread owns one key and sums exp(s - lse) over the group's queries
//    without cross-thread reduction [MC-Sparse summary: anchor two-pass paragraph].
//  * self-test kernels for the descriptor encodings and the TMA gathers.
//
// Warp roles of colsum_tc_kernel (288 threads): warps 0-3 column sums (thread =
// TMEM lane = key), warp 4 tensor-memory allocation and the single MMA-issuing
// thread, warps 5-8 producers (cp.async into 128-byte-swizzled shared memory).
// Every wait is bounded; on a timeout the CTA raises a status flag, drains its
// in-flight copies and MMAs, frees tensor memory and returns.
#include <cstdio>

#include "attn_tc.h"
#include "common.cuh"
#include "ptx.cuh"
#include "tc_common.cuh"
#include "tma.cuh"

namespace mcs {
namespace {

constexpr int kThreads = 288;

// ---------------------------------------------------------------- select pass 2
template <int D, int CQ>
struct ColsumSmem {
  static constexpr int kTile = (D / 64) * kRegion;
  static constexpr int kQ = 0;                 // [CQ x D] (stored with 128-row regions)
  static constexpr int kK = kQ + kTile;        // 2 stages of [128 x D]
  static constexpr int kBar = kK + 2 * kTile;
  static constexpr int kNumBars = 10;
  static constexpr int kMisc = kBar + kNumBars * 8;
  static constexpr int kLse = kMisc + 16;      // [CQ] fp32, log2 units
  static constexpr int kTok = kLse + 128 * 4;  // q tokens [128], k tokens [2][128]
  static constexpr int kBytes = kTok + 3 * 128 * 4;
  static constexpr int kAlloc = kBytes + 1024;
};

template <int D, int CQ>
__global__ void __launch_bounds__(kThreads, 1) colsum_tc_kernel(const TcColsumParams p) {
  using L = ColsumSmem<D, CQ>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(smem);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::kBar);
  uint64_t* q_full = bars + 0;
  uint64_t* k_full = bars + 1;   // [2]
  uint64_t* k_empty = bars + 3;  // [2]
  uint64_t* s_full = bars + 5;   // [2]
  uint64_t* s_free = bars + 7;   // [2]
  uint64_t* drain = bars + 9;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::kMisc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::kMisc + 4);
  float* lse2 = reinterpret_cast<float*>(smem + L::kLse);
  int32_t* q_tok = reinterpret_cast<int32_t*>(smem + L::kTok);
  int32_t* k_tok = q_tok + 128;

  constexpr uint32_t kCols = CQ <= 64 ? 128 : 256;  // two S^T buffers of CQ columns
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int grow = p.row0 + blockIdx.x;  // global group row = bh * G + g
  const int bh = grow / p.G, g = grow % p.G;
  const int T = (p.N + 127) / 128;
  uint32_t* st = p.status;

  if (tid == 0) {
    mbar_init(q_full, 128);
    for (int s = 0; s < 2; ++s) {
      mbar_init(k_full + s, 128);
      mbar_init(k_empty + s, 1);
      mbar_init(s_full + s, 1);
      mbar_init(s_free + s, 128);
    }
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 4) {
    tmem_alloc(tmem_slot, kCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp >= 5) {
    const int pt = tid - 160;
    {
      int tok = -1;
      if (pt < p.C && pt < CQ) {
        const int t = p.perm[size_t(bh) * p.N_pad + size_t(g) * p.C + pt];
        if (t < 0 || t >= p.N_pad) raise_status(st, kStatusBounds);
        else if (t < p.N) tok = t;
      }
      q_tok[pt] = tok;
      named_bar_sync(1, 128);
      const __nv_bfloat16* qb = p.q + size_t(bh) * p.N * D;
      for (int it = 0; it < D / 8; ++it) {
        const int id = it * 128 + pt, row = id / (D / 8), ch = id % (D / 8);
        if (row < CQ) {
          const int t = q_tok[row];
          cp_async16(sbase + L::kQ + sw128_off(row, ch), qb + size_t(t < 0 ? 0 : t) * D + ch * 8, t >= 0);
        }
      }
      cp_async_commit();
      cp_async_wait<0>();
      fence_proxy_async_smem();
      mbar_arrive(q_full);
    }
    const __nv_bfloat16* kb = p.k + size_t(bh) * p.N * D;
    // the leader's decision for iteration j lives in grp_stop[j & 1] (written by
    // the leader only), so a slow reader never sees the next iteration's write
    volatile int* grp_stop = abort_flag + 1;
    int j = 0;
    for (; j < T; ++j) {
      const int s = j & 1;
      const uint32_t u = uint32_t(j) >> 1;
      if (pt == 0) {
        int stop = *abort_flag;
        if (!stop && !mbar_wait(k_empty + s, (u & 1) ^ 1, st)) {
          raise_status(st, kStatusTimeout);
          *abort_flag = 1;
          stop = 1;
        }
        grp_stop[j & 1] = stop;
      }
      named_bar_sync(1, 128);
      if (grp_stop[j & 1]) break;
#pragma unroll 4
      for (int it = 0; it < D / 8; ++it) {
        const int id = it * 128 + pt, row = id / (D / 8), ch = id % (D / 8);
        const int t = j * 128 + row;
        cp_async16(sbase + L::kK + s * L::kTile + sw128_off(row, ch), kb + size_t(t < p.N ? t : 0) * D + ch * 8,
                   t < p.N);
      }
      cp_async_commit();
      if (j >= 1) {
        cp_async_wait<1>();
        fence_proxy_async_smem();
        mbar_arrive(k_full + ((j - 1) & 1));
      }
    }
    cp_async_wait<0>();
    fence_proxy_async_smem();
    if (j == T && T > 0) mbar_arrive(k_full + ((T - 1) & 1));
  } else if (warp == 4) {
    if (lane == 0) {
      constexpr uint32_t kIdesc = idesc_bf16_f32(128, CQ, 0, 0);
      bool ok = mbar_wait(q_full, 0, st);
      bool issued = false;
      for (int j = 0; ok && j < T; ++j) {
        const int s = j & 1;
        const uint32_t u = uint32_t(j) >> 1;
        ok = mbar_wait(k_full + s, u & 1, st) && mbar_wait(s_free + s, (u & 1) ^ 1, st);
        if (!ok) break;
        tc_fence_after();
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks)
          tc_mma_ss(tmem + s * CQ, desc_kmajor(sbase + L::kK + s * L::kTile, ks), desc_kmajor(sbase + L::kQ, ks),
                    kIdesc, ks > 0 ? 1u : 0u);
        tc_commit(s_full + s);
        tc_commit(k_empty + s);
        issued = true;
      }
      if (!ok) {
        raise_status(st, kStatusTimeout);
        *abort_flag = 1;
        if (issued) {
          tc_commit(drain);
          mbar_wait(drain, 0, st);
        }
      }
    }
  } else {
    // thread = key lane of the current 128-key tile
    if (tid < CQ) {
      int t = -1;
      if (tid < p.C) {
        const int v = p.perm[size_t(bh) * p.N_pad + size_t(g) * p.C + tid];
        if (v >= 0 && v < p.N) t = v;
      }
      lse2[tid] = t >= 0 ? p.lse[size_t(bh) * p.N + t] * kLog2e : INFINITY;
    }
    named_bar_sync(4, 128);
    const uint32_t lane_off = uint32_t(warp * 32) << 16;
    float* out = p.scores + size_t(blockIdx.x) * p.N;
    for (int j = 0; j < T; ++j) {
      const int b = j & 1;
      const uint32_t u = uint32_t(j) >> 1;
      if (!warp_all(mbar_wait(s_full + b, u & 1, st))) {
        raise_status(st, kStatusTimeout);
        *abort_flag = 1;
        break;
      }
      tc_fence_after();
      float acc = 0.f;
#pragma unroll
      for (int c = 0; c < CQ / 32; ++c) {
        uint32_t r[32];
        tmem_ld32(tmem + lane_off + b * CQ + c * 32, r);
#pragma unroll
        for (int i = 0; i < 32; ++i)
          acc += ex2_approx(fmaf(__uint_as_float(r[i]), p.scale_log2, -lse2[c * 32 + i]));
      }
      tc_fence_before();
      mbar_arrive(s_free + b);
      const int key = j * 128 + tid;
      if (key < p.N) out[key] = acc;
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 4) {
    tc_fence_after();
    tmem_dealloc(tmem, kCols);
  }
}

// ---------------------------------------------------------------- probe GEMM (self-test)
// D[128 x N] = A[128 x 64] * B, one MMA chain of 4 k-steps, for checking the
// descriptor encodings: mode 0: B given as [N x 64] K-major; mode 1: B given as
// [64 x N] MN-major (N contiguous), lbo/sbo of the MN-major descriptor are inputs;
// mode 2: as mode 0 but A is first written to tensor memory (bf16 pairs packed
// per 32-bit column, row r on lane r) and read from there by the MMA.
__global__ void __launch_bounds__(128, 1) tc_probe_kernel(const __nv_bfloat16* a, const __nv_bfloat16* b, float* d,
                                                          int mode, uint32_t mn_lbo, uint32_t mn_sbo,
                                                          uint32_t* status) {
  __shared__ __align__(1024) uint8_t sA[kRegion];
  __shared__ __align__(1024) uint8_t sB[2 * kRegion];
  __shared__ __align__(8) uint64_t bar;
  __shared__ uint32_t slot;
  const int tid = threadIdx.x, warp = tid >> 5;
  constexpr int N = 128;
  // A: 128 rows x 64 (K) -> one region
  for (int id = tid; id < 128 * 8; id += 128) {
    const int row = id >> 3, ch = id & 7;
    *reinterpret_cast<uint4*>(sA + sw128_off(row, ch)) = *reinterpret_cast<const uint4*>(a + row * 64 + ch * 8);
  }
  if (mode != 1) {  // B: N rows x 64 (K) -> one region
    for (int id = tid; id < N * 8; id += 128) {
      const int row = id >> 3, ch = id & 7;
      *reinterpret_cast<uint4*>(sB + sw128_off(row, ch)) = *reinterpret_cast<const uint4*>(b + row * 64 + ch * 8);
    }
  } else {  // B: 64 rows (K) x N (contiguous) -> N/64 regions, rows of 128 B
    for (int id = tid; id < 64 * (N / 8); id += 128) {
      const int row = id / (N / 8), ch = id % (N / 8);
      *reinterpret_cast<uint4*>(sB + sw128_off(row, ch)) = *reinterpret_cast<const uint4*>(b + row * N + ch * 8);
    }
  }
  fence_proxy_async_smem();
  if (tid == 0) {
    mbar_init(&bar, 1);
    fence_mbar_init();
  }
  if (warp == 0) {
    tmem_alloc(&slot, 256);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = slot;
  if (mode == 2) {  // A row `tid` -> lane `tid`, columns [128, 160): 32 packed bf16 pairs
    uint32_t r[32];
    for (int c = 0; c < 32; ++c) {
      const __nv_bfloat162 v2 = __halves2bfloat162(a[tid * 64 + 2 * c], a[tid * 64 + 2 * c + 1]);
      r[c] = *reinterpret_cast<const uint32_t*>(&v2);
    }
    tmem_st32(tmem + (uint32_t(warp * 32) << 16) + 128, r);
    tc_fence_before();
  }
  __syncthreads();
  tc_fence_after();
  if (tid == 0) {
    const uint32_t sa = smem_u32(sA), sb = smem_u32(sB);
    for (int ks = 0; ks < 4; ++ks) {
      const uint64_t da = desc_kmajor(sa, ks);
      if (mode == 2) {
        tc_mma_ts(tmem, tmem + 128 + ks * 8, desc_kmajor(sb, ks), idesc_bf16_f32(128, N, 0, 0), ks > 0 ? 1u : 0u);
        continue;
      }
      uint64_t db;
      uint32_t idesc;
      if (mode == 0) {
        db = desc_kmajor(sb, ks);
        idesc = idesc_bf16_f32(128, N, 0, 0);
      } else {
        db = smem_desc_sw128(sb + ks * 16 * 128, mn_lbo, mn_sbo);
        idesc = idesc_bf16_f32(128, N, 0, 1);
      }
      tc_mma_ss(tmem, da, db, idesc, ks > 0 ? 1u : 0u);
    }
    tc_commit(&bar);
  }
  const bool ok = mbar_wait(&bar, 0, status);
  if (!ok && tid == 0) raise_status(status, kStatusTimeout);
  __syncwarp();
  if (__all_sync(0xffffffffu, ok)) {
    tc_fence_after();
    for (int c = 0; c < N / 32; ++c) {
      uint32_t r[32];
      tmem_ld32(tmem + (uint32_t(warp * 32) << 16) + c * 32, r);
      for (int i = 0; i < 32; ++i) d[tid * N + c * 32 + i] = __uint_as_float(r[i]);
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, 256);
  }
}

// Gathers 128 rows of a bf16 [rows x 128] matrix with TMA tile::gather4 into the
// 128-byte-swizzled shared-memory layout the MMAs read, then writes them back out
// row-major (un-swizzled): out[i] = src[rows[i]] (zeros for rows out of range).
__global__ void __launch_bounds__(128, 1) tma_gather_probe_kernel(const __grid_constant__ CUtensorMap map,
                                                                  const int* rows, __nv_bfloat16* out,
                                                                  uint32_t* status) {
  __shared__ __align__(1024) uint8_t tile[2 * kRegion];
  __shared__ __align__(8) uint64_t bar;
  const int tid = threadIdx.x;
  if (tid == 0) {
    mbar_init(&bar, 1);
    fence_mbar_init();
  }
  __syncthreads();
  if (tid == 0) {
    const uint32_t b = smem_u32(&bar), t = smem_u32(tile);
    mbar_arrive_expect_tx(&bar, 2 * kRegion);
    for (int r4 = 0; r4 < 32; ++r4)
      for (int half = 0; half < 2; ++half)
        tma_gather4(t + half * kRegion + r4 * 512, &map, half * 64, rows[4 * r4], rows[4 * r4 + 1], rows[4 * r4 + 2],
                    rows[4 * r4 + 3], b);
  }
  const bool ok = mbar_wait(&bar, 0, status);
  if (!ok) {
    if (tid == 0) raise_status(status, kStatusTimeout);
    return;
  }
  for (int ch = 0; ch < 16; ++ch)
    *reinterpret_cast<uint4*>(out + tid * 128 + ch * 8) = *reinterpret_cast<const uint4*>(tile + sw128_off(tid, ch));
}

template <typename K>
cudaError_t set_smem(K kernel, int bytes) {
  return cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
}

}  // namespace

// ---------------------------------------------------------------- host launchers
template <int D, int CQ>
static cudaError_t launch_colsum(const TcColsumParams& p, int nrows, cudaStream_t stream) {
  using L = ColsumSmem<D, CQ>;
  auto kern = colsum_tc_kernel<D, CQ>;
  cudaError_t e = set_smem(kern, L::kAlloc);
  if (e != cudaSuccess) return e;
  kern<<<nrows, kThreads, L::kAlloc, stream>>>(p);
  note_launches(1);
  return cudaGetLastError();
}

cudaError_t tc_colsum(int D, int C, const TcColsumParams& p, int nrows, cudaStream_t stream) {
  if (D == 128 && C == 128) return launch_colsum<128, 128>(p, nrows, stream);
  if (D == 128 && C == 64) return launch_colsum<128, 64>(p, nrows, stream);
  if (D == 64 && C == 128) return launch_colsum<64, 128>(p, nrows, stream);
  if (D == 64 && C == 64) return launch_colsum<64, 64>(p, nrows, stream);
  return cudaErrorInvalidValue;
}

cudaError_t tma_gather_probe(const void* src, int nrows, const int* rows, void* out, uint32_t* status,
                             cudaStream_t stream) {
  CUtensorMap map;
  if (!make_gather_map(&map, src, uint64_t(nrows), 128)) return cudaErrorInvalidValue;
  tma_gather_probe_kernel<<<1, 128, 0, stream>>>(map, rows, static_cast<__nv_bfloat16*>(out), status);
  note_launches(1);
  return cudaGetLastError();
}

cudaError_t tc_probe(const void* a, const void* b, float* d, int mode, uint32_t lbo, uint32_t sbo, uint32_t* status,
                     cudaStream_t stream) {
  tc_probe_kernel<<<1, 128, 0, stream>>>(static_cast<const __nv_bfloat16*>(a), static_cast<const __nv_bfloat16*>(b),
                                         d, mode, lbo, sbo, status);
  note_launches(1);
  return cudaGetLastError();
}

}  // namespace mcs
