// Pass 2 of the anchor selection on the tcgen05 tensor cores, bf16 inputs
// (sm_103a): for one query group g, the summed softmax weight of every key,
//     S_g[j] = sum over the group's real queries i of exp(scale q_i.k_j - lse_i),
// with lse from pass 1 (the dense kernel) [MC-Sparse summary: anchor two-pass
// paragraph: the extra QK pass recomputes the probabilities].
//
// Two forms. At d = 128, C = 128 one CTA takes a pair of groups (see "group
// pairs" below). Otherwise (C = 64 or d = 64) one CTA per group, 320 threads:
//   warps 0-7   two warpgroups taking alternate key tiles: warps 0-3 first gather
//               the group's query rows (through perm); per key tile a warpgroup
//               reads the transposed logits S^T = K_tile Q_g^T from tensor
//               memory: the TMEM lane is the key, so each thread sums its key's
//               exp over the group's queries with no cross-thread reduction, and
//               writes the key's score (consecutive threads, consecutive keys);
//               two warps per sub-partition hide each other's load latency;
//   warp 8      tensor-memory allocation and the single MMA-issuing thread; four
//               (C = 128) or eight (C = 64) S^T buffers let it run ahead;
//   warp 9      TMA producer: key tiles of 128 rows as tiled boxes of a 3-D
//               tensor map into a 6-stage (d = 128) ring; rows >= N read zeros.
// All waits are bounded; on a timeout the CTA flags it, lets its copies and
// MMAs land, frees tensor memory and returns.
#include "attn_tc.h"
#include "common.cuh"
#include "ptx.cuh"
#include "tc_common.cuh"
#include "tma.cuh"

namespace mcs {
namespace {

constexpr int kColThreads = 320;
constexpr int kColMmaWarp = 8, kColTmaWarp = 9;

template <int D, int CQ>
struct ColCfg {
  static constexpr int kStages = (D == 128) ? 6 : 10;  // key tiles of 128 rows
  static constexpr int kTile = (D / 64) * kRegion;
  static constexpr int kQ = 0;  // [CQ x D] (regions of 128 rows)
  static constexpr int kK = kQ + kTile;
  static constexpr int kBar = kK + kStages * kTile;
  static constexpr int kNumBuf = 512 / CQ;  // S^T buffers of CQ columns
  static constexpr int kNumBars = 1 + 2 * kStages + 2 * kNumBuf + 1;
  static constexpr int kMisc = kBar + kNumBars * 8;
  static constexpr int kLse = kMisc + 16;  // [128] fp32: -lse_i * log2(e), -inf for pads
  static constexpr int kBytes = kLse + 128 * 4;
  static constexpr int kAlloc = kBytes + 1024;
};

template <int D, int CQ>
__global__ void __launch_bounds__(kColThreads, 1)
    colsum_kernel(const __grid_constant__ CUtensorMap map_k, const TcColsumParams p) {
  using L = ColCfg<D, CQ>;
  constexpr int S = L::kStages, NB = L::kNumBuf;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(smem);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::kBar);
  uint64_t* q_full = bars;
  uint64_t* k_full = bars + 1;
  uint64_t* k_empty = k_full + S;
  uint64_t* s_full = k_empty + S;  // [NB]
  uint64_t* s_free = s_full + NB;  // [NB]
  uint64_t* drain = s_free + NB;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::kMisc);
  float* nlse = reinterpret_cast<float*>(smem + L::kLse);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int grow = p.row0 + blockIdx.x;  // global group row = bh * G + g
  const int bh = grow / p.G, g = grow % p.G;
  const int T = (p.N + 127) / 128;
  uint32_t* st = p.status;

  if (tid == 0) {
    mbar_init(q_full, 128);
    for (int s = 0; s < S; ++s) {
      mbar_init(k_full + s, 1);
      mbar_init(k_empty + s, 1);
    }
    for (int b = 0; b < NB; ++b) {
      mbar_init(s_full + b, 1);
      mbar_init(s_free + b, 128);
    }
    mbar_init(drain, 1);
    fence_mbar_init();
  }
  if (warp == kColMmaWarp) {
    tmem_alloc(tmem_slot, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp < 8) {
    // ------------------------------------------------------------ query rows, then column sums
    const int32_t* permg = p.perm + size_t(bh) * p.N_pad + size_t(g) * p.C;
    if (warp < 4) {
      constexpr int kChunks = D / 8, kRowsPerPass = 128 / kChunks;
      const int ch = tid % kChunks, r0 = tid / kChunks;
      const __nv_bfloat16* qb = p.q + size_t(bh) * p.N * D;
#pragma unroll 4
      for (int it = 0; it < CQ / kRowsPerPass; ++it) {
        const int row = it * kRowsPerPass + r0;
        int t = -1;
        if (row < p.C) {
          const int v = __ldg(permg + row);
          if (v < 0 || v >= p.N_pad) raise_status(st, kStatusBounds);
          else if (v < p.N) t = v;
        }
        cp_async16(sbase + L::kQ + sw128_off(row, ch), qb + size_t(t < 0 ? 0 : t) * D + ch * 8, t >= 0);
      }
      cp_async_commit();
      if (tid < CQ) {
        int t = -1;
        if (tid < p.C) {
          const int v = __ldg(permg + tid);
          if (v >= 0 && v < p.N) t = v;
        }
        nlse[tid] = t >= 0 ? -__ldg(p.lse + size_t(bh) * p.N + t) * kLog2e : -INFINITY;
      }
      cp_async_wait<0>();
      fence_proxy_async_smem();
      mbar_arrive(q_full);
    }
    named_bar_sync(2, 256);  // nlse visible to all column threads
    // two warpgroups take alternate key tiles (tile j uses S^T buffer j % NB)
    const int wg = warp >> 2;
    const uint32_t lane_off = uint32_t((warp & 3) * 32) << 16;
    float* out = p.scores + size_t(blockIdx.x) * p.N;
    const float sl2 = p.scale_log2;
    const uint64_t sl2x2 = f2_pack(sl2, sl2);
    bool ok = true;
    for (int j = wg; j < T; j += 2) {
      const int b = j % NB;
      if (!warp_all(mbar_wait(s_full + b, uint32_t(j / NB) & 1, st))) {
        ok = false;
        break;
      }
      tc_fence_after();
      // the key's whole S^T row in one load (one wait), then the buffer goes
      // back to the MMA thread before the exponentials
      uint32_t r[CQ];
      if constexpr (CQ == 128) {
        tmem_ld128(tmem + lane_off + b * CQ, r);
      } else {
        uint32_t (&r0)[32] = *reinterpret_cast<uint32_t(*)[32]>(&r[0]);
        uint32_t (&r1)[32] = *reinterpret_cast<uint32_t(*)[32]>(&r[32]);
        tmem_ld32(tmem + lane_off + b * CQ, r0);
        tmem_ld32(tmem + lane_off + b * CQ + 32, r1);
      }
      tc_fence_before();
      mbar_arrive(s_free + b);
      // packed pairs: one FMA for two logits, two packed partial sums (four lanes)
      uint64_t acc2[2] = {f2_pack(0.f, 0.f), f2_pack(0.f, 0.f)};
#pragma unroll
      for (int i = 0; i < CQ; i += 4) {
        const float4 nl = *reinterpret_cast<const float4*>(nlse + i);
        float x0, x1, x2, x3;
        f2_unpack(f2_fma(f2_pack(__uint_as_float(r[i]), __uint_as_float(r[i + 1])), sl2x2, f2_pack(nl.x, nl.y)), x0, x1);
        f2_unpack(f2_fma(f2_pack(__uint_as_float(r[i + 2]), __uint_as_float(r[i + 3])), sl2x2, f2_pack(nl.z, nl.w)), x2, x3);
        acc2[0] = f2_add(acc2[0], f2_pack(ex2_approx(x0), ex2_approx(x1)));
        acc2[1] = f2_add(acc2[1], f2_pack(ex2_approx(x2), ex2_approx(x3)));
      }
      const int key = j * 128 + (tid & 127);
      float a0, a1;
      f2_unpack(f2_add(acc2[0], acc2[1]), a0, a1);
      if (key < p.N) out[key] = a0 + a1;
    }
    if (!ok && tid == 0) raise_status(st, kStatusTimeout);
  } else if (warp == kColTmaWarp) {
    // ------------------------------------------------------------ TMA producer
    int armed = 0;
    if (lane == 0) {
      tma_prefetch_map(&map_k);
      for (int j = 0; j < T; ++j) {
        const int s = j % S;
        if (!mbar_wait(k_empty + s, (uint32_t(j / S) & 1) ^ 1, st)) {
          raise_status(st, kStatusTimeout);
          break;
        }
        mbar_arrive_expect_tx(k_full + s, L::kTile);
#pragma unroll
        for (int rg = 0; rg < D / 64; ++rg)
          tma_load_3d(sbase + L::kK + s * L::kTile + rg * kRegion, &map_k, rg * 64, j * 128, bh,
                      smem_u32(k_full + s));
        armed = j + 1;
      }
      // let every armed copy land before the CTA can exit
      for (int t = (armed > S ? armed - S : 0); t < armed; ++t) mbar_wait(k_full + t % S, (t / S) & 1, st);
    }
    __syncwarp();
  } else if (warp == kColMmaWarp) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t kIdesc = idesc_bf16_f32(128, CQ, 0, 0);
      bool ok = mbar_wait(q_full, 0, st);
      bool issued = false;
      for (int j = 0; ok && j < T; ++j) {
        const int s = j % S, b = j % NB;
        ok = mbar_wait(k_full + s, uint32_t(j / S) & 1, st) && mbar_wait(s_free + b, (uint32_t(j / NB) & 1) ^ 1, st);
        if (!ok) break;
        tc_fence_after();
        const uint32_t klo = desc_lo_kmajor(sbase + L::kK + s * L::kTile), qlo = desc_lo_kmajor(sbase + L::kQ);
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks)
          tc_mma_ss_lo(tmem + b * CQ, klo + kstep_kmajor(ks), qlo + kstep_kmajor(ks), kIdesc, ks > 0 ? 1u : 0u);
        tc_commit(s_full + b);
        tc_commit(k_empty + s);
        issued = true;
      }
      if (!ok) {
        raise_status(st, kStatusTimeout);
        if (issued) {
          tc_commit(drain);
          mbar_wait(drain, 0, st);
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == kColMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

template <int D, int CQ>
cudaError_t launch_colsum(const TcColsumParams& p, int nrows, cudaStream_t stream) {
  using L = ColCfg<D, CQ>;
  CUtensorMap mk;
  if (!make_tile_map(&mk, p.k, p.BH, p.N, D, 128)) return cudaErrorInvalidValue;
  auto kern = colsum_kernel<D, CQ>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, L::kAlloc);
  if (e != cudaSuccess) return e;
  kern<<<nrows, kColThreads, L::kAlloc, stream>>>(mk, p);
  note_launches(1);
  return cudaGetLastError();
}


// ------------------------------------------------------------------ group pairs
// d = 128, C = 128: one CTA per pair of groups (2i, 2i+1) of one head, so that a
// key tile's MMA covers both groups' queries at once: S^T = K_tile [Q_a Q_b]^T is
// one N = 256 MMA per 16-deep slice (half the MMA issues per group of the
// single-group kernel, whose tile period the MMA issue rate and the exponential
// unit share; measured at the 720p layer: selection 59.4 -> 50.9 ms, identical
// indices). The query operand holds 256 rows in 256-row swizzled regions
// (one per 64 columns of d). Two 256-column S^T buffers fill tensor memory.
// 576 threads:
//   warps 0-15  four consumer warpgroups: warpgroup w takes the tiles of buffer
//               w % 2 (tiles j with j % 2 == w % 2) and the columns of group w / 2
//               (0-127 group a, 128-255 group b), so each warpgroup waits every
//               phase of its buffer's barriers in order; warps 0-7 first gather
//               both groups' query rows; a thread (key) reads its 128 columns 64
//               at a time and writes the key's score for its group;
//   warp 16     tensor-memory allocation and the MMA-issuing thread;
//   warp 17     TMA producer of the key tiles (4-stage ring).
// A pair is (head, i); the launch covers the pairs that touch its group rows,
// and a row outside the launch (or past G) is masked: its queries read zeros
// and its score row is not written.
constexpr int kPairThreads = 576;
constexpr int kPairWGs = 4;
constexpr int kPairMmaWarp = 16, kPairTmaWarp = 17;

struct PairCfg {
  static constexpr int D = 128;
  static constexpr int kStages = 4;
  static constexpr int kQRegion = 256 * 128;      // 256 rows x 128 bytes
  static constexpr int kQ = 0;                    // [256 x 128] bf16, two 256-row regions
  static constexpr int kK = kQ + 2 * kQRegion;    // key tiles [128 x 128], kRegion layout
  static constexpr int kTile = 2 * kRegion;
  static constexpr int kBar = kK + kStages * kTile;
  static constexpr int kNumBars = 1 + 2 * kStages + 2 * 2 + 1;  // q_full, k ring, s buffers, drain
  static constexpr int kMisc = kBar + kNumBars * 8;
  static constexpr int kLse = kMisc + 16;         // [256] fp32: -lse * log2(e), -inf for pads/masked
  static constexpr int kBytes = kLse + 256 * 4;
  static constexpr int kAlloc = kBytes + 1024;
  static_assert(kAlloc <= 227 * 1024, "shared memory");
};

// byte offset of 16-byte chunk ch of query row r (0..255) in the 256-row operand
__device__ __forceinline__ uint32_t q256_off(int r, int ch) {
  return uint32_t((ch >> 3) * PairCfg::kQRegion + r * 128 + (((ch & 7) ^ (r & 7)) << 4));
}
// K-major k-step s (16 elements of d) of the 256-row operand, in 16-byte units
__host__ __device__ constexpr uint32_t kstep_q256(int s) {
  return uint32_t((s >> 2) * (PairCfg::kQRegion >> 4) + (s & 3) * 2);
}

__global__ void __launch_bounds__(kPairThreads, 1)
    colsum_pair_kernel(const __grid_constant__ CUtensorMap map_k, const TcColsumParams p) {
  using L = PairCfg;
  constexpr int S = L::kStages, D = L::D;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(smem);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::kBar);
  uint64_t* q_full = bars;
  uint64_t* k_full = bars + 1;
  uint64_t* k_empty = k_full + S;
  uint64_t* s_full = k_empty + S;  // [2]
  uint64_t* s_free = s_full + 2;   // [2]
  uint64_t* drain = s_free + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::kMisc);
  float* nlse = reinterpret_cast<float*>(smem + L::kLse);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  // this CTA's pair and which of its rows belong to the launch
  const int G2 = (p.G + 1) / 2;
  const int row_end = p.row0 + p.nrows;
  const int P0 = (p.row0 / p.G) * G2 + (p.row0 % p.G) / 2;
  const int P = P0 + int(blockIdx.x);
  const int bh = P / G2, ga = 2 * (P % G2);
  const int row_a = bh * p.G + ga;
  const bool va = row_a >= p.row0 && row_a < row_end;
  const bool vb = ga + 1 < p.G && row_a + 1 >= p.row0 && row_a + 1 < row_end;
  const int T = (p.N + 127) / 128;
  uint32_t* st = p.status;

  if (tid == 0) {
    mbar_init(q_full, 256);
    for (int s = 0; s < S; ++s) {
      mbar_init(k_full + s, 1);
      mbar_init(k_empty + s, 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(s_full + b, 1);
      mbar_init(s_free + b, 256);  // both warpgroups of the buffer
    }
    mbar_init(drain, 1);
    fence_mbar_init();
  }
  if (warp == kPairMmaWarp) {
    tmem_alloc(tmem_slot, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp < 4 * kPairWGs) {
    // ------------------------------------------------------------ query rows, then column sums
    if (warp < 8) {  // 256 threads: row r of the pair operand is member r % 128 of group a or b
      constexpr int kChunks = D / 8, kRowsPerPass = 256 / kChunks;
      const int ch = tid % kChunks, r0 = tid / kChunks;
      const __nv_bfloat16* qb = p.q + size_t(bh) * p.N * D;
      const int32_t* permh = p.perm + size_t(bh) * p.N_pad;
#pragma unroll 4
      for (int it = 0; it < 256 / kRowsPerPass; ++it) {
        const int row = it * kRowsPerPass + r0;
        const int gsel = row >> 7, mem = row & 127;
        int t = -1;
        if ((gsel == 0 ? va : vb) && mem < p.C) {
          const int v = __ldg(permh + size_t(ga + gsel) * p.C + mem);
          if (v < 0 || v >= p.N_pad) raise_status(st, kStatusBounds);
          else if (v < p.N) t = v;
        }
        cp_async16(sbase + L::kQ + q256_off(row, ch), qb + size_t(t < 0 ? 0 : t) * D + ch * 8, t >= 0);
      }
      cp_async_commit();
      {
        const int gsel = tid >> 7, mem = tid & 127;
        int t = -1;
        if ((gsel == 0 ? va : vb) && mem < p.C) {
          const int v = __ldg(permh + size_t(ga + gsel) * p.C + mem);
          if (v >= 0 && v < p.N) t = v;
        }
        nlse[tid] = t >= 0 ? -__ldg(p.lse + size_t(bh) * p.N + t) * kLog2e : -INFINITY;
      }
      cp_async_wait<0>();
      fence_proxy_async_smem();
      mbar_arrive(q_full);
    }
    named_bar_sync(2, 128 * kPairWGs);  // nlse visible to all column threads
    const int wg = warp >> 2, b = wg & 1, gsel = wg >> 1;
    const bool mine = gsel == 0 ? va : vb;
    const uint32_t lane_off = uint32_t((warp & 3) * 32) << 16;
    float* out = p.scores + size_t(row_a + gsel - p.row0) * p.N;  // written only when `mine`
    const float sl2 = p.scale_log2;
    const uint64_t sl2x2 = f2_pack(sl2, sl2);
    bool ok = true;
    for (int j = b; j < T; j += 2) {
      if (!warp_all(mbar_wait(s_full + b, uint32_t(j >> 1) & 1, st))) {
        ok = false;
        break;
      }
      tc_fence_after();
      uint64_t acc[2] = {f2_pack(0.f, 0.f), f2_pack(0.f, 0.f)};
      // this group's 128 columns, 32 at a time, the next chunk's load in flight
      // while the current one is exponentiated
      const uint32_t tcol = tmem + lane_off + b * 256 + gsel * 128;
      auto chunk = [&](const uint32_t (&r)[32], int col) {
#pragma unroll
        for (int i = 0; i < 32; i += 4) {
          const float4 nl = *reinterpret_cast<const float4*>(nlse + gsel * 128 + col + i);
          const uint64_t x01 = f2_fma(f2_pack(__uint_as_float(r[i]), __uint_as_float(r[i + 1])), sl2x2, f2_pack(nl.x, nl.y));
          const uint64_t x23 =
              f2_fma(f2_pack(__uint_as_float(r[i + 2]), __uint_as_float(r[i + 3])), sl2x2, f2_pack(nl.z, nl.w));
          float x0, x1, x2, x3;
          f2_unpack(x01, x0, x1);
          f2_unpack(x23, x2, x3);
          acc[0] = f2_add(acc[0], f2_pack(ex2_approx(x0), ex2_approx(x1)));
          acc[1] = f2_add(acc[1], f2_pack(ex2_approx(x2), ex2_approx(x3)));
        }
      };
      uint32_t ra[32], rb[32];
      tmem_ld32_nowait(tcol, ra);
      tmem_wait_ld32(ra);
      tmem_ld32_nowait(tcol + 32, rb);
      chunk(ra, 0);
      tmem_wait_ld32(rb);
      tmem_ld32_nowait(tcol + 64, ra);
      chunk(rb, 32);
      tmem_wait_ld32(ra);
      tmem_ld32_nowait(tcol + 96, rb);
      chunk(ra, 64);
      tmem_wait_ld32(rb);
      tc_fence_before();  // this warpgroup's part of the row is in registers
      mbar_arrive(s_free + b);
      chunk(rb, 96);
      const int key = j * 128 + (tid & 127);
      if (mine && key < p.N) {
        float a0, a1;
        f2_unpack(f2_add(acc[0], acc[1]), a0, a1);
        out[key] = a0 + a1;
      }
    }
    if (!ok && tid == 0) raise_status(st, kStatusTimeout);
  } else if (warp == kPairTmaWarp) {
    // ------------------------------------------------------------ TMA producer
    int armed = 0;
    if (lane == 0) {
      tma_prefetch_map(&map_k);
      for (int j = 0; j < T; ++j) {
        const int s = j % S;
        if (!mbar_wait(k_empty + s, (uint32_t(j / S) & 1) ^ 1, st)) {
          raise_status(st, kStatusTimeout);
          break;
        }
        mbar_arrive_expect_tx(k_full + s, L::kTile);
#pragma unroll
        for (int rg = 0; rg < D / 64; ++rg)
          tma_load_3d(sbase + L::kK + s * L::kTile + rg * kRegion, &map_k, rg * 64, j * 128, bh,
                      smem_u32(k_full + s));
        armed = j + 1;
      }
      // let every armed copy land before the CTA can exit
      for (int t = (armed > S ? armed - S : 0); t < armed; ++t) mbar_wait(k_full + t % S, (t / S) & 1, st);
    }
    __syncwarp();
  } else if (warp == kPairMmaWarp) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t kIdesc = idesc_bf16_f32(128, 256, 0, 0);
      const uint32_t qlo = desc_lo_kmajor(sbase + L::kQ);
      bool ok = mbar_wait(q_full, 0, st);
      bool issued = false;
      for (int j = 0; ok && j < T; ++j) {
        const int s = j % S, b = j & 1;
        ok = mbar_wait(k_full + s, uint32_t(j / S) & 1, st) && mbar_wait(s_free + b, (uint32_t(j >> 1) & 1) ^ 1, st);
        if (!ok) break;
        tc_fence_after();
        const uint32_t klo = desc_lo_kmajor(sbase + L::kK + s * L::kTile);
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks)
          tc_mma_ss_lo(tmem + b * 256, klo + kstep_kmajor(ks), qlo + kstep_q256(ks), kIdesc, ks > 0 ? 1u : 0u);
        tc_commit(s_full + b);
        tc_commit(k_empty + s);
        issued = true;
      }
      if (!ok) {
        raise_status(st, kStatusTimeout);
        if (issued) {
          tc_commit(drain);
          mbar_wait(drain, 0, st);
        }
      }
    }
    __syncwarp();
  }
  tc_fence_before();
  __syncthreads();
  if (warp == kPairMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

cudaError_t launch_colsum_pair(const TcColsumParams& p, int nrows, cudaStream_t stream) {
  using L = PairCfg;
  CUtensorMap mk;
  if (!make_tile_map(&mk, p.k, p.BH, p.N, L::D, 128)) return cudaErrorInvalidValue;
  cudaError_t e = cudaFuncSetAttribute(colsum_pair_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, L::kAlloc);
  if (e != cudaSuccess) return e;
  TcColsumParams q = p;
  q.nrows = nrows;
  const int G2 = (p.G + 1) / 2;
  const int last = p.row0 + nrows - 1;
  const int P0 = (p.row0 / p.G) * G2 + (p.row0 % p.G) / 2;
  const int P1 = (last / p.G) * G2 + (last % p.G) / 2;
  colsum_pair_kernel<<<P1 - P0 + 1, kPairThreads, L::kAlloc, stream>>>(mk, q);
  note_launches(1);
  return cudaGetLastError();
}
}  // namespace

cudaError_t tc_colsum(int D, int C, const TcColsumParams& p, int nrows, cudaStream_t stream) {
  if (nrows <= 0) return cudaSuccess;
  if (D == 128 && C == 128) return launch_colsum_pair(p, nrows, stream);
  if (D == 128 && C == 64) return launch_colsum<128, 64>(p, nrows, stream);
  if (D == 64 && C == 128) return launch_colsum<64, 128>(p, nrows, stream);
  if (D == 64 && C == 64) return launch_colsum<64, 64>(p, nrows, stream);
  return cudaErrorInvalidValue;
}

}  // namespace mcs
