// Dense softmax attention with the row log-sum-exp on the tcgen05 tensor cores,
// bf16 inputs (sm_103a). Every anchor step runs it, and its LSE is pass 1 of
// the anchor selection [MC-Sparse summary: anchor two-pass paragraph; every
// anchor still runs full dense attention].
//
// One CTA owns one tile of 128 query rows (rows 128t..128t+127 of one head);
// 224 threads:
//   warp 5      TMA producer: the Q tile once, then a 3-stage ring of K and V
//               tiles of 128 keys as tiled boxes of a 3-D tensor map (rows >= N
//               of the last tile read as zeros); K runs one tile ahead of V.
//   warp 4      tensor-memory allocation and the thread issuing the S chain:
//               S_j = Q K_j^T (both operands in shared memory) into one of two
//               TMEM S buffers;
//   warp 6      the thread issuing the P V chain: O += P_j V_j with P read from
//               tensor memory (A operand) and V from shared memory (MN-major).
//               The two chains touch different tensor-memory columns and
//               separate key/value stages, so neither waits behind the other's
//               barriers (one thread issuing both, S_j then P_{j-1} V_{j-1},
//               measured 9 % slower at the 720p layer);
//   warps 0-3   softmax, one thread per query row (attn_common.cuh), then the
//               epilogue: O / l and the natural-log LSE.
// Tensor memory: S0 [0,128), S1 [128,256), O [256,256+D), P [384,448) columns.
// All waits are bounded; on a timeout the CTA flags it, lets its copies and
// MMAs land, frees tensor memory and returns.
#include "attn_common.cuh"
#include "attn_tc.h"
#include "common.cuh"
#include "ptx.cuh"
#include "tc_common.cuh"
#include "tma.cuh"

namespace mcs {
namespace {

constexpr int kDenseThreads = 224;

template <int D>
struct DenseCfg {
  static constexpr int kStages = (D == 128) ? 3 : 4;
  static constexpr int kTile = (D / 64) * kRegion;  // [128 x D] bf16
  static constexpr int kQ = 0;
  static constexpr int kK = kQ + kTile;
  static constexpr int kV = kK + kStages * kTile;
  static constexpr int kBar = kV + kStages * kTile;
  static constexpr int kNumBars = 1 + 4 * kStages + 4 + 5;
  static constexpr int kMisc = kBar + kNumBars * 8;
  static constexpr int kBytes = kMisc + 16;
  static constexpr int kAlloc = kBytes + 1024;
  static constexpr uint32_t kColS = 0, kColO = 256, kColP = 384;
};

template <int D, bool kPV>
__global__ void __launch_bounds__(kDenseThreads, 1)
    attn_dense_kernel(const __grid_constant__ CUtensorMap map_q, const __grid_constant__ CUtensorMap map_k,
                      const __grid_constant__ CUtensorMap map_v, const TcAttnParams p) {
  using L = DenseCfg<D>;
  constexpr int S = L::kStages;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(smem);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::kBar);
  uint64_t* q_full = bars;
  uint64_t* k_full = bars + 1;
  uint64_t* k_empty = k_full + S;
  uint64_t* v_full = k_empty + S;
  uint64_t* v_empty = v_full + S;
  uint64_t* s_full = v_empty + S;  // [2]
  uint64_t* s_free = s_full + 2;   // [2]
  uint64_t* p_full = s_free + 2;
  uint64_t* p_empty = p_full + 1;
  uint64_t* o_done = p_empty + 1;
  uint64_t* drain = o_done + 1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::kMisc);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int bh = blockIdx.y, tile = blockIdx.x;
  const int T = (p.N + 127) / 128;
  uint32_t* st = p.status;

  if (tid == 0) {
    mbar_init(q_full, 1);
    for (int s = 0; s < S; ++s) {
      mbar_init(k_full + s, 1);
      mbar_init(k_empty + s, 1);
      mbar_init(v_full + s, 1);
      mbar_init(v_empty + s, 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(s_full + b, 1);
      mbar_init(s_free + b, 128);
    }
    mbar_init(p_full, 128);
    mbar_init(p_empty, 1);
    mbar_init(o_done, 2);
    mbar_init(drain, 1);
    mbar_init(drain + 1, 1);
    fence_mbar_init();
  }
  if (warp == 4) {
    tmem_alloc(tmem_slot, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const uint32_t tS = tmem + L::kColS, tO = tmem + L::kColO, tP = tmem + L::kColP;

  if (warp == 5) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      tma_prefetch_map(&map_q);
      tma_prefetch_map(&map_k);
      if (kPV) tma_prefetch_map(&map_v);
      mbar_arrive_expect_tx(q_full, L::kTile);
#pragma unroll
      for (int rg = 0; rg < D / 64; ++rg)
        tma_load_3d(sbase + L::kQ + rg * kRegion, &map_q, rg * 64, tile * 128, bh, smem_u32(q_full));
    }
    int k_armed = 0, v_armed = 0;
    bool ok = true;
    for (int i = 0; i <= T && ok; ++i) {
      if (i < T) {
        const int s = i % S;
        const uint32_t u = uint32_t(i / S);
        bool w = true;
        if (lane == 0) w = mbar_wait(k_empty + s, (u & 1) ^ 1, st);
        ok = __shfl_sync(0xffffffffu, w, 0);
        if (!ok) break;
        if (lane == 0) {
          mbar_arrive_expect_tx(k_full + s, L::kTile);
#pragma unroll
          for (int rg = 0; rg < D / 64; ++rg)
            tma_load_3d(sbase + L::kK + s * L::kTile + rg * kRegion, &map_k, rg * 64, i * 128, bh,
                        smem_u32(k_full + s));
        }
        k_armed = i + 1;
      }
      if (kPV && i >= 1) {
        const int j = i - 1, s = j % S;
        const uint32_t u = uint32_t(j / S);
        bool w = true;
        if (lane == 0) w = mbar_wait(v_empty + s, (u & 1) ^ 1, st);
        ok = __shfl_sync(0xffffffffu, w, 0);
        if (!ok) break;
        if (lane == 0) {
          mbar_arrive_expect_tx(v_full + s, L::kTile);
#pragma unroll
          for (int rg = 0; rg < D / 64; ++rg)
            tma_load_3d(sbase + L::kV + s * L::kTile + rg * kRegion, &map_v, rg * 64, j * 128, bh,
                        smem_u32(v_full + s));
        }
        v_armed = j + 1;
      }
    }
    if (!ok && lane == 0) raise_status(st, kStatusTimeout);
    // let every armed copy land before the CTA can exit (normally already done)
    if (lane == 0) {
      mbar_wait(q_full, 0, st);
      for (int t = (k_armed > S ? k_armed - S : 0); t < k_armed; ++t) mbar_wait(k_full + t % S, (t / S) & 1, st);
      for (int t = (v_armed > S ? v_armed - S : 0); t < v_armed; ++t) mbar_wait(v_full + t % S, (t / S) & 1, st);
    }
    __syncwarp();
  } else if (warp == 4 || warp == 6) {
    // ------------------------------------------------------------ MMA issuers
    // lane 0 of warp 4 issues the S_j = Q K_j^T chain, lane 0 of warp 6 the
    // O += P_j V_j chain: the two touch different tensor-memory columns and
    // separate key/value stages, so neither waits behind the other's barriers
    if (lane == 0) {
      const bool pv_thread = warp == 6;
      constexpr uint32_t kIdescQK = idesc_bf16_f32(128, 128, 0, 0);
      constexpr uint32_t kIdescPV = idesc_bf16_f32(128, D, 0, 1);
      bool ok = mbar_wait(q_full, 0, st);
      bool issued = false;
      auto issue_pv = [&](int i) -> bool {
        const int s = i % S;
        const uint32_t u = uint32_t(i / S);
        if (!mbar_wait(v_full + s, u & 1, st)) return false;
        if (!mbar_wait(p_full, uint32_t(i) & 1, st)) return false;
        tc_fence_after();
        const uint32_t vlo = desc_lo_mnmajor(sbase + L::kV + s * L::kTile);
#pragma unroll
        for (int ks = 0; ks < 8; ++ks)
          tc_mma_ts_lo(tO, tP + ks * 8, vlo + kstep_mnmajor(ks), kIdescPV, (i > 0 || ks > 0) ? 1u : 0u);
        tc_commit(p_empty);
        tc_commit(v_empty + s);
        return true;
      };
      if (!pv_thread) {
        for (int j = 0; ok && j < T; ++j) {
          const int s = j % S, b = j & 1;
          const uint32_t u = uint32_t(j / S), ub = uint32_t(j >> 1);
          ok = mbar_wait(k_full + s, u & 1, st) && mbar_wait(s_free + b, (ub & 1) ^ 1, st);
          if (!ok) break;
          tc_fence_after();
          const uint32_t klo = desc_lo_kmajor(sbase + L::kK + s * L::kTile), qlo = desc_lo_kmajor(sbase + L::kQ);
#pragma unroll
          for (int ks = 0; ks < D / 16; ++ks)
            tc_mma_ss_lo(tS + b * 128, qlo + kstep_kmajor(ks), klo + kstep_kmajor(ks), kIdescQK, ks > 0 ? 1u : 0u);
          tc_commit(s_full + b);
          tc_commit(k_empty + s);
          issued = true;
        }
      } else if (kPV) {
        for (int j = 0; ok && j < T; ++j) {
          ok = issue_pv(j);
          issued = issued || ok;
        }
      }
      // o_done expects one commit from each issuing thread
      if (ok) tc_commit(o_done);
      if (!ok) {
        raise_status(st, kStatusTimeout);
        if (issued) {
          tc_commit(drain + (pv_thread ? 1 : 0));
          mbar_wait(drain + (pv_thread ? 1 : 0), 0, st);
        }
      }
    }
  } else {
    // ------------------------------------------------------------ softmax + epilogue
    const int row = tid;
    const uint32_t lane_off = uint32_t(warp * 32) << 16;
    float m, l;
    const SoftmaxSync sy{s_full, s_free, p_full, p_empty};
    bool ok = softmax_rows<D, kPV>(T, p.N, tS, tO, tP, lane_off, p.scale_log2, sy, st, m, l);
    const int t = tile * 128 + row;
    const int tok = t < p.N ? t : -1;
    if (ok && p.lse != nullptr && tok >= 0) p.lse[size_t(bh) * p.N + tok] = (m + __log2f(l)) * kLn2;
    if constexpr (kPV) {
      if (ok) ok = warp_all(mbar_wait(o_done, 0, st));
      if (ok) {
        tc_fence_after();
        store_row<D, kEpiPlain>(tO, lane_off, tok, (size_t(bh) * p.N + size_t(tok < 0 ? 0 : tok)) * D, 1.f / l, p.o,
                                nullptr);
      }
    }
    if (!ok && row == 0) raise_status(st, kStatusTimeout);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 4) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

template <int D, bool kPV>
cudaError_t launch_dense(const TcAttnParams& p, cudaStream_t stream) {
  using L = DenseCfg<D>;
  CUtensorMap mq, mk, mv;
  if (!(make_tile_map(&mq, p.q, p.BH, p.N, D, 128) && make_tile_map(&mk, p.k, p.BH, p.N, D, 128) &&
        make_tile_map(&mv, p.v, p.BH, p.N, D, 128)))
    return cudaErrorInvalidValue;
  auto kern = attn_dense_kernel<D, kPV>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, L::kAlloc);
  if (e != cudaSuccess) return e;
  dim3 grid(p.tiles_per_head, p.BH);
  kern<<<grid, kDenseThreads, L::kAlloc, stream>>>(mq, mk, mv, p);
  note_launches(1);
  return cudaGetLastError();
}

}  // namespace

cudaError_t tc_dense_attn(int D, const TcAttnParams& p, int BH, bool with_pv, cudaStream_t stream) {
  (void)BH;
  if (D == 128) return with_pv ? launch_dense<128, true>(p, stream) : launch_dense<128, false>(p, stream);
  if (D == 64) return with_pv ? launch_dense<64, true>(p, stream) : launch_dense<64, false>(p, stream);
  return cudaErrorInvalidValue;
}

}  // namespace mcs
