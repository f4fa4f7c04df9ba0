// Softmax attention on the tcgen05 tensor cores for bf16 inputs (sm_103a):
// dense attention with the row log-sum-exp, and the token-gather sparse
// attention of one query group over its K selected keys, whose key/value rows
// are fetched through the group's index list rather than repacked into blocks
// [MC-Sparse summary: index-gather / PDDP paragraph; residual paragraph].
//
// One CTA owns one tile of 128 query rows (dense: rows 128t..128t+127; sparse:
// the C members of group t, read through perm). K and V arrive in a 3-stage
// ring of tiles of 128 keys:
//   dense:  warp 5 is a TMA producer loading tiled boxes (Q once, then K_i ahead
//           of V_{i-1}); no thread waits on a copy.
//   sparse: warps 4-11 gather the rows with 16-byte cp.async copies at the group's
//           key indices (streamed through a shared-memory index ring) and signal
//           each tile two tiles after issuing it. Row gathers of 128-byte
//           segments are kept on the load/store path: on this GPU they move far
//           more bytes per cycle than 4-row TMA gathers.
//   warp 4      tensor-memory allocation and the single MMA-issuing thread:
//               S_j = Q K_j^T into one of two TMEM S buffers, then O += P_{j-1} V_{j-1}
//               with P read from tensor memory (A operand) and V from shared memory.
//   warps 0-3   softmax, one thread per query row (= TMEM lane): online base-2
//               softmax with a lazily rescaled running max (O is rescaled only when
//               the max grows by more than 2^8), P written to TMEM as bf16 pairs;
//               then the epilogue (O / l, optional residual add or residual store).
// Tensor memory: S0 [0,128), S1 [128,256), O [256,256+D), P [384,448) columns.
// All waits are bounded; on a timeout the CTA flags it, lets its copies and
// MMAs land, frees tensor memory and returns.
#include "attn_tc.h"
#include "common.cuh"
#include "ptx.cuh"
#include "tc_common.cuh"
#include "tma.cuh"

namespace mcs {
namespace {

// dense (192 threads): warps 0-3 softmax, warp 4 MMA, warp 5 TMA producer.
// sparse (512 threads, four warpgroups): warpgroup 0 softmax, warpgroups 1-2
// eight cp.async gather warps, warpgroup 3 the MMA warp (warp 12) and three idle
// warps. Row gathers need many warps in flight, so the registers are rebalanced
// with setmaxnreg: softmax up, gather and MMA down. The split below must fit in
// the 512 x (launch registers) the block starts with, which the launcher checks.
template <bool kSparse>
__host__ __device__ constexpr int fwd_threads() { return kSparse ? 512 : 192; }
constexpr int kGatherThreads = 256;
constexpr int kRegSoftmax = 224, kRegGather = 80, kRegMma = 64;
constexpr int kRegPool = 128 * kRegSoftmax + 256 * kRegGather + 128 * kRegMma;
template <bool kSparse>
__host__ __device__ constexpr int mma_warp() { return kSparse ? 12 : 4; }

template <int D>
struct FwdCfg {
  static constexpr int kStages = (D == 128) ? 3 : 4;
  static constexpr int kTile = (D / 64) * kRegion;  // [128 x D] bf16
  static constexpr int kQ = 0;
  static constexpr int kK = kQ + kTile;
  static constexpr int kV = kK + kStages * kTile;
  static constexpr int kBar = kV + kStages * kTile;
  static constexpr int kNumBars = 1 + 4 * kStages + 4 + 4;
  static constexpr int kMisc = kBar + kNumBars * 8;
  static constexpr int kIdxSlots = 3;              // sparse: index chunks of 128 keys in flight
  static constexpr int kIdx = kMisc + 16;
  static constexpr int kBytes = kIdx + kIdxSlots * 128 * 4;
  static constexpr int kAlloc = kBytes + 1024;
  static constexpr uint32_t kColS = 0, kColO = 256, kColP = 384;
};

template <int D, bool kSparse, int kEpi, bool kPV>
__global__ void __launch_bounds__(fwd_threads<kSparse>(), 1)
    attn_fwd_kernel(const __grid_constant__ CUtensorMap map_q, const __grid_constant__ CUtensorMap map_k,
                    const __grid_constant__ CUtensorMap map_v, const TcAttnParams p) {
  using L = FwdCfg<D>;
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
  const int nkv = kSparse ? p.K : p.N;
  const int T = (nkv + 127) / 128;
  uint32_t* st = p.status;

  if (tid == 0) {
    const uint32_t fill = kSparse ? kGatherThreads : 1;  // sparse: every gather thread arrives; dense: one TMA arm
    mbar_init(q_full, fill);
    for (int s = 0; s < S; ++s) {
      mbar_init(k_full + s, fill);
      mbar_init(k_empty + s, 1);
      mbar_init(v_full + s, fill);
      mbar_init(v_empty + s, 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(s_full + b, 1);
      mbar_init(s_free + b, 128);
    }
    mbar_init(p_full, 128);
    mbar_init(p_empty, 1);
    mbar_init(o_done, 1);
    mbar_init(drain, 1);
    fence_mbar_init();
  }
  if (warp == mma_warp<kSparse>()) {
    tmem_alloc(tmem_slot, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const uint32_t tS = tmem + L::kColS, tO = tmem + L::kColO, tP = tmem + L::kColP;

  // Registers move between warpgroups with setmaxnreg (sparse only): each
  // warpgroup executes its own instruction at the top of its role branch, so the
  // role code is dominated by its register budget.
  const bool producer = kSparse ? (warp >= 4 && warp < 12) : (warp == 5);
  if (producer) {
    if constexpr (kSparse) asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kRegGather));
    if constexpr (!kSparse) {
      // ---------------------------------------------------------- dense: one TMA producer warp
      if (lane == 0) {
        tma_prefetch_map(&map_q);
        tma_prefetch_map(&map_k);
        if (kPV) tma_prefetch_map(&map_v);
        mbar_arrive_expect_tx(q_full, L::kTile);
#pragma unroll
        for (int rg = 0; rg < D / 64; ++rg)
          tma_load_3d(sbase + L::kQ + rg * kRegion, &map_q, rg * 64, tile * 128, bh, smem_u32(q_full));
      }
      // K_i then V_{i-1}: K runs one tile ahead of V, as the MMA order needs.
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
      // Let every armed copy land before the CTA can exit (normally already done).
      if (lane == 0) {
        mbar_wait(q_full, 0, st);
        for (int t = (k_armed > S ? k_armed - S : 0); t < k_armed; ++t) mbar_wait(k_full + t % S, (t / S) & 1, st);
        for (int t = (v_armed > S ? v_armed - S : 0); t < v_armed; ++t) mbar_wait(v_full + t % S, (t / S) & 1, st);
      }
      __syncwarp();
    } else {
      // ---------------------------------------------------------- sparse: eight cp.async gather warps
      // Each thread copies 16-byte chunks of gathered rows into the swizzled
      // stage (a warp instruction covers whole 128-byte row segments). Per tile
      // j one cp.async group holds K_j, V_j and the index chunk of tile j+kLag;
      // group j is retired (waited, proxy-fenced, arrived on the full barriers)
      // kLag iterations later, so the row loads of kLag tiles are in flight.
      constexpr int kLag = L::kIdxSlots - 1;
      constexpr int kChunks = D / 8;               // 16-byte chunks per row
      constexpr int kRowsPerIt = kGatherThreads / kChunks;  // rows covered by one pass of the gather threads
      constexpr int kPasses = 128 / kRowsPerIt;
      const int pt = tid - 128;  // 0..255
      const int ch = pt % kChunks, r0 = pt / kChunks;
      int32_t* ring = reinterpret_cast<int32_t*>(smem + L::kIdx);  // [kIdxSlots][128]
      // decision of the leader for iteration j lives in stop[j & 1], so a slow
      // reader of iteration j never sees the leader's write for iteration j + 1
      volatile int* stop = reinterpret_cast<volatile int*>(smem + L::kMisc + 4);
      const int32_t* idxg = p.idx + (size_t(bh) * p.G + tile) * size_t(p.K);
      const int32_t* permg = p.perm + size_t(bh) * p.N_pad + size_t(tile) * p.C;
      const __nv_bfloat16* qb = p.q + size_t(bh) * p.N * D;
      const __nv_bfloat16* kb = p.k + size_t(bh) * p.N * D;
      const __nv_bfloat16* vb = p.v + size_t(bh) * p.N * D;
      // group 0: the Q rows of the group (through perm) and index chunks of tiles 0..kLag-1
#pragma unroll 4
      for (int it = 0; it < kPasses; ++it) {
        const int row = it * kRowsPerIt + r0;
        int t = -1;
        if (row < p.C) {
          const int v = __ldg(permg + row);
          if (v < 0 || v >= p.N_pad) raise_status(st, kStatusBounds);
          else if (v < p.N) t = v;
        }
        cp_async16(sbase + L::kQ + sw128_off(row, ch), qb + size_t(t < 0 ? 0 : t) * D + ch * 8, t >= 0);
      }
#pragma unroll
      for (int tt = 0; tt < kLag; ++tt)
        for (int e = pt; e < 128; e += kGatherThreads) {
          const int slot = tt * 128 + e;
          cp_async4(smem_u32(ring + tt * 128 + e), idxg + (slot < nkv ? slot : 0), slot < nkv);
        }
      cp_async_commit();
      cp_async_wait<0>();
      fence_proxy_async_smem();
      mbar_arrive(q_full);
      bool ok = true;
      int issued = 0;
      for (int j = 0; j < T; ++j) {
        const int s = j % S;
        if (j >= kLag) {  // retire tile j - kLag (also completes the index chunk of tile j)
          cp_async_wait<kLag - 1>();
          fence_proxy_async_smem();
          mbar_arrive(k_full + (j - kLag) % S);
          mbar_arrive(v_full + (j - kLag) % S);
        }
        if (pt == 0) {
          int stp = 0;
          if (!mbar_wait(v_empty + s, ((j / S) & 1) ^ 1, st)) {  // PV of tile j - S done: stage free
            raise_status(st, kStatusTimeout);
            stp = 1;
          }
          stop[j & 1] = stp;
        }
        named_bar_sync(1, kGatherThreads);
        if (stop[j & 1]) {
          ok = false;
          break;
        }
        const int32_t* rt = ring + (j % L::kIdxSlots) * 128;
        const uint32_t dk = sbase + L::kK + s * L::kTile, dv = sbase + L::kV + s * L::kTile;
        // all of this thread's row indices first, then the copies back to back: a
        // load between two copies would serialise the warp on its latency
        int toks[kPasses];
#pragma unroll
        for (int it = 0; it < kPasses; ++it) {
          const int row = it * kRowsPerIt + r0;
          toks[it] = (j * 128 + row < nkv) ? rt[row] : -1;
        }
#pragma unroll
        for (int it = 0; it < kPasses; ++it) {
          const int row = it * kRowsPerIt + r0;
          int t = toks[it];
          if (t >= p.N || (t < 0 && j * 128 + row < nkv)) {
            raise_status(st, kStatusBounds);
            t = -1;
          }
          const size_t off = size_t(t < 0 ? 0 : t) * D + ch * 8;
          cp_async16(dk + sw128_off(row, ch), kb + off, t >= 0);
          cp_async16(dv + sw128_off(row, ch), vb + off, t >= 0);
        }
        for (int e = pt; e < 128; e += kGatherThreads) {
          const int tn = j + kLag, slot = tn * 128 + e;
          cp_async4(smem_u32(ring + (tn % L::kIdxSlots) * 128 + e), idxg + (slot < nkv ? slot : 0), slot < nkv);
        }
        cp_async_commit();
        issued = j + 1;
      }
      cp_async_wait<0>();
      fence_proxy_async_smem();
      if (ok) {
        for (int t = (issued > kLag ? issued - kLag : 0); t < issued; ++t) {
          mbar_arrive(k_full + t % S);
          mbar_arrive(v_full + t % S);
        }
      }
    }
  } else if (warp < 4) {
    if constexpr (kSparse) asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kRegSoftmax));
    // ------------------------------------------------------------ softmax (thread = query row)
    const int row = tid;
    const uint32_t lane_off = uint32_t(warp * 32) << 16;
    const float sl2 = p.scale_log2;
    float m = -INFINITY, l = 0.f;
    bool ok = true;
    for (int j = 0; j < T; ++j) {
      const int b = j & 1;
      const uint32_t ub = uint32_t(j >> 1);
      ok = warp_all(mbar_wait(s_full + b, ub & 1, st));
      if (!ok) break;
      tc_fence_after();
      uint32_t r[128];
      tmem_ld128(tS + lane_off + b * 128, r);
      tc_fence_before();
      mbar_arrive(s_free + b);
      const int nvalid = min(128, nkv - j * 128);
      float mx = -INFINITY;
#pragma unroll
      for (int c = 0; c < 128; ++c) mx = fmaxf(mx, c < nvalid ? __uint_as_float(r[c]) : -INFINITY);
      const float m_new = fmaxf(m, mx * sl2);
      const bool need = m_new > m + 8.f;  // keep a stale max unless it grew by more than 2^8
      const float m_use = need ? m_new : m;
      const float alpha = need ? ex2_approx(m - m_new) : 1.f;
      const float neg_m = -m_use;
      float lsum = 0.f;
      uint32_t pk[64];
#pragma unroll
      for (int c = 0; c < 64; ++c) {
        const float p0 = (2 * c < nvalid) ? ex2_approx(fmaf(__uint_as_float(r[2 * c]), sl2, neg_m)) : 0.f;
        const float p1 = (2 * c + 1 < nvalid) ? ex2_approx(fmaf(__uint_as_float(r[2 * c + 1]), sl2, neg_m)) : 0.f;
        lsum += p0 + p1;
        pk[c] = pack_bf16x2(p0, p1);
      }
      l = l * alpha + lsum;
      m = m_use;
      if constexpr (kPV) {
        ok = warp_all(mbar_wait(p_empty, (uint32_t(j) & 1) ^ 1, st));  // PV of tile j-1 done
        if (!ok) break;
        tc_fence_after();
        if (__any_sync(0xffffffffu, need && j > 0)) {
#pragma unroll
          for (int c = 0; c < D / 32; ++c) {
            uint32_t o[32];
            tmem_ld32(tO + lane_off + c * 32, o);
#pragma unroll
            for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha);
            tmem_st32(tO + lane_off + c * 32, o);
          }
        }
        tmem_st64(tP + lane_off, pk);
        tc_fence_before();
        mbar_arrive(p_full);
      }
    }
    // ------------------------------------------------------------ epilogue
    int tok = -1;
    if constexpr (kSparse) {
      if (row < p.C) {
        const int t = p.perm[size_t(bh) * p.N_pad + size_t(tile) * p.C + row];
        if (t >= 0 && t < p.N) tok = t;
      }
    } else {
      const int t = tile * 128 + row;
      if (t < p.N) tok = t;
    }
    if (ok && !kSparse && p.lse != nullptr && tok >= 0) p.lse[size_t(bh) * p.N + tok] = (m + __log2f(l)) * kLn2;
    if constexpr (kPV) {
      if (ok) ok = warp_all(mbar_wait(o_done, 0, st));
      if (ok) {
        tc_fence_after();
        const float inv_l = 1.f / l;
        const size_t rowoff = (size_t(bh) * p.N + size_t(tok < 0 ? 0 : tok)) * D;
        __nv_bfloat16* dst = (kEpi == kEpiStoreResidual) ? p.res_out : p.o;
#pragma unroll
        for (int c = 0; c < D / 32; ++c) {
          uint32_t o[32];
          tmem_ld32(tO + lane_off + c * 32, o);
          if (tok >= 0 && dst != nullptr) {
#pragma unroll
            for (int q4 = 0; q4 < 4; ++q4) {
              float o8[8];
#pragma unroll
              for (int i = 0; i < 8; ++i) o8[i] = __uint_as_float(o[q4 * 8 + i]) * inv_l;
              const size_t off = rowoff + c * 32 + q4 * 8;
              if constexpr (kEpi != kEpiPlain) {
                const uint4 rv = *reinterpret_cast<const uint4*>(p.res_in + off);
                const __nv_bfloat16* rb = reinterpret_cast<const __nv_bfloat16*>(&rv);
#pragma unroll
                for (int i = 0; i < 8; ++i)
                  o8[i] = (kEpi == kEpiAddResidual) ? o8[i] + __bfloat162float(rb[i]) : __bfloat162float(rb[i]) - o8[i];
              }
              uint4 w;
              w.x = pack_bf16x2(o8[0], o8[1]);
              w.y = pack_bf16x2(o8[2], o8[3]);
              w.z = pack_bf16x2(o8[4], o8[5]);
              w.w = pack_bf16x2(o8[6], o8[7]);
              *reinterpret_cast<uint4*>(dst + off) = w;
            }
          }
        }
      }
    }
    if (!ok && row == 0) raise_status(st, kStatusTimeout);
  } else {
    // dense: warp 4; sparse: warpgroup 3 (warp 12 issues, warps 13-15 idle)
    if constexpr (kSparse) asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kRegMma));
    if (warp == mma_warp<kSparse>()) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
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
        const uint32_t vb = sbase + L::kV + s * L::kTile;
#pragma unroll
        for (int ks = 0; ks < 8; ++ks)
          tc_mma_ts(tO, tP + ks * 8, desc_mnmajor(vb, ks), kIdescPV, (i > 0 || ks > 0) ? 1u : 0u);
        tc_commit(p_empty);
        tc_commit(v_empty + s);
        return true;
      };
      for (int j = 0; ok && j < T; ++j) {
        const int s = j % S, b = j & 1;
        const uint32_t u = uint32_t(j / S), ub = uint32_t(j >> 1);
        ok = mbar_wait(k_full + s, u & 1, st) && mbar_wait(s_free + b, (ub & 1) ^ 1, st);
        if (!ok) break;
        tc_fence_after();
        const uint32_t kb = sbase + L::kK + s * L::kTile;
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks)
          tc_mma_ss(tS + b * 128, desc_kmajor(sbase + L::kQ, ks), desc_kmajor(kb, ks), kIdescQK, ks > 0 ? 1u : 0u);
        tc_commit(s_full + b);
        tc_commit(k_empty + s);
        issued = true;
        if (kPV && j >= 1) ok = issue_pv(j - 1);
      }
      if (ok && kPV && T > 0) ok = issue_pv(T - 1);
      if (ok) tc_commit(o_done);
      if (!ok) {
        raise_status(st, kStatusTimeout);
        if (issued) {
          tc_commit(drain);
          mbar_wait(drain, 0, st);
        }
      }
    }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == mma_warp<kSparse>()) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

template <int D, bool kSparse, int kEpi, bool kPV>
cudaError_t launch_fwd(const TcAttnParams& p, cudaStream_t stream) {
  using L = FwdCfg<D>;
  CUtensorMap mq, mk, mv;
  const uint64_t rows = uint64_t(p.BH) * p.N;
  bool ok;
  if (kSparse) {  // rows are gathered with cp.async; the maps are unused placeholders
    ok = make_gather_map(&mq, p.q, rows, D);
    mk = mq;
    mv = mq;
  } else {
    ok = make_tile_map(&mq, p.q, p.BH, p.N, D, 128) && make_tile_map(&mk, p.k, p.BH, p.N, D, 128) &&
         make_tile_map(&mv, p.v, p.BH, p.N, D, 128);
  }
  if (!ok) return cudaErrorInvalidValue;
  auto kern = attn_fwd_kernel<D, kSparse, kEpi, kPV>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, L::kAlloc);
  if (e != cudaSuccess) return e;
  if (kSparse) {
    // setmaxnreg.inc waits for registers released by the other warpgroups: never
    // launch unless the rebalanced split fits in what the block is launched with
    cudaFuncAttributes fa;
    if ((e = cudaFuncGetAttributes(&fa, kern)) != cudaSuccess) return e;
    if (fa.numRegs * fwd_threads<kSparse>() < kRegPool || fa.numRegs < kRegGather) return cudaErrorInvalidValue;
  }
  dim3 grid(p.tiles_per_head, p.BH);
  kern<<<grid, fwd_threads<kSparse>(), L::kAlloc, stream>>>(mq, mk, mv, p);
  note_launches(1);
  return cudaGetLastError();
}

}  // namespace

cudaError_t tc_dense_attn(int D, const TcAttnParams& p, int BH, bool with_pv, cudaStream_t stream) {
  (void)BH;
  if (D == 128) return with_pv ? launch_fwd<128, false, kEpiPlain, true>(p, stream)
                               : launch_fwd<128, false, kEpiPlain, false>(p, stream);
  if (D == 64) return with_pv ? launch_fwd<64, false, kEpiPlain, true>(p, stream)
                              : launch_fwd<64, false, kEpiPlain, false>(p, stream);
  return cudaErrorInvalidValue;
}

cudaError_t tc_sparse_attn(int D, int epi, const TcAttnParams& p, int BH, cudaStream_t stream) {
  (void)BH;
#define MCS_SPARSE_CASE(DD, EE) \
  if (D == DD && epi == EE) return launch_fwd<DD, true, EE, true>(p, stream);
  MCS_SPARSE_CASE(128, kEpiPlain)
  MCS_SPARSE_CASE(128, kEpiAddResidual)
  MCS_SPARSE_CASE(128, kEpiStoreResidual)
  MCS_SPARSE_CASE(64, kEpiPlain)
  MCS_SPARSE_CASE(64, kEpiAddResidual)
  MCS_SPARSE_CASE(64, kEpiStoreResidual)
#undef MCS_SPARSE_CASE
  return cudaErrorInvalidValue;
}

}  // namespace mcs
