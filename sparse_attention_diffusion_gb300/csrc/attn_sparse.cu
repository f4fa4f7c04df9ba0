// Token-gather sparse attention on the tcgen05 tensor cores, bf16 inputs
// (sm_103a): for one query group (the C members of group g, read through perm),
// softmax attention over the group's own K selected keys, whose key and value
// rows are fetched at the group's index list rather than repacked into blocks
// [MC-Sparse summary: index-gather / PDDP paragraph]. Epilogues add the cached
// residual (reuse step) or store R = O_dense - O_sparse (anchor step)
// [MC-Sparse summary: residual paragraph].
//
// One CTA per group, 512 threads in four warpgroups:
//   warpgroup 0 (warps 0-3)   softmax, one thread per query row, and the epilogue;
//   warpgroups 1-2 (4-11)     eight gather warps: the group's query rows (through
//                             perm) once, then per iteration i the key rows of
//                             tile i and the value rows of tile i-1 (128 keys per
//                             tile) at the group's index list, as 16-byte cp.async
//                             copies into a 3-stage K ring and a 3-stage V ring
//                             (128-byte swizzled); the index list streams through
//                             a shared-memory ring two tiles ahead;
//   warpgroup 3 (warp 12)     tensor-memory allocation and the single
//                             MMA-issuing thread (warps 13-15 idle).
// A K stage is released when S of its tile is done, a V stage when PV is done,
// so key rows are fetched well ahead of their use; iteration i's copies form one
// cp.async group, retired (waited, proxy-fenced, arrived on the full barriers)
// two iterations later. Each gather thread reads its row indices into registers
// before issuing its copies back to back (a load between two copies would
// serialise the warp on its latency) and keeps them for the value rows of the
// same tile one iteration later. The MMA thread issues P_j V_j as soon as P_j is
// written and only puts S_{j+1} first when its key rows have already landed.
// Row gathers of 128-byte segments are kept on the load/store path: on this GPU
// they move far more bytes per cycle than 4-row TMA gathers, and their
// throughput grows with the number of issuing warps. Registers are rebalanced
// with setmaxnreg (softmax 224, gather 80, MMA 64); the launcher checks that the
// split fits the registers the block is launched with.
// S = Q K^T reads both operands from shared memory; PV reads P from tensor memory.
// Tensor memory: S0 [0,128), S1 [128,256), O [256,256+D), P [384,448).
// All waits are bounded; on a timeout the CTA flags it, lets its copies and
// MMAs land, frees tensor memory and returns.
#include "attn_common.cuh"
#include "attn_tc.h"
#include "common.cuh"
#include "ptx.cuh"
#include "tc_common.cuh"

namespace mcs {
namespace {

constexpr int kSparseThreads = 512;
constexpr int kGather = 256;  // gather threads (warpgroups 1-2)
constexpr int kRegSoftmax = 224, kRegGather = 80, kRegMma = 64;
constexpr int kRegPool = 128 * kRegSoftmax + kGather * kRegGather + 128 * kRegMma;

template <int D>
struct SparseCfg {
  static constexpr int kSK = 3, kSV = 3;      // K and V stages
  static constexpr int kLag = 2;              // iterations between a copy group's issue and its retirement
  static constexpr int kRing = kLag + 1;      // index chunks of 128 keys in shared memory
  static constexpr int kTile = (D / 64) * kRegion;
  static constexpr int kQ = 0;
  static constexpr int kK = kQ + kTile;
  static constexpr int kV = kK + kSK * kTile;
  static constexpr int kBar = kV + kSV * kTile;
  static constexpr int kNumBars = 1 + 2 * kSK + 2 * kSV + 4 + 4;
  static constexpr int kMisc = kBar + kNumBars * 8;  // tmem slot, stop flags [2]
  static constexpr int kIdx = kMisc + 32;
  static constexpr int kBytes = kIdx + kRing * 128 * 4;
  static constexpr int kAlloc = kBytes + 1024;
  static constexpr uint32_t kColS = 0, kColO = 256, kColP = 384;
};

template <int D, int kEpi>
__global__ void __launch_bounds__(kSparseThreads, 1) attn_sparse_kernel(const TcAttnParams p) {
  using L = SparseCfg<D>;
  constexpr int SK = L::kSK, SV = L::kSV, kLag = L::kLag;
  constexpr int kChunks = D / 8;  // 16-byte chunks per row
  constexpr int kRowsPerPass = kGather / kChunks;
  constexpr int kPasses = 128 / kRowsPerPass;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(smem);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::kBar);
  uint64_t* q_full = bars;
  uint64_t* k_full = bars + 1;
  uint64_t* k_empty = k_full + SK;
  uint64_t* v_full = k_empty + SK;
  uint64_t* v_empty = v_full + SV;
  uint64_t* s_full = v_empty + SV;  // [2]
  uint64_t* s_free = s_full + 2;    // [2]
  uint64_t* p_full = s_free + 2;
  uint64_t* p_empty = p_full + 1;
  uint64_t* o_done = p_empty + 1;
  uint64_t* drain = o_done + 1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::kMisc);
  // the gather leader's decision for iteration i lives in stop[i & 1]: a slow
  // reader of iteration i never sees the leader's write for iteration i + 1
  volatile int* stop = reinterpret_cast<volatile int*>(smem + L::kMisc + 8);
  int32_t* ring = reinterpret_cast<int32_t*>(smem + L::kIdx);  // [kRing][128]

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int bh = blockIdx.y, g = blockIdx.x;
  const int nkv = p.K;
  const int T = (nkv + 127) / 128;
  uint32_t* st = p.status;
  const int32_t* idxg = p.idx + (size_t(bh) * p.G + g) * size_t(p.K);

  if (tid == 0) {
    mbar_init(q_full, kGather);
    for (int s = 0; s < SK; ++s) {
      mbar_init(k_full + s, kGather);
      mbar_init(k_empty + s, 1);
    }
    for (int s = 0; s < SV; ++s) {
      mbar_init(v_full + s, kGather);
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
  if (warp == 12) {
    tmem_alloc(tmem_slot, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const uint32_t tS = tmem + L::kColS, tO = tmem + L::kColO, tP = tmem + L::kColP;

  if (warp < 4) {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kRegSoftmax));
    // ------------------------------------------------------------ softmax, epilogue
    const int row = tid;
    const uint32_t lane_off = uint32_t(warp * 32) << 16;
    int tok = -1;
    if (row < p.C) {
      const int v = __ldg(p.perm + size_t(bh) * p.N_pad + size_t(g) * p.C + row);
      if (v < 0 || v >= p.N_pad) raise_status(st, kStatusBounds);
      else if (v < p.N) tok = v;
    }
    float m, l;
    const SoftmaxSync sy{s_full, s_free, p_full, p_empty};
    bool ok = softmax_rows<D, true>(T, nkv, tS, tO, tP, lane_off, p.scale_log2, sy, st, m, l);
    if (ok) ok = warp_all(mbar_wait(o_done, 0, st));
    if (ok) {
      tc_fence_after();
      __nv_bfloat16* dst = (kEpi == kEpiStoreResidual) ? p.res_out : p.o;
      store_row<D, kEpi>(tO, lane_off, tok, (size_t(bh) * p.N + size_t(tok < 0 ? 0 : tok)) * D, 1.f / l, dst,
                         p.res_in);
    }
    if (!ok && row == 0) raise_status(st, kStatusTimeout);
  } else if (warp < 12) {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kRegGather));
    // ------------------------------------------------------------ gather warps
    const int t = tid - 128;  // 0..255
    const int ch = t % kChunks, r0 = t / kChunks;
    const __nv_bfloat16* kb = p.k + size_t(bh) * p.N * D;
    const __nv_bfloat16* vb = p.v + size_t(bh) * p.N * D;
    {  // the group's query rows (through perm): operand A of S = Q K^T
      const __nv_bfloat16* qb = p.q + size_t(bh) * p.N * D;
      const int32_t* permg = p.perm + size_t(bh) * p.N_pad + size_t(g) * p.C;
#pragma unroll 4
      for (int it = 0; it < kPasses; ++it) {
        const int row = it * kRowsPerPass + r0;
        int tq = -1;
        if (row < p.C) {
          const int v = __ldg(permg + row);
          if (v < 0 || v >= p.N_pad) raise_status(st, kStatusBounds);
          else if (v < p.N) tq = v;
        }
        cp_async16(sbase + L::kQ + sw128_off(row, ch), qb + size_t(tq < 0 ? 0 : tq) * D + ch * 8, tq >= 0);
      }
    }
    // index chunks of tiles 0..kLag-1
#pragma unroll
    for (int tt = 0; tt < kLag; ++tt)
      for (int e = t; e < 128; e += kGather) {
        const int slot = tt * 128 + e;
        cp_async4(smem_u32(ring + tt * 128 + e), idxg + (slot < nkv ? slot : 0), slot < nkv);
      }
    cp_async_commit();
    cp_async_wait<0>();
    fence_proxy_async_smem();
    mbar_arrive(q_full);
    named_bar_sync(1, kGather);
    int prev[kPasses];  // this thread's key ids of tile i-1, for its value rows
#pragma unroll
    for (int it = 0; it < kPasses; ++it) prev[it] = -1;
    bool ok = true;
    int issued = 0;  // iterations whose copy group was committed
    for (int i = 0; i <= T; ++i) {
      if (i >= kLag) {  // retire iteration i - kLag: K of tile i-kLag, V of tile i-kLag-1
        cp_async_wait<kLag - 1>();
        fence_proxy_async_smem();
        const int r = i - kLag;
        if (r < T) mbar_arrive(k_full + r % SK);
        if (r >= 1) mbar_arrive(v_full + (r - 1) % SV);
      }
      if (t == 0) {
        int stp = 0;
        if (i < T && !mbar_wait(k_empty + i % SK, ((i / SK) & 1) ^ 1, st)) stp = 1;           // S of tile i-SK done
        if (!stp && i >= 1 && !mbar_wait(v_empty + (i - 1) % SV, (((i - 1) / SV) & 1) ^ 1, st))  // PV of tile i-1-SV
          stp = 1;
        if (stp) raise_status(st, kStatusTimeout);
        stop[i & 1] = stp;
      }
      named_bar_sync(1, kGather);
      if (stop[i & 1]) {
        ok = false;
        break;
      }
      int toks[kPasses];
      if (i < T) {
        const int32_t* rt = ring + (i % L::kRing) * 128;
#pragma unroll
        for (int it = 0; it < kPasses; ++it) {
          const int row = it * kRowsPerPass + r0;
          int tk = (i * 128 + row < nkv) ? rt[row] : -1;
          if (tk >= p.N || (tk < 0 && i * 128 + row < nkv)) {
            raise_status(st, kStatusBounds);
            tk = -1;
          }
          toks[it] = tk;
        }
        const uint32_t dk = sbase + L::kK + (i % SK) * L::kTile;
#pragma unroll
        for (int it = 0; it < kPasses; ++it) {
          const int row = it * kRowsPerPass + r0;
          cp_async16(dk + sw128_off(row, ch), kb + size_t(toks[it] < 0 ? 0 : toks[it]) * D + ch * 8, toks[it] >= 0);
        }
      }
      if (i >= 1) {
        const uint32_t dv = sbase + L::kV + ((i - 1) % SV) * L::kTile;
#pragma unroll
        for (int it = 0; it < kPasses; ++it) {
          const int row = it * kRowsPerPass + r0;
          cp_async16(dv + sw128_off(row, ch), vb + size_t(prev[it] < 0 ? 0 : prev[it]) * D + ch * 8, prev[it] >= 0);
        }
      }
      for (int e = t; e < 128; e += kGather) {
        const int tn = i + kLag, slot = tn * 128 + e;
        cp_async4(smem_u32(ring + (tn % L::kRing) * 128 + e), idxg + (slot < nkv ? slot : 0), slot < nkv);
      }
      cp_async_commit();
      issued = i + 1;
      if (i < T) {
#pragma unroll
        for (int it = 0; it < kPasses; ++it) prev[it] = toks[it];
      }
    }
    cp_async_wait<0>();
    fence_proxy_async_smem();
    if (ok) {  // iterations issued - kLag .. issued - 1 were not retired in the loop
      for (int r = (issued > kLag ? issued - kLag : 0); r < issued; ++r) {
        if (r < T) mbar_arrive(k_full + r % SK);
        if (r >= 1) mbar_arrive(v_full + (r - 1) % SV);
      }
    }
  } else {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kRegMma));
    // ------------------------------------------------------------ MMA issuer (warp 12)
    if (warp == 12 && lane == 0) {
      constexpr uint32_t kIdescQK = idesc_bf16_f32(128, 128, 0, 0);
      constexpr uint32_t kIdescPV = idesc_bf16_f32(128, D, 0, 1);
      bool ok = mbar_wait(q_full, 0, st);
      bool issued = false;
      if (ok) tc_fence_after();
      auto s_ready = [&](int j) {
        return mbar_test(k_full + j % SK, uint32_t(j / SK) & 1) && mbar_test(s_free + (j & 1), (uint32_t(j >> 1) & 1) ^ 1);
      };
      auto issue_s = [&](int j) -> bool {
        if (!mbar_wait(k_full + j % SK, uint32_t(j / SK) & 1, st)) return false;
        if (!mbar_wait(s_free + (j & 1), (uint32_t(j >> 1) & 1) ^ 1, st)) return false;
        tc_fence_after();
        const uint32_t kt = sbase + L::kK + (j % SK) * L::kTile;
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks)
          tc_mma_ss(tS + (j & 1) * 128, desc_kmajor(sbase + L::kQ, ks), desc_kmajor(kt, ks), kIdescQK, ks > 0 ? 1u : 0u);
        tc_commit(s_full + (j & 1));
        tc_commit(k_empty + j % SK);
        issued = true;
        return true;
      };
      auto issue_pv = [&](int i) -> bool {
        const int s = i % SV;
        if (!mbar_wait(v_full + s, uint32_t(i / SV) & 1, st)) return false;
        if (!mbar_wait(p_full, uint32_t(i) & 1, st)) return false;
        tc_fence_after();
        const uint32_t vt = sbase + L::kV + s * L::kTile;
#pragma unroll
        for (int ks = 0; ks < 8; ++ks)
          tc_mma_ts(tO, tP + ks * 8, desc_mnmajor(vt, ks), kIdescPV, (i > 0 || ks > 0) ? 1u : 0u);
        tc_commit(p_empty);
        tc_commit(v_empty + s);
        return true;
      };
      if (ok && T > 0) ok = issue_s(0);
      for (int j = 0; ok && j < T; ++j) {
        // S_{j+1} and PV_j are independent: take S_{j+1} first only if it can go now
        const bool s_next = j + 1 < T;
        bool s_done = false;
        if (s_next && s_ready(j + 1)) {
          ok = issue_s(j + 1);
          s_done = true;
        }
        if (ok) ok = issue_pv(j);
        if (ok && s_next && !s_done) ok = issue_s(j + 1);
      }
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
  tc_fence_before();
  __syncthreads();
  if (warp == 12) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

template <int D, int kEpi>
cudaError_t launch_sparse(const TcAttnParams& p, cudaStream_t stream) {
  using L = SparseCfg<D>;
  auto kern = attn_sparse_kernel<D, kEpi>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, L::kAlloc);
  if (e != cudaSuccess) return e;
  // setmaxnreg.inc waits for registers released by the other warpgroups: launch
  // only if the rebalanced split fits what the block is launched with
  cudaFuncAttributes fa;
  if ((e = cudaFuncGetAttributes(&fa, kern)) != cudaSuccess) return e;
  if (fa.numRegs * kSparseThreads < kRegPool || fa.numRegs < kRegGather) return cudaErrorInvalidValue;
  dim3 grid(p.tiles_per_head, p.BH);
  kern<<<grid, kSparseThreads, L::kAlloc, stream>>>(p);
  note_launches(1);
  return cudaGetLastError();
}

}  // namespace

cudaError_t tc_sparse_attn(int D, int epi, const TcAttnParams& p, int BH, cudaStream_t stream) {
  (void)BH;
#define MCS_SPARSE_CASE(DD, EE) \
  if (D == DD && epi == EE) return launch_sparse<DD, EE>(p, stream);
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
