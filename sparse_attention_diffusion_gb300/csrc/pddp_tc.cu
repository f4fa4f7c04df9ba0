// PDDP chunk moments on the tcgen05 tensor cores, bf16 queries with d = 128
// [MC-Sparse summary: PDDP paragraph: the principal direction of a node's
// queries]. For every chunk (<= 8 groups of one node, rows gathered through
// perm) it writes
//     pcov = sum_r x_r x_r^T   (d x d, fp32),   psum = sum_r x_r,   pcnt = #real rows,
// the raw second moment, from which the node covariance is
// sum_chunks pcov - n mu mu^T. The bf16 products are exact, so this is the
// same quantity the SIMT path forms, accumulated in fp32 in another order.
//
// The chunk tile X [128 rows x d] sits in shared memory in the 128-byte
// swizzled layout with d contiguous, which is the MN-major layout of X^T for
// both operands of D = X^T X (M = N = d, K = rows); a second MMA against a tile
// of ones (N = 16) gives the column sums in the same pass.
//
// Persistent CTAs walk the (head, chunk) items, 288 threads:
//   warps 0-3  gather: 16-byte copies of the tile's rows (pads and rows past
//              the chunk read zeros) into a 4-stage ring, each thread's copies
//              ended by an asynchronous arrive on the stage's full barrier;
//   warp 4     tensor-memory allocation and the single MMA-issuing thread; two
//              accumulator sets let a chunk accumulate while the previous one
//              drains;
//   warps 5-8  epilogue: tensor memory -> global (the accumulator's row i is
//              TMEM lane i; thread i writes column i of the stored matrix, so a
//              warp writes 128 contiguous bytes per store; D is symmetric) and
//              the chunk's real-row count from perm.
// All waits are bounded; on a timeout the CTA flags it, lets its copies and
// MMAs land, frees tensor memory and returns.
#include "common.cuh"
#include "kernels.h"
#include "ptx.cuh"
#include "status.cuh"
#include "tc_common.cuh"

namespace mcs {
namespace {

constexpr int kD = 128;
constexpr int kThreads = 288;
constexpr int kMmaWarp = 4, kEpiWarp0 = 5;
constexpr int kStages = 4;
constexpr int kTile = 2 * kRegion;  // 128 rows x 256 bytes
constexpr int kOnes = kStages * kTile;
constexpr int kBar = kOnes + kTile;
// full[S], empty[S], acc_full[2], acc_empty[2], drain
constexpr int kNumBars = 2 * kStages + 5;
constexpr int kSlot = kBar + kNumBars * 8;
constexpr int kCntRed = kSlot + 16;  // [4] per-warp row counts, then [4] per-warp wait results
constexpr int kBytes = kCntRed + 32;
constexpr int kAlloc = kBytes + 1024;
constexpr int kAccCols = 256;  // per accumulator set: D at +0 (128 cols), sums at +128 (16 cols)

struct CovParams {
  const __nv_bfloat16* x;   // [BH, N, d]
  const int32_t* perm;      // [BH, N_pad], current level's order
  const int* chunk_g0;      // [nch] this level
  const int* chunk_ng;      // [nch]
  float* psum;              // [BH, max_chunks, d]
  int* pcnt;                // [BH, max_chunks]
  float* pcov;              // [BH, max_chunks, d, d]
  int nch, BH, N, N_pad, C, max_chunks;
  uint32_t* status;
};

__global__ void __launch_bounds__(kThreads, 1) pddp_moments_kernel(const CovParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(smem);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kBar);
  uint64_t* full = bars;
  uint64_t* empty = full + kStages;
  uint64_t* acc_full = empty + kStages;
  uint64_t* acc_empty = acc_full + 2;
  uint64_t* drain = acc_empty + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kSlot);
  int* cnt_red = reinterpret_cast<int*>(smem + kCntRed);
  int* ok_red = cnt_red + 4;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int items = p.nch * p.BH;
  uint32_t* st = p.status;

  // the ones tile (B of the column-sum MMA): every element is 1.0, so its layout is moot
  for (int i = tid; i < kTile / 16; i += kThreads)
    reinterpret_cast<uint4*>(smem + kOnes)[i] = make_uint4(0x3F803F80u, 0x3F803F80u, 0x3F803F80u, 0x3F803F80u);
  fence_proxy_async_smem();
  if (tid == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(full + s, 128);
      mbar_init(empty + s, 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(acc_full + b, 1);
      mbar_init(acc_empty + b, 128);
    }
    mbar_init(drain, 1);
    fence_mbar_init();
  }
  if (warp == kMmaWarp) {
    tmem_alloc(tmem_slot, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp < 4) {
    // ------------------------------------------------------------ gather
    const int ch = tid & 15, r0 = tid >> 4;  // 8 rows per pass, 16 chunks of 16 bytes per row
    const uint32_t doff = sw128_off(r0, ch);
    int seq = 0;
    bool ok = true;
    for (int w = blockIdx.x; ok && w < items; w += gridDim.x) {
      const int bh = w / p.nch, c = w % p.nch;
      const int g0 = __ldg(p.chunk_g0 + c), rows = __ldg(p.chunk_ng + c) * p.C;
      const int32_t* pr = p.perm + size_t(bh) * p.N_pad + size_t(g0) * p.C;
      const __nv_bfloat16* xb = p.x + size_t(bh) * p.N * kD + ch * 8;
      for (int r = 0; r < rows; r += 128, ++seq) {
        const int s = seq % kStages;
        if (!warp_all(mbar_wait(empty + s, (uint32_t(seq / kStages) & 1) ^ 1, st))) {
          ok = false;
          break;
        }
        const uint32_t dst = sbase + s * kTile + doff;
#pragma unroll 4
        for (int it = 0; it < 16; ++it) {
          const int row = r + it * 8 + r0;
          int tok = -1;
          if (row < rows) {
            const int v = __ldg(pr + row);
            if (v < 0 || v >= p.N_pad) raise_status(st, kStatusBounds);
            else if (v < p.N) tok = v;
          }
          cp_async16(dst + it * 8 * 128, xb + size_t(tok < 0 ? 0 : tok) * kD, tok >= 0);
        }
        cp_async_arrive_noinc(full + s);
      }
    }
    if (!ok && tid == 0) raise_status(st, kStatusTimeout);
    asm volatile("cp.async.wait_all;" ::: "memory");
  } else if (warp == kMmaWarp) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t kIdescCov = idesc_bf16_f32(128, kD, 1, 1);
      constexpr uint32_t kIdescSum = idesc_bf16_f32(128, 16, 1, 0);
      const uint32_t ones_lo = desc_lo_kmajor(sbase + kOnes);
      int seq = 0, k = 0;
      bool ok = true, issued = false;
      for (int w = blockIdx.x; ok && w < items; w += gridDim.x, ++k) {
        const int c = w % p.nch;
        const int rows = __ldg(p.chunk_ng + c) * p.C;
        const int b = k & 1;
        if (!mbar_wait(acc_empty + b, (uint32_t(k >> 1) & 1) ^ 1, st)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t tD = tmem + b * kAccCols, tS = tD + 128;
        for (int r = 0; r < rows; r += 128, ++seq) {
          const int s = seq % kStages;
          if (!mbar_wait(full + s, uint32_t(seq / kStages) & 1, st)) {
            ok = false;
            break;
          }
          fence_proxy_async_smem();
          tc_fence_after();
          const uint32_t xlo = desc_lo_mnmajor(sbase + s * kTile);
#pragma unroll
          for (int ks = 0; ks < 8; ++ks) {
            const uint32_t acc = (r > 0 || ks > 0) ? 1u : 0u;
            tc_mma_ss_lo(tD, xlo + kstep_mnmajor(ks), xlo + kstep_mnmajor(ks), kIdescCov, acc);
            tc_mma_ss_lo(tS, xlo + kstep_mnmajor(ks), ones_lo + kstep_kmajor(ks), kIdescSum, acc);
          }
          tc_commit(empty + s);
          issued = true;
        }
        if (!ok) break;
        tc_commit(acc_full + b);
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
  } else {
    // ------------------------------------------------------------ epilogue
    const int et = tid - kEpiWarp0 * 32;             // 0..127
    const int i = (warp & 3) * 32 + lane;            // TMEM lane = accumulator row
    const uint32_t lane_off = uint32_t((warp & 3) * 32) << 16;
    int k = 0;
    for (int w = blockIdx.x; w < items; w += gridDim.x, ++k) {
      const int bh = w / p.nch, c = w % p.nch;
      const int g0 = __ldg(p.chunk_g0 + c), rows = __ldg(p.chunk_ng + c) * p.C;
      // real rows of the chunk (overlaps the accumulation)
      const int32_t* pr = p.perm + size_t(bh) * p.N_pad + size_t(g0) * p.C;
      int cnt = 0;
      for (int r = et; r < rows; r += 128) cnt += uint32_t(__ldg(pr + r)) < uint32_t(p.N) ? 1 : 0;
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) cnt += __shfl_xor_sync(0xffffffffu, cnt, off);
      const int b = k & 1;
      // every epilogue warp reaches both named barriers of an item, and all four
      // take the same decision after a timeout (no warp is left at a barrier)
      const bool okw = warp_all(mbar_wait(acc_full + b, uint32_t(k >> 1) & 1, st));
      if (lane == 0) {
        cnt_red[warp & 3] = cnt;
        ok_red[warp & 3] = okw ? 1 : 0;
      }
      named_bar_sync(1, 128);
      if (!(ok_red[0] & ok_red[1] & ok_red[2] & ok_red[3])) {
        if (et == 0) raise_status(st, kStatusTimeout);
        break;
      }
      tc_fence_after();
      const size_t item = size_t(bh) * p.max_chunks + c;
      float* out = p.pcov + item * kD * kD + i;
      const uint32_t tD = tmem + lane_off + b * kAccCols;
#pragma unroll 1
      for (int cb = 0; cb < kD / 32; ++cb) {
        uint32_t r[32];
        tmem_ld32(tD + cb * 32, r);
#pragma unroll
        for (int jj = 0; jj < 32; ++jj) out[size_t(cb * 32 + jj) * kD] = __uint_as_float(r[jj]);
      }
      {
        uint32_t r[32];
        tmem_ld32(tD + 128, r);
        p.psum[item * kD + i] = __uint_as_float(r[0]);
      }
      tc_fence_before();
      mbar_arrive(acc_empty + b);
      if (et == 0) p.pcnt[item] = cnt_red[0] + cnt_red[1] + cnt_red[2] + cnt_red[3];
      named_bar_sync(1, 128);  // cnt_red / ok_red are rewritten by the next item
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

}  // namespace

cudaError_t pddp_moments_tc(const __nv_bfloat16* x, const int32_t* perm, const int* chunk_g0, const int* chunk_ng,
                            int nch, int BH, int N, int N_pad, int C, float* psum, int* pcnt, float* pcov,
                            int max_chunks, uint32_t* status, int num_sms, cudaStream_t stream) {
  if (nch <= 0 || BH <= 0) return cudaSuccess;
  CovParams p{x, perm, chunk_g0, chunk_ng, psum, pcnt, pcov, nch, BH, N, N_pad, C, max_chunks, status};
  cudaError_t e = cudaFuncSetAttribute(pddp_moments_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kAlloc);
  if (e != cudaSuccess) return e;
  const int items = nch * BH;
  const int grid = items < num_sms ? items : num_sms;
  pddp_moments_kernel<<<grid, kThreads, kAlloc, stream>>>(p);
  note_launches(1);
  return cudaGetLastError();
}

}  // namespace mcs
