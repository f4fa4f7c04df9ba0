// Token-gather sparse attention on the tcgen05 tensor cores, bf16 inputs
// (sm_103a): for one query group (the C members of group g, read through perm),
// softmax attention over the group's own K selected keys, whose key and value
// rows are fetched at the group's index list rather than repacked into blocks
// [MC-Sparse summary: index-gather / PDDP paragraph]. Epilogues add the cached
// residual (reuse step) or store R = O_dense - O_sparse (anchor step)
// [MC-Sparse summary: residual paragraph].
//
// One CTA per group (kernels that hold tensor memory run one CTA per SM), in the
// structure of the dense kernel: S double-buffered in tensor memory, so S_{j+1}
// is computed while the softmax of S_j runs and P_j V_j while the softmax of
// S_{j+1} runs; one thread issues the S chain and another the P V chain. 640
// threads: warpgroups 0-1 softmax and epilogue, 2-3 gather, warp 16 tensor-memory
// allocation and the S chain, warp 17 the P V chain. The two softmax warpgroups
// work on the same tensor-memory lanes and split every tile's keys, each thread
// with its own running max and sum and its own O accumulator (warpgroup h into
// O_h: O_0 at column 256, O_1 at 384), writing its P as bf16 pairs over S
// columns it has read; the P V of a tile is two chains of four MMAs (one per
// accumulator), and S buffer b is refilled once the P V of its tile is done.
//   Groups of more than 64 queries: query r on lane r; warpgroup h takes keys
//     [64h, 64h + 64) of every tile. The two threads of a row each store half of
//     the output columns.
//   Groups of at most 64 (kQ64): query q on lanes q and q + 64 (the gather copies
//     its row into both rows of the query tile); lane q takes keys 0-63 and lane
//     q + 64 keys 64-127, split again between the warpgroups (32 keys per
//     thread), and each thread zeroes the P columns of its lane that its chain
//     reads for the other lane's keys. Lanes 64-127 hand their two partial rows
//     to lanes 0-63 through shared memory; four partial rows make each output.
// Eight gather warps copy the group's query rows (through perm) once, then per
// tile the key and value rows at the group's index list, as 16-byte cp.async
// copies into 3-stage K and V rings (6 stages at d = 64; 128-byte swizzled);
// eight threads per row, each copying one chunk of every 128-byte half, so a
// thread holds 4 row ids per tile; once idle they prefetch into L2 the group's
// residual rows and the first rows of the group starting about one SM count
// later. The gather warps never wait for their own copies: each thread ends a
// tile's key (value) copies with an asynchronous arrive on the stage's full
// barrier, which completes when every thread's rows have landed; the issuing
// threads then fence the generic-to-async proxy before the tensor core reads
// them. The gather warps only wait (through one leader and a named barrier) for
// the stages to be released: a K stage when S of its tile is done, a V stage when
// P V is done. Each gather thread reads its row indices for the next tile into
// registers while the leader waits, and issues a tile's copies back to back. The
// epilogue's residual row is loaded while the last P V runs. Registers are
// rebalanced with setmaxnreg; the launcher checks that the split fits the
// registers the block is launched with. All waits are bounded; on a timeout the
// CTA flags it, lets its copies and MMAs land, frees tensor memory and returns.
#include "attn_common.cuh"
#include "attn_tc.h"
#include "common.cuh"
#include "ptx.cuh"
#include "tc_common.cuh"

namespace mcs {
namespace {

constexpr int kGather = 256;  // gather threads (warpgroups 2-3)

// ---------------------------------------------------------------- layout
constexpr int kCsThreads = 640;
constexpr int kCsMmaWarp = 16, kCsPvWarp = 17;
constexpr int kCsRegSoftmax = 176, kCsRegGather = 48, kCsRegMma = 32;
constexpr int kCsRegPool = 256 * kCsRegSoftmax + kGather * kCsRegGather + 128 * kCsRegMma;

template <int D>
struct CsCfg {
  static constexpr int kSK = D == 64 ? 6 : 3, kSV = kSK;
  static constexpr int kTile = (D / 64) * kRegion;
  static constexpr int kQ = 0;
  static constexpr int kK = kQ + kTile;
  static constexpr int kV = kK + kSK * kTile;
  static constexpr int kBar = kV + kSV * kTile;
  static constexpr int kNumBars = 1 + 2 * kSK + 2 * kSV + 2 + 2 + 2 + 1 + 2;
  static constexpr int kMisc = kBar + kNumBars * 8;  // tmem slot, stop flags [2]
  static constexpr int kBytes = kMisc + 32;
  static constexpr int kAlloc = kBytes + 1024;
  static constexpr uint32_t kColOa = 256, kColOb = 384;  // S0, S1 at 0 and 128
  static_assert(kAlloc <= 227 * 1024, "shared memory");
  static_assert(4 * 256 * 4 <= kSK * kTile, "the epilogue's max / sum exchange fits the key ring");
};

template <int D, int kEpi, bool kQ64>
__global__ void __launch_bounds__(kCsThreads, 1) attn_sparse_cs_kernel(const TcAttnParams p) {
  using L = CsCfg<D>;
  constexpr int SK = L::kSK, SV = L::kSV;
  static_assert(SK == SV, "one stage index for tile i's key and value rows");
  constexpr int kChunks = 8;
  constexpr int kHalves = D / 64;
  constexpr int kRowsPerPass = kGather / kChunks;  // 32
  constexpr int kPasses = 128 / kRowsPerPass;      // 4 ids per thread per tile
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(smem);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::kBar);
  uint64_t* q_full = bars;
  uint64_t* k_full = bars + 1;
  uint64_t* k_empty = k_full + SK;
  uint64_t* v_full = k_empty + SK;
  uint64_t* v_empty = v_full + SV;
  uint64_t* s_full = v_empty + SV;   // [2] S buffer b written
  uint64_t* pv_done = s_full + 2;    // [2] P V of the tile in S buffer b done (buffer free)
  uint64_t* p_full = pv_done + 2;    // [2] both halves of P written over S buffer b
  uint64_t* o_done = p_full + 2;     // the last P V done
  uint64_t* drain = o_done + 1;      // [2] one per issuing thread
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::kMisc);
  volatile int* stop = reinterpret_cast<volatile int*>(smem + L::kMisc + 8);

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
      mbar_init(pv_done + b, 1);
      mbar_init(p_full + b, 256);
    }
    mbar_init(o_done, 1);
    mbar_init(drain, 1);
    mbar_init(drain + 1, 1);
    fence_mbar_init();
  }
  if (warp == kCsMmaWarp) {
    tmem_alloc(tmem_slot, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp < 8) {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kCsRegSoftmax));
    // ------------------------------------------------------------ softmax, epilogue
    const int h = warp >> 2;                 // which half of every tile (and of the output row)
    const int row = (warp & 3) * 32 + lane;  // tensor-memory lane
    const int qrow = kQ64 ? row & 63 : row;  // kQ64: query q on lanes q and q + 64
    const bool hi = kQ64 && row >= 64;
    const uint32_t lane_off = uint32_t((warp & 3) * 32) << 16;
    int tok = -1;
    if (qrow < p.C) {
      const int v = __ldg(p.perm + size_t(bh) * p.N_pad + size_t(g) * p.C + qrow);
      if (v < 0 || v >= p.N_pad) raise_status(st, kStatusBounds);
      else if (v < p.N) tok = v;
    }
    if (hi) tok = -1;  // lanes 64-127 hand their partial rows to lanes 0-63
    float m, l;
    bool ok;
    if constexpr (kQ64) {
      // keys [64 hi + 32 h, + 32) of every tile; zeros over [64 (1 - hi) + 32 h, + 16)
      ok = softmax_rows_cs<D, 32>(T, nkv, tmem, tmem + (h ? L::kColOb : L::kColOa), lane_off, (hi ? 64 : 0) + 32 * h,
                                  p.scale_log2, s_full, pv_done, p_full, st, m, l, (hi ? 0 : 64) + 32 * h);
    } else {
      ok = softmax_rows_cs<D>(T, nkv, tmem, tmem + (h ? L::kColOb : L::kColOa), lane_off, h * 64, p.scale_log2,
                              s_full, pv_done, p_full, st, m, l);
    }
    // this half of the row's residual (or O_dense), loaded while the last P V runs
    constexpr int kC = D / 2;  // output columns per thread
    uint4 rres[D / 16] = {};
    if constexpr (kEpi != kEpiPlain) {
      if (tok >= 0) {
        const uint4* src = reinterpret_cast<const uint4*>(p.res_in + (size_t(bh) * p.N + size_t(tok)) * D + h * kC);
#pragma unroll
        for (int i = 0; i < D / 16; ++i) rres[i] = src[i];
      }
    }
    // Every S has been read and every tile has landed, so the key ring is free:
    // the two halves of a row swap their max and sum through it. All 256 threads
    // meet at the named barrier whatever their wait status.
    float* xm = reinterpret_cast<float*>(smem + L::kK);  // [2][128] max, then [2][128] sum
    xm[h * 128 + row] = m;
    xm[512 + h * 128 + row] = l;
    if (ok) ok = warp_all(mbar_wait(o_done, 0, st));
    named_bar_sync(2, 256);
    __nv_bfloat16* dst = (kEpi == kEpiStoreResidual) ? p.res_out : p.o;
    const size_t rowoff = (size_t(bh) * p.N + size_t(tok < 0 ? 0 : tok)) * D;
    if constexpr (kQ64) {
      // four partial rows per query: (warpgroup 0 / 1) x (lane q / q + 64)
      const int q = qrow;
      const float m00 = xm[q], m10 = xm[128 + q], m01 = xm[64 + q], m11 = xm[192 + q];
      const float l00 = xm[512 + q], l10 = xm[640 + q], l01 = xm[576 + q], l11 = xm[704 + q];
      const float mm = fmaxf(fmaxf(m00, m10), fmaxf(m01, m11));
      auto wt = [&](float x) { return x == -INFINITY ? 0.f : ex2_approx(x - mm); };
      const float f00 = wt(m00), f10 = wt(m10), f01 = wt(m01), f11 = wt(m11);
      const float inv = 1.f / (l00 * f00 + l10 * f10 + l01 * f01 + l11 * f11);
      float4* xo = reinterpret_cast<float4*>(smem + L::kK + 4096);  // [D / 4][64] partials of lanes 64-127
      if (hi && ok) {
        tc_fence_after();
        partial_row_cs4<D>(tmem + L::kColOa, tmem + L::kColOb, lane_off, h * kC, f01, f11, xo + (h * kC / 4) * 64 + q);
      }
      named_bar_sync(2, 256);
      if (!hi && ok) {
        tc_fence_after();
        store_row_cs4<D, kEpi>(tmem + L::kColOa, tmem + L::kColOb, lane_off, h * kC, tok, rowoff, f00, f10, inv,
                               xo + (h * kC / 4) * 64 + q, dst, rres);
      }
    } else if (ok) {
      tc_fence_after();
      const float ma = xm[row], mb = xm[128 + row], la = xm[512 + row], lb = xm[640 + row];
      const float mm = fmaxf(ma, mb);
      const float fa = ma == -INFINITY ? 0.f : ex2_approx(ma - mm);
      const float fb = mb == -INFINITY ? 0.f : ex2_approx(mb - mm);
      const float inv = 1.f / (la * fa + lb * fb);
      store_row_cs<D, kEpi>(tmem + L::kColOa, tmem + L::kColOb, lane_off, h * kC, tok, rowoff, fa * inv, fb * inv,
                            dst, rres);
    }
    if (!ok && tid == 0) raise_status(st, kStatusTimeout);
  } else if (warp < 16) {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kCsRegGather));
    // ------------------------------------------------------------ gather warps
    const int t = tid - 256;  // 0..255
    const int ch = t % kChunks, r0 = t / kChunks;
    const __nv_bfloat16* kb = p.k + size_t(bh) * p.N * D;
    const __nv_bfloat16* vb = p.v + size_t(bh) * p.N * D;
    auto load_ids = [&](int i, int (&ids)[kPasses]) {
#pragma unroll
      for (int it = 0; it < kPasses; ++it) {
        const int slot = i * 128 + it * kRowsPerPass + r0;
        ids[it] = slot < nkv ? __ldg(idxg + slot) : -1;
      }
    };
    int ida[kPasses], idb[kPasses];
    load_ids(0, ida);
    {  // the group's query rows (through perm): operand A of S = Q K^T
      const __nv_bfloat16* qb = p.q + size_t(bh) * p.N * D;
      const int32_t* permg = p.perm + size_t(bh) * p.N_pad + size_t(g) * p.C;
#pragma unroll 4
      for (int it = 0; it < kPasses; ++it) {
        const int row = it * kRowsPerPass + r0;
        const int qr = kQ64 ? row & 63 : row;  // kQ64: rows q and q + 64 hold the same query
        int tq = -1;
        if (qr < p.C) {
          const int v = __ldg(permg + qr);
          if (v < 0 || v >= p.N_pad) raise_status(st, kStatusBounds);
          else if (v < p.N) tq = v;
        }
#pragma unroll
        for (int hh = 0; hh < kHalves; ++hh)
          cp_async16(sbase + L::kQ + hh * kRegion + sw128_off(row, ch), qb + size_t(tq < 0 ? 0 : tq) * D + hh * 64 + ch * 8,
                     tq >= 0);
      }
      cp_async_arrive_noinc(q_full);
    }
    static_assert(kRowsPerPass % 8 == 0, "a thread's rows share one swizzle phase");
    const uint32_t doff = sw128_off(r0, ch);
    const __nv_bfloat16* kbc = kb + ch * 8;
    const __nv_bfloat16* vbc = vb + ch * 8;
    auto tile = [&](int i, int (&ids)[kPasses], int (&next)[kPasses]) -> bool {
      if (i + 1 < T) load_ids(i + 1, next);
      const int s = i % SK;
      const uint32_t par = (uint32_t(i / SK) & 1) ^ 1;
      if (t == 0) {  // the K stage (S of tile i-SK) and the V stage (PV of tile i-SV) are free
        int stp = 0;
        if (!mbar_wait(k_empty + s, par, st) || !mbar_wait(v_empty + s, par, st)) stp = 1;
        if (stp) raise_status(st, kStatusTimeout);
        stop[i & 1] = stp;
      }
      named_bar_sync(1, kGather);
      if (stop[i & 1]) return false;
      bool all_valid = true;
#pragma unroll
      for (int it = 0; it < kPasses; ++it) all_valid &= uint32_t(ids[it]) < uint32_t(p.N);
      const uint32_t dk = sbase + L::kK + s * L::kTile + doff, dv = sbase + L::kV + s * L::kTile + doff;
      if (all_valid) {
#pragma unroll
        for (int it = 0; it < kPasses; ++it)
#pragma unroll
          for (int hh = 0; hh < kHalves; ++hh)
            cp_async16(dk + hh * kRegion + it * kRowsPerPass * 128, kbc + size_t(uint32_t(ids[it])) * D + hh * 64, true);
        cp_async_arrive_noinc(k_full + s);
#pragma unroll
        for (int it = 0; it < kPasses; ++it)
#pragma unroll
          for (int hh = 0; hh < kHalves; ++hh)
            cp_async16(dv + hh * kRegion + it * kRowsPerPass * 128, vbc + size_t(uint32_t(ids[it])) * D + hh * 64, true);
        cp_async_arrive_noinc(v_full + s);
      } else {
#pragma unroll
        for (int it = 0; it < kPasses; ++it) {
          const bool listed = i * 128 + it * kRowsPerPass + r0 < nkv;
          if (uint32_t(ids[it]) >= uint32_t(p.N)) {
            if (listed) raise_status(st, kStatusBounds);
            ids[it] = -1;
          }
        }
#pragma unroll
        for (int it = 0; it < kPasses; ++it)
#pragma unroll
          for (int hh = 0; hh < kHalves; ++hh)
            cp_async16(dk + hh * kRegion + it * kRowsPerPass * 128,
                       kbc + size_t(ids[it] < 0 ? 0 : ids[it]) * D + hh * 64, ids[it] >= 0);
        cp_async_arrive_noinc(k_full + s);
#pragma unroll
        for (int it = 0; it < kPasses; ++it)
#pragma unroll
          for (int hh = 0; hh < kHalves; ++hh)
            cp_async16(dv + hh * kRegion + it * kRowsPerPass * 128,
                       vbc + size_t(ids[it] < 0 ? 0 : ids[it]) * D + hh * 64, ids[it] >= 0);
        cp_async_arrive_noinc(v_full + s);
      }
      return true;
    };
    bool ok = true;
    for (int i = 0; ok && i < T; i += 2) {
      ok = tile(i, ida, idb);
      if (ok && i + 1 < T) ok = tile(i + 1, idb, ida);
    }
    // idle: warm L2 with this group's residual rows and the first rows of the
    // group starting about one SM count later (hints; addresses checked first)
    if (ok) {
      const int r = t >> 1, hh = t & 1;
      if (kEpi != kEpiPlain && hh < kHalves && r < p.C && (!kQ64 || r < 64)) {
        const int tq = __ldg(p.perm + size_t(bh) * p.N_pad + size_t(g) * p.C + r);
        if (tq >= 0 && tq < p.N)
          asm volatile("prefetch.global.L2 [%0];" ::"l"(p.res_in + (size_t(bh) * p.N + tq) * D + hh * 64));
      }
      uint32_t nsm;
      asm("mov.u32 %0, %%nsmid;" : "=r"(nsm));
      const long long nxt = (long long)bh * p.G + g + nsm;
      if (nxt < (long long)p.BH * p.G && hh < kHalves && r < 128) {
        const int bh2 = int(nxt / p.G), g2 = int(nxt % p.G);
        const int32_t* permg2 = p.perm + size_t(bh2) * p.N_pad + size_t(g2) * p.C;
        const int32_t* idx2 = p.idx + (size_t(bh2) * p.G + g2) * size_t(p.K);
        const int tq = r < p.C ? __ldg(permg2 + r) : -1;
        const int tk = r < p.K ? __ldg(idx2 + r) : -1;
        if (tq >= 0 && tq < p.N)
          asm volatile("prefetch.global.L2 [%0];" ::"l"(p.q + (size_t(bh2) * p.N + tq) * D + hh * 64));
        if (tk >= 0 && tk < p.N) {
          asm volatile("prefetch.global.L2 [%0];" ::"l"(p.k + (size_t(bh2) * p.N + tk) * D + hh * 64));
          asm volatile("prefetch.global.L2 [%0];" ::"l"(p.v + (size_t(bh2) * p.N + tk) * D + hh * 64));
        }
      }
    }
    asm volatile("cp.async.wait_all;" ::: "memory");
  } else {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kCsRegMma));
    // ------------------------------------------------------------ MMA issuers (warps 16, 17)
    if ((warp == kCsMmaWarp || warp == kCsPvWarp) && lane == 0) {
      const bool pv_thread = warp == kCsPvWarp;
      constexpr uint32_t kIdescQK = idesc_bf16_f32(128, 128, 0, 0);
      constexpr uint32_t kIdescPV = idesc_bf16_f32(128, D, 0, 1);
      bool ok = mbar_wait(q_full, 0, st);
      bool issued = false;
      if (ok) {
        fence_proxy_async_smem();
        tc_fence_after();
      }
      const uint32_t qlo = desc_lo_kmajor(sbase + L::kQ);
      if (!pv_thread) {
        // S chain: S_j = Q K_j^T into S buffer j % 2 once the P V of tile j-2 (whose P
        // sat in that buffer) is done
        for (int j = 0; ok && j < T; ++j) {
          const int s = j % SK, b = j & 1;
          ok = mbar_wait(k_full + s, uint32_t(j / SK) & 1, st) && mbar_wait(pv_done + b, (uint32_t(j >> 1) & 1) ^ 1, st);
          if (!ok) break;
          fence_proxy_async_smem();
          tc_fence_after();
          const uint32_t klo = desc_lo_kmajor(sbase + L::kK + s * L::kTile);
#pragma unroll
          for (int ks = 0; ks < D / 16; ++ks)
            tc_mma_ss_lo(tmem + uint32_t(b * 128), qlo + kstep_kmajor(ks), klo + kstep_kmajor(ks), kIdescQK,
                         ks > 0 ? 1u : 0u);
          tc_commit(s_full + b);
          tc_commit(k_empty + s);
          issued = true;
        }
      } else {
        // P V chains: O_a += P[:, keys 0-63] V[keys 0-63], O_b += P[:, keys 64-127] V[keys 64-127],
        // P read from the S buffer it was written over
        const uint32_t tOa = tmem + L::kColOa, tOb = tmem + L::kColOb;
        for (int j = 0; ok && j < T; ++j) {
          const int s = j % SV, b = j & 1;
          ok = mbar_wait(p_full + b, uint32_t(j >> 1) & 1, st) && mbar_wait(v_full + s, uint32_t(j / SV) & 1, st);
          if (!ok) break;
          fence_proxy_async_smem();
          tc_fence_after();
          const uint32_t vlo = desc_lo_mnmajor(sbase + L::kV + s * L::kTile);
          const uint32_t tP = tmem + uint32_t(b * 128);
          // 16-key slice s of a chain: its P sits over the S columns of its keys
          // (kQ64: warpgroup 0 holds keys 0-31 and 64-95, warpgroup 1 keys 32-63 and 96-127)
#pragma unroll
          for (int ks = 0; ks < 4; ++ks) {
            const int sa = kQ64 ? (ks < 2 ? ks : ks + 2) : ks;
            tc_mma_ts_lo(tOa, tP + (kQ64 ? 8 * sa + (sa >= 4 ? 32 : 0) : 8 * sa), vlo + kstep_mnmajor(sa), kIdescPV,
                         (j > 0 || ks > 0) ? 1u : 0u);
          }
#pragma unroll
          for (int ks = 0; ks < 4; ++ks) {
            const int sb = kQ64 ? (ks < 2 ? ks + 2 : ks + 4) : ks + 4;
            tc_mma_ts_lo(tOb, tP + (kQ64 ? 8 * sb + (sb >= 4 ? 48 : 16) : 8 * sb + 32), vlo + kstep_mnmajor(sb),
                         kIdescPV, (j > 0 || ks > 0) ? 1u : 0u);
          }
          tc_commit(pv_done + b);
          tc_commit(v_empty + s);
          issued = true;
        }
        if (ok) tc_commit(o_done);
      }
      if (!ok) {
        raise_status(st, kStatusTimeout);
        if (issued) {
          tc_commit(drain + (pv_thread ? 1 : 0));
          mbar_wait(drain + (pv_thread ? 1 : 0), 0, st);
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == kCsMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

template <int D, int kEpi, bool kQ64>
cudaError_t launch_sparse_cs(const TcAttnParams& p, cudaStream_t stream) {
  using L = CsCfg<D>;
  static_assert(4096 + 64 * D * 4 <= L::kSK * L::kTile, "the four-way merge fits the key ring");
  auto kern = attn_sparse_cs_kernel<D, kEpi, kQ64>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, L::kAlloc);
  if (e != cudaSuccess) return e;
  cudaFuncAttributes fa;
  if ((e = cudaFuncGetAttributes(&fa, kern)) != cudaSuccess) return e;
  if (fa.numRegs * kCsThreads < kCsRegPool || fa.numRegs < kCsRegGather) return cudaErrorInvalidValue;
  dim3 grid(p.tiles_per_head, p.BH);
  kern<<<grid, kCsThreads, L::kAlloc, stream>>>(p);
  note_launches(1);
  return cudaGetLastError();
}

}  // namespace

cudaError_t tc_sparse_attn(int D, int epi, const TcAttnParams& p, int BH, cudaStream_t stream) {
  (void)BH;
  // groups of more than 64 queries: two softmax warpgroups per row; of at most
  // 64: two lanes per query
#define MCS_SPARSE_CASE(DD, EE)                                          \
  if (D == DD && epi == EE)                                              \
    return p.C <= 64 ? launch_sparse_cs<DD, EE, true>(p, stream) : launch_sparse_cs<DD, EE, false>(p, stream);
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
