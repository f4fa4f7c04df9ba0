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
// S_{j+1} runs; one thread issues the S chain and another the P V chain; every
// query row is shared by two softmax threads, each taking one half of every
// tile's keys with its own running max, sum and O row, merged in the epilogue.
// Two forms:
//   attn_sparse_cs_kernel (C > 64, 640 threads): two softmax warpgroups on the
//     same tensor-memory lanes, warpgroup h taking keys [64h, 64h + 64) into its
//     own O accumulator and writing its P over the S columns it read; the P V
//     of a tile is two four-MMA chains, and S buffer b is refilled once the P V
//     of its tile is done. The two threads of a row each store half of the
//     output columns;
//   attn_sparse_kernel (C <= 64, 512 threads): one softmax warpgroup; query r
//     sits on lanes r and r + 64 (the gather copies its row into both rows of
//     the query tile), lane r taking keys 0-63 and lane r + 64 keys 64-127 of
//     every tile, with P in its own columns (the other half's P columns stay
//     zero); lanes 64-127 hand their O rows to lanes 0-63 through shared memory.
// In both, eight gather warps copy the group's query rows (through perm) once,
// then per tile the key and value rows at the group's index list, as 16-byte
// cp.async copies into 3-stage K and V rings (6 stages at d = 64; 128-byte
// swizzled); eight threads per row, each copying one chunk of every 128-byte
// half, so a thread holds 4 row ids per tile; once idle they prefetch into L2
// the group's residual rows and the first rows of the group starting about one
// SM count later. The gather warps never wait for their own copies: each thread
// ends a tile's key (value) copies with an asynchronous arrive on the stage's
// full barrier, which completes when every thread's rows have landed; the
// issuing threads then fence the generic-to-async proxy before the tensor core
// reads them. The gather warps only wait (through one leader and a named
// barrier) for the stages to be released: a K stage when S of its tile is done,
// a V stage when P V is done. Each gather thread reads its row indices for the
// next tile into registers while the leader waits, and issues a tile's copies
// back to back. The epilogue's residual row is loaded while the last P V runs.
// Registers are rebalanced with setmaxnreg; each launcher checks that the split
// fits the registers the block is launched with. All waits are bounded; on a
// timeout the CTA flags it, lets its copies and MMAs land, frees tensor memory
// and returns.
#include "attn_common.cuh"
#include "attn_tc.h"
#include "common.cuh"
#include "ptx.cuh"
#include "tc_common.cuh"

namespace mcs {
namespace {

// ---------------------------------------------------------------- two lanes per query (C <= 64)
// warpgroup 0 softmax and epilogue, 1-2 gather, warp 12 tensor-memory
// allocation and the S chain, warp 13 the P V chain. Tensor memory: S0 [0, 128),
// S1 [128, 256), O [256, 256 + D), P [384, 448).
constexpr int kSparseThreads = 512;
constexpr int kGather = 256;   // gather threads (warpgroups 1-2)
constexpr int kMmaWarp = 12;   // first warp of warpgroup 3: TMEM allocation and the S chain
constexpr int kPvWarp = 13;    // the P V chain
constexpr int kRegSoftmax = 240, kRegGather = 48, kRegMma = 32;  // the merge epilogue spills below 240
constexpr int kRegPool = 128 * kRegSoftmax + kGather * kRegGather + 128 * kRegMma;

template <int D>
struct SparseCfg {
  static constexpr int kSK = D == 64 ? 6 : 3, kSV = kSK;  // K and V stages (equal: tile i's key and value rows go together)
  static constexpr int kTile = (D / 64) * kRegion;
  static constexpr int kQ = 0;
  static constexpr int kK = kQ + kTile;
  static constexpr int kV = kK + kSK * kTile;
  static constexpr int kBar = kV + kSV * kTile;
  static constexpr int kNumBars = 1 + 2 * kSK + 2 * kSV + 2 + 2 + 1 + 1 + 1 + 2;
  static constexpr int kMisc = kBar + kNumBars * 8;  // tmem slot, stop flags [2]
  static constexpr int kBytes = kMisc + 32;
  static constexpr int kAlloc = kBytes + 1024;
  static constexpr uint32_t kColO = 256, kColP = 384;  // S0, S1 at 0 and 128
  static_assert(kAlloc <= 227 * 1024, "shared memory");
};

template <int D, int kEpi>
__global__ void __launch_bounds__(kSparseThreads, 1) attn_sparse_kernel(const TcAttnParams p) {
  using L = SparseCfg<D>;
  constexpr int SK = L::kSK, SV = L::kSV;
  static_assert(SK == SV, "one stage index for tile i's key and value rows");
  // gather mapping: a thread copies 16-byte chunk ch of the row's first 64
  // elements and chunk ch of the next 64 (d = 128: two 128-byte halves, each
  // copy instruction reading whole 128-byte segments), 8 threads per row
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
  uint64_t* s_full = v_empty + SV;  // [2] S buffer b written
  uint64_t* s_free = s_full + 2;    // [2] S buffer b read by the softmax
  uint64_t* p_full = s_free + 2;    // P_j written
  uint64_t* p_empty = p_full + 1;   // P_j V_j done (P free, O stable)
  uint64_t* o_done = p_empty + 1;
  uint64_t* drain = o_done + 1;     // [2] one per issuing thread
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::kMisc);
  // the gather leader's decision for iteration i lives in stop[i & 1]: a slow
  // reader of iteration i never sees the leader's write for iteration i + 1
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
      mbar_init(s_free + b, 128);
    }
    mbar_init(p_full, 128);
    mbar_init(p_empty, 1);
    mbar_init(o_done, 2);  // one commit from each issuing thread
    mbar_init(drain, 1);
    mbar_init(drain + 1, 1);
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
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kRegSoftmax));
    // ------------------------------------------------------------ softmax, epilogue
    // Query row r sits on lanes r and r + 64; lane r takes keys 0-63 of every
    // tile and lane r + 64 keys 64-127, each with its own running max, sum and O
    // row, merged in the epilogue. half is warp-uniform.
    const int row = tid;
    const int half = row >> 6;
    const int qrow = row & 63;
    const uint32_t lane_off = uint32_t(warp * 32) << 16;
    int tok = -1;
    if (qrow < p.C) {
      const int v = __ldg(p.perm + size_t(bh) * p.N_pad + size_t(g) * p.C + qrow);
      if (v < 0 || v >= p.N_pad) raise_status(st, kStatusBounds);
      else if (v < p.N) tok = v;
    }
    if (half) tok = -1;  // lane r + 64 hands its partial row to lane r
    float m, l;
    const SoftmaxSync sy{s_full, s_free, p_full, p_empty};
    {  // the other half's P columns stay zero for the whole group
      uint32_t z[32];
#pragma unroll
      for (int i = 0; i < 32; ++i) z[i] = 0u;
      tmem_st32(tmem + L::kColP + lane_off + uint32_t(32 - half * 32), z);
    }
    bool ok = softmax_rows<D, true, 64>(T, nkv, tmem, tmem + L::kColO, tmem + L::kColP, lane_off, p.scale_log2, sy,
                                        st, m, l, half * 64);
    // the row's residual (or O_dense), loaded while the last P V runs
    uint4 rres[D / 8] = {};
    if constexpr (kEpi != kEpiPlain) {
      if (tok >= 0) {
        const uint4* src = reinterpret_cast<const uint4*>(p.res_in + (size_t(bh) * p.N + size_t(tok)) * D);
#pragma unroll
        for (int i = 0; i < D / 8; ++i) rres[i] = src[i];
      }
    }
    if (ok) ok = warp_all(mbar_wait(o_done, 0, st));
    __nv_bfloat16* dst = (kEpi == kEpiStoreResidual) ? p.res_out : p.o;
    const size_t rowoff = (size_t(bh) * p.N + size_t(tok < 0 ? 0 : tok)) * D;
    {
      // Every tile has landed and every MMA is done (o_done), so the key ring's
      // shared memory is free: lanes 64-127 leave their O rows there (float4 k of
      // row r at k * 64 + r) with their max and sum; all 128 threads meet at the
      // named barrier whatever their wait status.
      float4* xo = reinterpret_cast<float4*>(smem + L::kK);
      float* xm = reinterpret_cast<float*>(smem + L::kK + 64 * D * 4);
      if (half) {
        if (ok) {
          tc_fence_after();
#pragma unroll
          for (int c = 0; c < D / 32; ++c) {
            uint32_t o[32];
            tmem_ld32(tmem + L::kColO + lane_off + c * 32, o);
#pragma unroll
            for (int k = 0; k < 8; ++k)
              xo[(c * 8 + k) * 64 + qrow] = make_float4(__uint_as_float(o[4 * k]), __uint_as_float(o[4 * k + 1]),
                                                        __uint_as_float(o[4 * k + 2]), __uint_as_float(o[4 * k + 3]));
          }
        }
        xm[qrow] = m;
        xm[64 + qrow] = l;
      }
      named_bar_sync(2, 128);
      if (!half && ok) {
        tc_fence_after();
        const float m1 = xm[qrow], l1 = xm[64 + qrow];
        const float mm = fmaxf(m, m1);
        const float a0 = m == -INFINITY ? 0.f : ex2_approx(m - mm);
        const float a1 = m1 == -INFINITY ? 0.f : ex2_approx(m1 - mm);
        const float inv = 1.f / (l * a0 + l1 * a1);
        store_row_pair<D, kEpi>(tmem + L::kColO, lane_off, tok, rowoff, a0 * inv, a1 * inv, xo + qrow, dst, rres);
      }
    }
    if (!ok && row == 0) raise_status(st, kStatusTimeout);
  } else if (warp < 12) {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kRegGather));
    // ------------------------------------------------------------ gather warps
    const int t = tid - 128;  // 0..255
    const int ch = t % kChunks, r0 = t / kChunks;
    const __nv_bfloat16* kb = p.k + size_t(bh) * p.N * D;
    const __nv_bfloat16* vb = p.v + size_t(bh) * p.N * D;
    // This thread's key ids of tile i (its rows r0 + k * kRowsPerPass), -1 past
    // the end of the list; read one tile ahead, so the loads complete while the
    // leader waits for the stages.
    auto load_ids = [&](int i, int (&ids)[kPasses]) {
#pragma unroll
      for (int it = 0; it < kPasses; ++it) {
        const int slot = i * 128 + it * kRowsPerPass + r0;
        ids[it] = slot < nkv ? __ldg(idxg + slot) : -1;
      }
    };
    int ida[kPasses], idb[kPasses];  // ids of even / odd tiles (no copies between them)
    load_ids(0, ida);  // tile 0's ids first: their loads overlap the query rows' copies
    {  // the group's query rows (through perm): operand A of S = Q K^T
      const __nv_bfloat16* qb = p.q + size_t(bh) * p.N * D;
      const int32_t* permg = p.perm + size_t(bh) * p.N_pad + size_t(g) * p.C;
#pragma unroll 4
      for (int it = 0; it < kPasses; ++it) {
        const int row = it * kRowsPerPass + r0;
        const int qr = row & 63;  // rows r and r + 64 hold the same query
        int tq = -1;
        if (qr < p.C) {
          const int v = __ldg(permg + qr);
          if (v < 0 || v >= p.N_pad) raise_status(st, kStatusBounds);
          else if (v < p.N) tq = v;
        }
#pragma unroll
        for (int h = 0; h < kHalves; ++h)
          cp_async16(sbase + L::kQ + h * kRegion + sw128_off(row, ch), qb + size_t(tq < 0 ? 0 : tq) * D + h * 64 + ch * 8,
                     tq >= 0);
      }
      cp_async_arrive_noinc(q_full);
    }
    static_assert(kRowsPerPass % 8 == 0, "a thread's rows share one swizzle phase");
    const uint32_t doff = sw128_off(r0, ch);  // + it * kRowsPerPass * 128 for pass it
    const __nv_bfloat16* kbc = kb + ch * 8;
    const __nv_bfloat16* vbc = vb + ch * 8;
    // one tile: wait for its stages, then key and value copies, each ended by an
    // asynchronous arrive on the stage's full barrier. Listed ids outside [0, N)
    // raise the bounds flag; they and the unlisted slots of the last tile read zeros.
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
          for (int h = 0; h < kHalves; ++h)
            cp_async16(dk + h * kRegion + it * kRowsPerPass * 128, kbc + size_t(uint32_t(ids[it])) * D + h * 64, true);
        cp_async_arrive_noinc(k_full + s);
#pragma unroll
        for (int it = 0; it < kPasses; ++it)
#pragma unroll
          for (int h = 0; h < kHalves; ++h)
            cp_async16(dv + h * kRegion + it * kRowsPerPass * 128, vbc + size_t(uint32_t(ids[it])) * D + h * 64, true);
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
          for (int h = 0; h < kHalves; ++h)
            cp_async16(dk + h * kRegion + it * kRowsPerPass * 128, kbc + size_t(ids[it] < 0 ? 0 : ids[it]) * D + h * 64,
                       ids[it] >= 0);
        cp_async_arrive_noinc(k_full + s);
#pragma unroll
        for (int it = 0; it < kPasses; ++it)
#pragma unroll
          for (int h = 0; h < kHalves; ++h)
            cp_async16(dv + h * kRegion + it * kRowsPerPass * 128, vbc + size_t(ids[it] < 0 ? 0 : ids[it]) * D + h * 64,
                       ids[it] >= 0);
        cp_async_arrive_noinc(v_full + s);
      }
      return true;
    };
    bool ok = true;
    for (int i = 0; ok && i < T; i += 2) {
      ok = tile(i, ida, idb);
      if (ok && i + 1 < T) ok = tile(i + 1, idb, ida);
    }
    // Idle from here on, a few tiles before the epilogue: warm L2 with this
    // group's residual (or O_dense) rows, which the epilogue reads, and with the
    // first rows of the group whose CTA starts about one SM count later (its query
    // rows through perm, the key and value rows of its first tile through its
    // index list). Prefetches are hints: no data is read into the CTA and every
    // address is checked first.
    if (ok && kEpi != kEpiPlain) {
      const int r = t >> 1, hh = t & 1;  // query row r of the group, 128-byte half hh
      const int qr = r;
      if (hh < kHalves && r < 64 && qr < p.C) {
        const int tq = __ldg(p.perm + size_t(bh) * p.N_pad + size_t(g) * p.C + qr);
        if (tq >= 0 && tq < p.N)
          asm volatile("prefetch.global.L2 [%0];" ::"l"(p.res_in + (size_t(bh) * p.N + tq) * D + hh * 64));
      }
    }
    if (ok) {
      uint32_t nsm;
      asm("mov.u32 %0, %%nsmid;" : "=r"(nsm));
      const long long nxt = (long long)bh * p.G + g + nsm;
      if (nxt < (long long)p.BH * p.G) {
        const int bh2 = int(nxt / p.G), g2 = int(nxt % p.G);
        const int r = t >> 1, hh = t & 1;
        if (hh < kHalves && r < 128) {
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
    }
    // let every copy land before the CTA can exit (normally long done)
    asm volatile("cp.async.wait_all;" ::: "memory");
    (void)ok;
  } else {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kRegMma));
    // ------------------------------------------------------------ MMA issuers (warps 12, 13)
    // Lane 0 of each runs its chain's schedule alone: its waits, MMAs and commits
    // (the other lanes go straight to the final barrier). Each thread's commits
    // cover only its own MMAs, so o_done expects one commit from each, and each
    // has its own drain barrier.
    if ((warp == kMmaWarp || warp == kPvWarp) && lane == 0) {
      const bool pv_thread = warp == kPvWarp;
      constexpr uint32_t kIdescQK = idesc_bf16_f32(128, 128, 0, 0);
      constexpr uint32_t kIdescPV = idesc_bf16_f32(128, D, 0, 1);
      bool ok = mbar_wait(q_full, 0, st);
      bool issued = false;
      if (ok) {
        fence_proxy_async_smem();  // rows written by the gather warps' cp.async copies
        tc_fence_after();
      }
      const uint32_t qlo = desc_lo_kmajor(sbase + L::kQ);
      if (!pv_thread) {
        // S chain: S_j = Q K_j^T into S buffer j % 2 once the softmax has read S_{j-2}
        for (int j = 0; ok && j < T; ++j) {
          const int s = j % SK, b = j & 1;
          ok = mbar_wait(k_full + s, uint32_t(j / SK) & 1, st) && mbar_wait(s_free + b, (uint32_t(j >> 1) & 1) ^ 1, st);
          if (!ok) break;
          fence_proxy_async_smem();  // key rows landed by cp.async, read by the tensor core
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
        // P V chain: O += P_j V_j with P from its own tensor-memory columns
        const uint32_t tO = tmem + L::kColO, tP = tmem + L::kColP;
        for (int j = 0; ok && j < T; ++j) {
          const int s = j % SV;
          ok = mbar_wait(p_full, uint32_t(j) & 1, st) && mbar_wait(v_full + s, uint32_t(j / SV) & 1, st);
          if (!ok) break;
          fence_proxy_async_smem();  // value rows landed by cp.async
          tc_fence_after();
          const uint32_t vlo = desc_lo_mnmajor(sbase + L::kV + s * L::kTile);
#pragma unroll
          for (int ks = 0; ks < 8; ++ks)
            tc_mma_ts_lo(tO, tP + ks * 8, vlo + kstep_mnmajor(ks), kIdescPV, (j > 0 || ks > 0) ? 1u : 0u);
          tc_commit(p_empty);
          tc_commit(v_empty + s);
          issued = true;
        }
      }
      if (ok) tc_commit(o_done);
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
  if (warp == kMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

template <int D, int kEpi>
cudaError_t launch_sparse(const TcAttnParams& p, cudaStream_t stream) {
  using L = SparseCfg<D>;
  static_assert(64 * D * 4 + 2 * 64 * 4 <= L::kSK * L::kTile, "the merge buffer fits the key ring");
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

// ---------------------------------------------------------------- column-split form (C > 64)
// Two softmax warpgroups share every query row: warpgroup h takes keys
// [64h, 64h + 64) of each tile with its own running max, sum and O accumulator
// (O_a at column 256, O_b at 384), writing its P over the S columns it has read;
// the P V of a tile is two chains of four MMAs (keys 0-63 into O_a, keys 64-127
// into O_b), and S buffer b is refilled once that P V is done. The epilogue
// merges the two partial rows (each thread stores half of the row's columns).
// 640 threads: warpgroups 0-1 softmax and epilogue, 2-3 gather (as above),
// warp 16 tensor-memory allocation and the S chain, warp 17 the P V chain.
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

template <int D, int kEpi>
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
    const int row = (warp & 3) * 32 + lane;  // query row = tensor-memory lane
    const uint32_t lane_off = uint32_t((warp & 3) * 32) << 16;
    int tok = -1;
    if (row < p.C) {
      const int v = __ldg(p.perm + size_t(bh) * p.N_pad + size_t(g) * p.C + row);
      if (v < 0 || v >= p.N_pad) raise_status(st, kStatusBounds);
      else if (v < p.N) tok = v;
    }
    float m, l;
    bool ok = softmax_rows_cs<D>(T, nkv, tmem, tmem + (h ? L::kColOb : L::kColOa), lane_off, h * 64, p.scale_log2,
                                 s_full, pv_done, p_full, st, m, l);
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
    if (ok) {
      tc_fence_after();
      const float ma = xm[row], mb = xm[128 + row], la = xm[512 + row], lb = xm[640 + row];
      const float mm = fmaxf(ma, mb);
      const float fa = ma == -INFINITY ? 0.f : ex2_approx(ma - mm);
      const float fb = mb == -INFINITY ? 0.f : ex2_approx(mb - mm);
      const float inv = 1.f / (la * fa + lb * fb);
      __nv_bfloat16* dst = (kEpi == kEpiStoreResidual) ? p.res_out : p.o;
      const size_t rowoff = (size_t(bh) * p.N + size_t(tok < 0 ? 0 : tok)) * D;
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
        int tq = -1;
        if (row < p.C) {
          const int v = __ldg(permg + row);
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
      if (kEpi != kEpiPlain && hh < kHalves && r < p.C) {
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
#pragma unroll
          for (int ks = 0; ks < 4; ++ks)
            tc_mma_ts_lo(tOa, tP + ks * 8, vlo + kstep_mnmajor(ks), kIdescPV, (j > 0 || ks > 0) ? 1u : 0u);
#pragma unroll
          for (int ks = 0; ks < 4; ++ks)
            tc_mma_ts_lo(tOb, tP + 64 + ks * 8, vlo + kstep_mnmajor(4 + ks), kIdescPV, (j > 0 || ks > 0) ? 1u : 0u);
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

template <int D, int kEpi>
cudaError_t launch_sparse_cs(const TcAttnParams& p, cudaStream_t stream) {
  using L = CsCfg<D>;
  auto kern = attn_sparse_cs_kernel<D, kEpi>;
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
    return p.C <= 64 ? launch_sparse<DD, EE>(p, stream) : launch_sparse_cs<DD, EE>(p, stream);
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
