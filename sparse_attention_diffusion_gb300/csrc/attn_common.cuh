// Softmax and epilogue of the tcgen05 attention kernels. The dense kernel runs
// one thread per query row (warps 0-3), the sparse kernel two warpgroups that
// split every tile's keys (two or four threads per query); a thread always works
// on the TMEM lane its row's accumulators live on.
#pragma once
#include <cuda_bf16.h>

#include "common.cuh"
#include "ptx.cuh"
#include "tc_common.cuh"

namespace mcs {

struct SoftmaxSync {
  uint64_t* s_full;   // [2] S buffer b written by the MMA
  uint64_t* s_free;   // [2] S buffer b read (128 arrivals)
  uint64_t* p_full;   // P written to TMEM (128 arrivals)
  uint64_t* p_empty;  // PV of the previous tile done (O stable, P free)
};

// Online base-2 softmax over T tiles of 128 keys (nkv keys in all). For tile j:
// load the S row from TMEM buffer j%2, update the running max m (log2 units,
// rescaled lazily: only when the max grows by more than 2^8) and the running sum
// l, write P = 2^(s*scale_log2 - m) to TMEM as bf16 pairs and, when the max
// moved, rescale the O accumulator row in TMEM. The exponentials are computed
// before waiting for the previous PV so they overlap it.
// Returns false if a bounded wait ran out.
template <int D, bool kPV>
__device__ __forceinline__ bool softmax_rows(int T, int nkv, uint32_t tS, uint32_t tO, uint32_t tP, uint32_t lane_off,
                                             float sl2, const SoftmaxSync& sy, const uint32_t* st, float& m_out,
                                             float& l_out) {
  float m = -INFINITY, l = 0.f;
  bool ok = true;
  for (int j = 0; j < T; ++j) {
    const int b = j & 1;
    const uint32_t ub = uint32_t(j >> 1);
    ok = warp_all(mbar_wait(sy.s_full + b, ub & 1, st));
    if (!ok) break;
    tc_fence_after();
    uint32_t r[128];
    tmem_ld128(tS + lane_off + b * 128, r);
    tc_fence_before();
    mbar_arrive(sy.s_free + b);
    const int nvalid = min(128, nkv - j * 128);
    if (nvalid < 128) {  // last, partial tile: logits of missing keys become -inf (p = 0)
#pragma unroll
      for (int c = 0; c < 128; ++c)
        if (c >= nvalid) r[c] = __float_as_uint(-INFINITY);
    }
    // independent partial maxima and sums: one warp per scheduler runs this, so
    // a single dependent chain of 128 max / 64 add operations would be pure latency
    float mp[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) mp[i] = __uint_as_float(r[i]);
#pragma unroll
    for (int c = 8; c < 128; c += 2) mp[(c >> 1) & 7] = fmax3(mp[(c >> 1) & 7], __uint_as_float(r[c]), __uint_as_float(r[c + 1]));
    const float mx = fmax3(fmax3(mp[0], mp[1], mp[2]), fmax3(mp[3], mp[4], mp[5]), fmaxf(mp[6], mp[7]));
    const float m_new = fmaxf(m, mx * sl2);
    const bool need = m_new > m + 8.f;
    const float m_use = need ? m_new : m;
    const float alpha = need ? ex2_approx(m - m_new) : 1.f;
    const float neg_m = -m_use;
    // two scores per packed FMA and two packed partial sums (four lanes)
    const uint64_t sl2x2 = f2_pack(sl2, sl2), negmx2 = f2_pack(neg_m, neg_m);
    uint64_t ls2[2] = {f2_pack(0.f, 0.f), f2_pack(0.f, 0.f)};
    uint32_t pk[64];
#pragma unroll
    for (int c = 0; c < 64; ++c) {
      float x0, x1;
      f2_unpack(f2_fma(f2_pack(__uint_as_float(r[2 * c]), __uint_as_float(r[2 * c + 1])), sl2x2, negmx2), x0, x1);
      const float p0 = ex2_approx(x0), p1 = ex2_approx(x1);
      ls2[c & 1] = f2_add(ls2[c & 1], f2_pack(p0, p1));
      pk[c] = pack_bf16x2(p0, p1);
    }
    float la, lb;
    f2_unpack(f2_add(ls2[0], ls2[1]), la, lb);
    const float lsum = la + lb;
    l = l * alpha + lsum;
    m = m_use;
    if constexpr (kPV) {
      ok = warp_all(mbar_wait(sy.p_empty, (uint32_t(j) & 1) ^ 1, st));  // PV of tile j-1 done
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
      mbar_arrive(sy.p_full);
    }
  }
  m_out = m;
  l_out = l;
  return ok;
}

// Epilogue for one row: O / l from TMEM, optionally plus (add-residual) or
// subtracted from (store-residual) a bf16 row, rounded once to bf16 and stored.
// Every thread of the warp must call it (the TMEM loads are warp-collective);
// rows with tok < 0 load but store nothing.
template <int D, int kEpi>
__device__ __forceinline__ void store_row(uint32_t tO, uint32_t lane_off, int tok, size_t rowoff, float inv_l,
                                          __nv_bfloat16* dst, const __nv_bfloat16* res_in) {
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
          const uint4 rv = *reinterpret_cast<const uint4*>(res_in + off);
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

// Column-split softmax: two threads (two warpgroups) share a tensor-memory lane,
// thread h taking keys [64h, 64h + 64) of every tile (col0 = 64h) with its own running
// max m and sum l and its own O accumulator row (tO). P is written as bf16 pairs
// over the S columns this thread has just read (columns b*128 + col0 ...), so S
// buffer b is free again once the P V of its tile is done (pv_done[b]); no other
// wait sits on the path to P. P of a tile in buffer b is announced on
// p_full[b], which therefore never runs more than one phase ahead of the P V
// thread's wait (its next phase needs S in buffer b again, behind that P V).
// The O row is rescaled only when the max grows by more than 2^8, after the
// previous tile's P V is done. A part of a row may see no key at all (m stays
// -inf, l 0, P 0). kW = 32 (64-query groups, four threads per query) reads 32
// columns from col0 and also zeroes the 16 P columns at zcol of its lane that
// its P V chain reads for the keys of the query's other lane.
// Returns false if a bounded wait ran out.
template <int D, int kW = 64>
__device__ __forceinline__ bool softmax_rows_cs(int T, int nkv, uint32_t tS, uint32_t tO, uint32_t lane_off, int col0,
                                                float sl2, uint64_t* s_full, uint64_t* pv_done, uint64_t* p_full,
                                                const uint32_t* st, float& m_out, float& l_out, int zcol = -1) {
  static_assert(kW == 64 || kW == 32, "a thread reads half or a quarter of a tile");
  float m = -INFINITY, l = 0.f;
  bool ok = true;
  for (int j = 0; j < T; ++j) {
    const int b = j & 1;
    ok = warp_all(mbar_wait(s_full + b, uint32_t(j >> 1) & 1, st));
    if (!ok) break;
    tc_fence_after();
    const uint32_t tSb = tS + lane_off + uint32_t(b * 128 + col0);
    uint32_t r[kW];
    if constexpr (kW == 64) tmem_ld64(tSb, r);
    else tmem_ld32(tSb, r);
    const int nvalid = min(kW, nkv - j * 128 - col0);
    if (nvalid < kW) {  // last, partial tile: logits of missing keys become -inf (p = 0)
#pragma unroll
      for (int c = 0; c < kW; ++c)
        if (c >= nvalid) r[c] = __float_as_uint(-INFINITY);
    }
    float mp[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) mp[i] = __uint_as_float(r[i]);
#pragma unroll
    for (int c = 8; c < kW; c += 2) mp[(c >> 1) & 7] = fmax3(mp[(c >> 1) & 7], __uint_as_float(r[c]), __uint_as_float(r[c + 1]));
    const float mx = fmax3(fmax3(mp[0], mp[1], mp[2]), fmax3(mp[3], mp[4], mp[5]), fmaxf(mp[6], mp[7]));
    const float m_new = fmaxf(m, mx * sl2);
    const bool need = m_new > m + 8.f;
    const float m_use = need ? m_new : m;
    const float alpha = need ? ex2_approx(m - m_new) : 1.f;
    const float neg_m = m_use == -INFINITY ? 0.f : -m_use;
    const uint64_t sl2x2 = f2_pack(sl2, sl2), negmx2 = f2_pack(neg_m, neg_m);
    uint64_t ls2[2] = {f2_pack(0.f, 0.f), f2_pack(0.f, 0.f)};
    uint32_t pk[kW / 2];
#pragma unroll
    for (int c = 0; c < kW / 2; ++c) {
      float x0, x1;
      f2_unpack(f2_fma(f2_pack(__uint_as_float(r[2 * c]), __uint_as_float(r[2 * c + 1])), sl2x2, negmx2), x0, x1);
      const float p0 = ex2_approx(x0), p1 = ex2_approx(x1);
      ls2[c & 1] = f2_add(ls2[c & 1], f2_pack(p0, p1));
      pk[c] = pack_bf16x2(p0, p1);
    }
    float la, lb;
    f2_unpack(f2_add(ls2[0], ls2[1]), la, lb);
    l = l * alpha + (la + lb);
    m = m_use;
    if (__any_sync(0xffffffffu, need && j > 0)) {
      // the previous tile's P V accumulates into this O row: let it finish first
      ok = warp_all(mbar_wait(pv_done + ((j - 1) & 1), uint32_t((j - 1) >> 1) & 1, st));
      if (!ok) break;
      tc_fence_after();
#pragma unroll
      for (int c = 0; c < D / 32; ++c) {
        uint32_t o[32];
        tmem_ld32(tO + lane_off + c * 32, o);
#pragma unroll
        for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha);
        tmem_st32(tO + lane_off + c * 32, o);
      }
    }
    if constexpr (kW == 64) {
      tmem_st32(tSb, pk);
    } else {
      // this lane's P columns of the other lane-half's keys must read as zero for
      // the P V chain this thread feeds (they hold S values otherwise)
      tmem_st16(tSb, pk);
      uint32_t z[16];
#pragma unroll
      for (int i = 0; i < 16; ++i) z[i] = 0u;
      tmem_st16(tS + lane_off + uint32_t(b * 128 + zcol), z);
    }
    tc_fence_before();
    mbar_arrive(p_full + b);
  }
  m_out = m;
  l_out = l;
  return ok;
}

// Epilogue of the column-split form: output columns [c0, c0 + D/2) of one row,
// o_a * fa + o_b * fb from the two accumulators (fa, fb: each half's weight
// 2^(m_half - m) times 1 / l), plus (add-residual) or subtracted from
// (store-residual) this half of the bf16 row held in rres, rounded once and
// stored. Every thread of the warp must call it (the TMEM loads are
// warp-collective); rows with tok < 0 load but store nothing.
template <int D, int kEpi>
__device__ __forceinline__ void store_row_cs(uint32_t tOa, uint32_t tOb, uint32_t lane_off, int c0, int tok,
                                             size_t rowoff, float fa, float fb, __nv_bfloat16* dst,
                                             const uint4 (&rres)[D / 16]) {
#pragma unroll
  for (int c = 0; c < D / 64; ++c) {
    uint32_t a[32], b[32];
    tmem_ld32(tOa + lane_off + c0 + c * 32, a);
    tmem_ld32(tOb + lane_off + c0 + c * 32, b);
    if (tok >= 0 && dst != nullptr) {
#pragma unroll
      for (int q4 = 0; q4 < 4; ++q4) {
        float o8[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) o8[i] = __uint_as_float(a[q4 * 8 + i]) * fa + __uint_as_float(b[q4 * 8 + i]) * fb;
        const size_t off = rowoff + c0 + c * 32 + q4 * 8;
        if constexpr (kEpi != kEpiPlain) {
          const uint4 rv = rres[c * 4 + q4];
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

// Epilogue pieces of the four-way split (64-query groups: query q on lanes q and
// q + 64, each lane shared by both warpgroups, four partial rows per query): a
// lane 64-127 thread leaves its two accumulators' weighted sum for output columns
// [c0, c0 + D/2) in shared memory (float4 k at xo[k * 64]); the lane q thread adds
// its own two, the partial from shared memory, scales by 1 / l, adds or subtracts
// the residual and stores. Every thread of the warp must call them (the TMEM
// loads are warp-collective).
template <int D>
__device__ __forceinline__ void partial_row_cs4(uint32_t tOa, uint32_t tOb, uint32_t lane_off, int c0, float fa, float fb,
                                                float4* xo) {
#pragma unroll
  for (int c = 0; c < D / 64; ++c) {
    uint32_t a[32], b[32];
    tmem_ld32(tOa + lane_off + c0 + c * 32, a);
    tmem_ld32(tOb + lane_off + c0 + c * 32, b);
#pragma unroll
    for (int k = 0; k < 8; ++k)
      xo[(c * 8 + k) * 64] = make_float4(__uint_as_float(a[4 * k]) * fa + __uint_as_float(b[4 * k]) * fb,
                                         __uint_as_float(a[4 * k + 1]) * fa + __uint_as_float(b[4 * k + 1]) * fb,
                                         __uint_as_float(a[4 * k + 2]) * fa + __uint_as_float(b[4 * k + 2]) * fb,
                                         __uint_as_float(a[4 * k + 3]) * fa + __uint_as_float(b[4 * k + 3]) * fb);
  }
}
template <int D, int kEpi>
__device__ __forceinline__ void store_row_cs4(uint32_t tOa, uint32_t tOb, uint32_t lane_off, int c0, int tok,
                                              size_t rowoff, float fa, float fb, float inv, const float4* xo,
                                              __nv_bfloat16* dst, const uint4 (&rres)[D / 16]) {
#pragma unroll
  for (int c = 0; c < D / 64; ++c) {
    uint32_t a[32], b[32];
    tmem_ld32(tOa + lane_off + c0 + c * 32, a);
    tmem_ld32(tOb + lane_off + c0 + c * 32, b);
    if (tok >= 0 && dst != nullptr) {
#pragma unroll
      for (int q4 = 0; q4 < 4; ++q4) {
        const float4 x0 = xo[(c * 8 + q4 * 2) * 64], x1 = xo[(c * 8 + q4 * 2 + 1) * 64];
        const float y[8] = {x0.x, x0.y, x0.z, x0.w, x1.x, x1.y, x1.z, x1.w};
        float o8[8];
#pragma unroll
        for (int i = 0; i < 8; ++i)
          o8[i] = (__uint_as_float(a[q4 * 8 + i]) * fa + __uint_as_float(b[q4 * 8 + i]) * fb + y[i]) * inv;
        const size_t off = rowoff + c0 + c * 32 + q4 * 8;
        if constexpr (kEpi != kEpiPlain) {
          const uint4 rv = rres[c * 4 + q4];
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

}  // namespace mcs
