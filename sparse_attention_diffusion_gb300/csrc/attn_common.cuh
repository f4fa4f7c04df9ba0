// Softmax and epilogue of the tcgen05 attention kernels (dense and sparse), run
// by warps 0-3: one thread per query row, which is the TMEM lane the row's
// accumulators live on.
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
// kW = 64 takes only keys [col0, col0 + 64) of every tile (S columns col0.., P
// columns col0/2..): two threads share a query row, each with its own running
// max and sum, and a row may then see no key at all (m stays -inf, l 0, P 0).
// Returns false if a bounded wait ran out.
template <int D, bool kPV, int kW = 128>
__device__ __forceinline__ bool softmax_rows(int T, int nkv, uint32_t tS, uint32_t tO, uint32_t tP, uint32_t lane_off,
                                             float sl2, const SoftmaxSync& sy, const uint32_t* st, float& m_out,
                                             float& l_out, int col0 = 0) {
  static_assert(kW == 128 || kW == 64, "a thread reads all 128 columns of a tile or one half");
  float m = -INFINITY, l = 0.f;
  bool ok = true;
  for (int j = 0; j < T; ++j) {
    const int b = j & 1;
    const uint32_t ub = uint32_t(j >> 1);
    ok = warp_all(mbar_wait(sy.s_full + b, ub & 1, st));
    if (!ok) break;
    tc_fence_after();
    uint32_t r[kW];
    if constexpr (kW == 128) tmem_ld128(tS + lane_off + b * 128, r);
    else tmem_ld64(tS + lane_off + b * 128 + col0, r);
    tc_fence_before();
    mbar_arrive(sy.s_free + b);
    const int nvalid = min(kW, nkv - j * 128 - col0);
    if (nvalid < kW) {  // last, partial tile: logits of missing keys become -inf (p = 0)
#pragma unroll
      for (int c = 0; c < kW; ++c)
        if (c >= nvalid) r[c] = __float_as_uint(-INFINITY);
    }
    // independent partial maxima and sums: one warp per scheduler runs this, so
    // a single dependent chain of 128 max / 64 add operations would be pure latency
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
    // (a half row with no key yet keeps m = -inf: exponents of -inf, not NaN)
    const float neg_m = (kW == 64 && m_use == -INFINITY) ? 0.f : -m_use;
    // two scores per packed FMA and two packed partial sums (four lanes)
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
      if constexpr (kW == 128) tmem_st64(tP + lane_off, pk);
      else tmem_st32(tP + lane_off + col0 / 2, pk);
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

// Epilogue for a query row whose keys were split over two threads (lanes r and
// r + 64, each with its own running max): o0 * f0 + o1 * f1, o0 from TMEM and o1
// from shared memory (float4 k of the row at o1[k * 64]), where f0 and f1 hold
// each half's weight 2^(m_half - m) and 1 / l; then plus (add-residual) or
// subtracted from (store-residual) the bf16 row held in rres, rounded once to
// bf16 and stored. Every thread of the warp must call it (the TMEM loads are
// warp-collective); rows with tok < 0 load but store nothing.
template <int D, int kEpi>
__device__ __forceinline__ void store_row_pair(uint32_t tO, uint32_t lane_off, int tok, size_t rowoff, float f0, float f1,
                                               const float4* o1, __nv_bfloat16* dst, const uint4 (&rres)[D / 8]) {
#pragma unroll
  for (int c = 0; c < D / 32; ++c) {
    uint32_t o[32];
    tmem_ld32(tO + lane_off + c * 32, o);
    if (tok >= 0 && dst != nullptr) {
#pragma unroll
      for (int q4 = 0; q4 < 4; ++q4) {
        const float4 x0 = o1[(c * 8 + q4 * 2) * 64], x1 = o1[(c * 8 + q4 * 2 + 1) * 64];
        const float y[8] = {x0.x, x0.y, x0.z, x0.w, x1.x, x1.y, x1.z, x1.w};
        float o8[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) o8[i] = __uint_as_float(o[q4 * 8 + i]) * f0 + y[i] * f1;
        const size_t off = rowoff + c * 32 + q4 * 8;
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

// Column-split softmax: two threads (two warpgroups) share a query row, thread
// h taking keys [64h, 64h + 64) of every tile (col0 = 64h) with its own running
// max m and sum l and its own O accumulator row (tO). P is written as bf16 pairs
// over the S columns this thread has just read (columns b*128 + col0 ...), so S
// buffer b is free again once the P V of its tile is done (pv_done[b]); no other
// wait sits on the path to P. P of a tile in buffer b is announced on
// p_full[b], which therefore never runs more than one phase ahead of the P V
// thread's wait (its next phase needs S in buffer b again, behind that P V). The O row is rescaled only when the max grows by
// more than 2^8, after the previous tile's P V is done. A half row may see no
// key at all (m stays -inf, l 0, P 0).
// Returns false if a bounded wait ran out.
template <int D>
__device__ __forceinline__ bool softmax_rows_cs(int T, int nkv, uint32_t tS, uint32_t tO, uint32_t lane_off, int col0,
                                                float sl2, uint64_t* s_full, uint64_t* pv_done, uint64_t* p_full,
                                                const uint32_t* st, float& m_out, float& l_out) {
  float m = -INFINITY, l = 0.f;
  bool ok = true;
  for (int j = 0; j < T; ++j) {
    const int b = j & 1;
    ok = warp_all(mbar_wait(s_full + b, uint32_t(j >> 1) & 1, st));
    if (!ok) break;
    tc_fence_after();
    const uint32_t tSb = tS + lane_off + uint32_t(b * 128 + col0);
    uint32_t r[64];
    tmem_ld64(tSb, r);
    const int nvalid = min(64, nkv - j * 128 - col0);
    if (nvalid < 64) {  // last, partial tile: logits of missing keys become -inf (p = 0)
#pragma unroll
      for (int c = 0; c < 64; ++c)
        if (c >= nvalid) r[c] = __float_as_uint(-INFINITY);
    }
    float mp[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) mp[i] = __uint_as_float(r[i]);
#pragma unroll
    for (int c = 8; c < 64; c += 2) mp[(c >> 1) & 7] = fmax3(mp[(c >> 1) & 7], __uint_as_float(r[c]), __uint_as_float(r[c + 1]));
    const float mx = fmax3(fmax3(mp[0], mp[1], mp[2]), fmax3(mp[3], mp[4], mp[5]), fmaxf(mp[6], mp[7]));
    const float m_new = fmaxf(m, mx * sl2);
    const bool need = m_new > m + 8.f;
    const float m_use = need ? m_new : m;
    const float alpha = need ? ex2_approx(m - m_new) : 1.f;
    const float neg_m = m_use == -INFINITY ? 0.f : -m_use;
    const uint64_t sl2x2 = f2_pack(sl2, sl2), negmx2 = f2_pack(neg_m, neg_m);
    uint64_t ls2[2] = {f2_pack(0.f, 0.f), f2_pack(0.f, 0.f)};
    uint32_t pk[32];
#pragma unroll
    for (int c = 0; c < 32; ++c) {
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
    tmem_st32(tSb, pk);
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

}  // namespace mcs
