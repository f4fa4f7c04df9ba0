// Residual store / apply: r = o_dense - o_sparse at the anchor step and
// o = o_sparse + r at reuse steps [MC-Sparse summary: residual paragraph].
// Element-wise and HBM-bound: 16-byte vector loads/stores, fp32 arithmetic,
// one rounding to the I/O type, grid sized to the SM count.
#include "common.cuh"
#include "kernels.h"

namespace mcs {
namespace {

template <typename T>
struct Vec;  // 16 bytes of T
template <>
struct Vec<float> {
  static constexpr int n = 4;
};
template <>
struct Vec<__nv_bfloat16> {
  static constexpr int n = 8;
};

template <typename T, bool kStore>
__global__ void __launch_bounds__(256) residual_kernel(const T* __restrict__ a, const T* __restrict__ b,
                                                      T* __restrict__ out, size_t nvec) {
  constexpr int n = Vec<T>::n;
  for (size_t i = blockIdx.x * size_t(blockDim.x) + threadIdx.x; i < nvec; i += size_t(gridDim.x) * blockDim.x) {
    const uint4 va = __ldcs(reinterpret_cast<const uint4*>(a) + i);
    const uint4 vb = __ldcs(reinterpret_cast<const uint4*>(b) + i);
    const T* ea = reinterpret_cast<const T*>(&va);
    const T* eb = reinterpret_cast<const T*>(&vb);
    uint4 vo;
    T* eo = reinterpret_cast<T*>(&vo);
#pragma unroll
    for (int k = 0; k < n; ++k) {
      const float x = to_f32(ea[k]), y = to_f32(eb[k]);
      eo[k] = from_f32<T>(kStore ? x - y : x + y);
    }
    __stcs(reinterpret_cast<uint4*>(out) + i, vo);
  }
}

template <typename T, bool kStore>
cudaError_t launch(const void* a, const void* b, void* out, size_t nelem, int num_sms, cudaStream_t s) {
  const size_t nvec = nelem / Vec<T>::n;
  if (nvec == 0) return cudaSuccess;
  const size_t want = (nvec + 255) / 256;
  const int grid = int(want < size_t(num_sms) * 8 ? want : size_t(num_sms) * 8);
  residual_kernel<T, kStore><<<grid, 256, 0, s>>>(static_cast<const T*>(a), static_cast<const T*>(b),
                                                  static_cast<T*>(out), nvec);
  note_launches(1);
  return cudaGetLastError();
}

}  // namespace

cudaError_t residual_op(bool store, bool bf16, const void* a, const void* b, void* out, size_t nelem, int num_sms,
                        cudaStream_t s) {
  if (bf16) return store ? launch<__nv_bfloat16, true>(a, b, out, nelem, num_sms, s)
                         : launch<__nv_bfloat16, false>(a, b, out, nelem, num_sms, s);
  return store ? launch<float, true>(a, b, out, nelem, num_sms, s) : launch<float, false>(a, b, out, nelem, num_sms, s);
}

}  // namespace mcs
