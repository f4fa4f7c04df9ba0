// Shared host/device definitions for the libmcs kernels.
#pragma once
#include <cstdint>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

namespace mcs {

// Element access for the two supported I/O types.
__device__ __forceinline__ float to_f32(float x) { return x; }
__device__ __forceinline__ float to_f32(__nv_bfloat16 x) { return __bfloat162float(x); }
template <typename T> __device__ __forceinline__ T from_f32(float x);
template <> __device__ __forceinline__ float from_f32<float>(float x) { return x; }
template <> __device__ __forceinline__ __nv_bfloat16 from_f32<__nv_bfloat16>(float x) {
  return __float2bfloat16_rn(x);
}

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

// Epilogue of the sparse attention kernels.
enum Epilogue : int {
  kEpiPlain = 0,      // o = attention
  kEpiAddResidual = 1,// o = attention + r            (reuse step)
  kEpiStoreResidual = 2 // r = o_dense - attention    (anchor step)
};

// Host-side launch bookkeeping and the device status word (defined in api.cu).
void note_launches(int n);
uint32_t* status_word_for_current_device();  // null if the CUDA runtime call failed

}  // namespace mcs
