// Self-test kernels (no counterpart in the method): a single tcgen05 MMA chain
// and a TMA 4-row gather, used to check on the GPU the shared-memory descriptor
// encodings, the tensor-memory A operand and the TMA gathers.
#include "attn_tc.h"
#include "common.cuh"
#include "ptx.cuh"
#include "tc_common.cuh"
#include "tma.cuh"

namespace mcs {
namespace {

// ---------------------------------------------------------------- probe GEMM (self-test)
// D[128 x N] = A[128 x 64] * B, one MMA chain of 4 k-steps, for checking the
// descriptor encodings: mode 0: B given as [N x 64] K-major; mode 1: B given as
// [64 x N] MN-major (N contiguous), lbo/sbo of the MN-major descriptor are inputs;
// mode 2: as mode 0 but A is first written to tensor memory (bf16 pairs packed
// per 32-bit column, row r on lane r) and read from there by the MMA.
__global__ void __launch_bounds__(128, 1) tc_probe_kernel(const __nv_bfloat16* a, const __nv_bfloat16* b, float* d,
                                                          int mode, uint32_t mn_lbo, uint32_t mn_sbo,
                                                          uint32_t* status) {
  __shared__ __align__(1024) uint8_t sA[kRegion];
  __shared__ __align__(1024) uint8_t sB[2 * kRegion];
  __shared__ __align__(8) uint64_t bar;
  __shared__ uint32_t slot;
  const int tid = threadIdx.x, warp = tid >> 5;
  constexpr int N = 128;
  // A: 128 rows x 64 (K) -> one region
  for (int id = tid; id < 128 * 8; id += 128) {
    const int row = id >> 3, ch = id & 7;
    *reinterpret_cast<uint4*>(sA + sw128_off(row, ch)) = *reinterpret_cast<const uint4*>(a + row * 64 + ch * 8);
  }
  if (mode != 1) {  // B: N rows x 64 (K) -> one region
    for (int id = tid; id < N * 8; id += 128) {
      const int row = id >> 3, ch = id & 7;
      *reinterpret_cast<uint4*>(sB + sw128_off(row, ch)) = *reinterpret_cast<const uint4*>(b + row * 64 + ch * 8);
    }
  } else {  // B: 64 rows (K) x N (contiguous) -> N/64 regions, rows of 128 B
    for (int id = tid; id < 64 * (N / 8); id += 128) {
      const int row = id / (N / 8), ch = id % (N / 8);
      *reinterpret_cast<uint4*>(sB + sw128_off(row, ch)) = *reinterpret_cast<const uint4*>(b + row * N + ch * 8);
    }
  }
  fence_proxy_async_smem();
  if (tid == 0) {
    mbar_init(&bar, 1);
    fence_mbar_init();
  }
  if (warp == 0) {
    tmem_alloc(&slot, 256);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = slot;
  if (mode == 2) {  // A row `tid` -> lane `tid`, columns [128, 160): 32 packed bf16 pairs
    uint32_t r[32];
    for (int c = 0; c < 32; ++c) {
      const __nv_bfloat162 v2 = __halves2bfloat162(a[tid * 64 + 2 * c], a[tid * 64 + 2 * c + 1]);
      r[c] = *reinterpret_cast<const uint32_t*>(&v2);
    }
    tmem_st32(tmem + (uint32_t(warp * 32) << 16) + 128, r);
    tc_fence_before();
  }
  __syncthreads();
  tc_fence_after();
  if (tid == 0) {
    const uint32_t sa = smem_u32(sA), sb = smem_u32(sB);
    for (int ks = 0; ks < 4; ++ks) {
      const uint64_t da = desc_kmajor(sa, ks);
      if (mode == 2) {
        tc_mma_ts(tmem, tmem + 128 + ks * 8, desc_kmajor(sb, ks), idesc_bf16_f32(128, N, 0, 0), ks > 0 ? 1u : 0u);
        continue;
      }
      uint64_t db;
      uint32_t idesc;
      if (mode == 0) {
        db = desc_kmajor(sb, ks);
        idesc = idesc_bf16_f32(128, N, 0, 0);
      } else {
        db = smem_desc_sw128(sb + ks * 16 * 128, mn_lbo, mn_sbo);
        idesc = idesc_bf16_f32(128, N, 0, 1);
      }
      tc_mma_ss(tmem, da, db, idesc, ks > 0 ? 1u : 0u);
    }
    tc_commit(&bar);
  }
  const bool ok = mbar_wait(&bar, 0, status);
  if (!ok && tid == 0) raise_status(status, kStatusTimeout);
  __syncwarp();
  if (__all_sync(0xffffffffu, ok)) {
    tc_fence_after();
    for (int c = 0; c < N / 32; ++c) {
      uint32_t r[32];
      tmem_ld32(tmem + (uint32_t(warp * 32) << 16) + c * 32, r);
      for (int i = 0; i < 32; ++i) d[tid * N + c * 32 + i] = __uint_as_float(r[i]);
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, 256);
  }
}

// Gathers 128 rows of a bf16 [rows x 128] matrix with TMA tile::gather4 into the
// 128-byte-swizzled shared-memory layout the MMAs read, then writes them back out
// row-major (un-swizzled): out[i] = src[rows[i]] (zeros for rows out of range).
__global__ void __launch_bounds__(128, 1) tma_gather_probe_kernel(const __grid_constant__ CUtensorMap map,
                                                                  const int* rows, __nv_bfloat16* out,
                                                                  uint32_t* status) {
  __shared__ __align__(1024) uint8_t tile[2 * kRegion];
  __shared__ __align__(8) uint64_t bar;
  const int tid = threadIdx.x;
  if (tid == 0) {
    mbar_init(&bar, 1);
    fence_mbar_init();
  }
  __syncthreads();
  if (tid == 0) {
    const uint32_t b = smem_u32(&bar), t = smem_u32(tile);
    mbar_arrive_expect_tx(&bar, 2 * kRegion);
    for (int r4 = 0; r4 < 32; ++r4)
      for (int half = 0; half < 2; ++half)
        tma_gather4(t + half * kRegion + r4 * 512, &map, half * 64, rows[4 * r4], rows[4 * r4 + 1], rows[4 * r4 + 2],
                    rows[4 * r4 + 3], b);
  }
  const bool ok = mbar_wait(&bar, 0, status);
  if (!ok) {
    if (tid == 0) raise_status(status, kStatusTimeout);
    return;
  }
  for (int ch = 0; ch < 16; ++ch)
    *reinterpret_cast<uint4*>(out + tid * 128 + ch * 8) = *reinterpret_cast<const uint4*>(tile + sw128_off(tid, ch));
}

// Waits on an mbarrier that nothing ever arrives at, with a wait limit of
// limit_ns, the way every pipeline wait in the library is bounded: the wait
// gives up, the kernel raises the timeout flag, releases the tensor memory it
// holds and returns, so the context stays usable. elapsed (nullable) receives
// the nanoseconds thread 0 spent waiting.
__global__ void __launch_bounds__(128, 1) wait_timeout_probe_kernel(uint64_t limit_ns, unsigned long long* elapsed,
                                                                    uint32_t* status) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ uint32_t slot;
  const int tid = threadIdx.x, warp = tid >> 5;
  if (tid == 0) {
    mbar_init(&bar, 1);  // one arrival expected, none ever made
    fence_mbar_init();
  }
  if (warp == 0) {
    tmem_alloc(&slot, 32);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = slot;
  const uint64_t t0 = globaltimer_ns();
  const bool ok = mbar_wait(&bar, 0, status, limit_ns);
  const uint64_t t1 = globaltimer_ns();
  if (!ok && tid == 0) raise_status(status, kStatusTimeout);
  if (tid == 0 && elapsed != nullptr) *elapsed = static_cast<unsigned long long>(t1 - t0);
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, 32);
  }
}

// Throughput of the exponential unit as the softmax uses it: every thread runs
// eight independent chains of ex2.approx.ftz.f32 (x <- 2^-x stays in (0.5, 1]),
// 32 warps per CTA; the dynamic shared memory it asks for (but does not use)
// keeps one CTA per SM, so a CTA's clock64 span is its SM's time for the count.
constexpr int kEx2Threads = 1024, kEx2Chains = 8;
__global__ void __launch_bounds__(kEx2Threads, 1) ex2_rate_kernel(int iters, unsigned long long* out) {
  float x[kEx2Chains];
#pragma unroll
  for (int k = 0; k < kEx2Chains; ++k) x[k] = 0.001f * float(threadIdx.x & 31) + 0.1f * float(k);
  __syncthreads();
  const long long t0 = clock64();
  for (int i = 0; i < iters; ++i) {
#pragma unroll
    for (int k = 0; k < kEx2Chains; ++k) x[k] = ex2_approx(-x[k]);
  }
  __syncthreads();
  const long long t1 = clock64();
  float acc = 0.f;
#pragma unroll
  for (int k = 0; k < kEx2Chains; ++k) acc += x[k];
  if (threadIdx.x == 0) {
    out[2 * blockIdx.x] = static_cast<unsigned long long>(t1 - t0);
    out[2 * blockIdx.x + 1] = static_cast<unsigned long long>(kEx2Threads) * kEx2Chains * unsigned(iters);
  }
  if (acc < 0.f) out[2 * blockIdx.x + 1] = 0;  // never true; keeps the chains live
}

}  // namespace

cudaError_t ex2_rate_probe(int iters, int nblocks, unsigned long long* out, cudaStream_t stream) {
  constexpr int kPad = 120 * 1024;  // more than half an SM's shared memory: one CTA per SM
  cudaError_t e = cudaFuncSetAttribute(ex2_rate_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kPad);
  if (e != cudaSuccess) return e;
  ex2_rate_kernel<<<nblocks, kEx2Threads, kPad, stream>>>(iters, out);
  note_launches(1);
  return cudaGetLastError();
}

cudaError_t wait_timeout_probe(uint64_t limit_ns, unsigned long long* elapsed, uint32_t* status, cudaStream_t stream) {
  wait_timeout_probe_kernel<<<1, 128, 0, stream>>>(limit_ns, elapsed, status);
  note_launches(1);
  return cudaGetLastError();
}

cudaError_t tma_gather_probe(const void* src, int nrows, const int* rows, void* out, uint32_t* status,
                             cudaStream_t stream) {
  CUtensorMap map;
  if (!make_gather_map(&map, src, uint64_t(nrows), 128)) return cudaErrorInvalidValue;
  tma_gather_probe_kernel<<<1, 128, 0, stream>>>(map, rows, static_cast<__nv_bfloat16*>(out), status);
  note_launches(1);
  return cudaGetLastError();
}

cudaError_t tc_probe(const void* a, const void* b, float* d, int mode, uint32_t lbo, uint32_t sbo, uint32_t* status,
                     cudaStream_t stream) {
  tc_probe_kernel<<<1, 128, 0, stream>>>(static_cast<const __nv_bfloat16*>(a), static_cast<const __nv_bfloat16*>(b),
                                         d, mode, lbo, sbo, status);
  note_launches(1);
  return cudaGetLastError();
}

}  // namespace mcs
