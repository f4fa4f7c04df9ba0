// Anchor selection without a caller-provided workspace.
//
// mcs_anchor_select needs scratch space for the pass-2 score rows (one fp32 row
// of N scores per query group) and takes it from a workspace the caller
// allocates. Some callers cannot allocate device memory at the point where they
// call us: code running under a CUDA-graph capture that forbids allocation, a
// host framework that owns the device heap and exposes no allocator to plug-ins,
// or a real-time loop where cudaMalloc's implicit synchronisation is not allowed.
// For them this file keeps the score rows in one fixed, file-scope device
// array, so mcs_anchor_select_noalloc allocates nothing: no cudaMalloc, no
// cudaFree, no allocating library routine.
//
// The array is kScratchBytes (64 MiB) and every GPU that loads the library
// holds it until the process exits. It is shared by all calls and keeps the
// previous call's contents; every score the top-K reads is written earlier in
// the same call, so nothing has to be cleared first. Calls whose kernels overlap
// on the GPU (different streams, or different host threads) race on it.
#include <mutex>

#include "mcs.h"
#include "api_internal.h"

namespace {

constexpr size_t kScratchBytes = size_t(64) << 20;
static __device__ __align__(256) unsigned char g_select_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
float* g_scratch_ptr[kMaxDevices] = {};
std::mutex g_setup_mutex;

// Device address of the scratch array on the current device. In host code the
// array's name is only a host-side stand-in, so the address is looked up once
// per device with that device current (the first call on a device does this).
float* scratch_for_current_device() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lock(g_setup_mutex);
  if (g_scratch_ptr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_select_scratch) != cudaSuccess) return nullptr;
    g_scratch_ptr[dev] = static_cast<float*>(p);
  }
  return g_scratch_ptr[dev];
}

bool aligned16(const void* p) { return p != nullptr && (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

extern "C" mcs_status mcs_anchor_select_noalloc(const mcs_desc* desc, const void* q, const void* k,
                                                const int32_t* perm, const float* lse, int K, int32_t* idx,
                                                float* mass, mcs_stream stream) {
  // argument checks (lse is required: pass 1 is not computed into the array) and
  // the launch loop are those of the workspace entry point; score rows per
  // launch are what fits in the array, at most 4,096
  if (desc == nullptr || desc->N < 1) return MCS_ERR_INVALID_ARG;
  if (static_cast<long long>(kScratchBytes) / (static_cast<long long>(desc->N) * 4) < 1) return MCS_ERR_UNSUPPORTED;
  if (!aligned16(lse)) return MCS_ERR_INVALID_ARG;
  float* scores = scratch_for_current_device();
  if (scores == nullptr) return MCS_ERR_CUDA;
  return mcs::anchor_select_rows(desc, q, k, perm, lse, K, idx, mass, scores, kScratchBytes,
                                 reinterpret_cast<cudaStream_t>(stream));
}
