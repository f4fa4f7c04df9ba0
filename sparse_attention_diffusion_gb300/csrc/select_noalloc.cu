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
#include <cmath>
#include <mutex>

#include "mcs.h"
#include "attn_tc.h"
#include "common.cuh"
#include "kernels.h"

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
  if (desc == nullptr || desc->B < 1 || desc->H < 1 || desc->N < 1) return MCS_ERR_INVALID_ARG;
  if ((desc->d != 64 && desc->d != 128) || (desc->C != 64 && desc->C != 128)) return MCS_ERR_UNSUPPORTED;
  if (desc->dtype != MCS_F32 && desc->dtype != MCS_BF16) return MCS_ERR_UNSUPPORTED;
  if (!std::isfinite(desc->scale)) return MCS_ERR_INVALID_ARG;
  const long long N = desc->N, C = desc->C, d = desc->d;
  const long long G = (N + C - 1) / C, BH = static_cast<long long>(desc->B) * desc->H;
  if (BH > 65535 || BH * G * C >= (1ll << 31)) return MCS_ERR_UNSUPPORTED;
  // one score row of N fp32 values must fit in the fixed scratch array
  const long long rows_fit = static_cast<long long>(kScratchBytes) / (N * 4);
  if (rows_fit < 1) return MCS_ERR_UNSUPPORTED;
  if (K < 1 || K > N) return MCS_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(perm) || !aligned16(idx) || !aligned16(lse))
    return MCS_ERR_INVALID_ARG;  // lse (pass 1) is required here: it is not computed into scratch
  if (mass != nullptr && !aligned16(mass)) return MCS_ERR_INVALID_ARG;
  float* scores = scratch_for_current_device();
  uint32_t* status = mcs::status_word_for_current_device();
  if (scores == nullptr || status == nullptr) return MCS_ERR_CUDA;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const float scale = desc->scale > 0.f ? desc->scale : 1.0f / sqrtf(static_cast<float>(d));
  const long long total = BH * G;
  for (long long r0 = 0; r0 < total; r0 += rows_fit) {
    const int nrows = static_cast<int>(total - r0 < rows_fit ? total - r0 : rows_fit);
    cudaError_t e;
    if (desc->dtype == MCS_BF16) {
      mcs::TcColsumParams p{};
      p.q = static_cast<const __nv_bfloat16*>(q);
      p.k = static_cast<const __nv_bfloat16*>(k);
      p.perm = perm;
      p.lse = lse;
      p.scores = scores;
      p.BH = static_cast<int>(BH);
      p.N = static_cast<int>(N);
      p.N_pad = static_cast<int>(G * C);
      p.C = static_cast<int>(C);
      p.G = static_cast<int>(G);
      p.row0 = static_cast<int>(r0);
      p.scale_log2 = scale * mcs::kLog2e;
      p.status = status;
      e = mcs::tc_colsum(static_cast<int>(d), static_cast<int>(C), p, nrows, s);
    } else {
      mcs::SimtColsumParams p{};
      p.q = static_cast<const float*>(q);
      p.k = static_cast<const float*>(k);
      p.perm = perm;
      p.lse = lse;
      p.scores = scores;
      p.N = static_cast<int>(N);
      p.N_pad = static_cast<int>(G * C);
      p.C = static_cast<int>(C);
      p.G = static_cast<int>(G);
      p.d = static_cast<int>(d);
      p.row0 = static_cast<int>(r0);
      p.scale = scale;
      p.status = status;
      e = mcs::simt_colsum(p, nrows, s);
    }
    if (e != cudaSuccess) return MCS_ERR_CUDA;
    mcs::TopkParams t{};
    t.scores = scores;
    t.perm = perm;
    t.idx = idx;
    t.mass = mass;
    t.N = static_cast<int>(N);
    t.N_pad = static_cast<int>(G * C);
    t.C = static_cast<int>(C);
    t.G = static_cast<int>(G);
    t.K = K;
    t.row0 = static_cast<int>(r0);
    t.status = status;
    if (mcs::topk_rows(t, nrows, s) != cudaSuccess) return MCS_ERR_CUDA;
  }
  return MCS_OK;
}
