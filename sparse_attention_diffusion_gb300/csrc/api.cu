// C ABI of libmcs (declared in include/mcs.h): argument validation, workspace
// layout, dispatch to the bf16 tcgen05 kernels or the fp32 SIMT kernels, and
// the device status word. Nothing here allocates device memory.
#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <mutex>

#include "mcs.h"
#include "api_internal.h"
#include "attn_tc.h"
#include "common.cuh"
#include "kernels.h"
#include "status.cuh"

namespace {

__device__ uint32_t g_status_word;  // OR of mcs::kStatus* bits raised by kernels
std::atomic<uint64_t> g_launches{0};

constexpr int kMaxDevices = 64;
uint32_t* g_status_ptr[kMaxDevices] = {};
int g_num_sms[kMaxDevices] = {};

// Rows of pass-2 scores kept in the workspace at once (each row is N fp32).
constexpr long long kSelectRows = 4096;

struct Dims {
  int B, H, N, d, C, G, N_pad, BH;
  bool bf16;
  float scale;
  int iters;
};

mcs_status check_desc(const mcs_desc* desc, Dims* o) {
  if (desc == nullptr) return MCS_ERR_INVALID_ARG;
  if (desc->B < 1 || desc->H < 1 || desc->N < 1) return MCS_ERR_INVALID_ARG;
  if (desc->d != 64 && desc->d != 128) return MCS_ERR_UNSUPPORTED;
  if (desc->C != 64 && desc->C != 128) return MCS_ERR_UNSUPPORTED;
  if (desc->dtype != MCS_F32 && desc->dtype != MCS_BF16) return MCS_ERR_UNSUPPORTED;
  if (!std::isfinite(desc->scale)) return MCS_ERR_INVALID_ARG;
  const long long G = (static_cast<long long>(desc->N) + desc->C - 1) / desc->C;
  const long long BH = static_cast<long long>(desc->B) * desc->H;
  if (BH > 65535 || BH * G * desc->C >= (1ll << 31)) return MCS_ERR_UNSUPPORTED;
  o->B = desc->B;
  o->H = desc->H;
  o->N = desc->N;
  o->d = desc->d;
  o->C = desc->C;
  o->G = static_cast<int>(G);
  o->N_pad = static_cast<int>(G * desc->C);
  o->BH = static_cast<int>(BH);
  o->bf16 = desc->dtype == MCS_BF16;
  o->scale = desc->scale > 0.f ? desc->scale : 1.0f / std::sqrt(static_cast<float>(desc->d));
  o->iters = desc->pddp_iters > 0 ? desc->pddp_iters : 20;
  return MCS_OK;
}

bool aligned16(const void* p) { return p != nullptr && (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool aligned16_or_null(const void* p) { return p == nullptr || aligned16(p); }

mcs_status device_state(uint32_t** status, int* sms) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return MCS_ERR_CUDA;
  if (g_status_ptr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_status_word) != cudaSuccess) return MCS_ERR_CUDA;
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return MCS_ERR_CUDA;
    g_num_sms[dev] = n;
    g_status_ptr[dev] = static_cast<uint32_t*>(p);
  }
  *status = g_status_ptr[dev];
  if (sms) *sms = g_num_sms[dev];
  return MCS_OK;
}

mcs_status from_cuda(cudaError_t e) { return e == cudaSuccess ? MCS_OK : MCS_ERR_CUDA; }

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

// Anchor-select workspace: [lse fp32 BH*N] [score rows: min(BH*G, kSelectRows) * N fp32]
size_t select_ws_bytes(const Dims& d) {
  const long long rows = std::min<long long>(static_cast<long long>(d.BH) * d.G, kSelectRows);
  return align256(size_t(d.BH) * d.N * 4) + align256(size_t(rows) * d.N * 4);
}

mcs_status dense_impl(const Dims& dm, const void* q, const void* k, const void* v, void* o, float* lse,
                      uint32_t* status, cudaStream_t s) {
  if (dm.bf16) {
    mcs::TcAttnParams p{};
    p.q = static_cast<const __nv_bfloat16*>(q);
    p.k = static_cast<const __nv_bfloat16*>(k);
    p.v = static_cast<const __nv_bfloat16*>(v);
    p.o = static_cast<__nv_bfloat16*>(o);
    p.lse = lse;
    p.BH = dm.BH;
    p.N = dm.N;
    p.N_pad = dm.N_pad;
    p.C = dm.C;
    p.G = dm.G;
    p.K = dm.N;
    p.tiles_per_head = (dm.N + 127) / 128;
    p.scale_log2 = dm.scale * mcs::kLog2e;
    p.status = status;
    return from_cuda(mcs::tc_dense_attn(dm.d, p, dm.BH, o != nullptr, s));
  }
  mcs::SimtAttnParams p{};
  p.q = static_cast<const float*>(q);
  p.k = static_cast<const float*>(k);
  p.v = static_cast<const float*>(v);
  p.o = static_cast<float*>(o);
  p.lse = lse;
  p.N = dm.N;
  p.N_pad = dm.N_pad;
  p.C = dm.C;
  p.G = dm.G;
  p.K = dm.N;
  p.d = dm.d;
  p.scale = dm.scale;
  p.status = status;
  return from_cuda(mcs::simt_dense_attn(p, dm.BH, s));
}

mcs_status sparse_impl(const Dims& dm, int epi, const void* q, const void* k, const void* v, const int32_t* perm,
                       const int32_t* idx, int K, const void* res_in, void* o, void* res_out, uint32_t* status,
                       cudaStream_t s) {
  if (dm.bf16) {
    mcs::TcAttnParams p{};
    p.q = static_cast<const __nv_bfloat16*>(q);
    p.k = static_cast<const __nv_bfloat16*>(k);
    p.v = static_cast<const __nv_bfloat16*>(v);
    p.o = static_cast<__nv_bfloat16*>(o);
    p.perm = perm;
    p.idx = idx;
    p.res_in = static_cast<const __nv_bfloat16*>(res_in);
    p.res_out = static_cast<__nv_bfloat16*>(res_out);
    p.BH = dm.BH;
    p.N = dm.N;
    p.N_pad = dm.N_pad;
    p.C = dm.C;
    p.G = dm.G;
    p.K = K;
    p.tiles_per_head = dm.G;
    p.scale_log2 = dm.scale * mcs::kLog2e;
    p.status = status;
    return from_cuda(mcs::tc_sparse_attn(dm.d, epi, p, dm.BH, s));
  }
  mcs::SimtAttnParams p{};
  p.q = static_cast<const float*>(q);
  p.k = static_cast<const float*>(k);
  p.v = static_cast<const float*>(v);
  p.o = static_cast<float*>(o);
  p.perm = perm;
  p.idx = idx;
  p.res_in = static_cast<const float*>(res_in);
  p.res_out = static_cast<float*>(res_out);
  p.N = dm.N;
  p.N_pad = dm.N_pad;
  p.C = dm.C;
  p.G = dm.G;
  p.K = K;
  p.d = dm.d;
  p.scale = dm.scale;
  p.status = status;
  return from_cuda(mcs::simt_sparse_attn(epi, p, dm.BH, s));
}

}  // namespace

namespace mcs {
mcs_status anchor_select_rows(const mcs_desc* desc, const void* q, const void* k, const int32_t* perm,
                              const float* lse, int K, int32_t* idx, float* mass, float* scores, size_t score_bytes,
                              cudaStream_t s) {
  Dims dm;
  mcs_status st = check_desc(desc, &dm);
  if (st != MCS_OK) return st;
  if (K < 1 || K > dm.N) return MCS_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(perm) || !aligned16(idx) || !aligned16(lse))
    return MCS_ERR_INVALID_ARG;
  if (!aligned16_or_null(mass) || !aligned16(scores)) return MCS_ERR_INVALID_ARG;
  // score rows per launch: what fits, at most kSelectRows (the launch grids stay small)
  const long long rows = std::min<long long>(kSelectRows, static_cast<long long>(score_bytes / (size_t(dm.N) * 4)));
  if (rows < 1) return MCS_ERR_UNSUPPORTED;
  uint32_t* status = nullptr;
  if ((st = device_state(&status, nullptr)) != MCS_OK) return st;
  const long long total = static_cast<long long>(dm.BH) * dm.G;
  for (long long r0 = 0; r0 < total; r0 += rows) {
    const int nrows = static_cast<int>(std::min<long long>(rows, total - r0));
    cudaError_t e;
    if (dm.bf16) {
      TcColsumParams p{};
      p.q = static_cast<const __nv_bfloat16*>(q);
      p.k = static_cast<const __nv_bfloat16*>(k);
      p.perm = perm;
      p.lse = lse;
      p.scores = scores;
      p.BH = dm.BH;
      p.N = dm.N;
      p.N_pad = dm.N_pad;
      p.C = dm.C;
      p.G = dm.G;
      p.row0 = static_cast<int>(r0);
      p.scale_log2 = dm.scale * kLog2e;
      p.status = status;
      e = tc_colsum(dm.d, dm.C, p, nrows, s);
    } else {
      SimtColsumParams p{};
      p.q = static_cast<const float*>(q);
      p.k = static_cast<const float*>(k);
      p.perm = perm;
      p.lse = lse;
      p.scores = scores;
      p.N = dm.N;
      p.N_pad = dm.N_pad;
      p.C = dm.C;
      p.G = dm.G;
      p.d = dm.d;
      p.row0 = static_cast<int>(r0);
      p.scale = dm.scale;
      p.status = status;
      e = simt_colsum(p, nrows, s);
    }
    if (e != cudaSuccess) return MCS_ERR_CUDA;
    TopkParams t{};
    t.scores = scores;
    t.perm = perm;
    t.idx = idx;
    t.mass = mass;
    t.N = dm.N;
    t.N_pad = dm.N_pad;
    t.C = dm.C;
    t.G = dm.G;
    t.K = K;
    t.row0 = static_cast<int>(r0);
    t.status = status;
    if ((e = topk_rows(t, nrows, s)) != cudaSuccess) return MCS_ERR_CUDA;
  }
  return MCS_OK;
}

void note_launches(int n) { g_launches.fetch_add(static_cast<uint64_t>(n), std::memory_order_relaxed); }
uint32_t* status_word_for_current_device() {
  uint32_t* st = nullptr;
  return device_state(&st, nullptr) == MCS_OK ? st : nullptr;
}
}  // namespace mcs

extern "C" {

size_t mcs_workspace_size(const mcs_desc* desc, int K) {
  Dims dm;
  if (check_desc(desc, &dm) != MCS_OK) return 0;
  (void)K;
  const size_t a = mcs::pddp_workspace_bytes(dm.BH, dm.N_pad, dm.C, dm.G, dm.d, dm.bf16);
  const size_t b = select_ws_bytes(dm);
  return a > b ? a : b;
}

size_t mcs_pddp_dirs_size(const mcs_desc* desc) {
  Dims dm;
  if (check_desc(desc, &dm) != MCS_OK) return 0;
  return size_t(dm.BH) * mcs::pddp_dir_slots(dm.G) * dm.d * sizeof(float);
}

mcs_status mcs_group_pddp_warm(const mcs_desc* desc, const void* q, const float* dirs_in, float* dirs_out,
                               int32_t* perm, int32_t* group_of, void* ws, size_t ws_bytes, mcs_stream stream) {
  Dims dm;
  mcs_status st = check_desc(desc, &dm);
  if (st != MCS_OK) return st;
  if (!aligned16(q) || !aligned16(perm) || !aligned16(group_of)) return MCS_ERR_INVALID_ARG;
  if (!aligned16_or_null(dirs_in) || !aligned16_or_null(dirs_out)) return MCS_ERR_INVALID_ARG;
  if (ws == nullptr || !aligned16(ws) || ws_bytes < mcs_workspace_size(desc, 1)) return MCS_ERR_WORKSPACE;
  uint32_t* status = nullptr;
  int sms = 0;
  if ((st = device_state(&status, &sms)) != MCS_OK) return st;
  mcs::PddpProblem p{};
  p.num_sms = sms;
  p.q = q;
  p.perm = perm;
  p.group_of = group_of;
  p.BH = dm.BH;
  p.N = dm.N;
  p.N_pad = dm.N_pad;
  p.C = dm.C;
  p.G = dm.G;
  p.d = dm.d;
  p.iters = desc->pddp_iters > 0 ? desc->pddp_iters : (desc->pddp_iters == 0 && dirs_in != nullptr ? 0 : 20);
  p.bf16 = dm.bf16;
  p.status = status;
  p.dirs_in = dirs_in;
  p.dirs_out = dirs_out;
  return from_cuda(mcs::pddp_run(p, ws, ws_bytes, reinterpret_cast<cudaStream_t>(stream)));
}

mcs_status mcs_group_pddp(const mcs_desc* desc, const void* q, int32_t* perm, int32_t* group_of, void* ws,
                          size_t ws_bytes, mcs_stream stream) {
  return mcs_group_pddp_warm(desc, q, nullptr, nullptr, perm, group_of, ws, ws_bytes, stream);
}

mcs_status mcs_dense_attn(const mcs_desc* desc, const void* q, const void* k, const void* v, void* o, float* lse,
                          mcs_stream stream) {
  Dims dm;
  mcs_status st = check_desc(desc, &dm);
  if (st != MCS_OK) return st;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v)) return MCS_ERR_INVALID_ARG;
  if (o == nullptr && lse == nullptr) return MCS_ERR_INVALID_ARG;
  if (!aligned16_or_null(o) || !aligned16_or_null(lse)) return MCS_ERR_INVALID_ARG;
  uint32_t* status = nullptr;
  if ((st = device_state(&status, nullptr)) != MCS_OK) return st;
  return dense_impl(dm, q, k, v, o, lse, status, reinterpret_cast<cudaStream_t>(stream));
}

mcs_status mcs_anchor_select(const mcs_desc* desc, const void* q, const void* k, const int32_t* perm, const float* lse,
                             int K, int32_t* idx, float* mass, void* ws, size_t ws_bytes, mcs_stream stream) {
  Dims dm;
  mcs_status st = check_desc(desc, &dm);
  if (st != MCS_OK) return st;
  if (K < 1 || K > dm.N) return MCS_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(perm) || !aligned16(idx)) return MCS_ERR_INVALID_ARG;
  if (!aligned16_or_null(lse) || !aligned16_or_null(mass)) return MCS_ERR_INVALID_ARG;
  if (ws == nullptr || !aligned16(ws) || ws_bytes < mcs_workspace_size(desc, K)) return MCS_ERR_WORKSPACE;
  uint32_t* status = nullptr;
  if ((st = device_state(&status, nullptr)) != MCS_OK) return st;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  uint8_t* w = static_cast<uint8_t*>(ws);
  const size_t lse_bytes = align256(size_t(dm.BH) * dm.N * 4);
  float* ws_lse = reinterpret_cast<float*>(w);
  float* scores = reinterpret_cast<float*>(w + lse_bytes);
  if (lse == nullptr) {
    // pass 1 computed here: row max / log-sum-exp only (no P V product)
    st = dense_impl(dm, q, k, k, nullptr, ws_lse, status, s);
    if (st != MCS_OK) return st;
    lse = ws_lse;
  }
  return mcs::anchor_select_rows(desc, q, k, perm, lse, K, idx, mass, scores, ws_bytes - lse_bytes, s);
}

mcs_status mcs_sparse_attn_gather(const mcs_desc* desc, const void* q, const void* k, const void* v,
                                  const int32_t* perm, const int32_t* idx, int K, const void* residual, void* o,
                                  mcs_stream stream) {
  Dims dm;
  mcs_status st = check_desc(desc, &dm);
  if (st != MCS_OK) return st;
  if (K < 1 || K > dm.N) return MCS_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(perm) || !aligned16(idx) || !aligned16(o))
    return MCS_ERR_INVALID_ARG;
  if (!aligned16_or_null(residual)) return MCS_ERR_INVALID_ARG;
  uint32_t* status = nullptr;
  if ((st = device_state(&status, nullptr)) != MCS_OK) return st;
  return sparse_impl(dm, residual ? mcs::kEpiAddResidual : mcs::kEpiPlain, q, k, v, perm, idx, K, residual, o,
                     nullptr, status, reinterpret_cast<cudaStream_t>(stream));
}

namespace {
// Heads per chunk and the 256-byte-rounded bytes of one staged tensor chunk.
bool host_chunking(const Dims& dm, int head_chunks, int* nch, int* hpc, size_t* chunk_bytes) {
  if (head_chunks < 1) return false;
  *nch = head_chunks < dm.BH ? head_chunks : dm.BH;
  *hpc = (dm.BH + *nch - 1) / *nch;
  *nch = (dm.BH + *hpc - 1) / *hpc;
  const size_t es = dm.bf16 ? 2 : 4;
  *chunk_bytes = ((size_t(*hpc) * dm.N * dm.d * es) + 255) & ~size_t(255);
  return true;
}
}  // namespace

size_t mcs_sparse_attn_gather_host_workspace_size(const mcs_desc* desc, int head_chunks) {
  Dims dm;
  int nch = 0, hpc = 0;
  size_t cb = 0;
  if (check_desc(desc, &dm) != MCS_OK || !host_chunking(dm, head_chunks, &nch, &hpc, &cb)) return 0;
  return 2 * 4 * cb;  // two slots of q, k, v, o
}

mcs_status mcs_sparse_attn_gather_host(const mcs_desc* desc, const void* q_host, const void* k_host,
                                       const void* v_host, const int32_t* perm, const int32_t* idx, int K,
                                       const void* residual, void* o_host, void* ws, size_t ws_bytes,
                                       int head_chunks, mcs_stream stream) {
  Dims dm;
  mcs_status st = check_desc(desc, &dm);
  if (st != MCS_OK) return st;
  if (K < 1 || K > dm.N) return MCS_ERR_INVALID_ARG;
  if (q_host == nullptr || k_host == nullptr || v_host == nullptr || o_host == nullptr) return MCS_ERR_INVALID_ARG;
  if (!aligned16(perm) || !aligned16(idx) || !aligned16_or_null(residual)) return MCS_ERR_INVALID_ARG;
  int nch = 0, hpc = 0;
  size_t cb = 0;
  if (!host_chunking(dm, head_chunks, &nch, &hpc, &cb)) return MCS_ERR_INVALID_ARG;
  if (ws == nullptr || !aligned16(ws) || ws_bytes < 2 * 4 * cb) return MCS_ERR_WORKSPACE;
  uint32_t* status = nullptr;
  if ((st = device_state(&status, nullptr)) != MCS_OK) return st;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const size_t es = dm.bf16 ? 2 : 4, head_bytes = size_t(dm.N) * dm.d * es;
  uint8_t* w = static_cast<uint8_t*>(ws);
  auto slot_ptr = [&](int slot, int t) { return w + (size_t(slot) * 4 + t) * cb; };  // t: q, k, v, o
  // copy-in and copy-out streams, two compute streams (even and odd chunks, so
  // that a chunk's kernel fills the SMs its predecessor's last wave leaves idle)
  // and the events that order them; destroying them right after enqueueing is
  // safe (released once the work ends)
  cudaStream_t h2d = nullptr, d2h = nullptr, cs[2] = {};
  cudaEvent_t start = nullptr, end = nullptr, ev_in[2] = {}, ev_done[2] = {}, ev_free[2] = {};
  auto cleanup = [&]() {
    for (int i = 0; i < 2; ++i) {
      if (ev_in[i]) cudaEventDestroy(ev_in[i]);
      if (ev_done[i]) cudaEventDestroy(ev_done[i]);
      if (ev_free[i]) cudaEventDestroy(ev_free[i]);
    }
    if (start) cudaEventDestroy(start);
    if (end) cudaEventDestroy(end);
    if (h2d) cudaStreamDestroy(h2d);
    if (d2h) cudaStreamDestroy(d2h);
    for (int i = 0; i < 2; ++i)
      if (cs[i]) cudaStreamDestroy(cs[i]);
  };
  bool okc = cudaStreamCreateWithFlags(&h2d, cudaStreamNonBlocking) == cudaSuccess &&
             cudaStreamCreateWithFlags(&d2h, cudaStreamNonBlocking) == cudaSuccess &&
             cudaStreamCreateWithFlags(&cs[0], cudaStreamNonBlocking) == cudaSuccess &&
             cudaStreamCreateWithFlags(&cs[1], cudaStreamNonBlocking) == cudaSuccess &&
             cudaEventCreateWithFlags(&start, cudaEventDisableTiming) == cudaSuccess &&
             cudaEventCreateWithFlags(&end, cudaEventDisableTiming) == cudaSuccess;
  for (int i = 0; okc && i < 2; ++i)
    okc = cudaEventCreateWithFlags(&ev_in[i], cudaEventDisableTiming) == cudaSuccess &&
          cudaEventCreateWithFlags(&ev_done[i], cudaEventDisableTiming) == cudaSuccess &&
          cudaEventCreateWithFlags(&ev_free[i], cudaEventDisableTiming) == cudaSuccess;
  okc = okc && cudaEventRecord(start, s) == cudaSuccess && cudaStreamWaitEvent(h2d, start, 0) == cudaSuccess &&
        cudaStreamWaitEvent(d2h, start, 0) == cudaSuccess && cudaStreamWaitEvent(cs[0], start, 0) == cudaSuccess &&
        cudaStreamWaitEvent(cs[1], start, 0) == cudaSuccess;
  for (int c = 0; okc && c < nch; ++c) {
    const int slot = c & 1, bh0 = c * hpc, nh = (dm.BH - bh0) < hpc ? (dm.BH - bh0) : hpc;
    const size_t off = size_t(bh0) * head_bytes, bytes = size_t(nh) * head_bytes;
    // slot reuse: chunk c - 2's output has been copied out (after its kernel)
    if (c >= 2) okc = cudaStreamWaitEvent(h2d, ev_free[slot], 0) == cudaSuccess;
    okc = okc &&
          cudaMemcpyAsync(slot_ptr(slot, 0), static_cast<const uint8_t*>(q_host) + off, bytes, cudaMemcpyHostToDevice,
                          h2d) == cudaSuccess &&
          cudaMemcpyAsync(slot_ptr(slot, 1), static_cast<const uint8_t*>(k_host) + off, bytes, cudaMemcpyHostToDevice,
                          h2d) == cudaSuccess &&
          cudaMemcpyAsync(slot_ptr(slot, 2), static_cast<const uint8_t*>(v_host) + off, bytes, cudaMemcpyHostToDevice,
                          h2d) == cudaSuccess &&
          cudaEventRecord(ev_in[slot], h2d) == cudaSuccess && cudaStreamWaitEvent(cs[slot], ev_in[slot], 0) == cudaSuccess;
    if (!okc) break;
    Dims dc = dm;
    dc.B = 1;
    dc.H = nh;
    dc.BH = nh;
    const void* rc = residual ? static_cast<const uint8_t*>(residual) + off : nullptr;
    st = sparse_impl(dc, residual ? mcs::kEpiAddResidual : mcs::kEpiPlain, slot_ptr(slot, 0), slot_ptr(slot, 1),
                     slot_ptr(slot, 2), perm + size_t(bh0) * dm.N_pad, idx + size_t(bh0) * dm.G * size_t(K), K, rc,
                     slot_ptr(slot, 3), nullptr, status, cs[slot]);
    if (st != MCS_OK) break;
    okc = cudaEventRecord(ev_done[slot], cs[slot]) == cudaSuccess &&
          cudaStreamWaitEvent(d2h, ev_done[slot], 0) == cudaSuccess &&
          cudaMemcpyAsync(static_cast<uint8_t*>(o_host) + off, slot_ptr(slot, 3), bytes, cudaMemcpyDeviceToHost, d2h) ==
              cudaSuccess &&
          cudaEventRecord(ev_free[slot], d2h) == cudaSuccess;
  }
  // the caller's stream completes after every copy (each copy-out follows its kernel)
  if (okc && st == MCS_OK)
    okc = cudaEventRecord(end, d2h) == cudaSuccess && cudaStreamWaitEvent(s, end, 0) == cudaSuccess;
  cleanup();
  if (st != MCS_OK) return st;
  return okc ? MCS_OK : MCS_ERR_CUDA;
}

mcs_status mcs_anchor_residual(const mcs_desc* desc, const void* q, const void* k, const void* v, const int32_t* perm,
                               const int32_t* idx, int K, const void* o_dense, void* r, mcs_stream stream) {
  Dims dm;
  mcs_status st = check_desc(desc, &dm);
  if (st != MCS_OK) return st;
  if (K < 1 || K > dm.N) return MCS_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(perm) || !aligned16(idx) ||
      !aligned16(o_dense) || !aligned16(r))
    return MCS_ERR_INVALID_ARG;
  uint32_t* status = nullptr;
  if ((st = device_state(&status, nullptr)) != MCS_OK) return st;
  return sparse_impl(dm, mcs::kEpiStoreResidual, q, k, v, perm, idx, K, o_dense, nullptr, r, status,
                     reinterpret_cast<cudaStream_t>(stream));
}

mcs_status mcs_residual_store(const mcs_desc* desc, const void* o_dense, const void* o_sparse, void* r,
                              mcs_stream stream) {
  Dims dm;
  mcs_status st = check_desc(desc, &dm);
  if (st != MCS_OK) return st;
  if (!aligned16(o_dense) || !aligned16(o_sparse) || !aligned16(r)) return MCS_ERR_INVALID_ARG;
  uint32_t* status = nullptr;
  int sms = 0;
  if ((st = device_state(&status, &sms)) != MCS_OK) return st;
  const size_t n = size_t(dm.BH) * dm.N * dm.d;
  return from_cuda(mcs::residual_op(true, dm.bf16, o_dense, o_sparse, r, n, sms, reinterpret_cast<cudaStream_t>(stream)));
}

mcs_status mcs_residual_apply(const mcs_desc* desc, const void* o_sparse, const void* r, void* o, mcs_stream stream) {
  Dims dm;
  mcs_status st = check_desc(desc, &dm);
  if (st != MCS_OK) return st;
  if (!aligned16(o_sparse) || !aligned16(r) || !aligned16(o)) return MCS_ERR_INVALID_ARG;
  uint32_t* status = nullptr;
  int sms = 0;
  if ((st = device_state(&status, &sms)) != MCS_OK) return st;
  const size_t n = size_t(dm.BH) * dm.N * dm.d;
  return from_cuda(mcs::residual_op(false, dm.bf16, o_sparse, r, o, n, sms, reinterpret_cast<cudaStream_t>(stream)));
}

mcs_status mcs_check_status(mcs_stream stream) {
  if (cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess) return MCS_ERR_CUDA;
  uint32_t* status = nullptr;
  mcs_status st = device_state(&status, nullptr);
  if (st != MCS_OK) return st;
  uint32_t v = 0;
  if (cudaMemcpy(&v, status, sizeof(v), cudaMemcpyDeviceToHost) != cudaSuccess) return MCS_ERR_CUDA;
  if (v != 0) {
    const uint32_t zero = 0;
    if (cudaMemcpy(status, &zero, sizeof(zero), cudaMemcpyHostToDevice) != cudaSuccess) return MCS_ERR_CUDA;
  }
  if (v & mcs::kStatusTimeout) return MCS_ERR_DEVICE_TIMEOUT;
  if (v & mcs::kStatusBounds) return MCS_ERR_DEVICE_BOUNDS;
  return MCS_OK;
}

const char* mcs_status_string(mcs_status status) {
  switch (status) {
    case MCS_OK: return "ok";
    case MCS_ERR_INVALID_ARG: return "invalid argument";
    case MCS_ERR_UNSUPPORTED: return "unsupported problem size or dtype";
    case MCS_ERR_WORKSPACE: return "workspace missing or too small";
    case MCS_ERR_CUDA: return "CUDA runtime error";
    case MCS_ERR_DEVICE_BOUNDS: return "device kernel met an out-of-range index";
    case MCS_ERR_DEVICE_TIMEOUT: return "device kernel wait timed out";
  }
  return "unknown status";
}

uint64_t mcs_launch_count(void) { return g_launches.load(std::memory_order_relaxed); }

mcs_status mcs_selftest_tc_mma(const void* a, const void* b, float* d, int mode, uint32_t mn_lbo, uint32_t mn_sbo,
                               mcs_stream stream) {
  if (!aligned16(a) || !aligned16(b) || !aligned16(d) || mode < 0 || mode > 2) return MCS_ERR_INVALID_ARG;
  uint32_t* status = nullptr;
  mcs_status st = device_state(&status, nullptr);
  if (st != MCS_OK) return st;
  return from_cuda(mcs::tc_probe(a, b, d, mode, mn_lbo, mn_sbo, status, reinterpret_cast<cudaStream_t>(stream)));
}

mcs_status mcs_selftest_wait_timeout(uint64_t limit_ns, uint64_t* elapsed_ns, mcs_stream stream) {
  if (limit_ns == 0 || limit_ns > 10ull * 1000 * 1000 * 1000) return MCS_ERR_INVALID_ARG;
  if (elapsed_ns != nullptr && (reinterpret_cast<uintptr_t>(elapsed_ns) & 7u) != 0) return MCS_ERR_INVALID_ARG;
  uint32_t* status = nullptr;
  mcs_status st = device_state(&status, nullptr);
  if (st != MCS_OK) return st;
  return from_cuda(mcs::wait_timeout_probe(limit_ns, reinterpret_cast<unsigned long long*>(elapsed_ns), status,
                                           reinterpret_cast<cudaStream_t>(stream)));
}

mcs_status mcs_selftest_ex2_rate(int iters, int nblocks, uint64_t* out, mcs_stream stream) {
  if (iters < 1 || iters > (1 << 24) || nblocks < 1 || nblocks > 65535 || out == nullptr ||
      (reinterpret_cast<uintptr_t>(out) & 7u) != 0)
    return MCS_ERR_INVALID_ARG;
  uint32_t* status = nullptr;
  mcs_status st = device_state(&status, nullptr);
  if (st != MCS_OK) return st;
  return from_cuda(mcs::ex2_rate_probe(iters, nblocks, reinterpret_cast<unsigned long long*>(out),
                                       reinterpret_cast<cudaStream_t>(stream)));
}

mcs_status mcs_selftest_tma_gather(const void* src, int nrows, const int32_t* rows, void* out, mcs_stream stream) {
  if (!aligned16(src) || !aligned16(rows) || !aligned16(out) || nrows < 1) return MCS_ERR_INVALID_ARG;
  uint32_t* status = nullptr;
  mcs_status st = device_state(&status, nullptr);
  if (st != MCS_OK) return st;
  return from_cuda(mcs::tma_gather_probe(src, nrows, rows, out, status, reinterpret_cast<cudaStream_t>(stream)));
}

}  // extern "C"

// ---------------------------------------------------------------- meta-cache ring
// One layer's entry: perm [BH, N_pad] int32 | idx [BH, G, K] int32 | residual
// [BH, N, d], each section starting on a 256-byte boundary. Two device slots
// take turns: the layer being computed sits in one while the next one is copied
// into the other on the ring's copy stream. Per slot, `copied` (recorded on the
// copy stream after every copy touching the slot) orders compute after copies,
// and `used` (recorded on the compute stream when the layer is released) orders
// copies after compute.
namespace {
struct EntryLayout {
  size_t perm, idx, res, total;
  size_t perm_bytes, idx_bytes, res_bytes;
};
EntryLayout entry_layout(const Dims& dm, int K) {
  EntryLayout e{};
  e.perm_bytes = size_t(dm.BH) * dm.N_pad * 4;
  e.idx_bytes = size_t(dm.BH) * dm.G * size_t(K) * 4;
  e.res_bytes = size_t(dm.BH) * dm.N * dm.d * (dm.bf16 ? 2 : 4);
  e.perm = 0;
  e.idx = align256(e.perm + e.perm_bytes);
  e.res = align256(e.idx + e.idx_bytes);
  e.total = align256(e.res + e.res_bytes);
  return e;
}
}  // namespace

struct mcs_cache_ring_s {
  Dims dm;
  int K = 0, n_layers = 0, device = 0;
  EntryLayout lay{};
  uint8_t* host = nullptr;  // [n_layers] entries, pinned (caller's)
  uint8_t* dev = nullptr;   // [2] slots (caller's)
  cudaStream_t copy = nullptr;
  cudaEvent_t copied[2] = {}, used[2] = {};
  int holds[2] = {-1, -1};  // layer whose entry the slot holds (or receives, once `copied` completes)
  int last = 1;             // slot of the most recent acquire
  int current[2] = {-1, -1};  // layer acquired into the slot and not yet released
  std::mutex mu;
};

namespace {
void ring_free(mcs_cache_ring r) {
  for (int i = 0; i < 2; ++i) {
    if (r->copied[i]) cudaEventDestroy(r->copied[i]);
    if (r->used[i]) cudaEventDestroy(r->used[i]);
  }
  if (r->copy) cudaStreamDestroy(r->copy);
  delete r;
}
bool ring_copy(mcs_cache_ring r, int slot, int layer, bool to_device) {
  uint8_t* d = r->dev + size_t(slot) * r->lay.total;
  uint8_t* h = r->host + size_t(layer) * r->lay.total;
  const cudaMemcpyKind kind = to_device ? cudaMemcpyHostToDevice : cudaMemcpyDeviceToHost;
  // copy after the slot's last compute use, then mark the slot's copies done
  if (cudaStreamWaitEvent(r->copy, r->used[slot], 0) != cudaSuccess) return false;
  const size_t off[3] = {r->lay.perm, r->lay.idx, r->lay.res};
  const size_t len[3] = {r->lay.perm_bytes, r->lay.idx_bytes, r->lay.res_bytes};
  for (int t = 0; t < 3; ++t) {
    void* dst = to_device ? static_cast<void*>(d + off[t]) : static_cast<void*>(h + off[t]);
    const void* src = to_device ? static_cast<const void*>(h + off[t]) : static_cast<const void*>(d + off[t]);
    if (cudaMemcpyAsync(dst, src, len[t], kind, r->copy) != cudaSuccess) return false;
  }
  return cudaEventRecord(r->copied[slot], r->copy) == cudaSuccess;
}
}  // namespace

size_t mcs_cache_entry_bytes(const mcs_desc* desc, int K) {
  Dims dm;
  if (check_desc(desc, &dm) != MCS_OK || K < 1 || K > dm.N) return 0;
  return entry_layout(dm, K).total;
}

mcs_status mcs_cache_ring_create(const mcs_desc* desc, int K, int n_layers, void* host_entries, void* device_slots,
                                 mcs_cache_ring* out) {
  if (out == nullptr) return MCS_ERR_INVALID_ARG;
  *out = nullptr;
  Dims dm;
  mcs_status st = check_desc(desc, &dm);
  if (st != MCS_OK) return st;
  if (K < 1 || K > dm.N || n_layers < 1) return MCS_ERR_INVALID_ARG;
  if (host_entries == nullptr || (reinterpret_cast<uintptr_t>(host_entries) & 255u) != 0) return MCS_ERR_INVALID_ARG;
  if (device_slots == nullptr || (reinterpret_cast<uintptr_t>(device_slots) & 255u) != 0) return MCS_ERR_INVALID_ARG;
  mcs_cache_ring r = new (std::nothrow) mcs_cache_ring_s();
  if (r == nullptr) return MCS_ERR_INVALID_ARG;
  r->dm = dm;
  r->K = K;
  r->n_layers = n_layers;
  r->lay = entry_layout(dm, K);
  r->host = static_cast<uint8_t*>(host_entries);
  r->dev = static_cast<uint8_t*>(device_slots);
  bool ok = cudaGetDevice(&r->device) == cudaSuccess &&
            cudaStreamCreateWithFlags(&r->copy, cudaStreamNonBlocking) == cudaSuccess;
  for (int i = 0; ok && i < 2; ++i)
    ok = cudaEventCreateWithFlags(&r->copied[i], cudaEventDisableTiming) == cudaSuccess &&
         cudaEventCreateWithFlags(&r->used[i], cudaEventDisableTiming) == cudaSuccess;
  if (!ok) {
    ring_free(r);
    return MCS_ERR_CUDA;
  }
  *out = r;
  return MCS_OK;
}

mcs_status mcs_cache_ring_acquire(mcs_cache_ring r, int layer, int load, int prefetch_next, mcs_stream stream,
                                  int32_t** perm, int32_t** idx, void** residual) {
  if (r == nullptr || layer < 0 || layer >= r->n_layers || perm == nullptr || idx == nullptr || residual == nullptr)
    return MCS_ERR_INVALID_ARG;
  std::lock_guard<std::mutex> lk(r->mu);
  if (r->current[0] == layer || r->current[1] == layer) return MCS_ERR_INVALID_ARG;  // already acquired
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  // the slot that holds (or is receiving) this layer, else the one not acquired last
  int slot = r->holds[0] == layer ? 0 : (r->holds[1] == layer ? 1 : (r->last ^ 1));
  if (r->current[slot] >= 0) return MCS_ERR_INVALID_ARG;  // both slots in use: release first
  if (load && r->holds[slot] != layer) {
    if (!ring_copy(r, slot, layer, true)) return MCS_ERR_CUDA;
  }
  r->holds[slot] = layer;  // the caller overwrites it when load == 0
  if (cudaStreamWaitEvent(s, r->copied[slot], 0) != cudaSuccess) return MCS_ERR_CUDA;
  r->current[slot] = layer;
  r->last = slot;
  if (prefetch_next && r->n_layers > 1) {
    const int nl = (layer + 1) % r->n_layers, ns = slot ^ 1;
    if (r->current[ns] < 0 && r->holds[ns] != nl) {
      if (!ring_copy(r, ns, nl, true)) return MCS_ERR_CUDA;
      r->holds[ns] = nl;
    }
  }
  uint8_t* d = r->dev + size_t(slot) * r->lay.total;
  *perm = reinterpret_cast<int32_t*>(d + r->lay.perm);
  *idx = reinterpret_cast<int32_t*>(d + r->lay.idx);
  *residual = d + r->lay.res;
  return MCS_OK;
}

mcs_status mcs_cache_ring_release(mcs_cache_ring r, int layer, int store, mcs_stream stream) {
  if (r == nullptr || layer < 0 || layer >= r->n_layers) return MCS_ERR_INVALID_ARG;
  std::lock_guard<std::mutex> lk(r->mu);
  const int slot = r->current[0] == layer ? 0 : (r->current[1] == layer ? 1 : -1);
  if (slot < 0) return MCS_ERR_INVALID_ARG;  // not acquired
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (cudaEventRecord(r->used[slot], s) != cudaSuccess) return MCS_ERR_CUDA;
  if (store && !ring_copy(r, slot, layer, false)) return MCS_ERR_CUDA;
  r->current[slot] = -1;
  return MCS_OK;
}

mcs_status mcs_cache_ring_destroy(mcs_cache_ring r) {
  if (r == nullptr) return MCS_ERR_INVALID_ARG;
  // the copies still queued read or write the caller's buffers: let them finish
  const bool ok = cudaStreamSynchronize(r->copy) == cudaSuccess;
  ring_free(r);
  return ok ? MCS_OK : MCS_ERR_CUDA;
}
