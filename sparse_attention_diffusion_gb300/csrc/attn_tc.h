// Host-side interface of the tcgen05 (bf16) attention and selection kernels.
#pragma once
#include <cstdint>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

namespace mcs {

struct TcAttnParams {
  const __nv_bfloat16* q;
  const __nv_bfloat16* k;
  const __nv_bfloat16* v;
  __nv_bfloat16* o;             // output rows (dense, plain, add-residual); may be null for lse-only
  float* lse;                   // dense: fp32 [BH, N] natural-log row LSE; may be null
  const int32_t* perm;          // sparse: [BH, N_pad]
  const int32_t* idx;           // sparse: [BH, G, K]
  const __nv_bfloat16* res_in;  // add-residual: R; store-residual: o_dense
  __nv_bfloat16* res_out;       // store-residual: R
  int BH, N, N_pad, C, G, K;
  int tiles_per_head;           // dense: ceil(N/128) query tiles; sparse: G groups
  float scale_log2;             // scale * log2(e)
  uint32_t* status;
};

struct TcColsumParams {
  const __nv_bfloat16* q;
  const __nv_bfloat16* k;
  const int32_t* perm;          // [BH, N_pad]
  const float* lse;             // [BH, N]
  float* scores;                // [nrows, N] fp32 rows of this launch
  int BH, N, N_pad, C, G;
  int row0;                     // first group row (bh * G + g) of this launch
  int nrows;                    // group rows of this launch (set by tc_colsum)
  float scale_log2;
  uint32_t* status;
};

cudaError_t tc_dense_attn(int D, const TcAttnParams& p, int BH, bool with_pv, cudaStream_t stream);
cudaError_t tc_sparse_attn(int D, int epi, const TcAttnParams& p, int BH, cudaStream_t stream);
cudaError_t tc_colsum(int D, int C, const TcColsumParams& p, int nrows, cudaStream_t stream);
cudaError_t tma_gather_probe(const void* src, int nrows, const int* rows, void* out, uint32_t* status,
                             cudaStream_t stream);
cudaError_t wait_timeout_probe(uint64_t limit_ns, unsigned long long* elapsed, uint32_t* status, cudaStream_t stream);
cudaError_t ex2_rate_probe(int iters, int nblocks, unsigned long long* out, cudaStream_t stream);
cudaError_t tc_probe(const void* a, const void* b, float* d, int mode, uint32_t lbo, uint32_t sbo, uint32_t* status,
                     cudaStream_t stream);

}  // namespace mcs
