// Host-side interface of the non-tensor-core kernels: residual, top-K, PDDP and
// the fp32 SIMT attention path.
#pragma once
#include <cstddef>
#include <cstdint>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

namespace mcs {

// ---------------------------------------------------------------- residual
cudaError_t residual_op(bool store, bool bf16, const void* a, const void* b, void* out, size_t nelem, int num_sms,
                        cudaStream_t s);

// ---------------------------------------------------------------- top-K
struct TopkParams {
  const float* scores;   // [nrows, N] score rows of this launch
  const int32_t* perm;   // [BH, N_pad] (for the real-query count of the mass)
  int32_t* idx;          // [BH*G, K]
  float* mass;           // [BH*G] or null
  int N, N_pad, C, G, K;
  int row0;              // first global group row of this launch
  uint32_t* status;
};
cudaError_t topk_rows(const TopkParams& p, int nrows, cudaStream_t stream);

// ---------------------------------------------------------------- PDDP
struct PddpProblem {
  const void* q;         // [BH, N, d] (fp32 or bf16)
  int32_t* perm;         // [BH, N_pad] output
  int32_t* group_of;     // [BH, N] output
  int BH, N, N_pad, C, G, d, iters;
  bool bf16;
  int num_sms;
  uint32_t* status;
  // optional direction tables [BH][2^L - 1][d] fp32 (L = ceil(log2 G)), node
  // (level, k) at row 2^level - 1 + k: start vectors (warm start) / final
  // directions; may alias (each row is read before it is written)
  const float* dirs_in;
  float* dirs_out;
};
// Rows of a PDDP direction table per head: 2^ceil(log2 G) - 1.
int pddp_dir_slots(int G);
// Workspace bytes for pddp_run (0 if unsupported).
size_t pddp_workspace_bytes(int BH, int N_pad, int C, int G, int d, bool bf16);
cudaError_t pddp_run(const PddpProblem& p, void* ws, size_t ws_bytes, cudaStream_t stream);
// Tensor-core chunk moments of one PDDP level (bf16, d = 128): per (head, chunk)
// the raw second moment sum x x^T [d x d], the sum of x [d] and the real-row
// count, for the chunks' rows gathered through perm (pddp_tc.cu).
cudaError_t pddp_moments_tc(const __nv_bfloat16* x, const int32_t* perm, const int* chunk_g0, const int* chunk_ng,
                            int nch, int BH, int N, int N_pad, int C, float* psum, int* pcnt, float* pcov,
                            int max_chunks, uint32_t* status, int num_sms, cudaStream_t stream);

// ---------------------------------------------------------------- fp32 SIMT attention
struct SimtAttnParams {
  const float* q;
  const float* k;
  const float* v;
  float* o;               // may be null (lse only, dense)
  float* lse;             // dense: [BH, N]; may be null
  const int32_t* perm;    // sparse
  const int32_t* idx;     // sparse
  const float* res_in;    // add-residual: R; store-residual: o_dense
  float* res_out;         // store-residual: R
  int N, N_pad, C, G, K, d;
  float scale;
  uint32_t* status;
};
cudaError_t simt_dense_attn(const SimtAttnParams& p, int BH, cudaStream_t stream);
cudaError_t simt_sparse_attn(int epi, const SimtAttnParams& p, int BH, cudaStream_t stream);

struct SimtColsumParams {
  const float* q;
  const float* k;
  const int32_t* perm;
  const float* lse;
  float* scores;          // [nrows, N]
  int N, N_pad, C, G, d, row0;
  float scale;
  uint32_t* status;
};
cudaError_t simt_colsum(const SimtColsumParams& p, int nrows, cudaStream_t stream);

}  // namespace mcs
