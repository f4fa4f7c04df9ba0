// Internal entry points shared by the C ABI's translation units.
#pragma once
#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>

#include "mcs.h"

namespace mcs {

// Pass 2 + exact top-K of the anchor selection over every group row of the
// problem, given the pass-1 lse (required) and a score buffer of score_bytes
// bytes (device, 16-byte aligned) that holds the fp32 score rows of one launch:
// min(4,096, score_bytes / (N * 4)) rows per launch. Validates the description
// and the pointers; MCS_ERR_UNSUPPORTED when not even one row fits.
mcs_status anchor_select_rows(const mcs_desc* desc, const void* q, const void* k, const int32_t* perm,
                              const float* lse, int K, int32_t* idx, float* mass, float* scores, size_t score_bytes,
                              cudaStream_t stream);

}  // namespace mcs
