// tcgen05 indexer scan (index_tc.cu).
#pragma once
#include <cuda_runtime.h>
#include "v4a.h"

namespace v4a {
// Scores every visible entry of every query on the tensor cores when the key
// format allows it (fp8 per-128 or fp4 per-32 keys with an fp8 query, 64
// heads x 128 dims).  Returns false (nothing launched) when the shape is not
// handled; otherwise launches and sets *rc.
// With `hist` non-null it also adds the top 12 bits of every score's
// order-preserving key to hist[t][4096] (which the caller has zeroed).
bool index_score_tc(const v4a_index_args* a, float* scores, int64_t row, uint32_t* hist, cudaStream_t stream,
                    int* rc);
// True when index_score_tc would launch for these arguments.
bool index_score_tc_supported(const v4a_index_args* a);
// The same for fp4 keys with power-of-two (MX) block scales, on the
// block-scaled MMA (index_mx.cu); V4A_IX_FP4_MX32 keys with an fp8 query, 64
// heads x 128 dims.
bool index_score_mx(const v4a_index_args* a, float* scores, int64_t row, uint32_t* hist, cudaStream_t stream,
                    int* rc);
bool index_score_mx_supported(const v4a_index_args* a);
}  // namespace v4a
