// tcgen05 indexer scan (index_tc.cu).
#pragma once
#include <cuda_runtime.h>
#include "v4a.h"

namespace v4a {
// Scores every visible entry of every query on the tensor cores when the key
// format allows it (fp8 per-128 or fp4 per-32 keys with an fp8 query).
// Returns false (nothing launched) when the shape is not handled; otherwise
// sets *rc and, when `hist` is non-null, also accumulates the 4096-bin
// score-key histogram per query and sets *hist_done.
bool index_score_tc(const v4a_index_args* a, float* scores, int64_t row, uint32_t* hist,
                    cudaStream_t stream, bool* hist_done, int* rc);
}  // namespace v4a
