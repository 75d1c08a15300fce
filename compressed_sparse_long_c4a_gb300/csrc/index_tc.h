// tcgen05 indexer scan (index_tc.cu).
#pragma once
#include <cuda_runtime.h>
#include "v4a.h"

namespace v4a {
// Scores every visible entry of every query on the tensor cores when the key
// format allows it (fp8 per-128 or fp4 per-32 keys with an fp8 query, 64
// heads x 128 dims).  Returns false (nothing launched) when the shape is not
// handled; otherwise launches and sets *rc.
bool index_score_tc(const v4a_index_args* a, float* scores, int64_t row, cudaStream_t stream, int* rc);
}  // namespace v4a
