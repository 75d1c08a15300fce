// tcgen05 indexer scan: placeholder until the tensor-core kernel lands.
#include "index_tc.h"

namespace v4a {
bool index_score_tc(const v4a_index_args*, float*, int64_t, uint32_t*, cudaStream_t, bool* hist_done,
                    int* rc) {
  *hist_done = false;
  *rc = V4A_OK;
  return false;
}
}  // namespace v4a
