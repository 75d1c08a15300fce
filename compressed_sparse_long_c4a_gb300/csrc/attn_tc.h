// tcgen05 sparse attention (attn_tc.cu).
#pragma once
#include <cuda_runtime.h>
#include "v4a.h"

namespace v4a {
size_t attn_tc_workspace_size(const v4a_attn_args* a);   // 0 when not handled

// The per-chunk results the attention kernel leaves in the workspace:
// o [T][splits][H][D] bf16 rows normalised by their chunk's softmax sum, and
// ml [T][splits][H][2] = (max in log2 units, sum); an empty chunk has max -inf.
// They are workspace: the fused output stage overwrites chunk 0's entries
// with the merged rows and their amax.
struct AttnPartials {
  uint16_t* o;
  float* ml;
  int splits;
};

// Launches the tensor-core attention when it handles the shapes (returns false
// otherwise, launching nothing); *rc is the call's result code.  With `keep`
// the chunk results stay in the workspace (described in *keep) and no merge
// kernel runs: the caller merges them.
//
// Long batches run as several launches of attn_tc_batch_queries(a) queries
// each, sharing the workspace.  With tn < 0 the call covers every query (with
// `keep`, only when they fit one launch); otherwise it covers queries
// [t0, t0 + tn), tn <= attn_tc_batch_queries(a), and a caller that merges the
// chunk results itself walks the launches one by one.
bool attn_tc(const v4a_attn_args* a, void* ws, size_t ws_bytes, cudaStream_t stream, int* rc,
             AttnPartials* keep = nullptr, int t0 = 0, int tn = -1);
int attn_tc_batch_queries(const v4a_attn_args* a);   // 0 when not handled
}  // namespace v4a
