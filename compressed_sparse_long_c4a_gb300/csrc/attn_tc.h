// tcgen05 sparse attention (attn_tc.cu).
#pragma once
#include <cuda_runtime.h>
#include "v4a.h"

namespace v4a {
size_t attn_tc_workspace_size(const v4a_attn_args* a);   // 0 when not handled
bool attn_tc(const v4a_attn_args* a, void* ws, size_t ws_bytes, cudaStream_t stream, int* rc);
}  // namespace v4a
