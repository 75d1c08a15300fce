// Internal entry points of libv4a (one per stage), called by the C ABI in api.cu.
#pragma once
#include <cuda_runtime.h>
#include "v4a.h"

namespace v4a {
int compress_insert(const v4a_compress_args* a, cudaStream_t stream);
size_t index_workspace_size(const v4a_index_args* a);
int index_scores_layout(const v4a_index_args* a, size_t* offset, int64_t* row_stride);
int index_topk(const v4a_index_args* a, void* ws, size_t ws_bytes, cudaStream_t stream);
int index_scores(const v4a_index_args* a, void* ws, size_t ws_bytes, cudaStream_t stream);
int index_select(const v4a_index_args* a, void* ws, size_t ws_bytes, cudaStream_t stream);
size_t attn_workspace_size(const v4a_attn_args* a);
int sparse_attn(const v4a_attn_args* a, void* ws, size_t ws_bytes, cudaStream_t stream);
int validate_attn(const v4a_attn_args* a);
int inv_rope_quant(const v4a_output_args* a, cudaStream_t stream);
int sparse_attn_out(const v4a_attn_args* attn, const v4a_output_args* out, void* ws, size_t ws_bytes,
                    cudaStream_t stream);
}  // namespace v4a
