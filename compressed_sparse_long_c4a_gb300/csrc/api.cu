// The extern "C" entry points of libv4a (declared in include/v4a.h).  Each one
// forwards to the stage implementation in the matching .cu file.

#include "v4a_internal.h"

extern "C" {

int v4a_compress_insert(const v4a_compress_args* args, void* stream) {
  return v4a::compress_insert(args, static_cast<cudaStream_t>(stream));
}

size_t v4a_index_workspace_size(const v4a_index_args* args) {
  return v4a::index_workspace_size(args);
}

int v4a_index_scores_layout(const v4a_index_args* args, size_t* offset, int64_t* row_stride) {
  return v4a::index_scores_layout(args, offset, row_stride);
}

int v4a_index_topk(const v4a_index_args* args, void* workspace, size_t workspace_bytes,
                   void* stream) {
  return v4a::index_topk(args, workspace, workspace_bytes, static_cast<cudaStream_t>(stream));
}

int v4a_index_scores(const v4a_index_args* args, void* workspace, size_t workspace_bytes,
                     void* stream) {
  return v4a::index_scores(args, workspace, workspace_bytes, static_cast<cudaStream_t>(stream));
}

int v4a_index_select(const v4a_index_args* args, void* workspace, size_t workspace_bytes,
                     void* stream) {
  return v4a::index_select(args, workspace, workspace_bytes, static_cast<cudaStream_t>(stream));
}

size_t v4a_attn_workspace_size(const v4a_attn_args* args) { return v4a::attn_workspace_size(args); }

int v4a_sparse_attn(const v4a_attn_args* args, void* workspace, size_t workspace_bytes,
                    void* stream) {
  return v4a::sparse_attn(args, workspace, workspace_bytes, static_cast<cudaStream_t>(stream));
}

int v4a_inv_rope_quant(const v4a_output_args* args, void* stream) {
  return v4a::inv_rope_quant(args, static_cast<cudaStream_t>(stream));
}

int v4a_sparse_attn_out(const v4a_attn_args* attn, const v4a_output_args* out, void* workspace,
                        size_t workspace_bytes, void* stream) {
  return v4a::sparse_attn_out(attn, out, workspace, workspace_bytes, static_cast<cudaStream_t>(stream));
}

const char* v4a_status_string(int code) {
  switch (code) {
    case V4A_OK: return "ok";
    case V4A_ERR_INVALID_ARG: return "invalid argument";
    case V4A_ERR_UNSUPPORTED: return "unsupported shape or format";
    case V4A_ERR_RING_TOO_SMALL: return "ring capacity below window - 1 + tokens per sequence";
    case V4A_ERR_OUT_OF_PAGES: return "a page-size bucket has too few free pages";
    case V4A_ERR_WORKSPACE: return "workspace missing or too small";
    case V4A_ERR_CUDA: return "CUDA launch failed";
    default: return "unknown status";
  }
}

int v4a_abi_version(void) { return V4A_ABI_VERSION; }

}  // extern "C"
