// v4a_index_topk_static: the indexer scan + top-k with its scratch in a
// fixed, file-scope device array instead of a caller-supplied workspace.
//
// Who needs it: a caller that may not allocate device memory on the step
// path.  Examples are a serving loop that hands all free HBM to the paged KV
// pool at start-up (a later cudaMalloc would fail, and it also synchronises
// the device) and a foreign-language binding that has no device allocator of
// its own to hand out a workspace.  Such a caller passes only the arguments;
// the scratch below is the workspace.
//
// Nothing here allocates: the array is part of this library's device image.
// Its address is looked up on every call, on the current device, with
// cudaGetSymbolAddress (a cached address would go stale when a caller resets
// the device and the module is loaded again; the lookup costs ~1 us of host
// time and no device work).
//
// Every call on a device shares the one array.  Calls whose lifetimes overlap
// on the device (two streams, or two host threads, without an ordering between
// them) race on it and may return each other's selections: order them on one
// stream or with events.  The histogram and counter part of the scratch must
// start at zero; each call clears it on its own stream before the scan
// (a clearing kernel), so nothing depends on the array's initial contents.

#include "v4a_internal.h"

namespace v4a {
namespace {

constexpr size_t kScratchBytes = size_t(V4A_INDEX_STATIC_SCRATCH_BYTES);
__device__ __align__(256) unsigned char g_index_scratch[kScratchBytes];

// Device address of g_index_scratch on the current device.
int scratch_of_current_device(void** out) {
  void* p = nullptr;
  if (cudaGetSymbolAddress(&p, g_index_scratch) != cudaSuccess || !p) return V4A_ERR_CUDA;
  *out = p;
  return V4A_OK;
}

}  // namespace

int index_topk_static(const v4a_index_args* a, cudaStream_t stream) {
  if (!a) return V4A_ERR_INVALID_ARG;
  const size_t need = index_workspace_size(a);
  if (need == 0) return index_topk(a, nullptr, 0, stream);   // bad shape (its code) or no tokens
  if (need > kScratchBytes) return V4A_ERR_WORKSPACE;        // beyond the fixed scratch
  void* scratch = nullptr;
  const int rc = scratch_of_current_device(&scratch);
  if (rc) return rc;
  return index_topk(a, scratch, kScratchBytes, stream);
}

}  // namespace v4a

extern "C" int v4a_index_topk_static(const v4a_index_args* args, void* stream) {
  return v4a::index_topk_static(args, static_cast<cudaStream_t>(stream));
}
