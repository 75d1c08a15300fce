// Test-only probe of the library's bounded mbarrier wait (tc::mbar_wait, the
// wait every tensor-core kernel's hand-offs use).  Never part of libv4a:
// tests/test_gpu_timeout.py compiles it on its own.
//
// probe_timeout: one CTA waits on an mbarrier that nothing ever arrives on, so
// the wait runs out its limit; the wait must then report V4A_DEV_TIMEOUT in the
// status word and return (no trap, no hang).
// probe_after: a trivial kernel that must still run and write its value, i.e.
// the context is usable after the timed-out wait.
#include <cuda_runtime.h>

#include "tc_common.cuh"

namespace {

__global__ void probe_timeout(int32_t* status, int32_t* gave_up) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    v4a::tc::mbar_init(&bar, 1);   // expects one arrival, which never comes
    abort_flag = 0;
    v4a::tc::mbar_fence_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) *gave_up = v4a::tc::mbar_wait(&bar, 0, status, &abort_flag) ? 0 : 1;
}

__global__ void probe_after(int32_t* out, int32_t v) {
  if (threadIdx.x == 0 && blockIdx.x == 0) *out = v;
}

}  // namespace

extern "C" int v4a_probe_wait_timeout(int32_t* status, int32_t* gave_up) {
  probe_timeout<<<1, 32>>>(status, gave_up);
  return static_cast<int>(cudaDeviceSynchronize());
}

extern "C" int v4a_probe_after(int32_t* out, int32_t v) {
  probe_after<<<1, 32>>>(out, v);
  return static_cast<int>(cudaDeviceSynchronize());
}
