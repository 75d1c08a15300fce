// Inverse RoPE on the attention output, fused with fp8 quantisation.
//
// Method: "DeepSeek V4 in vLLM: Efficient Long-context Attention", Method
// details fusion (2) (inverse RoPE then fp8 quant, feeding the o_lora fp8
// batched matmul) and Appendix "why inverse RoPE" (R_m^{-1} o_m removes the
// absolute position carried by V = K).
//
// One thread-block cluster of 8 CTAs per token; CTA r owns the r-th eighth
// of the token's H x D row bytes.  Each CTA brings its slice into shared
// memory with one bulk copy (one SM alone cannot pull a whole token quickly,
// eight can), rotates it by -angle while finding its amax, exchanges the amax
// with the other seven through distributed shared memory (one cluster
// barrier), then encodes and stores its slice: one pass over the data, no
// second kernel.

#include <cooperative_groups.h>

#include <mutex>

#include "tc_common.cuh"
#include "v4a_internal.h"

namespace cg = cooperative_groups;

namespace v4a {
namespace {

constexpr int kSlices = 8;               // CTAs per token (one cluster)
constexpr int kThreads = 256;
constexpr int kMaxSlice = 16 * 1024;     // bytes of one slice (H * D * 2 / 8 <= 16 KB)

struct OutDev {
  RopeFreq rope;
  int T, H, D, R, fmt;
  const int32_t* positions;
  const uint16_t* in;
  void* out;
  float* out_scale;
};

// The 8 values of a raw bf16 chunk starting at dim d0, rotated by -angle on
// the rope dims [first, first + R) (cs: cos [0, R/2), sin [R/2, R)).
__device__ __forceinline__ void rotated_chunk(const uint4 w, int d0, int first, int R, const float* cs, float* x) {
  const uint32_t u[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    float x0 = bf16_to_f32(uint16_t(u[i] & 0xffffu)), x1 = bf16_to_f32(uint16_t(u[i] >> 16));
    const int d = d0 + 2 * i;
    if (d >= first) {
      const int j = (d - first) >> 1;
      const float co = cs[j], si = -cs[R / 2 + j];
      const float y0 = x0 * co - x1 * si, y1 = x0 * si + x1 * co;
      x0 = y0; x1 = y1;
    }
    x[2 * i] = x0;
    x[2 * i + 1] = x1;
  }
}

__global__ void __cluster_dims__(kSlices, 1, 1) __launch_bounds__(kThreads)
inv_rope_quant_kernel(const OutDev a) {
  __shared__ __align__(128) uint4 rows_s[kMaxSlice / 16];
  __shared__ float cs[128];          // cos [0, R/2), sin [R/2, R)
  __shared__ float red[32];
  __shared__ float slice_amax;
  __shared__ uint64_t bar;
  cg::cluster_group cluster = cg::this_cluster();
  const int rank = int(cluster.block_rank());
  const int t = blockIdx.x / kSlices;
  const int per_head = a.D / 8;                        // 8-element chunks per head row
  const int nchunks = a.H * per_head / kSlices;        // chunks of this slice
  const int c0 = rank * nchunks;                       // first chunk of the slice within the token
  const int first = a.D - a.R;
  const uint16_t* in = a.in + int64_t(t) * a.H * a.D + int64_t(c0) * 8;
  if (threadIdx.x == 0) {
    tc::mbar_init(&bar, 1);
    tc::mbar_fence_init();
  }
  __syncthreads();   // the barrier is initialised before any thread waits on it
  pdl_trigger();
  pdl_wait();        // the attention output is the previous kernel's
  // the slice fits the buffer and the copy starts on 16 bytes (checked on the host as well)
  const bool copy_ok = nchunks > 0 && nchunks * 16 <= kMaxSlice && (reinterpret_cast<uintptr_t>(in) & 15) == 0;
  if (threadIdx.x == 0 && copy_ok) {
    tc::mbar_arrive_expect_tx(&bar, uint32_t(nchunks * 16));
    tc::bulk_load(rows_s, in, uint32_t(nchunks * 16), &bar);
  }
  rope_table(a.positions[t], a.R, a.rope, cs);
  // every thread waits for the copy (bounded; a copy that never lands leaves
  // this token's output unwritten rather than hanging the GPU)
  const long long t0 = clock64();
  bool landed = false;
  while (copy_ok && !(landed = tc::mbar_try_wait_sleep(&bar, 0, 20000u)) && clock64() - t0 < 2000000000LL) {}
  __syncthreads();

  if (a.fmt == V4A_OUT_BF16) {
    if (landed) {
      uint4* out = reinterpret_cast<uint4*>(static_cast<uint16_t*>(a.out) + int64_t(t) * a.H * a.D) + c0;
      for (int c = threadIdx.x; c < nchunks; c += kThreads) {
        float x[8];
        rotated_chunk(rows_s[c], ((c0 + c) % per_head) * 8, first, a.R, cs, x);
        uint32_t u[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) u[i] = uint32_t(f32_to_bf16(x[2 * i])) | (uint32_t(f32_to_bf16(x[2 * i + 1])) << 16);
        out[c] = make_uint4(u[0], u[1], u[2], u[3]);
      }
    }
    return;
  }
  // token amax over all heads and dims: CTA reduction, then across the cluster
  float amax = 0.f;
  for (int c = threadIdx.x; c < nchunks; c += kThreads) {
    float x[8];
    rotated_chunk(rows_s[c], ((c0 + c) % per_head) * 8, first, a.R, cs, x);
#pragma unroll
    for (int i = 0; i < 8; ++i) amax = fmaxf(amax, fabsf(x[i]));
  }
  amax = block_reduce<true>(amax, red);
  if (threadIdx.x == 0) slice_amax = amax;
  cluster.sync();
  if (threadIdx.x == 0) {
    float mx = 0.f;
    for (int r = 0; r < kSlices; ++r) mx = fmaxf(mx, *cluster.map_shared_rank(&slice_amax, r));
    red[0] = mx;
  }
  cluster.sync();   // no CTA leaves while others may still read its slice_amax
  const float tok = red[0];
  const float s = tok > 0.f ? tok / 448.f : 1.f;
  if (!landed) return;
  uint2* out = reinterpret_cast<uint2*>(static_cast<uint8_t*>(a.out) + int64_t(t) * a.H * a.D) + c0;
  for (int c = threadIdx.x; c < nchunks; c += kThreads) {
    float x[8];
    rotated_chunk(rows_s[c], ((c0 + c) % per_head) * 8, first, a.R, cs, x);
    uint32_t lo = 0, hi = 0;
#pragma unroll
    for (int i = 0; i < 4; ++i) lo |= uint32_t(f32_to_e4m3(x[i] / s)) << (8 * i);
#pragma unroll
    for (int i = 0; i < 4; ++i) hi |= uint32_t(f32_to_e4m3(x[4 + i] / s)) << (8 * i);
    out[c] = make_uint2(lo, hi);
  }
  if (rank == 0 && threadIdx.x == 0) a.out_scale[t] = s;
}

}  // namespace

int inv_rope_quant(const v4a_output_args* a, cudaStream_t stream) {
  if (!a) return V4A_ERR_INVALID_ARG;
  if (a->num_tokens < 0 || a->num_heads < 1 || a->dim < 8 || a->dim % 8) return V4A_ERR_INVALID_ARG;
  if (a->rope_dims < 0 || a->rope_dims > a->dim || a->rope_dims % 2) return V4A_ERR_INVALID_ARG;
  if (a->rope_dims > 128) return V4A_ERR_UNSUPPORTED;
  if (a->out_format != V4A_OUT_BF16 && a->out_format != V4A_OUT_FP8_TOKEN) return V4A_ERR_INVALID_ARG;
  // each of the 8 CTAs of a token takes a whole number of 16-byte chunks, at most 16 KB
  if ((int64_t(a->num_heads) * a->dim) % (8 * kSlices) != 0) return V4A_ERR_UNSUPPORTED;
  if (int64_t(a->num_heads) * a->dim * 2 / kSlices > kMaxSlice) return V4A_ERR_UNSUPPORTED;
  if (a->num_tokens == 0) return V4A_OK;
  if (!a->positions || !a->in || !a->out) return V4A_ERR_INVALID_ARG;
  if (reinterpret_cast<uintptr_t>(a->in) & 15) return V4A_ERR_UNSUPPORTED;   // bulk copies start on 16 bytes
  if (a->out_format == V4A_OUT_FP8_TOKEN && !a->out_scale) return V4A_ERR_INVALID_ARG;
  OutDev d;
  d.rope = make_rope_freq(a->rope_dims, a->rope_theta);
  d.T = a->num_tokens; d.H = a->num_heads; d.D = a->dim; d.R = a->rope_dims; d.fmt = a->out_format;
  d.positions = a->positions; d.in = a->in; d.out = a->out; d.out_scale = a->out_scale;
  if (launch_pdl(inv_rope_quant_kernel, dim3(a->num_tokens * kSlices), dim3(kThreads), 0, stream, d) != cudaSuccess)
    return V4A_ERR_CUDA;
  return cudaGetLastError() == cudaSuccess ? V4A_OK : V4A_ERR_CUDA;
}

}  // namespace v4a
