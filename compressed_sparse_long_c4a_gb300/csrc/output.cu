// Inverse RoPE on the attention output, fused with fp8 quantisation.
//
// Method: "DeepSeek V4 in vLLM: Efficient Long-context Attention", Method
// details fusion (2) (inverse RoPE then fp8 quant, feeding the o_lora fp8
// batched matmul) and Appendix "why inverse RoPE" (R_m^{-1} o_m removes the
// absolute position carried by V = K).
//
// One thread-block cluster of kSlices CTAs per token; CTA r of the cluster
// owns heads [r*hs, (r+1)*hs).  Each thread loads its 8-element chunks once
// (16-byte loads), rotates them by -angle in registers and keeps them there.
// For fp8 output the token's amax is reduced inside each CTA, exchanged
// across the cluster through distributed shared memory (one barrier.cluster
// on each side), and every CTA then encodes its own chunks: one pass over the
// data, no second kernel.

#include <cooperative_groups.h>

#include "v4a_common.cuh"
#include "v4a_internal.h"

namespace cg = cooperative_groups;

namespace v4a {
namespace {

constexpr int kSlices = 8;       // CTAs per token (one cluster)
constexpr int kThreads = 256;
constexpr int kMaxChunks = 8;    // 8-element chunks per thread (64 values in registers)

struct OutDev {
  RopeFreq rope;
  int T, H, D, R, fmt;
  const int32_t* positions;
  const uint16_t* in;
  void* out;
  float* out_scale;
};

__global__ void __cluster_dims__(kSlices, 1, 1) __launch_bounds__(kThreads)
inv_rope_quant_kernel(const OutDev a) {
  __shared__ float cs[128];          // cos [0, R/2), sin [R/2, R)
  __shared__ float red[32];
  __shared__ float cluster_amax;
  cg::cluster_group cluster = cg::this_cluster();
  const int rank = int(cluster.block_rank());
  const int t = blockIdx.x / kSlices;
  const int m = a.positions[t];
  rope_table(m, a.R, a.rope, cs);
  __syncthreads();
  const int hs = (a.H + kSlices - 1) / kSlices;
  const int h0 = rank * hs, h1 = min(a.H, h0 + hs);
  const int per_head = a.D / 8;                       // chunks per head row
  const int nchunks = max(0, h1 - h0) * per_head;
  const int first = a.D - a.R;
  const uint4* in = reinterpret_cast<const uint4*>(a.in + (int64_t(t) * a.H + h0) * a.D);

  float v[kMaxChunks][8];
  float amax = 0.f;
#pragma unroll
  for (int k = 0; k < kMaxChunks; ++k) {
    const int c = threadIdx.x + k * kThreads;
    if (c < nchunks) {
      const uint4 w = in[c];
      const uint32_t u[4] = {w.x, w.y, w.z, w.w};
      const int d0 = (c % per_head) * 8;
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        float x0 = bf16_to_f32(uint16_t(u[i] & 0xffffu)), x1 = bf16_to_f32(uint16_t(u[i] >> 16));
        const int d = d0 + 2 * i;
        if (d >= first) {
          const int j = (d - first) >> 1;
          const float co = cs[j], si = -cs[a.R / 2 + j];    // rotate by -angle
          const float y0 = x0 * co - x1 * si, y1 = x0 * si + x1 * co;
          x0 = y0; x1 = y1;
        }
        v[k][2 * i] = x0;
        v[k][2 * i + 1] = x1;
        amax = fmaxf(amax, fmaxf(fabsf(x0), fabsf(x1)));
      }
    }
  }
  if (a.fmt == V4A_OUT_BF16) {
    uint4* out = reinterpret_cast<uint4*>(static_cast<uint16_t*>(a.out) + (int64_t(t) * a.H + h0) * a.D);
#pragma unroll
    for (int k = 0; k < kMaxChunks; ++k) {
      const int c = threadIdx.x + k * kThreads;
      if (c < nchunks) {
        uint32_t u[4];
#pragma unroll
        for (int i = 0; i < 4; ++i)
          u[i] = uint32_t(f32_to_bf16(v[k][2 * i])) | (uint32_t(f32_to_bf16(v[k][2 * i + 1])) << 16);
        out[c] = make_uint4(u[0], u[1], u[2], u[3]);
      }
    }
    return;
  }
  // token amax: CTA reduction, then across the cluster through DSMEM
  amax = block_reduce<true>(amax, red);
  if (threadIdx.x == 0) cluster_amax = amax;
  cluster.sync();
  if (threadIdx.x == 0) {
    float mx = 0.f;
    for (int r = 0; r < kSlices; ++r) mx = fmaxf(mx, *cluster.map_shared_rank(&cluster_amax, r));
    red[0] = mx;
  }
  cluster.sync();   // no CTA leaves while others may still read its cluster_amax
  const float tok = red[0];
  const float s = tok > 0.f ? tok / 448.f : 1.f;
  uint2* out = reinterpret_cast<uint2*>(static_cast<uint8_t*>(a.out) + (int64_t(t) * a.H + h0) * a.D);
#pragma unroll
  for (int k = 0; k < kMaxChunks; ++k) {
    const int c = threadIdx.x + k * kThreads;
    if (c < nchunks) {
      uint32_t lo = 0, hi = 0;
#pragma unroll
      for (int i = 0; i < 4; ++i) lo |= uint32_t(f32_to_e4m3(v[k][i] / s)) << (8 * i);
#pragma unroll
      for (int i = 0; i < 4; ++i) hi |= uint32_t(f32_to_e4m3(v[k][4 + i] / s)) << (8 * i);
      out[c] = make_uint2(lo, hi);
    }
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
  const int hs = (a->num_heads + kSlices - 1) / kSlices;
  if (int64_t(hs) * (a->dim / 8) > int64_t(kThreads) * kMaxChunks) return V4A_ERR_UNSUPPORTED;
  if (a->num_tokens == 0) return V4A_OK;
  if (!a->positions || !a->in || !a->out) return V4A_ERR_INVALID_ARG;
  if (a->out_format == V4A_OUT_FP8_TOKEN && !a->out_scale) return V4A_ERR_INVALID_ARG;
  OutDev d;
  d.rope = make_rope_freq(a->rope_dims, a->rope_theta);
  d.T = a->num_tokens; d.H = a->num_heads; d.D = a->dim; d.R = a->rope_dims; d.fmt = a->out_format;
  d.positions = a->positions; d.in = a->in; d.out = a->out; d.out_scale = a->out_scale;
  inv_rope_quant_kernel<<<a->num_tokens * kSlices, kThreads, 0, stream>>>(d);
  return cudaGetLastError() == cudaSuccess ? V4A_OK : V4A_ERR_CUDA;
}

}  // namespace v4a
