// Inverse RoPE on the attention output, fused with fp8 quantisation.
//
// Method: "DeepSeek V4 in vLLM: Efficient Long-context Attention", Method
// details fusion (2) (inverse RoPE then fp8 quant, feeding the o_lora fp8
// batched matmul) and Appendix "why inverse RoPE" (R_m^{-1} o_m removes the
// absolute position carried by V = K).
//
// One CTA per token.  The R/2 rotation angles of position m are formed once
// (fp64, then reduced) into shared memory; every (head, pair) of the token is
// rotated by -angle.  For fp8 output the CTA first reduces the amax of the
// rotated token (one scale per token over all heads and dims), then encodes.

#include "v4a_common.cuh"
#include "v4a_internal.h"

namespace v4a {

__global__ void __launch_bounds__(512) inv_rope_quant_kernel(v4a_output_args a) {
  extern __shared__ float cs_s[];     // [R/2] cos, [R/2] sin
  __shared__ float red[32];
  const int t = blockIdx.x;
  const int m = a.positions[t];
  const int R = a.rope_dims, D = a.dim, HD = a.num_heads * a.dim;
  for (int j = threadIdx.x; j < R / 2; j += blockDim.x) {
    float c, s;
    rope_cos_sin(m, j, R, a.rope_theta, &c, &s);
    cs_s[j] = c;
    cs_s[R / 2 + j] = -s;             // inverse rotation
  }
  __syncthreads();
  const uint32_t* in = reinterpret_cast<const uint32_t*>(a.in + int64_t(t) * HD);
  const int first = D - R;
  auto rotated = [&](int pair, float* v0, float* v1) {
    const uint32_t w = in[pair];
    float x0 = bf16_to_f32(uint16_t(w & 0xffffu)), x1 = bf16_to_f32(uint16_t(w >> 16));
    const int d = (2 * pair) % D;
    if (d >= first) {
      const int j = (d - first) >> 1;
      const float c = cs_s[j], s = cs_s[R / 2 + j];
      const float y0 = x0 * c - x1 * s, y1 = x0 * s + x1 * c;
      x0 = y0; x1 = y1;
    }
    *v0 = x0; *v1 = x1;
  };
  const int npairs = HD / 2;
  if (a.out_format == V4A_OUT_BF16) {
    uint32_t* out = reinterpret_cast<uint32_t*>(static_cast<uint16_t*>(a.out) + int64_t(t) * HD);
    for (int p = threadIdx.x; p < npairs; p += blockDim.x) {
      float v0, v1;
      rotated(p, &v0, &v1);
      out[p] = uint32_t(f32_to_bf16(v0)) | (uint32_t(f32_to_bf16(v1)) << 16);
    }
    return;
  }
  float amax = 0.f;
  for (int p = threadIdx.x; p < npairs; p += blockDim.x) {
    float v0, v1;
    rotated(p, &v0, &v1);
    amax = fmaxf(amax, fmaxf(fabsf(v0), fabsf(v1)));
  }
  amax = block_reduce<true>(amax, red);
  const float s = amax > 0.f ? amax / 448.f : 1.f;
  uint16_t* out = reinterpret_cast<uint16_t*>(static_cast<uint8_t*>(a.out) + int64_t(t) * HD);
  for (int p = threadIdx.x; p < npairs; p += blockDim.x) {
    float v0, v1;
    rotated(p, &v0, &v1);
    out[p] = uint16_t(f32_to_e4m3(v0 / s)) | (uint16_t(f32_to_e4m3(v1 / s)) << 8);
  }
  if (threadIdx.x == 0) a.out_scale[t] = s;
}

int inv_rope_quant(const v4a_output_args* a, cudaStream_t stream) {
  if (!a) return V4A_ERR_INVALID_ARG;
  if (a->num_tokens < 0 || a->num_heads < 1 || a->dim < 2 || a->dim % 2) return V4A_ERR_INVALID_ARG;
  if (a->rope_dims < 0 || a->rope_dims > a->dim || a->rope_dims % 2) return V4A_ERR_INVALID_ARG;
  if (a->out_format != V4A_OUT_BF16 && a->out_format != V4A_OUT_FP8_TOKEN) return V4A_ERR_INVALID_ARG;
  if (a->num_tokens == 0) return V4A_OK;
  if (!a->positions || !a->in || !a->out) return V4A_ERR_INVALID_ARG;
  if (a->out_format == V4A_OUT_FP8_TOKEN && !a->out_scale) return V4A_ERR_INVALID_ARG;
  const size_t smem = size_t(a->rope_dims) * 4 + 16;
  inv_rope_quant_kernel<<<a->num_tokens, 512, smem, stream>>>(*a);
  return cudaGetLastError() == cudaSuccess ? V4A_OK : V4A_ERR_CUDA;
}

}  // namespace v4a
