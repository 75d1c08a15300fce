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

#include "attn_tc.h"
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
  // (non-blocking polls: a thread suspended in try_wait resumed up to ~0.5 us late on GB300)
  while (copy_ok && !(landed = tc::mbar_test(&bar, 0)) && clock64() - t0 < 2000000000LL) {}
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
  if (threadIdx.x < 32) {
    // one lane per CTA of the cluster, all remote reads in flight together
    float mx = threadIdx.x < unsigned(kSlices) ? *cluster.map_shared_rank(&slice_amax, int(threadIdx.x)) : 0.f;
    mx = warp_max(mx);
    if (threadIdx.x == 0) red[0] = mx;
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

// ---- attention merge fused with the output stage ------------------------------
//
// For the tensor-core attention's chunk results (normalised bf16 rows plus
// (max, sum) per chunk), two kernels that need no thread-block cluster, so
// that both spread over every SM:
//  merge_amax: one CTA per (head, token) merges the head's chunk rows with the
//    weights and the summation order of the stand-alone merge (four
//    interleaved groups of chunks, then group 0 + 1 + 2 + 3), rounds to bf16
//    as the stored attention output would be, and leaves the row in the
//    workspace in place of the head's chunk-0 row, with the amax of the row
//    rotated by -angle in place of chunk 0's (max, sum);
//  encode_rows: kEncSlices CTAs per token take the token amax over its heads,
//    rotate their share of the merged rows and encode it.
// The bf16 attention output never leaves the workspace, and the bytes equal
// those of the two-call path.
constexpr int kMergeGroups = 4;          // chunk groups: chunk sp belongs to group sp % 4
constexpr int kMergeMaxSplits = 1024;    // chunks per query (rounds of kPer per group)
constexpr int kEncSlices = 16;           // encode CTAs per token
constexpr int kEncPer = 4;               // 16-byte chunks per encode thread held in registers

struct MergeDev {
  RopeFreq rope;
  int H, D, R, fmt, splits;
  const int32_t* positions;
  uint16_t* part_o;   // [T][splits][H][D]; chunk 0's rows receive the merged rows
  float* part_ml;     // [T][splits][H][2]; chunk 0's pairs receive (row amax, 0)
};

// kPer: chunks per group held in registers per round (one round when
// splits <= 4 * kPer), as small as the split count allows so that four CTAs
// fit an SM and every (head, token) of a decode batch has its loads in
// flight in one wave.
template <int kPer>
__global__ void __launch_bounds__(256, kPer <= 9 ? 4 : 2) merge_amax_kernel(const MergeDev a) {
  __shared__ float wsm[kMergeMaxSplits];
  __shared__ float inv_s;
  __shared__ float4 part_s[kMergeGroups - 1][64][2];
  __shared__ float cs[128];
  __shared__ float red[2];
  const int t = blockIdx.y, h = blockIdx.x;
  const int grp = threadIdx.x >> 6, c = threadIdx.x & 63;
  const bool active = c < a.D / 8;
  const bool fp8 = a.fmt == V4A_OUT_FP8_TOKEN;
  pdl_trigger();
  if (fp8) rope_table(a.positions[t], a.R, a.rope, cs);   // positions are a step input
  pdl_wait();                                              // the chunk results are the previous kernel's
  uint16_t* po = a.part_o + (int64_t(t) * a.splits * a.H + h) * a.D + c * 8;
  float* ml = a.part_ml + (int64_t(t) * a.splits * a.H + h) * 2;
  uint4 row = make_uint4(0, 0, 0, 0);   // group 0: the merged 8 values of item c
  if (a.splits == 1) {
    // one chunk: its normalised row is the attention output as stored
    if (grp == 0 && active) row = __ldcg(reinterpret_cast<const uint4*>(po));
  } else {
    // 1. this thread's first round of chunk rows, in flight together
    uint4 v[kPer];
#pragma unroll
    for (int u = 0; u < kPer; ++u) {
      const int sp = grp + u * kMergeGroups;
      v[u] = (active && sp < a.splits) ? __ldcg(reinterpret_cast<const uint4*>(po + int64_t(sp) * a.H * a.D))
                                       : make_uint4(0, 0, 0, 0);
    }
    // 2. weights of every chunk (warp 0), while those loads are in flight;
    //    lane l takes chunks l, l + 32, ... in order
    if (threadIdx.x < 32) {
      const int lane = threadIdx.x;
      float mx = -INFINITY;
      for (int sp = lane; sp < a.splits; sp += 32) mx = fmaxf(mx, ml[int64_t(sp) * a.H * 2]);
      mx = warp_max(mx);
      float tl = 0.f;
      for (int sp = lane; sp < a.splits; sp += 32) {
        const float m = ml[int64_t(sp) * a.H * 2], l = ml[int64_t(sp) * a.H * 2 + 1];
        const float w = m == -INFINITY ? 0.f : l * exp2f(m - mx);
        wsm[sp] = w;
        tl += w;
      }
      const float tot = warp_sum(tl);
      if (lane == 0) inv_s = tot > 0.f ? 1.f / tot : 0.f;
    }
    __syncthreads();
    // 3. weighted sum of this thread's chunks in increasing order, round by
    //    round (an empty chunk has weight 0)
    float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    for (int u0 = 0;; u0 += kPer) {
#pragma unroll
      for (int u = 0; u < kPer; ++u) {
        const int sp = grp + (u0 + u) * kMergeGroups;
        const float w = sp < a.splits ? wsm[sp] : 0.f;
        if (w == 0.f) continue;
        const uint32_t q[4] = {v[u].x, v[u].y, v[u].z, v[u].w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          acc[2 * j] = fmaf(w, bf16_to_f32(uint16_t(q[j] & 0xffffu)), acc[2 * j]);
          acc[2 * j + 1] = fmaf(w, bf16_to_f32(uint16_t(q[j] >> 16)), acc[2 * j + 1]);
        }
      }
      if ((u0 + kPer) * kMergeGroups >= a.splits) break;
#pragma unroll
      for (int u = 0; u < kPer; ++u) {   // the next round's rows
        const int sp = grp + (u0 + kPer + u) * kMergeGroups;
        v[u] = (active && sp < a.splits) ? __ldcg(reinterpret_cast<const uint4*>(po + int64_t(sp) * a.H * a.D))
                                         : make_uint4(0, 0, 0, 0);
      }
    }
    if (grp > 0) {
      part_s[grp - 1][c][0] = make_float4(acc[0], acc[1], acc[2], acc[3]);
      part_s[grp - 1][c][1] = make_float4(acc[4], acc[5], acc[6], acc[7]);
    }
    __syncthreads();
    if (grp == 0 && active) {
#pragma unroll
      for (int g2 = 0; g2 < kMergeGroups - 1; ++g2) {
        const float4 x = part_s[g2][c][0], y = part_s[g2][c][1];
        acc[0] += x.x; acc[1] += x.y; acc[2] += x.z; acc[3] += x.w;
        acc[4] += y.x; acc[5] += y.y; acc[6] += y.z; acc[7] += y.w;
      }
      const float inv = inv_s;
      uint32_t o[4];
#pragma unroll
      for (int j = 0; j < 4; ++j)
        o[j] = uint32_t(f32_to_bf16(acc[2 * j] * inv)) | (uint32_t(f32_to_bf16(acc[2 * j + 1] * inv)) << 16);
      row = make_uint4(o[0], o[1], o[2], o[3]);
    }
  }
  // 4. group 0: the merged row in place of chunk 0's, and its rotated amax
  float amax = 0.f;
  if (grp == 0 && active) {
    *reinterpret_cast<uint4*>(po) = row;   // this thread read chunk 0's item c above (or never will)
    if (fp8) {
      float x[8];
      rotated_chunk(row, c * 8, a.D - a.R, a.R, cs, x);
#pragma unroll
      for (int i = 0; i < 8; ++i) amax = fmaxf(amax, fabsf(x[i]));
    }
  }
  if (threadIdx.x < 64) {
    amax = warp_max(amax);
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = amax;
  }
  __syncthreads();   // also orders warp 0's reads of chunk 0's (max, sum) before the write below
  if (threadIdx.x == 0) {
    ml[0] = fmaxf(red[0], red[1]);
    ml[1] = 0.f;
  }
}

struct EncDev {
  RopeFreq rope;
  int H, D, R, fmt, splits;
  const int32_t* positions;
  const uint16_t* part_o;   // merged rows: chunk 0's rows of each token
  const float* part_ml;     // row amax: chunk 0's pairs
  void* out;
  float* out_scale;
};

__global__ void __launch_bounds__(256) encode_rows_kernel(const EncDev a) {
  __shared__ float cs[128];
  __shared__ float tok_s;
  const int t = blockIdx.x / kEncSlices, r = blockIdx.x % kEncSlices;
  const int per_head = a.D / 8;
  const int nch = a.H * per_head;                       // 16-byte bf16 chunks of the token
  const int per = (nch + kEncSlices - 1) / kEncSlices;
  const int cb = r * per, ce = min(nch, cb + per);
  const int first = a.D - a.R;
  pdl_trigger();
  rope_table(a.positions[t], a.R, a.rope, cs);
  pdl_wait();                                           // the merged rows are the previous kernel's
  const uint4* rows = reinterpret_cast<const uint4*>(a.part_o + int64_t(t) * a.splits * a.H * a.D);
  // this thread's first kEncPer chunks, in flight while the token amax is formed
  uint4 w[kEncPer];
#pragma unroll
  for (int i = 0; i < kEncPer; ++i) {
    const int c = cb + threadIdx.x + i * int(blockDim.x);
    w[i] = c < ce ? __ldcg(rows + c) : make_uint4(0, 0, 0, 0);
  }
  if (a.fmt == V4A_OUT_BF16) {
    __syncthreads();   // cs
    uint4* out = reinterpret_cast<uint4*>(static_cast<uint16_t*>(a.out) + int64_t(t) * a.H * a.D);
    auto put = [&](int c, uint4 v) {
      float x[8];
      rotated_chunk(v, (c % per_head) * 8, first, a.R, cs, x);
      uint32_t u[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) u[i] = uint32_t(f32_to_bf16(x[2 * i])) | (uint32_t(f32_to_bf16(x[2 * i + 1])) << 16);
      out[c] = make_uint4(u[0], u[1], u[2], u[3]);
    };
#pragma unroll
    for (int i = 0; i < kEncPer; ++i) {
      const int c = cb + threadIdx.x + i * int(blockDim.x);
      if (c < ce) put(c, w[i]);
    }
    for (int c = cb + threadIdx.x + kEncPer * int(blockDim.x); c < ce; c += blockDim.x) put(c, __ldcg(rows + c));
    return;
  }
  if (threadIdx.x < 32) {   // token amax = max over the heads' row amax
    const float* ml = a.part_ml + int64_t(t) * a.splits * a.H * 2;
    float m = 0.f;
    for (int h = threadIdx.x; h < a.H; h += 32) m = fmaxf(m, __ldcg(ml + int64_t(h) * 2));
    m = warp_max(m);
    if (threadIdx.x == 0) tok_s = m > 0.f ? m / 448.f : 1.f;
  }
  __syncthreads();
  const float sc = tok_s;
  uint2* out = reinterpret_cast<uint2*>(static_cast<uint8_t*>(a.out) + int64_t(t) * a.H * a.D);
  auto put = [&](int c, uint4 v) {
    float x[8];
    rotated_chunk(v, (c % per_head) * 8, first, a.R, cs, x);
    uint32_t lo = 0, hi = 0;
#pragma unroll
    for (int i = 0; i < 4; ++i) lo |= uint32_t(f32_to_e4m3(x[i] / sc)) << (8 * i);
#pragma unroll
    for (int i = 0; i < 4; ++i) hi |= uint32_t(f32_to_e4m3(x[4 + i] / sc)) << (8 * i);
    out[c] = make_uint2(lo, hi);
  };
#pragma unroll
  for (int i = 0; i < kEncPer; ++i) {
    const int c = cb + threadIdx.x + i * int(blockDim.x);
    if (c < ce) put(c, w[i]);
  }
  for (int c = cb + threadIdx.x + kEncPer * int(blockDim.x); c < ce; c += blockDim.x) put(c, __ldcg(rows + c));
  if (r == 0 && threadIdx.x == 0) a.out_scale[t] = sc;
}

}  // namespace

// Output-stage argument checks shared by both entry points.
static int check_output_args(const v4a_output_args* a, bool need_in) {
  if (!a) return V4A_ERR_INVALID_ARG;
  if (a->num_tokens < 0 || a->num_heads < 1 || a->dim < 8 || a->dim % 8) return V4A_ERR_INVALID_ARG;
  if (a->rope_dims < 0 || a->rope_dims > a->dim || a->rope_dims % 2) return V4A_ERR_INVALID_ARG;
  if (a->rope_dims > 128) return V4A_ERR_UNSUPPORTED;
  if (a->out_format != V4A_OUT_BF16 && a->out_format != V4A_OUT_FP8_TOKEN) return V4A_ERR_INVALID_ARG;
  if (a->num_tokens == 0) return V4A_OK;
  if (!a->positions || !a->out || (need_in && !a->in)) return V4A_ERR_INVALID_ARG;
  if (a->out_format == V4A_OUT_FP8_TOKEN && !a->out_scale) return V4A_ERR_INVALID_ARG;
  return V4A_OK;
}

int sparse_attn_out(const v4a_attn_args* at, const v4a_output_args* a, void* ws, size_t ws_bytes,
                    cudaStream_t stream) {
  if (!at) return V4A_ERR_INVALID_ARG;
  int rc = check_output_args(a, false);
  if (rc) return rc;
  if (a->num_tokens != at->batch.num_tokens || a->num_heads != at->num_heads || a->dim != at->kv.dim)
    return V4A_ERR_INVALID_ARG;
  if (a->dim > 512) return V4A_ERR_UNSUPPORTED;   // one thread per 8 dims of a row, 64 per group
  rc = validate_attn(at);
  if (rc) return rc;
  if (a->num_tokens == 0) return V4A_OK;
  // one attention, merge and encode launch per group of queries (long
  // chunked-prefill batches take several, sharing the workspace)
  const int Tb = attn_tc_batch_queries(at);
  if (Tb == 0) return V4A_ERR_UNSUPPORTED;
  RopeFreq rope = make_rope_freq(a->rope_dims, a->rope_theta);
  const size_t out_elem = a->out_format == V4A_OUT_BF16 ? 2 : 1;
  for (int t0 = 0; t0 < a->num_tokens; t0 += Tb) {
    const int tn = a->num_tokens - t0 < Tb ? a->num_tokens - t0 : Tb;
    AttnPartials p{};
    if (!attn_tc(at, ws, ws_bytes, stream, &rc, &p, t0, tn)) return V4A_ERR_UNSUPPORTED;
    if (rc) return rc;
    if (p.splits > kMergeMaxSplits) return V4A_ERR_UNSUPPORTED;
    MergeDev m;
    m.rope = rope;
    m.H = a->num_heads; m.D = a->dim; m.R = a->rope_dims; m.fmt = a->out_format; m.splits = p.splits;
    m.positions = a->positions + t0; m.part_o = p.o; m.part_ml = p.ml;
    auto merge = p.splits <= 16 ? merge_amax_kernel<4> : p.splits <= 36 ? merge_amax_kernel<9> : merge_amax_kernel<16>;
    if (launch_pdl(merge, dim3(unsigned(a->num_heads), unsigned(tn)), dim3(256), 0, stream, m) != cudaSuccess)
      return V4A_ERR_CUDA;
    EncDev e;
    e.rope = rope;
    e.H = a->num_heads; e.D = a->dim; e.R = a->rope_dims; e.fmt = a->out_format; e.splits = p.splits;
    e.positions = a->positions + t0; e.part_o = p.o; e.part_ml = p.ml;
    e.out = static_cast<uint8_t*>(a->out) + size_t(t0) * a->num_heads * a->dim * out_elem;
    e.out_scale = a->out_scale ? a->out_scale + t0 : nullptr;
    if (launch_pdl(encode_rows_kernel, dim3(unsigned(tn * kEncSlices)), dim3(256), 0, stream, e) != cudaSuccess)
      return V4A_ERR_CUDA;
  }
  return cudaGetLastError() == cudaSuccess ? V4A_OK : V4A_ERR_CUDA;
}

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
