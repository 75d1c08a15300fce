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
// (max, sum) per chunk): one cluster of `csize` CTAs per token, CTA r owning
// heads [r*H/csize, (r+1)*H/csize).  Each thread merges one (head, 8-dim chunk)
// over all chunks of the query with the weights and the summation order of the
// stand-alone merge (four interleaved groups of chunks, then group 0 + 1 + 2 +
// 3), rounds to bf16 as the stored attention output would be, and leaves the
// row in shared memory; the rest is the output stage above (rotation by
// -angle, token amax through distributed shared memory, encode), so the bytes
// equal those of the two-call path.  The bf16 attention output never goes to
// HBM and one kernel boundary disappears.
constexpr int kMergeThreads = 1024;
constexpr int kMergeGroups = 4;          // chunk groups: chunk sp belongs to group sp % 4
constexpr int kMergeItems = kMergeThreads / kMergeGroups;   // (head, 8-dim chunk) items per round
constexpr int kMergeBatch = 9;           // chunk rows in flight per thread (34 chunks: one batch)
constexpr int kMergeMaxSplits = 64;
constexpr int kMergeMaxRows = 16;        // heads per CTA

struct MergeDev {
  RopeFreq rope;
  int T, H, D, R, fmt, splits;
  const int32_t* positions;
  const uint16_t* part_o;
  const float* part_ml;
  void* out;
  float* out_scale;
};

__global__ void __launch_bounds__(kMergeThreads) merge_out_kernel(const MergeDev a) {
  __shared__ __align__(128) uint4 rows_s[kMaxSlice / 16];
  __shared__ float4 part_s[kMergeGroups - 1][kMergeItems][2];
  __shared__ float wsm[kMergeMaxRows][kMergeMaxSplits];
  __shared__ float inv_s[kMergeMaxRows];
  __shared__ float cs[128];
  __shared__ float red[32];
  __shared__ float slice_amax;
  cg::cluster_group cluster = cg::this_cluster();
  const int csize = int(cluster.num_blocks());
  const int rank = int(cluster.block_rank());
  const int t = blockIdx.x / csize;
  const int hp = a.H / csize, h0 = rank * hp;
  const int per_head = a.D / 8;
  const int nchunks = hp * per_head;                   // 16-byte chunks of this CTA's rows
  const int first = a.D - a.R;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  pdl_trigger();
  rope_table(a.positions[t], a.R, a.rope, cs);        // positions are a step input
  pdl_wait();                                          // the chunk results are the previous kernel's
  // 1. chunk weights of every head of this CTA (as in the stand-alone merge)
  for (int hh = warp; hh < hp; hh += kMergeThreads / 32) {
    const float* ml = a.part_ml + (int64_t(t) * a.splits * a.H + h0 + hh) * 2;
    float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;
    if (lane < a.splits) { m0 = ml[int64_t(lane) * a.H * 2]; l0 = ml[int64_t(lane) * a.H * 2 + 1]; }
    if (lane + 32 < a.splits) { m1 = ml[int64_t(lane + 32) * a.H * 2]; l1 = ml[int64_t(lane + 32) * a.H * 2 + 1]; }
    const float mx = warp_max(fmaxf(m0, m1));
    const float w0 = m0 == -INFINITY ? 0.f : l0 * exp2f(m0 - mx);
    const float w1 = m1 == -INFINITY ? 0.f : l1 * exp2f(m1 - mx);
    if (lane < a.splits) wsm[hh][lane] = w0;
    if (lane + 32 < a.splits) wsm[hh][lane + 32] = w1;
    const float tot = warp_sum(w0 + w1);
    if (lane == 0) inv_s[hh] = tot > 0.f ? 1.f / tot : 0.f;
  }
  __syncthreads();
  // 2. merged rows, rounded to bf16, into shared memory.  Thread (g, i) sums
  //    the chunks of group g for item i of the round in increasing order (one
  //    warp = 32 consecutive items of one group: whole 512-byte runs per load);
  //    group 0 then adds groups 1, 2, 3 in that order.
  const int g = threadIdx.x / kMergeItems, il = threadIdx.x % kMergeItems;
  for (int base = 0; base < nchunks; base += kMergeItems) {
    const int c = base + il;
    float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    const bool live = c < nchunks;
    const int hh = live ? c / per_head : 0, cc = live ? c % per_head : 0;
    const uint16_t* po = a.part_o + (int64_t(t) * a.splits * a.H + h0 + hh) * a.D + cc * 8;
    if (a.splits == 1) {
      // one chunk: its normalised row is the attention output as stored
      if (live && g == 0) rows_s[c] = __ldcg(reinterpret_cast<const uint4*>(po));
      continue;
    }
    for (int u0 = 0; live && g + kMergeGroups * u0 < a.splits; u0 += kMergeBatch) {
      uint4 v[kMergeBatch];
#pragma unroll
      for (int u = 0; u < kMergeBatch; ++u) {
        const int sp = g + kMergeGroups * (u0 + u);
        v[u] = sp < a.splits ? __ldcg(reinterpret_cast<const uint4*>(po + int64_t(sp) * a.H * a.D))
                             : make_uint4(0, 0, 0, 0);
      }
#pragma unroll
      for (int u = 0; u < kMergeBatch; ++u) {
        const int sp = g + kMergeGroups * (u0 + u);
        const float w = sp < a.splits ? wsm[hh][sp] : 0.f;
        if (w == 0.f) continue;
        const uint32_t q[4] = {v[u].x, v[u].y, v[u].z, v[u].w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          acc[2 * j] = fmaf(w, bf16_to_f32(uint16_t(q[j] & 0xffffu)), acc[2 * j]);
          acc[2 * j + 1] = fmaf(w, bf16_to_f32(uint16_t(q[j] >> 16)), acc[2 * j + 1]);
        }
      }
    }
    if (g > 0) {
      part_s[g - 1][il][0] = make_float4(acc[0], acc[1], acc[2], acc[3]);
      part_s[g - 1][il][1] = make_float4(acc[4], acc[5], acc[6], acc[7]);
    }
    __syncthreads();
    if (g == 0 && live) {
#pragma unroll
      for (int g2 = 0; g2 < kMergeGroups - 1; ++g2) {
        const float4 x = part_s[g2][il][0], y = part_s[g2][il][1];
        acc[0] += x.x; acc[1] += x.y; acc[2] += x.z; acc[3] += x.w;
        acc[4] += y.x; acc[5] += y.y; acc[6] += y.z; acc[7] += y.w;
      }
      const float inv = inv_s[hh];
      uint32_t o[4];
#pragma unroll
      for (int j = 0; j < 4; ++j)
        o[j] = uint32_t(f32_to_bf16(acc[2 * j] * inv)) | (uint32_t(f32_to_bf16(acc[2 * j + 1] * inv)) << 16);
      rows_s[c] = make_uint4(o[0], o[1], o[2], o[3]);
    }
    __syncthreads();   // part_s is rewritten by the next round
  }
  __syncthreads();
  // 3. the output stage on those rows
  const int c0 = rank * nchunks;                       // first chunk of the slice within the token
  if (a.fmt == V4A_OUT_BF16) {
    uint4* out = reinterpret_cast<uint4*>(static_cast<uint16_t*>(a.out) + int64_t(t) * a.H * a.D) + c0;
    for (int c = threadIdx.x; c < nchunks; c += kMergeThreads) {
      float x[8];
      rotated_chunk(rows_s[c], ((c0 + c) % per_head) * 8, first, a.R, cs, x);
      uint32_t u[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) u[i] = uint32_t(f32_to_bf16(x[2 * i])) | (uint32_t(f32_to_bf16(x[2 * i + 1])) << 16);
      out[c] = make_uint4(u[0], u[1], u[2], u[3]);
    }
    return;
  }
  float amax = 0.f;
  for (int c = threadIdx.x; c < nchunks; c += kMergeThreads) {
    float x[8];
    rotated_chunk(rows_s[c], ((c0 + c) % per_head) * 8, first, a.R, cs, x);
#pragma unroll
    for (int i = 0; i < 8; ++i) amax = fmaxf(amax, fabsf(x[i]));
  }
  amax = block_reduce<true>(amax, red);
  if (threadIdx.x == 0) slice_amax = amax;
  cluster.sync();
  if (threadIdx.x < 32) {
    // one lane per CTA of the cluster: remote shared-memory reads take ~0.25 us
    // each on GB300, so they are issued together rather than one after another
    float mx = threadIdx.x < unsigned(csize) ? *cluster.map_shared_rank(&slice_amax, int(threadIdx.x)) : 0.f;
    mx = warp_max(mx);
    if (threadIdx.x == 0) red[0] = mx;
  }
  cluster.sync();   // no CTA leaves while others may still read its slice_amax
  const float tok = red[0];
  const float sc = tok > 0.f ? tok / 448.f : 1.f;
  uint2* out = reinterpret_cast<uint2*>(static_cast<uint8_t*>(a.out) + int64_t(t) * a.H * a.D) + c0;
  for (int c = threadIdx.x; c < nchunks; c += kMergeThreads) {
    float x[8];
    rotated_chunk(rows_s[c], ((c0 + c) % per_head) * 8, first, a.R, cs, x);
    uint32_t lo = 0, hi = 0;
#pragma unroll
    for (int i = 0; i < 4; ++i) lo |= uint32_t(f32_to_e4m3(x[i] / sc)) << (8 * i);
#pragma unroll
    for (int i = 0; i < 4; ++i) hi |= uint32_t(f32_to_e4m3(x[4 + i] / sc)) << (8 * i);
    out[c] = make_uint2(lo, hi);
  }
  if (rank == 0 && threadIdx.x == 0) a.out_scale[t] = sc;
}

// Largest cluster (16, else 8) the merge kernel can run with on this device.
int merge_cluster_size() {
  static int cached = 0;
  static std::once_flag once;
  std::call_once(once, [] {
    cudaFuncSetAttribute(merge_out_kernel, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    for (int cs : {16, 8}) {
      cudaLaunchConfig_t lc = {};
      lc.gridDim = dim3(cs);
      lc.blockDim = dim3(kMergeThreads);
      cudaLaunchAttribute at[1];
      at[0].id = cudaLaunchAttributeClusterDimension;
      at[0].val.clusterDim.x = cs;
      at[0].val.clusterDim.y = 1;
      at[0].val.clusterDim.z = 1;
      lc.attrs = at;
      lc.numAttrs = 1;
      int n = 0;
      if (cudaOccupancyMaxActiveClusters(&n, merge_out_kernel, &lc) == cudaSuccess && n > 0) {
        cached = cs;
        break;
      }
      cudaGetLastError();
    }
  });
  return cached;
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
  const int csize = merge_cluster_size();
  if (csize == 0 || a->num_heads % csize || a->num_heads / csize > kMergeMaxRows) return V4A_ERR_UNSUPPORTED;
  if (int64_t(a->num_heads / csize) * a->dim * 2 > kMaxSlice) return V4A_ERR_UNSUPPORTED;
  rc = validate_attn(at);
  if (rc) return rc;
  if (a->num_tokens == 0) return V4A_OK;
  // one attention launch and one merge launch per group of queries (long
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
    MergeDev d;
    d.rope = rope;
    d.T = tn; d.H = a->num_heads; d.D = a->dim; d.R = a->rope_dims; d.fmt = a->out_format;
    d.splits = p.splits; d.positions = a->positions + t0; d.part_o = p.o; d.part_ml = p.ml;
    d.out = static_cast<uint8_t*>(a->out) + size_t(t0) * a->num_heads * a->dim * out_elem;
    d.out_scale = a->out_scale ? a->out_scale + t0 : nullptr;
    cudaLaunchConfig_t lc = {};
    lc.gridDim = dim3(unsigned(tn * csize));
    lc.blockDim = dim3(kMergeThreads);
    lc.stream = stream;
    cudaLaunchAttribute la[2];
    la[0].id = cudaLaunchAttributeClusterDimension;
    la[0].val.clusterDim.x = unsigned(csize);
    la[0].val.clusterDim.y = 1;
    la[0].val.clusterDim.z = 1;
    la[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    la[1].val.programmaticStreamSerializationAllowed = 1;
    lc.attrs = la;
    lc.numAttrs = 2;
    if (cudaLaunchKernelEx(&lc, merge_out_kernel, d) != cudaSuccess) return V4A_ERR_CUDA;
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
