// Shared-K=V sparse attention over the selected compressed entries plus the
// uncompressed sliding window.
//
// Method: "DeepSeek V4 in vLLM: Efficient Long-context Attention",
// Background (shared key/value vectors; attend to the top-k compressed
// tokens; 128-token window over uncompressed tokens) and Appendix ("why
// inverse RoPE": with v_n = k_n the output is sum softmax(q.k_n) k_n; "why the
// short window": the window is [m-127, m]).
//
// Per query the key list is [selected entries (idx row, -1 skipped) or all
// visible entries] ++ [window positions max(0, m-W+1) .. m].  The list is cut
// into `splits` contiguous ranges; one CTA per (split, query, group of 16
// heads) walks its range in chunks of kChunk keys staged in shared memory
// (raw bf16 or e4m3 bytes + the per-row fp32 scale, so fp8 values stay
// exact).  Each warp owns one head and keeps its online-softmax state
// (m, l, o) in registers across chunks.  With one split the CTA writes the
// bf16 output directly; otherwise partials go to the workspace and
// attn_combine merges them.

#include "v4a_common.cuh"
#include "v4a_internal.h"
#include "attn_tc.h"

namespace v4a {

constexpr int kChunk = 128;

struct AttnDev {
  int T, H, D, ratio, fmt, wfmt, wlen, k, splits;
  const int32_t* seq_ids;
  const int32_t* positions;
  v4a_cache kv;
  int64_t block_bytes;
  const int32_t* idx;
  RingDev wring;
  const uint16_t* q;
  float scale;
  float* part_o;     // [T][splits][H][D]
  float* part_ml;    // [T][splits][H][2]
  uint16_t* out;     // [T][H][D] (written directly when splits == 1)
  float* lse;
  int32_t* status;
};

__device__ __forceinline__ int list_len(const AttnDev& a, int m, int* nsel, int* wstart) {
  const int nvis = (m + 1) / a.ratio;
  *nsel = a.idx ? a.k : nvis;
  *wstart = max(0, m - a.wlen + 1);
  return *nsel + (m - *wstart + 1);
}

template <int NJ>
__global__ void __launch_bounds__(512) attn_split_simt(AttnDev a) {
  extern __shared__ uint8_t smem[];
  const int t = blockIdx.y, sp = blockIdx.x;
  const int b = a.seq_ids[t], m = a.positions[t];
  int nsel, wstart;
  const int L = list_len(a, m, &nsel, &wstart);
  const int per = (L + a.splits - 1) / a.splits;
  const int lo = sp * per, hi = min(L, lo + per);
  const int D = a.D;
  const int rstride = 2 * D;
  uint8_t* rows = smem;                                                        // [kChunk][2D]
  float* kscale = reinterpret_cast<float*>(smem + size_t(kChunk) * rstride);  // [kChunk]
  int* kfmt = reinterpret_cast<int*>(kscale + kChunk);                         // [kChunk], -1 invalid
  const int nvis = (m + 1) / a.ratio;
  const int E = entries_per_block(a.ratio);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, nw = blockDim.x >> 5;
  const int h = blockIdx.z * nw + warp;
  const bool has_head = h < a.H;
  float q[NJ], o[NJ];
  if (has_head) {
    const uint16_t* qh = a.q + (int64_t(t) * a.H + h) * D;
#pragma unroll
    for (int j = 0; j < NJ; ++j) { q[j] = bf16_to_f32(qh[lane + 32 * j]); o[j] = 0.f; }
  }
  float mx = -INFINITY, l = 0.f;
  for (int c0 = lo; c0 < hi; c0 += kChunk) {
    const int c1 = min(hi, c0 + kChunk);
    __syncthreads();   // previous chunk fully consumed
    // stage keys: one warp per key row
    for (int li = c0 + warp; li < c1; li += nw) {
      const int r = li - c0;
      const uint8_t* src = nullptr;
      int f = -1;
      float s = 1.f;
      if (li < nsel) {
        const int e = a.idx ? a.idx[int64_t(t) * a.k + li] : li;
        if (e >= 0) {
          if (e >= nvis) {
            if (lane == 0 && blockIdx.z == 0) report(a.status, V4A_DEV_BAD_INDEX);
          } else {
            const int64_t blk = block_of(a.kv, b, e, (lane == 0 && blockIdx.z == 0) ? a.status : nullptr);
            if (blk >= 0) {
              const uint8_t* base = static_cast<const uint8_t*>(a.kv.pool) + blk * a.block_bytes;
              const int slot = e % E;
              f = a.fmt;
              src = base + int64_t(slot) * (a.fmt == V4A_KV_BF16 ? 2 * D : D);
              if (a.fmt == V4A_KV_FP8_TOKEN)
                s = reinterpret_cast<const float*>(base + int64_t(E) * D)[slot];
            }
          }
        }
      } else {
        const int p = wstart + (li - nsel);
        uint8_t* wrow;
        float* wsc;
        ring_slot(a.wring, b, p % a.wring.cap, &wrow, &wsc, (lane == 0 && blockIdx.z == 0) ? a.status : nullptr);
        if (wrow) {
          f = a.wfmt;
          src = wrow;
          if (wsc) s = *wsc;
        }
      }
      if (src) {
        const int nb = f == V4A_KV_BF16 ? 2 * D : D;
        for (int i = lane * 4; i < nb; i += 128)
          *reinterpret_cast<uint32_t*>(rows + size_t(r) * rstride + i) =
              *reinterpret_cast<const uint32_t*>(src + i);
      }
      if (lane == 0) { kscale[r] = s; kfmt[r] = f; }
    }
    __syncthreads();
    if (!has_head) continue;
    const int nk = c1 - c0;
    for (int r = 0; r < nk; ++r) {
      const int f = kfmt[r];
      if (f < 0) continue;
      float kv[NJ];
      const uint8_t* row = rows + size_t(r) * rstride;
      if (f == V4A_KV_BF16) {
#pragma unroll
        for (int j = 0; j < NJ; ++j)
          kv[j] = bf16_to_f32(reinterpret_cast<const uint16_t*>(row)[lane + 32 * j]);
      } else {
        const float s = kscale[r];
#pragma unroll
        for (int j = 0; j < NJ; ++j) kv[j] = e4m3_to_f32(row[lane + 32 * j]) * s;
      }
      float dot = 0.f;
#pragma unroll
      for (int j = 0; j < NJ; ++j) dot = fmaf(q[j], kv[j], dot);
      dot = warp_sum(dot);
      const float z = dot * a.scale;
      const float mn = fmaxf(mx, z);
      const float corr = expf(mx - mn);
      const float p = expf(z - mn);
      l = l * corr + p;
#pragma unroll
      for (int j = 0; j < NJ; ++j) o[j] = fmaf(p, kv[j], o[j] * corr);
      mx = mn;
    }
  }
  if (!has_head) return;
  if (a.splits == 1) {
    const float inv = 1.f / l;
    uint16_t* out = a.out + (int64_t(t) * a.H + h) * D;
#pragma unroll
    for (int j = 0; j < NJ; ++j) out[lane + 32 * j] = f32_to_bf16(o[j] * inv);
    if (a.lse && lane == 0) a.lse[int64_t(t) * a.H + h] = mx + logf(l);
    return;
  }
  const int64_t pi = (int64_t(t) * a.splits + sp) * a.H + h;
  float* po = a.part_o + pi * D;
#pragma unroll
  for (int j = 0; j < NJ; ++j) po[lane + 32 * j] = o[j];
  if (lane == 0) { a.part_ml[pi * 2] = mx; a.part_ml[pi * 2 + 1] = l; }
}

__global__ void attn_combine(int T, int H, int D, int splits, const float* part_o,
                             const float* part_ml, uint16_t* out, float* lse) {
  const int t = blockIdx.y, h = blockIdx.x;
  float mx = -INFINITY;
  for (int s = 0; s < splits; ++s) mx = fmaxf(mx, part_ml[((int64_t(t) * splits + s) * H + h) * 2]);
  float l = 0.f;
  for (int s = 0; s < splits; ++s) {
    const int64_t pi = (int64_t(t) * splits + s) * H + h;
    const float ms = part_ml[pi * 2];
    if (ms != -INFINITY) l += part_ml[pi * 2 + 1] * expf(ms - mx);
  }
  const float inv = 1.f / l;
  for (int d = threadIdx.x; d < D; d += blockDim.x) {
    float acc = 0.f;
    for (int s = 0; s < splits; ++s) {
      const int64_t pi = (int64_t(t) * splits + s) * H + h;
      const float ms = part_ml[pi * 2];
      if (ms != -INFINITY) acc = fmaf(part_o[pi * D + d], expf(ms - mx), acc);
    }
    out[(int64_t(t) * H + h) * D + d] = f32_to_bf16(acc * inv);
  }
  if (lse && threadIdx.x == 0) lse[int64_t(t) * H + h] = mx + logf(l);
}

// ------------------------------------------------------------------------------

// Shapes and formats only (enough to size the workspace).
static int validate_shape(const v4a_attn_args* a) {
  if (!a) return V4A_ERR_INVALID_ARG;
  const v4a_batch& B = a->batch;
  if (B.num_tokens < 0 || B.num_seqs <= 0) return V4A_ERR_INVALID_ARG;
  if (B.num_tokens > 65535) return V4A_ERR_UNSUPPORTED;
  const v4a_cache& c = a->kv;
  if (c.ratio != 4 && c.ratio != 128) return V4A_ERR_INVALID_ARG;
  if (c.num_blocks <= 0 || c.max_blocks <= 0) return V4A_ERR_INVALID_ARG;
  if (c.format != V4A_KV_BF16 && c.format != V4A_KV_FP8_TOKEN && c.format != V4A_KV_FP8_DSV4)
    return V4A_ERR_INVALID_ARG;
  if (a->window_format != V4A_KV_BF16 && a->window_format != V4A_KV_FP8_TOKEN) return V4A_ERR_INVALID_ARG;
  if (a->window_len < 1 || a->window_cap < 1) return V4A_ERR_INVALID_ARG;
  // every query's window [m - window_len + 1, m] must be in the ring at once
  // (the batch's newest positions were written by the compress call before)
  if (int64_t(a->window_cap) < int64_t(a->window_len) - 1 + B.max_new_per_seq) return V4A_ERR_RING_TOO_SMALL;
  if (a->idx && (a->k < 0 || a->k > 65536)) return V4A_ERR_INVALID_ARG;   // k = 0: window only
  const int D = c.dim;
  if (D != 64 && D != 128 && D != 256 && D != 512) return V4A_ERR_UNSUPPORTED;
  if (a->num_heads < 1 || a->num_heads > 256) return V4A_ERR_UNSUPPORTED;
  return V4A_OK;
}

static int validate(const v4a_attn_args* a, bool need_out = true) {
  const int rc = validate_shape(a);
  if (rc) return rc;
  if (a->batch.num_tokens == 0) return V4A_OK;
  if (!a->batch.seq_ids || !a->batch.positions || !a->q || (need_out && !a->out) || !a->kv.pool ||
      !a->kv.block_table)
    return V4A_ERR_INVALID_ARG;
  // key rows are read as 4-byte words (cache rows start on 4 bytes within a block)
  if ((reinterpret_cast<uintptr_t>(a->kv.pool) & 3) ||
      (!a->window_pages && (reinterpret_cast<uintptr_t>(a->window) & 3)))
    return V4A_ERR_INVALID_ARG;
  RingDev wr;
  return attn_window_ring(a, &wr);
}

// Splits of the key list per query: enough CTAs to cover the GPU twice,
// never more than one split per kChunk keys, and 1 (no combine) for large T.
static int splits_for(const v4a_attn_args* a) {
  const int E = entries_per_block(a->kv.ratio);
  const int64_t nsel = a->idx ? a->k : int64_t(a->kv.max_blocks) * E;
  const int64_t L = nsel + a->window_len;
  const int64_t chunks = (L + kChunk - 1) / kChunk;
  const int64_t groups = (a->num_heads + 15) / 16;
  const int64_t ctas = int64_t(a->batch.num_tokens) * groups;
  int64_t s = (2 * 152 + ctas - 1) / ctas;
  if (s > chunks) s = chunks;
  return int(s < 1 ? 1 : s);
}

size_t attn_workspace_size(const v4a_attn_args* a) {
  if (validate_shape(a)) return 0;
  size_t tc = attn_tc_workspace_size(a);
  if (tc) return tc;
  const size_t T = a->batch.num_tokens, S = splits_for(a), H = a->num_heads, D = a->kv.dim;
  return S == 1 ? 256 : T * S * H * (D + 2) * 4 + 256;
}

// For the fused attention + output call, which does not write a->out.
int validate_attn(const v4a_attn_args* a) { return validate(a, false); }

int sparse_attn(const v4a_attn_args* a, void* ws, size_t ws_bytes, cudaStream_t stream) {
  int rc = validate(a);
  if (rc) return rc;
  const int T = a->batch.num_tokens;
  if (T == 0) return V4A_OK;
  const size_t need = attn_workspace_size(a);
  if (!ws || ws_bytes < need) return V4A_ERR_WORKSPACE;
  if (attn_tc(a, ws, ws_bytes, stream, &rc)) return rc;
  // the CUDA-core kernels read the per-row-scale formats only
  if (a->kv.format == V4A_KV_FP8_DSV4) return V4A_ERR_UNSUPPORTED;
  const int S = splits_for(a);
  AttnDev d;
  d.T = T; d.H = a->num_heads; d.D = a->kv.dim; d.ratio = a->kv.ratio; d.fmt = a->kv.format;
  d.wfmt = a->window_format; d.wlen = a->window_len; d.k = a->k;
  attn_window_ring(a, &d.wring);     // validated above
  d.splits = S;
  d.seq_ids = a->batch.seq_ids; d.positions = a->batch.positions; d.kv = a->kv;
  d.block_bytes = kv_block_bytes(a->kv.format, a->kv.ratio, a->kv.dim);
  d.idx = a->idx;
  d.q = a->q; d.scale = a->softmax_scale;
  d.part_o = static_cast<float*>(ws);
  d.part_ml = d.part_o + size_t(T) * S * a->num_heads * a->kv.dim;
  d.out = a->out; d.lse = a->lse;
  d.status = a->status;
  const size_t smem = size_t(kChunk) * 2 * a->kv.dim + kChunk * 8;
  const int warps = a->num_heads < 16 ? a->num_heads : 16;
  const dim3 grid(S, T, (a->num_heads + warps - 1) / warps);
  switch (a->kv.dim / 32) {
#define V4A_ATTN_CASE(NJ)                                                                       \
  case NJ:                                                                                      \
    cudaFuncSetAttribute(attn_split_simt<NJ>, cudaFuncAttributeMaxDynamicSharedMemorySize,    \
                         int(smem));                                                            \
    attn_split_simt<NJ><<<grid, warps * 32, smem, stream>>>(d);                                        \
    break;
    V4A_ATTN_CASE(2)
    V4A_ATTN_CASE(4)
    V4A_ATTN_CASE(8)
    V4A_ATTN_CASE(16)
#undef V4A_ATTN_CASE
    default: return V4A_ERR_UNSUPPORTED;
  }
  if (S > 1)
    attn_combine<<<dim3(a->num_heads, T), 128, 0, stream>>>(T, a->num_heads, a->kv.dim, S,
                                                            d.part_o, d.part_ml, a->out, a->lse);
  return cudaGetLastError() == cudaSuccess ? V4A_OK : V4A_ERR_CUDA;
}

}  // namespace v4a
