// Fused KV compressor + RMSNorm + RoPE + paged-cache insert, and the
// sliding-window key RoPE + insert, in one launch.
//
// Method: "DeepSeek V4 in vLLM: Efficient Long-context Attention",
// Background (c4a: weighted sum of 8 tokens at stride 4; c128a: 128 tokens at
// stride 128), Method details fusion (1) (compress -> RMSNorm -> RoPE -> cache
// insert, separate for the indexer and the main cache) and fusion (3) (window
// key RoPE + insert), Appendix "exact position ranges and causality" (windows
// [4i-4, 4i+3] / [128i, 128i+127], RoPE once at the last native position).
//
// Grid: (T tokens, 2 + head groups).  Role 0 = main compressor, 1 = indexer
// compressor: each CTA owns one token; thread p owns the element pair
// (2p, 2p+1) of the row, which is also one RoPE pair.  A CTA of a compressor
// role always writes its token into the ring; if the token ends a window
// (position P with (P+1) % ratio == 0) it also builds the entry.  Role 2 is
// the window key (RoPE + encode + insert, thread p owning pair p as above).
// Roles >= 3 are the queries' side of the pages' horizontal fusion (3), with
// static warp roles: warp w of group g takes item g * warps + w of the
// token, a query head (RMSNorm + RoPE) or an indexer-query head (RoPE +
// per-head fp8 + head weight), with no communication between warps.  (The
// pages give the window key one warp as well; here it keeps a CTA of its
// own: with one warp per key the kernels after this launch ran 8 us slower
// per 1M-context decode step, measured, cause not found.)
// Window positions that belong to this call are read from the call's inputs,
// older ones from the ring; ring capacity >= window - 1 + tokens per sequence
// guarantees no ring slot written by this call is one of those older slots.

#include "v4a_common.cuh"
#include "v4a_internal.h"

namespace v4a {

struct CompressSide {
  RopeFreq rope;
  int active, is_indexer;
  int ratio, dim, rope_dims, format;
  float theta, eps;
  uint8_t* pool;
  int64_t num_blocks, block_bytes;
  const int32_t* bt;
  int max_blocks;
  const uint16_t* x;
  const float* gate;
  const float* bias;
  const float* gamma;
  RingDev ring;      // rows: bf16 x [dim]; side: gate
};

struct WindowSide {
  RopeFreq rope;
  int active, dim, rope_dims, format;
  float theta;
  const uint16_t* k;
  RingDev ring;      // rows: the encoded key; side: the fp8 scale
};

struct QuerySide {
  RopeFreq rope;
  int active, H, dim, rope_dims;
  float eps;
  const uint16_t* q_in;
  uint16_t* q_out;
  const float* gamma;
};

struct IndexQuerySide {
  RopeFreq rope;
  int active, H, dim, rope_dims;
  float w_mult;
  const uint16_t* q_in;
  uint8_t* q_out;
  float* q_scale;
  const float* w_in;
  float* w_out;
};

struct BatchDev {
  int T, B, max_new;
  const int32_t* seq_ids;
  const int32_t* positions;
};

__device__ __forceinline__ bool token_ok(const BatchDev& bt, int t, int b, int P) {
  if (b < 0 || b >= bt.B || P < 0) return false;
  if (t > 0 && bt.seq_ids[t - 1] == b && bt.positions[t - 1] != P - 1) return false;
  if (t >= bt.max_new && bt.seq_ids[t - bt.max_new] == b) return false;
  return true;
}

// Encodes the pair (v0, v1) owned by thread p into a row of the given format.
// All threads of the CTA must call it (it contains block reductions).
__device__ void store_kv_row(int format, int dim, int p, bool own, float v0, float v1,
                             uint8_t* row, float* scale_slot, float* red) {
  if (format == V4A_KV_FP8_DSV4) {
    // the DeepSeek-V4 584-byte row (dim 512, rope dims 64): pairs below 224
    // are the non-rope elements, 32 pairs (one warp) per 64-element scale
    // block; the rest are the rope elements, stored in bf16
    const int nope_pairs = kDsv4Nope / 2;
    const bool nope = own && p < nope_pairs;
    const float amax = warp_max(nope ? fmaxf(fabsf(v0), fabsf(v1)) : 0.f);
    if (nope) {
      // the smallest power of two s = 2^k with amax / s <= 448: amax = f 2^e,
      // f in [0.5, 1), 448 = 0.875 2^9, so k = e - 9, plus 1 when f > 0.875
      int k = 0;
      if (amax > 0.f) {
        int e;
        const float f = frexpf(amax, &e);
        k = e - 9 + (f > 0.875f ? 1 : 0);
      }
      const int b = min(max(k + 127, 1), 254);
      const uint16_t c = uint16_t(f32_to_e4m3(ldexpf(v0, 127 - b))) | (uint16_t(f32_to_e4m3(ldexpf(v1, 127 - b))) << 8);
      reinterpret_cast<uint16_t*>(row)[p] = c;
      if ((p & 31) == 0) row[kDsv4Nope + 2 * kDsv4Rope + (p >> 5)] = uint8_t(b);
    } else if (own) {
      const uint32_t packed = uint32_t(f32_to_bf16(v0)) | (uint32_t(f32_to_bf16(v1)) << 16);
      reinterpret_cast<uint32_t*>(row + kDsv4Nope)[p - nope_pairs] = packed;
    }
    if (p == 0) row[kDsv4Row - 1] = 0;
    return;
  }
  if (format == V4A_KV_BF16) {
    if (own) {
      const uint32_t packed = uint32_t(f32_to_bf16(v0)) | (uint32_t(f32_to_bf16(v1)) << 16);
      reinterpret_cast<uint32_t*>(row)[p] = packed;
    }
    return;
  }
  // fp8 e4m3 with one fp32 scale per row: amax / 448
  float a = own ? fmaxf(fabsf(v0), fabsf(v1)) : 0.f;
  const float amax = block_reduce<true>(a, red);
  const float s = amax > 0.f ? amax / 448.f : 1.f;
  if (own) {
    const uint16_t c = uint16_t(f32_to_e4m3(v0 / s)) | (uint16_t(f32_to_e4m3(v1 / s)) << 8);
    reinterpret_cast<uint16_t*>(row)[p] = c;
  }
  if (threadIdx.x == 0 && scale_slot) *scale_slot = s;
}

__device__ void store_ix_row(int format, int dim, int p, bool own, float v0, float v1,
                             uint8_t* row, float* scales, float* red) {
  if (format == V4A_IX_BF16) {
    if (own) {
      const uint32_t packed = uint32_t(f32_to_bf16(v0)) | (uint32_t(f32_to_bf16(v1)) << 16);
      reinterpret_cast<uint32_t*>(row)[p] = packed;
    }
    return;
  }
  const float a = own ? fmaxf(fabsf(v0), fabsf(v1)) : 0.f;
  if (ix_is_fp4(format)) {
    // 32 elements = 16 pairs = one half-warp
    float m = a;
#pragma unroll
    for (int o = 8; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    float s;
    if (format == V4A_IX_FP4_B32) {
      s = m > 0.f ? m / 6.f : 1.f;
    } else {
      // OCP MX shared scale: 2^(floor(log2 amax) - 2), 2 = the largest power
      // of two of e2m1; exponent clamped to the normal fp32 range
      const int e = int((__float_as_uint(m) >> 23) & 0xFFu) - 127;   // floor(log2 m) for normal m
      const int x = min(max(e - 2, -126), 127);
      s = m > 0.f ? __uint_as_float(uint32_t(x + 127) << 23) : 1.f;
    }
    if (own) {
      const uint32_t c0 = f32_to_e2m1(v0 / s), c1 = f32_to_e2m1(v1 / s);
      row[p] = uint8_t(c0 | (c1 << 4));
      if ((p & 15) == 0) scales[p >> 4] = s;
    }
    return;
  }
  // fp8 with one scale per 128 elements = 64 pairs = two warps
  const float wm = warp_max(a);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  __syncthreads();
  if (lane == 0) red[warp] = wm;
  __syncthreads();
  const float m = fmaxf(red[(warp & ~1)], red[(warp & ~1) + 1]);
  const float s = m > 0.f ? m / 448.f : 1.f;
  if (own) {
    const uint16_t c = uint16_t(f32_to_e4m3(v0 / s)) | (uint16_t(f32_to_e4m3(v1 / s)) << 8);
    reinterpret_cast<uint16_t*>(row)[p] = c;
    if ((p & 63) == 0) scales[p >> 6] = s;
  }
  __syncthreads();
}

// Latency matters more than bandwidth here (a handful of tokens per call), so
// every load that depends only on (token, sequence, position) is issued in
// one round before anything waits: this token's row, its block-table entry,
// gamma, and for each window position the gate of both possible sources (the
// call's inputs or the ring) with the sequence id that decides between them.
__device__ void compress_token(const CompressSide& c, const BatchDev& bt, int t, int b, int P, bool tok_ok,
                               int32_t* status) {
  __shared__ float w_s[128];
  __shared__ const uint16_t* src_s[128];
  __shared__ float red[32];
  __shared__ int64_t blk_s;
  const int p = threadIdx.x;
  const int npairs = c.dim >> 1;
  const bool own = p < npairs;
  const bool emit = (P + 1) % c.ratio == 0;
  const int i = (P + 1) / c.ratio - 1;
  const int W = c.ratio == 4 ? 8 : 128;
  const int p0 = c.ratio == 4 ? 4 * i - 4 : 128 * i;

  // ---- phase 1: independent loads ----
  const uint32_t* xin = reinterpret_cast<const uint32_t*>(c.x + int64_t(t) * c.dim);
  const uint32_t xv = own ? xin[p] : 0u;
  const float gt = p == 0 ? c.gate[t] : 0.f;
  float gm0 = 0.f, gm1 = 0.f;
  if (emit && own) { gm0 = c.gamma[2 * p]; gm1 = c.gamma[2 * p + 1]; }
  if (emit && p == blockDim.x - 1) {
    v4a_cache cc;
    cc.ratio = c.ratio; cc.block_table = c.bt; cc.max_blocks = c.max_blocks;
    cc.num_blocks = c.num_blocks;
    blk_s = block_of(cc, b, i, status);
  }
  float logit = -INFINITY;
  if (emit && p < W) {
    const int j = p, pos = p0 + j;
    const uint16_t* row = nullptr;
    if (pos >= 0) {
      const int d = P - pos;                 // 0 .. W-1
      uint8_t* rrow;
      float* rgate;
      ring_slot(c.ring, b, pos % c.ring.cap, &rrow, &rgate, status);
      const bool in_call_ok = t - d >= 0;
      const int sid = in_call_ok ? bt.seq_ids[t - d] : -1;
      const float g_call = in_call_ok ? c.gate[t - d] : 0.f;
      const float g_ring = rgate ? *rgate : 0.f;
      const float bias = c.bias[j];
      const bool in_call = in_call_ok && sid == b;
      // a ring slot whose page is missing drops out of the window (reported)
      row = in_call ? c.x + int64_t(t - d) * c.dim : reinterpret_cast<const uint16_t*>(rrow);
      if (row) logit = (in_call ? g_call : g_ring) + bias;
    }
    src_s[j] = row;
  }
  if (!tok_ok) return;                       // uniform: the whole CTA leaves before writing

  // this token's raw (x, gate) into the ring (no window position read below is
  // this slot: ring capacity >= window - 1 + tokens per sequence)
  {
    uint8_t* rrow;
    float* rgate;
    ring_slot(c.ring, b, P % c.ring.cap, &rrow, &rgate, p == 0 ? status : nullptr);
    if (rrow) {
      if (own) reinterpret_cast<uint32_t*>(rrow)[p] = xv;
      if (p == 0) *rgate = gt;
    }
  }
  if (!emit) return;

  // ---- window weights: softmax over the valid positions ----
  if (W <= 32) {
    if (p < 32) {                             // one warp
      const float mx = warp_max(logit);
      const float e = (p < W && logit > -INFINITY) ? expf(logit - mx) : 0.f;
      const float sum = warp_sum(e);
      if (p < W) w_s[p] = e / sum;
    }
    __syncthreads();
  } else {
    const float mx = block_reduce<true>(logit, red);
    const float e = (p < W && logit > -INFINITY) ? expf(logit - mx) : 0.f;
    const float sum = block_reduce<false>(e, red);
    if (p < W) w_s[p] = e / sum;
    __syncthreads();
  }

  // ---- phase 2: weighted sum of the window rows (pair per thread) ----
  // 32 rows' loads in flight per batch (a 128-token window takes 4 round
  // trips, not 16); the sum runs over the rows in window order either way
  constexpr int kRowsInFlight = 32;
  float a0 = 0.f, a1 = 0.f;
  if (own) {
    for (int j0 = 0; j0 < W; j0 += kRowsInFlight) {
      uint32_t v[kRowsInFlight];
#pragma unroll
      for (int u = 0; u < kRowsInFlight; ++u) {
        const uint16_t* row = j0 + u < W ? src_s[j0 + u] : nullptr;
        v[u] = row ? reinterpret_cast<const uint32_t*>(row)[p] : 0u;
      }
#pragma unroll
      for (int u = 0; u < kRowsInFlight; ++u) {
        if (j0 + u >= W) break;
        const float wj = w_s[j0 + u];
        a0 = fmaf(wj, bf16_to_f32(uint16_t(v[u] & 0xffffu)), a0);
        a1 = fmaf(wj, bf16_to_f32(uint16_t(v[u] >> 16)), a1);
      }
    }
  }
  // ---- RMSNorm ----
  const float ss = block_reduce<false>(own ? a0 * a0 + a1 * a1 : 0.f, red);
  const float r = 1.f / sqrtf(ss / float(c.dim) + c.eps);
  float v0 = 0.f, v1 = 0.f;
  if (own) {
    v0 = a0 * r * gm0;
    v1 = a1 * r * gm1;
    // RoPE at the anchor (= this token's position)
    const int first = c.dim - c.rope_dims;
    if (2 * p >= first) {
      float cs, sn;
      rope_cos_sin(P, c.rope.inv[(2 * p - first) >> 1], &cs, &sn);
      const float x0 = v0, x1 = v1;
      v0 = x0 * cs - x1 * sn;
      v1 = x0 * sn + x1 * cs;
    }
  }
  // ---- encode + insert at (block_table[b][i / E], i % E) ----
  const int E = entries_per_block(c.ratio);
  const int64_t blk = blk_s;                 // written before the reductions' barriers
  if (blk < 0) return;   // uniform across the CTA
  uint8_t* base = c.pool + blk * c.block_bytes;
  const int slot = i % E;
  if (!c.is_indexer) {
    const int64_t rb = kv_row_bytes(c.format, c.dim);
    store_kv_row(c.format, c.dim, p, own, v0, v1, base + slot * rb,
                 reinterpret_cast<float*>(base + E * rb) + slot, red);
  } else {
    const int64_t rb = ix_row_bytes(c.format, c.dim);
    const int ns = ix_scales_per_row(c.format, c.dim);
    store_ix_row(c.format, c.dim, p, own, v0, v1, base + slot * rb,
                 reinterpret_cast<float*>(base + 64 * rb) + int64_t(slot) * ns, red);
  }
}

// ---- fusion (3), the queries: one warp per query head ----
// Lane l holds the element pairs l, l + 32, ... (pairs never straddle lanes,
// so the rotation stays in the lane); dim % 64 == 0 and dim <= 1024.
constexpr int kWarpPairsMax = 16;

__device__ void query_head(const QuerySide& q, int t, int P, int h, int lane) {
  const int per = q.dim >> 6;                 // pairs per lane
  const int64_t row = (int64_t(t) * q.H + h) * q.dim;
  const uint32_t* in = reinterpret_cast<const uint32_t*>(q.q_in + row);
  const float2* g2 = reinterpret_cast<const float2*>(q.gamma);
  float v0[kWarpPairsMax], v1[kWarpPairsMax];
  float ss = 0.f;
#pragma unroll
  for (int i = 0; i < kWarpPairsMax; ++i) {
    if (i < per) {
      const uint32_t v = in[lane + 32 * i];
      v0[i] = bf16_to_f32(uint16_t(v & 0xffffu));
      v1[i] = bf16_to_f32(uint16_t(v >> 16));
      ss = fmaf(v0[i], v0[i], fmaf(v1[i], v1[i], ss));
    }
  }
  ss = warp_sum(ss);
  const float r = 1.f / sqrtf(ss / float(q.dim) + q.eps);
  const int first = q.dim - q.rope_dims;
  uint32_t* out = reinterpret_cast<uint32_t*>(q.q_out + row);
#pragma unroll
  for (int i = 0; i < kWarpPairsMax; ++i) {
    if (i < per) {
      const int j = lane + 32 * i;
      const float2 g = g2[j];
      float x0 = v0[i] * r * g.x, x1 = v1[i] * r * g.y;
      if (2 * j >= first) {
        float cs, sn;
        rope_cos_sin(P, q.rope.inv[(2 * j - first) >> 1], &cs, &sn);
        const float a0 = x0, a1 = x1;
        x0 = a0 * cs - a1 * sn;
        x1 = a0 * sn + a1 * cs;
      }
      out[j] = uint32_t(f32_to_bf16(x0)) | (uint32_t(f32_to_bf16(x1)) << 16);
    }
  }
}

// The indexer query: rotate, then e4m3 with one scale per head (amax / 448),
// and the head weight times w_mult; one warp per head, pairs as above.
__device__ void index_query_head(const IndexQuerySide& q, int t, int P, int h, int lane) {
  const int per = q.dim >> 6;
  const int64_t row = (int64_t(t) * q.H + h) * q.dim;
  const uint32_t* in = reinterpret_cast<const uint32_t*>(q.q_in + row);
  const int first = q.dim - q.rope_dims;
  float v0[kWarpPairsMax], v1[kWarpPairsMax];
  float amax = 0.f;
#pragma unroll
  for (int i = 0; i < kWarpPairsMax; ++i) {
    if (i < per) {
      const int j = lane + 32 * i;
      const uint32_t v = in[j];
      float x0 = bf16_to_f32(uint16_t(v & 0xffffu)), x1 = bf16_to_f32(uint16_t(v >> 16));
      if (2 * j >= first) {
        float cs, sn;
        rope_cos_sin(P, q.rope.inv[(2 * j - first) >> 1], &cs, &sn);
        const float a0 = x0, a1 = x1;
        x0 = a0 * cs - a1 * sn;
        x1 = a0 * sn + a1 * cs;
      }
      v0[i] = x0;
      v1[i] = x1;
      amax = fmaxf(amax, fmaxf(fabsf(x0), fabsf(x1)));
    }
  }
  amax = warp_max(amax);
  const float s = amax > 0.f ? amax / 448.f : 1.f;
  uint16_t* out = reinterpret_cast<uint16_t*>(q.q_out + row);
#pragma unroll
  for (int i = 0; i < kWarpPairsMax; ++i)
    if (i < per)
      out[lane + 32 * i] = uint16_t(f32_to_e4m3(v0[i] / s)) | (uint16_t(f32_to_e4m3(v1[i] / s)) << 8);
  if (lane == 0) {
    const int64_t th = int64_t(t) * q.H + h;
    q.q_scale[th] = s;
    q.w_out[th] = q.w_in[th] * q.w_mult;
  }
}

__device__ void window_token(const WindowSide& w, int t, int b, int P, int32_t* status) {
  __shared__ float red[32];
  const int p = threadIdx.x;
  const bool own = p < (w.dim >> 1);
  float v0 = 0.f, v1 = 0.f;
  if (own) {
    const uint32_t v = reinterpret_cast<const uint32_t*>(w.k + int64_t(t) * w.dim)[p];
    v0 = bf16_to_f32(uint16_t(v & 0xffffu));
    v1 = bf16_to_f32(uint16_t(v >> 16));
    const int first = w.dim - w.rope_dims;
    if (2 * p >= first) {
      float cs, sn;
      rope_cos_sin(P, w.rope.inv[(2 * p - first) >> 1], &cs, &sn);
      const float x0 = v0, x1 = v1;
      v0 = x0 * cs - x1 * sn;
      v1 = x0 * sn + x1 * cs;
    }
  }
  uint8_t* row;
  float* scale;
  ring_slot(w.ring, b, P % w.ring.cap, &row, &scale, p == 0 ? status : nullptr);
  if (!row) return;                          // uniform over the CTA
  store_kv_row(w.format, w.dim, p, own, v0, v1, row, scale, red);
}

__global__ void compress_insert_kernel(BatchDev bt, CompressSide mainc, CompressSide ixc,
                                       WindowSide win, QuerySide qs, IndexQuerySide iq, int32_t* status) {
  pdl_trigger();   // the next kernel may be scheduled now (it waits for this one in-kernel)
  const int t = blockIdx.x;
  const int role = blockIdx.y;
  const int b = bt.seq_ids[t];
  const int P = bt.positions[t];
  // a sequence id out of range or a negative position stops the CTA before any
  // address is formed from them; the run checks (consecutive positions, run
  // length) load while the compressor issues its own loads
  if (b < 0 || b >= bt.B || P < 0) {
    if (threadIdx.x == 0 && role == 0) report(status, V4A_DEV_BAD_BATCH);
    return;
  }
  const bool ok = token_ok(bt, t, b, P);
  if (!ok && threadIdx.x == 0 && role == 0) report(status, V4A_DEV_BAD_BATCH);
  if (role == 0 && mainc.active) compress_token(mainc, bt, t, b, P, ok, status);
  if (role == 1 && ixc.active) compress_token(ixc, bt, t, b, P, ok, status);
  if (role == 2 && win.active && ok) window_token(win, t, b, P, status);
  if (role >= 3) {
    // static warp roles: warp w of group g takes item g * warps + w, the
    // query heads first, then the indexer query's heads
    const int item = (role - 3) * int(blockDim.x >> 5) + int(threadIdx.x >> 5);
    const int nq = qs.active ? qs.H : 0, ni = iq.active ? iq.H : 0;
    if (item < nq) query_head(qs, t, P, item, threadIdx.x & 31);
    else if (item < nq + ni) index_query_head(iq, t, P, item - nq, threadIdx.x & 31);
  }
}

// True when pointer p is a multiple of `bytes` (the width of the loads and
// stores the kernel makes through it).
static bool aligned(const void* p, uintptr_t bytes) { return (reinterpret_cast<uintptr_t>(p) & (bytes - 1)) == 0; }

static int fill_side(const v4a_compressor* c, bool indexer, CompressSide* s, int max_new) {
  *s = CompressSide{};
  if (!c) return V4A_OK;
  const v4a_cache& k = c->cache;
  if (!k.pool || !k.block_table || !c->x || !c->gate || !c->bias || !c->gamma) return V4A_ERR_INVALID_ARG;
  // bf16 rows are read and written as element pairs
  if (!aligned(c->x, 4) || (!c->ring_pages && c->ring_x && !aligned(c->ring_x, 4))) return V4A_ERR_INVALID_ARG;
  if (k.ratio != 4 && k.ratio != 128) return V4A_ERR_INVALID_ARG;
  if (indexer && k.ratio != 4) return V4A_ERR_UNSUPPORTED;
  if (k.dim <= 0 || k.dim % 64 || k.dim > 1024) return V4A_ERR_UNSUPPORTED;
  if (k.rope_dims < 0 || k.rope_dims > k.dim || k.rope_dims % 2) return V4A_ERR_INVALID_ARG;
  if (k.num_blocks <= 0 || k.max_blocks <= 0 || c->ring_cap <= 0) return V4A_ERR_INVALID_ARG;
  const int W = k.ratio == 4 ? 8 : 128;
  if (c->ring_cap < W - 1 + max_new) return V4A_ERR_RING_TOO_SMALL;
  if (!indexer) {
    if (k.format != V4A_KV_BF16 && k.format != V4A_KV_FP8_TOKEN && k.format != V4A_KV_FP8_DSV4)
      return V4A_ERR_INVALID_ARG;
    if (k.format == V4A_KV_FP8_DSV4 && (k.dim != kDsv4Nope + kDsv4Rope || k.rope_dims != kDsv4Rope))
      return V4A_ERR_UNSUPPORTED;
  } else {
    if (k.format != V4A_IX_BF16 && k.format != V4A_IX_FP8_B128 && !ix_is_fp4(k.format))
      return V4A_ERR_INVALID_ARG;
    if (k.format == V4A_IX_FP8_B128 && k.dim % 128) return V4A_ERR_UNSUPPORTED;
  }
  if (k.rope_dims > 128) return V4A_ERR_UNSUPPORTED;
  s->rope = make_rope_freq(k.rope_dims, k.rope_theta);
  s->active = 1;
  s->is_indexer = indexer;
  s->ratio = k.ratio; s->dim = k.dim; s->rope_dims = k.rope_dims; s->format = k.format;
  s->theta = k.rope_theta; s->eps = c->eps;
  s->pool = static_cast<uint8_t*>(k.pool);
  s->num_blocks = k.num_blocks;
  s->block_bytes = indexer ? ix_block_bytes(k.format, k.dim) : kv_block_bytes(k.format, k.ratio, k.dim);
  s->bt = k.block_table; s->max_blocks = k.max_blocks;
  s->x = c->x; s->gate = c->gate; s->bias = c->bias; s->gamma = c->gamma;
  return ring_dev_fill(&s->ring, c->ring_x, c->ring_gate, c->ring_cap, 2 * k.dim, true, c->ring_pages);
}

int compress_insert(const v4a_compress_args* a, cudaStream_t stream) {
  if (!a) return V4A_ERR_INVALID_ARG;
  const v4a_batch& B = a->batch;
  if (B.num_tokens < 0 || B.num_seqs <= 0 || B.max_new_per_seq <= 0) return V4A_ERR_INVALID_ARG;
  if (B.num_tokens > 0 && (!B.seq_ids || !B.positions)) return V4A_ERR_INVALID_ARG;
  CompressSide mc, ic;
  int rc = fill_side(a->main, false, &mc, B.max_new_per_seq);
  if (rc) return rc;
  rc = fill_side(a->indexer, true, &ic, B.max_new_per_seq);
  if (rc) return rc;
  WindowSide ws{};
  if (a->window) {
    const v4a_window& w = *a->window;
    if (!w.k || w.ring_cap <= 0 || !aligned(w.k, 4)) return V4A_ERR_INVALID_ARG;
    if (w.dim <= 0 || w.dim % 64 || w.dim > 1024) return V4A_ERR_UNSUPPORTED;
    if (w.rope_dims < 0 || w.rope_dims > w.dim || w.rope_dims % 2) return V4A_ERR_INVALID_ARG;
    if (w.format != V4A_KV_BF16 && w.format != V4A_KV_FP8_TOKEN) return V4A_ERR_INVALID_ARG;
    if (w.window_len < 1) return V4A_ERR_INVALID_ARG;
    // a query's window [P - window_len + 1, P] must still be in the ring after
    // the call has written its max_new_per_seq positions
    if (int64_t(w.ring_cap) < int64_t(w.window_len) - 1 + B.max_new_per_seq) return V4A_ERR_RING_TOO_SMALL;
    if (w.rope_dims > 128) return V4A_ERR_UNSUPPORTED;
    ws.rope = make_rope_freq(w.rope_dims, w.rope_theta);
    ws.active = 1; ws.dim = w.dim; ws.rope_dims = w.rope_dims; ws.format = w.format;
    ws.theta = w.rope_theta; ws.k = w.k;
    rc = ring_dev_fill(&ws.ring, w.ring, w.ring_scale, w.ring_cap, int(kv_row_bytes(w.format, w.dim)),
                       w.format == V4A_KV_FP8_TOKEN, w.ring_pages);
    if (rc) return rc;
  }
  QuerySide qs{};
  if (a->query) {
    const v4a_query& q = *a->query;
    if (!q.q_in || !q.q_out || !q.gamma || q.num_heads < 1) return V4A_ERR_INVALID_ARG;
    if (!aligned(q.q_in, 4) || !aligned(q.q_out, 4) || !aligned(q.gamma, 8)) return V4A_ERR_INVALID_ARG;
    if (q.dim <= 0 || q.dim % 64 || q.dim > 1024) return V4A_ERR_UNSUPPORTED;
    if (q.rope_dims < 0 || q.rope_dims > q.dim || q.rope_dims % 2 || !(q.eps >= 0.f)) return V4A_ERR_INVALID_ARG;
    if (q.rope_dims > 128) return V4A_ERR_UNSUPPORTED;
    qs.rope = make_rope_freq(q.rope_dims, q.rope_theta);
    qs.active = 1; qs.H = q.num_heads; qs.dim = q.dim; qs.rope_dims = q.rope_dims; qs.eps = q.eps;
    qs.q_in = q.q_in; qs.q_out = q.q_out; qs.gamma = q.gamma;
  }
  IndexQuerySide iq{};
  if (a->index_query) {
    const v4a_index_query& q = *a->index_query;
    if (!q.q_in || !q.q_out || !q.q_scale || !q.w_in || !q.w_out || q.num_heads < 1) return V4A_ERR_INVALID_ARG;
    if (!aligned(q.q_in, 4) || !aligned(q.q_out, 2) || !aligned(q.q_scale, 4) || !aligned(q.w_in, 4) ||
        !aligned(q.w_out, 4))
      return V4A_ERR_INVALID_ARG;
    if (q.dim <= 0 || q.dim % 64 || q.dim > 1024) return V4A_ERR_UNSUPPORTED;
    if (q.rope_dims < 0 || q.rope_dims > q.dim || q.rope_dims % 2) return V4A_ERR_INVALID_ARG;
    if (q.rope_dims > 128) return V4A_ERR_UNSUPPORTED;
    iq.rope = make_rope_freq(q.rope_dims, q.rope_theta);
    iq.active = 1; iq.H = q.num_heads; iq.dim = q.dim; iq.rope_dims = q.rope_dims; iq.w_mult = q.w_mult;
    iq.q_in = q.q_in; iq.q_out = q.q_out; iq.q_scale = q.q_scale; iq.w_in = q.w_in; iq.w_out = q.w_out;
  }
  if (B.num_tokens == 0 || (!mc.active && !ic.active && !ws.active && !qs.active && !iq.active)) return V4A_OK;
  int maxdim = 64;
  if (mc.active) maxdim = max(maxdim, mc.dim);
  if (ic.active) maxdim = max(maxdim, ic.dim);
  int threads = ((maxdim / 2) + 31) / 32 * 32;
  // one thread per window position as well (128 for c128a compressors)
  if ((mc.active && mc.ratio == 128) || (ic.active && ic.ratio == 128)) threads = max(threads, 128);
  if (ws.active) threads = max(threads, ((ws.dim / 2) + 31) / 32 * 32);
  // query and indexer-query heads: one warp each, in groups of 8 warps (or
  // more) per CTA
  const int items = (qs.active ? qs.H : 0) + (iq.active ? iq.H : 0);
  if (items > 0) threads = max(threads, 256);
  threads = max(threads, 64);
  const int groups = (items + threads / 32 - 1) / (threads / 32);
  BatchDev bd{B.num_tokens, B.num_seqs, B.max_new_per_seq, B.seq_ids, B.positions};
  dim3 grid(B.num_tokens, 3 + groups);
  compress_insert_kernel<<<grid, threads, 0, stream>>>(bd, mc, ic, ws, qs, iq, a->status);
  return cudaGetLastError() == cudaSuccess ? V4A_OK : V4A_ERR_CUDA;
}

}  // namespace v4a
