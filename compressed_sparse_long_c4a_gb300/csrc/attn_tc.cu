// Shared-K=V sparse attention on the tensor cores (tcgen05, kind::f16, bf16
// operands, fp32 accumulate in TMEM), for decode-sized batches.
//
// Method: "DeepSeek V4 in vLLM: Efficient Long-context Attention", Background
// (keys and values share one vector; attend to the top-k compressed entries
// plus the 128 uncompressed window tokens) and Appendix ("why inverse RoPE":
// o_m = sum_n softmax(q_m . k_n) k_n).
//
// One CTA per (64-key chunk of a query's key list, query):
//   Q     [128 rows = heads, zero-padded][D] bf16  -> smem, K-major, 128-B swizzle
//   K     64 gathered rows [64][D] bf16 (fp8 codes are converted exactly to
//         bf16; their per-row scale is applied to the logits and to P)
//   S     = Q K^T           M=128, N=64,  K=D   -> TMEM columns [0, 64)
//   P     = exp(tau*s_n*S - m) * s_n, bf16 -> smem (one thread per head row)
//   O     = P K             M=128, N=256 per MMA (K as an MN-major operand),
//                           K=64              -> TMEM columns [0, D) (the S
//                           columns are reused once S has been read)
// The chunk's normalised O (bf16) and (max, sum) go to the workspace; a
// combine kernel merges the chunks of each query.  A single thread issues
// every MMA; completion is tracked with tcgen05.commit on mbarriers whose
// waits are bounded.

#include <mutex>

#include "attn_tc.h"
#include "tc_common.cuh"

namespace v4a {
namespace {

constexpr int kKeys = 64;            // keys per CTA (one chunk)
constexpr int kRows = 128;           // MMA M (heads, zero-padded)
constexpr int kThreads = 256;      // warps 0-3 own TMEM lane quarters for the softmax; all 8 drain

struct AtcArgs {
  int T, H, D, ratio, fmt, wfmt, wlen, wcap, k, splits;
  const int32_t* seq_ids;
  const int32_t* positions;
  const int32_t* bt;
  int max_blocks;
  int64_t num_blocks;
  const uint8_t* pool;
  int64_t block_bytes;
  const int32_t* idx;
  const uint8_t* window;
  const float* wscale;
  const uint16_t* q;
  float scale;
  uint16_t* out;
  float* lse;
  uint16_t* part_o;   // [T][splits][H][D] bf16, normalised by the chunk's sum
  float* part_ml;     // [T][splits][H][2] = (max, sum)
  int32_t* status;
  uint32_t idesc_s, idesc_pv;
};

struct ASmem {
  uint64_t bar_q, bar_s, bar_o;
  uint32_t tmem_base;
  int abort_flag;
  const uint8_t* src[kKeys];
  float kscale[kKeys];
  int kfmt[kKeys];                  // -1: no key in this slot
  float row_l[kRows], row_m[kRows];   // softmax sums / maxima handed to the drain warps
};

// MN-major operand (B of P*K): 64-element (128-byte) rows along N, consecutive
// K rows 128 bytes apart, 8-row groups 1024 bytes apart (SBO), the next
// 64-element N chunk `lbo` bytes further (LBO), 128-byte swizzle.
__device__ __forceinline__ uint64_t desc_sw128_mn(uint32_t saddr, uint32_t lbo) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);
  d |= static_cast<uint64_t>((lbo >> 4) & 0x3FFFu) << 16;
  d |= static_cast<uint64_t>(1024 >> 4) << 32;
  d |= static_cast<uint64_t>(1) << 46;
  d |= static_cast<uint64_t>(2) << 61;
  return d;
}

__device__ __forceinline__ uint32_t bf16x2_from_e4m3x2(uint16_t two) {
  const __half2_raw h = __nv_cvt_fp8x2_to_halfraw2(static_cast<__nv_fp8x2_storage_t>(two), __NV_E4M3);
  const float2 f = __half22float2(__half2(h));
  const __nv_bfloat162 b = __floats2bfloat162_rn(f.x, f.y);   // exact: e4m3 values are bf16 values
  return *reinterpret_cast<const uint32_t*>(&b);
}

__global__ void __launch_bounds__(kThreads, 1) attn_chunk_tc(const AtcArgs a,
                                                             const __grid_constant__ CUtensorMap qmap) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int D = a.D, nsub = D / 64;
  uint8_t* Qs = base;                                  // nsub x [128 rows][128 B]
  uint8_t* Ks = Qs + nsub * kRows * 128;               // nsub x [64 rows][128 B]
  uint8_t* Ps = Ks + nsub * kKeys * 128;               // [128 rows][128 B]
  ASmem& s = *reinterpret_cast<ASmem*>(Ps + kRows * 128);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int t = blockIdx.y, sp = blockIdx.x;
  const int b = a.seq_ids[t], m = a.positions[t];
  const int nvis = (m + 1) / a.ratio;
  const int nsel = a.idx ? a.k : nvis;
  const int wstart = max(0, m - a.wlen + 1);
  const int L = nsel + (m - wstart + 1);
  const int lo = sp * kKeys;
  const int64_t pi0 = int64_t(t) * a.splits + sp;

  if (lo >= L) {   // this query's list is shorter than the longest: empty chunk
    for (int h = tid; h < a.H; h += blockDim.x) {
      a.part_ml[(pi0 * a.H + h) * 2] = -INFINITY;
      a.part_ml[(pi0 * a.H + h) * 2 + 1] = 0.f;
    }
    return;
  }
  if (tid == 0) {
    tc::mbar_init(&s.bar_q, 1);
    tc::mbar_init(&s.bar_s, 1);
    tc::mbar_init(&s.bar_o, 1);
    s.abort_flag = 0;
    tc::mbar_fence_init();
    // Q: 128 rows from this query's first head (rows past the last head are
    // the next query's or zero-filled; their outputs are never stored), one
    // 64-column swizzled box per K sub-tile
    tc::mbar_arrive_expect_tx(&s.bar_q, uint32_t(nsub * kRows * 128));
    for (int sub = 0; sub < nsub; ++sub)
      tc::tma_load_2d(Qs + sub * (kRows * 128), &qmap, sub * 64, t * a.H, &s.bar_q);
  }
  __syncwarp();   // tcgen05.alloc is warp-collective: reconverge warp 0 after the init above
  if (warp == 0) tc::tmem_alloc(&s.tmem_base, D < 64 ? 64 : D);

  // ---- key slots of this chunk (sources, scales) ----
  if (tid < kKeys) {
    const int li = lo + tid;
    const uint8_t* src = nullptr;
    int f = -1;
    float sc = 1.f;
    if (li < L) {
      if (li < nsel) {
        const int e = a.idx ? a.idx[int64_t(t) * a.k + li] : li;
        if (e >= 0) {
          const int E = entries_per_block(a.ratio);
          const int lb = e / E;
          if (e >= nvis) {
            report(a.status, V4A_DEV_BAD_INDEX);
          } else if (lb >= a.max_blocks) {
            report(a.status, V4A_DEV_BAD_BLOCK);
          } else {
            const int32_t blk = a.bt[int64_t(b) * a.max_blocks + lb];
            if (blk < 0 || blk >= a.num_blocks) {
              report(a.status, V4A_DEV_BAD_BLOCK);
            } else {
              const uint8_t* bb = a.pool + int64_t(blk) * a.block_bytes;
              const int slot = e % E;
              f = a.fmt;
              src = bb + int64_t(slot) * (a.fmt == V4A_KV_BF16 ? 2 * D : D);
              if (a.fmt == V4A_KV_FP8_TOKEN) sc = reinterpret_cast<const float*>(bb + int64_t(E) * D)[slot];
            }
          }
        }
      } else {
        const int p = wstart + (li - nsel);
        const int64_t slot = int64_t(b) * a.wcap + p % a.wcap;
        f = a.wfmt;
        src = a.window + slot * (a.wfmt == V4A_KV_BF16 ? 2 * D : D);
        if (a.wfmt == V4A_KV_FP8_TOKEN) sc = a.wscale[slot];
      }
    }
    s.src[tid] = src;
    s.kscale[tid] = sc;
    s.kfmt[tid] = f;
  }
  __syncthreads();

  // ---- stage K into swizzled smem ----
  // keys: bf16 rows go straight to smem with cp.async; fp8 rows are loaded
  // into registers first (all loads in flight together), then converted
  // exactly to bf16 and stored swizzled.
  const int kchunks = kKeys * (D / 8);
  constexpr int kMaxPer = kKeys * (512 / 8) / kThreads;   // 16 for D = 512
  uint2 raw[kMaxPer];
#pragma unroll
  for (int i = 0; i < kMaxPer; ++i) {
    const int c = tid + i * kThreads;
    raw[i] = make_uint2(0, 0);
    if (c >= kchunks) continue;
    const int r = c / (D / 8), cc = c % (D / 8);
    const int f = s.kfmt[r];
    if (f == V4A_KV_BF16) {
      uint8_t* dst = Ks + (cc >> 3) * (kKeys * 128) + r * 128 + (((cc & 7) ^ (r & 7)) << 4);
      asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(tc::smem_u32(dst)),
                   "l"(s.src[r] + cc * 16)
                   : "memory");
    } else if (f == V4A_KV_FP8_TOKEN) {
      raw[i] = __ldg(reinterpret_cast<const uint2*>(s.src[r] + cc * 8));
    }
  }
#pragma unroll
  for (int i = 0; i < kMaxPer; ++i) {
    const int c = tid + i * kThreads;
    if (c >= kchunks) continue;
    const int r = c / (D / 8), cc = c % (D / 8);
    const int f = s.kfmt[r];
    if (f == V4A_KV_BF16) continue;
    uint8_t* dst = Ks + (cc >> 3) * (kKeys * 128) + r * 128 + (((cc & 7) ^ (r & 7)) << 4);
    uint4 v = make_uint4(0, 0, 0, 0);
    if (f == V4A_KV_FP8_TOKEN) {
      v.x = bf16x2_from_e4m3x2(uint16_t(raw[i].x & 0xffffu));
      v.y = bf16x2_from_e4m3x2(uint16_t(raw[i].x >> 16));
      v.z = bf16x2_from_e4m3x2(uint16_t(raw[i].y & 0xffffu));
      v.w = bf16x2_from_e4m3x2(uint16_t(raw[i].y >> 16));
    }
    *reinterpret_cast<uint4*>(dst) = v;
  }
  asm volatile("cp.async.wait_all;" ::: "memory");
  tc::mbar_wait(&s.bar_q, 0, a.status, &s.abort_flag);
  tc::fence_proxy_async();
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  const uint32_t tmem = s.tmem_base;
  volatile int* abort_flag = &s.abort_flag;

  // ---- S = Q K^T ----
  if (tid == 0) {
    const uint32_t q0 = tc::smem_u32(Qs), k0 = tc::smem_u32(Ks);
    for (int st = 0; st < D / 16; ++st) {
      const uint64_t ad = tc::desc_sw128(q0 + (st >> 2) * (kRows * 128)) + 2 * (st & 3);
      const uint64_t bd = tc::desc_sw128(k0 + (st >> 2) * (kKeys * 128)) + 2 * (st & 3);
      tc::mma_f16(tmem, ad, bd, a.idesc_s, st > 0);
    }
    tc::mma_commit(&s.bar_s);
  }
  // ---- softmax: warps 0-3, thread = head row ----
  const int row = tid & (kRows - 1);             // warp w reads TMEM lanes 32(w%4)..+31
  const uint32_t lane_addr = tmem + (uint32_t((warp & 3) * 32) << 16);
  // Collective tcgen05 loads below are always executed by whole warps; `ok`
  // is made warp-uniform and only gates the arithmetic and the stores.
  bool ok = __all_sync(0xffffffffu, tc::mbar_wait(&s.bar_s, 0, a.status, abort_flag));
  tc::tc_fence_after();
  float mx = -INFINITY, l = 0.f;
  if (warp < 4) {
    float v[64];
    tc::tmem_ld64(lane_addr, v);
#pragma unroll
    for (int n = 0; n < 64; ++n) {
      const float z = s.kfmt[n] >= 0 ? v[n] * a.scale * s.kscale[n] : -INFINITY;
      v[n] = z;
      mx = fmaxf(mx, z);
    }
    uint32_t pk[32];
#pragma unroll
    for (int n = 0; n < 64; n += 2) {
      const float p0 = s.kfmt[n] >= 0 ? __expf(v[n] - mx) : 0.f;
      const float p1 = s.kfmt[n + 1] >= 0 ? __expf(v[n + 1] - mx) : 0.f;
      l += p0 + p1;
      const __nv_bfloat162 pb = __floats2bfloat162_rn(p0 * s.kscale[n], p1 * s.kscale[n + 1]);
      pk[n >> 1] = *reinterpret_cast<const uint32_t*>(&pb);
    }
#pragma unroll
    for (int c = 0; c < 8; ++c)
      *reinterpret_cast<uint4*>(Ps + row * 128 + ((c ^ (row & 7)) << 4)) =
          make_uint4(pk[4 * c], pk[4 * c + 1], pk[4 * c + 2], pk[4 * c + 3]);
  }
  tc::fence_proxy_async();
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  // ---- O = P K (S columns are free again) ----
  if (tid == 0 && !*abort_flag) {
    const uint32_t p0 = tc::smem_u32(Ps), k0 = tc::smem_u32(Ks);
    const int halves = D > 256 ? D / 256 : 1;
    const int nchunk = D > 256 ? 4 : nsub;        // 64-column N chunks per MMA
    for (int st = 0; st < kKeys / 16; ++st) {
      const uint64_t ad = tc::desc_sw128(p0) + 2 * st;
      for (int hf = 0; hf < halves; ++hf) {
        const uint64_t bd =
            desc_sw128_mn(k0 + hf * nchunk * (kKeys * 128) + st * 16 * 128, kKeys * 128);
        tc::mma_f16(tmem + hf * 256, ad, bd, a.idesc_pv, st > 0);
      }
    }
    tc::mma_commit(&s.bar_o);
  }
  if (warp < 4) { s.row_l[row] = l; s.row_m[row] = mx; }
  ok = __all_sync(0xffffffffu, ok && tc::mbar_wait(&s.bar_o, 0, a.status, abort_flag));
  __syncthreads();
  tc::tc_fence_after();
  l = s.row_l[row];
  mx = s.row_m[row];
  const bool store = ok && row < a.H;   // H need not be a multiple of 32: loads stay warp-wide
  {
    const float inv = l > 0.f ? 1.f / l : 0.f;   // a chunk of only padding (-1) entries has l = 0
    const bool direct = a.splits == 1;
    uint16_t* dst = direct ? a.out + (int64_t(t) * a.H + row) * D : a.part_o + (pi0 * a.H + row) * D;
    // warps 0-3 drain the first half of the 64-column groups, warps 4-7 the rest
    const int half = nsub / 2;
    const int c0 = warp < 4 ? 0 : half, c1 = warp < 4 ? half : nsub;
    for (int c = c0; c < c1; ++c) {
      float v[64];
      tc::tmem_ld64(lane_addr + c * 64, v);
      if (!store) continue;
#pragma unroll
      for (int i = 0; i < 64; i += 8) {
        uint4 o;
        __nv_bfloat162 b0 = __floats2bfloat162_rn(v[i] * inv, v[i + 1] * inv);
        __nv_bfloat162 b1 = __floats2bfloat162_rn(v[i + 2] * inv, v[i + 3] * inv);
        __nv_bfloat162 b2 = __floats2bfloat162_rn(v[i + 4] * inv, v[i + 5] * inv);
        __nv_bfloat162 b3 = __floats2bfloat162_rn(v[i + 6] * inv, v[i + 7] * inv);
        o.x = *reinterpret_cast<uint32_t*>(&b0);
        o.y = *reinterpret_cast<uint32_t*>(&b1);
        o.z = *reinterpret_cast<uint32_t*>(&b2);
        o.w = *reinterpret_cast<uint32_t*>(&b3);
        *reinterpret_cast<uint4*>(dst + c * 64 + i) = o;
      }
    }
    if (!store || warp >= 4) {
    } else if (direct) {
      if (a.lse) a.lse[int64_t(t) * a.H + row] = mx + logf(l);
    } else {
      a.part_ml[(pi0 * a.H + row) * 2] = mx;
      a.part_ml[(pi0 * a.H + row) * 2 + 1] = l;
    }
  }
  tc::tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc::tc_fence_after();
    tc::tmem_dealloc(tmem, D < 64 ? 64 : D);
  }
}

// out = sum_s w_s * O_s with w_s = l_s e^{m_s} / sum_s' l_s' e^{m_s'}.
// One CTA of D/8 threads per (head, query); each thread owns 8 dims and
// keeps all of its split loads in flight together.
__global__ void attn_combine_bf16(int H, int D, int splits, const uint16_t* part_o, const float* part_ml,
                                  uint16_t* out, float* lse) {
  const int t = blockIdx.y, h = blockIdx.x;
  __shared__ float wsm[512];
  __shared__ float inv_s;
  const float* ml = part_ml + (int64_t(t) * splits * H + h) * 2;
  float mx = -INFINITY;
  for (int s = 0; s < splits; ++s) mx = fmaxf(mx, ml[int64_t(s) * H * 2]);
  for (int s = threadIdx.x; s < splits; s += blockDim.x) {
    const float ms = ml[int64_t(s) * H * 2];
    wsm[s] = ms == -INFINITY ? 0.f : ml[int64_t(s) * H * 2 + 1] * __expf(ms - mx);
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    float tot = 0.f;
    for (int s = 0; s < splits; ++s) tot += wsm[s];
    inv_s = 1.f / tot;
    if (lse) lse[int64_t(t) * H + h] = mx + logf(tot);
  }
  __syncthreads();
  const int d = threadIdx.x * 8;
  if (d >= D) return;
  float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
  const uint16_t* po = part_o + (int64_t(t) * splits * H + h) * D + d;
  constexpr int kUnroll = 8;
  for (int s0 = 0; s0 < splits; s0 += kUnroll) {
    uint4 v[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u)
      v[u] = (s0 + u < splits) ? *reinterpret_cast<const uint4*>(po + int64_t(s0 + u) * H * D)
                               : make_uint4(0, 0, 0, 0);
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const float w = (s0 + u < splits) ? wsm[s0 + u] : 0.f;
      if (w == 0.f) continue;   // empty chunk: its partial carries no weight (and may be garbage)
      const uint32_t q[4] = {v[u].x, v[u].y, v[u].z, v[u].w};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        acc[2 * i] = fmaf(w, bf16_to_f32(uint16_t(q[i] & 0xffffu)), acc[2 * i]);
        acc[2 * i + 1] = fmaf(w, bf16_to_f32(uint16_t(q[i] >> 16)), acc[2 * i + 1]);
      }
    }
  }
  const float inv = inv_s;
  uint32_t o[4];
#pragma unroll
  for (int i = 0; i < 4; ++i)
    o[i] = uint32_t(f32_to_bf16(acc[2 * i] * inv)) | (uint32_t(f32_to_bf16(acc[2 * i + 1] * inv)) << 16);
  *reinterpret_cast<uint4*>(out + (int64_t(t) * H + h) * D + d) = make_uint4(o[0], o[1], o[2], o[3]);
}

int splits_of(const v4a_attn_args* a) {
  const int E = entries_per_block(a->kv.ratio);
  const int64_t nsel = a->idx ? a->k : int64_t(a->kv.max_blocks) * E;
  return int((nsel + a->window_len + kKeys - 1) / kKeys);
}

// The chunked tensor-core path serves decode-sized batches: one CTA per 64
// keys of each query, so the CTA count is T * splits.  Long prefill batches
// use the CUDA-core path (one CTA walks a whole split of a query).
bool handled(const v4a_attn_args* a) {
  const int D = a->kv.dim;
  if (D != 128 && D != 256 && D != 512) return false;
  if (a->num_heads > kRows) return false;
  const int64_t ctas = int64_t(a->batch.num_tokens) * splits_of(a);
  if (ctas > 16 * 152) return false;
  if (splits_of(a) > 512) return false;
  return true;
}

}  // namespace

size_t attn_tc_workspace_size(const v4a_attn_args* a) {
  if (!handled(a)) return 0;
  const size_t T = a->batch.num_tokens, S = splits_of(a), H = a->num_heads, D = a->kv.dim;
  return T * S * H * D * 2 + T * S * H * 2 * 4 + 512;
}

bool attn_tc(const v4a_attn_args* a, void* ws, size_t ws_bytes, cudaStream_t stream, int* rc) {
  *rc = V4A_OK;
  if (!handled(a)) return false;
  if (ws_bytes < attn_tc_workspace_size(a)) { *rc = V4A_ERR_WORKSPACE; return true; }
  AtcArgs t{};
  t.T = a->batch.num_tokens;
  t.H = a->num_heads;
  t.D = a->kv.dim;
  t.ratio = a->kv.ratio;
  t.fmt = a->kv.format;
  t.wfmt = a->window_format;
  t.wlen = a->window_len;
  t.wcap = a->window_cap;
  t.k = a->k;
  t.splits = splits_of(a);
  t.seq_ids = a->batch.seq_ids;
  t.positions = a->batch.positions;
  t.bt = a->kv.block_table;
  t.max_blocks = a->kv.max_blocks;
  t.num_blocks = a->kv.num_blocks;
  t.pool = static_cast<const uint8_t*>(a->kv.pool);
  t.block_bytes = kv_block_bytes(a->kv.format, a->kv.ratio, a->kv.dim);
  t.idx = a->idx;
  t.window = static_cast<const uint8_t*>(a->window);
  t.wscale = a->window_scale;
  t.q = a->q;
  t.scale = a->softmax_scale;
  t.out = a->out;
  t.lse = a->lse;
  const size_t T = t.T, S = t.splits, H = t.H, D = t.D;
  t.part_o = static_cast<uint16_t*>(ws);
  t.part_ml = reinterpret_cast<float*>(static_cast<uint8_t*>(ws) + ((T * S * H * D * 2 + 255) & ~size_t(255)));
  t.status = a->status;
  t.idesc_s = tc::make_idesc(1, 1, kRows, kKeys);
  t.idesc_pv = tc::make_idesc(1, 1, kRows, D > 256 ? 256 : D) | (1u << 16);   // B is MN-major
  // At least 116 KB so that no two CTAs of a TMEM-allocating kernel ever share
  // an SM: every tcgen05 kernel in this library runs one CTA per SM.
  // Q as a 2-D tensor [T*H rows][D] bf16, boxes of 64 columns x 128 rows, 128-B swizzle
  CUtensorMap qmap;
  {
    auto encode = tc::encode_fn();
    if (!encode) return false;
    const cuuint64_t gdim[2] = {cuuint64_t(D), cuuint64_t(T) * H};
    const cuuint64_t gstride[1] = {cuuint64_t(D) * 2};
    const cuuint32_t box[2] = {64, kRows};
    const cuuint32_t es[2] = {1, 1};
    if (encode(&qmap, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<uint16_t*>(a->q), gdim, gstride, box, es,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return false;
  }
  size_t smem = 1024 + D * kRows * 2 + D * kKeys * 2 + kRows * 128 + sizeof(ASmem);
  if (smem < 116 * 1024) smem = 116 * 1024;
  static std::once_flag once;
  std::call_once(once, [] {
    cudaFuncSetAttribute(attn_chunk_tc, cudaFuncAttributeMaxDynamicSharedMemorySize, 227 * 1024);
  });
  if (smem > 227 * 1024) return false;
  attn_chunk_tc<<<dim3(t.splits, t.T), kThreads, smem, stream>>>(t, qmap);
  if (t.splits > 1)
    attn_combine_bf16<<<dim3(t.H, t.T), t.D / 8 < 32 ? 32 : t.D / 8, 0, stream>>>(t.H, t.D, t.splits, t.part_o,
                                                                                t.part_ml, t.out, t.lse);
  if (cudaGetLastError() != cudaSuccess) *rc = V4A_ERR_CUDA;
  return true;
}

}  // namespace v4a
