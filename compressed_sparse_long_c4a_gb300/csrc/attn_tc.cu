// Shared-K=V sparse attention on the tensor cores (tcgen05, kind::f16, bf16
// operands, fp32 accumulate in TMEM), for decode-sized batches.
//
// Method: "DeepSeek V4 in vLLM: Efficient Long-context Attention", Background
// (keys and values share one vector; attend to the top-k compressed entries
// plus the 128 uncompressed window tokens) and Appendix ("why inverse RoPE":
// o_m = sum_n softmax(q_m . k_n) k_n).
//
// One CTA per (64-key chunk of a query's key list, query):
//   Q     [128 rows = heads, zero-padded][D] bf16  -> smem by TMA, K-major,
//         128-B swizzle
//   K     64 gathered rows [64][D] bf16 (fp8 codes are converted exactly to
//         bf16 on the way in; their per-row scale is applied to the logits
//         and to P)
//   S     = Q K^T           M=128, N=64,  K=D   -> summed from 2-4 partial
//         accumulators of 64 TMEM columns, each over a quarter (half) of K
//   P     = 2^(S*f_n - max) * s_n, bf16 -> smem (one thread per head row;
//         f_n = tau * log2(e) * s_n folds the softmax scale and the key's
//         dequantisation scale into one factor per key)
//   O     = P K             M=128, N=256 per MMA (K as an MN-major operand),
//                           K=64              -> TMEM columns [0, D) (the S
//                           columns are reused once S has been read)
// The chunk's normalised O is written as bf16 rows into shared memory (the Q
// buffer, free once S is done) in the 128-byte swizzled layout of 64-column
// boxes, and leaves with TMA tensor stores: whole lines, no partial-sector
// writes.  With several chunks per query the rows go to the workspace with
// the chunk's (max, sum) and a combine kernel merges them; with one chunk
// they are the output.  The MMAs are issued by one lane of each of several
// warps (an issuing thread stalls ~0.1 us per instruction); completion is
// tracked with tcgen05.commit on mbarriers whose waits are bounded.

#include <mutex>

#include "attn_tc.h"
#include "tc_common.cuh"

namespace v4a {
namespace {

constexpr int kKeys = 64;            // keys per CTA (one chunk)
constexpr int kRows = 128;           // MMA M (heads, zero-padded)
constexpr int kThreads = 256;        // warps 0-3 own TMEM lane quarters for the softmax; all 8 drain
constexpr float kLog2e = 1.4426950408889634f;

struct AtcArgs {
  int T, H, D, ratio, fmt, wfmt, wlen, k, splits;
  const int32_t* seq_ids;
  const int32_t* positions;
  const int32_t* bt;
  int max_blocks;
  int64_t num_blocks;
  const uint8_t* pool;
  int64_t block_bytes;
  const int32_t* idx;
  RingDev wring;      // the window ring (dense or paged)
  const uint16_t* q;
  float scale;
  uint16_t* out;
  float* lse;
  uint16_t* part_o;   // [T][splits][H][D] bf16, normalised by the chunk's sum
  float* part_ml;     // [T][splits][H][2] = (max, sum); max in log2 units
  int32_t* status;
  uint32_t idesc_s, idesc_pv;
  int sparts;         // S partial accumulators (K split over that many MMA issuers)
  int rshift, eshift; // log2 of the compression ratio and of the entries per block
  int nq;             // N groups of O = P K (one MMA issuer each)
  int tma_out;        // rows leave through the output tensor map (H % 8 == 0)
  int kv_align8;      // cache rows start on 8 bytes only: read them as two 8-byte halves
  int direct;         // one chunk per query and no merge kernel after: rows are the output
};

struct ASmem {   // every field read with vector loads carries its alignment explicitly
  uint64_t bar_q, bar_s, bar_o[2];
  uint32_t tmem_base;
  int abort_flag;
  const uint8_t* src[kKeys];
  alignas(16) float kf[kKeys];      // tau * log2(e) * key scale, or 0 for an empty slot (read as float4)
  alignas(16) float ks[kKeys];      // key scale (applied to P), 0 for an empty slot (read as float4)
  int kfmt[kKeys];                  // -1: no key in this slot
  const float* sptr[kKeys];         // the key's dequantisation scale, or null (scale 1)
  float red_m[2][kRows], red_l[2][kRows];   // per-half row maxima / sums of the softmax
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

// 32 lanes x 16 consecutive fp32 columns into v[0..15], not waited for: the
// registers are valid only after tc::tmem_wait_ld on the array holding them.
__device__ __forceinline__ void tmem_ld16_nowait(uint32_t taddr, float* v) {
  uint32_t* r = reinterpret_cast<uint32_t*>(v);
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];\n"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr)
      : "memory");
}

// 16 bytes from an address that is 8-byte aligned only, as two 8-byte loads.
__device__ __forceinline__ uint4 ld16_8x2(const uint8_t* p) {
  const uint2 lo = __ldg(reinterpret_cast<const uint2*>(p)), hi = __ldg(reinterpret_cast<const uint2*>(p + 8));
  return make_uint4(lo.x, lo.y, hi.x, hi.y);
}

__device__ __forceinline__ uint32_t bf16x2_mul(uint32_t x, uint32_t m) {
  uint32_t r;
  asm("mul.rn.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(x), "r"(m));
  return r;
}

// Exact e4m3 -> bf16 of the four codes in w (lowest byte first), in integer
// and bf16 arithmetic only (the conversion instructions are the slow part of
// staging a key tile otherwise).  A code's sign goes to bit 15 and its 7
// magnitude bits to bits 4..10, giving the bf16 whose exponent field is the
// code's 4-bit exponent field: the code's value times 2^-120, a subnormal bf16
// for a subnormal code.  One bf16x2 multiply by 2^120 (bf16 arithmetic keeps
// subnormal inputs) restores it.  The NaN codes 0x7F / 0xFF, which the encoder
// never writes, come out as +-480.
__device__ __forceinline__ uint2 bf16x4_from_e4m3x4(uint32_t w) {
  const uint32_t a = __byte_perm(w, 0u, 0x1404);   // code 1 << 24 | code 0 << 8
  const uint32_t b = __byte_perm(w, 0u, 0x3424);   // code 3 << 24 | code 2 << 8
  const uint32_t ma = ((a >> 4) & 0x07F007F0u) | (a & 0x80008000u);
  const uint32_t mb = ((b >> 4) & 0x07F007F0u) | (b & 0x80008000u);
  uint2 r;
  asm("mul.rn.bf16x2 %0, %1, %2;" : "=r"(r.x) : "r"(ma), "r"(0x7B807B80u));   // 0x7B80 = bf16 2^120
  asm("mul.rn.bf16x2 %0, %1, %2;" : "=r"(r.y) : "r"(mb), "r"(0x7B807B80u));
  return r;
}

// Byte offset of 16-byte chunk `ch` (0..7) of row r inside a 128-byte swizzled box.
__device__ __forceinline__ uint32_t sw_off(int r, int ch) { return uint32_t(r * 128 + ((ch ^ (r & 7)) << 4)); }

// kD: the head dimension as a compile-time constant, so that the index
// arithmetic of the staging and drain loops is shifts and masks (these
// phases run on a few warps per SM and are bound by instruction latency).
// kDsv4: the cache holds DeepSeek-V4 584-byte rows (kD = 512); a separate
// instance, so that the other formats' staging keeps all its loads in
// flight without the extra registers that layout needs.
template <int kD, bool kDsv4 = false>
__global__ void __launch_bounds__(kThreads, 1) attn_chunk_tc(const AtcArgs a,
                                                             const __grid_constant__ CUtensorMap qmap,
                                                             const __grid_constant__ CUtensorMap omap) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  constexpr int D = kD, nsub = kD / 64;
  uint8_t* Qs = base;                                  // nsub x [128 rows][128 B]; later the O rows
  uint8_t* Ks = Qs + nsub * kRows * 128;               // nsub x [64 rows][128 B]
  uint8_t* Ps = Ks + nsub * kKeys * 128;               // [128 rows][128 B]
  ASmem& s = *reinterpret_cast<ASmem*>(Ps + kRows * 128);
  const int tid = threadIdx.x, warp = tid >> 5;
  const int t = blockIdx.y, sp = blockIdx.x;
  const int b = a.seq_ids[t], m = a.positions[t];
  const int nvis = (m + 1) >> a.rshift;
  const int nsel = a.idx ? a.k : nvis;
  const int wstart = max(0, m - a.wlen + 1);
  const int L = nsel + (m - wstart + 1);
  const int lo = sp * kKeys;
  const int64_t pi0 = int64_t(t) * a.splits + sp;
  pdl_trigger();

  if (lo >= L) {   // this query's list is shorter than the longest: empty chunk
    pdl_wait();
    for (int h = tid; h < a.H; h += blockDim.x) {
      a.part_ml[(pi0 * a.H + h) * 2] = -INFINITY;
      a.part_ml[(pi0 * a.H + h) * 2 + 1] = 0.f;
    }
    return;
  }
  if (tid == 0) {
    tc::mbar_init(&s.bar_q, 1);
    tc::mbar_init(&s.bar_s, uint32_t(a.sparts));           // every S issuer's commit
    const int halves = D > 256 ? D / 256 : 1;
    tc::mbar_init(&s.bar_o[0], uint32_t(a.nq / halves));   // the O issuers of each half
    tc::mbar_init(&s.bar_o[1], uint32_t(a.nq / halves));
    s.abort_flag = 0;
    tc::mbar_fence_init();
    if (a.tma_out) tc::prefetch_tmap(&omap);
    tc::prefetch_tmap(&qmap);
  }
  __syncwarp();   // tcgen05.alloc is warp-collective: reconverge warp 0 after the init above
  if (warp == 0) tc::tmem_alloc(&s.tmem_base, D < 64 ? 64 : D);
  // everything above overlaps the previous kernel; the queries (which the
  // compressor call may have just normalised and rotated), the selected
  // indices, the caches and the window ring are read only after it has
  // completed
  pdl_wait();
  if (tid == 0) {
    // Q: 128 rows from this query's first head (rows past the last head are
    // the next query's or zero-filled; their outputs are never stored), one
    // 64-column swizzled box per K sub-tile; waited for before the first MMA
    tc::mbar_arrive_expect_tx(&s.bar_q, uint32_t(nsub * kRows * 128));
    for (int sub = 0; sub < nsub; ++sub)
      tc::tma_load_2d(Qs + sub * (kRows * 128), &qmap, sub * 64, t * a.H, &s.bar_q);
  }

  // ---- key slots of this chunk (sources; the scales are loaded with the rows) ----
  if (tid < kKeys) {
    const int li = lo + tid;
    const uint8_t* src = nullptr;
    const float* sp = nullptr;
    int f = -1;
    if (li < L) {
      if (li < nsel) {
        const int e = a.idx ? a.idx[int64_t(t) * a.k + li] : li;
        if (e >= 0) {
          const int E = 1 << a.eshift;
          const int lb = e >> a.eshift;
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
              const int slot = e & (E - 1);
              f = a.fmt;
              src = bb + int64_t(slot) * kv_row_bytes(a.fmt, D);
              if (a.fmt == V4A_KV_FP8_TOKEN) sp = reinterpret_cast<const float*>(bb + int64_t(E) * D) + slot;
            }
          }
        }
      } else {
        const int p = wstart + (li - nsel);
        uint8_t* wrow;
        float* wsc;
        ring_slot(a.wring, b, p % a.wring.cap, &wrow, &wsc, a.status);
        if (wrow) {
          f = a.wfmt;
          src = wrow;
          sp = wsc;
        }
      }
    }
    s.src[tid] = src;
    s.sptr[tid] = sp;
    s.kfmt[tid] = f;
  }
  __syncthreads();

  // ---- stage K into swizzled smem ----
  // bf16 rows: 16-byte cp.async straight into place.  fp8 rows: 16-byte loads
  // (16 codes) into registers, all in flight together, then each converted
  // exactly to 16 bf16 values = two 16-byte chunks.
  {
    constexpr int kBchunks = kKeys * (D / 8);         // 16-byte bf16 chunks of the tile
    constexpr int kPer = kKeys * (D / 16) / kThreads;  // 16-byte fp8 chunks per thread
    // DeepSeek-V4 rows (D = 512): fp8 chunk slots below kNopeChunks hold 16
    // non-rope codes (scale byte cc / 4); each slot above holds 32 bytes of
    // the bf16 rope part (two bf16 chunks)
    constexpr int kNopeChunks = kDsv4Nope / 16;
    uint4 raw[kPer];
    uint4 raw2[kDsv4 ? kPer : 1];
    uint32_t sbyte[kDsv4 ? kPer : 1];
#pragma unroll
    for (int i = 0; i < kPer; ++i) {
      const int c = tid + i * kThreads;
      const int r = c / (D / 16), cc = c % (D / 16);
      raw[i] = make_uint4(0, 0, 0, 0);
      if (s.kfmt[r] == V4A_KV_FP8_TOKEN) {
        const uint8_t* src = s.src[r] + cc * 16;
        raw[i] = a.kv_align8 ? ld16_8x2(src) : __ldg(reinterpret_cast<const uint4*>(src));
      }
      if constexpr (kDsv4) {
        raw2[i] = make_uint4(0, 0, 0, 0);
        sbyte[i] = 127;
        if (s.kfmt[r] == V4A_KV_FP8_DSV4) {   // rows start on 8 bytes (584-byte stride)
          const uint8_t* row = s.src[r];
          if (cc < kNopeChunks) {
            raw[i] = ld16_8x2(row + cc * 16);
            sbyte[i] = __ldg(row + kDsv4Nope + 2 * kDsv4Rope + (cc >> 2));
          } else {
            const uint8_t* rp = row + kDsv4Nope + 32 * (cc - kNopeChunks);
            raw[i] = ld16_8x2(rp);
            raw2[i] = ld16_8x2(rp + 16);
          }
        }
      }
    }
    float sc = 1.f;   // thread tid < kKeys: key tid's scale, in flight with the rows
    if (tid < kKeys && s.sptr[tid]) sc = __ldg(s.sptr[tid]);
    if (a.fmt == V4A_KV_BF16 || a.wfmt == V4A_KV_BF16) {
      for (int c = tid; c < kBchunks; c += kThreads) {
        const int r = c / (D / 8), cc = c % (D / 8);
        if (s.kfmt[r] != V4A_KV_BF16) continue;
        uint8_t* dst = Ks + (cc >> 3) * (kKeys * 128) + sw_off(r, cc & 7);
        asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(tc::smem_u32(dst)), "l"(s.src[r] + cc * 16)
                     : "memory");
      }
    }
#pragma unroll
    for (int i = 0; i < kPer; ++i) {
      const int c = tid + i * kThreads;
      const int r = c / (D / 16), cc = c % (D / 16);   // fp8 chunk cc -> bf16 chunks 2cc, 2cc+1
      const int f = s.kfmt[r];
      if (f == V4A_KV_BF16) continue;
      uint4 v0 = make_uint4(0, 0, 0, 0), v1 = make_uint4(0, 0, 0, 0);
      bool codes = f == V4A_KV_FP8_TOKEN;
      if constexpr (kDsv4) codes = codes || (f == V4A_KV_FP8_DSV4 && cc < kNopeChunks);
      if (codes) {
        const uint2 b0 = bf16x4_from_e4m3x4(raw[i].x), b1 = bf16x4_from_e4m3x4(raw[i].y);
        const uint2 b2 = bf16x4_from_e4m3x4(raw[i].z), b3 = bf16x4_from_e4m3x4(raw[i].w);
        v0 = make_uint4(b0.x, b0.y, b1.x, b1.y);
        v1 = make_uint4(b2.x, b2.y, b3.x, b3.y);
        if constexpr (kDsv4) {
          if (f == V4A_KV_FP8_DSV4) {
            // times the block's power of two, a bf16 with exponent field = the
            // scale byte (exact while the product stays a normal bf16)
            const uint32_t m = (sbyte[i] << 7) | (sbyte[i] << 23);
            v0 = make_uint4(bf16x2_mul(v0.x, m), bf16x2_mul(v0.y, m), bf16x2_mul(v0.z, m), bf16x2_mul(v0.w, m));
            v1 = make_uint4(bf16x2_mul(v1.x, m), bf16x2_mul(v1.y, m), bf16x2_mul(v1.z, m), bf16x2_mul(v1.w, m));
          }
        }
      } else {
        if constexpr (kDsv4) {
          if (f == V4A_KV_FP8_DSV4) {   // rope: bf16 as stored
            v0 = raw[i];
            v1 = raw2[i];
          }
        }
      }
      const int c0 = 2 * cc;
      uint8_t* sub = Ks + (c0 >> 3) * (kKeys * 128);
      *reinterpret_cast<uint4*>(sub + sw_off(r, c0 & 7)) = v0;
      *reinterpret_cast<uint4*>(sub + sw_off(r, (c0 + 1) & 7)) = v1;
    }
    if (tid < kKeys) {   // read after the barrier before the MMAs
      const bool live = s.kfmt[tid] >= 0;
      s.kf[tid] = live ? sc * a.scale * kLog2e : 0.f;
      s.ks[tid] = live ? sc : 0.f;
    }
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
  // One thread issuing tcgen05.mma stalls ~0.1 us per instruction; several
  // issuing warps overlap up to the SM's rate of ~30 ns per instruction
  // (either measured on GB300, at N = 32 or 64).  The D/16 K steps are split
  // over `sparts` issuers (lane 0 of warps 0..sparts-1), each into its own
  // 64-column partial accumulator; the softmax sums the partials.
  if ((tid & 31) == 0 && warp < a.sparts) {
    const uint32_t q0 = tc::smem_u32(Qs), k0 = tc::smem_u32(Ks);
    constexpr int nst = D / 16;
    const int per = nst / a.sparts;
    for (int st = warp * per; st < (warp + 1) * per; ++st) {
      const uint64_t ad = tc::desc_sw128(q0 + (st >> 2) * (kRows * 128)) + 2 * (st & 3);
      const uint64_t bd = tc::desc_sw128(k0 + (st >> 2) * (kKeys * 128)) + 2 * (st & 3);
      tc::mma_f16(tmem + 64 * warp, ad, bd, a.idesc_s, st > warp * per);
    }
    tc::mma_commit(&s.bar_s);
  }
  // ---- softmax: all 8 warps; thread (row, hf) takes keys [32 hf, 32 hf + 32) of head row `row` ----
  // (warps w and w + 4 read the same TMEM lane quarter; the two halves of a
  // row meet through shared memory for the max and the sum)
  const int row = tid & (kRows - 1), hf = warp >> 2;
  const uint32_t lane_addr = tmem + (uint32_t((warp & 3) * 32) << 16);
  // Collective tcgen05 loads below are always executed by whole warps; `ok`
  // is made warp-uniform and only gates the arithmetic and the stores.
  bool ok = __all_sync(0xffffffffu, tc::mbar_wait(&s.bar_s, 0, a.status, abort_flag));
  tc::tc_fence_after();
  float mx, l;
  {
    float v[32];
    {
      float w0[64], w1[64];   // w0: partials 0 and 1, w1: partials 2 and 3 (32 columns each)
      tmem_ld16_nowait(lane_addr + 32 * hf, w0);
      tmem_ld16_nowait(lane_addr + 32 * hf + 16, w0 + 16);
      tmem_ld16_nowait(lane_addr + 64 + 32 * hf, w0 + 32);
      tmem_ld16_nowait(lane_addr + 64 + 32 * hf + 16, w0 + 48);
      if (a.sparts == 4) {
        tmem_ld16_nowait(lane_addr + 128 + 32 * hf, w1);
        tmem_ld16_nowait(lane_addr + 128 + 32 * hf + 16, w1 + 16);
        tmem_ld16_nowait(lane_addr + 192 + 32 * hf, w1 + 32);
        tmem_ld16_nowait(lane_addr + 192 + 32 * hf + 16, w1 + 48);
        tc::tmem_wait_ld(w0);
        tc::tmem_wait_ld(w1);
#pragma unroll
        for (int n = 0; n < 32; ++n) v[n] = (w0[n] + w0[32 + n]) + (w1[n] + w1[32 + n]);
      } else {
        tc::tmem_wait_ld(w0);
#pragma unroll
        for (int n = 0; n < 32; ++n) v[n] = w0[n] + w0[32 + n];
      }
    }
    const float4* kf4 = reinterpret_cast<const float4*>(s.kf) + 8 * hf;
    float m4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
    for (int n = 0; n < 32; n += 4) {
      const float4 f = kf4[n >> 2];
      // z in log2 units; an empty slot has factor 0 and is masked
      v[n] *= f.x; v[n + 1] *= f.y; v[n + 2] *= f.z; v[n + 3] *= f.w;
      if (f.x != 0.f) m4[0] = fmaxf(m4[0], v[n]);
      if (f.y != 0.f) m4[1] = fmaxf(m4[1], v[n + 1]);
      if (f.z != 0.f) m4[2] = fmaxf(m4[2], v[n + 2]);
      if (f.w != 0.f) m4[3] = fmaxf(m4[3], v[n + 3]);
    }
    s.red_m[hf][row] = fmaxf(fmaxf(m4[0], m4[1]), fmaxf(m4[2], m4[3]));
    __syncthreads();
    mx = fmaxf(s.red_m[0][row], s.red_m[1][row]);
    const float4* ks4 = reinterpret_cast<const float4*>(s.ks) + 8 * hf;
    uint32_t pk[16];
    float l4[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int n = 0; n < 32; n += 4) {
      const float4 k = ks4[n >> 2];
      const float p0 = k.x != 0.f ? exp2f(v[n] - mx) : 0.f;
      const float p1 = k.y != 0.f ? exp2f(v[n + 1] - mx) : 0.f;
      const float p2 = k.z != 0.f ? exp2f(v[n + 2] - mx) : 0.f;
      const float p3 = k.w != 0.f ? exp2f(v[n + 3] - mx) : 0.f;
      l4[0] += p0; l4[1] += p1; l4[2] += p2; l4[3] += p3;
      const __nv_bfloat162 b01 = __floats2bfloat162_rn(p0 * k.x, p1 * k.y);
      const __nv_bfloat162 b23 = __floats2bfloat162_rn(p2 * k.z, p3 * k.w);
      pk[n >> 1] = *reinterpret_cast<const uint32_t*>(&b01);
      pk[(n >> 1) + 1] = *reinterpret_cast<const uint32_t*>(&b23);
    }
#pragma unroll
    for (int c = 0; c < 4; ++c)
      *reinterpret_cast<uint4*>(Ps + sw_off(row, 4 * hf + c)) = make_uint4(pk[4 * c], pk[4 * c + 1], pk[4 * c + 2], pk[4 * c + 3]);
    s.red_l[hf][row] = (l4[0] + l4[1]) + (l4[2] + l4[3]);
  }
  tc::fence_proxy_async();
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  // ---- O = P K (S columns are free again) ----
  // D split into `nq` N groups, one MMA issuer each (lane 0 of warps
  // 0..nq-1); the groups of each N = 256 half commit to that half's barrier,
  // so the first half drains while the tensor core computes the second.
  const int halves = D > 256 ? D / 256 : 1;
  if ((tid & 31) == 0 && warp < a.nq && !*abort_flag) {
    const uint32_t p0 = tc::smem_u32(Ps), k0 = tc::smem_u32(Ks);
    const int N = D / a.nq, g = warp;              // this issuer's columns [g * N, g * N + N)
    for (int st = 0; st < kKeys / 16; ++st) {
      const uint64_t ad = tc::desc_sw128(p0) + 2 * st;
      const uint64_t bd = desc_sw128_mn(k0 + g * (N / 64) * (kKeys * 128) + st * 16 * 128, kKeys * 128);
      tc::mma_f16(tmem + g * N, ad, bd, a.idesc_pv, st > 0);
    }
    tc::mma_commit(&s.bar_o[(g * N) / (D / halves)]);
  }
  l = s.red_l[0][row] + s.red_l[1][row];   // written before the barrier above
  const bool store = ok && row < a.H;   // H need not be a multiple of 32: loads stay warp-wide
  const float inv = l > 0.f ? 1.f / l : 0.f;   // a chunk of only padding (-1) entries has l = 0
  const bool direct = a.direct != 0;
  // each half's 64-column groups: warps 0-3 drain the first half of them, warps 4-7 the rest
  const int per_half = nsub / halves;
  for (int half = 0; half < halves; ++half) {
    ok = __all_sync(0xffffffffu, ok && tc::mbar_wait(&s.bar_o[half], 0, a.status, abort_flag));
    tc::tc_fence_after();
    const int g0 = half * per_half, gh = per_half / 2;
    const int c0 = warp < 4 ? g0 : g0 + gh, c1 = warp < 4 ? g0 + gh : g0 + per_half;
    for (int c = c0; c < c1; ++c) {
      float v[64];
      tc::tmem_ld64(lane_addr + c * 64, v);
      if (!(store && ok)) continue;
      uint4 o[8];
#pragma unroll
      for (int i = 0; i < 64; i += 8) {
        __nv_bfloat162 b0 = __floats2bfloat162_rn(v[i] * inv, v[i + 1] * inv);
        __nv_bfloat162 b1 = __floats2bfloat162_rn(v[i + 2] * inv, v[i + 3] * inv);
        __nv_bfloat162 b2 = __floats2bfloat162_rn(v[i + 4] * inv, v[i + 5] * inv);
        __nv_bfloat162 b3 = __floats2bfloat162_rn(v[i + 6] * inv, v[i + 7] * inv);
        o[i >> 3] = make_uint4(*reinterpret_cast<uint32_t*>(&b0), *reinterpret_cast<uint32_t*>(&b1),
                               *reinterpret_cast<uint32_t*>(&b2), *reinterpret_cast<uint32_t*>(&b3));
      }
      if (a.tma_out) {
        // rows -> bf16 in the (free) Q buffer as a swizzled 64-column box
        uint8_t* box = Qs + c * (kRows * 128);
#pragma unroll
        for (int i = 0; i < 8; ++i) *reinterpret_cast<uint4*>(box + sw_off(row, i)) = o[i];
      } else {
        uint16_t* dst = direct ? a.out + (int64_t(t) * a.H + row) * D : a.part_o + (pi0 * a.H + row) * D;
#pragma unroll
        for (int i = 0; i < 8; ++i) *reinterpret_cast<uint4*>(dst + c * 64 + i * 8) = o[i];
      }
    }
    if (a.tma_out) {
      // this half's boxes leave with TMA tensor stores while the next half drains
      tc::fence_proxy_async();
      __syncthreads();
      if (tid == 0 && ok) {
        const int y = direct ? t * a.H : int(pi0) * a.H;
        for (int c = g0; c < g0 + per_half; ++c) tc::tma_store_2d(&omap, Qs + c * (kRows * 128), c * 64, y);
        tc::bulk_commit();
      }
    }
  }
  if (a.tma_out && tid == 0) tc::bulk_wait_read();   // shared memory stays valid until the stores have read it
  if (store && warp < 4) {
    if (direct) {
      if (a.lse) a.lse[int64_t(t) * a.H + row] = (mx + log2f(l)) * (1.f / kLog2e);
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

// out = sum_s w_s * O_s with w_s = l_s 2^{m_s} / sum_s' l_s' 2^{m_s'} (m in log2 units).
// One CTA per (head, query), 256 threads = 4 split groups x 64 threads; a
// thread owns one 8-dim chunk of the row (D <= 512) and the splits
// s = group (mod 4).  Its partial-row loads are issued first, before the
// split weights are known, so the whole CTA waits on one L2 round trip; the
// four groups are summed through shared memory.  Many small CTAs spread the
// partial rows over every SM (one SM alone streams them slowly).
constexpr int kCombGroups = 4;
constexpr int kCombMax = 16;     // splits per group held in registers per round (one round up to 64)
constexpr int kMaxSplits = 1024; // chunks per query (c128a at 1M: 130)

__global__ void __launch_bounds__(256, 2) attn_combine_bf16(int H, int D, int splits, const uint16_t* part_o,
                                                            const float* part_ml, uint16_t* out, float* lse) {
  pdl_trigger();
  pdl_wait();   // the partials are the previous kernel's output
  __shared__ float wsm[kMaxSplits];
  __shared__ float inv_s;
  __shared__ float4 part_s[kCombGroups - 1][64][2];
  const int t = blockIdx.y, h = blockIdx.x;
  const int grp = threadIdx.x >> 6, c = threadIdx.x & 63;
  const bool active = c < D / 8;
  const uint16_t* po = part_o + (int64_t(t) * splits * H + h) * D + c * 8;
  // 1. this thread's first round of partial chunks, in flight together
  uint4 v[kCombMax];
#pragma unroll
  for (int u = 0; u < kCombMax; ++u) {
    const int sp = grp + u * kCombGroups;
    v[u] = (active && sp < splits) ? __ldcg(reinterpret_cast<const uint4*>(po + int64_t(sp) * H * D))
                                   : make_uint4(0, 0, 0, 0);
  }
  // 2. weights of every split (warp 0), while those loads are in flight;
  //    lane l takes splits l, l + 32, ... in order
  if (threadIdx.x < 32) {
    const int lane = threadIdx.x;
    const float* ml = part_ml + (int64_t(t) * splits * H + h) * 2;
    float mx = -INFINITY;
    for (int sp = lane; sp < splits; sp += 32) mx = fmaxf(mx, ml[int64_t(sp) * H * 2]);
    mx = warp_max(mx);
    float tl = 0.f;
    for (int sp = lane; sp < splits; sp += 32) {
      const float m = ml[int64_t(sp) * H * 2], l = ml[int64_t(sp) * H * 2 + 1];
      const float w = m == -INFINITY ? 0.f : l * exp2f(m - mx);
      wsm[sp] = w;
      tl += w;
    }
    const float tot = warp_sum(tl);
    if (lane == 0) {
      inv_s = tot > 0.f ? 1.f / tot : 0.f;
      if (lse) lse[int64_t(t) * H + h] = (mx + log2f(tot)) * 0.6931471805599453f;
    }
  }
  __syncthreads();
  // 3. weighted sum of this thread's splits in increasing order, round by
  //    round (an empty chunk has weight 0 and its row is never read into the sum)
  float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
  for (int u0 = 0;; u0 += kCombMax) {
#pragma unroll
    for (int u = 0; u < kCombMax; ++u) {
      const int sp = grp + (u0 + u) * kCombGroups;
      const float w = sp < splits ? wsm[sp] : 0.f;
      if (w == 0.f) continue;
      const uint32_t q[4] = {v[u].x, v[u].y, v[u].z, v[u].w};
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        acc[2 * j] = fmaf(w, bf16_to_f32(uint16_t(q[j] & 0xffffu)), acc[2 * j]);
        acc[2 * j + 1] = fmaf(w, bf16_to_f32(uint16_t(q[j] >> 16)), acc[2 * j + 1]);
      }
    }
    if ((u0 + kCombMax) * kCombGroups >= splits) break;
#pragma unroll
    for (int u = 0; u < kCombMax; ++u) {   // the next round's rows
      const int sp = grp + (u0 + kCombMax + u) * kCombGroups;
      v[u] = (active && sp < splits) ? __ldcg(reinterpret_cast<const uint4*>(po + int64_t(sp) * H * D))
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
    for (int g2 = 0; g2 < kCombGroups - 1; ++g2) {
      const float4 x = part_s[g2][c][0], y = part_s[g2][c][1];
      acc[0] += x.x; acc[1] += x.y; acc[2] += x.z; acc[3] += x.w;
      acc[4] += y.x; acc[5] += y.y; acc[6] += y.z; acc[7] += y.w;
    }
    const float inv = inv_s;
    uint32_t o[4];
#pragma unroll
    for (int j = 0; j < 4; ++j)
      o[j] = uint32_t(f32_to_bf16(acc[2 * j] * inv)) | (uint32_t(f32_to_bf16(acc[2 * j + 1] * inv)) << 16);
    *reinterpret_cast<uint4*>(out + (int64_t(t) * H + h) * D + c * 8) = make_uint4(o[0], o[1], o[2], o[3]);
  }
}

int splits_of(const v4a_attn_args* a) {
  const int E = entries_per_block(a->kv.ratio);
  const int64_t nsel = a->idx ? a->k : int64_t(a->kv.max_blocks) * E;
  return int((nsel + a->window_len + kKeys - 1) / kKeys);
}

// One CTA per 64 keys of each query, so the CTA count is T * splits; long
// batches (chunked prefill) run as several launches of at most kMaxBatchCtas
// CTAs that share the chunk-result workspace (batch_queries below).
bool handled(const v4a_attn_args* a) {
  const int D = a->kv.dim;
  if (D != 128 && D != 256 && D != 512) return false;
  if (a->num_heads > kRows) return false;
  if (splits_of(a) > kMaxSplits) return false;
  // key rows are read with 16-byte loads, or two 8-byte loads when the block
  // size is a multiple of 8 only (an fp8 c128a block holds 2 x (512 + 4) B),
  // so the pool and the window ring must start on 16 bytes.  A window-only
  // call reads no cache entry.
  const bool reads_cache = !a->idx || a->k > 0;
  if (a->kv.format == V4A_KV_FP8_DSV4 && D != kDsv4Nope + kDsv4Rope) return false;
  if (reads_cache && ((kv_block_bytes(a->kv.format, a->kv.ratio, D) & 7) ||
                      (reinterpret_cast<uintptr_t>(a->kv.pool) & 15)))
    return false;
  // a paged window ring is 16-byte aligned by its descriptor's rules
  if (!a->window_pages && (reinterpret_cast<uintptr_t>(a->window) & 15)) return false;
  return true;
}

// Queries per launch: long batches (chunked prefill) run as several launches
// of at most kMaxBatchCtas CTAs, each reusing the same chunk-result workspace.
constexpr int64_t kMaxBatchCtas = 64 * 152;
int64_t batch_queries(const v4a_attn_args* a) {
  const int64_t T = a->batch.num_tokens, S = splits_of(a);
  const int64_t q = kMaxBatchCtas / S;
  return q < 1 ? 1 : (q < T ? q : T);
}

// 2-D bf16 tensor map [rows][D] with boxes of 64 columns x box_rows rows, 128-B swizzle.
bool encode_rows(CUtensorMap* map, const void* base, int64_t rows, int D, int box_rows) {
  auto encode = tc::encode_fn();
  if (!encode) return false;
  const cuuint64_t gdim[2] = {cuuint64_t(D), cuuint64_t(rows)};
  const cuuint64_t gstride[1] = {cuuint64_t(D) * 2};
  const cuuint32_t box[2] = {64, cuuint32_t(box_rows)};
  const cuuint32_t es[2] = {1, 1};
  return encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), gdim, gstride, box, es,
                CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

size_t attn_tc_workspace_size(const v4a_attn_args* a) {
  if (!handled(a)) return 0;
  const size_t T = size_t(batch_queries(a)), S = splits_of(a), H = a->num_heads, D = a->kv.dim;
  return T * S * H * D * 2 + T * S * H * 2 * 4 + 512;
}

int attn_tc_batch_queries(const v4a_attn_args* a) { return handled(a) ? int(batch_queries(a)) : 0; }

bool attn_tc(const v4a_attn_args* a, void* ws, size_t ws_bytes, cudaStream_t stream, int* rc,
             AttnPartials* keep, int t0, int tn) {
  *rc = V4A_OK;
  if (!handled(a)) return false;
  if (ws_bytes < attn_tc_workspace_size(a)) { *rc = V4A_ERR_WORKSPACE; return true; }
  const int Tall = a->batch.num_tokens, Tb = int(batch_queries(a));
  if (tn < 0) {
    // the whole batch: with the merge inside, launch batch after batch here;
    // a caller that merges itself (keep) walks the batches and passes each one
    if (keep && Tall > Tb) { *rc = V4A_ERR_INVALID_ARG; return true; }
    for (int b0 = 0; b0 < Tall && *rc == V4A_OK; b0 += Tb)
      attn_tc(a, ws, ws_bytes, stream, rc, keep, b0, Tall - b0 < Tb ? Tall - b0 : Tb);
    return true;
  }
  if (t0 < 0 || tn < 1 || tn > Tb || t0 + tn > Tall) { *rc = V4A_ERR_INVALID_ARG; return true; }
  const int64_t qrow = int64_t(t0) * a->num_heads;     // first query row of this launch
  AtcArgs t{};
  t.T = tn;
  t.H = a->num_heads;
  t.D = a->kv.dim;
  t.ratio = a->kv.ratio;
  t.rshift = a->kv.ratio == 4 ? 2 : 7;                 // ratio is 4 or 128 (validated by the caller)
  t.eshift = a->kv.ratio == 4 ? 6 : 1;                 // entries per 256-position block: 64 or 2
  t.fmt = a->kv.format;
  t.wfmt = a->window_format;
  t.wlen = a->window_len;
  t.k = a->k;
  t.splits = splits_of(a);
  t.seq_ids = a->batch.seq_ids + t0;
  t.positions = a->batch.positions + t0;
  t.bt = a->kv.block_table;
  t.max_blocks = a->kv.max_blocks;
  t.num_blocks = a->kv.num_blocks;
  t.pool = static_cast<const uint8_t*>(a->kv.pool);
  t.block_bytes = kv_block_bytes(a->kv.format, a->kv.ratio, a->kv.dim);
  t.kv_align8 = (t.block_bytes & 15) != 0 ? 1 : 0;   // (DeepSeek-V4 rows are always read as 8-byte halves)
  t.idx = a->idx ? a->idx + int64_t(t0) * a->k : nullptr;
  if (attn_window_ring(a, &t.wring)) { *rc = V4A_ERR_INVALID_ARG; return true; }
  t.q = a->q + qrow * a->kv.dim;
  t.scale = a->softmax_scale;
  t.out = a->out ? a->out + qrow * a->kv.dim : nullptr;
  t.lse = a->lse ? a->lse + qrow : nullptr;
  const size_t T = t.T, S = t.splits, H = t.H, D = t.D;
  t.part_o = static_cast<uint16_t*>(ws);
  t.part_ml = reinterpret_cast<float*>(static_cast<uint8_t*>(ws) + ((T * S * H * D * 2 + 255) & ~size_t(255)));
  t.direct = (S == 1 && !keep) ? 1 : 0;
  if (keep) *keep = AttnPartials{t.part_o, t.part_ml, int(S)};
  t.status = a->status;
  t.idesc_s = tc::make_idesc(1, 1, kRows, kKeys);
  // S partials: 64 columns each within the D columns allocated; O groups of >= 64 columns
  t.sparts = D >= 256 ? 4 : 2;
  t.nq = D >= 256 ? 4 : 2;
  t.idesc_pv = tc::make_idesc(1, 1, kRows, uint32_t(D / t.nq)) | (1u << 16);   // B is MN-major
  // Q as a 2-D tensor [T*H rows][D] bf16, boxes of 64 columns x 128 rows, 128-B swizzle
  CUtensorMap qmap, omap;
  if (!encode_rows(&qmap, t.q, int64_t(T) * H, int(D), kRows)) { *rc = V4A_ERR_CUDA; return true; }
  // output rows leave through a tensor map when whole boxes of H rows fit the swizzle atom
  t.tma_out = (H % 8 == 0) && (reinterpret_cast<uintptr_t>(t.direct ? static_cast<void*>(t.out) : ws) & 15) == 0;
  if (t.tma_out) {
    const void* dst = t.direct ? static_cast<const void*>(t.out) : static_cast<const void*>(t.part_o);
    const int64_t rows = t.direct ? int64_t(T) * H : int64_t(T) * S * H;
    if (!encode_rows(&omap, dst, rows, int(D), int(H))) t.tma_out = 0;
  }
  if (!t.tma_out) omap = qmap;   // unused
  size_t smem = 1024 + D * kRows * 2 + D * kKeys * 2 + kRows * 128 + sizeof(ASmem);
  // At least 116 KB so that no two CTAs of a TMEM-allocating kernel ever share
  // an SM: every tcgen05 kernel in this library runs one CTA per SM.
  if (smem < 116 * 1024) smem = 116 * 1024;
  static std::once_flag once;
  std::call_once(once, [] {
    cudaFuncSetAttribute(attn_chunk_tc<512>, cudaFuncAttributeMaxDynamicSharedMemorySize, 227 * 1024);
    cudaFuncSetAttribute(attn_chunk_tc<512, true>, cudaFuncAttributeMaxDynamicSharedMemorySize, 227 * 1024);
    cudaFuncSetAttribute(attn_chunk_tc<256>, cudaFuncAttributeMaxDynamicSharedMemorySize, 227 * 1024);
    cudaFuncSetAttribute(attn_chunk_tc<128>, cudaFuncAttributeMaxDynamicSharedMemorySize, 227 * 1024);
  });
  if (smem > 227 * 1024) { *rc = V4A_ERR_UNSUPPORTED; return true; }
  // both may start while the kernel before them runs (they wait in-kernel)
  auto kern = t.fmt == V4A_KV_FP8_DSV4 ? attn_chunk_tc<512, true>
             : D == 512                 ? attn_chunk_tc<512>
             : D == 256                 ? attn_chunk_tc<256>
                                        : attn_chunk_tc<128>;
  cudaError_t e = launch_pdl(kern, dim3(t.splits, t.T), dim3(kThreads), smem, stream, t, qmap, omap);
  if (e == cudaSuccess && !t.direct && !keep)
    e = launch_pdl(attn_combine_bf16, dim3(t.H, t.T), dim3(256), 0, stream, t.H, t.D, t.splits,
                   static_cast<const uint16_t*>(t.part_o), static_cast<const float*>(t.part_ml), t.out, t.lse);
  if (e != cudaSuccess || cudaGetLastError() != cudaSuccess) *rc = V4A_ERR_CUDA;
  return true;
}

}  // namespace v4a
