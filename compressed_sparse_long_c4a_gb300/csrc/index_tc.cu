// Indexer scan on the 5th-generation tensor cores (tcgen05, kind::f8f6f4).
//
// Method: "DeepSeek V4 in vLLM: Efficient Long-context Attention", Background
// "DeepSeek Sparse Attention" (score every compressed entry, keep the top-k),
// with the indexer cache in fp8 (one fp32 scale per 128 elements, the 132-B
// entry of the SGLang KV-pool article, section "DSA") or fp4 e2m1 (one fp32
// scale per 32 elements; vLLM page, Background: fp4 indexer cache).
//
// score_i = sum_h w_h * ReLU(q_h . k_i), q_h = qcode_h * qs_h (e4m3 + fp32
// scale per head), k_i = kcode_i * s_i,b per 32- or 128-element block b.
//
// Tile = 128 entries (two 64-entry physical blocks) x 64 heads x 128 dims.
//  The codes of each physical block arrive with one TMA tile copy through a
//  3-D tensor map over the pool ({128 elements, 64 rows, block}); the copy
//  itself writes the K-major, 128-byte-swizzled MMA operand: fp8 rows as they
//  are, fp4 rows expanded by the copy engine to 16 codes per 16-byte
//  container (the shared-memory form kind::f8f6f4 reads for e2m1).  The
//  block's scale words follow with one 1-D bulk copy.  No thread touches the
//  codes.
//  B = the query's e4m3 codes, N = 64 heads, staged once per query;
//  K = 128 in four MMAs of K = 32.  fp8 keys: the four MMAs accumulate into
//      one 64-column fp32 accumulator (one scale per entry, factored out of
//      the ReLU since scales are positive).  fp4 keys: each MMA writes its own
//      accumulator (one per 32-element scale block), combined in the epilogue
//      as sum_b s_b * acc_b before the ReLU.
// Products of e4m3 x e4m3 / e2m1 codes and their sums are exact or nearly so
// in the fp32 accumulator; the fp32 scales are applied in the epilogue.
//
// Warp roles (320 threads, one CTA per SM, persistent over a contiguous range
// of (query, tile) work items):
//   warp 0      producer: kStages-deep ring of tiles (block ids from a
//               shared-memory window of the block table); also stages the
//               query codes and w_h * qs_h, double-buffered.
//   warp 1      TMEM allocator and single-thread MMA issuer (double-buffered
//               TMEM accumulators).
//   warps 2..9  two epilogue warpgroups, one per accumulator (alternate
//               tiles): one thread per entry (TMEM lane) reads its scale
//               words as soon as the tile lands, then its accumulators, and
//               applies scales, ReLU and head weights with packed fp32x2 FMAs.
//               With a histogram requested it also counts the top 12 bits of
//               the score's order-preserving key in shared memory (flushed
//               to the query's global histogram at every query switch), the
//               first level of the long-row top-k.
// A stage is refilled once its MMAs have completed (commit) and the owning
// epilogue warpgroup has read its scale words.
// Every mbarrier wait is bounded (V4A_DEV_TIMEOUT, then a clean exit).

#include <mutex>

#include "index_tc.h"
#include "tc_common.cuh"

namespace v4a {
namespace {

constexpr int kStages = 10;
constexpr int kBoxBytes = 64 * 128;          // one physical block's codes as an MMA operand (64 rows)
constexpr int kOpBytes = 2 * kBoxBytes;      // 128 rows x 128 smem bytes
constexpr int kScaleBytes = 2 * 1024;        // scale words of two blocks (fp4: 64 x 16 B each)
constexpr int kStageBytes = kOpBytes + kScaleBytes;
constexpr int kQBytes = 64 * 128;            // 64 heads x 128 codes
constexpr int kHistBins = 4096;
constexpr int kEpiWarps = 8;                 // two epilogue warpgroups
constexpr int kEpi0 = 2;                     // first epilogue warp
constexpr int kThreads = 32 * kEpi0 + 32 * kEpiWarps;

struct TcArgs {
  int T, fmt, acc_cols;
  const int32_t* seq_ids;
  const int32_t* positions;
  const int32_t* bt;
  int max_blocks;
  int64_t num_blocks;
  const uint8_t* pool;
  int64_t block_bytes;
  int64_t scale_off;          // byte offset of the scale words inside a block
  uint32_t scale_bytes;       // scale bytes of one block (64 entries)
  uint32_t box_tx;            // transaction bytes of one code box: the packed bytes read (fp4: 4096)
  const uint8_t* q;           // [T][64][128] e4m3
  const float* qs;            // [T][64]
  const float* w;             // [T][64]
  float* scores;
  int64_t row;
  uint32_t* hist;             // [T][kHistBins] or null
  int32_t* status;
  uint32_t idesc;
};

struct Smem {
  uint64_t full[kStages], empty[kStages], tfull[2], tempty[2], qfull[2], qempty[2], done, hsync, hclear;
  uint32_t tmem_base;
  int abort_flag;
  int t0, j0, count;
  uint32_t valid[kStages];  // bit h: block h of the stage's tile was loaded
  int32_t btc[1024];        // producer's window of the current query's block-table row
  uint32_t part[kThreads];
  float wq[2][64];          // w_h * qs_h of the query in each query buffer
};

// Visible entries of query t, never beyond what its block-table row can address.
__device__ __forceinline__ int visible_of(const TcArgs& a, int t) {
  return min((a.positions[t] + 1) / 4, a.max_blocks * 64);
}

__device__ __forceinline__ int tiles_of(const TcArgs& a, int t) {
  return (visible_of(a, t) + 127) / 128;
}

// Walks the flattened (query, tile) list; the tile count of the current query
// is cached so the hot loop touches global memory only at query switches.
struct Cursor {
  int t, j, nt;
  __device__ void init(const TcArgs& a, int t0, int j0) {
    t = t0; j = j0; nt = t0 < a.T ? tiles_of(a, t0) : 0;
  }
  __device__ void next(const TcArgs& a) {
    if (++j >= nt) {
      j = 0;
      do { ++t; nt = t < a.T ? tiles_of(a, t) : 0; } while (t < a.T && nt == 0);
    }
  }
};

// Contiguous share of the flattened (query, tile) list for this CTA.  Each
// thread sums the tiles of a contiguous chunk of queries; the chunk holding
// the CTA's first item is then walked by its owner.
__device__ void plan(const TcArgs& a, Smem& s) {
  const int per = (a.T + blockDim.x - 1) / blockDim.x;
  const int c0 = threadIdx.x * per, c1 = min(a.T, c0 + per);
  uint32_t mine = 0;
  for (int t = c0; t < c1; ++t) mine += tiles_of(a, t);
  // exclusive scan of `mine` over the block: warp shuffles, then warp totals
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5, nw = (blockDim.x + 31) >> 5;
  uint32_t incl = mine;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t x = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += x;
  }
  if (lane == 31) s.part[wid] = incl;
  if (threadIdx.x == 0) { s.count = 0; s.t0 = a.T; s.j0 = 0; }
  __syncthreads();
  uint32_t before = incl - mine, all = 0;
  for (int w = 0; w < nw; ++w) {
    const uint32_t x = s.part[w];
    if (w < wid) before += x;
    all += x;
  }
  const uint32_t lo = uint32_t((uint64_t(all) * blockIdx.x) / gridDim.x);
  const uint32_t hi = uint32_t((uint64_t(all) * (blockIdx.x + 1)) / gridDim.x);
  if (hi > lo && lo >= before && lo < before + mine) {
    uint32_t acc = before;
    for (int t = c0; t < c1; ++t) {
      const uint32_t n = tiles_of(a, t);
      if (lo < acc + n) { s.t0 = t; s.j0 = int(lo - acc); break; }
      acc += n;
    }
    s.count = int(hi - lo);
  }
  __syncthreads();
}

// Adds the shared-memory histogram of query t to its global row and clears it.
// Called by all eight epilogue warps at the same item; they meet on two
// mbarriers (bounded waits, so a warp that gave up elsewhere cannot hang the
// others): every add of the old query is done before any bin is read, and
// every bin is cleared before any add of the next query.
__device__ __forceinline__ bool flush_hist(uint64_t* hsync, uint64_t* hclear, uint32_t& hph, uint32_t* h_s,
                                           uint32_t* g, int et, int32_t* status, volatile int* abort_flag) {
  const int lane = threadIdx.x & 31;
  __syncwarp();
  if (lane == 0) tc::mbar_arrive(hsync);
  bool ok = __all_sync(0xffffffffu, tc::mbar_wait(hsync, hph, status, abort_flag));
  if (ok) {
    for (int i = et; i < kHistBins; i += 32 * kEpiWarps) {
      const uint32_t v = h_s[i];
      if (v) {
        atomicAdd(&g[i], v);
        h_s[i] = 0;
      }
    }
  }
  __syncwarp();
  if (lane == 0) tc::mbar_arrive(hclear);
  ok = __all_sync(0xffffffffu, ok && tc::mbar_wait(hclear, hph, status, abort_flag));
  hph ^= 1;
  return ok;
}

__global__ void __launch_bounds__(kThreads, 1)
index_scan_tc(const TcArgs a, const __grid_constant__ CUtensorMap kmap) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* stages = base;                                   // kStages x (operand, scale words)
  uint8_t* qbuf = stages + kStages * kStageBytes;           // 2 x 8 KB
  uint32_t* hist_s = reinterpret_cast<uint32_t*>(qbuf + 2 * kQBytes);
  Smem& s = *reinterpret_cast<Smem*>(hist_s + kHistBins);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  volatile int* abort_flag = &s.abort_flag;

  if (threadIdx.x == 0) {
    for (int i = 0; i < kStages; ++i) {
      tc::mbar_init(&s.full[i], 1);
      tc::mbar_init(&s.empty[i], 1 + 4);            // MMA commit + the owning epilogue warpgroup
    }
    for (int i = 0; i < 2; ++i) {
      tc::mbar_init(&s.tfull[i], 1);
      tc::mbar_init(&s.tempty[i], 4);
      tc::mbar_init(&s.qfull[i], 1);
      tc::mbar_init(&s.qempty[i], 1 + kEpiWarps);   // MMA commit + every epilogue warp
    }
    tc::mbar_init(&s.done, 1);
    tc::mbar_init(&s.hsync, kEpiWarps);
    tc::mbar_init(&s.hclear, kEpiWarps);
    s.abort_flag = 0;
    tc::mbar_fence_init();
  }
  if (a.hist)
    for (int i = threadIdx.x; i < kHistBins; i += blockDim.x) hist_s[i] = 0;
  __syncwarp();   // tcgen05.alloc is warp-collective
  if (warp == 1) tc::tmem_alloc(&s.tmem_base, 2 * a.acc_cols);
  tc::tc_fence_before();
  plan(a, s);              // contains __syncthreads
  tc::tc_fence_after();
  const uint32_t tmem = s.tmem_base;
  const int count = s.count;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) tc::prefetch_tmap(&kmap);
    Cursor c;
    c.init(a, s.t0, s.j0);
    int cur_t = -1, qi = -1, stage = 0;
    uint32_t phase = 0;
    int issued = 0;
    int b = 0, nblk = 0, btc_base = 0, btc_end = 0;
    for (int it = 0; it < count; ++it) {
      if (c.t != cur_t) {
        cur_t = c.t;
        ++qi;
        const int qb = qi & 1;
        b = a.seq_ids[cur_t];
        nblk = (visible_of(a, cur_t) + 63) / 64;
        btc_base = btc_end = 0;                       // refill the block-table window below
        if (lane == 0 && (a.positions[cur_t] + 1) / 4 > a.max_blocks * 64) report(a.status, V4A_DEV_BAD_BLOCK);
        if (lane == 0 && qi >= 2) tc::mbar_wait(&s.qempty[qb], ((qi >> 1) - 1) & 1, a.status, abort_flag);
        __syncwarp();
        if (*abort_flag) break;
        const uint4* src = reinterpret_cast<const uint4*>(a.q + int64_t(cur_t) * kQBytes);
        uint8_t* dst = qbuf + qb * kQBytes;
        for (int cc = lane; cc < kQBytes / 16; cc += 32) {
          const int r = cc >> 3, ch = cc & 7;
          *reinterpret_cast<uint4*>(dst + r * 128 + ((ch ^ (r & 7)) << 4)) = src[cc];
        }
        for (int h = lane; h < 64; h += 32)
          s.wq[qb][h] = a.w[int64_t(cur_t) * 64 + h] * a.qs[int64_t(cur_t) * 64 + h];
        tc::fence_proxy_async();
        __syncwarp();
        if (lane == 0) tc::mbar_arrive(&s.qfull[qb]);
      }
      // block-table entries of this tile come from a shared-memory window of the
      // row, refilled with coalesced loads by the whole warp
      if (2 * c.j + 1 >= btc_end && 2 * c.j < nblk) {
        btc_base = 2 * c.j;
        btc_end = min(nblk, btc_base + 1024);
        __syncwarp();
        for (int i = lane; i < btc_end - btc_base; i += 32)
          s.btc[i] = a.bt[int64_t(b) * a.max_blocks + btc_base + i];
        __syncwarp();
      }
      if (lane == 0) {
        if (!tc::mbar_wait(&s.empty[stage], phase ^ 1, a.status, abort_flag)) *abort_flag = 1;
      }
      __syncwarp();
      if (*abort_flag) break;
      if (lane == 0) {
        int32_t p[2];
        uint32_t bytes = 0, valid = 0;
        for (int h = 0; h < 2; ++h) {
          const int lb = 2 * c.j + h;
          p[h] = -1;
          if (lb >= nblk) continue;
          p[h] = s.btc[lb - btc_base];
          if (p[h] < 0 || p[h] >= a.num_blocks) { p[h] = -1; report(a.status, V4A_DEV_BAD_BLOCK); continue; }
          bytes += a.box_tx + a.scale_bytes;
          valid |= 1u << h;
        }
        s.valid[stage] = valid;
        uint8_t* st = stages + stage * kStageBytes;
        tc::mbar_arrive_expect_tx(&s.full[stage], bytes);
        for (int h = 0; h < 2; ++h)
          if (p[h] >= 0) {
            tc::tma_load_3d(st + h * kBoxBytes, &kmap, 0, 0, p[h], &s.full[stage]);
            tc::bulk_load(st + kOpBytes + h * a.scale_bytes, a.pool + int64_t(p[h]) * a.block_bytes + a.scale_off,
                          a.scale_bytes, &s.full[stage]);
          }
      }
      ++issued;
      if (++stage == kStages) { stage = 0; phase ^= 1; }
      c.next(a);
    }
    // drain: every issued copy has landed before the CTA can exit (a stage's
    // full barrier completes once per use, so the last phase of each of the
    // last min(issued, kStages) stages is waited for)
    if (lane == 0) {
      const int nd = issued < kStages ? issued : kStages;
      for (int d = 0; d < nd; ++d) {
        stage = (stage + kStages - 1) % kStages;
        const int use = (issued - 1 - d) / kStages;    // how many times this stage was filled before
        const long long t0 = clock64();
        while (!tc::mbar_try_wait(&s.full[stage], uint32_t(use & 1)) && clock64() - t0 < 2000000000LL) {}
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      Cursor c;
      c.init(a, s.t0, s.j0);
      int cur_t = -1, qi = -1, acc = 0, stage = 0;
      uint32_t phase = 0, aphase = 0;
      const uint32_t q0 = tc::smem_u32(qbuf), op0 = tc::smem_u32(stages);
      for (int it = 0; it < count; ++it) {
        if (c.t != cur_t) {
          if (qi >= 0) tc::mma_commit(&s.qempty[qi & 1]);
          cur_t = c.t;
          ++qi;
          if (!tc::mbar_wait(&s.qfull[qi & 1], (qi >> 1) & 1, a.status, abort_flag)) break;
        }
        if (!tc::mbar_wait(&s.full[stage], phase, a.status, abort_flag)) break;
        if (!tc::mbar_wait(&s.tempty[acc], aphase ^ 1, a.status, abort_flag)) break;
        tc::tc_fence_after();
        const uint64_t adesc = tc::desc_sw128(op0 + stage * kStageBytes);
        const uint64_t bdesc = tc::desc_sw128(q0 + (qi & 1) * kQBytes);
        const uint32_t d = tmem + acc * a.acc_cols;
#pragma unroll
        for (int kb = 0; kb < 4; ++kb) {
          // advance 32 bytes of K inside the swizzled 128-byte rows
          if (a.fmt == V4A_IX_FP8_B128)
            tc::mma_f8f6f4(d, adesc + 2 * kb, bdesc + 2 * kb, a.idesc, kb > 0);
          else
            tc::mma_f8f6f4(d + 64 * kb, adesc + 2 * kb, bdesc + 2 * kb, a.idesc, 0);
        }
        tc::mma_commit(&s.empty[stage]);
        tc::mma_commit(&s.tfull[acc]);
        if (++acc == 2) { acc = 0; aphase ^= 1; }
        if (++stage == kStages) { stage = 0; phase ^= 1; }
        c.next(a);
      }
      // all issued MMAs complete before TMEM is released
      tc::mma_commit(&s.done);
      const long long t0 = clock64();
      while (!tc::mbar_try_wait(&s.done, 0) && clock64() - t0 < 2000000000LL) {}
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ epilogue
    // Warpgroup g (warps 2+4g .. 5+4g) owns accumulator g, i.e. every other
    // tile; both warpgroups walk every item to follow the query switches.
    const int g = (warp - kEpi0) >> 2;
    const int quarter = warp & 3;                // TMEM lanes 32*quarter .. +31
    const int row = quarter * 32 + lane;         // entry within the tile
    const int et = threadIdx.x - 32 * kEpi0;     // 0 .. 255
    const uint32_t lane_addr = tmem + (uint32_t(quarter * 32) << 16) + g * a.acc_cols;
    const bool fp8 = a.fmt == V4A_IX_FP8_B128;
    Cursor c;
    c.init(a, s.t0, s.j0);
    int cur_t = -1, qi = -1, n = 0, stage = 0;
    uint32_t phase = 0, aphase = 0, hph = 0;
    float* srow = nullptr;
    const float* wq = nullptr;
    bool aborted = false;
    for (int it = 0; it < count; ++it) {
      if (c.t != cur_t) {
        if (cur_t >= 0) {
          __syncwarp();
          if (lane == 0) tc::mbar_arrive(&s.qempty[qi & 1]);   // done with the old head weights
          if (a.hist && !flush_hist(&s.hsync, &s.hclear, hph, hist_s, a.hist + int64_t(cur_t) * kHistBins, et,
                                    a.status, abort_flag)) {
            aborted = true;
            break;
          }
        }
        cur_t = c.t;
        ++qi;
        n = visible_of(a, cur_t);
        srow = a.scores + int64_t(cur_t) * a.row;
        if (!__all_sync(0xffffffffu, tc::mbar_wait(&s.qfull[qi & 1], (qi >> 1) & 1, a.status, abort_flag))) {
          aborted = true;
          break;
        }
        wq = s.wq[qi & 1];
      }
      if ((it & 1) == g) {
        const int e = c.j * 128 + row;
        // scale words and validity land with the stage's copies: read them and
        // release the stage's scale part before the accumulator is ready
        if (!__all_sync(0xffffffffu, tc::mbar_wait(&s.full[stage], phase, a.status, abort_flag))) {
          aborted = true;
          break;
        }
        const bool blk_ok = (s.valid[stage] >> (row >> 6)) & 1u;
        const uint8_t* sp = stages + stage * kStageBytes + kOpBytes + (row >> 6) * a.scale_bytes;
        float sc0, sc1 = 0.f, sc2 = 0.f, sc3 = 0.f;
        if (fp8) {
          sc0 = reinterpret_cast<const float*>(sp)[row & 63];
        } else {
          const float4 v4 = reinterpret_cast<const float4*>(sp)[row & 63];
          sc0 = v4.x; sc1 = v4.y; sc2 = v4.z; sc3 = v4.w;
        }
        __syncwarp();
        if (lane == 0) tc::mbar_arrive(&s.empty[stage]);
        if (!__all_sync(0xffffffffu, tc::mbar_wait(&s.tfull[g], aphase, a.status, abort_flag))) {
          aborted = true;
          break;
        }
        tc::tc_fence_after();
        float score;
        if (fp8) {
          float v[64];
          tc::tmem_ld64(lane_addr, v);
          float2 sum = make_float2(0.f, 0.f);
#pragma unroll
          for (int h = 0; h < 64; h += 2) {
            const float2 r = make_float2(fmaxf(v[h], 0.f), fmaxf(v[h + 1], 0.f));
            sum = __ffma2_rn(r, make_float2(wq[h], wq[h + 1]), sum);
          }
          score = (sum.x + sum.y) * sc0;
        } else {
          float2 sum = make_float2(0.f, 0.f);
          const float2 s0 = make_float2(sc0, sc0), s1 = make_float2(sc1, sc1);
          const float2 s2 = make_float2(sc2, sc2), s3 = make_float2(sc3, sc3);
#pragma unroll
          for (int hg = 0; hg < 4; ++hg) {
            float v[64];
            tc::tmem_ld4x16(lane_addr + hg * 16, 64, v);
#pragma unroll
            for (int i = 0; i < 16; i += 2) {
              float2 d = __fmul2_rn(make_float2(v[i], v[i + 1]), s0);
              d = __ffma2_rn(make_float2(v[16 + i], v[17 + i]), s1, d);
              d = __ffma2_rn(make_float2(v[32 + i], v[33 + i]), s2, d);
              d = __ffma2_rn(make_float2(v[48 + i], v[49 + i]), s3, d);
              d.x = fmaxf(d.x, 0.f);
              d.y = fmaxf(d.y, 0.f);
              sum = __ffma2_rn(d, make_float2(wq[hg * 16 + i], wq[hg * 16 + i + 1]), sum);
            }
          }
          score = sum.x + sum.y;
        }
        tc::tc_fence_before();
        __syncwarp();
        if (lane == 0) tc::mbar_arrive(&s.tempty[g]);
        if (e < n) {
          const float sv = blk_ok ? score : -INFINITY;
          srow[e] = sv;
          if (a.hist) atomicAdd(&hist_s[float_key(sv) >> 20], 1u);
        }
        aphase ^= 1;
      }
      if (++stage == kStages) { stage = 0; phase ^= 1; }
      c.next(a);
    }
    // the last query's counts (a warp that gave up skips this; the others'
    // bounded waits then see the abort flag)
    if (a.hist && cur_t >= 0 && !aborted)
      flush_hist(&s.hsync, &s.hclear, hph, hist_s, a.hist + int64_t(cur_t) * kHistBins, et, a.status, abort_flag);
    __syncwarp();
  }
  tc::tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc::tc_fence_after();
    tc::tmem_dealloc(tmem, 2 * a.acc_cols);
  }
}

// ---- host side -------------------------------------------------------------------

}  // namespace

bool index_score_tc_supported(const v4a_index_args* a) {
  const v4a_cache& c = a->keys;
  if (c.format != V4A_IX_FP8_B128 && c.format != V4A_IX_FP4_B32) return false;
  if (a->q_format != V4A_Q_FP8_HEAD || a->num_heads != 64 || c.dim != 128) return false;
  // the fp4 tensor map wants a 32-byte aligned pool (block sizes are multiples of 32)
  if ((reinterpret_cast<uintptr_t>(c.pool) & 31) || (reinterpret_cast<uintptr_t>(a->q) & 15)) return false;
  if (c.num_blocks > INT32_MAX) return false;
  const size_t smem = 1024 + size_t(kStages) * kStageBytes + 2 * kQBytes + kHistBins * 4 + sizeof(Smem);
  return smem <= 227 * 1024;
}

bool index_score_tc(const v4a_index_args* a, float* scores, int64_t row, uint32_t* hist, cudaStream_t stream,
                    int* rc) {
  *rc = V4A_OK;
  if (!index_score_tc_supported(a)) return false;
  const v4a_cache& c = a->keys;
  const bool fp4 = c.format == V4A_IX_FP4_B32;
  TcArgs t{};
  t.T = a->batch.num_tokens;
  t.fmt = c.format;
  t.acc_cols = fp4 ? 256 : 64;
  t.seq_ids = a->batch.seq_ids;
  t.positions = a->batch.positions;
  t.bt = c.block_table;
  t.max_blocks = c.max_blocks;
  t.num_blocks = c.num_blocks;
  t.pool = static_cast<const uint8_t*>(c.pool);
  t.block_bytes = ix_block_bytes(c.format, c.dim);
  t.scale_off = 64 * ix_row_bytes(c.format, c.dim);
  t.scale_bytes = uint32_t(64 * 4 * ix_scales_per_row(c.format, c.dim));
  t.box_tx = uint32_t(64 * ix_row_bytes(c.format, c.dim));
  t.q = static_cast<const uint8_t*>(a->q);
  t.qs = a->q_scale;
  t.w = a->weights;
  t.scores = scores;
  t.row = row;
  t.hist = hist;
  t.status = a->status;
  t.idesc = tc::make_idesc(fp4 ? 5u : 0u, 0u, 128, 64);
  // The pool's codes as a 3-D tensor {128 elements, 64 rows, num_blocks}; one
  // box is one block's 64 rows, written as 128-byte swizzled K-major rows
  // (fp4: the 16U4_ALIGN16B type pads each 16 codes to 16 bytes on the way in).
  CUtensorMap kmap;
  {
    auto encode = tc::encode_fn();
    if (!encode) { *rc = V4A_ERR_CUDA; return true; }
    const cuuint64_t gdim[3] = {128, 64, cuuint64_t(c.num_blocks)};
    const cuuint64_t gstride[2] = {cuuint64_t(ix_row_bytes(c.format, c.dim)), cuuint64_t(t.block_bytes)};
    const cuuint32_t box[3] = {128, 64, 1};
    const cuuint32_t es[3] = {1, 1, 1};
    const CUtensorMapDataType dt = fp4 ? CU_TENSOR_MAP_DATA_TYPE_16U4_ALIGN16B : CU_TENSOR_MAP_DATA_TYPE_UINT8;
    if (encode(&kmap, dt, 3, const_cast<void*>(c.pool), gdim, gstride, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
               CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS) {
      *rc = V4A_ERR_CUDA;
      return true;
    }
  }
  const size_t smem = 1024 + size_t(kStages) * kStageBytes + 2 * kQBytes + kHistBins * 4 + sizeof(Smem);
  static std::once_flag attr_once;
  std::call_once(attr_once, [] {
    cudaFuncSetAttribute(index_scan_tc, cudaFuncAttributeMaxDynamicSharedMemorySize, 227 * 1024);
  });
  index_scan_tc<<<tc::sm_count(), kThreads, smem, stream>>>(t, kmap);
  if (cudaGetLastError() != cudaSuccess) { *rc = V4A_ERR_CUDA; return true; }
  return true;
}

}  // namespace v4a
