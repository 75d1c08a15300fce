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
//  The codes of each physical block arrive with ONE TMA tensor copy through a
//  3-D map over the pool ({128 elements, 64 rows, block}) that writes the
//  K-major, 128-byte-swizzled A operand itself (fp4: the 16U4_ALIGN16B type
//  expands each 16 codes to a 16-byte container, the layout kind::f8f6f4
//  reads for e2m1; fp8: plain swizzled rows).  The copy engine spends a
//  roughly fixed time on every copy (about 0.1 us on GB300, measured), so one
//  copy per block, issued by two producer warps, is what keeps HBM busy; the
//  scale words (1 KB or 256 B per block) travel on the load/store path
//  instead: each epilogue thread copies its own entry's words into shared
//  memory with cp.async a few tiles ahead of their use.
//  B = the query's e4m3 codes, N = 64 heads, staged once per query by a TMA
//  tensor copy (which writes the swizzled operand itself);
//  K = 128 in four MMAs of K = 32.  fp8 keys: the four MMAs accumulate into
//      one 64-column fp32 accumulator (one scale per entry, factored out of
//      the ReLU since scales are positive).  fp4 keys: each MMA writes its own
//      accumulator (one per 32-element scale block), combined in the epilogue
//      as sum_b s_b * acc_b before the ReLU.
// Products of e4m3 x e4m3 / e2m1 codes and their sums are exact or nearly so
// in the fp32 accumulator; the fp32 scales are applied in the epilogue.
//
// Warp roles (384 threads, one CTA per SM, persistent over a contiguous range
// of (query, tile) work items):
//   warp 0      TMEM allocator and single-thread MMA issuer (double-buffered
//               TMEM accumulators); a stage is released by the MMA's commit.
//   warps 1, 2  producers, alternating tiles: lanes 0 and 1 issue the two
//               block copies of a tile in one instruction (block ids from a
//               shared-memory window of the block table) and hand the ids to
//               the epilogue through a ring.
//   warp 3      query stager: TMA copy of each query's codes, w_h * qs_h,
//               double-buffered.
//   warps 4..11 two epilogue warpgroups, one per accumulator (alternate
//               tiles): one thread per entry (TMEM lane) reads its
//               accumulators and applies scales, ReLU and head weights with
//               packed fp32x2 FMAs, releasing the accumulator as soon as its
//               last TMEM load has landed.  With a histogram requested it also
//               counts the top 12 bits of the score's order-preserving key in
//               shared memory (flushed to the query's global histogram at
//               every query switch), the first level of the long-row top-k.
//               Lane 0 of each warp does the warp's barrier waits: a wait by
//               all 32 lanes of a warp costs several times more.
// Every mbarrier wait is bounded (V4A_DEV_TIMEOUT, then a clean exit).

#include <mutex>

#include "index_tc.h"
#include "scan_common.cuh"
#include "tc_common.cuh"

namespace v4a {
namespace {

constexpr int kMaxStages = 16;
constexpr int kBoxBytes = 64 * 128;          // one block's codes as 64 operand rows
constexpr int kStageBytes = 2 * kBoxBytes;   // one MMA A operand: 128 rows x 128 smem bytes
constexpr int kRing = 32;                    // per-tile block ids handed to the epilogue
constexpr int kQBytes = 64 * 128;            // 64 heads x 128 codes
constexpr int kHistBins = scan::kHistBins;
constexpr int kProd = 2;                     // producer warps (alternate tiles)
constexpr int kQw = 1 + kProd;               // query-stager warp
constexpr int kEpi0 = kQw + 1;               // first epilogue warp
constexpr int kEpiWarps = 8;                 // two epilogue warpgroups
constexpr int kThreads = 32 * (kEpi0 + kEpiWarps);
constexpr int kWin = 512;                    // block-table window of each producer
constexpr int kScLead = 3;                   // own tiles an epilogue thread copies its scale words ahead
constexpr int kScSlots = kScLead + 1;        // scale-word slots of each epilogue warpgroup
constexpr int kScSlot = 128 * 16;            // one tile's scale words (fp4: 16 B per entry; fp8: 4 B)

struct TcArgs {
  int T, fmt, acc_cols, stages;
  const int32_t* seq_ids;
  const int32_t* positions;
  const int32_t* bt;
  int max_blocks;
  int64_t num_blocks;
  const uint8_t* pool;
  int64_t block_bytes;
  int64_t scale_off;          // byte offset of the scale words inside a block
  uint32_t box_tx;            // transaction bytes of one code box (the packed bytes read: 4096 / 8192)
  const float* qs;            // [T][64]
  const float* w;             // [T][64]
  float* scores;
  int64_t row;
  uint32_t* hist;             // [T][kHistBins] or null
  int32_t* status;
  uint32_t idesc;
};

struct Smem {
  uint64_t full[kMaxStages], empty[kMaxStages], rfull[kRing], tfull[2], tempty[2], qfull[2], qempty[2], done,
      hsync, hclear;
  uint32_t tmem_base;
  int abort_flag;
  int t0, j0, count;
  int32_t rblk[kRing][2];           // physical blocks of each tile (-1: not loaded), for the scale words
  int32_t btc[kProd][kWin];         // each producer's window of the current query's block-table row
  uint32_t part[kThreads];
  float wq[2][64];                  // w_h * qs_h of the query in each query buffer
};

constexpr size_t kFixedSmem = 1024 + 2 * kQBytes + 2 * kScSlots * kScSlot + kHistBins * 4 + sizeof(Smem);

using scan::Cursor;
using scan::visible_of;
using scan::warp_wait;

// Layout constants of one key format (64 heads x 128 dims; 64 entries per block).
template <bool FP8>
struct Fmt {
  static constexpr int kRowBytes = FP8 ? 128 : 64;                 // codes of one entry
  static constexpr int kScaleOff = 64 * kRowBytes;                 // scale words after the 64 rows
  static constexpr int kScaleBytes = FP8 ? 4 : 16;                 // scale bytes of one entry
  static constexpr int kBlockBytes = kScaleOff + 64 * kScaleBytes; // 8448 / 5120
  static constexpr int kAccCols = FP8 ? 64 : 256;                  // fp32 columns of one accumulator
};

template <bool FP8>
__global__ void __launch_bounds__(kThreads, 1)
index_scan_tc(const TcArgs a, const __grid_constant__ CUtensorMap kmap, const __grid_constant__ CUtensorMap qmap) {
  using F = Fmt<FP8>;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* stages = base;                                   // stages x 16 KB: the MMA A operands
  uint8_t* qbuf = stages + size_t(a.stages) * kStageBytes;  // 2 x 8 KB
  uint8_t* scale_s = qbuf + 2 * kQBytes;                    // 2 x kScSlots x 2 KB: epilogue scale words
  uint32_t* hist_s = reinterpret_cast<uint32_t*>(scale_s + 2 * kScSlots * kScSlot);
  Smem& s = *reinterpret_cast<Smem*>(hist_s + kHistBins);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int S = a.stages;
  volatile int* abort_flag = &s.abort_flag;
  pdl_trigger();

  if (threadIdx.x == 0) {
    for (int i = 0; i < S; ++i) {
      tc::mbar_init(&s.full[i], 1);
      tc::mbar_init(&s.empty[i], 1);                // MMA commit
    }
    for (int i = 0; i < kRing; ++i) tc::mbar_init(&s.rfull[i], 1);   // producer
    for (int i = 0; i < 2; ++i) {
      tc::mbar_init(&s.tfull[i], 1);
      tc::mbar_init(&s.tempty[i], 4);   // the owning warpgroup's warps
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
  if (warp == 0) tc::tmem_alloc(&s.tmem_base, 2 * F::kAccCols);
  tc::tc_fence_before();
  scan::plan(a, s.part, &s.t0, &s.j0, &s.count);   // contains __syncthreads
  // the set-up above (inputs only) overlaps the previous kernels; the pool,
  // which they write, and the histogram, which they clear, are touched only
  // after they have completed
  pdl_wait();
  tc::tc_fence_after();
  const uint32_t tmem = s.tmem_base;
  const int count = s.count;

  if (warp >= 1 && warp <= kProd) {
    // ------------------------------------------------------------ producers
    const int pr = warp - 1;
    int32_t* btc = s.btc[pr];
    if (lane == 0) tc::prefetch_tmap(&kmap);
    Cursor c;
    c.init(a, s.t0, s.j0);
    int cur_t = -1, stage = 0;
    uint32_t phase = 0;
    int last_par[kMaxStages];              // parity of this producer's last fill of each stage, -1 if none
#pragma unroll
    for (int i = 0; i < kMaxStages; ++i) last_par[i] = -1;
    int b = 0, nblk = 0, btc_base = 0, btc_end = 0;
    for (int it = 0; it < count; ++it) {
      if (c.t != cur_t) {
        cur_t = c.t;
        b = a.seq_ids[cur_t];
        nblk = (visible_of(a, cur_t) + 63) / 64;
        btc_base = btc_end = 0;                       // refill the block-table window below
        if (pr == 0 && lane == 0 && (a.positions[cur_t] + 1) / 4 > a.max_blocks * 64)
          report(a.status, V4A_DEV_BAD_BLOCK);
      }
      if ((it % kProd) == pr) {
        // block-table entries come from a shared-memory window of the row,
        // refilled by the whole warp with all of its loads in flight together
        if (2 * c.j + 1 >= btc_end && 2 * c.j < nblk) {
          btc_base = 2 * c.j;
          btc_end = min(nblk, btc_base + kWin);
          const int n = btc_end - btc_base;
          const int32_t* row = a.bt + int64_t(b) * a.max_blocks + btc_base;
          __syncwarp();
          for (int i0 = 0; i0 < n; i0 += 32 * 8) {
            int32_t v[8];
#pragma unroll
            for (int u = 0; u < 8; ++u) {
              const int i = i0 + u * 32 + lane;
              v[u] = i < n ? row[i] : 0;
            }
#pragma unroll
            for (int u = 0; u < 8; ++u) {
              const int i = i0 + u * 32 + lane;
              if (i < n) btc[i] = v[u];
            }
          }
          __syncwarp();
        }
        bool ok = true;
        if (lane == 0) ok = tc::mbar_wait(&s.empty[stage], phase ^ 1, a.status, abort_flag);
        if (!__shfl_sync(0xffffffffu, ok, 0)) break;
        // lane h < 2 issues block h's copy; both copies leave in one instruction
        int32_t p = -1;
        if (lane < 2) {
          const int lb = 2 * c.j + lane;
          if (lb < nblk) {
            p = btc[lb - btc_base];
            if (p < 0 || p >= a.num_blocks) { p = -1; report(a.status, V4A_DEV_BAD_BLOCK); }
          }
          s.rblk[it % kRing][lane] = p;
        }
        const uint32_t valid = __ballot_sync(0xffffffffu, p >= 0) & 3u;
        if (lane == 0) {
          tc::mbar_arrive_expect_tx(&s.full[stage], uint32_t(__popc(valid)) * a.box_tx);
          last_par[stage] = int(phase);
        }
        __syncwarp();
        if (p >= 0) tc::tma_load_3d(stages + stage * kStageBytes + lane * kBoxBytes, &kmap, 0, 0, p, &s.full[stage]);
        if (lane == 0) tc::mbar_arrive(&s.rfull[it % kRing]);   // block ids for the epilogue
      }
      if (++stage == S) { stage = 0; phase ^= 1; }
      c.next(a);
    }
    // drain: every copy this producer issued has landed before the CTA can
    // exit (each stage belongs to one producer, so its last fill is the
    // barrier's latest phase)
    if (lane == 0) {
      for (int i = 0; i < S; ++i) {
        if (last_par[i] < 0) continue;
        const long long t0 = clock64();
        while (!tc::mbar_try_wait(&s.full[i], uint32_t(last_par[i])) && clock64() - t0 < 2000000000LL) {}
      }
    }
    __syncwarp();
  } else if (warp == kQw) {
    // ------------------------------------------------------------ query stager
    if (lane == 0) tc::prefetch_tmap(&qmap);
    Cursor c;
    c.init(a, s.t0, s.j0);
    int cur_t = -1, qi = -1;
    for (int it = 0; it < count; ++it) {
      if (c.t != cur_t) {
        cur_t = c.t;
        ++qi;
        const int qb = qi & 1;
        bool ok = true;
        if (lane == 0 && qi >= 2) ok = tc::mbar_wait(&s.qempty[qb], ((qi >> 1) - 1) & 1, a.status, abort_flag);
        if (!__shfl_sync(0xffffffffu, ok, 0)) { --qi; break; }
        for (int h = lane; h < 64; h += 32)
          s.wq[qb][h] = a.w[int64_t(cur_t) * 64 + h] * a.qs[int64_t(cur_t) * 64 + h];
        __syncwarp();
        if (lane == 0) {
          tc::mbar_arrive_expect_tx(&s.qfull[qb], uint32_t(kQBytes));
          tc::tma_load_2d(qbuf + qb * kQBytes, &qmap, 0, cur_t * 64, &s.qfull[qb]);
        }
      }
      c.next(a);
    }
    // the last copy into each query buffer has landed before the CTA can exit
    if (lane == 0)
      for (int q = qi; q >= 0 && q > qi - 2; --q) {
        const long long t0 = clock64();
        while (!tc::mbar_try_wait(&s.qfull[q & 1], uint32_t((q >> 1) & 1)) && clock64() - t0 < 2000000000LL) {}
      }
    __syncwarp();
  } else if (warp == 0) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      Cursor c;
      c.init(a, s.t0, s.j0);
      int cur_t = -1, qi = -1, acc = 0, stage = 0;
      uint32_t phase = 0, aphase = 0;
      const uint32_t q0 = tc::smem_u32(qbuf), st0 = tc::smem_u32(stages);
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
        const uint64_t adesc = tc::desc_sw128(st0 + stage * kStageBytes);
        const uint64_t bdesc = tc::desc_sw128(q0 + (qi & 1) * kQBytes);
        const uint32_t d = tmem + acc * F::kAccCols;
#pragma unroll
        for (int kb = 0; kb < 4; ++kb) {
          // advance 32 bytes of K inside the swizzled 128-byte rows
          if (FP8)
            tc::mma_f8f6f4(d, adesc + 2 * kb, bdesc + 2 * kb, a.idesc, kb > 0);
          else
            tc::mma_f8f6f4(d + 64 * kb, adesc + 2 * kb, bdesc + 2 * kb, a.idesc, 0);
        }
        tc::mma_commit(&s.empty[stage]);
        tc::mma_commit(&s.tfull[acc]);
        if (++acc == 2) { acc = 0; aphase ^= 1; }
        if (++stage == S) { stage = 0; phase ^= 1; }
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
    // Warpgroup g (warps 4+4g .. 7+4g) owns accumulator g, i.e. every other
    // tile; both warpgroups walk every item to follow the query switches.
    const int g = (warp - kEpi0) >> 2;
    const int quarter = warp & 3;                // TMEM lanes 32*quarter .. +31
    const int row = quarter * 32 + lane;         // entry within the tile
    const int et = threadIdx.x - 32 * kEpi0;     // 0 .. 255
    const uint32_t lane_addr = tmem + (uint32_t(quarter * 32) << 16) + g * F::kAccCols;
    Cursor c;
    c.init(a, s.t0, s.j0);
    int cur_t = -1, qi = -1, n = 0;
    uint32_t aphase = 0, hph = 0;
    float* srow = nullptr;
    const float* wq = nullptr;
    bool aborted = false;
    // Scale words: each thread copies its own entry's words for the tile
    // kScLead own tiles ahead into its warpgroup's ring with cp.async; one
    // commit group per own tile, so waiting until kScLead groups remain
    // pending means this tile's words have landed (no barrier needed: every
    // thread reads only what it copied itself).
    uint8_t* my_ring = scale_s + g * kScSlots * kScSlot;
    auto issue_scales = [&](int o) -> bool {   // own tile o = item 2o + g
      const int itn = 2 * o + g;
      if (itn < count) {
        if (!warp_wait(&s.rfull[itn % kRing], (itn / kRing) & 1, a.status, abort_flag)) return false;
        const int32_t b = s.rblk[itn % kRing][row >> 6];
        if (b >= 0) {
          uint8_t* dst = my_ring + (o % kScSlots) * kScSlot + row * F::kScaleBytes;
          const uint8_t* src = a.pool + int64_t(b) * F::kBlockBytes + F::kScaleOff + (row & 63) * F::kScaleBytes;
          if (FP8)
            tc::cp_async4(dst, src);
          else
            tc::cp_async16(dst, src);
        }
      }
      tc::cp_async_commit();
      return true;
    };
    for (int o = 0; o < kScLead && !aborted; ++o)
      if (!issue_scales(o)) aborted = true;
    for (int it = 0; it < count && !aborted; ++it) {
      if (c.t != cur_t) {
        if (cur_t >= 0) {
          __syncwarp();
          if (lane == 0) tc::mbar_arrive(&s.qempty[qi & 1]);   // done with the old head weights
          if (a.hist && !scan::flush_hist<kEpiWarps>(&s.hsync, &s.hclear, hph, hist_s, a.hist + int64_t(cur_t) * kHistBins, et,
                                    a.status, abort_flag)) {
            aborted = true;
            break;
          }
        }
        cur_t = c.t;
        ++qi;
        n = visible_of(a, cur_t);
        srow = a.scores + int64_t(cur_t) * a.row;
        if (!warp_wait(&s.qfull[qi & 1], (qi >> 1) & 1, a.status, abort_flag)) {
          aborted = true;
          break;
        }
        wq = s.wq[qi & 1];
      }
      if ((it & 1) == g) {
        const int e = c.j * 128 + row;
        const int o = it >> 1;
        if (!issue_scales(o + kScLead)) { aborted = true; break; }
        tc::cp_async_wait_group<kScLead>();
        // the block id was seen when this tile's copy was issued; the ring
        // slot is rewritten only kRing items later
        const int32_t blk = s.rblk[it % kRing][row >> 6];
        const uint8_t* slot = my_ring + (o % kScSlots) * kScSlot;
        float4 scv;
        if (FP8)
          scv = make_float4(reinterpret_cast<const float*>(slot)[row], 0.f, 0.f, 0.f);
        else
          scv = reinterpret_cast<const float4*>(slot)[row];
        if (!warp_wait(&s.tfull[g], aphase, a.status, abort_flag)) {
          aborted = true;
          break;
        }
        tc::tc_fence_after();
        float score;
        if (FP8) {
          float v[64];
          tc::tmem_ld64(lane_addr, v);
          tc::tc_fence_before();
          __syncwarp();
          if (lane == 0) tc::mbar_arrive(&s.tempty[g]);
          float2 sum = make_float2(0.f, 0.f), sum2 = make_float2(0.f, 0.f);
#pragma unroll
          for (int h = 0; h < 64; h += 4) {
            const float2 r = make_float2(fmaxf(v[h], 0.f), fmaxf(v[h + 1], 0.f));
            const float2 r2 = make_float2(fmaxf(v[h + 2], 0.f), fmaxf(v[h + 3], 0.f));
            sum = __ffma2_rn(r, make_float2(wq[h], wq[h + 1]), sum);
            sum2 = __ffma2_rn(r2, make_float2(wq[h + 2], wq[h + 3]), sum2);
          }
          score = ((sum.x + sum2.x) + (sum.y + sum2.y)) * scv.x;
        } else {
          // 16 heads per round (their 4 block accumulators = 64 columns); the
          // next round's TMEM loads are in flight while this round is summed,
          // and the accumulator is released as soon as the last round landed.
          // Two independent partial sums keep the FMA chains short.
          float2 sum = make_float2(0.f, 0.f), sum2 = make_float2(0.f, 0.f);
          const float2 s0 = make_float2(scv.x, scv.x), s1 = make_float2(scv.y, scv.y);
          const float2 s2 = make_float2(scv.z, scv.z), s3 = make_float2(scv.w, scv.w);
          float va[64], vb[64];
          tc::tmem_ld4x16_nowait(lane_addr, 64, va);
          tc::tmem_wait_ld(va);
#pragma unroll
          for (int hg = 0; hg < 4; ++hg) {
            float* v = (hg & 1) ? vb : va;
            float* nx = (hg & 1) ? va : vb;
            if (hg < 3) tc::tmem_ld4x16_nowait(lane_addr + (hg + 1) * 16, 64, nx);
#pragma unroll
            for (int i = 0; i < 16; i += 2) {
              float2 d = __fmul2_rn(make_float2(v[i], v[i + 1]), s0);
              d = __ffma2_rn(make_float2(v[16 + i], v[17 + i]), s1, d);
              d = __ffma2_rn(make_float2(v[32 + i], v[33 + i]), s2, d);
              d = __ffma2_rn(make_float2(v[48 + i], v[49 + i]), s3, d);
              d.x = fmaxf(d.x, 0.f);
              d.y = fmaxf(d.y, 0.f);
              if ((i & 2) == 0)
                sum = __ffma2_rn(d, make_float2(wq[hg * 16 + i], wq[hg * 16 + i + 1]), sum);
              else
                sum2 = __ffma2_rn(d, make_float2(wq[hg * 16 + i], wq[hg * 16 + i + 1]), sum2);
            }
            if (hg < 3) tc::tmem_wait_ld(nx);
            if (hg == 2) {
              tc::tc_fence_before();
              __syncwarp();
              if (lane == 0) tc::mbar_arrive(&s.tempty[g]);
            }
          }
          score = (sum.x + sum2.x) + (sum.y + sum2.y);
        }
        if (e < n) {
          const float sv = blk >= 0 ? score : -INFINITY;
          srow[e] = sv;
          if (a.hist) atomicAdd(&hist_s[float_key(sv) >> 20], 1u);
        }
        aphase ^= 1;
      }
      c.next(a);
    }
    // the last query's counts (a warp that gave up skips this; the others'
    // bounded waits then see the abort flag)
    if (a.hist && cur_t >= 0 && !aborted)
      scan::flush_hist<kEpiWarps>(&s.hsync, &s.hclear, hph, hist_s, a.hist + int64_t(cur_t) * kHistBins, et, a.status, abort_flag);
    tc::cp_async_wait_all();   // no copy into shared memory outlives the CTA
    __syncwarp();
  }
  tc::tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc::tc_fence_after();
    tc::tmem_dealloc(tmem, 2 * F::kAccCols);
  }
}

// ---- host side -------------------------------------------------------------------

// Operand stages that fit next to the fixed part of shared memory, an even
// number so that each stage always belongs to the same producer.
int stages_count() {
  const int64_t room = int64_t(227 * 1024) - int64_t(kFixedSmem);
  int n = int(room / kStageBytes);
  if (n > kMaxStages) n = kMaxStages;
  return n & ~1;
}

}  // namespace

bool index_score_tc_supported(const v4a_index_args* a) {
  const v4a_cache& c = a->keys;
  // power-of-two (MX) scales are a special case of the fp32 scales
  if (c.format != V4A_IX_FP8_B128 && !ix_is_fp4(c.format)) return false;
  if (a->q_format != V4A_Q_FP8_HEAD || a->num_heads != 64 || c.dim != 128) return false;
  // the fp4 tensor map wants a 32-byte aligned pool (block sizes are multiples of 32)
  if ((reinterpret_cast<uintptr_t>(c.pool) & 31) || (reinterpret_cast<uintptr_t>(a->q) & 15)) return false;
  if (c.num_blocks > INT32_MAX) return false;
  if (a->batch.num_tokens > (1 << 24)) return false;   // query rows of the tensor map stay in int range
  // an epilogue thread waits for the producer to issue the tile 2 * kScLead
  // items ahead, which needs the stages to hold more than that many tiles
  return stages_count() >= 2 * kScLead + 2;
}

bool index_score_tc(const v4a_index_args* a, float* scores, int64_t row, uint32_t* hist, cudaStream_t stream,
                    int* rc) {
  *rc = V4A_OK;
  if (!index_score_tc_supported(a)) return false;
  const v4a_cache& c = a->keys;
  const bool fp4 = ix_is_fp4(c.format);
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
  t.box_tx = uint32_t(64 * ix_row_bytes(c.format, c.dim));
  t.stages = stages_count();
  t.qs = a->q_scale;
  t.w = a->weights;
  t.scores = scores;
  t.row = row;
  t.hist = hist;
  t.status = a->status;
  t.idesc = tc::make_idesc(fp4 ? 5u : 0u, 0u, 128, 64);
  auto encode = tc::encode_fn();
  if (!encode) { *rc = V4A_ERR_CUDA; return true; }
  // The pool's codes as a 3-D tensor {128 elements, 64 rows, num_blocks}; one
  // box is one block's 64 rows, written as 128-byte swizzled K-major rows
  // (fp4: the 16U4_ALIGN16B type pads each 16 codes to 16 bytes on the way in).
  CUtensorMap kmap;
  {
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
  // the query codes as a 2-D tensor [T*64 rows][128 B]: one box = one query's
  // 64 heads, written as the 128-byte swizzled K-major B operand
  CUtensorMap qmap;
  {
    const cuuint64_t gdim[2] = {128, cuuint64_t(t.T) * 64};
    const cuuint64_t gstride[1] = {128};
    const cuuint32_t box[2] = {128, 64};
    const cuuint32_t es[2] = {1, 1};
    if (encode(&qmap, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(a->q), gdim, gstride, box, es,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS) {
      *rc = V4A_ERR_CUDA;
      return true;
    }
  }
  const size_t smem = kFixedSmem + size_t(t.stages) * kStageBytes;
  static std::once_flag attr_once;
  std::call_once(attr_once, [] {
    cudaFuncSetAttribute(index_scan_tc<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, 227 * 1024);
    cudaFuncSetAttribute(index_scan_tc<false>, cudaFuncAttributeMaxDynamicSharedMemorySize, 227 * 1024);
  });
  const cudaError_t e = fp4 ? launch_pdl(index_scan_tc<false>, dim3(tc::sm_count()), dim3(kThreads), smem, stream, t,
                                          kmap, qmap)
                           : launch_pdl(index_scan_tc<true>, dim3(tc::sm_count()), dim3(kThreads), smem, stream, t,
                                        kmap, qmap);
  if (e != cudaSuccess || cudaGetLastError() != cudaSuccess) { *rc = V4A_ERR_CUDA; return true; }
  return true;
}

}  // namespace v4a
