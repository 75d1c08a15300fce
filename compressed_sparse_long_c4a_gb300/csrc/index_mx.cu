// Indexer scan for fp4 keys with power-of-two (MX) block scales, on the
// 5th-generation tensor cores with the block-scaled MMA
// (tcgen05.mma kind::mxf8f6f4.block_scale).
//
// Method: "DeepSeek V4 in vLLM: Efficient Long-context Attention", Background
// "DeepSeek Sparse Attention" (score every compressed entry, keep the top-k)
// with the fp4 indexer cache (Background: fp4 indexer cache), computed in
// native fp4 as the summary article says the indexer does ("true FP4").
//
//   score_i = sum_h w_h * ReLU(q_h . k_i),  q_h = qcode_h * qs_h (e4m3 + one
//   fp32 scale per head), k_i = kcode_i * 2^x_{i,b} per 32-element block b.
//
// Why a kernel of its own: with power-of-two block scales the keys' scales
// ride inside the MMA as UE8M0 scale factors, so one 64-column fp32
// accumulator per 128-entry tile holds q_h . k_i directly and the epilogue
// is only the ReLU and the head weights.  (General fp32 scales need one
// accumulator per scale block, scaled in the epilogue: index_tc.cu.)
//
// Data path of one 128-entry tile (two physical blocks of 64 entries):
//   copy    each 5-KB block (codes, then scale words) arrives with ONE 1-D
//           bulk copy into a staging slot.  Every staging slot has two lanes
//           of its own that issue its next tile's copies as soon as the slot
//           is free.  Measured on GB300 for random 5-KB blocks: ~6.3-6.5 TB/s
//           in-kernel when 16-24 threads each keep one or two copies in
//           flight; the copy engine's cost goes with the number of copies
//           rather than their size, so one copy per block matters (copying
//           codes and scales separately halved the rate).
//   expand  one of two expansion warpgroups turns the slot into the MMA's
//           operands: each 16 packed bytes (32 codes) become two 16-byte
//           containers of the K-major, 128-byte-swizzled A operand, codes in
//           the first half and zeros in the second (the padded layout
//           kind::mxf8f6f4 reads for e2m1), and every fp32 scale word
//           becomes its exponent byte (UE8M0); the four bytes of an entry
//           are stored as one 32-bit TMEM word with tcgen05.st, in the layout
//           of the MMA's scale-factor operand: for rows r, 32+r, 64+r, 96+r
//           the words sit in lane r of every lane quarter, columns 0..3
//           (checked against a CPU sum on GB300 before this kernel was
//           written).  Step kb of the MMA selects byte kb (scale-factor id in
//           the instruction descriptor).
//   query   64 heads x 128 e4m3 codes by one TMA copy per query (B operand)
//           with scale factors 1.0 (UE8M0 127); the per-head fp32 query scale
//           is folded into the head weight (both are positive, so it commutes
//           with the ReLU).
//   MMA     M = 128 entries, N = 64 heads, K = 128 in four K = 32 steps, into
//           one of four TMEM accumulators.  A thread that issues tcgen05.mma
//           waits ~90-100 ns per instruction whatever its size (measured on
//           GB300: four issuing warps reach four times the rate of one), so
//           four MMA warps take the tiles in turn.
// Products of e2m1 and e4m3 codes, their sums over a block and the
// power-of-two scaling are exact in fp32.
//
// Warp roles (960 threads, one CTA per SM, persistent over a contiguous share
// of the (query, tile) items).  Tile it uses staging slot it % kStg and
// operand buffer, MMA issuer, accumulator and epilogue warpgroup it % 4.
//   warp 0      TMEM allocator and MMA issuer 0.
//   warp 1      query stager (TMA copy of the codes, w_h * qs_h).
//   warp 2      copy issuers: lanes 2s, 2s+1 copy the two blocks of staging
//               slot s.
//   warps 3-10  two expansion warpgroups (tiles of parity 0 and 1).
//   warps 11-26 four epilogue warpgroups: one thread per entry (TMEM lane)
//               -> score; with a histogram requested also the top 12 key bits
//               of the score (level 1 of the long-row top-k), one
//               shared-memory atomic per distinct bin of a warp.
//   warps 27-29 MMA issuers 1-3.
// Every wait is bounded (V4A_DEV_TIMEOUT, then a clean exit), and polls with
// a non-blocking test: a thread suspended in mbarrier.try_wait was measured
// to resume up to ~0.5 us after the phase completed.

#include <mutex>

#include "index_tc.h"
#include "scan_common.cuh"
#include "tc_common.cuh"

namespace v4a {
namespace {

using scan::Cursor;
using scan::visible_of;
using scan::warp_wait;

constexpr int kBlockBytes = 64 * 64 + 64 * 16;   // one physical block: codes, then scale words
constexpr int kCodeBytes = 64 * 64;         // packed codes of one block
constexpr int kStg = 12;                    // staging slots (tiles whose copies may be in flight)
constexpr int kStgBytes = 2 * kBlockBytes;  // one tile's two blocks, as copied
constexpr int kAcc = 4;                     // operand buffers, MMA issuers, TMEM accumulators, epilogue warpgroups
constexpr int kOpBytes = 128 * 128;         // padded A operand of one tile
constexpr int kQBytes = 64 * 128;           // 64 heads x 128 e4m3 codes
constexpr int kIss = 2;                     // the copy-issuer warp
constexpr int kExp0 = 3;                    // first expansion warp (two warpgroups)
constexpr int kEpi0 = kExp0 + 8;            // first epilogue warp (four warpgroups)
constexpr int kEpiW = 4 * kAcc;             // epilogue warps
constexpr int kMma1 = kEpi0 + kEpiW;        // MMA issuers 1..3 (issuer 0 is warp 0)
constexpr int kThreads = 32 * (kMma1 + kAcc - 1);
constexpr int kHistBins = scan::kHistBins;
constexpr uint32_t kSfaCol = 256;           // + 4 * operand buffer: scale factors of the keys
constexpr uint32_t kSfbCol = 320;           // scale factors of the query (all 1.0)
constexpr uint32_t kTmemCols = 512;
constexpr int kWin = 64;                    // block-table window of each epilogue warp
static_assert(2 * kStg <= 32, "two issuing lanes per staging slot, one warp");
static_assert(kStg % 2 == 0 && kStg > kAcc, "staging slot reuse");
static_assert(kSfaCol + 4 * kAcc <= kSfbCol && kSfbCol + 4 <= kTmemCols, "TMEM columns");

struct MxArgs {
  int T;
  const int32_t* seq_ids;
  const int32_t* positions;
  const int32_t* bt;
  int max_blocks;
  int64_t num_blocks;
  const uint8_t* pool;
  const float* qs;            // [T][64]
  const float* w;             // [T][64]
  float* scores;
  int64_t row;
  uint32_t* hist;             // [T][kHistBins] or null
  int32_t* status;
  uint32_t idesc;
};

struct MxSmem {
  uint64_t full[kStg], sempty[kStg], ready[kAcc], oempty[kAcc], afull[kAcc], aempty[kAcc], qfull[2], qempty[2],
      done, hsync, hclear;
  uint32_t tmem_base;
  int abort_flag;
  int t0, j0, count;
  uint32_t part[kThreads / 32];
  int32_t etw[kEpiW][kWin];         // each epilogue warp's window (the blocks of its 32 rows)
  alignas(16) float wq[2][64];      // w_h * qs_h of the query in each query buffer (read as float4)
};

constexpr size_t kSmemBytes =
    1024 + size_t(kAcc) * kOpBytes + 2 * kQBytes + size_t(kStg) * kStgBytes + kHistBins * 4 + sizeof(MxSmem);
static_assert(kSmemBytes <= 227 * 1024, "shared memory");

__device__ __forceinline__ void tmem_st4(uint32_t taddr, const uint32_t* v) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x4.b32 [%0], {%1, %2, %3, %4};" ::"r"(taddr), "r"(v[0]), "r"(v[1]),
               "r"(v[2]), "r"(v[3])
               : "memory");
}
__device__ __forceinline__ void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }
// 32 lanes x 16 consecutive fp32 columns, not waited for: the registers are
// valid only after tmem_wait_ld16 on the same array.
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
// Waits for this thread's outstanding TMEM loads; the 16 registers of `v` are
// tied to the wait so that no use of them is scheduled before it.
__device__ __forceinline__ void tmem_wait_ld16(float* v) {
  uint32_t* r = reinterpret_cast<uint32_t*>(v);
  asm volatile("tcgen05.wait::ld.sync.aligned;\n"
               : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]), "+r"(r[6]), "+r"(r[7]),
                 "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]), "+r"(r[12]), "+r"(r[13]), "+r"(r[14]),
                 "+r"(r[15])
               :
               : "memory");
}
__device__ __forceinline__ void mma_mx(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc, uint32_t sfa,
                                       uint32_t sfb, uint32_t accumulate) {
  asm volatile(
      "{\n.reg .pred p;\nsetp.ne.b32 p, %6, 0;\n"
      "tcgen05.mma.cta_group::1.kind::mxf8f6f4.block_scale [%0], %1, %2, %3, [%4], [%5], p;\n}\n" ::"r"(d_tmem),
      "l"(a), "l"(b), "r"(idesc), "r"(sfa), "r"(sfb), "r"(accumulate)
      : "memory");
}
// UE8M0 bytes of four fp32 power-of-two scale words (their exponent fields;
// the mantissa bits, zero for a power of two, are not read).
__device__ __forceinline__ uint32_t ue8m0x4(uint4 v) {
  return ((v.x >> 23) & 0xFFu) | (((v.y >> 23) & 0xFFu) << 8) | (((v.z >> 23) & 0xFFu) << 16) |
         (((v.w >> 23) & 0xFFu) << 24);
}

// A cursor over the items of one staging slot (every kStg-th item) that
// caches its query's sequence and block count, which change only at query
// switches.
struct Ahead {
  Cursor c;
  int t = -1, b = 0, nblk = 0;
  __device__ void skip(const MxArgs& a, int n) {
    for (int i = 0; i < n && c.t < a.T; ++i) c.next(a);
  }
  // block id of block q (0, 1) of the cursor's tile, or -1 past the row
  __device__ int32_t load(const MxArgs& a, int q) {
    if (c.t != t) {
      t = c.t;
      b = a.seq_ids[t];
      nblk = (visible_of(a, t) + 63) / 64;
    }
    const int lb = 2 * c.j + q;
    return lb < nblk ? a.bt[int64_t(b) * a.max_blocks + lb] : -1;
  }
};

__global__ void __launch_bounds__(kThreads, 1)
index_scan_mx(const MxArgs a, const __grid_constant__ CUtensorMap qmap) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* ops = base;                                         // kAcc x 16 KB: the A operands
  uint8_t* qbuf = ops + size_t(kAcc) * kOpBytes;               // 2 x 8 KB: the B operands
  uint8_t* stg = qbuf + 2 * kQBytes;                           // kStg x 10 KB: blocks as copied
  uint32_t* hist_s = reinterpret_cast<uint32_t*>(stg + size_t(kStg) * kStgBytes);
  MxSmem& s = *reinterpret_cast<MxSmem*>(hist_s + kHistBins);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  volatile int* abort_flag = &s.abort_flag;
  pdl_trigger();

  if (threadIdx.x == 0) {
    for (int i = 0; i < kStg; ++i) {
      tc::mbar_init(&s.full[i], 1);          // block 0's lane: expect_tx; then the copies' bytes
      tc::mbar_init(&s.sempty[i], 4);        // the expanding warpgroup's warps
    }
    for (int i = 0; i < kAcc; ++i) {
      tc::mbar_init(&s.ready[i], 4);         // the expanding warpgroup: operand and scale factors in place
      tc::mbar_init(&s.oempty[i], 1);        // MMA commit: operand buffer free
      tc::mbar_init(&s.afull[i], 1);         // MMA commit
      tc::mbar_init(&s.aempty[i], 4);        // the owning epilogue warpgroup
    }
    for (int i = 0; i < 2; ++i) {
      tc::mbar_init(&s.qfull[i], 1);
      tc::mbar_init(&s.qempty[i], kAcc + kEpiW);   // every MMA issuer's commit + every epilogue warp
    }
    tc::mbar_init(&s.done, kAcc);
    tc::mbar_init(&s.hsync, kEpiW);
    tc::mbar_init(&s.hclear, kEpiW);
    s.abort_flag = 0;
    tc::mbar_fence_init();
  }
  if (a.hist)
    for (int i = threadIdx.x; i < kHistBins; i += blockDim.x) hist_s[i] = 0;
  __syncwarp();   // tcgen05.alloc is warp-collective
  if (warp == 0) tc::tmem_alloc(&s.tmem_base, kTmemCols);
  tc::tc_fence_before();
  scan::plan(a, s.part, &s.t0, &s.j0, &s.count);   // contains __syncthreads
  tc::tc_fence_after();
  const uint32_t tmem = s.tmem_base;
  const int count = s.count;
  if (warp >= kEpi0 && warp < kEpi0 + 4) {
    // the query's scale factors: 1.0 in every byte of every lane
    const uint32_t one[4] = {0x7F7F7F7Fu, 0x7F7F7F7Fu, 0x7F7F7F7Fu, 0x7F7F7F7Fu};
    tmem_st4(tmem + (uint32_t((warp & 3) * 32) << 16) + kSfbCol, one);
    tmem_wait_st();
  }
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  // the set-up above (inputs only) overlaps the previous kernels; the pool,
  // which they write, and the scores and histogram are touched only after
  // they have completed
  pdl_wait();

  if (warp == kIss) {
    // ------------------------------------------------------------ copy issuers
    // lane 2s + k copies block k of staging slot s's tiles (s, s + kStg, ...)
    const int sl = lane >> 1, k = lane & 1;
    const unsigned pmask = 0x3u << (lane & 30);   // the slot's two lanes
    const bool mine = sl < kStg;                  // lanes past the last slot only keep step
    // cur: the tile being issued; nxt: this slot's next tile, whose block id
    // is loaded while the current one waits (a block-table load under full
    // HBM load takes microseconds, so it must never sit between a slot's
    // release and its next copy)
    Ahead cur, nxt;
    int32_t p = -1, pn = -1;
    int it = sl;
    if (mine) {
      cur.c.init(a, s.t0, s.j0);
      cur.skip(a, sl);
      nxt = cur;
      nxt.skip(a, kStg);
      if (sl < count) p = cur.load(a, k);
      if (sl + kStg < count) pn = nxt.load(a, k);
    }
    int cur_t = -1, last = -1;                     // last: this slot's last issued tile (for the drain)
    long long wait0 = 0;
    bool waiting = false;
    // Lock-step polling: every lane of the warp runs the same loop, and each
    // slot's pair tests its slot's release without blocking (a lane suspended
    // on one barrier would hold up the other slots' lanes).
    while (true) {
      const bool active = mine && it < count;
      if (!__any_sync(0xffffffffu, active)) break;
      if (__any_sync(0xffffffffu, *abort_flag != 0)) break;
      bool go = false;
      if (active) {
        if (k == 0) go = it < kStg || tc::mbar_test(&s.sempty[sl], ((it / kStg) & 1) ^ 1);
        go = __shfl_sync(pmask, go, lane & 30);
      }
      if (go) {
        waiting = false;
        if (cur.c.t != cur_t) {
          cur_t = cur.c.t;
          if (lane == 0 && (a.positions[cur_t] + 1) / 4 > a.max_blocks * 64) report(a.status, V4A_DEV_BAD_BLOCK);
        }
        const bool v = p >= 0 && p < a.num_blocks;
        if (p != -1 && !v) report(a.status, V4A_DEV_BAD_BLOCK);
        const uint32_t nv = __popc(__ballot_sync(pmask, v) & pmask);
        if (k == 0) tc::mbar_arrive_expect_tx(&s.full[sl], nv * uint32_t(kBlockBytes));
        // the expect_tx precedes both copies of this phase
        __syncwarp(pmask);
        if (v)
          tc::bulk_load(stg + size_t(sl) * kStgBytes + k * kBlockBytes, a.pool + int64_t(p) * kBlockBytes, kBlockBytes,
                        &s.full[sl]);
        last = it;
        // advance: the next tile's id was loaded a tile ago; load the one after
        cur = nxt;
        p = pn;
        nxt.skip(a, kStg);
        if (it + 2 * kStg < count) pn = nxt.load(a, k);
        it += kStg;
      } else if (active) {
        if (!waiting) {
          waiting = true;
          wait0 = clock64();
        } else if (clock64() - wait0 > 4000000000LL) {
          report(a.status, V4A_DEV_TIMEOUT);
          *abort_flag = 1;
        }
      }
      (void)0;
    }
    // no copy into shared memory outlives the CTA: wait (bounded) for the
    // slot's last fill (after a timeout its copies may still be in flight)
    if (mine && last >= 0) {
      const long long t0 = clock64();
      while (!tc::mbar_test(&s.full[sl], uint32_t((last / kStg) & 1)) && clock64() - t0 < 2000000000LL) {}
    }
    __syncwarp();
  } else if (warp >= kExp0 && warp < kEpi0) {
    // ------------------------------------------------------------ expansion
    const int g = (warp - kExp0) >> 2;            // the tiles of parity g
    const int pt = threadIdx.x - 32 * kExp0 - 128 * g;   // 0..127
    const int quarter = warp & 3;                 // TMEM lane quarter of this warp
    for (int it = g; it < count; it += 2) {
      const int sl = it % kStg, ob = it % kAcc;
      if (!warp_wait(&s.full[sl], (it / kStg) & 1, a.status, abort_flag)) break;
      // the operand buffer is free once the MMA of tile it - kAcc has completed
      if (it >= kAcc && !warp_wait(&s.oempty[ob], ((it / kAcc) & 1) ^ 1, a.status, abort_flag)) break;
      const uint8_t* src = stg + size_t(sl) * kStgBytes;
      uint8_t* dst = ops + size_t(ob) * kOpBytes;
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        // 16 packed bytes u: block h, entry eb, 32-code chunk c16 -> two containers of row R
        const int u = pt + 128 * i, h = u >> 8, eb = (u & 255) >> 2, c16 = u & 3, R = h * 64 + eb;
        const uint4 v = *reinterpret_cast<const uint4*>(src + h * kBlockBytes + eb * 64 + c16 * 16);
        *reinterpret_cast<uint4*>(dst + R * 128 + (((2 * c16) ^ (R & 7)) << 4)) = make_uint4(v.x, v.y, 0u, 0u);
        *reinterpret_cast<uint4*>(dst + R * 128 + (((2 * c16 + 1) ^ (R & 7)) << 4)) = make_uint4(v.z, v.w, 0u, 0u);
      }
      uint32_t wv[4];
#pragma unroll
      for (int gq = 0; gq < 4; ++gq) {
        const int e = 32 * gq + lane;             // row e's words go to lane `lane` of every lane quarter
        wv[gq] = ue8m0x4(*reinterpret_cast<const uint4*>(src + (e >> 6) * kBlockBytes + kCodeBytes + (e & 63) * 16));
      }
      tmem_st4(tmem + (uint32_t(quarter * 32) << 16) + kSfaCol + 4 * ob, wv);
      tmem_wait_st();
      tc::fence_proxy_async();   // the expanded operand (generic proxy) -> the tensor core (async proxy)
      tc::tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        tc::mbar_arrive(&s.ready[ob]);
        tc::mbar_arrive(&s.sempty[sl]);
      }
    }
    __syncwarp();
  } else if (warp == 1) {
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
        while (!tc::mbar_test(&s.qfull[q & 1], uint32_t((q >> 1) & 1)) && clock64() - t0 < 2000000000LL) {}
      }
    __syncwarp();
  } else if (warp == 0 || warp >= kMma1) {
    // ------------------------------------------------------------ MMA issuers
    // every issuer follows all items (query switches: it releases the old
    // query buffer with a commit and waits for the new one) and issues the
    // MMAs of its own tiles, into its own operand buffer and accumulator
    const int mi = warp == 0 ? 0 : warp - kMma1 + 1;
    if (lane == 0) {
      Cursor c;
      c.init(a, s.t0, s.j0);
      int cur_t = -1, qi = -1;
      const uint32_t op0 = tc::smem_u32(ops), q0 = tc::smem_u32(qbuf);
      for (int it = 0; it < count; ++it) {
        if (c.t != cur_t) {
          if (qi >= 0) tc::mma_commit(&s.qempty[qi & 1]);
          cur_t = c.t;
          ++qi;
          if (!tc::mbar_wait(&s.qfull[qi & 1], (qi >> 1) & 1, a.status, abort_flag)) break;
        }
        if ((it & 3) == mi) {
          if (!tc::mbar_wait(&s.ready[mi], (it / kAcc) & 1, a.status, abort_flag)) break;
          if (!tc::mbar_wait(&s.aempty[mi], ((it / kAcc) & 1) ^ 1, a.status, abort_flag)) break;
          tc::tc_fence_after();
          const uint64_t adesc = tc::desc_sw128(op0 + mi * kOpBytes);
          const uint64_t bdesc = tc::desc_sw128(q0 + (qi & 1) * kQBytes);
#pragma unroll
          for (int kb = 0; kb < 4; ++kb)
            // K step kb: 32 bytes further along the swizzled rows; scale byte kb
            mma_mx(tmem + 64 * mi, adesc + 2 * kb, bdesc + 2 * kb, a.idesc | (uint32_t(kb) << 29) | (uint32_t(kb) << 4),
                   tmem + kSfaCol + 4 * mi, tmem + kSfbCol, kb > 0);
          tc::mma_commit(&s.oempty[mi]);
          tc::mma_commit(&s.afull[mi]);
        }
        c.next(a);
      }
      // all issued MMAs complete before TMEM is released
      tc::mma_commit(&s.done);
      const long long t0 = clock64();
      while (!tc::mbar_test(&s.done, 0) && clock64() - t0 < 2000000000LL) {}
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ epilogue
    const int g = (warp - kEpi0) >> 2;               // warpgroup: the tiles it with it % 4 = g
    const int quarter = warp & 3;
    const int row = quarter * 32 + lane;             // entry within the tile = TMEM lane
    const int et = threadIdx.x - 32 * kEpi0;         // 0 .. 32 * kEpiW - 1
    const uint32_t lane_addr = tmem + (uint32_t(quarter * 32) << 16) + 64 * g;
    bool aborted = false;
    Cursor c;
    c.init(a, s.t0, s.j0);
    int cur_t = -1, qi = -1, n = 0, b = 0, nblk = 0, wbase = 0, wend = 0;
    int32_t* etw = s.etw[warp - kEpi0];
    const int half = row >> 6;                       // which of the tile's two blocks holds this warp's rows
    uint32_t hph = 0;
    float* srow = nullptr;
    const float* wq = nullptr;
    for (int it = 0; it < count && !aborted; ++it) {
      if (c.t != cur_t) {
        if (cur_t >= 0) {
          __syncwarp();
          if (lane == 0) tc::mbar_arrive(&s.qempty[qi & 1]);   // done with the old head weights
          if (a.hist && !scan::flush_hist<kEpiW>(&s.hsync, &s.hclear, hph, hist_s,
                                                 a.hist + int64_t(cur_t) * kHistBins, et, a.status, abort_flag)) {
            aborted = true;
            break;
          }
        }
        cur_t = c.t;
        ++qi;
        n = visible_of(a, cur_t);
        b = a.seq_ids[cur_t];
        nblk = (n + 63) / 64;
        wbase = wend = 0;
        srow = a.scores + int64_t(cur_t) * a.row;
        if (!warp_wait(&s.qfull[qi & 1], (qi >> 1) & 1, a.status, abort_flag)) {
          aborted = true;
          break;
        }
        wq = s.wq[qi & 1];
      }
      if ((it & 3) == g) {
        // this row's block id, from the warp's window of the block-table row
        // (refilled with all of its loads in flight together, once per kWin blocks)
        const int lb = 2 * c.j + half;
        if (lb >= wend && lb < nblk) {
          wbase = lb;
          wend = min(nblk, wbase + kWin);
          const int32_t* rowp = a.bt + int64_t(b) * a.max_blocks + wbase;
          __syncwarp();
          for (int i = lane; i < wend - wbase; i += 32) etw[i] = rowp[i];
          __syncwarp();
        }
        const int32_t blk = lb < nblk ? etw[lb - wbase] : -1;
        if (!warp_wait(&s.afull[g], (it / kAcc) & 1, a.status, abort_flag)) {
          aborted = true;
          break;
        }
        tc::tc_fence_after();
        // four groups of 16 heads, the next group's TMEM load in flight while
        // the current one is summed (two independent FMA chains)
        float2 sum = make_float2(0.f, 0.f), sum2 = make_float2(0.f, 0.f);
        float va[16], vb[16];
        tmem_ld16_nowait(lane_addr, va);
#pragma unroll
        for (int hg = 0; hg < 4; ++hg) {
          float* v = (hg & 1) ? vb : va;
          float* nx = (hg & 1) ? va : vb;
          tmem_wait_ld16(v);
          if (hg < 3) tmem_ld16_nowait(lane_addr + 16 * (hg + 1), nx);
          if (hg == 3) {
            tc::tc_fence_before();
            __syncwarp();
            if (lane == 0) tc::mbar_arrive(&s.aempty[g]);
          }
#pragma unroll
          for (int h = 0; h < 16; h += 4) {
            const float4 w4 = *reinterpret_cast<const float4*>(wq + 16 * hg + h);
            sum = __ffma2_rn(make_float2(fmaxf(v[h], 0.f), fmaxf(v[h + 1], 0.f)), make_float2(w4.x, w4.y), sum);
            sum2 = __ffma2_rn(make_float2(fmaxf(v[h + 2], 0.f), fmaxf(v[h + 3], 0.f)), make_float2(w4.z, w4.w), sum2);
          }
        }
        const int e = c.j * 128 + row;
        const float sv = (blk >= 0 && blk < a.num_blocks) ? (sum.x + sum2.x) + (sum.y + sum2.y) : -INFINITY;
        if (e < n) srow[e] = sv;
        if (a.hist) {
          // one shared-memory atomic per distinct bin of the warp (scores crowd into few bins)
          const uint32_t bin = e < n ? float_key(sv) >> 20 : 0xFFFFFFFFu;
          const uint32_t peers = __match_any_sync(0xffffffffu, bin);
          if (bin != 0xFFFFFFFFu && lane == __ffs(peers) - 1) atomicAdd(&hist_s[bin], uint32_t(__popc(peers)));
        }
      }
      c.next(a);
    }
    // the last query's counts (a warp that gave up skips this; the others'
    // bounded waits then see the abort flag)
    if (a.hist && cur_t >= 0 && !aborted)
      scan::flush_hist<kEpiW>(&s.hsync, &s.hclear, hph, hist_s, a.hist + int64_t(cur_t) * kHistBins, et, a.status,
                              abort_flag);
    __syncwarp();
  }
  tc::tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc::tc_fence_after();
    tc::tmem_dealloc(tmem, kTmemCols);
  }
}

}  // namespace

bool index_score_mx_supported(const v4a_index_args* a) {
  const v4a_cache& c = a->keys;
  if (c.format != V4A_IX_FP4_MX32) return false;
  if (a->q_format != V4A_Q_FP8_HEAD || a->num_heads != 64 || c.dim != 128) return false;
  // 16-byte bulk copies of the blocks; 16-byte aligned query rows for the tensor map
  if ((reinterpret_cast<uintptr_t>(c.pool) & 15) || (reinterpret_cast<uintptr_t>(a->q) & 15)) return false;
  if (c.num_blocks > INT32_MAX) return false;
  if (a->batch.num_tokens > (1 << 24)) return false;   // query rows of the tensor map stay in int range
  return true;
}

bool index_score_mx(const v4a_index_args* a, float* scores, int64_t row, uint32_t* hist, cudaStream_t stream,
                    int* rc) {
  *rc = V4A_OK;
  if (!index_score_mx_supported(a)) return false;
  const v4a_cache& c = a->keys;
  MxArgs t{};
  t.T = a->batch.num_tokens;
  t.seq_ids = a->batch.seq_ids;
  t.positions = a->batch.positions;
  t.bt = c.block_table;
  t.max_blocks = c.max_blocks;
  t.num_blocks = c.num_blocks;
  t.pool = static_cast<const uint8_t*>(c.pool);
  t.qs = a->q_scale;
  t.w = a->weights;
  t.scores = scores;
  t.row = row;
  t.hist = hist;
  t.status = a->status;
  // block-scaled descriptor: A e2m1 (5), B e4m3 (0), N = 64, UE8M0 scales
  // (bit 23), M = 128; the scale-factor ids (bits 4-5 and 29-30) are set per K step
  t.idesc = (5u << 7) | (0u << 10) | ((64u >> 3) << 17) | (1u << 23) | ((128u >> 4) << 24);
  auto encode = tc::encode_fn();
  if (!encode) { *rc = V4A_ERR_CUDA; return true; }
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
  static std::once_flag attr_once;
  std::call_once(attr_once, [] {
    cudaFuncSetAttribute(index_scan_mx, cudaFuncAttributeMaxDynamicSharedMemorySize, int(kSmemBytes));
  });
  const cudaError_t e = launch_pdl(index_scan_mx, dim3(tc::sm_count()), dim3(kThreads), kSmemBytes, stream, t, qmap);
  if (e != cudaSuccess || cudaGetLastError() != cudaSuccess) { *rc = V4A_ERR_CUDA; return true; }
  return true;
}

}  // namespace v4a
