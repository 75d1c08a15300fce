// Work planning and hand-off helpers shared by the persistent indexer scans
// (index_tc.cu, index_mx.cu).  A scan's work is the flattened list of
// (query, 128-entry tile) items; every CTA takes one contiguous share of it.
#pragma once

#include "tc_common.cuh"

namespace v4a {
namespace scan {

// Visible entries of query t ((m+1)/4, the c4a causality rule), never beyond
// what its block-table row can address.  A is any argument struct with
// `positions` and `max_blocks`.
template <class A>
__device__ __forceinline__ int visible_of(const A& a, int t) {
  return min((a.positions[t] + 1) / 4, a.max_blocks * 64);
}

template <class A>
__device__ __forceinline__ int tiles_of(const A& a, int t) {
  return (visible_of(a, t) + 127) / 128;
}

// Walks the flattened (query, tile) list; the tile count of the current query
// is cached so the hot loop touches global memory only at query switches.
struct Cursor {
  int t, j, nt;
  template <class A>
  __device__ void init(const A& a, int t0, int j0) {
    t = t0; j = j0; nt = t0 < a.T ? tiles_of(a, t0) : 0;
  }
  template <class A>
  __device__ void next(const A& a) {
    if (++j >= nt) {
      j = 0;
      do { ++t; nt = t < a.T ? tiles_of(a, t) : 0; } while (t < a.T && nt == 0);
    }
  }
};

// Contiguous share of the flattened (query, tile) list for this CTA: first
// item (*t0, *j0) and item count *count.  Each thread sums the tiles of a
// contiguous chunk of queries; the chunk holding the CTA's first item is then
// walked by its owner.  `part` holds one word per warp.  Contains
// __syncthreads; every thread of the CTA calls it.
template <class A>
__device__ void plan(const A& a, uint32_t* part, int* t0, int* j0, int* count) {
  const int per = (a.T + blockDim.x - 1) / blockDim.x;
  const int c0 = threadIdx.x * per, c1 = min(a.T, c0 + per);
  uint32_t mine = 0;
  for (int t = c0; t < c1; ++t) mine += tiles_of(a, t);
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5, nw = (blockDim.x + 31) >> 5;
  uint32_t incl = mine;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t x = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += x;
  }
  if (lane == 31) part[wid] = incl;
  if (threadIdx.x == 0) { *count = 0; *t0 = a.T; *j0 = 0; }
  __syncthreads();
  uint32_t before = incl - mine, all = 0;
  for (int w = 0; w < nw; ++w) {
    const uint32_t x = part[w];
    if (w < wid) before += x;
    all += x;
  }
  const uint32_t lo = uint32_t((uint64_t(all) * blockIdx.x) / gridDim.x);
  const uint32_t hi = uint32_t((uint64_t(all) * (blockIdx.x + 1)) / gridDim.x);
  if (hi > lo && lo >= before && lo < before + mine) {
    uint32_t acc = before;
    for (int t = c0; t < c1; ++t) {
      const uint32_t n = tiles_of(a, t);
      if (lo < acc + n) { *t0 = t; *j0 = int(lo - acc); break; }
      acc += n;
    }
    *count = int(hi - lo);
  }
  __syncthreads();
}

// Lane 0 waits for the phase (bounded) and the warp proceeds together; the
// warp barrier orders the other lanes' reads after lane 0's observation.
__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, int32_t* status, volatile int* abort_flag) {
  bool ok = true;
  if ((threadIdx.x & 31) == 0) ok = tc::mbar_wait(bar, parity, status, abort_flag);
  ok = __shfl_sync(0xffffffffu, ok, 0);
  __syncwarp();
  return ok;
}

constexpr int kHistBins = 4096;   // top 12 bits of a score's order-preserving key

// Adds the shared-memory histogram of one query to its global row and clears
// it.  Called by all kWarps epilogue warps at the same item; they meet on two
// mbarriers (bounded waits, so a warp that gave up elsewhere cannot hang the
// others): every add of the old query is done before any bin is read, and
// every bin is cleared before any add of the next query.  `et` is the
// thread's index within the epilogue warps.
template <int kWarps>
__device__ __forceinline__ bool flush_hist(uint64_t* hsync, uint64_t* hclear, uint32_t& hph, uint32_t* h_s,
                                           uint32_t* g, int et, int32_t* status, volatile int* abort_flag) {
  const int lane = threadIdx.x & 31;
  __syncwarp();
  if (lane == 0) tc::mbar_arrive(hsync);
  bool ok = __all_sync(0xffffffffu, tc::mbar_wait(hsync, hph, status, abort_flag));
  if (ok) {
    for (int i = et; i < kHistBins; i += 32 * kWarps) {
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

}  // namespace scan
}  // namespace v4a
