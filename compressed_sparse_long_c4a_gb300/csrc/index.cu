// Indexer scoring and top-k selection.
//
// Method: "DeepSeek V4 in vLLM: Efficient Long-context Attention", Background
// "DeepSeek Sparse Attention" (the query attends only to the top-k compressed
// entries; a 1M-token sequence still holds ~250k c4a entries) and Appendix
// "exact values of k".  Score rule: score_i = sum_h w_h * ReLU(q_h . k_i) over
// the entries the query may see (anchor 4i+3 <= m).  Ties go to the lower
// index; the selected set is written in ascending index order, -1 padded.
//
// Kernels:
//  * index_score_simt  - CUDA-core scores for bf16 / fp8 / fp4 key caches
//                         (one CTA per (query, 64-entry physical block)).
//  * index_score_tc / index_score_mx - tcgen05 scores for fp8 / fp4 caches
//                         (index_tc.cu, index_mx.cu); both also leave the
//                         4096-bin histogram of the score keys' top 12 bits.
//  * topk_smem         - one CTA per query when the row fits in shared memory:
//                         level 1 from that histogram when there is one (only
//                         the threshold bin's entries go through the radix
//                         passes), else a radix select over the whole row of
//                         the k-th largest (score, -index) composite; then an
//                         ordered compaction.
//  * topk_hist         - the same histogram for long rows scored on the CUDA
//                         cores.
//  * topk_cluster      - long rows (up to 2^20 entries): one thread-block
//                         cluster per query finds the exact k-th largest key
//                         from three histogram levels (the cluster barrier's
//                         release / acquire orders the levels' global
//                         counts), then every CTA writes its selected indices
//                         in ascending order.

#include <cooperative_groups.h>
#include <cstdio>
#include <algorithm>
#include <mutex>

#include "v4a_common.cuh"
#include "v4a_internal.h"
#include "index_tc.h"
#include "tc_common.cuh"

namespace cg = cooperative_groups;

namespace v4a {

constexpr int kSmemTopkMax = 32768;   // rows up to this length use topk_smem
constexpr int kHistBins = 4096;       // top 12 bits of the order-preserving key
constexpr int kMaxK = 16384;
constexpr int kSlice = 8192;          // scores per CTA of the long-row top-k (8 per thread)
constexpr int kBitmapMax = 1 << 20;   // longest supported row (entries; 4M native positions)

struct IndexWs {
  float* scores;        // [T][row]
  uint32_t* hist;       // [T][kHistBins]   top 12 key bits of every score
  uint32_t* hist2;      // [T][kHistBins]   next 12 bits of the threshold bin's scores (long rows)
  uint32_t* hist3;      // [T][256]         last 8 bits of the threshold sub-bin's scores (long rows)
  uint2* gteq;          // [T][16]          each cluster CTA's entries above / equal to the exact cut
  int64_t row;
  size_t zero_bytes;    // bytes of hist, hist2 and hist3 (cleared per call)
  size_t total;
};

static int64_t round_up(int64_t v, int64_t a) { return (v + a - 1) / a * a; }

static IndexWs ws_layout(const v4a_index_args* a, void* base) {
  IndexWs w{};
  const int64_t T = a->batch.num_tokens;
  w.row = round_up(int64_t(a->keys.max_blocks) * 64, 128);
  char* p = static_cast<char*>(base);
  size_t off = 0;
  auto take = [&](size_t bytes) { char* r = p ? p + off : nullptr; off += round_up(bytes, 256); return r; };
  w.hist = reinterpret_cast<uint32_t*>(take(size_t(T) * kHistBins * 4));
  w.hist2 = reinterpret_cast<uint32_t*>(take(size_t(T) * kHistBins * 4));
  w.hist3 = reinterpret_cast<uint32_t*>(take(size_t(T) * 256 * 4));
  w.zero_bytes = off;
  w.gteq = reinterpret_cast<uint2*>(take(size_t(T) * 16 * 8));
  w.scores = reinterpret_cast<float*>(take(size_t(T) * w.row * 4));
  w.total = off;
  return w;
}

// ------------------------------------------------------------------------------
// CUDA-core scores
// ------------------------------------------------------------------------------

struct ScoreArgs {
  int T, H, dim, k_fmt, q_fmt;
  const int32_t* seq_ids;
  const int32_t* positions;
  v4a_cache keys;
  int64_t block_bytes;
  const void* q;
  const float* q_scale;
  const float* w;
  float* scores;
  int64_t row;
  int32_t* status;
};

__global__ void __launch_bounds__(256) index_score_simt(ScoreArgs a) {
  extern __shared__ float smem[];
  const int t = blockIdx.y;
  const int j = blockIdx.x;                  // logical 64-entry block
  const int m = a.positions[t];
  const int n = min((m + 1) / 4, a.keys.max_blocks * 64);
  if (j == 0 && threadIdx.x == 0 && (m + 1) / 4 > n) report(a.status, V4A_DEV_BAD_BLOCK);
  if (j * 64 >= n) return;
  const int b = a.seq_ids[t];
  const int H = a.H, D = a.dim, DP = a.dim + 1;
  float* q_s = smem;                         // [H][D+1]
  float* w_s = q_s + H * DP;                 // [H]
  float* k_s = w_s + H;                      // [64][D+1]
  for (int i = threadIdx.x; i < H * D; i += blockDim.x) {
    const int h = i / D, d = i % D;
    float v;
    if (a.q_fmt == V4A_Q_BF16) {
      v = bf16_to_f32(static_cast<const uint16_t*>(a.q)[(int64_t(t) * H + h) * D + d]);
    } else {
      v = e4m3_to_f32(static_cast<const uint8_t*>(a.q)[(int64_t(t) * H + h) * D + d]) *
          a.q_scale[int64_t(t) * H + h];
    }
    q_s[h * DP + d] = v;
  }
  for (int h = threadIdx.x; h < H; h += blockDim.x) w_s[h] = a.w[int64_t(t) * H + h];
  __shared__ int64_t blk_s;
  if (threadIdx.x == 0) blk_s = block_of(a.keys, b, j * 64, a.status);
  __syncthreads();
  const int64_t blk = blk_s;
  if (blk < 0) {
    for (int e = threadIdx.x; e < 64; e += blockDim.x)
      if (j * 64 + e < n) a.scores[int64_t(t) * a.row + j * 64 + e] = -INFINITY;
    return;
  }
  const uint8_t* base = static_cast<const uint8_t*>(a.keys.pool) + blk * a.block_bytes;
  for (int i = threadIdx.x; i < 64 * D; i += blockDim.x) {
    const int e = i / D, d = i % D;
    float v;
    if (a.k_fmt == V4A_IX_BF16) {
      v = bf16_to_f32(reinterpret_cast<const uint16_t*>(base)[i]);
    } else if (a.k_fmt == V4A_IX_FP8_B128) {
      const float* sc = reinterpret_cast<const float*>(base + 64 * D);
      v = e4m3_to_f32(base[i]) * sc[e * (D / 128) + d / 128];
    } else {
      const float* sc = reinterpret_cast<const float*>(base + 64 * (D / 2));
      const uint8_t byte = base[e * (D / 2) + d / 2];
      v = e2m1_to_f32((d & 1) ? (byte >> 4) : (byte & 15)) * sc[e * (D / 32) + d / 32];
    }
    k_s[e * DP + d] = v;
  }
  __syncthreads();
  const int e = threadIdx.x >> 2, part = threadIdx.x & 3;
  float acc = 0.f;
  for (int h = part; h < H; h += 4) {
    float dot = 0.f;
    const float* qh = q_s + h * DP;
    const float* ke = k_s + e * DP;
    for (int d = 0; d < D; ++d) dot = fmaf(qh[d], ke[d], dot);
    acc = fmaf(w_s[h], fmaxf(dot, 0.f), acc);
  }
  acc += __shfl_xor_sync(0xffffffffu, acc, 1);
  acc += __shfl_xor_sync(0xffffffffu, acc, 2);
  if (part == 0 && j * 64 + e < n) a.scores[int64_t(t) * a.row + j * 64 + e] = acc;
}

// ------------------------------------------------------------------------------
// Radix select over unique 64-bit composites (key << 32 | ~index)
// ------------------------------------------------------------------------------

__device__ __forceinline__ uint64_t composite(uint32_t key, int idx) {
  return (uint64_t(key) << 32) | uint64_t(0xFFFFFFFFu - uint32_t(idx));
}

// Returns thr such that exactly `need` (>= 1) of the n composites are >= thr.
// All threads of the CTA call it; hist = 256 words of shared memory.
// Passes before `first_pass` are skipped: the caller guarantees that all n
// composites agree on their top 8 * first_pass bits.
template <class Get>
__device__ uint64_t select_threshold(int n, int need, Get get, uint32_t* hist, uint32_t* sh,
                                     int first_pass = 0) {
  uint64_t prefix = 0, mask = 0;
  if (first_pass > 0) {
    mask = ~uint64_t(0) << (64 - 8 * first_pass);
    prefix = get(0) & mask;
  }
  for (int pass = first_pass; pass < 8; ++pass) {
    const int shift = 56 - 8 * pass;
    for (int i = threadIdx.x; i < 256; i += blockDim.x) hist[i] = 0;
    __syncthreads();
    // one shared-memory atomic per distinct digit of a warp: the keys crowd
    // into few digits in the first passes, and same-address atomics serialise
    // (a 32K-entry row took ~50 us with one atomic per entry on GB300)
    for (int base = 0; base < n; base += blockDim.x) {   // the same trip count in every lane
      const int i = base + int(threadIdx.x);
      uint32_t digit = 0xFFFFFFFFu;
      if (i < n) {
        const uint64_t c = get(i);
        if ((c & mask) == prefix) digit = uint32_t((c >> shift) & 255);
      }
      const uint32_t peers = __match_any_sync(0xffffffffu, digit);
      if (digit != 0xFFFFFFFFu && (threadIdx.x & 31) == uint32_t(__ffs(peers) - 1))
        atomicAdd(&hist[digit], uint32_t(__popc(peers)));
    }
    __syncthreads();
    if (threadIdx.x < 32) {
      // warp 0: find the digit where the running count from the top reaches need
      uint32_t loc[8], s = 0;
#pragma unroll
      for (int q = 0; q < 8; ++q) { loc[q] = hist[255 - (threadIdx.x * 8 + q)]; s += loc[q]; }
      uint32_t incl = s;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const uint32_t v = __shfl_up_sync(0xffffffffu, incl, o);
        if (threadIdx.x >= o) incl += v;
      }
      const uint32_t excl = incl - s;
      if (excl < uint32_t(need) && uint32_t(need) <= incl) {
        uint32_t acc = excl;
        int q = 0;
        for (; q < 8; ++q) {
          if (acc + loc[q] >= uint32_t(need)) break;
          acc += loc[q];
        }
        sh[0] = 255 - (threadIdx.x * 8 + q);
        sh[1] = acc;
        sh[2] = loc[q];
      }
    }
    __syncthreads();
    const int d = int(sh[0]);
    const uint32_t above = sh[1], inbin = sh[2];
    __syncthreads();
    need -= int(above);
    prefix |= uint64_t(d) << shift;
    mask |= uint64_t(255) << shift;
    if (inbin == uint32_t(need)) return prefix;
  }
  return prefix;
}

// Block-wide exclusive scan of one value per thread (blockDim <= 1024).
__device__ __forceinline__ uint32_t block_excl_scan(uint32_t v, uint32_t* scratch, uint32_t* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = (blockDim.x + 31) >> 5;
  uint32_t incl = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t x = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += x;
  }
  if (lane == 31) scratch[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    uint32_t s = lane < nw ? scratch[lane] : 0;
    uint32_t si = s;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t x = __shfl_up_sync(0xffffffffu, si, o);
      if (lane >= o) si += x;
    }
    if (lane < nw) scratch[lane] = si - s;
    if (lane == nw - 1) scratch[32] = si;
  }
  __syncthreads();
  const uint32_t r = scratch[warp] + incl - v;
  if (total) *total = scratch[32];
  __syncthreads();
  return r;
}

// Threshold bin of a 4096-bin histogram whose counts this thread holds for
// bins kHistBins-1-(4*tid+q), q < 4: the bin b with fewer than `need` counts
// strictly above it and at least `need` at or above it; *above receives the
// count strictly above.  All 1024 threads call it.
__device__ int threshold_bin4(const uint32_t (&loc)[4], uint32_t need, uint32_t* scan, int* bin_s,
                              uint32_t* above_s, uint32_t* above) {
  const uint32_t s4 = (loc[0] + loc[1]) + (loc[2] + loc[3]);
  uint32_t total;
  const uint32_t excl = block_excl_scan(s4, scan, &total);
  if (excl < need && need <= excl + s4) {
    uint32_t acc = excl;
    int q = 0;
    for (; q < 4; ++q) {
      if (acc + loc[q] >= need) break;
      acc += loc[q];
    }
    *bin_s = kHistBins - 1 - (int(threadIdx.x) * 4 + q);
    *above_s = acc;
  }
  __syncthreads();
  *above = *above_s;
  const int b = *bin_s;
  __syncthreads();
  return b;
}

__device__ void write_all_visible(int32_t* out, int n, int k) {
  for (int i = threadIdx.x; i < k; i += blockDim.x) out[i] = i < n ? i : -1;
}

// ------------------------------------------------------------------------------
// Single-CTA top-k (rows that fit in shared memory)
// ------------------------------------------------------------------------------

// hist1: the scan's histogram of the top 12 key bits of every score (or null).
// With it, level 1 comes from the histogram and only the entries of the
// threshold bin (the candidates, usually ~1% of the row) go through the
// 8-bit radix passes; every pass over the whole row costs a histogram whose
// counts crowd into a few bins.
constexpr int kCandMax = 8192;          // candidates held in shared memory (else: every entry)

__global__ void __launch_bounds__(1024) topk_smem(const float* scores, int64_t row, int max_entries,
                                                 const int32_t* positions, int k, const uint32_t* hist1,
                                                 int32_t* out) {
  extern __shared__ __align__(16) uint32_t keys_s[];   // [row] keys, then [kCandMax] candidate indices
  __shared__ uint32_t hist[256];
  __shared__ uint32_t sh[4];
  __shared__ uint32_t scan[40];
  __shared__ int bin_s;
  __shared__ uint32_t above_s, ncand_s;
  const int t = blockIdx.x;
  const int n = min((positions[t] + 1) / 4, max_entries);
  int32_t* o = out + int64_t(t) * k;
  if (n <= k) { write_all_visible(o, n, k); return; }
  const float* s = scores + int64_t(t) * row;
  // the row into shared memory, kU 16-byte loads in flight per thread (one
  // load at a time left a 32K-entry row waiting ~30 us on memory latency)
  {
    constexpr int kU = 8;
    const float4* s4 = reinterpret_cast<const float4*>(s);   // rows start on 512 bytes
    const int n4 = n >> 2;
    for (int base = 0; base < n4; base += kU * int(blockDim.x)) {
      float4 v[kU];
#pragma unroll
      for (int u = 0; u < kU; ++u) {
        const int j = base + u * int(blockDim.x) + int(threadIdx.x);
        v[u] = j < n4 ? __ldcg(s4 + j) : make_float4(0.f, 0.f, 0.f, 0.f);
      }
#pragma unroll
      for (int u = 0; u < kU; ++u) {
        const int j = base + u * int(blockDim.x) + int(threadIdx.x);
        if (j < n4)
          reinterpret_cast<uint4*>(keys_s)[j] =
              make_uint4(float_key(v[u].x), float_key(v[u].y), float_key(v[u].z), float_key(v[u].w));
      }
    }
    for (int i = 4 * n4 + int(threadIdx.x); i < n; i += blockDim.x) keys_s[i] = float_key(s[i]);
  }
  __syncthreads();
  uint64_t thr;
  bool done = false;
  if (hist1) {
    // level 1 from the scan's histogram: bin b1 holds the k-th largest key
    const uint32_t* g1 = hist1 + int64_t(t) * kHistBins;
    uint32_t loc[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) loc[q] = __ldcg(&g1[kHistBins - 1 - (int(threadIdx.x) * 4 + q)]);
    uint32_t above1;
    const uint32_t b1 = uint32_t(threshold_bin4(loc, uint32_t(k), scan, &bin_s, &above_s, &above1));
    const uint32_t in_b1 = __ldcg(&g1[b1]);
    if (in_b1 <= uint32_t(kCandMax)) {   // uniform: every thread read the same counts
      // the candidates (key in bin b1) into a list, in any order
      uint32_t* cand_s = keys_s + ((row + 3) & ~int64_t(3));
      if (threadIdx.x == 0) ncand_s = 0;
      __syncthreads();
      const int lane = threadIdx.x & 31;
      for (int base = 0; base < n; base += blockDim.x) {
        const int i = base + int(threadIdx.x);
        const bool c = i < n && (keys_s[i] >> 20) == b1;
        const uint32_t bal = __ballot_sync(0xffffffffu, c);
        uint32_t slot = 0;
        if (lane == 0 && bal) slot = atomicAdd(&ncand_s, uint32_t(__popc(bal)));
        slot = __shfl_sync(0xffffffffu, slot, 0);
        if (c) cand_s[slot + __popc(bal & ((1u << lane) - 1u))] = uint32_t(i);
      }
      __syncthreads();
      const int nc = int(ncand_s);
      // the candidates agree on their top 12 key bits, so the radix passes
      // start at the second byte of the composite
      thr = select_threshold(
          nc, int(uint32_t(k) - above1),
          [&](int j) { const uint32_t i = cand_s[j]; return composite(keys_s[i], int(i)); }, hist, sh, 1);
      done = true;
    }
  }
  if (!done)
    thr = select_threshold(n, k, [&](int i) { return composite(keys_s[i], i); }, hist, sh);
  // ordered compaction: warp w owns indices [w*per_w, (w+1)*per_w), read 32
  // consecutive keys at a time (no bank conflicts) and written in order with
  // ballots
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, nw = blockDim.x >> 5;
  const int per_w = ((n + nw - 1) / nw + 31) & ~31;
  const int wlo = min(n, warp * per_w), whi = min(n, wlo + per_w);
  uint32_t cnt = 0;
  for (int b = wlo; b < whi; b += 32) {
    const int i = b + lane;
    cnt += __popc(__ballot_sync(0xffffffffu, i < whi && composite(keys_s[i], i) >= thr));
  }
  uint32_t off = block_excl_scan(lane == 0 ? cnt : 0u, scan, nullptr);
  off = __shfl_sync(0xffffffffu, off, 0);
  const uint32_t lt = (1u << lane) - 1u;
  for (int b = wlo; b < whi; b += 32) {
    const int i = b + lane;
    const bool sel = i < whi && composite(keys_s[i], i) >= thr;
    const uint32_t bal = __ballot_sync(0xffffffffu, sel);
    if (sel) o[off + __popc(bal & lt)] = i;
    off += __popc(bal);
  }
}

// ------------------------------------------------------------------------------
// Multi-CTA top-k for long rows
// ------------------------------------------------------------------------------

__global__ void __launch_bounds__(512) topk_hist(const float* scores, int64_t row, int max_entries,
                                                const int32_t* positions, int k, int slices,
                                                uint32_t* hist) {
  __shared__ uint32_t h_s[kHistBins];
  const int t = blockIdx.y;
  const int n = min((positions[t] + 1) / 4, max_entries);
  if (n <= k) return;
  for (int i = threadIdx.x; i < kHistBins; i += blockDim.x) h_s[i] = 0;
  __syncthreads();
  const int per = (n + slices - 1) / slices;
  const int lo = blockIdx.x * per, hi = min(n, lo + per);
  const float* s = scores + int64_t(t) * row;
  const int lane = threadIdx.x & 31;
  constexpr int kU = 4;   // loads in flight per thread
  for (int base = lo; base < hi; base += kU * blockDim.x) {
    float v[kU];
#pragma unroll
    for (int u = 0; u < kU; ++u) {
      const int i = base + u * blockDim.x + threadIdx.x;
      v[u] = i < hi ? s[i] : 0.f;
    }
#pragma unroll
    for (int u = 0; u < kU; ++u) {
      const int i = base + u * blockDim.x + threadIdx.x;
      const uint32_t bin = i < hi ? (float_key(v[u]) >> 20) : 0xFFFFFFFFu;
      // one shared atomic per distinct bin of the warp (scores cluster in few bins)
      const uint32_t peers = __match_any_sync(0xffffffffu, bin);
      if (bin != 0xFFFFFFFFu && lane == __ffs(peers) - 1) atomicAdd(&h_s[bin], __popc(peers));
    }
  }
  __syncthreads();
  uint32_t* g = hist + int64_t(t) * kHistBins;
  for (int i = threadIdx.x; i < kHistBins; i += blockDim.x)
    if (h_s[i]) atomicAdd(&g[i], h_s[i]);
}

// ------------------------------------------------------------------------------
// Cluster long-row top-k
// ------------------------------------------------------------------------------
//
// One thread-block cluster per query (16 CTAs, else 8), 1024 threads per CTA,
// PER consecutive scores of the row per thread, held in registers.  The exact
// k-th largest key K* comes from three histogram levels of the
// order-preserving key: the top 12 bits (built by the scan), the next 12 bits
// and the last 8 bits of the entries in the threshold bins.  Each CTA counts
// a level in shared memory and adds its nonzero counts to the query's global
// histogram; after a cluster barrier (a hardware barrier of co-scheduled
// CTAs whose release / acquire also orders global memory: no CTA waits on a
// grid) every CTA reads the level whole.  Then every CTA learns, from the
// counts of the CTAs before it (one lane each), its share of the ties at K*
// (lowest indices first) and its output offset, and writes its selected
// indices in ascending order.  The level-1 counts are loaded together with the
// scores, and the above / equal counts share one block scan.  Three cluster barriers in all: measured on
// GB300, a cluster barrier costs ~1 us and a distributed-shared-memory read
// ~0.25 us, so the levels are combined in L2 rather than through remote
// shared memory.

// Exclusive block-wide prefix sum of two 32-bit counts packed in one 64-bit
// word (no carry crosses between them while both sums stay below 2^32).
__device__ __forceinline__ uint64_t block_excl_scan64(uint64_t v, uint64_t* scratch, uint64_t* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = (blockDim.x + 31) >> 5;
  uint64_t incl = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint64_t x = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += x;
  }
  if (lane == 31) scratch[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    const uint64_t s = lane < nw ? scratch[lane] : 0;
    uint64_t si = s;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint64_t x = __shfl_up_sync(0xffffffffu, si, o);
      if (lane >= o) si += x;
    }
    if (lane < nw) scratch[lane] = si - s;
    if (lane == nw - 1) scratch[32] = si;
  }
  __syncthreads();
  const uint64_t r = scratch[warp] + incl - v;
  *total = scratch[32];
  __syncthreads();
  return r;
}

template <int PER>
__global__ void __launch_bounds__(1024, 1) topk_cluster(const float* scores, int64_t row, int max_entries,
                                                    const int32_t* positions, int k, const uint32_t* hist1,
                                                    uint32_t* hist2, uint32_t* hist3, uint2* gteq, int32_t* out) {
  pdl_trigger();
  __shared__ uint32_t scan[40];
  __shared__ uint64_t scan64[40];
  __shared__ uint32_t h_s[kHistBins];  // this CTA's counts of the level being built
  __shared__ uint32_t pre_s[2];        // ties in and entries selected by the CTAs before this one
  __shared__ int bin_s;
  __shared__ uint32_t above_s;
  cg::cluster_group cluster = cg::this_cluster();
  const int r = int(cluster.block_rank());
  const int t = blockIdx.y;
  for (int i = threadIdx.x; i < kHistBins; i += blockDim.x) h_s[i] = 0;
  pdl_wait();   // the scores and the first-level histogram are the previous kernel's output
  const int n = min((positions[t] + 1) / 4, max_entries);
  int32_t* o = out + int64_t(t) * k;
  if (n <= k) {   // every CTA of the cluster takes this branch together
    if (r == 0) write_all_visible(o, n, k);
    return;
  }
  // the level-1 counts of this thread's four bins and its PER consecutive
  // entries, in flight together
  const uint32_t* g1 = hist1 + int64_t(t) * kHistBins;
  uint32_t loc[4];
#pragma unroll
  for (int q = 0; q < 4; ++q) loc[q] = __ldcg(&g1[kHistBins - 1 - (int(threadIdx.x) * 4 + q)]);
  const int i0 = (r * int(blockDim.x) + int(threadIdx.x)) * PER;
  const float* sc = scores + int64_t(t) * row;
  uint32_t key[PER];
  if (i0 + PER <= n) {
#pragma unroll
    for (int u = 0; u < PER; u += 4) {
      const float4 f = __ldcg(reinterpret_cast<const float4*>(sc + i0 + u));
      key[u] = float_key(f.x); key[u + 1] = float_key(f.y); key[u + 2] = float_key(f.z); key[u + 3] = float_key(f.w);
    }
  } else {
#pragma unroll
    for (int u = 0; u < PER; ++u) key[u] = i0 + u < n ? float_key(__ldcg(sc + i0 + u)) : 0u;
  }
  // level 1: the top 12 bits (histogram from the scan)
  uint32_t above1;
  const uint32_t b1 = uint32_t(threshold_bin4(loc, uint32_t(k), scan, &bin_s, &above_s, &above1));
  const uint32_t need1 = uint32_t(k) - above1;
  // level 2: the next 12 bits of the entries in bin b1; each CTA's nonzero
  // counts go to the query's global histogram, complete after the cluster
  // barrier (its release / acquire covers global memory)
#pragma unroll
  for (int u = 0; u < PER; ++u)
    if (i0 + u < n && (key[u] >> 20) == b1) atomicAdd(&h_s[(key[u] >> 8) & (kHistBins - 1)], 1u);
  __syncthreads();
  uint32_t* g2 = hist2 + int64_t(t) * kHistBins;
  for (int i = threadIdx.x; i < kHistBins; i += blockDim.x) {
    const uint32_t c = h_s[i];
    if (c) {
      atomicAdd(&g2[i], c);
      h_s[i] = 0;
    }
  }
  cluster.sync();
  uint32_t above2;
#pragma unroll
  for (int q = 0; q < 4; ++q) loc[q] = __ldcg(&g2[kHistBins - 1 - (int(threadIdx.x) * 4 + q)]);
  const uint32_t b2 = uint32_t(threshold_bin4(loc, need1, scan, &bin_s, &above_s, &above2));
  const uint32_t need2 = need1 - above2;
  // level 3: the last 8 bits of the entries in sub-bin (b1, b2)
  const uint32_t top24 = (b1 << 12) | b2;
#pragma unroll
  for (int u = 0; u < PER; ++u)
    if (i0 + u < n && (key[u] >> 8) == top24) atomicAdd(&h_s[key[u] & 255u], 1u);
  __syncthreads();
  uint32_t* g3 = hist3 + int64_t(t) * 256;
  if (threadIdx.x < 256 && h_s[threadIdx.x]) atomicAdd(&g3[threadIdx.x], h_s[threadIdx.x]);
  cluster.sync();
  if (threadIdx.x < 32) {
    const int lane = threadIdx.x;
    uint32_t loc[8], s8 = 0;
#pragma unroll
    for (int q = 0; q < 8; ++q) { loc[q] = __ldcg(&g3[255 - (lane * 8 + q)]); s8 += loc[q]; }
    uint32_t incl = s8;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const uint32_t x = __shfl_up_sync(0xffffffffu, incl, off);
      if (lane >= off) incl += x;
    }
    const uint32_t excl = incl - s8;
    if (excl < need2 && need2 <= incl) {
      uint32_t acc = excl;
      int q = 0;
      for (; q < 8; ++q) {
        if (acc + loc[q] >= need2) break;
        acc += loc[q];
      }
      bin_s = 255 - (lane * 8 + q);
      above_s = acc;
    }
  }
  __syncthreads();
  const uint32_t K = (top24 << 8) | uint32_t(bin_s);   // exact key of the k-th largest
  const uint32_t need = need2 - above_s;               // entries equal to K to take (>= 1)
  // this thread's entries above K and equal to K
  uint32_t gt = 0, eq = 0;
#pragma unroll
  for (int u = 0; u < PER; ++u) {
    const bool in = i0 + u < n;
    gt += in && key[u] > K;
    eq += in && key[u] == K;
  }
  uint64_t tot64;
  const uint64_t pre64 = block_excl_scan64((uint64_t(gt) << 32) | eq, scan64, &tot64);
  const uint32_t eq_before = uint32_t(pre64);         // ties of this CTA before this thread
  uint2* ge = gteq + int64_t(t) * 16;
  if (threadIdx.x == 0) ge[r] = make_uint2(uint32_t(tot64 >> 32), uint32_t(tot64));
  cluster.sync();
  if (threadIdx.x < 32) {
    // the CTAs before this one, one lane each: ties are taken in index order,
    // CTA rr takes min(eq_rr, need - ties before it)
    const int lane = threadIdx.x;
    const uint2 x = lane < r ? __ldcg(&ge[lane]) : make_uint2(0u, 0u);
    uint32_t ie = x.y;                              // inclusive prefix of the ties
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const uint32_t v = __shfl_up_sync(0xffffffffu, ie, off);
      if (lane >= off) ie += v;
    }
    const uint32_t e_before = ie - x.y;
    const uint32_t take = e_before >= need ? 0u : min(x.y, need - e_before);
    uint32_t sel = x.x + take;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) sel += __shfl_xor_sync(0xffffffffu, sel, off);
    const uint32_t all_e = __shfl_sync(0xffffffffu, ie, 31);
    if (lane == 0) { pre_s[0] = all_e; pre_s[1] = sel; }
  }
  __syncthreads();
  const uint32_t pre_eq = pre_s[0];
  // selected: key > K, or key == K and among the first `need` ties of the row
  uint32_t mine = 0;
  {
    uint32_t rk = pre_eq + eq_before;
#pragma unroll
    for (int u = 0; u < PER; ++u) {
      const bool in = i0 + u < n;
      if (in && key[u] > K) ++mine;
      else if (in && key[u] == K) { if (rk < need) ++mine; ++rk; }
    }
  }
  uint32_t tot;
  uint32_t pos = pre_s[1] + block_excl_scan(mine, scan, &tot);
  {
    uint32_t rk = pre_eq + eq_before;
#pragma unroll
    for (int u = 0; u < PER; ++u) {
      const bool in = i0 + u < n;
      bool take = false;
      if (in && key[u] > K) take = true;
      else if (in && key[u] == K) { take = rk < need; ++rk; }
      if (take && pos < uint32_t(k)) o[pos++] = i0 + u;   // the bound holds unless the histograms were incomplete
    }
  }
}

// ------------------------------------------------------------------------------
// Host side
// ------------------------------------------------------------------------------

// Largest cluster (16, else 8) topk_cluster runs with on this device (0 if none).
static int topk_cluster_size() {
  static int cached = 0;
  static std::once_flag once;
  std::call_once(once, [] {
    for (auto f : {topk_cluster<16>, topk_cluster<32>, topk_cluster<64>})
      cudaFuncSetAttribute(f, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    for (int cs : {16, 8}) {
      cudaLaunchConfig_t lc = {};
      lc.gridDim = dim3(unsigned(cs));
      lc.blockDim = dim3(1024);
      cudaLaunchAttribute at[1];
      at[0].id = cudaLaunchAttributeClusterDimension;
      at[0].val.clusterDim.x = unsigned(cs);
      at[0].val.clusterDim.y = 1;
      at[0].val.clusterDim.z = 1;
      lc.attrs = at;
      lc.numAttrs = 1;
      int n = 0;
      if (cudaOccupancyMaxActiveClusters(&n, topk_cluster<64>, &lc) == cudaSuccess && n > 0) {
        cached = cs;
        break;
      }
      cudaGetLastError();
    }
  });
  return cached;
}

// Shapes and formats only (enough to size the workspace).
static int validate_shape(const v4a_index_args* a) {
  if (!a) return V4A_ERR_INVALID_ARG;
  const v4a_batch& B = a->batch;
  if (B.num_tokens < 0 || B.num_seqs <= 0) return V4A_ERR_INVALID_ARG;
  if (B.num_tokens > 65535) return V4A_ERR_UNSUPPORTED;
  const v4a_cache& c = a->keys;
  if (c.ratio != 4) return V4A_ERR_UNSUPPORTED;
  if (c.num_blocks <= 0 || c.max_blocks <= 0) return V4A_ERR_INVALID_ARG;
  if (int64_t(c.max_blocks) * 64 > kBitmapMax) return V4A_ERR_UNSUPPORTED;
  if (a->k < 1 || a->k > kMaxK) return V4A_ERR_UNSUPPORTED;
  if (a->num_heads < 1 || a->num_heads > 128) return V4A_ERR_UNSUPPORTED;
  if (c.dim < 32 || c.dim > 256 || c.dim % 32) return V4A_ERR_UNSUPPORTED;
  if (c.format == V4A_IX_BF16) {
    if (a->q_format != V4A_Q_BF16) return V4A_ERR_UNSUPPORTED;
  } else if (c.format == V4A_IX_FP8_B128 || ix_is_fp4(c.format)) {
    if (a->q_format != V4A_Q_FP8_HEAD) return V4A_ERR_UNSUPPORTED;
    if (c.format == V4A_IX_FP8_B128 && c.dim % 128) return V4A_ERR_UNSUPPORTED;
  } else {
    return V4A_ERR_INVALID_ARG;
  }
  return V4A_OK;
}

static int validate(const v4a_index_args* a) {
  const int rc = validate_shape(a);
  if (rc) return rc;
  if (a->batch.num_tokens == 0) return V4A_OK;
  if (!a->batch.seq_ids || !a->batch.positions || !a->q || !a->weights || !a->out_idx ||
      !a->keys.pool || !a->keys.block_table)
    return V4A_ERR_INVALID_ARG;
  if (a->q_format == V4A_Q_FP8_HEAD && !a->q_scale) return V4A_ERR_INVALID_ARG;
  return V4A_OK;
}

int index_scores_layout(const v4a_index_args* a, size_t* offset, int64_t* row_stride) {
  if (validate_shape(a)) return V4A_ERR_INVALID_ARG;
  char* fake = reinterpret_cast<char*>(size_t(1) << 40);
  const IndexWs w = ws_layout(a, fake);
  if (offset) *offset = size_t(reinterpret_cast<char*>(w.scores) - fake);
  if (row_stride) *row_stride = w.row;
  return V4A_OK;
}

size_t index_workspace_size(const v4a_index_args* a) {
  if (validate_shape(a)) return 0;
  return ws_layout(a, nullptr).total;
}

// Zeroes the histogram/counter part of the workspace.  Launched so that it may
// start early; it waits for the kernel before it (which may still be reading
// the previous call's histograms) before it writes.
__global__ void __launch_bounds__(256) clear_words(uint32_t* p, size_t n) {
  pdl_trigger();
  pdl_wait();
  for (size_t i = size_t(blockIdx.x) * blockDim.x + threadIdx.x; i < n; i += size_t(gridDim.x) * blockDim.x) p[i] = 0u;
}

// Stage 1: clear the histogram/counters and score every visible entry.
int index_scores(const v4a_index_args* a, void* ws, size_t ws_bytes, cudaStream_t stream) {
  int rc = validate(a);
  if (rc) return rc;
  const int T = a->batch.num_tokens;
  if (T == 0) return V4A_OK;
  IndexWs w = ws_layout(a, nullptr);
  if (!ws || ws_bytes < w.total) return V4A_ERR_WORKSPACE;
  w = ws_layout(a, ws);
  const v4a_cache& c = a->keys;
  {
    const size_t words = w.zero_bytes / 4;
    const unsigned blocks = unsigned(std::min<size_t>((words + 255) / 256, 1024));
    if (launch_pdl(clear_words, dim3(blocks), dim3(256), 0, stream, w.hist, words) != cudaSuccess) return V4A_ERR_CUDA;
  }
  // the tensor-core scans always leave the level-1 histogram (both top-k paths use it)
  if (index_score_mx(a, w.scores, w.row, w.hist, stream, &rc)) return rc;
  if (index_score_tc(a, w.scores, w.row, w.hist, stream, &rc)) return rc;
  ScoreArgs sa;
  sa.T = T; sa.H = a->num_heads; sa.dim = c.dim; sa.k_fmt = c.format; sa.q_fmt = a->q_format;
  sa.seq_ids = a->batch.seq_ids; sa.positions = a->batch.positions; sa.keys = c;
  sa.block_bytes = ix_block_bytes(c.format, c.dim);
  sa.q = a->q; sa.q_scale = a->q_scale; sa.w = a->weights; sa.scores = w.scores; sa.row = w.row;
  sa.status = a->status;
  const size_t smem = size_t(a->num_heads * (c.dim + 1) + a->num_heads + 64 * (c.dim + 1)) * 4;
  if (smem > 227 * 1024) return V4A_ERR_UNSUPPORTED;
  cudaFuncSetAttribute(index_score_simt, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem));
  index_score_simt<<<dim3(unsigned(c.max_blocks), unsigned(T)), 256, smem, stream>>>(sa);
  return cudaGetLastError() == cudaSuccess ? V4A_OK : V4A_ERR_CUDA;
}

// Stage 2: top-k of the scores left in the workspace by stage 1.
int index_select(const v4a_index_args* a, void* ws, size_t ws_bytes, cudaStream_t stream) {
  int rc = validate(a);
  if (rc) return rc;
  const int T = a->batch.num_tokens;
  if (T == 0) return V4A_OK;
  IndexWs w = ws_layout(a, nullptr);
  if (!ws || ws_bytes < w.total) return V4A_ERR_WORKSPACE;
  w = ws_layout(a, ws);
  const bool tc_hist = index_score_mx_supported(a) || index_score_tc_supported(a);
  // Rows past kSmemTopkMax take the cluster path.  So do rows of more than
  // 8192 entries with a level-1 histogram when every query's cluster fits one
  // wave: its phases cost about the same at 32K entries as at 1M, below one
  // CTA's passes over a 32K-entry row.
  const int csz = topk_cluster_size();
  const bool cluster_wave = tc_hist && csz > 0 && w.row > 8192 && int64_t(T) * csz <= tc::sm_count() / 2;
  if (w.row <= kSmemTopkMax && !cluster_wave) {
    const uint32_t* h1 = tc_hist ? w.hist : nullptr;
    const size_t smem = (size_t(w.row) + (h1 ? size_t(kCandMax) : 0)) * 4;
    cudaFuncSetAttribute(topk_smem, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem));
    topk_smem<<<T, 1024, smem, stream>>>(w.scores, w.row, a->keys.max_blocks * 64, a->batch.positions,
                                         a->k, h1, a->out_idx);
  } else {
    const int slices = int((w.row + kSlice - 1) / kSlice);
    // the tensor-core scans already left the first-level histogram
    if (!index_score_mx_supported(a) && !index_score_tc_supported(a))
      topk_hist<<<dim3(slices, T), 512, 0, stream>>>(w.scores, w.row, a->keys.max_blocks * 64,
                                                     a->batch.positions, a->k, slices, w.hist);
    // one cluster per query; each thread holds PER consecutive scores
    const int cs = topk_cluster_size();
    if (cs == 0) return V4A_ERR_UNSUPPORTED;
    const int64_t per_needed = (w.row + int64_t(cs) * 1024 - 1) / (int64_t(cs) * 1024);
    if (per_needed > 64) return V4A_ERR_UNSUPPORTED;
    cudaLaunchConfig_t lc = {};
    lc.gridDim = dim3(unsigned(cs), unsigned(T));
    lc.blockDim = dim3(1024);
    lc.stream = stream;
    cudaLaunchAttribute at[2];
    at[0].id = cudaLaunchAttributeClusterDimension;
    at[0].val.clusterDim.x = unsigned(cs);
    at[0].val.clusterDim.y = 1;
    at[0].val.clusterDim.z = 1;
    at[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[1].val.programmaticStreamSerializationAllowed = 1;
    lc.attrs = at;
    lc.numAttrs = 2;
    const float* sc = w.scores;
    const uint32_t* h1 = w.hist;
    const int me = a->keys.max_blocks * 64;
    cudaError_t e;
    if (per_needed <= 16)
      e = cudaLaunchKernelEx(&lc, topk_cluster<16>, sc, w.row, me, a->batch.positions, a->k, h1, w.hist2, w.hist3,
                             w.gteq, a->out_idx);
    else if (per_needed <= 32)
      e = cudaLaunchKernelEx(&lc, topk_cluster<32>, sc, w.row, me, a->batch.positions, a->k, h1, w.hist2, w.hist3,
                             w.gteq, a->out_idx);
    else
      e = cudaLaunchKernelEx(&lc, topk_cluster<64>, sc, w.row, me, a->batch.positions, a->k, h1, w.hist2, w.hist3,
                             w.gteq, a->out_idx);
    if (e != cudaSuccess) return V4A_ERR_CUDA;
  }
  return cudaGetLastError() == cudaSuccess ? V4A_OK : V4A_ERR_CUDA;
}

int index_topk(const v4a_index_args* a, void* ws, size_t ws_bytes, cudaStream_t stream) {
  const int rc = index_scores(a, ws, ws_bytes, stream);
  return rc ? rc : index_select(a, ws, ws_bytes, stream);
}

}  // namespace v4a
