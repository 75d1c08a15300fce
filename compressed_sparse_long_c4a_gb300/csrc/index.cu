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
//  * index_score_tc    - tcgen05 scores for fp8 / fp4 caches (index_tc.cu).
//  * topk_smem         - one CTA per query when the row fits in shared memory:
//                         radix select of the k-th largest (score, -index)
//                         composite, then an ordered compaction.
//  * topk_hist / topk_select - long rows, one CTA per 8192-score slice: a
//                         4096-bin histogram of the score keys' top 12 bits
//                         (built by the tensor-core scan itself when that
//                         path scored the row, else by topk_hist) gives the
//                         threshold bin; every slice then compacts,
//                         in index order, its entries above that bin ("takes")
//                         and those in it ("candidates", plus a histogram of
//                         their next 12 bits).  The last slice CTA of a query
//                         resolves the exact threshold among the candidates
//                         and merges the two ordered lists into the output.
//                         The "last CTA" is found with an atomic counter; no
//                         CTA ever waits on another.  It holds up to 8
//                         candidates per thread in registers, so the
//                         candidates are read from L2 once.
//  * topk_coop          - long rows when every slice CTA of the batch fits on
//                         the GPU at once (cooperative launch): the exact
//                         k-th largest key comes from three histogram levels
//                         (12 + 12 + 8 bits) shared by the query's slices
//                         through bounded global barriers, then each slice
//                         writes its share in ascending index order.  This
//                         is the path of the 1M-context decode; topk_select
//                         covers batches too large for one wave.

#include <cstdio>
#include <algorithm>
#include <mutex>

#include "v4a_common.cuh"
#include "v4a_internal.h"
#include "index_tc.h"

namespace v4a {

constexpr int kSmemTopkMax = 32768;   // rows up to this length use topk_smem
constexpr int kHistBins = 4096;       // top 12 bits of the order-preserving key
constexpr int kMaxK = 16384;
constexpr int kSlice = 8192;          // scores per CTA of the long-row top-k (8 per thread)
constexpr int kMaxSlices = 1024;      // rows up to 8M entries

struct IndexWs {
  float* scores;        // [T][row]
  uint32_t* hist;       // [T][kHistBins]   top 12 key bits of every score
  uint32_t* hist2;      // [T][kHistBins]   next 12 bits of the threshold bin's scores
  uint32_t* hist3;      // [T][256]         last 8 bits of the threshold sub-bin's scores
  uint32_t* counters;   // [T][4]: arrivals at the cooperative select's barriers / "done" of the fallback
  uint64_t* cand;       // [T][row]: slice s keeps its takes at [lo, ..) and its candidates at [.., hi)
  uint32_t* info;       // [T][slices]: takes | candidates << 16 of each slice
  uint2* gteq;          // [T][slices]: entries above / equal to the exact threshold key, per slice
  int64_t row;
  size_t zero_bytes;    // bytes of hist + counters (cleared per call)
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
  w.counters = reinterpret_cast<uint32_t*>(take(size_t(T) * 4 * 4));
  w.zero_bytes = off;
  w.scores = reinterpret_cast<float*>(take(size_t(T) * w.row * 4));
  if (w.row > kSmemTopkMax) {
    w.cand = reinterpret_cast<uint64_t*>(take(size_t(T) * w.row * 8));
    w.info = reinterpret_cast<uint32_t*>(take(size_t(T) * ((w.row + kSlice - 1) / kSlice) * 4));
    w.gteq = reinterpret_cast<uint2*>(take(size_t(T) * ((w.row + kSlice - 1) / kSlice) * 8));
  }
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
    for (int i = threadIdx.x; i < n; i += blockDim.x) {
      const uint64_t c = get(i);
      if ((c & mask) == prefix) atomicAdd(&hist[(c >> shift) & 255], 1u);
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

__device__ void write_all_visible(int32_t* out, int n, int k) {
  for (int i = threadIdx.x; i < k; i += blockDim.x) out[i] = i < n ? i : -1;
}

// ------------------------------------------------------------------------------
// Single-CTA top-k (rows that fit in shared memory)
// ------------------------------------------------------------------------------

__global__ void __launch_bounds__(1024) topk_smem(const float* scores, int64_t row, int max_entries,
                                                 const int32_t* positions, int k, int32_t* out) {
  extern __shared__ uint32_t keys_s[];
  __shared__ uint32_t hist[256];
  __shared__ uint32_t sh[4];
  __shared__ uint32_t scan[40];
  const int t = blockIdx.x;
  const int n = min((positions[t] + 1) / 4, max_entries);
  int32_t* o = out + int64_t(t) * k;
  if (n <= k) { write_all_visible(o, n, k); return; }
  const float* s = scores + int64_t(t) * row;
  for (int i = threadIdx.x; i < n; i += blockDim.x) keys_s[i] = float_key(s[i]);
  __syncthreads();
  const uint64_t thr = select_threshold(
      n, k, [&](int i) { return composite(keys_s[i], i); }, hist, sh);
  // ordered compaction: thread c owns indices [c*chunk, (c+1)*chunk)
  const int chunk = (n + blockDim.x - 1) / blockDim.x;
  const int lo = threadIdx.x * chunk, hi = min(n, lo + chunk);
  uint32_t cnt = 0;
  for (int i = lo; i < hi; ++i) cnt += composite(keys_s[i], i) >= thr;
  uint32_t off = block_excl_scan(cnt, scan, nullptr);
  for (int i = lo; i < hi; ++i)
    if (composite(keys_s[i], i) >= thr) o[off++] = i;
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

// Threshold bin of a 4096-bin histogram: the bin b such that fewer than `need`
// counts lie strictly above it and at least `need` at or above it.  Block of
// 1024 threads, 4 bins each (scanned from the top).  Returns b and, through
// *above, the count strictly above it.
__device__ int threshold_bin(const uint32_t* h, uint32_t need, uint32_t* scan, int* bin_s,
                             uint32_t* above_s, uint32_t* above) {
  uint32_t loc[4], s4 = 0;
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const int bin = kHistBins - 1 - (threadIdx.x * 4 + q);
    loc[q] = bin >= 0 ? h[bin] : 0;
    s4 += loc[q];
  }
  uint32_t total;
  const uint32_t excl = block_excl_scan(s4, scan, &total);
  if (excl < need && need <= excl + s4) {
    uint32_t acc = excl;
    int q = 0;
    for (; q < 4; ++q) {
      if (acc + loc[q] >= need) break;
      acc += loc[q];
    }
    *bin_s = kHistBins - 1 - (threadIdx.x * 4 + q);
    *above_s = acc;
  }
  __syncthreads();
  *above = *above_s;
  const int b = *bin_s;
  __syncthreads();
  return b;
}

constexpr int kFine = 2048;   // capacity of the resolving CTA's exact-select list
constexpr int kRegCands = 8;  // threshold-bin candidates per thread held in registers while resolving

// Position of j among the slices' ranges: the largest s with pre[s] <= j.
__device__ __forceinline__ int slice_of(const uint32_t* pre, int nsl, uint32_t j) {
  int lo = 0, hi = nsl - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (pre[mid] <= j) lo = mid; else hi = mid - 1;
  }
  return lo;
}

// Number of elements of the ascending list l[0..n) below x.
__device__ __forceinline__ int count_below(const int32_t* l, int n, int32_t x) {
  int lo = 0, hi = n;
  while (lo < hi) {
    const int mid = (lo + hi) >> 1;
    if (l[mid] < x) lo = mid + 1; else hi = mid;
  }
  return lo;
}

__global__ void __launch_bounds__(1024, 1) topk_select(const float* scores, int64_t row, int max_entries,
                                                   const int32_t* positions, int k, int slices,
                                                   const uint32_t* hist, uint32_t* hist2,
                                                   uint32_t* counters, uint64_t* cand, uint32_t* info,
                                                   int32_t* out) {
  extern __shared__ int32_t lists_s[];   // resolving CTA: [k] takes, then [k] selected candidates
  __shared__ uint32_t scan[40];
  __shared__ uint32_t h2_s[kHistBins];
  __shared__ uint64_t fine_s[kFine];
  __shared__ uint32_t pre_s[2][kMaxSlices + 1];
  __shared__ uint32_t hist256[256];
  __shared__ uint32_t sh[4];
  __shared__ int bin_s;
  __shared__ uint32_t above_s;
  __shared__ int last_s;
  __shared__ uint32_t nfine_s;
  const int t = blockIdx.y, sl = blockIdx.x;
  const int n = min((positions[t] + 1) / 4, max_entries);
  int32_t* o = out + int64_t(t) * k;
  if (n <= k) {
    if (sl == 0) write_all_visible(o, n, k);
    return;
  }
  const int nsl = (n + kSlice - 1) / kSlice;
  if (sl >= nsl) return;
  // 1. this slice's scores (thread c owns entries lo + 8c .. lo + 8c + 7), loaded
  //    first so that their latency overlaps the threshold search below
  constexpr int kPer = kSlice / 1024;
  const int lo = sl * kSlice, hi = min(n, lo + kSlice);
  const float* sc = scores + int64_t(t) * row;
  const int i0 = lo + kPer * int(threadIdx.x);
  float v[kPer];
  if (i0 + kPer - 1 < hi) {
#pragma unroll
    for (int u = 0; u < kPer; u += 4) {
      const float4 f = __ldcg(reinterpret_cast<const float4*>(sc + i0 + u));
      v[u] = f.x; v[u + 1] = f.y; v[u + 2] = f.z; v[u + 3] = f.w;
    }
  } else {
#pragma unroll
    for (int u = 0; u < kPer; ++u) v[u] = i0 + u < hi ? __ldcg(sc + i0 + u) : 0.f;
  }
  for (int i = threadIdx.x; i < kHistBins; i += blockDim.x) h2_s[i] = 0;
  // 2. threshold bin of the top 12 key bits
  uint32_t above1;
  const uint32_t tbin = uint32_t(threshold_bin(hist + int64_t(t) * kHistBins, uint32_t(k), scan, &bin_s,
                                               &above_s, &above1));
  // 3. ordered compaction of this slice into its range of the candidate array:
  //    entries above the threshold bin ("takes", as indices) from the front,
  //    entries in it (as composites) at the back
  uint32_t key[kPer], ntk = 0, ncd = 0;
#pragma unroll
  for (int u = 0; u < kPer; ++u) {
    key[u] = float_key(v[u]);
    const bool in = i0 + u < hi;
    ntk += in && (key[u] >> 20) > tbin;
    ncd += in && (key[u] >> 20) == tbin;
  }
  uint32_t tot;
  const uint32_t off = block_excl_scan(ntk | (ncd << 16), scan, &tot);   // both halves <= kSlice < 2^16
  const uint32_t NCD = tot >> 16;
  uint32_t otk = off & 0xFFFFu, ocd = off >> 16;
  uint64_t* cd = cand + int64_t(t) * row;
#pragma unroll
  for (int u = 0; u < kPer; ++u) {
    const int i = i0 + u;
    if (i >= hi) continue;
    const uint32_t b = key[u] >> 20;
    if (b > tbin) {
      cd[lo + otk++] = uint64_t(i);
    } else if (b == tbin) {
      cd[hi - NCD + ocd++] = composite(key[u], i);
      atomicAdd(&h2_s[(key[u] >> 8) & (kHistBins - 1)], 1u);
    }
  }
  __syncthreads();
  uint32_t* g2 = hist2 + int64_t(t) * kHistBins;
  for (int i = threadIdx.x; i < kHistBins; i += blockDim.x)
    if (h2_s[i]) atomicAdd(&g2[i], h2_s[i]);
  if (threadIdx.x == 0) info[int64_t(t) * slices + sl] = tot;
  // 4. the last slice CTA of this query resolves the threshold and merges
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) last_s = atomicAdd(&counters[int64_t(t) * 4 + 2], 1u) == uint32_t(nsl - 1);
  __syncthreads();
  if (!last_s) return;
  __threadfence();
  {
    // slice counts and the second-level histogram, both loads in flight together
    const uint32_t x = int(threadIdx.x) < nsl ? __ldcg(&info[int64_t(t) * slices + threadIdx.x]) : 0u;
    for (int i = threadIdx.x; i < kHistBins; i += blockDim.x) h2_s[i] = __ldcg(&g2[i]);
    uint32_t tk_tot, cd_tot;
    const uint32_t ptk = block_excl_scan(x & 0xFFFFu, scan, &tk_tot);
    const uint32_t pcd = block_excl_scan(x >> 16, scan, &cd_tot);
    if (int(threadIdx.x) < nsl) { pre_s[0][threadIdx.x] = ptk; pre_s[1][threadIdx.x] = pcd; }
    if (threadIdx.x == 0) { pre_s[0][nsl] = tk_tot; pre_s[1][nsl] = cd_tot; nfine_s = 0; }
  }
  __syncthreads();
  const int above = int(pre_s[0][nsl]);      // entries above the threshold bin (< k)
  const int nc = int(pre_s[1][nsl]);         // entries in it (>= k - above)
  const int need = k - above;
  int32_t* take_l = lists_s;
  int32_t* csel_l = lists_s + k;
  auto cand_at = [&](int j) -> uint64_t {    // j-th candidate in index order
    const int s2 = slice_of(pre_s[1], nsl, uint32_t(j));
    const int hi2 = min(n, (s2 + 1) * kSlice);
    const int ncd2 = int(pre_s[1][s2 + 1] - pre_s[1][s2]);
    return __ldcg(reinterpret_cast<const unsigned long long*>(&cd[hi2 - ncd2 + (j - int(pre_s[1][s2]))]));
  };
  // takes, in index order (independent of the exact threshold)
  for (int j = threadIdx.x; j < above; j += blockDim.x) {
    const int s2 = slice_of(pre_s[0], nsl, uint32_t(j));
    take_l[j] = int32_t(__ldcg(reinterpret_cast<const unsigned long long*>(
        &cd[int64_t(s2) * kSlice + (j - int(pre_s[0][s2]))])));
  }
  if (nc <= int(blockDim.x) * kRegCands) {
    // common case: every candidate is read once into registers; thread c owns
    // the run [c*R, c*R + R) of the candidates, so its selected ones are
    // consecutive in index order
    const int R = (nc + int(blockDim.x) - 1) / int(blockDim.x);
    const int j0 = int(threadIdx.x) * R;
    uint64_t c[kRegCands];
#pragma unroll
    for (int u = 0; u < kRegCands; ++u) c[u] = (u < R && j0 + u < nc) ? cand_at(j0 + u) : 0ull;
    uint32_t above2;
    const uint32_t tbin2 = uint32_t(threshold_bin(h2_s, uint32_t(need), scan, &bin_s, &above_s, &above2));
    const int need2 = need - int(above2);
    uint64_t thr;
    if (h2_s[tbin2] <= uint32_t(kFine)) {
#pragma unroll
      for (int u = 0; u < kRegCands; ++u)
        if (u < R && j0 + u < nc && ((uint32_t(c[u] >> 40) & (kHistBins - 1)) == tbin2))
          fine_s[atomicAdd(&nfine_s, 1u)] = c[u];
      __syncthreads();
      // the sub-bin's candidates share their top 24 key bits: select on the rest
      thr = select_threshold(int(nfine_s), need2, [&](int i) { return fine_s[i]; }, hist256, sh, 3);
    } else {
      // degenerate (e.g. all scores equal): exact select over every candidate of the sub-bin
      thr = select_threshold(nc, need2, [&](int j) {
        const uint64_t cc = cand_at(j);
        return (uint32_t(cc >> 40) & (kHistBins - 1)) == tbin2 ? cc : uint64_t(0);
      }, hist256, sh);
    }
    uint32_t cnt = 0;
#pragma unroll
    for (int u = 0; u < kRegCands; ++u) cnt += (u < R && j0 + u < nc && c[u] >= thr) ? 1u : 0u;
    uint32_t pos = block_excl_scan(cnt, scan, nullptr);
#pragma unroll
    for (int u = 0; u < kRegCands; ++u)
      if (u < R && j0 + u < nc && c[u] >= thr) csel_l[pos++] = int32_t(0xFFFFFFFFu - uint32_t(c[u]));
  } else {
    // more candidates than registers hold: stream them from L2 in each pass
    uint32_t above2;
    const uint32_t tbin2 = uint32_t(threshold_bin(h2_s, uint32_t(need), scan, &bin_s, &above_s, &above2));
    const int need2 = need - int(above2);
    const uint64_t thr = select_threshold(nc, need2, [&](int j) {
      const uint64_t cc = cand_at(j);
      return (uint32_t(cc >> 40) & (kHistBins - 1)) == tbin2 ? cc : uint64_t(0);
    }, hist256, sh);
    uint32_t carry = 0;
    for (int b0 = 0; b0 < nc; b0 += blockDim.x) {
      const int j = b0 + int(threadIdx.x);
      const uint64_t cc = j < nc ? cand_at(j) : 0ull;
      const bool f = j < nc && cc >= thr;
      uint32_t cnt;
      const uint32_t pos = block_excl_scan(f ? 1u : 0u, scan, &cnt);
      if (f) csel_l[carry + pos] = int32_t(0xFFFFFFFFu - uint32_t(cc));
      carry += cnt;
    }
  }
  __syncthreads();
  // merge the two ascending lists (disjoint indices) into the output
  for (int j = threadIdx.x; j < above; j += blockDim.x) {
    const int32_t x = take_l[j];
    const int d = j + count_below(csel_l, need, x);
    if (d < k) o[d] = x;
  }
  for (int j = threadIdx.x; j < need; j += blockDim.x) {
    const int32_t y = csel_l[j];
    const int d = j + count_below(take_l, above, y);
    if (d < k) o[d] = y;
  }
}

// ------------------------------------------------------------------------------
// Cooperative long-row top-k (all CTAs of the grid co-resident)
// ------------------------------------------------------------------------------
//
// One CTA per 8192-score slice of a query, every slice kept in registers.
// The exact k-th largest key K* is found with three histogram levels of the
// order-preserving key (top 12 bits: built by the tensor-core scan; next 12
// bits; last 8 bits), each level a global histogram filled by the query's
// CTAs and read by all of them after a barrier of the query's CTAs.  Then
// every CTA publishes how many of its entries lie above K* and at K*; after a
// last barrier each CTA knows, from the prefix over the slices before it, its
// share of the ties at K* (lowest indices first) and its output offset, and
// writes its selected indices in ascending order.  No candidate lists, no
// single resolving CTA.

// Waits until `target` CTAs have arrived at *counter (bounded; false if it gave up).
__device__ __forceinline__ bool slice_barrier(uint32_t* counter, uint32_t target, int32_t* status, int* give_up) {
  __syncthreads();
  if (threadIdx.x == 0) {
    __threadfence();
    atomicAdd(counter, 1u);
    const long long t0 = clock64();
    uint32_t v = 0;
    while (true) {
      asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(counter) : "memory");
      if (v >= target) break;
      if (clock64() - t0 > 2000000000LL) {
        report(status, V4A_DEV_TIMEOUT);
        *give_up = 1;
        break;
      }
      __nanosleep(64);
    }
    __threadfence();
  }
  __syncthreads();
  return *give_up == 0;
}

// Threshold of a 256-bin histogram (warp 0 scans; result broadcast through shared memory).
__device__ int threshold_bin256(const uint32_t* h, uint32_t need, int* bin_s, uint32_t* above_s,
                                uint32_t* above) {
  if (threadIdx.x < 32) {
    const int lane = threadIdx.x;
    uint32_t loc[8], s8 = 0;
#pragma unroll
    for (int q = 0; q < 8; ++q) { loc[q] = __ldcg(&h[255 - (lane * 8 + q)]); s8 += loc[q]; }
    uint32_t incl = s8;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t x = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += x;
    }
    const uint32_t excl = incl - s8;
    if (excl < need && need <= incl) {
      uint32_t acc = excl;
      int q = 0;
      for (; q < 8; ++q) {
        if (acc + loc[q] >= need) break;
        acc += loc[q];
      }
      *bin_s = 255 - (lane * 8 + q);
      *above_s = acc;
    }
  }
  __syncthreads();
  *above = *above_s;
  const int b = *bin_s;
  __syncthreads();
  return b;
}

__global__ void __launch_bounds__(1024, 1) topk_coop(const float* scores, int64_t row, int max_entries,
                                                 const int32_t* positions, int k, int slices,
                                                 const uint32_t* hist1, uint32_t* hist2, uint32_t* hist3,
                                                 uint32_t* counters, uint2* gteq, int32_t* out, int32_t* status) {
  pdl_trigger();   // the attention kernel may be scheduled on SMs this grid leaves free
  __shared__ uint32_t scan[40];
  __shared__ uint32_t h_s[kHistBins];
  __shared__ int bin_s, give_up;
  __shared__ uint32_t above_s;
  constexpr int kPer = kSlice / 1024;
  const int t = blockIdx.y, sl = blockIdx.x;
  const int n = min((positions[t] + 1) / 4, max_entries);
  int32_t* o = out + int64_t(t) * k;
  if (n <= k) {                        // every CTA of this query leaves together
    if (sl == 0) write_all_visible(o, n, k);
    return;
  }
  const int nsl = (n + kSlice - 1) / kSlice;
  if (sl >= nsl) return;               // not one of this query's slices
  if (threadIdx.x == 0) give_up = 0;
  const int lo = sl * kSlice, hi = min(n, lo + kSlice);
  const float* sc = scores + int64_t(t) * row;
  const int i0 = lo + kPer * int(threadIdx.x);
  uint32_t key[kPer];
  {
    float v[kPer];
    if (i0 + kPer - 1 < hi) {
#pragma unroll
      for (int u = 0; u < kPer; u += 4) {
        const float4 f = __ldcg(reinterpret_cast<const float4*>(sc + i0 + u));
        v[u] = f.x; v[u + 1] = f.y; v[u + 2] = f.z; v[u + 3] = f.w;
      }
    } else {
#pragma unroll
      for (int u = 0; u < kPer; ++u) v[u] = i0 + u < hi ? __ldcg(sc + i0 + u) : 0.f;
    }
#pragma unroll
    for (int u = 0; u < kPer; ++u) key[u] = i0 + u < hi ? float_key(v[u]) : 0u;   // key 0: below every score
  }
  uint32_t* cnt = counters + int64_t(t) * 4;
  // level 1: top 12 bits (histogram from the scan)
  for (int i = threadIdx.x; i < kHistBins; i += blockDim.x) h_s[i] = 0;
  uint32_t above1;
  const uint32_t b1 = uint32_t(threshold_bin(hist1 + int64_t(t) * kHistBins, uint32_t(k), scan, &bin_s, &above_s,
                                             &above1));
  // level 2: next 12 bits of the entries in bin b1
#pragma unroll
  for (int u = 0; u < kPer; ++u)
    if (i0 + u < hi && (key[u] >> 20) == b1) atomicAdd(&h_s[(key[u] >> 8) & (kHistBins - 1)], 1u);
  __syncthreads();
  uint32_t* g2 = hist2 + int64_t(t) * kHistBins;
  for (int i = threadIdx.x; i < kHistBins; i += blockDim.x) {
    if (h_s[i]) atomicAdd(&g2[i], h_s[i]);
    h_s[i] = 0;
  }
  if (!slice_barrier(&cnt[0], uint32_t(nsl), status, &give_up)) return;
  const uint32_t need1 = uint32_t(k) - above1;
  uint32_t above2;
  const uint32_t b2 = uint32_t(threshold_bin(g2, need1, scan, &bin_s, &above_s, &above2));
  // level 3: last 8 bits of the entries in sub-bin (b1, b2)
  const uint32_t top24 = (b1 << 12) | b2;
#pragma unroll
  for (int u = 0; u < kPer; ++u)
    if (i0 + u < hi && (key[u] >> 8) == top24) atomicAdd(&h_s[key[u] & 255u], 1u);
  __syncthreads();
  uint32_t* g3 = hist3 + int64_t(t) * 256;
  for (int i = threadIdx.x; i < 256; i += blockDim.x)
    if (h_s[i]) atomicAdd(&g3[i], h_s[i]);
  if (!slice_barrier(&cnt[1], uint32_t(nsl), status, &give_up)) return;
  const uint32_t need2 = need1 - above2;
  uint32_t above3;
  const uint32_t b3 = uint32_t(threshold_bin256(g3, need2, &bin_s, &above_s, &above3));
  const uint32_t K = (top24 << 8) | b3;                       // exact key of the k-th largest
  const uint32_t need = need2 - above3;                       // entries equal to K to take (>= 1)
  // this slice's entries above K and equal to K
  uint32_t gt = 0, eq = 0;
#pragma unroll
  for (int u = 0; u < kPer; ++u) {
    const bool in = i0 + u < hi;
    gt += in && key[u] > K;
    eq += in && key[u] == K;
  }
  uint32_t tot;
  const uint32_t eq_before = block_excl_scan(eq, scan, &tot);   // ties of this slice before this thread
  const uint32_t eq_slice = tot;
  const uint32_t gt_slice = block_excl_scan(gt, scan, &tot), gt_total = tot;
  (void)gt_slice;
  if (threadIdx.x == 0) gteq[int64_t(t) * slices + sl] = make_uint2(gt_total, eq_slice);
  if (!slice_barrier(&cnt[2], uint32_t(nsl), status, &give_up)) return;
  // ties taken by the slices before this one, and this slice's output offset
  __shared__ uint32_t pre_eq_s, pre_sel_s;
  {
    uint32_t e = 0, sel = 0, ge = 0;
    if (int(threadIdx.x) < sl) {
      const uint2 x = __ldcg(&gteq[int64_t(t) * slices + threadIdx.x]);
      ge = x.x;
      e = x.y;
    }
    const uint32_t pe = block_excl_scan(e, scan, &tot);         // ties in slices before slice threadIdx.x
    if (int(threadIdx.x) < sl) {
      const uint32_t take = pe >= need ? 0u : min(e, need - pe);
      sel = ge + take;
    }
    uint32_t sel_tot;
    block_excl_scan(sel, scan, &sel_tot);
    if (threadIdx.x == 0) { pre_eq_s = tot; pre_sel_s = sel_tot; }
    __syncthreads();
  }
  const uint32_t pre_eq = pre_eq_s, pre_sel = pre_sel_s;
  // ordered compaction: entry selected if key > K, or key == K and it is among
  // the first `need` ties of the row in index order
  uint32_t mine = 0;
  {
    uint32_t r = pre_eq + eq_before;
#pragma unroll
    for (int u = 0; u < kPer; ++u) {
      const bool in = i0 + u < hi;
      if (in && key[u] > K) ++mine;
      else if (in && key[u] == K) { if (r < need) ++mine; ++r; }
    }
  }
  uint32_t pos = pre_sel + block_excl_scan(mine, scan, &tot);
  {
    uint32_t r = pre_eq + eq_before;
#pragma unroll
    for (int u = 0; u < kPer; ++u) {
      const bool in = i0 + u < hi;
      bool take = false;
      if (in && key[u] > K) take = true;
      else if (in && key[u] == K) { take = r < need; ++r; }
      if (take && pos < uint32_t(k)) o[pos++] = i0 + u;   // the bound holds unless the histograms were incomplete
    }
  }
}

// ------------------------------------------------------------------------------
// Host side
// ------------------------------------------------------------------------------

// CTAs of topk_coop that can be resident at once on this device (its grid
// must not exceed this: its CTAs wait for one another).
static int64_t coop_capacity() {
  static int64_t cap = -1;
  static std::once_flag once;
  std::call_once(once, [] {
    int dev = 0, sms = 0, per = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per, topk_coop, 1024, 0) != cudaSuccess) per = 0;
    cap = int64_t(sms) * per;
  });
  return cap;
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
  if (int64_t(c.max_blocks) * 64 > int64_t(kMaxSlices) * kSlice) return V4A_ERR_UNSUPPORTED;
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
  uint32_t* hist = w.row > kSmemTopkMax ? w.hist : nullptr;
  if (index_score_mx(a, w.scores, w.row, hist, stream, &rc)) return rc;
  if (index_score_tc(a, w.scores, w.row, hist, stream, &rc)) return rc;
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
  if (w.row <= kSmemTopkMax) {
    const size_t smem = size_t(w.row) * 4;
    cudaFuncSetAttribute(topk_smem, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem));
    topk_smem<<<T, 1024, smem, stream>>>(w.scores, w.row, a->keys.max_blocks * 64, a->batch.positions,
                                         a->k, a->out_idx);
  } else {
    const int slices = int((w.row + kSlice - 1) / kSlice);
    // the tensor-core scans already left the first-level histogram
    if (!index_score_mx_supported(a) && !index_score_tc_supported(a))
      topk_hist<<<dim3(slices, T), 512, 0, stream>>>(w.scores, w.row, a->keys.max_blocks * 64,
                                                     a->batch.positions, a->k, slices, w.hist);
    // all of a query's slices resolve together in one cooperative grid when
    // the whole grid fits on the GPU at once; otherwise one CTA per query
    // resolves after the others have compacted their slices
    if (int64_t(slices) * T <= coop_capacity()) {
      cudaLaunchConfig_t lc = {};
      lc.gridDim = dim3(unsigned(slices), unsigned(T));
      lc.blockDim = dim3(1024);
      lc.stream = stream;
      cudaLaunchAttribute at[1];
      at[0].id = cudaLaunchAttributeCooperative;
      at[0].val.cooperative = 1;
      lc.attrs = at;
      lc.numAttrs = 1;
      if (cudaLaunchKernelEx(&lc, topk_coop, static_cast<const float*>(w.scores), w.row, a->keys.max_blocks * 64,
                             a->batch.positions, a->k, slices, static_cast<const uint32_t*>(w.hist), w.hist2,
                             w.hist3, w.counters, w.gteq, a->out_idx, a->status) != cudaSuccess)
        return V4A_ERR_CUDA;
    } else {
      const size_t smem = size_t(2) * a->k * 4;
      cudaFuncSetAttribute(topk_select, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem));
      topk_select<<<dim3(slices, T), 1024, smem, stream>>>(w.scores, w.row, a->keys.max_blocks * 64,
                                                           a->batch.positions, a->k, slices, w.hist,
                                                           w.hist2, w.counters, w.cand, w.info, a->out_idx);
    }
  }
  return cudaGetLastError() == cudaSuccess ? V4A_OK : V4A_ERR_CUDA;
}

int index_topk(const v4a_index_args* a, void* ws, size_t ws_bytes, cudaStream_t stream) {
  const int rc = index_scores(a, ws, ws_bytes, stream);
  return rc ? rc : index_select(a, ws, ws_bytes, stream);
}

}  // namespace v4a
