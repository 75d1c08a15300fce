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
// Tile = 128 entries (two 64-entry physical blocks) x 64 heads x 128 dims:
//  A = key codes, M = 128 rows (TMEM lane = entry), K-major, 128-byte swizzle,
//      loaded by TMA straight from the paged pool (3-D tensor map: row bytes,
//      64 rows, block id; fp4 rows land in the padded 16-elements-per-16-bytes
//      layout the f8f6f4 MMA reads);
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
//   warp 0      TMA producer: kStages-deep ring of key tiles, each with the
//               two blocks' fp32 scale words (1-D bulk copies); also copies
//               the query codes and w_h * qs_h into double-buffered smem.
//   warp 1      TMEM allocator and single-thread MMA issuer; accumulators are
//               double-buffered in TMEM.
//   warps 2..9  two epilogue warpgroups, one per accumulator (alternate
//               tiles): one thread per entry (TMEM lane) reads its
//               accumulators, applies scales, ReLU and head weights with
//               packed fp32x2 FMAs and writes the score.
// A stage is refilled only after the MMA (commit) and the owning epilogue
// warpgroup (scale words read) have released it.
// Every mbarrier wait is bounded (V4A_DEV_TIMEOUT, then a clean exit).

#include <cuda.h>
#include <cudaTypedefs.h>

#include <mutex>

#include "index_tc.h"
#include "tc_common.cuh"

namespace v4a {
namespace {

constexpr int kStages = 8;
constexpr int kTileBytes = 128 * 128;    // 128 rows x 128 smem bytes (one MMA operand)
constexpr int kBlockSmem = 64 * 128;     // one 64-entry block in smem
constexpr int kScaleBytes = 2048;        // scale words of the two blocks of a tile (fp4: 2 x 1 KB)
constexpr int kQBytes = 64 * 128;        // 64 heads x 128 codes
constexpr int kEpiWarps = 8;             // two epilogue warpgroups
constexpr int kThreads = 64 + 32 * kEpiWarps;

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
  const uint8_t* q;           // [T][64][128] e4m3
  const float* qs;            // [T][64]
  const float* w;             // [T][64]
  float* scores;
  int64_t row;
  int32_t* status;
  uint32_t idesc;
  uint32_t tx_per_block;
};

struct Smem {
  uint64_t full[kStages], empty[kStages], tfull[2], tempty[2], qfull[2], qempty[2], done;
  uint32_t tmem_base;
  int abort_flag;
  int t0, j0, count;
  uint32_t valid[kStages];  // bit h: block h of the stage's tile was loaded
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
  s.part[threadIdx.x] = mine;
  if (threadIdx.x == 0) { s.count = 0; s.t0 = a.T; s.j0 = 0; }
  __syncthreads();
  uint32_t before = 0, all = 0;
  for (int i = 0; i < int(blockDim.x); ++i) {
    const uint32_t v = s.part[i];
    if (i < int(threadIdx.x)) before += v;
    all += v;
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

__global__ void __launch_bounds__(kThreads, 1)
index_scan_tc(const TcArgs a, const __grid_constant__ CUtensorMap tmap) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* tiles = base;                                   // kStages x 16 KB
  uint8_t* qbuf = tiles + kStages * kTileBytes;            // 2 x 8 KB
  uint8_t* scl = qbuf + 2 * kQBytes;                       // kStages x 2 KB
  Smem& s = *reinterpret_cast<Smem*>(scl + kStages * kScaleBytes);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  volatile int* abort_flag = &s.abort_flag;

  if (threadIdx.x == 0) {
    for (int i = 0; i < kStages; ++i) {
      tc::mbar_init(&s.full[i], 1);
      tc::mbar_init(&s.empty[i], 1 + 4);            // MMA commit + the owning warpgroup
    }
    for (int i = 0; i < 2; ++i) {
      tc::mbar_init(&s.tfull[i], 1);
      tc::mbar_init(&s.tempty[i], 4);
      tc::mbar_init(&s.qfull[i], 1);
      tc::mbar_init(&s.qempty[i], 1 + kEpiWarps);   // MMA commit + every epilogue warp
    }
    tc::mbar_init(&s.done, 1);
    s.abort_flag = 0;
    tc::mbar_fence_init();
  }
  if (warp == 0 && lane == 0) tc::prefetch_tmap(&tmap);
  __syncwarp();   // tcgen05.alloc is warp-collective
  if (warp == 1) tc::tmem_alloc(&s.tmem_base, 2 * a.acc_cols);
  tc::tc_fence_before();
  plan(a, s);              // contains __syncthreads
  tc::tc_fence_after();
  const uint32_t tmem = s.tmem_base;
  const int count = s.count;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    Cursor c;
    c.init(a, s.t0, s.j0);
    int cur_t = -1, qi = -1, stage = 0;
    uint32_t phase = 0;
    uint32_t last_phase[kStages];
    int issued = 0;
    int b = 0, nblk = 0;
    for (int it = 0; it < count; ++it) {
      if (c.t != cur_t) {
        cur_t = c.t;
        ++qi;
        const int qb = qi & 1;
        b = a.seq_ids[cur_t];
        nblk = (visible_of(a, cur_t) + 63) / 64;
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
      if (lane == 0) {
        if (!tc::mbar_wait(&s.empty[stage], phase ^ 1, a.status, abort_flag)) *abort_flag = 1;
      }
      __syncwarp();
      if (*abort_flag) break;
      if (lane == 0) {
        int64_t p[2];
        uint32_t bytes = 0, valid = 0;
        for (int h = 0; h < 2; ++h) {
          const int lb = 2 * c.j + h;
          p[h] = -1;
          if (lb >= nblk) continue;
          p[h] = a.bt[int64_t(b) * a.max_blocks + lb];
          if (p[h] < 0 || p[h] >= a.num_blocks) { p[h] = -1; report(a.status, V4A_DEV_BAD_BLOCK); continue; }
          bytes += a.tx_per_block + a.scale_bytes;
          valid |= 1u << h;
        }
        s.valid[stage] = valid;
        tc::mbar_arrive_expect_tx(&s.full[stage], bytes);
        for (int h = 0; h < 2; ++h) {
          if (p[h] < 0) continue;
          tc::tma_load_3d(tiles + stage * kTileBytes + h * kBlockSmem, &tmap, 0, 0, int(p[h]), &s.full[stage]);
          tc::bulk_load(scl + stage * kScaleBytes + h * (kScaleBytes / 2),
                        a.pool + p[h] * a.block_bytes + a.scale_off, a.scale_bytes, &s.full[stage]);
        }
        last_phase[stage] = phase;
      }
      ++issued;
      if (++stage == kStages) { stage = 0; phase ^= 1; }
      c.next(a);
    }
    // drain: every issued copy has landed before the CTA can exit
    if (lane == 0) {
      const int nd = issued < kStages ? issued : kStages;
      for (int d = 0; d < nd; ++d) {
        stage = (stage + kStages - 1) % kStages;
        const long long t0 = clock64();
        while (!tc::mbar_try_wait(&s.full[stage], last_phase[stage]) && clock64() - t0 < 2000000000LL) {}
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      Cursor c;
      c.init(a, s.t0, s.j0);
      int cur_t = -1, qi = -1, stage = 0, acc = 0;
      uint32_t phase = 0, aphase = 0;
      const uint32_t q0 = tc::smem_u32(qbuf), t0a = tc::smem_u32(tiles);
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
        const uint64_t adesc = tc::desc_sw128(t0a + stage * kTileBytes);
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
        if (++stage == kStages) { stage = 0; phase ^= 1; }
        if (++acc == 2) { acc = 0; aphase ^= 1; }
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
    const int g = (warp - 2) >> 2;
    const int quarter = warp & 3;                // TMEM lanes 32*quarter .. +31
    const int row = quarter * 32 + lane;         // entry within the tile
    const uint32_t lane_addr = tmem + (uint32_t(quarter * 32) << 16) + g * a.acc_cols;
    Cursor c;
    c.init(a, s.t0, s.j0);
    int cur_t = -1, qi = -1, n = 0, stage = 0;
    uint32_t phase = 0, aphase = 0;
    float* srow = nullptr;
    const float* wq = nullptr;
    for (int it = 0; it < count; ++it) {
      if (c.t != cur_t) {
        if (cur_t >= 0) {
          __syncwarp();
          if (lane == 0) tc::mbar_arrive(&s.qempty[qi & 1]);   // done with the old head weights
        }
        cur_t = c.t;
        ++qi;
        n = visible_of(a, cur_t);
        srow = a.scores + int64_t(cur_t) * a.row;
        if (!__all_sync(0xffffffffu, tc::mbar_wait(&s.qfull[qi & 1], (qi >> 1) & 1, a.status, abort_flag)))
          break;
        wq = s.wq[qi & 1];
      }
      if ((it & 1) == g) {
        const int e = c.j * 128 + row;
        // the stage's scale words and validity came with its TMA copies
        bool ok = tc::mbar_wait(&s.full[stage], phase, a.status, abort_flag);
        ok = __all_sync(0xffffffffu, ok && tc::mbar_wait(&s.tfull[g], aphase, a.status, abort_flag));
        if (!ok) break;
        const bool blk_ok = (s.valid[stage] >> (row >> 6)) & 1u;
        const uint8_t* sp = scl + stage * kScaleBytes + (row >> 6) * (kScaleBytes / 2);
        float sc0, sc1 = 0.f, sc2 = 0.f, sc3 = 0.f;
        if (a.fmt == V4A_IX_FP8_B128) {
          sc0 = reinterpret_cast<const float*>(sp)[row & 63];
        } else {
          const float4 v4 = reinterpret_cast<const float4*>(sp)[row & 63];
          sc0 = v4.x; sc1 = v4.y; sc2 = v4.z; sc3 = v4.w;
        }
        __syncwarp();
        if (lane == 0) tc::mbar_arrive(&s.empty[stage]);     // scales read: stage may be refilled
        tc::tc_fence_after();
        float score;
        if (a.fmt == V4A_IX_FP8_B128) {
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
        if (e < n) srow[e] = blk_ok ? score : -INFINITY;
        aphase ^= 1;
      }
      if (++stage == kStages) { stage = 0; phase ^= 1; }
      c.next(a);
    }
  }
  tc::tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc::tc_fence_after();
    tc::tmem_dealloc(tmem, 2 * a.acc_cols);
  }
}

// ---- host side -------------------------------------------------------------------

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

int sm_count() {
  static int n = 0;
  static std::once_flag once;
  std::call_once(once, [] {
    int dev = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    if (n <= 0) n = 148;
  });
  return n;
}

}  // namespace

bool index_score_tc(const v4a_index_args* a, float* scores, int64_t row, cudaStream_t stream, int* rc) {
  *rc = V4A_OK;
  const v4a_cache& c = a->keys;
  if (c.format != V4A_IX_FP8_B128 && c.format != V4A_IX_FP4_B32) return false;
  if (a->q_format != V4A_Q_FP8_HEAD || a->num_heads != 64 || c.dim != 128) return false;
  if ((reinterpret_cast<uintptr_t>(c.pool) & 31) || (reinterpret_cast<uintptr_t>(a->q) & 15)) return false;
  auto encode = encode_fn();
  if (!encode) return false;
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
  t.q = static_cast<const uint8_t*>(a->q);
  t.qs = a->q_scale;
  t.w = a->weights;
  t.scores = scores;
  t.row = row;
  t.status = a->status;
  t.idesc = tc::make_idesc(fp4 ? 5u : 0u, 0u, 128, 64);
  // transaction bytes of one block's TMA copy: the global bytes read (for the
  // padded 4-bit type that is half of what lands in shared memory)
  t.tx_per_block = uint32_t(64 * ix_row_bytes(c.format, c.dim));

  CUtensorMap map;
  const cuuint64_t gdim[3] = {128, 64, cuuint64_t(c.num_blocks)};
  const cuuint64_t gstride[2] = {cuuint64_t(ix_row_bytes(c.format, c.dim)), cuuint64_t(t.block_bytes)};
  const cuuint32_t box[3] = {128, 64, 1};
  const cuuint32_t estride[3] = {1, 1, 1};
  CUresult r = encode(&map, fp4 ? CU_TENSOR_MAP_DATA_TYPE_16U4_ALIGN16B : CU_TENSOR_MAP_DATA_TYPE_UINT8, 3,
                      const_cast<void*>(c.pool), gdim, gstride, box, estride, CU_TENSOR_MAP_INTERLEAVE_NONE,
                      CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                      CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return false;
  const size_t smem = 1024 + size_t(kStages) * (kTileBytes + kScaleBytes) + 2 * kQBytes + sizeof(Smem);
  static std::once_flag attr_once;
  std::call_once(attr_once, [smem] {
    cudaFuncSetAttribute(index_scan_tc, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem));
  });
  index_scan_tc<<<sm_count(), kThreads, smem, stream>>>(t, map);
  if (cudaGetLastError() != cudaSuccess) { *rc = V4A_ERR_CUDA; return true; }
  return true;
}

}  // namespace v4a
