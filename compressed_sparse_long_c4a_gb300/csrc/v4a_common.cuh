// Device helpers shared by the libv4a kernels: bf16/e4m3/e2m1 conversions,
// rotary angles, slot mapping, status reporting and block reductions.
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <cuda_fp8.h>
#include <cuda_fp4.h>
#include <stdint.h>

#include <cmath>

#include "v4a.h"

namespace v4a {

constexpr int kBlockPositions = 256;   // one logical block = 256 native positions

__device__ __forceinline__ void report(int32_t* status, int bits) {
  if (status) atomicOr(status, bits);
}

// ---- programmatic dependent launch -----------------------------------------------
// A kernel launched with launch_pdl may start while the kernel before it on the
// stream is still running.  Every CTA of such a kernel calls pdl_wait() before
// it reads anything an earlier kernel writes (or writes anything an earlier
// kernel reads); pdl_wait returns once the earlier kernel has completed and its
// writes are visible.  pdl_trigger() lets the next such kernel be scheduled.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                              cudaStream_t stream, Args... args) {
  cudaLaunchConfig_t lc = {};
  lc.gridDim = grid;
  lc.blockDim = block;
  lc.dynamicSmemBytes = smem;
  lc.stream = stream;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[0].val.programmaticStreamSerializationAllowed = 1;
  lc.attrs = at;
  lc.numAttrs = 1;
  return cudaLaunchKernelEx(&lc, kernel, static_cast<KArgs>(args)...);
}

// ---- bf16 -------------------------------------------------------------------
__device__ __forceinline__ float bf16_to_f32(uint16_t b) {
  return __uint_as_float(static_cast<uint32_t>(b) << 16);
}
__device__ __forceinline__ uint16_t f32_to_bf16(float f) {
  __nv_bfloat16 h = __float2bfloat16_rn(f);
  return *reinterpret_cast<uint16_t*>(&h);
}

// ---- fp8 e4m3 ------------------------------------------------------------------
__device__ __forceinline__ float e4m3_to_f32(uint8_t c) {
  __half_raw h = __nv_cvt_fp8_to_halfraw(static_cast<__nv_fp8_storage_t>(c), __NV_E4M3);
  return __half2float(__half(h));
}
__device__ __forceinline__ uint8_t f32_to_e4m3(float f) {
  return static_cast<uint8_t>(__nv_cvt_float_to_fp8(f, __NV_SATFINITE, __NV_E4M3));
}

// ---- fp4 e2m1 ------------------------------------------------------------------
// Magnitudes of the OCP e2m1 codes 0..7 (sign in bit 3).
__device__ __forceinline__ float e2m1_to_f32(uint32_t nib) {
  const float mag[8] = {0.f, 0.5f, 1.f, 1.5f, 2.f, 3.f, 4.f, 6.f};
  float v = mag[nib & 7u];
  return (nib & 8u) ? -v : v;
}
__device__ __forceinline__ uint32_t f32_to_e2m1(float f) {
  return static_cast<uint32_t>(__nv_cvt_float_to_fp4(f, __NV_E2M1, cudaRoundNearest)) & 0xFu;
}

// ---- rotary angles ------------------------------------------------------------
// angle_j = pos * theta^(-2j/R).  inv_freq_j = theta^(-2j/R) is computed on the
// host in fp64; the angle is formed and reduced to [-pi, pi] in fp64 on the
// device (positions reach 1e6, where an fp32 angle would be off by ~0.06 rad)
// and only then rotated with fp32 sincosf.
struct RopeFreq {
  double inv[64];   // inv_freq_j for j < rope_dims / 2 (rope_dims <= 128)
};

inline RopeFreq make_rope_freq(int rope_dims, float theta) {
  RopeFreq f{};
  for (int j = 0; j < rope_dims / 2 && j < 64; ++j)
    f.inv[j] = std::pow(static_cast<double>(theta), -2.0 * j / static_cast<double>(rope_dims));
  return f;
}

__device__ __forceinline__ void rope_cos_sin(int pos, double inv_freq, float* c, float* s) {
  const double ang = static_cast<double>(pos) * inv_freq;
  const double two_pi = 6.283185307179586476925286766559;
  const double red = fma(-rint(ang * (1.0 / two_pi)), two_pi, ang);
  sincosf(static_cast<float>(red), s, c);
}

// cos/sin of the R/2 angles of position `pos` into cs[0..R/2) and cs[R/2..R),
// computed by threads 0..R/2-1 of the block (the caller synchronises).
__device__ __forceinline__ void rope_table(int pos, int rope_dims, const RopeFreq& f, float* cs) {
  for (int j = threadIdx.x; j < rope_dims / 2; j += blockDim.x)
    rope_cos_sin(pos, f.inv[j], &cs[j], &cs[rope_dims / 2 + j]);
}

// ---- paged cache geometry ----------------------------------------------------
__host__ __device__ __forceinline__ int entries_per_block(int ratio) {
  return kBlockPositions / ratio;
}

constexpr int kDsv4Row = 584, kDsv4Nope = 448, kDsv4Rope = 64, kDsv4Unit = 576;

__host__ __device__ __forceinline__ int64_t kv_block_bytes(int fmt, int ratio, int dim) {
  const int64_t e = entries_per_block(ratio);
  if (fmt == V4A_KV_FP8_DSV4) return (e * kDsv4Row + kDsv4Unit - 1) / kDsv4Unit * kDsv4Unit;
  return fmt == V4A_KV_BF16 ? e * dim * 2 : e * (dim + 4);
}

__host__ __device__ __forceinline__ int64_t kv_row_bytes(int fmt, int dim) {
  if (fmt == V4A_KV_FP8_DSV4) return kDsv4Row;
  return fmt == V4A_KV_BF16 ? int64_t(dim) * 2 : int64_t(dim);
}

__host__ __device__ __forceinline__ bool ix_is_fp4(int fmt) {
  return fmt == V4A_IX_FP4_B32 || fmt == V4A_IX_FP4_MX32;
}

__host__ __device__ __forceinline__ int64_t ix_row_bytes(int fmt, int dim) {
  return fmt == V4A_IX_BF16 ? int64_t(dim) * 2 : (fmt == V4A_IX_FP8_B128 ? dim : dim / 2);
}

__host__ __device__ __forceinline__ int ix_scales_per_row(int fmt, int dim) {
  return fmt == V4A_IX_FP8_B128 ? dim / 128 : (ix_is_fp4(fmt) ? dim / 32 : 0);
}

__host__ __device__ __forceinline__ int64_t ix_block_bytes(int fmt, int dim) {
  return 64 * (ix_row_bytes(fmt, dim) + 4 * ix_scales_per_row(fmt, dim));
}

// Physical block of logical entry i, or -1 (and a status bit) if unusable.
__device__ __forceinline__ int64_t block_of(const v4a_cache& c, int seq, int i,
                                            int32_t* status) {
  const int e = entries_per_block(c.ratio);
  const int lb = i / e;
  if (lb >= c.max_blocks) { report(status, V4A_DEV_BAD_BLOCK); return -1; }
  const int32_t blk = c.block_table[int64_t(seq) * c.max_blocks + lb];
  if (blk < 0 || blk >= c.num_blocks) { report(status, V4A_DEV_BAD_BLOCK); return -1; }
  return blk;
}

// ---- reductions -----------------------------------------------------------------
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}
__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

// Block-wide reduction; `red` must hold >= 32 floats.  All threads get the result.
template <bool kMax>
__device__ __forceinline__ float block_reduce(float v, float* red) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int nw = (blockDim.x + 31) >> 5;
  v = kMax ? warp_max(v) : warp_sum(v);
  __syncthreads();
  if (lane == 0) red[warp] = v;
  __syncthreads();
  float r = (lane < nw) ? red[lane] : (kMax ? -INFINITY : 0.f);
  if (warp == 0) {
    r = kMax ? warp_max(r) : warp_sum(r);
    if (lane == 0) red[0] = r;
  }
  __syncthreads();
  r = red[0];
  __syncthreads();
  return r;
}

// A ring (compressor state or sliding-window keys) as the kernels address it:
// a per-sequence buffer ([B][cap][row] plus an optional [B][cap] fp32 side
// array), or slots in pages of a shared pool (table != nullptr; the page
// holds [slots][row] then [slots] fp32).
struct RingDev {
  uint8_t* rows;          // dense rows, or the page pool
  float* side;            // dense side array (nullptr: none); unused when paged
  const int32_t* table;   // [B][cap / slots] page ids, or nullptr
  int64_t num_pages, page_bytes;
  int cap, slots, row_bytes, has_side;
};

// Addresses of slot s (0 <= s < cap) of sequence b.  A page id out of range
// reports V4A_DEV_BAD_BLOCK and gives null addresses.
__device__ __forceinline__ void ring_slot(const RingDev& r, int b, int s, uint8_t** row, float** side,
                                          int32_t* status) {
  if (!r.table) {
    const int64_t i = int64_t(b) * r.cap + s;
    *row = r.rows + i * r.row_bytes;
    *side = r.has_side ? r.side + i : nullptr;
    return;
  }
  const int q = s / r.slots, j = s - q * r.slots;
  const int32_t pg = r.table[int64_t(b) * (r.cap / r.slots) + q];
  if (pg < 0 || pg >= r.num_pages) {
    report(status, V4A_DEV_BAD_BLOCK);
    *row = nullptr;
    *side = nullptr;
    return;
  }
  uint8_t* base = r.rows + int64_t(pg) * r.page_bytes;
  *row = base + int64_t(j) * r.row_bytes;
  *side = r.has_side ? reinterpret_cast<float*>(base + int64_t(r.slots) * r.row_bytes) + j : nullptr;
}

// Fills a RingDev from a dense buffer pair or a v4a_ring_pages descriptor;
// V4A_OK or V4A_ERR_INVALID_ARG.
inline int ring_dev_fill(RingDev* r, void* rows, float* side, int cap, int row_bytes, bool has_side,
                         const v4a_ring_pages* pg) {
  *r = RingDev{};
  r->cap = cap;
  r->row_bytes = row_bytes;
  r->has_side = has_side ? 1 : 0;
  if (cap <= 0) return V4A_ERR_INVALID_ARG;
  if (!pg) {
    if (!rows || (has_side && !side)) return V4A_ERR_INVALID_ARG;
    r->rows = static_cast<uint8_t*>(rows);
    r->side = side;
    return V4A_OK;
  }
  if (!pg->pool || !pg->table || pg->num_pages <= 0 || pg->slots <= 0 || cap % pg->slots) return V4A_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(pg->pool) & 15) || (pg->page_bytes & 15)) return V4A_ERR_INVALID_ARG;
  if (pg->page_bytes < int64_t(pg->slots) * (row_bytes + (has_side ? 4 : 0))) return V4A_ERR_INVALID_ARG;
  r->rows = static_cast<uint8_t*>(pg->pool);
  r->table = pg->table;
  r->num_pages = pg->num_pages;
  r->page_bytes = pg->page_bytes;
  r->slots = pg->slots;
  return V4A_OK;
}

// The window ring of an attention call (dense or paged).
inline int attn_window_ring(const v4a_attn_args* a, RingDev* r) {
  return ring_dev_fill(r, const_cast<void*>(a->window), const_cast<float*>(a->window_scale), a->window_cap,
                       int(kv_row_bytes(a->window_format, a->kv.dim)), a->window_format == V4A_KV_FP8_TOKEN,
                       a->window_pages);
}

// Order-preserving map of a float to uint32 (larger float -> larger key).
__device__ __forceinline__ uint32_t float_key(float f) {
  uint32_t u = __float_as_uint(f);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

}  // namespace v4a
