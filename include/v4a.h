/*
 * v4a.h - C ABI of libv4a, a GB300 (sm_103a) implementation of the
 * DeepSeek-V4-style compressed sparse attention layer (c4a / c128a) in
 * decode and chunked prefill.
 *
 * Source of the method: "DeepSeek V4 in vLLM: Efficient Long-context
 * Attention" (vLLM blog, April 2026), sections Background (shared K=V,
 * compression, sparse attention, sliding window), Method details (single
 * logical block size, compressor state as a sliding window, kernel fusions)
 * and Appendix (inverse RoPE, exact position ranges and causality, values of
 * k, why the short window).  Byte layouts of the fp8 indexer entry follow the
 * SGLang KV-pool article, section "DSA", and the DeepSeek-V4 584-byte cache
 * row its section "DeepSeek-V4".  The host page allocator (page-size
 * buckets) is declared in v4a_pages.h.
 *
 * General rules for every entry point:
 *  - All pointers inside the argument structs are DEVICE pointers unless a
 *    field says otherwise; the structs themselves live in host memory and are
 *    read only during the call.
 *  - The caller owns and allocates every buffer (caches, rings, block tables,
 *    inputs, outputs, workspace).  The library never allocates or frees device
 *    memory, never synchronises, and launches only on the given stream
 *    (a cudaStream_t passed as void*; NULL = legacy default stream).
 *  - Calls are ordered by the stream: compress_insert -> index_topk ->
 *    sparse_attn -> inv_rope_quant.
 *  - A nonzero return code means nothing was launched, except V4A_ERR_CUDA,
 *    which reports a launch failure.  Problems that only the device can see
 *    (an unallocated block, a bad index) are OR-ed into the optional device
 *    word `status` as V4A_DEV_* bits; the offending read or write is skipped.
 *    No kernel traps and no kernel waits on another.
 *  - bf16 tensors are passed as uint16_t bit patterns; fp8 is OCP e4m3fn,
 *    fp4 is OCP e2m1 (element 2j in the low nibble of byte j).
 *  - Rows are read and written in element pairs: bf16 row pointers must be
 *    4-byte aligned, e4m3 rows written by the compressor launch 2-byte
 *    aligned, fp32 pairs (the query norm's gamma) 8-byte aligned; pools,
 *    rings and tables should start on 16 bytes (the tensor-core paths need
 *    it and take another path or return V4A_ERR_UNSUPPORTED otherwise).
 *    v4a_compress_insert returns V4A_ERR_INVALID_ARG for a misaligned input
 *    or output row pointer.
 */
#ifndef V4A_H
#define V4A_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define V4A_ABI_VERSION 5

#if defined(__GNUC__)
#define V4A_API __attribute__((visibility("default")))
#else
#define V4A_API
#endif

/* ---- host return codes ---------------------------------------------------- */
#define V4A_OK                 0
#define V4A_ERR_INVALID_ARG    1  /* null pointer, bad size, bad enum */
#define V4A_ERR_UNSUPPORTED    2  /* valid but not implemented (dim, heads, format pairing) */
#define V4A_ERR_RING_TOO_SMALL 3  /* ring capacity < window - 1 + max_new_per_seq */
#define V4A_ERR_WORKSPACE      4  /* workspace missing or smaller than *_workspace_size */
#define V4A_ERR_CUDA           5  /* a kernel launch failed */
#define V4A_ERR_OUT_OF_PAGES   6  /* page allocator (v4a_pages.h): a bucket has too few free pages */

/* ---- device status bits (OR-ed into *status when status != NULL) ---------- */
#define V4A_DEV_BAD_BLOCK  1  /* a needed block-table entry is < 0 or >= num_blocks */
#define V4A_DEV_BAD_BATCH  2  /* seq id out of range, positions not consecutive in a
                                 sequence's run, or a run longer than max_new_per_seq */
#define V4A_DEV_BAD_INDEX  4  /* a selected entry index is >= the visible count */
#define V4A_DEV_TIMEOUT    8  /* a bounded wait inside a tensor-core kernel gave up; that call's
                                 outputs are incomplete (never expected; reported, never hung) */

/* ---- formats ---------------------------------------------------------------- */
/* Shared-K=V cache and window ring rows. */
#define V4A_KV_BF16       0  /* row = dim bf16 */
#define V4A_KV_FP8_TOKEN  1  /* row = dim e4m3 codes; one fp32 scale per row (amax/448) */
#define V4A_KV_FP8_DSV4   2  /* compressed cache only, dim 512 with 64 rope dims: the DeepSeek-V4
                                row of the SGLang KV-pool article ("DeepSeek-V4"), 584 B =
                                448 e4m3 codes of the non-rope dims, the 64 rope dims in bf16,
                                7 UE8M0 scale bytes (one per 64 codes: the smallest power of
                                two s with amax/s <= 448; value = code * 2^(byte-127)), 1 zero
                                pad byte; the scales live inside the row */
/* Indexer key cache rows. */
#define V4A_IX_BF16       0  /* row = dim bf16 */
#define V4A_IX_FP8_B128   1  /* row = dim e4m3; one fp32 scale per 128 elements (132 B at dim 128) */
#define V4A_IX_FP4_B32    2  /* row = dim/2 bytes e2m1; one fp32 scale per 32 elements */
#define V4A_IX_FP4_MX32   3  /* the V4A_IX_FP4_B32 bytes with every scale a power of two, chosen by the
                                OCP Microscaling (MX) rule 2^(floor(log2 amax) - 2); the tensor cores
                                then apply the scales inside the MMA.  A scale word that is not a
                                power of two is read as its power-of-two part by the tensor-core
                                scan (its mantissa bits are ignored). */
/* Indexer query. */
#define V4A_Q_BF16        0  /* [T][H_I][dim] bf16 */
#define V4A_Q_FP8_HEAD    1  /* [T][H_I][dim] e4m3 + [T][H_I] fp32 scale */
/* Output of the inverse-RoPE stage. */
#define V4A_OUT_BF16      0
#define V4A_OUT_FP8_TOKEN 1  /* e4m3 codes + one fp32 scale per token over H*dim (amax/448) */

/*
 * Ragged batch of new tokens.  Token t belongs to sequence seq_ids[t] and sits
 * at absolute 0-based position positions[t].  The tokens of one sequence are
 * contiguous in t and at consecutive increasing positions.  In decode each
 * sequence has one token; in chunked prefill a sequence has up to
 * max_new_per_seq tokens.  The same tokens are the queries of the step.
 */
typedef struct {
  int32_t num_tokens;          /* T >= 0 */
  const int32_t* seq_ids;      /* [T], each in [0, num_seqs) */
  const int32_t* positions;    /* [T] */
  int32_t num_seqs;            /* B: rows of every block table and ring */
  int32_t max_new_per_seq;     /* host-side bound on one sequence's tokens in this call */
} v4a_batch;

/*
 * A paged compressed cache ("a single logical block size": every physical
 * block covers 256 native positions, i.e. 256/ratio entries).  Entry i of
 * sequence b lives in physical block block_table[b][i / E], slot i % E, with
 * E = 256/ratio.  Inside a block all data rows come first ([E][row bytes]),
 * then the fp32 scale words ([E][scales per row]) if the format has any.
 * Block bytes:  KV_BF16 E*dim*2;  KV_FP8_TOKEN E*(dim+4);
 *               KV_FP8_DSV4 ceil(E*584/576)*576 (rows from the block's first
 *               byte, the page padded to 576-byte units as in the article);
 *               IX_BF16 64*dim*2;  IX_FP8_B128 64*(dim + 4*dim/128);
 *               IX_FP4_B32, IX_FP4_MX32 64*(dim/2 + 4*dim/32).
 */
typedef struct {
  int32_t ratio;               /* 4 (c4a) or 128 (c128a); indexer caches use 4 */
  int32_t dim;                 /* row length in elements */
  int32_t rope_dims;           /* the last rope_dims dims are rotated (interleaved pairs) */
  float rope_theta;            /* base of the rotary frequencies */
  int32_t format;              /* V4A_KV_* or V4A_IX_* */
  void* pool;                  /* num_blocks * block bytes */
  int64_t num_blocks;
  const int32_t* block_table;  /* [num_seqs][max_blocks]; -1 = unallocated */
  int32_t max_blocks;
} v4a_cache;

/*
 * A ring kept in pages of a shared pool instead of a per-sequence buffer
 * (vLLM page, Method details, "compressor state as a sliding window": the
 * rolling compressor residual, like the sliding-window keys, is registered as
 * sliding-window KV and lives in the same page pools as the compressed
 * caches).  Slot s (0 <= s < ring_cap) of sequence b lives in page
 * table[b][s / slots] at index s % slots.  Inside a page the rows come first
 * ([slots][row bytes]: the bf16 x of a compressor ring, the key row of a
 * window ring), then one fp32 per slot (the compressor's gate, the fp8
 * window's scale; absent for a bf16 window).  A page id outside
 * [0, num_pages) sets V4A_DEV_BAD_BLOCK and the slot is skipped.
 */
typedef struct {
  void* pool;                  /* page pool base; 16-byte aligned */
  int64_t num_pages;
  int64_t page_bytes;          /* page stride: a multiple of 16, >= slots * row bytes, plus
                                  slots * 4 when the ring keeps an fp32 per slot */
  const int32_t* table;        /* [num_seqs][ring_cap / slots] page ids */
  int32_t slots;               /* slots per page; ring_cap must be a multiple of it */
} v4a_ring_pages;

/*
 * One compressor (the main KV compressor or the indexer's own).  For token t
 * at position P with (P+1) % ratio == 0 it emits entry i = (P+1)/ratio - 1 over
 * the native positions [4i-4, 4i+3] (c4a; positions < 0 take no weight) or
 * [128i, 128i+127] (c128a):  w = softmax_j(gate[p_j] + bias[j]),
 * c = sum_j w_j x[p_j], c <- c / sqrt(mean(c^2) + eps) * gamma, RoPE at the
 * anchor P, encode, store at the entry's slot.  Every new token's (x, gate) is
 * also stored in the ring at slot P % ring_cap; positions older than the
 * call's first token of that sequence are read from the ring.
 */
typedef struct {
  v4a_cache cache;             /* destination */
  const uint16_t* x;           /* [T][cache.dim] bf16 */
  const float* gate;           /* [T] */
  const float* bias;           /* [8] (c4a) or [128] (c128a) */
  const float* gamma;          /* [cache.dim] */
  float eps;                   /* RMSNorm epsilon (1e-6) */
  uint16_t* ring_x;            /* [num_seqs][ring_cap][cache.dim] bf16 (NULL with ring_pages) */
  float* ring_gate;            /* [num_seqs][ring_cap] (NULL with ring_pages) */
  int32_t ring_cap;            /* >= window - 1 + max_new_per_seq (window 8 or 128) */
  const v4a_ring_pages* ring_pages; /* host pointer or NULL.  Non-NULL: the ring lives in
                                       these pages and ring_x / ring_gate are not read */
} v4a_compressor;

/* Uncompressed sliding-window keys: k[t] rotated at P, encoded, stored at
 * ring[seq][P % ring_cap]. */
typedef struct {
  const uint16_t* k;           /* [T][dim] bf16 (normalised upstream) */
  int32_t dim, rope_dims;
  float rope_theta;
  int32_t format;              /* V4A_KV_BF16 or V4A_KV_FP8_TOKEN */
  void* ring;                  /* [num_seqs][ring_cap][dim] bf16 or e4m3 (NULL with ring_pages) */
  float* ring_scale;           /* [num_seqs][ring_cap] (fp8 only; NULL with ring_pages) */
  int32_t ring_cap;            /* >= window_len - 1 + max_new_per_seq, else V4A_ERR_RING_TOO_SMALL */
  int32_t window_len;          /* the sliding window the ring serves (128); >= 1 */
  const v4a_ring_pages* ring_pages; /* host pointer or NULL.  Non-NULL: the ring lives in
                                       these pages and ring / ring_scale are not read */
} v4a_window;

/*
 * The queries' elementwise work before attention (vLLM page, Method details,
 * fusion (3): the Q norm, fused horizontally with the window keys' RoPE +
 * insert, one warp per query head or key head).  For token t at position P
 * and head h:  q_out[t][h] = RoPE_P(q_in[t][h] / sqrt(mean(q_in[t][h]^2) + eps)
 * * gamma), the rotation on the last rope_dims dims (interleaved pairs) as for
 * the keys.  q_out is what v4a_sparse_attn takes as its already rotated q.
 */
typedef struct {
  const uint16_t* q_in;        /* [T][H][dim] bf16 */
  uint16_t* q_out;             /* [T][H][dim] bf16; may equal q_in (in place) */
  const float* gamma;          /* [dim] RMSNorm weight, shared by the heads */
  float eps;                   /* RMSNorm epsilon (1e-6) */
  int32_t num_heads;           /* H >= 1 */
  int32_t dim;                 /* a multiple of 64, <= 1024 */
  int32_t rope_dims;           /* even, <= min(dim, 128) */
  float rope_theta;
} v4a_query;

/*
 * The indexer query's preparation (vLLM page, Method details: the reused
 * DeepSeek-V3.2 fusion of Q RoPE, quantisation and the weight
 * multiplication), one warp per indexer head.  For token t at position P
 * and head h: v = RoPE_P(q_in[t][h]) on the last rope_dims dims (interleaved
 * pairs), q_scale[t][h] = amax|v| / 448 (1 when 0), q_out[t][h] =
 * e4m3(v / q_scale[t][h]), w_out[t][h] = w_in[t][h] * w_mult.  The outputs
 * are the V4A_Q_FP8_HEAD query, its scales and the head weights that
 * v4a_index_topk takes.
 */
typedef struct {
  const uint16_t* q_in;        /* [T][H_I][dim] bf16 */
  uint8_t* q_out;              /* [T][H_I][dim] e4m3 */
  float* q_scale;              /* [T][H_I] */
  const float* w_in;           /* [T][H_I] */
  float* w_out;                /* [T][H_I]; may equal w_in */
  float w_mult;
  int32_t num_heads;           /* H_I >= 1 */
  int32_t dim;                 /* a multiple of 64, <= 1024 */
  int32_t rope_dims;           /* even, <= min(dim, 128) */
  float rope_theta;
} v4a_index_query;

typedef struct {
  v4a_batch batch;
  const v4a_compressor* main;     /* host pointer; may be NULL */
  const v4a_compressor* indexer;  /* host pointer; may be NULL (c128a layers) */
  const v4a_window* window;       /* host pointer; may be NULL */
  int32_t* status;                /* optional device word */
  const v4a_query* query;         /* host pointer; may be NULL */
  const v4a_index_query* index_query; /* host pointer; may be NULL */
} v4a_compress_args;

/*
 * Fused compressor + RMSNorm + RoPE + cache insert for the main and indexer
 * caches, and the queries' norm + RoPE beside the window keys' RoPE + insert
 * (vLLM page, Method details, fusions (1) and (3); appendix "exact position
 * ranges and causality"), and the indexer query's RoPE + fp8 + weights.
 * One launch: one CTA per token for each compressor and for the window key,
 * then warps that each take one query head or one indexer-query head.
 * Returns V4A_ERR_RING_TOO_SMALL when a ring cannot hold the call's tokens
 * without overwriting positions a window still reads.
 */
V4A_API int v4a_compress_insert(const v4a_compress_args* args, void* stream);

/*
 * Indexer scoring and top-k (vLLM page, Background "DeepSeek Sparse
 * Attention"; appendix "values of k").  For query t at position m:
 *   score_i = sum_h weights[t][h] * ReLU(q_h . key_i),  i < (m+1)/4,
 * with q_h = q[t][h] (* q_scale[t][h] for fp8) and key_i the decoded indexer
 * entry.  out_idx[t] receives the k entries with the largest scores (ties to
 * the lower index) in ascending order, padded with -1 when fewer than k are
 * visible.
 */
typedef struct {
  v4a_batch batch;
  v4a_cache keys;              /* indexer cache, ratio 4 */
  int32_t num_heads;           /* H_I */
  int32_t q_format;            /* V4A_Q_BF16 (with IX_BF16 keys) or V4A_Q_FP8_HEAD */
  const void* q;               /* [T][H_I][keys.dim] */
  const float* q_scale;        /* [T][H_I] (fp8 query only) */
  const float* weights;        /* [T][H_I] */
  int32_t k;                   /* 1 <= k <= 16384; V4A_ERR_UNSUPPORTED when a block-table row
                                  addresses more than 2^20 entries (keys.max_blocks * 64) */
  int32_t* out_idx;            /* [T][k] */
  int32_t* status;
} v4a_index_args;

/* Bytes of device workspace v4a_index_topk / _scores / _select need (0 on a bad
 * shape).  The workspace holds the scores of every visible entry of every
 * query plus selection scratch; it is only read and written by these calls. */
V4A_API size_t v4a_index_workspace_size(const v4a_index_args* args);
V4A_API int v4a_index_topk(const v4a_index_args* args, void* workspace, size_t workspace_bytes,
                   void* stream);
/* v4a_index_topk in two launches-groups on the same stream: _scores writes
 * every visible entry's score into the workspace, _select reads them and
 * writes out_idx.  Calling _scores then _select with the same arguments and
 * workspace is exactly v4a_index_topk. */
V4A_API int v4a_index_scores(const v4a_index_args* args, void* workspace, size_t workspace_bytes,
                     void* stream);
/* Where v4a_index_scores leaves the scores: query t's score of entry i is the
 * float at byte offset (*offset + 4 * (t * *row_stride + i)) of the workspace,
 * for i < the query's visible count. */
V4A_API int v4a_index_scores_layout(const v4a_index_args* args, size_t* offset, int64_t* row_stride);
V4A_API int v4a_index_select(const v4a_index_args* args, void* workspace, size_t workspace_bytes,
                     void* stream);

/* v4a_index_topk without a workspace argument.  The method itself has no
 * counterpart: this variant exists for callers that may not allocate device
 * memory on the step path (a serving loop that gave all free HBM to the paged
 * KV pool at start-up; a binding with no device allocator of its own).
 *
 * Scratch is one fixed array of V4A_INDEX_STATIC_SCRATCH_BYTES inside this
 * library's device image (device memory it holds once its device code is
 * loaded on a device); the call allocates and frees nothing.  Returns
 * V4A_ERR_WORKSPACE, launching nothing, when the arguments need more than that
 * (v4a_index_workspace_size(args) > V4A_INDEX_STATIC_SCRATCH_BYTES; the
 * scratch is 4 bytes per entry a query's block-table row can address plus
 * 16 KB per query, so 16 MiB holds 15 queries over 262,144 entries each);
 * otherwise it returns exactly what v4a_index_topk would with a workspace of
 * that size, and writes the same out_idx.
 *
 * Every call looks up the array's address on the current device
 * (cudaGetSymbolAddress; V4A_ERR_CUDA if that fails; nothing is cached, so a
 * device reset between calls is harmless).  The first call on a device may
 * load this library's device code: make it before any stream capture starts.
 * All calls on a device share the array, so calls that may be in flight at the
 * same time (other streams or host threads, unordered) race and must be
 * ordered by the caller.  The part of the scratch that must start at zero
 * (histograms and counters) is cleared by every call on its own stream. */
#define V4A_INDEX_STATIC_SCRATCH_BYTES (16u << 20)
V4A_API int v4a_index_topk_static(const v4a_index_args* args, void* stream);

/*
 * Sparse attention with shared K=V (vLLM page, Background and appendix "why
 * inverse RoPE").  For query t at position m and head h, over the keys
 *   S = {selected compressed entries} U {window tokens max(0,m-W+1) .. m}:
 *   z_n = softmax_scale * q_h . k_n,  o_h = sum_n softmax(z)_n k_n.
 * idx == NULL selects every visible entry i < (m+1)/ratio (c128a layers).
 * Entries of idx that are -1 are skipped.  idx != NULL with k == 0 selects no
 * compressed entry: the window alone (the pages' pure sliding-window layers;
 * idx is then not read, and the kv cache fields must still pass the shape
 * checks but no entry of it is read).  out is bf16; lse (optional) is the
 * natural-log sum of exp(z) per (t, h).
 */
typedef struct {
  v4a_batch batch;
  v4a_cache kv;                /* main compressed cache */
  const int32_t* idx;          /* [T][k] or NULL */
  int32_t k;                   /* 1..65536 with idx; 0 with a non-NULL idx: window only */
  const void* window;          /* [num_seqs][window_cap][row bytes]; unread with window_pages */
  const float* window_scale;   /* [num_seqs][window_cap] (fp8 window only); unread with window_pages */
  int32_t window_cap;          /* >= window_len - 1 + max_new_per_seq, else V4A_ERR_RING_TOO_SMALL */
  int32_t window_format;       /* V4A_KV_* */
  int32_t window_len;          /* 128 */
  int32_t num_heads;           /* H */
  const uint16_t* q;           /* [T][H][kv.dim] bf16, already rotated */
  float softmax_scale;         /* 1/sqrt(dim) */
  uint16_t* out;               /* [T][H][kv.dim] bf16 */
  float* lse;                  /* [T][H] or NULL */
  int32_t* status;
  const v4a_ring_pages* window_pages; /* host pointer or NULL.  Non-NULL: the window ring
                                         lives in these pages (window / window_scale unread) */
} v4a_attn_args;

/* Bytes of device workspace v4a_sparse_attn needs: the per-chunk results of
 * the queries of one launch (long batches such as chunked prefill run as
 * several launches that reuse it, in stream order); 0 on a bad shape.
 * Caller-owned; its contents need no initialisation. */
V4A_API size_t v4a_attn_workspace_size(const v4a_attn_args* args);
V4A_API int v4a_sparse_attn(const v4a_attn_args* args, void* workspace, size_t workspace_bytes,
                    void* stream);

/*
 * Inverse RoPE on the attention output, fused with fp8 quantisation (vLLM
 * page, Method details, fusion (2); appendix "why inverse RoPE"):
 * out[t][h] = R_{-m} in[t][h] on the last rope_dims dims, m = positions[t];
 * for V4A_OUT_FP8_TOKEN one scale per token, amax over all heads and dims / 448.
 */
typedef struct {
  int32_t num_tokens;
  const int32_t* positions;    /* [T] */
  int32_t num_heads, dim, rope_dims;
  float rope_theta;
  const uint16_t* in;          /* [T][H][dim] bf16 */
  int32_t out_format;          /* V4A_OUT_* */
  void* out;                   /* [T][H][dim] bf16 or e4m3 */
  float* out_scale;            /* [T] (fp8 only) */
} v4a_output_args;

V4A_API int v4a_inv_rope_quant(const v4a_output_args* args, void* stream);

/*
 * v4a_sparse_attn followed by v4a_inv_rope_quant, as one call whose bf16
 * attention output never goes to memory.  Same passages as the two calls,
 * with the pages' fusion (2) ("DeepSeek V4 in vLLM: Efficient Long-context
 * Attention", Method details) extended to the merge of the attention's key
 * chunks: the chunk results are merged (with each row's amax after the
 * inverse rotation) by one kernel and inverse-rotated and encoded by the
 * next, the merged rows staying in the workspace.  The bytes of `out` and
 * `out_scale` equal those of the two calls.
 *
 *   attn: as for v4a_sparse_attn; attn->out and attn->lse are not written and
 *         may be NULL.
 *   out:  as for v4a_inv_rope_quant; out->in is not read and may be NULL.
 *         num_tokens, num_heads and dim must equal the attention's, and
 *         out->positions must hold the same positions as attn->batch.
 *   workspace: at least v4a_attn_workspace_size(attn) bytes (caller-owned).
 * Errors: as for the two calls; V4A_ERR_UNSUPPORTED (nothing launched) when
 * the shapes are outside the fused path (the tensor-core attention must take
 * them), in which case the two calls serve.
 */
V4A_API int v4a_sparse_attn_out(const v4a_attn_args* attn, const v4a_output_args* out, void* workspace,
                                size_t workspace_bytes, void* stream);

/* Human-readable text of a V4A_* return code. */
V4A_API const char* v4a_status_string(int code);
V4A_API int v4a_abi_version(void);

#ifdef __cplusplus
}
#endif
#endif /* V4A_H */
