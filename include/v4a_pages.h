/*
 * v4a_pages.h - host page allocator of libv4a: every layer's compressed
 * caches, sliding-window rings and compressor states in a few page-size
 * buckets, one shared page pool per bucket.
 *
 * Source: "DeepSeek V4 in vLLM: Efficient Long-context Attention", Method
 * details, "keeping the KV cache memory packed":
 *  (1) one logical block = 256 native positions in every layer, so a c4a
 *      block holds 64 entries and a c128a block 2; allocating a block for a
 *      sequence reserves its next 256 positions in all layers at once;
 *  (2) the compressor state (and the sliding-window keys) is sliding-window
 *      state: a fixed number of pages per sequence, advanced as decoding
 *      goes on, in the same pools as the caches;
 *  (3) page bytes = entries per block x bytes per entry; the caches are
 *      folded into a few page sizes ("buckets"), each backed by one pool that
 *      is sized once at load, so that an allocation is a lookup in the
 *      kind's bucket, with no repartitioning and no per-kind pools.  For
 *      DeepSeek-V4 the five cache kinds fold into three buckets: c4a KV, SWA
 *      KV and both compressor states in the largest; the indexer KV and the
 *      indexer's compressor state in the middle one; c128a KV in the
 *      smallest.
 *
 * Readings: the pages do not give the per-entry sizes of the compressor
 * states nor how the block size of a sliding-window kind is chosen.  Here a
 * compressed cache ("BLOCK" kind) has the page size of its 256-position block
 * (v4a_cache rules), the buckets are the distinct BLOCK page sizes, and a
 * sliding-window kind ("RING" kind) joins the bucket the caller names by
 * rank (0 = largest page), holding floor(page bytes / slot bytes) ring slots
 * per page.  A RING kind's slot layout is that of v4a_ring_pages (v4a.h).
 *
 * The allocator is host bookkeeping only: the caller allocates the device
 * pools (v4a_pages_bucket gives their sizes) and copies the block tables
 * (v4a_pages_tables, one host array holding every table) to the device
 * whenever they change.  Not thread-safe: one thread, or a lock around it.
 */
#ifndef V4A_PAGES_H
#define V4A_PAGES_H

#include <stdint.h>

#include "v4a.h"

#ifdef __cplusplus
extern "C" {
#endif

#define V4A_PAGES_BLOCK 0   /* a compressed cache: one page per 256-position logical block */
#define V4A_PAGES_RING  1   /* a sliding-window ring: a fixed set of pages per sequence */

typedef struct {
  int32_t kind;         /* V4A_PAGES_BLOCK or V4A_PAGES_RING */
  int32_t layers;       /* >= 1: layers holding one cache of this kind each */
  int64_t page_bytes;   /* BLOCK: bytes of the cache's 256-position block (> 0) */
  int64_t slot_bytes;   /* RING: bytes of one slot, row plus its fp32 side value (> 0) */
  int32_t ring_slots;   /* RING: slots the ring must hold (window - 1 + new tokens per call) */
  int32_t bucket;       /* RING: rank of the bucket it joins, 0 = largest page; the
                           bucket's page bytes must be a multiple of 16 */
} v4a_pages_kind;

typedef struct {
  int32_t bucket;       /* the bucket holding this kind's pages */
  int32_t slots;        /* RING: slots per page (0 for BLOCK) */
  int32_t ring_pages;   /* RING: pages per ring (0 for BLOCK) */
  int32_t ring_cap;     /* RING: slots * ring_pages >= ring_slots (0 for BLOCK) */
  int32_t table_cols;   /* BLOCK: max_blocks; RING: ring_pages */
  int64_t table_offset; /* int32 elements from the start of v4a_pages_tables to the
                           table [max_seqs][table_cols] of the kind's layer 0 */
  int64_t table_stride; /* int32 elements between consecutive layers' tables */
} v4a_pages_kind_info;

typedef struct v4a_pages v4a_pages;  /* opaque */

/*
 * Plans the buckets and sizes the pools once.  RING kinds take
 * max_seqs * layers * ring_pages pages of their bucket; what budget_bytes
 * leaves is divided into logical blocks (each needs one page per BLOCK kind
 * and layer), at most max_seqs * max_blocks of them.  Every table entry
 * starts at -1.  Errors: V4A_ERR_INVALID_ARG (a bad kind, a RING kind that
 * names no bucket, fits no slot in a page or joins a bucket whose page is
 * not a multiple of 16 bytes, no BLOCK kind, max_seqs or max_blocks < 1, a
 * page count beyond 2^31 - 1), V4A_ERR_OUT_OF_PAGES (the budget holds the
 * rings of max_seqs sequences plus less than one logical block).
 */
V4A_API int v4a_pages_create(const v4a_pages_kind* kinds, int32_t num_kinds, int32_t max_seqs,
                             int32_t max_blocks, int64_t budget_bytes, v4a_pages** out);
V4A_API void v4a_pages_destroy(v4a_pages* p);

V4A_API int32_t v4a_pages_num_buckets(const v4a_pages* p);
/* Page bytes, page count and free pages of a bucket (buckets by decreasing page size). */
V4A_API int v4a_pages_bucket(const v4a_pages* p, int32_t bucket, int64_t* page_bytes, int64_t* num_pages,
                             int64_t* free_pages);
V4A_API int v4a_pages_info(const v4a_pages* p, int32_t kind, v4a_pages_kind_info* info);
/* Every table in one host array of *num_entries int32 (owned by the allocator). */
V4A_API const int32_t* v4a_pages_tables(const v4a_pages* p, int64_t* num_entries);

/* Calls that allocate return V4A_ERR_OUT_OF_PAGES (defined in v4a.h) when a
 * bucket has too few free pages, and then allocate nothing. */

/* Starts sequence seq: the pages of every RING kind's ring in every layer. */
V4A_API int v4a_pages_open(v4a_pages* p, int32_t seq);
/* Grows an open sequence's blocks to cover native positions [0, positions):
 * ceil(positions / 256) logical blocks, each one page per BLOCK kind and
 * layer.  Never shrinks.  V4A_ERR_INVALID_ARG beyond max_blocks. */
V4A_API int v4a_pages_reserve(v4a_pages* p, int32_t seq, int64_t positions);
/* Ends a sequence: every page it holds goes back to its bucket. */
V4A_API int v4a_pages_close(v4a_pages* p, int32_t seq);
/* Logical blocks an open sequence holds (-1 when it is not open). */
V4A_API int64_t v4a_pages_blocks(const v4a_pages* p, int32_t seq);

#ifdef __cplusplus
}
#endif
#endif /* V4A_PAGES_H */
