// Host page allocator: page-size buckets with one shared pool (a free list
// of page ids) each, serving the compressed caches (one page per logical
// block of 256 native positions, per layer) and the sliding-window rings
// (a fixed set of pages per sequence and layer) of a whole model.
//
// Method: "DeepSeek V4 in vLLM: Efficient Long-context Attention", Method
// details, "keeping the KV cache memory packed" (single logical block size,
// compressor state as a sliding window, unified page sizes in three
// buckets).  The declarations and the readings are in v4a_pages.h.

#include <algorithm>
#include <climits>
#include <cstdint>
#include <memory>
#include <new>
#include <vector>

#include "v4a_pages.h"

namespace {
constexpr int64_t kBlockPositions = 256;
constexpr int64_t kMaxTableEntries = int64_t(1) << 31;
}  // namespace

struct v4a_pages {
  struct Bucket {
    int64_t page_bytes = 0;
    int64_t num_pages = 0;
    int64_t block_pages = 0;      // pages one logical block takes (BLOCK kinds x layers)
    int64_t ring_pages = 0;       // pages one open sequence's rings take
    std::vector<int32_t> free;    // free page ids; the next allocation takes the back
  };
  struct Kind {
    v4a_pages_kind k;
    v4a_pages_kind_info info;
  };
  std::vector<Bucket> buckets;
  std::vector<Kind> kinds;
  std::vector<int32_t> tables;
  std::vector<int64_t> blocks;    // per sequence: logical blocks held, -1 = not open
  int32_t max_seqs = 0, max_blocks = 0;

  int32_t* row(const Kind& k, int32_t layer, int32_t seq) {
    return tables.data() + k.info.table_offset + int64_t(layer) * k.info.table_stride +
           int64_t(seq) * k.info.table_cols;
  }
};

namespace {

int create(const v4a_pages_kind* kinds, int32_t num_kinds, int32_t max_seqs, int32_t max_blocks,
           int64_t budget_bytes, v4a_pages** out) {
  if (!kinds || num_kinds < 1 || max_seqs < 1 || max_blocks < 1 || budget_bytes < 0) return V4A_ERR_INVALID_ARG;

  // the buckets: the distinct page sizes of the compressed caches, largest first
  std::vector<int64_t> sizes;
  for (int32_t i = 0; i < num_kinds; ++i) {
    const v4a_pages_kind& k = kinds[i];
    if (k.layers < 1) return V4A_ERR_INVALID_ARG;
    if (k.kind == V4A_PAGES_BLOCK) {
      if (k.page_bytes <= 0) return V4A_ERR_INVALID_ARG;
      sizes.push_back(k.page_bytes);
    } else if (k.kind == V4A_PAGES_RING) {
      if (k.slot_bytes <= 0 || k.ring_slots < 1 || k.bucket < 0) return V4A_ERR_INVALID_ARG;
    } else {
      return V4A_ERR_INVALID_ARG;
    }
  }
  if (sizes.empty()) return V4A_ERR_INVALID_ARG;
  std::sort(sizes.begin(), sizes.end(), [](int64_t a, int64_t b) { return a > b; });
  sizes.erase(std::unique(sizes.begin(), sizes.end()), sizes.end());

  std::unique_ptr<v4a_pages> p(new (std::nothrow) v4a_pages);
  if (!p) return V4A_ERR_INVALID_ARG;
  p->max_seqs = max_seqs;
  p->max_blocks = max_blocks;
  p->buckets.resize(sizes.size());
  for (size_t b = 0; b < sizes.size(); ++b) p->buckets[b].page_bytes = sizes[b];

  int64_t offset = 0;
  int rc = V4A_OK;
  for (int32_t i = 0; i < num_kinds && rc == V4A_OK; ++i) {
    v4a_pages::Kind K{};
    K.k = kinds[i];
    v4a_pages_kind_info& info = K.info;
    if (K.k.kind == V4A_PAGES_BLOCK) {
      info.bucket = int32_t(std::find(sizes.begin(), sizes.end(), K.k.page_bytes) - sizes.begin());
      info.table_cols = max_blocks;
      p->buckets[info.bucket].block_pages += K.k.layers;
    } else {
      if (K.k.bucket >= int32_t(sizes.size())) { rc = V4A_ERR_INVALID_ARG; break; }
      const int64_t pb = sizes[K.k.bucket];
      const int64_t slots = pb / K.k.slot_bytes;
      if ((pb & 15) || slots < 1 || slots > INT32_MAX) { rc = V4A_ERR_INVALID_ARG; break; }
      const int64_t pages = (K.k.ring_slots + slots - 1) / slots;
      if (slots * pages > INT32_MAX) { rc = V4A_ERR_INVALID_ARG; break; }
      info.bucket = K.k.bucket;
      info.slots = int32_t(slots);
      info.ring_pages = int32_t(pages);
      info.ring_cap = int32_t(slots * pages);
      info.table_cols = int32_t(pages);
      p->buckets[info.bucket].ring_pages += int64_t(K.k.layers) * pages;
    }
    info.table_offset = offset;
    info.table_stride = int64_t(max_seqs) * info.table_cols;
    offset += int64_t(K.k.layers) * info.table_stride;
    if (offset > kMaxTableEntries) rc = V4A_ERR_INVALID_ARG;
    p->kinds.push_back(K);
  }
  if (rc) return rc;

  // pool sizes: the rings of max_seqs sequences, then as many logical blocks
  // (one page per BLOCK kind and layer each) as the rest of the budget holds
  int64_t ring_bytes = 0, block_bytes = 0;
  for (const auto& B : p->buckets) {
    if (B.ring_pages > 0 && int64_t(max_seqs) * B.ring_pages > INT32_MAX) return V4A_ERR_INVALID_ARG;
    ring_bytes += int64_t(max_seqs) * B.ring_pages * B.page_bytes;
    block_bytes += B.block_pages * B.page_bytes;
  }
  if (ring_bytes > budget_bytes) return V4A_ERR_OUT_OF_PAGES;
  int64_t nblk = (budget_bytes - ring_bytes) / block_bytes;
  nblk = std::min<int64_t>(nblk, int64_t(max_seqs) * max_blocks);
  for (const auto& B : p->buckets)
    if (B.block_pages > 0)
      nblk = std::min<int64_t>(nblk, (INT32_MAX - int64_t(max_seqs) * B.ring_pages) / B.block_pages);
  if (nblk < 1) return V4A_ERR_OUT_OF_PAGES;
  for (auto& B : p->buckets) {
    B.num_pages = int64_t(max_seqs) * B.ring_pages + nblk * B.block_pages;
    B.free.resize(size_t(B.num_pages));
    for (int64_t j = 0; j < B.num_pages; ++j) B.free[size_t(j)] = int32_t(B.num_pages - 1 - j);
  }
  p->tables.assign(size_t(offset), -1);
  p->blocks.assign(size_t(max_seqs), -1);
  *out = p.release();
  return V4A_OK;
}

}  // namespace

extern "C" {

// No exception leaves the C ABI: an allocation failure while planning is
// reported as V4A_ERR_INVALID_ARG with nothing created.
V4A_API int v4a_pages_create(const v4a_pages_kind* kinds, int32_t num_kinds, int32_t max_seqs,
                             int32_t max_blocks, int64_t budget_bytes, v4a_pages** out) {
  if (!out) return V4A_ERR_INVALID_ARG;
  *out = nullptr;
  try {
    return create(kinds, num_kinds, max_seqs, max_blocks, budget_bytes, out);
  } catch (...) {
    return V4A_ERR_INVALID_ARG;
  }
}

V4A_API void v4a_pages_destroy(v4a_pages* p) { delete p; }

V4A_API int32_t v4a_pages_num_buckets(const v4a_pages* p) { return p ? int32_t(p->buckets.size()) : 0; }

V4A_API int v4a_pages_bucket(const v4a_pages* p, int32_t bucket, int64_t* page_bytes, int64_t* num_pages,
                             int64_t* free_pages) {
  if (!p || bucket < 0 || bucket >= int32_t(p->buckets.size())) return V4A_ERR_INVALID_ARG;
  const auto& B = p->buckets[bucket];
  if (page_bytes) *page_bytes = B.page_bytes;
  if (num_pages) *num_pages = B.num_pages;
  if (free_pages) *free_pages = int64_t(B.free.size());
  return V4A_OK;
}

V4A_API int v4a_pages_info(const v4a_pages* p, int32_t kind, v4a_pages_kind_info* info) {
  if (!p || !info || kind < 0 || kind >= int32_t(p->kinds.size())) return V4A_ERR_INVALID_ARG;
  *info = p->kinds[kind].info;
  return V4A_OK;
}

V4A_API const int32_t* v4a_pages_tables(const v4a_pages* p, int64_t* num_entries) {
  if (!p) return nullptr;
  if (num_entries) *num_entries = int64_t(p->tables.size());
  return p->tables.data();
}

V4A_API int v4a_pages_open(v4a_pages* p, int32_t seq) {
  if (!p || seq < 0 || seq >= p->max_seqs || p->blocks[seq] >= 0) return V4A_ERR_INVALID_ARG;
  for (const auto& B : p->buckets)
    if (int64_t(B.free.size()) < B.ring_pages) return V4A_ERR_OUT_OF_PAGES;
  for (const auto& K : p->kinds) {
    if (K.k.kind != V4A_PAGES_RING) continue;
    auto& fl = p->buckets[K.info.bucket].free;
    for (int32_t l = 0; l < K.k.layers; ++l) {
      int32_t* r = p->row(K, l, seq);
      for (int32_t j = 0; j < K.info.ring_pages; ++j) {
        r[j] = fl.back();
        fl.pop_back();
      }
    }
  }
  p->blocks[seq] = 0;
  return V4A_OK;
}

V4A_API int v4a_pages_reserve(v4a_pages* p, int32_t seq, int64_t positions) {
  if (!p || seq < 0 || seq >= p->max_seqs || p->blocks[seq] < 0 || positions < 0) return V4A_ERR_INVALID_ARG;
  const int64_t need = (positions + kBlockPositions - 1) / kBlockPositions;
  if (need > p->max_blocks) return V4A_ERR_INVALID_ARG;
  const int64_t have = p->blocks[seq];
  if (need <= have) return V4A_OK;
  for (const auto& B : p->buckets)
    if (int64_t(B.free.size()) < (need - have) * B.block_pages) return V4A_ERR_OUT_OF_PAGES;
  for (int64_t lb = have; lb < need; ++lb) {
    for (const auto& K : p->kinds) {
      if (K.k.kind != V4A_PAGES_BLOCK) continue;
      auto& fl = p->buckets[K.info.bucket].free;
      for (int32_t l = 0; l < K.k.layers; ++l) {
        p->row(K, l, seq)[lb] = fl.back();
        fl.pop_back();
      }
    }
  }
  p->blocks[seq] = need;
  return V4A_OK;
}

V4A_API int v4a_pages_close(v4a_pages* p, int32_t seq) {
  if (!p || seq < 0 || seq >= p->max_seqs || p->blocks[seq] < 0) return V4A_ERR_INVALID_ARG;
  for (const auto& K : p->kinds) {
    auto& fl = p->buckets[K.info.bucket].free;
    for (int32_t l = 0; l < K.k.layers; ++l) {
      int32_t* r = p->row(K, l, seq);
      for (int32_t j = 0; j < K.info.table_cols; ++j) {
        if (r[j] >= 0) fl.push_back(r[j]);
        r[j] = -1;
      }
    }
  }
  p->blocks[seq] = -1;
  return V4A_OK;
}

V4A_API int64_t v4a_pages_blocks(const v4a_pages* p, int32_t seq) {
  if (!p || seq < 0 || seq >= p->max_seqs) return -1;
  return p->blocks[seq];
}

}  // extern "C"
