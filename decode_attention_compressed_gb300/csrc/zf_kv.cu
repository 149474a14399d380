// zf_kv: host-side page manager for the compressed paged caches (ZipFusion §III.D, KV Cache
// Management and Scheduling; §II.C, Compression for Higher Serving Capacity).
//
// What the pages fix, restated for this library's cache layout:
//  * a page stays uncompressed while it fills, so that tokens can be appended to it in place; a
//    full page is compressed afterwards and keeps its page id;
//  * new pages must accept writes before they are compressed, so capacity for new pages is
//    counted in uncompressed storage, and it grows back as compression releases that storage;
//  * one logical page needs storage in every layer.
// Here a page id names one compressed slot in every layer's cache.  Uncompressed pages live in
// raw slots drawn from one pool that all layers share (every layer's cache points at the same raw
// arrays): a page being written holds one raw slot per layer, and once its encodes have run each
// layer gives its slot back on its own — so storage that compression frees in one layer is
// reused by any layer, and a page left raw in one layer holds one slot, not one in every layer.
// A partial last page holds its slots for as long as it fills; a full page holds them until the
// caller reports, layer by layer, whether the encode compressed it (a page-head whose blocks need
// more than six escapes stays in its raw slot for good).  With one layer, or with separate
// per-layer raw pools addressed by the same slot index (a caller that reports a page raw when it
// is raw in any layer), this is the same bookkeeping for every layer at once.  Host code only;
// one manager must not be used from two threads at once.
#include <algorithm>
#include <cstdint>
#include <new>
#include <vector>

#include "../../include/zf.h"

struct zf_kv {
  int32_t num_pages = 0, num_raw = 0, num_layers = 0, page_size = 0, max_requests = 0, max_pages = 0;
  std::vector<int32_t> free_pages;      // stacks of free ids / slots
  std::vector<int32_t> free_raw;
  struct Request {
    bool active = false;
    int32_t len = 0;
    std::vector<int32_t> pages;
    std::vector<int32_t> tail_raw;      // per layer, raw slot of the partial last page; empty if the last is full
  };
  std::vector<Request> reqs;
  std::vector<int32_t> owner;           // per page id: request holding it, -1 if free
  std::vector<int32_t> held_raw;        // [page id][layer]: raw slot a full page holds, -1 if none
  std::vector<uint8_t> pending;         // per page id: full, raw slots held until the caller reclaims
  std::vector<int32_t> kept;            // per page id: layers in which it is full and left raw
  std::vector<int32_t> pending_ids;     // the pending page ids, unordered
  std::vector<int32_t> pending_at;      // per page id: its index in pending_ids, -1 if not pending
  int32_t kept_pages = 0;               // full pages left raw in at least one layer
  int64_t kept_slots = 0;               // raw slots those pages hold
};

namespace {

int32_t pages_for(const zf_kv* kv, int64_t len) {
  return static_cast<int32_t>((len + kv->page_size - 1) / kv->page_size);
}

int32_t take(std::vector<int32_t>& stack) {
  const int32_t v = stack.back();
  stack.pop_back();
  return v;
}

int32_t* held(zf_kv* kv, int32_t pid) { return kv->held_raw.data() + static_cast<size_t>(pid) * kv->num_layers; }

// a page that just became full: its per-layer raw slots are held until the caller reclaims them
void set_pending(zf_kv* kv, int32_t pid, const std::vector<int32_t>& slots) {
  std::copy(slots.begin(), slots.end(), held(kv, pid));
  kv->pending[pid] = 1;
  kv->pending_at[pid] = static_cast<int32_t>(kv->pending_ids.size());
  kv->pending_ids.push_back(pid);
}

void clear_pending(zf_kv* kv, int32_t pid) {
  if (!kv->pending[pid]) return;
  const int32_t at = kv->pending_at[pid], last = kv->pending_ids.back();
  kv->pending_ids[at] = last;
  kv->pending_at[last] = at;
  kv->pending_ids.pop_back();
  kv->pending_at[pid] = -1;
  kv->pending[pid] = 0;
}

void give_back_raw(zf_kv* kv, int32_t pid) {
  int32_t* h = held(kv, pid);
  for (int32_t l = 0; l < kv->num_layers; ++l) {
    if (h[l] >= 0) kv->free_raw.push_back(h[l]);
    h[l] = -1;
  }
  clear_pending(kv, pid);
  if (kv->kept[pid]) {
    --kv->kept_pages;
    kv->kept_slots -= kv->kept[pid];
  }
  kv->kept[pid] = 0;
}

// a new page takes one raw slot per layer
std::vector<int32_t> take_slots(zf_kv* kv) {
  std::vector<int32_t> slots(kv->num_layers);
  for (int32_t& v : slots) v = take(kv->free_raw);
  return slots;
}

// pages that can be opened from the free pools: one id and num_layers raw slots each
int32_t openable(const zf_kv* kv) {
  return std::min(static_cast<int32_t>(kv->free_pages.size()),
                  static_cast<int32_t>(kv->free_raw.size()) / kv->num_layers);
}

}  // namespace

extern "C" zf_status zf_kv_create(int32_t num_pages, int32_t num_raw_slots, int32_t num_layers, int32_t page_size,
                                  int32_t max_requests, int32_t max_pages_per_req, zf_kv** out) {
  if (!out) return ZF_ERR_INVALID_ARGUMENT;
  *out = nullptr;
  if (num_pages < 1 || num_layers < 1 || num_raw_slots < num_layers || max_requests < 1 || max_pages_per_req < 1 ||
      page_size < ZF_BLOCK_TOKENS || page_size % ZF_BLOCK_TOKENS || page_size > ZF_MAX_PAGE_SIZE)
    return ZF_ERR_INVALID_ARGUMENT;
  zf_kv* kv = new (std::nothrow) zf_kv;
  if (!kv) return ZF_ERR_UNSUPPORTED;
  kv->num_pages = num_pages;
  kv->num_raw = num_raw_slots;
  kv->num_layers = num_layers;
  kv->page_size = page_size;
  kv->max_requests = max_requests;
  kv->max_pages = max_pages_per_req;
  // lowest ids and slots are handed out first
  for (int32_t i = num_pages - 1; i >= 0; --i) kv->free_pages.push_back(i);
  for (int32_t i = num_raw_slots - 1; i >= 0; --i) kv->free_raw.push_back(i);
  kv->reqs.resize(max_requests);
  kv->owner.assign(num_pages, -1);
  kv->held_raw.assign(static_cast<size_t>(num_pages) * num_layers, -1);
  kv->pending.assign(num_pages, 0);
  kv->kept.assign(num_pages, 0);
  kv->pending_at.assign(num_pages, -1);
  *out = kv;
  return ZF_OK;
}

extern "C" void zf_kv_destroy(zf_kv* kv) { delete kv; }

extern "C" zf_status zf_kv_admit(zf_kv* kv, int32_t req, int32_t len, int32_t* page_ids, int32_t* n_valid,
                                 int32_t* raw_slots, int32_t* n) {
  if (!kv || !n || req < 0 || req >= kv->max_requests || len < 0 || kv->reqs[req].active)
    return ZF_ERR_INVALID_ARGUMENT;
  const int32_t np = pages_for(kv, len);
  if (np > kv->max_pages) return ZF_ERR_INVALID_ARGUMENT;
  if (np > 0 && (!page_ids || !n_valid || !raw_slots)) return ZF_ERR_INVALID_ARGUMENT;
  // every page is written uncompressed first: np ids and np raw slots in every layer
  if (np > openable(kv)) return ZF_ERR_CAPACITY;
  zf_kv::Request& r = kv->reqs[req];
  r = zf_kv::Request{};
  r.active = true;
  r.len = len;
  for (int32_t i = 0; i < np; ++i) {
    const int32_t pid = take(kv->free_pages);
    const std::vector<int32_t> slots = take_slots(kv);
    const int32_t fill = std::min(kv->page_size, len - i * kv->page_size);
    kv->owner[pid] = req;
    r.pages.push_back(pid);
    if (fill == kv->page_size) {
      set_pending(kv, pid, slots);
    } else {
      r.tail_raw = slots;
    }
    page_ids[i] = pid;
    n_valid[i] = fill;
    for (int32_t l = 0; l < kv->num_layers; ++l) raw_slots[static_cast<size_t>(l) * np + i] = slots[l];
  }
  *n = np;
  return ZF_OK;
}

extern "C" zf_status zf_kv_append(zf_kv* kv, const int32_t* reqs, int32_t n, int32_t* page_ids, int32_t* n_valid,
                                  int32_t* raw_slots) {
  if (!kv || n < 0 || (n > 0 && (!reqs || !page_ids || !n_valid || !raw_slots))) return ZF_ERR_INVALID_ARGUMENT;
  // check everything first, so that a refused call changes nothing
  int32_t need = 0;
  std::vector<uint8_t> seen(kv->max_requests, 0);
  for (int32_t i = 0; i < n; ++i) {
    const int32_t q = reqs[i];
    if (q < 0 || q >= kv->max_requests || !kv->reqs[q].active || seen[q]) return ZF_ERR_INVALID_ARGUMENT;
    seen[q] = 1;
    if (kv->reqs[q].len % kv->page_size == 0) {            // the next token opens a new page
      if (pages_for(kv, kv->reqs[q].len) + 1 > kv->max_pages) return ZF_ERR_INVALID_ARGUMENT;
      ++need;
    }
  }
  if (need > openable(kv)) return ZF_ERR_CAPACITY;
  for (int32_t i = 0; i < n; ++i) {
    zf_kv::Request& r = kv->reqs[reqs[i]];
    if (r.len % kv->page_size == 0) {
      const int32_t pid = take(kv->free_pages);
      kv->owner[pid] = reqs[i];
      r.pages.push_back(pid);
      r.tail_raw = take_slots(kv);
    }
    ++r.len;
    const int32_t pid = r.pages.back();
    const int32_t fill = r.len - (static_cast<int32_t>(r.pages.size()) - 1) * kv->page_size;
    page_ids[i] = pid;
    n_valid[i] = fill;
    for (int32_t l = 0; l < kv->num_layers; ++l) raw_slots[static_cast<size_t>(l) * n + i] = r.tail_raw[l];
    if (fill == kv->page_size) {                            // full: compressed by this encode
      set_pending(kv, pid, r.tail_raw);
      r.tail_raw.clear();
    }
  }
  return ZF_OK;
}

extern "C" zf_status zf_kv_pending(const zf_kv* kv, int32_t* page_ids, int32_t* raw_slots, int32_t capacity,
                                   int32_t* n) {
  if (!kv || !n || capacity < 0 || (capacity > 0 && (!page_ids || !raw_slots))) return ZF_ERR_INVALID_ARGUMENT;
  const int32_t k = static_cast<int32_t>(kv->pending_ids.size());
  *n = k;
  if (k > capacity) return ZF_ERR_INVALID_ARGUMENT;
  std::vector<int32_t> ids(kv->pending_ids);
  std::sort(ids.begin(), ids.end());
  for (int32_t i = 0; i < k; ++i) {
    page_ids[i] = ids[i];
    const int32_t* h = kv->held_raw.data() + static_cast<size_t>(ids[i]) * kv->num_layers;
    for (int32_t l = 0; l < kv->num_layers; ++l) raw_slots[static_cast<size_t>(l) * k + i] = h[l];
  }
  return ZF_OK;
}

extern "C" zf_status zf_kv_reclaim(zf_kv* kv, const int32_t* page_ids, const int32_t* kept_raw, int32_t n) {
  if (!kv || n < 0 || (n > 0 && (!page_ids || !kept_raw))) return ZF_ERR_INVALID_ARGUMENT;
  std::vector<uint8_t> seen(kv->num_pages, 0);
  for (int32_t i = 0; i < n; ++i) {
    const int32_t pid = page_ids[i];
    if (pid < 0 || pid >= kv->num_pages || !kv->pending[pid] || seen[pid]) return ZF_ERR_INVALID_ARGUMENT;
    seen[pid] = 1;
  }
  for (int32_t i = 0; i < n; ++i) {
    const int32_t pid = page_ids[i];
    int32_t* h = held(kv, pid);
    int32_t keep = 0;
    for (int32_t l = 0; l < kv->num_layers; ++l) {
      if (kept_raw[static_cast<size_t>(l) * n + i]) {
        ++keep;
      } else {                                              // compressed in this layer: slot back to the pool
        kv->free_raw.push_back(h[l]);
        h[l] = -1;
      }
    }
    clear_pending(kv, pid);
    if (keep) {
      kv->kept[pid] = keep;
      ++kv->kept_pages;
      kv->kept_slots += keep;
    }
  }
  return ZF_OK;
}

extern "C" zf_status zf_kv_release(zf_kv* kv, int32_t req) {
  if (!kv || req < 0 || req >= kv->max_requests || !kv->reqs[req].active) return ZF_ERR_INVALID_ARGUMENT;
  zf_kv::Request& r = kv->reqs[req];
  for (const int32_t pid : r.pages) {
    give_back_raw(kv, pid);
    kv->owner[pid] = -1;
    kv->free_pages.push_back(pid);
  }
  for (const int32_t slot : r.tail_raw) kv->free_raw.push_back(slot);
  r = zf_kv::Request{};
  return ZF_OK;
}

extern "C" zf_status zf_kv_export(const zf_kv* kv, int32_t* page_table, int32_t* seq_lens) {
  if (!kv || !page_table || !seq_lens) return ZF_ERR_INVALID_ARGUMENT;
  for (int32_t q = 0; q < kv->max_requests; ++q) {
    const zf_kv::Request& r = kv->reqs[q];
    int32_t* row = page_table + static_cast<int64_t>(q) * kv->max_pages;
    for (int32_t i = 0; i < kv->max_pages; ++i)
      row[i] = i < static_cast<int32_t>(r.pages.size()) ? r.pages[i] : -1;
    seq_lens[q] = r.active ? r.len : 0;
  }
  return ZF_OK;
}

extern "C" zf_status zf_kv_get_stats(const zf_kv* kv, zf_kv_stats* out) {
  if (!kv || !out) return ZF_ERR_INVALID_ARGUMENT;
  zf_kv_stats s{};
  s.free_pages = static_cast<int32_t>(kv->free_pages.size());
  s.free_raw_slots = static_cast<int32_t>(kv->free_raw.size());
  for (const zf_kv::Request& r : kv->reqs) {
    if (!r.active) continue;
    ++s.active_requests;
    s.tokens += r.len;
    if (!r.tail_raw.empty()) ++s.partial_pages;
  }
  const int32_t owned = kv->num_pages - s.free_pages;
  s.pending_pages = static_cast<int32_t>(kv->pending_ids.size());
  s.raw_full_pages = kv->kept_pages;
  s.raw_full_slots = static_cast<int32_t>(kv->kept_slots);
  s.compressed_pages = owned - s.partial_pages - s.pending_pages - s.raw_full_pages;
  // new pages are written uncompressed first: each needs a page id and a raw slot in every layer
  s.new_page_capacity = openable(kv);
  *out = s;
  return ZF_OK;
}

extern "C" zf_status zf_kv_plan_pages(int64_t bytes_per_layer, int32_t num_kv_heads, int32_t page_size,
                                      int32_t num_raw_slots, int32_t* num_pages, int32_t* dense_pages) {
  if (!num_pages || !dense_pages || bytes_per_layer < 0 || num_kv_heads < 1 || num_raw_slots < 0 ||
      page_size < ZF_BLOCK_TOKENS || page_size % ZF_BLOCK_TOKENS || page_size > ZF_MAX_PAGE_SIZE)
    return ZF_ERR_INVALID_ARGUMENT;
  const int64_t blocks = page_size / 4;                     // 512-value blocks per page head
  const int64_t raw_page = 2LL * num_kv_heads * blocks * ZF_RAW_BLOCK_BYTES;          // K and V
  const int64_t comp_page = 2LL * num_kv_heads * blocks * ZF_SLOT_BYTES + 4LL * num_kv_heads;   // + directory
  const int64_t left = bytes_per_layer - static_cast<int64_t>(num_raw_slots) * raw_page;
  const int64_t pages = left > 0 ? left / comp_page : 0;
  const int64_t dense = bytes_per_layer / raw_page;
  *num_pages = static_cast<int32_t>(std::min<int64_t>(pages, INT32_MAX));
  *dense_pages = static_cast<int32_t>(std::min<int64_t>(dense, INT32_MAX));
  return ZF_OK;
}
