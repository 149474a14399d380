// Pieces shared by the attention kernels of libzf (the warp-MMA kernel in zf_attn.cu and the
// tensor-memory kernel in zf_attn_tc.cu): launch arguments, the work split over CTAs (host planner
// and the in-kernel walk over page ranges or chunks), the page resolve through the page table and
// the directory, per-warp tile copies, and the merge arguments.
#pragma once

#include <cuda_runtime.h>
#include <math_constants.h>
#include <stdint.h>

#include <climits>
#include <mutex>

#include "zf_device.cuh"
#include "zf_host.h"

namespace zf {

// Per-variant shape: the compressed kernel runs 15 consumer warps with 6272-byte stages (one
// compressed K+V tile; raw tiles load K, then V, into the same stage); the dense kernel runs 10
// consumer warps with 8192-byte stages (one raw K+V tile).  Plus one metadata warp.
template <bool kCompressed>
struct Cfg {
  static constexpr int kWarps = kCompressed ? 15 : 10;
  static constexpr int kStageBytes = kCompressed ? 6272 : 8192;
  static constexpr int kVOffset = kCompressed ? 3136 : 4096;   // V tile within a stage
  static constexpr int kThreads = (kWarps + 1) * 32;
  // tiles per CTA prefetched into L2 at start-up (measured best on a 32-layer MHA step: two per
  // warp for the compressed kernel, four per warp for the dense one)
  static constexpr int kPrefetchTiles = kCompressed ? 2 * kWarps : 4 * kWarps;
};
constexpr int kWarpStages = 2;
constexpr int kTileCompBytes = 4 * kSlotBytes;      // 3136: one 16-token tile of K (or V), compressed
constexpr int kTileRawBytes = 4 * kRawBlockBytes;   // 4096
constexpr int kHeadsPerSlice = 8;                   // MMA n of the warp-MMA kernel
constexpr int kMaxItemTiles = 512;                  // 16-token tiles per work item (metadata buffer size)
constexpr int kMaxItemPages = 256;                  // pages per work item (page-table loads per lane: /32)
// q rows in shared memory: channel words permuted so that lane (gi, ti) finds the four B-fragment
// words of k-steps 2j and 2j+1 (words 16j + ti + {0, 4, 8, 12}) in one 16-byte read at word
// 16j + 4ti; rows padded to 320 bytes so the eight rows of a warp's reads hit distinct banks.
constexpr int kQRowBytes = 320;
constexpr int kOStride = 132;                       // padded combine row (conflict-free writes)
// partial chunks per pair are sized for ranges of at least (balanced range) / kMinRangeDivisor pages
constexpr int kMinRangeDivisor = 16;
// start-up prefetch: used when a CTA's balanced share is between these numbers of tiles (below,
// the preceding call's tail is too short to hide the extra planning)
constexpr int kPrefetchMinTilesPerCta = 16;
constexpr int kPrefetchMaxTilesPerCta = 512;
constexpr int kPlanMinTilesPerCta = 4;            // early planning of the first item: from here up to the max
// planner: items of at least this many rounds (tiles per consumer warp) count as long
constexpr int kLongItemRounds = 5;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kRescaleThreshold = 8.0f;           // log2 units: p <= 2^8 between max updates
// running max before any visible score: finite, so that a column whose scores are all hidden (a
// new token that sees none of an item's positions) gets p = 2^(-inf - kNoScore) = 0, not NaN
constexpr float kNoScore = -1e30f;

enum : int { kKindComp = 0, kKindRaw = 1, kKindInvalid = 2 };

struct AttnArgs {
  const uint8_t* k_comp;
  const uint8_t* v_comp;
  const uint8_t* k_raw;
  const uint8_t* v_raw;
  const int32_t* dir;
  int32_t* status;
  const uint16_t* q;
  const int32_t* page_table;
  const int32_t* seq_lens;
  float* out;
  float* lse;
  float* part_o;
  float* part_lse;
  int32_t* chunk_counts;     // [batch][hkv * slices] partials per pair, for the merge kernel
  int32_t batch, hq, hkv, group, slices, page_size, num_pages, num_raw, max_pages, max_chunks;
  int32_t tokens;            // new tokens per request T: query head qh = head * T + token (hq, group count them)
  int32_t hps;               // query heads (MMA columns) per head slice: kHeadsPerSlice, or 16 / 32
  int32_t min_range_pages;   // lower bound of the pages per CTA range
  int32_t chunk_pages;       // > 0: fixed chunks of this many pages, items dealt round-robin
  int32_t prefetch;          // prefetch the first tiles into L2 while the preceding grid drains
  int32_t plan_first;        // plan the first item while the preceding grid drains
  int64_t comp_head_bytes;   // bytes of one (page, kv head) K record, compressed
  int64_t raw_head_bytes;    // bytes of one (page, kv head) K record, raw
  float scale_log2;          // softmax_scale * log2(e)
  uint64_t wait_limit_ns;    // limit of the waits for the metadata warp's items (kWaitTimeoutNs; tests shorten it)
  uint64_t publish_delay_ns; // the metadata warp's first item is published this much later (0; tests only)
};

struct Plan {
  int grid = 0, max_chunks = 0, slices = 1, min_range_pages = 1, chunk_pages = 0;
  bool prefetch = false, plan_first = false;
  size_t part_o_bytes = 0, part_lse_bytes = 0, ws_bytes = 0;
};

// What the metadata warp publishes for an item.
struct ItemDesc {
  int b, c, g, t0, t1, units, h0, nh, single, pg0, npg;   // pg0, npg: the item's pages in the request
  int planned;   // first item only: the plan made before the wait held, its first tiles are in flight
};

// Row of q, out and lse (stored [batch][T][heads]) for query head qh = head * T + token of request b.
__device__ __forceinline__ size_t query_row(int b, int qh, int T, int hq) {
  const int h = qh / T, t = qh - h * T;
  return (static_cast<size_t>(b) * T + t) * (hq / T) + h;
}

__device__ __forceinline__ bool same_piece(const ItemDesc& x, const ItemDesc& y) {
  return x.b == y.b && x.c == y.c && x.g == y.g && x.t0 == y.t0 && x.t1 == y.t1 && x.units == y.units &&
         x.h0 == y.h0 && x.nh == y.nh && x.single == y.single && x.pg0 == y.pg0 && x.npg == y.npg;
}

// Geometry of the page sequence: pair p = (request b, r = kv head * slices + slice) owns pages
// [S_p, S_p + n_b) with S_p = HS * prefix[b] + r * n_b (HS pairs per request, n_b pages each).
// CTA k owns [k W, (k + 1) W); within one CTA range a pair's pages are cut every pmax pages from
// where they start.  Partials of a pair are numbered in page order across CTAs.
struct Ranges {
  int W, pmax, ppc;   // pages per CTA range, pages per item, items of a full range
};

// Partials of the pair starting at S that lie in CTA ranges before range k.
__device__ __forceinline__ int chunks_before(const Ranges& g, int S, int k) {
  const int k0 = S / g.W;
  if (k <= k0) return 0;
  const int first = (k0 + 1) * g.W - S;
  return (first + g.pmax - 1) / g.pmax + (k - k0 - 1) * g.ppc;
}

// Partials of the pair with pages [S, S + n), n >= 1.
__device__ __forceinline__ int pair_chunks(const Ranges& g, int S, int n) {
  const int kl = (S + n - 1) / g.W;
  const int tail = S + n - max(S, kl * g.W);
  return chunks_before(g, S, kl) + (tail + g.pmax - 1) / g.pmax;
}

// The item covering pages [pg0, pg1) of pair (b, r) as partial c; L: the length of request b.
__device__ __forceinline__ ItemDesc describe_piece(const AttnArgs& a, int b, int r, int pg0, int pg1, int c,
                                                   bool single, int L) {
  ItemDesc d;
  d.b = b;
  d.c = c;
  d.planned = 0;
  d.g = a.slices == 1 ? r : r / a.slices;
  const int s = r - d.g * a.slices;
  d.single = single;
  d.pg0 = pg0;
  d.npg = pg1 - pg0;
  d.t0 = pg0 * a.page_size;
  d.t1 = min(pg1 * a.page_size, L);
  d.units = (d.t1 - d.t0 + 15) >> 4;
  d.h0 = d.g * a.group + s * a.hps;
  d.nh = min(a.hps, a.group - s * a.hps);
  return d;
}

// Resolve the item's pages into one entry per tile: meta[u] = slot << 5 | tile_in_page << 2 | kind
// (all 32 lanes).  Two rounds of independent loads: every page-table entry, then every directory
// entry they name; only then are the entries classified and written (classifying each page as
// its directory entry arrives made one dependent round trip per page and lane: up to 8 in a row).
// kSpec: relaxed loads of values that may still change, and no error reports (prefetch planning).
// keep_pid / keep_dir (optional): the page ids and directory entries read, per k (-1 past npg).
constexpr int kPagesPerLane = kMaxItemPages / 32;
template <bool kCompressed, bool kSpec = false>
__device__ __forceinline__ void resolve_tiles(const AttnArgs& a, const ItemDesc& d, int* meta, int lane,
                                              int* keep_pid = nullptr, int* keep_dir = nullptr) {
  constexpr int kPer = kPagesPerLane;
  const int tpp = a.page_size >> 4;
  const int npg = d.npg;
  const int32_t* row = a.page_table + static_cast<size_t>(d.b) * a.max_pages + d.pg0;
  int pid[kPer], dir[kPer];
#pragma unroll
  for (int k = 0; k < kPer; ++k) {
    const int i = lane + 32 * k;
    pid[k] = i < npg ? (kSpec ? ld_relaxed(row + i) : row[i]) : -1;
  }
#pragma unroll
  for (int k = 0; k < kPer; ++k) {
    dir[k] = -2;                                   // no entry read (never a valid one)
    if (kCompressed && pid[k] >= 0 && pid[k] < a.num_pages) {
      const int32_t* dp = a.dir + static_cast<size_t>(pid[k]) * a.hkv + d.g;
      dir[k] = kSpec ? ld_relaxed(dp) : *dp;
    }
  }
  if (keep_pid != nullptr) {
#pragma unroll
    for (int k = 0; k < kPer; ++k) {
      keep_pid[k] = pid[k];
      keep_dir[k] = dir[k] == -2 ? -1 : dir[k];
    }
  }
#pragma unroll
  for (int k = 0; k < kPer; ++k) {
    const int i = lane + 32 * k;
    if (i >= npg) break;
    int kind = kKindInvalid, slot = 0;
    if (kCompressed) {
      if (pid[k] >= 0 && pid[k] < a.num_pages) {
        const int dd = dir[k];
        if (dd == ZF_DIR_COMPRESSED) {
          kind = kKindComp;
          slot = pid[k];
        } else if (dd >= 0 && dd < a.num_raw) {
          kind = kKindRaw;
          slot = dd;
        } else if (!kSpec) {
          report(a.status, ZF_DEV_BAD_DIR);
        }
      } else if (!kSpec) {
        report(a.status, ZF_DEV_BAD_PAGE_ID);
      }
    } else if (pid[k] >= 0 && pid[k] < a.num_raw) {
      kind = kKindRaw;
      slot = pid[k];
    } else if (!kSpec) {
      report(a.status, ZF_DEV_BAD_PAGE_ID);
    }
    for (int t = 0; t < tpp; ++t) {
      const int u = i * tpp + t;
      if (u < d.units) meta[u] = (slot << 5) | (t << 2) | kind;
    }
  }
}

// Start the copies of tile u of an item into `stage` (K at 0, V at kVOffset), signalled on the
// warp's own barrier `bar`: one lane issues 1-D bulk copies (each consumer warp issues its own, so
// an SM has 10-15 copy streams in flight).  In the compressed kernel a raw tile does not fit one
// stage: only its K half is started here and the V half is fetched after QK^T (issue_raw_v).
// Returns whether anything was armed on `bar`.
template <bool kCompressed>
__device__ __forceinline__ bool issue_tile(const AttnArgs& a, const ItemDesc& d, const int* meta, int u,
                                           uint8_t* stage, uint64_t* bar, int lane, uint64_t policy) {
  using C = Cfg<kCompressed>;
  const int m = meta[u];
  const int kind = m & 3;
  const size_t head = static_cast<size_t>(m >> 5) * a.hkv + d.g;
  const int t = (m >> 2) & 7;
  if (kCompressed && kind == kKindComp) {
    if (lane == 0) {
      const size_t off = head * a.comp_head_bytes + static_cast<size_t>(t) * kTileCompBytes;
      mbar_arrive_expect_tx(bar, 2 * kTileCompBytes);
      bulk_copy_g2s(stage, a.k_comp + off, kTileCompBytes, bar, policy);
      bulk_copy_g2s(stage + C::kVOffset, a.v_comp + off, kTileCompBytes, bar, policy);
    }
    return true;
  }
  if (kind == kKindRaw) {
    if (lane == 0) {
      const size_t off = head * a.raw_head_bytes + static_cast<size_t>(t) * kTileRawBytes;
      mbar_arrive_expect_tx(bar, (kCompressed ? 1 : 2) * kTileRawBytes);
      bulk_copy_g2s(stage, a.k_raw + off, kTileRawBytes, bar, policy);
      if (!kCompressed) bulk_copy_g2s(stage + C::kVOffset, a.v_raw + off, kTileRawBytes, bar, policy);
    }
    return true;
  }
  return false;
}

// Compressed kernel, raw tile: after QK^T, fetch the V half into the same stage.
__device__ __forceinline__ void issue_raw_v(const AttnArgs& a, const ItemDesc& d, const int* meta, int u,
                                            uint8_t* stage, uint64_t* bar, int lane, uint64_t policy) {
  const int m = meta[u];
  const size_t head = static_cast<size_t>(m >> 5) * a.hkv + d.g;
  const size_t off = head * a.raw_head_bytes + static_cast<size_t>((m >> 2) & 7) * kTileRawBytes;
  if (lane == 0) {
    mbar_arrive_expect_tx(bar, kTileRawBytes);
    bulk_copy_g2s(stage, a.v_raw + off, kTileRawBytes, bar, policy);
  }
}

// L2 prefetch of the K and V records of tiles [0, n) of an item (lanes split the tiles).
template <bool kCompressed>
__device__ __forceinline__ void prefetch_item_tiles(const AttnArgs& a, const ItemDesc& d, const int* meta, int n,
                                                    int lane) {
  for (int u = lane; u < n; u += 32) {
    const int m = meta[u];
    const int kind = m & 3;
    const size_t head = static_cast<size_t>(m >> 5) * a.hkv + d.g;
    const int t = (m >> 2) & 7;
    if (kCompressed && kind == kKindComp) {
      const size_t off = head * a.comp_head_bytes + static_cast<size_t>(t) * kTileCompBytes;
      bulk_prefetch_l2(a.k_comp + off, kTileCompBytes);
      bulk_prefetch_l2(a.v_comp + off, kTileCompBytes);
    } else if (kind == kKindRaw) {
      const size_t off = head * a.raw_head_bytes + static_cast<size_t>(t) * kTileRawBytes;
      bulk_prefetch_l2(a.k_raw + off, kTileRawBytes);
      bulk_prefetch_l2(a.v_raw + off, kTileRawBytes);
    }
  }
}

// Pages of every request (chunks, when chunk_pages > 0) into prefix[b + 1], then prefix sums
// (prefix[0] = 0); each request's length (clamped) into lens[b].  All threads; ends
// with a barrier.
// kSpec: relaxed loads, no error reports.
// Returns the (clamped) length of request tid, -1 past the batch.  changed (batch <= kThreads, one
// request per thread): set when that length differs from held, the one an earlier pass returned.
template <bool kSpec, int kThreads>
__device__ __forceinline__ int load_lengths(const AttnArgs& a, int* prefix, int* lens, int tid, int held = -1,
                                            volatile int* changed = nullptr) {
  int mine = -1;
  const int warp = tid >> 5, lane = tid & 31;
  const int max_len = a.max_pages * a.page_size;
  for (int b = tid; b < a.batch; b += kThreads) {
    int len = kSpec ? ld_relaxed(a.seq_lens + b) : a.seq_lens[b];
    if (len < 0 || len > max_len) {
      if (!kSpec && blockIdx.x == 0) report(a.status, ZF_DEV_BAD_SEQ_LEN);
      len = min(max(len, 0), max_len);
    }
    if (b == tid) mine = len;
    if (changed != nullptr && b == tid && len != held) *changed = 1;
    const int pages = (len + a.page_size - 1) / a.page_size;
    prefix[b + 1] = a.chunk_pages > 0 ? (pages + a.chunk_pages - 1) / a.chunk_pages : pages;
    lens[b] = len;
  }
  __syncthreads();
  if (warp == 0) {
    int carry = 0;
    for (int base = 0; base < a.batch; base += 32) {
      const int i = base + lane;
      int v = i < a.batch ? prefix[i + 1] : 0;
#pragma unroll
      for (int d = 1; d < 32; d <<= 1) {
        const int t = __shfl_up_sync(0xFFFFFFFFu, v, d);
        if (lane >= d) v += t;
      }
      if (i < a.batch) prefix[i + 1] = carry + v;
      carry += __shfl_sync(0xFFFFFFFFu, v, 31);
    }
    if (lane == 0) prefix[0] = 0;
  }
  __syncthreads();
  return mine;
}

__device__ __forceinline__ Ranges make_ranges(const AttnArgs& a, int total) {
  Ranges g;
  g.W = max((total + static_cast<int>(gridDim.x) - 1) / static_cast<int>(gridDim.x), a.min_range_pages);
  g.pmax = min(kMaxItemTiles / (a.page_size / ZF_BLOCK_TOKENS), kMaxItemPages);
  g.ppc = (g.W + g.pmax - 1) / g.pmax;
  return g;
}

// Walk this CTA's items and hand each to emit(desc) (uniform across the warp); stops early when emit
// returns false.  Returns whether the walk ran to its end.
//  * balanced mode (chunk_pages == 0): this CTA's page range, pair by pair;
//  * chunked mode: items (request, chunk, kv head / slice) of chunk_pages pages, dealt round-robin
//    (item i to CTA i % grid); prefix holds chunk counts.
template <typename Emit>
__device__ __forceinline__ bool walk_range(const AttnArgs& a, const int* prefix, const int* lens, const Ranges& g,
                                           int HS, Emit&& emit) {
  if (a.chunk_pages > 0) {
    const int cp = a.chunk_pages;
    const int items = HS * prefix[a.batch];
    for (int item = blockIdx.x; item < items; item += gridDim.x) {
      const int j = item / HS, r = item - j * HS;
      int l = 0, h = a.batch;                 // prefix[l] <= j < prefix[l + 1]
      while (h - l > 1) {
        const int mid = (l + h) >> 1;
        if (prefix[mid] <= j) l = mid; else h = mid;
      }
      const int c = j - prefix[l];
      const int len = lens[l];
      const int n = (len + a.page_size - 1) / a.page_size;
      if (!emit(describe_piece(a, l, r, c * cp, min(c * cp + cp, n), c, prefix[l + 1] - prefix[l] == 1, len)))
        return false;
    }
    return true;
  }
  const int total = HS * prefix[a.batch];
  const long long lo_l = static_cast<long long>(blockIdx.x) * g.W;
  const int hi = static_cast<int>(min(lo_l + g.W, static_cast<long long>(total)));
  int t = static_cast<int>(min(lo_l, static_cast<long long>(total)));
  if (t >= hi) return true;
  int b = 0;
  {   // the request holding page t: largest b with HS * prefix[b] <= t
    int l = 0, h = a.batch;
    while (h - l > 1) {
      const int mid = (l + h) >> 1;
      if (HS * prefix[mid] <= t) l = mid; else h = mid;
    }
    b = l;
  }
  // the first pair may have started in an earlier range; every later one starts in this range,
  // so only the first needs the division-based geometry
  while (HS * prefix[b + 1] <= t) ++b;
  int n = prefix[b + 1] - prefix[b];
  int r = (t - HS * prefix[b]) / n;
  int S = HS * prefix[b] + r * n;
  int c = chunks_before(g, S, blockIdx.x);
  bool single = pair_chunks(g, S, n) == 1;
  const long long range_end = lo_l + g.W;
  while (true) {
    const int seg_end = min(hi, S + n);
    for (int pt = t; pt < seg_end; pt += g.pmax, ++c)
      if (!emit(describe_piece(a, b, r, pt - S, min(pt + g.pmax, seg_end) - S, c, single, lens[b])))
        return false;
    t = seg_end;
    if (t >= hi) return true;
    if (++r == HS) {                           // next request with pages
      r = 0;
      do { ++b; } while (prefix[b + 1] == prefix[b]);
      n = prefix[b + 1] - prefix[b];
    }
    S = t;
    c = 0;
    single = n <= g.pmax && S + n <= range_end;
  }
}

struct MergeArgs {
  const float* part_o;
  const float* part_lse;
  float* out;
  float* lse;
  const int32_t* chunk_counts;
  int32_t batch, hq, group, slices, max_chunks, tokens, hps;
};

// ------------------------------------------------------------------------------- host planner
// Work split for one call, from the sizes alone (requests assumed at max_pages).  Two modes, whichever
// the cost model (rounds of tiles per warp on the busiest CTA, plus one round per item) prefers:
//  * balanced ranges: every CTA gets the same number of pages, wherever requests start and end;
//    best for long and ragged contexts;
//  * fixed chunks of cp pages, items dealt round-robin: for short contexts, where the per-item cost
//    dominates and chunks that never straddle a request boundary save items.
// hps: query heads per head slice (the columns one kernel pass gives a kv head's tiles).
static Plan make_plan(int batch, int hq, int hkv, int page_size, int max_pages, int num_sms, int warps,
                      int hps = kHeadsPerSlice) {
  Plan p;
  const int group = hq / hkv;
  p.slices = (group + hps - 1) / hps;
  const long long pairs = static_cast<long long>(batch) * hkv * p.slices;
  const long long total_max = pairs * max_pages;     // pages when every request is full length
  const int tpp = page_size / ZF_BLOCK_TOKENS;
  const int pmax = kMaxItemTiles / tpp < kMaxItemPages ? kMaxItemTiles / tpp : kMaxItemPages;
  const int grid_b = static_cast<int>(total_max < num_sms ? (total_max > 0 ? total_max : 1) : num_sms);
  const long long balanced = (total_max + grid_b - 1) / grid_b;
  auto rounds = [&](long long tiles) { return (tiles + warps - 1) / warps; };
  // balanced: the busiest CTA meets up to 1 + W / max_pages requests and cuts every pmax pages
  const long long cost_b = rounds(balanced * tpp) + 1 + 1 + (balanced + max_pages - 1) / max_pages + balanced / pmax;
  long long cost_c = LLONG_MAX;
  int best_cp = 0;
  const int cp_max = max_pages < pmax ? max_pages : pmax;
  long long best_item_rounds = 0, best_load = 0;
  for (int cp = 1; cp <= cp_max; ++cp) {
    const long long items = pairs * ((max_pages + cp - 1) / cp);
    const long long grid = items < num_sms ? items : num_sms;
    const long long item_rounds = (items + grid - 1) / grid;
    const long long cost = item_rounds * (rounds(static_cast<long long>(cp) * tpp) + 1);
    const long long load = item_rounds * cp;            // pages per CTA
    // Ties: fewer items per CTA first; then, for long items, the lighter CTA (measured on GB300:
    // 128 instead of 135 tiles per CTA, both nine rounds per warp, is 4% faster); else the larger
    // chunk (fewer partials to merge: 45 instead of 32 tiles, both three rounds, is 2% faster).
    bool better = cost < cost_c;
    if (cost == cost_c) {
      if (item_rounds != best_item_rounds) better = item_rounds < best_item_rounds;
      else if (rounds(static_cast<long long>(cp) * tpp) >= kLongItemRounds) better = load <= best_load;
      else better = true;
    }
    if (better) {
      cost_c = cost;
      best_cp = cp;
      best_item_rounds = item_rounds;
      best_load = load;
    }
  }
  if (best_cp > 0 && cost_c < cost_b) {
    p.chunk_pages = best_cp;
    p.max_chunks = (max_pages + best_cp - 1) / best_cp;
    const long long items = pairs * p.max_chunks;
    p.grid = static_cast<int>(items < num_sms ? items : num_sms);
  } else {
    p.grid = grid_b;
    // The kernel gives each CTA max(ceil(total / grid), min_range_pages) pages; a floor keeps the
    // number of partials per pair, and so the workspace, bounded when requests are short.
    p.min_range_pages = static_cast<int>(balanced / kMinRangeDivisor > 1 ? balanced / kMinRangeDivisor : 1);
    // A pair of n pages meets at most ceil(n / W) + 1 CTA ranges and is cut every pmax pages in
    // each, so it has at most floor(n / pmax) + ceil(n / W) + 1 partials.
    p.max_chunks = max_pages / pmax + (max_pages + p.min_range_pages - 1) / p.min_range_pages + 1;
  }
  // Short calls (a few rounds of tiles per CTA) are dominated by their start-up: they plan their
  // first item while the preceding grid drains, and those above a few tiles per CTA also prefetch
  // their first tiles into L2.  Long calls do neither (measured on GB300: planning early made the
  // Llama-3-8B batch-64 call 2.7% slower, the prefetch slower still).  Below the prefetch range
  // the plan still pays (LLaMA-7B MHA at 512 tokens, 7 tiles per CTA: 11.2 -> 10.5 us per call),
  // down to a few tiles per CTA (a single 8-head 512-token call, 2 tiles per CTA, lost 0.1-1.6 us).
  p.prefetch = balanced * tpp >= kPrefetchMinTilesPerCta && balanced * tpp <= kPrefetchMaxTilesPerCta;
  p.plan_first = balanced * tpp >= kPlanMinTilesPerCta && balanced * tpp <= kPrefetchMaxTilesPerCta;
  const size_t n = static_cast<size_t>(batch) * hq * p.max_chunks;
  p.part_o_bytes = n * ZF_HEAD_DIM * 4;
  p.part_lse_bytes = (n * 4 + 255) & ~static_cast<size_t>(255);
  p.ws_bytes = p.part_o_bytes + p.part_lse_bytes + ((static_cast<size_t>(pairs) * 4 + 255) & ~static_cast<size_t>(255));
  return p;
}

// Raise a kernel's dynamic shared-memory limit once per (device, kernel); the limit only grows.
// `which` (0-3) names the kernel among those of the calling file: each file that includes this
// header keeps its own records, so two kernels of one file must not share a number.
static zf_status ensure_smem_limit(const void* kernel, int which, size_t bytes) {
  static std::mutex mu;
  static size_t done[64][4] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return ZF_ERR_CUDA;
  if (dev < 0 || dev >= 64) return ZF_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(mu);
  if (done[dev][which] >= bytes) return ZF_OK;
  if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(bytes)) !=
      cudaSuccess)
    return ZF_ERR_CUDA;
  done[dev][which] = bytes;
  return ZF_OK;
}

static zf_status current_sm_count(int* sms) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return ZF_ERR_CUDA;
  if (cudaDeviceGetAttribute(sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return ZF_ERR_CUDA;
  return ZF_OK;
}

static bool attn_shape_ok(int batch, int hq, int hkv, int max_pages) {
  if (!(batch >= 0 && batch <= ZF_MAX_BATCH && hkv >= 1 && hq >= hkv && hq % hkv == 0 && max_pages >= 1 &&
        static_cast<long long>(max_pages) * ZF_MAX_PAGE_SIZE < INT_MAX))
    return false;
  // the kernel indexes the pages of all (request, kv head, head slice) pairs with 32-bit ints
  const long long slices = (hq / hkv + kHeadsPerSlice - 1) / kHeadsPerSlice;
  return static_cast<long long>(batch) * hkv * slices * max_pages < (1ll << 30);
}

// Query heads as the kernel counts them: every (head, new token) pair of a request is one, so a
// call with T tokens is planned like a call with T times the heads (and T times the GQA group).
static bool tokens_ok(int32_t tokens, int32_t hq) {
  return tokens >= 1 && tokens <= ZF_MAX_TOKENS && static_cast<long long>(hq) * tokens <= INT_MAX / ZF_HEAD_DIM;
}


// Launches shared by the two attention translation units.
// The split-result merge of a call's partials (zf_attn.cu); multi: rows of out / lse are
// [batch][T][heads].
zf_status launch_merge(const MergeArgs& m, bool multi, cudaStream_t stream);
// The tensor-memory kernel (zf_attn_tc.cu) for calls whose kv heads have more than
// kHeadsPerSlice query columns: whether its shared memory holds the lengths of `batch` requests,
// its plan, and its launch (attention + merge) with `base` holding every other argument.
// columns per pass of the tensor-memory kernel for hq / hkv query columns per kv head: 16 or 32
int attention_tc_cols(int hq, int hkv);
bool attention_tc_fits(int32_t batch, int hq, int hkv);
Plan attention_tc_plan(int batch, int hq, int hkv, int page_size, int max_pages, int num_sms);
zf_status launch_attention_tc(const AttnArgs& base, const Plan& p, int32_t tokens, cudaStream_t stream);

}  // namespace zf
