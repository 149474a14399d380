// zf_decode_attn / zf_dense_decode_attn (and their _multi forms for several new tokens per
// request): split-KV decode attention over a paged KV cache whose full pages are stored
// compressed, plus the split-result merge.
//
// ZipFusion §III.C (Attention over the Compressed KV Cache): compressed blocks are copied
// HBM -> shared memory as they are, each thread rebuilds the exact BF16 operands of a
// tensor-core instruction in registers right before use, raw blocks need no rebuild, and page
// metadata for later pages is fetched while earlier pages are attended.  ZipFusion §IV.B:
// split-KV partial results are combined by a split-result merge.
//
// Design for sm_103a (one CTA per SM, persistent):
//  * work split (host planner, from the sizes): either balanced page ranges — the pages of all
//    (request b, kv head g, head slice) pairs, laid end to end, cut into one equal contiguous range
//    per CTA, so a ragged batch gives every SM the same number of tiles; where a range meets a
//    pair it forms that pair's partial(s), cut further into items of at most 256 pages and 512
//    tiles — or, for short contexts, fixed chunks of pages dealt round-robin; each item yields
//    one partial;
//  * the last warp is the metadata warp: it walks the CTA's items, and runs one item ahead,
//    resolving the item's page ids through the page table and the directory into shared memory
//    and staging the item's q rows; an end marker closes the CTA's item stream;
//  * the consumer warps each stream their own 16-token tiles (tile u of an item goes to warp
//    u % warps) into two private shared-memory stages, prefetching the next tile while computing
//    the current one: one lane of the warp issues 1-D bulk copies (cp.async.bulk, L2 evict-first)
//    on the warp's own mbarrier.  (Measured on GB300: bulk copies of 3-8 KB complete at about one
//    per 0.55 us per issuing warp, so one producer warp per SM tops out at 0.9-2.3 TB/s on this
//    traffic, while 8+ issuing warps reach 5.3-6.4 TB/s.)
//  * per tile, a warp rebuilds K blocks straight into m16n8k16 A fragments (the storage order is
//    the fragment order), computes S^T = K Q^T for up to 8 query heads of the GQA group (one MMA
//    n-tile), runs the online softmax in the log2 domain (the running max is only raised, after a
//    warp vote, when a score exceeds it by more than 8), transposes P^T into B fragments with
//    movmatrix, and accumulates O^T = V^T P^T with P split into a BF16 high part and a BF16
//    remainder (two MMAs) so P keeps ~16 significant bits; V blocks are rebuilt right before use;
//  * at the end of an item the warps' (m, l, O) are merged through shared memory and written as
//    the item's partial (or as the final output when the pair has a single partial);
//  * a second kernel merges each (request, head)'s partials by log-sum-exp;
//  * consecutive calls overlap: the merge kernel lets the next grid launch at once, and that grid
//    warms L2 while it waits for this one; a short call also plans its first item (and prefetches
//    its first tiles into L2) then, and after the wait keeps that plan if what it read is unchanged.
#include <cuda_runtime.h>
#include <math_constants.h>
#include <stdint.h>

#include <climits>
#include <mutex>

#include "zf_attn_common.cuh"

namespace zf {

struct SmemLayout {
  size_t stages, item_full, q_full, item_empty, misc, desc, meta, qbuf, bars, prefix, lens, total;
};

template <bool kCompressed>
__host__ __device__ inline SmemLayout smem_layout(int batch) {
  using C = Cfg<kCompressed>;
  SmemLayout s;
  size_t at = 0;
  s.stages = at; at += static_cast<size_t>(C::kWarps) * kWarpStages * C::kStageBytes;
  s.item_full = at; at += 2 * 8;                          // count 1: tiles of the item resolved
  s.q_full = at; at += 2 * 8;                             // count 1: q rows of the item staged
  s.item_empty = at; at += 2 * 8;
  s.misc = at; at += 16 + 16 * 4;    // [0] abort flag, [4] lengths changed, [16..] combine stage per warp
  s.desc = at; at += 2 * 64;
  s.meta = at; at += 2 * kMaxItemTiles * 4;
  s.qbuf = at; at += 2 * kHeadsPerSlice * kQRowBytes;
  s.bars = at; at += static_cast<size_t>(C::kWarps) * kWarpStages * 8;
  s.prefix = at; at += static_cast<size_t>(batch + 1) * 4;
  s.lens = at; at += static_cast<size_t>(batch) * 4;     // each request's length, clamped
  s.total = (at + 127) & ~static_cast<size_t>(127);
  return s;
}

template <int kWarps>
__device__ __forceinline__ void consumer_barrier() {
  asm volatile("bar.sync 1, %0;" ::"n"(kWarps * 32) : "memory");
}

// Barrier over the consumer warps that also ORs a predicate across them (the same answer in all).
template <int kWarps>
__device__ __forceinline__ bool consumer_any(bool v) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.u32 p, %1, 0;\n\t"
      "bar.red.or.pred q, 1, %2, p;\n\t"
      "selp.u32 %0, 1, 0, q;\n\t}"
      : "=r"(r)
      : "r"(static_cast<uint32_t>(v)), "n"(kWarps * 32)
      : "memory");
  return r != 0;
}


// Stage q rows of an item into qbuf (permuted, padded layout; rows past nh are zero).
// q rows of an item: 8 rows x 64 words, lane holds words lane and lane + 32 of every row (rows
// past nh are zero); store_q writes them to qbuf in the permuted, padded layout.
template <bool kMulti>
__device__ __forceinline__ void load_q(const AttnArgs& a, const ItemDesc& d, int lane, uint32_t (&v)[2 * kHeadsPerSlice]) {
#pragma unroll
  for (int r = 0; r < kHeadsPerSlice; ++r) {
    const int qh = d.h0 + min(r, d.nh - 1);
    const size_t row = kMulti ? query_row(d.b, qh, a.tokens, a.hq) : static_cast<size_t>(d.b) * a.hq + qh;
    const uint32_t* src = reinterpret_cast<const uint32_t*>(a.q + row * ZF_HEAD_DIM);
#pragma unroll
    for (int h = 0; h < 2; ++h) v[2 * r + h] = r < d.nh ? src[lane + 32 * h] : 0u;
  }
}

__device__ __forceinline__ void store_q(uint8_t* qb, int lane, const uint32_t (&v)[2 * kHeadsPerSlice]) {
#pragma unroll
  for (int r = 0; r < kHeadsPerSlice; ++r) {
    uint32_t* dst = reinterpret_cast<uint32_t*>(qb + r * kQRowBytes);
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int w = lane + 32 * h;              // channel word w = 16j + 4r' + t  (t < 4, r' < 4)
      const int j = w >> 4, rr = (w >> 2) & 3, t = w & 3;
      dst[16 * j + 4 * t + rr] = v[2 * r + h];
    }
  }
}

// kMulti: several new tokens per request (query head qh = head * T + token, a causal mask on the
// last positions, rows of q / out / lse mapped through query_row); a separate instantiation, so
// the single-token kernels are compiled exactly as without it.
template <bool kCompressed, bool kMulti>
// At most 112 registers per thread (the compiler needs 104 for the compressed variant, without
// spills): 16 warps then leave room on every SM sub-partition for a merge warp, so the merge grid
// of the previous call and this grid's CTAs can be resident together.
__global__ void __maxnreg__(112) attn_kernel(const AttnArgs a) {
  using C = Cfg<kCompressed>;
  constexpr int kWarps = C::kWarps;
  extern __shared__ __align__(128) uint8_t smem[];
  const SmemLayout L = smem_layout<kCompressed>(a.batch);
  uint64_t* item_full = reinterpret_cast<uint64_t*>(smem + L.item_full);
  uint64_t* item_empty = reinterpret_cast<uint64_t*>(smem + L.item_empty);
  uint64_t* q_full = reinterpret_cast<uint64_t*>(smem + L.q_full);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L.misc);
  volatile int* lengths_changed = reinterpret_cast<volatile int*>(smem + L.misc + 4);
  int* combine_stage = reinterpret_cast<int*>(smem + L.misc + 16);
  ItemDesc* desc = reinterpret_cast<ItemDesc*>(smem + L.desc);
  int* meta = reinterpret_cast<int*>(smem + L.meta);
  uint8_t* qbuf = smem + L.qbuf;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L.bars);
  int* prefix = reinterpret_cast<int*>(smem + L.prefix);
  int* lens = reinterpret_cast<int*>(smem + L.lens);
  uint8_t* stages = smem + L.stages;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  // ---- prologue: barriers, pages per request and their prefix sums, the CTA ranges
  if (tid < 2) {
    mbar_init(&item_full[tid], 1);
    mbar_init(&q_full[tid], 1);
    mbar_init(&item_empty[tid], kWarps);
  }
  if (tid < kWarps * kWarpStages) mbar_init(&bars[tid], 1);
  if (tid == 0) {
    *abort_flag = 0;
    *lengths_changed = 0;
  }
  fence_mbar_init();
  const int HS = a.hkv * a.slices;
  // A call plans its first item before the wait and checks the plan after it (one request per
  // thread, so each thread can hold the length it read).
  const bool plan_early = a.plan_first && a.batch <= C::kThreads;
  int held_len = -1;                      // the length of request tid read before the wait
  int plan_pid[kPagesPerLane], plan_dir[kPagesPerLane];   // metadata warp: what the plan read
  // While the preceding grid drains (this grid is launched early, see allow_next_grid): L2 hints.
  // (1) lines of seq_lens, the page table and, up to 8 MB, the directory, spread over the grid;
  // (2) for short calls, the K/V records of this CTA's first kPrefetchTiles tiles, planned from
  //     relaxed reads of lengths, page table and directory that may still change.  The first
  //     item's plan (desc[0], meta buffer 0) is kept: after the wait it is used only if every
  //     value it was made from reads the same again.
  {
    const size_t n_len = (static_cast<size_t>(a.batch) * 4 + 127) / 128;
    const size_t n_tab = (static_cast<size_t>(a.batch) * a.max_pages * 4 + 127) / 128;
    const size_t dir_bytes = static_cast<size_t>(a.num_pages) * a.hkv * 4;
    const size_t n_dir = kCompressed && dir_bytes <= (8u << 20) ? (dir_bytes + 127) / 128 : 0;
    const size_t stride = static_cast<size_t>(gridDim.x) * C::kThreads;
    for (size_t i = static_cast<size_t>(blockIdx.x) * C::kThreads + tid; i < n_len + n_tab + n_dir; i += stride) {
      const void* line = i < n_len ? static_cast<const void*>(reinterpret_cast<const uint8_t*>(a.seq_lens) + 128 * i)
                         : i < n_len + n_tab
                             ? static_cast<const void*>(reinterpret_cast<const uint8_t*>(a.page_table) + 128 * (i - n_len))
                             : static_cast<const void*>(reinterpret_cast<const uint8_t*>(a.dir) + 128 * (i - n_len - n_tab));
      prefetch_l2(line);
    }
    const bool spec = a.prefetch || plan_early;
    if (spec) held_len = load_lengths<true, C::kThreads>(a, prefix, lens, tid);
    if (spec && warp == kWarps) {
      if (lane == 0) desc[0].b = -1;     // no planned first item (yet)
      const Ranges g = make_ranges(a, HS * prefix[a.batch]);
      int budget = a.prefetch ? C::kPrefetchTiles : 0;
      bool first = true;
      walk_range(a, prefix, lens, g, HS, [&](const ItemDesc& d) -> bool {
        int* mb = meta + (first ? 0 : kMaxItemTiles);
        if (first) resolve_tiles<kCompressed, true>(a, d, mb, lane, plan_pid, plan_dir);
        else resolve_tiles<kCompressed, true>(a, d, mb, lane);
        __syncwarp();
        if (first && lane == 0) desc[0] = d;
        first = false;
        const int n = min(d.units, budget);
        if (n > 0) prefetch_item_tiles<kCompressed>(a, d, mb, n, lane);
        __syncwarp();
        budget -= n;
        return budget > 0;
      });
    }
    __syncthreads();
  }
  wait_prior_grid();          // inputs may come from the preceding grid
  allow_next_grid();
  const uint64_t policy = l2_evict_first_policy();
  uint32_t inflight = 0;        // consumer: bit s: stage s has copies armed and not yet waited for
  bool prefetched = false;      // consumer: this warp's first tile of the current item is already in flight
  // The planned first item.  The metadata warp re-reads the plan's page-table and directory
  // entries and loads its q rows alongside the lengths below (one round trip instead of lengths,
  // then page table, then directory); each consumer warp then starts the copy of its first tile
  // (K/V are final after the wait, and the plan's addresses are in range whatever it read), before
  // the plan is confirmed.  The copies go out after the lengths, not before: a burst of tile copies
  // ahead of them slows those small loads down.
  ItemDesc plan{};
  plan.b = -1;
  int check_pid[kPagesPerLane], check_dir[kPagesPerLane];
  uint32_t qv[2 * kHeadsPerSlice];
  int plan_tile = kKindInvalid;     // consumer: the plan's entry for this warp's first tile
  if (plan_early) {
    plan = desc[0];
    if (warp < kWarps && plan.b >= 0 && warp < plan.units) plan_tile = meta[warp];   // read before the barrier
    if (warp == kWarps && plan.b >= 0) {
      const int32_t* row = a.page_table + static_cast<size_t>(plan.b) * a.max_pages + plan.pg0;
#pragma unroll
      for (int k = 0; k < kPagesPerLane; ++k) {
        const int i = lane + 32 * k;
        check_pid[k] = i < plan.npg ? row[i] : -1;
        check_dir[k] = kCompressed && i < plan.npg && plan_pid[k] >= 0 && plan_pid[k] < a.num_pages
                           ? a.dir[static_cast<size_t>(plan_pid[k]) * a.hkv + plan.g]
                           : -1;
      }
      load_q<kMulti>(a, plan, lane, qv);
    }
  }
  load_lengths<false, C::kThreads>(a, prefix, lens, tid, held_len, plan_early ? lengths_changed : nullptr);
  if (warp < kWarps && (plan_tile & 3) != kKindInvalid &&
      issue_tile<kCompressed>(a, plan, &plan_tile, 0, stages + static_cast<size_t>(warp) * kWarpStages * C::kStageBytes,
                              &bars[warp * kWarpStages], lane, policy)) {
    inflight = 1u;
    prefetched = true;
  }
  const int total = HS * prefix[a.batch];       // pages (items) of all pairs (the host bounds it below 2^30)
  const Ranges g = make_ranges(a, total);

  if (warp == kWarps) {
    // ============================================================== metadata warp
    // Walk this CTA's page range, publishing one item at a time (double buffered), then an end
    // marker.
    // The plan holds if no length changed and every page of the planned item reads the same page
    // id and directory entry as before, all of them valid (so the skipped resolve would have
    // reported nothing).
    bool plan_ok = false;
    if (plan.b >= 0) {
      bool ok = true;
#pragma unroll
      for (int k = 0; k < kPagesPerLane; ++k) {
        const int i = lane + 32 * k;
        if (i < plan.npg) {
          const int pid = plan_pid[k], dd = plan_dir[k];
          ok = ok && check_pid[k] == pid;
          if (kCompressed)
            ok = ok && pid >= 0 && pid < a.num_pages && check_dir[k] == dd &&
                 (dd == ZF_DIR_COMPRESSED || (dd >= 0 && dd < a.num_raw));
          else
            ok = ok && pid >= 0 && pid < a.num_raw;
        }
      }
      plan_ok = __all_sync(0xFFFFFFFFu, ok) && !*lengths_changed;
    }
    int k = 0;
    if (a.publish_delay_ns) sleep_for_ns(a.publish_delay_ns);    // tests: the consumers' waits run out
    auto publish = [&](const ItemDesc& piece) -> bool {
      const int buf = k & 1;
      bool good = true;
      if (lane == 0) good = !*abort_flag && mbar_wait(&item_empty[buf], ((k >> 1) & 1u) ^ 1u);
      good = __shfl_sync(0xFFFFFFFFu, good, 0);
      if (!good) {
        if (lane == 0) {
          report(a.status, ZF_DEV_TIMEOUT);
          *abort_flag = 1;
        }
        return false;
      }
      ItemDesc d = piece;
      // the first item as planned: meta buffer 0 already holds its tiles and qv its q rows
      d.planned = k == 0 && plan_ok && d.b >= 0 && same_piece(d, plan);
      if (d.b >= 0 && !d.planned) resolve_tiles<kCompressed>(a, d, meta + buf * kMaxItemTiles, lane);
      __syncwarp();
      if (lane == 0) {
        desc[buf] = d;
        mbar_arrive(&item_full[buf]);        // release: the tiles can be fetched
      }
      if (d.b >= 0) {
        if (!d.planned) load_q<kMulti>(a, d, lane, qv);
        store_q(qbuf + buf * kHeadsPerSlice * kQRowBytes, lane, qv);
        __syncwarp();
        if (lane == 0) mbar_arrive(&q_full[buf]);   // release: the q rows
      }
      ++k;
      return true;
    };
    if (walk_range(a, prefix, lens, g, HS, publish)) {
      ItemDesc end_marker{};
      end_marker.b = -1;
      publish(end_marker);
    }
    return;
  }

  // ================================================================== consumer warps
  // partials per pair, for the merge kernel (spread over all CTAs; off the metadata warp's path)
  for (int p = blockIdx.x * (kWarps * 32) + tid; p < a.batch * HS; p += gridDim.x * (kWarps * 32)) {
    const int b = p / HS, r = p - b * HS;
    const int n = prefix[b + 1] - prefix[b];
    a.chunk_counts[p] = a.chunk_pages > 0 ? n : n > 0 ? pair_chunks(g, HS * prefix[b] + r * n, n) : 0;
  }
  const int gi = lane >> 2, ti = lane & 3;
  uint8_t* my_stages = stages + static_cast<size_t>(warp) * kWarpStages * C::kStageBytes;
  uint64_t* my_bars = bars + warp * kWarpStages;
  bool aborted = false;
  int sidx = 0;                 // stage of the next tile to consume
  uint32_t phase = 0;           // bit s: parity of the next wait on stage s
  for (int k = 0;; ++k) {
    const int buf = k & 1;
    if (!aborted && (*abort_flag || !mbar_wait(&item_full[buf], (k >> 1) & 1u, a.wait_limit_ns))) {
      aborted = true;
      *abort_flag = 1;
      report(a.status, ZF_DEV_TIMEOUT);
    }
    // one decision for all consumer warps: stop at the end marker, or once any wait gave up
    if (consumer_any<kWarps>(aborted || desc[buf].b < 0)) break;
    const ItemDesc d = desc[buf];
    const int* m = meta + buf * kMaxItemTiles;
    if (k == 0 && prefetched && !d.planned) {
      // the copy started from the plan is not this item's: let it land, then start over
      prefetched = false;
      if (!aborted) {
        if (*abort_flag || !mbar_wait(&my_bars[0], phase & 1u)) {
          aborted = true;
          *abort_flag = 1;
          report(a.status, ZF_DEV_TIMEOUT);
        } else {
          phase ^= 1u;
          inflight &= ~1u;
        }
      }
    }
    // Q^T as the B operand (k = channel, n = head): one 16-byte read gives this lane's words of
    // k-steps 2j and 2j+1 (rows past the group's heads are zero)
    const uint8_t* qrow = qbuf + (buf * kHeadsPerSlice + gi) * kQRowBytes + 16 * ti;

    float m0 = kMulti ? kNoScore : -CUDART_INF_F, m1 = m0, l0 = 0.f, l1 = 0.f;
    // several new tokens: the token of column c (query head d.h0 + c) is (d.h0 + c) % T and sees
    // positions up to causal_lim + token
    const int causal_lim = kMulti ? lens[d.b] - a.tokens : 0;
    float o[8][4];
#pragma unroll
    for (int mt = 0; mt < 8; ++mt) o[mt][0] = o[mt][1] = o[mt][2] = o[mt][3] = 0.f;

    // this warp's first tile of the item, unless it was prefetched during the previous item
    if (!prefetched && warp < d.units) {
      if (issue_tile<kCompressed>(a, d, m, warp, my_stages + sidx * C::kStageBytes, &my_bars[sidx], lane, policy))
        inflight |= 1u << sidx;
    }
    prefetched = false;
    if (!aborted && (*abort_flag || !mbar_wait(&q_full[buf], (k >> 1) & 1u, a.wait_limit_ns))) {
      aborted = true;
      *abort_flag = 1;
      report(a.status, ZF_DEV_TIMEOUT);
    }

    for (int u = warp; u < d.units && !aborted; u += kWarps) {
      // prefetch the warp's next tile: the next one of this item, or its first one of the next item
      const int un = u + kWarps;
      const int ns = sidx ^ 1;
      uint8_t* next_stage = my_stages + ns * C::kStageBytes;
      if (un < d.units) {
        if (issue_tile<kCompressed>(a, d, m, un, next_stage, &my_bars[ns], lane, policy)) inflight |= 1u << ns;
      } else {
        const int nb = buf ^ 1;       // the next item (or the end marker) is published after this one
        if (*abort_flag || !mbar_wait(&item_full[nb], ((k + 1) >> 1) & 1u, a.wait_limit_ns)) {
          aborted = true;
          *abort_flag = 1;
          report(a.status, ZF_DEV_TIMEOUT);
          break;
        } else if (desc[nb].b >= 0 && warp < desc[nb].units) {
          if (issue_tile<kCompressed>(a, desc[nb], meta + nb * kMaxItemTiles, warp, next_stage, &my_bars[ns], lane,
                                      policy))
            inflight |= 1u << ns;
          prefetched = true;
        }
      }
      // wait for the current tile
      if (inflight & (1u << sidx)) {
        if (*abort_flag || !mbar_wait(&my_bars[sidx], (phase >> sidx) & 1u)) {
          aborted = true;
          *abort_flag = 1;
          report(a.status, ZF_DEV_TIMEOUT);
          break;
        }
        phase ^= 1u << sidx;
        inflight &= ~(1u << sidx);
      }

      const int kind = m[u] & 3;
      if (kind != kKindInvalid) {
        uint8_t* kp = my_stages + sidx * C::kStageBytes;
        const bool comp = kCompressed && kind == kKindComp;
        const int ntok = min(16, d.t1 - (d.t0 + 16 * u));

        // ---- S^T (16 tokens x 8 heads) = K (16 x 128) . Q^T (128 x 8); two accumulation chains.
        // The common case (compressed, no escape in the four K blocks) runs a branch-free loop.
        float sa[4] = {0.f, 0.f, 0.f, 0.f}, sb[4] = {0.f, 0.f, 0.f, 0.f};
        uint32_t hdr[4] = {0u, 0u, 0u, 0u};
        bool fast = false;
        if (comp) {
#pragma unroll
          for (int j = 0; j < 4; ++j) hdr[j] = *reinterpret_cast<const uint32_t*>(kp + j * kSlotBytes + kHeaderAt);
          fast = ((hdr[0] | hdr[1] | hdr[2] | hdr[3]) & kHeaderEscMask) == 0;
        }
        if (fast) {
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            uint32_t ka[8];
            rebuild_lane_noesc(kp + j * kSlotBytes, lane, __byte_perm(hdr[j], 0u, 0x0000u), ka);
            const uint4 q = *reinterpret_cast<const uint4*>(qrow + 64 * j);
            float(&acc)[4] = (j & 1) ? sb : sa;
            mma_bf16(acc, ka[0], ka[1], ka[2], ka[3], q.x, q.y);
            mma_bf16(acc, ka[4], ka[5], ka[6], ka[7], q.z, q.w);
          }
        } else {
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            uint32_t ka[8];
            if (comp) rebuild_lane(kp + j * kSlotBytes, lane, ka);
            else load_raw_lane(kp + j * kRawBlockBytes, lane, ka);
            const uint4 q = *reinterpret_cast<const uint4*>(qrow + 64 * j);
            float(&acc)[4] = (j & 1) ? sb : sa;
            mma_bf16(acc, ka[0], ka[1], ka[2], ka[3], q.x, q.y);
            mma_bf16(acc, ka[4], ka[5], ka[6], ka[7], q.z, q.w);
          }
        }
        const uint8_t* vp = kp + C::kVOffset;
        if (kCompressed && !comp) {      // raw tile in the compressed kernel: V goes where K was
          __syncwarp();                  // every lane is done reading the K half
          issue_raw_v(a, d, m, u, kp, &my_bars[sidx], lane, policy);
          if (*abort_flag || !mbar_wait(&my_bars[sidx], (phase >> sidx) & 1u)) {
            aborted = true;
            *abort_flag = 1;
            report(a.status, ZF_DEV_TIMEOUT);
            break;
          }
          phase ^= 1u << sidx;
          vp = kp;
        }

        // ---- online softmax, log2 domain.  lane: tokens gi, gi+8 x heads 2ti, 2ti+1
        float x0 = (sa[0] + sb[0]) * a.scale_log2, x1 = (sa[1] + sb[1]) * a.scale_log2;
        float x2 = (sa[2] + sb[2]) * a.scale_log2, x3 = (sa[3] + sb[3]) * a.scale_log2;
        uint32_t keep_a = 0xFFFFFFFFu, keep_b = 0xFFFFFFFFu;
        if (ntok < 16) {
          if (gi >= ntok) x0 = x1 = -CUDART_INF_F;
          if (gi + 8 >= ntok) x2 = x3 = -CUDART_INF_F;
          // tokens past the context may hold anything (even NaN): their values are zeroed so that
          // p = 0 times them stays 0.  V^T columns of this lane: tokens 2ti, 2ti+1 (regs 0,1,4,5)
          // and 2ti+8, 2ti+9 (regs 2,3,6,7).
          keep_a = (2 * ti < ntok ? 0x0000FFFFu : 0u) | (2 * ti + 1 < ntok ? 0xFFFF0000u : 0u);
          keep_b = (2 * ti + 8 < ntok ? 0x0000FFFFu : 0u) | (2 * ti + 9 < ntok ? 0xFFFF0000u : 0u);
        }
        if (kMulti) {
          const int pos = d.t0 + 16 * u + gi;          // this lane's first row; the second is pos + 8
          if (pos + 8 > causal_lim) {
            const int ta = causal_lim + (d.h0 + 2 * ti) % a.tokens;
            const int tb = causal_lim + (d.h0 + 2 * ti + 1) % a.tokens;
            if (pos > ta) x0 = -CUDART_INF_F;
            if (pos > tb) x1 = -CUDART_INF_F;
            if (pos + 8 > ta) x2 = -CUDART_INF_F;
            if (pos + 8 > tb) x3 = -CUDART_INF_F;
          }
        }
        const bool grow = fmaxf(x0, x2) > m0 + kRescaleThreshold || fmaxf(x1, x3) > m1 + kRescaleThreshold;
        if (__any_sync(0xFFFFFFFFu, grow)) {
          float mx0 = fmaxf(x0, x2), mx1 = fmaxf(x1, x3);
#pragma unroll
          for (int dd = 4; dd < 32; dd <<= 1) {
            mx0 = fmaxf(mx0, __shfl_xor_sync(0xFFFFFFFFu, mx0, dd));
            mx1 = fmaxf(mx1, __shfl_xor_sync(0xFFFFFFFFu, mx1, dd));
          }
          const float mn0 = fmaxf(m0, mx0), mn1 = fmaxf(m1, mx1);   // finite: token 0 is valid (kNoScore at least)
          const float al0 = fast_exp2(m0 - mn0), al1 = fast_exp2(m1 - mn1);
          m0 = mn0;
          m1 = mn1;
          l0 *= al0;
          l1 *= al1;
#pragma unroll
          for (int mt = 0; mt < 8; ++mt) {
            o[mt][0] *= al0;
            o[mt][1] *= al1;
            o[mt][2] *= al0;
            o[mt][3] *= al1;
          }
        }
        const float p0 = fast_exp2(x0 - m0), p1 = fast_exp2(x1 - m1);
        const float p2 = fast_exp2(x2 - m0), p3 = fast_exp2(x3 - m1);
        l0 += p0 + p2;
        l1 += p1 + p3;
        // P^T as the B operand (k = token, n = head): high BF16 part and BF16 remainder
        const uint32_t h01 = pack_bf16x2(p0, p1), h23 = pack_bf16x2(p2, p3);
        const uint32_t r01 = pack_bf16x2(p0 - bf16lo_to_f32(h01), p1 - bf16hi_to_f32(h01));
        const uint32_t r23 = pack_bf16x2(p2 - bf16lo_to_f32(h23), p3 - bf16hi_to_f32(h23));
        const uint32_t bh0 = transpose8x8(h01), bh1 = transpose8x8(h23);
        const uint32_t bl0 = transpose8x8(r01), bl1 = transpose8x8(r23);

        // ---- O^T (128 channels x 8 heads) += V^T (128 x 16 tokens) . P^T (16 x 8).  Branch-free
        // loop for a full compressed tile without escapes in its V blocks.
        fast = false;
        if (comp && ntok == 16) {
#pragma unroll
          for (int j = 0; j < 4; ++j) hdr[j] = *reinterpret_cast<const uint32_t*>(vp + j * kSlotBytes + kHeaderAt);
          fast = ((hdr[0] | hdr[1] | hdr[2] | hdr[3]) & kHeaderEscMask) == 0;
        }
        if (fast) {
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            uint32_t va[8];
            rebuild_lane_noesc(vp + j * kSlotBytes, lane, __byte_perm(hdr[j], 0u, 0x0000u), va);
            mma_bf16(o[2 * j], va[0], va[1], va[2], va[3], bh0, bh1);
            mma_bf16(o[2 * j + 1], va[4], va[5], va[6], va[7], bh0, bh1);
            mma_bf16(o[2 * j], va[0], va[1], va[2], va[3], bl0, bl1);
            mma_bf16(o[2 * j + 1], va[4], va[5], va[6], va[7], bl0, bl1);
          }
        } else {
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            uint32_t va[8];
            if (comp) rebuild_lane(vp + j * kSlotBytes, lane, va);
            else load_raw_lane(vp + j * kRawBlockBytes, lane, va);
            if (ntok < 16) {         // the context's last tile only
              va[0] &= keep_a; va[1] &= keep_a; va[4] &= keep_a; va[5] &= keep_a;
              va[2] &= keep_b; va[3] &= keep_b; va[6] &= keep_b; va[7] &= keep_b;
            }
            mma_bf16(o[2 * j], va[0], va[1], va[2], va[3], bh0, bh1);
            mma_bf16(o[2 * j + 1], va[4], va[5], va[6], va[7], bh0, bh1);
            mma_bf16(o[2 * j], va[0], va[1], va[2], va[3], bl0, bl1);
            mma_bf16(o[2 * j + 1], va[4], va[5], va[6], va[7], bl0, bl1);
          }
        }
      }
      __syncwarp();                // the stage may now be refilled
      sidx ^= 1;
    }

    // ---- merge the warps' states of this item through shared memory.  Each warp writes its state
    // into its stage that holds no tile in flight (the one it consumed last).
#pragma unroll
    for (int dd = 4; dd < 32; dd <<= 1) {
      l0 += __shfl_xor_sync(0xFFFFFFFFu, l0, dd);
      l1 += __shfl_xor_sync(0xFFFFFFFFu, l1, dd);
    }
    float* my_combine = reinterpret_cast<float*>(my_stages + (sidx ^ 1) * C::kStageBytes);
    float* cm = my_combine + kHeadsPerSlice * kOStride;
    float* cl = cm + kHeadsPerSlice;
    if (lane == 0) combine_stage[warp] = sidx ^ 1;
    if (gi == 0) {
      cm[2 * ti] = m0;
      cm[2 * ti + 1] = m1;
      cl[2 * ti] = l0;
      cl[2 * ti + 1] = l1;
    }
#pragma unroll
    for (int mt = 0; mt < 8; ++mt) {
      my_combine[(2 * ti) * kOStride + 16 * mt + gi] = o[mt][0];
      my_combine[(2 * ti + 1) * kOStride + 16 * mt + gi] = o[mt][1];
      my_combine[(2 * ti) * kOStride + 16 * mt + gi + 8] = o[mt][2];
      my_combine[(2 * ti + 1) * kOStride + 16 * mt + gi + 8] = o[mt][3];
    }
    consumer_barrier<kWarps>();
    if (!aborted) {
      const int hh = warp;                     // warps 0..7 finish head hh, channels 4*lane..+3
      if (hh < d.nh) {
        float mw[kWarps];
        float M = -CUDART_INF_F;
#pragma unroll
        for (int w = 0; w < kWarps; ++w) {
          const float* cwp = reinterpret_cast<const float*>(
              stages + (static_cast<size_t>(w) * kWarpStages + combine_stage[w]) * C::kStageBytes);
          mw[w] = cwp[kHeadsPerSlice * kOStride + hh];
          M = fmaxf(M, mw[w]);
        }
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
        float lsum = 0.f;
        if (M != -CUDART_INF_F) {
#pragma unroll
          for (int w = 0; w < kWarps; ++w) {
            const float* cwp = reinterpret_cast<const float*>(
                stages + (static_cast<size_t>(w) * kWarpStages + combine_stage[w]) * C::kStageBytes);
            const float f = exp2f(mw[w] - M);
            lsum += f * cwp[kHeadsPerSlice * kOStride + kHeadsPerSlice + hh];
            const float4 v = *reinterpret_cast<const float4*>(cwp + hh * kOStride + 4 * lane);
            acc.x += f * v.x;
            acc.y += f * v.y;
            acc.z += f * v.z;
            acc.w += f * v.w;
          }
        }
        const float inv = lsum > 0.f ? 1.f / lsum : 0.f;
        acc.x *= inv;
        acc.y *= inv;
        acc.z *= inv;
        acc.w *= inv;
        const float lse2 = lsum > 0.f ? M + log2f(lsum) : -CUDART_INF_F;
        const size_t bh = static_cast<size_t>(d.b) * a.hq + d.h0 + hh;
        if (d.single) {
          const size_t row = kMulti ? query_row(d.b, d.h0 + hh, a.tokens, a.hq) : bh;
          *reinterpret_cast<float4*>(a.out + row * ZF_HEAD_DIM + 4 * lane) = acc;
          if (lane == 0) a.lse[row] = lse2 * kLn2;
        } else {
          const size_t pidx = bh * a.max_chunks + d.c;
          *reinterpret_cast<float4*>(a.part_o + pidx * ZF_HEAD_DIM + 4 * lane) = acc;
          if (lane == 0) a.part_lse[pidx] = lse2;
        }
      }
    }
    consumer_barrier<kWarps>();
    if (lane == 0) mbar_arrive(&item_empty[buf]);     // this item's metadata and q are free
  }
  // copies still in flight (only after a wait gave up) must land before the CTA exits
  for (int st = 0; st < kWarpStages; ++st)
    if (inflight & (1u << st)) mbar_wait(&my_bars[st], (phase >> st) & 1u);
}

// One warp per (request, query head): lse = log2 sum_i 2^lse_i, out = sum_i 2^(lse_i - lse) o_i.
// Requests with one chunk were finished by the attention kernel; empty requests get 0 / -inf.
// The first 32 chunk LSEs and the first kPreload chunk outputs are loaded together with the chunk
// count (slots past the count hold stale values and are never used), so the chain is one round
// trip to L2 instead of three.  Blocks of two warps; the kernel's 64 registers per thread fit on an
// SM sub-partition beside four attention warps of at most 112 registers.
constexpr int kPreload = 8;
constexpr int kMergeWarps = 2;
template <bool kMulti>
__global__ void __launch_bounds__(kMergeWarps * 32) merge_kernel(const MergeArgs a) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // The next grid (the next call's attention) may launch right away: its CTAs take SMs as this
  // call's attention CTAs retire and use the wait to prefetch; they read nothing final before
  // this grid completes.
  allow_next_grid();
  wait_prior_grid();                       // the attention grid's partials
  const int idx = blockIdx.x * kMergeWarps + warp;
  if (idx >= a.batch * a.hq) return;
  const int b = idx / a.hq, h = idx - b * a.hq;
  const int gq = h / a.group;
  const float* pl = a.part_lse + static_cast<size_t>(idx) * a.max_chunks;
  const float4* po = reinterpret_cast<const float4*>(a.part_o + static_cast<size_t>(idx) * a.max_chunks * ZF_HEAD_DIM) + lane;
  const float lse_lane = lane < a.max_chunks ? pl[lane] : -CUDART_INF_F;
  float4 pre[kPreload];
#pragma unroll
  for (int j = 0; j < kPreload; ++j)
    pre[j] = j < a.max_chunks ? po[static_cast<size_t>(j) * (ZF_HEAD_DIM / 4)] : make_float4(0.f, 0.f, 0.f, 0.f);
  const int nch = a.chunk_counts[(b * (a.hq / a.group) + gq) * a.slices + (h - gq * a.group) / a.hps];
  const size_t row = kMulti ? query_row(b, h, a.tokens, a.hq) : static_cast<size_t>(idx);
  float4* outp = reinterpret_cast<float4*>(a.out + row * ZF_HEAD_DIM) + lane;
  if (nch == 1) return;
  // chunk log-sum-exps, one per lane: max and sum of 2^(lse_i - max) by warp reductions
  float M = lane < nch ? lse_lane : -CUDART_INF_F;
  for (int i = lane + 32; i < nch; i += 32) M = fmaxf(M, pl[i]);
#pragma unroll
  for (int d = 16; d > 0; d >>= 1) M = fmaxf(M, __shfl_xor_sync(0xFFFFFFFFu, M, d));
  if (nch == 0 || M == -CUDART_INF_F) {
    *outp = make_float4(0.f, 0.f, 0.f, 0.f);
    if (lane == 0) a.lse[row] = -CUDART_INF_F;
    return;
  }
  const float w0 = lane < nch ? fast_exp2(lse_lane - M) : 0.f;
  float lsum = w0;
  for (int i = lane + 32; i < nch; i += 32) lsum += fast_exp2(pl[i] - M);
#pragma unroll
  for (int d = 16; d > 0; d >>= 1) lsum += __shfl_xor_sync(0xFFFFFFFFu, lsum, d);
  // weighted sum of the chunk outputs: lane owns 4 channels; weights come from the owning lane
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
  for (int j = 0; j < kPreload; ++j) {
    const float f = __shfl_sync(0xFFFFFFFFu, w0, j);
    if (j < nch) {
      acc.x += f * pre[j].x;
      acc.y += f * pre[j].y;
      acc.z += f * pre[j].z;
      acc.w += f * pre[j].w;
    }
  }
  for (int c0 = 0; c0 < nch; c0 += 32) {
    const float w = c0 == 0 ? w0 : (c0 + lane < nch ? fast_exp2(pl[c0 + lane] - M) : 0.f);
    const int n = min(32, nch - c0);
    for (int j = c0 == 0 ? kPreload : 0; j < n; ++j) {
      const float f = __shfl_sync(0xFFFFFFFFu, w, j);
      const float4 v = po[static_cast<size_t>(c0 + j) * (ZF_HEAD_DIM / 4)];
      acc.x += f * v.x;
      acc.y += f * v.y;
      acc.z += f * v.z;
      acc.w += f * v.w;
    }
  }
  const float inv = __fdividef(1.f, lsum);
  *outp = make_float4(acc.x * inv, acc.y * inv, acc.z * inv, acc.w * inv);
  if (lane == 0) a.lse[row] = (M + fast_log2(lsum)) * kLn2;
}

// Which kernel a compressed call runs.  ZF_KERNEL_AUTO runs the tensor-memory kernel when a kv head
// has more than 8 query columns (query heads per kv head x new tokens), where the warp-MMA kernel
// would read its tiles twice or more, and the warp-MMA kernel otherwise.  Measured on GB300 (the
// benchmark's CUDA-graph step, one layer of 8192-token contexts): 28-32 columns 1.88-2.00x faster
// (GQA-7 with 4 new tokens 526 against 990 us), 14-16 columns 1.18-1.26x faster (GQA-7 with 2 new
// tokens 427 against 503 us, GQA-4 with 4 new tokens 274 against 340 us).
// Returns whether it is the tensor-memory kernel, or -1 when that kernel was asked for and cannot
// run these sizes.
static int pick_tc(int32_t kernel, int batch, int hq, int hkv) {
  if (kernel == ZF_KERNEL_TCGEN05) return attention_tc_fits(batch, hq, hkv) ? 1 : -1;
  if (kernel == ZF_KERNEL_AUTO && hq / hkv > 8 && attention_tc_fits(batch, hq, hkv)) return 1;
  return 0;
}

static Plan compressed_plan(bool tc, int batch, int hq, int hkv, int page_size, int max_pages, int num_sms) {
  return tc ? attention_tc_plan(batch, hq, hkv, page_size, max_pages, num_sms)
            : make_plan(batch, hq, hkv, page_size, max_pages, num_sms, Cfg<true>::kWarps);
}

// Workspace that serves every attention kernel (the largest of their plans).
static size_t plan_workspace(int batch, int hq, int hkv, int page_size, int max_pages, int num_sms) {
  size_t w = make_plan(batch, hq, hkv, page_size, max_pages, num_sms, Cfg<true>::kWarps).ws_bytes;
  const size_t d = make_plan(batch, hq, hkv, page_size, max_pages, num_sms, Cfg<false>::kWarps).ws_bytes;
  w = w > d ? w : d;
  if (attention_tc_fits(batch, hq, hkv)) {
    const size_t t = attention_tc_plan(batch, hq, hkv, page_size, max_pages, num_sms).ws_bytes;
    w = w > t ? w : t;
  }
  return w;
}

template <bool kCompressed>
static zf_status launch_attention(const zf_cache* c, const uint16_t* q, int32_t batch, int32_t tokens, int32_t hq_in,
                                  const int32_t* page_table, int32_t max_pages, const int32_t* seq_lens,
                                  float scale, float* out, float* lse, void* workspace, size_t ws_bytes,
                                  void* stream, int32_t kernel = ZF_KERNEL_AUTO,
                                  uint64_t wait_limit_ns = kWaitTimeoutNs, uint64_t publish_delay_ns = 0) {
  if (kernel != ZF_KERNEL_AUTO && kernel != ZF_KERNEL_WARP_MMA && kernel != ZF_KERNEL_TCGEN05)
    return ZF_ERR_INVALID_ARGUMENT;
  zf_status st = check_cache(c, kCompressed, true, kCompressed);
  if (st != ZF_OK) return st;
  if (!tokens_ok(tokens, hq_in)) return ZF_ERR_INVALID_ARGUMENT;
  const int32_t hq = hq_in * tokens;
  if (!attn_shape_ok(batch, hq_in, c->num_kv_heads, max_pages) || !attn_shape_ok(batch, hq, c->num_kv_heads, max_pages))
    return ZF_ERR_INVALID_ARGUMENT;
  if (batch == 0) return ZF_OK;
  if (!q || !page_table || !seq_lens || !out || !lse || !workspace) return ZF_ERR_INVALID_ARGUMENT;
  if (!aligned16(q) || !aligned16(out) || !aligned16(workspace) || (reinterpret_cast<uintptr_t>(lse) & 3u) ||
      (reinterpret_cast<uintptr_t>(page_table) & 3u) || (reinterpret_cast<uintptr_t>(seq_lens) & 3u))
    return ZF_ERR_INVALID_ARGUMENT;
  if (!(scale == scale)) return ZF_ERR_INVALID_ARGUMENT;
  // tile entries pack a slot id into 26 bits
  if (c->num_pages >= (1 << 26) || c->num_raw_slots >= (1 << 26)) return ZF_ERR_UNSUPPORTED;
  int sms = 0;
  if ((st = current_sm_count(&sms)) != ZF_OK) return st;
  const int tc = kCompressed ? pick_tc(kernel, batch, hq, c->num_kv_heads) : 0;
  if (tc < 0) return ZF_ERR_UNSUPPORTED;
  const Plan p = kCompressed ? compressed_plan(tc > 0, batch, hq, c->num_kv_heads, c->page_size, max_pages, sms)
                             : make_plan(batch, hq, c->num_kv_heads, c->page_size, max_pages, sms, Cfg<false>::kWarps);
  if (ws_bytes < p.ws_bytes) return ZF_ERR_WORKSPACE_TOO_SMALL;

  AttnArgs a{};
  a.k_comp = c->k_comp;
  a.v_comp = c->v_comp;
  a.k_raw = reinterpret_cast<const uint8_t*>(c->k_raw);
  a.v_raw = reinterpret_cast<const uint8_t*>(c->v_raw);
  a.dir = c->dir;
  a.status = c->status;
  a.q = q;
  a.page_table = page_table;
  a.seq_lens = seq_lens;
  a.out = out;
  a.lse = lse;
  a.part_o = static_cast<float*>(workspace);
  a.part_lse = reinterpret_cast<float*>(static_cast<uint8_t*>(workspace) + p.part_o_bytes);
  a.chunk_counts = reinterpret_cast<int32_t*>(static_cast<uint8_t*>(workspace) + p.part_o_bytes + p.part_lse_bytes);
  a.batch = batch;
  a.hq = hq;
  a.hkv = c->num_kv_heads;
  a.group = hq / c->num_kv_heads;
  a.tokens = tokens;
  a.hps = kHeadsPerSlice;
  a.slices = p.slices;
  a.page_size = c->page_size;
  a.num_pages = c->num_pages;
  a.num_raw = c->num_raw_slots;
  a.max_pages = max_pages;
  a.max_chunks = p.max_chunks;
  a.min_range_pages = p.min_range_pages;
  a.chunk_pages = p.chunk_pages;
  a.prefetch = p.prefetch ? 1 : 0;
  a.plan_first = p.plan_first ? 1 : 0;
  a.comp_head_bytes = static_cast<int64_t>(c->page_size / 4) * kSlotBytes;
  a.raw_head_bytes = static_cast<int64_t>(c->page_size / 4) * kRawBlockBytes;
  a.scale_log2 = scale * 1.4426950408889634f;
  a.wait_limit_ns = wait_limit_ns;
  a.publish_delay_ns = publish_delay_ns;

  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (tc > 0) return launch_attention_tc(a, p, tokens, s);
  const size_t smem = smem_layout<kCompressed>(batch).total;
  const bool multi = tokens > 1;
  const void* fn = multi ? reinterpret_cast<const void*>(attn_kernel<kCompressed, true>)
                         : reinterpret_cast<const void*>(attn_kernel<kCompressed, false>);
  if ((st = ensure_smem_limit(fn, (kCompressed ? 1 : 0) + (multi ? 2 : 0), smem)) != ZF_OK) return st;
  // programmatic dependent launch: each kernel may start while its predecessor in the stream
  // drains, and waits for it (griddepcontrol.wait) before touching inputs or the workspace
  cudaLaunchAttribute pdl[1];
  pdl[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  pdl[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(p.grid);
  cfg.blockDim = dim3(Cfg<kCompressed>::kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cfg.attrs = pdl;
  cfg.numAttrs = 1;
  if ((multi ? cudaLaunchKernelEx(&cfg, attn_kernel<kCompressed, true>, a)
             : cudaLaunchKernelEx(&cfg, attn_kernel<kCompressed, false>, a)) != cudaSuccess)
    return ZF_ERR_CUDA;

  MergeArgs m{};
  m.part_o = a.part_o;
  m.part_lse = a.part_lse;
  m.out = out;
  m.lse = lse;
  m.batch = batch;
  m.hq = hq;
  m.chunk_counts = a.chunk_counts;
  m.group = a.group;
  m.slices = a.slices;
  m.max_chunks = p.max_chunks;
  m.tokens = tokens;
  m.hps = kHeadsPerSlice;
  return launch_merge(m, multi, s);
}

zf_status launch_merge(const MergeArgs& m, bool multi, cudaStream_t stream) {
  // programmatic dependent launch: it starts while the attention grid drains and waits for it
  cudaLaunchAttribute pdl[1];
  pdl[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  pdl[0].val.programmaticStreamSerializationAllowed = 1;
  const int rows = m.batch * m.hq;
  cudaLaunchConfig_t mcfg = {};
  mcfg.gridDim = dim3((rows + kMergeWarps - 1) / kMergeWarps);
  mcfg.blockDim = dim3(kMergeWarps * 32);
  mcfg.dynamicSmemBytes = 0;
  mcfg.stream = stream;
  mcfg.attrs = pdl;
  mcfg.numAttrs = 1;
  if ((multi ? cudaLaunchKernelEx(&mcfg, merge_kernel<true>, m) : cudaLaunchKernelEx(&mcfg, merge_kernel<false>, m)) !=
      cudaSuccess)
    return ZF_ERR_CUDA;
  return ZF_OK;
}

}  // namespace zf

using namespace zf;

extern "C" size_t zf_decode_attn_workspace_size(int32_t batch, int32_t num_q_heads, int32_t num_kv_heads,
                                                int32_t page_size, int32_t max_pages_per_req) {
  if (!attn_shape_ok(batch, num_q_heads, num_kv_heads, max_pages_per_req)) return 0;
  if (page_size < ZF_BLOCK_TOKENS || page_size % ZF_BLOCK_TOKENS || page_size > ZF_MAX_PAGE_SIZE) return 0;
  int sms = 0;
  if (current_sm_count(&sms) != ZF_OK) return 0;
  const size_t ws = plan_workspace(batch, num_q_heads, num_kv_heads, page_size, max_pages_per_req, sms);
  return ws > 0 ? ws : 256;
}

extern "C" size_t zf_decode_attn_multi_workspace_size(int32_t batch, int32_t tokens, int32_t num_q_heads,
                                                      int32_t num_kv_heads, int32_t page_size,
                                                      int32_t max_pages_per_req) {
  if (!tokens_ok(tokens, num_q_heads) || !attn_shape_ok(batch, num_q_heads, num_kv_heads, max_pages_per_req)) return 0;
  return zf_decode_attn_workspace_size(batch, num_q_heads * tokens, num_kv_heads, page_size, max_pages_per_req);
}

extern "C" zf_status zf_decode_attn(const zf_cache* cache, const uint16_t* q, int32_t batch, int32_t num_q_heads,
                                    const int32_t* page_table, int32_t max_pages_per_req, const int32_t* seq_lens,
                                    float softmax_scale, float* out, float* lse, void* workspace,
                                    size_t workspace_bytes, void* stream) {
  return launch_attention<true>(cache, q, batch, 1, num_q_heads, page_table, max_pages_per_req, seq_lens,
                                softmax_scale, out, lse, workspace, workspace_bytes, stream);
}

extern "C" zf_status zf_decode_attn_multi(const zf_cache* cache, const uint16_t* q, int32_t batch, int32_t tokens,
                                          int32_t num_q_heads, const int32_t* page_table, int32_t max_pages_per_req,
                                          const int32_t* seq_lens, float softmax_scale, float* out, float* lse,
                                          void* workspace, size_t workspace_bytes, void* stream) {
  return launch_attention<true>(cache, q, batch, tokens, num_q_heads, page_table, max_pages_per_req, seq_lens,
                                softmax_scale, out, lse, workspace, workspace_bytes, stream);
}

extern "C" zf_status zf_decode_attn_multi_kernel(const zf_cache* cache, const uint16_t* q, int32_t batch,
                                                 int32_t tokens, int32_t num_q_heads, const int32_t* page_table,
                                                 int32_t max_pages_per_req, const int32_t* seq_lens,
                                                 float softmax_scale, float* out, float* lse, void* workspace,
                                                 size_t workspace_bytes, int32_t kernel, void* stream) {
  return launch_attention<true>(cache, q, batch, tokens, num_q_heads, page_table, max_pages_per_req, seq_lens,
                                softmax_scale, out, lse, workspace, workspace_bytes, stream, kernel);
}

extern "C" zf_status zf_decode_attn_wait_test(const zf_cache* cache, const uint16_t* q, int32_t batch, int32_t tokens,
                                              int32_t num_q_heads, const int32_t* page_table,
                                              int32_t max_pages_per_req, const int32_t* seq_lens,
                                              float softmax_scale, float* out, float* lse, void* workspace,
                                              size_t workspace_bytes, int32_t kernel, uint64_t wait_limit_ns,
                                              uint64_t publish_delay_ns, void* stream) {
  if (wait_limit_ns < 1000 || wait_limit_ns > kWaitTimeoutNs || publish_delay_ns > kWaitTimeoutNs)
    return ZF_ERR_INVALID_ARGUMENT;
  return launch_attention<true>(cache, q, batch, tokens, num_q_heads, page_table, max_pages_per_req, seq_lens,
                                softmax_scale, out, lse, workspace, workspace_bytes, stream, kernel, wait_limit_ns,
                                publish_delay_ns);
}

extern "C" zf_status zf_dense_decode_attn(const zf_cache* cache, const uint16_t* q, int32_t batch,
                                          int32_t num_q_heads, const int32_t* page_table, int32_t max_pages_per_req,
                                          const int32_t* seq_lens, float softmax_scale, float* out, float* lse,
                                          void* workspace, size_t workspace_bytes, void* stream) {
  return launch_attention<false>(cache, q, batch, 1, num_q_heads, page_table, max_pages_per_req, seq_lens,
                                 softmax_scale, out, lse, workspace, workspace_bytes, stream);
}

extern "C" zf_status zf_dense_decode_attn_multi(const zf_cache* cache, const uint16_t* q, int32_t batch,
                                                int32_t tokens, int32_t num_q_heads, const int32_t* page_table,
                                                int32_t max_pages_per_req, const int32_t* seq_lens,
                                                float softmax_scale, float* out, float* lse, void* workspace,
                                                size_t workspace_bytes, void* stream) {
  return launch_attention<false>(cache, q, batch, tokens, num_q_heads, page_table, max_pages_per_req, seq_lens,
                                 softmax_scale, out, lse, workspace, workspace_bytes, stream);
}

// ---------------------------------------------------------------------------------------------
// zf_decode_attn_static: the same attention for callers that cannot allocate device memory.
// Its split-KV scratch is this file-scope device array (held by every GPU that loads the library
// until exit).  Host code must not pass `g_static_workspace` itself to a kernel: on the host the
// name is only a stand-in, so the device address is looked up with the caller's device current.
static __device__ __align__(256) unsigned char g_static_workspace[ZF_STATIC_WORKSPACE_BYTES];

namespace {
// Address of g_static_workspace in the current context.  Looked up on every call rather than
// cached per device ordinal: after a device reset, or with another context of the same device
// made current, a cached address would name memory that context does not map.  Once the module
// is loaded the lookup allocates nothing; the first lookup in a context may load it (lazy module
// loading), which is when the array is reserved.
zf_status static_workspace_address(void** out) {
  void* p = nullptr;
  const cudaError_t e = cudaGetSymbolAddress(&p, g_static_workspace);
  if (e == cudaErrorMemoryAllocation) {
    (void)cudaGetLastError();          // not sticky: clear it for the caller's next call
    return ZF_ERR_STATIC_WORKSPACE_UNAVAILABLE;
  }
  if (e != cudaSuccess || !p) return ZF_ERR_CUDA;
  *out = p;
  return ZF_OK;
}
}  // namespace

extern "C" zf_status zf_decode_attn_static(const zf_cache* cache, const uint16_t* q, int32_t batch,
                                           int32_t num_q_heads, const int32_t* page_table,
                                           int32_t max_pages_per_req, const int32_t* seq_lens,
                                           float softmax_scale, float* out, float* lse, void* stream) {
  if (!cache) return ZF_ERR_INVALID_ARGUMENT;
  if (!attn_shape_ok(batch, num_q_heads, cache->num_kv_heads, max_pages_per_req)) return ZF_ERR_INVALID_ARGUMENT;
  const int P = cache->page_size;
  if (P < ZF_BLOCK_TOKENS || P % ZF_BLOCK_TOKENS || P > ZF_MAX_PAGE_SIZE) return ZF_ERR_INVALID_ARGUMENT;
  int sms = 0;
  zf_status st = current_sm_count(&sms);
  if (st != ZF_OK) return st;
  const bool tc = pick_tc(ZF_KERNEL_AUTO, batch, num_q_heads, cache->num_kv_heads) > 0;
  const Plan p = compressed_plan(tc, batch, num_q_heads, cache->num_kv_heads, P, max_pages_per_req, sms);
  if (p.ws_bytes > ZF_STATIC_WORKSPACE_BYTES) return ZF_ERR_STATIC_WORKSPACE_EXCEEDED;
  void* ws = nullptr;
  if ((st = static_workspace_address(&ws)) != ZF_OK) return st;
  return launch_attention<true>(cache, q, batch, 1, num_q_heads, page_table, max_pages_per_req, seq_lens,
                                softmax_scale, out, lse, ws, ZF_STATIC_WORKSPACE_BYTES, stream);
}
