// Decode attention over the compressed paged cache when a kv head has more than 8 query columns
// (GQA groups above 8, or several new tokens per request: columns = query heads per kv head x new
// tokens), on the 5th-generation tensor cores: the rebuilt K and V tiles go to shared memory as
// MMA operands and the scores and the output accumulate in tensor memory, so each kv head's tiles
// are read from HBM once for up to 32 columns (the warp-MMA kernel takes 8 columns per pass and
// reads the tiles once per 8).
//
// ZipFusion §III.C (Attention over the Compressed KV Cache): compressed blocks are copied
// HBM -> shared memory as they are and the exact BF16 values are rebuilt from them with integer
// operations right before the tensor-core instructions; raw blocks need no rebuild.  §IV.B: split
// chunks are combined by a split-result merge.
//
// One CTA per SM, 14 warps:
//  * warps 0-7 (rebuild): warp r takes tile r of every 128-token group of an item (16 tokens of
//    one kv head); it copies its tiles HBM -> its two private stages with 1-D bulk copies (the next
//    tile in flight while it works on this one), rebuilds the tile's K rows into the K operand
//    (A of S^T = K Q^T: 128 tokens x 128 channels) and its V^T columns into the V operand (A of
//    O^T = V^T P^T: 128 channels x 128 tokens), K-major core-matrix layout, straight from the
//    m16n8k16 fragment registers the rebuild produces (one conflict-free 32-bit store per lane
//    fills one 8 x 16-byte core matrix);
//  * warps 8-11 (softmax warpgroup; warp w reads TMEM lanes 32(w%4)..): S^T comes out of tensor
//    memory in the m16n8 accumulator layout, the online softmax runs in the log2 domain with one
//    running max per column shared by the warpgroup (raised only when a score exceeds it by more
//    than 8, after a warpgroup vote; the output in tensor memory is then rescaled in place), and
//    P^T (BF16 high part + BF16 remainder) is transposed with movmatrix into the P operand; at the
//    end of an item it divides O^T by the column sums and writes the output or the partial;
//  * warp 12 (MMA): allocates tensor memory and one lane issues the MMAs: per group 8 x
//    (M128 N{16,32} K16) for S^T into one of two TMEM score buffers, then 2 x 8 for O^T += V^T P^T
//    (high and low parts), signalling completion through tcgen05.commit on mbarriers;
//  * warp 13 (metadata): walks the CTA's items (the warp-MMA kernel's planner and page walk), one
//    item ahead: resolves the pages through the page table and the directory and stages the
//    item's query rows as the B operand of S^T.
// Every wait is bounded (2 s); a wait that gives up sets ZF_DEV_TIMEOUT and the CTA winds down
// (the softmax warpgroup decides together, so its named barriers are always met).
#include <cuda_runtime.h>
#include <math_constants.h>
#include <stdint.h>

#include "zf_attn_common.cuh"

namespace zf {
namespace {

constexpr int kRebuildWarps = 8;
constexpr int kSoftmaxWarp0 = 8;                  // warps 8..11: TMEM lane quadrants 0..3
constexpr int kMmaWarp = 12;
constexpr int kMetaWarp = 13;
constexpr int kTcWarps = 14;
constexpr int kTcThreads = kTcWarps * 32;
constexpr int kTcStageBytes = Cfg<true>::kStageBytes;   // one compressed K + V tile (a raw tile: K, then V)
constexpr int kTcVOffset = Cfg<true>::kVOffset;
constexpr int kOpBytes = 128 * 128 * 2;           // one 128 x 128 BF16 operand
constexpr int kCoreRow = 2048;                    // bytes between core-matrix rows along M/N (16 along K)
constexpr uint32_t kTmemCols = 128;               // two score buffers + the output, <= 32 columns each
constexpr int kSoftmaxBarrier = 1;                // named barrier of the softmax warpgroup

// Barriers (mbarrier index in the shared array).
enum : int {
  kBarStage = 0,                // 2 per rebuild warp: its tile copies
  kBarItemFull = 16,            // [2] the metadata warp published an item
  kBarItemEmpty = 18,           // [2] rebuild + softmax warps are done with it
  kBarQFull = 20,               // [2] the item's query operand is staged
  kBarKFull = 22,               // the 8 rebuild warps wrote a group's K operand
  kBarVFull = 23,               // ... and its V operand
  kBarKFree = 24,               // S^T = K Q^T of a group completed (commit)
  kBarVFree = 25,               // O^T += V^T P^T of a group completed (commit): V and P operands free
  kBarSFull = 26,               // [2] scores of a group in TMEM buffer (commit)
  kBarSFree = 28,               // [2] the softmax warpgroup read that score buffer
  kBarPFull = 30,               // the softmax warpgroup wrote a group's P operand
  kBarOFree = 31,               // the softmax warpgroup read an item's output from TMEM
  kBarDrain = 32,               // end of the CTA: every MMA issued has completed
  kNumBars = 33,
};

struct TcLayout {
  size_t kop, vop, pop, qop, stages, meta, desc, bars, misc, red, prefix, lens, total;
};

template <int kCols>
__host__ __device__ inline TcLayout tc_layout(int batch) {
  TcLayout s;
  size_t at = 0;
  s.kop = at; at += kOpBytes;
  s.vop = at; at += kOpBytes;
  s.pop = at; at += 2 * kCols * 256;              // P^T: high part, then low part (kCols x 128 BF16 each)
  s.qop = at; at += 2 * kCols * 256;              // Q of two items (kCols x 128 BF16 each)
  s.stages = at; at += static_cast<size_t>(kRebuildWarps) * kWarpStages * kTcStageBytes;
  s.meta = at; at += 2 * kMaxItemTiles * 4;
  s.desc = at; at += 2 * 64;
  s.bars = at; at += kNumBars * 8;
  s.misc = at; at += 16;                          // [0] abort flag, [4] TMEM base address
  s.red = at; at += static_cast<size_t>(10 * kCols) * 4;   // column maxima [4][kCols], sums [4][kCols], alpha, max
  s.prefix = at; at += static_cast<size_t>(batch + 1) * 4;
  s.lens = at; at += static_cast<size_t>(batch) * 4;
  s.total = (at + 127) & ~static_cast<size_t>(127);
  return s;
}

// A bounded wait that also gives up at once when another warp already has (abort flag set).
__device__ __forceinline__ bool wait_or_abort(uint64_t* bar, uint32_t parity, volatile int* abort_flag,
                                              int32_t* status) {
  if (*abort_flag) return false;
  if (mbar_wait(bar, parity)) return true;
  *abort_flag = 1;
  report(status, ZF_DEV_TIMEOUT);
  return false;
}

// The softmax warpgroup's barrier, and the same barrier ORing a predicate over its 128 threads.
__device__ __forceinline__ void wg_sync() { asm volatile("bar.sync %0, 128;" ::"n"(kSoftmaxBarrier) : "memory"); }
__device__ __forceinline__ bool wg_any(bool v) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.u32 p, %1, 0;\n\t"
      "bar.red.or.pred q, %2, 128, p;\n\t"
      "selp.u32 %0, 1, 0, q;\n\t}"
      : "=r"(r)
      : "r"(static_cast<uint32_t>(v)), "n"(kSoftmaxBarrier)
      : "memory");
  return r != 0;
}

// K rows of tile p (tokens 16p .. 16p+15 of the group) into the K operand.  Register i of a half
// of a lane's fragment (rows g = lane/4 (+8 for i odd), columns 2(lane%4) (+8 for i >= 2)) is core
// matrix (m-block 2p + (i & 1), k-block 4j + 2h + (i >> 1)) of channel group j, half h.
__device__ __forceinline__ void write_k_tile(const uint8_t* st, bool comp, uint8_t* kop, int p, int lane) {
  uint8_t* base = kop + (2 * p) * kCoreRow + (lane >> 2) * 16 + (lane & 3) * 4;
  uint32_t hdr[4] = {0u, 0u, 0u, 0u};
  bool fast = false;
  if (comp) {
#pragma unroll
    for (int j = 0; j < 4; ++j) hdr[j] = *reinterpret_cast<const uint32_t*>(st + j * kSlotBytes + kHeaderAt);
    fast = ((hdr[0] | hdr[1] | hdr[2] | hdr[3]) & kHeaderEscMask) == 0;
  }
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    uint32_t ka[8];
    if (fast) rebuild_lane_noesc(st + j * kSlotBytes, lane, __byte_perm(hdr[j], 0u, 0x0000u), ka);
    else if (comp) rebuild_lane(st + j * kSlotBytes, lane, ka);
    else load_raw_lane(st + j * kRawBlockBytes, lane, ka);
#pragma unroll
    for (int h = 0; h < 2; ++h)
#pragma unroll
      for (int i = 0; i < 4; ++i)
        *reinterpret_cast<uint32_t*>(base + (i & 1) * kCoreRow + (4 * j + 2 * h + (i >> 1)) * 128) = ka[4 * h + i];
  }
}

// V^T columns of tile p (tokens 16p ..) into the V operand; values of tokens at or past ntok are
// zeroed (they may hold anything).  Register i of a half (V^T rows = channels g (+8 for i odd),
// columns = tokens 2(lane%4) (+8 for i >= 2)) is core matrix (m-block 4j + 2h + (i & 1), k-block
// 2p + (i >> 1)).
__device__ __forceinline__ void write_v_tile(const uint8_t* st, bool comp, int ntok, uint8_t* vop, int p, int lane) {
  const int ti = lane & 3;
  uint8_t* base = vop + (2 * p) * 128 + (lane >> 2) * 16 + ti * 4;
  uint32_t keep_a = 0xFFFFFFFFu, keep_b = 0xFFFFFFFFu;
  if (ntok < 16) {
    keep_a = (2 * ti < ntok ? 0x0000FFFFu : 0u) | (2 * ti + 1 < ntok ? 0xFFFF0000u : 0u);
    keep_b = (2 * ti + 8 < ntok ? 0x0000FFFFu : 0u) | (2 * ti + 9 < ntok ? 0xFFFF0000u : 0u);
  }
  uint32_t hdr[4] = {0u, 0u, 0u, 0u};
  bool fast = false;
  if (comp) {
#pragma unroll
    for (int j = 0; j < 4; ++j) hdr[j] = *reinterpret_cast<const uint32_t*>(st + j * kSlotBytes + kHeaderAt);
    fast = ((hdr[0] | hdr[1] | hdr[2] | hdr[3]) & kHeaderEscMask) == 0;
  }
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    uint32_t va[8];
    if (fast) rebuild_lane_noesc(st + j * kSlotBytes, lane, __byte_perm(hdr[j], 0u, 0x0000u), va);
    else if (comp) rebuild_lane(st + j * kSlotBytes, lane, va);
    else load_raw_lane(st + j * kRawBlockBytes, lane, va);
#pragma unroll
    for (int h = 0; h < 2; ++h)
#pragma unroll
      for (int i = 0; i < 4; ++i)
        *reinterpret_cast<uint32_t*>(base + (4 * j + 2 * h + (i & 1)) * kCoreRow + (i >> 1) * 128) =
            va[4 * h + i] & ((i >> 1) ? keep_b : keep_a);
  }
}

// Zero V^T columns of tile slot p (a group with fewer than 8 tiles, or a page that could not be
// resolved): 16 m-blocks x 2 k-blocks of 128 bytes.
__device__ __forceinline__ void zero_v_tile(uint8_t* vop, int p, int lane) {
#pragma unroll
  for (int e = lane; e < 256; e += 32) {
    const int core = e >> 3;
    *reinterpret_cast<uint4*>(vop + (core >> 1) * kCoreRow + (2 * p + (core & 1)) * 128 + (e & 7) * 16) =
        make_uint4(0u, 0u, 0u, 0u);
  }
}

// The item's query rows as the B operand of S^T = K Q^T (column n = query head d.h0 + n, K-major:
// core matrix (n / 8, channel / 8)); columns past d.nh are zero.
template <int kCols>
__device__ __forceinline__ void stage_q(const AttnArgs& a, const ItemDesc& d, uint8_t* qb, int lane) {
#pragma unroll 4
  for (int it = 0; it < kCols / 2; ++it) {
    const int n = 2 * it + (lane >> 4), ck = lane & 15;
    uint4 v = make_uint4(0u, 0u, 0u, 0u);
    if (n < d.nh) {
      const size_t row = query_row(d.b, d.h0 + n, a.tokens, a.hq);
      v = *reinterpret_cast<const uint4*>(a.q + row * ZF_HEAD_DIM + 8 * ck);
    }
    *reinterpret_cast<uint4*>(qb + (n >> 3) * kCoreRow + ck * 128 + (n & 7) * 16) = v;
  }
}

template <int kCols>
__device__ __forceinline__ void tmem_ld_scores(uint32_t taddr, uint32_t (&r)[kCols / 2]) {
  if constexpr (kCols == 16) tmem_ld_16x256b_x2(taddr, r);
  else tmem_ld_16x256b_x4(taddr, r);
}

template <int kCols>
__global__ void __launch_bounds__(kTcThreads, 1) attn_tc_kernel(const AttnArgs a) {
  constexpr int NJ = kCols / 8;                   // 8-column blocks
  constexpr uint32_t kIdesc = umma_idesc_bf16(128, kCols);
  extern __shared__ __align__(1024) uint8_t smem[];
  const TcLayout L = tc_layout<kCols>(a.batch);
  uint8_t* kop = smem + L.kop;
  uint8_t* vop = smem + L.vop;
  uint8_t* pop = smem + L.pop;                    // high part; the low part follows at + kCols * 256
  uint8_t* qop = smem + L.qop;
  uint8_t* stages = smem + L.stages;
  int* meta = reinterpret_cast<int*>(smem + L.meta);
  ItemDesc* desc = reinterpret_cast<ItemDesc*>(smem + L.desc);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L.bars);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L.misc);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L.misc + 4);
  float* red = reinterpret_cast<float*>(smem + L.red);
  int* prefix = reinterpret_cast<int*>(smem + L.prefix);
  int* lens = reinterpret_cast<int*>(smem + L.lens);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  if (tid == 0) {
    for (int i = 0; i < 2 * kRebuildWarps; ++i) mbar_init(&bars[kBarStage + i], 1);
    for (int b = 0; b < 2; ++b) {
      mbar_init(&bars[kBarItemFull + b], 1);
      mbar_init(&bars[kBarItemEmpty + b], kRebuildWarps + 4);
      mbar_init(&bars[kBarQFull + b], 1);
      mbar_init(&bars[kBarSFull + b], 1);
      mbar_init(&bars[kBarSFree + b], 4);
    }
    mbar_init(&bars[kBarKFull], kRebuildWarps);
    mbar_init(&bars[kBarVFull], kRebuildWarps);
    mbar_init(&bars[kBarKFree], 1);
    mbar_init(&bars[kBarVFree], 1);
    mbar_init(&bars[kBarPFull], 4);
    mbar_init(&bars[kBarOFree], 4);
    mbar_init(&bars[kBarDrain], 1);
    *abort_flag = 0;
  }
  fence_mbar_init();
  if (warp == kMmaWarp) tmem_alloc(tmem_slot, kTmemCols);
  tcgen05_before_sync();
  wait_prior_grid();          // inputs may come from the preceding grid
  allow_next_grid();
  load_lengths<false, kTcThreads>(a, prefix, lens, tid);      // ends with a CTA barrier
  tcgen05_after_sync();
  const uint32_t tmem = *tmem_slot;
  const int HS = a.hkv * a.slices;
  const int total = HS * prefix[a.batch];
  const Ranges g = make_ranges(a, total);

  if (warp == kMetaWarp) {
    // ================================================================== metadata warp
    int k = 0;
    auto publish = [&](const ItemDesc& piece) -> bool {
      const int buf = k & 1;
      bool good = true;
      if (lane == 0) good = wait_or_abort(&bars[kBarItemEmpty + buf], ((k >> 1) & 1) ^ 1, abort_flag, a.status);
      good = __shfl_sync(0xFFFFFFFFu, good, 0);
      if (!good) return false;
      ItemDesc d = piece;
      d.planned = 0;
      if (d.b >= 0) resolve_tiles<true>(a, d, meta + buf * kMaxItemTiles, lane);
      __syncwarp();
      if (lane == 0) {
        desc[buf] = d;
        mbar_arrive(&bars[kBarItemFull + buf]);
      }
      if (d.b >= 0) {
        stage_q<kCols>(a, d, qop + buf * kCols * 256, lane);
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars[kBarQFull + buf]);
      }
      ++k;
      return true;
    };
    if (walk_range(a, prefix, lens, g, HS, publish)) {
      ItemDesc end_marker{};
      end_marker.b = -1;
      publish(end_marker);
    }
  } else if (warp < kRebuildWarps) {
    // ================================================================== rebuild warps
    // partials per pair, for the merge kernel
    for (int p = blockIdx.x * (kRebuildWarps * 32) + tid; p < a.batch * HS; p += gridDim.x * (kRebuildWarps * 32)) {
      const int b = p / HS, r = p - b * HS;
      const int n = prefix[b + 1] - prefix[b];
      a.chunk_counts[p] = a.chunk_pages > 0 ? n : n > 0 ? pair_chunks(g, HS * prefix[b] + r * n, n) : 0;
    }
    const int r = warp;
    uint8_t* my_stages = stages + static_cast<size_t>(r) * kWarpStages * kTcStageBytes;
    uint64_t* my_bars = &bars[kBarStage + kWarpStages * r];
    const uint64_t policy = l2_evict_first_policy();
    uint32_t inflight = 0, phase = 0;
    int sidx = 0, G = 0;
    bool prefetched = false, aborted = false;
    for (int k = 0; !aborted; ++k) {
      const int buf = k & 1;
      if (!wait_or_abort(&bars[kBarItemFull + buf], (k >> 1) & 1, abort_flag, a.status)) break;
      const ItemDesc d = desc[buf];
      if (d.b < 0) break;
      const int* m = meta + buf * kMaxItemTiles;
      const int ng = (d.units + 7) >> 3;
      if (!prefetched && r < d.units &&
          issue_tile<true>(a, d, m, r, my_stages + sidx * kTcStageBytes, &my_bars[sidx], lane, policy))
        inflight |= 1u << sidx;
      prefetched = false;
      for (int gl = 0; gl < ng; ++gl) {
        const int u = 8 * gl + r;
        const int Gg = G + gl;
        if (u < d.units) {
          const int un = u + 8, ns = sidx ^ 1;
          uint8_t* next_stage = my_stages + ns * kTcStageBytes;
          if (un < d.units && issue_tile<true>(a, d, m, un, next_stage, &my_bars[ns], lane, policy))
            inflight |= 1u << ns;
          if (inflight & (1u << sidx)) {
            if (!wait_or_abort(&my_bars[sidx], (phase >> sidx) & 1, abort_flag, a.status)) { aborted = true; break; }
            phase ^= 1u << sidx;
            inflight &= ~(1u << sidx);
          }
          const int kind = m[u] & 3;
          uint8_t* st = my_stages + sidx * kTcStageBytes;
          if (Gg > 0 && !wait_or_abort(&bars[kBarKFree], (Gg - 1) & 1, abort_flag, a.status)) { aborted = true; break; }
          if (kind != kKindInvalid) write_k_tile(st, kind == kKindComp, kop, r, lane);
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) mbar_arrive(&bars[kBarKFull]);
          const uint8_t* vsrc = st + kTcVOffset;
          if (kind == kKindRaw) {                 // a raw tile's V half goes where its K half was
            issue_raw_v(a, d, m, u, st, &my_bars[sidx], lane, policy);
            if (!wait_or_abort(&my_bars[sidx], (phase >> sidx) & 1, abort_flag, a.status)) {
              inflight |= 1u << sidx;            // still in flight: waited for at the end
              aborted = true;
              break;
            }
            phase ^= 1u << sidx;
            vsrc = st;
          }
          if (Gg > 0 && !wait_or_abort(&bars[kBarVFree], (Gg - 1) & 1, abort_flag, a.status)) { aborted = true; break; }
          if (kind != kKindInvalid) write_v_tile(vsrc, kind == kKindComp, min(16, d.t1 - (d.t0 + 16 * u)), vop, r, lane);
          else zero_v_tile(vop, r, lane);
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) mbar_arrive(&bars[kBarVFull]);
          sidx ^= 1;
          if (un >= d.units) {
            // this warp's first tile of the next item (waiting for it only now, after this tile's
            // operands are written: its publication waits for an item whose last MMA needs them)
            const int nb = buf ^ 1;
            if (!wait_or_abort(&bars[kBarItemFull + nb], ((k + 1) >> 1) & 1, abort_flag, a.status)) {
              aborted = true;
              break;
            }
            if (desc[nb].b >= 0 && r < desc[nb].units) {
              if (issue_tile<true>(a, desc[nb], meta + nb * kMaxItemTiles, r, my_stages + sidx * kTcStageBytes,
                                   &my_bars[sidx], lane, policy))
                inflight |= 1u << sidx;
              prefetched = true;
            }
          }
        } else {
          // no tile in this slot of the item's last group: V^T columns zero, K rows unused
          if (Gg > 0 && !wait_or_abort(&bars[kBarKFree], (Gg - 1) & 1, abort_flag, a.status)) { aborted = true; break; }
          if (lane == 0) mbar_arrive(&bars[kBarKFull]);
          if (Gg > 0 && !wait_or_abort(&bars[kBarVFree], (Gg - 1) & 1, abort_flag, a.status)) { aborted = true; break; }
          zero_v_tile(vop, r, lane);
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) mbar_arrive(&bars[kBarVFull]);
        }
      }
      if (aborted) break;
      G += ng;
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars[kBarItemEmpty + buf]);
    }
    // copies still in flight (only after a wait gave up) must land before the CTA exits
    for (int s = 0; s < kWarpStages; ++s)
      if (inflight & (1u << s)) mbar_wait(&my_bars[s], (phase >> s) & 1);
  } else if (warp == kMmaWarp) {
    // ================================================================== MMA warp
    if (lane == 0) {
      struct GroupRef {
        int buf, item, G;
        bool first, last;
      };
      int k = -1, gl = 0, ng = 0, Gnext = 0;
      // The next group in order; a group that opens an item waits for the item's publication.
      auto advance = [&](GroupRef& x) -> bool {
        if (gl >= ng) {
          ++k;
          if (!wait_or_abort(&bars[kBarItemFull + (k & 1)], (k >> 1) & 1, abort_flag, a.status)) return false;
          const ItemDesc d = desc[k & 1];
          if (d.b < 0) return false;
          ng = (d.units + 7) >> 3;
          gl = 0;
        }
        x.buf = k & 1;
        x.item = k;
        x.G = Gnext++;
        x.first = gl == 0;
        x.last = gl == ng - 1;
        ++gl;
        return true;
      };
      auto issue_qk = [&](const GroupRef& x) -> bool {
        if (!wait_or_abort(&bars[kBarKFull], x.G & 1, abort_flag, a.status)) return false;
        if (x.G >= 2 && !wait_or_abort(&bars[kBarSFree + (x.G & 1)], ((x.G >> 1) - 1) & 1, abort_flag, a.status))
          return false;
        if (x.first && !wait_or_abort(&bars[kBarQFull + x.buf], (x.item >> 1) & 1, abort_flag, a.status)) return false;
        tcgen05_after_sync();
        const uint32_t d_tmem = tmem + (x.G & 1) * kCols;
        const uint8_t* qb = qop + x.buf * kCols * 256;
#pragma unroll
        for (int j = 0; j < 8; ++j)
          umma_bf16(d_tmem, umma_desc_kmajor(kop + j * 256), umma_desc_kmajor(qb + j * 256), kIdesc, j > 0);
        umma_commit(&bars[kBarSFull + (x.G & 1)]);
        umma_commit(&bars[kBarKFree]);
        return true;
      };
      auto issue_pv = [&](const GroupRef& x) -> bool {
        if (!wait_or_abort(&bars[kBarPFull], x.G & 1, abort_flag, a.status)) return false;
        if (!wait_or_abort(&bars[kBarVFull], x.G & 1, abort_flag, a.status)) return false;
        if (x.first && x.item > 0 && !wait_or_abort(&bars[kBarOFree], (x.item - 1) & 1, abort_flag, a.status))
          return false;
        tcgen05_after_sync();
        const uint32_t o_tmem = tmem + 2 * kCols;
#pragma unroll
        for (int j = 0; j < 8; ++j)
          umma_bf16(o_tmem, umma_desc_kmajor(vop + j * 256), umma_desc_kmajor(pop + j * 256), kIdesc,
                    !(x.first && j == 0));
#pragma unroll
        for (int j = 0; j < 8; ++j)
          umma_bf16(o_tmem, umma_desc_kmajor(vop + j * 256), umma_desc_kmajor(pop + kCols * 256 + j * 256), kIdesc, 1);
        umma_commit(&bars[kBarVFree]);
        return true;
      };
      GroupRef cur, nxt;
      if (advance(cur) && issue_qk(cur)) {
        while (true) {
          if (cur.last) {
            // close the item before waiting for the next one to be published
            if (!issue_pv(cur) || !advance(nxt) || !issue_qk(nxt)) break;
          } else {
            advance(nxt);                      // same item: no wait
            if (!issue_qk(nxt) || !issue_pv(cur)) break;
          }
          cur = nxt;
        }
      }
      // every MMA issued has completed before tensor memory is released
      umma_commit(&bars[kBarDrain]);
      mbar_wait(&bars[kBarDrain], 0);
    }
    __syncwarp();
  } else {
    // ================================================================== softmax warpgroup
    const int q = warp - kSoftmaxWarp0;           // TMEM lane quadrant (warp % 4)
    const int gi = lane >> 2, ti = lane & 3;
    float* red_max = red;                         // [4][kCols]
    float* red_sum = red + 4 * kCols;             // [4][kCols]
    float* alpha_s = red + 8 * kCols;             // [kCols]
    float* m_s = red + 9 * kCols;                 // [kCols]
    const uint32_t lane_base = static_cast<uint32_t>(32 * q) << 16;
    int G = 0;
    for (int k = 0;; ++k) {
      const int buf = k & 1;
      const bool ok_item = wait_or_abort(&bars[kBarItemFull + buf], (k >> 1) & 1, abort_flag, a.status);
      const ItemDesc d = desc[buf];
      if (wg_any(!ok_item || d.b < 0)) break;
      const int* mt = meta + buf * kMaxItemTiles;
      const int ng = (d.units + 7) >> 3;
      const int causal_lim = lens[d.b] - a.tokens;   // token t of a request sees positions <= causal_lim + t
      float mcol[NJ][2], lsum[NJ][2];
#pragma unroll
      for (int j = 0; j < NJ; ++j) {
        mcol[j][0] = mcol[j][1] = kNoScore;
        lsum[j][0] = lsum[j][1] = 0.f;
      }
      bool stop = false;
      for (int gl = 0; gl < ng; ++gl, ++G) {
        const int sb = G & 1;
        bool ok = wait_or_abort(&bars[kBarSFull + sb], (G >> 1) & 1, abort_flag, a.status);
        tcgen05_after_sync();
        uint32_t sr[2][kCols / 2];
#pragma unroll
        for (int s = 0; s < 2; ++s)
          tmem_ld_scores<kCols>(tmem + (static_cast<uint32_t>(32 * q + 16 * s) << 16) + sb * kCols, sr[s]);
        tmem_wait_ld();
        tcgen05_before_sync();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars[kBarSFree + sb]);
        // the P operand (and the output) are free once the previous group's PV completed
        if (G > 0) ok = wait_or_abort(&bars[kBarVFree], (G - 1) & 1, abort_flag, a.status) && ok;
        tcgen05_after_sync();
        // scores in the log2 domain; hidden: past the item, unresolved pages, padding columns,
        // positions past a new token's own
        float x[2][NJ][4];
#pragma unroll
        for (int s = 0; s < 2; ++s) {
#pragma unroll
          for (int i2 = 0; i2 < 2; ++i2) {
            const int tok = 128 * gl + 32 * q + 16 * s + gi + 8 * i2;     // token offset within the item
            const int u = tok >> 4;
            const int pos = d.t0 + tok;
            const bool valid = u < d.units && (mt[u] & 3) != kKindInvalid && pos < d.t1;
#pragma unroll
            for (int j = 0; j < NJ; ++j) {
#pragma unroll
              for (int e = 0; e < 2; ++e) {
                const int col = 8 * j + 2 * ti + e;
                const bool vis = valid && col < d.nh && pos <= causal_lim + (d.h0 + col) % a.tokens;
                x[s][j][2 * i2 + e] = vis ? __uint_as_float(sr[s][4 * j + 2 * i2 + e]) * a.scale_log2 : -CUDART_INF_F;
              }
            }
          }
        }
        bool grow = false;
#pragma unroll
        for (int j = 0; j < NJ; ++j)
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            const float mx = fmaxf(fmaxf(x[0][j][e], x[0][j][2 + e]), fmaxf(x[1][j][e], x[1][j][2 + e]));
            grow = grow || mx > mcol[j][e] + kRescaleThreshold;
          }
        if (wg_any(grow || !ok)) {
          if (wg_any(!ok)) {
            stop = true;
            break;
          }
          // column maxima over the warpgroup's 128 tokens, then the new running max
          float cm[NJ][2];
#pragma unroll
          for (int j = 0; j < NJ; ++j)
#pragma unroll
            for (int e = 0; e < 2; ++e) {
              float v = fmaxf(fmaxf(x[0][j][e], x[0][j][2 + e]), fmaxf(x[1][j][e], x[1][j][2 + e]));
#pragma unroll
              for (int dd = 4; dd < 32; dd <<= 1) v = fmaxf(v, __shfl_xor_sync(0xFFFFFFFFu, v, dd));
              cm[j][e] = v;
            }
          if (gi == 0) {
#pragma unroll
            for (int j = 0; j < NJ; ++j)
#pragma unroll
              for (int e = 0; e < 2; ++e) red_max[q * kCols + 8 * j + 2 * ti + e] = cm[j][e];
          }
          wg_sync();
#pragma unroll
          for (int j = 0; j < NJ; ++j)
#pragma unroll
            for (int e = 0; e < 2; ++e) {
              const int c = 8 * j + 2 * ti + e;
              const float nm = fmaxf(fmaxf(mcol[j][e], fmaxf(red_max[c], red_max[kCols + c])),
                                     fmaxf(red_max[2 * kCols + c], red_max[3 * kCols + c]));   // finite: >= kNoScore
              const float al = fast_exp2(mcol[j][e] - nm);
              mcol[j][e] = nm;
              lsum[j][e] *= al;
              if (q == 0 && gi == 0) alpha_s[c] = al;
            }
          wg_sync();
          if (gl > 0) {
            // the output holds this item's earlier groups: rescale it in tensor memory (the
            // previous group's PV has completed)
#pragma unroll
            for (int c0 = 0; c0 < kCols; c0 += 16) {
              uint32_t o[16];
              tmem_ld_32x32b_x16(tmem + lane_base + 2 * kCols + c0, o);
              tmem_wait_ld();
#pragma unroll
              for (int i = 0; i < 16; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha_s[c0 + i]);
              tmem_st_32x32b_x16(tmem + lane_base + 2 * kCols + c0, o);
            }
            tmem_wait_st();
          }
        }
        // P = 2^(x - m): BF16 high part and BF16 remainder, transposed into P^T core matrices
        // (n-block j, k-block 4q + 2s (+1 for tokens 8-15 of the 16))
#pragma unroll
        for (int s = 0; s < 2; ++s) {
#pragma unroll
          for (int j = 0; j < NJ; ++j) {
            const float p0 = fast_exp2(x[s][j][0] - mcol[j][0]), p1 = fast_exp2(x[s][j][1] - mcol[j][1]);
            const float p2 = fast_exp2(x[s][j][2] - mcol[j][0]), p3 = fast_exp2(x[s][j][3] - mcol[j][1]);
            lsum[j][0] += p0 + p2;
            lsum[j][1] += p1 + p3;
            const uint32_t h01 = pack_bf16x2(p0, p1), h23 = pack_bf16x2(p2, p3);
            const uint32_t r01 = pack_bf16x2(p0 - bf16lo_to_f32(h01), p1 - bf16hi_to_f32(h01));
            const uint32_t r23 = pack_bf16x2(p2 - bf16lo_to_f32(h23), p3 - bf16hi_to_f32(h23));
            uint8_t* ph = pop + j * kCoreRow + (4 * q + 2 * s) * 128 + gi * 16 + ti * 4;
            *reinterpret_cast<uint32_t*>(ph) = transpose8x8(h01);
            *reinterpret_cast<uint32_t*>(ph + 128) = transpose8x8(h23);
            *reinterpret_cast<uint32_t*>(ph + kCols * 256) = transpose8x8(r01);
            *reinterpret_cast<uint32_t*>(ph + kCols * 256 + 128) = transpose8x8(r23);
          }
        }
        fence_proxy_async_smem();
        tcgen05_before_sync();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars[kBarPFull]);
      }
      if (stop) break;
      // ---- the item's output: O^T / column sums (the last group's PV has completed)
      const bool ok = wait_or_abort(&bars[kBarVFree], (G - 1) & 1, abort_flag, a.status);
      tcgen05_after_sync();
#pragma unroll
      for (int j = 0; j < NJ; ++j)
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          float v = lsum[j][e];
#pragma unroll
          for (int dd = 4; dd < 32; dd <<= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, dd);
          if (gi == 0) {
            red_sum[q * kCols + 8 * j + 2 * ti + e] = v;
            if (q == 0) m_s[8 * j + 2 * ti + e] = mcol[j][e];
          }
        }
      if (wg_any(!ok)) break;                     // also makes red_sum and m_s visible
      const int ch = 32 * q + lane;               // this thread's output channel (TMEM lane)
#pragma unroll
      for (int c0 = 0; c0 < kCols; c0 += 16) {
        uint32_t o[16];
        tmem_ld_32x32b_x16(tmem + lane_base + 2 * kCols + c0, o);
        tmem_wait_ld();
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const int n = c0 + i;
          if (n < d.nh) {
            const float lsum_n = red_sum[n] + red_sum[kCols + n] + red_sum[2 * kCols + n] + red_sum[3 * kCols + n];
            const float inv = lsum_n > 0.f ? 1.f / lsum_n : 0.f;
            const float lse2 = lsum_n > 0.f ? m_s[n] + log2f(lsum_n) : -CUDART_INF_F;
            const float val = __uint_as_float(o[i]) * inv;
            if (d.single) {
              const size_t row = query_row(d.b, d.h0 + n, a.tokens, a.hq);
              a.out[row * ZF_HEAD_DIM + ch] = val;
              if (ch == 0) a.lse[row] = lse2 * kLn2;
            } else {
              const size_t pidx = (static_cast<size_t>(d.b) * a.hq + d.h0 + n) * a.max_chunks + d.c;
              a.part_o[pidx * ZF_HEAD_DIM + ch] = val;
              if (ch == 0) a.part_lse[pidx] = lse2;
            }
          }
        }
      }
      tcgen05_before_sync();
      wg_sync();                                  // every warp read the output and the sums
      if (lane == 0) {
        mbar_arrive(&bars[kBarOFree]);
        mbar_arrive(&bars[kBarItemEmpty + buf]);
      }
    }
  }
  tcgen05_before_sync();
  __syncthreads();
  tcgen05_after_sync();
  if (warp == kMmaWarp) tmem_dealloc(tmem, kTmemCols);
}

}  // namespace

bool attention_tc_fits(int32_t batch) {
  return tc_layout<kTcMaxCols>(batch).total <= 227 * 1024;
}

Plan attention_tc_plan(int batch, int hq, int hkv, int page_size, int max_pages, int num_sms) {
  return make_plan(batch, hq, hkv, page_size, max_pages, num_sms, kRebuildWarps, kTcMaxCols);
}

zf_status launch_attention_tc(const AttnArgs& base, const Plan& p, int32_t tokens, cudaStream_t stream) {
  AttnArgs a = base;
  a.hps = kTcMaxCols;
  a.slices = p.slices;
  a.max_chunks = p.max_chunks;
  a.min_range_pages = p.min_range_pages;
  a.chunk_pages = p.chunk_pages;
  a.prefetch = 0;
  a.plan_first = 0;
  const int cols = a.group < kTcMaxCols ? a.group : kTcMaxCols;   // columns of the widest slice
  const bool narrow = cols <= 16;
  const size_t smem = narrow ? tc_layout<16>(a.batch).total : tc_layout<32>(a.batch).total;
  const void* kernel = narrow ? reinterpret_cast<const void*>(attn_tc_kernel<16>)
                              : reinterpret_cast<const void*>(attn_tc_kernel<32>);
  zf_status st = ensure_smem_limit(kernel, narrow ? 0 : 1, smem);
  if (st != ZF_OK) return st;
  cudaLaunchAttribute pdl[1];
  pdl[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  pdl[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(p.grid);
  cfg.blockDim = dim3(kTcThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cfg.attrs = pdl;
  cfg.numAttrs = 1;
  if ((narrow ? cudaLaunchKernelEx(&cfg, attn_tc_kernel<16>, a) : cudaLaunchKernelEx(&cfg, attn_tc_kernel<32>, a)) !=
      cudaSuccess)
    return ZF_ERR_CUDA;
  MergeArgs m{};
  m.part_o = a.part_o;
  m.part_lse = a.part_lse;
  m.out = a.out;
  m.lse = a.lse;
  m.chunk_counts = a.chunk_counts;
  m.batch = a.batch;
  m.hq = a.hq;
  m.group = a.group;
  m.slices = a.slices;
  m.max_chunks = a.max_chunks;
  m.tokens = tokens;
  m.hps = kTcMaxCols;
  return launch_merge(m, tokens > 1, stream);
}

}  // namespace zf
