// Decode attention over the compressed paged cache when a kv head has more than 8 query columns
// (GQA groups above 8, or several new tokens per request: columns = query heads per kv head x new
// tokens), on the 5th-generation tensor cores: the rebuilt K and V tiles become MMA operands (K in
// tensor memory, V^T in shared memory) and the scores and the output accumulate in tensor memory,
// so each kv head's tiles are read from HBM once per N = 16 or 32 columns (the warp-MMA kernel
// takes 8 columns per pass and reads the tiles once per 8).
//
// ZipFusion §III.C (Attention over the Compressed KV Cache): compressed blocks are copied
// HBM -> shared memory as they are and the exact BF16 values are rebuilt from them with integer
// operations right before the tensor-core instructions; raw blocks need no rebuild.  §IV.B: split
// chunks are combined by a split-result merge.
//
// One CTA per SM, 27 warps:
//  * warps 0-7 rebuild K, warps 8-15 rebuild V: warp r (mod 8) takes tile slot r of every
//    128-token group of an item (16 tokens of one kv head).  Its half of the tile comes HBM ->
//    its private stages by 1-D bulk copies (at N = 16 three stages per K warp and two per V warp,
//    started by the copy warp; at N = 32 two each, started by the warp itself: the next copies are
//    in flight while it works on this one), and it rebuilds the half straight from the m16n8k16
//    fragment registers the rebuild produces: K (A of S^T = K Q^T: 128 tokens x 128 channels) into
//    one of two tensor-memory buffers with tcgen05.st, V^T (A of O^T = V^T P^T: 128 channels x 128
//    tokens) into one of two shared-memory buffers in the K-major core-matrix layout (one
//    conflict-free 32-bit store per lane fills one 8 x 16-byte core matrix).  K and V warps wait
//    only for the MMA that last read their buffer, so the keys of the next group are rebuilt while
//    this group's softmax runs;
//  * warps 16-23 (two softmax warpgroups, each owning half of the columns; warp w reads TMEM
//    lanes 32(w%4)..): S^T comes out of tensor memory in the m16n8 accumulator layout, the online
//    softmax runs in the log2 domain with one running max per column shared by the warpgroup
//    (raised only when a score exceeds it by more than 8, after a warpgroup vote; the warpgroup's
//    output columns in tensor memory are then rescaled in place), and P^T (BF16 high part + BF16
//    remainder) is transposed with movmatrix into one of two P operand buffers; at the end of an
//    item each warpgroup divides its O^T columns by their sums and writes the output or the
//    partial;
//  * warp 24 (MMA): allocates tensor memory; the warp runs the issue loop and one elected lane
//    issues both products, whichever is ready first: S^T = K Q^T (8 x M128 N K16, A from tensor
//    memory) into one of two TMEM score buffers, and O^T += V^T P^T (8 MMAs of 2N: P's high part
//    and its remainder side by side) into the TMEM output, each completion signalled by
//    tcgen05.commit to an mbarrier;
//  * warp 25 (metadata): walks the CTA's items (the warp-MMA kernel's planner and page walk), one
//    item ahead: resolves the pages through the page table and the directory and stages the
//    item's query rows as the B operand of S^T;
//  * warp 26 (copy, N = 16): lane w starts rebuild warp w's copies as soon as it hands a stage back.
// Every wait is bounded (2 s); a wait that gives up sets ZF_DEV_TIMEOUT and the CTA winds down
// (each softmax warpgroup decides together, so its named barriers are always met).
#include <cuda_runtime.h>
#include <math_constants.h>
#include <stdint.h>

#include "zf_attn_common.cuh"

namespace zf {
namespace {

constexpr int kHalfWarps = 8;                     // warps per half: 8 rebuild K rows, 8 rebuild V^T columns
constexpr int kRebuildWarps = 2 * kHalfWarps;
constexpr int kSoftmaxWarp0 = 16;                 // warps 16..23: warpgroup (w - 16) / 4, TMEM lane quadrant w % 4
constexpr int kSoftmaxWarps = 8;                  // two warpgroups, each owns half of the columns
constexpr int kMmaWarp = kSoftmaxWarp0 + kSoftmaxWarps;
constexpr int kMetaWarp = kMmaWarp + 1;
constexpr int kCopyWarp = kMetaWarp + 1;          // lane i keeps rebuild warp i's copy stages filled
constexpr int kTcWarps = kCopyWarp + 1;
constexpr int kTcThreads = kTcWarps * 32;
constexpr int kHalfStageBytes = kTileCompBytes;   // one compressed K (or V) half tile; a raw half: 3 + 1 blocks
constexpr int kOpBytes = 128 * 128 * 2;           // one 128 x 128 BF16 operand
constexpr int kCoreRow = 2048;                    // bytes between core-matrix rows along M/N (16 along K)
// Tensor memory: two score buffers (kCols columns each) at columns 0 .. 2 kCols, the output
// (2 kCols columns: high and low parts of P) at 2 kCols .. 4 kCols, and two K operands (128 tokens
// x 128 channels as BF16 pairs: 64 columns each) from column 128.
constexpr uint32_t kTmemCols = 256;
constexpr uint32_t kTmemK = 128;
constexpr int kSoftmaxBarrier = 1;                // named barriers of the softmax warpgroups: 1 and 2

// Barriers (mbarrier index in the shared array).
// Copy stages per rebuild warp (measured on GB300: the K warps' copies, which the first product
// waits for, gain most from a third stage; at 32 columns the larger operands leave room for two
// each).  kNumStages: the stage barriers allocated (the most any width uses).
template <int kCols>
struct TcStages {
  static constexpr int kK = kCols == 16 ? 3 : 2;
  static constexpr int kV = 2;
  static constexpr int kTotal = kHalfWarps * (kK + kV);
};
constexpr int kNumStages = kHalfWarps * 5;

enum : int {
  kBarStage = 0,                // one per copy stage of the rebuild warps (K warps first): data landed
  kBarStageEmpty = kNumStages,  // one per copy stage: its rebuild warp is done with it
  kBarItemFull = 2 * kNumStages,      // [2] the metadata warp published an item
  kBarItemEmpty = kBarItemFull + 2,   // [2] rebuild + softmax warps are done with it
  kBarQFull = kBarItemEmpty + 2,      // [2] the item's query operand is staged
  kBarKFull = kBarQFull + 2,          // [2] the 8 K warps wrote a group's K operand (per K buffer)
  kBarVFull = kBarKFull + 2,          // [2] the 8 V warps wrote a group's V operand (per V buffer)
  kBarKFree = kBarVFull + 2,          // [2] S^T = K Q^T of a group completed, per K buffer (commit)
  kBarSFull = kBarKFree + 2,          // [2] scores of a group in TMEM buffer (commit)
  kBarSFree = kBarSFull + 2,          // [2] the softmax warpgroups read that score buffer
  kBarPFull = kBarSFree + 2,          // [2] the softmax warpgroups wrote a group's P operand (per P buffer)
  kBarPvDone = kBarPFull + 2,         // [2] O^T += V^T P^T of a group completed, per V / P buffer (commit)
  kBarOFree = kBarPvDone + 2,         // the softmax warpgroups read an item's output from tensor memory
  kBarDrain = kBarOFree + 1,          // end of the CTA: every MMA issued has completed
  kNumBars = kBarDrain + 1,
};

struct TcLayout {
  size_t vop, pop, qop, stages, meta, desc, bars, misc, spar, red, prefix, lens, total;
};

template <int kCols>
__host__ __device__ inline TcLayout tc_layout(int batch) {
  TcLayout s;
  size_t at = 0;
  s.vop = at; at += 2 * kOpBytes;                 // two V operands (groups alternate)
  s.pop = at; at += 4 * kCols * 256;              // P^T, two buffers: high part, then low part (kCols x 128 BF16 each)
  s.qop = at; at += 2 * kCols * 256;              // Q of two items (kCols x 128 BF16 each)
  s.stages = at; at += static_cast<size_t>(TcStages<kCols>::kTotal) * kHalfStageBytes;
  s.meta = at; at += 2 * kMaxItemTiles * 4;
  s.desc = at; at += 2 * 64;
  s.bars = at; at += kNumBars * 8;
  s.misc = at; at += 16;                          // [0] abort flag, [4] TMEM base address
  s.spar = at; at += kNumStages * 4;              // per stage: parity of its data barrier's next phase
  s.red = at; at += static_cast<size_t>(10 * kCols) * 4;   // column maxima [4][kCols], sums [4][kCols], alpha, max
  s.prefix = at; at += static_cast<size_t>(batch + 1) * 4;
  s.lens = at; at += static_cast<size_t>(batch) * 4;
  s.total = (at + 127) & ~static_cast<size_t>(127);
  return s;
}

// A bounded wait that also gives up at once when another warp already has (abort flag set).
__device__ __forceinline__ bool wait_or_abort(uint64_t* bar, uint32_t parity, volatile int* abort_flag,
                                              int32_t* status, uint64_t limit_ns = kWaitTimeoutNs) {
  if (*abort_flag) return false;
  if (mbar_wait(bar, parity, limit_ns)) return true;
  *abort_flag = 1;
  report(status, ZF_DEV_TIMEOUT);
  return false;
}

// A softmax warpgroup's barrier (id), and the same barrier ORing a predicate over its 128 threads.
__device__ __forceinline__ void wg_sync(uint32_t id) { asm volatile("bar.sync %0, 128;" ::"r"(id) : "memory"); }
__device__ __forceinline__ bool wg_any(uint32_t id, bool v) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.u32 p, %1, 0;\n\t"
      "bar.red.or.pred q, %2, 128, p;\n\t"
      "selp.u32 %0, 1, 0, q;\n\t}"
      : "=r"(r)
      : "r"(static_cast<uint32_t>(v)), "r"(id)
      : "memory");
  return r != 0;
}

// Tensor-memory accesses of the softmax warpgroups beyond the shared set: 8 score columns
// (16x256b.x1), and 8 output columns per lane (32x32b.x8).
__device__ __forceinline__ void tmem_ld_16x256b_x1(uint32_t taddr, uint32_t (&r)[4]) {
  asm volatile("tcgen05.ld.sync.aligned.16x256b.x1.b32 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(taddr));
}
__device__ __forceinline__ void tmem_st_32x32b_x8(uint32_t taddr, const uint32_t (&r)[8]) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"r"(taddr), "r"(r[0]),
               "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7])
               : "memory");
}

// Start the copy of the K (is_v false) or V half of tile u of an item into `stage`: a compressed
// half (3136 bytes) whole, a raw half's first three blocks (its fourth is fetched once those are
// used, see fetch_raw_block3).  Returns the tile's kind (nothing is armed for an invalid one).
// The MMA warp's issue forms: the whole warp runs the issue loop and one lane, chosen by
// elect.sync (the lowest active lane, so always the same one in a converged warp), issues each
// tcgen05.mma and tcgen05.commit.  Issued from warp-uniform code this way, an MMA costs its warp
// about 32 cycles against about 59 from a lane running the loop alone (measured on GB300, 16 MMAs
// per group as here).
__device__ __forceinline__ void umma_bf16_elect(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                                uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p, e;\n\t"
      "elect.sync _|e, 0xffffffff;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}
__device__ __forceinline__ void umma_bf16_ta_elect(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc,
                                                   uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p, e;\n\t"
      "elect.sync _|e, 0xffffffff;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}
__device__ __forceinline__ void umma_commit_elect(uint64_t* bar) {
  asm volatile(
      "{\n\t.reg .pred e;\n\t"
      "elect.sync _|e, 0xffffffff;\n\t"
      "@e tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n\t}" ::"r"(smem_addr(bar))
      : "memory");
}
// A barrier test that holds for the warp only when every lane saw the phase complete (each lane
// then has its own acquire, and the warp's control flow stays uniform).
__device__ __forceinline__ bool mbar_test_warp(uint64_t* bar, uint32_t parity) {
  return __all_sync(0xFFFFFFFFu, mbar_test(bar, parity));
}

__device__ __forceinline__ int issue_half(const AttnArgs& a, const ItemDesc& d, const int* meta, int u, bool is_v,
                                          uint8_t* stage, uint64_t* bar, int lane, uint64_t policy) {
  const int m = meta[u];
  const int kind = m & 3;
  const size_t head = static_cast<size_t>(m >> 5) * a.hkv + d.g;
  const int t = (m >> 2) & 7;
  if (lane == 0) {
    if (kind == kKindComp) {
      mbar_arrive_expect_tx(bar, kTileCompBytes);
      bulk_copy_g2s(stage, (is_v ? a.v_comp : a.k_comp) + head * a.comp_head_bytes + static_cast<size_t>(t) * kTileCompBytes,
                    kTileCompBytes, bar, policy);
    } else if (kind == kKindRaw) {
      mbar_arrive_expect_tx(bar, 3 * kRawBlockBytes);
      bulk_copy_g2s(stage, (is_v ? a.v_raw : a.k_raw) + head * a.raw_head_bytes + static_cast<size_t>(t) * kTileRawBytes,
                    3 * kRawBlockBytes, bar, policy);
    }
  }
  return kind;
}

// The fourth block of a raw half of tile u, into the start of `stage` (its first three blocks
// have been used).
__device__ __forceinline__ void fetch_raw_block3(const AttnArgs& a, const ItemDesc& d, const int* meta, int u,
                                                 bool is_v, uint8_t* stage, uint64_t* bar, int lane, uint64_t policy) {
  const int m = meta[u];
  const size_t head = static_cast<size_t>(m >> 5) * a.hkv + d.g;
  const int t = (m >> 2) & 7;
  if (lane == 0) {
    mbar_arrive_expect_tx(bar, kRawBlockBytes);
    bulk_copy_g2s(stage, (is_v ? a.v_raw : a.k_raw) + head * a.raw_head_bytes + static_cast<size_t>(t) * kTileRawBytes +
                             3 * kRawBlockBytes,
                  kRawBlockBytes, bar, policy);
  }
}

// Fragment registers -> operand.  K (A of S^T = K Q^T, rows = tokens) goes to tensor memory:
// the rows of tile slot p are TMEM lanes 16p .. 16p+15 and the 128 channels are 64 columns of BF16
// pairs, in a channel order permuted within each 16-channel span (element 4c + m of a span holds
// channel {2c, 2c+1, 2c+8, 2c+9}[m]; the query operand uses the same order, which leaves q.k
// unchanged).  That order is the one tcgen05.st.16x256b takes from the m16n8k16 fragments: a
// thread's registers for span 2j + h are {a0a1, a4a5, a2a3, a6a7} of half h of channel group j.
// V^T (A of O^T = V^T P^T, rows = channels) goes to shared memory: register i of half h of channel
// group j (rows g = lane/4 (+8 for i odd), columns 2(lane%4) (+8 for i >= 2)) is core matrix
// (m-block 4j + 2h + (i & 1), k-block 2p + (i >> 1)); values of tokens at or past the context's end
// are zeroed by keep_a / keep_b.
__device__ __forceinline__ void store_k_block(const uint32_t (&ka)[8], int j, uint32_t k_tmem) {
  const uint32_t r[8] = {ka[0], ka[2], ka[1], ka[3], ka[4], ka[6], ka[5], ka[7]};
  tmem_st_16x256b_x2(k_tmem + 16 * j, r);
}
__device__ __forceinline__ void store_v_block(const uint32_t (&va)[8], int j, uint8_t* vop, int p, int lane,
                                              uint32_t keep_a, uint32_t keep_b) {
  uint8_t* base = vop + (2 * p) * 128 + (lane >> 2) * 16 + (lane & 3) * 4;
#pragma unroll
  for (int h = 0; h < 2; ++h)
#pragma unroll
    for (int i = 0; i < 4; ++i)
      *reinterpret_cast<uint32_t*>(base + (4 * j + 2 * h + (i & 1)) * kCoreRow + (i >> 1) * 128) =
          va[4 * h + i] & ((i >> 1) ? keep_b : keep_a);
}

// One half tile (K or V, 4 blocks) from its stage into its operand.  kind: compressed or raw (a raw
// half holds its first three blocks; fetch3() brings the fourth into the start of the stage and
// returns false when its wait gave up).  Returns false only then.
// One copy of this code serves the K and the V warps (kV picks the store per block at run time):
// measured on GB300, separate K and V copies were 1-4% slower, and the kernel is sensitive to its
// code size (a K / V-specialised rebuild loop was 17-25% slower).
template <typename Fetch3>
__device__ __forceinline__ bool rebuild_half(bool kV, const uint8_t* st, int kind, uint32_t keep_a, uint32_t keep_b, uint8_t* vop_g,
                                             int p, uint32_t k_tmem, int lane, Fetch3&& fetch3) {
  auto put = [&](const uint32_t (&x)[8], int j) {
    if (kV) store_v_block(x, j, vop_g, p, lane, keep_a, keep_b);
    else store_k_block(x, j, k_tmem);
  };
  if (kind == kKindComp) {
    uint32_t hdr[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) hdr[j] = *reinterpret_cast<const uint32_t*>(st + j * kSlotBytes + kHeaderAt);
    const bool escapes = ((hdr[0] | hdr[1] | hdr[2] | hdr[3]) & kHeaderEscMask) != 0;
    // header byte 0 (base/2) of the four blocks in one register, so that the loop below picks
    // block j's with a byte permute rather than an indexed (local-memory) array
    const uint32_t bases = __byte_perm(__byte_perm(hdr[0], hdr[1], 0x0040u), __byte_perm(hdr[2], hdr[3], 0x0040u), 0x5410u);
    if (escapes) {
#pragma unroll 1
      for (int j = 0; j < 4; ++j) {
        uint32_t x[8];
        rebuild_lane(st + j * kSlotBytes, lane, x);
        put(x, j);
      }
    } else {
      // the next block's low bytes and codes are loaded while this one is rebuilt
      uint4 lo_n = *reinterpret_cast<const uint4*>(st + 16 * lane);
      uint2 cd_n = *reinterpret_cast<const uint2*>(st + 512 + 8 * lane);
#pragma unroll 1
      for (int j = 0; j < 4; ++j) {
        const uint4 lo = lo_n;
        const uint2 cd = cd_n;
        const uint8_t* nx = st + (j < 3 ? j + 1 : 3) * kSlotBytes;
        lo_n = *reinterpret_cast<const uint4*>(nx + 16 * lane);
        cd_n = *reinterpret_cast<const uint2*>(nx + 512 + 8 * lane);
        uint32_t h[4], x[8];
        high_bytes(cd, __byte_perm(bases, 0u, 0x1111u * j), h);
        interleave(lo, h, x);
        put(x, j);
      }
    }
    return true;
  }
#pragma unroll 1
  for (int j = 0; j < 3; ++j) {
    uint32_t x[8];
    load_raw_lane(st + j * kRawBlockBytes, lane, x);
    put(x, j);
  }
  if (!fetch3()) return false;
  uint32_t x[8];
  load_raw_lane(st, lane, x);
  put(x, 3);
  return true;
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
// core matrix (n / 8, k / 8)); columns past d.nh are zero.  K index k holds channel
// 16 (k / 16) + {2c, 2c+1, 2c+8, 2c+9}[k % 4], c = (k % 16) / 4: the order of the K operand.
template <int kCols>
__device__ __forceinline__ void stage_q(const AttnArgs& a, const ItemDesc& d, uint8_t* qb, int lane) {
#pragma unroll 2
  for (int it = 0; it < kCols / 4; ++it) {
    // lane: column n, 16-channel span sp (two 16-byte chunks of the operand)
    const int n = 4 * it + (lane >> 3), sp = lane & 7;
    uint4 lo = make_uint4(0u, 0u, 0u, 0u), hi = lo;
    if (n < d.nh) {
      const size_t row = query_row(d.b, d.h0 + n, a.tokens, a.hq);
      const uint4* src = reinterpret_cast<const uint4*>(a.q + row * ZF_HEAD_DIM + 16 * sp);
      lo = src[0];      // channel pairs 0..3 of the span
      hi = src[1];      // channel pairs 4..7
    }
    // chunk 0: pairs (0,1) (8,9) (2,3) (10,11) -> words 0, 4, 1, 5; chunk 1: words 2, 6, 3, 7
    *reinterpret_cast<uint4*>(qb + (n >> 3) * kCoreRow + (2 * sp) * 128 + (n & 7) * 16) =
        make_uint4(lo.x, hi.x, lo.y, hi.y);
    *reinterpret_cast<uint4*>(qb + (n >> 3) * kCoreRow + (2 * sp + 1) * 128 + (n & 7) * 16) =
        make_uint4(lo.z, hi.z, lo.w, hi.w);
  }
}

template <int kN>
__device__ __forceinline__ void tmem_ld_scores(uint32_t taddr, uint32_t (&r)[kN / 2]) {
  if constexpr (kN == 8) tmem_ld_16x256b_x1(taddr, r);
  else if constexpr (kN == 16) tmem_ld_16x256b_x2(taddr, r);
  else tmem_ld_16x256b_x4(taddr, r);
}

template <int kCols>
__global__ void __launch_bounds__(kTcThreads, 1) attn_tc_kernel(const AttnArgs a) {
  static_assert(4 * kCols <= static_cast<int>(kTmemK), "scores and output must end before the K operands");
  static_assert((kCols & (kCols - 1)) == 0 && 2 * kCols <= 256, "the PV MMA takes N = 2 kCols");
  // At 16 columns the copy warp keeps the rebuild warps' stages filled (measured on GB300: GQA-7 x 2
  // tokens 503 -> 466 us per call); at 32 columns, with two stages per rebuild warp, each rebuild
  // warp starts its own copies (there the copy warp's reaction added to every copy's latency:
  // GQA-7 x 4 tokens 567 -> 632 us).
  constexpr bool kCopyWarpFeeds = kCols == 16;
  constexpr uint32_t kIdesc = umma_idesc_bf16(128, kCols);
  // O^T += V^T P^T takes P's high part and its remainder as 2 kCols columns of one operand: the
  // output holds V^T P_hi^T in its first kCols columns and V^T P_lo^T in the rest, summed at the
  // end (an MMA's issue cost does not grow with N at these sizes, so this halves the PV issues)
  constexpr uint32_t kIdescPv = umma_idesc_bf16(128, 2 * kCols);
  extern __shared__ __align__(1024) uint8_t smem[];
  const TcLayout L = tc_layout<kCols>(a.batch);
  uint8_t* vop = smem + L.vop;
  uint8_t* pop = smem + L.pop;                    // buffer b at + b * 2 * kCols * 256: high part, then low part
  uint8_t* qop = smem + L.qop;
  uint8_t* stages = smem + L.stages;
  int* meta = reinterpret_cast<int*>(smem + L.meta);
  ItemDesc* desc = reinterpret_cast<ItemDesc*>(smem + L.desc);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L.bars);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L.misc);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L.misc + 4);
  float* red = reinterpret_cast<float*>(smem + L.red);
  int* prefix = reinterpret_cast<int*>(smem + L.prefix);
  int* spar = reinterpret_cast<int*>(smem + L.spar);
  int* lens = reinterpret_cast<int*>(smem + L.lens);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  if (tid == 0) {
    for (int i = 0; i < kNumStages; ++i) {
      mbar_init(&bars[kBarStage + i], 1);
      mbar_init(&bars[kBarStageEmpty + i], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&bars[kBarItemFull + b], 1);
      mbar_init(&bars[kBarItemEmpty + b], kRebuildWarps + kSoftmaxWarps + (kCopyWarpFeeds ? 1 : 0));
      mbar_init(&bars[kBarQFull + b], 1);
      mbar_init(&bars[kBarSFull + b], 1);
      mbar_init(&bars[kBarSFree + b], kSoftmaxWarps);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&bars[kBarKFull + b], kHalfWarps);
      mbar_init(&bars[kBarVFull + b], kHalfWarps);
      mbar_init(&bars[kBarKFree + b], 1);
    }
    mbar_init(&bars[kBarDrain], 1);
    mbar_init(&bars[kBarOFree], kSoftmaxWarps);
    for (int b = 0; b < 2; ++b) {
      mbar_init(&bars[kBarPvDone + b], 1);
      mbar_init(&bars[kBarPFull + b], kSoftmaxWarps);
    }
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
    if (a.publish_delay_ns) sleep_for_ns(a.publish_delay_ns);    // tests: the other warps' waits run out
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
    const bool is_v = warp >= kHalfWarps;          // warps 0-7: K rows; 8-15: V^T columns
    // tile slot of every group: a K warp writes its rows (TMEM lanes 16 r ..) in its own lane
    // quadrant (warp % 4), so K warp w takes slot 2 (w % 4) + w / 4
    const int r = is_v ? warp - kHalfWarps : 2 * (warp & 3) + (warp >> 2);
    // the barrier that group Gg's operand is announced on: one per operand buffer, so that warps
    // running two groups ahead of the MMA warp never move it two phases past that warp's test
    auto full_bar = [&](int Gg) { return &bars[(is_v ? kBarVFull : kBarKFull) + (Gg & 1)]; };
    // group G's operands (one of two K and one of two V buffers) are free once S^T, respectively
    // O^T += V^T P^T, of group G - 2 is computed
    auto wait_operand_free = [&](int Gg) -> bool {
      return Gg < 2 || wait_or_abort(&bars[(is_v ? kBarPvDone : kBarKFree) + (Gg & 1)], ((Gg >> 1) - 1) & 1,
                                     abort_flag, a.status);
    };
    // this warp's ring of copy stages: its tiles, across items, go to stages 0, 1, .., ns-1, 0, ..
    constexpr int kKSt = TcStages<kCols>::kK, kVSt = TcStages<kCols>::kV;
    static_assert(TcStages<kCols>::kTotal <= kNumStages, "stage barriers");
    const int ns = is_v ? kVSt : kKSt;
    const int first_stage = is_v ? kHalfWarps * kKSt + (warp - kHalfWarps) * kVSt : warp * kKSt;
    uint8_t* ring = stages + static_cast<size_t>(first_stage) * kHalfStageBytes;
    uint64_t* ring_bars = &bars[kBarStage + first_stage];
    if constexpr (kCopyWarpFeeds) {
      uint64_t* ring_empty = &bars[kBarStageEmpty + first_stage];
      const uint64_t policy = l2_evict_first_policy();
      uint32_t phase = 0;                            // per stage: parity of its data barrier's next wait
      int st_use = 0;                                // the stage of the next tile (its index mod ns)
      bool aborted = false, fetch3_pending = false;
      int G = 0;
      const ItemDesc* dcur = nullptr;
      const int* mcur = nullptr;
      // the fourth block of a raw half tile into the start of its stage (the first three are used)
      auto fetch_block3 = [&](int sidx, int u) -> bool {
        __syncwarp();
        fetch_raw_block3(a, *dcur, mcur, u, is_v, ring + sidx * kHalfStageBytes, &ring_bars[sidx], lane, policy);
        if (!wait_or_abort(&ring_bars[sidx], (phase >> sidx) & 1, abort_flag, a.status)) {
          fetch3_pending = true;                     // still in flight: waited for at the end
          return false;
        }
        phase ^= 1u << sidx;
        return true;
      };
      for (int k = 0; !aborted; ++k) {
        const int buf = k & 1;
        if (!wait_or_abort(&bars[kBarItemFull + buf], (k >> 1) & 1, abort_flag, a.status, a.wait_limit_ns)) break;
        const ItemDesc d = desc[buf];
        if (d.b < 0) break;
        const int* m = meta + buf * kMaxItemTiles;
        dcur = &desc[buf];                           // (the shared copy: taking d's address would put d in local memory)
        mcur = m;
        const int ng = (d.units + 7) >> 3;
        for (int gl = 0; gl < ng && !aborted; ++gl) {
          const int u = 8 * gl + r;
          const int Gg = G + gl;
          if (u < d.units) {
            // every tile of this warp has a stage: its copy, or a plain arrival for a page that
            // could not be resolved, comes from the copy warp
            const int sidx = st_use;
            if (!wait_or_abort(&ring_bars[sidx], (phase >> sidx) & 1, abort_flag, a.status)) { aborted = true; break; }
            phase ^= 1u << sidx;
            const int kind = m[u] & 3;
            uint8_t* st = ring + sidx * kHalfStageBytes;
            if (!wait_operand_free(Gg)) { aborted = true; break; }
            uint8_t* op = vop + (Gg & 1) * kOpBytes;
            const uint32_t k_tmem = tmem + (static_cast<uint32_t>(16 * r) << 16) + kTmemK + (Gg & 1) * 64;
            if (kind == kKindInvalid) {
              if (is_v) zero_v_tile(op, r, lane);
            } else {
              uint32_t keep_a = 0xFFFFFFFFu, keep_b = 0xFFFFFFFFu;
              if (is_v) {
                const int ntok = min(16, d.t1 - (d.t0 + 16 * u));
                const int ti = lane & 3;
                if (ntok < 16) {
                  keep_a = (2 * ti < ntok ? 0x0000FFFFu : 0u) | (2 * ti + 1 < ntok ? 0xFFFF0000u : 0u);
                  keep_b = (2 * ti + 8 < ntok ? 0x0000FFFFu : 0u) | (2 * ti + 9 < ntok ? 0xFFFF0000u : 0u);
                }
              }
              const bool ok_half = rebuild_half(is_v, st, kind, keep_a, keep_b, op, r, k_tmem, lane, [&]() {
                                            return fetch_block3(sidx, u);
                                          });
              if (!ok_half) {
                aborted = true;
                break;
              }
            }
            // the stage is read: hand it back to the copy warp with its data barrier's next parity
            __syncwarp();
            if (lane == 0) {
              spar[first_stage + sidx] = (phase >> sidx) & 1;
              mbar_arrive(&ring_empty[sidx]);
            }
            if (++st_use == ns) st_use = 0;
            if (is_v) {
              fence_proxy_async_smem();
            } else {
              tmem_wait_st();
              tcgen05_before_sync();
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(full_bar(Gg));
          } else {
            // no tile in this slot of the item's last group: V^T columns zero, K rows unused
            if (!wait_operand_free(Gg)) { aborted = true; break; }
            if (is_v) zero_v_tile(vop + (Gg & 1) * kOpBytes, r, lane);
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(full_bar(Gg));
          }
        }
        if (aborted) break;
        G += ng;
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars[kBarItemEmpty + buf]);
      }
      // a raw block this warp fetched itself and never waited for must land before the CTA exits
      if (fetch3_pending && !mbar_wait(&ring_bars[st_use], (phase >> st_use) & 1)) report(a.status, ZF_DEV_TIMEOUT);
    } else {
      // at 32 columns each rebuild warp starts its own copies
      const uint64_t policy = l2_evict_first_policy();
      uint32_t armed = 0, phase = 0;                 // per stage: a copy is in flight / parity of its next wait
      int n_issued = 0, n_used = 0;                  // this warp's tiles started / consumed
      int st_issue = 0, st_use = 0;                  // their stages (n mod ns, kept without a division)
      int iss_k = 0, iss_u = r;                      // the next tile to start: item iss_k, unit iss_u
      bool iss_end = false, aborted = false;
      // Start copies while stages are free, up to the item after the one being consumed (k_cur);
      // an item not yet published is tested, not waited for.
      auto pump = [&](int k_cur) {
        while (!iss_end && n_issued - n_used < ns && iss_k <= k_cur + 1) {
          if (iss_k > k_cur && !mbar_test(&bars[kBarItemFull + (iss_k & 1)], (iss_k >> 1) & 1)) break;
          const ItemDesc& di = desc[iss_k & 1];
          if (di.b < 0) {
            iss_end = true;
            break;
          }
          if (iss_u >= di.units) {
            ++iss_k;
            iss_u = r;
            continue;
          }
          const int st = st_issue;
          if (issue_half(a, di, meta + (iss_k & 1) * kMaxItemTiles, iss_u, is_v, ring + st * kHalfStageBytes,
                         &ring_bars[st], lane, policy) != kKindInvalid)
            armed |= 1u << st;
          ++n_issued;
          if (++st_issue == ns) st_issue = 0;
          iss_u += 8;
        }
      };
      int G = 0;
      const ItemDesc* dcur = nullptr;
      const int* mcur = nullptr;
      // the fourth block of a raw half tile into the start of its stage (the first three are used)
      auto fetch_block3 = [&](int sidx, int u) -> bool {
        __syncwarp();
        fetch_raw_block3(a, *dcur, mcur, u, is_v, ring + sidx * kHalfStageBytes, &ring_bars[sidx], lane, policy);
        if (!wait_or_abort(&ring_bars[sidx], (phase >> sidx) & 1, abort_flag, a.status)) return false;
        phase ^= 1u << sidx;
        return true;
      };
      for (int k = 0; !aborted; ++k) {
        const int buf = k & 1;
        if (!wait_or_abort(&bars[kBarItemFull + buf], (k >> 1) & 1, abort_flag, a.status, a.wait_limit_ns)) break;
        const ItemDesc d = desc[buf];
        if (d.b < 0) break;
        const int* m = meta + buf * kMaxItemTiles;
        dcur = &desc[buf];                           // (the shared copy: taking d's address would put d in local memory)
        mcur = m;
        const int ng = (d.units + 7) >> 3;
        pump(k);
        for (int gl = 0; gl < ng && !aborted; ++gl) {
          const int u = 8 * gl + r;
          const int Gg = G + gl;
          if (u < d.units) {
            const int sidx = st_use;
            if (armed & (1u << sidx)) {
              if (!wait_or_abort(&ring_bars[sidx], (phase >> sidx) & 1, abort_flag, a.status)) { aborted = true; break; }
              phase ^= 1u << sidx;
              armed &= ~(1u << sidx);
            }
            const int kind = m[u] & 3;
            uint8_t* st = ring + sidx * kHalfStageBytes;
            if (!wait_operand_free(Gg)) { aborted = true; break; }
            uint8_t* op = vop + (Gg & 1) * kOpBytes;
            const uint32_t k_tmem = tmem + (static_cast<uint32_t>(16 * r) << 16) + kTmemK + (Gg & 1) * 64;
            if (kind == kKindInvalid) {
              if (is_v) zero_v_tile(op, r, lane);
            } else {
              uint32_t keep_a = 0xFFFFFFFFu, keep_b = 0xFFFFFFFFu;
              if (is_v) {
                const int ntok = min(16, d.t1 - (d.t0 + 16 * u));
                const int ti = lane & 3;
                if (ntok < 16) {
                  keep_a = (2 * ti < ntok ? 0x0000FFFFu : 0u) | (2 * ti + 1 < ntok ? 0xFFFF0000u : 0u);
                  keep_b = (2 * ti + 8 < ntok ? 0x0000FFFFu : 0u) | (2 * ti + 9 < ntok ? 0xFFFF0000u : 0u);
                }
              }
              const bool ok_half = rebuild_half(is_v, st, kind, keep_a, keep_b, op, r, k_tmem, lane, [&]() {
                                            return fetch_block3(sidx, u);
                                          });
              if (!ok_half) {
                armed |= 1u << sidx;               // still in flight: waited for at the end
                aborted = true;
                break;
              }
            }
            if (is_v) {
              fence_proxy_async_smem();
            } else {
              tmem_wait_st();
              tcgen05_before_sync();
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(full_bar(Gg));
            ++n_used;
            if (++st_use == ns) st_use = 0;
            pump(k);
          } else {
            // no tile in this slot of the item's last group: V^T columns zero, K rows unused
            if (!wait_operand_free(Gg)) { aborted = true; break; }
            if (is_v) zero_v_tile(vop + (Gg & 1) * kOpBytes, r, lane);
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(full_bar(Gg));
          }
        }
        if (aborted) break;
        G += ng;
        // every tile of this item was consumed, so started: the start pointer leaves the item before
        // its descriptor buffer is released (and reused for item k + 2)
        if (iss_k == k) {
          iss_k = k + 1;
          iss_u = r;
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars[kBarItemEmpty + buf]);
      }
      // copies still in flight (only after a wait gave up, or started for an item never reached)
      // must land before the CTA exits
      for (int s2 = 0; s2 < ns; ++s2)
        if ((armed & (1u << s2)) && !mbar_wait(&ring_bars[s2], (phase >> s2) & 1)) report(a.status, ZF_DEV_TIMEOUT);
    }
  } else if (warp == kCopyWarp) {
    if constexpr (kCopyWarpFeeds) {
      // ================================================================== copy warp
      // Lane w (< 16) keeps rebuild warp w's stages filled: it follows that warp's tiles (units r,
      // r + 8, .. of every item), and as soon as a stage is handed back (and the item published) it
      // starts the next tile's copy into it, or arrives on its data barrier for a page that could not
      // be resolved.  It leaves an item as soon as it has started that item's last tile for its warp;
      // the warp releases an item once every lane has left it.
      constexpr int kKSt = TcStages<kCols>::kK, kVSt = TcStages<kCols>::kV;
      const bool act = lane < kRebuildWarps;
      const int w = act ? lane : 0;
      const bool is_v = w >= kHalfWarps;
      const int r = is_v ? w - kHalfWarps : 2 * (w & 3) + (w >> 2);
      const int ns = is_v ? kVSt : kKSt;
      const int first_stage = is_v ? kHalfWarps * kKSt + (w - kHalfWarps) * kVSt : w * kKSt;
      uint8_t* ring = stages + static_cast<size_t>(first_stage) * kHalfStageBytes;
      uint64_t* ring_bars = &bars[kBarStage + first_stage];
      uint64_t* ring_empty = &bars[kBarStageEmpty + first_stage];
      const uint64_t policy = l2_evict_first_policy();
      int iss_k = 0, iss_u = r, st = 0, released = 0;
      bool done = !act, ready = false;              // ready: item iss_k is published
      uint32_t used = 0, epar = 0, ipar = 0;        // per stage: started once / next handback parity / last start's parity
      uint64_t idle_since = 0;                      // start of the current run of idle iterations (0: none)
      while (true) {
        bool progress = false, left = false;
        if (!done && !ready) ready = mbar_test(&bars[kBarItemFull + (iss_k & 1)], (iss_k >> 1) & 1);
        if (ready) {
          const ItemDesc& di = desc[iss_k & 1];
          if (di.b < 0) {
            done = true;
            ready = false;
          } else if (iss_u >= di.units) {           // no tile of this warp in the item
            ++iss_k;
            iss_u = r;
            ready = false;
            progress = left = true;
          } else if (!((used >> st) & 1) || mbar_test(&ring_empty[st], (epar >> st) & 1)) {
            uint32_t par = 0;
            if ((used >> st) & 1) {
              epar ^= 1u << st;
              par = static_cast<uint32_t>(spar[first_stage + st]);
            }
            used |= 1u << st;
            ipar = (ipar & ~(1u << st)) | (par << st);
            const int mu = meta[(iss_k & 1) * kMaxItemTiles + iss_u];
            const int kind = mu & 3;
            const size_t head = static_cast<size_t>(mu >> 5) * a.hkv + di.g;
            const int t = (mu >> 2) & 7;
            uint8_t* dst = ring + st * kHalfStageBytes;
            if (kind == kKindComp) {
              mbar_arrive_expect_tx(&ring_bars[st], kTileCompBytes);
              bulk_copy_g2s(dst, (is_v ? a.v_comp : a.k_comp) + head * a.comp_head_bytes + static_cast<size_t>(t) * kTileCompBytes,
                            kTileCompBytes, &ring_bars[st], policy);
            } else if (kind == kKindRaw) {
              mbar_arrive_expect_tx(&ring_bars[st], 3 * kRawBlockBytes);
              bulk_copy_g2s(dst, (is_v ? a.v_raw : a.k_raw) + head * a.raw_head_bytes + static_cast<size_t>(t) * kTileRawBytes,
                            3 * kRawBlockBytes, &ring_bars[st], policy);
            } else {
              mbar_arrive(&ring_bars[st]);
            }
            if (++st == ns) st = 0;
            iss_u += 8;
            if (iss_u >= di.units) {                // leave the item at once: its buffer may be reused
              ++iss_k;
              iss_u = r;
              ready = false;
              left = true;
            }
            progress = true;
          }
        }
        // items every lane has left go back to the metadata warp
        if (__any_sync(0xFFFFFFFFu, left)) {
          const int min_k = __reduce_min_sync(0xFFFFFFFFu, act ? iss_k : INT_MAX);
          while (released < min_k) {
            if (lane == 0) mbar_arrive(&bars[kBarItemEmpty + (released & 1)]);
            ++released;
          }
        }
        if (__any_sync(0xFFFFFFFFu, progress)) {
          idle_since = 0;
          continue;
        }
        if (__all_sync(0xFFFFFFFFu, done)) break;
        if (*abort_flag) break;
        const uint64_t now = global_timer_ns();
        if (idle_since == 0) {
          idle_since = now;
        } else if (now - idle_since > a.wait_limit_ns + kWaitTimeoutNs) {
          *abort_flag = 1;
          report(a.status, ZF_DEV_TIMEOUT);
          break;
        }
      }
      // Every copy started must land before the CTA exits.  Normally its rebuild warp hands the stage
      // back once it has used it; after a wait gave up (abort flag) the copy's own barrier phase is
      // waited for instead (a rebuild warp gives up only before its handback of a stage can be
      // preceded by its own fetch of a raw fourth block, so that phase is still the copy's).
      if (act) {
        const uint64_t t0 = global_timer_ns();
        for (int s2 = 0; s2 < ns; ++s2) {
          if (!((used >> s2) & 1)) continue;
          while (!mbar_test(&ring_empty[s2], (epar >> s2) & 1)) {
            if (*abort_flag) {
              if (!mbar_wait(&ring_bars[s2], (ipar >> s2) & 1)) report(a.status, ZF_DEV_TIMEOUT);
              break;
            }
            if (global_timer_ns() - t0 > kWaitTimeoutNs) {
              report(a.status, ZF_DEV_TIMEOUT);
              break;
            }
          }
        }
      }
    }
  } else if (warp == kMmaWarp) {
    // ================================================================== MMA warp
    // The warp issues both products, whichever is ready first (non-blocking tests), so that
    // neither waits behind the other: S^T = K Q^T of group qk_G and O^T += V^T P^T of group pv_G
    // (pv_G < qk_G).  Every lane runs the loop; one elected lane issues.
    {
      // The item of a group whose S^T is issued and O^T is not yet: the current item k or the one
      // before (item k is published only once item k - 2's outputs were read, so every O^T of
      // item k - 2 was issued by then).  Their first groups tell which.
      int cur_item = -1, cur_first = 0, prev_item = -1, prev_first = 0;
      int qk_G = 0, pv_G = 0, k = -1, gl = 0, ng = 0;
      bool end_seen = false;
      uint64_t t_last = global_timer_ns();
      while (true) {
        bool progress = false;
        if (!end_seen && gl >= ng && mbar_test_warp(&bars[kBarItemFull + ((k + 1) & 1)], ((k + 1) >> 1) & 1)) {
          ++k;
          const ItemDesc d = desc[k & 1];
          if (d.b < 0) {
            end_seen = true;
          } else {
            ng = (d.units + 7) >> 3;
            gl = 0;
            prev_item = cur_item;
            prev_first = cur_first;
            cur_item = k;
            cur_first = qk_G;
          }
          progress = true;
        }
        if (!end_seen && gl < ng) {
          const int G = qk_G;
          if (mbar_test_warp(&bars[kBarKFull + (G & 1)], (G >> 1) & 1) &&
              (G < 2 || mbar_test_warp(&bars[kBarSFree + (G & 1)], ((G >> 1) - 1) & 1)) &&
              (gl != 0 || mbar_test_warp(&bars[kBarQFull + (k & 1)], (k >> 1) & 1))) {
            tcgen05_after_sync();
            const uint32_t d_tmem = tmem + (G & 1) * kCols;
            const uint32_t k_tmem = tmem + kTmemK + (G & 1) * 64;
            const uint8_t* qb = qop + (k & 1) * kCols * 256;
#pragma unroll
            for (int j = 0; j < 8; ++j)
              umma_bf16_ta_elect(d_tmem, k_tmem + 8 * j, umma_desc_kmajor(qb + j * 256), kIdesc, j > 0);
            umma_commit_elect(&bars[kBarSFull + (G & 1)]);
            umma_commit_elect(&bars[kBarKFree + (G & 1)]);
            ++qk_G;
            ++gl;
            progress = true;
          }
        }
        if (pv_G < qk_G) {
          const int G = pv_G;
          const int x_item = G >= cur_first ? cur_item : prev_item;
          const bool x_first = G == cur_first || G == prev_first;
          if (mbar_test_warp(&bars[kBarPFull + (G & 1)], (G >> 1) & 1) &&
              mbar_test_warp(&bars[kBarVFull + (G & 1)], (G >> 1) & 1) &&
              (!x_first || x_item == 0 || mbar_test_warp(&bars[kBarOFree], (x_item - 1) & 1))) {
            tcgen05_after_sync();
            const uint32_t o_tmem = tmem + 2 * kCols;
            const uint8_t* vb = vop + (G & 1) * kOpBytes;
            const uint8_t* pb = pop + (G & 1) * (2 * kCols * 256);
#pragma unroll
            for (int j = 0; j < 8; ++j)
              umma_bf16_elect(o_tmem, umma_desc_kmajor(vb + j * 256), umma_desc_kmajor(pb + j * 256), kIdescPv,
                        !(x_first && j == 0));
            umma_commit_elect(&bars[kBarPvDone + (G & 1)]);
            ++pv_G;
            progress = true;
          }
        }
        if (end_seen && pv_G == qk_G) break;
        if (progress) {
          t_last = global_timer_ns();
        } else if (__nanosleep(64), __any_sync(0xFFFFFFFFu, *abort_flag != 0)) {   // idle: leave the issue slots to the other warps
          break;
        } else if (__any_sync(0xFFFFFFFFu, global_timer_ns() - t_last > a.wait_limit_ns)) {
          if (lane == 0) {
            *abort_flag = 1;
            report(a.status, ZF_DEV_TIMEOUT);
          }
          break;
        }
      }
      // every MMA issued has completed before tensor memory is released
      umma_commit_elect(&bars[kBarDrain]);
      const bool drained = mbar_wait(&bars[kBarDrain], 0);
      if (lane == 0 && !drained) report(a.status, ZF_DEV_TIMEOUT);
    }
    __syncwarp();
  } else {
    // ================================================================== softmax warpgroups
    // Warpgroup hf owns columns hf * kHalf .. + kHalf: their running maxima, sums, P^T columns and
    // output columns (high and low halves), so the two warpgroups never wait for each other.
    constexpr int kHalf = kCols / 2;
    constexpr int NJh = kHalf / 8;                // 8-column blocks of a warpgroup
    const int q = (warp - kSoftmaxWarp0) & 3;     // TMEM lane quadrant (warp % 4)
    const int hf = (warp - kSoftmaxWarp0) >> 2;
    const int c0h = hf * kHalf;                   // first column of this warpgroup
    const uint32_t nb = kSoftmaxBarrier + hf;     // its named barrier
    const int gi = lane >> 2, ti = lane & 3;
    float* red_max = red;                         // [4][kCols]
    float* red_sum = red + 4 * kCols;             // [4][kCols]
    float* alpha_s = red + 8 * kCols;             // [kCols]
    float* m_s = red + 9 * kCols;                 // [kCols]
    const uint32_t lane_base = static_cast<uint32_t>(32 * q) << 16;
    int G = 0;
    for (int k = 0;; ++k) {
      const int buf = k & 1;
      const bool ok_item = wait_or_abort(&bars[kBarItemFull + buf], (k >> 1) & 1, abort_flag, a.status, a.wait_limit_ns);
      const ItemDesc d = desc[buf];
      if (wg_any(nb, !ok_item || d.b < 0)) break;
      const int* mt = meta + buf * kMaxItemTiles;
      const int ng = (d.units + 7) >> 3;
      const int causal_lim = lens[d.b] - a.tokens;   // token t of a request sees positions <= causal_lim + t
      float mcol[NJh][2], lsum[NJh][2];
      float cap[NJh][2];                          // +inf: a column of the slice, -inf: padding
      int lim[NJh][2];                            // last position a column sees (-1: padding column)
#pragma unroll
      for (int j = 0; j < NJh; ++j) {
        mcol[j][0] = mcol[j][1] = kNoScore;
        lsum[j][0] = lsum[j][1] = 0.f;
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const int col = c0h + 8 * j + 2 * ti + e;
          cap[j][e] = col < d.nh ? CUDART_INF_F : -CUDART_INF_F;
          lim[j][e] = col < d.nh ? causal_lim + (d.h0 + col) % a.tokens : -1;
        }
      }
      // the last position every column of the slice sees: columns h0 .. h0 + nh - 1 are tokens
      // (h0 + c) mod T, the earliest of which is 0 unless they stay within one token cycle
      const int r0 = d.h0 % a.tokens;
      const int lim_all = causal_lim + (r0 + d.nh > a.tokens ? 0 : r0);
      bool stop = false;
      for (int gl = 0; gl < ng; ++gl, ++G) {
        const int sb = G & 1;
        bool ok = wait_or_abort(&bars[kBarSFull + sb], (G >> 1) & 1, abort_flag, a.status);
        tcgen05_after_sync();
        uint32_t sr[2][kHalf / 2];
#pragma unroll
        for (int s = 0; s < 2; ++s)
          tmem_ld_scores<kHalf>(tmem + (static_cast<uint32_t>(32 * q + 16 * s) << 16) + sb * kCols + c0h, sr[s]);
        tmem_wait_ld();
        tcgen05_before_sync();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars[kBarSFree + sb]);
        // this group's P buffer is free once the PV two groups back completed
        if (G >= 2) ok = wait_or_abort(&bars[kBarPvDone + sb], ((G >> 1) - 1) & 1, abort_flag, a.status) && ok;
        // scores in the log2 domain; hidden: past the item, unresolved pages, padding columns,
        // positions past a new token's own
        // This thread's rows are tokens tok0 + {0, 8} of tile u0 and tok0 + {16, 24} of tile u0 + 1.
        // Fast path (32 columns, where the softmax paces the kernel; at 16 it measured slower):
        // both tiles resolved, and every row inside the item and seen by every column.
        float x[2][NJh][4];
        const int tok0 = 128 * gl + 32 * q + gi;
        const int u0 = tok0 >> 4;
        const bool all_seen = kCols == 32 && u0 + 1 < d.units && (mt[u0] & 3) != kKindInvalid && (mt[u0 + 1] & 3) != kKindInvalid &&
                              d.t0 + tok0 + 24 < d.t1 && d.t0 + tok0 + 24 <= lim_all;
        if (all_seen) {
#pragma unroll
          for (int s = 0; s < 2; ++s)
#pragma unroll
            for (int j = 0; j < NJh; ++j)
#pragma unroll
              for (int i = 0; i < 4; ++i)
                x[s][j][i] = fminf(__uint_as_float(sr[s][4 * j + i]) * a.scale_log2, cap[j][i & 1]);
        } else {
#pragma unroll
          for (int s = 0; s < 2; ++s) {
#pragma unroll
            for (int i2 = 0; i2 < 2; ++i2) {
              const int tok = tok0 + 16 * s + 8 * i2;     // token offset within the item
              const int u = tok >> 4;
              const int pos = (u < d.units && (mt[u] & 3) != kKindInvalid && d.t0 + tok < d.t1) ? d.t0 + tok : INT_MAX;
#pragma unroll
              for (int j = 0; j < NJh; ++j)
#pragma unroll
                for (int e = 0; e < 2; ++e)
                  x[s][j][2 * i2 + e] =
                      pos <= lim[j][e] ? __uint_as_float(sr[s][4 * j + 2 * i2 + e]) * a.scale_log2 : -CUDART_INF_F;
            }
          }
        }
        bool grow = false;
#pragma unroll
        for (int j = 0; j < NJh; ++j)
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            const float mx = fmaxf(fmaxf(x[0][j][e], x[0][j][2 + e]), fmaxf(x[1][j][e], x[1][j][2 + e]));
            grow = grow || mx > mcol[j][e] + kRescaleThreshold;
          }
        if (wg_any(nb, grow || !ok)) {
          // the output holds this item's earlier groups: its rescale needs the previous PV done
          if (gl > 0) ok = wait_or_abort(&bars[kBarPvDone + (sb ^ 1)], ((G - 1) >> 1) & 1, abort_flag, a.status) && ok;
          if (wg_any(nb, !ok)) {
            stop = true;
            break;
          }
          tcgen05_after_sync();
          // column maxima over the warpgroup's 128 tokens, then the new running max
#pragma unroll
          for (int j = 0; j < NJh; ++j)
#pragma unroll
            for (int e = 0; e < 2; ++e) {
              float v = fmaxf(fmaxf(x[0][j][e], x[0][j][2 + e]), fmaxf(x[1][j][e], x[1][j][2 + e]));
#pragma unroll
              for (int dd = 4; dd < 32; dd <<= 1) v = fmaxf(v, __shfl_xor_sync(0xFFFFFFFFu, v, dd));
              if (gi == 0) red_max[q * kCols + c0h + 8 * j + 2 * ti + e] = v;
            }
          wg_sync(nb);
#pragma unroll
          for (int j = 0; j < NJh; ++j)
#pragma unroll
            for (int e = 0; e < 2; ++e) {
              const int c = c0h + 8 * j + 2 * ti + e;
              const float nm = fmaxf(fmaxf(mcol[j][e], fmaxf(red_max[c], red_max[kCols + c])),
                                     fmaxf(red_max[2 * kCols + c], red_max[3 * kCols + c]));   // finite: >= kNoScore
              const float al = fast_exp2(mcol[j][e] - nm);
              mcol[j][e] = nm;
              lsum[j][e] *= al;
              if (q == 0 && gi == 0) alpha_s[c] = al;
            }
          wg_sync(nb);
          if (gl > 0) {
            // rescale this warpgroup's output columns in tensor memory: high halves at 2 kCols + c,
            // low halves at 3 kCols + c
#pragma unroll 1
            for (int c0 = 0; c0 < 2 * kHalf; c0 += 8) {
              const int c = c0h + (c0 & (kHalf - 1));
              const uint32_t col = (c0 < kHalf ? 2 * kCols : 3 * kCols) + c;
              uint32_t o[8];
              tmem_ld_32x32b_x8(tmem + lane_base + col, o);
              tmem_wait_ld();
#pragma unroll
              for (int i = 0; i < 8; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha_s[c + i]);
              tmem_st_32x32b_x8(tmem + lane_base + col, o);
            }
            tmem_wait_st();
          }
        }
        // P = 2^(x - m): BF16 high part and BF16 remainder, transposed into P^T core matrices
        // (n-block c0h / 8 + j, k-block 4q + 2s (+1 for tokens 8-15 of the 16)) of buffer G & 1
        uint8_t* pb = pop + sb * (2 * kCols * 256) + (c0h / 8) * kCoreRow;
#pragma unroll
        for (int s = 0; s < 2; ++s) {
#pragma unroll
          for (int j = 0; j < NJh; ++j) {
            const float p0 = fast_exp2(x[s][j][0] - mcol[j][0]), p1 = fast_exp2(x[s][j][1] - mcol[j][1]);
            const float p2 = fast_exp2(x[s][j][2] - mcol[j][0]), p3 = fast_exp2(x[s][j][3] - mcol[j][1]);
            lsum[j][0] += p0 + p2;
            lsum[j][1] += p1 + p3;
            const uint32_t h01 = pack_bf16x2(p0, p1), h23 = pack_bf16x2(p2, p3);
            const uint32_t r01 = pack_bf16x2(p0 - bf16lo_to_f32(h01), p1 - bf16hi_to_f32(h01));
            const uint32_t r23 = pack_bf16x2(p2 - bf16lo_to_f32(h23), p3 - bf16hi_to_f32(h23));
            uint8_t* ph = pb + j * kCoreRow + (4 * q + 2 * s) * 128 + gi * 16 + ti * 4;
            *reinterpret_cast<uint32_t*>(ph) = transpose8x8(h01);
            *reinterpret_cast<uint32_t*>(ph + 128) = transpose8x8(h23);
            *reinterpret_cast<uint32_t*>(ph + kCols * 256) = transpose8x8(r01);
            *reinterpret_cast<uint32_t*>(ph + kCols * 256 + 128) = transpose8x8(r23);
          }
        }
        fence_proxy_async_smem();
        tcgen05_before_sync();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars[kBarPFull + sb]);   // P written (and the output rescaled)
      }
      if (stop) break;
      // ---- the item's output: O^T / column sums (once the last group's PV has completed)
      const bool ok = wait_or_abort(&bars[kBarPvDone + ((G - 1) & 1)], ((G - 1) >> 1) & 1, abort_flag, a.status);
      tcgen05_after_sync();
#pragma unroll
      for (int j = 0; j < NJh; ++j)
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          float v = lsum[j][e];
#pragma unroll
          for (int dd = 4; dd < 32; dd <<= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, dd);
          if (gi == 0) {
            red_sum[q * kCols + c0h + 8 * j + 2 * ti + e] = v;
            if (q == 0) m_s[c0h + 8 * j + 2 * ti + e] = mcol[j][e];
          }
        }
      if (wg_any(nb, !ok)) break;                 // also makes red_sum and m_s visible
      const int ch = 32 * q + lane;               // this thread's output channel (TMEM lane)
#pragma unroll 1
      for (int c0 = c0h; c0 < c0h + kHalf; c0 += 8) {
        uint32_t o[8], olo[8];
        tmem_ld_32x32b_x8(tmem + lane_base + 2 * kCols + c0, o);
        tmem_ld_32x32b_x8(tmem + lane_base + 3 * kCols + c0, olo);
        tmem_wait_ld();
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const int n = c0 + i;
          if (n < d.nh) {
            const float lsum_n = red_sum[n] + red_sum[kCols + n] + red_sum[2 * kCols + n] + red_sum[3 * kCols + n];
            const float inv = lsum_n > 0.f ? 1.f / lsum_n : 0.f;
            const float lse2 = lsum_n > 0.f ? m_s[n] + log2f(lsum_n) : -CUDART_INF_F;
            const float val = (__uint_as_float(o[i]) + __uint_as_float(olo[i])) * inv;
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
      wg_sync(nb);                                // every warp read the output and the sums
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

int attention_tc_cols(int hq, int hkv) { return hq / hkv > 16 ? 32 : 16; }

bool attention_tc_fits(int32_t batch, int hq, int hkv) {
  const size_t bytes = attention_tc_cols(hq, hkv) == 32 ? tc_layout<32>(batch).total : tc_layout<16>(batch).total;
  return bytes <= 227 * 1024;
}

Plan attention_tc_plan(int batch, int hq, int hkv, int page_size, int max_pages, int num_sms) {
  return make_plan(batch, hq, hkv, page_size, max_pages, num_sms, kHalfWarps, attention_tc_cols(hq, hkv));
}

template <int kCols>
static zf_status launch_tc(const AttnArgs& base, const Plan& p, int32_t tokens, cudaStream_t stream) {
  AttnArgs a = base;
  a.hps = kCols;
  a.slices = p.slices;
  a.max_chunks = p.max_chunks;
  a.min_range_pages = p.min_range_pages;
  a.chunk_pages = p.chunk_pages;
  a.prefetch = 0;
  a.plan_first = 0;
  const size_t smem = tc_layout<kCols>(a.batch).total;
  // one record per instantiation (16 columns: 0, 32 columns: 1)
  zf_status st = ensure_smem_limit(reinterpret_cast<const void*>(attn_tc_kernel<kCols>), kCols / 32, smem);
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
  if (cudaLaunchKernelEx(&cfg, attn_tc_kernel<kCols>, a) != cudaSuccess) return ZF_ERR_CUDA;
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
  m.hps = kCols;
  return launch_merge(m, tokens > 1, stream);
}

zf_status launch_attention_tc(const AttnArgs& base, const Plan& p, int32_t tokens, cudaStream_t stream) {
  return attention_tc_cols(base.hq, base.hkv) == 32 ? launch_tc<32>(base, p, tokens, stream)
                                                   : launch_tc<16>(base, p, tokens, stream);
}

}  // namespace zf
