// zf_decode_attn / zf_dense_decode_attn: split-KV decode attention over a paged KV cache whose
// full pages are stored compressed, plus the split-result merge.
//
// ZipFusion §III.C (Attention over the Compressed KV Cache): compressed blocks are copied
// HBM -> shared memory as they are, each thread rebuilds the exact BF16 operands of a
// tensor-core instruction in registers right before use, raw blocks need no rebuild, and page
// metadata for later pages is fetched while earlier pages are attended.  ZipFusion §IV.B:
// split-KV partial results are combined by a split-result merge.
//
// Design for sm_103a (one CTA per SM, persistent over a static list of work items):
//  * work item = (request b, kv head g, head slice, chunk of pages); the chunk size is picked on
//    the host so that items fill the SMs in whole rounds;
//  * warp 8 is the producer: it resolves page ids through the page table and the directory and
//    streams every 16-token tile (K 4 blocks + V 4 blocks) into a 16-stage shared-memory ring
//    with 1-D bulk copies (cp.async.bulk, mbarrier transaction counts, L2 evict-first);
//  * warps 0-7 consume tiles round-robin.  A warp rebuilds K blocks straight into m16n8k16
//    A fragments (the storage order is the fragment order), computes S^T = K Q^T for up to 8
//    query heads of the GQA group (one MMA n-tile), runs the online softmax in the log2 domain,
//    transposes P^T into B fragments with movmatrix, and accumulates O^T = V^T P^T with P split
//    into a BF16 high part and a BF16 remainder (two MMAs) so P keeps ~16 significant bits;
//  * at the end of an item the 8 warps' (m, l, O) are merged through shared memory and written
//    as the item's partial (or as the final output when the request has a single chunk);
//  * a second kernel merges each (request, head)'s chunk partials by log-sum-exp.
#include <cuda_runtime.h>
#include <math_constants.h>
#include <stdint.h>

#include <climits>
#include <mutex>

#include "zf_device.cuh"
#include "zf_host.h"

namespace zf {

constexpr int kConsumerWarps = 8;
constexpr int kAttnThreads = (kConsumerWarps + 1) * 32;
constexpr int kStages = 16;
constexpr int kStageBytes = 8192;                   // K tile + V tile, raw size
constexpr int kHalfStage = 4096;
constexpr int kTileCompBytes = 4 * kSlotBytes;      // 3136: one 16-token tile of K (or V), compressed
constexpr int kTileRawBytes = 4 * kRawBlockBytes;   // 4096
constexpr int kHeadsPerSlice = 8;                   // MMA n
constexpr int kOStride = 132;                       // padded combine row (conflict-free writes)
constexpr int kCombineWarpFloats = kHeadsPerSlice * kOStride + 16;
constexpr int kItemOverheadTiles = 4;               // planner: fixed cost of an item, in tiles
constexpr float kLn2 = 0.6931471805599453f;

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
  int32_t batch, hq, hkv, group, slices, page_size, num_pages, num_raw, max_pages, chunk_pages, max_chunks;
  int64_t comp_head_bytes;   // bytes of one (page, kv head) K record, compressed
  int64_t raw_head_bytes;    // bytes of one (page, kv head) K record, raw
  float scale_log2;          // softmax_scale * log2(e)
};

struct Plan {
  int grid = 0, chunk_pages = 1, max_chunks = 0, slices = 1;
  size_t part_o_bytes = 0, ws_bytes = 0, smem = 0;
};

struct SmemLayout {
  size_t stages, full, empty, kinds, flag, combine, lens, prefix, total;
};

__host__ __device__ inline SmemLayout smem_layout(int batch) {
  SmemLayout s;
  size_t at = 0;
  s.stages = at; at += static_cast<size_t>(kStages) * kStageBytes;
  s.full = at; at += kStages * 8;
  s.empty = at; at += kStages * 8;
  s.kinds = at; at += kStages * 4;
  s.flag = at; at += 16;
  s.combine = at; at += static_cast<size_t>(kConsumerWarps) * kCombineWarpFloats * 4;
  s.lens = at; at += static_cast<size_t>(batch) * 4;
  s.prefix = at; at += static_cast<size_t>(batch + 1) * 4;
  s.total = (at + 127) & ~static_cast<size_t>(127);
  return s;
}

struct Item {
  int b, g, s, c, p0, p1, t0, t1, units;
};

__device__ __forceinline__ Item decode_item(const AttnArgs& a, const int* lens, const int* prefix, int item) {
  Item it;
  const int per = a.hkv * a.slices;
  const int j = item / per;
  const int r = item - j * per;
  it.g = r / a.slices;
  it.s = r - it.g * a.slices;
  int lo = 0, hi = a.batch;                 // prefix[lo] <= j < prefix[hi]
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (prefix[mid] <= j) lo = mid; else hi = mid;
  }
  it.b = lo;
  it.c = j - prefix[lo];
  const int L = lens[lo];
  const int pages = (L + a.page_size - 1) / a.page_size;
  it.p0 = it.c * a.chunk_pages;
  it.p1 = min(it.p0 + a.chunk_pages, pages);
  it.t0 = it.p0 * a.page_size;
  it.t1 = min(it.p1 * a.page_size, L);
  it.units = (it.t1 - it.t0 + 15) >> 4;
  return it;
}

__device__ __forceinline__ void consumer_barrier() {
  asm volatile("bar.sync 1, %0;" ::"n"(kConsumerWarps * 32) : "memory");
}

template <bool kCompressed>
__global__ void __launch_bounds__(kAttnThreads, 1) attn_kernel(const AttnArgs a) {
  extern __shared__ __align__(128) uint8_t smem[];
  const SmemLayout L = smem_layout(a.batch);
  uint8_t* stages = smem + L.stages;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + L.full);
  uint64_t* empty = reinterpret_cast<uint64_t*>(smem + L.empty);
  int* kinds = reinterpret_cast<int*>(smem + L.kinds);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L.flag);
  float* combine = reinterpret_cast<float*>(smem + L.combine);
  int* lens = reinterpret_cast<int*>(smem + L.lens);
  int* prefix = reinterpret_cast<int*>(smem + L.prefix);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  // ---- prologue: barriers, clamped lengths, chunk counts and their prefix sums
  if (tid < kStages) {
    mbar_init(&full[tid], 1);
    mbar_init(&empty[tid], 1);
  }
  if (tid == 0) *abort_flag = 0;
  const int max_len = a.max_pages * a.page_size;
  for (int b = tid; b < a.batch; b += kAttnThreads) {
    int len = a.seq_lens[b];
    if (len < 0 || len > max_len) {
      if (blockIdx.x == 0) report(a.status, ZF_DEV_BAD_SEQ_LEN);
      len = min(max(len, 0), max_len);
    }
    lens[b] = len;
    const int pages = (len + a.page_size - 1) / a.page_size;
    prefix[b + 1] = (pages + a.chunk_pages - 1) / a.chunk_pages;
  }
  fence_mbar_init();
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
  const int total_items = prefix[a.batch] * a.hkv * a.slices;

  if (warp == kConsumerWarps) {
    // ================================================================ producer warp
    const uint64_t policy = l2_evict_first_policy();
    uint32_t seq = 0;
    bool ok = true;
    for (int item = blockIdx.x; item < total_items && ok; item += gridDim.x) {
      const Item it = decode_item(a, lens, prefix, item);
      const int32_t* row = a.page_table + static_cast<size_t>(it.b) * a.max_pages;
      for (int pb = it.p0; pb < it.p1 && ok; pb += 32) {
        // page metadata for the next 32 pages, one lane each
        const int pi = pb + lane;
        int kind = kKindInvalid, slot = 0;
        if (pi < it.p1) {
          const int pid = row[pi];
          if (kCompressed) {
            if (pid >= 0 && pid < a.num_pages) {
              const int d = a.dir[static_cast<size_t>(pid) * a.hkv + it.g];
              if (d == ZF_DIR_COMPRESSED) {
                kind = kKindComp;
                slot = pid;
              } else if (d >= 0 && d < a.num_raw) {
                kind = kKindRaw;
                slot = d;
              } else {
                report(a.status, ZF_DEV_BAD_DIR);
              }
            } else {
              report(a.status, ZF_DEV_BAD_PAGE_ID);
            }
          } else if (pid >= 0 && pid < a.num_raw) {
            kind = kKindRaw;
            slot = pid;
          } else {
            report(a.status, ZF_DEV_BAD_PAGE_ID);
          }
        }
        const int npg = min(32, it.p1 - pb);
        for (int j = 0; j < npg; ++j) {
          const int kind_j = __shfl_sync(0xFFFFFFFFu, kind, j);
          const int slot_j = __shfl_sync(0xFFFFFFFFu, slot, j);
          const int ntok = min(a.page_size, it.t1 - (pb + j) * a.page_size);
          const int ntiles = (ntok + 15) >> 4;
          if (lane == 0) {
            const size_t head = static_cast<size_t>(slot_j) * a.hkv + it.g;
            for (int t = 0; t < ntiles; ++t) {
              const int stage = static_cast<int>(seq % kStages);
              const uint32_t phase = (seq / kStages) & 1u;
              if (*abort_flag || !mbar_wait(&empty[stage], phase ^ 1u)) {
                report(a.status, ZF_DEV_TIMEOUT);
                *abort_flag = 1;
                ok = false;
                break;
              }
              kinds[stage] = kind_j;
              uint8_t* dst = stages + static_cast<size_t>(stage) * kStageBytes;
              if (kind_j == kKindComp) {
                const size_t off = head * a.comp_head_bytes + static_cast<size_t>(t) * kTileCompBytes;
                mbar_arrive_expect_tx(&full[stage], 2 * kTileCompBytes);
                bulk_copy_g2s(dst, a.k_comp + off, kTileCompBytes, &full[stage], policy);
                bulk_copy_g2s(dst + kHalfStage, a.v_comp + off, kTileCompBytes, &full[stage], policy);
              } else if (kind_j == kKindRaw) {
                const size_t off = head * a.raw_head_bytes + static_cast<size_t>(t) * kTileRawBytes;
                mbar_arrive_expect_tx(&full[stage], 2 * kTileRawBytes);
                bulk_copy_g2s(dst, a.k_raw + off, kTileRawBytes, &full[stage], policy);
                bulk_copy_g2s(dst + kHalfStage, a.v_raw + off, kTileRawBytes, &full[stage], policy);
              } else {
                mbar_arrive(&full[stage]);
              }
              ++seq;
            }
          }
          ok = __shfl_sync(0xFFFFFFFFu, ok, 0);
          if (!ok) break;
        }
      }
    }
    if (lane == 0 && !ok) {
      // give copies already in flight a bounded chance to land before the CTA exits
      for (int s = 0; s < kStages; ++s) {
        if (seq > static_cast<uint32_t>(s)) {
          const uint32_t last = seq - 1 - ((seq - 1 - s) % kStages);
          mbar_wait(&full[s], (last / kStages) & 1u);
        }
      }
    }
    return;
  }

  // ================================================================== consumer warps
  const int gi = lane >> 2, ti = lane & 3;
  uint32_t seq_base = 0;
  bool aborted = false;
  float* my_combine = combine + warp * kCombineWarpFloats;
  for (int item = blockIdx.x; item < total_items; item += gridDim.x) {
    const Item it = decode_item(a, lens, prefix, item);
    const int h0 = it.g * a.group + it.s * kHeadsPerSlice;
    const int nh = min(kHeadsPerSlice, a.group - it.s * kHeadsPerSlice);

    // Q^T as the B operand (k = channel, n = head): lane holds head gi, channels 2ti(+1), +8(+9)
    uint32_t qb[8][2];
    {
      const uint32_t* qrow = reinterpret_cast<const uint32_t*>(
          a.q + (static_cast<size_t>(it.b) * a.hq + h0 + min(gi, nh - 1)) * ZF_HEAD_DIM);
#pragma unroll
      for (int ks = 0; ks < 8; ++ks) {
        qb[ks][0] = gi < nh ? qrow[8 * ks + ti] : 0u;
        qb[ks][1] = gi < nh ? qrow[8 * ks + ti + 4] : 0u;
      }
    }
    float m0 = -CUDART_INF_F, m1 = -CUDART_INF_F, l0 = 0.f, l1 = 0.f;
    float o[8][4];
#pragma unroll
    for (int mt = 0; mt < 8; ++mt) o[mt][0] = o[mt][1] = o[mt][2] = o[mt][3] = 0.f;

    for (int k = warp; k < it.units; k += kConsumerWarps) {
      const uint32_t s = seq_base + k;
      const int stage = static_cast<int>(s % kStages);
      if (!aborted && (*abort_flag || !mbar_wait(&full[stage], (s / kStages) & 1u))) {
        aborted = true;
        *abort_flag = 1;
        report(a.status, ZF_DEV_TIMEOUT);
      }
      if (aborted) continue;
      const int kind = kinds[stage];
      const int ntok = min(16, it.t1 - (it.t0 + 16 * k));
      const uint8_t* kp = stages + static_cast<size_t>(stage) * kStageBytes;
      const uint8_t* vp = kp + kHalfStage;

      // ---- S^T (16 tokens x 8 heads) = K (16 x 128) . Q^T (128 x 8)
      float sacc[4] = {0.f, 0.f, 0.f, 0.f};
      uint32_t va[4][8];
      if (kCompressed && kind == kKindComp) {
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          uint32_t ka[8];
          rebuild_lane(kp + j * kSlotBytes, lane, ka);
          mma_bf16(sacc, ka[0], ka[1], ka[2], ka[3], qb[2 * j][0], qb[2 * j][1]);
          mma_bf16(sacc, ka[4], ka[5], ka[6], ka[7], qb[2 * j + 1][0], qb[2 * j + 1][1]);
        }
#pragma unroll
        for (int j = 0; j < 4; ++j) rebuild_lane(vp + j * kSlotBytes, lane, va[j]);
      } else if (kind == kKindRaw) {
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          uint32_t ka[8];
          load_raw_lane(kp + j * kRawBlockBytes, lane, ka);
          mma_bf16(sacc, ka[0], ka[1], ka[2], ka[3], qb[2 * j][0], qb[2 * j][1]);
          mma_bf16(sacc, ka[4], ka[5], ka[6], ka[7], qb[2 * j + 1][0], qb[2 * j + 1][1]);
        }
#pragma unroll
        for (int j = 0; j < 4; ++j) load_raw_lane(vp + j * kRawBlockBytes, lane, va[j]);
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[stage]);   // the stage is free once its bytes are in registers
      if (kind == kKindInvalid) continue;
      if (ntok < 16) {
        // tokens past the context may hold anything (even NaN): zero their values so that
        // p = 0 times them stays 0.  V^T fragment columns of this lane: tokens 2ti, 2ti+1 (regs
        // 0,1,4,5) and 2ti+8, 2ti+9 (regs 2,3,6,7).
        const uint32_t keep_a = (2 * ti < ntok ? 0x0000FFFFu : 0u) | (2 * ti + 1 < ntok ? 0xFFFF0000u : 0u);
        const uint32_t keep_b = (2 * ti + 8 < ntok ? 0x0000FFFFu : 0u) | (2 * ti + 9 < ntok ? 0xFFFF0000u : 0u);
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          va[j][0] &= keep_a; va[j][1] &= keep_a; va[j][4] &= keep_a; va[j][5] &= keep_a;
          va[j][2] &= keep_b; va[j][3] &= keep_b; va[j][6] &= keep_b; va[j][7] &= keep_b;
        }
      }

      // ---- online softmax (log2 domain).  sacc: (token gi | gi+8) x (head 2ti | 2ti+1)
      float x0 = sacc[0] * a.scale_log2, x1 = sacc[1] * a.scale_log2;
      float x2 = sacc[2] * a.scale_log2, x3 = sacc[3] * a.scale_log2;
      if (gi >= ntok) x0 = x1 = -CUDART_INF_F;
      if (gi + 8 >= ntok) x2 = x3 = -CUDART_INF_F;
      float mx0 = fmaxf(x0, x2), mx1 = fmaxf(x1, x3);
#pragma unroll
      for (int d = 4; d < 32; d <<= 1) {
        mx0 = fmaxf(mx0, __shfl_xor_sync(0xFFFFFFFFu, mx0, d));
        mx1 = fmaxf(mx1, __shfl_xor_sync(0xFFFFFFFFu, mx1, d));
      }
      const float mn0 = fmaxf(m0, mx0), mn1 = fmaxf(m1, mx1);   // finite: token 0 of a tile is valid
      const float al0 = exp2f(m0 - mn0), al1 = exp2f(m1 - mn1);
      const float p0 = exp2f(x0 - mn0), p1 = exp2f(x1 - mn1);
      const float p2 = exp2f(x2 - mn0), p3 = exp2f(x3 - mn1);
      m0 = mn0;
      m1 = mn1;
      l0 = l0 * al0 + (p0 + p2);
      l1 = l1 * al1 + (p1 + p3);
#pragma unroll
      for (int mt = 0; mt < 8; ++mt) {
        o[mt][0] *= al0;
        o[mt][1] *= al1;
        o[mt][2] *= al0;
        o[mt][3] *= al1;
      }
      // P^T as the B operand (k = token, n = head): high BF16 part and BF16 remainder
      const uint32_t h01 = pack_bf16x2(p0, p1), h23 = pack_bf16x2(p2, p3);
      const uint32_t r01 = pack_bf16x2(p0 - bf16lo_to_f32(h01), p1 - bf16hi_to_f32(h01));
      const uint32_t r23 = pack_bf16x2(p2 - bf16lo_to_f32(h23), p3 - bf16hi_to_f32(h23));
      const uint32_t bh0 = transpose8x8(h01), bh1 = transpose8x8(h23);
      const uint32_t bl0 = transpose8x8(r01), bl1 = transpose8x8(r23);

      // ---- O^T (128 channels x 8 heads) += V^T (128 x 16 tokens) . P^T (16 x 8)
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        mma_bf16(o[2 * j], va[j][0], va[j][1], va[j][2], va[j][3], bh0, bh1);
        mma_bf16(o[2 * j], va[j][0], va[j][1], va[j][2], va[j][3], bl0, bl1);
        mma_bf16(o[2 * j + 1], va[j][4], va[j][5], va[j][6], va[j][7], bh0, bh1);
        mma_bf16(o[2 * j + 1], va[j][4], va[j][5], va[j][6], va[j][7], bl0, bl1);
      }
    }
    seq_base += static_cast<uint32_t>(it.units);

    // ---- merge the 8 warps' states of this item through shared memory
#pragma unroll
    for (int d = 4; d < 32; d <<= 1) {
      l0 += __shfl_xor_sync(0xFFFFFFFFu, l0, d);
      l1 += __shfl_xor_sync(0xFFFFFFFFu, l1, d);
    }
    float* cm = my_combine + kHeadsPerSlice * kOStride;
    float* cl = cm + kHeadsPerSlice;
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
    consumer_barrier();
    {
      const int hh = warp;                 // this thread finishes head hh, channels 4*lane..+3
      if (hh < nh) {
        float mw[kConsumerWarps];
        float M = -CUDART_INF_F;
#pragma unroll
        for (int w = 0; w < kConsumerWarps; ++w) {
          mw[w] = combine[w * kCombineWarpFloats + kHeadsPerSlice * kOStride + hh];
          M = fmaxf(M, mw[w]);
        }
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
        float lsum = 0.f;
        if (M != -CUDART_INF_F) {
#pragma unroll
          for (int w = 0; w < kConsumerWarps; ++w) {
            const float* cwp = combine + w * kCombineWarpFloats;
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
        const size_t bh = static_cast<size_t>(it.b) * a.hq + h0 + hh;
        if (prefix[it.b + 1] - prefix[it.b] == 1) {
          *reinterpret_cast<float4*>(a.out + bh * ZF_HEAD_DIM + 4 * lane) = acc;
          if (lane == 0) a.lse[bh] = lse2 * kLn2;
        } else {
          const size_t pidx = bh * a.max_chunks + it.c;
          *reinterpret_cast<float4*>(a.part_o + pidx * ZF_HEAD_DIM + 4 * lane) = acc;
          if (lane == 0) a.part_lse[pidx] = lse2;
        }
      }
    }
    consumer_barrier();
  }
}

struct MergeArgs {
  const int32_t* seq_lens;
  const float* part_o;
  const float* part_lse;
  float* out;
  float* lse;
  int32_t batch, hq, page_size, max_pages, chunk_pages, max_chunks;
};

// One warp per (request, query head): lse = log2 sum_i 2^lse_i, out = sum_i 2^(lse_i - lse) o_i.
// Requests with one chunk were finished by the attention kernel; empty requests get 0 / -inf.
__global__ void __launch_bounds__(128) merge_kernel(const MergeArgs a) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int idx = blockIdx.x * 4 + warp;
  if (idx >= a.batch * a.hq) return;
  const int b = idx / a.hq;
  const int len = min(max(a.seq_lens[b], 0), a.max_pages * a.page_size);
  const int pages = (len + a.page_size - 1) / a.page_size;
  const int nch = (pages + a.chunk_pages - 1) / a.chunk_pages;
  float4* outp = reinterpret_cast<float4*>(a.out + static_cast<size_t>(idx) * ZF_HEAD_DIM) + lane;
  if (nch == 1) return;
  const float* pl = a.part_lse + static_cast<size_t>(idx) * a.max_chunks;
  float M = -CUDART_INF_F;
  for (int i = lane; i < nch; i += 32) M = fmaxf(M, pl[i]);
#pragma unroll
  for (int d = 16; d > 0; d >>= 1) M = fmaxf(M, __shfl_xor_sync(0xFFFFFFFFu, M, d));
  if (nch == 0 || M == -CUDART_INF_F) {
    *outp = make_float4(0.f, 0.f, 0.f, 0.f);
    if (lane == 0) a.lse[idx] = -CUDART_INF_F;
    return;
  }
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  float lsum = 0.f;
  const float4* po = reinterpret_cast<const float4*>(a.part_o + static_cast<size_t>(idx) * a.max_chunks * ZF_HEAD_DIM) + lane;
  for (int i = 0; i < nch; ++i) {
    const float f = exp2f(pl[i] - M);
    const float4 v = po[static_cast<size_t>(i) * (ZF_HEAD_DIM / 4)];
    lsum += f;
    acc.x += f * v.x;
    acc.y += f * v.y;
    acc.z += f * v.z;
    acc.w += f * v.w;
  }
  const float inv = 1.f / lsum;
  *outp = make_float4(acc.x * inv, acc.y * inv, acc.z * inv, acc.w * inv);
  if (lane == 0) a.lse[idx] = (M + log2f(lsum)) * kLn2;
}

// ------------------------------------------------------------------------------- host planner
static Plan make_plan(int batch, int hq, int hkv, int page_size, int max_pages, int num_sms) {
  Plan p;
  const int group = hq / hkv;
  p.slices = (group + kHeadsPerSlice - 1) / kHeadsPerSlice;
  const long long pairs = static_cast<long long>(batch) * hkv * p.slices;
  const int tiles = page_size / ZF_BLOCK_TOKENS;
  long long best = LLONG_MAX;
  int best_cp = max_pages;
  for (int cp = 1; cp <= max_pages; ++cp) {
    const long long chunks = (max_pages + cp - 1) / cp;
    const long long items = pairs * chunks;
    const long long grid = items < num_sms ? items : num_sms;
    const long long rounds = (items + grid - 1) / grid;
    const long long cost = rounds * (static_cast<long long>(cp) * tiles + kItemOverheadTiles);
    if (cost <= best) {          // ties go to the larger chunk (fewer partials)
      best = cost;
      best_cp = cp;
    }
  }
  p.chunk_pages = best_cp;
  p.max_chunks = (max_pages + best_cp - 1) / best_cp;
  const long long items = pairs * p.max_chunks;
  p.grid = static_cast<int>(items < num_sms ? (items > 0 ? items : 1) : num_sms);
  const size_t n = static_cast<size_t>(batch) * hq * p.max_chunks;
  p.part_o_bytes = n * ZF_HEAD_DIM * 4;
  p.ws_bytes = p.part_o_bytes + ((n * 4 + 255) & ~static_cast<size_t>(255));
  p.smem = smem_layout(batch).total;
  return p;
}

static zf_status current_sm_count(int* sms) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return ZF_ERR_CUDA;
  if (cudaDeviceGetAttribute(sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return ZF_ERR_CUDA;
  return ZF_OK;
}

static bool attn_shape_ok(int batch, int hq, int hkv, int max_pages) {
  return batch >= 0 && batch <= ZF_MAX_BATCH && hkv >= 1 && hq >= hkv && hq % hkv == 0 && max_pages >= 1 &&
         static_cast<long long>(max_pages) * ZF_MAX_PAGE_SIZE < INT_MAX;
}

template <bool kCompressed>
static zf_status launch_attention(const zf_cache* c, const uint16_t* q, int32_t batch, int32_t hq,
                                  const int32_t* page_table, int32_t max_pages, const int32_t* seq_lens,
                                  float scale, float* out, float* lse, void* workspace, size_t ws_bytes,
                                  void* stream) {
  zf_status st = check_cache(c, kCompressed, true, kCompressed);
  if (st != ZF_OK) return st;
  if (!attn_shape_ok(batch, hq, c->num_kv_heads, max_pages)) return ZF_ERR_INVALID_ARGUMENT;
  if (batch == 0) return ZF_OK;
  if (!q || !page_table || !seq_lens || !out || !lse || !workspace) return ZF_ERR_INVALID_ARGUMENT;
  if (!aligned16(q) || !aligned16(out) || !aligned16(workspace) || (reinterpret_cast<uintptr_t>(lse) & 3u) ||
      (reinterpret_cast<uintptr_t>(page_table) & 3u) || (reinterpret_cast<uintptr_t>(seq_lens) & 3u))
    return ZF_ERR_INVALID_ARGUMENT;
  if (!(scale == scale)) return ZF_ERR_INVALID_ARGUMENT;
  int sms = 0;
  if ((st = current_sm_count(&sms)) != ZF_OK) return st;
  const Plan p = make_plan(batch, hq, c->num_kv_heads, c->page_size, max_pages, sms);
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
  a.batch = batch;
  a.hq = hq;
  a.hkv = c->num_kv_heads;
  a.group = hq / c->num_kv_heads;
  a.slices = p.slices;
  a.page_size = c->page_size;
  a.num_pages = c->num_pages;
  a.num_raw = c->num_raw_slots;
  a.max_pages = max_pages;
  a.chunk_pages = p.chunk_pages;
  a.max_chunks = p.max_chunks;
  a.comp_head_bytes = static_cast<int64_t>(c->page_size / 4) * kSlotBytes;
  a.raw_head_bytes = static_cast<int64_t>(c->page_size / 4) * kRawBlockBytes;
  a.scale_log2 = scale * 1.4426950408889634f;

  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (cudaFuncSetAttribute(attn_kernel<kCompressed>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(p.smem)) != cudaSuccess)
    return ZF_ERR_CUDA;
  attn_kernel<kCompressed><<<p.grid, kAttnThreads, p.smem, s>>>(a);
  if (cudaGetLastError() != cudaSuccess) return ZF_ERR_CUDA;

  MergeArgs m{};
  m.seq_lens = seq_lens;
  m.part_o = a.part_o;
  m.part_lse = a.part_lse;
  m.out = out;
  m.lse = lse;
  m.batch = batch;
  m.hq = hq;
  m.page_size = c->page_size;
  m.max_pages = max_pages;
  m.chunk_pages = p.chunk_pages;
  m.max_chunks = p.max_chunks;
  const int rows = batch * hq;
  merge_kernel<<<(rows + 3) / 4, 128, 0, s>>>(m);
  return cudaGetLastError() == cudaSuccess ? ZF_OK : ZF_ERR_CUDA;
}

}  // namespace zf

using namespace zf;

extern "C" size_t zf_decode_attn_workspace_size(int32_t batch, int32_t num_q_heads, int32_t num_kv_heads,
                                                int32_t page_size, int32_t max_pages_per_req) {
  if (!attn_shape_ok(batch, num_q_heads, num_kv_heads, max_pages_per_req)) return 0;
  if (page_size < ZF_BLOCK_TOKENS || page_size % ZF_BLOCK_TOKENS || page_size > ZF_MAX_PAGE_SIZE) return 0;
  int sms = 0;
  if (current_sm_count(&sms) != ZF_OK) return 0;
  const Plan p = make_plan(batch, num_q_heads, num_kv_heads, page_size, max_pages_per_req, sms);
  return p.ws_bytes > 0 ? p.ws_bytes : 256;
}

extern "C" zf_status zf_decode_attn(const zf_cache* cache, const uint16_t* q, int32_t batch, int32_t num_q_heads,
                                    const int32_t* page_table, int32_t max_pages_per_req, const int32_t* seq_lens,
                                    float softmax_scale, float* out, float* lse, void* workspace,
                                    size_t workspace_bytes, void* stream) {
  return launch_attention<true>(cache, q, batch, num_q_heads, page_table, max_pages_per_req, seq_lens, softmax_scale,
                                out, lse, workspace, workspace_bytes, stream);
}

extern "C" zf_status zf_dense_decode_attn(const zf_cache* cache, const uint16_t* q, int32_t batch,
                                          int32_t num_q_heads, const int32_t* page_table, int32_t max_pages_per_req,
                                          const int32_t* seq_lens, float softmax_scale, float* out, float* lse,
                                          void* workspace, size_t workspace_bytes, void* stream) {
  return launch_attention<false>(cache, q, batch, num_q_heads, page_table, max_pages_per_req, seq_lens,
                                 softmax_scale, out, lse, workspace, workspace_bytes, stream);
}

// ---------------------------------------------------------------------------------------------
// zf_decode_attn_static: the same attention for callers that cannot allocate device memory.
// Its split-KV scratch is this file-scope device array (held by every GPU that loads the library
// until exit).  Host code must not pass `g_static_workspace` itself to a kernel: on the host the
// name is only a stand-in, so the device address is looked up once per device below.
static __device__ __align__(256) unsigned char g_static_workspace[ZF_STATIC_WORKSPACE_BYTES];

namespace {
constexpr int kStaticMaxDevices = 64;
std::mutex g_static_mutex;
void* g_static_address[kStaticMaxDevices] = {};

// Address of g_static_workspace on the current device (looked up on the first call per device).
zf_status static_workspace_address(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return ZF_ERR_CUDA;
  if (dev < 0 || dev >= kStaticMaxDevices) return ZF_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_static_mutex);
  if (!g_static_address[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_static_workspace) != cudaSuccess || !p) return ZF_ERR_CUDA;
    g_static_address[dev] = p;
  }
  *out = g_static_address[dev];
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
  const Plan p = make_plan(batch, num_q_heads, cache->num_kv_heads, P, max_pages_per_req, sms);
  if (p.ws_bytes > ZF_STATIC_WORKSPACE_BYTES) return ZF_ERR_STATIC_WORKSPACE_EXCEEDED;
  void* ws = nullptr;
  if ((st = static_workspace_address(&ws)) != ZF_OK) return st;
  return launch_attention<true>(cache, q, batch, num_q_heads, page_table, max_pages_per_req, seq_lens,
                                softmax_scale, out, lse, ws, ZF_STATIC_WORKSPACE_BYTES, stream);
}
