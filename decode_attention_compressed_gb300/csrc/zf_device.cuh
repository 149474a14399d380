// Device-side building blocks shared by the libzf kernels (sm_103a): PTX wrappers for mbarriers,
// 1-D bulk (TMA) copies, the warp MMA and matrix transpose, the block storage order, and the
// in-register rebuild of BF16 values from a compressed block.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/zf.h"

namespace zf {

constexpr int kSlotBytes = ZF_SLOT_BYTES;        // 784
constexpr int kRawBlockBytes = ZF_RAW_BLOCK_BYTES;
constexpr int kHeaderAt = 768;
constexpr int kEscapesAt = 772;
constexpr uint32_t kHeaderEscMask = 0x700u;    // header bits 8-10: number of escapes
constexpr uint64_t kWaitTimeoutNs = 2000000000ull;  // a pipeline wait gives up after 2 s

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t global_timer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// ------------------------------------------------------------------------------------ mbarrier
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.release.cta.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)),
               "r"(bytes)
               : "memory");
}

// try_wait blocks for a system-dependent time before it returns false, so a waiting warp spends
// few issue slots polling.
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t done;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(done)
      : "r"(smem_addr(bar)), "r"(parity)
      : "memory");
  return done != 0;
}

// Non-blocking test of the same condition.
__device__ __forceinline__ bool mbar_test(uint64_t* bar, uint32_t parity) {
  uint32_t done;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.test_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(done)
      : "r"(smem_addr(bar)), "r"(parity)
      : "memory");
  return done != 0;
}

// Wait for the phase with the given parity to complete.  Bounded: returns false after
// kWaitTimeoutNs (checked at every retry), so a broken pipeline never hangs the GPU.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, uint64_t limit_ns = kWaitTimeoutNs) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  for (uint32_t i = 1; i < (1u << 30); ++i) {
    if (mbar_try_wait(bar, parity)) return true;
    if (global_timer_ns() - t0 > limit_ns) return false;
  }
  return false;
}

// Sleep for about `ns` nanoseconds (bounded by the argument itself).
__device__ __forceinline__ void sleep_for_ns(uint64_t ns) {
  const uint64_t t0 = global_timer_ns();
  while (global_timer_ns() - t0 < ns) __nanosleep(1000);
}

// Programmatic dependent launch: wait for the preceding grid's results / let the next grid start.
__device__ __forceinline__ void wait_prior_grid() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void allow_next_grid() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// ------------------------------------------------------------------------------- bulk copies
__device__ __forceinline__ uint64_t l2_evict_first_policy() {
  uint64_t policy;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(policy));
  return policy;
}

// Hint: bring the 128-byte line holding `p` into L2 (no value is read; safe on any valid address).
__device__ __forceinline__ void prefetch_l2(const void* p) {
  asm volatile("prefetch.global.L2 [%0];" ::"l"(p));
}

// Hint: bring `bytes` (a multiple of 16, `src` 16-byte aligned) starting at `src` into L2.
__device__ __forceinline__ void bulk_prefetch_l2(const void* src, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src), "r"(bytes) : "memory");
}

// Relaxed (atomic, unordered) 32-bit load: a well-defined read of a value another grid may be
// writing at the same time.
__device__ __forceinline__ int ld_relaxed(const int32_t* p) {
  int v;
  asm volatile("ld.relaxed.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

// 1-D bulk copy global -> shared, completion signalled on `bar` as transaction bytes.
// dst, src and bytes must be multiples of 16.
__device__ __forceinline__ void bulk_copy_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar,
                                              uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;" ::"r"(
          smem_addr(dst)),
      "l"(src), "r"(bytes), "r"(smem_addr(bar)), "l"(policy)
      : "memory");
}

// ------------------------------------------------------------------------------- warp MMA
// D (16x8 fp32) += A (16x16 bf16, row) * B (16x8 bf16, col).
__device__ __forceinline__ void mma_bf16(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// Transpose of an 8x8 16-bit matrix held one row pair per lane (lane l: row l/4, cols 2(l%4)..+1).
__device__ __forceinline__ uint32_t transpose8x8(uint32_t x) {
  uint32_t y;
  asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(y) : "r"(x));
  return y;
}

// Four 8x8 16-bit matrices from shared memory, lane l supplying the address of row l % 8 of
// matrix l / 8; lane l receives elements (l / 4, 2(l % 4) .. +1) of each matrix (transposed with
// .trans), one 32-bit register per matrix.
__device__ __forceinline__ void ldmatrix_x4(const void* row, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                            uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(smem_addr(row))
               : "memory");
}
__device__ __forceinline__ void ldmatrix_x4_trans(const void* row, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                                  uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(smem_addr(row))
               : "memory");
}

// 2^x with the hardware approximation (PTX ex2.approx.ftz.f32); ex2(-inf) = 0.
__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// log2(x) with the hardware approximation (PTX lg2.approx.ftz.f32).
__device__ __forceinline__ float fast_log2(float x) {
  float y;
  asm("lg2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Round two floats to BF16 (nearest even) and pack: `lo` in bits 0-15, `hi` in bits 16-31.
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}
__device__ __forceinline__ float bf16lo_to_f32(uint32_t x) { return __uint_as_float(x << 16); }
__device__ __forceinline__ float bf16hi_to_f32(uint32_t x) { return __uint_as_float(x & 0xFFFF0000u); }

// ------------------------------------------------------------------- 5th-generation tensor cores
// tcgen05 MMA with operands in shared memory and the accumulator in tensor memory (TMEM; 128 lanes
// x 512 32-bit columns per SM; address = lane << 16 | column).

// Shared-memory operand descriptor, K-major without swizzle: 8-row x 16-byte core matrices of
// 128 contiguous bytes, adjacent along K at 128 bytes (leading byte offset) and along M/N at
// 2048 bytes (stride byte offset: one row of 16 core matrices = 128 K-elements of 16 bits);
// bits 46-47 hold the descriptor version 1.
__device__ __forceinline__ uint64_t umma_desc_kmajor(const void* p) {
  return static_cast<uint64_t>((smem_addr(p) & 0x3FFFFu) >> 4) | (static_cast<uint64_t>(128 >> 4) << 16) |
         (static_cast<uint64_t>(2048 >> 4) << 32) | (1ull << 46);
}

// Instruction descriptor of kind::f16: FP32 accumulator (bits 4-5 = 1), BF16 A and B (bits 7-9 and
// 10-12 = 1), both K-major (bits 15, 16 = 0), N >> 3 in bits 17-22, M >> 4 in bits 24-28.
__host__ __device__ constexpr uint32_t umma_idesc_bf16(int m, int n) {
  return (1u << 4) | (1u << 7) | (1u << 10) | (static_cast<uint32_t>(n >> 3) << 17) |
         (static_cast<uint32_t>(m >> 4) << 24);
}

// D (TMEM) = A (smem) * B^T (smem) + (accumulate ? D : 0), issued by one thread.
__device__ __forceinline__ void umma_bf16(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                          uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// D (TMEM) = A (TMEM) * B^T (smem) + (accumulate ? D : 0), issued by one thread.
__device__ __forceinline__ void umma_bf16_ta(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc,
                                             uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Arrive once on `bar` when every tcgen05.mma this thread issued before has completed.
__device__ __forceinline__ void umma_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_addr(bar))
               : "memory");
}

// Whole-warp TMEM allocation of `cols` columns (a power of two >= 32); the base address is
// written to `slot` in shared memory.
__device__ __forceinline__ void tmem_alloc(uint32_t* slot, uint32_t cols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_addr(slot)), "r"(cols)
               : "memory");
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t base, uint32_t cols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(base), "r"(cols) : "memory");
}
__device__ __forceinline__ void tcgen05_before_sync() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tcgen05_after_sync() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tmem_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }
__device__ __forceinline__ void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }
// Generic-proxy shared-memory writes become visible to the tensor cores (async proxy).
__device__ __forceinline__ void fence_proxy_async_smem() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

// 16 TMEM lanes x 8 columns per repeat, in the m16n8 accumulator layout: thread t gets rows
// t/4 and t/4 + 8, columns 2(t%4) and +1 of each 8-column block (registers 4j .. 4j+3).
__device__ __forceinline__ void tmem_ld_16x256b_x2(uint32_t taddr, uint32_t (&r)[8]) {
  asm volatile("tcgen05.ld.sync.aligned.16x256b.x2.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7])
               : "r"(taddr));
}
__device__ __forceinline__ void tmem_ld_16x256b_x4(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.16x256b.x4.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
        "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
}
// Store in the same 16x256b layout, two 8-column repeats.
__device__ __forceinline__ void tmem_st_16x256b_x2(uint32_t taddr, const uint32_t (&r)[8]) {
  asm volatile("tcgen05.st.sync.aligned.16x256b.x2.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"r"(taddr), "r"(r[0]),
               "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7])
               : "memory");
}
// 32 TMEM lanes (thread t: lane t), 16 consecutive columns.
__device__ __forceinline__ void tmem_ld_32x32b_x16(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
        "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
}
__device__ __forceinline__ void tmem_ld_32x32b_x8(uint32_t taddr, uint32_t (&r)[8]) {
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7])
               : "r"(taddr));
}
__device__ __forceinline__ void tmem_st_32x32b_x16(uint32_t taddr, const uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(
          taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]), "r"(r[9]),
      "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
      : "memory");
}

// ------------------------------------------------------------------------- block storage order
// Storage position of natural (token tau, channel gamma) of a 16x32 block.  The block is stored
// in the register order of the m16n8k16 A operand: lane = 4*groupID + threadID_in_group holds
// rows groupID (+8) and columns 2*threadID_in_group (+1, +8, +9) of each 16x16 half.
__host__ __device__ __forceinline__ int block_position(bool is_value, int tau, int gamma) {
  const int half = gamma >> 4;
  const int row = is_value ? (gamma & 15) : tau;
  const int col = is_value ? tau : (gamma & 15);
  const int lane = 4 * (row & 7) + ((col & 7) >> 1);
  const int r = 4 * (col >> 3) + 2 * (row >> 3) + (col & 1);
  return 16 * lane + 8 * half + r;
}

// ------------------------------------------------------------------------- in-register rebuild
// High bytes of a lane's 16 values from its two code words (byte k of a word = code k | code k+4
// << 4).  A code is sign << 3 | exponent offset; the high byte of a value is sign << 7 |
// (base/2 + offset).  `base4` holds base/2 in every byte: base/2 + offset is the 7-bit exponent>>1
// field, so one 32-bit add fills four high bytes without any carry crossing a byte.
// Output: word w holds the high bytes of values 4w..4w+3, one per byte.
__device__ __forceinline__ void high_bytes(uint2 code, uint32_t base4, uint32_t (&h)[4]) {
  // values 0..3 of a word (low nibbles): offset bits 0-2 stay, sign bit 3 moves to bit 7;
  // values 4..7 (high nibbles): offset bits 4-6 move to bits 0-2, sign bit 7 stays.
  h[0] = base4 + (code.x & 0x07070707u) + ((code.x & 0x08080808u) << 4);
  h[1] = base4 + ((code.x >> 4) & 0x07070707u) + (code.x & 0x80808080u);
  h[2] = base4 + (code.y & 0x07070707u) + ((code.y & 0x08080808u) << 4);
  h[3] = base4 + ((code.y >> 4) & 0x07070707u) + (code.y & 0x80808080u);
}

// Interleave low and high bytes into four BF16 pairs per 8 values: value 2i in the low half of
// a[i].
__device__ __forceinline__ void interleave(uint4 lo, const uint32_t (&h)[4], uint32_t (&a)[8]) {
  a[0] = __byte_perm(lo.x, h[0], 0x5140);
  a[1] = __byte_perm(lo.x, h[0], 0x7362);
  a[2] = __byte_perm(lo.y, h[1], 0x5140);
  a[3] = __byte_perm(lo.y, h[1], 0x7362);
  a[4] = __byte_perm(lo.z, h[2], 0x5140);
  a[5] = __byte_perm(lo.z, h[2], 0x7362);
  a[6] = __byte_perm(lo.w, h[3], 0x5140);
  a[7] = __byte_perm(lo.w, h[3], 0x7362);
}

// Replace the exponent>>1 field of the escaped values this lane owns (positions 16*lane..+15).
// `tail` is the block's last 16 bytes: the header word, then the six escape entries
// (position << 7 | exponent >> 1).  Entry position p is value p & 15 of lane p >> 4, whose high
// byte is byte p & 3 of h[(p >> 2) & 3].
__device__ __forceinline__ void patch_escapes(uint4 tail, uint32_t n_esc, int lane, uint32_t (&h)[4]) {
  for (uint32_t e = 0; e < n_esc; ++e) {
    const uint32_t pair = e < 2 ? tail.y : (e < 4 ? tail.z : tail.w);
    const uint32_t entry = (e & 1u) ? pair >> 16 : pair & 0xFFFFu;
    const uint32_t p = entry >> 7;
    // branch-free: lanes that do not own the value apply an empty mask
    const uint32_t sh = (p & 3u) * 8u, w = (p >> 2) & 3u;
    const uint32_t mask = (p >> 4) == static_cast<uint32_t>(lane) ? 0x7Fu << sh : 0u;
    const uint32_t val = ((entry & 0x7Fu) << sh) & mask;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const uint32_t mi = w == static_cast<uint32_t>(i) ? mask : 0u;
      h[i] = (h[i] & ~mi) | (val & mi);
    }
  }
}

// This lane's 16 values of a compressed block that has no escapes; base4 = header byte 0 (base/2)
// in every byte.
__device__ __forceinline__ void rebuild_lane_noesc(const uint8_t* slot, int lane, uint32_t base4,
                                                   uint32_t (&a)[8]) {
  const uint4 lo = *reinterpret_cast<const uint4*>(slot + 16 * lane);
  const uint2 code = *reinterpret_cast<const uint2*>(slot + 512 + 8 * lane);
  uint32_t h[4];
  high_bytes(code, base4, h);
  interleave(lo, h, a);
}

// This lane's 16 values (storage positions 16*lane..16*lane+15) of a compressed block in
// shared or global memory.  The header and the escape entries come in one 16-byte load.
__device__ __forceinline__ void rebuild_lane(const uint8_t* slot, int lane, uint32_t (&a)[8]) {
  const uint4 tail = *reinterpret_cast<const uint4*>(slot + kHeaderAt);
  const uint4 lo = *reinterpret_cast<const uint4*>(slot + 16 * lane);
  const uint2 code = *reinterpret_cast<const uint2*>(slot + 512 + 8 * lane);
  const uint32_t base4 = __byte_perm(tail.x, 0u, 0x0000u);   // header byte 0 = base/2 (bit 7 clear)
  uint32_t h[4];
  high_bytes(code, base4, h);
  const uint32_t n_esc = (tail.x >> 8) & 7u;
  if (n_esc) patch_escapes(tail, n_esc, lane, h);
  interleave(lo, h, a);
}

// This lane's 16 values of a raw block.  Raw blocks are half-major (position 256*half + 8*lane + r
// holds storage position 16*lane + 8*half + r), so each 16-byte read of a warp is conflict-free.
__device__ __forceinline__ void load_raw_lane(const uint8_t* block, int lane, uint32_t (&a)[8]) {
  const uint4 x = *reinterpret_cast<const uint4*>(block + 16 * lane);
  const uint4 y = *reinterpret_cast<const uint4*>(block + 512 + 16 * lane);
  a[0] = x.x; a[1] = x.y; a[2] = x.z; a[3] = x.w;
  a[4] = y.x; a[5] = y.y; a[6] = y.z; a[7] = y.w;
}

__device__ __forceinline__ void report(int32_t* status, int32_t bits) {
  if (status) atomicOr(status, bits);
}

}  // namespace zf
