// zf_encode_pages, zf_append_tokens, zf_decompress and zf_validate_pages: page compression,
// token appends into uncompressed pages, the bit-exact inverse, and a check of stored metadata.
//
// ZipFusion §III.B (Lossless KV Cache Format, Fig. 2): a block is compressed when its exponents
// fit [b, b+15], b = minimum exponent rounded down to even; each value keeps its low byte and a
// 4-bit code (sign, exponent offset).  This format adds up to six escapes for blocks whose range
// is wider (window anchored at the maximum exponent).  ZipFusion §III.D: partial pages stay raw;
// full pages are compressed under their page id.
//
// One CTA encodes one (page, kv head): each warp classifies and encodes whole blocks straight into
// the page's compressed slot (coalesced 16-byte stores); a page head with a block that cannot be
// compressed is then written to its raw slot instead.
#include <cuda_runtime.h>
#include <stdint.h>

#include "zf_device.cuh"
#include "zf_host.h"

namespace zf {

constexpr int kCodecWarps = 8;
constexpr int kCodecThreads = kCodecWarps * 32;
static_assert(kCodecThreads == 2 * ZF_HEAD_DIM, "append_kernel: one thread per K and per V channel");

struct CodecArgs {
  uint8_t* k_comp;
  uint8_t* v_comp;
  uint16_t* k_raw;
  uint16_t* v_raw;
  int32_t* dir;
  int32_t* status;
  const uint16_t* src_k;   // encode: source pages; decompress: unused
  const uint16_t* src_v;
  uint16_t* dst_k;         // decompress: destination pages
  uint16_t* dst_v;
  const int32_t* page_ids;
  const int32_t* n_valid;
  const int32_t* raw_slots;
  const int32_t* positions;  // append: token index within the page
  int32_t num_pages, hkv, page_size, num_raw, flags;
  int32_t raw_out;         // decompress: 1 = write the raw block layout of a dense cache
};

// Natural-layout address of this lane's 16 values of block (tile, group): token tau = lane/2,
// channels 32*group + 16*(lane%2) .. +15 of a [P][128] page head.
__device__ __forceinline__ size_t natural_offset(int tile, int group, int lane) {
  return static_cast<size_t>(16 * tile + (lane >> 1)) * ZF_HEAD_DIM + 32 * group + 16 * (lane & 1);
}

struct uint4x2 {
  uint4 a, b;
};

// One warp encodes one block.  u: this lane's 16 values at storage positions 16*lane .. +15
// (two per word, low half first).  Writes the 784-byte slot, or sets *fail when the block needs
// more than ZF_MAX_ESCAPES escapes.  Base: the minimum exponent rounded down to even when every
// exponent fits [base, base+15], else the smallest even base whose window reaches the maximum
// exponent, values below it becoming escapes.
//
// Four values per 32-bit operation: with h = sign << 7 | exponent >> 1 (a value's high byte) and
// eh = h & 0x7F, the rule reads base/2 = min eh when max eh <= min eh + 7, else max eh - 7; a value
// is an escape when eh < base/2, and its code is sign << 3 | (eh - base/2) (offset 0 for escapes).
__device__ __forceinline__ uint32_t byte_signs(uint32_t x) {
  uint32_t r;       // prmt with the sign-replicate selector bit: byte i = 0xFF if bit 7 of byte i is set
  asm("prmt.b32 %0, %1, 0, 0xBA98;" : "=r"(r) : "r"(x));
  return r;
}

__device__ __forceinline__ void encode_block_lane(const uint32_t (&u)[8], uint8_t* slot, int lane, int* fail) {
  uint32_t eh[4], lo4[4];
#pragma unroll
  for (int k = 0; k < 4; ++k) {            // values 4k .. 4k+3: word 2k holds 4k, 4k+1
    eh[k] = __byte_perm(u[2 * k], u[2 * k + 1], 0x7531);    // high bytes
    lo4[k] = __byte_perm(u[2 * k], u[2 * k + 1], 0x6420);   // low bytes, stored as they are
  }
  // min and max of the 16 exponent>>1 fields, two per 16-bit lane
  uint32_t f[8];
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    f[2 * k] = eh[k] & 0x007F007Fu;
    f[2 * k + 1] = (eh[k] >> 8) & 0x007F007Fu;
  }
  uint32_t mn = __vimin3_u16x2(__vimin3_u16x2(f[0], f[1], f[2]), __vimin3_u16x2(f[3], f[4], f[5]),
                               __vimin3_u16x2(f[6], f[7], f[7]));
  uint32_t mx = __vimax3_u16x2(__vimax3_u16x2(f[0], f[1], f[2]), __vimax3_u16x2(f[3], f[4], f[5]),
                               __vimax3_u16x2(f[6], f[7], f[7]));
  mn = __reduce_min_sync(0xFFFFFFFFu, min(mn & 0xFFFFu, mn >> 16));
  mx = __reduce_max_sync(0xFFFFFFFFu, max(mx & 0xFFFFu, mx >> 16));
  const uint32_t half_base = mx > mn + 7 ? mx - 7 : mn;
  const uint32_t hb4 = half_base * 0x01010101u;
  // per byte: d = 0x80 + eh - base/2 (no borrow crosses a byte: eh, base/2 <= 127), bit 7 set
  // exactly when the value is not an escape
  uint32_t code[4], esc[4], cnt = 0;
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const uint32_t d = (eh[k] | 0x80808080u) - hb4;
    const uint32_t keep = byte_signs(d);                        // 0xFF per non-escape byte
    esc[k] = ~d & 0x80808080u;
    code[k] = (d & keep & 0x07070707u) | ((eh[k] >> 4) & 0x08080808u);
    cnt += __popc(esc[k]);
  }
  const uint32_t total = __reduce_add_sync(0xFFFFFFFFu, cnt);
  if (total > ZF_MAX_ESCAPES) {
    if (lane == 0) atomicOr(fail, 1);
    return;
  }
  *reinterpret_cast<uint4*>(slot + 16 * lane) = make_uint4(lo4[0], lo4[1], lo4[2], lo4[3]);
  // byte m of a code word = code of value m | code of value m + 4 << 4
  *reinterpret_cast<uint2*>(slot + 512 + 8 * lane) = make_uint2(code[0] | code[1] << 4, code[2] | code[3] << 4);
  uint16_t* escs = reinterpret_cast<uint16_t*>(slot + kEscapesAt);
  if (lane < ZF_MAX_ESCAPES && static_cast<uint32_t>(lane) >= total) escs[lane] = 0;
  if (total > 0) {
    uint32_t before = cnt;                   // inclusive scan over lanes, then exclusive
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
      const uint32_t t = __shfl_up_sync(0xFFFFFFFFu, before, d);
      if (lane >= d) before += t;
    }
    uint32_t k = before - cnt;
#pragma unroll
    for (int j = 0; j < 16; ++j) {
      if (esc[j >> 2] & (0x80u << (8 * (j & 3)))) {     // entry: position << 7 | exponent >> 1
        escs[k++] = static_cast<uint16_t>(((16 * lane + j) << 7) | ((eh[j >> 2] >> (8 * (j & 3))) & 0x7Fu));
      }
    }
  }
  if (lane == 0)
    *reinterpret_cast<uint32_t*>(slot + kHeaderAt) =
        half_base | (total << 8) | (static_cast<uint32_t>(ZF_FORMAT_VERSION) << 24);
}

// This lane's 16 source values of block `bi` (tile bi/4, channel group bi%4) of a [P][128] page
// head in natural layout: token lane/2, channels 16*(lane%2) .. +15 of the group.
__device__ __forceinline__ uint4x2 load_block_lane(const uint16_t* src_head, int bi, int lane) {
  const uint16_t* p = src_head + natural_offset(bi >> 2, bi & 3, lane);
  uint4x2 x;
  x.a = *reinterpret_cast<const uint4*>(p);
  x.b = *reinterpret_cast<const uint4*>(p + 8);
  return x;
}

// Rows of a warp's staging block: 16 tokens x 32 channels, rows padded to 80 bytes so that the
// eight 16-byte rows one ldmatrix phase reads fall in distinct banks.
constexpr int kStageRowBytes = 80;
constexpr int kStageBytes = 16 * kStageRowBytes;

// A lane's natural-layout values -> the warp's stage -> the lane's own 16 storage positions
// (16*lane .. +15, two per word).  The storage order is the m16n8k16 A-operand register order of
// each 16x16 half, so ldmatrix delivers it: for keys the A operand is the block itself (rows
// tokens), for values its transpose (rows channels), read with .trans.
__device__ __forceinline__ void to_storage_order(const uint4x2& x, bool is_value, uint8_t* stage, int lane,
                                                 uint32_t (&u)[8]) {
  uint8_t* row = stage + (lane >> 1) * kStageRowBytes + 32 * (lane & 1);
  *reinterpret_cast<uint4*>(row) = x.a;
  *reinterpret_cast<uint4*>(row + 16) = x.b;
  __syncwarp();
  // matrix q = lane / 8 of the four, row lane % 8 of it.  Keys: q selects (tokens +8 for q odd,
  // channels +8 for q >= 2); values: (channels +8 for q odd, tokens +8 for q >= 2).
  const int q = lane >> 3, r = lane & 7;
  const int tok = r + 8 * (is_value ? (q >> 1) : (q & 1));
  const int ch = 8 * (is_value ? (q & 1) : (q >> 1));
#pragma unroll
  for (int half = 0; half < 2; ++half) {
    const uint8_t* p = stage + tok * kStageRowBytes + 2 * (16 * half + ch);
    if (is_value) ldmatrix_x4_trans(p, u[4 * half], u[4 * half + 1], u[4 * half + 2], u[4 * half + 3]);
    else ldmatrix_x4(p, u[4 * half], u[4 * half + 1], u[4 * half + 2], u[4 * half + 3]);
  }
  __syncwarp();                                  // the stage is rewritten by the next block
}

// One CTA per (page, kv head) with W warps: warp w takes blocks w, w + W, ... of the page head's K
// blocks then V blocks, kEncodeBatch at a time.  The source address does not depend on the
// page id, so the first batch of loads is issued before the page id and fill count are read.  A
// full page is encoded straight into its compressed slot; if any block needs more than
// ZF_MAX_ESCAPES escapes, the page head is then written raw instead (the compressed slot's
// contents are unused while the directory names the raw slot).  Partial and forced-raw pages go
// to the raw slot directly.  Launched with programmatic stream serialisation: it waits for the
// preceding grid before reading anything, and lets the next grid launch at once.
// Two blocks in flight per warp and 8 warps per CTA (measured on GB300 against 2, 4 and 16
// warps, and against loading the next pair while encoding this one: 8 warps without that was
// fastest); at most 64 registers so that four CTAs fit an SM.
constexpr int kEncodeBatch = 2;
constexpr int kEncodeWarps = 8;
__global__ void __launch_bounds__(kEncodeWarps * 32, 4) encode_kernel(CodecArgs a) {
  __shared__ __align__(16) uint8_t stage[kEncodeWarps][kStageBytes];
  __shared__ int fail;
  wait_prior_grid();
  allow_next_grid();
  const int P = a.page_size;
  const int nblk = P / 4;                    // blocks per K (or V) page head
  const int nb = 2 * nblk;
  const int i = blockIdx.x, h = blockIdx.y;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  constexpr int kStep = kEncodeWarps * kEncodeBatch;
  const size_t head_elems = static_cast<size_t>(P) * ZF_HEAD_DIM;
  const uint16_t* src_k = a.src_k + (static_cast<size_t>(i) * a.hkv + h) * head_elems;
  const uint16_t* src_v = a.src_v + (static_cast<size_t>(i) * a.hkv + h) * head_elems;
  uint4x2 x[kEncodeBatch];
  auto load = [&](int b0) {
#pragma unroll
    for (int k = 0; k < kEncodeBatch; ++k) {
      const int blk = b0 + k * kEncodeWarps;
      if (blk < nb) x[k] = load_block_lane(blk >= nblk ? src_v : src_k, blk >= nblk ? blk - nblk : blk, lane);
    }
  };
  // walk the warp's blocks a batch at a time: fn(block, values) for each; batch 0 is already in x
  auto walk = [&](auto&& fn) {
    for (int b0 = warp; b0 < nb; b0 += kStep) {
      if (b0 != warp) load(b0);
#pragma unroll
      for (int k = 0; k < kEncodeBatch; ++k) {
        const int blk = b0 + k * kEncodeWarps;
        if (blk < nb) fn(blk, x[k]);
      }
    }
  };
  load(warp);
  if (threadIdx.x == 0) fail = 0;
  const int pid = a.page_ids[i];
  const int nv = a.n_valid[i];
  if (pid < 0 || pid >= a.num_pages) {
    if (threadIdx.x == 0) report(a.status, ZF_DEV_BAD_PAGE_ID);
    return;
  }
  const size_t dir_at = static_cast<size_t>(pid) * a.hkv + h;
  if (nv < 0 || nv > P) {
    if (threadIdx.x == 0) {
      report(a.status, ZF_DEV_BAD_N_VALID);
      a.dir[dir_at] = ZF_DIR_INVALID;
    }
    return;
  }
  uint8_t* my_stage = stage[warp];
  __syncthreads();                           // `fail` is initialised
  if (!((a.flags & ZF_ENCODE_FORCE_RAW) || nv < P)) {
    const size_t rec = static_cast<size_t>(nblk) * kSlotBytes;     // bytes per K (or V) record
    uint8_t* dk = a.k_comp + dir_at * rec;
    uint8_t* dv = a.v_comp + dir_at * rec;
    walk([&](int blk, const uint4x2& v) {
      const bool is_value = blk >= nblk;
      const int bi = is_value ? blk - nblk : blk;
      uint32_t u[8];
      to_storage_order(v, is_value, my_stage, lane, u);
      encode_block_lane(u, (is_value ? dv : dk) + static_cast<size_t>(bi) * kSlotBytes, lane, &fail);
    });
    __syncthreads();
    if (!fail) {
      if (threadIdx.x == 0) a.dir[dir_at] = ZF_DIR_COMPRESSED;
      return;
    }
    load(warp);                              // a block overflowed its escapes: the page head goes raw
  }
  const int rs = a.raw_slots ? a.raw_slots[i] : -1;
  if (rs < 0 || rs >= a.num_raw) {
    if (threadIdx.x == 0) {
      a.dir[dir_at] = ZF_DIR_INVALID;
      report(a.status, ZF_DEV_BAD_RAW_SLOT);
    }
    return;
  }
  const size_t rrec = static_cast<size_t>(nblk) * 512;             // uint16 per K (or V) record
  uint16_t* rk = a.k_raw + (static_cast<size_t>(rs) * a.hkv + h) * rrec;
  uint16_t* rv = a.v_raw + (static_cast<size_t>(rs) * a.hkv + h) * rrec;
  walk([&](int blk, const uint4x2& v) {
    const bool is_value = blk >= nblk;
    const int bi = is_value ? blk - nblk : blk;
    uint32_t u[8];
    to_storage_order(v, is_value, my_stage, lane, u);
    // raw blocks are half-major: the lane's storage positions 16*lane + 8*half + r sit at
    // 256*half + 8*lane + r
    uint8_t* dst = reinterpret_cast<uint8_t*>((is_value ? rv : rk) + static_cast<size_t>(bi) * 512);
    *reinterpret_cast<uint4*>(dst + 16 * lane) = make_uint4(u[0], u[1], u[2], u[3]);
    *reinterpret_cast<uint4*>(dst + 512 + 16 * lane) = make_uint4(u[4], u[5], u[6], u[7]);
  });
  if (threadIdx.x == 0) a.dir[dir_at] = rs;
}

// Raw record index of storage position e of a block: 16-byte group 2*lane + half of the storage
// order sits at group 32*half + lane of a raw block (the layout load_raw_lane reads).
__device__ __forceinline__ int raw_position(int e) { return ((e >> 3) & 1) * 256 + (e >> 4) * 8 + (e & 7); }

// One CTA appends one token to one (page, kv head) in its raw slot (ZipFusion §III.D: a page that
// is still filling stays uncompressed, so a decode step writes its token in place).  Threads
// 0-127 write the K channels, 128-255 the V channels, each to its block's raw position.  The
// token that fills the page (position P-1) is followed by the page head's compression from the
// slot: every warp encodes blocks from the raw record (a lane's 16 storage-order values are its
// two 16-byte groups there), and the page goes to its compressed slot unless a block needs more
// than ZF_MAX_ESCAPES escapes, in which case it stays in the raw slot.
__global__ void __launch_bounds__(kCodecThreads) append_kernel(CodecArgs a) {
  extern __shared__ __align__(16) uint8_t smem[];
  const int P = a.page_size;
  const int nblk = P / 4;
  uint8_t* comp = smem;                      // [2*nblk][784]
  int* fail = reinterpret_cast<int*>(smem + 2 * nblk * kSlotBytes);
  const int i = blockIdx.x, h = blockIdx.y;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int pid = a.page_ids[i], pos = a.positions[i], rs = a.raw_slots[i];
  if (pid < 0 || pid >= a.num_pages) {
    if (threadIdx.x == 0) report(a.status, ZF_DEV_BAD_PAGE_ID);
    return;
  }
  const size_t dir_at = static_cast<size_t>(pid) * a.hkv + h;
  if (pos < 0 || pos >= P || rs < 0 || rs >= a.num_raw) {
    if (threadIdx.x == 0) {
      report(a.status, (pos < 0 || pos >= P) ? ZF_DEV_BAD_N_VALID : ZF_DEV_BAD_RAW_SLOT);
      a.dir[dir_at] = ZF_DIR_INVALID;
    }
    return;
  }
  const size_t rec = static_cast<size_t>(nblk) * 512;            // uint16 per K (or V) record
  uint16_t* rk = a.k_raw + (static_cast<size_t>(rs) * a.hkv + h) * rec;
  uint16_t* rv = a.v_raw + (static_cast<size_t>(rs) * a.hkv + h) * rec;
  {
    const bool is_value = threadIdx.x >= ZF_HEAD_DIM;
    const int c = threadIdx.x & (ZF_HEAD_DIM - 1);
    const int bi = (pos >> 4) * 4 + (c >> 5);
    const int at = bi * 512 + raw_position(block_position(is_value, pos & 15, c & 31));
    const size_t from = (static_cast<size_t>(i) * a.hkv + h) * ZF_HEAD_DIM + c;
    (is_value ? rv : rk)[at] = (is_value ? a.src_v : a.src_k)[from];
  }
  if (pos < P - 1) {
    if (threadIdx.x == 0) a.dir[dir_at] = rs;
    return;
  }
  if (threadIdx.x == 0) *fail = 0;
  __syncthreads();                           // the token is in the slot for every warp of the CTA
  for (int blk = warp; blk < 2 * nblk; blk += kCodecWarps) {
    const bool is_value = blk >= nblk;
    const int bi = is_value ? blk - nblk : blk;
    const uint4* src = reinterpret_cast<const uint4*>((is_value ? rv : rk) + static_cast<size_t>(bi) * 512);
    const uint4 y0 = src[lane], y1 = src[lane + 32];
    const uint32_t u[8] = {y0.x, y0.y, y0.z, y0.w, y1.x, y1.y, y1.z, y1.w};
    encode_block_lane(u, comp + blk * kSlotBytes, lane, fail);
  }
  __syncthreads();
  if (*fail) {
    if (threadIdx.x == 0) a.dir[dir_at] = rs;
    return;
  }
  const size_t crec = static_cast<size_t>(nblk) * kSlotBytes;
  uint8_t* dk = a.k_comp + (static_cast<size_t>(pid) * a.hkv + h) * crec;
  uint8_t* dv = a.v_comp + (static_cast<size_t>(pid) * a.hkv + h) * crec;
  const int n16 = static_cast<int>(crec / 16);
  for (int t = threadIdx.x; t < 2 * n16; t += kCodecThreads) {
    const uint4 val = reinterpret_cast<const uint4*>(comp)[t];
    if (t < n16) reinterpret_cast<uint4*>(dk)[t] = val;
    else reinterpret_cast<uint4*>(dv)[t - n16] = val;
  }
  if (threadIdx.x == 0) a.dir[dir_at] = ZF_DIR_COMPRESSED;
}

// Metadata check of one compressed slot (shared by the device validator and the host entry).
// The header word is b/2 (bits 0-6) | escape count (bits 8-10) | format version (bits 24-31);
// every other bit is zero, at most ZF_MAX_ESCAPES escapes are listed with strictly ascending
// positions, and unused entries are 0.
__host__ __device__ inline bool slot_header_ok(uint32_t header, const uint16_t (&esc)[ZF_MAX_ESCAPES]) {
  const uint32_t n_esc = (header >> 8) & 0x7u;
  if ((header >> 24) != ZF_FORMAT_VERSION || (header & 0x00FFF880u) != 0 || n_esc > ZF_MAX_ESCAPES)
    return false;
  int last = -1;
  for (int k = 0; k < ZF_MAX_ESCAPES; ++k) {
    if (static_cast<uint32_t>(k) < n_esc) {
      const int p = esc[k] >> 7;
      if (p <= last) return false;
      last = p;
    } else if (esc[k] != 0) {
      return false;
    }
  }
  return true;
}

// ... and every code's offset added to b/2 stays within 7 bits (the rebuild's additions carry
// into no sign bit, ZipFusion §III.C), which can only fail when b/2 > 120.
__host__ __device__ inline bool slot_ok(const uint8_t* slot) {
  uint32_t header = 0;
  for (int b = 0; b < 4; ++b) header |= static_cast<uint32_t>(slot[kHeaderAt + b]) << (8 * b);
  uint16_t esc[ZF_MAX_ESCAPES];
  for (int k = 0; k < ZF_MAX_ESCAPES; ++k)
    esc[k] = static_cast<uint16_t>(slot[kEscapesAt + 2 * k] | slot[kEscapesAt + 2 * k + 1] << 8);
  if (!slot_header_ok(header, esc)) return false;
  const uint32_t half_base = header & 0x7Fu;
  if (half_base > 120) {
    for (int j = 0; j < 256; ++j) {
      const uint32_t c = slot[512 + j];
      if (half_base + (c & 7u) > 127 || half_base + ((c >> 4) & 7u) > 127) return false;
    }
  }
  return true;
}

// One CTA per (page, kv head): thread t checks slot t of the page head's K and V records.
__global__ void __launch_bounds__(kCodecThreads) validate_kernel(CodecArgs a, int32_t* bad) {
  const int P = a.page_size;
  const int nblk = P / 4;
  const int i = blockIdx.x, h = blockIdx.y;
  const int pid = a.page_ids[i];
  if (pid < 0 || pid >= a.num_pages) {
    if (threadIdx.x == 0) {
      report(a.status, ZF_DEV_BAD_PAGE_ID);
      if (bad) bad[i] = 1;
    }
    return;
  }
  const int d = a.dir[static_cast<size_t>(pid) * a.hkv + h];
  if (d != ZF_DIR_COMPRESSED) {
    if (threadIdx.x == 0 && (d < 0 || d >= a.num_raw)) {
      report(a.status, ZF_DEV_BAD_DIR);
      if (bad) bad[i] = 1;
    }
    return;
  }
  for (int t = threadIdx.x; t < 2 * nblk; t += kCodecThreads) {
    const bool is_value = t >= nblk;
    const uint8_t* slot = (is_value ? a.v_comp : a.k_comp) +
                          ((static_cast<size_t>(pid) * a.hkv + h) * nblk + (is_value ? t - nblk : t)) * kSlotBytes;
    if (!slot_ok(slot)) {
      report(a.status, ZF_DEV_BAD_SLOT);
      if (bad) bad[i] = 1;
    }
  }
}

__global__ void __launch_bounds__(kCodecThreads) decompress_kernel(CodecArgs a) {
  __shared__ __align__(16) uint16_t stage[kCodecWarps][512];
  const int P = a.page_size;
  const int nblk = P / 4;
  const int i = blockIdx.x, h = blockIdx.y;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int pid = a.page_ids[i];
  int kind = 2;                         // 0 compressed, 1 raw, 2 invalid
  int slot = 0;
  if (pid >= 0 && pid < a.num_pages) {
    const int d = a.dir[static_cast<size_t>(pid) * a.hkv + h];
    if (d == ZF_DIR_COMPRESSED) {
      kind = 0;
      slot = pid;
    } else if (d >= 0 && d < a.num_raw) {
      kind = 1;
      slot = d;
    }
  }
  if (kind == 2 && threadIdx.x == 0)
    report(a.status, (pid >= 0 && pid < a.num_pages) ? ZF_DEV_BAD_DIR : ZF_DEV_BAD_PAGE_ID);

  const size_t head_elems = static_cast<size_t>(P) * ZF_HEAD_DIM;
  for (int blk = warp; blk < 2 * nblk; blk += kCodecWarps) {
    const bool is_value = blk >= nblk;
    const int bi = is_value ? blk - nblk : blk;
    const int tile = bi >> 2, group = bi & 3;
    uint32_t v[8] = {0, 0, 0, 0, 0, 0, 0, 0};
    if (kind == 0) {
      const uint8_t* base = (is_value ? a.v_comp : a.k_comp) +
                            (static_cast<size_t>(slot) * a.hkv + h) * nblk * kSlotBytes + static_cast<size_t>(bi) * kSlotBytes;
      rebuild_lane(base, lane, v);
    } else if (kind == 1) {
      const uint16_t* base = (is_value ? a.v_raw : a.k_raw) +
                             (static_cast<size_t>(slot) * a.hkv + h) * nblk * 512 + static_cast<size_t>(bi) * 512;
      load_raw_lane(reinterpret_cast<const uint8_t*>(base), lane, v);
    }
    if (a.raw_out) {                     // raw block layout: the inverse of load_raw_lane
      uint8_t* blk = reinterpret_cast<uint8_t*>(is_value ? a.dst_v : a.dst_k) +
                     ((static_cast<size_t>(i) * a.hkv + h) * nblk + bi) * kRawBlockBytes;
      *reinterpret_cast<uint4*>(blk + 16 * lane) = make_uint4(v[0], v[1], v[2], v[3]);
      *reinterpret_cast<uint4*>(blk + 512 + 16 * lane) = make_uint4(v[4], v[5], v[6], v[7]);
      continue;
    }
    uint16_t* st = stage[warp];
    *reinterpret_cast<uint4*>(st + 16 * lane) = make_uint4(v[0], v[1], v[2], v[3]);
    *reinterpret_cast<uint4*>(st + 16 * lane + 8) = make_uint4(v[4], v[5], v[6], v[7]);
    __syncwarp();
    const int tau = lane >> 1, g0 = 16 * (lane & 1);
    uint32_t o[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const uint32_t lo = st[block_position(is_value, tau, g0 + 2 * j)];
      const uint32_t hi = st[block_position(is_value, tau, g0 + 2 * j + 1)];
      o[j] = lo | hi << 16;
    }
    uint16_t* dst = (is_value ? a.dst_v : a.dst_k) + (static_cast<size_t>(i) * a.hkv + h) * head_elems +
                    natural_offset(tile, group, lane);
    *reinterpret_cast<uint4*>(dst) = make_uint4(o[0], o[1], o[2], o[3]);
    *reinterpret_cast<uint4*>(dst + 8) = make_uint4(o[4], o[5], o[6], o[7]);
    __syncwarp();
  }
}

}  // namespace zf

using namespace zf;

extern "C" zf_status zf_encode_pages(const zf_cache* cache, const uint16_t* src_k, const uint16_t* src_v,
                                     const int32_t* page_ids, const int32_t* n_valid, const int32_t* raw_slots,
                                     int32_t n, int32_t flags, void* stream) {
  if (flags & ~ZF_ENCODE_FORCE_RAW) return ZF_ERR_INVALID_ARGUMENT;
  // a forced-raw encode never writes the compressed pools, so they may be absent
  zf_status st = check_cache(cache, /*need_comp=*/!(flags & ZF_ENCODE_FORCE_RAW), /*need_raw=*/false, /*need_dir=*/true);
  if (st != ZF_OK) return st;
  if (n < 0) return ZF_ERR_INVALID_ARGUMENT;
  if (n == 0) return ZF_OK;
  if (!src_k || !src_v || !page_ids || !n_valid || !aligned16(src_k) || !aligned16(src_v))
    return ZF_ERR_INVALID_ARGUMENT;
  if (cache->num_raw_slots > 0 && (!cache->k_raw || !cache->v_raw || !aligned16(cache->k_raw) || !aligned16(cache->v_raw)))
    return ZF_ERR_INVALID_ARGUMENT;
  if (cache->num_kv_heads > 65535) return ZF_ERR_UNSUPPORTED;
  CodecArgs a{};
  a.k_comp = cache->k_comp; a.v_comp = cache->v_comp; a.k_raw = cache->k_raw; a.v_raw = cache->v_raw;
  a.dir = cache->dir; a.status = cache->status;
  a.src_k = src_k; a.src_v = src_v;
  a.page_ids = page_ids; a.n_valid = n_valid; a.raw_slots = raw_slots;
  a.num_pages = cache->num_pages; a.hkv = cache->num_kv_heads; a.page_size = cache->page_size;
  a.num_raw = cache->num_raw_slots; a.flags = flags;
  // programmatic stream serialisation: the grid may launch while its predecessor drains and waits
  // for it (griddepcontrol.wait) before reading anything
  cudaLaunchAttribute pdl[1];
  pdl[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  pdl[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(n, cache->num_kv_heads);
  cfg.blockDim = dim3(32 * kEncodeWarps);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = static_cast<cudaStream_t>(stream);
  cfg.attrs = pdl;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, encode_kernel, a) == cudaSuccess ? ZF_OK : ZF_ERR_CUDA;
}

extern "C" zf_status zf_append_tokens(const zf_cache* cache, const uint16_t* k_tok, const uint16_t* v_tok,
                                      const int32_t* page_ids, const int32_t* positions, const int32_t* raw_slots,
                                      int32_t n, void* stream) {
  zf_status st = check_cache(cache, /*need_comp=*/true, /*need_raw=*/true, /*need_dir=*/true);
  if (st != ZF_OK) return st;
  if (n < 0) return ZF_ERR_INVALID_ARGUMENT;
  if (n == 0) return ZF_OK;
  if (!k_tok || !v_tok || !page_ids || !positions || !raw_slots) return ZF_ERR_INVALID_ARGUMENT;
  if (cache->num_kv_heads > 65535) return ZF_ERR_UNSUPPORTED;
  CodecArgs a{};
  a.k_comp = cache->k_comp; a.v_comp = cache->v_comp; a.k_raw = cache->k_raw; a.v_raw = cache->v_raw;
  a.dir = cache->dir; a.status = cache->status;
  a.src_k = k_tok; a.src_v = v_tok;
  a.page_ids = page_ids; a.positions = positions; a.raw_slots = raw_slots;
  a.num_pages = cache->num_pages; a.hkv = cache->num_kv_heads; a.page_size = cache->page_size;
  a.num_raw = cache->num_raw_slots;
  const int nblk = cache->page_size / 4;
  const size_t smem = static_cast<size_t>(2 * nblk) * kSlotBytes + 16;
  if (cudaFuncSetAttribute(append_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem)) !=
      cudaSuccess)
    return ZF_ERR_CUDA;
  append_kernel<<<dim3(n, cache->num_kv_heads), kCodecThreads, smem, static_cast<cudaStream_t>(stream)>>>(a);
  return cudaGetLastError() == cudaSuccess ? ZF_OK : ZF_ERR_CUDA;
}

extern "C" zf_status zf_validate_pages(const zf_cache* cache, const int32_t* page_ids, int32_t n, int32_t* bad,
                                       void* stream) {
  zf_status st = check_cache(cache, /*need_comp=*/true, /*need_raw=*/false, /*need_dir=*/true);
  if (st != ZF_OK) return st;
  if (n < 0) return ZF_ERR_INVALID_ARGUMENT;
  if (n == 0) return ZF_OK;
  if (!page_ids || (reinterpret_cast<uintptr_t>(bad) & 3u)) return ZF_ERR_INVALID_ARGUMENT;
  if (cache->num_kv_heads > 65535) return ZF_ERR_UNSUPPORTED;
  CodecArgs a{};
  a.k_comp = cache->k_comp; a.v_comp = cache->v_comp; a.dir = cache->dir; a.status = cache->status;
  a.page_ids = page_ids;
  a.num_pages = cache->num_pages; a.hkv = cache->num_kv_heads; a.page_size = cache->page_size;
  a.num_raw = cache->num_raw_slots;
  validate_kernel<<<dim3(n, cache->num_kv_heads), kCodecThreads, 0, static_cast<cudaStream_t>(stream)>>>(a, bad);
  return cudaGetLastError() == cudaSuccess ? ZF_OK : ZF_ERR_CUDA;
}

extern "C" int32_t zf_slot_is_valid(const uint8_t* slot) { return slot && slot_ok(slot) ? 1 : 0; }

static zf_status launch_decompress(const zf_cache* cache, const int32_t* page_ids, int32_t n, uint16_t* dst_k,
                                   uint16_t* dst_v, int raw_out, void* stream) {
  // the directory may name any compressed slot or raw slot, so every pool the descriptor sizes
  // must be present (a NULL pool would otherwise be read on the device)
  zf_status st = check_cache(cache, /*need_comp=*/true, /*need_raw=*/true, /*need_dir=*/true);
  if (st != ZF_OK) return st;
  if (n < 0) return ZF_ERR_INVALID_ARGUMENT;
  if (n == 0) return ZF_OK;
  if (!page_ids || !dst_k || !dst_v || !aligned16(dst_k) || !aligned16(dst_v)) return ZF_ERR_INVALID_ARGUMENT;
  if (cache->num_kv_heads > 65535) return ZF_ERR_UNSUPPORTED;
  CodecArgs a{};
  a.k_comp = cache->k_comp; a.v_comp = cache->v_comp; a.k_raw = cache->k_raw; a.v_raw = cache->v_raw;
  a.dir = cache->dir; a.status = cache->status;
  a.dst_k = dst_k; a.dst_v = dst_v; a.page_ids = page_ids;
  a.num_pages = cache->num_pages; a.hkv = cache->num_kv_heads; a.page_size = cache->page_size;
  a.num_raw = cache->num_raw_slots;
  a.raw_out = raw_out;
  decompress_kernel<<<dim3(n, cache->num_kv_heads), kCodecThreads, 0, static_cast<cudaStream_t>(stream)>>>(a);
  return cudaGetLastError() == cudaSuccess ? ZF_OK : ZF_ERR_CUDA;
}

extern "C" zf_status zf_decompress(const zf_cache* cache, const int32_t* page_ids, int32_t n, uint16_t* dst_k,
                                   uint16_t* dst_v, void* stream) {
  return launch_decompress(cache, page_ids, n, dst_k, dst_v, 0, stream);
}

extern "C" zf_status zf_decompress_to_raw(const zf_cache* cache, const int32_t* page_ids, int32_t n,
                                          uint16_t* dst_k_raw, uint16_t* dst_v_raw, void* stream) {
  return launch_decompress(cache, page_ids, n, dst_k_raw, dst_v_raw, 1, stream);
}
