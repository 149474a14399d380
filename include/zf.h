/*
 * zf.h — C ABI of libzf: decode attention over a losslessly compressed BF16 paged KV cache,
 * hand-written CUDA for GB300 (sm_103a).
 *
 * The method follows "ZipFusion: Fusing Lossless KV Decompression with Attention for Efficient
 * LLM Decoding": full pages are compressed into fixed-layout blocks (§III.B, Fig. 2), the
 * attention kernel copies compressed blocks from HBM to shared memory and rebuilds the exact
 * BF16 bit patterns in registers with integer operations right before the tensor-core
 * instructions (§III.C), partially filled pages stay uncompressed (§III.D), and split-KV partial
 * results are combined by a split-result merge (§IV.B).
 *
 * General rules for every call below
 *  - All tensor pointers are DEVICE pointers owned by the caller; the library never allocates,
 *    frees or keeps them.  All arrays are dense, row-major, and 16-byte aligned.  (The host-side
 *    page manager zf_kv_* and zf_slot_is_valid work on host memory instead.)
 *  - BF16 values are passed as their 16-bit patterns (uint16_t).
 *  - `stream` is a cudaStream_t (NULL = the legacy default stream).  Every call only enqueues
 *    work on `stream` and returns; results are ready when the stream reaches that point.
 *  - Host-side argument errors are detected before anything is launched and returned as a
 *    negative zf_status.  Data-dependent errors found on the device (an out-of-range page id,
 *    a page that needed raw storage but got none, a pipeline wait that gave up) never fault:
 *    the offending page is skipped and a bit is OR-ed into the optional device status word
 *    zf_cache.status (ZF_DEV_* below), which the caller may read after synchronising.
 *  - Concurrent calls on different streams are safe as long as they do not write the same memory.
 *    The library's only global state is (a) the scratch array of zf_decode_attn_static (below),
 *    which that entry point's calls share, and (b) a per-device record, behind a mutex, of the
 *    shared-memory limits already raised for its kernels.  Every other entry point works only
 *    on the memory it is given.
 *
 * Data layout of one layer's cache (head_dim is fixed at 128, page_size P is a multiple of 16):
 *  - A BLOCK is 16 consecutive tokens x 32 consecutive channels of one (page, kv head, K|V):
 *    512 values.  A page head holds P/16 tiles x 4 channel groups = P/4 blocks, tile-major.
 *  - Storage order inside a block (ZipFusion §III.C: keys and values are arranged for their
 *    operand roles): position p = 16*lane + 8*half + r is element r of `lane` in the A operand of
 *    the warp MMA m16n8k16 (PTX ISA, "Matrix Fragments for mma.m16n8k16"): for K the A operand
 *    is the 16x16 tile (rows tokens, columns channels 16*half..+15); for V it is the transposed
 *    tile (rows channels 16*half..+15, columns tokens).
 *  - Compressed block, 784 bytes: [0,512) the values' low bytes in storage order;
 *    [512,768) 4-bit codes (bit 3 sign, bits 0-2 exponent offset), byte 4m+k = code[8m+k] |
 *    code[8m+k+4] << 4; [768,772) header u32 = base/2 | n_escapes << 8 | 1 << 24 (format 1,
 *    other bits 0); [772,784) up to six u16 escapes (position << 7 | exponent >> 1), ascending.
 *    base is the block's minimum exponent rounded down to even when every exponent fits
 *    [base, base+15] (ZipFusion's rule); otherwise the smallest even base whose window reaches
 *    the maximum exponent, with the (at most 6) lower values listed as escapes.
 *  - Raw block, 1024 bytes: the 512 BF16 values, half-major: position 256*half + 8*lane + r
 *    holds storage position 16*lane + 8*half + r (conflict-free 16-byte reads per half).
 *  - k_comp/v_comp: [num_pages][num_kv_heads][P/4 blocks][784 bytes]  (slot of each page id)
 *    k_raw/v_raw:   [num_raw_slots][num_kv_heads][P/4 blocks][512 BF16]
 *    dir:           [num_pages][num_kv_heads] int32: ZF_DIR_COMPRESSED, a raw slot index >= 0,
 *                   or ZF_DIR_INVALID.
 */
#ifndef ZF_H
#define ZF_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef int32_t zf_status;
#define ZF_OK 0
#define ZF_ERR_INVALID_ARGUMENT (-1)   /* null pointer, bad size, misaligned pointer, bad shape */
#define ZF_ERR_UNSUPPORTED (-2)        /* valid but outside what this build handles */
#define ZF_ERR_WORKSPACE_TOO_SMALL (-3)
#define ZF_ERR_CUDA (-4)               /* a CUDA runtime call failed (launch or attribute) */
#define ZF_ERR_STATIC_WORKSPACE_EXCEEDED (-5) /* zf_decode_attn_static: sizes need more than ZF_STATIC_WORKSPACE_BYTES */
#define ZF_ERR_CAPACITY (-6)           /* zf_kv: not enough free page ids or raw slots; nothing changed */
#define ZF_ERR_STATIC_WORKSPACE_UNAVAILABLE (-7) /* zf_decode_attn_static: the device had no memory left to
                                                    load the library's scratch array (see that call) */

/* Bits of the device status word (zf_cache.status). */
#define ZF_DEV_BAD_PAGE_ID 0x1         /* page id outside [0, num_pages) */
#define ZF_DEV_BAD_RAW_SLOT 0x2        /* a page head needed raw storage and its raw slot was missing or out of range */
#define ZF_DEV_BAD_N_VALID 0x4         /* n_valid outside [0, page_size] */
#define ZF_DEV_BAD_SEQ_LEN 0x8         /* seq_len outside [0, max_pages_per_req * page_size] */
#define ZF_DEV_BAD_DIR 0x10            /* directory entry neither compressed nor a valid raw slot */
#define ZF_DEV_TIMEOUT 0x20            /* a shared-memory pipeline wait gave up */
#define ZF_DEV_BAD_SLOT 0x40           /* zf_validate_pages: a compressed slot's metadata is malformed */

#define ZF_HEAD_DIM 128
#define ZF_BLOCK_TOKENS 16
#define ZF_BLOCK_CHANNELS 32
#define ZF_SLOT_BYTES 784
#define ZF_RAW_BLOCK_BYTES 1024
#define ZF_MAX_ESCAPES 6
#define ZF_FORMAT_VERSION 1
#define ZF_DIR_COMPRESSED (-1)
#define ZF_DIR_INVALID (-2)
#define ZF_MAX_BATCH 4096              /* requests per zf_decode_attn call */
#define ZF_MAX_TOKENS 64               /* new tokens per request in zf_decode_attn_multi */
#define ZF_MAX_PAGE_SIZE 128

#define ZF_ENCODE_FORCE_RAW 1          /* zf_encode_pages flag: store every page raw */

/* One layer's cache.  Only the pointers a call uses must be valid for that call. */
typedef struct zf_cache {
  int32_t num_pages;      /* page ids are in [0, num_pages) */
  int32_t num_kv_heads;
  int32_t head_dim;       /* must be 128 */
  int32_t page_size;      /* tokens per page, multiple of 16, <= ZF_MAX_PAGE_SIZE */
  int32_t num_raw_slots;  /* raw page slots in k_raw / v_raw (may be 0) */
  int32_t reserved;       /* must be 0 */
  uint8_t* k_comp;        /* [num_pages][num_kv_heads][page_size/4][784] */
  uint8_t* v_comp;
  uint16_t* k_raw;        /* [num_raw_slots][num_kv_heads][page_size/4][512]; several layers' caches
                             may point at the same raw arrays (one pool, each slot written only by
                             the encode it was listed for; see zf_kv) */
  uint16_t* v_raw;
  int32_t* dir;           /* [num_pages][num_kv_heads] */
  int32_t* status;        /* optional device word; ZF_DEV_* bits are OR-ed in; NULL = not reported */
} zf_cache;

/* Human-readable name of a status code.  Never returns NULL. */
const char* zf_status_string(zf_status status);

/* Bytes of one (page, kv head) record of K (or of V): compressed = page_size/4 * 784,
 * raw = page_size/4 * 1024.  Returns 0 for an unsupported page size. */
size_t zf_page_head_bytes(int32_t page_size, int32_t compressed);

/*
 * zf_encode_pages — compress (or store raw) n full or partial pages.
 * ZipFusion §III.B (format) and §III.D (page lifecycle: a partially filled page stays
 * uncompressed so decoding can keep appending to it; a full page is compressed later and keeps
 * its page id).
 *   src_k, src_v: [n][num_kv_heads][page_size][128] BF16, natural (token, channel) layout; page i
 *                 of the call is written under id page_ids[i].
 *   page_ids:     [n] distinct ids in [0, num_pages).
 *   n_valid:      [n] tokens filled in each page, 0..page_size.  Pages with n_valid < page_size,
 *                 pages with a block that needs more than 6 escapes, and every page when
 *                 flags & ZF_ENCODE_FORCE_RAW are stored raw in slot raw_slots[i] (values past
 *                 n_valid are stored as given).  Otherwise the page goes to its compressed slot.
 *   raw_slots:    [n] raw slot per page, or -1 when none is available (a page that then needs
 *                 raw storage gets ZF_DIR_INVALID and ZF_DEV_BAD_RAW_SLOT).
 *   Writes k_comp/v_comp or k_raw/v_raw and dir[page_ids[i]][*].  A full page head that ends up
 *   raw (a block with more than 6 escapes) may also have had its compressed slot overwritten;
 *   that slot is not read while the directory names the raw slot.  All pointers are device
 *   pointers; n == 0 is a no-op.  The source must not alias the cache.  Launched with
 *   programmatic stream serialisation (it waits for the preceding kernel before reading).
 */
zf_status zf_encode_pages(const zf_cache* cache, const uint16_t* src_k, const uint16_t* src_v,
                          const int32_t* page_ids, const int32_t* n_valid,
                          const int32_t* raw_slots, int32_t n, int32_t flags, void* stream);

/*
 * zf_append_tokens — write one new token into each of n uncompressed pages, in place.
 * ZipFusion §III.D (KV Cache Management and Scheduling): a page that is still filling stays
 * uncompressed so decoding appends its values directly; once full it is compressed under its
 * page id.
 *   k_tok, v_tok: [n][num_kv_heads][128] BF16: entry i is the token at index positions[i]
 *                 (0..page_size-1) of page page_ids[i], written into raw slot raw_slots[i], which
 *                 must already hold the page's earlier tokens (from earlier appends, or from
 *                 zf_encode_pages with that slot and n_valid >= positions[i]).
 *   page_ids:     [n] distinct ids in [0, num_pages); raw_slots: [n] in [0, num_raw_slots).
 *   The directory entry of each page head becomes the raw slot; when positions[i] is
 *   page_size - 1 the page head is then compressed from the slot into its compressed slot
 *   (directory ZF_DIR_COMPRESSED), unless a block needs more than 6 escapes (it stays raw).
 *   The result is bit-for-bit what zf_encode_pages writes for the page's tokens so far.  A bad
 *   page id sets ZF_DEV_BAD_PAGE_ID; a bad position or raw slot sets ZF_DEV_BAD_N_VALID /
 *   ZF_DEV_BAD_RAW_SLOT and makes the page's directory entries invalid.  Needs k_comp, v_comp,
 *   k_raw, v_raw and dir; device pointers; n == 0 is a no-op.
 */
zf_status zf_append_tokens(const zf_cache* cache, const uint16_t* k_tok, const uint16_t* v_tok,
                           const int32_t* page_ids, const int32_t* positions, const int32_t* raw_slots,
                           int32_t n, void* stream);

/*
 * zf_validate_pages — check the stored form of n pages, for example after a cache was saved to a
 * file and loaded again (its pools are plain bytes).  Per page head: the directory entry must be
 * ZF_DIR_COMPRESSED or a raw slot in [0, num_raw_slots) (else ZF_DEV_BAD_DIR); every K and V
 * slot of a compressed page head must pass zf_slot_is_valid (else ZF_DEV_BAD_SLOT).  Raw records
 * hold plain BF16 values, where every bit pattern is valid.  Bad page ids set ZF_DEV_BAD_PAGE_ID.
 *   page_ids: [n] device; bad: optional [n] device int32, set to 1 for each page with a problem
 *   (entries of good pages are left as they are: zero it first).  Needs k_comp, v_comp and dir.
 */
zf_status zf_validate_pages(const zf_cache* cache, const int32_t* page_ids, int32_t n, int32_t* bad,
                            void* stream);

/* One 784-byte compressed slot in host memory: 1 when its metadata is well formed — format
 * version 1, header bits 7 and 11-23 zero, at most 6 escapes, escape positions strictly
 * ascending, unused escape entries zero, and base/2 + every code's 3-bit offset within 7 bits
 * (the rebuild adds them without a carry, ZipFusion §III.C) — else 0.  The same test
 * zf_validate_pages runs on the device. */
int32_t zf_slot_is_valid(const uint8_t* slot);

/*
 * zf_decompress — bit-exact inverse of zf_encode_pages, used for verification.
 *   page_ids: [n] ids; dst_k, dst_v: [n][num_kv_heads][page_size][128] BF16 in natural layout.
 *   A page head whose directory entry is invalid is written as zeros (and ZF_DEV_BAD_DIR set).
 */
zf_status zf_decompress(const zf_cache* cache, const int32_t* page_ids, int32_t n,
                        uint16_t* dst_k, uint16_t* dst_v, void* stream);

/*
 * zf_decompress_to_raw — zf_decompress into the raw block layout of a dense cache: page_ids[i] is
 * written to raw slot i of dst_k_raw / dst_v_raw ([n][num_kv_heads][page_size/4][512] BF16, the
 * layout of zf_cache.k_raw / v_raw), so zf_dense_decode_attn can attend over the result directly.
 * This is the restore-then-attend pattern that ZipFusion §II.B (Compression for Faster Decode
 * Attention) measures: each layer is restored into a shared buffer before a dense attention
 * kernel reads it.  It is kept as a measured baseline for the fused path.  The bytes written equal
 * those zf_encode_pages with ZF_ENCODE_FORCE_RAW writes for the same source pages.  Same argument
 * checks and device error reporting as zf_decompress.
 */
zf_status zf_decompress_to_raw(const zf_cache* cache, const int32_t* page_ids, int32_t n,
                               uint16_t* dst_k_raw, uint16_t* dst_v_raw, void* stream);

/* Workspace bytes zf_decode_attn / zf_dense_decode_attn need for these sizes on the current
 * device (split-KV partial outputs and log-sum-exps).  0 on invalid sizes. */
size_t zf_decode_attn_workspace_size(int32_t batch, int32_t num_q_heads, int32_t num_kv_heads,
                                     int32_t page_size, int32_t max_pages_per_req);

/*
 * zf_decode_attn — batched single-token decode attention over the compressed paged cache.
 * ZipFusion §III.C (attention consumes compressed blocks copied HBM->shared memory and rebuilt in
 * registers, raw blocks need no rebuild; page metadata for later pages is fetched while earlier
 * pages are attended) and §IV.B (split-KV with a split-result merge).
 *   q:          [batch][num_q_heads][128] BF16.  Query head h reads kv head h / (num_q_heads /
 *               num_kv_heads); num_q_heads must be a multiple of num_kv_heads.
 *   page_table: [batch][max_pages_per_req] page ids; token t of request b is slot t % page_size
 *               of page page_table[b][t / page_size].  Entries past a request's pages are unread.
 *   seq_lens:   [batch] device int32 context lengths, 0..max_pages_per_req * page_size.
 *   softmax_scale: multiplies q.k before the softmax.
 *   out:        [batch][num_q_heads][128] float32 = sum_t softmax(scale * q.k)_t v_t.
 *   lse:        [batch][num_q_heads] float32, natural-log log-sum-exp of scale * q.k.
 *               A request with seq_len 0 gets out = 0 and lse = -inf.
 *   workspace:  device buffer of at least zf_decode_attn_workspace_size(...) bytes, any contents;
 *               it must not be shared with a concurrent call.
 *   batch <= ZF_MAX_BATCH.  Two kernels are enqueued (attention, then merge); results are
 *   deterministic (no atomics).  The attention kernel is the one ZF_KERNEL_AUTO picks (see
 *   zf_decode_attn_multi_kernel): the warp-MMA kernel when a kv head has at most 8 query heads,
 *   the tcgen05 kernel above that (where it fits the batch).
 *   Both are launched with programmatic stream serialisation: when the kernel ahead of them in
 *   the stream allows it (griddepcontrol.launch_dependents; this library's merge kernel does), the
 *   attention grid starts early.  Before its grid-dependency wait it only warms L2 and, for short
 *   calls, plans its first item from relaxed reads of seq_lens, page_table and the directory and
 *   prefetches the first tiles into L2; after the wait every length, page-table and directory
 *   entry it uses is read again (a plan whose inputs changed is dropped) and q and the K/V data
 *   are read only then, so inputs written by that preceding kernel are always seen.
 */
zf_status zf_decode_attn(const zf_cache* cache, const uint16_t* q, int32_t batch,
                         int32_t num_q_heads, const int32_t* page_table, int32_t max_pages_per_req,
                         const int32_t* seq_lens, float softmax_scale, float* out, float* lse,
                         void* workspace, size_t workspace_bytes, void* stream);

/* Workspace bytes zf_decode_attn_multi / zf_dense_decode_attn_multi need (0 on invalid sizes). */
size_t zf_decode_attn_multi_workspace_size(int32_t batch, int32_t tokens, int32_t num_q_heads,
                                           int32_t num_kv_heads, int32_t page_size,
                                           int32_t max_pages_per_req);

/*
 * zf_decode_attn_multi — decode attention for `tokens` (T) new tokens per request at once
 * (speculative verification, multi-token decode).  The pages treat one new token per step; this
 * call takes the plain causal reading of several: the T tokens of request b sit at positions
 * L-T .. L-1 (L = seq_lens[b]; their keys and values are already in the cache) and token t
 * attends to positions 0 .. L-T+t, exactly as zf_decode_attn over that prefix would.
 *   q:   [batch][T][num_q_heads][128] BF16.
 *   out: [batch][T][num_q_heads][128] float32;  lse: [batch][T][num_q_heads] float32.
 *   1 <= T <= ZF_MAX_TOKENS.  A token that sees no position (L - T + t < 0) gets out = 0 and
 *   lse = -inf.  The (head, token) pairs of one kv head are computed like a GQA group T times
 *   larger: the 8 columns of a tensor-core tile take 8 of them, and each group of 8 reads the kv
 *   head's K/V tiles once, so the bytes read do not grow with T while (q heads per kv head) x T
 *   <= 8 (MHA up to 8 tokens, GQA-4 up to 2) and grow by one read per further 8.  Other arguments,
 *   workspace and ordering as zf_decode_attn (workspace: zf_decode_attn_multi_workspace_size).
 *   T = 1 is zf_decode_attn.
 */
zf_status zf_decode_attn_multi(const zf_cache* cache, const uint16_t* q, int32_t batch, int32_t tokens,
                               int32_t num_q_heads, const int32_t* page_table, int32_t max_pages_per_req,
                               const int32_t* seq_lens, float softmax_scale, float* out, float* lse,
                               void* workspace, size_t workspace_bytes, void* stream);

/* Kernels zf_decode_attn_multi_kernel can be asked for. */
#define ZF_KERNEL_AUTO 0       /* what zf_decode_attn and zf_decode_attn_multi run (below) */
#define ZF_KERNEL_WARP_MMA 1   /* warp-level MMA, 8 query columns per pass over a kv head's tiles */
#define ZF_KERNEL_TCGEN05 2    /* 5th-generation tensor cores, 16 or 32 columns per pass */

/*
 * zf_decode_attn_multi_kernel — zf_decode_attn_multi with the attention kernel chosen by `kernel`.
 * ZipFusion §III.C: the compressed blocks are rebuilt into exact BF16 operands right before the
 * tensor-core instructions.  The columns of a kv head are its query heads x new tokens
 * ((num_q_heads / num_kv_heads) x T).
 *  - ZF_KERNEL_WARP_MMA rebuilds each block in registers straight into warp-MMA (m16n8k16)
 *    fragments: 8 columns per pass, so a kv head's K/V tiles are read once per 8 columns.
 *  - ZF_KERNEL_TCGEN05 rebuilds each 16-token tile into operands of tcgen05.mma (K in tensor
 *    memory, V^T in shared memory; M = 128 tokens or channels) whose scores and output accumulate
 *    in tensor memory: N = 16 columns per pass when a kv head has at most 16 columns, else 32,
 *    so a kv head's tiles are read once per 16 or 32 columns.  Its shared memory also holds the
 *    request lengths: batch above 1379 (16 columns) or 1363 (32 columns) returns
 *    ZF_ERR_UNSUPPORTED.
 *  - ZF_KERNEL_AUTO (what zf_decode_attn / zf_decode_attn_multi do) runs ZF_KERNEL_TCGEN05 when
 *    a kv head has more than 8 columns (where the warp-MMA kernel would read its tiles twice or
 *    more) and the batch fits it, else ZF_KERNEL_WARP_MMA.
 *   Both give the same results within floating-point rounding (different summation order).
 *   Workspace: zf_decode_attn_multi_workspace_size covers every kernel.  Other arguments as for
 *   zf_decode_attn_multi.  Returns ZF_ERR_INVALID_ARGUMENT for an unknown `kernel`.
 */
zf_status zf_decode_attn_multi_kernel(const zf_cache* cache, const uint16_t* q, int32_t batch, int32_t tokens,
                                      int32_t num_q_heads, const int32_t* page_table, int32_t max_pages_per_req,
                                      const int32_t* seq_lens, float softmax_scale, float* out, float* lse,
                                      void* workspace, size_t workspace_bytes, int32_t kernel, void* stream);

/*
 * zf_decode_attn_wait_test — for tests of the failure path: zf_decode_attn_multi_kernel with the
 * kernel's waits for its metadata warp's items limited to wait_limit_ns (1 us .. 2 s; the normal
 * limit is 2 s) and that warp's first item published publish_delay_ns (<= 2 s) late.  With a delay
 * above the limit the waits run out: the call then sets ZF_DEV_TIMEOUT in the cache's status
 * word, the CTAs wind down (copies in flight land first, tensor memory is released), no output is
 * guaranteed, and the context and the stream stay usable for the next call.  No fault, trap or
 * endless wait is involved.  The paper has no counterpart; it exists so that tests can exercise the
 * bounded waits.  ZF_ERR_INVALID_ARGUMENT for limits out of range; other arguments as for
 * zf_decode_attn_multi_kernel.
 */
zf_status zf_decode_attn_wait_test(const zf_cache* cache, const uint16_t* q, int32_t batch, int32_t tokens,
                                   int32_t num_q_heads, const int32_t* page_table, int32_t max_pages_per_req,
                                   const int32_t* seq_lens, float softmax_scale, float* out, float* lse,
                                   void* workspace, size_t workspace_bytes, int32_t kernel, uint64_t wait_limit_ns,
                                   uint64_t publish_delay_ns, void* stream);

/*
 * zf_dense_decode_attn — the same decode attention over an uncompressed BF16 paged cache: page
 * id p of the page table is read from raw slot p of cache->k_raw / cache->v_raw (raw block
 * layout above; zf_encode_pages with ZF_ENCODE_FORCE_RAW and raw_slots = page_ids builds it).
 * cache->num_raw_slots bounds the page ids; dir and the compressed pools are not used.
 * Same grid, pipeline and merge as zf_decode_attn; it reads 1024-byte blocks instead of
 * 784-byte ones and skips the reconstruction.  Arguments as for zf_decode_attn.
 */
zf_status zf_dense_decode_attn(const zf_cache* cache, const uint16_t* q, int32_t batch,
                               int32_t num_q_heads, const int32_t* page_table,
                               int32_t max_pages_per_req, const int32_t* seq_lens,
                               float softmax_scale, float* out, float* lse, void* workspace,
                               size_t workspace_bytes, void* stream);

/* zf_dense_decode_attn_multi — zf_decode_attn_multi over the uncompressed cache (the comparator). */
zf_status zf_dense_decode_attn_multi(const zf_cache* cache, const uint16_t* q, int32_t batch,
                                     int32_t tokens, int32_t num_q_heads, const int32_t* page_table,
                                     int32_t max_pages_per_req, const int32_t* seq_lens,
                                     float softmax_scale, float* out, float* lse, void* workspace,
                                     size_t workspace_bytes, void* stream);

/*
 * zf_decode_attn_static — zf_decode_attn for callers that cannot allocate device memory.
 * The paper has no counterpart to this entry point; it exists for integration only.
 *   Some callers have no way to hand the library a workspace: for example a kernel plugin inside
 *   a host engine that owns every byte of device memory through its own pool and exposes no
 *   scratch hook, or a latency-critical path where cudaMalloc (which can synchronise the device)
 *   is not allowed.  This call takes the same arguments as zf_decode_attn minus the workspace and
 *   uses a scratch array compiled into the library instead: ZF_STATIC_WORKSPACE_BYTES (32 MiB) of
 *   device memory that every GPU which loads libzf holds until the process exits.  It calls no
 *   cudaMalloc, cudaFree or allocating library routine.
 *   - Sizes whose split-KV partials need more than ZF_STATIC_WORKSPACE_BYTES (see
 *     zf_decode_attn_workspace_size) are rejected with ZF_ERR_STATIC_WORKSPACE_EXCEEDED before
 *     anything is launched.
 *   - When the array comes into being: CUDA loads the library's device code into a context lazily
 *     by default (CUDA_MODULE_LOADING=LAZY), and the array is reserved when the module holding
 *     it is loaded — at the first libzf attention call in that context, which may be the first
 *     zf_decode_attn_static call itself.  That first call can therefore reserve the 32 MiB and
 *     synchronise.  A caller that cannot allocate later should make one call (any shape) at
 *     initialisation, before its engine takes the rest of device memory and before any stream
 *     capture.  If the device has no memory left to load it, the call returns
 *     ZF_ERR_STATIC_WORKSPACE_UNAVAILABLE and launches nothing.
 *   - Every call looks up the array's address in the current context (cheap once the module is
 *     loaded, and it allocates nothing), so it stays correct after a device reset or with another
 *     context of the device current.
 *   - All calls share the one array and it keeps the previous call's contents (nothing in it has
 *     to start at zero).  Calls that overlap on the GPU (other streams, other threads) race on it:
 *     serialise them.
 *   Results are bit-for-bit those of zf_decode_attn for the same inputs (same kernels, same work
 *   split; only the scratch memory differs).
 */
#define ZF_STATIC_WORKSPACE_BYTES (32u << 20)
zf_status zf_decode_attn_static(const zf_cache* cache, const uint16_t* q, int32_t batch,
                                int32_t num_q_heads, const int32_t* page_table,
                                int32_t max_pages_per_req, const int32_t* seq_lens,
                                float softmax_scale, float* out, float* lse, void* stream);

/* ------------------------------------------------------------------------------------------
 * zf_kv — host-side page manager for the caches above.  ZipFusion §III.D (KV Cache Management and
 * Scheduling): a page stays uncompressed while it fills so that tokens can be appended in place,
 * a full page is compressed afterwards and keeps its page id, new pages must accept writes before
 * compression (so capacity for them is counted in uncompressed storage) and capacity grows back as
 * compression releases that storage.  §II.C (Compression for Higher Serving Capacity): the
 * storage compression frees is what lets more requests in.
 * A page id names one compressed slot in every layer's cache.  Raw slots come from one pool that
 * all num_layers layers share (every layer's zf_cache points its k_raw / v_raw at the same arrays
 * of num_raw_slots slots): a page being written holds one raw slot per layer — a request's partial
 * last page while it fills, a full page until the caller reports, layer by layer, whether its
 * encode compressed it (zf_kv_reclaim).  A layer whose page-heads of that page all compressed
 * returns its slot to the pool, where any layer can take it (§III.D: storage released in one layer
 * is reassigned to another once the reads of it have finished — here, once the caller has read
 * the directory after the encode, and the slot is only written again by a later encode on the
 * caller's stream); a layer with a page-head left raw (more than six escapes in a block) keeps its
 * slot until the request is released.  With num_layers = 1 the same bookkeeping also serves
 * per-layer raw pools addressed by one slot index (report a page raw when it is raw in any layer).
 * Per-layer outputs and inputs are layer-major: entry (layer l, item i) of an n-item list is at
 * l * n + i, so row l is the raw_slots array of layer l's zf_encode_pages / zf_append_tokens
 * call.  The manager only does the bookkeeping: the caller writes the listed pages (a prompt with
 * zf_encode_pages, a decode step's tokens with zf_append_tokens) and uploads the page table and
 * lengths.
 * Host code; not thread-safe; no GPU calls.
 * ------------------------------------------------------------------------------------------ */
typedef struct zf_kv zf_kv;

typedef struct zf_kv_stats {
  int64_t tokens;             /* tokens held by active requests */
  int32_t free_pages;         /* page ids not held */
  int32_t free_raw_slots;     /* raw slots not held */
  int32_t active_requests;
  int32_t partial_pages;      /* last pages still filling (each holds a raw slot) */
  int32_t pending_pages;      /* full pages whose raw slot awaits zf_kv_reclaim */
  int32_t raw_full_pages;     /* full pages left raw in at least one layer */
  int32_t compressed_pages;   /* full pages compressed in every layer (no raw slot) */
  int32_t new_page_capacity;  /* pages that can be opened now: min(free ids, free raw slots / num_layers) */
  int32_t raw_full_slots;     /* raw slots held by the raw_full_pages (one per layer left raw) */
} zf_kv_stats;

/* A manager for num_pages page ids and a pool of num_raw_slots raw slots (>= num_layers) shared by
 * num_layers layers, pages of page_size tokens, request slots 0 .. max_requests-1 of at most
 * max_pages_per_req pages each.  *out = NULL on error. */
zf_status zf_kv_create(int32_t num_pages, int32_t num_raw_slots, int32_t num_layers, int32_t page_size,
                       int32_t max_requests, int32_t max_pages_per_req, zf_kv** out);
void zf_kv_destroy(zf_kv* kv);

/* Admit request slot `req` (inactive) with a prompt of `len` tokens: takes n = ceil(len /
 * page_size) page ids and n raw slots per layer (every page is written uncompressed first) and
 * writes the encode list for the prompt in page order — page_ids / n_valid [n], raw_slots
 * [num_layers][n] — and *n = n.  ZF_ERR_CAPACITY when the pools cannot hold it. */
zf_status zf_kv_admit(zf_kv* kv, int32_t req, int32_t len, int32_t* page_ids, int32_t* n_valid,
                      int32_t* raw_slots, int32_t* n);

/* One new token for each of the n distinct active requests reqs[i]: entry i of the outputs is the
 * page that holds it (page_ids[i], tokens in it n_valid[i], its raw slot in layer l
 * raw_slots[l * n + i]) — one zf_append_tokens call per layer (positions n_valid[i] - 1) writes
 * them all.  A request whose last page is full opens a new page (an id + a raw slot per layer)
 * first; a page that becomes full here is compressed by those calls and its raw slots are
 * pending until zf_kv_reclaim.  All or nothing: ZF_ERR_CAPACITY (or an invalid request) changes
 * no request. */
zf_status zf_kv_append(zf_kv* kv, const int32_t* reqs, int32_t n, int32_t* page_ids, int32_t* n_valid,
                       int32_t* raw_slots);

/* Full pages whose raw slots are pending, ascending page id: *n = their count k; page_ids[i] and,
 * per layer, raw_slots[l * k + i] (raw_slots holds num_layers * capacity entries).
 * ZF_ERR_INVALID_ARGUMENT, with *n set, when k exceeds capacity. */
zf_status zf_kv_pending(const zf_kv* kv, int32_t* page_ids, int32_t* raw_slots, int32_t capacity, int32_t* n);

/* After the encodes of these n pending pages have run: kept_raw[l * n + i] != 0 when any
 * page-head of page_ids[i] is stored raw in layer l (directory entry >= 0); that layer keeps its
 * raw slot, every other layer returns its slot to the shared pool.  Every id must be pending,
 * with no repeats. */
zf_status zf_kv_reclaim(zf_kv* kv, const int32_t* page_ids, const int32_t* kept_raw, int32_t n);

/* Return request `req`'s page ids and raw slots to the pools. */
zf_status zf_kv_release(zf_kv* kv, int32_t req);

/* page_table [max_requests][max_pages_per_req] (-1 past a request's pages) and seq_lens
 * [max_requests] (0 for inactive slots), host arrays, as zf_decode_attn takes them. */
zf_status zf_kv_export(const zf_kv* kv, int32_t* page_table, int32_t* seq_lens);

zf_status zf_kv_get_stats(const zf_kv* kv, zf_kv_stats* out);

/* Sizing: page ids a layer's cache of bytes_per_layer holds next to num_raw_slots raw slots of
 * its own (with one shared pool: its share, pool slots / layers), counting compressed K and V
 * slots plus directory entries per page id, and the pages the same bytes hold as a dense BF16
 * cache. */
zf_status zf_kv_plan_pages(int64_t bytes_per_layer, int32_t num_kv_heads, int32_t page_size,
                           int32_t num_raw_slots, int32_t* num_pages, int32_t* dense_pages);

#ifdef __cplusplus
}
#endif

#endif /* ZF_H */
