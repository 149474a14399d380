// Host-side argument checks shared by the libzf entry points.
#pragma once

#include <stdint.h>

#include "../../include/zf.h"

namespace zf {

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Shape and pointer checks of a cache descriptor.  Pools a call does not use may be NULL.
inline zf_status check_cache(const zf_cache* c, bool need_comp, bool need_raw, bool need_dir) {
  if (!c) return ZF_ERR_INVALID_ARGUMENT;
  if (c->head_dim != ZF_HEAD_DIM || c->reserved != 0) return ZF_ERR_INVALID_ARGUMENT;
  if (c->page_size < ZF_BLOCK_TOKENS || c->page_size % ZF_BLOCK_TOKENS != 0) return ZF_ERR_INVALID_ARGUMENT;
  if (c->page_size > ZF_MAX_PAGE_SIZE) return ZF_ERR_UNSUPPORTED;
  if (c->num_kv_heads < 1 || c->num_pages < 0 || c->num_raw_slots < 0) return ZF_ERR_INVALID_ARGUMENT;
  if (need_comp && c->num_pages > 0) {
    if (!c->k_comp || !c->v_comp || !aligned16(c->k_comp) || !aligned16(c->v_comp)) return ZF_ERR_INVALID_ARGUMENT;
  }
  if (need_raw && c->num_raw_slots > 0) {
    if (!c->k_raw || !c->v_raw || !aligned16(c->k_raw) || !aligned16(c->v_raw)) return ZF_ERR_INVALID_ARGUMENT;
  }
  if (need_dir && c->num_pages > 0 && !c->dir) return ZF_ERR_INVALID_ARGUMENT;
  if (c->status && (reinterpret_cast<uintptr_t>(c->status) & 3u)) return ZF_ERR_INVALID_ARGUMENT;
  return ZF_OK;
}

}  // namespace zf
