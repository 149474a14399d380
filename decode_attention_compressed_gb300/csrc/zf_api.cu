// Status strings and size helpers of the libzf C ABI.
#include <stddef.h>
#include <stdint.h>

#include "../../include/zf.h"

extern "C" const char* zf_status_string(zf_status status) {
  switch (status) {
    case ZF_OK: return "ok";
    case ZF_ERR_INVALID_ARGUMENT: return "invalid argument";
    case ZF_ERR_UNSUPPORTED: return "unsupported configuration";
    case ZF_ERR_WORKSPACE_TOO_SMALL: return "workspace too small";
    case ZF_ERR_CUDA: return "CUDA runtime error";
    case ZF_ERR_STATIC_WORKSPACE_EXCEEDED: return "sizes need more scratch than the library's static workspace";
    case ZF_ERR_CAPACITY: return "not enough free page ids or raw slots";
    case ZF_ERR_STATIC_WORKSPACE_UNAVAILABLE: return "no device memory left to load the library's static workspace";
    default: return "unknown status";
  }
}

extern "C" size_t zf_page_head_bytes(int32_t page_size, int32_t compressed) {
  if (page_size < ZF_BLOCK_TOKENS || page_size % ZF_BLOCK_TOKENS || page_size > ZF_MAX_PAGE_SIZE) return 0;
  return static_cast<size_t>(page_size / 4) * (compressed ? ZF_SLOT_BYTES : ZF_RAW_BLOCK_BYTES);
}
