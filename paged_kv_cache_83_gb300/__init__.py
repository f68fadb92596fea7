"""GB300-native paged KV-cache hot path: slot-mapped K/V store, paged GQA decode and varlen
prefill with a cached prefix, as hand-written sm_103a CUDA kernels behind a C ABI
(``include/pa.h``). ``binding`` holds the Python marshalling layer; ``build`` compiles the
library in-tree."""
from .binding import (PA_BM_DEGENERATE_HASH, BlockManager, BlockManagerError,
                      PA_DECODE_NOALLOC_SCRATCH_BYTES, PA_DEVERR_LENGTH, PA_DEVERR_SLOT,
                      PA_DEVERR_TABLE, PA_DEVERR_TIMEOUT, PagedAttnError, load, pa_decode,
                      pa_decode_debug_tail_units, pa_decode_noalloc,
                      pa_decode_workspace_size, pa_prefill_varlen, pa_store_decode,
                      pa_store_decode_host, pa_store_decode_host_layout,
                      pa_store_decode_host_workspace_size, pa_store_kv)

__all__ = ["load", "pa_store_kv", "pa_decode", "pa_store_decode", "pa_store_decode_host",
           "pa_store_decode_host_layout", "pa_store_decode_host_workspace_size", "pa_decode_workspace_size",
           "pa_prefill_varlen",
           "pa_decode_noalloc", "PA_DECODE_NOALLOC_SCRATCH_BYTES", "BlockManager",
           "BlockManagerError", "PA_BM_DEGENERATE_HASH",
           "PagedAttnError", "PA_DEVERR_SLOT", "PA_DEVERR_TABLE", "PA_DEVERR_LENGTH",
           "PA_DEVERR_TIMEOUT", "pa_decode_debug_tail_units"]
