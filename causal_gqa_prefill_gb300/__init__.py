"""GB300-native causal GQA prefill attention (forward, decode and backward).

The computation runs in a hand-written sm_103a CUDA library
(``lib/libattn_prefill.so``, C ABI in ``include/attn_prefill.h``); this
package is a thin binding plus the seeded workload generators. Importing it
does not load the library; the first call does, and raises if it is missing.
"""

from ._abi import (ATTN_OK, ATTN_ERR_INVALID_ARG, ATTN_ERR_UNSUPPORTED, ATTN_ERR_CUDA,
                   ATTN_ERR_TIMEOUT, ATTN_ERR_CHECK, load as load_library, library_path,
                   status_string)
from .api import (AttnError, attn_decode, attn_decode_fwd, attn_decode_workspace_bytes,
                  attn_prefill, attn_prefill_fp8, attn_prefill_fwd, attn_prefill_fwd_chunk,
                  attn_prefill_fwd_fp8, attn_device_check, attn_prefill_grid_size,
                  attn_prefill_backward, attn_prefill_bwd, attn_prefill_bwd_workspace_bytes,
                  attn_selftest_wait_timeout, attn_selftest_wait_timeout_noalloc,
                  attn_prefill_fwd_host,
                  attn_prefill_host_staging_bytes)

__all__ = [
    "ATTN_OK", "ATTN_ERR_INVALID_ARG", "ATTN_ERR_UNSUPPORTED", "ATTN_ERR_CUDA",
    "ATTN_ERR_TIMEOUT", "ATTN_ERR_CHECK", "AttnError", "attn_prefill", "attn_prefill_fwd", "attn_prefill_fwd_chunk",
    "attn_prefill_fp8", "attn_prefill_fwd_fp8", "attn_decode", "attn_decode_fwd",
    "attn_decode_workspace_bytes", "attn_device_check", "attn_prefill_backward",
    "attn_prefill_bwd", "attn_prefill_bwd_workspace_bytes", "attn_selftest_wait_timeout",
    "attn_selftest_wait_timeout_noalloc", "attn_prefill_fwd_host", "attn_prefill_host_staging_bytes",
    "attn_prefill_grid_size", "load_library", "library_path", "status_string",
]
