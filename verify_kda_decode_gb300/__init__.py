"""GB300-native KDA (Kimi Delta Attention) mixer step: decode, draft verify + commit, prefill.

The compute lives in libkda.so (hand-written sm_103a CUDA behind the C ABI in include/kda.h);
``verify_kda_decode_gb300.kda`` is its ctypes binding.  Importing the package loads the library
(building it in-tree with nvcc first if it is missing) and fails if that is not possible.
"""
from .kda import (  # noqa: F401
    EXPORTS, KdaError, KdaLayer, KdaPool, kda_commit, kda_decode, kda_decode_resume, kda_get_error,
    kda_prefill, kda_prefill_varlen, kda_prefill_varlen_workspace_size,
    kda_prefill_noalloc, kda_prefill_noalloc_max_bytes, kda_prefill_workspace_size, kda_verify,
    kda_verify_resume,
    library, prepare_decode, prepare_verify, PreparedCall,
)
