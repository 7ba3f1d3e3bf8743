"""GB300-native (sm_103a) DSA sparse decode attention over a paged KV cache.

The compute lives in libsdattn.so (CUDA kernels behind the C ABI of
include/sdattn.h); this package is its thin ctypes binding plus the seeded
synthetic workload generators (``inputs``).  Importing the package does not
load the library; the first call does, and raises if it is not built.
"""
from ._binding import (  # noqa: F401
    FLAG_BOUNDS,
    FLAG_TIMEOUT,
    SdaError,
    declared_functions,
    default_workspace,
    load,
    no_alloc_read_errors,
    read_errors,
    set_wait_limit_ns,
    sparse_decode_attention,
    sparse_decode_attention_no_alloc,
    sparse_decode_select_regions,
    sparse_decode_splits,
    sparse_decode_summary_scores,
    sparse_decode_swa_attention,
    sparse_decode_swa_splits,
    status_string,
    timeline_buffer,
    use_library,
    workspace_bytes,
)
