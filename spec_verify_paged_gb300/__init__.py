"""Paged decode/verify attention, KV append and speculative acceptance for
one GB300 GPU (sm_103a).

The computation lives in libsvp.so (CUDA kernels behind the C ABI declared in
include/svp.h); this package is its thin Python binding.  Importing it loads
nothing; the first call loads the library and raises if it is not built.
"""
from .binding import (  # noqa: F401
    StepRunner,
    SvpError,
    kv_append,
    last_launch_count,
    load_library,
    paged_decode_attention,
    paged_tree_attention,
    read_device_status,
    spec_accept,
    spec_accept_tree,
    workspace_for,
)
