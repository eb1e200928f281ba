"""Low-bit MLA KV-cache decode for one GB300 (sm_103a).

The compute lives in ``libmla_lowbit.so`` (hand-written CUDA kernels behind the
C ABI in include/mla_lowbit.h); this package is its thin Python binding.
"""

from .binding import (  # noqa: F401
    EXPORTS,
    Layout,
    LibraryError,
    bytes_per_token,
    decode,
    decode_multi,
    decode_noalloc,
    decode_plan,
    layout,
    load,
    page_bytes,
    read_error,
    set_fault_injection,
    strerror,
    version,
    write,
    write_decode,
)
from .cache import PagedCache  # noqa: F401
