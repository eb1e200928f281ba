"""CPU oracle for low-bit MLA decode (test infrastructure, not product code).

A plain, slow, obviously correct numpy restatement of what the decode path
computes, written from "QuantMLA: Function-Aligned Dual-Path Quantization for
Low-Bit MLA KV Caching" (Abstract; Figure 3 and Figure 8 captions) plus the
quantiser details those pages leave open and the workload fixes (per-token
asymmetric 64-channel groups, fp16 scale and min, round-half-to-even codes,
sink 4 / recent 128 bf16 tokens).

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  It shares no code with the CUDA path
and never imports it.

Every function here is pinned by ``tests/test_oracle.py`` against closed
forms, textbook IEEE facts, brute force and ``torch`` fp64 attention; the one
part the pages give no numbers for -- agreement with the authors' own kernel --
is "parity unpinned" (the pages print no worked example or kernel output).
"""

from .quant import (  # noqa: F401
    bf16_bits_to_f64,
    dequantize,
    f16_satfinite,
    pack_codes,
    quantize_group,
    quantize_token,
    unpack_codes,
    hadamard_matrix64,
    hadamard_rotate_f32,
    rotate_latent_bits,
)
from .layout import Layout, bytes_per_token, compression_ratio, page_geometry  # noqa: F401
from .cache import PagedCacheModel, is_protected, reference_keys  # noqa: F401
from .attention import mla_decode_fp64, mla_decode_multi_fp64  # noqa: F401
