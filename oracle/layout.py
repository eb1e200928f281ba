"""Physical cache layout of the oracle (its own definition; nothing shared with
the CUDA library).

QuantMLA (Abstract; Figure 3 and Figure 5a captions) stores packed content and
RoPE-key codes plus per-group metadata, with bf16 buffers for protected
tokens; the pages leave the byte geometry open.  Adopted geometry, per 64-token
page, every region 16-byte aligned:

* content codes ``[64][512 * content_bits / 8]`` bytes,
* RoPE codes ``[64][64 * rope_bits / 8]`` bytes,
* metadata ``[64][9][2]`` fp16 = (scale, min) for groups 0..7 (content) then 8 (RoPE).

A bf16 page (``content_bits == 16``) is ``[64][576]`` bf16 with no metadata.
"""

from __future__ import annotations

import dataclasses

LATENT = 512
ROPE = 64
GROUP = 64
PAGE_TOKENS = 64
SINK = 4
LOCAL = 128
N_GROUPS = (LATENT + ROPE) // GROUP  # 8 content + 1 rope


@dataclasses.dataclass(frozen=True)
class Layout:
    content_bits: int = 4   # 4, 2 or 16 (bf16 pages)
    rope_bits: int = 4      # 4, or 16 with bf16 pages
    rotate: bool = False    # online Hadamard rotation of the content latent (packed only)

    def __post_init__(self):
        ok = (self.content_bits, self.rope_bits) in ((4, 4), (2, 4), (16, 16))
        if not ok:
            raise ValueError(f"unsupported layout C{self.content_bits}R{self.rope_bits}")
        if self.rotate and not self.packed:
            raise ValueError("rotation applies to packed layouts")

    @property
    def packed(self) -> bool:
        return self.content_bits != 16


def page_geometry(layout: Layout) -> dict:
    if not layout.packed:
        return dict(page_bytes=PAGE_TOKENS * (LATENT + ROPE) * 2, row_bytes=(LATENT + ROPE) * 2)
    content_row = LATENT * layout.content_bits // 8
    rope_row = ROPE * layout.rope_bits // 8
    meta_row = N_GROUPS * 2 * 2
    content_off = 0
    rope_off = content_off + PAGE_TOKENS * content_row
    meta_off = rope_off + PAGE_TOKENS * rope_row
    page_bytes = meta_off + PAGE_TOKENS * meta_row
    return dict(page_bytes=page_bytes, content_off=content_off, content_row=content_row,
                rope_off=rope_off, rope_row=rope_row, meta_off=meta_off, meta_row=meta_row)


def bytes_per_token(layout: Layout) -> int:
    """Closed form: codes plus one fp16 (scale, min) pair per 64-channel group."""
    if not layout.packed:
        return (LATENT + ROPE) * 2
    return (LATENT * layout.content_bits // 8 + ROPE * layout.rope_bits // 8
            + N_GROUPS * 2 * 2)


def compression_ratio(layout: Layout, context: int = 0) -> float:
    """bf16 bytes over packed bytes for ``context`` tokens of one sequence.

    With ``context == 0`` the ratio of bare bytes per token.  Otherwise the
    packed side also holds the bf16 copies of the protected tokens (every
    token keeps a packed copy, Figure 8 caption), ``min(context, 132)`` of them.
    """
    bf16 = (LATENT + ROPE) * 2
    if context == 0:
        return bf16 / bytes_per_token(layout)
    prot = min(context, SINK + LOCAL)
    return context * bf16 / (context * bytes_per_token(layout) + prot * bf16)
