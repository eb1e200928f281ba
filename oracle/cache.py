"""Model of the paged low-bit cache with bf16 sink and recent buffers.

QuantMLA, Figure 8 caption: the fused writer makes a packed copy of every
incoming token and keeps the pre-quantisation bf16 values of the protected
sink and recent tokens in dedicated buffers; attention reads those bf16 values
for protected tokens and the dequantised packed values for all others; a token
leaving the recent window switches to the packed copy it already has, with no
second quantisation.  Figure 5 and Table 9 fix the policy as sink 4 / local 128.

Readings adopted where the pages are silent:

* the window counts the token just written: with ``L`` tokens held, token ``t``
  is protected iff ``t < 4`` or ``t >= L - 128``;
* for ``L <= 132`` every token is protected (the two rules overlap);
* sink tokens get packed copies too (the writer packs all tokens alike);
* the recent buffer is a ring of 128 rows indexed by ``pos mod 128``; within one
  write call a token reaches the ring only if it is among the last 128 of its
  sequence after the call, so a bulk prefill leaves the same ring as
  token-by-token writes.

Page geometry: ``oracle.layout``.  Logical token ``pos`` of sequence ``b`` lives
in page ``block_table[b][pos // 64]`` at row ``pos % 64``.
"""

from __future__ import annotations

import numpy as np

from .layout import LATENT, LOCAL, PAGE_TOKENS, ROPE, SINK, Layout, page_geometry
from .quant import (bf16_bits_to_f64, dequantize, pack_codes, quantize_token, rotate_latent_bits,
                    unpack_codes)


def is_protected(t: np.ndarray, L: int) -> np.ndarray:
    t = np.asarray(t)
    return (t < SINK) | (t >= L - LOCAL)


class PagedCacheModel:
    """Byte-level model of the page pool and the bf16 buffers."""

    def __init__(self, layout: Layout, num_pages: int, block_table: np.ndarray):
        self.layout = layout
        self.geom = page_geometry(layout)
        self.block_table = np.asarray(block_table, dtype=np.int64)
        self.num_seqs = self.block_table.shape[0]
        self.pool = np.zeros((num_pages, self.geom["page_bytes"]), dtype=np.uint8)
        self.sink = np.zeros((self.num_seqs, SINK, LATENT + ROPE), dtype=np.uint16)
        self.recent = np.zeros((self.num_seqs, LOCAL, LATENT + ROPE), dtype=np.uint16)

    def _rows(self, seq, pos):
        page = self.block_table[seq, pos // PAGE_TOKENS]
        if np.any(page < 0) or np.any(page >= self.pool.shape[0]):
            raise IndexError("block table entry out of range")
        return page, pos % PAGE_TOKENS

    def write(self, seq, pos, ckv_bits, krope_bits, lens_after):
        """Write tokens ``ckv_bits[i], krope_bits[i]`` at ``(seq[i], pos[i])``.

        ``lens_after[b]`` is sequence b's length once this call is done; it
        decides which tokens reach the recent ring.
        """
        seq = np.asarray(seq, dtype=np.int64)
        pos = np.asarray(pos, dtype=np.int64)
        ckv_bits = np.asarray(ckv_bits, dtype=np.uint16).reshape(-1, LATENT)
        krope_bits = np.asarray(krope_bits, dtype=np.uint16).reshape(-1, ROPE)
        lens_after = np.asarray(lens_after, dtype=np.int64)
        page, row = self._rows(seq, pos)
        g = self.geom
        lay = self.layout
        if lay.rotate:
            # the token is stored (packed and bf16 copies alike) in the rotated basis
            ckv_bits = rotate_latent_bits(ckv_bits)
        if lay.packed:
            cc, rc, s16, m16 = quantize_token(ckv_bits, krope_bits, lay.content_bits,
                                              lay.rope_bits)
            cbytes = pack_codes(cc, lay.content_bits)
            rbytes = pack_codes(rc, lay.rope_bits)
            meta = np.stack([s16, m16], axis=-1).reshape(-1, 18)
            meta_bytes = np.ascontiguousarray(meta).view(np.uint8).reshape(-1, 36)
            for off, width, data in (("content_off", "content_row", cbytes),
                                     ("rope_off", "rope_row", rbytes),
                                     ("meta_off", "meta_row", meta_bytes)):
                cols = g[off] + row[:, None] * g[width] + np.arange(g[width])[None, :]
                self.pool[page[:, None], cols] = data
            tok16 = np.concatenate([ckv_bits, krope_bits], axis=1)
            sink = pos < SINK
            self.sink[seq[sink], pos[sink]] = tok16[sink]
            ring = pos >= lens_after[seq] - LOCAL
            self.recent[seq[ring], pos[ring] % LOCAL] = tok16[ring]
        else:
            tok = np.ascontiguousarray(np.concatenate([ckv_bits, krope_bits], axis=1))
            tok = tok.view(np.uint8)
            cols = row[:, None] * g["row_bytes"] + np.arange(g["row_bytes"])[None, :]
            self.pool[page[:, None], cols] = tok

    def token_bytes(self, seq: int, pos: int) -> bytes:
        """All packed bytes (codes + metadata) of one token, for change detection."""
        page, row = self._rows(np.int64(seq), np.int64(pos))
        g = self.geom
        if not self.layout.packed:
            a = row * g["row_bytes"]
            return self.pool[page, a:a + g["row_bytes"]].tobytes()
        parts = []
        for off, width in (("content_off", "content_row"), ("rope_off", "rope_row"),
                           ("meta_off", "meta_row")):
            a = g[off] + row * g[width]
            parts.append(self.pool[page, a:a + g[width]].tobytes())
        return b"".join(parts)

    def dequantized_keys(self, seq: int, L: int) -> np.ndarray:
        """Dequantised packed copies of tokens ``0..L-1`` (float64 ``[L][576]``)."""
        g = self.geom
        lay = self.layout
        n_pages = (L + PAGE_TOKENS - 1) // PAGE_TOKENS
        pages = self.block_table[seq, :n_pages]
        if not lay.packed:
            rows = self.pool[pages].reshape(n_pages * PAGE_TOKENS, -1)[:L]
            return bf16_bits_to_f64(rows.view(np.uint16))
        pg = self.pool[pages]
        cb = pg[:, g["content_off"]:g["rope_off"]].reshape(-1, g["content_row"])[:L]
        rb = pg[:, g["rope_off"]:g["meta_off"]].reshape(-1, g["rope_row"])[:L]
        mb = pg[:, g["meta_off"]:].reshape(-1, g["meta_row"])[:L]
        meta = np.ascontiguousarray(mb).view(np.float16).reshape(L, 9, 2)
        codes = np.concatenate([unpack_codes(cb, lay.content_bits),
                                unpack_codes(rb, lay.rope_bits)], axis=1)
        return dequantize(codes, meta[..., 0], meta[..., 1])

    def effective_keys(self, seq: int, L: int) -> np.ndarray:
        """Keys attention sees for ``L`` tokens: bf16 buffers for protected
        tokens, dequantised packed copies otherwise (float64 ``[L][576]``)."""
        keys = self.dequantized_keys(seq, L)
        if not self.layout.packed:
            return keys
        t = np.arange(L)
        for i in t[is_protected(t, L)]:
            if i < SINK:
                keys[i] = bf16_bits_to_f64(self.sink[seq, i])
            else:
                keys[i] = bf16_bits_to_f64(self.recent[seq, i % LOCAL])
        return keys


def reference_keys(ckv_bits: np.ndarray, krope_bits: np.ndarray, L: int,
                   layout: Layout) -> np.ndarray:
    """Effective keys straight from the definition, without the page model:
    bf16 input for protected tokens, quantise-then-dequantise otherwise."""
    ckv_bits = np.asarray(ckv_bits, dtype=np.uint16)[:L]
    krope_bits = np.asarray(krope_bits, dtype=np.uint16)[:L]
    exact = np.concatenate([bf16_bits_to_f64(ckv_bits), bf16_bits_to_f64(krope_bits)], axis=1)
    if not layout.packed:
        return exact
    cc, rc, s16, m16 = quantize_token(ckv_bits, krope_bits, layout.content_bits,
                                      layout.rope_bits)
    deq = dequantize(np.concatenate([cc, rc], axis=1), s16, m16)
    prot = is_protected(np.arange(L), L)
    deq[prot] = exact[prot]
    return deq
