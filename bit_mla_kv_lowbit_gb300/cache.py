"""Device-side state of one paged low-bit MLA cache, allocated with PyTorch.

PyTorch supplies the memory and the stream; every computation is a call into
the C ABI through ``binding``.
"""

from __future__ import annotations

from typing import Optional, Sequence

import numpy as np

from . import binding


class PagedCache:
    """Page pool, bf16 sink/recent buffers, block table and device error word."""

    def __init__(self, content_bits: int, rope_bits: int, block_table, num_pages: int,
                 device: str = "cuda", rotate: bool = False):
        import torch
        self.torch = torch
        self.layout = binding.layout(content_bits, rope_bits, rotate)
        self.page_bytes = binding.page_bytes(self.layout)
        bt = torch.as_tensor(np.asarray(block_table, dtype=np.int32))
        self.block_table = bt.to(device).contiguous()
        self.num_seqs, self.max_pages = self.block_table.shape
        self.pool = torch.zeros(num_pages, self.page_bytes, dtype=torch.uint8, device=device)
        packed = content_bits != 16
        self.sink = (torch.zeros(self.num_seqs, 4, 576, dtype=torch.bfloat16, device=device)
                     if packed else None)
        self.recent = (torch.zeros(self.num_seqs, 128, 576, dtype=torch.bfloat16, device=device)
                       if packed else None)
        self.err = torch.zeros(1, dtype=torch.int32, device=device)
        self.device = device
        self._ws = None

    def write(self, ckv, krope, pos, seq_idx=None, seq_lens_after=None, stream=None):
        binding.write(self.layout, ckv, krope, pos, self.block_table, self.pool, self.sink,
                      self.recent, self.err, seq_idx=seq_idx, seq_lens_after=seq_lens_after,
                      stream=stream)

    def workspace(self, heads: int, seq_lens_host: Sequence[int]):
        _, _, nbytes = binding.decode_plan(self.layout, heads, seq_lens_host)
        nbytes = max(int(nbytes), 16)
        if self._ws is None or self._ws.numel() < nbytes:
            self._ws = self.torch.empty(nbytes, dtype=self.torch.uint8, device=self.device)
        return self._ws

    def decode(self, q, seq_lens, seq_lens_host, softmax_scale: float, out=None, lse=None,
               workspace=None, stream=None):
        torch = self.torch
        B, H, _ = q.shape
        if out is None:
            out = torch.empty(B, H, 512, dtype=torch.float32, device=self.device)
        if workspace is None:
            workspace = self.workspace(H, seq_lens_host)
        binding.decode(self.layout, q, self.pool, self.block_table, seq_lens, seq_lens_host,
                       self.sink, self.recent, out, workspace, self.err, softmax_scale, lse=lse,
                       stream=stream)
        return out

    def write_decode(self, ckv_new, krope_new, q, seq_lens, seq_lens_host, softmax_scale: float,
                     out=None, lse=None, workspace=None, stream=None):
        """Append one token per sequence (at position seq_lens[s] - 1) and decode."""
        torch = self.torch
        B, H, _ = q.shape
        if out is None:
            out = torch.empty(B, H, 512, dtype=torch.float32, device=self.device)
        if workspace is None:
            workspace = self.workspace(H, seq_lens_host)
        binding.write_decode(self.layout, q, ckv_new, krope_new, self.pool, self.block_table,
                             seq_lens, seq_lens_host, self.sink, self.recent, out, workspace,
                             self.err, softmax_scale, lse=lse, stream=stream)
        return out

    def decode_multi(self, q, seq_lens, seq_lens_host, softmax_scale: float, out=None, lse=None,
                     workspace=None, stream=None):
        """n causal queries per sequence (q [B][n][H][576]) over the cache."""
        torch = self.torch
        B, n, H, _ = q.shape
        if out is None:
            out = torch.empty(B, n, H, 512, dtype=torch.float32, device=self.device)
        if workspace is None:
            workspace = self.workspace(n * H, seq_lens_host)
        binding.decode_multi(self.layout, q, self.pool, self.block_table, seq_lens, seq_lens_host,
                             self.sink, self.recent, out, workspace, self.err, softmax_scale,
                             lse=lse, stream=stream)
        return out

    def error(self) -> int:
        return binding.read_error(self.err)

    def clear_error(self):
        self.err.zero_()
