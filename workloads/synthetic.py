"""Synthetic decode workloads with the shapes and value distributions of the
low-bit MLA decode benchmarks (QuantMLA: Function-Aligned Dual-Path
Quantization for Low-Bit MLA KV Caching -- Figure 5 and Table 9 describe the
decode measurements; the shapes follow DeepSeek-V2-Lite and DeepSeek-V3).

Recipe (every draw comes from ``numpy.random.default_rng`` on children of one
``SeedSequence(seed)``, so any single sequence can be regenerated alone):

* child 0: per-channel latent scales, ``lognormal(0, 0.5)`` for the 512 content
  channels, then 4 outlier channels (drawn without replacement) times 10;
* child 1: context lengths (fixed, integer-uniform or log-uniform);
* child 2: the physical page permutation of the paged cache;
* child 3 + b: sequence b, itself split into (tokens, queries).
  Content latents are ``N(0,1) * scale[channel]``; RoPE keys are ``N(0,1)``
  pairs ``(a, b)`` for the adjacent channels ``(2i, 2i+1)``, rotated by
  ``pos * 10000**(-2i/64)``; queries are ``N(0,1)``.  All three are rounded to
  bf16 (round to nearest even) and handed out as ``uint16`` bit patterns.

The module only draws numbers: it contains no quantisation and no attention.
"""

from __future__ import annotations

import dataclasses
import math
from typing import Optional, Sequence, Tuple

import numpy as np

LATENT = 512
ROPE = 64
QK_DIM = LATENT + ROPE
PAGE_TOKENS = 64
ROPE_THETA = 10000.0


def bf16_bits_from_f32(x: np.ndarray) -> np.ndarray:
    """Round float32 values to bf16 (nearest, ties to even); return uint16 bits."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    u = x.view(np.uint32).astype(np.uint64)
    u = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    return u.astype(np.uint16)


def f32_from_bf16_bits(bits: np.ndarray) -> np.ndarray:
    """Widen bf16 bit patterns to float32 (exact)."""
    bits = np.ascontiguousarray(bits, dtype=np.uint16)
    return (bits.astype(np.uint32) << 16).view(np.float32)


@dataclasses.dataclass(frozen=True)
class Workload:
    """One decode workload.

    ``lengths`` holds each sequence's context length after the first decode
    step's append; step ``s`` (0-based) decodes over ``L_b + s`` tokens after
    writing the token at position ``L_b + s - 1``.
    """

    name: str
    batch: int
    heads: int
    length_kind: str              # "fixed" | "uniform" | "loguniform" | "explicit"
    length_args: Tuple[int, ...]  # (L,) | (lo, hi) | (lo, hi) | explicit lengths
    content_bits: int             # 4, 2 or 16 (bf16 pages)
    rope_bits: int                # 4 or 16
    steps: int = 1                # decode steps, each appending one token per sequence
    seed: int = 0
    writer_in_step: bool = False  # the timed step also runs the cache writer
    softmax_scale: float = 1.0 / math.sqrt(192.0)
    # Global indices of this workload's sequences in the batch they were drawn
    # from (a rank's shard); None means sequence b is global sequence b.  Token
    # and query draws follow the global index, so a shard holds exactly the
    # values its sequences have in the global batch.
    seq_ids: Optional[Tuple[int, ...]] = None

    def with_(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)


WORKLOADS = {
    # B1 H16 L1024 C4R4, the small case the oracle finishes in seconds.
    "tiny_c4r4": Workload("tiny_c4r4", 1, 16, "fixed", (1024,), 4, 4, 1, 0),
    # DeepSeek-V2-Lite-shaped: B8 H16 L32768, writer + decode each step.
    "v2lite_c4r4": Workload("v2lite_c4r4", 8, 16, "fixed", (32768,), 4, 4, 1, 1,
                            writer_in_step=True),
    # DeepSeek-V3-shaped: B32, 128 heads sharing one latent, L ~ U{4096..16384}.
    "v3_c4r4": Workload("v3_c4r4", 32, 128, "uniform", (4096, 16384), 4, 4, 1, 2),
    # Long context, 128 heads, packed vs bf16 pages on the same values.
    "long_c4r4": Workload("long_c4r4", 4, 128, "fixed", (131072,), 4, 4, 1, 3),
    "long_bf16": Workload("long_bf16", 4, 128, "fixed", (131072,), 16, 16, 1, 3),
    # Long context with 16 heads (the HBM-bound variant of the same cache).
    "long16_c4r4": Workload("long16_c4r4", 4, 16, "fixed", (131072,), 4, 4, 1, 3),
    "long16_bf16": Workload("long16_bf16", 4, 16, "fixed", (131072,), 16, 16, 1, 3),
    # Mixed precision C2R4: B64 H16, L log-uniform in [1024, 131072], 16 steps.
    "mixed_c2r4": Workload("mixed_c2r4", 64, 16, "loguniform", (1024, 131072), 2, 4, 16, 4,
                           writer_in_step=True),
}


def get(name: str) -> Workload:
    return WORKLOADS[name]


def layout_of(w: Workload) -> dict:
    return dict(content_bits=w.content_bits, rope_bits=w.rope_bits, group=64,
                sink=4, local=128, page_tokens=PAGE_TOKENS, latent=LATENT, rope=ROPE)


def _children(w: Workload):
    return np.random.SeedSequence(w.seed).spawn(3 + w.batch)


def channel_scales(w: Workload) -> np.ndarray:
    rng = np.random.default_rng(_children(w)[0])
    scale = rng.lognormal(0.0, 0.5, LATENT)
    outliers = rng.choice(LATENT, 4, replace=False)
    scale[outliers] *= 10.0
    return scale.astype(np.float32)


def sequence_lengths(w: Workload) -> np.ndarray:
    """Context length of each sequence after the first step's append."""
    rng = np.random.default_rng(_children(w)[1])
    if w.length_kind == "fixed":
        lens = np.full(w.batch, w.length_args[0], dtype=np.int64)
    elif w.length_kind == "uniform":
        lo, hi = w.length_args
        lens = rng.integers(lo, hi + 1, size=w.batch)
    elif w.length_kind == "loguniform":
        lo, hi = w.length_args
        lens = np.rint(np.exp(rng.uniform(math.log(lo), math.log(hi), size=w.batch)))
        lens = np.clip(lens, lo, hi).astype(np.int64)
    elif w.length_kind == "explicit":
        lens = np.asarray(w.length_args, dtype=np.int64)
        assert lens.shape == (w.batch,)
    else:
        raise ValueError(w.length_kind)
    return lens.astype(np.int64)


def tokens_per_sequence(w: Workload) -> np.ndarray:
    """Tokens each sequence holds after the last step."""
    return sequence_lengths(w) + (w.steps - 1)


def make_paging(w: Workload, spare_pages: int = 0):
    """Random physical page ids for each sequence.

    Returns ``(block_table [B][max_pages] int32, num_pages)``; entries past a
    sequence's last page are -1.
    """
    n_tok = tokens_per_sequence(w)
    n_pages = (n_tok + PAGE_TOKENS - 1) // PAGE_TOKENS
    total = int(n_pages.sum()) + spare_pages
    rng = np.random.default_rng(_children(w)[2])
    perm = rng.permutation(total).astype(np.int32)
    max_pages = max(int(n_pages.max()), 1)
    table = np.full((w.batch, max_pages), -1, dtype=np.int32)
    off = 0
    for b in range(w.batch):
        k = int(n_pages[b])
        table[b, :k] = perm[off:off + k]
        off += k
    return table, total


def _seq_streams(w: Workload, b: int):
    g = b if w.seq_ids is None else int(w.seq_ids[b])
    return np.random.SeedSequence(w.seed).spawn(3 + g + 1)[3 + g].spawn(2)


def sequence_tokens(w: Workload, b: int, n_tokens: Optional[int] = None,
                    scales: Optional[np.ndarray] = None):
    """bf16 bits of sequence b's tokens at positions 0..n_tokens-1.

    Returns ``(ckv [n][512] uint16, krope [n][64] uint16)``.  The draw always
    covers every token the sequence will hold, so the values at a position do
    not depend on ``n_tokens``.
    """
    total = int(tokens_per_sequence(w)[b])
    n = total if n_tokens is None else int(n_tokens)
    assert 0 <= n <= total
    if scales is None:
        scales = channel_scales(w)
    rng = np.random.default_rng(_seq_streams(w, b)[0])
    lat = rng.standard_normal((total, LATENT), dtype=np.float32)[:n]
    lat *= scales[None, :]
    ckv = bf16_bits_from_f32(lat)
    del lat
    ab = rng.standard_normal((total, 2, ROPE // 2), dtype=np.float32)[:n]
    pos = np.arange(n, dtype=np.float64)[:, None]
    inv_freq = ROPE_THETA ** (-2.0 * np.arange(ROPE // 2, dtype=np.float64) / ROPE)
    ang = pos * inv_freq[None, :]
    cos, sin = np.cos(ang), np.sin(ang)
    a = ab[:, 0, :].astype(np.float64)
    bb = ab[:, 1, :].astype(np.float64)
    rot = np.empty((n, ROPE), dtype=np.float32)
    rot[:, 0::2] = a * cos - bb * sin
    rot[:, 1::2] = a * sin + bb * cos
    krope = bf16_bits_from_f32(rot)
    return ckv, krope


def queries(w: Workload, b: int) -> np.ndarray:
    """bf16 bits of sequence b's absorbed queries for every step: [steps][H][576]."""
    rng = np.random.default_rng(_seq_streams(w, b)[1])
    q = rng.standard_normal((w.steps, w.heads, QK_DIM), dtype=np.float32)
    return bf16_bits_from_f32(q)


def shard_workload(w: Workload, rank: int, world: int) -> Workload:
    """Rank ``rank``'s shard of the global batch of ``world * w.batch`` sequences
    drawn from ``w``'s recipe: global sequence g goes to rank g mod world, so
    every sequence is decoded by exactly one rank and ranks share nothing (no
    data-path exchange).  The shard keeps the global lengths and values of its
    sequences; its page pool and block table are its own.  With world == 1 the
    shard is ``w`` itself (same lengths, values and paging)."""
    if world < 1 or not 0 <= rank < world:
        raise ValueError(f"rank {rank} of {world}")
    glob = w.with_(batch=w.batch * world)
    if world > 1 and w.length_kind == "explicit":
        raise ValueError("explicit lengths name one batch; shard a recipe workload")
    lens = sequence_lengths(glob)
    ids = tuple(g for g in range(glob.batch) if g % world == rank)
    return w.with_(batch=len(ids), length_kind="explicit",
                   length_args=tuple(int(lens[g]) for g in ids), seq_ids=ids)


def custom(name: str, lengths: Sequence[int], heads: int = 16, content_bits: int = 4,
           rope_bits: int = 4, steps: int = 1, seed: int = 0) -> Workload:
    """A small workload with explicit lengths (for tests)."""
    lengths = tuple(int(x) for x in lengths)
    return Workload(name, len(lengths), heads, "explicit", lengths, content_bits, rope_bits,
                    steps, seed)


def device_tokens(n: int, seed: int, device, start_pos: int = 0):
    """Seeded bf16 tokens generated on a torch device, for timing sweeps whose
    sizes make host generation too slow (up to millions of tokens per
    sequence).  Same recipe as ``sequence_tokens`` (lognormal(0, 0.5)
    per-channel latent scales with 4 outlier channels x 10; N(0,1) RoPE pairs
    rotated by ``pos * 10000**(-2i/64)``), drawn with torch's generator, so
    the values differ from the host generator's.  Returns ``(ckv [n][512],
    krope [n][64])`` as torch bf16 tensors.  Nothing checks these values
    against the oracle; they only give the cache realistic statistics."""
    import torch
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    scale = torch.exp(0.5 * torch.randn(LATENT, generator=g, device=device))
    outliers = torch.randperm(LATENT, generator=g, device=device)[:4]
    scale[outliers] *= 10.0
    ckv = (torch.randn(n, LATENT, generator=g, device=device) * scale).to(torch.bfloat16)
    ab = torch.randn(n, 2, ROPE // 2, generator=g, device=device)
    pos = torch.arange(start_pos, start_pos + n, device=device, dtype=torch.float64)[:, None]
    inv_freq = ROPE_THETA ** (-2.0 * torch.arange(ROPE // 2, device=device, dtype=torch.float64) / ROPE)
    ang = pos * inv_freq[None, :]
    cos, sin = torch.cos(ang), torch.sin(ang)
    a, b = ab[:, 0, :].double(), ab[:, 1, :].double()
    rot = torch.empty(n, ROPE, device=device, dtype=torch.float32)
    rot[:, 0::2] = (a * cos - b * sin).float()
    rot[:, 1::2] = (a * sin + b * cos).float()
    return ckv, rot.to(torch.bfloat16)
