"""MLA decode attention in absorbed form, float64.

QuantMLA (Abstract; Figure 8 caption): one query attends to every cached
token of its sequence; the cached key is the content latent (512) followed by
the decoupled RoPE key (64); the reconstructed content latent serves both the
matching (QK) and the latent aggregation (PV) -- the value is the key's first
512 channels -- and every valid token shares one softmax normalisation.

Adopted readings: the query is already absorbed (``q_nope @ W_UK`` next to the
rotated ``q_pe``), so the output stays in latent space ``[H][512]`` with no
up-projection; the softmax scale is given by the caller (1/sqrt(192) in the
workloads).
"""

from __future__ import annotations

import numpy as np

from .quant import bf16_bits_to_f64, hadamard_matrix64


def _rotate_groups(x: np.ndarray) -> np.ndarray:
    """R applied to each 64-channel group of ``[..., 512]`` (float64, R = R^T)."""
    R = hadamard_matrix64()
    lead = x.shape[:-1]
    return (x.reshape(lead + (8, 64)) @ R.T).reshape(lead + (512,))


def mla_decode_fp64(q_bits: np.ndarray, keys: np.ndarray, softmax_scale: float,
                    rotate: bool = False):
    """Softmax attention of ``H`` heads over ``L`` keys.

    ``q_bits``: bf16 bits ``[H][576]``; ``keys``: float64 ``[L][576]``.
    Returns ``(out [H][512] float64, lse [H] float64)`` where ``lse`` is the
    natural-log sum of ``exp(logit)``.  With ``L == 0`` the output is zero and
    ``lse`` is ``-inf``.

    ``rotate``: the keys' content channels are in the rotated basis of an
    online-rotated cache (``quant.rotate_latent_bits``); the query's content
    channels are rotated by the same R and the output rotated back, so the
    logits are ``q . R^T k'`` and the output ``R^T sum p k'``.
    """
    q = bf16_bits_to_f64(q_bits)
    keys = np.asarray(keys, dtype=np.float64)
    H = q.shape[0]
    L = keys.shape[0]
    if L == 0:
        return np.zeros((H, 512)), np.full(H, -np.inf)
    if rotate:
        q = q.copy()
        q[:, :512] = _rotate_groups(q[:, :512])
    z = float(softmax_scale) * (q @ keys.T)          # [H][L]
    zmax = z.max(axis=1, keepdims=True)
    e = np.exp(z - zmax)
    denom = e.sum(axis=1)
    out = (e @ keys[:, :512]) / denom[:, None]
    if rotate:
        out = _rotate_groups(out)
    lse = zmax[:, 0] + np.log(denom)
    return out, lse


def mla_decode_multi_fp64(q_bits: np.ndarray, keys: np.ndarray, softmax_scale: float,
                          rotate: bool = False):
    """Several queries of one sequence decoded in one step, causally.

    Group-Query Latent Attention abstract (Shi, Meng, Zhang): multi-token
    prediction decodes s_q = 2 query tokens per step on the same latent cache
    that the absorbed path reads with s_q = 1.  Adopted reading: the ``n``
    queries are the sequence's last ``n`` tokens (positions ``L - n .. L - 1``,
    all already cached), and query ``i`` attends to the tokens up to and
    including its own position, ``keys[: L - n + i + 1]`` -- ordinary causal
    attention, each query exactly ``mla_decode_fp64`` over its prefix.

    ``q_bits``: bf16 bits ``[n][H][576]``; ``keys``: float64 ``[L][576]``
    with ``L >= n``.  Returns ``(out [n][H][512], lse [n][H])``.
    """
    q_bits = np.asarray(q_bits)
    n = q_bits.shape[0]
    L = np.asarray(keys).shape[0]
    assert L >= n, "the queries' own tokens must be cached"
    outs, lses = [], []
    for i in range(n):
        o, l = mla_decode_fp64(q_bits[i], np.asarray(keys)[: L - n + i + 1], softmax_scale,
                               rotate=rotate)
        outs.append(o)
        lses.append(l)
    return np.stack(outs), np.stack(lses)
