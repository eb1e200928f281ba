"""Per-token asymmetric group quantisation, packing and dequantisation.

QuantMLA (Abstract) caches the content latent at INT4 or INT2 and the RoPE key
at INT4; the Figure 8 caption has the fused writer pack a low-bit copy of
every incoming token.  The pages do not fix the quantiser; the adopted
definition (an RTN-style asymmetric quantiser, named as a baseline in Table 3)
is, per token and per 64-channel group, in this order:

1. ``mn, mx`` = min and max of the group's bf16 values (exact in float32); a
   zero minimum is taken as +0, so the stored fp16 min never holds -0;
2. ``s32 = float32(mx - mn) / float32(2**bits - 1)`` (IEEE float32, nearest);
3. ``s16 = fp16(s32)``, ``m16 = fp16(mn)``: nearest-even, saturating at +-65504;
4. ``r = float32(x - float32(m16)) / float32(s16)`` (two float32 operations,
   each rounded to nearest; a true division, no reciprocal, no fused op);
5. ``code = clamp(round_half_even(r), 0, 2**bits - 1)``; every code is 0 when
   ``s16 == 0``;
6. dequantised value ``x_hat = float64(s16) * code + float64(m16)`` (exact).

Inputs with ``|x| > 65504`` are outside the contract (the fp16 metadata cannot
hold them) and raise.
"""

from __future__ import annotations

import numpy as np

F16_MAX = 65504.0


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    bits = np.ascontiguousarray(bits, dtype=np.uint16)
    return (bits.astype(np.uint32) << 16).view(np.float32)


def bf16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    return bf16_bits_to_f32(bits).astype(np.float64)


def f16_satfinite(x32: np.ndarray) -> np.ndarray:
    """float32 -> fp16, round to nearest even, finite values saturate to +-65504."""
    x32 = np.asarray(x32, dtype=np.float32)
    return np.clip(x32, np.float32(-F16_MAX), np.float32(F16_MAX)).astype(np.float16)


def quantize_group(x_bits: np.ndarray, bits: int):
    """Quantise groups of bf16 values along the last axis.

    ``x_bits``: uint16 bf16 bit patterns ``[..., G]``.
    Returns ``(codes uint8 [..., G], scale fp16 [...], min fp16 [...])``.
    """
    x = bf16_bits_to_f32(x_bits)
    if np.any(~np.isfinite(x)) or np.any(np.abs(x) > F16_MAX):
        raise ValueError("input outside the fp16 metadata range (|x| > 65504)")
    levels = np.float32(2 ** bits - 1)
    mn = x.min(axis=-1) + np.float32(0.0)   # -0 + 0 = +0 under round-to-nearest
    mx = x.max(axis=-1)
    s32 = np.subtract(mx, mn, dtype=np.float32) / levels
    s16 = f16_satfinite(s32)
    m16 = f16_satfinite(mn)
    s_f = s16.astype(np.float32)[..., None]
    m_f = m16.astype(np.float32)[..., None]
    diff = np.subtract(x, m_f, dtype=np.float32)
    with np.errstate(divide="ignore", invalid="ignore"):
        r = np.divide(diff, s_f, dtype=np.float32)
    r = np.where(s_f == 0, np.float32(0), r)
    codes = np.clip(np.rint(r), 0, levels).astype(np.uint8)
    return codes, s16, m16


def quantize_token(ckv_bits: np.ndarray, krope_bits: np.ndarray, content_bits: int,
                   rope_bits: int):
    """Quantise tokens ``[..., 512]`` + ``[..., 64]`` into 9 groups.

    Returns ``(content codes [..., 512], rope codes [..., 64], scale fp16 [..., 9],
    min fp16 [..., 9])`` with groups 0..7 content and 8 RoPE.
    """
    lead = ckv_bits.shape[:-1]
    cg = ckv_bits.reshape(lead + (8, 64))
    c_codes, c_s, c_m = quantize_group(cg, content_bits)
    r_codes, r_s, r_m = quantize_group(krope_bits, rope_bits)
    scale = np.concatenate([c_s, r_s[..., None]], axis=-1)
    mins = np.concatenate([c_m, r_m[..., None]], axis=-1)
    return c_codes.reshape(lead + (512,)), r_codes, scale, mins


def pack_codes(codes: np.ndarray, bits: int) -> np.ndarray:
    """Pack codes along the last axis: channel ``k*i + j`` goes to bits
    ``bits*j .. bits*j + bits - 1`` of byte ``i`` (k = 8 / bits)."""
    codes = np.asarray(codes, dtype=np.uint8)
    per = 8 // bits
    n = codes.shape[-1]
    assert n % per == 0
    out = np.zeros(codes.shape[:-1] + (n // per,), dtype=np.uint8)
    for j in range(per):
        out |= (codes[..., j::per] << (bits * j)).astype(np.uint8)
    return out


def unpack_codes(packed: np.ndarray, bits: int) -> np.ndarray:
    packed = np.asarray(packed, dtype=np.uint8)
    per = 8 // bits
    mask = (1 << bits) - 1
    out = np.empty(packed.shape[:-1] + (packed.shape[-1] * per,), dtype=np.uint8)
    for j in range(per):
        out[..., j::per] = (packed >> (bits * j)) & mask
    return out


def dequantize(codes: np.ndarray, scale16: np.ndarray, min16: np.ndarray) -> np.ndarray:
    """``x_hat = s16 * code + m16`` in float64 (exact); groups of 64 along the last axis."""
    lead = codes.shape[:-1]
    n = codes.shape[-1]
    g = codes.reshape(lead + (n // 64, 64)).astype(np.float64)
    s = scale16.astype(np.float64)[..., None]
    m = min16.astype(np.float64)[..., None]
    return (s * g + m).reshape(lead + (n,))


# ---------------------------------------------------------------- online rotation
# QuaRot-style online rotation of the content latent (QuantMLA, Table 1: QuaRot
# as an MLA-adapted baseline; the pages' own transforms are fused offline).
# Adopted reading for an un-fused model: each 64-channel content group x is
# replaced, as it is written, by R x with R = H_64 / 8 the orthonormal
# Sylvester-Hadamard matrix (R symmetric, R R = I), computed in float32 and
# rounded to bf16; queries are rotated the same way and attention outputs
# rotated back, so attention sees the same inner products.  RoPE keys are not
# rotated.

def hadamard_matrix64() -> np.ndarray:
    """R = H_64 / 8 in float64: R[i][j] = (-1)^popcount(i & j) / 8."""
    i = np.arange(64)
    pc = np.vectorize(lambda v: bin(v).count("1"))(i[:, None] & i[None, :])
    return np.where(pc % 2 == 0, 1.0, -1.0) / 8.0


def hadamard_rotate_f32(x: np.ndarray) -> np.ndarray:
    """R x for groups of 64 along the last axis, in float32 with a fixed order of
    operations: butterfly stages h = 1, 2, 4, ..., 32, where element i (bit h
    clear) and element i + h become (a + b, a - b); then a scale by 1/8 (exact)."""
    y = np.array(x, dtype=np.float32, copy=True)
    h = 1
    while h < 64:
        lo = np.array([i for i in range(64) if not i & h])
        a = y[..., lo].copy()
        b = y[..., lo + h].copy()
        y[..., lo] = a + b
        y[..., lo + h] = a - b
        h *= 2
    return y * np.float32(0.125)


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 to bf16 (nearest, ties to even); finite inputs only."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    return ((u + 0x7FFF + ((u >> 16) & 1)) >> 16).astype(np.uint16)


def rotate_latent_bits(ckv_bits: np.ndarray) -> np.ndarray:
    """The rotated content latent as bf16 bits: the 8 groups of ``[..., 512]``
    each rotated by R (float32) and rounded to bf16."""
    x = bf16_bits_to_f32(ckv_bits)
    lead = x.shape[:-1]
    y = hadamard_rotate_f32(x.reshape(lead + (8, 64))).reshape(lead + (512,))
    return f32_to_bf16_bits(y)
