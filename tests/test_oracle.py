"""Pins for the CPU oracle: closed forms, IEEE facts, brute force, invariants.

None of these checks re-types the oracle's own formula: each compares it with
something the definition or the mathematics fixes independently (hand-derived
values, textbook rounding facts, exact grids, constant-logit and one-hot
attention, loops without max-subtraction, torch's fp64 attention).
"""

import math

import numpy as np
import pytest

import oracle
from oracle import Layout, PagedCacheModel
from workloads import synthetic as syn

C4R4 = Layout(4, 4)
C2R4 = Layout(2, 4)
BF16 = Layout(16, 16)


def bf16(x):
    return syn.bf16_bits_from_f32(np.asarray(x, dtype=np.float32))


# ---------------------------------------------------------------- fp16 rounding

@pytest.mark.parametrize("x, want", [
    (1.0 + 2.0 ** -11, 1.0),                     # tie -> even mantissa (down)
    (1.0 + 3 * 2.0 ** -11, 1.0 + 2.0 ** -9),     # tie -> even mantissa (up)
    (1.0 + 2.0 ** -11 + 2.0 ** -20, 1.0 + 2.0 ** -10),  # above the tie -> up
    (65504.0, 65504.0),
    (65519.0, 65504.0),                          # below the RNE overflow threshold
    (65520.0, 65504.0),                          # RNE would give inf; saturates
    (1.0e6, 65504.0),
    (-1.0e6, -65504.0),
    (2.0 ** -24, 2.0 ** -24),                    # smallest subnormal
    (2.0 ** -25, 0.0),                           # tie between 0 and 2^-24 -> 0 (even)
    (3 * 2.0 ** -26, 2.0 ** -24),
    (0.1, 0.0999755859375),                      # nearest fp16 to 0.1
])
def test_f16_satfinite_textbook(x, want):
    got = float(oracle.f16_satfinite(np.float32(x)))
    assert got == want


# ---------------------------------------------------------------- packing

def test_pack_bit_positions_by_hand():
    # INT4: channel 2i -> low nibble, 2i+1 -> high nibble.
    assert oracle.pack_codes(np.array([1, 2, 15, 0], np.uint8), 4).tolist() == [0x21, 0x0F]
    # INT2: channel 4i+j -> bits 2j..2j+1.
    assert oracle.pack_codes(np.array([1, 2, 3, 0], np.uint8), 2).tolist() == [0b00111001]


@pytest.mark.parametrize("bits", [2, 4])
def test_pack_unpack_roundtrip(bits):
    rng = np.random.default_rng(7)
    codes = rng.integers(0, 2 ** bits, size=(37, 512), dtype=np.uint8)
    packed = oracle.pack_codes(codes, bits)
    assert packed.shape == (37, 512 * bits // 8)
    assert np.array_equal(oracle.unpack_codes(packed, bits), codes)


# ---------------------------------------------------------------- closed-form layout

def test_page_and_token_bytes_closed_form():
    assert oracle.page_geometry(C4R4)["page_bytes"] == 20736
    assert oracle.page_geometry(C2R4)["page_bytes"] == 12544
    assert oracle.page_geometry(BF16)["page_bytes"] == 73728
    assert oracle.bytes_per_token(BF16) == 1152
    assert oracle.bytes_per_token(C4R4) == 256 + 32 + 32 + 4
    assert oracle.bytes_per_token(C2R4) == 128 + 32 + 32 + 4
    for lay in (C4R4, C2R4):
        g = oracle.page_geometry(lay)
        for k in ("content_off", "rope_off", "meta_off", "page_bytes"):
            assert g[k] % 128 == 0
    assert oracle.compression_ratio(C4R4) == pytest.approx(1152 / 324)
    assert oracle.compression_ratio(C2R4) == pytest.approx(1152 / 196)
    n = 131072
    assert oracle.compression_ratio(C4R4, n) == pytest.approx(n * 1152 / (n * 324 + 132 * 1152))
    assert oracle.compression_ratio(C4R4, n) == pytest.approx(3.5428, abs=1e-4)
    assert oracle.compression_ratio(C2R4, n) == pytest.approx(5.8429, abs=1e-4)


# ---------------------------------------------------------------- quantiser

@pytest.mark.parametrize("bits", [2, 4])
def test_exact_grid_is_recovered(bits):
    levels = 2 ** bits - 1
    s, m = 0.25, -2.0   # fp16- and bf16-exact
    rng = np.random.default_rng(1)
    k = rng.integers(0, levels + 1, size=64)
    k[0], k[1] = 0, levels  # both ends present so (max-min)/levels == s exactly
    x = m + s * k
    codes, s16, m16 = oracle.quantize_group(bf16(x), bits)
    assert float(s16) == s and float(m16) == m
    assert np.array_equal(codes, k)
    assert np.array_equal(oracle.dequantize(codes[None], s16[None], m16[None])[0], x)


def test_ties_round_to_half_even():
    # s = 1, m = 0: r equals the value itself, so halves are exact ties.
    x = np.zeros(64, np.float32)
    x[1] = 15.0
    x[2:9] = [2.5, 3.5, 0.5, 1.5, 14.5, 7.5, 8.5]
    codes, s16, m16 = oracle.quantize_group(bf16(x), 4)
    assert float(s16) == 1.0 and float(m16) == 0.0
    assert codes[:9].tolist() == [0, 15, 2, 4, 0, 2, 14, 8, 8]


def test_constant_group_gives_zero_scale():
    x = np.full(64, 3.25, np.float32)
    codes, s16, m16 = oracle.quantize_group(bf16(x), 4)
    assert float(s16) == 0.0 and float(m16) == 3.25
    assert not codes.any()
    assert np.all(oracle.dequantize(codes[None], s16[None], m16[None]) == 3.25)


def test_hand_worked_group():
    # mn = -1, mx = 2: s32 = 3/15 = 0.2 (float32 0.2000000030), s16 = 0.199951171875,
    # m16 = -1; x = 0.5 -> r = 1.5 / 0.199951171875 = 7.5018... -> code 8.
    x = np.zeros(64, np.float32)
    x[0], x[1], x[2] = -1.0, 2.0, 0.5
    codes, s16, m16 = oracle.quantize_group(bf16(x), 4)
    assert float(s16) == 0.199951171875 and float(m16) == -1.0
    assert codes[:3].tolist() == [0, 15, 8]
    # x = 0 -> r = 1 / 0.199951171875 = 5.0012 -> 5
    assert codes[3] == 5


@pytest.mark.parametrize("bits", [2, 4])
def test_code_range_and_error_bound(bits):
    rng = np.random.default_rng(3)
    x = (rng.standard_normal((500, 64)) * np.exp(rng.normal(0, 2, (500, 1)))).astype(np.float32)
    xb = bf16(x)
    xf = syn.f32_from_bf16_bits(xb).astype(np.float64)
    codes, s16, m16 = oracle.quantize_group(xb, bits)
    assert codes.max() <= 2 ** bits - 1
    xh = oracle.dequantize(codes, s16[:, None], m16[:, None])
    mn, mx = xf.min(1), xf.max(1)
    s32 = (mx - mn) / (2 ** bits - 1)
    s = s16.astype(np.float64)
    m = m16.astype(np.float64)
    bound = s / 2 + np.abs(m - mn) + (2 ** bits - 1) * np.abs(s - s32) + 1e-6 * np.abs(xf).max(1)
    assert np.all(np.abs(xh - xf).max(1) <= bound)


def test_zero_minimum_is_stored_as_plus_zero():
    x = np.zeros(64, np.float32)
    x[3] = -0.0
    x[7] = 2.0
    codes, s16, m16 = oracle.quantize_group(bf16(x), 4)
    assert m16.view(np.uint16) == 0 and float(s16) == np.float16(2.0 / 15)


def test_out_of_contract_inputs_raise():
    x = np.zeros(64, np.float32)
    x[5] = 65536.0   # bf16-representable, beyond fp16
    with pytest.raises(ValueError):
        oracle.quantize_group(bf16(x), 4)


# ---------------------------------------------------------------- attention

def _tokens(L, seed=0, scale=1.0):
    rng = np.random.default_rng(seed)
    ckv = bf16(rng.standard_normal((L, 512)) * scale)
    kr = bf16(rng.standard_normal((L, 64)))
    return ckv, kr


def test_zero_query_gives_mean_of_values():
    L = 300
    ckv, kr = _tokens(L)
    keys = oracle.reference_keys(ckv, kr, L, C4R4)
    q = np.zeros((4, 576), np.uint16)
    out, lse = oracle.mla_decode_fp64(q, keys, 0.1)
    assert np.allclose(out, keys[:, :512].mean(0)[None], rtol=0, atol=1e-12)
    assert np.allclose(lse, math.log(L))


def test_equal_logits_from_grid_exact_rope_keys():
    # Content query zero, every rope key the same grid-exact vector: all logits
    # equal even though most tokens are dequantised, so out = mean of values.
    L = 400
    ckv, _ = _tokens(L, 1)
    rope = -1.0 + 0.125 * (np.arange(64) % 16)
    kr = np.tile(bf16(rope), (L, 1))
    keys = oracle.reference_keys(ckv, kr, L, C4R4)
    assert np.array_equal(keys[:, 512:], np.tile(rope, (L, 1)))
    rng = np.random.default_rng(2)
    q = np.zeros((2, 576), np.float32)
    q[:, 512:] = rng.standard_normal((2, 64))
    out, _ = oracle.mla_decode_fp64(bf16(q), keys, 1 / math.sqrt(192))
    assert np.allclose(out, keys[:, :512].mean(0)[None], rtol=0, atol=1e-11)


def test_one_hot_logit_selects_one_token():
    L, star = 700, 333
    ckv, _ = _tokens(L, 4)
    kr = np.zeros((L, 64), np.uint16)
    kr[star, 0] = bf16([1.0])[0]
    keys = oracle.reference_keys(ckv, kr, L, C4R4)
    q = np.zeros((3, 576), np.float32)
    q[:, 512] = 1024.0
    scale = 1 / math.sqrt(192)
    out, _ = oracle.mla_decode_fp64(bf16(q), keys, scale)
    gap = scale * 1024.0 * keys[star, 512]
    assert gap > 50
    bound = math.exp(-gap) * L * np.abs(keys[:, :512]).max() * 2
    assert np.abs(out - keys[star, :512][None]).max() <= bound + 1e-13


def test_multi_query_causal_boundary_selects_own_token():
    # Logits grow by 0.25 * 1024 * scale per position (key channel 512 = t / 4),
    # so every query's softmax concentrates on the latest token it may see:
    # query i of n sits at position L - n + i and must select exactly that
    # token (seeing one more, or one fewer, would select a neighbour).
    L, n = 300, 4
    rng = np.random.default_rng(11)
    keys = rng.standard_normal((L, 576))
    keys[:, 512:] = 0.0
    keys[:, 512] = np.arange(L) / 4.0
    q = np.zeros((n, 3, 576), np.float32)
    q[:, :, 512] = 1024.0
    scale = 1 / math.sqrt(192)
    out, lse = oracle.mla_decode_multi_fp64(bf16(q.reshape(n * 3, 576)).reshape(n, 3, 576),
                                            keys, scale)
    gap = scale * 1024.0 * 0.25
    assert gap > 18
    for i in range(n):
        own = L - n + i
        bound = 2 * math.exp(-gap) * np.abs(keys[:, :512]).max() / (1 - math.exp(-gap))
        assert np.abs(out[i] - keys[own, :512][None]).max() <= bound
        # lse is the log of the visible tokens' exp(logit): dominated by the own token
        assert abs(lse[i, 0] - scale * 1024.0 * keys[own, 512]) < 1e-6


def test_multi_query_matches_masked_torch_sdpa():
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(12)
    L, n, H = 40, 3, 2
    keys = rng.standard_normal((L, 576))
    q = bf16(rng.standard_normal((n * H, 576)) * 0.3).reshape(n, H, 576)
    scale = 0.05
    out, _ = oracle.mla_decode_multi_fp64(q, keys, scale)
    qf = torch.from_numpy(syn.f32_from_bf16_bits(q).astype(np.float64))      # [n][H][576]
    k = torch.from_numpy(keys)                                               # [L][576]
    # MQA layout: heads as the batch, queries as the sequence; explicit mask
    mask = torch.tensor([[t <= L - n + i for t in range(L)] for i in range(n)])
    got = torch.nn.functional.scaled_dot_product_attention(
        qf.permute(1, 0, 2), k[None].expand(H, L, 576), k[None, :, :512].expand(H, L, 512),
        attn_mask=mask, scale=scale).permute(1, 0, 2).numpy()
    assert np.abs(got - out).max() < 1e-12


def test_hadamard_rotation_closed_forms():
    R = oracle.hadamard_matrix64()
    # orthonormal and symmetric: R R = I
    assert np.array_equal(R @ R, np.eye(64)) and np.array_equal(R, R.T)
    # the butterfly on e_k is column k of R, exactly (entries +-1/8)
    eye = np.eye(64, dtype=np.float32)
    assert np.array_equal(oracle.hadamard_rotate_f32(eye), R.T.astype(np.float32))
    # small integers: every partial sum is exact in float32
    rng = np.random.default_rng(21)
    xi = rng.integers(-1000, 1000, size=(50, 64)).astype(np.float32)
    assert np.array_equal(oracle.hadamard_rotate_f32(xi).astype(np.float64), xi.astype(np.float64) @ R.T)
    # bf16 inputs: within float32 rounding of six butterfly stages
    xb = syn.f32_from_bf16_bits(bf16(rng.standard_normal((50, 64)) * 10)).astype(np.float32)
    want = xb.astype(np.float64) @ R.T
    err = np.abs(oracle.hadamard_rotate_f32(xb).astype(np.float64) - want)
    assert np.all(err <= 6 * 2.0 ** -24 * np.abs(xb).astype(np.float64).sum(axis=1, keepdims=True))


# ---------------------------------------------------------------- bf16 rounding

@pytest.mark.parametrize("x, want", [
    (1.0 + 2.0 ** -8, 0x3F80),                   # tie -> even mantissa (down to 1.0)
    (1.0 + 3 * 2.0 ** -8, 0x3F82),               # tie -> even mantissa (up to 1 + 2^-6)
    (1.0 + 2.0 ** -8 + 2.0 ** -20, 0x3F81),      # just above the tie -> up
    (1.0 + 2.0 ** -8 - 2.0 ** -20, 0x3F80),      # just below the tie -> down
    (-(1.0 + 2.0 ** -8), 0xBF80),
    (-(1.0 + 3 * 2.0 ** -8), 0xBF82),
    (0.0, 0x0000),
    (-0.0, 0x8000),
    (2.0 ** -126, 0x0080),                       # smallest normal
    (2.0 ** -130, 0x0008),                       # subnormal, exact in bf16
    (3.0 * 2.0 ** -134, 0x0000 + 2),             # subnormal tie (1.5 ulp) -> 2 (even)
    (65504.0, 0x4780),                           # 65504 = 1.999 x 2^15 rounds up to 65536
])
def test_f32_to_bf16_bits_textbook(x, want):
    # the rotation's bf16 rounding: nearest, ties to even (textbook bf16 facts)
    got = oracle.quant.f32_to_bf16_bits(np.array([x], dtype=np.float32))[0]
    assert int(got) == want
    # the input generator's rounding obeys the same facts
    assert int(bf16(np.array([x]))[0]) == want


def test_f32_to_bf16_bits_matches_torch():
    # an independent implementation of the same IEEE rounding: torch's
    # float32 -> bfloat16 conversion, over many magnitudes and both signs
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(23)
    x = (rng.standard_normal(200000) * np.exp2(rng.integers(-60, 60, 200000))).astype(np.float32)
    # ties: random finite high halves (exponent below 0xFF) with the low 16 bits
    # exactly 0x8000
    ties = ((rng.integers(0, 0x7F7F, 20000).astype(np.uint32) << 16) | 0x8000).view(np.float32)
    x = np.concatenate([x, ties, -ties])
    want = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(oracle.quant.f32_to_bf16_bits(x), want)
    assert np.array_equal(bf16(x), want)


def test_rotate_latent_bits_rounds_a_hand_derived_group():
    # x = e_0 + (3/256) e_1 in every content group.  Every butterfly stage only
    # copies sums: element i becomes 1 + 3/256 (i even) or 1 - 3/256 (i odd),
    # exact in float32; the 1/8 scale is exact too.  Rounded to bf16:
    #   (1 + 3/256) / 8 = 1.00000011b x 2^-3: a tie between mantissas 0000001
    #       and 0000010 -> even -> 1.0000010b x 2^-3 = bits 0x3E02;
    #   (1 - 3/256) / 8 = 253/2048 = 1.1111101b x 2^-4: exact -> bits 0x3DFD.
    x = np.zeros((2, 512), dtype=np.float32)
    x[:, 0::64] = 1.0
    x[:, 1::64] = 3.0 / 256.0
    x[1] = -x[1]
    got = oracle.rotate_latent_bits(bf16(x))
    want = np.where(np.arange(512) % 2 == 0, 0x3E02, 0x3DFD).astype(np.uint16)
    assert np.array_equal(got[0], want)
    assert np.array_equal(got[1], want | 0x8000)


def test_rotated_attention_equals_unrotated_on_exact_keys():
    # keys stored in the rotated basis (exactly, in float64) must give the same
    # logits and outputs as the plain keys: q is rotated, the output rotated back
    rng = np.random.default_rng(22)
    L, H = 60, 3
    keys = rng.standard_normal((L, 576)) * 3
    R = oracle.hadamard_matrix64()
    rk = keys.copy()
    rk[:, :512] = (keys[:, :512].reshape(L, 8, 64) @ R.T).reshape(L, 512)
    q = bf16(rng.standard_normal((H, 576)))
    o0, l0 = oracle.mla_decode_fp64(q, keys, 0.05)
    o1, l1 = oracle.mla_decode_fp64(q, rk, 0.05, rotate=True)
    assert np.abs(o0 - o1).max() < 1e-12 and np.abs(l0 - l1).max() < 1e-12


def test_rotated_cache_stores_the_rotated_latent():
    L = 200
    ckv, kr = _tokens(L, 4)
    lay = oracle.Layout(4, 4, rotate=True)
    table = np.arange(4, dtype=np.int32)[None, :]
    m = oracle.PagedCacheModel(lay, 4, table)
    m.write(np.zeros(L, np.int64), np.arange(L), ckv, kr, np.array([L]))
    rot = oracle.rotate_latent_bits(ckv)
    # bf16 copies (sink and ring) hold the rotated latent and the unrotated RoPE key
    assert np.array_equal(m.sink[0, :4, :512], rot[:4])
    assert np.array_equal(m.recent[0, np.arange(L - 128, L) % 128, :512], rot[L - 128:])
    assert np.array_equal(m.recent[0, np.arange(L - 128, L) % 128, 512:], kr[L - 128:])
    # packed codes are those of the rotated latent: same bytes as an unrotated
    # cache fed the rotated bits
    plain = oracle.PagedCacheModel(oracle.Layout(4, 4), 4, table)
    plain.write(np.zeros(L, np.int64), np.arange(L), rot, kr, np.array([L]))
    assert np.array_equal(m.pool, plain.pool)
    with pytest.raises(ValueError):
        oracle.Layout(16, 16, rotate=True)


def test_bruteforce_tiny_softmax_without_max_subtraction():
    rng = np.random.default_rng(5)
    for L in (1, 2, 5, 8):
        H = 2
        keys = rng.standard_normal((L, 576))
        q = bf16(rng.standard_normal((H, 576)) * 0.3)
        qf = syn.f32_from_bf16_bits(q).astype(np.float64)
        scale = 0.05
        out, lse = oracle.mla_decode_fp64(q, keys, scale)
        for h in range(H):
            w = [math.exp(scale * sum(qf[h, c] * keys[t, c] for c in range(576)))
                 for t in range(L)]
            tot = sum(w)
            for c in range(0, 512, 37):
                want = sum(w[t] * keys[t, c] for t in range(L)) / tot
                assert abs(out[h, c] - want) <= 1e-12 * max(1.0, abs(want))
            assert abs(lse[h] - math.log(tot)) <= 1e-12


def test_matches_torch_sdpa_fp64_as_mqa():
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(6)
    H, L = 16, 257
    keys = rng.standard_normal((L, 576))
    q = bf16(rng.standard_normal((H, 576)))
    scale = 1 / math.sqrt(192)
    out, _ = oracle.mla_decode_fp64(q, keys, scale)
    qt = torch.from_numpy(syn.f32_from_bf16_bits(q).astype(np.float64)).view(1, H, 1, 576)
    kt = torch.from_numpy(keys).view(1, 1, L, 576).expand(1, H, L, 576)
    vt = torch.from_numpy(keys[:, :512].copy()).view(1, 1, L, 512).expand(1, H, L, 512)
    ref = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, scale=scale)
    assert np.abs(out - ref.view(H, 512).numpy()).max() < 1e-12


def test_empty_sequence():
    out, lse = oracle.mla_decode_fp64(np.zeros((2, 576), np.uint16), np.zeros((0, 576)), 0.1)
    assert not out.any() and np.all(np.isneginf(lse))


# ---------------------------------------------------------------- protection policy

def test_short_sequences_are_plain_bf16_attention():
    for L in (1, 4, 5, 131, 132):
        ckv, kr = _tokens(L, 8)
        keys = oracle.reference_keys(ckv, kr, L, C4R4)
        exact = np.concatenate([syn.f32_from_bf16_bits(ckv), syn.f32_from_bf16_bits(kr)], 1)
        assert np.array_equal(keys, exact.astype(np.float64))


def test_length_133_packs_exactly_token_4():
    L = 133
    ckv, kr = _tokens(L, 9)
    keys = oracle.reference_keys(ckv, kr, L, C4R4)
    exact = np.concatenate([syn.f32_from_bf16_bits(ckv), syn.f32_from_bf16_bits(kr)], 1)
    diff_rows = np.nonzero(np.any(keys != exact, axis=1))[0]
    assert diff_rows.tolist() == [4]


@pytest.mark.parametrize("lay", [C4R4, C2R4])
def test_window_transition_token_by_token(lay):
    # 200 single-token steps: a token is served packed exactly when L > pos + 128
    # (and pos >= 4), and its packed bytes never change after it was written.
    n = 200
    ckv, kr = _tokens(n, 10)
    table = np.arange(4, dtype=np.int32)[None, :]
    model = PagedCacheModel(lay, 4, table)
    written = {}
    for L in range(1, n + 1):
        t = L - 1
        model.write([0], [t], ckv[t:t + 1], kr[t:t + 1], [L])
        written[t] = model.token_bytes(0, t)
        for u in range(L):
            assert model.token_bytes(0, u) == written[u]
        keys = model.effective_keys(0, L)
        ref = oracle.reference_keys(ckv, kr, L, lay)
        assert np.array_equal(keys, ref)
        packed_rows = [u for u in range(L) if not oracle.is_protected(np.array(u), L)]
        assert packed_rows == [u for u in range(4, L) if L > u + 128]


def test_bulk_prefill_equals_token_by_token():
    n = 300
    ckv, kr = _tokens(n, 11)
    table = np.array([[3, 0, 4, 1, 2]], dtype=np.int32)
    a = PagedCacheModel(C4R4, 5, table)
    b = PagedCacheModel(C4R4, 5, table)
    a.write(np.zeros(n, int), np.arange(n), ckv, kr, [n])
    for t in range(n):
        b.write([0], [t], ckv[t:t + 1], kr[t:t + 1], [t + 1])
    assert np.array_equal(a.pool, b.pool)
    assert np.array_equal(a.sink, b.sink) and np.array_equal(a.recent, b.recent)


def test_page_bytes_decode_by_hand():
    # One token, hand-checked against the byte layout.
    table = np.array([[1]], dtype=np.int32)
    model = PagedCacheModel(C4R4, 2, table)
    ckv = np.zeros(512, np.float32)
    ckv[0], ckv[1], ckv[63] = 15.0, 1.0, 0.0   # group 0: s = 1, m = 0
    kr = np.zeros(64, np.float32)
    model.write([0], [5], bf16(ckv)[None], bf16(kr)[None], [6])
    page = model.pool[1]
    row = 5
    assert page[row * 256 + 0] == 0x1F           # codes 15 (low) and 1 (high)
    meta = page[18432 + row * 36: 18432 + row * 36 + 36].view(np.float16)
    assert meta[0] == 1.0 and meta[1] == 0.0      # group 0 (scale, min)
    assert meta[2] == 0.0 and meta[3] == 0.0      # group 1: constant zeros
    assert not model.pool[0].any()


def test_cache_model_matches_definition_on_workload_slice():
    w = syn.custom("t", [520, 77], content_bits=4)
    table, npages = syn.make_paging(w)
    model = PagedCacheModel(C4R4, npages, table)
    for b, L in enumerate(syn.sequence_lengths(w)):
        ckv, kr = syn.sequence_tokens(w, b)
        model.write(np.full(L, b), np.arange(L), ckv, kr, syn.sequence_lengths(w))
        assert np.array_equal(model.effective_keys(b, L), oracle.reference_keys(ckv, kr, L, C4R4))
