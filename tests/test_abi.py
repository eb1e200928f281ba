"""Host-side checks of the C ABI that need no GPU: symbols, sizes, argument
validation and split planning."""

import ctypes
import math
import os
import re

import numpy as np
import pytest

import bit_mla_kv_lowbit_gb300 as pkg
import oracle

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "mla_lowbit.h")


def declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(mla_lowbit_\w+)\s*\(", src)))


def test_library_exports_every_declared_symbol():
    lib = pkg.load()
    names = declared_functions()
    assert names, "no declarations parsed"
    for n in names:
        assert hasattr(lib, n), f"{n} declared in mla_lowbit.h but not exported"
    assert set(names) == set(pkg.EXPORTS)


def test_sizes_agree_with_oracle_closed_form():
    for cb, rb in ((4, 4), (2, 4), (16, 16)):
        lay = pkg.layout(cb, rb)
        olay = oracle.Layout(cb, rb)
        assert pkg.page_bytes(lay) == oracle.page_geometry(olay)["page_bytes"]
        assert pkg.bytes_per_token(lay) == oracle.bytes_per_token(olay)


@pytest.mark.parametrize("fields", [
    dict(content_bits=3), dict(rope_bits=2), dict(group=32), dict(sink=0), dict(local=64),
    dict(page_tokens=128), dict(latent=256), dict(rope=32), dict(rotate=2), dict(rotate=-1),
])
def test_invalid_layouts_rejected(fields):
    lay = pkg.layout(4, 4)
    for k, v in fields.items():
        setattr(lay, k, v)
    assert pkg.page_bytes(lay) == 0
    with pytest.raises(pkg.LibraryError):
        pkg.decode_plan(lay, 16, [100], num_sms=152)


def test_rotation_only_on_packed_layouts():
    # the online rotation re-encodes the content latent before quantisation:
    # accepted for the packed layouts, refused for bf16 pages
    for cb in (4, 2):
        assert pkg.page_bytes(pkg.layout(cb, 4, rotate=True)) == pkg.page_bytes(pkg.layout(cb, 4))
    assert pkg.page_bytes(pkg.layout(16, 16, rotate=True)) == 0


def test_strerror_and_version():
    assert pkg.strerror(0) == "ok"
    for st in range(-6, 0):
        assert pkg.strerror(st) != "unknown status"
    assert pkg.strerror(-99) == "unknown status"
    assert pkg.version() >= 100


def _call_write(lay, **over):
    lib = pkg.load()
    args = dict(n=4, ckv=0x1000, krope=0x2000, seq_idx=None, pos=0x3000, lens=None, num_seqs=4,
                table=0x4000, max_pages=8, pool=0x5000, num_pages=16, sink=0x6000,
                recent=0x7000, err=0x8000, stream=None)
    args.update(over)
    return lib.mla_lowbit_write(ctypes.byref(lay), args["n"], args["ckv"], args["krope"],
                                args["seq_idx"], args["pos"], args["lens"], args["num_seqs"],
                                args["table"], args["max_pages"], args["pool"], args["num_pages"],
                                args["sink"], args["recent"], args["err"], args["stream"])


def test_write_host_validation_without_launch():
    lay = pkg.layout(4, 4)
    assert _call_write(lay, n=0) == 0                 # nothing to do
    assert _call_write(lay, ckv=None) == -2
    assert _call_write(lay, err=None) == -2
    assert _call_write(lay, sink=None) == -2
    assert _call_write(lay, pool=0x5004) == -3        # misaligned
    assert _call_write(lay, n=-1) == -4
    assert _call_write(lay, n=5, num_seqs=4) == -1    # identity seq_idx needs n <= num_seqs
    assert _call_write(pkg.layout(16, 16), sink=None, recent=None, ckv=None) == -2
    bad = pkg.layout(4, 4)
    bad.content_bits = 8
    assert _call_write(bad) == -1


def _call_decode(lay, **over):
    lib = pkg.load()
    lens = np.array([100, 200], np.int32)
    args = dict(B=2, H=16, scale=0.07, q=0x1000, pool=0x2000, num_pages=8, table=0x3000,
                max_pages=4, lens=0x4000, lens_host=lens.ctypes.data, sink=0x5000, recent=0x6000,
                out=0x7000, lse=None, ws=0x8000, ws_bytes=1 << 30, err=0x9000, stream=None)
    args.update(over)
    return lib.mla_lowbit_decode(ctypes.byref(lay), args["B"], args["H"],
                                 ctypes.c_float(args["scale"]), args["q"], args["pool"],
                                 args["num_pages"], args["table"], args["max_pages"], args["lens"],
                                 args["lens_host"], args["sink"], args["recent"], args["out"],
                                 args["lse"], args["ws"], args["ws_bytes"], args["err"],
                                 args["stream"])


def test_decode_host_validation_without_launch():
    lay = pkg.layout(4, 4)
    assert _call_decode(lay, H=24) == -4
    assert _call_decode(lay, H=144) == -4
    assert _call_decode(lay, B=0) == -4
    assert _call_decode(lay, q=None) == -2
    assert _call_decode(lay, lens_host=None) == -2
    assert _call_decode(lay, out=0x7008) == -3
    assert _call_decode(lay, scale=0.0) == -1
    assert _call_decode(lay, scale=float("nan")) == -1
    too_long = np.array([100, 4 * 64 + 1], np.int32)
    assert _call_decode(lay, lens_host=too_long.ctypes.data) == -1


def _call_write_decode(lay, B=2, H=16, ckv=0x8000, kr=0x9000, lens_host=None):
    # fake, aligned device pointers: every case is rejected before any launch
    lens = np.array([100, 300], np.int32) if lens_host is None else lens_host
    return pkg.load().mla_lowbit_write_decode(
        ctypes.byref(lay), B, H, ctypes.c_float(0.07), 0x1000, ckv, kr, 0x2000, 64, 0x3000, 16,
        0x4000, lens.ctypes.data, 0x5000, 0x6000, 0x7000, None, 0xA000, 1 << 20, 0xB000, None)


def test_write_decode_host_validation_without_launch():
    lay = pkg.layout(4, 4)
    assert _call_write_decode(lay, ckv=None) == -2
    assert _call_write_decode(lay, kr=None) == -2
    assert _call_write_decode(lay, ckv=0x8008) == -3          # new-token rows not 16-byte aligned
    zero = np.array([100, 0], np.int32)                        # every sequence appends a token
    assert _call_write_decode(lay, lens_host=zero) == -1
    assert _call_write_decode(lay, H=24) == -4


def _expected_splits(L, packed, chunk):
    # Work units of a sequence: for packed layouts the pages that hold at least
    # one token served from packed codes (positions 4 .. L-129), then the
    # protected tokens (sink 0..3 and recent L-128..L-1, each counted once) in
    # 64-token tiles; for bf16 pages every page.  Splits cut the units into
    # chunks, at least one split per sequence.
    if packed:
        served = [t for t in range(4, max(4, L - 128))]
        pages = len({t // 64 for t in served})
        protected = len({t for t in range(L) if t < 4 or t >= L - 128})
        units = pages + 3 * math.ceil(protected / 64)  # a bf16 tile counts 3 units
    else:
        units = math.ceil(L / 64)
    return max(1, math.ceil(units / chunk))


@pytest.mark.parametrize("cb", [4, 2, 16])
def test_plan_matches_definition(cb):
    lay = pkg.layout(cb, 4 if cb != 16 else 16)
    rng = np.random.default_rng(0)
    lens = [0, 1, 4, 5, 131, 132, 133, 192, 193, 196, 197, 260, 1000, 4099]
    lens += rng.integers(0, 20000, 10).tolist()
    for heads in (16, 64, 128):
        total, chunk, ws = pkg.decode_plan(lay, heads, lens, num_sms=152)
        assert chunk >= 1
        assert total == sum(_expected_splits(L, cb != 16, chunk) for L in lens)
        assert ws == total * heads * (512 + 2) * 4 + len(lens) * 8


def test_plan_fills_one_wave_on_uniform_lengths():
    # one CTA per SM: 8 sequences of 510 packed-served pages + 3 protected-token
    # tiles of 3 units each (519 units) -> 4,152 units in chunks of
    # ceil(4152 / 152) = 28 -> 19 splits per sequence: one wave of 152 CTAs
    total, chunk, _ = pkg.decode_plan(pkg.layout(4, 4), 16, [32768] * 8, num_sms=152)
    assert (total, chunk) == (152, 28)
    # bf16 pages: 8 x 512 pages in chunks of 27 -> 19 splits per sequence
    total, chunk, _ = pkg.decode_plan(pkg.layout(16, 16), 16, [32768] * 8, num_sms=152)
    assert (total, chunk) == (152, 27)


def test_plan_spreads_work_over_full_waves():
    # one CTA per SM; 128 heads run as 2-CTA clusters.  The planner picks the
    # fewest waves the split cap allows (128 pages for the cluster kernel, 64
    # for the 16-row kernel), then the smallest chunk whose splits fit those
    # waves, so the last wave is not a short tail.
    lay = pkg.layout(4, 4)
    for heads, lens in [(128, [8192] * 32), (128, [131072] * 4), (128, [10240] * 32),
                        (16, [2000] * 1000), (16, [32768] * 8)]:
        total, chunk, _ = pkg.decode_plan(lay, heads, lens, num_sms=152)
        cps = 2 * (heads // 128) if heads % 128 == 0 else heads // 16
        cap = 128 if heads % 128 == 0 else 64
        assert 1 <= chunk <= cap
        waves = -(-total * cps // 152)
        capped = sum(_expected_splits(L, True, cap) for L in lens)
        assert waves == -(-capped * cps // 152) or waves == -(-total * cps // 152)
        assert waves >= -(-capped * cps // 152)          # never fewer than possible
        if chunk > 1:                                      # smallest chunk for these waves
            smaller = sum(_expected_splits(L, True, chunk - 1) for L in lens)
            assert smaller * cps > waves * 152
    # the cases that motivated it: one wave each (32 x 131 units in chunks of 68;
    # 4 x 8,201 units in chunks of 109 -> 76 clusters), and several waves past
    # the cap (4 x 1M tokens: chunks of 124, 532 splits)
    assert pkg.decode_plan(lay, 128, [8192] * 32, num_sms=152)[:2] == (64, 68)
    assert pkg.decode_plan(lay, 128, [131072] * 4, num_sms=152)[:2] == (76, 109)
    assert pkg.decode_plan(lay, 128, [1048576] * 4, num_sms=152)[:2] == (532, 124)
    # rotation runs on the 16-row kernel: the 64-page cap
    assert pkg.decode_plan(pkg.layout(4, 4, rotate=True), 128, [131072] * 4, num_sms=152)[1] <= 64


def test_plan_takes_more_waves_when_they_are_faster():
    # 32 sequences of 4K-16K tokens at 128 heads: the fewest waves (one) need
    # 96-unit chunks, because each sequence's splits round up; two waves of
    # 43-unit chunks take about waves * (chunk + 3) = 92 units against 99, so
    # the planner takes two.  The 128K headline keeps its single wave.
    from workloads import synthetic as syn
    lay = pkg.layout(4, 4)
    lens = [int(x) for x in syn.sequence_lengths(syn.get("v3_c4r4"))]
    total, chunk, _ = pkg.decode_plan(lay, 128, lens, num_sms=152)
    waves = -(-total * 2 // 152)
    assert (total, chunk, waves) == (151, 43, 2)
    one_wave = sum(_expected_splits(L, True, 96) for L in lens)
    assert one_wave * 2 <= 152 and sum(_expected_splits(L, True, 95) for L in lens) * 2 > 152
    assert waves * (chunk + 3) * 20 < 1 * (96 + 3) * 19
    assert pkg.decode_plan(lay, 128, [131072] * 4, num_sms=152)[:2] == (76, 109)
