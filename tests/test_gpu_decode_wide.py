"""The 128-row tcgen05 decode (2-CTA clusters, decode_wide.cu) vs the fp64 oracle.

Packed layouts and bf16 pages with exactly 128 query rows per sequence (128
heads, or n_q query blocks of 128 / n_q heads) take this kernel by default.  Same bar as
the other decode tests: max-abs <= 2e-3 and rel-L2 <= 1e-3 per sequence, lse
within 1e-4, writer bytes bit-exact.
"""

import numpy as np
import pytest

import oracle
from tests.gpu_util import GpuRun, check_attention, oracle_model, to_dev
from tests.test_gpu_decode import EDGE_LENGTHS, _check_run_step
from workloads import synthetic as syn

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("cb", [4, 2, 16])
def test_wide_edge_lengths(cb):
    w = syn.custom(f"wide_edge_c{cb}", EDGE_LENGTHS, heads=128, content_bits=cb,
                   rope_bits=16 if cb == 16 else 4, seed=81)
    run = GpuRun(w)
    run.prefill()
    _check_run_step(run, 0, lse=True)


@pytest.mark.parametrize("cb", [4, 16])
def test_wide_long_sequences_many_splits(cb):
    # sequences long enough for several splits each, with a short one beside
    w = syn.custom(f"wide_long_c{cb}", [17000, 9000, 133, 1], heads=128, content_bits=cb,
                   rope_bits=16 if cb == 16 else 4, seed=82)
    run = GpuRun(w)
    run.prefill()
    _check_run_step(run, 0, lse=True)


def test_wide_write_decode_steps():
    w = syn.custom("wide_wd", [1, 64, 131, 132, 133, 700, 3000], heads=128, content_bits=4,
                   steps=3, seed=83)
    run = GpuRun(w)
    run.prefill()
    for s in range(3):
        _check_run_step(run, s, lse=True, fused=True)


@pytest.mark.parametrize("cb,heads,n", [(4, 64, 2), (4, 16, 8), (2, 32, 4), (16, 64, 2), (16, 32, 4)])
def test_wide_multi_query_blocks(cb, heads, n):
    # n_q * heads = 128 rows: per-row causal masks inside the 128-row kernel
    import torch
    w = syn.custom(f"wide_mq_c{cb}_h{heads}_n{n}", [8, 131, 134, 700, 2500], heads=heads,
                   content_bits=cb, rope_bits=16 if cb == 16 else 4, steps=n, seed=85 + n)
    run = GpuRun(w)
    run.prefill()
    ckv, kr, _ = run.step_inputs(0)
    lens = run.lens.astype(np.int32)
    run.cache.write(to_dev(ckv, torch.bfloat16), to_dev(kr, torch.bfloat16),
                    to_dev(lens - 1, torch.int32), seq_lens_after=to_dev(lens, torch.int32))
    q = np.stack([syn.queries(w, b)[:n] for b in range(w.batch)])
    lse = torch.empty(w.batch, n, heads, dtype=torch.float32, device="cuda")
    out = run.cache.decode_multi(to_dev(q, torch.bfloat16), to_dev(lens, torch.int32),
                                 [int(x) for x in lens], w.softmax_scale, lse=lse)
    torch.cuda.synchronize()
    assert run.cache.error() == 0
    out, lse = out.cpu().numpy(), lse.cpu().numpy()
    for b in range(w.batch):
        model, L = oracle_model(run, b, 0)
        ref, ref_lse = oracle.mla_decode_multi_fp64(q[b], model.effective_keys(b, L),
                                                    w.softmax_scale)
        for i in range(n):
            check_attention(out[b, i], ref[i], f"seq {b} (L={L}) query {i}")
            assert np.allclose(lse[b, i], ref_lse[i], rtol=0, atol=1e-4), f"lse seq {b} query {i}"


def test_wide_large_scales_under_the_lazy_max():
    # Content groups spanning +-3000 (fp16 scales near 400) and logits that
    # climb slowly along the sequence, so the running max trails the tile max
    # by up to the lazy threshold: P * s would pass the fp16 range unless the
    # tile's largest scale lowers the threshold.  Outputs are O(1e3), so the
    # bar is relative: rel-L2 <= 1e-3 and max-abs <= 1e-5 of the largest value.
    import torch
    import bit_mla_kv_lowbit_gb300 as pkg
    rng = np.random.default_rng(91)
    L, H = 2000, 128
    ckv = rng.uniform(-3000.0, 3000.0, (L, 512))
    u = np.where(rng.random(64) < 0.5, -0.125, 0.125)
    ramp = 0.5 + 3.0 * np.arange(L) / L
    kr = ramp[:, None] * u[None, :]
    q = np.zeros((H, 576))
    q[:, 512:] = 130.0 * u[None, :] * (1.0 + 0.01 * np.arange(H))[:, None]
    to_bits = lambda x: syn.bf16_bits_from_f32(np.asarray(x, dtype=np.float32))
    ckv_b, kr_b, q_b = to_bits(ckv), to_bits(kr), to_bits(q)
    table = np.arange(32, dtype=np.int32)[None, :]
    cache = pkg.PagedCache(4, 4, table, 32, "cuda")
    lens = torch.tensor([L], dtype=torch.int32, device="cuda")
    cache.write(to_dev(ckv_b, torch.bfloat16), to_dev(kr_b, torch.bfloat16),
                torch.arange(L, dtype=torch.int32, device="cuda"),
                seq_idx=torch.zeros(L, dtype=torch.int32, device="cuda"), seq_lens_after=lens)
    scale = 1.0 / np.sqrt(192.0)
    out = cache.decode(to_dev(q_b[None], torch.bfloat16), lens, [L], scale)
    torch.cuda.synchronize()
    assert cache.error() == 0
    got = out.cpu().numpy()[0].astype(np.float64)
    model = oracle.PagedCacheModel(oracle.Layout(4, 4), 32, table)
    model.write(np.zeros(L, np.int64), np.arange(L), ckv_b, kr_b, np.array([L]))
    ref, _ = oracle.mla_decode_fp64(q_b, model.effective_keys(0, L), scale)
    assert np.all(np.isfinite(got))
    rel = np.linalg.norm(got - ref) / np.linalg.norm(ref)
    assert rel <= 1e-3 and np.abs(got - ref).max() <= 1e-5 * np.abs(ref).max(), (rel, np.abs(got - ref).max())


def test_wide_scales_beyond_the_fp16_plane_range():
    # Content groups spanning +-31000: the fp16 scale is ~4100, so s * |c - 8|
    # reaches ~33000 and the kernel stores those tokens' planes scaled by 2^-4
    # (and scales their logits and P back).  Relative bar, as the outputs are
    # O(1e4): rel-L2 <= 1e-3 and max-abs <= 1e-3 of the largest value (fp32
    # tensor-core accumulation over 1,500 products of this size carries ~1e-4
    # relative error; a wrong compensation would be off by a factor of 16).
    import torch
    import bit_mla_kv_lowbit_gb300 as pkg
    rng = np.random.default_rng(92)
    L, H = 1500, 128
    ckv = rng.uniform(-31000.0, 31000.0, (L, 512))
    ckv[::3, 64:128] *= 1e-3          # some groups on every third token stay small
    kr = rng.standard_normal((L, 64))
    q = rng.standard_normal((H, 576)) * 1e-4
    to_bits = lambda x: syn.bf16_bits_from_f32(np.asarray(x, dtype=np.float32))
    ckv_b, kr_b, q_b = to_bits(ckv), to_bits(kr), to_bits(q)
    table = np.arange(24, dtype=np.int32)[None, :]
    cache = pkg.PagedCache(4, 4, table, 24, "cuda")
    lens = torch.tensor([L], dtype=torch.int32, device="cuda")
    cache.write(to_dev(ckv_b, torch.bfloat16), to_dev(kr_b, torch.bfloat16),
                torch.arange(L, dtype=torch.int32, device="cuda"),
                seq_idx=torch.zeros(L, dtype=torch.int32, device="cuda"), seq_lens_after=lens)
    scale = 1.0 / np.sqrt(192.0)
    lse = torch.empty(1, H, dtype=torch.float32, device="cuda")
    out = cache.decode(to_dev(q_b[None], torch.bfloat16), lens, [L], scale, lse=lse)
    torch.cuda.synchronize()
    assert cache.error() == 0
    got = out.cpu().numpy()[0].astype(np.float64)
    model = oracle.PagedCacheModel(oracle.Layout(4, 4), 24, table)
    model.write(np.zeros(L, np.int64), np.arange(L), ckv_b, kr_b, np.array([L]))
    ref, ref_lse = oracle.mla_decode_fp64(q_b, model.effective_keys(0, L), scale)
    assert np.all(np.isfinite(got))
    rel = np.linalg.norm(got - ref) / np.linalg.norm(ref)
    assert rel <= 1e-3 and np.abs(got - ref).max() <= 1e-3 * np.abs(ref).max(), (rel, np.abs(got - ref).max())
    # each logit sums 576 products of size ~3 here: fp32 accumulation alone
    # leaves ~1e-4 in the log-sum-exp, hence a 1e-3 bar instead of 1e-4
    assert np.allclose(lse.cpu().numpy()[0], ref_lse, rtol=0, atol=1e-3)


@pytest.mark.parametrize("cb", [4, 2])
def test_wide_two_row_blocks_mtp_128_heads(cb):
    # 2 causal queries of 128 heads (256 rows: two 128-row clusters per split),
    # the multi-token prediction step of a 128-head model
    import torch
    heads, n = 128, 2
    w = syn.custom(f"wide_mtp128_c{cb}", [6, 133, 700, 3100], heads=heads, content_bits=cb,
                   steps=n, seed=95)
    run = GpuRun(w)
    run.prefill()
    ckv, kr, _ = run.step_inputs(0)
    lens = run.lens.astype(np.int32)
    run.cache.write(to_dev(ckv, torch.bfloat16), to_dev(kr, torch.bfloat16),
                    to_dev(lens - 1, torch.int32), seq_lens_after=to_dev(lens, torch.int32))
    q = np.stack([syn.queries(w, b)[:n] for b in range(w.batch)])
    lse = torch.empty(w.batch, n, heads, dtype=torch.float32, device="cuda")
    out = run.cache.decode_multi(to_dev(q, torch.bfloat16), to_dev(lens, torch.int32),
                                 [int(x) for x in lens], w.softmax_scale, lse=lse)
    torch.cuda.synchronize()
    assert run.cache.error() == 0
    out, lse = out.cpu().numpy(), lse.cpu().numpy()
    for b in range(w.batch):
        model, L = oracle_model(run, b, 0)
        ref, ref_lse = oracle.mla_decode_multi_fp64(q[b], model.effective_keys(b, L),
                                                    w.softmax_scale)
        for i in range(n):
            check_attention(out[b, i], ref[i], f"seq {b} (L={L}) query {i}")
            assert np.allclose(lse[b, i], ref_lse[i], rtol=0, atol=1e-4), f"lse seq {b} query {i}"


@pytest.mark.parametrize("heads", [128, 16])
def test_min_terms_with_q_group_sums_beyond_fp16(heads):
    # Content q near 1100, so each group's q sum (the factor of the logits'
    # min terms) is ~70,400, past the fp16 maximum, over a cache of values
    # 0.05 +- 1e-3 (m' ~ 0.05).  The min terms then carry ~2,000 of each
    # scaled logit and move it by O(1) from token to token (the oracle's
    # softmax spreads over ~550 effective tokens, top weight ~1.6 %).  The
    # 128-row kernel computes them on the tensor core from three bf16 parts
    # per factor, the 16-head kernel (the control) in fp32.  The log-sum-exp
    # (~2,039) is the sensitive check: fp32 sums of min terms of ~3,500 each
    # leave ~1e-4 in it, so the bar is 1e-3.
    import torch
    import bit_mla_kv_lowbit_gb300 as pkg
    rng = np.random.default_rng(94)
    L = 900
    ckv = 0.05 + rng.uniform(-1e-3, 1e-3, (L, 512))
    kr = rng.standard_normal((L, 64))
    q = np.concatenate([1100.0 + 10.0 * rng.standard_normal((heads, 512)),
                        1e-3 * rng.standard_normal((heads, 64))], axis=1)
    to_bits = lambda x: syn.bf16_bits_from_f32(np.asarray(x, dtype=np.float32))
    ckv_b, kr_b, q_b = to_bits(ckv), to_bits(kr), to_bits(q)
    table = np.arange(16, dtype=np.int32)[None, :]
    cache = pkg.PagedCache(4, 4, table, 16, "cuda")
    lens = torch.tensor([L], dtype=torch.int32, device="cuda")
    cache.write(to_dev(ckv_b, torch.bfloat16), to_dev(kr_b, torch.bfloat16),
                torch.arange(L, dtype=torch.int32, device="cuda"),
                seq_idx=torch.zeros(L, dtype=torch.int32, device="cuda"), seq_lens_after=lens)
    scale = 1.0 / np.sqrt(192.0)
    lse = torch.empty(1, heads, dtype=torch.float32, device="cuda")
    out = cache.decode(to_dev(q_b[None], torch.bfloat16), lens, [L], scale, lse=lse)
    torch.cuda.synchronize()
    assert cache.error() == 0
    got = out.cpu().numpy()[0]
    model = oracle.PagedCacheModel(oracle.Layout(4, 4), 16, table)
    model.write(np.zeros(L, np.int64), np.arange(L), ckv_b, kr_b, np.array([L]))
    ref, ref_lse = oracle.mla_decode_fp64(q_b, model.effective_keys(0, L), scale)
    check_attention(got, ref, f"{heads} heads")
    assert np.allclose(lse.cpu().numpy()[0], ref_lse, rtol=0, atol=1e-3)


def _lengths_for_chunk(lay, chunk, num_sms, batch=2):
    """Equal sequence lengths for which the planner cuts 128-head work into splits
    of `chunk` pages (found with the library's own planner for this GPU's SM count)."""
    import bit_mla_kv_lowbit_gb300 as pkg
    for L in range(2000, 60000, 64):
        if pkg.decode_plan(lay, 128, [L] * batch, num_sms=num_sms)[1] == chunk:
            return [L] * batch
    return None


@pytest.mark.parametrize("chunk", [2, 3, 4, 5])
def test_wide_tiles_spanning_pages(chunk):
    # Packed caches run 48-token tiles over a split's pages: with `chunk` pages
    # per split (64 * chunk tokens) the tiles cross page boundaries at 16, 32 or
    # 0 tokens in and the last tile of a split is ragged for chunk = 1, 2, 4, 5.
    # Every split size from 2 to 5 pages, checked against the oracle.
    import torch
    import bit_mla_kv_lowbit_gb300 as pkg
    nsm = torch.cuda.get_device_properties(0).multi_processor_count
    lens = _lengths_for_chunk(pkg.layout(4, 4), chunk, nsm)
    if lens is None:
        pytest.skip(f"no length gives {chunk}-page splits on {nsm} SMs")
    w = syn.custom(f"wide_span_k{chunk}", lens, heads=128, content_bits=4, seed=90 + chunk)
    run = GpuRun(w)
    run.prefill()
    _check_run_step(run, 0, lse=True)
