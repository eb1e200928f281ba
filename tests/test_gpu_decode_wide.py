"""The 128-row tcgen05 decode (2-CTA clusters, decode_wide.cu) vs the fp64 oracle.

Packed layouts with exactly 128 query rows per sequence (128 heads, or n_q
query blocks of 128 / n_q heads) take this kernel by default.  Same bar as
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


@pytest.mark.parametrize("cb", [4, 2])
def test_wide_edge_lengths(cb):
    w = syn.custom(f"wide_edge_c{cb}", EDGE_LENGTHS, heads=128, content_bits=cb, seed=81)
    run = GpuRun(w)
    run.prefill()
    _check_run_step(run, 0, lse=True)


def test_wide_long_sequences_many_splits():
    # sequences long enough for several splits each, with a short one beside
    w = syn.custom("wide_long", [17000, 9000, 133, 1], heads=128, content_bits=4, seed=82)
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


def test_wide_matches_mma_kernel(monkeypatch):
    # the same decode through the 16-head mma.sync kernel (forced by the
    # environment) and through the 128-row kernel agree to the oracle's bar
    import torch
    w = syn.custom("wide_vs_mma", [2100, 5000, 140], heads=128, content_bits=4, seed=84)
    run = GpuRun(w)
    run.prefill()
    ckv, kr, q = run.step_inputs(0)
    lens = (run.lens).astype(np.int32)
    run.cache.write(to_dev(ckv, torch.bfloat16), to_dev(kr, torch.bfloat16),
                    to_dev(lens - 1, torch.int32), seq_lens_after=to_dev(lens, torch.int32))
    outs = []
    for env in (None, "m"):
        if env:
            monkeypatch.setenv("MLA_LOWBIT_DECODE", env)
        else:
            monkeypatch.delenv("MLA_LOWBIT_DECODE", raising=False)
        out = run.cache.decode(to_dev(q, torch.bfloat16), to_dev(lens, torch.int32),
                               [int(x) for x in lens], w.softmax_scale)
        torch.cuda.synchronize()
        outs.append(out.cpu().numpy())
    assert run.cache.error() == 0
    for b in range(w.batch):
        check_attention(outs[0][b], outs[1][b].astype(np.float64), f"seq {b}")


@pytest.mark.parametrize("cb,heads,n", [(4, 64, 2), (4, 16, 8), (2, 32, 4)])
def test_wide_multi_query_blocks(cb, heads, n):
    # n_q * heads = 128 rows: per-row causal masks inside the 128-row kernel
    import torch
    w = syn.custom(f"wide_mq_c{cb}_h{heads}_n{n}", [8, 131, 134, 700, 2500], heads=heads,
                   content_bits=cb, steps=n, seed=85 + n)
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
