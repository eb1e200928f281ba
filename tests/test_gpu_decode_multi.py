"""Multi-token query decode (mla_lowbit_decode_multi) vs the fp64 oracle:
n queries per sequence at positions L - n .. L - 1, each attending causally
over the same dequantised cache.  Bar: max-abs <= 2e-3, rel-L2 <= 1e-3 per
query and sequence; lse within 1e-4."""

import numpy as np
import pytest

import oracle
from tests.gpu_util import GpuRun, check_attention, oracle_model, to_dev
from workloads import synthetic as syn

pytestmark = pytest.mark.gpu


def _run_multi(cb, heads, n, lengths, seed):
    import torch
    w = syn.custom(f"mq_c{cb}_h{heads}_n{n}", lengths, heads=heads, content_bits=cb,
                   rope_bits=4 if cb != 16 else 16, steps=n, seed=seed)
    run = GpuRun(w)
    run.prefill()
    ckv, kr, _ = run.step_inputs(0)          # token L - 1 of every sequence
    lens = run.lens.astype(np.int32)
    run.cache.write(to_dev(ckv, torch.bfloat16), to_dev(kr, torch.bfloat16),
                    to_dev(lens - 1, torch.int32), seq_lens_after=to_dev(lens, torch.int32))
    q = np.stack([syn.queries(w, b)[:n] for b in range(w.batch)])      # [B][n][H][576]
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


@pytest.mark.parametrize("cb,heads,n", [(4, 16, 2), (4, 16, 4), (2, 16, 2), (4, 32, 2)])
def test_multi_query_matches_oracle(cb, heads, n):
    _run_multi(cb, heads, n, [4, 5, 131, 133, 134, 700, 2500, 4099], seed=61 + n)


def test_multi_query_bf16_pages():
    _run_multi(16, 16, 3, [3, 64, 700, 1500], seed=66)
