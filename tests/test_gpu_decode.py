"""Decode kernels vs the fp64 oracle on the same dequantised cache.

Bar (from the workload definition): max-abs error <= 2e-3 and rel-L2 <= 1e-3
per sequence, over all heads and channels; writer bytes bit-exact.
"""

import math

import numpy as np
import pytest

import oracle
from tests.gpu_util import GpuRun, check_attention, oracle_model, to_dev
from workloads import synthetic as syn

pytestmark = pytest.mark.gpu

EDGE_LENGTHS = [1, 2, 4, 5, 63, 64, 65, 100, 131, 132, 133, 134, 192, 196, 197, 200, 260, 1000,
                1500, 4099]


def _check_run_step(run, s, seqs=None, lse=None, fused=False):
    out, lse_got = run.run_step(s, lse=lse is not None, fused=fused)
    assert run.cache.error() == 0, f"device error word {run.cache.error()}"
    seqs = range(run.w.batch) if seqs is None else seqs
    for b in seqs:
        model, L = oracle_model(run, b, s)
        pages = run.pages_of(b, L)
        got_pages = run.cache.pool[run.torch.from_numpy(pages.astype(np.int64)).to(run.dev)]
        assert np.array_equal(got_pages.cpu().numpy(), model.pool[pages]), f"writer bytes, seq {b}"
        q = syn.queries(run.w, b)[s]
        ref, ref_lse = oracle.mla_decode_fp64(q, model.effective_keys(b, L), run.w.softmax_scale,
                                              rotate=run.rotate)
        check_attention(out[b], ref, f"{run.w.name} seq {b} (L={L}) step {s}")
        if lse_got is not None:
            assert np.allclose(lse_got[b], ref_lse, rtol=0, atol=1e-4), f"lse seq {b}"
    return out


@pytest.mark.parametrize("cb,rb", [(4, 4), (2, 4), (16, 16)])
def test_edge_lengths_16_heads(cb, rb):
    w = syn.custom(f"edge_c{cb}", EDGE_LENGTHS, heads=16, content_bits=cb, rope_bits=rb, seed=31)
    run = GpuRun(w)
    run.prefill()
    _check_run_step(run, 0, lse=True)


@pytest.mark.parametrize("heads", [32, 64, 128])
def test_head_counts(heads):
    w = syn.custom(f"heads{heads}", [133, 700, 2500], heads=heads, content_bits=4, seed=32)
    run = GpuRun(w)
    run.prefill()
    _check_run_step(run, 0, lse=True)


def test_tiny_config_exact_workload():
    w = syn.get("tiny_c4r4")
    run = GpuRun(w)
    run.prefill()
    _check_run_step(run, 0, lse=True)


@pytest.mark.parametrize("cb", [4, 2])
def test_window_transition_200_steps(cb):
    # One sequence grown token by token from length 1 to 200 through the writer;
    # at every step the decode must match the oracle, so each token switches from
    # its bf16 copy to its packed copy exactly when it leaves the recent window.
    w = syn.custom(f"win_c{cb}", [1], heads=16, content_bits=cb, steps=200, seed=33)
    run = GpuRun(w)
    for s in range(200):
        seqs = [0] if (s % 7 == 0 or 120 <= s <= 140 or s == 199) else []
        if seqs:
            _check_run_step(run, s, seqs)
        else:
            run.run_step(s)


def test_zero_query_returns_mean_of_keys():
    # Closed form independent of the softmax path: all logits equal.
    import torch
    w = syn.custom("zq", [900], heads=16, content_bits=4, seed=34)
    run = GpuRun(w)
    run.prefill()
    ckv, kr, _ = run.step_inputs(0)
    L = int(run.lens[0])
    run.cache.write(to_dev(ckv, torch.bfloat16), to_dev(kr, torch.bfloat16),
                    torch.tensor([L - 1], dtype=torch.int32, device="cuda"))
    q = torch.zeros(1, 16, 576, dtype=torch.bfloat16, device="cuda")
    out = run.cache.decode(q, torch.tensor([L], dtype=torch.int32, device="cuda"), [L], 0.07)
    torch.cuda.synchronize()
    model, _ = oracle_model(run, 0, 0)
    mean = model.effective_keys(0, L)[:, :512].mean(0)
    assert np.abs(out[0].cpu().numpy() - mean[None]).max() < 1e-4


def test_empty_and_single_token_sequences():
    import torch
    import bit_mla_kv_lowbit_gb300 as pkg
    table = np.array([[0], [1]], dtype=np.int32)
    cache = pkg.PagedCache(4, 4, table, 2)
    ckv = torch.randn(1, 512, device="cuda").to(torch.bfloat16)
    kr = torch.randn(1, 64, device="cuda").to(torch.bfloat16)
    cache.write(ckv, kr, torch.tensor([0], dtype=torch.int32, device="cuda"),
                seq_idx=torch.tensor([1], dtype=torch.int32, device="cuda"))
    q = torch.randn(2, 16, 576, device="cuda").to(torch.bfloat16)
    lse = torch.empty(2, 16, device="cuda")
    out = cache.decode(q, torch.tensor([0, 1], dtype=torch.int32, device="cuda"), [0, 1], 0.07,
                       lse=lse)
    torch.cuda.synchronize()
    assert cache.error() == 0
    assert not out[0].any() and torch.isneginf(lse[0]).all()
    assert torch.allclose(out[1], ckv.float().expand(16, 512), atol=1e-6, rtol=0)


def test_bad_page_sets_error_and_stays_finite():
    import torch
    w = syn.custom("badpage", [700], heads=16, content_bits=4, seed=35)
    run = GpuRun(w)
    run.prefill()
    run.run_step(0)
    run.cache.clear_error()
    bt = run.cache.block_table.clone()
    run.cache.block_table[0, 3] = -5
    _, _, q = run.step_inputs(0)
    L = int(run.lens[0])
    out = run.cache.decode(to_dev(q, torch.bfloat16), torch.tensor([L], dtype=torch.int32,
                                                                    device="cuda"), [L], 0.07)
    torch.cuda.synchronize()
    run.cache.block_table.copy_(bt)
    assert run.cache.error() & 4
    assert torch.isfinite(out).all()


def test_host_device_length_mismatch_is_reported():
    import torch
    w = syn.custom("mismatch", [700, 300], heads=16, content_bits=4, seed=36)
    run = GpuRun(w)
    run.prefill()
    run.run_step(0)
    run.cache.clear_error()
    _, _, q = run.step_inputs(0)
    lens_host = [int(x) for x in run.lens]
    lens_dev = torch.tensor([run.lens[0], run.lens[1] + 200], dtype=torch.int32, device="cuda")
    ws = run.cache.workspace(16, [int(run.lens[0]), int(run.lens[1]) + 200])
    run.cache.decode(to_dev(q, torch.bfloat16), lens_dev, lens_host, 0.07, workspace=ws)
    torch.cuda.synchronize()
    assert run.cache.error() & 16


# ---------------------------------------------------------------- full sizes

def _full(name, steps=(0,), seqs=None):
    w = syn.get(name)
    run = GpuRun(w)
    run.prefill(keep_tokens=True)
    for s in range(max(steps) + 1):
        if s in steps:
            _check_run_step(run, s, seqs)
        else:
            run.run_step(s)


def test_full_v2lite_all_sequences():
    _full("v2lite_c4r4")


def test_full_v3_sampled_sequences():
    _full("v3_c4r4", seqs=[0, 13, 31])


@pytest.mark.parametrize("name", ["long_c4r4", "long_bf16", "long16_c4r4", "long16_bf16"])
def test_full_long_context_sampled(name):
    _full(name, seqs=[2])


@pytest.mark.parametrize("cb", [4, 2])
def test_quarter_million_tokens(cb):
    # past the 128K configurations: 262,144 cached tokens in one sequence (4,096
    # pages, the most splits per sequence the planner makes for 16 heads);
    # writer bytes bit-exact over the whole pool, decode within the bar, error
    # word 0, guard bytes intact
    w = syn.custom(f"q262k_c{cb}", [262144], heads=16, content_bits=cb, rope_bits=4, seed=37)
    run = GpuRun(w)
    run.prefill(keep_tokens=True)
    _check_run_step(run, 0, lse=True)


def test_full_mixed_c2r4_sixteen_steps():
    w = syn.get("mixed_c2r4")
    lens = syn.sequence_lengths(w)
    seqs = [int(np.argmin(lens)), int(np.argmax(lens)), 17]
    _full("mixed_c2r4", steps=(0, 7, 15), seqs=seqs)
