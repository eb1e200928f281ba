"""Writer kernel vs the oracle writer: bit-exact page bytes and bf16 buffers."""

import numpy as np
import pytest

import oracle
from tests.gpu_util import GpuRun, oracle_model, to_dev
from workloads import synthetic as syn

pytestmark = pytest.mark.gpu


def _compare_sequence(run, b, s):
    model, L = oracle_model(run, b, s)
    pages = run.pages_of(b, L)
    got = run.cache.pool[run.torch.from_numpy(pages.astype(np.int64)).to(run.dev)].cpu().numpy()
    assert np.array_equal(got, model.pool[pages]), f"pages of sequence {b} differ"
    if run.w.content_bits != 16:
        sink = run.cache.sink[b].cpu().view(run.torch.int16).numpy().view(np.uint16)
        rec = run.cache.recent[b].cpu().view(run.torch.int16).numpy().view(np.uint16)
        n_sink = min(L, 4)
        assert np.array_equal(sink[:n_sink], model.sink[b, :n_sink])
        for t in range(max(4, L - 128), L):
            assert np.array_equal(rec[t % 128], model.recent[b, t % 128]), f"ring slot of {t}"


@pytest.mark.parametrize("cb,rb", [(4, 4), (2, 4), (16, 16)])
def test_writer_bitexact_small_batch(cb, rb):
    w = syn.custom("wr", [1, 5, 133, 300, 777, 64, 65], heads=16, content_bits=cb, rope_bits=rb,
                   steps=3, seed=21)
    run = GpuRun(w)
    run.prefill()
    for s in range(3):
        run.run_step(s)
    assert run.cache.error() == 0
    for b in range(w.batch):
        _compare_sequence(run, b, 2)


def _edge_tokens(n_rep=3):
    """Hand-made groups: constant, exact grids, ties, signed zeros, extremes, tiny."""
    rows = []
    rows.append(np.zeros(64, np.float32))                         # constant zero
    rows.append(np.full(64, -3.5, np.float32))                    # constant non-zero
    r = np.zeros(64, np.float32); r[1] = 15.0
    r[2:9] = [2.5, 3.5, 0.5, 1.5, 14.5, 7.5, 8.5]; rows.append(r)  # ties at s = 1
    r = -2.0 + 0.25 * (np.arange(64) % 16); rows.append(r.astype(np.float32))  # exact grid
    r = np.zeros(64, np.float32); r[3] = -0.0; r[7] = 2.0; rows.append(r)    # -0 minimum
    r = np.linspace(-65280, 65280, 64).astype(np.float32); rows.append(r)    # extremes (bf16-exact ends)
    r = (np.arange(64, dtype=np.float32) - 32) * 1e-39; rows.append(r)       # subnormals
    r = np.full(64, 1e-30, np.float32); r[0] = -1e-30; rows.append(r)
    rng = np.random.default_rng(4)
    r = (rng.standard_normal(64) * 1e4).astype(np.float32); rows.append(r)
    r = np.zeros(64, np.float32); r[0] = 65280.0; r[1] = -65280.0; rows.append(r)
    r = np.array([(-1) ** k * 2.0 ** (-k) for k in range(64)], np.float32); rows.append(r)
    base = np.stack(rows)                                   # [R][64]
    toks = []
    for k in range(n_rep * len(rows)):
        groups = [base[(k + i) % len(rows)] for i in range(9)]
        toks.append(np.concatenate(groups))
    x = np.stack(toks)
    bits = syn.bf16_bits_from_f32(x)
    return bits[:, :512].copy(), bits[:, 512:].copy()


@pytest.mark.parametrize("cb", [4, 2])
def test_writer_bitexact_edge_values(cb):
    import torch
    ckv, kr = _edge_tokens()
    n = ckv.shape[0]
    table = np.arange((n + 63) // 64 + 1, dtype=np.int32)[None, :][:, ::-1].copy()
    npages = table.shape[1]
    import bit_mla_kv_lowbit_gb300 as pkg
    cache = pkg.PagedCache(cb, 4, table, npages)
    cache.write(to_dev(ckv, torch.bfloat16), to_dev(kr, torch.bfloat16),
                torch.arange(n, dtype=torch.int32, device="cuda"),
                seq_idx=torch.zeros(n, dtype=torch.int32, device="cuda"),
                seq_lens_after=torch.tensor([n], dtype=torch.int32, device="cuda"))
    torch.cuda.synchronize()
    assert cache.error() == 0
    model = oracle.PagedCacheModel(oracle.Layout(cb, 4), npages, table)
    model.write(np.zeros(n, int), np.arange(n), ckv, kr, [n])
    got = cache.pool.cpu().numpy()
    diff = np.nonzero(got != model.pool)
    assert diff[0].size == 0, f"first differing bytes at {list(zip(*diff))[:5]}"


def test_writer_device_errors_skip_work():
    import torch
    import bit_mla_kv_lowbit_gb300 as pkg
    table = np.array([[0, 1], [2, -1]], dtype=np.int32)
    cache = pkg.PagedCache(4, 4, table, 3)
    ckv = torch.ones(4, 512, dtype=torch.bfloat16, device="cuda")
    kr = torch.ones(4, 64, dtype=torch.bfloat16, device="cuda")
    # token 0: fine; 1: page -1; 2: position past the table; 3: sequence 7
    seq = torch.tensor([0, 1, 0, 7], dtype=torch.int32, device="cuda")
    pos = torch.tensor([3, 70, 128, 0], dtype=torch.int32, device="cuda")
    cache.write(ckv, kr, pos, seq_idx=seq)
    torch.cuda.synchronize()
    err = cache.error()
    assert err & pkg.binding.DEV_BAD_PAGE and err & pkg.binding.DEV_BAD_POS
    assert err & pkg.binding.DEV_BAD_SEQ
    pool = cache.pool.cpu().numpy()
    assert pool[0].any() and not pool[1].any() and not pool[2].any()
