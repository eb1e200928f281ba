"""Randomised decode configurations against the fp64 oracle.

The twelve cases cover every (layout, head count) pair of C4R4, C2R4 and bf16
pages with 16, 32, 64 and 128 heads (so both the 16-row kernel and the 128-row
cluster kernel run); each draws from its own seed a batch of 1-3 sequences and
log-uniform lengths from 1 to 8,000 tokens.  The cache is filled through the
writer and one decode step is checked: writer bytes bit-exact, attention within
max-abs 2e-3 / rel-L2 1e-3, lse within 1e-4, device error word 0."""

import numpy as np
import pytest

from tests.gpu_util import GpuRun
from tests.test_gpu_decode import _check_run_step
from workloads import synthetic as syn

pytestmark = pytest.mark.gpu

LAYOUTS = [(4, 4), (2, 4), (16, 16)]
HEADS = [16, 32, 64, 128]


def _draw(seed):
    rng = np.random.default_rng(1000 + seed)
    cb, rb = LAYOUTS[(seed // len(HEADS)) % len(LAYOUTS)]
    heads = HEADS[seed % len(HEADS)]
    batch = int(rng.integers(1, 4))
    lens = np.exp(rng.uniform(0.0, np.log(8000.0), batch)).astype(int).clip(1, 8000)
    return cb, rb, heads, [int(x) for x in lens]


@pytest.mark.parametrize("seed", range(12))
def test_random_config(seed):
    cb, rb, heads, lens = _draw(seed)
    w = syn.custom(f"rand{seed}_c{cb}_h{heads}", lens, heads=heads, content_bits=cb, rope_bits=rb,
                   seed=200 + seed)
    run = GpuRun(w)
    run.prefill()
    _check_run_step(run, 0, lse=True)


def test_draws_cover_both_kernels_and_every_layout():
    draws = [_draw(s) for s in range(12)]
    assert {(d[0], d[2]) for d in draws} == {(cb, h) for cb, _ in LAYOUTS for h in HEADS}


# multi-token query decode: (layout, heads, queries per sequence) so that the
# query rows per sequence are 32, 64 (16-row kernel) and 128, 256 (cluster kernel)
MULTI = [(4, 16, 2), (2, 16, 4), (4, 16, 8), (16, 32, 4), (4, 128, 2), (2, 64, 2)]


@pytest.mark.parametrize("case", range(len(MULTI)))
def test_random_multi_query(case):
    from tests.test_gpu_decode_multi import _run_multi
    cb, heads, n = MULTI[case]
    rng = np.random.default_rng(2000 + case)
    batch = int(rng.integers(1, 4))
    # every sequence holds at least its n query tokens
    lens = np.exp(rng.uniform(np.log(n), np.log(6000.0), batch)).astype(int).clip(n, 6000)
    _run_multi(cb, heads, n, [int(x) for x in lens], seed=300 + case)


@pytest.mark.parametrize("seed", range(4))
def test_random_rotated(seed):
    # the rotated cache (writer rotation, rotated queries, output rotated back)
    rng = np.random.default_rng(3000 + seed)
    cb = (4, 2)[seed % 2]
    heads = (16, 128)[seed // 2]
    batch = int(rng.integers(1, 4))
    lens = np.exp(rng.uniform(0.0, np.log(6000.0), batch)).astype(int).clip(1, 6000)
    w = syn.custom(f"randrot{seed}_c{cb}_h{heads}", [int(x) for x in lens], heads=heads,
                   content_bits=cb, seed=400 + seed)
    run = GpuRun(w, rotate=True)
    run.prefill()
    _check_run_step(run, 0, lse=True)
