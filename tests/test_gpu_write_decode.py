"""mla_lowbit_write_decode (append + decode in one call) against the separate
writer + decode calls and against the fp64 oracle.

The fused call must leave the same pool bytes and bf16 buffers and return the
same output and lse as mla_lowbit_write followed by mla_lowbit_decode (the
arithmetic is the same; only where the new token's bf16 values are read
from differs)."""

import numpy as np
import pytest

from tests.gpu_util import GpuRun
from tests.test_gpu_decode import _check_run_step
from workloads import synthetic as syn

pytestmark = pytest.mark.gpu

LENGTHS = [1, 2, 4, 5, 64, 131, 132, 133, 197, 1000, 4099]


def _pair(cb, heads, seed):
    w = syn.custom(f"wd_c{cb}_h{heads}", LENGTHS, heads=heads, content_bits=cb,
                   rope_bits=4 if cb != 16 else 16, seed=seed)
    a, b = GpuRun(w), GpuRun(w)
    a.prefill()
    b.prefill()
    return a, b


@pytest.mark.parametrize("cb,heads", [(4, 16), (2, 16), (4, 32), (16, 16)])
def test_fused_equals_separate(cb, heads):
    a, b = _pair(cb, heads, seed=51)
    out_a, lse_a = a.run_step(0, lse=True)
    out_b, lse_b = b.run_step(0, lse=True, fused=True)
    assert a.cache.error() == 0 and b.cache.error() == 0
    t = a.torch
    assert t.equal(a.cache.pool, b.cache.pool), "pool bytes differ"
    if cb != 16:
        assert t.equal(a.cache.sink, b.cache.sink), "sink buffer differs"
        assert t.equal(a.cache.recent, b.cache.recent), "recent ring differs"
    assert np.array_equal(out_a, out_b)
    assert np.array_equal(lse_a, lse_b)


@pytest.mark.parametrize("cb,heads", [(4, 128), (2, 128)])
def test_unfused_kernels_take_the_writer_path(cb, heads):
    # the 128-row kernel appends with the writer kernel first: same results
    a, b = _pair(cb, heads, seed=52)
    out_a, _ = a.run_step(0)
    out_b, _ = b.run_step(0, fused=True)
    assert a.cache.error() == 0 and b.cache.error() == 0
    assert a.torch.equal(a.cache.pool, b.cache.pool)
    assert a.torch.equal(a.cache.recent, b.cache.recent)
    assert np.array_equal(out_a, out_b)


@pytest.mark.parametrize("cb", [4, 2])
def test_fused_window_transition_vs_oracle(cb):
    # one sequence grown from length 1 to 160 only through the fused call
    w = syn.custom(f"wd_win_c{cb}", [1], heads=16, content_bits=cb, steps=160, seed=53)
    run = GpuRun(w)
    for s in range(160):
        if s % 9 == 0 or 126 <= s <= 134 or s == 159:
            _check_run_step(run, s, [0], lse=True, fused=True)
        else:
            run.run_step(s, fused=True)
