"""The alternative split kernels vs the fp64 oracle: the hybrid mma.sync +
tcgen05 kernel (MLA_LOWBIT_DECODE=hy), the all-tcgen05 kernel
(MLA_LOWBIT_DECODE=tc) and the group-per-warp kernel (MLA_LOWBIT_DECODE=gw);
the default kernel is covered by test_gpu_decode.py.

Same bar as the default kernel: max-abs error <= 2e-3 and rel-L2 <= 1e-3 per
sequence; writer bytes bit-exact.
"""

import numpy as np
import pytest

from tests.test_gpu_decode import EDGE_LENGTHS, _check_run_step, _full
from tests.gpu_util import GpuRun
from workloads import synthetic as syn

pytestmark = pytest.mark.gpu


@pytest.fixture(params=["hy", "tc", "gw"], autouse=True)
def kernel(request, monkeypatch):
    monkeypatch.setenv("MLA_LOWBIT_DECODE", request.param)
    return request.param


@pytest.mark.parametrize("cb", [4, 2])
def test_kernel_edge_lengths_16_heads(cb):
    w = syn.custom(f"k_edge_c{cb}", EDGE_LENGTHS, heads=16, content_bits=cb, rope_bits=4, seed=41)
    run = GpuRun(w)
    run.prefill()
    _check_run_step(run, 0, lse=True)


def test_kernel_head_counts_128():
    w = syn.custom("k_heads128", [133, 700, 2500], heads=128, content_bits=4, seed=42)
    run = GpuRun(w)
    run.prefill()
    _check_run_step(run, 0, lse=True)


def test_kernel_full_v2lite_all_sequences():
    _full("v2lite_c4r4")


def test_kernel_full_long_c4r4_sampled():
    _full("long_c4r4", seqs=[2])


def test_kernel_full_mixed_c2r4():
    w = syn.get("mixed_c2r4")
    lens = syn.sequence_lengths(w)
    _full("mixed_c2r4", steps=(0, 3), seqs=[int(np.argmin(lens)), int(np.argmax(lens)), 17])
