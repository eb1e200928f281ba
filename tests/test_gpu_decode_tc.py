"""The tcgen05 split kernel (selected with MLA_LOWBIT_DECODE=tc) vs the fp64 oracle.

Same bar as the default kernel: max-abs error <= 2e-3 and rel-L2 <= 1e-3 per
sequence; writer bytes bit-exact.
"""

import pytest

from tests.test_gpu_decode import EDGE_LENGTHS, _check_run_step, _full
from tests.gpu_util import GpuRun
from workloads import synthetic as syn

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _tc_kernel(monkeypatch):
    monkeypatch.setenv("MLA_LOWBIT_DECODE", "tc")


@pytest.mark.parametrize("cb", [4, 2])
def test_tc_edge_lengths_16_heads(cb):
    w = syn.custom(f"tc_edge_c{cb}", EDGE_LENGTHS, heads=16, content_bits=cb, rope_bits=4, seed=41)
    run = GpuRun(w)
    run.prefill()
    _check_run_step(run, 0, lse=True)


def test_tc_head_counts_128():
    w = syn.custom("tc_heads128", [133, 700, 2500], heads=128, content_bits=4, seed=42)
    run = GpuRun(w)
    run.prefill()
    _check_run_step(run, 0, lse=True)


def test_tc_full_v2lite_all_sequences():
    _full("v2lite_c4r4")


def test_tc_full_long_c4r4_sampled():
    _full("long_c4r4", seqs=[2])


def test_tc_full_mixed_c2r4():
    w = syn.get("mixed_c2r4")
    lens = syn.sequence_lengths(w)
    import numpy as np
    _full("mixed_c2r4", steps=(0, 3), seqs=[int(np.argmin(lens)), int(np.argmax(lens)), 17])
