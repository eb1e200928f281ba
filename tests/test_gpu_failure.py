"""Failure detection of the tcgen05 decode kernels, made on purpose without a
GPU fault: every mbarrier wait is bounded, and a self-test setting withholds
one hand-off between warp roles so that the waits behind it run out after a
short limit.  The call must return, report MLA_LOWBIT_DEV_PIPELINE in the
device error word, and leave the context usable: the next normal decode in
the same process matches the oracle (tensor memory was freed, the drained
MMAs left nothing behind).  Also the device-side checks of the 128-row kernel
on bad inputs: a block-table entry outside the pool and device lengths that
disagree with the host plan."""

import numpy as np
import pytest

from tests.gpu_util import GpuRun, to_dev
from tests.test_gpu_decode import _check_run_step
from workloads import synthetic as syn

pytestmark = pytest.mark.gpu

PIPELINE = 32


@pytest.mark.parametrize("cb", [4, 16])
def test_bounded_wait_runs_out_and_context_recovers(cb):
    import torch
    import bit_mla_kv_lowbit_gb300 as pkg
    w = syn.custom(f"fault128_c{cb}", [700, 2100, 140], heads=128, content_bits=cb,
                   rope_bits=16 if cb == 16 else 4, steps=2, seed=91)
    run = GpuRun(w)
    run.prefill()
    run.run_step(0)
    assert run.cache.error() == 0
    _, _, q = run.step_inputs(0)
    lens = [int(x) for x in run.lens]
    try:
        # about 1 ms of SM cycles instead of about 1 s
        pkg.set_fault_injection(1, 2_000_000)
        out = run.cache.decode(to_dev(q, torch.bfloat16),
                               to_dev(np.asarray(lens, np.int32), torch.int32), lens,
                               w.softmax_scale)
        torch.cuda.synchronize()
        err = run.cache.error()
    finally:
        pkg.set_fault_injection(0, 0)
    assert err & PIPELINE, f"error word {err}: the bounded wait did not report"
    assert torch.isfinite(out).all()
    # the same process decodes correctly afterwards
    run.cache.clear_error()
    _check_run_step(run, 1, lse=True)


def test_fault_setting_is_validated():
    import bit_mla_kv_lowbit_gb300 as pkg
    with pytest.raises(pkg.LibraryError):
        pkg.set_fault_injection(2, 0)
    with pytest.raises(pkg.LibraryError):
        pkg.set_fault_injection(0, -1)
    pkg.set_fault_injection(0, 0)


@pytest.mark.parametrize("cb", [4, 16])
def test_bad_page_128_rows(cb):
    import torch
    w = syn.custom(f"badpage128_c{cb}", [700], heads=128, content_bits=cb,
                   rope_bits=16 if cb == 16 else 4, seed=92)
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


@pytest.mark.parametrize("cb", [4, 16])
def test_host_device_length_mismatch_128_rows(cb):
    import torch
    w = syn.custom(f"mismatch128_c{cb}", [700, 300], heads=128, content_bits=cb,
                   rope_bits=16 if cb == 16 else 4, seed=93)
    run = GpuRun(w)
    run.prefill()
    run.run_step(0)
    run.cache.clear_error()
    _, _, q = run.step_inputs(0)
    lens_host = [int(x) for x in run.lens]
    lens_dev = torch.tensor([run.lens[0], run.lens[1] + 200], dtype=torch.int32, device="cuda")
    ws = run.cache.workspace(128, [int(run.lens[0]), int(run.lens[1]) + 200])
    run.cache.decode(to_dev(q, torch.bfloat16), lens_dev, lens_host, 0.07, workspace=ws)
    torch.cuda.synchronize()
    assert run.cache.error() & 16
