"""Two GPUs in one process: the kernels' shared-memory limits are per-device
attributes, and every call runs on the device of its page pool whatever the
current device is.  Decodes on the second device after the first (16 and 128
heads) must match the oracle.  Needs two visible GPUs; skipped otherwise."""

import pytest

from tests.gpu_util import GpuRun
from tests.test_gpu_decode import _check_run_step
from workloads import synthetic as syn

pytestmark = pytest.mark.gpu


def _two_gpus():
    import torch
    return torch.cuda.is_available() and torch.cuda.device_count() >= 2


@pytest.mark.skipif(not _two_gpus(), reason="needs two visible GPUs")
@pytest.mark.parametrize("heads", [16, 128])
def test_second_device_after_first(heads):
    import torch
    w = syn.custom(f"dev2_h{heads}", [700, 2100, 140], heads=heads, content_bits=4, seed=53)
    for dev in ("cuda:0", "cuda:1"):
        torch.cuda.set_device(0)  # the current device stays the first one
        run = GpuRun(w, dev=dev)
        run.prefill()
        _check_run_step(run, 0, lse=True)


@pytest.mark.skipif(not _two_gpus(), reason="needs two visible GPUs")
def test_tensors_on_another_device_are_rejected():
    import torch
    w = syn.custom("dev2_mix", [300], heads=16, content_bits=4, seed=54)
    run = GpuRun(w, dev="cuda:0")
    run.prefill()
    q1 = torch.zeros(1, 16, 576, dtype=torch.bfloat16, device="cuda:1")
    lens = [int(x) for x in run.lens]
    with pytest.raises(ValueError, match="page pool"):
        run.cache.decode(q1, torch.tensor(lens, dtype=torch.int32, device="cuda:0"), lens,
                         w.softmax_scale)
