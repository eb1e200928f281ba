"""The allocation-free decode entry point against the regular one.

mla_lowbit_decode_noalloc serves hosts that may not allocate device memory
(their cache pool already holds nearly all of HBM, or their plug-in interface
has no workspace argument): it keeps the split partials in a fixed array the
library owns.  Two calls in a row, each checked against mla_lowbit_decode on
the same inputs within the parity tolerance, show that the shared array's
leftover contents from the previous call do not leak into the next one.

This file is named to be collected last.
"""

import ctypes

import numpy as np
import pytest

from tests.gpu_util import GpuRun, MAX_ABS, REL_L2, to_dev
from workloads import synthetic as syn

pytestmark = pytest.mark.gpu


def _close(a, b):
    a = a.double().cpu().numpy()
    b = b.double().cpu().numpy()
    err = np.abs(a - b).max()
    rel = np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-30)
    assert np.all(np.isfinite(a)) and err <= MAX_ABS and rel <= REL_L2, (err, rel)


def test_noalloc_matches_workspace_decode_twice():
    import torch
    import bit_mla_kv_lowbit_gb300 as pkg
    w = syn.custom("noalloc", [5000, 133, 2100, 77], heads=16, content_bits=4, steps=2, seed=41)
    run = GpuRun(w)
    run.prefill()
    for s in range(2):
        ckv, kr, q = run.step_inputs(s)
        lens_now = (run.lens + s).astype(np.int32)
        run.cache.write(to_dev(ckv, torch.bfloat16), to_dev(kr, torch.bfloat16),
                        to_dev((run.lens - 1 + s).astype(np.int32), torch.int32),
                        seq_lens_after=to_dev(lens_now, torch.int32))
        qd = to_dev(q, torch.bfloat16)
        lens_d = to_dev(lens_now, torch.int32)
        B, H = w.batch, w.heads
        ref = torch.empty(B, H, 512, device="cuda")
        ref_lse = torch.empty(B, H, device="cuda")
        run.cache.decode(qd, lens_d, lens_now, w.softmax_scale, out=ref, lse=ref_lse)
        got = torch.full((B, H, 512), float("nan"), device="cuda")
        got_lse = torch.full((B, H), float("nan"), device="cuda")
        pkg.decode_noalloc(run.cache.layout, qd, run.cache.pool, run.cache.block_table, lens_d,
                           lens_now, run.cache.sink, run.cache.recent, got, run.cache.err,
                           w.softmax_scale, lse=got_lse)
        torch.cuda.synchronize()
        assert run.cache.error() == 0
        _close(got, ref)
        _close(got_lse, ref_lse)


def test_noalloc_rejects_plans_beyond_its_array():
    import bit_mla_kv_lowbit_gb300 as pkg
    lay = pkg.layout(4, 4)
    # 128 heads over many long sequences: the plan's workspace exceeds 32 MiB.
    lens = np.full(256, 131072, np.int32)
    _, _, need = pkg.decode_plan(lay, 128, lens)
    assert need > (32 << 20)
    lib = pkg.load()
    st = lib.mla_lowbit_decode_noalloc(ctypes.byref(lay), len(lens), 128, ctypes.c_float(0.07),
                                       0x1000, 0x2000, 1, 0x3000, 2048, 0x4000,
                                       lens.ctypes.data_as(ctypes.c_void_p), 0x5000, 0x6000,
                                       0x7000, None, 0x8000, None)
    assert st == -4 and "size" in pkg.strerror(st)
