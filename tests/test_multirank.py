"""The replica path of bench.py with two ranks on CPU (gloo): the decode path
shards by sequence with no data-path collective, so N GPUs run N replicas and
the only communication is the barrier and the max over ranks of the step
times.  Whole-job throughput counts the tokens of every rank."""

import os
import socket
import subprocess
import sys
import textwrap

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _run_ranks(body: str, world: int = 2, timeout: int = 120):
    port = _free_port()
    script = textwrap.dedent(body)
    procs = []
    for r in range(world):
        env = dict(os.environ, RANK=str(r), LOCAL_RANK=str(r), WORLD_SIZE=str(world),
                   MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), PYTHONPATH=ROOT)
        procs.append(subprocess.Popen([sys.executable, "-c", script], cwd=ROOT, env=env,
                                      stdout=subprocess.PIPE, stderr=subprocess.PIPE, text=True))
    outs = []
    for p in procs:
        try:
            out, err = p.communicate(timeout=timeout)
        finally:
            if p.poll() is None:
                p.kill()
        assert p.returncode == 0, err
        outs.append(out)
    return outs


def test_max_over_ranks_and_whole_job_throughput():
    outs = _run_ranks("""
        import os, json
        import torch.distributed as dist
        import bench
        dist.init_process_group("gloo")
        r = dist.get_rank()
        # rank r measured step r + 1 ms and decode 2 - r ms
        t = bench.reduce_max_over_ranks([r + 1.0, 2.0 - r], dist, "cpu")
        tok = bench.whole_job_tokens_per_s(dist.get_world_size(), 8, t[0])
        print(json.dumps({"rank": r, "t": t, "tok": tok}))
        dist.destroy_process_group()
    """)
    import json
    res = [json.loads(o.strip().splitlines()[-1]) for o in outs]
    for d in res:
        assert d["t"] == [2.0, 2.0]          # every rank sees the slowest rank's times
        assert d["tok"] == 2 * 8 / 2e-3      # both ranks' sequences over the max time


def test_reference_arm_runs_on_rank_zero_only():
    outs = _run_ranks("""
        import sys
        import bench
        sys.argv = ["bench.py", "--impl", "reference", "--workload", "tiny_c4r4",
                    "--steps", "1", "--warmup", "0"]
        bench.main()
    """, timeout=300)
    import json
    line = json.loads(outs[0].strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["n_gpus"] == 2
    assert outs[1].strip() == ""             # the other rank exits without work or output
