"""The multi-GPU path of bench.py with two ranks on CPU (gloo): the decode
shards a seeded global batch by sequence (global sequence g on rank g mod N)
with no data-path collective; the only communication is the barrier and the
max over ranks of the step times.  Whole-job throughput counts the tokens of
every rank."""

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


def test_sequence_shards_cover_the_global_batch_once():
    # Each rank builds only its sequences' lengths, pages and block table; the
    # union over ranks is the global batch exactly once, each shard carries the
    # global values of its sequences, and the oracle's outputs of the shards,
    # put back in global order, are the single-rank result.
    outs = _run_ranks("""
        import json
        import numpy as np
        import torch
        import torch.distributed as dist
        import oracle
        from workloads import synthetic as syn
        dist.init_process_group("gloo")
        r, n = dist.get_rank(), dist.get_world_size()
        w = syn.get("tiny_c4r4").with_(name="tiny_u", batch=3, length_kind="uniform",
                                        length_args=(140, 400), seed=17)
        sh = syn.shard_workload(w, r, n)
        glob = w.with_(batch=w.batch * n)
        ids = list(sh.seq_ids)
        # every rank's ids, gathered
        allids = [None] * n
        dist.all_gather_object(allids, ids)
        # this shard against the global draw: lengths and token values
        gl = syn.sequence_lengths(glob)
        lens = syn.sequence_lengths(sh)
        assert [int(x) for x in lens] == [int(gl[g]) for g in ids]
        table, npages = syn.make_paging(sh)
        assert table.shape[0] == len(ids) and table.max() < npages
        for b, g in enumerate(ids):
            t_s, k_s = syn.sequence_tokens(sh, b)
            t_g, k_g = syn.sequence_tokens(glob, g)
            assert np.array_equal(t_s, t_g) and np.array_equal(k_s, k_g)
            assert np.array_equal(syn.queries(sh, b), syn.queries(glob, g))
        # the oracle decode of every shard sequence on this rank's own cache
        model = oracle.PagedCacheModel(oracle.Layout(4, 4), npages, table)
        outs = {}
        for b, g in enumerate(ids):
            L = int(lens[b])
            ckv, kr = syn.sequence_tokens(sh, b)
            la = np.zeros(len(ids), np.int64)
            la[b] = L
            model.write(np.full(L, b), np.arange(L), ckv, kr, la)
            o, _ = oracle.mla_decode_fp64(syn.queries(sh, b)[0], model.effective_keys(b, L),
                                          w.softmax_scale)
            outs[g] = o.tolist()
        gathered = [None] * n
        dist.all_gather_object(gathered, outs)
        if r == 0:
            merged = {}
            for d in gathered:
                merged.update({int(k): v for k, v in d.items()})
            print(json.dumps({"ids": allids, "outs": merged}))
        dist.destroy_process_group()
    """, timeout=300)
    import json

    import numpy as np

    import oracle
    from workloads import synthetic as syn
    res = json.loads(outs[0].strip().splitlines()[-1])
    flat = [g for ids in res["ids"] for g in ids]
    assert sorted(flat) == list(range(6)) and len(flat) == len(set(flat))   # once each
    assert res["ids"] == [[0, 2, 4], [1, 3, 5]]                              # g mod N
    # single-rank reference: the global batch on one cache
    w = syn.get("tiny_c4r4").with_(name="tiny_u", batch=6, length_kind="uniform",
                                    length_args=(140, 400), seed=17)
    table, npages = syn.make_paging(w)
    model = oracle.PagedCacheModel(oracle.Layout(4, 4), npages, table)
    lens = syn.sequence_lengths(w)
    for g in range(6):
        L = int(lens[g])
        ckv, kr = syn.sequence_tokens(w, g)
        la = np.zeros(6, np.int64)
        la[g] = L
        model.write(np.full(L, g), np.arange(L), ckv, kr, la)
        ref, _ = oracle.mla_decode_fp64(syn.queries(w, g)[0], model.effective_keys(g, L),
                                        w.softmax_scale)
        assert np.array_equal(np.asarray(res["outs"][str(g)]), ref)
