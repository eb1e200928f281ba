"""Benchmark: low-bit MLA decode step on one GB300 (or N sequence shards under
torchrun).

One step = the split-KV decode (+ log-sum-exp combine) over the whole cache of
the long-context C4R4 workload: 4 sequences x 131072 tokens, 128 heads sharing
one latent (512) + RoPE (64) cache, 64-token pages in random physical order
(the 128K configuration of the low-bit MLA decode benchmarks), unless
``--workload`` names another; workloads with the writer in the step append one
token per sequence first.  The same line reports, under ``configs``, the same
step on bf16 pages, with 16 heads, and on the 32K DeepSeek-V2-Lite shape.
Inputs are synthetic and seeded (workloads/).  Under torchrun each rank decodes
its own shard of a global batch (world x batch sequences), no collective.

Prints one JSON line.  ``--impl reference`` times the CPU oracle instead (the
reference arm; bounded sample of the same workload).
"""

from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from workloads import synthetic as syn  # noqa: E402

METRIC = "C4R4 MLA decode: tokens/s and packed-cache HBM GB/s (% of peak) at 1 GPU"
L2_FLUSH_BYTES = 512 << 20


# ---------------------------------------------------------------- helpers

def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


def tensor_peak():
    """Dense fp16/bf16 tensor peak in TFLOP/s (the same rate for both types):
    the measured burst figure, else the fallback."""
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return float(json.load(f)["bf16_tflops"]), "measured"
    except Exception:
        return 1900.0, "fallback"


def algorithmic_flops(w: syn.Workload, lens) -> float:
    """Flops the decode must do per step: QK over 576 channels and PV over 512
    for every cached token and head (2 flops per multiply-add)."""
    return 2.0 * w.heads * (576 + 512) * float(np.sum(lens))


def percentiles(xs, qs=(10, 50, 90)):
    ys = sorted(xs)
    return {f"p{q}": round(ys[min(len(ys) - 1, int(round(q / 100 * (len(ys) - 1))))], 5) for q in qs}


def algorithmic_bytes(w: syn.Workload, lens) -> dict:
    """Bytes the decode must move per step, from the closed form: packed bytes of
    the packed-served tokens, bf16 bytes of the protected tokens, queries,
    outputs and block-table entries (split partials are implementation overhead
    and not counted)."""
    bpt = {4: 324, 2: 196, 16: 1152}[w.content_bits]
    packed = w.content_bits != 16
    tot = 0
    for L in lens:
        L = int(L)
        prot = min(L, 132) if packed else 0
        tot += (L - prot) * bpt + prot * 1152 + math.ceil(L / 64) * 4
    tot += w.batch * w.heads * 576 * 2 + w.batch * w.heads * 512 * 4
    writer = w.batch * (576 * 2 + bpt + (1152 if packed else 0)) if w.writer_in_step else 0
    return {"decode": tot, "writer": writer}


class ClockSampler:
    """Polls nvidia-smi (SM clock, max clock, throttle reasons) in a thread.

    Started before the warm-up; ``mark()`` brackets the timed region and the
    summary uses the samples taken inside it (or the nearest ones when the
    region is shorter than one poll)."""

    QUERY = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
             "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
             "clocks_event_reasons.sw_power_cap")
    NAMES = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]

    def __init__(self, index: int):
        self.index = index
        self.samples = []  # (t, sm, max, reasons)
        self.stop = threading.Event()
        self.window = [None, None]

    def _poll(self):
        while not self.stop.is_set():
            try:
                out = subprocess.run(["nvidia-smi", "-i", str(self.index),
                                      f"--query-gpu={self.QUERY}",
                                      "--format=csv,noheader,nounits"],
                                     capture_output=True, text=True, timeout=5).stdout
                parts = [p.strip() for p in out.strip().split(",")]
                sm, mx = float(parts[0]), float(parts[1])
                reasons = {n for n, v in zip(self.NAMES, parts[3:7]) if v.lower() == "active"}
                self.samples.append((time.perf_counter(), sm, mx, reasons))
            except Exception:
                time.sleep(0.05)

    def __enter__(self):
        self.thread = threading.Thread(target=self._poll, daemon=True)
        self.thread.start()
        return self

    def mark(self, which: int):
        self.window[which] = time.perf_counter()

    def __exit__(self, *exc):
        self.stop.set()
        self.thread.join(timeout=10)

    def summary(self):
        t0, t1 = self.window
        inside = [s for s in self.samples if t0 is not None and t0 <= s[0] <= t1]
        note = "inside timed region"
        if not inside and self.samples and t0 is not None:
            mid = 0.5 * (t0 + t1)
            inside = sorted(self.samples, key=lambda s: abs(s[0] - mid))[:3]
            note = "timed region shorter than one poll; nearest samples"
        sm = [s[1] for s in inside]
        reasons = sorted(set().union(*[s[3] for s in inside])) if inside else []
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": inside[0][2] if inside else None,
                "reasons": reasons, "samples": len(inside), "note": note}


def traffic_record(kernel_key: str):
    """DRAM bytes per launch from a committed ncu summary, only while the kernel
    sources still hash to the value recorded with it."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            rec = json.load(f).get(kernel_key)
    except Exception:
        return None
    if not rec:
        return None
    if rec.get("sources_sha256") != sources_sha256(rec.get("sources", [])):
        return None
    return rec


def sources_sha256(files):
    """Hash of the files (repo-relative) that define a captured kernel and its launch."""
    import hashlib
    h = hashlib.sha256()
    if not files:
        return None
    for name in files:
        with open(os.path.join(ROOT, name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()


# ---------------------------------------------------------------- the GPU arm

class Setup:
    def __init__(self, w: syn.Workload, dev: str, rotate: bool = False):
        import torch
        import bit_mla_kv_lowbit_gb300 as pkg
        self.torch = torch
        self.w = w
        self.dev = dev
        self.lens = syn.sequence_lengths(w).astype(np.int32)
        self.table, self.npages = syn.make_paging(w)
        self.cache = pkg.PagedCache(w.content_bits, w.rope_bits, self.table, self.npages, dev,
                                    rotate=rotate)
        scales = syn.channel_scales(w)
        B = w.batch
        new_ckv = np.empty((B, 512), np.uint16)
        new_kr = np.empty((B, 64), np.uint16)
        lens_prev = (self.lens - 1).astype(np.int32)
        lens_prev_d = torch.from_numpy(lens_prev).to(dev)
        for b in range(B):
            ckv, kr = syn.sequence_tokens(w, b, scales=scales)
            n = int(self.lens[b]) - 1
            new_ckv[b], new_kr[b] = ckv[n], kr[n]
            if n > 0:
                self.cache.write(torch.from_numpy(ckv[:n]).to(dev).view(torch.bfloat16),
                                 torch.from_numpy(kr[:n]).to(dev).view(torch.bfloat16),
                                 torch.arange(n, dtype=torch.int32, device=dev),
                                 seq_idx=torch.full((n,), b, dtype=torch.int32, device=dev),
                                 seq_lens_after=lens_prev_d)
            del ckv, kr
        q = np.stack([syn.queries(w, b)[0] for b in range(B)])
        # one pinned host buffer and one device buffer hold a step's inputs
        # (q, then the new tokens' latent and RoPE key), so the end-to-end step
        # moves them with a single host-to-device copy
        nq, nc, nk = q.size, new_ckv.size, new_kr.size
        self.h_in = torch.empty(nq + nc + nk, dtype=torch.bfloat16).pin_memory()
        self.h_in[:nq].view(torch.int16).copy_(torch.from_numpy(q.reshape(-1).view(np.int16)))
        self.h_in[nq:nq + nc].view(torch.int16).copy_(torch.from_numpy(new_ckv.reshape(-1).view(np.int16)))
        self.h_in[nq + nc:].view(torch.int16).copy_(torch.from_numpy(new_kr.reshape(-1).view(np.int16)))
        self.d_in = self.h_in.to(dev)
        self.n_in = nq + (nc + nk if w.writer_in_step else 0)  # elements copied per step
        self.h_q = self.h_in[:nq].view(q.shape)
        self.q = self.d_in[:nq].view(q.shape)
        self.ckv = self.d_in[nq:nq + nc].view(new_ckv.shape)
        self.kr = self.d_in[nq + nc:].view(new_kr.shape)
        self.pos = torch.from_numpy(self.lens - 1).to(dev)
        self.lens_d = torch.from_numpy(self.lens).to(dev)
        self.lens_h = [int(x) for x in self.lens]
        self.out = torch.empty(B, w.heads, 512, dtype=torch.float32, device=dev)
        self.h_out = torch.empty(B, w.heads, 512, dtype=torch.float32).pin_memory()
        self.ws = self.cache.workspace(w.heads, self.lens_h)
        self.flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
        torch.cuda.synchronize()
        assert self.cache.error() == 0, "device error during prefill"

    def decode(self):
        self.cache.decode(self.q, self.lens_d, self.lens_h, self.w.softmax_scale, out=self.out,
                          workspace=self.ws)

    def step(self):
        """One decode step: with the writer in the step, the append of each
        sequence's new token and the decode are one mla_lowbit_write_decode call."""
        if self.w.writer_in_step:
            self.cache.write_decode(self.ckv, self.kr, self.q, self.lens_d, self.lens_h,
                                    self.w.softmax_scale, out=self.out, workspace=self.ws)
        else:
            self.decode()

    def step_e2e(self):
        """Same step through the public API from pinned host buffers."""
        self.d_in[:self.n_in].copy_(self.h_in[:self.n_in], non_blocking=True)
        self.step()
        self.h_out.copy_(self.out, non_blocking=True)


def reduce_max_over_ranks(values, dist, device):
    """Element-wise max of per-rank values over all ranks (every rank gets the
    result); the values themselves when there is one rank."""
    if dist is None:
        return list(values)
    import torch
    t = torch.tensor(list(values), dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return t.tolist()


def whole_job_tokens_per_s(world: int, batch: int, t_ms: float) -> float:
    """Output tokens of all ranks (one per sequence per step) per second, for a
    step time that is already the max over ranks."""
    return world * batch / (t_ms * 1e-3)


def time_steps(s, step, passes: int, steps: int, warmup: int, stream, clk=None):
    """Per-step device times (ms): ``passes`` independent passes, each with its own
    warm-up, of ``steps`` timed steps; L2 is flushed (a write larger than L2)
    before every step, outside the events."""
    import torch
    out = []
    for p in range(passes):
        for _ in range(warmup):
            step()
        torch.cuda.synchronize()
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
              for _ in range(steps)]
        if clk is not None and p == 0:
            clk.mark(0)
        for i in range(steps):
            s.flush.zero_()
            ev[i][0].record(stream)
            step()
            ev[i][1].record(stream)
        torch.cuda.synchronize()
        if clk is not None and p == passes - 1:
            clk.mark(1)
        out += [a_.elapsed_time(b_) for a_, b_ in ev]
    return out


def bytes_per_token(w: syn.Workload) -> int:
    return {4: 324, 2: 196, 16: 1152}[w.content_bits]


def config_record(w: syn.Workload, lens, ms, peak, tpk, kind: str):
    """Measurements of one workload's decode step: times over all samples
    (median, p10, p90, mean), throughput and the roofline fraction of the bound
    that applies (tensor for packed caches read by 128 heads, else HBM)."""
    mean = sum(ms) / len(ms)
    by = algorithmic_bytes(w, lens)
    step_bytes = by["decode"] + by["writer"]
    gbs = step_bytes / (mean * 1e-3) / 1e9
    tf = algorithmic_flops(w, lens) / (mean * 1e-3) / 1e12
    tensor_bound = w.heads > 32 and w.content_bits != 16
    rec = {"workload": w.name, "batch": w.batch, "heads": w.heads,
           "layout": f"C{w.content_bits}R{w.rope_bits}" if w.content_bits != 16 else "bf16",
           "context": int(lens[0]) if len(set(int(x) for x in lens)) == 1 else "mixed",
           "writer_in_step": w.writer_in_step, "samples": len(ms),
           "step_us": {"mean": round(mean * 1e3, 2),
                       **{k: round(v * 1e3, 2) for k, v in percentiles(ms).items()}},
           "tokens_per_s": round(w.batch / (mean * 1e-3), 1),
           "kv_tokens_per_s": round(float(np.sum(lens)) / (mean * 1e-3), 1),
           "bytes_per_token": bytes_per_token(w),
           "packed_cache_gbs": round(gbs, 1), "hbm_frac": round(gbs / peak, 4),
           "tensor_tflops": round(tf, 2), "tensor_frac": round(tf / tpk, 4),
           "bound": "tensor" if tensor_bound else "hbm", "kernel": kind}
    # the same roofline object as the headline's, for this workload's bound
    trec = traffic_record(f"decode_{w.name}")
    rec["roofline"] = {
        "bound": rec["bound"], "kernel": kind,
        "achieved": round(tf, 2) if tensor_bound else round(gbs, 1),
        "peak": tpk if tensor_bound else peak,
        "unit": "TFLOP/s" if tensor_bound else "GB/s",
        "frac": rec["tensor_frac"] if tensor_bound else rec["hbm_frac"],
        "traffic": (trec or {}).get("dram_bytes_per_launch"),
        "traffic_source": (f"ncu capture: {trec.get('source')}" if trec else
                           "no ncu capture of the current kernel sources (null)")}
    return rec


def run_gpu(args, w):
    import torch
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    dev = f"cuda:{local}"
    torch.cuda.set_device(local)
    # this rank's shard of the global batch (world x the workload's batch):
    # every sequence of the global batch is decoded by exactly one rank
    ws_ = syn.shard_workload(w, rank, world)
    s = Setup(ws_, dev)
    stream = torch.cuda.current_stream()

    def barrier():
        if dist is not None:
            dist.barrier()

    passes = 2
    per_pass = max(1, args.steps // passes)
    clk = ClockSampler(local).__enter__()
    barrier()
    torch.cuda.synchronize()
    step_ms = time_steps(s, s.step, passes, per_pass, args.warmup, stream, clk)
    clk.__exit__(None, None, None)
    barrier()

    # ---- end to end through the public API with host buffers
    e2e_steps = min(len(step_ms), 200)
    for _ in range(2):
        s.step_e2e()
    torch.cuda.synchronize()
    ev2 = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(e2e_steps)]
    for i in range(e2e_steps):
        s.flush.zero_()
        ev2[i][0].record(stream)
        s.step_e2e()
        ev2[i][1].record(stream)
    torch.cuda.synchronize()
    e2e_ms = [a_.elapsed_time(b_) for a_, b_ in ev2]
    assert s.cache.error() == 0, f"device error word {s.cache.error()}"
    assert bool(torch.isfinite(s.out).all()), "non-finite output"

    t_step = sum(step_ms) / len(step_ms)
    t_e2e = sum(e2e_ms) / len(e2e_ms)
    t_step, t_e2e = reduce_max_over_ranks([t_step, t_e2e], dist, dev)
    B = ws_.batch
    tokens_per_s = whole_job_tokens_per_s(world, B, t_step)
    e2e_tokens_per_s = whole_job_tokens_per_s(world, B, t_e2e)
    peak, peak_kind = peaks()
    tpk, tpk_kind = tensor_peak()
    # split + combine; the library fuses the append into the split kernel for
    # packed caches whose rows are not a multiple of 128 (the 128-row kernel
    # and bf16 pages run the writer kernel first)
    fused = w.writer_in_step and w.content_bits != 16 and w.heads % 128 != 0
    n_launch_step = 2 + (1 if w.writer_in_step and not fused else 0)
    kernel_desc = ("append + decode (split kernel with fused append, combine)" if fused else
                   "writer + decode (split + combine)" if w.writer_in_step else
                   "decode (split + combine)")
    head = config_record(ws_, s.lens, step_ms, peak, tpk, kernel_desc)
    trec = traffic_record(f"decode_{w.name}")
    by = algorithmic_bytes(ws_, s.lens)
    step_bytes = by["decode"] + by["writer"]
    dec_gbs = step_bytes / (t_step * 1e-3) / 1e9
    dec_tflops = algorithmic_flops(ws_, s.lens) / (t_step * 1e-3) / 1e12
    tensor_bound = head["bound"] == "tensor"
    traffic = {"traffic": (trec or {}).get("dram_bytes_per_launch"),
               "traffic_source": (f"ncu capture: {trec.get('source')}" if trec else
                                  "no ncu capture of the current kernel sources (null)")}
    roofline = ({"bound": "tensor", "kernel": kernel_desc, "achieved": round(dec_tflops, 2),
                 "peak": tpk, "peak_source": f"{tpk_kind} bf16_tflops (fp16 runs at the same rate)",
                 "unit": "TFLOP/s", "frac": round(dec_tflops / tpk, 4),
                 "algorithmic_flops": algorithmic_flops(ws_, s.lens),
                 "hbm_frac": round(dec_gbs / peak, 4), **traffic}
                if tensor_bound else
                {"bound": "hbm", "kernel": kernel_desc, "achieved": round(dec_gbs, 1),
                 "peak": peak, "peak_source": f"{peak_kind} hbm_gbs", "unit": "GB/s",
                 "frac": round(dec_gbs / peak, 4), "algorithmic_bytes": step_bytes, **traffic})

    # ---- the other configurations of the same metric, one GPU (rank 0 alone)
    configs = {}
    if rank == 0 and world == 1 and not args.no_extra_configs:
        del s
        torch.cuda.empty_cache()
        for name in EXTRA_CONFIGS.get(w.name, ()):
            wx = syn.get(name)
            sx = Setup(wx, dev)
            fused_x = wx.writer_in_step and wx.content_bits != 16 and wx.heads % 128 != 0
            ms = time_steps(sx, sx.step, passes, max(1, args.extra_steps // passes),
                            args.warmup, stream)
            assert sx.cache.error() == 0, f"device error word {sx.cache.error()} ({name})"
            configs[name] = config_record(
                wx, sx.lens, ms, peak, tpk,
                ("append + decode" if fused_x else "writer + decode") if wx.writer_in_step
                else "decode")
            del sx
            torch.cuda.empty_cache()
        # the pages' comparison: packed against bf16 pages on the same values
        for packed, plain in (("long_c4r4", "long_bf16"), ("long16_c4r4", "long16_bf16")):
            recs = {**configs, w.name: head}
            if packed in recs and plain in recs:
                a_, b_ = recs[packed], recs[plain]
                L = 131072
                comp = (L * 1152) / ((L - 132) * 324 + 132 * 1152)
                configs[f"{packed}_vs_{plain}"] = {
                    "speedup": round(b_["step_us"]["mean"] / a_["step_us"]["mean"], 3),
                    "delta_pct_table9": round(100.0 * (a_["step_us"]["mean"] / b_["step_us"]["mean"] - 1), 1),
                    "bytes_per_token": [324, 1152],
                    "compression_closed_form_at_128k": round(comp, 3)}

    if rank == 0:
        line = {
            "metric": METRIC,
            "value": round(tokens_per_s, 1),
            "unit": "tokens/s",
            "n_gpus": world,
            "steps": len(step_ms),
            "warmup": args.warmup,
            "ms_per_step": round(t_step, 5),
            "higher_is_better": True,
            "scaling": "weak",
            "vs_baseline": None,
            "dtype": "f16-mma/f32 (int codes exact)",
            "data": "synthetic (seeded; workloads/synthetic.py)",
            "config": {"workload": w.name, "batch_per_gpu": B, "global_batch": B * world,
                       "heads": w.heads, "context": [int(x) for x in s_lens(ws_)][:8],
                       "layout": head["layout"], "page_tokens": 64,
                       "writer_in_step": w.writer_in_step,
                       "l2": f"flushed before every step ({L2_FLUSH_BYTES >> 20} MiB write)",
                       "sampling": f"{passes} independent passes x {per_pass} steps, each pass "
                                   f"after its own {args.warmup} warm-up steps",
                       "parallelism": f"sequence shards x{world} (no collective)"},
            "packed_cache_gbs": round(dec_gbs, 1),
            "hbm_frac": round(dec_gbs / peak, 4),
            "tensor_frac": round(dec_tflops / tpk, 4),
            "decode_us": round(t_step * 1e3, 2),
            "kv_tokens_per_s": round(world * float(np.sum(s_lens(ws_))) / (t_step * 1e-3), 1),
            "roofline": roofline,
            "step_us_percentiles": head["step_us"],
            "e2e": {"value": round(e2e_tokens_per_s, 1), "unit": "tokens/s",
                    "h2d_bytes_per_step": int(e2e_in_bytes(ws_)),
                    "d2h_bytes_per_step": int(ws_.batch * ws_.heads * 512 * 4)},
            "gpu_launches": n_launch_step * len(step_ms),
            "clocks": clk.summary(),
            "configs": configs,
        }
        if not args.no_cpu_baseline and world == 1:
            line["cpu_baseline"] = cpu_baseline(w, args.cpu_seconds)
        print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()


# the other workloads reported beside a headline workload (one GPU)
EXTRA_CONFIGS = {
    "long_c4r4": ("long_bf16", "long16_c4r4", "long16_bf16", "v2lite_c4r4"),
    "long16_c4r4": ("long16_bf16",),
    "v2lite_c4r4": (),
}


def s_lens(w: syn.Workload):
    return syn.sequence_lengths(w)


def e2e_in_bytes(w: syn.Workload) -> int:
    """Host-to-device bytes of one end-to-end step: q, plus the new tokens when
    the writer is in the step."""
    n = w.batch * w.heads * 576
    if w.writer_in_step:
        n += w.batch * (512 + 64)
    return 2 * n


# ---------------------------------------------------------------- the oracle arm

# heads of sequence 0 that one oracle step decodes (a bounded sample of the
# workload's step); the step counts as ORACLE_HEADS / heads of an output token
ORACLE_HEADS = 16
REFERENCE_SECONDS = 150.0   # cap on the reference arm's timed region


def _oracle_sample(w: syn.Workload):
    """Oracle state for sequence 0 of the workload (prefilled, not timed)."""
    import oracle
    lens = syn.sequence_lengths(w)
    table, npages = syn.make_paging(w)
    b = 0
    L = int(lens[b])
    ckv, kr = syn.sequence_tokens(w, b)
    lay = oracle.Layout(w.content_bits, w.rope_bits)
    model = oracle.PagedCacheModel(lay, npages, table)
    lens_after = np.zeros(w.batch, np.int64)
    lens_after[b] = L - 1
    model.write(np.full(L - 1, b), np.arange(L - 1), ckv[:L - 1], kr[:L - 1], lens_after)
    q = syn.queries(w, b)[0][:ORACLE_HEADS]
    return model, b, L, ckv[L - 1:L], kr[L - 1:L], q


def _oracle_step(w, model, b, L, ckv1, kr1, q):
    import oracle
    lens_after = np.zeros(w.batch, np.int64)
    lens_after[b] = L
    if w.writer_in_step:
        model.write([b], [L - 1], ckv1, kr1, lens_after)
    return oracle.mla_decode_fp64(q, model.effective_keys(b, L), w.softmax_scale)


def _sample_text(w, n, L, el):
    nh = min(ORACLE_HEADS, w.heads)
    return (f"{n} oracle steps of sequence 0 (L={L}, {nh} of {w.heads} heads per step = "
            f"{nh / w.heads:g} output token{', writer + ' if w.writer_in_step else ', '}"
            f"fp64 attention) of {w.name}, {el:.1f} s")


def cpu_baseline(w: syn.Workload, budget_s: float):
    """The oracle as it stands, timed on this host for a bounded sample of the
    workload's step, repeated until ``budget_s`` seconds; tokens/s = output
    tokens (the sampled fraction of each) / time."""
    model, b, L, ckv1, kr1, q = _oracle_sample(w)
    frac = min(ORACLE_HEADS, w.heads) / w.heads
    n, t0 = 0, time.perf_counter()
    while True:
        _oracle_step(w, model, b, L, ckv1, kr1, q)
        n += 1
        el = time.perf_counter() - t0
        if el >= budget_s:
            break
    return {"value": round(n * frac / el, 4), "unit": "tokens/s", "cores": os.cpu_count(),
            "kind": "oracle", "sample": _sample_text(w, n, L, el)}


def run_reference(args, w):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    model, b, L, ckv1, kr1, q = _oracle_sample(w)
    frac = min(ORACLE_HEADS, w.heads) / w.heads
    for _ in range(min(max(args.warmup, 0), 1)):
        _oracle_step(w, model, b, L, ckv1, kr1, q)
    n, t0 = 0, time.perf_counter()
    while n < args.steps:
        _oracle_step(w, model, b, L, ckv1, kr1, q)
        n += 1
        if time.perf_counter() - t0 > REFERENCE_SECONDS:
            break
    el = time.perf_counter() - t0
    value = n * frac / el
    world = int(os.environ.get("WORLD_SIZE", "1"))
    line = {
        "impl": "reference",
        "metric": METRIC, "value": round(value, 4), "unit": "tokens/s", "n_gpus": world,
        "steps": n, "warmup": args.warmup, "ms_per_step": round(el / n * 1e3, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded; workloads/synthetic.py)",
        "config": {"workload": w.name, "batch_per_gpu": w.batch, "heads": w.heads,
                   "sample": f"sequence 0, {min(ORACLE_HEADS, w.heads)} heads per step "
                             f"(CPU oracle; at most {REFERENCE_SECONDS:.0f} s of steps)"},
        "cpu_baseline": {"value": round(value, 4), "unit": "tokens/s", "cores": os.cpu_count(),
                         "kind": "oracle", "sample": _sample_text(w, n, L, el)},
        "e2e": {"value": round(value, 4), "unit": "tokens/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------- context sweep

TABLE9_CONTEXTS = (1024, 4096, 16384, 65536, 262144, 1048576)


def run_table9(args):
    """Decode latency against context length (QuantMLA, Table 9 caption and
    Figure 5b: latency from 1K to 1M context at batch 8 and 32, C4R4 against
    bf16 pages). One JSON line per (batch, context, layout); decode only (split
    + combine), L2 flushed before each timed call. The caches are filled
    through the library's writer from seeded device-generated tokens."""
    import torch
    import bit_mla_kv_lowbit_gb300 as pkg
    dev = "cuda:0"
    torch.cuda.set_device(0)
    heads = args.sweep_heads
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    peak, peak_kind = peaks()
    chunk = 1 << 18
    for B in (8, 32):
        for L in TABLE9_CONTEXTS:
            res = {}
            for cb in [c for c in (4, 16) if ("c4r4" if c == 4 else "bf16") in args.sweep_layouts]:
                w = syn.custom(f"t9_b{B}_l{L}_c{cb}", [L] * B, heads=heads, content_bits=cb,
                               rope_bits=4 if cb == 4 else 16, seed=9)
                table, npages = syn.make_paging(w)
                cache = pkg.PagedCache(cb, 4 if cb == 4 else 16, table, npages, dev)
                lens_after = torch.full((B,), L, dtype=torch.int32, device=dev)
                for b in range(B):
                    for p0 in range(0, L, chunk):
                        n = min(chunk, L - p0)
                        ckv, kr = syn.device_tokens(n, seed=1000 * b + p0 // chunk, device=dev,
                                                    start_pos=p0)
                        cache.write(ckv, kr, torch.arange(p0, p0 + n, dtype=torch.int32, device=dev),
                                    seq_idx=torch.full((n,), b, dtype=torch.int32, device=dev),
                                    seq_lens_after=lens_after)
                        del ckv, kr
                g = torch.Generator(device=dev)
                g.manual_seed(L + B)
                q = torch.randn(B, heads, 576, generator=g, device=dev).to(torch.bfloat16)
                out = torch.empty(B, heads, 512, dtype=torch.float32, device=dev)
                lens_h = [L] * B
                ws = cache.workspace(heads, lens_h)
                for _ in range(3):
                    cache.decode(q, lens_after, lens_h, w.softmax_scale, out=out, workspace=ws)
                torch.cuda.synchronize()
                ts = []
                for _ in range(args.sweep_reps):
                    flush.zero_()
                    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                    e0.record()
                    cache.decode(q, lens_after, lens_h, w.softmax_scale, out=out, workspace=ws)
                    e1.record()
                    torch.cuda.synchronize()
                    ts.append(e0.elapsed_time(e1) * 1e3)
                    # every call: a device-detected error (bad page, plan mismatch,
                    # a bounded wait that ran out) fails the sweep
                    err = cache.error()
                    assert err == 0, f"device error word {err} (B={B}, L={L}, {cb}-bit)"
                assert bool(torch.isfinite(out).all()), f"non-finite output (B={B}, L={L})"
                by = algorithmic_bytes(w, np.full(B, L))["decode"]
                med = sorted(ts)[len(ts) // 2]
                res[cb] = med
                print(json.dumps({
                    "sweep": "table9", "batch": B, "context": L, "heads": heads,
                    "layout": "C4R4" if cb == 4 else "bf16",
                    "decode_us": round(med, 2), **{k: round(v, 2) for k, v in
                                                   percentiles(ts).items()},
                    "algorithmic_bytes": by, "gbs": round(by / (med * 1e-6) / 1e9, 1),
                    "hbm_frac": round(by / (med * 1e-6) / 1e9 / peak, 4),
                    "peak_source": f"{peak_kind} hbm_gbs",
                    "c4r4_vs_bf16_pct": (round(100.0 * (res[4] - med) / med, 1)
                                         if cb == 16 and 4 in res else None),
                    # every call's time, so that runs in separate processes can be
                    # pooled (the Table 9 entries average 120 samples of two runs)
                    "samples_us": [round(t, 2) for t in ts]}), flush=True)
                del cache, ws, out, q
                torch.cuda.empty_cache()


def run_mtp(args):
    """Multi-token query decode: decode time for several causal queries per
    sequence over the same cache (the Group-Query Latent Attention abstract's
    s_q = 2 multi-token prediction step).  On the v2lite shape (B8 H16 L32768
    C4R4) 1, 2, 4 and 8 queries (8 queries of 16 heads are 128 rows, which the
    2-CTA tcgen05 kernel takes); on a 128-head shape (--sweep-workload v3_c4r4)
    1 and 2 queries (128 and 256 rows).  One JSON line per query count; L2
    flushed before each timed call."""
    import torch
    w = syn.get(args.sweep_workload)
    s = Setup(w, "cuda:0")
    peak, peak_kind = peaks()
    tpk, tpk_kind = tensor_peak()
    base = None
    for n in ((1, 2, 4, 8) if w.heads <= 16 else (1, 2)):
        g = torch.Generator(device="cuda")
        g.manual_seed(100 + n)
        q = torch.randn(w.batch, n, w.heads, 576, generator=g, device="cuda").to(torch.bfloat16)
        out = torch.empty(w.batch, n, w.heads, 512, dtype=torch.float32, device="cuda")
        ws = s.cache.workspace(n * w.heads, s.lens_h)
        for _ in range(3):
            s.cache.decode_multi(q, s.lens_d, s.lens_h, w.softmax_scale, out=out, workspace=ws)
        torch.cuda.synchronize()
        ts = []
        for _ in range(args.sweep_reps):
            s.flush.zero_()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            s.cache.decode_multi(q, s.lens_d, s.lens_h, w.softmax_scale, out=out, workspace=ws)
            e1.record()
            torch.cuda.synchronize()
            ts.append(e0.elapsed_time(e1) * 1e3)
        assert s.cache.error() == 0, f"device error word {s.cache.error()}"
        med = sorted(ts)[len(ts) // 2]
        base = base or med
        by = algorithmic_bytes(w.with_(heads=n * w.heads), s.lens)["decode"]
        fl = 2.0 * n * w.heads * (576 + 512) * float(np.sum(s.lens))
        print(json.dumps({"sweep": "mtp", "workload": w.name, "queries_per_seq": n,
                          "decode_us": round(med, 2), **{k: round(v, 2) for k, v in
                                                         percentiles(ts).items()},
                          "output_tokens_per_s": round(w.batch * n / (med * 1e-6), 1),
                          "time_vs_one_query": round(med / base, 3),
                          "hbm_frac": round(by / (med * 1e-6) / 1e9 / peak, 4),
                          "tensor_frac": round(fl / (med * 1e-6) / 1e12 / tpk, 4),
                          "peak_source": f"{peak_kind} hbm_gbs, {tpk_kind} bf16_tflops"}),
              flush=True)


def run_rotate(args):
    """Cost of the online Hadamard rotation: the write + decode step (one
    mla_lowbit_write_decode call) on the same workload with a plain and a
    rotated cache.  One JSON line per (workload, rotation); L2 flushed before
    each timed call."""
    import torch
    v2 = syn.get("v2lite_c4r4")
    for w in (v2, v2.with_(name="v2lite_c2r4", content_bits=2)):
        base = None
        for rot in (False, True):
            s = Setup(w, "cuda:0", rotate=rot)
            for _ in range(3):
                s.step()
            torch.cuda.synchronize()
            ts = []
            for _ in range(args.sweep_reps):
                s.flush.zero_()
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record()
                s.step()
                e1.record()
                torch.cuda.synchronize()
                ts.append(e0.elapsed_time(e1) * 1e3)
            assert s.cache.error() == 0, f"device error word {s.cache.error()}"
            med = sorted(ts)[len(ts) // 2]
            base = base or med
            print(json.dumps({"sweep": "rotate", "workload": w.name, "rotate": rot,
                              "step_us": round(med, 2),
                              **{k: round(v, 2) for k, v in percentiles(ts).items()},
                              "time_vs_plain": round(med / base, 3)}), flush=True)
            del s
            torch.cuda.empty_cache()


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=600,
                    help="timed steps of the headline workload, in two independent passes")
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--extra-steps", type=int, default=120,
                    help="timed steps of each other configuration in the line")
    ap.add_argument("--no-extra-configs", action="store_true")
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="long_c4r4", choices=sorted(syn.WORKLOADS))
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--sweep", choices=["table9", "mtp", "rotate"], default=None,
                    help="context-length sweep, multi-token query decode or the cost of the "
                         "online rotation, instead of the benchmark line")
    ap.add_argument("--sweep-heads", type=int, default=16)
    ap.add_argument("--sweep-workload", default="v2lite_c4r4", choices=sorted(syn.WORKLOADS),
                    help="workload of the multi-query sweep")
    ap.add_argument("--sweep-reps", type=int, default=15)
    ap.add_argument("--sweep-layouts", default="c4r4,bf16",
                    help="table9 sweep: comma-separated layouts to time (c4r4, bf16)")
    args = ap.parse_args()
    if args.sweep == "table9":
        run_table9(args)
        return
    if args.sweep == "mtp":
        run_mtp(args)
        return
    if args.sweep == "rotate":
        run_rotate(args)
        return
    w = syn.get(args.workload)
    if args.impl == "reference":
        run_reference(args, w)
    else:
        run_gpu(args, w)


if __name__ == "__main__":
    main()
